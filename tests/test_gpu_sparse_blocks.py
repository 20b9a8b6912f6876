"""The forward over lists per sparse block ("[CuTe,Flex] varlen blocksparsity",
flash-attention #2224: block-sparse tensors per q_subtile_factor x tile_m
sparse block; "[feat] VSA-256 fastpath on Blackwell via FA4 CuTe block-sparse
attention", FastVideo #1354: 256-token blocks): metadata with tile_m = 256 and
tile_n = 256 or 128, which the metadata kernel classifies per block and the
forward walks directly (one list entry, its KV tiles as consecutive items).

- K-META at block granularity against the oracle's lists for the same block
  size: bit for bit.
- The forward against the oracle on the same block-granular workload: O within
  5e-3 and LSE within 1e-3 max abs on the fp32 output, bf16 = RNE(fp32).
- Config 4 at VSA's native 256-token blocks against the per-tile forward of the
  expanded map: every output bit equal (same tiles, same order, same
  arithmetic), and sampled rows against the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads import make_workload  # noqa: E402
from workloads.configs import (MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE, MASK_PREFIX,  # noqa: E402
                               MASK_SLIDING_WINDOW, as_sparse_blocks, random_workload)
from workloads.device import DeviceWorkload, meta_to_numpy  # noqa: E402

pytestmark = pytest.mark.gpu

KEYS = ("full_cnt", "full_idx", "mask_cnt", "mask_idx")

CASES = {
    "none_valid_256x256": dict(seed=251, B=2, H=2, D=128, seqlens_q=[700, 700], kind=MASK_NONE,
                               valid_len=True, tile_m=256, tile_n=256),
    "causal_256x256": dict(seed=252, B=1, H=3, D=64, seqlens_q=[1024], kind=MASK_CAUSAL,
                           tile_m=256, tile_n=256),
    "window_256x128": dict(seed=253, B=1, H=2, D=128, seqlens_q=[1000], kind=MASK_SLIDING_WINDOW,
                           window_left=300, sink_tokens=100, tile_m=256, tile_n=128),
    "prefix_256x256": dict(seed=254, B=2, H=2, D=128, seqlens_q=[512, 512], seqlens_k=[900, 900],
                           kind=MASK_PREFIX, prefix_len=300, tile_m=256, tile_n=256),
    "document_256x128": dict(seed=255, B=1, H=2, D=64, seqlens_q=[768], kind=MASK_DOCUMENT,
                             n_docs=4, tile_m=256, tile_n=128),
    "empty_256x256": dict(seed=256, B=1, H=2, D=128, seqlens_q=[512], kind=MASK_NONE, density=0.0,
                          force_diag=False, tile_m=256, tile_n=256),
    "ragged_none_256x256": dict(seed=257, B=1, H=2, D=128, seqlens_q=[400], seqlens_k=[1100],
                                kind=MASK_NONE, valid_len=True, density=0.7, tile_m=256,
                                tile_n=256),
}


def _run(wl, q, k, v):
    dw = DeviceWorkload(wl, "cuda", qkv=(q, k, v))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    out32, lse = dw.forward(meta, err_flag=err, out_dtype=torch.float32)
    out16, lse16 = dw.forward(meta, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out16.view(torch.int16), out32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lse, lse16)
    return meta, out32, lse


def _check_rows(got_o, got_l, ref_o, ref_l):
    assert np.max(np.abs(got_o - ref_o), initial=0.0) <= 5e-3
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(got_l), fin)
    assert np.all(got_l[~fin] == -np.inf)
    assert np.max(np.abs(got_l[fin] - ref_l[fin]), initial=0.0) <= 1e-3


@pytest.mark.parametrize("name", list(CASES))
def test_block_lists_match_the_oracle(name):
    wl = random_workload(**CASES[name])
    q, k, v = wl.qkv()
    meta, out, lse = _run(wl, q, k, v)
    ref_meta = oracle.build_meta(wl)
    got = meta_to_numpy(meta)
    for key in KEYS:
        assert np.array_equal(got[key], ref_meta[key]), key
    ref_o, ref_l = oracle.fwd(wl, q, k, v, ref_meta)
    _check_rows(out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                ref_o, ref_l)


def test_vsa_native_blocks_equal_the_per_tile_forward():
    wl = make_workload(4)
    w2 = as_sparse_blocks(wl)
    q, k, v = wl.qkv()
    meta2, out2, lse2 = _run(w2, q, k, v)
    ref_meta2 = oracle.build_meta(w2)
    got = meta_to_numpy(meta2)
    for key in KEYS:
        assert np.array_equal(got[key], ref_meta2[key]), key
    meta1, out1, lse1 = _run(wl, q, k, v)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    # and against the oracle's own block-granular definition on sampled rows
    rng = np.random.default_rng(4)
    S = int(wl.seqlens_q[0])
    tok = np.concatenate([rng.integers(0, S, 200), [0, 127, 128, 255, S - 1]]).astype(np.int32)
    head = rng.integers(0, wl.H, tok.size).astype(np.int32)
    ref_o, ref_l = oracle.fwd_rows(w2, q, k, v, ref_meta2, tok, head)
    o = out2.cpu().numpy().astype(np.float64).reshape(S, wl.H, wl.D)[tok, head]
    l = lse2.cpu().numpy().astype(np.float64).reshape(wl.H, S)[head, tok]
    _check_rows(o, l, ref_o, ref_l)
