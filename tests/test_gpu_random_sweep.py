"""A seeded sweep over random problem shapes, forward and backward against the
oracle: batch or varlen packing, 1-3 heads, d 64 or 128, sequence lengths from
1 to 700 (keys possibly longer or shorter than queries), every mask kind with
random window, sink and prefix lengths, random per-KV-tile valid lengths, and
block densities from empty to full.  Tolerances are those of the forward and
backward parity tests: O within 5e-3 and LSE within 1e-3 max abs (fp32 output),
identical empty rows, and each gradient within 2e-2 of its largest reference
value (plus 1e-4)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads.configs import (MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE, MASK_PREFIX,  # noqa: E402
                               MASK_SLIDING_WINDOW, random_workload)
from workloads.device import DeviceWorkload, bf16_to_device  # noqa: E402

pytestmark = pytest.mark.gpu

KINDS = (MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT, MASK_PREFIX)


def _case(i):
    rng = np.random.default_rng(9000 + i)
    varlen = bool(rng.integers(0, 2))
    B = int(rng.integers(1, 4))
    H = int(rng.integers(1, 4))
    D = int(rng.choice([64, 128]))
    kind = int(KINDS[i % len(KINDS)])
    if varlen:
        sq = [int(x) for x in rng.integers(1, 701, B)]
        sk = sq if kind != MASK_NONE else [int(x) for x in rng.integers(1, 701, B)]
    else:
        sq = [int(rng.integers(1, 701))] * B
        sk = sq if kind != MASK_NONE else [int(rng.integers(1, 701))] * B
    return dict(seed=9100 + i, B=B, H=H, D=D, seqlens_q=sq, seqlens_k=sk, varlen=varlen, kind=kind,
                density=float(rng.choice([0.0, 0.3, 0.7, 1.0])), window_left=int(rng.integers(1, 400)),
                sink_tokens=int(rng.integers(0, 150)), prefix_len=int(rng.integers(0, 500)),
                valid_len=bool(rng.integers(0, 2)), n_docs=int(rng.integers(1, 5)),
                force_diag=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("i", range(48))
def test_random_problem_matches_the_oracle(i):
    c = _case(i)
    wl = random_workload(**c)
    q, k, v = wl.qkv()
    g_bits = wl.tensor("do")
    dw = DeviceWorkload(wl, "cuda", qkv=(q, k, v))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    out, lse = dw.forward(meta, err_flag=err, out_dtype=torch.float32)
    grads = bsa.backward(dw.q, dw.k, dw.v, out, lse, bf16_to_device(g_bits, "cuda"), meta,
                         cu_seqlens_q=dw.cu_q, cu_seqlens_k=dw.cu_k, kv_valid_len=dw.vl,
                         kind=wl.kind, mask_params=dw.mask_params, softmax_scale=wl.scale,
                         grad_dtype=torch.float32, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, c
    ref_meta = oracle.build_meta(wl)
    o_ref, l_ref = oracle.fwd(wl, q, k, v, ref_meta)
    o = out.cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(o - o_ref), initial=0.0) <= 5e-3, c
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(l), fin), c
    assert np.all(l[~fin] == -np.inf)
    assert np.max(np.abs(l[fin] - l_ref[fin]), initial=0.0) <= 1e-3, c
    refs = oracle.bwd(wl, q, k, v, ref_meta, g_bits)
    for got, ref in zip(grads, refs):
        got = got.cpu().numpy().astype(np.float64)
        scale = float(np.max(np.abs(ref), initial=0.0))
        assert np.max(np.abs(got - ref), initial=0.0) <= 2e-2 * scale + 1e-4, c
