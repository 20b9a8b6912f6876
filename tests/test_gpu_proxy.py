"""Proxy-compensated forward ("feat(prims-ts): support proxy-compensated
block-sparse attention", FlashInfer #4872) and the KV summaries against the
oracle: O within 5e-3 and LSE within 1e-3 of the fp64 definition fed the same
bf16 summaries; summaries within one bf16 ulp of the fp64 mean / sum; with every
tile selected the proxy forward equals the exact forward bit for bit.  At full
size, on the video sparse attention map (B 1, H 24, S 61440, mask kind none, as
bench.py's proxy A/B runs it), every row of the last head and 400 random rows
are compared with the oracle's per-row form, and the bf16 output is RNE of the
fp32 one everywhere."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads.device import DeviceWorkload  # noqa: E402
from workloads.configs import MASK_NONE, random_workload  # noqa: E402
from workloads.formats import to_bitmask  # noqa: E402

pytestmark = pytest.mark.gpu

CASES = [
    dict(seed=91, B=1, H=2, D=64, sq=256, sk=300, density=0.5),
    dict(seed=92, B=2, H=2, D=128, sq=384, sk=1000, density=0.3),     # pairs straddle sequences
    dict(seed=93, B=1, H=3, D=128, sq=300, sk=640, density=0.0),      # every tile a proxy
    dict(seed=94, B=1, H=1, D=64, sq=256, sk=20000, density=0.05),    # 157 tiles: two chunks
    dict(seed=95, B=1, H=2, D=128, sq=512, sk=512, density=0.6),
]


def _setup(c):
    wl = random_workload(c["seed"], B=c["B"], H=c["H"], D=c["D"], seqlens_q=[c["sq"]] * c["B"],
                         seqlens_k=[c["sk"]] * c["B"], kind=MASK_NONE, density=c["density"],
                         force_diag=c["density"] > 0)
    dw = DeviceWorkload(wl, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    nn = math.ceil(c["sk"] / 128)
    ks = torch.empty((c["B"], nn, c["H"], c["D"]), dtype=torch.bfloat16, device="cuda")
    vs = torch.empty_like(ks)
    stream = torch.cuda.current_stream().cuda_stream
    st = bsa.bsattn_kv_summaries(dw.k, dw.v, c["B"], c["sk"], c["H"], c["D"], ks, vs, stream)
    assert st == bsa.BSATTN_OK, bsa.status_string(st)
    words, W = to_bitmask(wl, wl.block_map)
    d_words = torch.from_numpy(words.view(np.int32)).to("cuda")
    return wl, dw, err, meta, ks, vs, d_words, W


def _proxy(wl, dw, err, meta, ks, vs, d_words, W, out_dtype=torch.float32):
    sq, sk = dw.seqlens()
    out = torch.empty(dw.q.shape, dtype=out_dtype, device="cuda")
    lse = torch.empty((wl.B, wl.H, sq), dtype=torch.float32, device="cuda")
    ws = bsa.alloc_workspace(meta)
    st = bsa.bsattn_fwd_proxy(dw.q, dw.k, dw.v, wl.B, sq, sk, wl.H, wl.D, meta, d_words, W, ks, vs,
                              wl.scale, out, bsa.OUT_F32 if out_dtype == torch.float32 else bsa.OUT_BF16,
                              lse, workspace=ws, err_flag=err,
                              stream=torch.cuda.current_stream().cuda_stream)
    assert st == bsa.BSATTN_OK, bsa.status_string(st)
    torch.cuda.synchronize()
    return out, lse


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_summaries_match_oracle(idx):
    wl, dw, err, meta, ks, vs, _, _ = _setup(CASES[idx])
    torch.cuda.synchronize()
    q, k, v = wl.qkv()
    km, vsum = oracle.kv_summaries(wl, k, v)
    for got, ref in ((ks, km), (vs, vsum)):
        g = got.float().cpu().numpy().astype(np.float64)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
        assert np.all(np.abs(g - ref) <= ulp + 1e-6)


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_proxy_forward_matches_oracle(idx):
    wl, dw, err, meta, ks, vs, d_words, W = _setup(CASES[idx])
    out, lse = _proxy(wl, dw, err, meta, ks, vs, d_words, W)
    assert int(err.item()) == 0
    q, k, v = wl.qkv()
    o_ref, l_ref = oracle.fwd_proxy(wl, q, k, v, _bits(ks), _bits(vs), wl.block_map)
    e_o = np.max(np.abs(out.cpu().numpy().astype(np.float64) - o_ref))
    e_l = np.max(np.abs(lse.cpu().numpy().astype(np.float64) - l_ref))
    assert e_o <= 5e-3 and e_l <= 1e-3, (e_o, e_l)
    out16, lse16 = _proxy(wl, dw, err, meta, ks, vs, d_words, W, out_dtype=torch.bfloat16)
    assert torch.equal(out16.view(torch.int16), out.to(torch.bfloat16).view(torch.int16))


def test_proxy_with_every_tile_selected_equals_exact_forward():
    c = dict(seed=96, B=1, H=2, D=128, sq=384, sk=700, density=1.0)
    wl, dw, err, meta, ks, vs, d_words, W = _setup(c)
    out, lse = _proxy(wl, dw, err, meta, ks, vs, d_words, W)
    out_e, lse_e = dw.forward(meta, err_flag=err, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, out_e) and torch.equal(lse, lse_e)


def test_proxy_forward_full_size_on_the_benchmark_map():
    from workloads import make_workload
    from workloads.device import DeviceWorkload as DW
    wl = make_workload(4)
    q, k, v = wl.qkv()
    dw = DW(wl, "cuda", qkv=(q, k, v))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sq, sk = dw.seqlens()
    meta = dw.alloc_meta()
    stream = torch.cuda.current_stream().cuda_stream
    st = bsa.bsattn_build_meta(dw.block_map, None, None, sq, sk, None, bsa.MASK_NONE, None, meta, err, stream)
    assert st == bsa.BSATTN_OK, bsa.status_string(st)
    nn = math.ceil(sk / 128)
    ks = torch.empty((wl.B, nn, wl.H, wl.D), dtype=torch.bfloat16, device="cuda")
    vs = torch.empty_like(ks)
    st = bsa.bsattn_kv_summaries(dw.k, dw.v, wl.B, sk, wl.H, wl.D, ks, vs, stream)
    assert st == bsa.BSATTN_OK, bsa.status_string(st)
    words, W = to_bitmask(wl, wl.block_map)
    d_words = torch.from_numpy(words.view(np.int32)).to("cuda")
    out, lse = _proxy(wl, dw, err, meta, ks, vs, d_words, W)
    out16, _ = _proxy(wl, dw, err, meta, ks, vs, d_words, W, out_dtype=torch.bfloat16)
    assert int(err.item()) == 0
    assert torch.equal(out16.view(torch.int16), out.to(torch.bfloat16).view(torch.int16))
    o = out.cpu().numpy()[0]            # [S, H, D]
    l = lse.cpu().numpy()[0]            # [H, S]
    rng = np.random.default_rng(404)
    tok = np.concatenate([np.arange(sq), rng.integers(0, sq, 400)])
    head = np.concatenate([np.full(sq, wl.H - 1), rng.integers(0, wl.H, 400)])
    o_ref, l_ref = oracle.fwd_proxy_rows(wl, q, k, v, _bits(ks), _bits(vs), wl.block_map, tok, head)
    e_o = float(np.max(np.abs(o[tok, head].astype(np.float64) - o_ref)))
    e_l = float(np.max(np.abs(l[head, tok].astype(np.float64) - l_ref)))
    assert e_o <= 5e-3 and e_l <= 1e-3, (e_o, e_l)
