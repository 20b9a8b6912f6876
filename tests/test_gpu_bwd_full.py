"""Backward at the benchmark workloads' full sizes, in the launch configuration
bench.py times (bf16 forward output, bf16 gradients), against the oracle.

The batched random workload (B 2, H 4, S 1024) and the varlen workload (8
sequences of 100-4096 tokens, H 16) are compared element by element with the
dense fp64 backward (per sequence for varlen).  The VSA (H 24, S 61440) and
long-context (H 32, S 131072) workloads are compared on every row of their
first and last heads (dQ, dK, dV of the whole head, by the oracle's per-head
backward, which walks the head's Q tiles) and on sampled Q tiles (dQ rows) and
KV tiles (dK, dV rows) of random heads.  Tolerance as in test_gpu_bwd.py, per
compared tensor: max |G - G_ref| <= 2e-2 max |G_ref| and
||G - G_ref||_F <= 1e-2 ||G_ref||_F."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads.device import DeviceWorkload, bf16_to_device  # noqa: E402
from workloads import make_workload  # noqa: E402

pytestmark = pytest.mark.gpu

MAX_TOL, FRO_TOL = 2e-2, 1e-2


def _run(wl):
    q, k, v = wl.qkv()
    g = wl.tensor("do")
    dw = DeviceWorkload(wl, "cuda", qkv=(q, k, v))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    out, lse = dw.forward(meta, err_flag=err)
    grads = bsa.backward(dw.q, dw.k, dw.v, out, lse, bf16_to_device(g, "cuda"), meta,
                         cu_seqlens_q=dw.cu_q, cu_seqlens_k=dw.cu_k, kv_valid_len=dw.vl,
                         kind=wl.kind, mask_params=dw.mask_params, softmax_scale=wl.scale,
                         err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    host = [t.float().cpu().numpy().astype(np.float64) for t in grads]
    del grads, out, lse, dw
    torch.cuda.empty_cache()
    return (q, k, v, g), host


def _close(got, ref, what):
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    assert float(np.max(np.abs(got - ref))) <= MAX_TOL * scale, what
    assert float(np.linalg.norm(got - ref)) <= FRO_TOL * max(float(np.linalg.norm(ref)), 1e-30), what


def test_bwd_batched_random_workload_elementwise():
    wl = make_workload(2)
    (q, k, v, g), (dq, dk, dv) = _run(wl)
    ref = oracle.bwd(wl, q, k, v, oracle.build_meta(wl), g)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        _close(got, r, name)


@pytest.mark.parametrize("cfg", [4, 5])
def test_bwd_full_size_whole_heads_and_sampled_tiles(cfg):
    wl = make_workload(cfg)
    (q, k, v, g), (dq, dk, dv) = _run(wl)
    assert all(np.all(np.isfinite(t)) for t in (dq, dk, dv))
    meta = oracle.build_meta(wl)
    rng = np.random.default_rng(700 + cfg)
    b = 0
    # Q tiles: three random ones and the last one of the last head
    tiles = [(int(rng.integers(wl.H)), int(rng.integers(wl.num_m))) for _ in range(3)]
    tiles.append((wl.H - 1, wl.num_m - 1))
    for h, m in tiles:
        ref = oracle.bwd_dq_tile(wl, q, k, v, g, meta, b, h, m)
        r0 = m * wl.tile_m
        _close(dq[b, r0:r0 + ref.shape[0], h], ref, f"dq h={h} m={m}")
    # KV tiles: two random ones past the first four (on the long-context map every
    # Q tile names those, which the per-tile oracle would walk one by one) and the last
    kv = [(int(rng.integers(wl.H)), int(rng.integers(4, wl.num_n))) for _ in range(2)]
    kv.append((wl.H - 1, wl.num_n - 1))
    for h, n in kv:
        rk, rv = oracle.bwd_dkdv_tile(wl, q, k, v, g, meta, b, h, n)
        c0 = n * wl.tile_n
        _close(dk[b, c0:c0 + rk.shape[0], h], rk, f"dk h={h} n={n}")
        _close(dv[b, c0:c0 + rv.shape[0], h], rv, f"dv h={h} n={n}")
    # whole heads: the first and the last, every row of dQ, dK and dV
    for h in (0, wl.H - 1):
        hq, hk, hv = oracle.bwd_head(wl, q, k, v, g, meta, b, h)
        _close(dq[b, :, h], hq, f"dq head {h}")
        _close(dk[b, :, h], hk, f"dk head {h}")
        _close(dv[b, :, h], hv, f"dv head {h}")


def test_bwd_varlen_workload_elementwise():
    wl = make_workload(3)
    (q, k, v, g), (dq, dk, dv) = _run(wl)
    ref = oracle.bwd(wl, q, k, v, oracle.build_meta(wl), g)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        _close(got, r, name)
