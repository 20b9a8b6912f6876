"""The fixed-scratch forward (bsattn_fwd_static_scratch), for callers that
cannot allocate device memory at call time, against the forward with a caller
workspace (same inputs, two calls in a row, results equal) and against the
oracle (O within 5e-3, LSE within 1e-3 max abs).  Calls after the first on a
device must leave the device's free memory unchanged: the entry point allocates
nothing.

Named to be collected last, so it also runs after every other GPU test in the
same process; it must pass alone in a fresh process as well."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads.device import DeviceWorkload  # noqa: E402
from workloads import make_workload  # noqa: E402
from workloads.configs import random_workload  # noqa: E402

pytestmark = pytest.mark.gpu


def _cases():
    return [make_workload(1), make_workload(3),
            random_workload(7, B=2, H=3, D=128, seqlens_q=[700, 700], kind=bsa.MASK_SLIDING_WINDOW,
                            window_left=300, sink_tokens=64)]


@pytest.mark.parametrize("idx", [0, 1, 2])
@pytest.mark.parametrize("out_dtype", [bsa.OUT_F32, bsa.OUT_BF16])
def test_static_scratch_matches_workspace_forward(idx, out_dtype):
    wl = _cases()[idx]
    dw = DeviceWorkload(wl, "cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    meta = dw.build_meta(err_flag=err)
    tdt = torch.float32 if out_dtype == bsa.OUT_F32 else torch.bfloat16
    ref_out, ref_lse = dw.forward(meta, err_flag=err, out_dtype=tdt)   # caller workspace
    torch.cuda.synchronize()
    sq, sk = dw.seqlens()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = bsa.bsattn_fwd_static_scratch(
            dw.q, dw.k, dw.v, wl.B, sq, sk, wl.H, wl.D, dw.cu_q, dw.cu_k, meta, dw.vl, wl.kind,
            dw.mask_params, wl.scale, out, out_dtype, lse, err_flag=err, stream=stream)
        assert st == bsa.BSATTN_OK, bsa.status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        # same kernel and per-unit arithmetic: equal within a zero tolerance
        assert torch.equal(out, ref_out), f"call {call}: output differs"
        assert torch.equal(lse, ref_lse), f"call {call}: LSE differs"


@pytest.mark.parametrize("cfg", [1, 3])
def test_static_scratch_matches_the_oracle_and_allocates_nothing(cfg):
    wl = make_workload(cfg)
    q, k, v = wl.qkv()
    dw = DeviceWorkload(wl, "cuda:0", qkv=(q, k, v))
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    meta = dw.build_meta(err_flag=err)
    sq, sk = dw.seqlens()
    stream = torch.cuda.current_stream().cuda_stream
    outs = [torch.empty(dw.q.shape, dtype=torch.float32, device="cuda:0") for _ in range(3)]
    lse_shape = (wl.H, wl.rows_q) if wl.varlen else (wl.B, wl.H, sq)
    lses = [torch.empty(lse_shape, dtype=torch.float32, device="cuda:0") for _ in range(3)]
    torch.cuda.synchronize()
    free = []
    for call in range(3):
        st = bsa.bsattn_fwd_static_scratch(
            dw.q, dw.k, dw.v, wl.B, sq, sk, wl.H, wl.D, dw.cu_q, dw.cu_k, meta, dw.vl, wl.kind,
            dw.mask_params, wl.scale, outs[call], bsa.OUT_F32, lses[call], err_flag=err,
            stream=stream)
        assert st == bsa.BSATTN_OK, bsa.status_string(st)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    assert int(err.item()) == 0
    # the first call may load the library's device data; later calls allocate nothing
    assert free[1] == free[2], f"free device memory changed: {free}"
    ref_o, ref_l = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    fin = np.isfinite(ref_l)
    for call in (1, 2):
        o = outs[call].cpu().numpy().astype(np.float64)
        lse = lses[call].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(o - ref_o)) <= 5e-3
        assert np.array_equal(np.isfinite(lse), fin)
        assert np.max(np.abs(lse[fin] - ref_l[fin])) <= 1e-3
