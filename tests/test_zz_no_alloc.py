"""The fixed-scratch forward (bsattn_fwd_static_scratch) against the forward
with a caller workspace: same inputs, two calls in a row, results equal.

Named to be collected last, so it also runs after every other GPU test in the
same process; it must pass alone in a fresh process as well."""
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
from tests.gpu_run import DeviceWorkload  # noqa: E402
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
