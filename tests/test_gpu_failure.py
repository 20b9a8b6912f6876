"""Device-side failure handling of the forward, without a GPU fault.

- Varlen offsets that reach past the packed rows: the sequence is skipped and
  BSATTN_FLAG_BAD_SEQLENS is set.  The output and LSE buffers carry 128 spare
  rows past the sizes given to the call, so that even a kernel without the
  guard would store into memory this test owns, never past an allocation.
- A pipeline wait that runs out: the wait limit is lowered through the testing
  hook so that waits of an ordinary launch expire (no signal is removed).  The
  call must return with BSATTN_FLAG_TIMEOUT set, and the next call on the same
  stream, at the default limit, must give exactly a fresh run's result.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads import make_workload  # noqa: E402
from workloads.configs import MASK_CAUSAL, random_workload  # noqa: E402
from workloads.device import DeviceWorkload  # noqa: E402

pytestmark = pytest.mark.gpu

SPARE = 128
SENTINEL = 7.0


def test_varlen_offsets_past_the_packed_rows_are_skipped_and_flagged():
    wl = random_workload(241, B=3, H=2, D=128, seqlens_q=[200, 300, 150], varlen=True,
                         kind=MASK_CAUSAL, density=0.7)
    q, k, v = wl.qkv()
    dw = DeviceWorkload(wl, "cuda", qkv=(q, k, v))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows_q, rows_k = wl.rows_q, wl.rows_k
    cu_bad = dw.cu_q.clone()
    cu_bad[wl.B] = rows_q + 64            # the last sequence now ends past the packed rows
    out = torch.full((rows_q + SPARE, wl.H, wl.D), SENTINEL, dtype=torch.float32, device="cuda")
    lse = torch.full((wl.H * rows_q + SPARE,), SENTINEL, dtype=torch.float32, device="cuda")
    st = bsa.bsattn_fwd(dw.q, dw.k, dw.v, wl.B, rows_q, rows_k, wl.H, wl.D, cu_bad, dw.cu_k, meta,
                        dw.vl, wl.kind, dw.mask_params, wl.scale, out, bsa.OUT_F32, lse,
                        err_flag=err)
    assert st == bsa.BSATTN_OK, bsa.status_string(st)
    torch.cuda.synchronize()
    assert int(err.item()) & bsa.FLAG_BAD_SEQLENS
    o = out.cpu().numpy().astype(np.float64)
    lse_np = lse.cpu().numpy().astype(np.float64)
    last = int(wl.cu_seqlens_q[wl.B - 1])
    # the spare rows and every row of the skipped sequence keep the sentinel
    assert np.all(o[last:] == SENTINEL)
    assert np.all(lse_np[wl.H * rows_q:] == SENTINEL)
    l2 = lse_np[:wl.H * rows_q].reshape(wl.H, rows_q)
    assert np.all(l2[:, last:] == SENTINEL)
    # the other sequences are computed as usual
    ref_o, ref_l = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    assert np.max(np.abs(o[:last] - ref_o[:last])) <= 5e-3
    fin = np.isfinite(ref_l[:, :last])
    assert np.array_equal(np.isfinite(l2[:, :last]), fin)
    assert np.max(np.abs(l2[:, :last][fin] - ref_l[:, :last][fin])) <= 1e-3


@pytest.mark.parametrize("workspace", ["auto", None])
def test_expired_wait_sets_timeout_and_the_next_call_is_exact(workspace):
    wl = make_workload(2)
    dw = DeviceWorkload(wl, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    ref_o, ref_l = dw.forward(meta, err_flag=err, out_dtype=torch.float32, workspace=workspace)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # 1,000 cycles: far shorter than a K/V tile load, so waits of this launch expire
    bsa.bsattn_testing_set_wait_limit(1000)
    try:
        t0 = time.perf_counter()
        out, lse = dw.forward(meta, err_flag=err, out_dtype=torch.float32, workspace=workspace)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        bsa.bsattn_testing_set_wait_limit(0)
    assert int(err.item()) & bsa.FLAG_TIMEOUT
    # the aborting CTAs drain what they issued and exit promptly (no wait runs
    # to the one-second default limit)
    assert elapsed < 0.5, f"aborted launch took {elapsed:.3f} s"
    err.zero_()
    out2, lse2 = dw.forward(meta, err_flag=err, out_dtype=torch.float32, workspace=workspace)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out2, ref_o) and torch.equal(lse2, ref_l)
