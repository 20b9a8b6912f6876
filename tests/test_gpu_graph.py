"""The library's calls are stream-ordered and allocate nothing, so a whole step
(metadata, forward, backward) can be captured into a CUDA graph and replayed:
the replay must equal the eager calls bit for bit, also after new inputs are
written into the captured buffers (the graph reads them at replay time)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
from workloads.device import DeviceWorkload, bf16_to_device  # noqa: E402
from workloads import make_workload  # noqa: E402

pytestmark = pytest.mark.gpu


def _buffers(wl, dw, meta):
    dev = dw.q.device
    sq, _ = dw.seqlens()
    return dict(out=torch.empty(dw.q.shape, dtype=torch.float32, device=dev),
                lse=torch.empty((wl.B, wl.H, sq), dtype=torch.float32, device=dev),
                dq=torch.empty(dw.q.shape, dtype=torch.float32, device=dev),
                dk=torch.empty(dw.k.shape, dtype=torch.float32, device=dev),
                dv=torch.empty(dw.v.shape, dtype=torch.float32, device=dev),
                ws=bsa.alloc_workspace(meta, dev),
                wsb=torch.empty(bsa.bsattn_bwd_workspace_size(meta), dtype=torch.uint8, device=dev),
                err=torch.zeros(1, dtype=torch.int32, device=dev))


def _step(wl, dw, meta, dout, b):
    """Metadata, forward and backward on the current stream, into preallocated buffers."""
    stream = torch.cuda.current_stream()
    sq, sk = dw.seqlens()
    dw.build_meta(meta, err_flag=b["err"], stream=stream)
    dw.forward(meta, out=b["out"], lse=b["lse"], err_flag=b["err"], workspace=b["ws"], stream=stream)
    st = bsa.bsattn_bwd(dw.q, dw.k, dw.v, b["out"], bsa.OUT_F32, b["lse"], dout, wl.B, sq, sk, wl.H,
                        wl.D, None, None, meta, dw.vl, wl.kind, dw.mask_params, wl.scale, b["dq"],
                        b["dk"], b["dv"], bsa.OUT_F32, b["wsb"], err_flag=b["err"], stream=stream)
    assert st == bsa.BSATTN_OK


def _snapshot(b):
    return {k: b[k].clone() for k in ("out", "lse", "dq", "dk", "dv")}


def _spoil(b):
    for k in ("out", "lse", "dq", "dk", "dv"):
        b[k].fill_(float("nan"))


def test_captured_step_replays_bitwise():
    wl = make_workload(2)  # B 2, H 4, S 1024, d 128, random map, causal
    dw = DeviceWorkload(wl, "cuda")
    meta = dw.alloc_meta()
    dout = bf16_to_device(wl.tensor("do"), "cuda")
    b = _buffers(wl, dw, meta)
    _step(wl, dw, meta, dout, b)          # eager (also sets the kernels' attributes)
    torch.cuda.synchronize()
    eager = _snapshot(b)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(wl, dw, meta, dout, b)      # warm-up on a side stream before capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(wl, dw, meta, dout, b)
    _spoil(b)
    graph.replay()
    torch.cuda.synchronize()
    assert int(b["err"].item()) == 0
    for k, v in eager.items():
        assert torch.equal(b[k], v), k
    # new inputs in the same buffers: the replay computes on them
    gen = torch.Generator(device="cuda").manual_seed(7)
    dw.q.copy_(torch.randn(dw.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
    _step(wl, dw, meta, dout, b)
    torch.cuda.synchronize()
    eager2 = _snapshot(b)
    assert not torch.equal(eager2["out"], eager["out"])
    _spoil(b)
    graph.replay()
    torch.cuda.synchronize()
    for k, v in eager2.items():
        assert torch.equal(b[k], v), k


def test_captured_static_scratch_forward():
    wl = make_workload(4)
    from workloads.configs import with_heads
    wl = with_heads(wl, 2)
    dw = DeviceWorkload(wl, "cuda")
    meta = dw.build_meta()
    sq, sk = dw.seqlens()
    out = torch.empty(dw.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.B, wl.H, sq), dtype=torch.float32, device="cuda")

    def fwd():
        st = bsa.bsattn_fwd_static_scratch(dw.q, dw.k, dw.v, wl.B, sq, sk, wl.H, wl.D, None, None,
                                           meta, dw.vl, wl.kind, dw.mask_params, wl.scale, out,
                                           bsa.OUT_BF16, lse, stream=torch.cuda.current_stream())
        assert st == bsa.BSATTN_OK

    fwd()  # the first call resolves the scratch address, outside any capture
    torch.cuda.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fwd()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd()
    out.zero_()
    lse.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    assert np.isfinite(lse.cpu().numpy()).all()
