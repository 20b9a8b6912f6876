"""``block_sparse_attention``: the forward and backward through torch.autograd.

The loss L = sum(out * G) for a seeded bf16 G gives dL/dout = G exactly, so the
gradients autograd accumulates into q, k and v must equal, bit for bit, a direct
``backward`` call with dout = G on the same forward output; and, against the
oracle's fp64 gradients, each gradient tensor holds the backward tolerance
(max |g - g_ref| <= 2e-2 max |g_ref| + 1e-4: one bf16 rounding of P and one of
dS per term) plus the bf16 rounding of the gradient itself (half an ulp, at most
2^-8 max |g_ref|).  The output is the bf16 forward: the fp32 tolerance 5e-3 plus
half an ulp of bf16 (at most 2^-8 max |O_ref|)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads.configs import MASK_CAUSAL, MASK_SLIDING_WINDOW, random_workload  # noqa: E402
from workloads.device import DeviceWorkload, bf16_to_device  # noqa: E402

pytestmark = pytest.mark.gpu

CASES = {
    "batched_causal": dict(seed=421, B=2, H=2, D=128, seqlens_q=[300, 300], kind=MASK_CAUSAL,
                           density=0.6),
    "varlen_window": dict(seed=422, B=3, H=2, D=64, seqlens_q=[200, 333, 129], varlen=True,
                          kind=MASK_SLIDING_WINDOW, window_left=100, sink_tokens=20, density=0.8,
                          valid_len=True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_autograd_matches_direct_backward_and_oracle(name):
    wl = random_workload(**CASES[name])
    q_bits, k_bits, v_bits = wl.qkv()
    g_bits = wl.tensor("do")
    dw = DeviceWorkload(wl, "cuda", qkv=(q_bits, k_bits, v_bits))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    kw = dict(cu_seqlens_q=dw.cu_q, cu_seqlens_k=dw.cu_k, kv_valid_len=dw.vl, kind=wl.kind,
              mask_params=dw.mask_params, softmax_scale=wl.scale, err_flag=err)
    q = dw.q.detach().clone().requires_grad_(True)
    k = dw.k.detach().clone().requires_grad_(True)
    v = dw.v.detach().clone().requires_grad_(True)
    g = bf16_to_device(g_bits, "cuda")
    out = bsa.block_sparse_attention(q, k, v, meta, **kw)
    assert out.dtype == torch.bfloat16 and out.shape == q.shape
    (out.float() * g.float()).sum().backward()
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # the same kernels called directly
    out2, lse2 = bsa.forward(dw.q, dw.k, dw.v, meta, **kw)
    dq2, dk2, dv2 = bsa.backward(dw.q, dw.k, dw.v, out2, lse2, g, meta, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), out2)
    for a, b in ((q.grad, dq2), (k.grad, dk2), (v.grad, dv2)):
        assert a.dtype == torch.bfloat16 and torch.equal(a, b)

    # against the oracle
    ref_meta = oracle.build_meta(wl)
    o_ref, _ = oracle.fwd(wl, q_bits, k_bits, v_bits, ref_meta)
    o = out.detach().float().cpu().numpy().astype(np.float64)
    assert np.max(np.abs(o - o_ref)) <= 5e-3 + 2 ** -8 * np.max(np.abs(o_ref))
    refs = oracle.bwd(wl, q_bits, k_bits, v_bits, ref_meta, g_bits)
    for got, ref in zip((q.grad, k.grad, v.grad), refs):
        got = got.float().cpu().numpy().astype(np.float64)
        scale = float(np.max(np.abs(ref), initial=0.0))
        assert np.max(np.abs(got - ref), initial=0.0) <= 2e-2 * scale + 1e-4 + scale * 2 ** -8
