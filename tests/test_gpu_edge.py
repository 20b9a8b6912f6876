"""Degenerate inputs through the forward and the backward, against the oracle:
a varlen batch with a sequence that has no queries and one that has no keys,
sequences of one token, a batched sequence shorter than one tile, and an empty
selection (every row's key set empty: O = 0, LSE = -inf, all gradients 0)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_sparse_flashattention_gb300 as bsa  # noqa: E402
import oracle  # noqa: E402
from workloads.device import DeviceWorkload, bf16_to_device  # noqa: E402
from workloads.configs import MASK_CAUSAL, MASK_NONE, MASK_SLIDING_WINDOW, random_workload  # noqa: E402

pytestmark = pytest.mark.gpu

CASES = {
    "no_queries_no_keys": dict(seed=331, B=3, H=2, D=64, seqlens_q=[200, 0, 150],
                               seqlens_k=[100, 300, 0], varlen=True, kind=MASK_NONE, density=0.7),
    "one_token": dict(seed=332, B=3, H=2, D=128, seqlens_q=[1, 1, 130], seqlens_k=[1, 129, 1],
                      varlen=True, kind=MASK_CAUSAL, density=1.0),
    "short_batched": dict(seed=333, B=2, H=3, D=64, seqlens_q=[77, 77], seqlens_k=[45, 45],
                          kind=MASK_SLIDING_WINDOW, window_left=20, sink_tokens=3, density=1.0),
    "empty_selection": dict(seed=334, B=1, H=2, D=128, seqlens_q=[300], seqlens_k=[260],
                            kind=MASK_NONE, density=0.0, force_diag=False),
}


def _run(c):
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
    assert int(err.item()) == 0
    f64 = lambda t: t.cpu().numpy().astype(np.float64)  # noqa: E731
    return wl, (q, k, v, g_bits), f64(out), f64(lse), [f64(t) for t in grads]


@pytest.mark.parametrize("name", list(CASES))
def test_degenerate_inputs_match_the_oracle(name):
    wl, (q, k, v, g_bits), out, lse, grads = _run(CASES[name])
    meta = oracle.build_meta(wl)
    o_ref, l_ref = oracle.fwd(wl, q, k, v, meta)
    assert np.max(np.abs(out - o_ref), initial=0.0) <= 5e-3
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(lse[~fin] == -np.inf)
    assert np.max(np.abs(lse[fin] - l_ref[fin]), initial=0.0) <= 1e-3
    refs = oracle.bwd(wl, q, k, v, meta, g_bits)
    for got, ref in zip(grads, refs):
        # relative to the tensor's largest gradient, with an absolute floor: a
        # one-key row has dS = P (dP - D) = 0 exactly (P = 1, dP = D), which the
        # oracle reaches and the kernel reaches to summation-order rounding
        scale = float(np.max(np.abs(ref), initial=0.0))
        assert np.max(np.abs(got - ref), initial=0.0) <= 2e-2 * scale + 1e-4
    # structural zeros are exact: rows with no keys get dq = 0, keys that no query
    # attends get dk = dv = 0
    dq, dk, dv = grads
    no_keys = ~fin.T if wl.varlen else ~fin.transpose(0, 2, 1)
    assert np.all(dq[no_keys] == 0.0)
    unused = np.all(refs[2] == 0.0, axis=-1)
    assert np.all(dk[unused] == 0.0) and np.all(dv[unused] == 0.0)


def test_empty_selection_gives_zero_output_and_gradients():
    wl, _, out, lse, grads = _run(CASES["empty_selection"])
    assert np.all(out == 0.0) and np.all(lse == -np.inf)
    for g in grads:
        assert np.all(g == 0.0)


def test_sequences_without_queries_or_keys():
    wl, _, out, lse, (dq, dk, dv) = _run(CASES["no_queries_no_keys"])
    cq, ck = wl.cu_seqlens_q, wl.cu_seqlens_k
    # sequence 1 has no queries: its keys get no gradient
    assert np.all(dk[ck[1]:ck[2]] == 0.0) and np.all(dv[ck[1]:ck[2]] == 0.0)
    # sequence 2 has no keys: its rows are empty
    assert np.all(out[cq[2]:cq[3]] == 0.0) and np.all(dq[cq[2]:cq[3]] == 0.0)
    assert np.all(lse[:, cq[2]:cq[3]] == -np.inf)
