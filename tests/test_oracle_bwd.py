"""The oracle's backward pinned to things other than itself: its allowed-key
masks reproduce the C oracle's forward; its gradients match central finite
differences of L = sum(O * G); on a dense causal map they match torch autograd
in fp64."""
import numpy as np
import pytest

import oracle
from workloads.configs import (MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE, MASK_PREFIX,
                               MASK_SLIDING_WINDOW, random_workload)


def _w(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


CASES = [
    dict(seed=201, B=1, H=2, D=16, seqlens_q=[300], seqlens_k=[260], kind=MASK_CAUSAL),
    dict(seed=202, B=2, H=1, D=8, seqlens_q=[200, 200], kind=MASK_SLIDING_WINDOW, window_left=90,
         sink_tokens=20, valid_len=True),
    dict(seed=203, B=1, H=1, D=8, seqlens_q=[256], seqlens_k=[400], kind=MASK_PREFIX,
         prefix_len=150, valid_len=True),
    dict(seed=204, B=1, H=2, D=8, seqlens_q=[260], kind=MASK_NONE, density=0.6),
    dict(seed=205, B=2, H=1, D=8, seqlens_q=[300, 300], kind=MASK_DOCUMENT, density=0.8),
]


@pytest.mark.parametrize("c", CASES)
def test_allowed_masks_reproduce_the_c_oracle_forward(c):
    wl = random_workload(**c)
    q, k, v = wl.qkv()
    meta = oracle.build_meta(wl)
    o_c, _ = oracle.fwd(wl, q, k, v, meta)
    o_np = oracle.fwd_f64(wl, meta, _w(q), _w(k), _w(v))
    assert np.max(np.abs(o_c - o_np)) < 1e-12


@pytest.mark.parametrize("c", CASES[:3])
def test_gradients_match_finite_differences(c):
    wl = random_workload(**c)
    q, k, v = (_w(x) for x in wl.qkv())
    meta = oracle.build_meta(wl)
    rng = np.random.default_rng(c["seed"])
    G = rng.standard_normal(q.shape[:3] + (v.shape[3],))
    dq, dk, dv = oracle.bwd_f64(wl, meta, q, k, v, G)

    def loss(qq, kk, vv):
        return float((oracle.fwd_f64(wl, meta, qq, kk, vv) * G).sum())

    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                  loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_dense_causal_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    wl = random_workload(205, B=1, H=2, D=16, seqlens_q=[256], kind=MASK_CAUSAL, density=1.0)
    wl.block_map[:] = 1
    q, k, v = (_w(x) for x in wl.qkv())
    meta = oracle.build_meta(wl)
    G = np.random.default_rng(5).standard_normal(q.shape)
    dq, dk, dv = oracle.bwd_f64(wl, meta, q, k, v, G)
    tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3), requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=wl.scale)
    o.backward(torch.tensor(G.transpose(0, 2, 1, 3)))
    for ref, got in ((tq.grad, dq), (tk.grad, dk), (tv.grad, dv)):
        assert np.max(np.abs(ref.numpy().transpose(0, 2, 1, 3) - got)) < 1e-10


@pytest.mark.parametrize("c", CASES)
def test_per_tile_backward_equals_the_dense_one(c):
    # the per-tile forms (for sampled checks at full size) against bwd_f64 on
    # every Q tile and KV tile, and their allowed sets against allowed_mask
    wl = random_workload(**c)
    q, k, v = wl.qkv()
    g = wl.tensor("do")
    meta = oracle.build_meta(wl)
    dq, dk, dv = oracle.bwd(wl, q, k, v, meta, g)
    for b in range(wl.B):
        for h in range(wl.H):
            A = oracle.allowed_mask(wl, meta, b, h)
            for m in range(wl.num_m):
                r0, r1, keys, At = oracle.tile_allowed(wl, meta, b, h, m)
                full = np.zeros((r1 - r0, A.shape[1]), bool)
                full[:, keys] = At
                assert np.array_equal(full, A[r0:r1])
                t = oracle.bwd_dq_tile(wl, q, k, v, g, meta, b, h, m)
                assert np.max(np.abs(t - dq[b, r0:r1, h]), initial=0) < 1e-12
            for n in range(wl.num_n):
                tk, tv = oracle.bwd_dkdv_tile(wl, q, k, v, g, meta, b, h, n)
                c0 = n * wl.tile_n
                assert np.max(np.abs(tk - dk[b, c0:c0 + tk.shape[0], h]), initial=0) < 1e-12
                assert np.max(np.abs(tv - dv[b, c0:c0 + tv.shape[0], h]), initial=0) < 1e-12


@pytest.mark.parametrize("c", CASES)
def test_per_head_backward_equals_the_dense_one(c):
    # the whole-head form (Q tile by Q tile, for full-size checks) against bwd_f64
    wl = random_workload(**c)
    q, k, v = wl.qkv()
    g = wl.tensor("do")
    meta = oracle.build_meta(wl)
    dq, dk, dv = oracle.bwd(wl, q, k, v, meta, g)
    for b in range(wl.B):
        for h in range(wl.H):
            hq, hk, hv = oracle.bwd_head(wl, q, k, v, g, meta, b, h)
            for got, ref in ((hq, dq[b, :, h]), (hk, dk[b, :, h]), (hv, dv[b, :, h])):
                assert got.shape == ref.shape
                assert np.max(np.abs(got - ref), initial=0) < 1e-12


VARLEN_CASES = [
    dict(seed=211, B=3, H=2, D=8, seqlens_q=[300, 129, 200], seqlens_k=[260, 400, 128],
         varlen=True, kind=MASK_CAUSAL),
    dict(seed=212, B=3, H=1, D=8, seqlens_q=[250, 90, 310], varlen=True,
         kind=MASK_SLIDING_WINDOW, window_left=100, sink_tokens=30, valid_len=True),
    dict(seed=213, B=2, H=2, D=8, seqlens_q=[280, 170], varlen=True, kind=MASK_DOCUMENT,
         density=0.7),
    dict(seed=214, B=2, H=1, D=8, seqlens_q=[200, 330], seqlens_k=[310, 150], varlen=True,
         kind=MASK_PREFIX, prefix_len=140, valid_len=True),
]


@pytest.mark.parametrize("c", VARLEN_CASES)
def test_sequence_views_reproduce_the_c_oracle_varlen_forward(c):
    # each sequence of a varlen workload, taken as a batched workload of one with
    # its slice of the packed lists, gives the C oracle's varlen forward rows
    wl = random_workload(**c)
    q, k, v = wl.qkv()
    meta = oracle.build_meta(wl)
    o_c, _ = oracle.fwd(wl, q, k, v, meta)
    for b in range(wl.B):
        view, mb, qs, ks = oracle.seq_view(wl, meta, b)
        o = oracle.fwd_f64(view, mb, _w(q[qs])[None], _w(k[ks])[None], _w(v[ks])[None])[0]
        assert np.max(np.abs(o - o_c[qs])) < 1e-12


@pytest.mark.parametrize("c", VARLEN_CASES[:2])
def test_varlen_gradients_match_finite_differences(c):
    wl = random_workload(**c)
    q, k, v = wl.qkv()
    meta = oracle.build_meta(wl)
    rng = np.random.default_rng(c["seed"])
    g_bits = wl.tensor("do")
    dq, dk, dv = oracle.bwd(wl, q, k, v, meta, g_bits)
    G = _w(g_bits)
    qf, kf, vf = _w(q), _w(k), _w(v)

    def loss(qq, kk, vv):
        tot = 0.0
        for b in range(wl.B):
            view, mb, qs, ks = oracle.seq_view(wl, meta, b)
            o = oracle.fwd_f64(view, mb, qq[qs][None], kk[ks][None], vv[ks][None])[0]
            tot += float((o * G[qs]).sum())
        return tot

    eps = 1e-6
    for name, x, grad in (("q", qf, dq), ("k", kf, dk), ("v", vf, dv)):
        for _ in range(4):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            a_p = {"q": qf, "k": kf, "v": vf}
            a_m = dict(a_p)
            a_p[name], a_m[name] = xp, xm
            fd = (loss(a_p["q"], a_p["k"], a_p["v"]) - loss(a_m["q"], a_m["k"], a_m["v"])) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx)
