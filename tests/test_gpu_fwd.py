"""Attention kernel vs the oracle: O within 5e-3 and LSE within 1e-3 max abs
(the bar the block-sparse forward is held to, on bf16 inputs with fp32
accumulation), with identical -inf positions for empty rows.  O is compared in
the kernel's fp32 output; the bf16 output is checked to be exactly the
round-to-nearest-even of that fp32 output (a bf16 result cannot meet an
absolute 5e-3 bar on its own once |O| >= 2, where half a bf16 ulp is 0.0078).

Small configs are compared element by element; the two full-size configs on
every row of their first and last head and at sampled (row, head) outputs of
the rest, in the same launch configuration the benchmark times, plus properties
that hold at any size."""
import numpy as np
import pytest
import torch

import block_sparse_flashattention_gb300 as bsa
import oracle
from workloads.device import DeviceWorkload, meta_from_numpy
from workloads import bf16_bits_to_f32, make_workload
from workloads.configs import (MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE, MASK_PREFIX,
                               MASK_SLIDING_WINDOW, random_workload)

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 5e-3, 1e-3


def _compare(got_o, got_l, ref_o, ref_l):
    assert got_o.shape == ref_o.shape and got_l.shape == ref_l.shape
    assert np.all(np.isfinite(got_o))
    e_o = float(np.max(np.abs(got_o - ref_o))) if ref_o.size else 0.0
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(got_l), fin), "empty-row pattern differs"
    assert np.all(got_l[~fin] == -np.inf)
    e_l = float(np.max(np.abs(got_l[fin] - ref_l[fin]))) if fin.any() else 0.0
    assert e_o <= TOL_O, f"max |dO| = {e_o:.3e}"
    assert e_l <= TOL_LSE, f"max |dLSE| = {e_l:.3e}"
    return e_o, e_l


def _run(wl, meta_arrays=None, expect_flags=0):
    """Runs the forward twice (fp32 and bf16 outputs); returns the fp32 O and LSE
    after checking that the bf16 output is exactly RNE(fp32 output)."""
    q, k, v = wl.qkv()
    dw = DeviceWorkload(wl, "cuda", qkv=(q, k, v))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if meta_arrays is None:
        meta = dw.build_meta(err_flag=err)
    else:
        meta = meta_from_numpy(wl, meta_arrays)
    out32, lse = dw.forward(meta, err_flag=err, out_dtype=torch.float32)
    out16, lse16 = dw.forward(meta, err_flag=err, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert int(err.item()) == expect_flags
    assert torch.equal(out16.view(torch.int16), out32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lse, lse16)
    return (q, k, v), out32.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _full_check(wl):
    (q, k, v), got_o, got_l = _run(wl)
    ref_meta = oracle.build_meta(wl)
    ref_o, ref_l = oracle.fwd(wl, q, k, v, ref_meta)
    return _compare(got_o, got_l, ref_o, ref_l)


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_fwd_configs_small(cfg):
    _full_check(make_workload(cfg))


CASES = [
    dict(seed=201, B=1, H=2, D=128, seqlens_q=[256], kind=MASK_CAUSAL, density=1.0),
    dict(seed=202, B=2, H=3, D=64, seqlens_q=[384, 384], kind=MASK_CAUSAL),          # 3 tiles: odd
    dict(seed=203, B=1, H=2, D=128, seqlens_q=[300], seqlens_k=[520], kind=MASK_NONE,
         valid_len=True),
    dict(seed=204, B=4, H=2, D=128, seqlens_q=[130, 257, 40, 1], varlen=True, kind=MASK_CAUSAL,
         valid_len=True),
    dict(seed=205, B=2, H=2, D=64, seqlens_q=[200, 450], seqlens_k=[333, 129], varlen=True,
         kind=MASK_SLIDING_WINDOW, window_left=150, sink_tokens=70, valid_len=True),
    dict(seed=206, B=1, H=2, D=128, seqlens_q=[1000], kind=MASK_SLIDING_WINDOW, window_left=256,
         sink_tokens=200, density=0.8),
    dict(seed=207, B=1, H=2, D=128, seqlens_q=[512], kind=MASK_PREFIX, prefix_len=200),
    dict(seed=208, B=2, H=1, D=128, seqlens_q=[300, 77], varlen=True, kind=MASK_DOCUMENT,
         n_docs=4),
    dict(seed=209, B=1, H=2, D=64, seqlens_q=[640], seqlens_k=[1300], kind=MASK_PREFIX,
         prefix_len=700, valid_len=True),
    dict(seed=210, B=3, H=2, D=128, seqlens_q=[4096, 100, 2000], varlen=True, kind=MASK_CAUSAL,
         density=0.3),
    dict(seed=211, B=1, H=2, D=128, seqlens_q=[256], kind=MASK_CAUSAL, density=0.0,
         force_diag=False),                                                           # all empty
    dict(seed=212, B=1, H=3, D=128, seqlens_q=[2048], kind=MASK_NONE, density=0.5,
         force_diag=False),                                                           # some empty
    dict(seed=213, B=5, H=2, D=64, seqlens_q=[1, 127, 128, 129, 255], varlen=True,
         kind=MASK_NONE, density=1.0),
    dict(seed=214, B=1, H=1, D=128, seqlens_q=[128], seqlens_k=[100_000], kind=MASK_NONE,
         density=0.05, force_diag=False),                                            # long rows
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fwd_random_cases(case):
    _full_check(random_workload(**CASES[case]))


def test_fwd_large_logits_do_not_overflow():
    """Scores up to ~100 in the exponent: the running maximum keeps exp() finite."""
    wl = random_workload(215, B=1, H=2, D=128, seqlens_q=[512], kind=MASK_CAUSAL, density=0.7,
                         scale=1.0)
    _full_check(wl)


# ------------------------------------------------------- caller-made lists

def _edit_lists(wl, fn):
    meta = oracle.build_meta(wl)
    edited = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in meta.items()}
    fn(edited)
    return meta, edited


def test_fwd_list_order_is_free():
    """Lists given in a shuffled order give the same result (within tolerance)."""
    wl = random_workload(221, B=2, H=2, D=128, seqlens_q=[768, 768], kind=MASK_CAUSAL,
                         density=0.6)
    rng = np.random.default_rng(0)

    def shuffle(m):
        for key in ("full", "mask"):
            cnt, idx = m[key + "_cnt"], m[key + "_idx"]
            for pos in np.ndindex(cnt.shape):
                c = int(cnt[pos])
                idx[pos][:c] = rng.permutation(idx[pos][:c])
    meta, edited = _edit_lists(wl, shuffle)
    (q, k, v), got_o, got_l = _run(wl, edited)
    ref_o, ref_l = oracle.fwd(wl, q, k, v, meta)
    _compare(got_o, got_l, ref_o, ref_l)


def test_fwd_ragged_tile_in_full_list_is_clipped():
    wl = random_workload(222, B=1, H=2, D=128, seqlens_q=[200], seqlens_k=[200], kind=MASK_NONE,
                         density=1.0)

    def all_full(m):
        m["full_idx"][0, :, :, :] = -1
        m["full_idx"][0, :, :, :2] = [1, 0]
        m["full_cnt"][:] = 2
        m["mask_idx"][:] = -1
        m["mask_cnt"][:] = 0
    _, edited = _edit_lists(wl, all_full)
    (q, k, v), got_o, got_l = _run(wl, edited)
    ref_o, ref_l = oracle.fwd(wl, q, k, v, edited)
    _compare(got_o, got_l, ref_o, ref_l)


def test_fwd_bad_indices_are_skipped_and_flagged():
    wl = random_workload(223, B=1, H=2, D=128, seqlens_q=[512], kind=MASK_CAUSAL, density=0.8)

    def corrupt(m):
        # row (0, 0, 3): replace its first full entry by an out-of-range id and
        # give row (0, 1, 2) a count above num_n
        c = int(m["full_cnt"][0, 0, 3])
        assert c >= 1
        m["full_idx"][0, 0, 3, 0] = 99
        m["mask_cnt"][0, 1, 2] = 50
    meta, edited = _edit_lists(wl, corrupt)
    (q, k, v), got_o, got_l = _run(wl, edited,
                                   expect_flags=bsa.FLAG_BAD_INDEX | bsa.FLAG_BAD_COUNT)
    # what the kernel computes: the bad entry dropped, the count clamped to num_n
    # (the -1 padding it then meets is skipped as well)
    fixed = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in edited.items()}
    row = fixed["full_idx"][0, 0, 3]
    c = int(fixed["full_cnt"][0, 0, 3])
    keep = [x for x in row[:c].tolist() if 0 <= x < wl.num_n]
    row[:] = -1
    row[:len(keep)] = keep
    fixed["full_cnt"][0, 0, 3] = len(keep)
    mrow = fixed["mask_idx"][0, 1, 2]
    keep = [x for x in mrow.tolist() if 0 <= x < wl.num_n]
    mrow[:] = -1
    mrow[:len(keep)] = keep
    fixed["mask_cnt"][0, 1, 2] = len(keep)
    ref_o, ref_l = oracle.fwd(wl, q, k, v, fixed)
    _compare(got_o, got_l, ref_o, ref_l)


# ---------------------------------------------------------- full-size configs

def _sample_rows(wl, n_tiles, seed):
    """(packed row, head) pairs: a few rows of randomly chosen tiles, always
    including each tile's first and last row."""
    rng = np.random.default_rng(seed)
    S = int(wl.seqlens_q[0])
    tiles = rng.integers(0, S // 128, size=n_tiles)
    heads = rng.integers(0, wl.H, size=n_tiles)
    toks, hs = [], []
    for t, h in zip(tiles, heads):
        for r in (0, 1, 63, 64, 126, 127, int(rng.integers(0, 128))):
            toks.append(int(t) * 128 + r)
            hs.append(int(h))
    toks += [0, S - 1]
    hs += [0, wl.H - 1]
    return np.array(toks, np.int32), np.array(hs, np.int32)


@pytest.mark.parametrize("cfg", [4, 5])
def test_fwd_full_size_whole_heads_and_samples(cfg):
    """Every output row of the first and the last head, element by element, plus
    sampled rows of randomly chosen tiles and heads across the rest."""
    wl = make_workload(cfg)
    (q, k, v), got_o, got_l = _run(wl)
    ref_meta = oracle.build_meta(wl)
    S = int(wl.seqlens_q[0])
    g_o_all = got_o.reshape(S, wl.H, wl.D)
    g_l_all = got_l.reshape(wl.H, S)
    for h in (0, wl.H - 1):
        tok = np.arange(S, dtype=np.int32)
        ref_o, ref_l = oracle.fwd_rows(wl, q, k, v, ref_meta, tok, np.full(S, h, np.int32))
        _compare(g_o_all[:, h], g_l_all[h], ref_o, ref_l)
    tok, head = _sample_rows(wl, 48, seed=cfg)
    ref_o, ref_l = oracle.fwd_rows(wl, q, k, v, ref_meta, tok, head)
    _compare(g_o_all[tok, head], g_l_all[head, tok], ref_o, ref_l)
    # properties at every output: finite, no empty rows in these configs, and each
    # O row a convex combination of V rows (bounded by the largest |v|)
    assert np.all(np.isfinite(got_l))
    vmax = float(np.max(np.abs(bf16_to_f32(v))))
    assert float(np.max(np.abs(got_o))) <= vmax + 1e-2


def bf16_to_f32(x):
    return bf16_bits_to_f32(x)


def test_fwd_has_no_hidden_stall():
    """Every wait in the kernel gives up after about a second; a small launch must
    finish far below that, or some wait is running to its limit."""
    wl = make_workload(2)
    dw = DeviceWorkload(wl, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    dw.forward(meta, err_flag=err)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(5):
        dw.forward(meta, err_flag=err)
    b.record()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert a.elapsed_time(b) / 5 < 50.0, f"{a.elapsed_time(b) / 5:.1f} ms per launch"


@pytest.mark.parametrize("which", ["cfg2", "cfg3", "odd", "varlen_ragged"])
def test_fwd_schedules_agree_bitwise(which):
    """The scheduled path (work units claimed heaviest first) and the fixed-stride
    path compute every unit identically, so their outputs agree bit for bit."""
    wl = {"cfg2": lambda: make_workload(2), "cfg3": lambda: make_workload(3),
          "odd": lambda: random_workload(231, B=2, H=3, D=64, seqlens_q=[384, 384]),
          "varlen_ragged": lambda: random_workload(232, B=5, H=2, D=128,
                                                    seqlens_q=[1, 300, 129, 1000, 77],
                                                    varlen=True, density=0.4)}[which]()
    dw = DeviceWorkload(wl, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    meta = dw.build_meta(err_flag=err)
    ws = bsa.alloc_workspace(meta)
    assert ws is not None
    out_a, lse_a = dw.forward(meta, err_flag=err, workspace=None)
    out_b, lse_b = dw.forward(meta, err_flag=err, workspace=ws)
    out_c, lse_c = dw.forward(meta, err_flag=err, workspace=ws)     # workspace reused
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for o, l in ((out_b, lse_b), (out_c, lse_c)):
        assert torch.equal(out_a.view(torch.int16), o.view(torch.int16))
        assert torch.equal(lse_a, l)
