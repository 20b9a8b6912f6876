"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: values the pages
print for a worked example (tests/golden), hand-worked closed forms, special
cases that reduce to a library routine (torch scaled_dot_product_attention and
logsumexp in fp64 on the CPU), a dense brute force on tiny inputs
(tests/dense_ref.py) and invariants of the method.
"""
import math
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits_to_f32, make_workload
from workloads.configs import (MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE, MASK_PREFIX,
                               MASK_SLIDING_WINDOW, Workload, random_workload)
from tests import dense_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cdiv(a, b):
    return -(-a // b)


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


def _single_row_workload(row, kind=MASK_NONE, D=64):
    nn = len(row)
    bm = np.asarray(row, np.uint8).reshape(1, 1, 1, nn)
    return Workload(name="row", B=1, H=1, D=D, varlen=False,
                    seqlens_q=np.array([128], np.int32),
                    seqlens_k=np.array([128 * nn], np.int32), block_map=bm, kind=kind,
                    scale=1.0 / math.sqrt(D), data_seed=7)


def _map_row(wl, b, h, m):
    if wl.varlen:
        off = wl.map_row_offsets()
        nn = _cdiv(int(wl.seqlens_k[b]), wl.tile_n)
        return wl.block_map[h, off[b] + m * nn: off[b] + (m + 1) * nn]
    return wl.block_map[b, h, m]


def _rows(wl):
    for b in range(wl.B):
        for h in range(wl.H):
            for m in range(_cdiv(int(wl.seqlens_q[b]), wl.tile_m)):
                yield b, h, m


def _f64(x):
    return bf16_bits_to_f32(x).astype(np.float64)


# ------------------------------------------------------------- worked examples

def test_worked_example_reversed_list():
    (line,) = _golden_lines("reversed_list_worked_example.txt")
    lhs, rhs = line.split("->")
    row = [int(t) for t in lhs.split()]
    expect = [int(t) for t in rhs.split()]
    wl = _single_row_workload(row)
    meta = oracle.build_meta(wl)
    assert meta["full_idx"][0, 0, 0].tolist() == expect
    assert int(meta["full_cnt"][0, 0, 0]) == sum(row)
    assert meta["mask_idx"][0, 0, 0].tolist() == [-1] * len(row)
    assert int(meta["mask_cnt"][0, 0, 0]) == 0


def test_tiny_walk_example():
    nb, sel, visit, leaps = _golden_lines("sparse_walk_tiny_example.txt")
    nb = int(nb)
    sel = [int(t) for t in sel.split()]
    row = [1 if n in sel else 0 for n in range(nb)]
    meta = oracle.build_meta(_single_row_workload(row))
    cnt = int(meta["full_cnt"][0, 0, 0])
    lst = meta["full_idx"][0, 0, 0][:cnt].tolist()
    assert lst == [int(t) for t in visit.split()]
    assert [a - b for a, b in zip(lst, lst[1:])] == [int(t) for t in leaps.split()]


def test_varlen_offsets_hand_worked():
    kv = {}
    for ln in _golden_lines("varlen_offsets_hand_worked.txt"):
        key, val = ln.split("=")
        kv[key.strip()] = [int(t) for t in val.split()]
    sq = np.array(kv["seqlens_q"], np.int32)
    sk = np.array(kv["seqlens_k"], np.int32)
    wl = Workload(name="v", B=len(sq), H=1, D=64, varlen=True, seqlens_q=sq, seqlens_k=sk,
                  block_map=np.zeros(1, np.uint8), kind=MASK_NONE, scale=0.125, data_seed=1)
    cm, cn = oracle.varlen_offsets(wl)
    assert cm.tolist() == kv["cu_total_m_blocks"]
    assert cn.tolist() == kv["cu_block_idx_offsets"]
    wl.block_map = np.ones((1, kv["total_n_blocks"][0]), np.uint8)
    meta = oracle.build_meta(wl)
    assert meta["total_m_blocks"] == kv["total_m_blocks"][0]
    assert meta["total_n_blocks"] == kv["total_n_blocks"][0]


@pytest.mark.parametrize("seed", range(5))
def test_varlen_identities_random_lengths(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 9))
    sq = rng.integers(1, 1000, size=B).astype(np.int32)
    sk = rng.integers(1, 1000, size=B).astype(np.int32)
    wl = Workload(name="v", B=B, H=2, D=64, varlen=True, seqlens_q=sq, seqlens_k=sk,
                  block_map=np.zeros(1, np.uint8), kind=MASK_NONE, scale=0.125, data_seed=1)
    cm, cn = oracle.varlen_offsets(wl)
    nm = [math.ceil(int(s) / 128) for s in sq]
    nn = [math.ceil(int(s) / 128) for s in sk]
    assert cm[-1] == sum(nm)
    assert cn[-1] == sum(a * b for a, b in zip(nm, nn))
    assert np.all(np.diff(cm) == nm) and np.all(np.diff(cn) == [a * b for a, b in zip(nm, nn)])


# ----------------------------------------------------------- metadata checks

META_CASES = [
    dict(seed=11, B=2, H=2, D=64, seqlens_q=[384, 384], kind=MASK_CAUSAL),
    dict(seed=12, B=1, H=3, D=64, seqlens_q=[300], seqlens_k=[520], kind=MASK_NONE,
         valid_len=True),
    dict(seed=13, B=3, H=2, D=64, seqlens_q=[130, 257, 40], varlen=True, kind=MASK_CAUSAL),
    dict(seed=14, B=2, H=2, D=64, seqlens_q=[200, 450], seqlens_k=[333, 129], varlen=True,
         kind=MASK_SLIDING_WINDOW, window_left=150, sink_tokens=70, valid_len=True),
    dict(seed=15, B=1, H=2, D=64, seqlens_q=[512], kind=MASK_PREFIX, prefix_len=200),
    dict(seed=16, B=2, H=1, D=64, seqlens_q=[300, 77], varlen=True, kind=MASK_DOCUMENT,
         n_docs=4),
    dict(seed=17, B=1, H=2, D=64, seqlens_q=[640], kind=MASK_SLIDING_WINDOW, window_left=128,
         sink_tokens=128, density=0.7),
]


def _case(c):
    c = dict(c)
    return random_workload(**c)


@pytest.mark.parametrize("case", range(len(META_CASES)))
def test_meta_partition_and_format(case):
    wl = _case(META_CASES[case])
    meta = oracle.build_meta(wl)
    for b, h, m in _rows(wl):
        nn = _cdiv(int(wl.seqlens_k[b]), wl.tile_n)
        full, mask = dense_ref.row_lists(wl, meta, b, h, m)
        sel = set(np.flatnonzero(_map_row(wl, b, h, m)).tolist())
        assert not set(full) & set(mask)
        assert set(full) | set(mask) <= sel
        for lst in (full, mask):
            assert all(0 <= n < nn for n in lst)
            assert lst == sorted(lst, reverse=True) and len(set(lst)) == len(lst)
        # padding
        if wl.varlen:
            base = int(meta["cu_block_idx_offsets"][b]) + m * nn
            fi = meta["full_idx"][h, base: base + nn]
            mi = meta["mask_idx"][h, base: base + nn]
        else:
            fi, mi = meta["full_idx"][b, h, m], meta["mask_idx"][b, h, m]
        assert np.all(fi[len(full):] == -1) and np.all(mi[len(mask):] == -1)


@pytest.mark.parametrize("case", range(len(META_CASES)))
def test_meta_classification_matches_dense_predicate(case):
    wl = _case(META_CASES[case])
    meta = oracle.build_meta(wl)
    for b, h, m in _rows(wl):
        sq, sk = int(wl.seqlens_q[b]), int(wl.seqlens_k[b])
        full, mask = dense_ref.row_lists(wl, meta, b, h, m)
        for n in np.flatnonzero(_map_row(wl, b, h, m)).tolist():
            ii = np.arange(m * 128, min(m * 128 + 128, sq))[:, None]
            jj = np.arange(n * 128, n * 128 + 128)[None, :]
            pred = (jj < sk) & dense_ref.mask_matrix(wl, b, ii, np.minimum(jj, sk - 1))
            if wl.kv_valid_len is not None:
                pred &= jj - n * 128 < wl.kv_valid_len[b, n]
            if pred.all():
                assert n in full
            elif pred.any():
                assert n in mask
            else:
                assert n not in full and n not in mask


def test_config1_lists():
    """Tiny causal: per head, full {(1,0)} and mask {(0,0),(1,1)}."""
    wl = make_workload(1)
    meta = oracle.build_meta(wl)
    for h in range(wl.H):
        assert meta["full_cnt"][0, h].tolist() == [0, 1]
        assert meta["mask_cnt"][0, h].tolist() == [1, 1]
        assert meta["full_idx"][0, h, 1].tolist() == [0, -1]
        assert meta["mask_idx"][0, h, 0].tolist() == [0, -1]
        assert meta["mask_idx"][0, h, 1].tolist() == [1, -1]


def _head_slice(wl, heads):
    return replace(wl, H=heads, block_map=np.ascontiguousarray(wl.block_map[:, :heads]))


def test_config5_closed_form_counts():
    """Window [m-32, m] + sinks {0..3}, window 4096 tokens, 512 sink tokens, causal.

    Closed form: mask = the diagonal tile of every row plus tile m-32 whenever it
    is not a sink tile (m >= 36); every other selected tile with n <= m is full.
    Totals per head: 37,222 tiles of which 2,012 are mask tiles."""
    wl = _head_slice(make_workload(5), 1)
    meta = oracle.build_meta(wl)
    nm = wl.num_m
    exp_full, exp_mask = np.zeros(nm, int), np.zeros(nm, int)
    for m in range(nm):
        sel = set(range(max(0, m - 32), m + 1)) | set(range(min(4, m + 1)))
        masks = {m} | ({m - 32} if m - 32 >= 4 else set())
        exp_mask[m] = len(masks)
        exp_full[m] = len(sel - masks)
    assert meta["mask_cnt"][0, 0].tolist() == exp_mask.tolist()
    assert meta["full_cnt"][0, 0].tolist() == exp_full.tolist()
    assert int(exp_full.sum() + exp_mask.sum()) == 37222 and int(exp_mask.sum()) == 2012


def test_config4_valid_length_classification():
    """VSA: each selected logical block gives tile 2kb (valid 128, full) and tile
    2kb+1 (valid v-128: full iff v == 256, else mask)."""
    full_wl = make_workload(4)
    wl = _head_slice(full_wl, 2)
    meta = oracle.build_meta(wl)
    v = full_wl.extra["logical_block_valid_len"]
    logical = full_wl.extra["logical_map"]
    for h in range(2):
        for qb in range(0, 240, 17):
            kbs = np.flatnonzero(logical[h, qb])
            full = {2 * kb for kb in kbs} | {2 * kb + 1 for kb in kbs if v[kb] == 256}
            mask = {2 * kb + 1 for kb in kbs if v[kb] < 256}
            for m in (2 * qb, 2 * qb + 1):
                f, mk = dense_ref.row_lists(wl, meta, 0, h, m)
                assert set(f) == full and set(mk) == mask


# ------------------------------------------------------------ forward checks

FWD_CASES = META_CASES + [
    dict(seed=21, B=1, H=2, D=128, seqlens_q=[256], kind=MASK_CAUSAL, density=1.0),
    dict(seed=22, B=2, H=1, D=32, seqlens_q=[129, 1], varlen=True, kind=MASK_NONE,
         valid_len=True),
]


@pytest.mark.parametrize("case", range(len(FWD_CASES)))
def test_fwd_matches_dense_bruteforce(case):
    wl = _case(FWD_CASES[case])
    q, k, v = wl.qkv()
    meta = oracle.build_meta(wl)
    O, L = oracle.fwd(wl, q, k, v, meta)
    Od, Ld = dense_ref.dense_attention(wl, q, k, v, meta)
    assert np.max(np.abs(O - Od)) <= 1e-12
    fin = np.isfinite(Ld)
    assert np.array_equal(fin, np.isfinite(L))
    assert np.all(L[~fin] == -np.inf)
    assert np.max(np.abs(L[fin] - Ld[fin])) <= 1e-12


def _sdpa(q, k, v, scale, causal):
    """torch SDPA in fp64 on [B,S,H,D] float64 arrays -> O [B,S,H,D], LSE [B,H,S]."""
    Q, K, V = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale, is_causal=causal)
    S = scale * Q @ K.transpose(-1, -2)
    if causal:
        S = S.masked_fill(torch.ones_like(S, dtype=torch.bool).triu(1), float("-inf"))
    return O.permute(0, 2, 1, 3).numpy(), torch.logsumexp(S, dim=-1).numpy()


@pytest.mark.parametrize("kind,causal", [(MASK_NONE, False), (MASK_CAUSAL, True)])
def test_all_ones_map_equals_library_attention(kind, causal):
    wl = random_workload(31, B=2, H=3, D=64, seqlens_q=[320, 320], kind=kind, density=1.0)
    q, k, v = wl.qkv()
    O, L = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    Oref, Lref = _sdpa(_f64(q), _f64(k), _f64(v), wl.scale, causal)
    assert np.max(np.abs(O - Oref)) <= 1e-12
    assert np.max(np.abs(L - Lref)) <= 1e-12


def test_sliding_window_of_one_is_identity():
    """window_left = 1, no sinks: each query sees only its own key, so O_i = v_i
    and LSE_i = scale * q_i . k_i."""
    wl = random_workload(32, B=1, H=2, D=64, seqlens_q=[300], kind=MASK_SLIDING_WINDOW,
                         window_left=1, sink_tokens=0, density=1.0)
    q, k, v = wl.qkv()
    O, L = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    assert np.array_equal(O, _f64(v))
    qk = np.einsum("bshd,bshd->bhs", _f64(q), _f64(k))
    assert np.max(np.abs(L - wl.scale * qk)) <= 1e-12


@pytest.mark.parametrize("sinks", [5, 130])
def test_window_of_one_with_sinks_is_library_attention_on_gathered_keys(sinks):
    """window_left = 1 with s sink tokens: query i sees exactly the keys
    j < min(s, i + 1) and itself, so each row equals torch SDPA over those keys
    gathered out of the sequence (s = 130 puts the sink edge inside tile 1)."""
    wl = random_workload(37, B=1, H=2, D=64, seqlens_q=[300], kind=MASK_SLIDING_WINDOW,
                         window_left=1, sink_tokens=sinks, density=1.0)
    q, k, v = wl.qkv()
    O, L = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    worst_o = worst_l = 0.0
    for i in range(300):
        keys = sorted(set(range(min(sinks, i + 1))) | {i})
        Oi, Li = _sdpa(qf[:, i:i + 1], kf[:, keys], vf[:, keys], wl.scale, False)
        worst_o = max(worst_o, float(np.max(np.abs(O[:, i:i + 1] - Oi))))
        worst_l = max(worst_l, float(np.max(np.abs(L[:, :, i:i + 1] - Li))))
    assert worst_o <= 1e-12 and worst_l <= 1e-12


def test_wide_sliding_window_equals_causal_library():
    wl = random_workload(33, B=1, H=2, D=64, seqlens_q=[300], kind=MASK_SLIDING_WINDOW,
                         window_left=10_000, sink_tokens=0, density=1.0)
    q, k, v = wl.qkv()
    O, L = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    Oref, Lref = _sdpa(_f64(q), _f64(k), _f64(v), wl.scale, True)
    assert np.max(np.abs(O - Oref)) <= 1e-12 and np.max(np.abs(L - Lref)) <= 1e-12


@pytest.mark.parametrize("prefix,causal", [(0, True), (10_000, False)])
def test_prefix_extremes_equal_library(prefix, causal):
    wl = random_workload(34, B=1, H=2, D=64, seqlens_q=[260], kind=MASK_PREFIX,
                         prefix_len=prefix, density=1.0)
    q, k, v = wl.qkv()
    O, L = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    Oref, Lref = _sdpa(_f64(q), _f64(k), _f64(v), wl.scale, causal)
    assert np.max(np.abs(O - Oref)) <= 1e-12 and np.max(np.abs(L - Lref)) <= 1e-12


def test_document_single_and_distinct():
    wl = random_workload(35, B=1, H=2, D=64, seqlens_q=[260], kind=MASK_DOCUMENT,
                         density=1.0, n_docs=1)
    q, k, v = wl.qkv()
    O, L = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    Oref, Lref = _sdpa(_f64(q), _f64(k), _f64(v), wl.scale, False)
    assert np.max(np.abs(O - Oref)) <= 1e-12 and np.max(np.abs(L - Lref)) <= 1e-12
    wl.doc_id_q = np.arange(260, dtype=np.int32)
    wl.doc_id_k = wl.doc_id_q.copy()
    O, L = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    assert np.array_equal(O, _f64(v))


def test_valid_length_one_is_strided_library_attention():
    """kind NONE, valid length 1 in every tile: query i sees keys 0, 128, 256, ..."""
    wl = random_workload(36, B=1, H=2, D=64, seqlens_q=[384], kind=MASK_NONE, density=1.0,
                         valid_len=True)
    wl.kv_valid_len[:] = 1
    q, k, v = wl.qkv()
    O, L = oracle.fwd(wl, q, k, v, oracle.build_meta(wl))
    Oref, Lref = _sdpa(_f64(q), _f64(k)[:, ::128], _f64(v)[:, ::128], wl.scale, False)
    assert np.max(np.abs(O - Oref)) <= 1e-12 and np.max(np.abs(L - Lref)) <= 1e-12


# --------------------------------------------------------------- invariants

def _permute_lists(wl, meta, seed):
    rng = np.random.default_rng(seed)
    out = {k: v.copy() if isinstance(v, np.ndarray) else v for k, v in meta.items()}
    for b, h, m in _rows(wl):
        nn = _cdiv(int(wl.seqlens_k[b]), wl.tile_n)
        for kind in ("full", "mask"):
            if wl.varlen:
                base = int(meta["cu_block_idx_offsets"][b]) + m * nn
                cnt = int(meta[kind + "_cnt"][h, int(meta["cu_total_m_blocks"][b]) + m])
                seg = out[kind + "_idx"][h, base: base + cnt]
            else:
                cnt = int(meta[kind + "_cnt"][b, h, m])
                seg = out[kind + "_idx"][b, h, m, :cnt]
            seg[:] = rng.permutation(seg)
    return out


@pytest.mark.parametrize("case", [0, 3, 6])
def test_list_order_does_not_matter(case):
    wl = _case(FWD_CASES[case])
    q, k, v = wl.qkv()
    meta = oracle.build_meta(wl)
    O1, L1 = oracle.fwd(wl, q, k, v, meta)
    O2, L2 = oracle.fwd(wl, q, k, v, _permute_lists(wl, meta, 5))
    assert np.max(np.abs(O1 - O2)) <= 1e-12
    fin = np.isfinite(L1)
    assert np.max(np.abs(L1[fin] - L2[fin])) <= 1e-12


def test_full_block_moved_to_mask_list_is_unchanged():
    """With kind NONE and no valid length, the token predicate is true on every
    interior tile, so listing a full tile as a mask tile changes nothing."""
    wl = random_workload(41, B=1, H=2, D=64, seqlens_q=[512], kind=MASK_NONE, density=0.6,
                         force_diag=False)
    q, k, v = wl.qkv()
    meta = oracle.build_meta(wl)
    moved = {k: v.copy() if isinstance(v, np.ndarray) else v for k, v in meta.items()}
    moved["mask_idx"], moved["full_idx"] = meta["full_idx"].copy(), meta["mask_idx"].copy()
    moved["mask_cnt"], moved["full_cnt"] = meta["full_cnt"].copy(), meta["mask_cnt"].copy()
    O1, L1 = oracle.fwd(wl, q, k, v, meta)
    O2, L2 = oracle.fwd(wl, q, k, v, moved)
    assert np.max(np.abs(O1 - O2)) <= 1e-12
    fin = np.isfinite(L1)
    assert np.array_equal(fin, np.isfinite(L2)) and np.max(np.abs(L1[fin] - L2[fin])) <= 1e-12


def test_empty_rows_give_zero_and_minus_inf():
    wl = random_workload(42, B=1, H=2, D=64, seqlens_q=[256], kind=MASK_CAUSAL, density=0.0,
                         force_diag=False)
    q, k, v = wl.qkv()
    meta = oracle.build_meta(wl)
    assert meta["full_cnt"].sum() == 0 and meta["mask_cnt"].sum() == 0
    O, L = oracle.fwd(wl, q, k, v, meta)
    assert np.all(O == 0) and np.all(L == -np.inf)


def test_partial_tail_tile_never_full():
    """A KV tile that runs past seqlen_k has keys outside the sequence, so the
    token predicate is false there and the tile can only be a mask tile."""
    wl = random_workload(43, B=1, H=1, D=64, seqlens_q=[128], seqlens_k=[200], kind=MASK_NONE,
                         density=1.0)
    meta = oracle.build_meta(wl)
    assert dense_ref.row_lists(wl, meta, 0, 0, 0) == ([0], [1])


def test_full_list_tile_past_seqlen_is_clipped():
    """Caller-supplied lists may put a ragged last tile in the full list; keys at
    or past seqlen_k are still outside the sequence.  With every tile listed as
    full and kind NONE the result is plain attention over the 200 real keys."""
    wl = random_workload(44, B=1, H=2, D=64, seqlens_q=[128], seqlens_k=[200], kind=MASK_NONE,
                         density=1.0)
    q, k, v = wl.qkv()
    meta = oracle.build_meta(wl)
    meta["full_idx"][0, :, 0] = [1, 0]
    meta["full_cnt"][0, :, 0] = 2
    meta["mask_idx"][0, :, 0] = -1
    meta["mask_cnt"][0, :, 0] = 0
    O, L = oracle.fwd(wl, q, k, v, meta)
    Oref, Lref = _sdpa(_f64(q), _f64(k), _f64(v), wl.scale, False)
    assert np.max(np.abs(O - Oref)) <= 1e-12 and np.max(np.abs(L - Lref)) <= 1e-12
