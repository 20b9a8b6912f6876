"""Dense brute force used to pin the oracle on tiny inputs (tests only).

The block lists are expanded to a token-level boolean matrix per (sequence,
head), and attention is then the textbook masked softmax over the whole
S_q x S_k score matrix, computed with numpy in fp64.  This shares nothing with
the oracle's C code: it has no per-row gather, no per-tile loop and no
two-pass running state.
"""
import numpy as np

from workloads import bf16_bits_to_f32
from workloads.configs import (MASK_CAUSAL, MASK_DOCUMENT, MASK_NONE, MASK_PREFIX,
                               MASK_SLIDING_WINDOW)


def _cdiv(a, b):
    return -(-a // b)


def mask_matrix(wl, b, i, j):
    """mask_mod of workload wl on broadcastable sequence-local positions i, j."""
    if wl.kind == MASK_NONE:
        return np.ones(np.broadcast(i, j).shape, bool)
    if wl.kind == MASK_CAUSAL:
        return j <= i
    if wl.kind == MASK_SLIDING_WINDOW:
        return (j <= i) & ((i - j < wl.window_left) | (j < wl.sink_tokens))
    if wl.kind == MASK_PREFIX:
        return (j < wl.prefix_len) | (j <= i)
    if wl.kind == MASK_DOCUMENT:
        dq = wl.doc_id_q[wl.cu_seqlens_q[b] + i]
        dk = wl.doc_id_k[wl.cu_seqlens_k[b] + j]
        return dq == dk
    raise ValueError(wl.kind)


def row_lists(wl, meta, b, h, m):
    """(full list, mask list) of row (b, h, m), first `cnt` entries only."""
    if wl.varlen:
        nn = _cdiv(int(wl.seqlens_k[b]), wl.tile_n)
        cnt_at = (h, int(meta["cu_total_m_blocks"][b]) + m)
        base = int(meta["cu_block_idx_offsets"][b]) + m * nn
        fi = meta["full_idx"][h, base: base + nn]
        mi = meta["mask_idx"][h, base: base + nn]
    else:
        cnt_at = (b, h, m)
        fi = meta["full_idx"][b, h, m]
        mi = meta["mask_idx"][b, h, m]
    return (fi[: int(meta["full_cnt"][cnt_at])].tolist(),
            mi[: int(meta["mask_cnt"][cnt_at])].tolist())


def allowed(wl, meta, b, h):
    """Token-level allowed matrix [S_q(b), S_k(b)] expanded from the lists."""
    sq, sk = int(wl.seqlens_q[b]), int(wl.seqlens_k[b])
    A = np.zeros((sq, sk), bool)
    for m in range(_cdiv(sq, wl.tile_m)):
        r0, r1 = m * wl.tile_m, min((m + 1) * wl.tile_m, sq)
        full, mask = row_lists(wl, meta, b, h, m)
        for n in full:
            A[r0:r1, n * wl.tile_n: min((n + 1) * wl.tile_n, sk)] = True
        for n in mask:
            c0, c1 = n * wl.tile_n, min((n + 1) * wl.tile_n, sk)
            ii = np.arange(r0, r1)[:, None]
            jj = np.arange(c0, c1)[None, :]
            pred = mask_matrix(wl, b, ii, jj)
            if wl.kv_valid_len is not None:
                pred = pred & (jj - n * wl.tile_n < wl.kv_valid_len[b, n])
            A[r0:r1, c0:c1] |= pred
    return A


def seq_slices(wl, x, cu, b):
    """Rows of sequence b from a q/k/v tensor (batched or packed), as float64 [S, H, D]."""
    if wl.varlen:
        t = x[cu[b]: cu[b + 1]]
    else:
        t = x[b]
    return bf16_bits_to_f32(t).astype(np.float64)


def dense_attention(wl, q, k, v, meta):
    """Returns O (fp64, q's layout) and LSE (fp64, [B,H,S] or [H,total])."""
    cuq, cuk = wl.cu_seqlens_q, wl.cu_seqlens_k
    O = np.zeros(q.shape, np.float64)
    L = (np.zeros((wl.H, wl.rows_q)) if wl.varlen
         else np.zeros((wl.B, wl.H, int(wl.seqlens_q[0]))))
    for b in range(wl.B):
        Q, K, V = seq_slices(wl, q, cuq, b), seq_slices(wl, k, cuk, b), seq_slices(wl, v, cuk, b)
        for h in range(wl.H):
            A = allowed(wl, meta, b, h)
            S = wl.scale * (Q[:, h, :] @ K[:, h, :].T)
            S = np.where(A, S, -np.inf)
            any_ = A.any(axis=1)
            mx = np.where(any_, S.max(axis=1), 0.0)
            P = np.exp(S - mx[:, None])
            den = P.sum(axis=1)
            o = np.where(any_[:, None], (P @ V[:, h, :]) / np.where(any_, den, 1.0)[:, None], 0.0)
            lse = np.where(any_, mx + np.log(np.where(any_, den, 1.0)), -np.inf)
            if wl.varlen:
                O[cuq[b]: cuq[b + 1], h] = o
                L[h, cuq[b]: cuq[b + 1]] = lse
            else:
                O[b, :, h] = o
                L[b, h] = lse
    return O, L
