"""CPU oracle for the block-sparse attention forward and its backward -- TEST
INFRASTRUCTURE ONLY.

Loads ``bsattn_oracle.c`` (plain C, fp64; compiled here with gcc) through
ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library,
and nothing in the product path imports it.

Functions follow the varlen block-sparsity pull request (flash-attention
#2224, description and review) for the metadata layout and the block-sparse
learning note ("Dense FlashAttention vs Block-Sparse Attention", section 2) for
the reversed, -1-padded index lists; the C file's header lists each source and
every reading taken where the pages leave a step open.  The backward (numpy,
fp64: ``bwd_f64`` and its per-tile and per-head forms) differentiates the same definition;
it is pinned by central finite differences and fp64 torch autograd, and the
per-tile and per-head forms by the dense one (tests/test_oracle_bwd.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsattn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.POINTER(ctypes.c_int32)


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
                ("varlen", ctypes.c_int32), ("num_m", ctypes.c_int32), ("num_n", ctypes.c_int32),
                ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("cu_q", _P), ("cu_k", _P), ("kv_valid_len", _P), ("vl_stride", ctypes.c_int32),
                ("kind", ctypes.c_int32), ("window_left", ctypes.c_int32),
                ("sink_tokens", ctypes.c_int32), ("prefix_len", ctypes.c_int32),
                ("doc_q", _P), ("doc_k", _P)]


class Meta(ctypes.Structure):
    _fields_ = [("full_cnt", _P), ("full_idx", _P), ("mask_cnt", _P), ("mask_idx", _P),
                ("cu_total_m_blocks", _P), ("cu_block_idx_offsets", _P),
                ("total_m_blocks", ctypes.c_int32), ("total_n_blocks", ctypes.c_int32)]


def build(force: bool = False) -> str:
    """Compile the oracle into liboracle.so next to its source."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = f"{_LIB}.tmp.{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                    "-lm", "-lpthread"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load(path=None):
    global _lib
    with _lock:
        if _lib is None or path is not None:
            if path is None:
                build()
            lib = ctypes.CDLL(path or _LIB)
            lib.oracle_varlen_offsets.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Meta)]
            lib.oracle_varlen_offsets.restype = ctypes.c_int
            lib.oracle_build_meta.argtypes = [ctypes.POINTER(Problem), ctypes.c_void_p,
                                              ctypes.POINTER(Meta), ctypes.c_int]
            lib.oracle_build_meta.restype = ctypes.c_int
            lib.oracle_fwd_rows.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Meta),
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_double, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_int]
            lib.oracle_fwd_rows.restype = ctypes.c_int
            _lib = lib
    return _lib


def _use_library(path=None):
    """Point this module at another compiled copy of the oracle (the mutation
    tests use it to check that planted mistakes are caught); None restores the
    library built from bsattn_oracle.c."""
    global _lib
    if path is None:
        with _lock:
            _lib = None
        _load()
    else:
        _load(path)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


class _Holder:
    """Keeps the numpy arrays behind a Problem alive while C uses them."""

    def __init__(self, wl):
        self.cu_q = np.ascontiguousarray(wl.cu_seqlens_q, dtype=np.int32)
        self.cu_k = np.ascontiguousarray(wl.cu_seqlens_k, dtype=np.int32)
        self.vl = (None if wl.kv_valid_len is None
                   else np.ascontiguousarray(wl.kv_valid_len, dtype=np.int32))
        self.dq = None if wl.doc_id_q is None else np.ascontiguousarray(wl.doc_id_q, np.int32)
        self.dk = None if wl.doc_id_k is None else np.ascontiguousarray(wl.doc_id_k, np.int32)
        self.p = Problem(B=wl.B, H=wl.H, D=wl.D, varlen=int(wl.varlen), num_m=wl.num_m,
                         num_n=wl.num_n, tile_m=wl.tile_m, tile_n=wl.tile_n,
                         cu_q=_ptr(self.cu_q), cu_k=_ptr(self.cu_k), kv_valid_len=_ptr(self.vl),
                         vl_stride=(0 if self.vl is None else self.vl.shape[-1]),
                         kind=wl.kind, window_left=wl.window_left, sink_tokens=wl.sink_tokens,
                         prefix_len=wl.prefix_len, doc_q=_ptr(self.dq), doc_k=_ptr(self.dk))


def meta_shapes(wl):
    """Shapes of (cnt, idx) arrays: batched [B,H,num_m] / [B,H,num_m,num_n];
    varlen [H,total_m_blocks] / [H,total_n_blocks]."""
    if wl.varlen:
        return (wl.H, wl.total_m_blocks), (wl.H, wl.total_n_blocks)
    return (wl.B, wl.H, wl.num_m), (wl.B, wl.H, wl.num_m, wl.num_n)


def build_meta(wl, block_map=None, threads=None) -> dict:
    """Metadata lists for workload `wl` (its own block map unless one is given)."""
    lib = _load()
    hold = _Holder(wl)
    bm = np.ascontiguousarray(wl.block_map if block_map is None else block_map, dtype=np.uint8)
    cs, is_ = meta_shapes(wl)
    out = {"full_cnt": np.empty(cs, np.int32), "full_idx": np.empty(is_, np.int32),
           "mask_cnt": np.empty(cs, np.int32), "mask_idx": np.empty(is_, np.int32),
           "cu_total_m_blocks": np.zeros(wl.B + 1, np.int32),
           "cu_block_idx_offsets": np.zeros(wl.B + 1, np.int32)}
    mt = Meta(full_cnt=_ptr(out["full_cnt"]), full_idx=_ptr(out["full_idx"]),
              mask_cnt=_ptr(out["mask_cnt"]), mask_idx=_ptr(out["mask_idx"]),
              cu_total_m_blocks=_ptr(out["cu_total_m_blocks"]),
              cu_block_idx_offsets=_ptr(out["cu_block_idx_offsets"]),
              total_m_blocks=0, total_n_blocks=0)
    rc = lib.oracle_build_meta(ctypes.byref(hold.p), bm.ctypes.data, ctypes.byref(mt),
                               threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_build_meta rejected the problem")
    if wl.varlen:
        out["total_m_blocks"], out["total_n_blocks"] = mt.total_m_blocks, mt.total_n_blocks
    return out


def tile_rows(wl):
    """Every Q-tile row as (row index, map slice, num_n(b)).  Row indices follow
    the count arrays: batched (b, h, m) -> (b * H + h) * num_m + m, varlen
    (h, packed tile T) -> h * total_m_blocks + T; the map slice is where that
    row's num_n(b) selection bytes sit in the block map."""
    out = []
    if not wl.varlen:
        for b in range(wl.B):
            for h in range(wl.H):
                for m in range(wl.num_m):
                    out.append(((b * wl.H + h) * wl.num_m + m, (b, h, m, slice(0, wl.num_n)), wl.num_n))
        return out
    tm = [-(-int(s) // wl.tile_m) for s in wl.seqlens_q]
    nn = [-(-int(s) // wl.tile_n) for s in wl.seqlens_k]
    offs = wl.map_row_offsets()
    cum = np.concatenate([[0], np.cumsum(tm)]).astype(np.int64)
    for h in range(wl.H):
        for b in range(wl.B):
            for m in range(tm[b]):
                base = int(offs[b]) + m * nn[b]
                out.append((h * int(cum[-1]) + int(cum[b]) + m, (h, slice(base, base + nn[b])), nn[b]))
    return out


def expand_blocks(block_map, q_block_tiles, kv_block_tiles, num_m, num_n):
    """Per-tile map [B, H, num_m, num_n] of a map given per sparse block of
    q_block_tiles x kv_block_tiles tiles ("[CuTe,Flex] varlen blocksparsity",
    flash-attention #2224, q_subtile_factor; "[feat] VSA-256 fastpath",
    FastVideo #1354: each 256-token block runs as 128-token tiles): tile (m, n)
    takes block (m // q_block_tiles, n // kv_block_tiles)."""
    bm = np.asarray(block_map)
    out = np.zeros(bm.shape[:2] + (num_m, num_n), dtype=bm.dtype)
    for m in range(num_m):
        for n in range(num_n):
            out[:, :, m, n] = bm[:, :, m // q_block_tiles, n // kv_block_tiles]
    return out


def split_valid_len(valid_blocks, kv_block_tiles, num_n, tile=128):
    """Per-tile valid lengths [B, num_n] of lengths given per sparse KV block: tile
    j of a block keeps clamp(v - tile * j, 0, tile) keys (the VSA split of a
    256-token block into min(v, 128) and v - min(v, 128), FastVideo #1354)."""
    vb = np.asarray(valid_blocks, dtype=np.int64)
    out = np.zeros((vb.shape[0], num_n), np.int32)
    for n in range(num_n):
        v = vb[:, n // kv_block_tiles] - tile * (n % kv_block_tiles)
        out[:, n] = np.clip(v, 0, tile)
    return out


def map_from_bitmask(wl, words, words_per_row):
    """The block map that packed 32-bit selection words describe ("feat(prims-ts):
    support proxy-compensated block-sparse attention", FlashInfer #4872, bitmask
    format): one bit per KV tile of a row, bit n % 32 of word n // 32 (least
    significant bit first -- a reading: the page does not fix the bit order), and
    bits past the row's num_n(b) tiles ignored."""
    words = np.asarray(words, dtype=np.uint32).reshape(-1, words_per_row)
    bm = np.zeros_like(wl.block_map)
    for r, sl, nn in tile_rows(wl):
        n = np.arange(min(nn, 32 * words_per_row))
        bits = (words[r, n >> 5] >> (n & 31).astype(np.uint32)) & 1
        row = bm[sl]
        row[: n.size] = bits.astype(bm.dtype)
        bm[sl] = row
    return bm


def map_from_bsr(wl, indptr, indices):
    """The block map that BSR rows describe (same page: canonical block_indptr /
    block_indices): row r selects the KV tiles indices[indptr[r]:indptr[r+1]], in
    any order, each once however often it is listed.  Readings: an id outside
    [0, num_n(b)) selects nothing, and a row whose end lies below its start
    selects nothing."""
    indptr = np.asarray(indptr, dtype=np.int64)
    indices = np.asarray(indices, dtype=np.int64)
    bm = np.zeros_like(wl.block_map)
    for r, sl, nn in tile_rows(wl):
        a, z = int(indptr[r]), int(indptr[r + 1])
        if z < a:
            continue
        ids = indices[a:z]
        ids = ids[(ids >= 0) & (ids < nn)]
        row = bm[sl]
        row[ids] = 1
        bm[sl] = row
    return bm


def varlen_offsets(wl):
    """(cu_total_m_blocks, cu_block_idx_offsets) for a varlen workload."""
    lib = _load()
    hold = _Holder(wl)
    cm = np.zeros(wl.B + 1, np.int32)
    cn = np.zeros(wl.B + 1, np.int32)
    mt = Meta(cu_total_m_blocks=_ptr(cm), cu_block_idx_offsets=_ptr(cn))
    if lib.oracle_varlen_offsets(ctypes.byref(hold.p), ctypes.byref(mt)) != 0:
        raise ValueError("bad sequence lengths")
    return cm, cn


def fwd_rows(wl, q, k, v, meta, tok, head, threads=None):
    """O (fp64 [n, D]) and LSE (fp64 [n]) for packed query rows `tok`, heads `head`.

    q/k/v are raw bf16 bits (uint16) in the workload's layout; `meta` is a dict
    as returned by build_meta (lists of this oracle, never of the CUDA path)."""
    lib = _load()
    hold = _Holder(wl)
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    head = np.ascontiguousarray(head, dtype=np.int32)
    n = tok.size
    o = np.empty((n, wl.D), np.float64)
    lse = np.empty(n, np.float64)
    arrs = {key: np.ascontiguousarray(meta[key], dtype=np.int32)
            for key in ("full_cnt", "full_idx", "mask_cnt", "mask_idx",
                        "cu_total_m_blocks", "cu_block_idx_offsets")}
    mt = Meta(full_cnt=_ptr(arrs["full_cnt"]), full_idx=_ptr(arrs["full_idx"]),
              mask_cnt=_ptr(arrs["mask_cnt"]), mask_idx=_ptr(arrs["mask_idx"]),
              cu_total_m_blocks=_ptr(arrs["cu_total_m_blocks"]),
              cu_block_idx_offsets=_ptr(arrs["cu_block_idx_offsets"]),
              total_m_blocks=int(meta.get("total_m_blocks", 0)),
              total_n_blocks=int(meta.get("total_n_blocks", 0)))
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    rc = lib.oracle_fwd_rows(ctypes.byref(hold.p), ctypes.byref(mt), q.ctypes.data,
                             k.ctypes.data, v.ctypes.data, float(wl.scale), n,
                             tok.ctypes.data, head.ctypes.data, o.ctypes.data, lse.ctypes.data,
                             threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_fwd_rows rejected a row")
    return o, lse


def fwd(wl, q, k, v, meta, threads=None):
    """Every query row of every head.

    Returns O as fp64 in q's layout and LSE as fp64 in the library's layout:
    batched [B, H, S_q], varlen [H, total_q]."""
    rows = wl.rows_q
    tok = np.tile(np.arange(rows, dtype=np.int32), wl.H)
    head = np.repeat(np.arange(wl.H, dtype=np.int32), rows)
    o, lse = fwd_rows(wl, q, k, v, meta, tok, head, threads)
    o = o.reshape(wl.H, rows, wl.D).transpose(1, 0, 2)           # [rows, H, D]
    lse = lse.reshape(wl.H, rows)                                  # [H, rows]
    if wl.varlen:
        return np.ascontiguousarray(o), np.ascontiguousarray(lse)
    S = int(wl.seqlens_q[0])
    o = o.reshape(wl.B, S, wl.H, wl.D)
    lse = lse.reshape(wl.H, wl.B, S).transpose(1, 0, 2)            # [B, H, S]
    return np.ascontiguousarray(o), np.ascontiguousarray(lse)


# ---- proxy compensation ("feat(prims-ts): support proxy-compensated block-sparse
# attention", FlashInfer #4872): selected blocks exact, each omitted KV block
# represented by its arithmetic-mean K and summed V, the softmax denominator
# counting the block's true number of keys.  Batched, mask kind none.

def _widen(bits):
    """bf16 bits -> float64 (exact)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def kv_summaries(wl, k, v):
    """Per (b, KV tile n, h): mean of the tile's keys and sum of its values over
    the keys j < seqlen_k, in fp64.  Returns (k_mean, v_sum) [B, num_n, H, D]."""
    kf, vf = _widen(k), _widen(v)
    B, S, H, D = kf.shape
    nn = -(-S // wl.tile_n)
    km = np.zeros((B, nn, H, D))
    vs = np.zeros((B, nn, H, D))
    for n in range(nn):
        j0, j1 = n * wl.tile_n, min((n + 1) * wl.tile_n, S)
        km[:, n] = kf[:, j0:j1].mean(axis=1)
        vs[:, n] = vf[:, j0:j1].sum(axis=1)
    return km, vs


def fwd_proxy(wl, q, k, v, k_sum, v_sum, sel_map):
    """Proxy-compensated forward, fp64.  sel_map [B, H, num_m, num_n] marks the
    exactly computed tiles; k_sum / v_sum [B, num_n, H, D] are the summaries the
    kernel is given (bf16 bits, or float64).  For row i of (b, h): E = keys of the selected
    tiles below seqlen_k, O = unselected tiles n < num_n with w_n keys each;
    den = sum_E e^{s_j} + sum_O w_n e^{t_n}, out = (sum_E e^{s_j} v_j +
    sum_O e^{t_n} v_sum_n) / den, lse = ln den (s_j = scale q.k_j,
    t_n = scale q.k_sum_n).  Returns O [B, S_q, H, D] and LSE [B, H, S_q]."""
    qf, kf, vf = _widen(q), _widen(k), _widen(v)
    # summaries as bf16 bits (what the kernel reads) or as exact float64 values
    ks = _widen(k_sum) if np.asarray(k_sum).dtype == np.uint16 else np.asarray(k_sum, np.float64)
    vs = _widen(v_sum) if np.asarray(v_sum).dtype == np.uint16 else np.asarray(v_sum, np.float64)
    B, Sq, H, D = qf.shape
    Sk = kf.shape[1]
    tm, tn = wl.tile_m, wl.tile_n
    nn = -(-Sk // tn)
    w = np.array([min(tn, Sk - n * tn) for n in range(nn)], np.float64)
    out = np.zeros((B, Sq, H, D))
    lse = np.zeros((B, H, Sq))
    tile_of_key = np.arange(Sk) // tn
    for b in range(B):
        for h in range(H):
            s = wl.scale * qf[b, :, h] @ kf[b, :, h].T                   # [Sq, Sk]
            t = wl.scale * qf[b, :, h] @ ks[b, :, h].T                   # [Sq, nn]
            sel = np.asarray(sel_map[b, h], dtype=bool)                  # [num_m, nn]
            row_sel = sel[np.arange(Sq) // tm]                           # [Sq, nn]
            exact = row_sel[:, tile_of_key]                              # [Sq, Sk]
            s = np.where(exact, s, -np.inf)
            t = np.where(row_sel, -np.inf, t)
            m = np.maximum(s.max(axis=1), t.max(axis=1))[:, None]
            es = np.exp(s - m)
            et = np.exp(t - m)
            den = es.sum(axis=1) + (et * w[None]).sum(axis=1)
            num = es @ vf[b, :, h] + et @ vs[b, :, h]
            out[b, :, h] = num / den[:, None]
            lse[b, h] = m[:, 0] + np.log(den)
    return out, lse


def fwd_proxy_rows(wl, q, k, v, k_sum, v_sum, sel_map, tok, head, batch=None):
    """fwd_proxy's definition for selected rows only: row tok[r] of head head[r]
    (of sequence batch[r], default 0).  Rows are grouped by their Q tile, whose
    selected tiles' keys enter exactly and whose other tiles enter as the
    weighted summaries, so a long sequence needs no [S_q, S_k] matrix.  Returns
    O [R, D] and LSE [R] (natural log), fp64."""
    ks = _widen(k_sum) if np.asarray(k_sum).dtype == np.uint16 else np.asarray(k_sum, np.float64)
    vs = _widen(v_sum) if np.asarray(v_sum).dtype == np.uint16 else np.asarray(v_sum, np.float64)
    tok = np.asarray(tok, np.int64)
    head = np.asarray(head, np.int64)
    batch = np.zeros_like(tok) if batch is None else np.asarray(batch, np.int64)
    Sk = k.shape[1]
    D = q.shape[3]
    tm, tn = wl.tile_m, wl.tile_n
    nn = -(-Sk // tn)
    w = np.array([min(tn, Sk - n * tn) for n in range(nn)], np.float64)
    out = np.zeros((tok.size, D))
    lse = np.zeros(tok.size)
    groups = {}
    for r in range(tok.size):
        groups.setdefault((int(batch[r]), int(head[r]), int(tok[r]) // tm), []).append(r)
    for (b, h, m), rows in groups.items():
        rows = np.asarray(rows)
        sel = np.asarray(sel_map[b, h, m], dtype=bool)               # [nn]
        keys = np.concatenate([np.arange(n * tn, min((n + 1) * tn, Sk)) for n in np.flatnonzero(sel)]
                              ) if sel.any() else np.zeros(0, np.int64)
        qf = _widen(q[b, tok[rows], h])                              # [R, D]
        s = wl.scale * qf @ _widen(k[b, keys, h]).T                  # exact keys
        t = wl.scale * qf @ ks[b, ~sel, h].T                         # summaries of the others
        mx = np.maximum(s.max(axis=1, initial=-np.inf), t.max(axis=1, initial=-np.inf))[:, None]
        es, et = np.exp(s - mx), np.exp(t - mx)
        den = es.sum(axis=1) + (et * w[~sel][None]).sum(axis=1)
        num = es @ _widen(v[b, keys, h]) + et @ vs[b, ~sel, h]
        out[rows] = num / den[:, None]
        lse[rows] = mx[:, 0] + np.log(den)
    return out, lse


# ---- backward (the gradients of the forward defined above; batched) ---------

def allowed_mask(wl, meta, b, h):
    """bool [S_q, S_k]: key j is in query row i's allowed set for (b, h): j in a
    full-list tile of row i's Q tile and below seqlen_k, or in a mask-list tile and
    also passing the token predicate and the tile's valid length."""
    Sq, Sk = int(wl.seqlens_q[b]), int(wl.seqlens_k[b])
    tm, tn = wl.tile_m, wl.tile_n
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    if wl.kind == 0:
        pred = np.ones((Sq, Sk), bool)
    elif wl.kind == 1:
        pred = j <= i
    elif wl.kind == 2:
        pred = (j <= i) & ((i - j < wl.window_left) | (j < wl.sink_tokens))
    elif wl.kind == 4:
        pred = (j < wl.prefix_len) | (j <= i)
    elif wl.kind == 3:
        dq = np.asarray(wl.doc_id_q)[b * Sq:(b + 1) * Sq]
        dk = np.asarray(wl.doc_id_k)[b * Sk:(b + 1) * Sk]
        pred = dq[:, None] == dk[None, :]
    else:
        raise ValueError(wl.kind)
    out = np.zeros((Sq, Sk), bool)
    for m in range(-(-Sq // tm)):
        r0, r1 = m * tm, min((m + 1) * tm, Sq)
        for key, masked in (("full", False), ("mask", True)):
            cnt = int(meta[key + "_cnt"][b, h, m])
            for n in meta[key + "_idx"][b, h, m, :cnt]:
                c0, c1 = int(n) * tn, min((int(n) + 1) * tn, Sk)
                if c1 <= c0:
                    continue
                blk = np.ones((r1 - r0, c1 - c0), bool)
                if masked:
                    blk &= pred[r0:r1, c0:c1]
                    if wl.kv_valid_len is not None:
                        blk &= (np.arange(c1 - c0) < int(wl.kv_valid_len[b, int(n)]))[None, :]
                out[r0:r1, c0:c1] |= blk
    return out


def _probs(wl, meta, b, h, qf, kf):
    A = allowed_mask(wl, meta, b, h)
    s = np.where(A, wl.scale * qf[b, :, h] @ kf[b, :, h].T, -np.inf)
    mx = s.max(axis=1, keepdims=True)
    mx = np.where(np.isfinite(mx), mx, 0.0)
    e = np.where(A, np.exp(s - mx), 0.0)
    den = e.sum(axis=1, keepdims=True)
    return np.divide(e, den, out=np.zeros_like(e), where=den > 0)


def fwd_f64(wl, meta, qf, kf, vf):
    """O = P V over the allowed keys, for float64 inputs [B, S, H, D] (batched)."""
    out = np.zeros(qf.shape[:3] + (vf.shape[3],))
    for b in range(wl.B):
        for h in range(wl.H):
            out[b, :, h] = _probs(wl, meta, b, h, qf, kf) @ vf[b, :, h]
    return out


def bwd_f64(wl, meta, qf, kf, vf, gf):
    """Gradients of fwd_f64 for upstream gradient gf (float64, batched):
    P = softmax over the allowed keys of scale q.k (a row with none has P = 0),
    O = P V,  dV = P^T dO,  dP = dO V^T,  D_i = sum_d dO_i O_i,
    dS = P (dP - D),  dQ = scale dS K,  dK = scale dS^T Q."""
    dq, dk, dv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    for b in range(wl.B):
        for h in range(wl.H):
            P = _probs(wl, meta, b, h, qf, kf)
            O = P @ vf[b, :, h]
            g = gf[b, :, h]
            dv[b, :, h] = P.T @ g
            dP = g @ vf[b, :, h].T
            Dv = (g * O).sum(axis=1, keepdims=True)
            dS = P * (dP - Dv)
            dq[b, :, h] = wl.scale * dS @ kf[b, :, h]
            dk[b, :, h] = wl.scale * dS.T @ qf[b, :, h]
    return dq, dk, dv


def seq_view(wl, meta, b):
    """Sequence b of a varlen workload as a batched workload of one sequence with
    its own slice of the lists (varlen layout, flash-attention #2224: counts
    [H, total_m_blocks] from cu_total_m_blocks[b], indices [H, total_n_blocks]
    with row (b, m) at cu_block_idx_offsets[b] + m num_n(b)).  Returns (view,
    meta of the view, packed q-row slice, packed k-row slice)."""
    from dataclasses import replace
    sq, sk = int(wl.seqlens_q[b]), int(wl.seqlens_k[b])
    nm, nn = -(-sq // wl.tile_m), -(-sk // wl.tile_n)
    t0 = int(meta["cu_total_m_blocks"][b])
    off = int(meta["cu_block_idx_offsets"][b])
    mb = {}
    for key in ("full", "mask"):
        mb[key + "_cnt"] = np.asarray(meta[key + "_cnt"])[:, t0:t0 + nm][None]
        mb[key + "_idx"] = np.asarray(meta[key + "_idx"])[:, off:off + nm * nn].reshape(wl.H, nm, nn)[None]
    cq, ck = wl.cu_seqlens_q, wl.cu_seqlens_k
    qs, ks = slice(int(cq[b]), int(cq[b + 1])), slice(int(ck[b]), int(ck[b + 1]))
    view = replace(wl, B=1, varlen=False, seqlens_q=np.array([sq], np.int32),
                   seqlens_k=np.array([sk], np.int32),
                   block_map=np.zeros((1, wl.H, nm, nn), np.uint8),
                   kv_valid_len=None if wl.kv_valid_len is None else np.asarray(wl.kv_valid_len)[b:b + 1],
                   doc_id_q=None if wl.doc_id_q is None else np.asarray(wl.doc_id_q)[qs],
                   doc_id_k=None if wl.doc_id_k is None else np.asarray(wl.doc_id_k)[ks])
    return view, mb, qs, ks


def bwd(wl, q, k, v, meta, dout):
    """bwd_f64 on bf16 inputs (raw bits); dQ, dK, dV in the layouts of q, k, v.
    Varlen: every sequence on its own (no key of one sequence is in another's
    allowed sets), through seq_view."""
    if not wl.varlen:
        return bwd_f64(wl, meta, _widen(q), _widen(k), _widen(v), _widen(dout))
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(wl.B):
        view, mb, qs, ks = seq_view(wl, meta, b)
        if qs.stop == qs.start or ks.stop == ks.start:
            continue
        g = bwd_f64(view, mb, _widen(q[qs])[None], _widen(k[ks])[None], _widen(v[ks])[None],
                    _widen(dout[qs])[None])
        dq[qs], dk[ks], dv[ks] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv


# ---- per-tile backward, for sampled checks at full size.  The same definition
# as bwd_f64 (gradients of softmax attention over each row's allowed keys),
# evaluated for one Q tile's rows or one KV tile's keys: a row's probabilities
# involve only the keys its Q tile's lists name, so nothing outside them is
# formed, and only the slices used are widened from bf16.

def _pred(wl, b, i, j):
    """Token predicate of the mask kind for query rows i (column vector) and keys
    j (row vector) of sequence b, as in allowed_mask."""
    if wl.kind == 0:
        return np.ones((i.shape[0], j.shape[1]), bool)
    if wl.kind == 1:
        return j <= i
    if wl.kind == 2:
        return (j <= i) & ((i - j < wl.window_left) | (j < wl.sink_tokens))
    if wl.kind == 4:
        return (j < wl.prefix_len) | (j <= i)
    if wl.kind == 3:
        Sq, Sk = int(wl.seqlens_q[b]), int(wl.seqlens_k[b])
        dq = np.asarray(wl.doc_id_q)[b * Sq:(b + 1) * Sq]
        dk = np.asarray(wl.doc_id_k)[b * Sk:(b + 1) * Sk]
        return dq[i[:, 0]][:, None] == dk[j[0]][None, :]
    raise ValueError(wl.kind)


def tile_allowed(wl, meta, b, h, m):
    """Q tile m of (b, h): (r0, r1, keys, A) with rows [r0, r1), `keys` the
    ascending key indices of the tiles its lists name, and A bool [rows, keys]
    the allowed pairs (full tiles: keys below seqlen_k; mask tiles: also the
    token predicate and the tile's valid length); a tile named twice is one
    tile whose allowed pairs are the union."""
    Sq, Sk = int(wl.seqlens_q[b]), int(wl.seqlens_k[b])
    tm, tn = wl.tile_m, wl.tile_n
    r0, r1 = m * tm, min((m + 1) * tm, Sq)
    i = np.arange(r0, r1)[:, None]
    blocks = {}
    for key, masked in (("full", False), ("mask", True)):
        cnt = int(meta[key + "_cnt"][b, h, m])
        for n in meta[key + "_idx"][b, h, m, :cnt]:
            n = int(n)
            c0, c1 = n * tn, min((n + 1) * tn, Sk)
            if c1 <= c0:
                continue
            blk = np.ones((r1 - r0, c1 - c0), bool)
            if masked:
                blk &= _pred(wl, b, i, np.arange(c0, c1)[None, :])
                if wl.kv_valid_len is not None:
                    blk &= (np.arange(c1 - c0) < int(wl.kv_valid_len[b, n]))[None, :]
            blocks[n] = blocks[n] | blk if n in blocks else blk
    if not blocks:
        return r0, r1, np.zeros(0, np.int64), np.zeros((r1 - r0, 0), bool)
    ns = sorted(blocks)
    keys = np.concatenate([np.arange(n * tn, n * tn + blocks[n].shape[1]) for n in ns])
    return r0, r1, keys, np.concatenate([blocks[n] for n in ns], axis=1)


def _tile_grads(wl, q, k, v, dout, meta, b, h, m):
    """For Q tile m: rows, keys, P, dS (fp64) and the widened q rows / keys."""
    r0, r1, keys, A = tile_allowed(wl, meta, b, h, m)
    qf = _widen(q[b, r0:r1, h])
    kf, vf = _widen(k[b, keys, h]), _widen(v[b, keys, h])
    g = _widen(dout[b, r0:r1, h])
    s = np.where(A, wl.scale * (qf @ kf.T), -np.inf)
    mx = s.max(axis=1, keepdims=True) if keys.size else np.zeros((r1 - r0, 1))
    mx = np.where(np.isfinite(mx), mx, 0.0)
    e = np.where(A, np.exp(s - mx), 0.0)
    den = e.sum(axis=1, keepdims=True)
    P = np.divide(e, den, out=np.zeros_like(e), where=den > 0)
    O = P @ vf
    dS = P * (g @ vf.T - (g * O).sum(axis=1, keepdims=True))
    return r0, r1, keys, P, dS, qf, kf, g


def bwd_dq_tile(wl, q, k, v, dout, meta, b, h, m):
    """dQ (fp64 [rows, D]) of Q tile m of (b, h); inputs are raw bf16 bits in the
    batched layout, `meta` the oracle's own lists."""
    _, _, keys, _, dS, _, kf, _ = _tile_grads(wl, q, k, v, dout, meta, b, h, m)
    return wl.scale * (dS @ kf) if keys.size else np.zeros((dS.shape[0], q.shape[3]))


def bwd_head(wl, q, k, v, dout, meta, b, h):
    """(dQ, dK, dV) (fp64 [S_q, D], [S_k, D], [S_k, D]) of head h of sequence b:
    bwd_f64's definition evaluated one Q tile at a time.  Each Q tile's rows
    give their dQ rows directly and add P^T dO and scale dS^T Q into the dV and
    dK rows of the keys its lists name, so a head of a long sequence needs no
    dense [S_q, S_k] matrix."""
    Sq, Sk = int(wl.seqlens_q[b]), int(wl.seqlens_k[b])
    D = q.shape[3]
    dq, dk, dv = np.zeros((Sq, D)), np.zeros((Sk, D)), np.zeros((Sk, D))
    for m in range(-(-Sq // wl.tile_m)):
        r0, r1, keys, P, dS, qf, kf, g = _tile_grads(wl, q, k, v, dout, meta, b, h, m)
        if not keys.size:
            continue
        dq[r0:r1] = wl.scale * (dS @ kf)
        dv[keys] += P.T @ g
        dk[keys] += wl.scale * (dS.T @ qf)
    return dq, dk, dv


def bwd_dkdv_tile(wl, q, k, v, dout, meta, b, h, n):
    """(dK, dV) (fp64 [keys, D] each) of KV tile n of (b, h): the sums over every Q
    tile whose lists name n."""
    Sk = int(wl.seqlens_k[b])
    c0, c1 = n * wl.tile_n, min((n + 1) * wl.tile_n, Sk)
    D = q.shape[3]
    dk, dv = np.zeros((c1 - c0, D)), np.zeros((c1 - c0, D))
    for m in range(meta["full_cnt"].shape[2]):
        named = any(n in meta[key + "_idx"][b, h, m, :int(meta[key + "_cnt"][b, h, m])]
                    for key in ("full", "mask"))
        if not named:
            continue
        _, _, keys, P, dS, qf, _, g = _tile_grads(wl, q, k, v, dout, meta, b, h, m)
        sel = (keys >= c0) & (keys < c1)
        pos = keys[sel] - c0
        dv[pos] += P[:, sel].T @ g
        dk[pos] += wl.scale * (dS[:, sel].T @ qf)
    return dk, dv
