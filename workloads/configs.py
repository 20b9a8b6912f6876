"""The five benchmark workloads and small randomised variants, built from seeds.

Each workload is a set of inputs to the block-sparse forward: bf16 Q/K/V in
BSHD layout (batched ``[B, S, H, D]`` or varlen-packed ``[total, H, D]``), a
boolean block map over 128x128 tiles, an optional per-KV-tile valid length and
a mask kind with its parameters.  The map layouts follow the varlen
block-sparsity pull request (flash-attention #2224, description): batched maps
are ``[B, H, num_m, num_n]``; varlen maps are packed ``[H, total_n_blocks]``
with sequence b's rows starting at the sum over earlier sequences of
num_m * num_n and each row holding num_n(b) entries.

Seeds: data seed = 1000 + config number, map seed = 2000 + config number.
Streams inside a seed: 0 q, 1 k, 2 v, 3 block map, 4 lengths, 5 scores,
6 valid lengths, 7 document ids.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

TILE = 128

# Mask kinds, numbered as in the C ABI (include/bsattn.h).
MASK_NONE, MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_DOCUMENT, MASK_PREFIX = 0, 1, 2, 3, 4

S_Q, S_K, S_V, S_MAP, S_LEN, S_SCORE, S_VALID, S_DOC, S_DO = range(9)


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class Workload:
    name: str
    B: int
    H: int
    D: int
    varlen: bool
    seqlens_q: np.ndarray            # int32 [B]
    seqlens_k: np.ndarray            # int32 [B]
    block_map: np.ndarray            # uint8, batched [B,H,num_m,num_n] or varlen [H,total_n]
    kind: int
    scale: float
    data_seed: int
    kv_valid_len: Optional[np.ndarray] = None   # int32 [B, num_n_stride]
    window_left: int = 0
    sink_tokens: int = 0
    prefix_len: int = 0
    doc_id_q: Optional[np.ndarray] = None       # int32 per packed q row
    doc_id_k: Optional[np.ndarray] = None       # int32 per packed k row
    tile_m: int = TILE
    tile_n: int = TILE
    notes: str = ""
    extra: dict = field(default_factory=dict)

    # ---- shapes -----------------------------------------------------------
    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens_q)]).astype(np.int32)

    @property
    def cu_seqlens_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens_k)]).astype(np.int32)

    @property
    def rows_q(self) -> int:
        return int(self.seqlens_q.sum())

    @property
    def rows_k(self) -> int:
        return int(self.seqlens_k.sum())

    @property
    def num_m(self) -> int:
        """Batched: Q tiles per sequence.  Varlen: the largest per-sequence count."""
        return max(_cdiv(int(s), self.tile_m) for s in self.seqlens_q)

    @property
    def num_n(self) -> int:
        """Batched: KV tiles per sequence.  Varlen: the largest per-sequence count
        (the row stride of kv_valid_len)."""
        return max(_cdiv(int(s), self.tile_n) for s in self.seqlens_k)

    @property
    def total_m_blocks(self) -> int:
        return sum(_cdiv(int(s), self.tile_m) for s in self.seqlens_q)

    @property
    def total_n_blocks(self) -> int:
        return sum(_cdiv(int(sq), self.tile_m) * _cdiv(int(sk), self.tile_n)
                   for sq, sk in zip(self.seqlens_q, self.seqlens_k))

    def q_shape(self):
        if self.varlen:
            return (self.rows_q, self.H, self.D)
        return (self.B, int(self.seqlens_q[0]), self.H, self.D)

    def k_shape(self):
        if self.varlen:
            return (self.rows_k, self.H, self.D)
        return (self.B, int(self.seqlens_k[0]), self.H, self.D)

    def fill(self, which: str, ptr: int) -> None:
        """Write the bf16 bits of tensor `which` ('q', 'k', 'v', or 'do': the
        upstream gradient of the output, shaped like q) to host memory at ptr."""
        from . import normal_bf16_into
        stream = {"q": S_Q, "k": S_K, "v": S_V, "do": S_DO}[which]
        shape = self.q_shape() if which in ("q", "do") else self.k_shape()
        normal_bf16_into(ptr, int(np.prod(shape)), self.data_seed, stream)

    def tensor(self, which: str) -> np.ndarray:
        shape = self.q_shape() if which in ("q", "do") else self.k_shape()
        out = np.empty(shape, dtype=np.uint16)
        self.fill(which, out.ctypes.data)
        return out

    def qkv(self):
        return self.tensor("q"), self.tensor("k"), self.tensor("v")

    def map_row_offsets(self) -> np.ndarray:
        """Varlen only: where sequence b's rows start inside a packed [total_n] map row."""
        sizes = [_cdiv(int(sq), self.tile_m) * _cdiv(int(sk), self.tile_n)
                 for sq, sk in zip(self.seqlens_q, self.seqlens_k)]
        return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


# ---------------------------------------------------------------------------
# Generic random workload (tests)
# ---------------------------------------------------------------------------

def random_workload(seed: int, B: int, H: int, D: int, seqlens_q: List[int],
                    seqlens_k: Optional[List[int]] = None, varlen: bool = False,
                    density: float = 0.5, kind: int = MASK_CAUSAL, window_left: int = 0,
                    sink_tokens: int = 0, prefix_len: int = 0, valid_len: bool = False,
                    n_docs: int = 3, scale: Optional[float] = None,
                    force_diag: bool = True, name: str = "random", tile_m: int = TILE,
                    tile_n: int = TILE) -> Workload:
    """A seeded workload with Bernoulli(density) block maps.

    For batched workloads seqlens_q (and seqlens_k) must hold B equal lengths.
    tile_m / tile_n: the listed block size (batched only when not 128), which the
    map, the diagonal and the valid lengths (1..tile_n per block) refer to.
    """
    from . import uniform01, u64
    if seqlens_k is None:
        seqlens_k = list(seqlens_q)
    sq = np.asarray(seqlens_q, dtype=np.int32)
    sk = np.asarray(seqlens_k, dtype=np.int32)
    assert len(sq) == B and len(sk) == B
    if not varlen:
        assert len(set(sq.tolist())) == 1 and len(set(sk.tolist())) == 1
    wl = Workload(name=name, B=B, H=H, D=D, varlen=varlen, seqlens_q=sq, seqlens_k=sk,
                  block_map=np.zeros(1, np.uint8), kind=kind,
                  scale=(1.0 / math.sqrt(D)) if scale is None else scale,
                  data_seed=seed, window_left=window_left, sink_tokens=sink_tokens,
                  prefix_len=prefix_len, tile_m=tile_m, tile_n=tile_n)
    assert not varlen or (tile_m == TILE and tile_n == TILE)
    mseed = seed + 1000
    if varlen:
        off = wl.map_row_offsets()
        total_n = int(off[-1])
        u = uniform01(H * total_n, mseed, S_MAP).reshape(H, total_n)
        bm = (u < density).astype(np.uint8)
        if force_diag:
            for b in range(B):
                nm, nn = _cdiv(int(sq[b]), TILE), _cdiv(int(sk[b]), TILE)
                for m in range(min(nm, nn)):
                    bm[:, off[b] + m * nn + m] = 1
        wl.block_map = bm
    else:
        nm, nn = wl.num_m, wl.num_n
        u = uniform01(B * H * nm * nn, mseed, S_MAP).reshape(B, H, nm, nn)
        bm = (u < density).astype(np.uint8)
        if force_diag:
            d = np.arange(min(nm, nn))
            bm[:, :, d, d] = 1
        wl.block_map = bm
    if valid_len:
        nn = wl.num_n
        r = u64(B * nn, mseed, S_VALID).reshape(B, nn)
        wl.kv_valid_len = (1 + (r % tile_n)).astype(np.int32)    # 1..tile_n
    if kind == MASK_DOCUMENT:
        def docs(lengths, stream):
            out = []
            for b, L in enumerate(lengths):
                L = int(L)
                cuts = np.sort(u64(max(n_docs - 1, 0), mseed + b, stream) % max(L, 1))
                ids = np.zeros(L, np.int32)
                for c in cuts:
                    ids[int(c):] += 1
                out.append(ids + 1000 * b)
            return np.concatenate(out).astype(np.int32) if out else np.zeros(0, np.int32)
        wl.doc_id_q = docs(sq, S_DOC)
        wl.doc_id_k = docs(sk, S_DOC) if list(sk) != list(sq) else wl.doc_id_q.copy()
    return wl


# ---------------------------------------------------------------------------
# The five benchmark workloads
# ---------------------------------------------------------------------------

def _cfg1() -> Workload:
    """tiny causal: B=1 H=2 S=256 d=64, causal block map (n <= m)."""
    B, H, S, D = 1, 2, 256, 64
    nm = S // TILE
    bm = np.zeros((B, H, nm, nm), np.uint8)
    for m in range(nm):
        bm[:, :, m, : m + 1] = 1
    return Workload(name="tiny_causal_b1_h2_s256_d64", B=B, H=H, D=D, varlen=False,
                    seqlens_q=np.full(B, S, np.int32), seqlens_k=np.full(B, S, np.int32),
                    block_map=bm, kind=MASK_CAUSAL, scale=1.0 / math.sqrt(D), data_seed=1001)


def _cfg2() -> Workload:
    """batched random: B=2 H=4 S=1024 d=128, Bernoulli(0.3) map, diagonal forced, causal."""
    from . import uniform01
    B, H, S, D = 2, 4, 1024, 128
    nm = S // TILE
    u = uniform01(B * H * nm * nm, 2002, S_MAP).reshape(B, H, nm, nm)
    bm = (u < 0.3).astype(np.uint8)
    d = np.arange(nm)
    bm[:, :, d, d] = 1
    return Workload(name="batched_random_b2_h4_s1024_d128_p0.3", B=B, H=H, D=D, varlen=False,
                    seqlens_q=np.full(B, S, np.int32), seqlens_k=np.full(B, S, np.int32),
                    block_map=bm, kind=MASK_CAUSAL, scale=1.0 / math.sqrt(D), data_seed=1002)


def _cfg3() -> Workload:
    """varlen packed: 8 sequences, lengths ~U[100,4096], H=16 d=128, causal +
    Bernoulli(0.5) below the diagonal, diagonal forced."""
    from . import uniform01
    B, H, D, lo, hi = 8, 16, 128, 100, 4096
    attempt = 0
    while True:
        u = uniform01(B, 2003, S_LEN, offset=attempt * B)
        lens = (lo + np.floor(u * (hi - lo + 1))).astype(np.int32)
        if np.any(lens % TILE != 0):
            break
        attempt += 1
    wl = Workload(name="varlen_8seq_u100_4096_h16_d128_p0.5", B=B, H=H, D=D, varlen=True,
                  seqlens_q=lens, seqlens_k=lens.copy(), block_map=np.zeros(1, np.uint8),
                  kind=MASK_CAUSAL, scale=1.0 / math.sqrt(D), data_seed=1003)
    off = wl.map_row_offsets()
    total_n = int(off[-1])
    u = uniform01(H * total_n, 2003, S_MAP).reshape(H, total_n)
    bm = np.zeros((H, total_n), np.uint8)
    for b in range(B):
        n_b = _cdiv(int(lens[b]), TILE)
        m_idx, n_idx = np.meshgrid(np.arange(n_b), np.arange(n_b), indexing="ij")
        flat = off[b] + m_idx * n_b + n_idx
        sel = np.where(n_idx < m_idx, u[:, flat] < 0.5, n_idx == m_idx)
        bm[:, flat] = sel.astype(np.uint8)
    wl.block_map = bm
    return wl


def _cfg4() -> Workload:
    """video sparse attention: B=1 H=24 S=61440 (240 logical 256-token blocks),
    top-32 logical KV blocks per logical Q block by seeded U(0,1) scores with the
    own block forced, valid length ~U[192,256] per logical KV block; run as
    128-token tiles (each logical block -> two tiles; valid length split as
    min(v,128) and v - min(v,128))."""
    from . import uniform01
    B, H, S, D, NB, TOPK = 1, 24, 61440, 128, 240, 32
    scores = uniform01(H * NB * NB, 2004, S_SCORE).reshape(H, NB, NB)
    ar = np.arange(NB)
    scores[:, ar, ar] = np.inf
    top = np.argsort(-scores, axis=-1, kind="stable")[..., :TOPK]
    logical = np.zeros((H, NB, NB), np.uint8)
    np.put_along_axis(logical, top, 1, axis=-1)
    bm = np.repeat(np.repeat(logical, 2, axis=1), 2, axis=2)[None]      # [1,H,480,480]
    u = uniform01(NB, 2004, S_VALID)
    v = (192 + np.floor(u * 65)).astype(np.int32)                        # 192..256
    child0 = np.minimum(v, TILE)
    child1 = v - child0
    vl = np.stack([child0, child1], axis=1).reshape(1, 2 * NB).astype(np.int32)
    return Workload(name="vsa_b1_h24_s61440_d128_top32of240", B=B, H=H, D=D, varlen=False,
                    seqlens_q=np.full(B, S, np.int32), seqlens_k=np.full(B, S, np.int32),
                    block_map=np.ascontiguousarray(bm), kind=MASK_NONE,
                    scale=1.0 / math.sqrt(D), data_seed=1004, kv_valid_len=vl,
                    extra={"logical_block_valid_len": v, "logical_map": logical})


def _cfg5() -> Workload:
    """long context: B=1 H=32 S=131072 d=128, blocks [m-32, m] plus sink blocks
    {0,1,2,3}; sliding window of 4096 tokens (self included), 512 sink tokens, causal."""
    B, H, S, D = 1, 32, 131072, 128
    nm = S // TILE
    m = np.arange(nm)[:, None]
    n = np.arange(nm)[None, :]
    row = ((n >= m - 32) & (n <= m)) | (n < 4)
    bm = np.broadcast_to(row.astype(np.uint8)[None, None], (B, H, nm, nm)).copy()
    return Workload(name="long_ctx_b1_h32_s131072_d128_win4096_sink4", B=B, H=H, D=D,
                    varlen=False, seqlens_q=np.full(B, S, np.int32),
                    seqlens_k=np.full(B, S, np.int32), block_map=bm,
                    kind=MASK_SLIDING_WINDOW, scale=1.0 / math.sqrt(D), data_seed=1005,
                    window_left=4096, sink_tokens=512)


CONFIGS = {1: _cfg1, 2: _cfg2, 3: _cfg3, 4: _cfg4, 5: _cfg5}


def as_sparse_blocks(wl: Workload) -> Workload:
    """Config 4 stated at its native sparse-block size: the map per 256-token
    logical block (240 x 240 per head) with one valid length per logical KV
    block, listed as 256 x 256 blocks (q/k/v are the same draws)."""
    from dataclasses import replace
    logical = wl.extra["logical_map"]
    return replace(wl, tile_m=2 * TILE, tile_n=2 * TILE,
                   block_map=np.ascontiguousarray(logical[None]),
                   kv_valid_len=np.ascontiguousarray(
                       wl.extra["logical_block_valid_len"].reshape(wl.B, -1).astype(np.int32)),
                   name=wl.name + "_256blocks")


def with_heads(wl: Workload, heads: int) -> Workload:
    """The first `heads` heads of a workload's block map (q/k/v are drawn for the
    new shape): a smaller case with the same sparsity structure, for profiling."""
    from dataclasses import replace
    bm = wl.block_map[:heads] if wl.varlen else wl.block_map[:, :heads]
    return replace(wl, H=heads, block_map=np.ascontiguousarray(bm),
                   name=f"{wl.name}_first{heads}heads")


def make_workload(cfg: int) -> Workload:
    return CONFIGS[cfg]()
