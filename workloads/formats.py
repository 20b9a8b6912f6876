"""Encoders of a boolean block map into the two other selection formats the
metadata entry points accept ("feat(prims-ts): support proxy-compensated
block-sparse attention", FlashInfer #4872, bitmask format): packed 32-bit words
per Q-tile row (bit n % 32 of word n // 32 selects KV tile n) and BSR rows
(block_indptr / block_indices).  Input preparation only."""
import numpy as np


def tile_rows(wl):
    """Every Q-tile row as (row index, map slice, num_n(b)); rows in the order of
    the count arrays (batched (b, h, m) -> (b * H + h) * num_m + m; varlen
    (h, packed tile T) -> h * total_m_blocks + T)."""
    out = []
    if not wl.varlen:
        for b in range(wl.B):
            for h in range(wl.H):
                for m in range(wl.num_m):
                    out.append(((b * wl.H + h) * wl.num_m + m, (b, h, m, slice(0, wl.num_n)), wl.num_n))
        return out
    tm = [-(-int(s) // wl.tile_m) for s in wl.seqlens_q]
    nn = [-(-int(s) // wl.tile_n) for s in wl.seqlens_k]
    sizes = [a * b for a, b in zip(tm, nn)]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    cum = np.concatenate([[0], np.cumsum(tm)]).astype(np.int64)
    for h in range(wl.H):
        for b in range(wl.B):
            for m in range(tm[b]):
                base = int(offs[b]) + m * nn[b]
                out.append((h * int(cum[-1]) + int(cum[b]) + m, (h, slice(base, base + nn[b])), nn[b]))
    return out


def to_bitmask(wl, block_map, words_per_row=None, pad_seed=None):
    """uint32 [rows, words_per_row] and words_per_row; with pad_seed the bits past
    each row's tiles are filled at random (readers must ignore them).  A row wider
    than 32 * words_per_row keeps its first 32 * words_per_row tiles."""
    rows = tile_rows(wl)
    nn_max = max(nn for _, _, nn in rows)
    W = words_per_row or (nn_max + 31) // 32
    rng = np.random.default_rng(pad_seed) if pad_seed is not None else None
    bits = np.zeros((len(rows), 32 * W), dtype=bool)
    for r, sl, nn in rows:
        k = min(nn, 32 * W)
        bits[r, :k] = np.asarray(block_map[sl], dtype=bool)[:k]
        if rng is not None and k < 32 * W:
            bits[r, k:] = rng.integers(0, 2, 32 * W - k).astype(bool)
    # bit x of word w = byte 4w + x // 8, bit x % 8 of little-endian words
    words = np.packbits(bits, axis=1, bitorder="little").view("<u4").astype(np.uint32)
    return words, W


def to_bsr(wl, block_map, shuffle_seed=None, dup_every=0):
    """(indptr int32 [rows + 1], indices int32); with shuffle_seed the ids of a row
    come in random order, and dup_every > 0 repeats every dup_every-th id."""
    rows = sorted(tile_rows(wl), key=lambda t: t[0])
    rng = np.random.default_rng(shuffle_seed) if shuffle_seed is not None else None
    indptr = [0]
    chunks = []
    for r, sl, nn in rows:
        ids = np.nonzero(np.asarray(block_map[sl]))[0].astype(np.int32)
        if dup_every:
            ids = np.concatenate([ids, ids[::dup_every]])
        if rng is not None:
            rng.shuffle(ids)
        chunks.append(ids)
        indptr.append(indptr[-1] + ids.size)
    indices = np.concatenate(chunks) if chunks else np.zeros(0, np.int32)
    if indices.size == 0:
        indices = np.zeros(1, np.int32)
    return np.asarray(indptr, np.int32), indices.astype(np.int32)
