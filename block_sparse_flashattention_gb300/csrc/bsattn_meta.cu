// Metadata kernels: varlen offsets and the boolean-block-map -> full / mask list
// compaction ("[CuTe,Flex] varlen blocksparsity", flash-attention #2224,
// description and review; list format from "Dense FlashAttention vs Block-Sparse
// Attention", section 2).  The selection may also come as packed 32-bit bitmask
// words or as BSR indptr / indices rows ("feat(prims-ts): support
// proxy-compensated block-sparse attention", FlashInfer #4872, bitmask format);
// all three give the same lists.
//
// A selected KV tile is classified over the rectangle of (query row, key) pairs
// it covers: full if the token predicate holds on every pair, mask if on some,
// dropped if on none.  For the interval-shaped mask kinds (none, causal, sliding
// window with sinks, prefix) the three outcomes follow in closed form from the
// corner rows/columns of the rectangle; the document kind, whose ids are
// arbitrary, is decided by scanning the pairs.
#include "bsattn_internal.h"

namespace bsattn {

namespace {

__device__ __forceinline__ long long cdiv_ll(long long a, long long b) { return (a + b - 1) / b; }

// Running sums of num_m(b) and num_m(b) * num_n(b) over the batch (one warp).
__global__ void __launch_bounds__(32) bsattn_meta_offsets_kernel(MetaParams p) {
    const int lane = threadIdx.x;
    long long carry_m = 0, carry_n = 0;
    bool bad = false;
    if (lane == 0) {
        p.cu_tm[0] = 0;
        p.cu_off[0] = 0;
    }
    for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        long long nm = 0, nmn = 0;
        if (b < p.B) {
            long long sq = (long long)p.cu_q[b + 1] - p.cu_q[b];
            long long sk = (long long)p.cu_k[b + 1] - p.cu_k[b];
            if (sq < 0 || sk < 0) {
                bad = true;
                sq = sk = 0;
            }
            nm = cdiv_ll(sq, kTile);
            nmn = nm * cdiv_ll(sk, kTile);
        }
        for (int d = 1; d < 32; d <<= 1) {  // inclusive scan
            long long um = __shfl_up_sync(0xffffffffu, nm, d);
            long long un = __shfl_up_sync(0xffffffffu, nmn, d);
            if (lane >= d) {
                nm += um;
                nmn += un;
            }
        }
        if (b < p.B) {
            long long vm = carry_m + nm, vn = carry_n + nmn;
            if (vm > INT32_MAX || vn > INT32_MAX) bad = true;
            p.cu_tm[b + 1] = (int32_t)(vm > INT32_MAX ? INT32_MAX : vm);
            p.cu_off[b + 1] = (int32_t)(vn > INT32_MAX ? INT32_MAX : vn);
        }
        carry_m += __shfl_sync(0xffffffffu, nm, 31);
        carry_n += __shfl_sync(0xffffffffu, nmn, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0 && p.err && (bad || carry_m != p.total_m || carry_n != p.total_n))
        atomicOr(p.err, BSATTN_FLAG_BAD_SEQLENS);
}

struct RowGeom {
    long long i_min, i_max;  // query rows of the tile inside the sequence (sequence-local)
    long long sk;            // seqlen_k of the sequence
    long long qbase, kbase;  // packed row of the sequence's first query / key
    int b;
};

// Sparse KV block of tile n (a shift for the usual power-of-two block sizes).
__device__ __forceinline__ int kv_block_of(const MetaParams &p, int n) {
    return p.kv_block_shift >= 0 ? (n >> p.kv_block_shift) : n / p.kv_block_tiles;
}

// Valid keys at the start of KV tile n of sequence b: given per tile, or per
// sparse KV block of kv_block_tiles tiles (tile j of the block keeps
// clamp(v - 128 j, 0, 128) of the block's v valid keys).
__device__ __forceinline__ long long tile_valid_len(const MetaParams &p, int b, int n) {
    if (!p.vl_per_block) return p.vl[(long long)b * p.vl_stride + n];
    const int blk = kv_block_of(p, n);
    const long long v = p.vl[(long long)b * p.vl_stride + blk] - (long long)kTile * (n - blk * p.kv_block_tiles);
    return v < 0 ? 0 : (v > kTile ? kTile : v);
}

// 0 = drop, 1 = mask list, 2 = full list, for listed block n (p.tile_k keys) of
// the row's rectangle of query rows.
__device__ int classify(const MetaParams &p, const RowGeom &g, int n) {
    const long long j_lo = (long long)n * p.tile_k, j_end = j_lo + p.tile_k;
    long long j_hi = j_end < g.sk ? j_end : g.sk;
    if (p.vl) {
        const long long lim = j_lo + tile_valid_len(p, g.b, n);
        if (lim < j_hi) j_hi = lim;
    }
    if (j_hi <= j_lo) return 0;
    const bool full_cols = (j_hi == j_end);
    const long long jmin = j_lo, jmax = j_hi - 1, imin = g.i_min, imax = g.i_max;
    bool some = false, all = false;
    switch (p.kind) {
    case BSATTN_MASK_NONE:
        some = true;
        all = true;
        break;
    case BSATTN_MASK_CAUSAL:
        some = jmin <= imax;
        all = jmax <= imin;
        break;
    case BSATTN_MASK_PREFIX: {
        const long long P = p.prefix_len;
        some = (jmin < P) || (jmin <= imax);
        all = (jmax < P) || (jmax <= imin);
        break;
    }
    case BSATTN_MASK_SLIDING_WINDOW: {
        const long long W = p.window_left, S = p.sink_tokens;
        const bool sink_some = (jmin < S) && (jmin <= imax);
        const bool win_some = (W > 0) && (imax - jmin >= 0) && (imin - jmax <= W - 1);
        some = sink_some || win_some;
        const long long js = jmin > S ? jmin : S;  // first non-sink key of the tile
        all = (jmax <= imin) && (js > jmax || imax - js < W);
        break;
    }
    case BSATTN_MASK_DOCUMENT: {
        all = true;
        for (long long i = imin; i <= imax && !(some && !all); ++i) {
            const int32_t dq = p.doc_q[g.qbase + i];
            for (long long j = jmin; j <= jmax; ++j) {
                const bool eq = dq == p.doc_k[g.kbase + j];
                some |= eq;
                all &= eq;
                if (some && !all) break;
            }
        }
        break;
    }
    default:
        return 0;
    }
    if (!some) return 0;
    return (all && full_cols) ? 2 : 1;
}

// One warp per (b, h, m) row: lanes take 32 consecutive block ids from the top
// down, classify them, and compact the ballots into the two descending lists.
// A BSR row is first turned into a bit set in the warp's shared memory.
__global__ void __launch_bounds__(256) bsattn_meta_classify_kernel(MetaParams p) {
    extern __shared__ uint32_t bitset_smem[];
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const long long rows =
        p.varlen ? (long long)p.H * p.total_m : (long long)p.B * p.H * p.num_m;
    if (row >= rows) return;

    RowGeom g;
    long long cnt_at, idx_at;
    int nn, m;
    if (!p.varlen) {
        const long long bh = row / p.num_m;
        m = (int)(row % p.num_m);
        g.b = (int)(bh / p.H);
        g.sk = p.seqlen_k;
        const long long sq = p.seqlen_q;
        g.i_min = (long long)m * p.tile_q;
        g.i_max = (g.i_min + p.tile_q < sq ? g.i_min + p.tile_q : sq) - 1;
        g.qbase = (long long)g.b * p.seqlen_q;
        g.kbase = (long long)g.b * p.seqlen_k;
        nn = p.num_n;
        cnt_at = row;
        idx_at = row * p.num_n;
    } else {
        const int h = (int)(row / p.total_m);
        const int T = (int)(row % p.total_m);
        if (T >= p.cu_tm[p.B]) return;  // caller's total exceeds the sequences' (flagged)
        int lo = 0, hi = p.B - 1;       // largest b with cu_tm[b] <= T
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.cu_tm[mid] <= T) lo = mid;
            else hi = mid - 1;
        }
        g.b = lo;
        m = T - p.cu_tm[lo];
        const long long sq = (long long)p.cu_q[lo + 1] - p.cu_q[lo];
        g.sk = (long long)p.cu_k[lo + 1] - p.cu_k[lo];
        // A sequence outside the packed arrays (when their row counts are given),
        // with negative offsets, or with more KV tiles than the valid-length row
        // stride has no rows here.
        const bool outside = p.cu_q[lo] < 0 || p.cu_k[lo] < 0 || sq < 0 || g.sk < 0 ||
                             (p.seqlen_q > 0 && p.cu_q[lo + 1] > p.seqlen_q) ||
                             (p.seqlen_k > 0 && p.cu_k[lo + 1] > p.seqlen_k) ||
                             (p.vl && cdiv_ll(g.sk, kTile) > p.vl_stride);
        if (outside) {
            if (lane == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_SEQLENS);
            return;
        }
        g.i_min = (long long)m * kTile;
        g.i_max = (g.i_min + kTile < sq ? g.i_min + kTile : sq) - 1;
        g.qbase = p.cu_q[lo];
        g.kbase = p.cu_k[lo];
        nn = (int)cdiv_ll(g.sk, kTile);
        cnt_at = (long long)h * p.total_m + T;
        idx_at = (long long)h * p.total_n + p.cu_off[lo] + (long long)m * nn;
        if (p.cu_off[lo] < 0 || (long long)p.cu_off[lo] + (long long)(m + 1) * nn > p.total_n) {
            if (lane == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_SEQLENS);
            return;
        }
    }
    if (g.i_max < g.i_min) return;  // cannot happen for m < num_m(b)

    // selection source of this row
    const uint8_t *map = p.map ? p.map + idx_at : nullptr;
    const bool coarse = p.block_n > 0;  // map given per sparse block
    if (coarse) {  // batched only: row = (b H + h) num_m + m
        const long long bh = row / p.num_m;
        map = p.map + (bh * p.block_m + m / p.q_block_tiles) * p.block_n;
        if (p.vl_tiles_out && (bh % p.H) == 0 && m == 0)  // once per sequence
            for (int n = lane; n < nn; n += 32)
                p.vl_tiles_out[(long long)g.b * nn + n] = p.vl ? (int32_t)tile_valid_len(p, g.b, n) : kTile;
    }
    const uint32_t *words = nullptr;
    int nbits = nn;  // tiles the row's selection covers
    uint32_t *bits = bitset_smem + (threadIdx.x >> 5) * p.bitset_words;
    if (p.src == kSrcBitmask) {
        words = p.words + cnt_at * p.words_per_row;
        if ((long long)p.words_per_row * 32 < nn) {  // the row's words cannot cover its tiles
            nbits = p.words_per_row * 32;
            if (lane == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_COUNT);
        }
    } else if (p.src == kSrcBsr) {
        const int nw = (nn + 31) >> 5;
        if (nw > p.bitset_words) {  // more tiles than the bit set holds (sizes disagree)
            nbits = p.bitset_words * 32;
            if (lane == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_COUNT);
        }
        for (int w = lane; w < p.bitset_words; w += 32) bits[w] = 0u;
        __syncwarp();
        const long long a = p.indptr[cnt_at], z = p.indptr[cnt_at + 1];
        if (z < a) {
            if (lane == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_COUNT);
        } else {
            bool bad = false;
            for (long long e = a + lane; e < z; e += 32) {
                const int32_t n = p.indices[e];
                if (n >= 0 && n < nbits) atomicOr(&bits[n >> 5], 1u << (n & 31));
                else bad = true;
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_INDEX);
        }
        __syncwarp();
    }
    auto selected = [&](int n) -> bool {
        if (n >= nbits) return false;
        if (p.src == kSrcBitmask) return (__ldg(words + (n >> 5)) >> (n & 31)) & 1u;
        if (p.src == kSrcBsr) return (bits[n >> 5] >> (n & 31)) & 1u;
        return (coarse ? map[kv_block_of(p, n)] : map[n]) != 0;
    };
    int32_t *fidx = p.full_idx + idx_at;
    int32_t *midx = p.mask_idx + idx_at;
    int nf = 0, nmk = 0;
    const unsigned lt = (1u << lane) - 1u;
    for (int top = nn - 1; top >= 0; top -= 32) {
        const int n = top - lane;
        int cls = 0;
        if (n >= 0 && selected(n)) cls = classify(p, g, n);
        const unsigned fb = __ballot_sync(0xffffffffu, cls == 2);
        const unsigned mb = __ballot_sync(0xffffffffu, cls == 1);
        if (cls == 2) fidx[nf + __popc(fb & lt)] = n;
        if (cls == 1) midx[nmk + __popc(mb & lt)] = n;
        nf += __popc(fb);
        nmk += __popc(mb);
    }
    for (int e = nf + lane; e < nn; e += 32) fidx[e] = -1;
    for (int e = nmk + lane; e < nn; e += 32) midx[e] = -1;
    if (lane == 0) {
        p.full_cnt[cnt_at] = nf;
        p.mask_cnt[cnt_at] = nmk;
    }
}

}  // namespace

cudaError_t launch_meta(const MetaParams &p, cudaStream_t stream) {
    if (p.varlen) {
        bsattn_meta_offsets_kernel<<<1, 32, 0, stream>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const long long rows =
        p.varlen ? (long long)p.H * p.total_m : (long long)p.B * p.H * p.num_m;
    if (rows <= 0) return cudaSuccess;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t smem = p.src == kSrcBsr ? (size_t)8 * p.bitset_words * sizeof(uint32_t) : 0;
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(bsattn_meta_classify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
    }
    bsattn_meta_classify_kernel<<<(unsigned)blocks, 256, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace bsattn
