// Backward of the block-sparse attention forward, batched or varlen.  With P the
// forward's probabilities over each row's allowed keys, O = P V and upstream
// gradient dO:
//   D_i = sum_d dO_i O_i,  dV = P^T dO,  dP = dO V^T,  dS = P (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
// Training needs the backward, which the pages list as missing ("[CuTe,Flex]
// varlen blocksparsity", flash-attention #2224, which also names the transposed
// metadata it needs; "[feat] VSA-256 fastpath", FastVideo #1354).  It runs as
//   0. (varlen) a prefix of the sequences' KV tile counts;
//   1. list transpose: every forward list entry sets a byte code (1 full, 2
//      mask) for its (KV tile, Q tile) pair, stored in the layout of the
//      KV-major lists; one warp per KV tile then compacts its codes into
//      KV-major full / mask lists, Q tiles in descending order;
//   2. an order pass: KV tiles sorted by list length, longest first, so the
//      dK / dV grid starts its longest CTAs first;
//   3. a row pass writing -D and -LSE * log2(e) into rows padded to 128 per Q
//      tile (negated, so that the gradient kernels add them);
//   4. the dK / dV kernel: one CTA per KV tile, S^T = K Q^T and dP^T = V dO^T per
//      listed Q tile on tcgen05 as full-width products in two alternating TMEM
//      regions, P^T and dS^T formed per key row into the S^T region, dV += P^T dO
//      and dK += dS^T Q accumulated in TMEM; the next Q tile's S^T goes into the
//      dP^T region as soon as dP^T is in registers, so each product overlaps the
//      elementwise step the next one waits for;
//   5. the dQ kernel: one CTA per Q tile, S = Q K^T and dP = dO V^T per listed KV
//      tile as full-width products, dS per query row into one of two TMEM
//      buffers, dQ += dS K accumulated in TMEM; the next KV tile's S and dP are
//      issued once this tile's are in the elementwise warps' registers.
// Both elementwise passes form P and dS two columns per packed f32x2
// instruction, a dropped column entering the exponential as -inf.
// P is recomputed from the forward's LSE (no running maximum) and rounded to
// bf16 before the P^T dO product, as the forward rounds it before P V; dS is
// rounded to bf16 before its products.
// Layouts.  Batched: sequence b of length S at rows b S; forward lists
// [B, H, num_m(, num_n)]; KV-major lists [B, H, num_n(, num_m)].  Varlen:
// sequence b at rows cu_q[b] / cu_k[b]; forward lists [H, total_m] /
// [H, total_n]; KV-major counts [H, B num_n] (tile cu_tn[b] + n of head h, the
// rest unused), KV-major lists [H, total_n] with column (b, n) at
// cu_block_idx_offsets[b] + n num_m(b) (the block of sequence b holds num_m(b)
// num_n(b) entries in either order).
#include <cuda_bf16.h>

#include <type_traits>

#include "bsattn_internal.h"
#include "sm100_ptx.cuh"

namespace bsattn {

namespace {

// Geometry of sequence b.  A varlen sequence whose offsets disagree with the
// metadata (num_m(b) != ceil(len_q / 128), num_n(b) above the kv_valid_len
// stride, or its list block past total_n) has no tiles here.
struct Seq {
    int sq, sk, nm, nn;  // lengths, Q tiles, KV tiles
    long long q0, k0;    // first packed row
    int T0, Tk0;         // first packed Q tile, first KV tile (varlen: cu_tn[b])
    long long off;       // varlen: first entry of the sequence's list block
    int bad;             // varlen offsets rejected (then nm = nn = 0)
};

__device__ __forceinline__ Seq seq_of(const BwdParams &p, int b) {
    Seq s;
    if (!p.varlen) {
        s.sq = p.seqlen_q;
        s.sk = p.seqlen_k;
        s.nm = p.num_m;
        s.nn = p.num_n;
        s.q0 = (long long)b * p.seqlen_q;
        s.k0 = (long long)b * p.seqlen_k;
        s.T0 = b * p.num_m;
        s.Tk0 = b * p.num_n;
        s.off = 0;
        s.bad = 0;
        return s;
    }
    s.q0 = p.cu_q[b];
    s.k0 = p.cu_k[b];
    s.sq = p.cu_q[b + 1] - p.cu_q[b];
    s.sk = p.cu_k[b + 1] - p.cu_k[b];
    s.nm = p.cu_tm[b + 1] - p.cu_tm[b];
    s.nn = s.sk > 0 ? (s.sk + kTile - 1) / kTile : 0;
    s.T0 = p.cu_tm[b];
    s.Tk0 = p.cu_tn ? p.cu_tn[b] : 0;
    s.off = p.cu_off[b];
    // the sequence must lie inside the packed arrays and agree with the metadata
    const bool ok = s.q0 >= 0 && s.k0 >= 0 && s.sq >= 0 && s.sk >= 0 && s.q0 + s.sq <= p.rows_q &&
                    s.k0 + s.sk <= p.rows_k && s.nm == (s.sq + kTile - 1) / kTile && s.nn <= p.num_n &&
                    s.off >= 0 && s.off + (long long)s.nm * s.nn <= p.total_n;
    s.bad = ok ? 0 : 1;
    if (!ok) s.nm = s.nn = 0;
    return s;
}

// Largest b in [0, B) with cu[b] <= x (cu ascending).
__device__ __forceinline__ int seq_search(const int32_t *cu, int B, long long x) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Forward list row of (b, h, m): count index and first index entry.
__device__ __forceinline__ long long fwd_cnt_at(const BwdParams &p, const Seq &s, int b, int h, int m) {
    return p.varlen ? (long long)h * p.total_m + s.T0 + m : ((long long)b * p.H + h) * p.num_m + m;
}
__device__ __forceinline__ long long fwd_idx_at(const BwdParams &p, const Seq &s, int b, int h, int m) {
    return p.varlen ? (long long)h * p.total_n + s.off + (long long)m * s.nn
                    : (((long long)b * p.H + h) * p.num_m + m) * p.num_n;
}
// KV-major column of (b, h, n): count index (also the order pass's item id) and
// first list entry (also the first selection code).
__device__ __forceinline__ long long kv_cnt_at(const BwdParams &p, const Seq &s, int b, int h, int n) {
    return p.varlen ? (long long)h * p.B * p.num_n + s.Tk0 + n : ((long long)b * p.H + h) * p.num_n + n;
}
__device__ __forceinline__ long long kv_idx_at(const BwdParams &p, const Seq &s, int b, int h, int n) {
    return p.varlen ? (long long)h * p.total_n + s.off + (long long)n * s.nm
                    : (((long long)b * p.H + h) * p.num_n + n) * p.num_m;
}
// First of the 128 padded rows of Q tile (b, h, m) in the LSE2 / D workspace.
__device__ __forceinline__ long long vec_at(const BwdParams &p, const Seq &s, int b, int h, int m) {
    return (p.varlen ? (long long)h * p.total_m + s.T0 + m : ((long long)b * p.H + h) * p.num_m + m) * kTile;
}

// Decodes a KV-major item id into (b, h, n); false for ids past the last tile.
__device__ __forceinline__ bool kv_item(const BwdParams &p, long long c, int &b, int &h, int &n, Seq &s) {
    if (!p.varlen) {
        n = (int)(c % p.num_n);
        const long long bh = c / p.num_n;
        b = (int)(bh / p.H);
        h = (int)(bh - (long long)b * p.H);
        if (b >= p.B) return false;
        s = seq_of(p, b);
        return true;
    }
    const long long per_head = (long long)p.B * p.num_n;
    h = (int)(c / per_head);
    const long long Tk = c - (long long)h * per_head;
    if (h >= p.H || Tk >= p.cu_tn[p.B]) return false;
    b = seq_search(p.cu_tn, p.B, Tk);
    s = seq_of(p, b);
    n = (int)(Tk - s.Tk0);
    return n < s.nn;
}

// Decodes a packed Q tile id (batched: (b H + h) num_m + m; varlen: h total_m + T)
// into (b, h, m); false when the tile holds no rows.
__device__ __forceinline__ bool q_item(const BwdParams &p, long long t, int &b, int &h, int &m, Seq &s) {
    if (!p.varlen) {
        m = (int)(t % p.num_m);
        const long long bh = t / p.num_m;
        b = (int)(bh / p.H);
        h = (int)(bh - (long long)b * p.H);
        if (b >= p.B) return false;
        s = seq_of(p, b);
        return true;
    }
    h = (int)(t / p.total_m);
    const int T = (int)(t - (long long)h * p.total_m);
    if (h >= p.H || T >= p.cu_tm[p.B]) return false;
    b = seq_search(p.cu_tm, p.B, T);
    s = seq_of(p, b);
    m = T - s.T0;
    return m < s.nm;
}

// ------------------------------------------------ 0. KV tile prefix (varlen) --
// One CTA: cu_tn[b] = sum of num_n over the sequences before b (0 for a
// sequence seq_of rejects, which is flagged BSATTN_FLAG_BAD_SEQLENS).
__global__ void __launch_bounds__(1024) bsattn_bwd_seq_kernel(BwdParams p) {
    __shared__ int warp_sums[32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    bool bad = false;
    for (int b0 = 0; b0 < p.B; b0 += blockDim.x) {
        const int b = b0 + (int)threadIdx.x;
        int v = 0;
        if (b < p.B) {
            const Seq s = seq_of(p, b);  // (its Tk0, read before this pass wrote it, is unused)
            bad |= s.bad != 0;
            v = s.nn;
        }
        int incl = v;
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += u;
        }
        if (lane == 31) warp_sums[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += u;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int before = carry + (wid > 0 ? warp_sums[wid - 1] : 0) + incl - v;
        if (b < p.B) p.cu_tn[b] = before;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = before + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) p.cu_tn[p.B] = carry;
    if (__syncthreads_or(bad) && threadIdx.x == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_SEQLENS);
}

// ------------------------------------------------------- 1. list transpose --
// One warp per forward list row (b, h, m): every valid entry n sets code 1
// (full) or 2 (mask) for (KV tile n, Q tile m).  A count outside [0, num_n(b)],
// an index outside [0, num_n(b)) or a tile listed twice sets
// BSATTN_FLAG_BAD_INDEX; the bad entry is skipped (a repeat keeps the OR of the
// codes, so a tile in both lists is treated as a mask tile).
__global__ void __launch_bounds__(256) bsattn_bwd_scatter_kernel(BwdParams p) {
    const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    int b, h, m;
    Seq s;
    if (!q_item(p, w, b, h, m, s)) return;
    const long long ca = fwd_cnt_at(p, s, b, h, m), ia = fwd_idx_at(p, s, b, h, m);
    bool bad = false;
    for (int list = 0; list < 2; ++list) {
        int c = (list ? p.mask_cnt : p.full_cnt)[ca];
        const int32_t *idx_in = (list ? p.mask_idx : p.full_idx) + ia;
        if (c < 0 || c > s.nn) {
            bad = true;
            c = c < 0 ? 0 : s.nn;
        }
        const uint32_t code = list ? 2u : 1u;
        for (int e = lane; e < c; e += 32) {
            const int n = idx_in[e];
            if (n < 0 || n >= s.nn) {
                bad = true;
                continue;
            }
            const long long at = kv_idx_at(p, s, b, h, n) + m;  // byte of (n, m)
            const uint32_t sh = 8u * (uint32_t)(at & 3);
            const uint32_t old = atomicOr(reinterpret_cast<uint32_t *>(p.codes + (at & ~3ll)), code << sh);
            if ((old >> sh) & 0xffu) bad = true;
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_INDEX);
}

// One warp per KV tile (b, h, n): its codes, read from the last Q tile to the
// first 32 at a time, compacted by ballot into the full and mask lists.
__global__ void __launch_bounds__(256) bsattn_bwd_scan_kernel(BwdParams p) {
    const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const uint32_t lane = threadIdx.x & 31u;
    int b, h, n;
    Seq s;
    if (!kv_item(p, w, b, h, n, s)) return;
    const long long at = kv_idx_at(p, s, b, h, n);
    const uint8_t *col = p.codes + at;
    int32_t *fi = p.t_full_idx + at;
    int32_t *mi = p.t_mask_idx + at;
    const uint32_t below = (1u << lane) - 1u;
    int nf = 0, nm = 0;
    for (int top = s.nm - 1; top >= 0; top -= 32) {
        const int m = top - (int)lane;
        const uint32_t code = m >= 0 ? col[m] : 0u;
        const uint32_t bf = __ballot_sync(0xffffffffu, code == 1u);
        const uint32_t bm = __ballot_sync(0xffffffffu, code >= 2u);
        if (code == 1u) fi[nf + __popc(bf & below)] = m;
        if (code >= 2u) mi[nm + __popc(bm & below)] = m;
        nf += __popc(bf);
        nm += __popc(bm);
    }
    if (lane == 0) {
        const long long ci = kv_cnt_at(p, s, b, h, n);
        p.t_full_cnt[ci] = nf;
        p.t_mask_cnt[ci] = nm;
    }
}

// One CTA: the ids of the KV tiles ordered by their number of listed Q tiles,
// longest first (a counting sort; the order among equal lengths is unspecified
// and affects only which CTA starts first, never a result).  Ids of no tile
// (varlen padding of the count array) sort last and are written as -1.
constexpr int kOrderBins = 8192;
__global__ void __launch_bounds__(1024) bsattn_bwd_order_kernel(BwdParams p) {
    __shared__ int hist[kOrderBins];
    __shared__ int warp_sums[32];
    const long long items = (long long)p.B * p.H * p.num_n;
    const int top = min(p.num_m_max, kOrderBins - 2);  // lengths above `top` share bin 0
    const int nb = top + 2;                            // bin top + 1: not a tile
    auto bin_of = [&](long long c) -> int {
        int b, h, n;
        Seq s;
        if (!kv_item(p, c, b, h, n, s)) return top + 1;
        const long long ci = kv_cnt_at(p, s, b, h, n);
        return top - min(p.t_full_cnt[ci] + p.t_mask_cnt[ci], top);
    };
    for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (long long c = threadIdx.x; c < items; c += blockDim.x) atomicAdd(&hist[bin_of(c)], 1);
    __syncthreads();
    // exclusive scan over the bins: each thread owns a contiguous run of bins
    const int per = (nb + (int)blockDim.x - 1) / (int)blockDim.x;
    const int b0 = min((int)threadIdx.x * per, nb), b1 = min(b0 + per, nb);
    int run = 0;
    for (int i = b0; i < b1; ++i) run += hist[i];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = run;
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        warp_sums[lane] = v;
    }
    __syncthreads();
    int base = incl - run + (wid > 0 ? warp_sums[wid - 1] : 0);
    for (int i = b0; i < b1; ++i) {
        const int c = hist[i];
        hist[i] = base;
        base += c;
    }
    __syncthreads();
    for (long long c = threadIdx.x; c < items; c += blockDim.x) {
        const int bin = bin_of(c);
        p.order[atomicAdd(&hist[bin], 1)] = bin == top + 1 ? -1 : (int32_t)c;
    }
}

// ------------------------------------------------------------ 2. row pass --
// One warp per 4 padded query rows (Q tile, r .. r + 3): D = sum_d dO O in fp32
// and LSE * log2(e), both stored negated.  Each lane takes D / 32 consecutive elements of every row
// (one 8- or 4-byte load of dO and one of O per row), the four rows' loads issued
// before any is used.  Rows past the sequence, and rows with no keys
// (LSE = -inf), get LSE2 = +inf (-inf stored), so every probability they would form is 0.
constexpr int kRowsPerWarp = 4;
__global__ void __launch_bounds__(256) bsattn_bwd_rows_kernel(BwdParams p) {
    const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const long long row0 = w * kRowsPerWarp;
    int b, h, m;
    Seq s;
    if (!q_item(p, row0 / kTile, b, h, m, s)) return;
    const int r0 = (int)(row0 % kTile);
    const bool wide = p.D == 128;  // 4 elements per lane (else 2)
    uint2 g[kRowsPerWarp];         // dO, bf16 pairs
    float4 o[kRowsPerWarp];        // O as fp32
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
        const int i = m * kTile + r0 + k;
        g[k] = make_uint2(0u, 0u);
        o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i >= s.sq) continue;
        const long long e = ((s.q0 + i) * p.H + h) * p.D + (long long)lane * (wide ? 4 : 2);
        if (wide) {
            g[k] = *reinterpret_cast<const uint2 *>(p.dout + e);
            if (p.o_f32) {
                o[k] = *reinterpret_cast<const float4 *>(static_cast<const float *>(p.o) + e);
            } else {
                const uint2 ob = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.o) + e);
                o[k] = make_float4(__uint_as_float(ob.x << 16), __uint_as_float(ob.x & 0xffff0000u),
                                   __uint_as_float(ob.y << 16), __uint_as_float(ob.y & 0xffff0000u));
            }
        } else {
            g[k].x = *reinterpret_cast<const uint32_t *>(p.dout + e);
            if (p.o_f32) {
                const float2 of = *reinterpret_cast<const float2 *>(static_cast<const float *>(p.o) + e);
                o[k] = make_float4(of.x, of.y, 0.f, 0.f);
            } else {
                const uint32_t ob = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(p.o) + e);
                o[k] = make_float4(__uint_as_float(ob << 16), __uint_as_float(ob & 0xffff0000u), 0.f, 0.f);
            }
        }
    }
    float d[kRowsPerWarp];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
        float acc = __uint_as_float(g[k].x << 16) * o[k].x;
        acc = fmaf(__uint_as_float(g[k].x & 0xffff0000u), o[k].y, acc);
        acc = fmaf(__uint_as_float(g[k].y << 16), o[k].z, acc);
        acc = fmaf(__uint_as_float(g[k].y & 0xffff0000u), o[k].w, acc);
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        d[k] = acc;
    }
    if (lane < kRowsPerWarp) {  // lane k writes row r0 + k
        const int i = m * kTile + r0 + lane;
        float dk = 0.f, l2 = INFINITY;
#pragma unroll
        for (int k = 0; k < kRowsPerWarp; ++k)
            if (k == lane) dk = d[k];
        if (i < s.sq) {
            const long long li = p.varlen ? (long long)h * p.rows_q + s.q0 + i : ((long long)b * p.H + h) * s.sq + i;
            const float lse = p.lse[li];
            l2 = lse == -INFINITY ? INFINITY : lse * 1.4426950408889634f;
        }
        const long long at = vec_at(p, s, b, h, m) + r0 + lane;
        p.dvec[at] = -dk;  // negated: the gradient kernels form s log2(e) - LSE2 and dP - D as sums
        p.lse2[at] = -l2;
    }
}

// Shared memory of the dK/dV kernel: K and V resident, a ring of Q tiles (each
// with its queries' -LSE2 and -D vectors) and a ring of dO tiles, barriers,
// item info, misc.  dO leaves the ring after the dV product, Q after the dK
// product, one product later.
template <int D>
struct BwdCfg {
    static constexpr uint32_t kTileBytes = kTile * D * 2;
    static constexpr int kSub = D / 64;                       // 64-column swizzle spans per tile
    static constexpr uint32_t kSubBytes = kTile * 64 * 2;
    static constexpr int kQStages = 2, kOStages = 2;
    static constexpr uint32_t kRes0 = 0, kRes1 = kTileBytes;  // K, V
    static constexpr uint32_t kQ = 2 * kTileBytes;            // Q stage s at kQ + s * kTileBytes
    static constexpr uint32_t kO = kQ + kQStages * kTileBytes;  // dO stage s at kO + s * kTileBytes
    static constexpr uint32_t kVec = kO + kOStages * kTileBytes;  // Q stage s: 2 x 128 floats at kVec + 1024 s
    static constexpr uint32_t kBar = kVec + 1024 * kQStages;
    // barriers: resident tiles full, Q full / empty [kQStages], dO full / empty
    // [kOStages], S^T done, dP^T done, P^T written [2: query halves], dP^T in
    // the elementwise warps' registers, dS^T written [2: query halves],
    // accumulators done, MMA drain
    static constexpr int bRF = 0, bQF = 1, bQE = bQF + kQStages, bOF = bQE + kQStages, bOE = bOF + kOStages;
    static constexpr int bS = bOE + kOStages, bP = bS + 1, bPt = bP + 1, bDL = bPt + 2, bDS = bDL + 1;
    static constexpr int bDone = bDS + 2, bDrain = bDone + 1, kNumBars = bDrain + 1;
    static constexpr uint32_t kInfo = kBar + kNumBars * 8;    // int32 [kQStages][2]: Q tile, mask flag
    static constexpr uint32_t kMisc = kInfo + 8 * kQStages;   // [0] tmem base, [1] abort
    static constexpr uint32_t kBytes = kMisc + 16;
    static constexpr uint32_t kSmemAlloc = kBytes + 1024;     // slack for 1024-byte alignment
};

constexpr int kBwdThreads = 384;  // warps 0-3: roles; warps 4-11: elementwise
constexpr int kEwWarps = 8;

__device__ __forceinline__ uint32_t bwd_span_bits(long long lo, long long hi) {
    lo = lo < 0 ? 0 : lo;
    hi = hi > 32 ? 32 : hi;
    if (hi <= lo) return 0u;
    const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
    return below_hi & ~((1u << lo) - 1u);
}

template <int D>
__device__ __forceinline__ void bwd_init(uint8_t *gbase, uint32_t base, uint32_t warp) {
    using C = BwdCfg<D>;
    uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + C::kMisc);
    auto bar = [&](int i) -> uint32_t { return base + C::kBar + 8u * (uint32_t)i; };
    if (threadIdx.x == 0) {
        mbar_init(bar(C::bRF), 1);
        for (int s = 0; s < C::kQStages; ++s) {
            mbar_init(bar(C::bQF + s), 1);
            mbar_init(bar(C::bQE + s), 1);
        }
        for (int s = 0; s < C::kOStages; ++s) {
            mbar_init(bar(C::bOF + s), 1);
            mbar_init(bar(C::bOE + s), 1);
        }
        mbar_init(bar(C::bS), 1);
        mbar_init(bar(C::bP), 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(bar(C::bPt + k), kEwWarps);  // one arrival per elementwise warp
            mbar_init(bar(C::bDS + k), kEwWarps);
        }
        mbar_init(bar(C::bDL), kEwWarps);
        mbar_init(bar(C::bDone), 1);
        mbar_init(bar(C::bDrain), 1);
        misc[1] = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 2) {
        tmem_alloc(base + C::kMisc, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Stores 32 fp32 accumulator columns, times `mul`, at element `off` of a
// gradient tensor (fp32, or bf16 rounded to nearest even).
__device__ __forceinline__ void bwd_store_row32(void *dst, int f32, long long off, const uint32_t (&v)[32],
                                                float mul) {
    if (f32) {
        float *o = static_cast<float *>(dst) + off;
#pragma unroll
        for (int x = 0; x < 32; x += 4)
            *reinterpret_cast<float4 *>(o + x) =
                make_float4(__uint_as_float(v[x]) * mul, __uint_as_float(v[x + 1]) * mul,
                            __uint_as_float(v[x + 2]) * mul, __uint_as_float(v[x + 3]) * mul);
    } else {
        uint16_t *o = static_cast<uint16_t *>(dst) + off;
#pragma unroll
        for (int x = 0; x < 32; x += 8)
            *reinterpret_cast<uint4 *>(o + x) =
                make_uint4(pack_bf16x2(__uint_as_float(v[x]) * mul, __uint_as_float(v[x + 1]) * mul),
                           pack_bf16x2(__uint_as_float(v[x + 2]) * mul, __uint_as_float(v[x + 3]) * mul),
                           pack_bf16x2(__uint_as_float(v[x + 4]) * mul, __uint_as_float(v[x + 5]) * mul),
                           pack_bf16x2(__uint_as_float(v[x + 6]) * mul, __uint_as_float(v[x + 7]) * mul));
    }
}

// Epilogue of an elementwise warp: its 32 rows x D/2 columns of an fp32 TMEM
// accumulator (columns [cg * D/2, (cg + 1) * D/2)), times `mul`, to global rows
// (zeros when `have` is false; nothing stored when `store` is false).
template <int D>
__device__ __forceinline__ void bwd_epilogue_half(uint32_t tacc, bool have, bool store, void *dst, int f32,
                                                  long long orow, int cg, float mul) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        const int col = cg * (D / 2) + 32 * c;
        uint32_t v[32];
        if (have) {
            tmem_ld32(tacc + (uint32_t)col, v);
            tmem_wait_ld();
            reg_fence(v);
        } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = 0u;
        }
        if (store) bwd_store_row32(dst, f32, orow + col, v, mul);
    }
}


// ----------------------------------------------------------- 4. dK and dV --
// One CTA per (b, h, KV tile n), taken in the order of the order pass; 384
// threads: warp 0 loads (K and V of the tile once, then Q with LSE2 and D, and
// dO of each listed Q tile into their rings), warp 1 issues the MMAs, warp 2
// owns TMEM, warps 4-11 form P^T and dS^T (warp w: TMEM lane quarter w % 4,
// thread = key row; column group cg = (w - 4) / 4 takes query chunks cg and
// cg + 2, 32 columns each) and write the gradients.
// TMEM: two 128-column regions R0 = [0, 128), R1 = [128, 256), dV [256, 256 + D),
// dK [256 + D, 256 + 2D).  Q tile t: S^T (N = 128) in R(t % 2), dP^T in
// R((t + 1) % 2).  P^T (bf16) of query chunk c goes to columns [32 c, 32 c + 16)
// of R(t % 2) and dS^T to [32 c + 16, 32 c + 32), inside the chunk's own S^T
// columns, so dP^T's region is free as soon as the elementwise warps hold it in
// registers: S^T of tile t + 1 goes there, and dP^T of tile t + 1 into R(t % 2)
// after tile t's dK product (products run in issue order).  Tensor core order
// per tile: dV_t, S_t+1, dK_t, dP_t+1, so each product covers the elementwise
// step the next one waits for (P^T of t + 1 forms under dK_t and dP_t+1, dS^T
// of t under dV_t and S_t+1).
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bsattn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tq,
                           const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                           const __grid_constant__ CUtensorMap tdo) {
    using C = BwdCfg<D>;
    constexpr int kQS = C::kQStages, kOS = C::kOStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    int32_t *info = reinterpret_cast<int32_t *>(gbase + C::kInfo);
    uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + C::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    auto bar = [&](int i) -> uint32_t { return base + C::kBar + 8u * (uint32_t)i; };
    const uint32_t warp = warp_id(), lane = lane_id();
    const uint32_t lead = lane == 0 ? 1u : 0u;

    const long long item = p.order[blockIdx.x];  // (b, h, n) of this CTA; -1: none
    int b, h, n;
    Seq sg;
    if (item < 0 || !kv_item(p, item, b, h, n, sg)) return;
    const long long ci = kv_cnt_at(p, sg, b, h, n), li = kv_idx_at(p, sg, b, h, n);
    const int cm = min(max(p.t_mask_cnt[ci], 0), sg.nm);
    const int cf = min(max(p.t_full_cnt[ci], 0), sg.nm);
    const int total = cm + cf;  // listed Q tiles: the mask list, then the full list

    bwd_init<D>(gbase, base, warp);
    const uint32_t tmem = misc[0];
    const uint32_t tdV = tmem + 256u, tdK = tmem + 256u + D;
    auto region = [&](int t) -> uint32_t { return tmem + 128u * (uint32_t)(t & 1); };  // S^T of tile t

    if (warp == 0) {
        // ------------------------------------------------------- loads --
        const int kvrow = (int)(sg.k0 + n * kTile);
        mbar_arrive_expect_tx_lead(lead, bar(C::bRF), 2 * C::kTileBytes);
        for (int x = 0; x < C::kSub; ++x) {
            tma_load_3d_lead(lead, base + C::kRes0 + x * C::kSubBytes, &tk, bar(C::bRF), x * 64, h, kvrow);
            tma_load_3d_lead(lead, base + C::kRes1 + x * C::kSubBytes, &tv, bar(C::bRF), x * 64, h, kvrow);
        }
        int nq = 0, no = 0;  // Q and dO tiles issued
        for (int it = 0; it < total; ++it) {
            const int qs = it % kQS, os = it % kOS;
            if (!mbar_wait(bar(C::bQE + qs), ((it / kQS) & 1) ^ 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT)) break;
            const int m = it < cm ? p.t_mask_idx[li + it] : p.t_full_idx[li + (it - cm)];
            info[qs * 2 + 0] = m;
            info[qs * 2 + 1] = it < cm ? 1 : 0;
            const int qrow = (int)(sg.q0 + m * kTile);
            const long long vrow = vec_at(p, sg, b, h, m);
            mbar_arrive_expect_tx_lead(lead, bar(C::bQF + qs), C::kTileBytes + 1024u);
            for (int x = 0; x < C::kSub; ++x)
                tma_load_3d_lead(lead, base + C::kQ + qs * C::kTileBytes + x * C::kSubBytes, &tq, bar(C::bQF + qs),
                                 x * 64, h, qrow);
            bulk_g2s_lead(lead, base + C::kVec + 1024u * qs, p.lse2 + vrow, 512u, bar(C::bQF + qs));
            bulk_g2s_lead(lead, base + C::kVec + 1024u * qs + 512u, p.dvec + vrow, 512u, bar(C::bQF + qs));
            ++nq;
            if (!mbar_wait(bar(C::bOE + os), ((it / kOS) & 1) ^ 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT)) break;
            mbar_arrive_expect_tx_lead(lead, bar(C::bOF + os), C::kTileBytes);
            for (int x = 0; x < C::kSub; ++x)
                tma_load_3d_lead(lead, base + C::kO + os * C::kTileBytes + x * C::kSubBytes, &tdo, bar(C::bOF + os),
                                 x * 64, h, qrow);
            ++no;
        }
        // every copy issued has landed before the CTA may exit
        mbar_wait_drain(bar(C::bRF), 0);
        for (int s = 0; s < kQS; ++s) {
            const int uses = (nq + kQS - 1 - s) / kQS;
            if (uses > 0) mbar_wait_drain(bar(C::bQF + s), (uint32_t)(uses - 1) & 1u);
        }
        for (int s = 0; s < kOS; ++s) {
            const int uses = (no + kOS - 1 - s) / kOS;
            if (uses > 0) mbar_wait_drain(bar(C::bOF + s), (uint32_t)(uses - 1) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMAs --
        constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false);
        constexpr uint32_t idesc_ts = idesc_bf16_f32(128, D, true);
        constexpr uint64_t kSubUnits = C::kSubBytes >> 4;
        const uint64_t dKk = smem_desc_sw128(base + C::kRes0, 16, 1024);
        const uint64_t dVk = smem_desc_sw128(base + C::kRes1, 16, 1024);
        // S^T = K Q_t^T into region(t), or dP^T = V dO_t^T into region(t + 1)
        auto issue_mm = [&](int t, bool dp) {
            const uint32_t st = dp ? base + C::kO + (uint32_t)(t % kOS) * C::kTileBytes
                                   : base + C::kQ + (uint32_t)(t % kQS) * C::kTileBytes;
            const uint64_t dB = smem_desc_sw128(st, 16, 1024);
            const uint64_t dA = dp ? dVk : dKk;
            const uint32_t td = region(dp ? t + 1 : t);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (uint64_t)((kk >> 2) * kSubUnits + (kk & 3) * 2);
                mma_ss_lead(lead, td, dA + off, dB + off, idesc_ss, kk > 0 ? 1u : 0u);
            }
        };
        // dV += P^T_t dO_t, or dK += dS^T_t Q_t, over query half `half` (16 queries per step)
        auto issue_grad = [&](int t, bool dk, int half) {
            const uint32_t st = dk ? base + C::kQ + (uint32_t)(t % kQS) * C::kTileBytes
                                   : base + C::kO + (uint32_t)(t % kOS) * C::kTileBytes;
            const uint64_t dBm = smem_desc_sw128(st, C::kSubBytes, 1024);
            const uint32_t ta = region(t) + (dk ? 16u : 0u);
#pragma unroll
            for (int kk = 4 * half; kk < 4 * half + 4; ++kk)
                mma_ts_lead(lead, dk ? tdK : tdV, ta + 32u * (kk >> 1) + 8u * (kk & 1),
                            dBm + (uint64_t)(kk * (2048 >> 4)), idesc_ts, (t > 0 || kk > 0) ? 1u : 0u);
        };
        auto wait = [&](int bi, int par) -> bool {
            const bool r = mbar_wait(bar(bi), (uint32_t)par & 1u, abort_flag, p.err, BSATTN_FLAG_TIMEOUT);
            tc_fence_after();
            return r;
        };
        bool ok = wait(C::bRF, 0);
        if (ok && total > 0) {
            if ((ok = wait(C::bQF, 0))) {
                issue_mm(0, false);
                mma_commit_lead(lead, bar(C::bS));
            }
            if (ok && (ok = wait(C::bOF, 0))) {
                issue_mm(0, true);
                mma_commit_lead(lead, bar(C::bP));
            }
        }
        for (int it = 0; ok && it < total; ++it) {
            const bool more = it + 1 < total;
            if (!(ok = wait(C::bPt, it))) break;
            issue_grad(it, false, 0);
            if (!(ok = wait(C::bPt + 1, it))) break;
            issue_grad(it, false, 1);
            mma_commit_lead(lead, bar(C::bOE + it % kOS));  // dO stage free once dV has read it
            if (more) {
                if (!(ok = wait(C::bDL, it))) break;
                if (!(ok = wait(C::bQF + (it + 1) % kQS, (it + 1) / kQS))) break;
                issue_mm(it + 1, false);
                mma_commit_lead(lead, bar(C::bS));
            }
            if (!(ok = wait(C::bDS, it))) break;
            issue_grad(it, true, 0);
            if (!(ok = wait(C::bDS + 1, it))) break;
            issue_grad(it, true, 1);
            mma_commit_lead(lead, bar(C::bQE + it % kQS));  // Q stage and its vectors free
            if (more) {
                if (!(ok = wait(C::bOF + (it + 1) % kOS, (it + 1) / kOS))) break;
                issue_mm(it + 1, true);
                mma_commit_lead(lead, bar(C::bP));
            }
        }
        if (ok) mma_commit_lead(lead, bar(C::bDone));
        mma_commit_lead(lead, bar(C::bDrain));
        mbar_wait_drain(bar(C::bDrain), 0);
    } else if (warp >= 4) {
        // ------------------------------------------------- elementwise --
        const uint32_t q4 = warp & 3u;
        const int cg = (int)(warp - 4) >> 2;   // column group
        const int r = (int)(q4 * 32u + lane);  // key row of the tile
        const uint32_t la = (q4 * 32u) << 16;  // TMEM lane offset of this warp
        const int j = n * kTile + r;           // sequence-local key
        const int klim_full = min(kTile, sg.sk - n * kTile);
        int klim_mask = klim_full;
        if (p.vl) klim_mask = min(klim_mask, p.vl[(long long)b * p.num_n + n]);
        const float sl2 = p.scale_log2;
        const float *vecs = reinterpret_cast<const float *>(gbase + C::kVec);
        bool ok = true;
        for (int it = 0; it < total; ++it) {
            const int qs = it % kQS;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(C::bQF + qs), (it / kQS) & 1, abort_flag, p.err,
                                                         BSATTN_FLAG_TIMEOUT))))
                break;
            if (!(ok = __all_sync(0xffffffffu,
                                  mbar_wait(bar(C::bS), it & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT))))
                break;
            tc_fence_after();
            const int m = reinterpret_cast<volatile int32_t *>(info)[qs * 2 + 0];
            const bool msk = reinterpret_cast<volatile int32_t *>(info)[qs * 2 + 1] != 0;
            // kept query columns of this key row: [lo, hi) (query i = m * 128 + column)
            long long lo = 0, hi = kTile;
            const bool row_on = r < (msk ? klim_mask : klim_full);
            const long long d0 = (long long)j - (long long)m * kTile;  // column of query i == j
            if (!row_on) {
                hi = 0;
            } else if (msk) {
                if (p.kind == BSATTN_MASK_CAUSAL) {
                    lo = d0;
                } else if (p.kind == BSATTN_MASK_SLIDING_WINDOW) {
                    lo = d0;
                    if (j >= p.sink_tokens) hi = d0 + p.window_left;
                } else if (p.kind == BSATTN_MASK_PREFIX) {
                    if (j >= p.prefix_len) lo = d0;
                }
            }
            const bool doc = msk && row_on && p.kind == BSATTN_MASK_DOCUMENT;
            const int32_t dk = doc ? p.doc_k[sg.k0 + j] : 0;
            const float *nl2 = vecs + qs * 256, *ndd = nl2 + 128;  // -LSE2, -D of the stage's queries
            const uint32_t tS = region(it) + la, tP = region(it + 1) + la;
            // P = 2^(s log2(e) scale - LSE2), two columns per packed instruction;
            // dropped columns enter the exponential as -inf.  A chunk every lane
            // keeps whole takes the form without selects.
            float pr[2][32];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = cg + 2 * k;  // query chunk: columns [32 c, 32 c + 32)
                uint32_t vs[32];
                tmem_ld32(tS + 32u * c, vs);
                tmem_wait_ld();
                reg_fence(vs);
                uint32_t keep = bwd_span_bits(lo - 32 * c, hi - 32 * c);
                if (doc) {
                    keep = 0u;
                    for (int x = 0; x < 32; ++x) {
                        const int i = m * kTile + 32 * c + x;
                        if (i < sg.sq && __ldg(p.doc_q + sg.q0 + i) == dk)
                            keep |= 1u << x;
                    }
                }
                uint32_t pw[16];
                auto form = [&](auto masked) {
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const float2 nl = *reinterpret_cast<const float2 *>(nl2 + 32 * c + 2 * x);
                        float x0, x1;
                        ffma2(x0, x1, __uint_as_float(vs[2 * x]), __uint_as_float(vs[2 * x + 1]), sl2, sl2,
                              nl.x, nl.y);
                        if constexpr (decltype(masked)::value) {
                            x0 = ((keep >> (2 * x)) & 1u) ? x0 : -INFINITY;
                            x1 = ((keep >> (2 * x + 1)) & 1u) ? x1 : -INFINITY;
                        }
                        pr[k][2 * x] = ex2_approx(x0);
                        pr[k][2 * x + 1] = ex2_approx(x1);
                        pw[x] = pack_bf16x2(pr[k][2 * x], pr[k][2 * x + 1]);
                    }
                };
                if (__all_sync(0xffffffffu, keep == 0xffffffffu)) form(std::false_type{});
                else form(std::true_type{});
                tmem_st16(tS + 32u * c, pw);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::bPt + k));
            }
            // dS = P (dP - D): dP^T of this tile into registers, its region
            // released, then dS^T of each chunk
            if (!(ok = __all_sync(0xffffffffu,
                                  mbar_wait(bar(C::bP), it & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT))))
                break;
            tc_fence_after();
            uint32_t vp[2][32];
            tmem_ld32(tP + 32u * cg, vp[0]);
            tmem_ld32(tP + 32u * (cg + 2), vp[1]);
            tmem_wait_ld();
            reg_fence(vp[0]);
            reg_fence(vp[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::bDL));
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = cg + 2 * k;
                uint32_t dw[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float2 nd = *reinterpret_cast<const float2 *>(ndd + 32 * c + 2 * x);
                    float t0, t1, d0, d1;
                    fadd2(t0, t1, __uint_as_float(vp[k][2 * x]), __uint_as_float(vp[k][2 * x + 1]), nd.x, nd.y);
                    fmul2(d0, d1, pr[k][2 * x], pr[k][2 * x + 1], t0, t1);
                    dw[x] = pack_bf16x2(d0, d1);
                }
                tmem_st16(tS + 32u * c + 16u, dw);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::bDS + k));
            }
        }
        // ------------------------------------------------- epilogue --
        if (ok && total > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::bDone), 0, abort_flag, p.err, BSATTN_FLAG_TIMEOUT));
            tc_fence_after();
        }
        if (ok) {
            const long long orow = ((sg.k0 + j) * p.H + h) * D;
            bwd_epilogue_half<D>(tdV + la, total > 0, j < sg.sk, p.dv, p.grad_f32, orow, cg, 1.f);
            bwd_epilogue_half<D>(tdK + la, total > 0, j < sg.sk, p.dk, p.grad_f32, orow, cg, p.scale);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Shared memory of the dQ kernel: Q and dO resident, a ring of three K tiles and
// one of two V tiles (V is done with one item earlier than K: after the item's
// dP products, K only after its dQ products), barriers, item info, misc.
template <int D>
struct DqCfg {
    static constexpr uint32_t kTileBytes = kTile * D * 2;
    static constexpr int kSub = D / 64;
    static constexpr uint32_t kSubBytes = kTile * 64 * 2;
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr uint32_t kRes0 = 0, kRes1 = kTileBytes;     // Q, dO
    static constexpr uint32_t kK = 2 * kTileBytes;               // K stage s at kK + s * kTileBytes
    static constexpr uint32_t kV = kK + kKStages * kTileBytes;   // V stage s at kV + s * kTileBytes
    static constexpr uint32_t kBar = kV + kVStages * kTileBytes;
    // barriers: resident tiles, K full [3], K empty [3], V full [2], V empty [2],
    // S and dP ready, S and dP in the elementwise warps' registers [2: even and
    // odd items], dS done [2: even and odd items], dQ done, MMA drain
    static constexpr int bRF = 0, bKF = 1, bKE = 4, bVF = 7, bVE = 9, bSR = 11, bSL = 12, bPR = 14;
    static constexpr int bDone = 16, bDrain = 17, kNumBars = 18;
    static constexpr uint32_t kInfo = kBar + kNumBars * 8;       // int32 [3][2]: tile, mask flag
    static constexpr uint32_t kMisc = kInfo + 32;                // [0] tmem base, [1] abort
    static constexpr uint32_t kBytes = kMisc + 16;
    static constexpr uint32_t kSmemAlloc = kBytes + 1024;        // slack for 1024-byte alignment
};

template <int D>
__device__ __forceinline__ void dq_init(uint8_t *gbase, uint32_t base, uint32_t warp) {
    using C = DqCfg<D>;
    uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + C::kMisc);
    auto bar = [&](int i) -> uint32_t { return base + C::kBar + 8u * (uint32_t)i; };
    if (threadIdx.x == 0) {
        mbar_init(bar(C::bRF), 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(bar(C::bKF + s), 1);
            mbar_init(bar(C::bKE + s), 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(bar(C::bVF + s), 1);
            mbar_init(bar(C::bVE + s), 1);
        }
        mbar_init(bar(C::bSR), 1);
        for (int e = 0; e < 2; ++e) {
            mbar_init(bar(C::bSL + e), kEwWarps);
            mbar_init(bar(C::bPR + e), kEwWarps);
        }
        mbar_init(bar(C::bDone), 1);
        mbar_init(bar(C::bDrain), 1);
        misc[1] = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 2) {
        tmem_alloc(base + C::kMisc, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// ------------------------------------------------------------------ 5. dQ --
// One CTA per (b, h, Q tile m), 384 threads, the same roles: Q and dO of the
// tile stay resident, K and V of each listed KV tile (the forward's mask list,
// then its full list; entries outside [0, num_n) skipped by every role alike)
// pass through the K and V rings.  Thread = query row; column group cg of the
// elementwise warps takes key chunk 2 h + cg of key half h.
// TMEM: S [0, 128), dP [128, 256), dS buffers (bf16) [256, 320) and [320, 384),
// dQ [384, 384 + D).  S and dP are full-width (N = 128) products; those of tile
// t + 1 are issued as soon as the elementwise warps hold tile t's in registers,
// so they run under tile t's elementwise work, ahead of tile t's dQ product,
// which reads dS buffer t % 2 while the elementwise warps fill the other one.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bsattn_bwd_dq_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                         const __grid_constant__ CUtensorMap tdo) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    int32_t *info = reinterpret_cast<int32_t *>(gbase + C::kInfo);
    uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + C::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    auto bar = [&](int i) -> uint32_t { return base + C::kBar + 8u * (uint32_t)i; };
    const uint32_t warp = warp_id(), lane = lane_id();
    const uint32_t lead = lane == 0 ? 1u : 0u;

    int b, h, m;
    Seq sg;
    if (!q_item(p, blockIdx.x, b, h, m, sg)) return;
    const long long ca = fwd_cnt_at(p, sg, b, h, m), ia = fwd_idx_at(p, sg, b, h, m);
    const int cm = min(max(p.mask_cnt[ca], 0), sg.nn);
    const int cf = min(max(p.full_cnt[ca], 0), sg.nn);
    // raw entry e of the item sequence (mask list first); -1 when out of range
    auto entry = [&](int e) -> int {
        const int n = e < cm ? __ldg(p.mask_idx + ia + e) : __ldg(p.full_idx + ia + (e - cm));
        return (n >= 0 && n < sg.nn) ? n : -1;
    };
    int total = 0;  // valid entries: every warp counts them 32 at a time
    for (int e0 = 0; e0 < cm + cf; e0 += 32) {
        const int e = e0 + (int)(threadIdx.x & 31u);
        total += __popc(__ballot_sync(0xffffffffu, e < cm + cf && entry(e) >= 0));
    }

    dq_init<D>(gbase, base, warp);
    const uint32_t tmem = misc[0];
    const uint32_t tS = tmem, tP = tmem + 128u, tDS = tmem + 256u, tdQ = tmem + 384u;

    if (warp == 0) {
        // ------------------------------------------------------- loads --
        const int qrow = (int)(sg.q0 + m * kTile);
        mbar_arrive_expect_tx_lead(lead, bar(C::bRF), 2 * C::kTileBytes);
        for (int x = 0; x < C::kSub; ++x) {
            tma_load_3d_lead(lead, base + C::kRes0 + x * C::kSubBytes, &tq, bar(C::bRF), x * 64, h, qrow);
            tma_load_3d_lead(lead, base + C::kRes1 + x * C::kSubBytes, &tdo, bar(C::bRF), x * 64, h, qrow);
        }
        int nk = 0, nv = 0;  // K and V tiles issued
        for (int e = 0; e < cm + cf; ++e) {
            const int n = entry(e);
            if (n < 0) continue;
            const int ks = nk % C::kKStages, vs = nv % C::kVStages;
            const int kvrow = (int)(sg.k0 + n * kTile);
            // K first (S needs it), then V (dP needs it), each on its own ring
            if (!mbar_wait(bar(C::bKE + ks), ((nk / C::kKStages) & 1) ^ 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT))
                break;
            info[ks * 2 + 0] = n;
            info[ks * 2 + 1] = e < cm ? 1 : 0;
            mbar_arrive_expect_tx_lead(lead, bar(C::bKF + ks), C::kTileBytes);
            for (int x = 0; x < C::kSub; ++x)
                tma_load_3d_lead(lead, base + C::kK + ks * C::kTileBytes + x * C::kSubBytes, &tk, bar(C::bKF + ks),
                                 x * 64, h, kvrow);
            ++nk;
            if (!mbar_wait(bar(C::bVE + vs), ((nv / C::kVStages) & 1) ^ 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT))
                break;
            mbar_arrive_expect_tx_lead(lead, bar(C::bVF + vs), C::kTileBytes);
            for (int x = 0; x < C::kSub; ++x)
                tma_load_3d_lead(lead, base + C::kV + vs * C::kTileBytes + x * C::kSubBytes, &tv, bar(C::bVF + vs),
                                 x * 64, h, kvrow);
            ++nv;
        }
        mbar_wait_drain(bar(C::bRF), 0);
        for (int s = 0; s < C::kKStages; ++s) {
            const int uses = (nk + C::kKStages - 1 - s) / C::kKStages;
            if (uses > 0) mbar_wait_drain(bar(C::bKF + s), (uint32_t)(uses - 1) & 1u);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            const int uses = (nv + C::kVStages - 1 - s) / C::kVStages;
            if (uses > 0) mbar_wait_drain(bar(C::bVF + s), (uint32_t)(uses - 1) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMAs --
        // Per listed KV tile, in two key halves h (N = 64): S_h, dP_h -> SR_h.  After
        // PR_h of tile t: dQ += dS_h K_h of tile t, then half h of tile t + 1 (its
        // first half waits for K and then V of tile t + 1, so the dQ product runs
        // while they land).
        constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false);
        constexpr uint32_t idesc_ts = idesc_bf16_f32(128, D, true);
        constexpr uint64_t kSubUnits = C::kSubBytes >> 4;
        const uint64_t dQk = smem_desc_sw128(base + C::kRes0, 16, 1024);
        const uint64_t dOk = smem_desc_sw128(base + C::kRes1, 16, 1024);
        // S = Q K^T over the 128 keys of the item's K stage, or dP = dO V^T
        auto issue_mm = [&](int it, bool dp) {
            const uint32_t st = base + (dp ? C::kV + (uint32_t)(it % C::kVStages) * C::kTileBytes
                                           : C::kK + (uint32_t)(it % C::kKStages) * C::kTileBytes);
            const uint64_t dB = smem_desc_sw128(st, 16, 1024);
            const uint64_t dA = dp ? dOk : dQk;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (uint64_t)((kk >> 2) * kSubUnits + (kk & 3) * 2);
                mma_ss_lead(lead, dp ? tP : tS, dA + off, dB + off, idesc_ss, kk > 0 ? 1u : 0u);
            }
        };
        auto issue_dq = [&](int it) {  // dQ += dS K (16 keys per step)
            const uint64_t dKm =
                smem_desc_sw128(base + C::kK + (uint32_t)(it % C::kKStages) * C::kTileBytes, C::kSubBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ts_lead(lead, tdQ, tDS + 64u * (uint32_t)(it & 1) + 8u * kk, dKm + (uint64_t)(kk * (2048 >> 4)),
                            idesc_ts, (it > 0 || kk > 0) ? 1u : 0u);
        };
        // S of item it after its K lands, dP after its V lands; the V stage is
        // free once dP has read it
        auto issue_s = [&](int it) -> bool {
            if (!mbar_wait(bar(C::bKF + it % C::kKStages), (it / C::kKStages) & 1, abort_flag, p.err,
                           BSATTN_FLAG_TIMEOUT))
                return false;
            tc_fence_after();
            issue_mm(it, false);
            if (!mbar_wait(bar(C::bVF + it % C::kVStages), (it / C::kVStages) & 1, abort_flag, p.err,
                           BSATTN_FLAG_TIMEOUT))
                return false;
            tc_fence_after();
            issue_mm(it, true);
            mma_commit_lead(lead, bar(C::bSR));
            mma_commit_lead(lead, bar(C::bVE + it % C::kVStages));
            return true;
        };
        bool ok = mbar_wait(bar(C::bRF), 0, abort_flag, p.err, BSATTN_FLAG_TIMEOUT);
        tc_fence_after();
        if (ok && total > 0) ok = issue_s(0);
        for (int it = 0; ok && it < total; ++it) {
            if (it + 1 < total) {
                // S and dP of this item are in the elementwise warps' registers
                if (!(ok = mbar_wait(bar(C::bSL + (it & 1)), (it >> 1) & 1, abort_flag, p.err,
                                     BSATTN_FLAG_TIMEOUT)))
                    break;
                tc_fence_after();
                if (!(ok = issue_s(it + 1))) break;
            }
            if (!(ok = mbar_wait(bar(C::bPR + (it & 1)), (it >> 1) & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT)))
                break;
            tc_fence_after();
            issue_dq(it);
            mma_commit_lead(lead, bar(C::bKE + it % C::kKStages));  // K stage free once dQ has read it
        }
        if (ok) mma_commit_lead(lead, bar(C::bDone));
        mma_commit_lead(lead, bar(C::bDrain));
        mbar_wait_drain(bar(C::bDrain), 0);
    } else if (warp >= 4) {
        // ------------------------------------------------- elementwise --
        const uint32_t q4 = warp & 3u;
        const int cg = (int)(warp - 4) >> 2;
        const int r = (int)(q4 * 32u + lane);  // query row of the tile
        const uint32_t la = (q4 * 32u) << 16;
        const int i = m * kTile + r;           // sequence-local query
        const long long vrow = vec_at(p, sg, b, h, m) + r;
        const float nl2 = p.lse2[vrow], ndd = p.dvec[vrow];  // -LSE2, -D of this query row
        const float sl2 = p.scale_log2;
        const int32_t dqid = (p.kind == BSATTN_MASK_DOCUMENT && i < sg.sq) ? p.doc_q[sg.q0 + i] : 0;
        bool ok = true;
        for (int it = 0; it < total; ++it) {
            const int s = it & 1;            // dS buffer
            const int ks = it % C::kKStages;  // K stage (item info)
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(C::bKF + ks), (it / C::kKStages) & 1, abort_flag,
                                                         p.err, BSATTN_FLAG_TIMEOUT))))
                break;
            const int n = reinterpret_cast<volatile int32_t *>(info)[ks * 2 + 0];
            const bool msk = reinterpret_cast<volatile int32_t *>(info)[ks * 2 + 1] != 0;
            int lim = min(kTile, sg.sk - n * kTile);
            if (msk && p.vl) lim = min(lim, __ldg(p.vl + (long long)b * p.num_n + n));
            // kept key columns: span [lo0, hi0) plus span [lo1, hi1), cut to [0, lim)
            const long long d = (long long)i - (long long)n * kTile;  // column of key j == i
            long long lo0 = 0, hi0 = lim, lo1 = 0, hi1 = 0;
            if (msk) {
                if (p.kind == BSATTN_MASK_CAUSAL) {
                    hi0 = min((long long)lim, d + 1);
                } else if (p.kind == BSATTN_MASK_SLIDING_WINDOW) {
                    lo0 = d - p.window_left + 1;
                    hi0 = min((long long)lim, d + 1);
                    hi1 = min((long long)lim, min((long long)p.sink_tokens - (long long)n * kTile, d + 1));
                } else if (p.kind == BSATTN_MASK_PREFIX) {
                    hi0 = min((long long)lim, max((long long)p.prefix_len - (long long)n * kTile, d + 1));
                }
            }
            const bool doc = msk && p.kind == BSATTN_MASK_DOCUMENT;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(C::bSR), it & 1, abort_flag, p.err,
                                                         BSATTN_FLAG_TIMEOUT))))
                break;
            tc_fence_after();
            // key chunks cg and cg + 2 (32 columns each) of S and dP; once both are
            // in registers the MMA warp may overwrite them with the next tile's
            uint32_t dw[2][16];
            uint32_t vsa[2][32], vpa[2][32];
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                tmem_ld32(tS + la + 32u * (cg + 2 * k2), vsa[k2]);
                tmem_ld32(tP + la + 32u * (cg + 2 * k2), vpa[k2]);
            }
            tmem_wait_ld();
            reg_fence(vsa[0]);
            reg_fence(vpa[0]);
            reg_fence(vsa[1]);
            reg_fence(vpa[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::bSL + s));
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int c = cg + 2 * k2;  // key chunk: columns [32 c, 32 c + 32)
                const uint32_t (&vs)[32] = vsa[k2];
                const uint32_t (&vp)[32] = vpa[k2];
                uint32_t keep = bwd_span_bits(lo0 - 32 * c, hi0 - 32 * c) | bwd_span_bits(lo1 - 32 * c, hi1 - 32 * c);
                if (doc) {
                    keep = 0u;
                    const uint32_t in_lim = bwd_span_bits(0, (long long)lim - 32 * c);
                    for (int x = 0; x < 32; ++x) {
                        const int j = n * kTile + 32 * c + x;
                        if (((in_lim >> x) & 1u) && __ldg(p.doc_k + sg.k0 + j) == dqid)
                            keep |= 1u << x;
                    }
                }
                // dS = 2^(s log2(e) scale - LSE2) (dP - D), two columns per packed
                // instruction; dropped columns enter the exponential as -inf.  A
                // chunk every lane keeps whole takes the form without selects.
                auto form = [&](auto masked) {
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        float x0, x1, t0, t1, d0, d1;
                        ffma2(x0, x1, __uint_as_float(vs[2 * x]), __uint_as_float(vs[2 * x + 1]), sl2, sl2, nl2,
                              nl2);
                        if constexpr (decltype(masked)::value) {
                            x0 = ((keep >> (2 * x)) & 1u) ? x0 : -INFINITY;
                            x1 = ((keep >> (2 * x + 1)) & 1u) ? x1 : -INFINITY;
                        }
                        fadd2(t0, t1, __uint_as_float(vp[2 * x]), __uint_as_float(vp[2 * x + 1]), ndd, ndd);
                        fmul2(d0, d1, ex2_approx(x0), ex2_approx(x1), t0, t1);
                        dw[k2][x] = pack_bf16x2(d0, d1);
                    }
                };
                if (__all_sync(0xffffffffu, keep == 0xffffffffu)) form(std::false_type{});
                else form(std::true_type{});
            }
            tmem_st16(tDS + 64u * s + la + 16u * cg, dw[0]);
            tmem_st16(tDS + 64u * s + la + 16u * (cg + 2), dw[1]);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::bPR + s));
        }
        // ------------------------------------------------- epilogue --
        if (ok && total > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::bDone), 0, abort_flag, p.err, BSATTN_FLAG_TIMEOUT));
            tc_fence_after();
        }
        if (ok) {
            const long long orow = ((sg.q0 + i) * p.H + h) * D;
            bwd_epilogue_half<D>(tdQ + la, total > 0, i < sg.sq, p.dq, p.grad_f32, orow, cg, p.scale);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Dynamic shared memory of the gradient kernels: at least 120 KB, so that one
// CTA holds an SM (each allocates all 512 TMEM columns).
template <int D>
constexpr uint32_t bwd_smem_bytes() {
    return BwdCfg<D>::kSmemAlloc > 120u * 1024u ? BwdCfg<D>::kSmemAlloc : 120u * 1024u;
}
template <int D>
constexpr uint32_t dq_smem_bytes() {
    return DqCfg<D>::kSmemAlloc > 120u * 1024u ? DqCfg<D>::kSmemAlloc : 120u * 1024u;
}
static_assert(DqCfg<128>::kSmemAlloc <= 232448u, "dQ kernel shared memory exceeds 227 KB");

template <int D>
cudaError_t prepare_bwd_kernels() {
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(bsattn_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bwd_smem_bytes<D>());
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(bsattn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dq_smem_bytes<D>());
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    return cudaSuccess;
}

unsigned warp_blocks(long long warps) { return (unsigned)((warps + 7) / 8); }

template <int D>
cudaError_t launch_bwd_d(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                         const CUtensorMap &tv, const CUtensorMap &tdo, cudaStream_t stream) {
    cudaError_t e = prepare_bwd_kernels<D>();
    if (e != cudaSuccess) return e;
    const long long q_tiles = p.varlen ? (long long)p.H * p.total_m : (long long)p.B * p.H * p.num_m;
    const long long kv_items = (long long)p.B * p.H * p.num_n;
    const size_t code_bytes = p.varlen ? (size_t)p.H * p.total_n : (size_t)kv_items * p.num_m;
    if ((e = cudaMemsetAsync(p.codes, 0, (code_bytes + 3) & ~(size_t)3, stream)) != cudaSuccess) return e;
    if (p.varlen) {
        bsattn_bwd_seq_kernel<<<1, 1024, 0, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (q_tiles > 0) {
        bsattn_bwd_scatter_kernel<<<warp_blocks(q_tiles), 256, 0, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    bsattn_bwd_scan_kernel<<<warp_blocks(kv_items), 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bsattn_bwd_order_kernel<<<1, 1024, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (q_tiles > 0) {
        bsattn_bwd_rows_kernel<<<warp_blocks(q_tiles * kTile / kRowsPerWarp), 256, 0, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // every KV tile writes its dK / dV rows (zeros without listed Q tiles)
    bsattn_bwd_dkdv_kernel<D><<<(unsigned)kv_items, kBwdThreads, bwd_smem_bytes<D>(), stream>>>(p, tq, tk, tv, tdo);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (q_tiles > 0)
        bsattn_bwd_dq_kernel<D><<<(unsigned)q_tiles, kBwdThreads, dq_smem_bytes<D>(), stream>>>(p, tq, tk, tv, tdo);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, cudaStream_t stream) {
    const long long q_tiles = p.varlen ? (long long)p.H * p.total_m : (long long)p.B * p.H * p.num_m;
    const long long kv_items = (long long)p.B * p.H * p.num_n;
    if (kv_items <= 0) return cudaSuccess;
    if (kv_items > 0x7fffffffLL || q_tiles > 0x7fffffffLL || (q_tiles * kTile + 7) / 8 > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    if (p.D == 64) return launch_bwd_d<64>(p, tq, tk, tv, tdo, stream);
    if (p.D == 128) return launch_bwd_d<128>(p, tq, tk, tv, tdo, stream);
    return cudaErrorInvalidValue;
}

}  // namespace bsattn
