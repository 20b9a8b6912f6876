// Backward of the block-sparse attention forward (batched).  With P the
// forward's probabilities over each row's allowed keys, O = P V and upstream
// gradient dO:
//   D_i = sum_d dO_i O_i,  dV = P^T dO,  dP = dO V^T,  dS = P (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
// Training needs the backward, which the pages list as missing ("[CuTe,Flex]
// varlen blocksparsity", flash-attention #2224; "[feat] VSA-256 fastpath",
// FastVideo #1354).  It runs as
//   1. a transpose of the forward's lists into KV-major lists (for each KV tile,
//      the Q tiles that selected it, full and mask separately, descending);
//   2. a row pass writing D and LSE * log2(e) into padded per-(b, h) rows;
//   3. the dK / dV kernel: one CTA per KV tile, S^T = K Q^T and dP^T = V dO^T per
//      listed Q tile on tcgen05, P^T and dS^T formed per key row in TMEM, then
//      dV += P^T dO and dK += dS^T Q accumulated in TMEM;
//   4. the dQ kernel: one CTA per Q tile, S = Q K^T and dP = dO V^T per listed KV
//      tile, dS per query row, dQ += dS K accumulated in TMEM.
// P is recomputed from the forward's LSE (no running maximum) and rounded to
// bf16 before the P^T dO product, as the forward rounds it before P V; dS is
// rounded to bf16 before its products.
#include <cuda_bf16.h>

#include "bsattn_internal.h"
#include "sm100_ptx.cuh"

namespace bsattn {

namespace {

// ------------------------------------------------------------ 1. transpose --
// One CTA per (b, h): Q-tile rows are taken from the last to the first, each
// row's entries appended to their KV tile's list, so every KV-major list is
// descending in m.  Entries outside [0, num_n) are skipped and flagged.
__global__ void __launch_bounds__(256) bsattn_bwd_transpose_kernel(BwdParams p) {
    const int bh = blockIdx.x;
    const long long crow = (long long)bh * p.num_n;  // first KV-major count of (b, h)
    for (int n = threadIdx.x; n < p.num_n; n += blockDim.x) {
        p.t_full_cnt[crow + n] = 0;
        p.t_mask_cnt[crow + n] = 0;
    }
    __syncthreads();
    bool bad = false;
    for (int m = p.num_m - 1; m >= 0; --m) {
        const long long r = (long long)bh * p.num_m + m;
        for (int list = 0; list < 2; ++list) {
            const int32_t *cnt_in = list ? p.mask_cnt : p.full_cnt;
            const int32_t *idx_in = list ? p.mask_idx : p.full_idx;
            int32_t *cnt_out = list ? p.t_mask_cnt : p.t_full_cnt;
            int32_t *idx_out = list ? p.t_mask_idx : p.t_full_idx;
            int c = cnt_in[r];
            if (c < 0 || c > p.num_n) {
                bad = true;
                c = c < 0 ? 0 : p.num_n;
            }
            for (int e = threadIdx.x; e < c; e += blockDim.x) {
                const int n = idx_in[r * p.num_n + e];
                if (n < 0 || n >= p.num_n) {
                    bad = true;
                    continue;
                }
                const int pos = atomicAdd(&cnt_out[crow + n], 1);
                if (pos < p.num_m) idx_out[(crow + n) * p.num_m + pos] = m;
                else bad = true;  // a tile listed twice in one row overflows its column
            }
        }
        __syncthreads();  // the next (smaller) m is appended after this one
    }
    for (long long e = threadIdx.x; e < (long long)p.num_n * p.num_m; e += blockDim.x) {
        const long long n = e / p.num_m;
        const int k = (int)(e - n * p.num_m);
        if (k >= min(p.t_full_cnt[crow + n], p.num_m)) p.t_full_idx[(crow + n) * p.num_m + k] = -1;
        if (k >= min(p.t_mask_cnt[crow + n], p.num_m)) p.t_mask_idx[(crow + n) * p.num_m + k] = -1;
    }
    __syncthreads();
    for (int n = threadIdx.x; n < p.num_n; n += blockDim.x) {
        p.t_full_cnt[crow + n] = min(p.t_full_cnt[crow + n], p.num_m);
        p.t_mask_cnt[crow + n] = min(p.t_mask_cnt[crow + n], p.num_m);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0 && p.err) atomicOr(p.err, BSATTN_FLAG_BAD_INDEX);
}

// ------------------------------------------------------------ 2. row pass --
// One warp per query row (b, i, h): D = sum_d dO O in fp32 and LSE * log2(e), in
// rows of num_m * 128 per (b, h).  Rows past seqlen_q, and rows with no keys
// (LSE = -inf), get LSE2 = +inf, so every probability they would form is 0.
__global__ void __launch_bounds__(256) bsattn_bwd_rows_kernel(BwdParams p) {
    const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const long long per_bh = (long long)p.num_m * kTile;
    if (w >= (long long)p.B * p.H * per_bh) return;
    const long long bh = w / per_bh;
    const int i = (int)(w - bh * per_bh);
    const int b = (int)(bh / p.H), h = (int)(bh - (long long)b * p.H);
    float d = 0.f, l2 = INFINITY;
    if (i < p.seqlen_q) {
        const long long row = ((long long)b * p.seqlen_q + i) * p.H + h;  // [B, S, H] row
        for (int c = lane; c < p.D; c += 32) {
            const float g = __uint_as_float((uint32_t)p.dout[row * p.D + c] << 16);
            const float o = p.o_f32 ? static_cast<const float *>(p.o)[row * p.D + c]
                                    : __uint_as_float((uint32_t)static_cast<const uint16_t *>(p.o)[row * p.D + c] << 16);
            d = fmaf(g, o, d);
        }
        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        const float lse = p.lse[bh * p.seqlen_q + i];
        l2 = lse == -INFINITY ? INFINITY : lse * 1.4426950408889634f;
    }
    if (lane == 0) {
        p.dvec[bh * per_bh + i] = d;
        p.lse2[bh * per_bh + i] = l2;
    }
}

// Shared memory of both gradient kernels: two resident tiles, a ring of two
// stages of two tiles plus two 128-float vectors, barriers, item info, misc.
template <int D>
struct BwdCfg {
    static constexpr uint32_t kTileBytes = kTile * D * 2;
    static constexpr int kSub = D / 64;                       // 64-column swizzle spans per tile
    static constexpr uint32_t kSubBytes = kTile * 64 * 2;
    static constexpr uint32_t kRes0 = 0, kRes1 = kTileBytes;  // resident tiles
    static constexpr uint32_t kSt = 2 * kTileBytes;           // stage s: kSt + s * 2 * kTileBytes
    static constexpr uint32_t kVec = kSt + 4 * kTileBytes;   // stage s: 2 x 128 floats at kVec + 1024 s
    static constexpr uint32_t kBar = kVec + 2048;
    static constexpr int bRF = 0, bF = 1, bE = 3, bSR = 5, bPR = 6, bDone = 7, bDrain = 8, kNumBars = 9;
    static constexpr uint32_t kInfo = kBar + kNumBars * 8;    // int32 [2][4]
    static constexpr uint32_t kMisc = kInfo + 32;             // [0] tmem base, [1] abort
    static constexpr uint32_t kBytes = kMisc + 16;
    static constexpr uint32_t kSmemAlloc = kBytes + 1024;     // slack for 1024-byte alignment
};

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
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::bF + s), 1);
            mbar_init(bar(C::bE + s), 1);
        }
        mbar_init(bar(C::bSR), 1);
        mbar_init(bar(C::bPR), 4);  // one arrival per elementwise warp
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

// ----------------------------------------------------------- 3. dK and dV --
// One CTA per (b, h, KV tile n), 256 threads: warp 0 loads (K and V of the tile
// once, then Q, dO, LSE2 and D of each listed Q tile into a two-stage ring),
// warp 1 issues the MMAs, warp 2 owns TMEM, warps 4-7 (one per TMEM lane
// quarter; thread = key row) form P^T and dS^T and write the gradients.
// TMEM: S^T [0, 128), dP^T [128, 256), dV [256, 256 + D), dK [256 + D, 256 + 2D);
// P^T (bf16) overwrites the first 64 columns of S^T, dS^T those of dP^T.
template <int D>
__global__ void __launch_bounds__(256, 1)
    bsattn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tq,
                           const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                           const __grid_constant__ CUtensorMap tdo) {
    using C = BwdCfg<D>;
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

    const int n = (int)(blockIdx.x % (unsigned)p.num_n);
    const int bh = (int)(blockIdx.x / (unsigned)p.num_n);
    const int b = bh / p.H, h = bh - b * p.H;
    const long long crow = (long long)bh * p.num_n + n;
    const int cm = min(max(p.t_mask_cnt[crow], 0), p.num_m);
    const int cf = min(max(p.t_full_cnt[crow], 0), p.num_m);
    const int total = cm + cf;  // listed Q tiles: the mask list, then the full list

    bwd_init<D>(gbase, base, warp);
    const uint32_t tmem = misc[0];
    const uint32_t tS = tmem, tP = tmem + 128u, tdV = tmem + 256u, tdK = tmem + 256u + D;

    if (warp == 0) {
        // ------------------------------------------------------- loads --
        const int kvrow = b * p.seqlen_k + n * kTile;
        mbar_arrive_expect_tx_lead(lead, bar(C::bRF), 2 * C::kTileBytes);
        for (int x = 0; x < C::kSub; ++x) {
            tma_load_3d_lead(lead, base + C::kRes0 + x * C::kSubBytes, &tk, bar(C::bRF), x * 64, h, kvrow);
            tma_load_3d_lead(lead, base + C::kRes1 + x * C::kSubBytes, &tv, bar(C::bRF), x * 64, h, kvrow);
        }
        int it = 0;
        for (; it < total; ++it) {
            const int s = it & 1;
            if (!mbar_wait(bar(C::bE + s), ((it >> 1) & 1) ^ 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT)) break;
            const int m = it < cm ? p.t_mask_idx[crow * p.num_m + it] : p.t_full_idx[crow * p.num_m + (it - cm)];
            info[s * 4 + 0] = m;
            info[s * 4 + 1] = it < cm ? 1 : 0;
            const int qrow = b * p.seqlen_q + m * kTile;
            const uint32_t st = base + C::kSt + (uint32_t)s * 2u * C::kTileBytes;
            mbar_arrive_expect_tx_lead(lead, bar(C::bF + s), 2 * C::kTileBytes + 1024u);
            for (int x = 0; x < C::kSub; ++x) {
                tma_load_3d_lead(lead, st + x * C::kSubBytes, &tq, bar(C::bF + s), x * 64, h, qrow);
                tma_load_3d_lead(lead, st + C::kTileBytes + x * C::kSubBytes, &tdo, bar(C::bF + s), x * 64,
                                 h, qrow);
            }
            const long long vrow = (long long)bh * p.num_m * kTile + (long long)m * kTile;
            bulk_g2s_lead(lead, base + C::kVec + 1024u * s, p.lse2 + vrow, 512u, bar(C::bF + s));
            bulk_g2s_lead(lead, base + C::kVec + 1024u * s + 512u, p.dvec + vrow, 512u, bar(C::bF + s));
        }
        // every copy issued has landed before the CTA may exit
        mbar_wait_drain(bar(C::bRF), 0);
        for (int s = 0; s < 2; ++s) {
            const int uses = (it + 1 - s) / 2;
            if (uses > 0) mbar_wait_drain(bar(C::bF + s), (uint32_t)(uses - 1) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMAs --
        constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false);
        constexpr uint32_t idesc_ts = idesc_bf16_f32(128, D, true);
        constexpr uint64_t kSubUnits = C::kSubBytes >> 4;
        const uint64_t dKk = smem_desc_sw128(base + C::kRes0, 16, 1024);
        const uint64_t dVk = smem_desc_sw128(base + C::kRes1, 16, 1024);
        bool ok = mbar_wait(bar(C::bRF), 0, abort_flag, p.err, BSATTN_FLAG_TIMEOUT);
        tc_fence_after();
        for (int it = 0; ok && it < total; ++it) {
            const int s = it & 1;
            if (!(ok = mbar_wait(bar(C::bF + s), (it >> 1) & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT))) break;
            tc_fence_after();
            const uint32_t st = base + C::kSt + (uint32_t)s * 2u * C::kTileBytes;
            const uint64_t dQk = smem_desc_sw128(st, 16, 1024);
            const uint64_t dOk = smem_desc_sw128(st + C::kTileBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // S^T = K Q^T
                const uint64_t off = (uint64_t)((kk >> 2) * kSubUnits + (kk & 3) * 2);
                mma_ss_lead(lead, tS, dKk + off, dQk + off, idesc_ss, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // dP^T = V dO^T
                const uint64_t off = (uint64_t)((kk >> 2) * kSubUnits + (kk & 3) * 2);
                mma_ss_lead(lead, tP, dVk + off, dOk + off, idesc_ss, kk > 0 ? 1u : 0u);
            }
            mma_commit_lead(lead, bar(C::bSR));
            if (!(ok = mbar_wait(bar(C::bPR), it & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT))) break;
            tc_fence_after();
            const uint64_t dOm = smem_desc_sw128(st + C::kTileBytes, C::kSubBytes, 1024);
            const uint64_t dQm = smem_desc_sw128(st, C::kSubBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)  // dV += P^T dO
                mma_ts_lead(lead, tdV, tS + kk * 8, dOm + (uint64_t)(kk * (2048 >> 4)), idesc_ts,
                            (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)  // dK += dS^T Q
                mma_ts_lead(lead, tdK, tP + kk * 8, dQm + (uint64_t)(kk * (2048 >> 4)), idesc_ts,
                            (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit_lead(lead, bar(C::bE + s));  // stage free once these have read it
        }
        if (ok) mma_commit_lead(lead, bar(C::bDone));
        mma_commit_lead(lead, bar(C::bDrain));
        mbar_wait_drain(bar(C::bDrain), 0);
    } else if (warp >= 4) {
        // ------------------------------------------------- elementwise --
        const uint32_t q4 = warp & 3u;
        const int r = (int)(q4 * 32u + lane);  // key row of the tile
        const uint32_t la = (q4 * 32u) << 16;  // TMEM lane offset of this warp
        const int j = n * kTile + r;           // sequence-local key
        const int klim_full = min(kTile, p.seqlen_k - n * kTile);
        int klim_mask = klim_full;
        if (p.vl) klim_mask = min(klim_mask, p.vl[(long long)b * p.num_n + n]);
        const float sl2 = p.scale_log2;
        const float *vecs = reinterpret_cast<const float *>(gbase + C::kVec);
        bool ok = true;
        for (int it = 0; it < total; ++it) {
            const int s = it & 1;
            bool w = mbar_wait(bar(C::bF + s), (it >> 1) & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT);
            w = w && mbar_wait(bar(C::bSR), it & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT);
            if (!(ok = __all_sync(0xffffffffu, w))) break;
            tc_fence_after();
            const int m = reinterpret_cast<volatile int32_t *>(info)[s * 4 + 0];
            const bool msk = reinterpret_cast<volatile int32_t *>(info)[s * 4 + 1] != 0;
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
            const int32_t dk = doc ? p.doc_k[(long long)b * p.seqlen_k + j] : 0;
            const float *l2 = vecs + s * 256, *dd = l2 + 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t vs[32], vp[32];
                tmem_ld32(tS + la + 32u * c, vs);
                tmem_ld32(tP + la + 32u * c, vp);
                tmem_wait_ld();
                reg_fence(vs);
                reg_fence(vp);
                uint32_t keep = bwd_span_bits(lo - 32 * c, hi - 32 * c);
                if (doc) {
                    keep = 0u;
                    for (int x = 0; x < 32; ++x) {
                        const int i = m * kTile + 32 * c + x;
                        if (i < p.seqlen_q && __ldg(p.doc_q + (long long)b * p.seqlen_q + i) == dk)
                            keep |= 1u << x;
                    }
                }
                uint32_t pw[16], dw[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int c0 = 32 * c + 2 * x;
                    const float p0 = ((keep >> (2 * x)) & 1u)
                                         ? ex2_approx(fmaf(__uint_as_float(vs[2 * x]), sl2, -l2[c0])) : 0.f;
                    const float p1 = ((keep >> (2 * x + 1)) & 1u)
                                         ? ex2_approx(fmaf(__uint_as_float(vs[2 * x + 1]), sl2, -l2[c0 + 1]))
                                         : 0.f;
                    const float ds0 = p0 * (__uint_as_float(vp[2 * x]) - dd[c0]);
                    const float ds1 = p1 * (__uint_as_float(vp[2 * x + 1]) - dd[c0 + 1]);
                    pw[x] = pack_bf16x2(p0, p1);
                    dw[x] = pack_bf16x2(ds0, ds1);
                }
                tmem_st16(tS + la + 16u * c, pw);
                tmem_st16(tP + la + 16u * c, dw);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::bPR));
        }
        // ------------------------------------------------- epilogue --
        if (ok && total > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::bDone), 0, abort_flag, p.err, BSATTN_FLAG_TIMEOUT));
            tc_fence_after();
        }
        if (ok) {
            const bool store = j < p.seqlen_k;
            const long long orow = (((long long)b * p.seqlen_k + j) * p.H + h) * D;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const uint32_t tacc = g ? tdK : tdV;
                const float mul = g ? p.scale : 1.f;
                void *dst = g ? p.dk : p.dv;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    if (total > 0) {
                        tmem_ld32(tacc + la + 32u * c, v);
                        tmem_wait_ld();
                        reg_fence(v);
                    } else {
#pragma unroll
                        for (int x = 0; x < 32; ++x) v[x] = 0u;
                    }
                    if (!store) continue;
                    bwd_store_row32(dst, p.grad_f32, orow + 32 * c, v, mul);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 4. dQ --
// One CTA per (b, h, Q tile m), 256 threads, the same roles: Q and dO of the tile
// stay resident, K and V of each listed KV tile (the forward's mask list, then
// its full list; entries outside [0, num_n) skipped by every role alike) pass
// through the two-stage ring.  Thread = query row.
// TMEM: S [0, 128), dP [128, 256), dQ [256, 256 + D); dS (bf16) overwrites the
// first 64 columns of dP.
template <int D>
__global__ void __launch_bounds__(256, 1)
    bsattn_bwd_dq_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                         const __grid_constant__ CUtensorMap tdo) {
    using C = BwdCfg<D>;
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

    const int m = (int)(blockIdx.x % (unsigned)p.num_m);
    const int bh = (int)(blockIdx.x / (unsigned)p.num_m);
    const int b = bh / p.H, h = bh - b * p.H;
    const long long crow = (long long)bh * p.num_m + m;
    const int cm = min(max(p.mask_cnt[crow], 0), p.num_n);
    const int cf = min(max(p.full_cnt[crow], 0), p.num_n);
    // raw entry e of the item sequence (mask list first); -1 when out of range
    auto entry = [&](int e) -> int {
        const int n = e < cm ? __ldg(p.mask_idx + crow * p.num_n + e) : __ldg(p.full_idx + crow * p.num_n + (e - cm));
        return (n >= 0 && n < p.num_n) ? n : -1;
    };
    int total = 0;  // valid entries: counted by every thread the same way
    for (int e = 0; e < cm + cf; ++e) total += entry(e) >= 0 ? 1 : 0;

    bwd_init<D>(gbase, base, warp);
    const uint32_t tmem = misc[0];
    const uint32_t tS = tmem, tP = tmem + 128u, tdQ = tmem + 256u;

    if (warp == 0) {
        // ------------------------------------------------------- loads --
        const int qrow = b * p.seqlen_q + m * kTile;
        mbar_arrive_expect_tx_lead(lead, bar(C::bRF), 2 * C::kTileBytes);
        for (int x = 0; x < C::kSub; ++x) {
            tma_load_3d_lead(lead, base + C::kRes0 + x * C::kSubBytes, &tq, bar(C::bRF), x * 64, h, qrow);
            tma_load_3d_lead(lead, base + C::kRes1 + x * C::kSubBytes, &tdo, bar(C::bRF), x * 64, h, qrow);
        }
        int it = 0;
        for (int e = 0; e < cm + cf; ++e) {
            const int n = entry(e);
            if (n < 0) continue;
            const int s = it & 1;
            if (!mbar_wait(bar(C::bE + s), ((it >> 1) & 1) ^ 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT)) break;
            info[s * 4 + 0] = n;
            info[s * 4 + 1] = e < cm ? 1 : 0;
            const int kvrow = b * p.seqlen_k + n * kTile;
            const uint32_t st = base + C::kSt + (uint32_t)s * 2u * C::kTileBytes;
            mbar_arrive_expect_tx_lead(lead, bar(C::bF + s), 2 * C::kTileBytes);
            for (int x = 0; x < C::kSub; ++x) {
                tma_load_3d_lead(lead, st + x * C::kSubBytes, &tk, bar(C::bF + s), x * 64, h, kvrow);
                tma_load_3d_lead(lead, st + C::kTileBytes + x * C::kSubBytes, &tv, bar(C::bF + s), x * 64, h,
                                 kvrow);
            }
            ++it;
        }
        mbar_wait_drain(bar(C::bRF), 0);
        for (int s = 0; s < 2; ++s) {
            const int uses = (it + 1 - s) / 2;
            if (uses > 0) mbar_wait_drain(bar(C::bF + s), (uint32_t)(uses - 1) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMAs --
        constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false);
        constexpr uint32_t idesc_ts = idesc_bf16_f32(128, D, true);
        constexpr uint64_t kSubUnits = C::kSubBytes >> 4;
        const uint64_t dQk = smem_desc_sw128(base + C::kRes0, 16, 1024);
        const uint64_t dOk = smem_desc_sw128(base + C::kRes1, 16, 1024);
        bool ok = mbar_wait(bar(C::bRF), 0, abort_flag, p.err, BSATTN_FLAG_TIMEOUT);
        tc_fence_after();
        for (int it = 0; ok && it < total; ++it) {
            const int s = it & 1;
            if (!(ok = mbar_wait(bar(C::bF + s), (it >> 1) & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT))) break;
            tc_fence_after();
            const uint32_t st = base + C::kSt + (uint32_t)s * 2u * C::kTileBytes;
            const uint64_t dKk = smem_desc_sw128(st, 16, 1024);
            const uint64_t dVk = smem_desc_sw128(st + C::kTileBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // S = Q K^T
                const uint64_t off = (uint64_t)((kk >> 2) * kSubUnits + (kk & 3) * 2);
                mma_ss_lead(lead, tS, dQk + off, dKk + off, idesc_ss, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // dP = dO V^T
                const uint64_t off = (uint64_t)((kk >> 2) * kSubUnits + (kk & 3) * 2);
                mma_ss_lead(lead, tP, dOk + off, dVk + off, idesc_ss, kk > 0 ? 1u : 0u);
            }
            mma_commit_lead(lead, bar(C::bSR));
            if (!(ok = mbar_wait(bar(C::bPR), it & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT))) break;
            tc_fence_after();
            const uint64_t dKm = smem_desc_sw128(st, C::kSubBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)  // dQ += dS K
                mma_ts_lead(lead, tdQ, tP + kk * 8, dKm + (uint64_t)(kk * (2048 >> 4)), idesc_ts,
                            (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit_lead(lead, bar(C::bE + s));
        }
        if (ok) mma_commit_lead(lead, bar(C::bDone));
        mma_commit_lead(lead, bar(C::bDrain));
        mbar_wait_drain(bar(C::bDrain), 0);
    } else if (warp >= 4) {
        // ------------------------------------------------- elementwise --
        const uint32_t q4 = warp & 3u;
        const int r = (int)(q4 * 32u + lane);  // query row of the tile
        const uint32_t la = (q4 * 32u) << 16;
        const int i = m * kTile + r;           // sequence-local query
        const long long vrow = (long long)bh * p.num_m * kTile + (long long)m * kTile + r;
        const float l2 = p.lse2[vrow], dd = p.dvec[vrow];
        const float sl2 = p.scale_log2;
        const int32_t dqid = (p.kind == BSATTN_MASK_DOCUMENT && i < p.seqlen_q)
                                 ? p.doc_q[(long long)b * p.seqlen_q + i] : 0;
        bool ok = true;
        for (int it = 0; it < total; ++it) {
            const int s = it & 1;
            bool w = mbar_wait(bar(C::bF + s), (it >> 1) & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT);
            w = w && mbar_wait(bar(C::bSR), it & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT);
            if (!(ok = __all_sync(0xffffffffu, w))) break;
            tc_fence_after();
            const int n = reinterpret_cast<volatile int32_t *>(info)[s * 4 + 0];
            const bool msk = reinterpret_cast<volatile int32_t *>(info)[s * 4 + 1] != 0;
            int lim = min(kTile, p.seqlen_k - n * kTile);
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
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t vs[32], vp[32];
                tmem_ld32(tS + la + 32u * c, vs);
                tmem_ld32(tP + la + 32u * c, vp);
                tmem_wait_ld();
                reg_fence(vs);
                reg_fence(vp);
                uint32_t keep = bwd_span_bits(lo0 - 32 * c, hi0 - 32 * c) | bwd_span_bits(lo1 - 32 * c, hi1 - 32 * c);
                if (doc) {
                    keep = 0u;
                    const uint32_t in_lim = bwd_span_bits(0, (long long)lim - 32 * c);
                    for (int x = 0; x < 32; ++x) {
                        const int j = n * kTile + 32 * c + x;
                        if (((in_lim >> x) & 1u) && __ldg(p.doc_k + (long long)b * p.seqlen_k + j) == dqid)
                            keep |= 1u << x;
                    }
                }
                uint32_t dw[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float p0 = ((keep >> (2 * x)) & 1u) ? ex2_approx(fmaf(__uint_as_float(vs[2 * x]), sl2, -l2)) : 0.f;
                    const float p1 =
                        ((keep >> (2 * x + 1)) & 1u) ? ex2_approx(fmaf(__uint_as_float(vs[2 * x + 1]), sl2, -l2)) : 0.f;
                    dw[x] = pack_bf16x2(p0 * (__uint_as_float(vp[2 * x]) - dd), p1 * (__uint_as_float(vp[2 * x + 1]) - dd));
                }
                tmem_st16(tP + la + 16u * c, dw);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::bPR));
        }
        // ------------------------------------------------- epilogue --
        if (ok && total > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::bDone), 0, abort_flag, p.err, BSATTN_FLAG_TIMEOUT));
            tc_fence_after();
        }
        if (ok) {
            const bool store = i < p.seqlen_q;
            const long long orow = (((long long)b * p.seqlen_q + i) * p.H + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                if (total > 0) {
                    tmem_ld32(tdQ + la + 32u * c, v);
                    tmem_wait_ld();
                    reg_fence(v);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] = 0u;
                }
                if (!store) continue;
                bwd_store_row32(p.dq, p.grad_f32, orow + 32 * c, v, p.scale);
            }
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
                                 (int)bwd_smem_bytes<D>());
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    return cudaSuccess;
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                         const CUtensorMap &tv, const CUtensorMap &tdo, cudaStream_t stream) {
    cudaError_t e = prepare_bwd_kernels<D>();
    if (e != cudaSuccess) return e;
    const long long bh = (long long)p.B * p.H;
    bsattn_bwd_transpose_kernel<<<(unsigned)bh, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long long rows = bh * p.num_m * kTile;
    bsattn_bwd_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bsattn_bwd_dkdv_kernel<D><<<(unsigned)(bh * p.num_n), 256, bwd_smem_bytes<D>(), stream>>>(p, tq, tk, tv, tdo);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bsattn_bwd_dq_kernel<D><<<(unsigned)(bh * p.num_m), 256, bwd_smem_bytes<D>(), stream>>>(p, tq, tk, tv, tdo);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, cudaStream_t stream) {
    const long long bh = (long long)p.B * p.H;
    if (bh <= 0 || p.num_m <= 0 || p.num_n <= 0) return cudaSuccess;
    if (bh * p.num_n > 0x7fffffffLL || bh * p.num_m > 0x7fffffffLL ||
        (bh * p.num_m * kTile + 7) / 8 > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    if (p.D == 64) return launch_bwd_d<64>(p, tq, tk, tv, tdo, stream);
    if (p.D == 128) return launch_bwd_d<128>(p, tq, tk, tv, tdo, stream);
    return cudaErrorInvalidValue;
}

}  // namespace bsattn
