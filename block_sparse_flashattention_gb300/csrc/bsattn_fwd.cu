// Block-sparse attention forward for sm_103a: TMA + tcgen05 + TMEM, persistent,
// warp-specialised.
//
// What it computes ("[CuTe,Flex] varlen blocksparsity", flash-attention #2224):
// for each (head, Q tile) it visits only the KV tiles of the row's mask list and
// full list, runs an online softmax over them (mask_mod only on mask tiles) and
// writes O and LSE.  The K/V loads follow the listed blocks ("Dense
// FlashAttention vs Block-Sparse Attention", sections 4 and 6: the next tile's
// address is only known from the list) and both K and V jump to each listed tile.
//
// Work unit = (head, pair of consecutive packed Q tiles).  The two tiles' lists
// are merged on the fly, largest global KV row first; a KV tile listed by both
// tiles is loaded once and used by both (the paired 128-row halves of a 256-token
// VSA block share their whole list; neighbouring sliding-window tiles share all
// but one tile).
//
// Roles (384 threads, one CTA per SM, all of TMEM):
//   warp 0      TMA producer: walks the lists (next index read one step ahead),
//               loads Q tiles and K/V tiles into rings of shared-memory stages
//   warp 1      tcgen05 issuer: S_t = Q_t K^T into TMEM, O_t += P_t V with P in TMEM
//   warp 2      owns the TMEM allocation
//   warp 3      scheduler: claims work units and reads the head of their lists
//               one unit ahead of the producer
//   warps 4-7   softmax + O rescale + epilogue for tile 0 of the pair
//   warps 8-11  the same for tile 1
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D);
// P_t (bf16 pairs) overwrites the first 64 columns of S_t.
#include "bsattn_internal.h"
#include "sm100_ptx.cuh"

namespace bsattn {

namespace {

constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
// Register split: the kernel is built for 168 registers per thread at launch
// (65536 / 384, rounded down to a multiple of 8), i.e. 64512 for the CTA.  The
// control warpgroup gives registers back and the two softmax warpgroups take
// them: 128 * 120 + 2 * 128 * 192 = 64512, exactly the launch allocation.
// (setmaxnreg sits inside each role's branch so that ptxas applies the budget there.)
constexpr int kLaunchRegs = 168;
constexpr int kStagesK128 = 2;  // K ring depth at d = 128 (3 measured no faster)
constexpr uint32_t kCtrlRegs = 120, kSoftmaxRegs = 192;
static_assert(128 * kCtrlRegs + 2 * 128 * kSoftmaxRegs <= (uint32_t)kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint32_t kSubTileBytes = kTile * 64 * 2;  // 128 rows x 64 bf16 (one 128-byte swizzle span)

// Item flags (producer -> MMA issuer).
constexpr uint32_t kPart0 = 1u, kPart1 = 2u, kMask0 = 4u, kMask1 = 8u, kEnd = 16u, kBound0 = 32u,
                   kBound1 = 64u, kLast0 = 128u, kLast1 = 256u,  // kLast_t: tile t's last item
                   kStop = 512u,                                  // no further units
                   kSummary = 1024u;                              // K/V from the tile summaries
// Per-tile flags (MMA issuer -> softmax).
constexpr uint32_t kSMask = 1u, kSBound = 2u, kSEnd = 4u, kSStop = 8u, kSSummary = 16u;
constexpr int kUnitRing = 4;  // unit ids in flight between the producer and the softmax

struct Item {
    int32_t krow;  // packed K/V row of the tile
    int32_t n0, n1;
    uint32_t flags;
    int32_t lim0, lim1;  // per tile: keys of the tile that may be kept (sequence end,
                         // and the valid length on mask tiles)
    int32_t pad0, pad1;
};

struct SInfo {
    int32_t n;
    uint32_t flags;
    int32_t lim;
    int32_t pad;
};

struct TileInfo {
    int valid;
    int b, m;
    int qrow0;    // packed q row of the tile's first row
    int nvalid;   // rows of the tile inside the sequence
    int krow0;    // packed k row of the sequence's first key
    int sk;       // seqlen_k(b)
    int nn;       // num_n(b)
    long long cnt_at, idx_at;
};

// What the scheduler warp hands the producer for one unit: the unit id, where
// its two Q tiles sit, and the head of each of their lists (counts, first two
// entries, and the valid length of the first mask tile), so that the producer
// can issue the unit's first loads without waiting on global memory.
struct UnitDesc {
    TileInfo ti[2];
    int32_t u;       // unit id; -1: no further units
    int32_t cnt[4];  // [2t] mask count, [2t + 1] full count of tile t, as stored
    int32_t e0[4];   // first entry of each list (-1 if the list has no room for it)
    int32_t e1[4];   // second entry
    int32_t vl[2];   // valid length of tile t's first mask entry (kTile without one)
    int32_t pad;
};
constexpr int kUnitDescs = 2;

template <int D>
struct Cfg {
    static constexpr int kStagesK = D == 128 ? kStagesK128 : 4;
    static constexpr int kStagesV = D == 128 ? 2 : 4;
    static constexpr uint32_t kTileBytes = kTile * D * 2;
    static constexpr int kSub = D / 64;  // 64-column swizzle spans per tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + 2 * kTileBytes;
    static constexpr uint32_t kV = kK + kStagesK * kTileBytes;
    static constexpr uint32_t kBar = kV + kStagesV * kTileBytes;
    // barrier indices.  bKF + s completes when item s's K tile and its V tile have
    // both landed (one wait per item covers both loads); bKE / bVE release the
    // K and V stages.
    static constexpr int bKF = 0, bKE = kStagesK, bVE = 2 * kStagesK;
    static constexpr int bQF = 2 * kStagesK + kStagesV, bQE = bQF + 2, bSR = bQF + 4,
                         bPR = bQF + 6,  // bPR + 2t + half
                         bED = bQF + 10, bUF = bQF + 12, bUE = bQF + 14, bDrain = bQF + 16,
                         kNumBars = bQF + 17;
    static constexpr uint32_t kItems = kBar + kNumBars * 8;
    static constexpr uint32_t kSInfo = kItems + kStagesK * sizeof(Item);
    static constexpr uint32_t kUnits = kSInfo + 2 * sizeof(SInfo);
    static constexpr uint32_t kMisc = kUnits + kUnitRing * 4;  // [0] tmem base, [1] abort
    static constexpr uint32_t kUDesc = kMisc + 16;               // 2 unit descriptors
    // Epilogue scratch: 4 KB per softmax warp (32 rows x 128 bytes).
    static constexpr uint32_t kEpi = (kUDesc + kUnitDescs * sizeof(UnitDesc) + 127u) & ~127u;
    static constexpr uint32_t kBytes = kEpi + 8u * 4096u;
    static constexpr uint32_t kSmemAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};


// Geometry of packed Q tile T of head h.  A varlen sequence whose offsets leave
// the packed arrays (cu_q[b] < 0, cu_q[b + 1] past the packed query rows, or the
// same for keys), or whose KV tiles outnumber the valid-length row stride, yields
// no tile; then, when `err` is given, BSATTN_FLAG_BAD_SEQLENS is set.
__device__ __forceinline__ TileInfo tile_info(const FwdParams &p, int h, int T, int32_t *err = nullptr) {
    TileInfo t;
    t.valid = 0;
    t.b = t.m = t.qrow0 = t.nvalid = t.krow0 = t.sk = t.nn = 0;
    t.cnt_at = t.idx_at = 0;
    if (T >= p.total_m) return t;
    int sq;
    if (!p.varlen) {
        t.b = T / p.num_m;
        t.m = T - t.b * p.num_m;
        sq = p.seqlen_q;
        t.sk = p.seqlen_k;
        t.qrow0 = t.b * p.seqlen_q + t.m * kTile;
        t.krow0 = t.b * p.seqlen_k;
        t.nn = p.num_n;
        t.cnt_at = ((long long)t.b * p.H + h) * p.num_m + t.m;
        t.idx_at = t.cnt_at * p.num_n;
    } else {
        if (T >= p.cu_tm[p.B]) return t;
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.cu_tm[mid] <= T) lo = mid;
            else hi = mid - 1;
        }
        t.b = lo;
        t.m = T - p.cu_tm[lo];
        // every load first (they go out together), then the checks
        const int q0 = p.cu_q[lo], q1 = p.cu_q[lo + 1], k0 = p.cu_k[lo], k1 = p.cu_k[lo + 1];
        const int off = p.cu_off[lo];
        sq = q1 - q0;
        t.sk = k1 - k0;
        t.qrow0 = q0 + t.m * kTile;
        t.krow0 = k0;
        t.nn = (t.sk + kTile - 1) / kTile;
        t.cnt_at = (long long)h * p.total_m + T;
        t.idx_at = (long long)h * p.total_n + off + (long long)t.m * t.nn;
        const bool bad = q0 < 0 || q1 < q0 || q1 > p.seqlen_q || k0 < 0 || k1 < k0 || k1 > p.seqlen_k ||
                         (p.vl && t.nn > p.vl_stride) || off < 0 ||
                         (long long)off + (long long)(t.m + 1) * t.nn > p.total_n;
        if (bad) {
            if (err) atomicOr(err, BSATTN_FLAG_BAD_SEQLENS);
            return t;
        }
    }
    t.nvalid = sq - t.m * kTile;
    if (t.nvalid > kTile) t.nvalid = kTile;
    if (t.nvalid <= 0) return t;
    t.valid = 1;
    return t;
}

// Bits [lo, hi) of a 32-bit word (positions relative to the word; clamped).
__device__ __forceinline__ uint32_t span_bits(int lo, int hi) {
    lo = lo < 0 ? 0 : lo;
    hi = hi > 32 ? 32 : hi;
    if (hi <= lo) return 0u;
    const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
    return below_hi & ~((1u << lo) - 1u);
}

// A list cursor whose next raw entry is loaded one step before it is needed.
struct Cursor {
    const int32_t *ptr;
    int cnt, pos, head, pre;
};

__device__ __forceinline__ void cur_advance(Cursor &c, int nn, int32_t *err) {
    while (true) {
        ++c.pos;
        if (c.pos >= c.cnt) {
            c.head = -1;
            return;
        }
        c.head = c.pre;
        c.pre = (c.pos + 1 < c.cnt) ? __ldg(c.ptr + c.pos + 1) : -1;
        if (c.head >= 0 && c.head < nn) return;
        if (err) atomicOr(err, BSATTN_FLAG_BAD_INDEX);
    }
}

// Starts a cursor on a list whose count and first two entries were read ahead
// (e1 is only used when the list has two entries).
__device__ __forceinline__ void cur_init(Cursor &c, const int32_t *ptr, int cnt, int e0, int e1,
                                         int nn, int32_t *err) {
    if (cnt < 0 || cnt > nn) {
        if (err) atomicOr(err, BSATTN_FLAG_BAD_COUNT);
        cnt = cnt < 0 ? 0 : nn;
    }
    c.ptr = ptr;
    c.cnt = cnt;
    c.pos = 0;
    if (cnt == 0) {
        c.head = -1;
        return;
    }
    c.head = e0;
    c.pre = cnt > 1 ? e1 : -1;
    if (c.head >= 0 && c.head < nn) return;
    if (err) atomicOr(err, BSATTN_FLAG_BAD_INDEX);
    cur_advance(c, nn, err);
}

// Softmax, O rescale and epilogue of one tile slot t (warps 4-7: t = 0, 8-11:
// t = 1).  Events come from the slot's S-ready barrier (bar_sr) with the item's
// description in *sinfo_t; P is published in two halves (bar_pr, bar_pr + 8);
// bar_ed acknowledges an end of unit.  The unit of each end-to-end run of events
// is read from unit_ring_t (a unit is a pair of consecutive Q tiles).
template <int D, bool kProxy, bool kPolled>
__device__ __forceinline__ void softmax_role(const FwdParams &p, const uint32_t tmem, const int t,
                                             const uint32_t warp, const uint32_t lane,
                                             const uint32_t bar_sr, const uint32_t bar_pr,
                                             const uint32_t bar_ed, const SInfo *sinfo_t,
                                             const int32_t *unit_ring_t, uint8_t *epi,
                                             volatile int *abort_flag) {
    using C = Cfg<D>;
    const uint32_t quarter = warp & 3u;
    const int r = (int)(quarter * 32 + lane);                 // row of the tile
    const uint32_t lane_addr = tmem + ((quarter * 32u) << 16);
    const uint32_t s_col = (uint32_t)t * 128u;
    const uint32_t o_col = 256u + (uint32_t)t * D;
    const float sl2 = p.scale_log2;
    uint32_t scount = 0, ucs = 0;
    bool ok = true;
    SInfo si;
    // Next event (S tile, end of unit, or stop) for this tile.
    auto wait_s = [&]() -> bool {
        bool w = mbar_wait_lim<kPolled>(bar_sr, scount & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT, p.wait_limit);
        w = __all_sync(0xffffffffu, w);
        if (!w) return false;
        ++scount;
        tc_fence_after();
        const volatile SInfo *vs = sinfo_t;
        si.n = vs->n;
        si.flags = vs->flags;
        si.lim = vs->lim;
        return true;
    };
    while (ok) {
        if (!(ok = wait_s())) break;
        if (si.flags & kSStop) break;
        // The producer wrote this unit's id before the events that led here.
        const int u = *reinterpret_cast<const volatile int32_t *>(&unit_ring_t[ucs % kUnitRing]);
        const int h = u / p.pairs_per_head;
        const TileInfo ti = tile_info(p, h, 2 * (u - h * p.pairs_per_head) + t);
        const int i_seq = ti.m * kTile + r;  // sequence-local query position
        float m_run = -INFINITY, l_run = 0.f;
        int j = 0;
        while (true) {
            if (si.flags & kSEnd) {
                // Acknowledge the end of the unit: the MMA warp may signal again.
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_ed);
                break;
            }
            float s[128];
            // Summary items: the sequence's last KV tile, if partial, counts with
            // its true number of keys; its score column is read on its own (P
            // overwrites the first half of the S columns).
            const bool summary = kProxy && (si.flags & kSSummary) != 0;
            int c_tail = -1;
            if (summary && p.proxy_tail < kTile) {
                const int ct = (p.num_n - 1) - si.n * kTile;
                if (ct >= 0 && ct < kTile) c_tail = ct;
            }
            uint32_t s_tail_bits = 0u;
            float hm0, hm1, hm2, hm3;  // maxima of the four 32-column groups, as loaded
            {
                uint32_t v0[32], v1[32], v2[32], v3[32];
                tmem_ld32_max(lane_addr + s_col + 0, v0, hm0);
                tmem_ld32_max(lane_addr + s_col + 32, v1, hm1);
                tmem_ld32_max(lane_addr + s_col + 64, v2, hm2);
                tmem_ld32_max(lane_addr + s_col + 96, v3, hm3);
                if (c_tail >= 0) tmem_ld1(lane_addr + s_col + (uint32_t)c_tail, s_tail_bits);
                tmem_wait_ld();
                reg_fence(v0);
                reg_fence(v1);
                reg_fence(v2);
                reg_fence(v3);
                reg_fence(hm0);
                reg_fence(hm1);
                reg_fence(hm2);
                reg_fence(hm3);
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    s[x] = __uint_as_float(v0[x]);
                    s[32 + x] = __uint_as_float(v1[x]);
                    s[64 + x] = __uint_as_float(v2[x]);
                    s[96 + x] = __uint_as_float(v3[x]);
                }
            }
            bool tail_kept = false;
            const bool masked = (si.flags & (kSMask | kSBound | (kProxy ? kSSummary : 0u))) != 0;
            if (masked) {
                // Keep-mask of the 128 columns as four 32-bit words; columns at or
                // past si.lim (sequence end, valid length) are always dropped.
                const int j0 = si.n * kTile;
                const int lim = si.lim;
                uint32_t keep[4];
                if (summary) {
                    // keep the summary columns whose tile is not computed exactly
                    const uint32_t *sw = p.sel_words + ti.cnt_at * p.sel_words_per_row;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int wi = 4 * si.n + w;
                        const uint32_t sel = wi < p.sel_words_per_row ? __ldg(sw + wi) : 0u;
                        keep[w] = ~sel & span_bits(0, lim - 32 * w);
                    }
                    if (c_tail >= 0) {
                        const uint32_t kw = (c_tail >> 5) == 0 ? keep[0]
                                          : (c_tail >> 5) == 1 ? keep[1]
                                          : (c_tail >> 5) == 2 ? keep[2] : keep[3];
                        tail_kept = (kw >> (c_tail & 31)) & 1u;
                    }
                } else if (!(si.flags & kSMask) || p.kind == BSATTN_MASK_NONE) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) keep[w] = span_bits(0, lim - 32 * w);
                } else if (p.kind == BSATTN_MASK_DOCUMENT) {
                    const int32_t dq = __ldg(p.doc_q + ti.qrow0 + min(r, ti.nvalid - 1));
                    const int32_t *dk = p.doc_k + (long long)ti.krow0 + j0;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t bits = 0;
#pragma unroll 1
                        for (int x = 0; x < 32; ++x) {
                            const int c = 32 * w + x;
                            if (c < lim && __ldg(dk + c) == dq) bits |= 1u << x;
                        }
                        keep[w] = bits;
                    }
                } else {
                    const int diag = i_seq - j0 + 1;  // columns c < diag have j <= i
                    int la = 0, ha = lim, hb = 0;
                    if (p.kind == BSATTN_MASK_CAUSAL) {
                        ha = min(lim, diag);
                    } else if (p.kind == BSATTN_MASK_SLIDING_WINDOW) {
                        la = diag <= p.window_left ? 0 : diag - p.window_left;
                        ha = min(lim, diag);
                        hb = min(ha, p.sink_tokens - j0);
                    } else if (p.kind == BSATTN_MASK_PREFIX) {
                        ha = min(lim, max(p.prefix_len - j0, diag));
                    }
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        keep[w] = span_bits(la - 32 * w, ha - 32 * w) | span_bits(0, hb - 32 * w);
                }
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    if (keep[w] == 0xffffffffu) continue;
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (!((keep[w] >> x) & 1u)) s[32 * w + x] = -INFINITY;
                    // this group's maximum over its kept scores (the load's covers all 32)
                    float g = fmax3(s[32 * w], s[32 * w + 1], s[32 * w + 2]);
#pragma unroll
                    for (int x = 3; x < 31; x += 2) g = fmax3(g, s[32 * w + x], s[32 * w + x + 1]);
                    g = fmaxf(g, s[32 * w + 31]);
                    if (w == 0) hm0 = g;
                    else if (w == 1) hm1 = g;
                    else if (w == 2) hm2 = g;
                    else hm3 = g;
                }
            }
            const float m_new = fmaxf(m_run, fmax3(hm0, hm1, fmaxf(hm2, hm3)) * sl2);
            // Rescale O only when some row's running maximum grew by more than 2^8;
            // otherwise keep the stale maximum (O / l at the end is the same).
            const bool rescale = (j > 0) && __any_sync(0xffffffffu, (m_new - m_run) > 8.0f);
            float alpha = 1.f;
            if (j == 0 || rescale) {
                if (rescale && m_new != -INFINITY) alpha = ex2_approx(m_run - m_new);
                m_run = m_new;
            }
            const float nm = (m_run == -INFINITY) ? 0.f : -m_run;
            float la0 = 0.f, la1 = 0.f, lb0 = 0.f, lb1 = 0.f;
            auto p_half = [&](int c) {
                uint32_t pk[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    float x0, x1;
                    ffma2(x0, x1, s[c * 64 + 2 * x], s[c * 64 + 2 * x + 1], sl2, sl2, nm, nm);
                    const float p0 = ex2_approx(x0);
                    const float p1 = ex2_approx(x1);
                    if (x & 1) fadd2(lb0, lb1, lb0, lb1, p0, p1);
                    else fadd2(la0, la1, la0, la1, p0, p1);
                    pk[x] = pack_bf16x2(p0, p1);
                }
                tmem_st32(lane_addr + s_col + c * 32, pk);
            };
            // Publish P to the MMA warp in two halves (keys 0-63, then 64-127).
            auto publish = [&](int half) {
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pr + 8u * (uint32_t)half);
            };
            p_half(0);
            if (rescale) {
                // S_t of this item was issued after the previous item's P.V, so
                // its completion (observed above) means O_t is up to date.
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(lane_addr + o_col + c * 32, v);
                    tmem_wait_ld();
                    reg_fence(v);
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        v[x] = __float_as_uint(__uint_as_float(v[x]) * alpha);
                    tmem_st32(lane_addr + o_col + c * 32, v);
                }
            }
            publish(0);
            p_half(1);
            publish(1);
            const float l0 = la0 + lb0, l1 = la1 + lb1;
            float l_item = l0 + l1;
            if (summary) {
                // a summary column stands for the 128 keys of its tile (the tail
                // tile for proxy_tail keys)
                l_item *= (float)kTile;
                if (tail_kept) {
                    const float pt = ex2_approx(fmaf(__uint_as_float(s_tail_bits), sl2, nm));
                    l_item += (float)(p.proxy_tail - kTile) * pt;
                }
            }
            l_run = l_run * alpha + l_item;
            ++j;
            if (!(ok = wait_s())) break;
        }
        if (!ok) break;
        // Epilogue: O / l and LSE = ln(sum of exp(scale * s)).  Each lane holds one
        // row of 128-byte blocks (64 columns in bf16, 32 in fp32).  A block goes
        // through the warp's shared-memory scratch (16-byte pieces placed at
        // piece ^ (row & 7), so that neither side conflicts on banks) and comes
        // back with lane 8g + j holding piece j of rows 8g..8g+7: every store
        // instruction then writes 4 whole 128-byte row segments.
        const bool row_ok = ti.valid && r < ti.nvalid;
        const bool empty = (j == 0) || !(l_run > 0.f);
        const float inv = empty ? 0.f : 1.f / l_run;
        const int gl = (int)(lane & 7u);
        const int row0 = (int)(quarter * 32u) + 8 * (int)(lane >> 3);  // first row this lane stores
        const int nrows = ti.valid ? min(max(ti.nvalid - row0, 0), 8) : 0;
        // The lane number is re-read here (opaque to the compiler) so that the
        // scratch addresses below are formed in the epilogue instead of being
        // hoisted out of the unit loop and held in registers through it.
        uint32_t ln;
        asm volatile("mov.u32 %0, %%laneid;" : "=r"(ln));
        uint4 *scr = reinterpret_cast<uint4 *>(epi + (warp - 4u) * 4096u);
        // Writes this lane's block (row = lane) and reads back the 8 pieces it stores.
        auto exchange = [&](uint32_t (&w)[32]) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                scr[ln * 8u + ((uint32_t)i ^ (ln & 7u))] =
                    make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint4 x = scr[(ln >> 3) * 64u + (uint32_t)k * 8u + ((ln & 7u) ^ (uint32_t)k)];
                w[4 * k] = x.x;
                w[4 * k + 1] = x.y;
                w[4 * k + 2] = x.z;
                w[4 * k + 3] = x.w;
            }
            __syncwarp();
        };
        const long long row_step = (long long)p.H * D;             // elements between rows
        const long long out0 = ((long long)(ti.qrow0 + row0) * p.H + h) * D;
        if (p.out_f32) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t w[32];
                if (j > 0) {
                    tmem_ld32(lane_addr + o_col + c * 32, w);
                    tmem_wait_ld();
                    reg_fence(w);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) w[x] = 0u;
                }
#pragma unroll
                for (int x = 0; x < 32; ++x) w[x] = __float_as_uint(__uint_as_float(w[x]) * inv);
                exchange(w);
                float *dst = static_cast<float *>(p.out) + out0 + c * 32 + 4 * gl;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (k < nrows)
                        *reinterpret_cast<uint4 *>(dst + k * row_step) =
                            make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t w[32];
                if (j > 0) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t v[32];
                        tmem_ld32(lane_addr + o_col + c * 64 + hf * 32, v);
                        tmem_wait_ld();
                        reg_fence(v);
#pragma unroll
                        for (int x = 0; x < 16; ++x)
                            w[16 * hf + x] = pack_bf16x2(__uint_as_float(v[2 * x]) * inv,
                                                         __uint_as_float(v[2 * x + 1]) * inv);
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) w[x] = 0u;
                }
                exchange(w);
                uint16_t *dst = static_cast<uint16_t *>(p.out) + out0 + c * 64 + 8 * gl;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (k < nrows)
                        *reinterpret_cast<uint4 *>(dst + k * row_step) =
                            make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            }
        }
        if (row_ok) {
            const float lse = empty ? -INFINITY : (m_run * 0.69314718055994530942f + logf(l_run));
            const long long li = p.varlen
                                     ? (long long)h * p.lse_row_stride + ti.qrow0 + r
                                     : ((long long)ti.b * p.H + h) * p.lse_row_stride +
                                           (long long)ti.m * kTile + r;
            p.lse[li] = lse;
        }
        tc_fence_before();
        ++ucs;
    }
}

// kProxy: proxy-compensation build (summary items after each unit); the exact
// build carries none of that code.  kPolled: pipeline waits poll without
// suspending and give up after p.wait_limit cycles (the build a lowered wait
// limit runs; the waits of the default build use their fixed one-second limit).
// kBlocks: lists per sparse block of two Q tiles (one list row per unit), each
// entry covering p.list_kv_tiles KV tiles; the per-tile builds carry none of it.
template <int D, bool kProxy, bool kPolled, bool kBlocks>
__global__ void __launch_bounds__(kThreads, 1)
    bsattn_fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const __grid_constant__ CUtensorMap tks,
                      const __grid_constant__ CUtensorMap tvs) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    Item *items = reinterpret_cast<Item *>(gbase + C::kItems);
    SInfo *sinfo = reinterpret_cast<SInfo *>(gbase + C::kSInfo);
    int32_t *unit_ring = reinterpret_cast<int32_t *>(gbase + C::kUnits);
    UnitDesc *udesc = reinterpret_cast<UnitDesc *>(gbase + C::kUDesc);
    uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + C::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    auto bar = [&](int i) -> uint32_t { return base + C::kBar + 8u * (uint32_t)i; };
    const uint32_t sQ = base + C::kQ, sK = base + C::kK, sV = base + C::kV;

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStagesK; ++s) {
            mbar_init(bar(C::bKF + s), 1);
            mbar_init(bar(C::bKE + s), 1);
        }
        for (int s = 0; s < C::kStagesV; ++s) mbar_init(bar(C::bVE + s), 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::bQF + t), 1);
            mbar_init(bar(C::bQE + t), 1);
            mbar_init(bar(C::bSR + t), 2);
            mbar_init(bar(C::bPR + 2 * t), 4);      // first half of P_t: one arrival per warp
            mbar_init(bar(C::bPR + 2 * t + 1), 4);  // second half
            mbar_init(bar(C::bED + t), 4);          // softmax t has seen the end of a unit
        }
        for (int s = 0; s < kUnitDescs; ++s) {
            mbar_init(bar(C::bUF + s), 1);  // unit descriptor written (scheduler warp)
            mbar_init(bar(C::bUE + s), 1);  // unit descriptor taken (producer)
        }
        mbar_init(bar(C::bDrain), 1);
        misc[1] = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 2) {
        tmem_alloc(base + C::kMisc, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // Launched as a dependent of the scheduling pass (or of whatever preceded it
    // on the stream): nothing global is read or written before this point.
    grid_dependency_wait();

    if (warp == 0) {
        regs_release<kCtrlRegs>();
        // ------------------------------------------------------- producer --
        // The whole warp runs the producer's control flow in step (list reads are
        // broadcast loads); lane 0 alone arms the barriers and issues the copies.
        const uint32_t lead = lane == 0 ? 1u : 0u;
        {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            // kc / vc count every use of a K / V stage (TMA arm or end marker); qn
            // counts the uses of each Q stage.  The drain below derives from them the
            // last phase of every full barrier.
            uint32_t kc = 0, vc = 0, uc = 0, qn0 = 0, qn1 = 0;
            for (uint32_t un = 0;; ++un) {
                // The next unit, prepared by the scheduler warp.
                const uint32_t slot = un % kUnitDescs;
                if (!mbar_wait_lim<kPolled>(bar(C::bUF + slot), (un / kUnitDescs) & 1, abort_flag, p.err,
                               BSATTN_FLAG_TIMEOUT, p.wait_limit))
                    goto producer_done;
                const UnitDesc d = udesc[slot];
                mbar_arrive_lead(lead, bar(C::bUE + slot));
                const int u = d.u;
                if (u < 0) break;
                unit_ring[uc % kUnitRing] = u;
                const int h = u / p.pairs_per_head;
                const TileInfo ti[2] = {d.ti[0], d.ti[1]};
                for (int t = 0; t < 2; ++t) {
                    if (!mbar_wait_lim<kPolled>(bar(C::bQE + t), (uc & 1) ^ 1, abort_flag, p.err,
                                   BSATTN_FLAG_TIMEOUT, p.wait_limit))
                        goto producer_done;
                    if (ti[t].valid) {
                        mbar_arrive_expect_tx_lead(lead, bar(C::bQF + t), C::kTileBytes);
                        for (int x = 0; x < C::kSub; ++x)
                            tma_load_3d_lead(lead, sQ + t * C::kTileBytes + x * kSubTileBytes, &tq,
                                        bar(C::bQF + t), x * 64, h, ti[t].qrow0);
                    } else {
                        mbar_arrive_lead(lead, bar(C::bQF + t));
                    }
                    if (t == 0) ++qn0;
                    else ++qn1;
                }
                Cursor cm[2], cf[2];
                // With lists per sparse Q block the unit is one block: its two Q
                // tiles walk the block's one list, each entry's KV tiles in turn.
                constexpr bool block_lists = kBlocks;
                for (int t = 0; t < 2; ++t) {
                    if (block_lists) {
                        const long long idx_at =
                            (((long long)ti[0].b * p.H + h) * p.list_m + (ti[0].m >> 1)) * p.list_n;
                        if (t == 0 && ti[0].valid) {
                            cur_init(cm[0], p.mask_idx + idx_at, d.cnt[0], d.e0[0], d.e1[0], p.list_n, p.err);
                            cur_init(cf[0], p.full_idx + idx_at, d.cnt[1], d.e0[1], d.e1[1], p.list_n, p.err);
                        } else {
                            cm[t].head = cf[t].head = -1;
                            cm[t].cnt = cf[t].cnt = 0;
                            cm[t].pos = cf[t].pos = 0;
                        }
                    } else if (ti[t].valid) {
                        cur_init(cm[t], p.mask_idx + ti[t].idx_at, d.cnt[2 * t], d.e0[2 * t],
                                 d.e1[2 * t], ti[t].nn, p.err);
                        cur_init(cf[t], p.full_idx + ti[t].idx_at, d.cnt[2 * t + 1], d.e0[2 * t + 1],
                                 d.e1[2 * t + 1], ti[t].nn, p.err);
                    } else {
                        cm[t].head = cf[t].head = -1;
                        cm[t].cnt = cf[t].cnt = 0;
                        cm[t].pos = cf[t].pos = 0;
                    }
                }
                while (block_lists) {
                    // next entry of the block's lists: KV block c, its tiles from the
                    // top down as dual items (both Q tiles share the block's list)
                    const int c = max(cm[0].head, cf[0].head);
                    if (c < 0) break;
                    const bool mblk = cm[0].head == c;
                    const int kvt = p.list_kv_tiles;
                    int vlb = kvt * kTile;  // valid keys of the block (mask blocks only)
                    if (mblk) {
                        if (p.vl)
                            vlb = cm[0].pos == 0 ? d.vl[0] : __ldg(p.vl + (long long)ti[0].b * p.vl_stride + c);
                        cur_advance(cm[0], p.list_n, p.err);
                    } else {
                        cur_advance(cf[0], p.list_n, p.err);
                    }
                    const bool list_done = max(cm[0].head, cf[0].head) < 0;
                    // keys of tile c * kvt + j that may be kept: the sequence end, and on
                    // a mask block the valid length, tile j of the block keeping
                    // clamp(v - 128 j, 0, 128) of the block's v valid keys
                    const int n_lo = c * kvt;
                    int lim[2];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int n = n_lo + j;
                        int l = (j < kvt && n < ti[0].nn) ? min(kTile, ti[0].sk - n * kTile) : 0;
                        if (mblk) l = min(l, max(0, min(kTile, vlb - j * kTile)));
                        lim[j] = l;
                    }
#pragma unroll
                    for (int j = 1; j >= 0; --j) {
                        if (lim[j] <= 0) continue;  // no key of this tile is kept
                        const int n = n_lo + j;
                        const uint32_t both = ti[1].valid ? 3u : 1u;  // kPart1 = 2 kPart0
                        Item it;
                        it.krow = ti[0].krow0 + n * kTile;
                        it.n0 = n;
                        it.n1 = ti[1].valid ? n : -1;
                        it.flags = both;  // kPart0 | kPart1
                        // mask_mod runs on mask blocks; without one, a tile whose keys
                        // are all valid needs no mask at all
                        if (mblk && !(p.kind == BSATTN_MASK_NONE && lim[j] == kTile)) it.flags |= both * kMask0;
                        if ((n + 1) * kTile > ti[0].sk) it.flags |= both * kBound0;
                        if (list_done && (j == 0 || lim[0] <= 0)) it.flags |= both * kLast0;
                        it.lim0 = it.lim1 = lim[j];
                        it.pad0 = it.pad1 = 0;
                        const uint32_t ks = kc % C::kStagesK;
                        if (!mbar_wait_lim<kPolled>(bar(C::bKE + ks), ((kc / C::kStagesK) & 1) ^ 1, abort_flag,
                                                    p.err, BSATTN_FLAG_TIMEOUT, p.wait_limit))
                            goto producer_done;
                        items[ks] = it;
                        mbar_arrive_expect_tx_lead(lead, bar(C::bKF + ks), 2 * C::kTileBytes);
                        for (int x = 0; x < C::kSub; ++x)
                            tma_load_3d_lead(lead, sK + ks * C::kTileBytes + x * kSubTileBytes, &tk,
                                             bar(C::bKF + ks), x * 64, h, it.krow);
                        ++kc;
                        const uint32_t vs = vc % C::kStagesV;
                        if (!mbar_wait_lim<kPolled>(bar(C::bVE + vs), ((vc / C::kStagesV) & 1) ^ 1, abort_flag,
                                                    p.err, BSATTN_FLAG_TIMEOUT, p.wait_limit)) {
                            mbar_complete_tx_lead(lead, bar(C::bKF + ks), C::kTileBytes);
                            goto producer_done;
                        }
                        for (int x = 0; x < C::kSub; ++x)
                            tma_load_3d_lead(lead, sV + vs * C::kTileBytes + x * kSubTileBytes, &tv,
                                             bar(C::bKF + ks), x * 64, h, it.krow);
                        ++vc;
                    }
                }
                while (!block_lists) {
                    const int c0 = max(cm[0].head, cf[0].head);
                    const int c1 = max(cm[1].head, cf[1].head);
                    if (c0 < 0 && c1 < 0) break;
                    const long long g0 = c0 >= 0 ? (long long)ti[0].krow0 + (long long)c0 * kTile : -1;
                    const long long g1 = c1 >= 0 ? (long long)ti[1].krow0 + (long long)c1 * kTile : -1;
                    const bool p0 = c0 >= 0 && g0 >= g1;
                    const bool p1 = c1 >= 0 && g1 >= g0;
                    Item it;
                    it.krow = (int32_t)(p0 ? g0 : g1);
                    it.n0 = p0 ? c0 : -1;
                    it.n1 = p1 ? c1 : -1;
                    it.flags = 0;
                    it.lim0 = it.lim1 = kTile;
                    it.pad0 = it.pad1 = 0;
                    int vl0 = kTile, vl1 = kTile;  // valid lengths, loaded before the stage wait
                    if (p0) {
                        it.flags |= kPart0;
                        if (cm[0].head == c0) {
                            it.flags |= kMask0;
                            if (p.vl)
                                vl0 = cm[0].pos == 0 ? d.vl[0]
                                                     : __ldg(p.vl + (long long)ti[0].b * p.vl_stride + c0);
                            cur_advance(cm[0], ti[0].nn, p.err);
                        } else {
                            cur_advance(cf[0], ti[0].nn, p.err);
                        }
                        if ((c0 + 1) * kTile > ti[0].sk) it.flags |= kBound0;
                    }
                    if (p1) {
                        it.flags |= kPart1;
                        if (cm[1].head == c1) {
                            it.flags |= kMask1;
                            if (p.vl)
                                vl1 = cm[1].pos == 0 ? d.vl[1]
                                                     : __ldg(p.vl + (long long)ti[1].b * p.vl_stride + c1);
                            cur_advance(cm[1], ti[1].nn, p.err);
                        } else {
                            cur_advance(cf[1], ti[1].nn, p.err);
                        }
                        if ((c1 + 1) * kTile > ti[1].sk) it.flags |= kBound1;
                    }
                    // A tile whose lists are now exhausted is done with its Q tile after
                    // this item's S: the MMA warp releases that Q buffer early.
                    // (with proxy compensation the tile's last item is a summary item)
                    if (!kProxy && p0 && max(cm[0].head, cf[0].head) < 0) it.flags |= kLast0;
                    if (!kProxy && p1 && max(cm[1].head, cf[1].head) < 0) it.flags |= kLast1;
                    const uint32_t ks = kc % C::kStagesK;
                    if (!mbar_wait_lim<kPolled>(bar(C::bKE + ks), ((kc / C::kStagesK) & 1) ^ 1, abort_flag, p.err,
                                   BSATTN_FLAG_TIMEOUT, p.wait_limit))
                        goto producer_done;
                    if (p0) it.lim0 = min(min(kTile, ti[0].sk - c0 * kTile), vl0);
                    if (p1) it.lim1 = min(min(kTile, ti[1].sk - c1 * kTile), vl1);
                    items[ks] = it;
                    // K and V of the item complete one barrier (V lands in its own ring).
                    mbar_arrive_expect_tx_lead(lead, bar(C::bKF + ks), 2 * C::kTileBytes);
                    for (int x = 0; x < C::kSub; ++x)
                        tma_load_3d_lead(lead, sK + ks * C::kTileBytes + x * kSubTileBytes, &tk, bar(C::bKF + ks),
                                    x * 64, h, it.krow);
                    ++kc;
                    const uint32_t vs = vc % C::kStagesV;
                    if (!mbar_wait_lim<kPolled>(bar(C::bVE + vs), ((vc / C::kStagesV) & 1) ^ 1, abort_flag, p.err,
                                   BSATTN_FLAG_TIMEOUT, p.wait_limit)) {
                        // V is not loaded: the K-stage barrier stops expecting its bytes,
                        // so that the drain below sees the phase complete with K.
                        mbar_complete_tx_lead(lead, bar(C::bKF + ks), C::kTileBytes);
                        goto producer_done;
                    }
                    for (int x = 0; x < C::kSub; ++x)
                        tma_load_3d_lead(lead, sV + vs * C::kTileBytes + x * kSubTileBytes, &tv, bar(C::bKF + ks),
                                    x * 64, h, it.krow);
                    ++vc;
                }
                if constexpr (kProxy) {
                    // Summary items: every chunk of 128 KV-tile summaries of each tile's
                    // sequence (row b * num_n + 128 c of the summary tensors), from the
                    // last chunk down; two tiles of one sequence share each chunk.
                    const int nc = (p.num_n + kTile - 1) / kTile;
                    int sc0 = ti[0].valid ? nc - 1 : -1, sc1 = ti[1].valid ? nc - 1 : -1;
                    while (sc0 >= 0 || sc1 >= 0) {
                        const long long g0 = sc0 >= 0 ? (long long)ti[0].b * p.num_n + (long long)sc0 * kTile : -1;
                        const long long g1 = sc1 >= 0 ? (long long)ti[1].b * p.num_n + (long long)sc1 * kTile : -1;
                        const bool p0 = sc0 >= 0 && g0 >= g1, p1 = sc1 >= 0 && g1 >= g0;
                        Item it;
                        it.krow = (int32_t)(p0 ? g0 : g1);
                        it.n0 = p0 ? sc0 : -1;
                        it.n1 = p1 ? sc1 : -1;
                        it.flags = kSummary | (p0 ? kPart0 : 0u) | (p1 ? kPart1 : 0u);
                        it.lim0 = p0 ? min(kTile, p.num_n - sc0 * kTile) : kTile;
                        it.lim1 = p1 ? min(kTile, p.num_n - sc1 * kTile) : kTile;
                        it.pad0 = it.pad1 = 0;
                        if (p0 && --sc0 < 0) it.flags |= kLast0;
                        if (p1 && --sc1 < 0) it.flags |= kLast1;
                        const uint32_t ks = kc % C::kStagesK;
                        if (!mbar_wait_lim<kPolled>(bar(C::bKE + ks), ((kc / C::kStagesK) & 1) ^ 1, abort_flag, p.err,
                                       BSATTN_FLAG_TIMEOUT, p.wait_limit))
                            goto producer_done;
                        items[ks] = it;
                        mbar_arrive_expect_tx_lead(lead, bar(C::bKF + ks), 2 * C::kTileBytes);
                        for (int x = 0; x < C::kSub; ++x)
                            tma_load_3d_lead(lead, sK + ks * C::kTileBytes + x * kSubTileBytes, &tks,
                                             bar(C::bKF + ks), x * 64, h, it.krow);
                        ++kc;
                        const uint32_t vs = vc % C::kStagesV;
                        if (!mbar_wait_lim<kPolled>(bar(C::bVE + vs), ((vc / C::kStagesV) & 1) ^ 1, abort_flag, p.err,
                                       BSATTN_FLAG_TIMEOUT, p.wait_limit)) {
                            mbar_complete_tx_lead(lead, bar(C::bKF + ks), C::kTileBytes);
                            goto producer_done;
                        }
                        for (int x = 0; x < C::kSub; ++x)
                            tma_load_3d_lead(lead, sV + vs * C::kTileBytes + x * kSubTileBytes, &tvs,
                                             bar(C::bKF + ks), x * 64, h, it.krow);
                        ++vc;
                    }
                }
                {
                    const uint32_t ks = kc % C::kStagesK;
                    if (!mbar_wait_lim<kPolled>(bar(C::bKE + ks), ((kc / C::kStagesK) & 1) ^ 1, abort_flag, p.err,
                                   BSATTN_FLAG_TIMEOUT, p.wait_limit))
                        goto producer_done;
                    Item end;
                    end.krow = 0;
                    end.n0 = end.n1 = -1;
                    end.flags = kEnd;
                    end.lim0 = end.lim1 = 0;
                    end.pad0 = end.pad1 = 0;
                    items[ks] = end;
                    mbar_arrive_lead(lead, bar(C::bKF + ks));
                    ++kc;
                }
                ++uc;
            }
            {
                const uint32_t ks = kc % C::kStagesK;
                if (!mbar_wait_lim<kPolled>(bar(C::bKE + ks), ((kc / C::kStagesK) & 1) ^ 1, abort_flag, p.err,
                               BSATTN_FLAG_TIMEOUT, p.wait_limit))
                    goto producer_done;
                Item stop;
                stop.krow = 0;
                stop.n0 = stop.n1 = -1;
                stop.flags = kStop;
                stop.lim0 = stop.lim1 = 0;
                stop.pad0 = stop.pad1 = 0;
                items[ks] = stop;
                mbar_arrive_lead(lead, bar(C::bKF + ks));
                ++kc;
            }
        producer_done:
            // Make sure no TMA write into this CTA's shared memory is still in flight.
            // Stage s was last used by item (kc - 1 - s) / kStages * kStages + s, whose
            // phase is (kc - 1 - s) / kStages; its barrier also counts that item's V tile.
#pragma unroll
            for (uint32_t s = 0; s < (uint32_t)C::kStagesK; ++s)
                if (kc > s) mbar_wait_drain(bar(C::bKF + s), ((kc - 1 - s) / C::kStagesK) & 1u);
            if (qn0 > 0) mbar_wait_drain(bar(C::bQF + 0), (qn0 - 1) & 1u);
            if (qn1 > 0) mbar_wait_drain(bar(C::bQF + 1), (qn1 - 1) & 1u);
        }
    } else if (warp == 1) {
        regs_release<kCtrlRegs>();
        // ---------------------------------------------------- MMA issuer --
        // The whole warp runs the issuer's control flow in step (waits, item reads
        // and bookkeeping are warp-uniform); lane 0 alone issues the MMAs, commits
        // and arrivals, through predicated instructions.
        const uint32_t lead = lane == 0 ? 1u : 0u;
        {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
            // Descriptors are built once; per K step only the 16-byte-unit start
            // address moves (every operand address is below 2^18, so the 14-bit
            // address field never carries into the neighbouring fields).
            const uint64_t desc_q = smem_desc_sw128(sQ, 16, 1024);
            const uint64_t desc_k = smem_desc_sw128(sK, 16, 1024);
            const uint64_t desc_v = smem_desc_sw128(sV, kSubTileBytes, 1024);
            constexpr uint64_t kTileUnits = C::kTileBytes >> 4;
            constexpr uint64_t kSubUnits = kSubTileBytes >> 4;
            uint32_t kc = 0, vc = 0, uc = 0;
            uint32_t pc[2] = {0, 0}, edc[2] = {0, 0};
            bool need_ed[2] = {false, false};
            // per-unit state
            bool have_q[2] = {false, false};
            bool q_released[2] = {false, false};
            bool first_pv[2] = {true, true};
            int pend[2] = {-1, -1};  // V-ring item counter of the tile's pending P.V
            bool ok = true;
            // O_t += P_t V for the tile's pending item.  P_t arrives in two halves of
            // 64 keys, each with its own barrier (one barrier signalled twice per item
            // could run two phases ahead of this wait); the first four K steps go out
            // as soon as the first half is in TMEM.
            auto issue_pv = [&](int t) -> bool {
                // Each softmax warp arrives on the first-half barrier before the second,
                // so a completed second half implies a completed first half: one test
                // then covers both (the common case when the MMA warp runs behind).
                const bool both = mbar_test_wait(bar(C::bPR + 2 * t + 1), pc[t] & 1);
                if (!both &&
                    !mbar_wait_lim<kPolled>(bar(C::bPR + 2 * t), pc[t] & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT, p.wait_limit))
                    return false;
                // The item's V tile landed before its K-stage wait completed.
                const uint32_t vs = (uint32_t)pend[t] % C::kStagesV;
                tc_fence_after();
                const uint64_t vdesc = desc_v + vs * kTileUnits;
                const uint32_t o_tmem = tmem + 256 + t * D, p_tmem = tmem + t * 128;
                const uint32_t acc0 = first_pv[t] ? 0u : 1u;
#pragma unroll
                for (int kk = 0; kk < kTile / 32; ++kk)
                    mma_ts_lead(lead, o_tmem, p_tmem + kk * 8, vdesc + (uint64_t)(kk * (2048 >> 4)), idesc_pv,
                           kk > 0 ? 1u : acc0);
                if (!both && !mbar_wait_lim<kPolled>(bar(C::bPR + 2 * t + 1), pc[t] & 1, abort_flag, p.err,
                                        BSATTN_FLAG_TIMEOUT, p.wait_limit))
                    return false;
                ++pc[t];
                tc_fence_after();
#pragma unroll
                for (int kk = kTile / 32; kk < kTile / 16; ++kk)
                    mma_ts_lead(lead, o_tmem, p_tmem + kk * 8, vdesc + (uint64_t)(kk * (2048 >> 4)), idesc_pv, 1u);
                first_pv[t] = false;
                if (pend[1 - t] != pend[t]) mma_commit_lead(lead, bar(C::bVE + vs));
                pend[t] = -1;
                return true;
            };
            // Publishes sinfo[t] and signals tile t's S-ready barrier.  After an end
            // of unit, the softmax must first acknowledge that end: the barrier could
            // otherwise complete two phases before the softmax waits on it.
            auto signal_s = [&](int t, int32_t n, int32_t lim, uint32_t fl) -> bool {
                if (need_ed[t]) {
                    if (!mbar_wait_lim<kPolled>(bar(C::bED + t), edc[t] & 1, abort_flag, p.err, BSATTN_FLAG_TIMEOUT, p.wait_limit))
                        return false;
                    ++edc[t];
                    need_ed[t] = false;
                }
                sinfo[t].n = n;
                sinfo[t].lim = lim;
                sinfo[t].flags = fl;
                mma_commit_lead(lead, bar(C::bSR + t));
                mbar_arrive_lead(lead, bar(C::bSR + t));
                return true;
            };
            while (ok) {
                const uint32_t ks = kc % C::kStagesK;
                if (!(ok = mbar_wait_lim<kPolled>(bar(C::bKF + ks), (kc / C::kStagesK) & 1, abort_flag, p.err,
                                     BSATTN_FLAG_TIMEOUT, p.wait_limit)))
                    break;
                Item it;
                {
                    const volatile Item *vi = &items[ks];
                    it.krow = vi->krow;
                    it.n0 = vi->n0;
                    it.n1 = vi->n1;
                    it.flags = vi->flags;
                    it.lim0 = vi->lim0;
                    it.lim1 = vi->lim1;
                }
                if (it.flags & kStop) {
                    
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (ok) ok = signal_s(t, -1, 0, kSStop);
                    ++kc;
                    break;
                }
                if (it.flags & kEnd) {
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (ok && pend[t] >= 0) ok = issue_pv(t);
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (ok && !have_q[t])
                            ok = mbar_wait_lim<kPolled>(bar(C::bQF + t), uc & 1, abort_flag, p.err,
                                           BSATTN_FLAG_TIMEOUT, p.wait_limit);
                    if (!ok) break;
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (!q_released[t]) mma_commit_lead(lead, bar(C::bQE + t));
                    mbar_arrive_lead(lead, bar(C::bKE + ks));
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (ok) ok = signal_s(t, -1, 0, kSEnd);
                        need_ed[t] = true;
                    }
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        have_q[t] = q_released[t] = false;
                        first_pv[t] = true;
                        pend[t] = -1;
                    }
                    ++uc;
                    ++kc;
                    continue;
                }
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!ok) break;
                    if (!(it.flags & (t ? kPart1 : kPart0))) continue;
                    if (pend[t] >= 0 && !(ok = issue_pv(t))) break;
                    if (!have_q[t]) {
                        if (!(ok = mbar_wait_lim<kPolled>(bar(C::bQF + t), uc & 1, abort_flag, p.err,
                                             BSATTN_FLAG_TIMEOUT, p.wait_limit)))
                            break;
                        have_q[t] = true;
                        tc_fence_after();
                    }
                    const uint64_t qd = desc_q + t * kTileUnits;
                    const uint64_t kd = desc_k + ks * kTileUnits;
                    const uint32_t s_tmem = tmem + t * 128;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = (uint64_t)((kk >> 2) * kSubUnits + (kk & 3) * 2);
                        mma_ss_lead(lead, s_tmem, qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    const uint32_t sfl = ((it.flags & (t ? kMask1 : kMask0)) ? kSMask : 0u) |
                                         ((it.flags & (t ? kBound1 : kBound0)) ? kSBound : 0u) |
                                         ((it.flags & kSummary) ? kSSummary : 0u);
                    if (!(ok = signal_s(t, t ? it.n1 : it.n0, t ? it.lim1 : it.lim0, sfl))) break;
                    if (it.flags & (t ? kLast1 : kLast0)) {
                        mma_commit_lead(lead, bar(C::bQE + t));  // no further S_t in this unit
                        q_released[t] = true;
                    }
                    pend[t] = (int)vc;
                }
                if (!ok) break;
                // A tile that sits this item out retires its pending P.V now, so a
                // V stage is never held across more than one item.
#pragma unroll
                for (int t = 0; t < 2; ++t)
                    if (ok && !(it.flags & (t ? kPart1 : kPart0)) && pend[t] >= 0) ok = issue_pv(t);
                if (!ok) break;
                mma_commit_lead(lead, bar(C::bKE + ks));
                ++kc;
                ++vc;
            }
            // Wait until every tcgen05 operation issued above has completed.
            mma_commit_lead(lead, bar(C::bDrain));
            mbar_wait_drain(bar(C::bDrain), 0);
        }
    } else if (warp == 3) {
        regs_release<kCtrlRegs>();
        // ------------------------------------------------------ scheduler --
        // Claims units and reads the head of their lists one unit ahead of the
        // producer.  Units come either from a fixed stride over the CTAs, or, with a
        // schedule, from an order array claimed slot by slot through an atomic
        // counter.
        // The whole warp runs in step; lane 0 alone claims (the slot is broadcast)
        // and arrives.
        const uint32_t lead = lane == 0 ? 1u : 0u;
        auto claim_slot = [&]() -> uint32_t {
            uint32_t pos = 0;
            if (lead) pos = atomicAdd(p.sched_counter, 1u);
            return __shfl_sync(0xffffffffu, pos, 0);
        };
        {
            int u;
            if (p.dynamic) {
                const uint32_t pos = claim_slot();
                u = pos < (uint32_t)p.num_units ? __ldg(p.sched_order + pos) : -1;
            } else {
                u = (int)blockIdx.x < p.num_units ? (int)blockIdx.x : -1;
            }
            for (uint32_t n = 0;; ++n) {
                const uint32_t slot = n % kUnitDescs;
                if (!mbar_wait_lim<kPolled>(bar(C::bUE + slot), ((n / kUnitDescs) & 1) ^ 1, abort_flag, p.err,
                               BSATTN_FLAG_TIMEOUT, p.wait_limit))
                    break;
                UnitDesc &d = udesc[slot];
                d.u = u;
                if (u < 0) {
                    mbar_arrive_lead(lead, bar(C::bUF + slot));
                    break;
                }
                const uint32_t claim = p.dynamic ? claim_slot() : 0u;
                const int h = u / p.pairs_per_head;
                const int pr = u - h * p.pairs_per_head;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const TileInfo ti = tile_info(p, h, 2 * pr + t, lead ? p.err : nullptr);
                    d.ti[t] = ti;
                    int cm = 0, cf = 0, m0 = -1, m1 = -1, f0 = -1, f1 = -1, vl = kTile;
                    // the lists of tile t, or, with lists per sparse Q block, the
                    // block's one list (read for tile 0; tile 1 has none of its own)
                    long long cnt_at = ti.cnt_at, idx_at = ti.idx_at;
                    int nn = ti.nn;
                    const bool has_list = ti.valid && (!kBlocks || t == 0);
                    if constexpr (kBlocks) {
                        cnt_at = ((long long)ti.b * p.H + h) * p.list_m + (ti.m >> 1);
                        idx_at = cnt_at * p.list_n;
                        nn = p.list_n;
                    }
                    if (has_list) {
                        cm = __ldg(p.mask_cnt + cnt_at);
                        cf = __ldg(p.full_cnt + cnt_at);
                        m0 = __ldg(p.mask_idx + idx_at);
                        f0 = __ldg(p.full_idx + idx_at);
                        if (nn > 1) {
                            m1 = __ldg(p.mask_idx + idx_at + 1);
                            f1 = __ldg(p.full_idx + idx_at + 1);
                        }
                        if (p.vl && cm > 0 && m0 >= 0 && m0 < nn)
                            vl = __ldg(p.vl + (long long)ti.b * p.vl_stride + m0);
                    }
                    d.cnt[2 * t] = cm;
                    d.cnt[2 * t + 1] = cf;
                    d.e0[2 * t] = m0;
                    d.e0[2 * t + 1] = f0;
                    d.e1[2 * t] = m1;
                    d.e1[2 * t + 1] = f1;
                    d.vl[t] = vl;
                }
                mbar_arrive_lead(lead, bar(C::bUF + slot));
                if (p.dynamic)
                    u = claim < (uint32_t)p.num_units ? __ldg(p.sched_order + claim) : -1;
                else
                    u = (long long)u + gridDim.x < p.num_units ? u + (int)gridDim.x : -1;
            }
        }
    } else if (warp < 4) {
        regs_release<kCtrlRegs>();  // warp 2: idle until the teardown
    } else if (warp >= 4) {
        // ------------------------------------------------------- softmax --
        regs_claim<kSoftmaxRegs>();
        const int t = (warp >= 8) ? 1 : 0;
        softmax_role<D, kProxy, kPolled>(p, tmem, t, warp, lane, bar(C::bSR + t), bar(C::bPR + 2 * t),
                                                bar(C::bED + t), &sinfo[t], unit_ring, gbase + C::kEpi,
                                                abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Work of one Q tile = its listed KV tiles (counts clamped to [0, 2^15)).  With
// lists per sparse Q block the block's list counts for its first tile only.
__device__ __forceinline__ int tile_weight(const FwdParams &p, int h, int T) {
    if (T >= p.total_m) return 0;
    long long at;
    if (p.varlen) {
        at = (long long)h * p.total_m + T;
    } else {
        const int b = T / p.num_m, m = T - b * p.num_m;
        if (p.list_q_tiles == 2) {
            if (m & 1) return 0;
            at = ((long long)b * p.H + h) * p.list_m + (m >> 1);
        } else {
            at = ((long long)b * p.H + h) * p.num_m + m;
        }
    }
    const int w = (max(__ldg(p.full_cnt + at), 0) + max(__ldg(p.mask_cnt + at), 0)) * p.list_kv_tiles;
    return min(w, 32767);
}

// Scheduling pass (one CTA): orders the work units by decreasing work, stable
// (units of equal work keep their head-major order, which keeps one head's K/V
// resident in L2 while the CTAs work on it), and resets the claim counter.
// Heaviest-first claiming is the longest-processing-time rule for list scheduling.
//
// A counting sort over 1024 work keys, split into kSchedChunks contiguous runs
// of units: every run's key histogram, one exclusive scan over (key, run), then
// each warp scatters its own run in unit order.  The attention kernel launched
// after it starts at once and waits for its completion before its first claim.
constexpr int kSchedBuckets = 1024;
constexpr int kSchedThreads = 1024;
constexpr int kSchedChunks = kSchedThreads / 32;  // one run per warp
constexpr size_t kSchedSmemBytes = (size_t)kSchedChunks * kSchedBuckets * sizeof(int);
static_assert(kSchedThreads == kSchedBuckets, "one thread per work key in the scan");

__device__ __forceinline__ int unit_key(const FwdParams &p, int u) {
    const int h = u / p.pairs_per_head, pr = u - h * p.pairs_per_head;
    const int w = tile_weight(p, h, 2 * pr) + tile_weight(p, h, 2 * pr + 1);
    return kSchedBuckets - 1 - min(w, kSchedBuckets - 1);
}

__global__ void __launch_bounds__(kSchedThreads, 1) bsattn_schedule_kernel(const __grid_constant__ FwdParams p) {
    grid_launch_dependents();
    extern __shared__ int run_at[];  // [kSchedChunks][kSchedBuckets]: count, then start
    __shared__ int warp_sum[kSchedChunks];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = p.num_units;
    const int run_len = (n + kSchedChunks - 1) / kSchedChunks;
    for (int i = tid; i < kSchedChunks * kSchedBuckets; i += kSchedThreads) run_at[i] = 0;
    if (tid == 0) *p.sched_counter = 0u;
    __syncthreads();
    for (int u = tid; u < n; u += kSchedThreads)
        atomicAdd(&run_at[(u / run_len) * kSchedBuckets + unit_key(p, u)], 1);
    __syncthreads();
    // Thread k owns key k: its total over the runs, scanned across keys.
    const int k = tid;
    int total = 0;
#pragma unroll 8
    for (int c = 0; c < kSchedChunks; ++c) total += run_at[c * kSchedBuckets + k];
    int incl = total;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = warp_sum[lane];
        int x = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x += o;
        }
        warp_sum[lane] = x - v;
    }
    __syncthreads();
    int at = warp_sum[warp] + incl - total;  // first position of key k
#pragma unroll 8
    for (int c = 0; c < kSchedChunks; ++c) {
        const int v = run_at[c * kSchedBuckets + k];
        run_at[c * kSchedBuckets + k] = at;
        at += v;
    }
    __syncthreads();
    // Warp w scatters run w, 32 units at a time in unit order.
    int *start = run_at + warp * kSchedBuckets;
    const unsigned lt = (1u << lane) - 1u;
    const int u_end = min(n, (warp + 1) * run_len);
    for (int base = warp * run_len; base < u_end; base += 32) {
        const int u = base + lane;
        const int key = u < u_end ? unit_key(p, u) : 0xFFFF;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (u < u_end) p.sched_order[start[key] + __popc(peers & lt)] = u;
        __syncwarp();
        if (u < u_end && lane == __ffs(peers) - 1) start[key] += __popc(peers);
        __syncwarp();
    }
}

cudaError_t prepare_schedule_kernel() {
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set_for_device[dev]) {
        e = cudaFuncSetAttribute(bsattn_schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSchedSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    return cudaSuccess;
}

template <int D, bool kProxy, bool kPolled, bool kBlocks>
cudaError_t prepare_fwd_kernel() {
    using C = Cfg<D>;
    static int attr_set_for_device[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set_for_device[dev]) {
        // The register split inside the kernel assumes exactly kLaunchRegs per
        // thread at launch; refuse to run a build where that does not hold.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, bsattn_fwd_kernel<D, kProxy, kPolled, kBlocks>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(bsattn_fwd_kernel<D, kProxy, kPolled, kBlocks>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_set_for_device[dev] = 1;
    }
    return cudaSuccess;
}

template <int D, bool kProxy, bool kPolled, bool kBlocks>
cudaError_t launch_fwd_kernel(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv, const CUtensorMap &tks, const CUtensorMap &tvs,
                              int grid, cudaStream_t stream) {
    cudaError_t e = prepare_fwd_kernel<D, kProxy, kPolled, kBlocks>();
    if (e != cudaSuccess) return e;
    // After the scheduling pass the kernel is a programmatic dependent: its CTAs
    // set up shared memory and TMEM while the pass runs, then wait for it.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<D>::kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.dynamic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, bsattn_fwd_kernel<D, kProxy, kPolled, kBlocks>, p, tq, tk, tv, tks, tvs);
}

template <int D>
cudaError_t launch_fwd_d(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                         const CUtensorMap &tv, const CUtensorMap &tks, const CUtensorMap &tvs,
                         int num_sms, cudaStream_t stream) {
    if (p.num_units <= 0) return cudaSuccess;
    cudaError_t e;
    if (p.dynamic) {
        e = prepare_schedule_kernel();
        if (e != cudaSuccess) return e;
        bsattn_schedule_kernel<<<1, kSchedThreads, kSchedSmemBytes, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int grid = p.num_units < num_sms ? p.num_units : num_sms;
    // A wait limit below the default (a test lowering it) runs the build whose
    // waits poll against that limit; the proxy build keeps its fixed limit.
    // Lists per sparse block run their own build (with the default limit).
    if (p.proxy) return launch_fwd_kernel<D, true, false, false>(p, tq, tk, tv, tks, tvs, grid, stream);
    if (p.list_q_tiles == 2) return launch_fwd_kernel<D, false, false, true>(p, tq, tk, tv, tks, tvs, grid, stream);
    if (p.wait_limit < kDefaultWaitLimitCycles)
        return launch_fwd_kernel<D, false, true, false>(p, tq, tk, tv, tks, tvs, grid, stream);
    return launch_fwd_kernel<D, false, false, false>(p, tq, tk, tv, tks, tvs, grid, stream);
}

}  // namespace

cudaError_t launch_fwd(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tks, const CUtensorMap &tvs, int D,
                       int num_sms, cudaStream_t stream) {
    if (D == 128) return launch_fwd_d<128>(p, tq, tk, tv, tks, tvs, num_sms, stream);
    if (D == 64) return launch_fwd_d<64>(p, tq, tk, tv, tks, tvs, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace bsattn
