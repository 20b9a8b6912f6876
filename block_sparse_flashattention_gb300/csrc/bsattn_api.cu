// C-ABI entry points: host-side validation, TMA tensor maps, kernel launches.
// Nothing here allocates device memory or synchronises with the device.
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "bsattn_internal.h"

namespace {

using bsattn::kTile;

// Workspace: the claim counter in the first 256 bytes, then the unit order.
constexpr size_t kWorkspaceHeader = 256;

// Pipeline wait limit of the forward launches (0: the default); tests lower it.
std::atomic<long long> g_wait_limit{0};

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bsattn_status check_mask(bsattn_mask_kind kind, const bsattn_mask_params *mp) {
    switch (kind) {
    case BSATTN_MASK_NONE:
    case BSATTN_MASK_CAUSAL:
        return BSATTN_OK;
    case BSATTN_MASK_SLIDING_WINDOW:
        if (!mp || mp->window_left < 0 || mp->sink_tokens < 0) return BSATTN_ERR_INVALID_ARG;
        return BSATTN_OK;
    case BSATTN_MASK_PREFIX:
        if (!mp || mp->prefix_len < 0) return BSATTN_ERR_INVALID_ARG;
        return BSATTN_OK;
    case BSATTN_MASK_DOCUMENT:
        if (!mp || !mp->doc_id_q || !mp->doc_id_k) return BSATTN_ERR_INVALID_ARG;
        return BSATTN_OK;
    default:
        return BSATTN_ERR_INVALID_ARG;
    }
}

// Metadata listed per 128 x 128 tile (every entry point), or, batched only, per
// sparse block of two Q tiles and one or two KV tiles (bsattn_build_meta and the
// forward).
bool per_tile(const bsattn_meta *m) { return m->tile_m == kTile && m->tile_n == kTile; }
bool per_block(const bsattn_meta *m) {
    return !m->varlen && m->tile_m == 2 * kTile && (m->tile_n == kTile || m->tile_n == 2 * kTile);
}

// Work units of the forward: pairs of consecutive Q tiles of a head; with
// metadata per sparse block of two Q tiles, one unit per block.
long long fwd_units(const bsattn_meta *m) {
    if (per_block(m)) return (long long)m->H * m->B * m->num_m;
    const long long total_m = m->varlen ? (long long)m->total_m_blocks : (long long)m->B * m->num_m;
    return (long long)m->H * cdiv(total_m, 2);
}

// Common checks on the metadata descriptor.
bsattn_status check_meta(const bsattn_meta *m) {
    if (!m) return BSATTN_ERR_INVALID_ARG;
    if (!per_tile(m) && !per_block(m)) return BSATTN_ERR_UNSUPPORTED;
    if (m->B <= 0 || m->H <= 0) return BSATTN_ERR_INVALID_ARG;
    if (!m->full_cnt || !m->full_idx || !m->mask_cnt || !m->mask_idx) return BSATTN_ERR_INVALID_ARG;
    if (m->varlen != 0 && m->varlen != 1) return BSATTN_ERR_INVALID_ARG;
    if (m->varlen) {
        if (!m->cu_total_m_blocks || !m->cu_block_idx_offsets) return BSATTN_ERR_INVALID_ARG;
        if (m->total_m_blocks < 0 || m->total_n_blocks < 0 || m->num_n < 0)
            return BSATTN_ERR_INVALID_ARG;
    } else {
        if (m->num_m < 0 || m->num_n < 0) return BSATTN_ERR_INVALID_ARG;
        if ((long long)m->B * m->H * m->num_m > INT32_MAX) return BSATTN_ERR_INVALID_ARG;
    }
    return BSATTN_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [rows, H, D] bf16 tensor; box = 128 rows x 1 head x 64 columns, 128-byte swizzle.
bool encode_bshd(CUtensorMap *map, const void *ptr, long long rows, int H, int D) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kTile};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms_current_device() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

// Validation and launch shared by the three metadata entry points; `p` arrives
// with its selection source set.
bsattn_status build_meta_impl(bsattn::MetaParams p, const int32_t *cu_seqlens_q,
                              const int32_t *cu_seqlens_k, int32_t seqlen_q, int32_t seqlen_k,
                              const int32_t *kv_valid_len, bsattn_mask_kind kind,
                              const bsattn_mask_params *mp, const bsattn_meta *meta,
                              int32_t *err_flag, void *stream) {
    bsattn_status st = check_meta(meta);
    if (st != BSATTN_OK) return st;
    if ((st = check_mask(kind, mp)) != BSATTN_OK) return st;
    p.varlen = meta->varlen;
    p.B = meta->B;
    p.H = meta->H;
    p.num_m = meta->num_m;
    p.num_n = meta->num_n;
    if (meta->varlen) {
        if (!cu_seqlens_q || !cu_seqlens_k) return BSATTN_ERR_INVALID_ARG;
        if (kv_valid_len && meta->num_n <= 0) return BSATTN_ERR_INVALID_ARG;
        p.total_m = meta->total_m_blocks;
        p.total_n = meta->total_n_blocks;
        if ((long long)p.H * p.total_m > INT32_MAX * 8LL) return BSATTN_ERR_INVALID_ARG;
    } else {
        if (cu_seqlens_q || cu_seqlens_k) return BSATTN_ERR_INVALID_ARG;
        if (seqlen_q < 0 || seqlen_k < 0) return BSATTN_ERR_INVALID_ARG;
        if (meta->num_m != cdiv(seqlen_q, meta->tile_m) || meta->num_n != cdiv(seqlen_k, meta->tile_n))
            return BSATTN_ERR_INVALID_ARG;
        if ((long long)meta->B * seqlen_q > INT32_MAX || (long long)meta->B * seqlen_k > INT32_MAX)
            return BSATTN_ERR_INVALID_ARG;
    }
    p.tile_q = meta->tile_m;
    p.tile_k = meta->tile_n;
    p.seqlen_q = seqlen_q;
    p.seqlen_k = seqlen_k;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.cu_tm = meta->cu_total_m_blocks;
    p.cu_off = meta->cu_block_idx_offsets;
    p.vl = kv_valid_len;
    p.vl_stride = p.vl_per_block ? p.block_n : meta->num_n;
    p.kind = (int)kind;
    if (mp) {
        p.window_left = mp->window_left;
        p.sink_tokens = mp->sink_tokens;
        p.prefix_len = mp->prefix_len;
        p.doc_q = mp->doc_id_q;
        p.doc_k = mp->doc_id_k;
    }
    p.full_cnt = meta->full_cnt;
    p.full_idx = meta->full_idx;
    p.mask_cnt = meta->mask_cnt;
    p.mask_idx = meta->mask_idx;
    p.err = err_flag;
    cudaError_t e = bsattn::launch_meta(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

struct ProxyArgs {
    const uint32_t *sel_words;
    int32_t words_per_row;
    const void *k_sum, *v_sum;
};

bsattn_status fwd_impl(const void *q, const void *k, const void *v, int32_t B, int32_t seqlen_q,
                         int32_t seqlen_k, int32_t H, int32_t D, const int32_t *cu_seqlens_q,
                         const int32_t *cu_seqlens_k, const bsattn_meta *meta,
                         const int32_t *kv_valid_len, bsattn_mask_kind kind,
                         const bsattn_mask_params *mp, float softmax_scale, void *out,
                         bsattn_out_dtype out_dtype, float *lse, void *workspace,
                         size_t workspace_bytes, int32_t *err_flag, void *stream,
                      const ProxyArgs *proxy) {
    bsattn_status st = check_meta(meta);
    if (st != BSATTN_OK) return st;
    if ((st = check_mask(kind, mp)) != BSATTN_OK) return st;
    if (!q || !k || !v || !out || !lse) return BSATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return BSATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || seqlen_q < 0 || seqlen_k < 0) return BSATTN_ERR_INVALID_ARG;
    if (meta->B != B || meta->H != H) return BSATTN_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return BSATTN_ERR_INVALID_ARG;
    if (out_dtype != BSATTN_OUT_BF16 && out_dtype != BSATTN_OUT_F32) return BSATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return BSATTN_ERR_UNSUPPORTED;

    bsattn::FwdParams p = {};
    p.varlen = meta->varlen;
    p.B = B;
    p.H = H;
    long long rows_q, rows_k;
    if (meta->varlen) {
        if (!cu_seqlens_q || !cu_seqlens_k) return BSATTN_ERR_INVALID_ARG;
        if (kv_valid_len && meta->num_n <= 0) return BSATTN_ERR_INVALID_ARG;
        rows_q = seqlen_q;
        rows_k = seqlen_k;
        p.total_m = meta->total_m_blocks;
        p.total_n = meta->total_n_blocks;
        p.lse_row_stride = seqlen_q;
    } else {
        if (cu_seqlens_q || cu_seqlens_k) return BSATTN_ERR_INVALID_ARG;
        if (meta->num_m != cdiv(seqlen_q, meta->tile_m) || meta->num_n != cdiv(seqlen_k, meta->tile_n))
            return BSATTN_ERR_INVALID_ARG;
        rows_q = (long long)B * seqlen_q;
        rows_k = (long long)B * seqlen_k;
        p.num_m = (int)cdiv(seqlen_q, kTile);
        p.num_n = (int)cdiv(seqlen_k, kTile);
        // a list row per sparse Q block is one work unit: every block whole
        if (per_block(meta) && (p.num_m & 1)) return BSATTN_ERR_UNSUPPORTED;
        if ((long long)B * p.num_m > INT32_MAX) return BSATTN_ERR_INVALID_ARG;
        p.total_m = B * p.num_m;
        p.lse_row_stride = seqlen_q;
    }
    p.list_q_tiles = meta->tile_m / kTile;
    p.list_kv_tiles = meta->tile_n / kTile;
    p.list_m = meta->num_m;
    p.list_n = meta->num_n;
    if (rows_q > INT32_MAX || rows_k > INT32_MAX) return BSATTN_ERR_INVALID_ARG;
    p.seqlen_q = seqlen_q;
    p.seqlen_k = seqlen_k;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.full_cnt = meta->full_cnt;
    p.full_idx = meta->full_idx;
    p.mask_cnt = meta->mask_cnt;
    p.mask_idx = meta->mask_idx;
    p.cu_tm = meta->cu_total_m_blocks;
    p.cu_off = meta->cu_block_idx_offsets;
    p.vl = kv_valid_len;
    p.vl_stride = meta->num_n;
    p.kind = (int)kind;
    if (mp) {
        p.window_left = mp->window_left;
        p.sink_tokens = mp->sink_tokens;
        p.prefix_len = mp->prefix_len;
        p.doc_q = mp->doc_id_q;
        p.doc_k = mp->doc_id_k;
    }
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634074);
    p.out = out;
    p.out_f32 = out_dtype == BSATTN_OUT_F32 ? 1 : 0;
    p.lse = lse;
    p.err = err_flag;
    const long long wl = g_wait_limit.load(std::memory_order_relaxed);
    p.wait_limit = wl > 0 ? wl : bsattn::kDefaultWaitLimitCycles;
    p.pairs_per_head = (int)cdiv(p.total_m, 2);
    if ((long long)H * p.pairs_per_head > INT32_MAX) return BSATTN_ERR_INVALID_ARG;
    p.num_units = H * p.pairs_per_head;
    if (p.num_units == 0 || rows_q == 0) return BSATTN_OK;
    if (workspace) {
        if (!aligned16(workspace)) return BSATTN_ERR_INVALID_ARG;
        size_t need = 0;
        if ((st = bsattn_fwd_workspace_size(meta, &need)) != BSATTN_OK) return st;
        if (need > 0) {
            if (workspace_bytes < need) return BSATTN_ERR_INVALID_ARG;
            p.dynamic = 1;
            p.sched_counter = static_cast<uint32_t *>(workspace);
            p.sched_order = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + kWorkspaceHeader);
        }
    }

    CUtensorMap tq, tk, tv;
    if (!encode_bshd(&tq, q, rows_q, H, D) || !encode_bshd(&tk, k, rows_k > 0 ? rows_k : 1, H, D) ||
        !encode_bshd(&tv, v, rows_k > 0 ? rows_k : 1, H, D))
        return BSATTN_ERR_CUDA;
    CUtensorMap tks = tk, tvs = tv;  // summary maps: unused unless proxy summaries are given
    if (proxy) {
        const long long sum_rows = (long long)B * meta->num_n;
        if (!encode_bshd(&tks, proxy->k_sum, sum_rows, H, D) ||
            !encode_bshd(&tvs, proxy->v_sum, sum_rows, H, D))
            return BSATTN_ERR_CUDA;
        p.proxy = 1;
        p.sel_words = proxy->sel_words;
        p.sel_words_per_row = proxy->words_per_row;
        p.proxy_tail = seqlen_k - (meta->num_n - 1) * kTile;
    }
    const int sms = num_sms_current_device();
    if (sms <= 0) return BSATTN_ERR_CUDA;
    cudaError_t e = bsattn::launch_fwd(p, tq, tk, tv, tks, tvs, D, sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

// Workspace of bsattn_bwd, in 256-byte aligned regions: the KV-major counts
// (full, mask) and the KV tile order, [B, H, num_n] int32 each (varlen: [H,
// B num_n]); the KV-major lists (full, mask), int32, and the selection codes,
// one byte each, all in the layout of the forward's index lists ([B, H, num_n,
// num_m] batched, [H, total_n] varlen); the KV tile prefix [B + 1]; then
// LSE * log2(e) and D, fp32, 128 per Q tile ([B, H, num_m] or [H, total_m]).
struct BwdLayout {
    size_t t_full_cnt, t_mask_cnt, order, t_full_idx, t_mask_idx, codes, cu_tn, lse2, dvec, total;
};

BwdLayout bwd_layout(const bsattn_meta *m) {
    auto up = [](size_t x) { return (x + 255u) & ~(size_t)255u; };
    const size_t cols = (size_t)m->B * (size_t)m->H * (size_t)m->num_n;
    const size_t entries = m->varlen ? (size_t)m->H * (size_t)m->total_n_blocks : cols * (size_t)m->num_m;
    const size_t q_tiles = m->varlen ? (size_t)m->H * (size_t)m->total_m_blocks
                                     : (size_t)m->B * (size_t)m->H * (size_t)m->num_m;
    BwdLayout L;
    L.t_full_cnt = 0;
    L.t_mask_cnt = L.t_full_cnt + up(cols * 4u);
    L.order = L.t_mask_cnt + up(cols * 4u);
    L.t_full_idx = L.order + up(cols * 4u);
    L.t_mask_idx = L.t_full_idx + up(entries * 4u);
    L.codes = L.t_mask_idx + up(entries * 4u);
    L.cu_tn = L.codes + up(entries);
    L.lse2 = L.cu_tn + up(((size_t)m->B + 1u) * 4u);
    L.dvec = L.lse2 + up(q_tiles * (size_t)kTile * 4u);
    L.total = L.dvec + up(q_tiles * (size_t)kTile * 4u);
    return L;
}

}  // namespace

extern "C" {

const char *bsattn_status_string(bsattn_status s) {
    switch (s) {
    case BSATTN_OK: return "BSATTN_OK";
    case BSATTN_ERR_INVALID_ARG: return "BSATTN_ERR_INVALID_ARG";
    case BSATTN_ERR_UNSUPPORTED: return "BSATTN_ERR_UNSUPPORTED";
    case BSATTN_ERR_CUDA: return "BSATTN_ERR_CUDA";
    case BSATTN_ERR_CAPACITY: return "BSATTN_ERR_CAPACITY";
    default: return "BSATTN_ERR_UNKNOWN";
    }
}

int32_t bsattn_abi_version(void) { return BSATTN_ABI_VERSION; }

bsattn_status bsattn_testing_set_wait_limit(long long cycles) {
    g_wait_limit.store(cycles > 0 ? cycles : 0, std::memory_order_relaxed);
    return BSATTN_OK;
}

bsattn_status bsattn_fwd_workspace_size(const bsattn_meta *meta, size_t *bytes) {
    if (!bytes) return BSATTN_ERR_INVALID_ARG;
    *bytes = 0;
    bsattn_status st = check_meta(meta);
    if (st != BSATTN_OK) return st;
    const long long units = fwd_units(meta);
    if (units <= 0 || units > bsattn::kMaxScheduledUnits) return BSATTN_OK;
    *bytes = (size_t)(kWorkspaceHeader + 4 * units);
    return BSATTN_OK;
}

bsattn_status bsattn_build_meta(const uint8_t *block_map, const int32_t *cu_seqlens_q,
                                const int32_t *cu_seqlens_k, int32_t seqlen_q, int32_t seqlen_k,
                                const int32_t *kv_valid_len, bsattn_mask_kind kind,
                                const bsattn_mask_params *mp, const bsattn_meta *meta,
                                int32_t *err_flag, void *stream) {
    if (!block_map) return BSATTN_ERR_INVALID_ARG;
    bsattn::MetaParams p = {};
    p.src = bsattn::kSrcByteMap;
    p.map = block_map;
    return build_meta_impl(p, cu_seqlens_q, cu_seqlens_k, seqlen_q, seqlen_k, kv_valid_len, kind, mp,
                           meta, err_flag, stream);
}

bsattn_status bsattn_kv_summaries(const void *k, const void *v, int32_t B, int32_t seqlen_k,
                                  int32_t H, int32_t D, void *k_sum, void *v_sum, void *stream) {
    if (!k || !v || !k_sum || !v_sum) return BSATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || seqlen_k <= 0 || D <= 0 || (D & 1) || D > 256) return BSATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(k_sum) | reinterpret_cast<uintptr_t>(v_sum)) & 3u)
        return BSATTN_ERR_INVALID_ARG;
    if ((long long)B * seqlen_k * H * D > (1LL << 40)) return BSATTN_ERR_INVALID_ARG;
    const cudaError_t e = bsattn::launch_kv_summary(k, v, B, seqlen_k, H, D, k_sum, v_sum,
                                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

bsattn_status bsattn_build_meta_blocks(const uint8_t *block_map, int32_t q_block_tiles,
                                       int32_t kv_block_tiles, int32_t seqlen_q, int32_t seqlen_k,
                                       const int32_t *kv_valid_len_blocks,
                                       int32_t *kv_valid_len_tiles, bsattn_mask_kind kind,
                                       const bsattn_mask_params *mp, const bsattn_meta *meta,
                                       int32_t *err_flag, void *stream) {
    if (!block_map || !meta) return BSATTN_ERR_INVALID_ARG;
    if (q_block_tiles < 1 || kv_block_tiles < 1 || q_block_tiles > 1024 || kv_block_tiles > 1024)
        return BSATTN_ERR_INVALID_ARG;
    if (meta->varlen) return BSATTN_ERR_UNSUPPORTED;  // batched layouts only
    if (!per_tile(meta)) return BSATTN_ERR_UNSUPPORTED;  // writes per-tile lists
    if (kv_valid_len_blocks && !kv_valid_len_tiles) return BSATTN_ERR_INVALID_ARG;
    bsattn::MetaParams p = {};
    p.src = bsattn::kSrcByteMap;
    p.map = block_map;
    p.q_block_tiles = q_block_tiles;
    p.kv_block_tiles = kv_block_tiles;
    p.block_m = (int)cdiv(meta->num_m, q_block_tiles);
    p.block_n = (int)cdiv(meta->num_n, kv_block_tiles);
    p.kv_block_shift = -1;
    for (int s = 0; s < 11; ++s)
        if ((1 << s) == kv_block_tiles) p.kv_block_shift = s;
    p.vl_tiles_out = kv_valid_len_tiles;
    p.vl_per_block = kv_valid_len_blocks ? 1 : 0;
    return build_meta_impl(p, nullptr, nullptr, seqlen_q, seqlen_k, kv_valid_len_blocks, kind, mp,
                           meta, err_flag, stream);
}

bsattn_status bsattn_build_meta_bitmask(const uint32_t *words, int32_t words_per_row,
                                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                        int32_t seqlen_q, int32_t seqlen_k,
                                        const int32_t *kv_valid_len, bsattn_mask_kind kind,
                                        const bsattn_mask_params *mp, const bsattn_meta *meta,
                                        int32_t *err_flag, void *stream) {
    if (!words || words_per_row <= 0) return BSATTN_ERR_INVALID_ARG;
    // batched rows must hold num_n bits; varlen rows are checked per sequence on the device
    if (meta && !meta->varlen && (long long)words_per_row * 32 < meta->num_n) return BSATTN_ERR_INVALID_ARG;
    bsattn::MetaParams p = {};
    p.src = bsattn::kSrcBitmask;
    p.words = words;
    p.words_per_row = words_per_row;
    return build_meta_impl(p, cu_seqlens_q, cu_seqlens_k, seqlen_q, seqlen_k, kv_valid_len, kind, mp,
                           meta, err_flag, stream);
}

bsattn_status bsattn_build_meta_bsr(const int32_t *block_indptr, const int32_t *block_indices,
                                    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                    int32_t seqlen_q, int32_t seqlen_k, const int32_t *kv_valid_len,
                                    bsattn_mask_kind kind, const bsattn_mask_params *mp,
                                    const bsattn_meta *meta, int32_t *err_flag, void *stream) {
    if (!block_indptr || !block_indices) return BSATTN_ERR_INVALID_ARG;
    if (seqlen_k <= 0) return BSATTN_ERR_INVALID_ARG;  // sizes the per-row bit set
    bsattn::MetaParams p = {};
    p.src = bsattn::kSrcBsr;
    p.indptr = block_indptr;
    p.indices = block_indices;
    const long long nn_max = cdiv(seqlen_k, kTile);
    p.bitset_words = (int)((nn_max + 31) / 32);
    if ((long long)p.bitset_words * 8 * 4 > 200 * 1024) return BSATTN_ERR_UNSUPPORTED;
    return build_meta_impl(p, cu_seqlens_q, cu_seqlens_k, seqlen_q, seqlen_k, kv_valid_len, kind, mp,
                           meta, err_flag, stream);
}

bsattn_status bsattn_fwd(const void *q, const void *k, const void *v, int32_t B, int32_t seqlen_q,
                         int32_t seqlen_k, int32_t H, int32_t D, const int32_t *cu_seqlens_q,
                         const int32_t *cu_seqlens_k, const bsattn_meta *meta,
                         const int32_t *kv_valid_len, bsattn_mask_kind kind,
                         const bsattn_mask_params *mp, float softmax_scale, void *out,
                         bsattn_out_dtype out_dtype, float *lse, void *workspace,
                         size_t workspace_bytes, int32_t *err_flag, void *stream) {
    return fwd_impl(q, k, v, B, seqlen_q, seqlen_k, H, D, cu_seqlens_q, cu_seqlens_k, meta, kv_valid_len,
                    kind, mp, softmax_scale, out, out_dtype, lse, workspace, workspace_bytes, err_flag,
                    stream, nullptr);
}

bsattn_status bsattn_fwd_proxy(const void *q, const void *k, const void *v, int32_t B,
                               int32_t seqlen_q, int32_t seqlen_k, int32_t H, int32_t D,
                               const bsattn_meta *meta, const uint32_t *sel_words,
                               int32_t words_per_row, const void *k_sum, const void *v_sum,
                               float softmax_scale, void *out, bsattn_out_dtype out_dtype, float *lse,
                               void *workspace, size_t workspace_bytes, int32_t *err_flag,
                               void *stream) {
    if (!meta) return BSATTN_ERR_INVALID_ARG;
    if (meta->varlen || !per_tile(meta)) return BSATTN_ERR_UNSUPPORTED;  // batched, per tile
    if (!sel_words || !k_sum || !v_sum) return BSATTN_ERR_INVALID_ARG;
    if (!aligned16(k_sum) || !aligned16(v_sum)) return BSATTN_ERR_INVALID_ARG;
    if (words_per_row <= 0 || (long long)words_per_row * 32 < meta->num_n) return BSATTN_ERR_INVALID_ARG;
    if ((long long)B * meta->num_n > INT32_MAX) return BSATTN_ERR_INVALID_ARG;
    ProxyArgs pa{sel_words, words_per_row, k_sum, v_sum};
    return fwd_impl(q, k, v, B, seqlen_q, seqlen_k, H, D, nullptr, nullptr, meta, nullptr,
                    BSATTN_MASK_NONE, nullptr, softmax_scale, out, out_dtype, lse, workspace,
                    workspace_bytes, err_flag, stream, &pa);
}

bsattn_status bsattn_bwd_workspace_size(const bsattn_meta *meta, size_t *bytes) {
    bsattn_status st = check_meta(meta);
    if (st != BSATTN_OK) return st;
    if (!per_tile(meta)) return BSATTN_ERR_UNSUPPORTED;
    if (!bytes) return BSATTN_ERR_INVALID_ARG;
    if (meta->varlen && meta->num_n <= 0) return BSATTN_ERR_INVALID_ARG;
    *bytes = bwd_layout(meta).total;
    return BSATTN_OK;
}

bsattn_status bsattn_bwd(const void *q, const void *k, const void *v, const void *out,
                         bsattn_out_dtype out_dtype, const float *lse, const void *dout, int32_t B,
                         int32_t seqlen_q, int32_t seqlen_k, int32_t H, int32_t D,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                         const bsattn_meta *meta, const int32_t *kv_valid_len, bsattn_mask_kind kind,
                         const bsattn_mask_params *mp, float softmax_scale, void *dq, void *dk, void *dv,
                         bsattn_out_dtype grad_dtype, void *workspace, size_t workspace_bytes,
                         int32_t *err_flag, void *stream) {
    bsattn_status st = check_meta(meta);
    if (st != BSATTN_OK) return st;
    if (!per_tile(meta)) return BSATTN_ERR_UNSUPPORTED;
    if ((st = check_mask(kind, mp)) != BSATTN_OK) return st;
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace)
        return BSATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return BSATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || seqlen_q < 0 || seqlen_k < 0) return BSATTN_ERR_INVALID_ARG;
    if (meta->B != B || meta->H != H) return BSATTN_ERR_INVALID_ARG;
    long long rows_q, rows_k;
    if (meta->varlen) {
        // seqlen_q / seqlen_k: total packed rows, as for bsattn_fwd
        if (!cu_seqlens_q || !cu_seqlens_k || meta->num_n <= 0) return BSATTN_ERR_INVALID_ARG;
        rows_q = seqlen_q;
        rows_k = seqlen_k;
    } else {
        if (cu_seqlens_q || cu_seqlens_k) return BSATTN_ERR_INVALID_ARG;
        if (meta->num_m != cdiv(seqlen_q, kTile) || meta->num_n != cdiv(seqlen_k, kTile))
            return BSATTN_ERR_INVALID_ARG;
        rows_q = (long long)B * seqlen_q;
        rows_k = (long long)B * seqlen_k;
    }
    if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return BSATTN_ERR_INVALID_ARG;
    if (out_dtype != BSATTN_OUT_BF16 && out_dtype != BSATTN_OUT_F32) return BSATTN_ERR_INVALID_ARG;
    if (grad_dtype != BSATTN_OUT_BF16 && grad_dtype != BSATTN_OUT_F32) return BSATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return BSATTN_ERR_UNSUPPORTED;
    if (rows_q > INT32_MAX || rows_k > INT32_MAX) return BSATTN_ERR_INVALID_ARG;
    const BwdLayout L = bwd_layout(meta);
    if (workspace_bytes < L.total) return BSATTN_ERR_INVALID_ARG;
    if (rows_q == 0 || rows_k == 0) {
        // no keys (every row's key set is empty) or no queries: all gradients are 0
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        const size_t el = grad_dtype == BSATTN_OUT_F32 ? 4u : 2u;
        if (cudaMemsetAsync(dq, 0, (size_t)rows_q * H * D * el, s) != cudaSuccess ||
            cudaMemsetAsync(dk, 0, (size_t)rows_k * H * D * el, s) != cudaSuccess ||
            cudaMemsetAsync(dv, 0, (size_t)rows_k * H * D * el, s) != cudaSuccess)
            return BSATTN_ERR_CUDA;
        return BSATTN_OK;
    }

    char *ws = static_cast<char *>(workspace);
    bsattn::BwdParams p = {};
    p.varlen = meta->varlen ? 1 : 0;
    p.B = B;
    p.H = H;
    p.D = D;
    p.seqlen_q = seqlen_q;
    p.seqlen_k = seqlen_k;
    p.num_m = meta->varlen ? 0 : meta->num_m;
    p.num_n = meta->num_n;
    p.rows_q = rows_q;
    p.rows_k = rows_k;
    p.total_m = meta->total_m_blocks;
    p.total_n = meta->total_n_blocks;
    p.num_m_max = meta->varlen ? meta->total_m_blocks : meta->num_m;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.cu_tm = meta->cu_total_m_blocks;
    p.cu_off = meta->cu_block_idx_offsets;
    p.cu_tn = reinterpret_cast<int32_t *>(ws + L.cu_tn);
    p.scale = softmax_scale;
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634074);
    p.full_cnt = meta->full_cnt;
    p.full_idx = meta->full_idx;
    p.mask_cnt = meta->mask_cnt;
    p.mask_idx = meta->mask_idx;
    p.t_full_cnt = reinterpret_cast<int32_t *>(ws + L.t_full_cnt);
    p.t_mask_cnt = reinterpret_cast<int32_t *>(ws + L.t_mask_cnt);
    p.t_full_idx = reinterpret_cast<int32_t *>(ws + L.t_full_idx);
    p.t_mask_idx = reinterpret_cast<int32_t *>(ws + L.t_mask_idx);
    p.codes = reinterpret_cast<uint8_t *>(ws + L.codes);
    p.order = reinterpret_cast<int32_t *>(ws + L.order);
    p.vl = kv_valid_len;
    p.kind = (int)kind;
    if (mp) {
        p.window_left = mp->window_left;
        p.sink_tokens = mp->sink_tokens;
        p.prefix_len = mp->prefix_len;
        p.doc_q = mp->doc_id_q;
        p.doc_k = mp->doc_id_k;
    }
    p.o = out;
    p.o_f32 = out_dtype == BSATTN_OUT_F32 ? 1 : 0;
    p.dout = static_cast<const uint16_t *>(dout);
    p.lse = lse;
    p.lse2 = reinterpret_cast<float *>(ws + L.lse2);
    p.dvec = reinterpret_cast<float *>(ws + L.dvec);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.grad_f32 = grad_dtype == BSATTN_OUT_F32 ? 1 : 0;
    p.err = err_flag;

    CUtensorMap tq, tk, tv, tdo;
    if (!encode_bshd(&tq, q, rows_q, H, D) || !encode_bshd(&tk, k, rows_k, H, D) ||
        !encode_bshd(&tv, v, rows_k, H, D) || !encode_bshd(&tdo, dout, rows_q, H, D))
        return BSATTN_ERR_CUDA;
    cudaError_t e = bsattn::launch_bwd(p, tq, tk, tv, tdo, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------- fixed scheduling scratch --
// For callers that cannot allocate device memory at call time (a host program
// with no device allocator of its own, or a loop that must not call cudaMalloc /
// cudaFree, the latter being device-synchronising): a scheduling workspace of a
// fixed size that lives in the library's own device data.  One array per device
// (a __device__ variable has one instance per device); every call on a device
// uses it, so overlapping calls would race on it.
namespace {

constexpr size_t kStaticScratchBytes = kWorkspaceHeader + 4u * (size_t)BSATTN_STATIC_SCRATCH_UNITS;
static_assert(BSATTN_STATIC_SCRATCH_UNITS <= bsattn::kMaxScheduledUnits,
              "the fixed scratch must stay within the scheduling pass's limit");

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

CtxGetCurrentFn get_ctx_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Device address of the current device's scratch.  It is resolved with the
// device current and kept per CUDA context: a reset device gets a new context
// (and a new copy of the library's device data), so the address is resolved
// again after one.
bsattn_status static_scratch_address(void **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSATTN_ERR_CUDA;
    CtxGetCurrentFn ctx_fn = get_ctx_fn();
    if (!ctx_fn) return BSATTN_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (ctx_fn(&ctx) != CUDA_SUCCESS) return BSATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!ctx || !g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
        // cudaGetSymbolAddress also makes the device's primary context current on
        // this thread when none is.
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return BSATTN_ERR_CUDA;
        if (ctx_fn(&ctx) != CUDA_SUCCESS || !ctx) return BSATTN_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *addr = g_scratch_addr[dev];
    return BSATTN_OK;
}

}  // namespace

extern "C" bsattn_status bsattn_fwd_static_scratch(
    const void *q, const void *k, const void *v, int32_t B, int32_t seqlen_q, int32_t seqlen_k,
    int32_t H, int32_t D, const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
    const bsattn_meta *meta, const int32_t *kv_valid_len, bsattn_mask_kind kind,
    const bsattn_mask_params *mp, float softmax_scale, void *out, bsattn_out_dtype out_dtype,
    float *lse, int32_t *err_flag, void *stream) {
    bsattn_status st = check_meta(meta);
    if (st != BSATTN_OK) return st;
    const long long units = fwd_units(meta);
    if (units > BSATTN_STATIC_SCRATCH_UNITS) return BSATTN_ERR_CAPACITY;
    void *scratch = nullptr;
    if ((st = static_scratch_address(&scratch)) != BSATTN_OK) return st;
    return bsattn_fwd(q, k, v, B, seqlen_q, seqlen_k, H, D, cu_seqlens_q, cu_seqlens_k, meta,
                      kv_valid_len, kind, mp, softmax_scale, out, out_dtype, lse, scratch,
                      kStaticScratchBytes, err_flag, stream);
}
