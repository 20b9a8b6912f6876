// Parameters passed from the C-ABI entry points to the kernels (internal).
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "bsattn.h"

namespace bsattn {

constexpr int kTile = 128;  // tile_m = tile_n = 128 in this build

// Where the metadata kernel reads which KV tiles a Q-tile row selects.
enum MetaSource { kSrcByteMap = 0, kSrcBitmask = 1, kSrcBsr = 2 };

struct MetaParams {
    int src;                       // MetaSource
    const uint8_t *map;            // byte map, laid out like the index lists
    const uint32_t *words;         // bitmask: [rows][words_per_row], bit n % 32 of word n / 32
    int words_per_row;
    const int32_t *indptr;         // BSR: [rows + 1] into indices
    const int32_t *indices;        // BSR: selected KV tiles of each row, any order
    int bitset_words;              // BSR: 32-bit words of the per-warp bit set
    // Sparse blocks of q_block_tiles x kv_block_tiles tiles (batched byte map
    // only; block_n > 0 selects this form): the map is [B, H, block_m, block_n].
    int q_block_tiles, kv_block_tiles, block_m, block_n;
    int kv_block_shift;            // log2(kv_block_tiles) when a power of two, else -1
    // kv_valid_len given per sparse KV block ([B, vl_stride] blocks): tile j of a
    // block keeps clamp(v - 128 j, 0, 128) keys; vl_tiles_out, if set, receives
    // the per-tile values [B, num_n].
    int vl_per_block;
    int32_t *vl_tiles_out;
    int varlen, B, H;
    int num_m, num_n;              // batched sizes (varlen: num_n = kv_valid_len stride)
    int tile_q, tile_k;            // rows / keys of a listed block: 128, or (batched) a
                                   // sparse block of two tiles
    int total_m, total_n;          // varlen packed sizes as allocated by the caller
    int seqlen_q, seqlen_k;        // batched
    const int32_t *cu_q, *cu_k;    // varlen [B+1]
    int32_t *cu_tm, *cu_off;       // varlen [B+1], written by the offsets kernel
    const int32_t *vl;             // [B, vl_stride] or null
    int vl_stride;
    int kind, window_left, sink_tokens, prefix_len;
    const int32_t *doc_q, *doc_k;
    int32_t *full_cnt, *full_idx, *mask_cnt, *mask_idx;
    int32_t *err;
};

struct FwdParams {
    int varlen, B, H;
    int seqlen_q, seqlen_k;        // batched per-sequence lengths
    const int32_t *cu_q, *cu_k;    // varlen [B+1]
    int num_m, num_n;              // batched: 128-row tiles per sequence
    int total_m, total_n;          // Q tiles per head over the batch; varlen idx row size
    // Lists per sparse block (batched): list_q_tiles = 2 Q tiles share a list row
    // (one work unit), each entry covers list_kv_tiles (1 or 2) KV tiles; list_m
    // rows per sequence, list_n entries per row.  list_q_tiles = 1: per-tile lists.
    int list_q_tiles, list_kv_tiles, list_m, list_n;
    const int32_t *full_cnt, *full_idx, *mask_cnt, *mask_idx;
    const int32_t *cu_tm, *cu_off; // varlen
    const int32_t *vl;
    int vl_stride;
    int kind, window_left, sink_tokens, prefix_len;
    const int32_t *doc_q, *doc_k;
    float scale_log2;              // softmax_scale * log2(e)
    void *out;                     // bf16 or fp32 (out_f32)
    int out_f32;
    float *lse;
    int32_t *err;
    int lse_row_stride;            // batched: seqlen_q; varlen: total q rows
    int pairs_per_head;            // ceil(total_m / 2)
    int num_units;                 // H * pairs_per_head
    int dynamic;                   // units claimed from sched_order through sched_counter
    // Proxy compensation (batched): after each unit's listed tiles, summary items
    // over the KV-tile summaries (mean K, summed V) of the tiles' sequences; a
    // summary column counts only if its tile is not in the row's exact selection
    // (sel_words, bit n % 32 of word n / 32), with a denominator mass of 128 keys,
    // proxy_tail for the sequence's last tile.
    int proxy;
    const uint32_t *sel_words;
    int sel_words_per_row;
    int proxy_tail;
    uint32_t *sched_counter;       // workspace: next slot of sched_order
    int32_t *sched_order;          // workspace: units, heaviest first
    long long wait_limit;          // cycles after which a pipeline wait gives up
};

// Cycles after which a forward pipeline wait gives up unless a test lowers it
// (about one second at 2 GHz).
constexpr long long kDefaultWaitLimitCycles = 1ll << 31;

// Units the scheduling pass can order (its per-unit keys live in shared memory).
constexpr int kMaxScheduledUnits = 98304;

// Backward (batched): dK/dV per KV tile over the KV-major lists, dQ per Q tile
// over the forward lists.
struct BwdParams {
    int varlen;
    int B, H, D, seqlen_q, seqlen_k, num_m, num_n;  // varlen: num_m unused, num_n = vl stride
    long long rows_q, rows_k;     // packed rows (batched: B * seqlen)
    int total_m, total_n;         // varlen metadata totals
    int num_m_max;                // longest possible KV-major list (batched num_m, varlen total_m)
    const int32_t *cu_q, *cu_k, *cu_tm, *cu_off;  // varlen offsets (cu_seqlens, metadata)
    int32_t *cu_tn;               // varlen workspace [B + 1]: KV tile prefix
    float scale, scale_log2;
    const int32_t *full_cnt, *full_idx, *mask_cnt, *mask_idx;  // forward lists
    int32_t *t_full_cnt, *t_full_idx, *t_mask_cnt, *t_mask_idx; // KV-major lists
    uint8_t *codes;               // selection code per (KV tile, Q tile), list layout
    int32_t *order;               // [B * H * num_n] KV tile ids, longest list first, -1 padding
    const int32_t *vl;            // [B, num_n] or null (mask tiles only)
    int kind, window_left, sink_tokens, prefix_len;
    const int32_t *doc_q, *doc_k;
    const void *o;                // forward output, bf16 or fp32, layout of q
    int o_f32;
    const uint16_t *dout;         // bf16, layout of q
    const float *lse;             // batched [B, H, S_q], varlen [H, rows_q]; natural log
    float *lse2, *dvec;           // workspace, 128 rows per Q tile: -LSE * log2(e), -D (negated:
                                  // the gradient kernels add them)
    void *dq, *dk, *dv;           // gradients in q / k / v layouts
    int grad_f32;
    int32_t *err;
};

cudaError_t launch_bwd(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, cudaStream_t stream);

cudaError_t launch_meta(const MetaParams &p, cudaStream_t stream);
cudaError_t launch_kv_summary(const void *k, const void *v, int B, int S, int H, int D, void *k_sum,
                              void *v_sum, cudaStream_t stream);
cudaError_t launch_fwd(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tks, const CUtensorMap &tvs, int D,
                       int num_sms, cudaStream_t stream);

}  // namespace bsattn
