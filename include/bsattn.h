/*
 * bsattn -- block-sparse attention for NVIDIA GB300 (sm_103a): metadata from a
 * block map (byte map, bitmask, BSR or coarse blocks), the forward (exact, or
 * with proxy compensation), and the backward of the exact forward.
 *
 * C ABI.  Every pointer argument is caller-owned memory; the library allocates
 * nothing and keeps no state between calls.  Device pointers must be CUDA
 * device memory on the current device.  Calls are asynchronous on `stream`
 * (a cudaStream_t passed as void*; NULL = the legacy default stream) and never
 * synchronise with the host.  The returned status covers host-side argument
 * validation and kernel-launch errors only; faults in the metadata that only the
 * device can see are reported through the optional `err_flag` word (bits
 * BSATTN_FLAG_*), which the kernels OR into and never clear.  No kernel traps.
 *
 * Sources for the operations (page titles and the part of the page):
 *  - "[CuTe,Flex] varlen blocksparsity", flash-attention pull request #2224:
 *    description (batched and varlen-packed *_block_cnt / *_block_idx shapes,
 *    num_m(b), num_n(b), total_m_blocks, total_n_blocks) and review thread
 *    (metadata tuple (mask_block_cnt, mask_block_idx, full_block_cnt,
 *    full_block_idx); cu_total_m_blocks and cu_block_idx_offsets, the latter
 *    the running sum of num_m(b) * num_n(b); mask_mod only on mask blocks).
 *  - "Dense FlashAttention vs Block-Sparse Attention" (learning note on
 *    Block-Sparse-Attention), sections 2 and 4: boolean block rows become
 *    reversed index lists padded with -1; the kernel walks only the listed
 *    blocks and the K/V loads jump to each listed block.
 *  - "[feat] VSA-256 fastpath on Blackwell via FA4 CuTe block-sparse
 *    attention" (FastVideo #1354): Q/K/V in BSHD layout; a per-KV-block valid
 *    length read by mask_mod; LSE in [B, H, S] layout.
 *  - "feat(prims-ts): support proxy-compensated block-sparse attention"
 *    (FlashInfer #4872): the bitmask and BSR selection formats and proxy
 *    compensation (see bsattn_build_meta_bitmask, bsattn_build_meta_bsr,
 *    bsattn_fwd_proxy).
 *  The backward (bsattn_bwd) is the gradient of the forward's definition; the
 *  first two pages name it as the missing step for training.
 */
#ifndef BSATTN_H
#define BSATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BSATTN_ABI_VERSION 2

typedef enum {
    BSATTN_OK = 0,
    BSATTN_ERR_INVALID_ARG = 1, /* a pointer, size or layout argument is invalid     */
    BSATTN_ERR_UNSUPPORTED = 2, /* valid, but not served by this build (e.g. D=96)   */
    BSATTN_ERR_CUDA = 3,        /* a CUDA call or a kernel launch failed             */
    BSATTN_ERR_CAPACITY = 4     /* the problem exceeds a fixed capacity: see
                                   bsattn_fwd_static_scratch                         */
} bsattn_status;

/* Token-level mask_mod applied on mask-list blocks.  Positions are
 * sequence-local: i = query position, j = key position inside the sequence. */
typedef enum {
    BSATTN_MASK_NONE = 0,           /* all keys                                      */
    BSATTN_MASK_CAUSAL = 1,         /* j <= i                                        */
    BSATTN_MASK_SLIDING_WINDOW = 2, /* j <= i && (i - j < window_left || j < sink_tokens) */
    BSATTN_MASK_DOCUMENT = 3,       /* doc_id_q[q row] == doc_id_k[k row]            */
    BSATTN_MASK_PREFIX = 4          /* j < prefix_len || j <= i                      */
} bsattn_mask_kind;

/* Element type of the attention output. */
typedef enum {
    BSATTN_OUT_BF16 = 0, /* round-to-nearest-even of the fp32 result */
    BSATTN_OUT_F32 = 1   /* the fp32 result itself                   */
} bsattn_out_dtype;

/* Device-side error bits ORed into *err_flag. */
#define BSATTN_FLAG_BAD_COUNT 0x1   /* a block count outside [0, num_n(b)] was clamped        */
#define BSATTN_FLAG_BAD_INDEX 0x2   /* a block index outside [0, num_n(b)) was skipped        */
#define BSATTN_FLAG_TIMEOUT 0x4     /* a pipeline wait exceeded its limit; the CTA stopped   */
#define BSATTN_FLAG_BAD_SEQLENS 0x8 /* cu_seqlens disagree with the meta or leave the packed rows */

typedef struct {
    int32_t window_left;      /* SLIDING_WINDOW: keys with 0 <= i - j < window_left      */
    int32_t sink_tokens;      /* SLIDING_WINDOW: keys j < sink_tokens (still causal)     */
    int32_t prefix_len;       /* PREFIX: keys j < prefix_len, else causal                */
    const int32_t *doc_id_q;  /* DOCUMENT: device int32, one id per packed q row        */
    const int32_t *doc_id_k;  /* DOCUMENT: device int32, one id per packed k row        */
} bsattn_mask_params;

/*
 * Block-sparse metadata (all arrays device int32, caller-allocated).
 *
 * Batched (varlen = 0), sequences of equal length:
 *   full_cnt, mask_cnt  [B, H, num_m]
 *   full_idx, mask_idx  [B, H, num_m, num_n]
 *   cu_total_m_blocks, cu_block_idx_offsets: unused (may be NULL)
 * Varlen (varlen = 1), sequences packed back to back:
 *   full_cnt, mask_cnt  [H, total_m_blocks]
 *   full_idx, mask_idx  [H, total_n_blocks]; row (b, m) of head h starts at
 *                       h * total_n_blocks + cu_block_idx_offsets[b] + m * num_n(b)
 *   cu_total_m_blocks   [B+1], running sum of num_m(b)
 *   cu_block_idx_offsets[B+1], running sum of num_m(b) * num_n(b)
 *   num_m               unused; num_n = the row stride of kv_valid_len (at least
 *                       the largest num_n(b))
 * Each index row lists KV block ids in descending order; entries at and after
 * the row's count are -1.
 *
 * tile_m x tile_n is the size of a listed block: 128 x 128 (one tile; every
 * entry point), or, batched only, a sparse block of two Q tiles and one or two
 * KV tiles: 256 x 128 or 256 x 256 ("[CuTe,Flex] varlen blocksparsity",
 * flash-attention #2224: lists per q_subtile_factor x tile_m sparse block;
 * "[feat] VSA-256 fastpath on Blackwell via FA4 CuTe block-sparse attention",
 * FastVideo #1354: 256-token blocks).  Then num_m = ceil(seqlen_q / tile_m),
 * num_n = ceil(seqlen_k / tile_n), bsattn_build_meta classifies whole blocks
 * (the token predicate over the block's query rows and keys), kv_valid_len
 * holds one value per KV block ([B, num_n], tile j of a block keeping
 * clamp(v - 128 j, 0, 128) keys), and bsattn_fwd walks the block lists
 * directly: a block's two Q tiles form one work unit, each entry's KV tiles
 * are visited in turn.  The forward then needs ceil(seqlen_q / 128) even (each
 * Q block whole); bsattn_bwd, bsattn_fwd_proxy and bsattn_build_meta_blocks
 * take 128 x 128 metadata only.  Other sizes -> BSATTN_ERR_UNSUPPORTED.
 */
typedef struct {
    int32_t *full_cnt, *full_idx, *mask_cnt, *mask_idx;
    int32_t *cu_total_m_blocks, *cu_block_idx_offsets;
    int32_t varlen, B, H, num_m, num_n;
    int32_t total_m_blocks, total_n_blocks;
    int32_t tile_m, tile_n;
} bsattn_meta;

/*
 * bsattn_build_meta -- boolean block map -> full / mask lists (and, for
 * varlen, the two offset tensors).
 *
 * Every selected KV block n of row (b, h, m) is classified by the token
 * predicate P(i, j) = j < seqlen_k(b) && mask_mod(i, j) && (j - tile_n n) <
 * kv_valid_len[b, n] over the row's query rows i < seqlen_q(b) (tile_m of them
 * from tile_m m) and the block's tile_n keys j: true for every pair -> full list,
 * for some pair -> mask list, for none -> dropped (tile_m = tile_n = 128 unless
 * the metadata is per sparse block, see above).  Result is bit-exact and
 * deterministic.
 *
 * block_map     device uint8; batched [B, H, num_m, num_n], varlen [H, total_n_blocks]
 *               in the packed layout above; nonzero = selected.
 * cu_seqlens_q  varlen: device int32 [B+1] packed row offsets; batched: NULL.
 * cu_seqlens_k  likewise for keys.
 * seqlen_q/_k   batched: per-sequence lengths (num_m == ceil(seqlen_q/128),
 *               num_n == ceil(seqlen_k/128) is checked); varlen: the packed row
 *               counts of q and k, or 0.  When positive, a sequence whose offsets
 *               reach past them (or are negative) is rejected: its rows are not
 *               written and BSATTN_FLAG_BAD_SEQLENS is set.
 * kv_valid_len  optional device int32 [B, meta->num_n]: valid keys at the start
 *               of each listed KV block (the rest of it is masked on mask blocks).
 * kind, mp      mask_mod (mp may be NULL unless the kind needs it).
 * meta          sizes in, device output pointers in; varlen also writes
 *               cu_total_m_blocks / cu_block_idx_offsets.  If the totals the
 *               device computes differ from meta->total_*_blocks, rows past the
 *               given totals are not written and BSATTN_FLAG_BAD_SEQLENS is set.
 * err_flag      optional device int32 word (see BSATTN_FLAG_*).
 */
bsattn_status bsattn_build_meta(const uint8_t *block_map, const int32_t *cu_seqlens_q,
                                const int32_t *cu_seqlens_k, int32_t seqlen_q, int32_t seqlen_k,
                                const int32_t *kv_valid_len, bsattn_mask_kind kind,
                                const bsattn_mask_params *mp, const bsattn_meta *meta,
                                int32_t *err_flag, void *stream);

/*
 * bsattn_kv_summaries -- per-KV-tile summaries for proxy compensation
 * ("feat(prims-ts): support proxy-compensated block-sparse attention", FlashInfer
 * #4872: one arithmetic-mean K summary and one summed-V summary per KV block).
 * For sequence b, KV tile n and head h, over the keys j of the tile
 * (128 n <= j < min(128 n + 128, seqlen_k)):
 *   k_sum[b, n, h, :] = mean_j k[b, j, h, :],   v_sum[b, n, h, :] = sum_j v[b, j, h, :]
 * accumulated in fp32 in ascending j, rounded to bf16 (round to nearest even).
 *
 * k, v          device bf16 [B, seqlen_k, H, D], contiguous, 4-byte aligned.
 * k_sum, v_sum  device bf16 [B, ceil(seqlen_k / 128), H, D] (written).
 * D even, at most 256; B, H, seqlen_k > 0.
 */
bsattn_status bsattn_kv_summaries(const void *k, const void *v, int32_t B, int32_t seqlen_k,
                                  int32_t H, int32_t D, void *k_sum, void *v_sum, void *stream);

/*
 * bsattn_build_meta_blocks -- bsattn_build_meta for a block map given at a
 * sparse block size that is a multiple of the 128-token tile ("[CuTe,Flex]
 * varlen blocksparsity", flash-attention #2224: q_subtile_factor; "[feat] VSA-256
 * fastpath on Blackwell via FA4 CuTe block-sparse attention", FastVideo #1354:
 * 256-token blocks run as 128-token tiles).  A sparse block covers q_block_tiles
 * x kv_block_tiles tiles; tile (m, n) is selected iff its block
 * (m / q_block_tiles, n / kv_block_tiles) is.  The lists written are identical
 * to those bsattn_build_meta writes for the expanded per-tile map.
 *
 * block_map            device uint8 [B, H, ceil(num_m / q_block_tiles),
 *                      ceil(num_n / kv_block_tiles)]; nonzero = selected.
 * q_block_tiles,
 * kv_block_tiles       tiles per sparse block along Q and KV, 1..1024.
 * seqlen_q, seqlen_k   per-sequence lengths, as for bsattn_build_meta (batched).
 * kv_valid_len_blocks  optional device int32 [B, ceil(num_n / kv_block_tiles)]:
 *                      valid keys at the start of each sparse KV block; tile j
 *                      of a block keeps clamp(v - 128 j, 0, 128) of them (the
 *                      VSA split of a 256-token block into min(v, 128) and
 *                      v - min(v, 128)).
 * kv_valid_len_tiles   device int32 [B, num_n], written with those per-tile
 *                      lengths (128 where none are given) for bsattn_fwd; required
 *                      when kv_valid_len_blocks is given, else optional (NULL).
 * Varlen metadata -> BSATTN_ERR_UNSUPPORTED.  Other arguments and errors as for
 * bsattn_build_meta.
 */
bsattn_status bsattn_build_meta_blocks(const uint8_t *block_map, int32_t q_block_tiles,
                                       int32_t kv_block_tiles, int32_t seqlen_q, int32_t seqlen_k,
                                       const int32_t *kv_valid_len_blocks,
                                       int32_t *kv_valid_len_tiles, bsattn_mask_kind kind,
                                       const bsattn_mask_params *mp, const bsattn_meta *meta,
                                       int32_t *err_flag, void *stream);

/*
 * bsattn_build_meta_bitmask -- bsattn_build_meta with the selected KV tiles of
 * each Q-tile row given as packed 32-bit words ("feat(prims-ts): support
 * proxy-compensated block-sparse attention", FlashInfer #4872, bitmask format:
 * one bit per semantic KV block; padding bits past the last block are ignored).
 * The lists written are identical to those bsattn_build_meta writes for the
 * equivalent byte map.
 *
 * words          device uint32 [rows][words_per_row]; KV tile n of a row is
 *                selected iff bit (n % 32) of word (n / 32) is set (least
 *                significant bit first).  Rows are ordered like the count arrays:
 *                batched (b, h, m) -> (b * H + h) * num_m + m; varlen
 *                (h, packed Q tile T) -> h * total_m_blocks + T.  Bits for
 *                tiles n >= num_n(b) are ignored.
 * words_per_row  > 0; batched: at least ceil(num_n / 32) (else
 *                BSATTN_ERR_INVALID_ARG); varlen: a sequence with more KV tiles
 *                than 32 * words_per_row sets BSATTN_FLAG_BAD_COUNT and only its
 *                first 32 * words_per_row tiles can be selected.
 * Other arguments and errors as for bsattn_build_meta.
 */
bsattn_status bsattn_build_meta_bitmask(const uint32_t *words, int32_t words_per_row,
                                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                        int32_t seqlen_q, int32_t seqlen_k,
                                        const int32_t *kv_valid_len, bsattn_mask_kind kind,
                                        const bsattn_mask_params *mp, const bsattn_meta *meta,
                                        int32_t *err_flag, void *stream);

/*
 * bsattn_build_meta_bsr -- bsattn_build_meta with the selected KV tiles given in
 * BSR form, block_indptr / block_indices over the Q-tile rows (same page:
 * canonical BSR block_indptr / block_indices).  The lists written are identical
 * to those for the equivalent byte map.
 *
 * block_indptr   device int32 [rows + 1], rows ordered as for the bitmask form;
 *                row r selects block_indices[block_indptr[r] .. block_indptr[r+1]).
 *                A row whose end is below its start selects nothing and sets
 *                BSATTN_FLAG_BAD_COUNT.
 * block_indices  device int32 [block_indptr[rows]], KV tile ids of each row in
 *                any order; a repeated id selects its tile once; an id outside
 *                [0, num_n(b)) is skipped and sets BSATTN_FLAG_BAD_INDEX.
 * seqlen_k       must be > 0: batched keys per sequence, varlen total packed keys
 *                (it bounds num_n(b), which sizes a per-row bit set of
 *                ceil(ceil(seqlen_k / 128) / 32) words in shared memory;
 *                BSATTN_ERR_UNSUPPORTED when that exceeds 6400 words).
 * Other arguments and errors as for bsattn_build_meta.
 */
bsattn_status bsattn_build_meta_bsr(const int32_t *block_indptr, const int32_t *block_indices,
                                    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                    int32_t seqlen_q, int32_t seqlen_k, const int32_t *kv_valid_len,
                                    bsattn_mask_kind kind, const bsattn_mask_params *mp,
                                    const bsattn_meta *meta, int32_t *err_flag, void *stream);

/*
 * bsattn_fwd -- block-sparse attention forward.
 *
 * For each head h, sequence b and query row i (tile m = i / 128), the allowed
 * key set is every key j < seqlen_k(b) of the tiles in the full list of row
 * (b, h, m), plus every key of the tiles in its mask list that passes the token
 * predicate of bsattn_build_meta.  Then, with s_j = softmax_scale * q_i . k_j,
 *   lse_i = ln(sum_j exp(s_j)),  out_i = sum_j exp(s_j - lse_i) v_j,
 * and an empty key set gives out_i = 0, lse_i = -inf.  Accumulation is fp32;
 * the probabilities are rounded to bf16 before the P.V product.
 *
 * q             device bf16, batched [B, seqlen_q, H, D], varlen [seqlen_q, H, D]
 *               (seqlen_q = total packed rows); contiguous, 16-byte aligned.
 * k, v          device bf16, same layout with seqlen_k.
 * B, H, D       D in {64, 128}; H equal for q and k/v.
 * cu_seqlens_*  varlen: device int32 [B+1]; batched: NULL.  A sequence whose
 *               offsets are negative, decrease, or reach past seqlen_q / seqlen_k
 *               (the packed row counts), or that has more KV tiles than
 *               meta->num_n while kv_valid_len is given, is skipped: none of its
 *               out / lse rows is written and BSATTN_FLAG_BAD_SEQLENS is set.
 * meta          lists as written by bsattn_build_meta (or the caller, same format;
 *               indices out of range are skipped and flagged).
 * kv_valid_len, kind, mp   as for bsattn_build_meta (applied on mask-list tiles).
 * softmax_scale > 0.
 * out           device, same shape as q; element type out_dtype.
 * out_dtype     BSATTN_OUT_BF16 or BSATTN_OUT_F32.
 * workspace     optional device scratch of at least bsattn_fwd_workspace_size() bytes,
 *               16-byte aligned, contents need not be initialised.  With it, a
 *               scheduling pass orders the work units (pairs of Q tiles of one head)
 *               by decreasing work and the persistent CTAs claim them in that order
 *               (longest-processing-time list scheduling); without it (NULL), CTAs take
 *               units by a fixed stride.  Results are identical either way.  Two calls
 *               that may run concurrently must not share a workspace.
 * lse           device fp32, batched [B, H, seqlen_q], varlen [H, seqlen_q].
 * err_flag      optional device int32 word.
 */
bsattn_status bsattn_fwd(const void *q, const void *k, const void *v, int32_t B, int32_t seqlen_q,
                         int32_t seqlen_k, int32_t H, int32_t D, const int32_t *cu_seqlens_q,
                         const int32_t *cu_seqlens_k, const bsattn_meta *meta,
                         const int32_t *kv_valid_len, bsattn_mask_kind kind,
                         const bsattn_mask_params *mp, float softmax_scale, void *out,
                         bsattn_out_dtype out_dtype, float *lse, void *workspace,
                         size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * bsattn_fwd_proxy -- block-sparse forward with proxy compensation ("feat(prims-ts):
 * support proxy-compensated block-sparse attention", FlashInfer #4872: selected
 * blocks stay exact; each omitted KV block is represented by its mean-K and
 * summed-V summaries, and the softmax denominator counts the block's true number
 * of keys).  Batched, mask kind none (the page's proxy mode needs a dense mask),
 * no kv_valid_len.  For query row i of sequence b, head h, Q tile m:
 *   E = keys j < seqlen_k of the tiles in the lists of (b, h, m)  (exact),
 *   O = KV tiles n < num_n whose bit is clear in sel_words row (b, h, m) (omitted),
 *   s_j = scale q_i.k_j,  t_n = scale q_i.k_sum[b, n, h],  w_n = keys of tile n,
 *   den = sum_E exp(s_j) + sum_O w_n exp(t_n),
 *   out_i = (sum_E exp(s_j) v_j + sum_O exp(t_n) v_sum[b, n, h]) / den,
 *   lse_i = ln(den).
 * The exact lists and sel_words describe the same selection (e.g. lists from
 * bsattn_build_meta with kind none and the same map, and the bitmask form of that
 * map); a tile in the lists but not in sel_words would be counted twice.
 *
 * sel_words      device uint32 [B * H * num_m][words_per_row], bit n % 32 of word
 *                n / 32 = tile n is computed exactly; words_per_row >= ceil(num_n / 32).
 * k_sum, v_sum   device bf16 [B, num_n, H, D], 16-byte aligned (bsattn_kv_summaries).
 * Other arguments as for bsattn_fwd.  Varlen -> BSATTN_ERR_UNSUPPORTED.
 */
bsattn_status bsattn_fwd_proxy(const void *q, const void *k, const void *v, int32_t B,
                               int32_t seqlen_q, int32_t seqlen_k, int32_t H, int32_t D,
                               const bsattn_meta *meta, const uint32_t *sel_words,
                               int32_t words_per_row, const void *k_sum, const void *v_sum,
                               float softmax_scale, void *out, bsattn_out_dtype out_dtype, float *lse,
                               void *workspace, size_t workspace_bytes, int32_t *err_flag,
                               void *stream);

/*
 * bsattn_fwd_workspace_size -- bytes of workspace bsattn_fwd can use for this
 * metadata (0 when the problem is too large for the scheduling pass, in which
 * case bsattn_fwd ignores any workspace and uses the fixed stride).
 */
bsattn_status bsattn_fwd_workspace_size(const bsattn_meta *meta, size_t *bytes);

/*
 * bsattn_fwd_static_scratch -- bsattn_fwd with the scheduling workspace taken
 * from a fixed scratch array inside the library, for callers that cannot
 * allocate device memory at call time: a C or C++ host program that has no
 * device allocator of its own to hand a workspace from, or a latency-critical
 * loop that must not call cudaMalloc / cudaFree (cudaFree synchronises the
 * device).  This call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).  It is an engineering addition: the pages describe no
 * counterpart.
 *
 * Arguments are those of bsattn_fwd without workspace / workspace_bytes, with
 * the same meaning, layout, ownership and results.
 *
 * Capacity: problems of up to BSATTN_STATIC_SCRATCH_UNITS work units
 * (units = H * ceil(total Q tiles / 2)); larger ones return
 * BSATTN_ERR_CAPACITY before any CUDA call (use bsattn_fwd with a workspace).
 * Setup: the first call on each device resolves the scratch array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  The address is kept per CUDA context: after
 * cudaDeviceReset (or any re-creation of the device's primary context) the next
 * call resolves it again, so that first call after a reset also belongs before
 * any capture.  Zeroing: the claim counter in the scratch is
 * reset on the stream by the scheduling pass of every call.
 * Concurrency: all calls on one device share the one scratch array, so calls
 * that may overlap (different streams, or threads without ordering) race on it
 * and must not be issued.
 */
#define BSATTN_STATIC_SCRATCH_UNITS 65536
bsattn_status bsattn_fwd_static_scratch(const void *q, const void *k, const void *v, int32_t B,
                                        int32_t seqlen_q, int32_t seqlen_k, int32_t H, int32_t D,
                                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                        const bsattn_meta *meta, const int32_t *kv_valid_len,
                                        bsattn_mask_kind kind, const bsattn_mask_params *mp,
                                        float softmax_scale, void *out, bsattn_out_dtype out_dtype,
                                        float *lse, int32_t *err_flag, void *stream);

/*
 * bsattn_bwd -- gradients of bsattn_fwd with respect to q, k and v, for batched
 * and varlen metadata.  The backward is the step the pages report as missing
 * for training ("[CuTe,Flex] varlen blocksparsity", flash-attention #2224:
 * backward not yet supported with block sparsity and would need transposed
 * metadata; "[feat] VSA-256 fastpath", FastVideo #1354: forward only).
 * With P_ij the forward's probabilities (0 outside row i's allowed set A_i, the
 * set bsattn_fwd sums over) and dO the upstream gradient of out:
 *   D_i = sum_d dO_id out_id,   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i),
 *   dv_j = sum_i P_ij dO_i,  dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i.
 * P is recomputed as exp(scale q_i.k_j - lse_i) from the forward's lse; a row
 * with an empty key set (lse = -inf) contributes nothing.  Products run on the
 * tensor cores in bf16 (P and dS rounded to bf16) with fp32 accumulation; the
 * result does not depend on the order in which the KV tiles are processed.
 *
 * q, k, v, B, seqlen_q, seqlen_k, H, D, cu_seqlens_q, cu_seqlens_k, meta,
 *               kv_valid_len, kind, mp, softmax_scale: exactly those given to
 *               bsattn_fwd (layouts, varlen packing and checks as there).
 * out, lse      the forward's results for these arguments: out in the layout of
 *               q in out_dtype; lse fp32 batched [B, H, seqlen_q], varlen
 *               [H, total q rows].
 * dout          device bf16, layout of q, 16-byte aligned.
 * dq, dk, dv    device outputs in the layouts of q, k, v, grad_dtype (fp32 or
 *               bf16), 16-byte aligned; every row of a sequence the metadata
 *               describes is written (rows whose key or query set is empty get 0).
 * workspace     device, 256-byte aligned, at least bsattn_bwd_workspace_size
 *               bytes; overwritten; needs no zeroing.
 * err_flag      optional device int32 word: BSATTN_FLAG_BAD_INDEX when a list
 *               entry lies outside [0, num_n(b)) (skipped), a count outside
 *               [0, num_n(b)] (clamped) or a row lists a tile twice;
 *               BSATTN_FLAG_BAD_SEQLENS when a varlen sequence's offsets disagree
 *               with the metadata or reach past the packed rows (its rows are not
 *               written);
 *               BSATTN_FLAG_TIMEOUT as for bsattn_fwd.
 * D other than 64 or 128 -> BSATTN_ERR_UNSUPPORTED.
 * Asynchronous on `stream`; the arrays must stay valid until it completes.
 */
bsattn_status bsattn_bwd(const void *q, const void *k, const void *v, const void *out,
                         bsattn_out_dtype out_dtype, const float *lse, const void *dout, int32_t B,
                         int32_t seqlen_q, int32_t seqlen_k, int32_t H, int32_t D,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                         const bsattn_meta *meta, const int32_t *kv_valid_len, bsattn_mask_kind kind,
                         const bsattn_mask_params *mp, float softmax_scale, void *dq, void *dk, void *dv,
                         bsattn_out_dtype grad_dtype, void *workspace, size_t workspace_bytes,
                         int32_t *err_flag, void *stream);

/*
 * bsattn_bwd_workspace_size -- bytes of workspace bsattn_bwd needs for this
 * metadata: per KV tile and head (B * num_n per head; varlen: num_n is the
 * kv_valid_len stride) two list counts and an order slot (12 bytes); per entry
 * of the forward's index lists two KV-major list entries and a selection code
 * (9 bytes); B + 1 prefix entries; two fp32 values per Q tile row (1 KB per Q
 * tile and head); each of the nine regions rounded up to 256 bytes.
 */
bsattn_status bsattn_bwd_workspace_size(const bsattn_meta *meta, size_t *bytes);

/*
 * bsattn_testing_set_wait_limit -- testing hook, not for production use; the
 * pages have no counterpart.  Sets the number of SM clock cycles after which a
 * pipeline wait (an mbarrier wait between the roles of a CTA) of later
 * bsattn_fwd and bsattn_fwd_static_scratch launches from this process gives up.
 * A limit below the default runs a build of the same kernel whose waits poll
 * without suspending the thread (a suspended wait could outlast a short limit);
 * the default build is used otherwise.  A CTA whose wait gives up sets
 * BSATTN_FLAG_TIMEOUT in err_flag, waits for the copies and tensor-core products
 * it has already issued, frees its tensor memory and exits; out / lse are then
 * incomplete.  cycles <= 0 restores the default of 2^31 cycles (about one
 * second at 2 GHz).  bsattn_fwd_proxy, and bsattn_fwd with metadata listed
 * per sparse block, keep the default.  The setting is process-wide and read
 * when a call is made; always BSATTN_OK.
 */
bsattn_status bsattn_testing_set_wait_limit(long long cycles);

/* Human-readable name of a status code (static string). */
const char *bsattn_status_string(bsattn_status status);

/* BSATTN_ABI_VERSION of the loaded library. */
int32_t bsattn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSATTN_H */
