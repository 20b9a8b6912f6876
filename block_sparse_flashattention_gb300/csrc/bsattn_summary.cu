// K/V summaries of the KV tiles for proxy compensation ("feat(prims-ts): support
// proxy-compensated block-sparse attention", FlashInfer #4872: one arithmetic-mean
// K summary and one summed-V summary per semantic KV block).
//
// For sequence b, KV tile n and head h, over the tile's keys j in
// [128 n, min(128 n + 128, seqlen_k)):
//   k_sum[b, n, h, :] = mean_j K[b, j, h, :],   v_sum[b, n, h, :] = sum_j V[b, j, h, :]
// accumulated in fp32 in ascending j and rounded to bf16 (RNE).  HBM-bound: K and
// V are read once and the summaries written once.
#include <cuda_bf16.h>

#include "bsattn_internal.h"

namespace bsattn {

namespace {

// One warp per (b, n, h); lane l handles the bf16 pairs l, l + 32, ... of the row.
__global__ void __launch_bounds__(256) bsattn_kv_summary_kernel(const __nv_bfloat162 *k,
                                                                const __nv_bfloat162 *v, int B, int S,
                                                                int H, int D, int nn,
                                                                __nv_bfloat162 *k_sum,
                                                                __nv_bfloat162 *v_sum) {
    const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= (long long)B * nn * H) return;
    const int h = (int)(w % H);
    const long long bn = w / H;
    const int n = (int)(bn % nn), b = (int)(bn / nn);
    const int j0 = n * kTile, j1 = min(j0 + kTile, S);
    const int pairs = D / 2;
    const float cnt = (float)(j1 - j0);
    for (int c = lane; c < pairs; c += 32) {
        float ka = 0.f, kb = 0.f, va = 0.f, vb = 0.f;
        for (int j = j0; j < j1; ++j) {
            const long long at = (((long long)b * S + j) * H + h) * pairs + c;
            const float2 kf = __bfloat1622float2(k[at]);
            const float2 vf = __bfloat1622float2(v[at]);
            ka += kf.x;
            kb += kf.y;
            va += vf.x;
            vb += vf.y;
        }
        const long long o = (((long long)b * nn + n) * H + h) * pairs + c;
        k_sum[o] = __floats2bfloat162_rn(__fdiv_rn(ka, cnt), __fdiv_rn(kb, cnt));
        v_sum[o] = __floats2bfloat162_rn(va, vb);
    }
}

}  // namespace

cudaError_t launch_kv_summary(const void *k, const void *v, int B, int S, int H, int D, void *k_sum,
                              void *v_sum, cudaStream_t stream) {
    const int nn = (S + kTile - 1) / kTile;
    const long long warps = (long long)B * nn * H;
    if (warps <= 0) return cudaSuccess;
    const long long blocks = (warps + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    bsattn_kv_summary_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat162 *>(k), static_cast<const __nv_bfloat162 *>(v), B, S, H, D, nn,
        static_cast<__nv_bfloat162 *>(k_sum), static_cast<__nv_bfloat162 *>(v_sum));
    return cudaGetLastError();
}

}  // namespace bsattn
