// fa_merge.cu -- K6: merge of split-KV partial results, fp32 on the CUDA cores.
//
// Method (FlashAttention DAC'24 reading note, paper.adslab.icu, Methods, the update of m, l and O
// after each block): two results over disjoint key sets combine by rescaling each with e^{m_s - m}
// and its sum l_s.  With each partial already normalised and carried as LSE_s = m_s + ln l_s, the
// same update over S partials reads
//     LSE = ln sum_s e^{LSE_s},   O = sum_s e^{LSE_s - LSE} O_s,
// which is why a plain average of the block results is not enough (FlashAttention note,
// paweldubiel.com: the per-block outputs need their normalisers).  A partial with LSE_s = -inf
// (no allowed key in its range) has weight 0 and is not read.
//
// HBM-bound: one warp per query row; the lanes first reduce the S log-sum-exps, then stream the
// S partial rows in float4 columns.  Bytes per row: S (d + 1) 4 read (less the skipped parts) +
// d (2 or 4) + 4 written.
#include <algorithm>
#include <cmath>

#include <cuda_bf16.h>

#include "fa_internal.h"

namespace fa {
namespace merge {

constexpr int WARPS = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(WARPS * 32)
    merge_kernel(const float *__restrict__ O_parts, const float *__restrict__ LSE_parts, int S,
                 long long rows, int d, void *__restrict__ O, float *__restrict__ LSE) {
    const int lane = threadIdx.x & 31;
    const long long warps_total = static_cast<long long>(gridDim.x) * WARPS;
    const int d4 = d >> 2;
    for (long long r = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5); r < rows;
         r += warps_total) {
        // LSE = M + ln sum_s e^{LSE_s - M}, M the largest finite LSE_s
        float mx = -INFINITY;
        for (int s = lane; s < S; s += 32) mx = fmaxf(mx, LSE_parts[static_cast<size_t>(s) * rows + r]);
        mx = warp_max(mx);
        float sum = 0.f;
        if (mx != -INFINITY)
            for (int s = lane; s < S; s += 32)
                sum += expf(LSE_parts[static_cast<size_t>(s) * rows + r] - mx);
        sum = warp_sum(sum);
        const float lse = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
        if (lane == 0) LSE[r] = lse;
        for (int c = lane; c < d4; c += 32) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lse != -INFINITY) {
                for (int s = 0; s < S; ++s) {
                    const float ls = LSE_parts[static_cast<size_t>(s) * rows + r];
                    if (ls == -INFINITY) continue;
                    const float w = expf(ls - lse);
                    const float4 v = reinterpret_cast<const float4 *>(
                        O_parts + (static_cast<size_t>(s) * rows + r) * d)[c];
                    acc.x = fmaf(w, v.x, acc.x);
                    acc.y = fmaf(w, v.y, acc.y);
                    acc.z = fmaf(w, v.z, acc.z);
                    acc.w = fmaf(w, v.w, acc.w);
                }
            }
            if constexpr (OUT_BF16) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
                __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
                uint2 u;
                u.x = *reinterpret_cast<uint32_t *>(&lo);
                u.y = *reinterpret_cast<uint32_t *>(&hi);
                reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(O) + static_cast<size_t>(r) * d)[c] = u;
            } else {
                reinterpret_cast<float4 *>(static_cast<float *>(O) + static_cast<size_t>(r) * d)[c] = acc;
            }
        }
    }
}

}  // namespace merge

cudaError_t launch_merge(const float *O_parts, const float *LSE_parts, int S, long long rows, int d,
                         void *O, bool out_bf16, float *LSE, cudaStream_t stream) {
    const long long blocks_needed = (rows + merge::WARPS - 1) / merge::WARPS;
    // grid-stride: a few waves of 8-warp blocks on every SM
    const int grid = static_cast<int>(std::min<long long>(blocks_needed, 8LL * num_sms()));
    if (out_bf16)
        merge::merge_kernel<true><<<grid, merge::WARPS * 32, 0, stream>>>(O_parts, LSE_parts, S, rows,
                                                                          d, O, LSE);
    else
        merge::merge_kernel<false><<<grid, merge::WARPS * 32, 0, stream>>>(O_parts, LSE_parts, S,
                                                                           rows, d, O, LSE);
    return cudaGetLastError();
}

}  // namespace fa
