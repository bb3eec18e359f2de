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
// partial rows that have a key in their range in float4 columns, four parts' loads in flight
// before their FMAs.  Bytes per row: S (d + 1) 4 read (less the skipped parts) +
// d (2 or 4) + 4 written.
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
    const long long r = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int d4 = d >> 2;
    // LSE = M + ln sum_s e^{LSE_s - M}, M the largest LSE_s; lane l reads parts l, l+32, ...
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
    // the column loop runs the same number of times on every lane (its shuffles need all 32)
    for (int c0 = 0; c0 < d4; c0 += 32) {
        const int c = c0 + lane;
        const bool col = c < d4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lse != -INFINITY) {
            for (int s0 = 0; s0 < S; s0 += 32) {
                // parts s0 .. s0+31: weight of part s0+l held by lane l, 0 for an empty part
                const int sl = s0 + lane;
                const float ls = sl < S ? LSE_parts[static_cast<size_t>(sl) * rows + r] : -INFINITY;
                const float wl = (ls == -INFINITY) ? 0.f : expf(ls - lse);
                unsigned live = __ballot_sync(0xffffffffu, wl != 0.f);
                // four parts at a time: their loads are issued before any of their FMAs
                while (live) {
                    int idx[4];
                    float w[4];
                    float4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        idx[u] = live ? __ffs(live) - 1 : -1;
                        if (live) live &= live - 1;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        w[u] = __shfl_sync(0xffffffffu, wl, idx[u] < 0 ? 0 : idx[u]);
                        v[u] = (idx[u] < 0 || !col) ? make_float4(0.f, 0.f, 0.f, 0.f)
                                          : reinterpret_cast<const float4 *>(
                                                O_parts + (static_cast<size_t>(s0 + idx[u]) * rows + r) * d)[c];
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (idx[u] < 0) continue;
                        acc.x = fmaf(w[u], v[u].x, acc.x);
                        acc.y = fmaf(w[u], v[u].y, acc.y);
                        acc.z = fmaf(w[u], v[u].z, acc.z);
                        acc.w = fmaf(w[u], v[u].w, acc.w);
                    }
                }
            }
        }
        if (!col) continue;
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

}  // namespace merge

cudaError_t launch_merge(const float *O_parts, const float *LSE_parts, int S, long long rows, int d,
                         void *O, bool out_bf16, float *LSE, cudaStream_t stream) {
    // one warp per row, every row in flight at once (the hardware schedules the waves)
    const long long blocks = (rows + merge::WARPS - 1) / merge::WARPS;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int grid = static_cast<int>(blocks);
    if (out_bf16)
        merge::merge_kernel<true><<<grid, merge::WARPS * 32, 0, stream>>>(O_parts, LSE_parts, S, rows,
                                                                          d, O, LSE);
    else
        merge::merge_kernel<false><<<grid, merge::WARPS * 32, 0, stream>>>(O_parts, LSE_parts, S,
                                                                           rows, d, O, LSE);
    return cudaGetLastError();
}

}  // namespace fa
