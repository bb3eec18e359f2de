// fa_simt_fp32.cu -- K5: exact attention forward and backward in fp32 on the CUDA cores.
//
// For checks that need fp32 accuracy (tensor-core tf32 keeps a 10-bit mantissa).  One warp per
// output row; each lane holds up to four of the d <= 128 features (lane, lane + 32, ...), dot
// products are reduced across the warp.  The forward is the per-key form of the online-softmax
// recurrence (FlashAttention note, paweldubiel.com: m, l = sum e^{s-m}, u = sum e^{s-m} v,
// rescaled by e^{m-m'} when the max grows; result u / l).  The backward follows the formulas of
// the "Attention's hidden recurrence" blog (mzeromiko), section "standard attention / backward":
// D_i = <dO_i, O_i>, dS_ij = P_ij (<dO_i, v_j> - D_i), with P_ij = exp(s_ij - LSE_i) recomputed.
// dQ rows and dK/dV rows are written by separate warps, so nothing is accumulated atomically.
#include <cmath>

#include "fa_internal.h"

namespace fa {
namespace simt {

constexpr int WARPS = 8;
constexpr int MAXE = 4;   // features per lane (d <= 128)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ void load_row(const float *p, int d, int lane, float (&x)[MAXE]) {
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        x[e] = c < d ? p[c] : 0.f;
    }
}

__device__ __forceinline__ float dot_row(const float (&x)[MAXE], const float *p, int d, int lane) {
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        if (c < d) acc = fmaf(x[e], p[c], acc);
    }
    return warp_sum(acc);
}

// grid: (ceil(N / WARPS), B * Hq); one warp per query row.
__global__ void __launch_bounds__(WARPS * 32) fwd_kernel(const float *__restrict__ Q,
                                                         const float *__restrict__ K,
                                                         const float *__restrict__ V,
                                                         float *__restrict__ O,
                                                         float *__restrict__ LSE, int Hq, int Hkv,
                                                         int N, int d, int causal, float scale) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * WARPS + (threadIdx.x >> 5);
    const int bh = blockIdx.y;
    if (i >= N) return;
    const int b = bh / Hq, hq = bh % Hq, hk = hq / (Hq / Hkv);
    const size_t nd = static_cast<size_t>(N) * d;
    const float *q = Q + bh * nd + static_cast<size_t>(i) * d;
    const float *k = K + (static_cast<size_t>(b) * Hkv + hk) * nd;
    const float *v = V + (static_cast<size_t>(b) * Hkv + hk) * nd;
    float qr[MAXE], acc[MAXE];
    load_row(q, d, lane, qr);
#pragma unroll
    for (int e = 0; e < MAXE; ++e) acc[e] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int jend = causal ? i + 1 : N;
    for (int j = 0; j < jend; ++j) {
        const float s = scale * dot_row(qr, k + static_cast<size_t>(j) * d, d, lane);
        const float mn = fmaxf(m, s);
        const float alpha = expf(m - mn);   // 0 on the first key (m = -inf)
        const float p = expf(s - mn);
        l = l * alpha + p;
        const float *vj = v + static_cast<size_t>(j) * d;
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
            const int c = lane + 32 * e;
            acc[e] = acc[e] * alpha + (c < d ? p * vj[c] : 0.f);
        }
        m = mn;
    }
    float *o = O + bh * nd + static_cast<size_t>(i) * d;
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        if (c < d) o[c] = acc[e] / l;
    }
    if (lane == 0) LSE[static_cast<size_t>(bh) * N + i] = m + logf(l);
}

// D_i = <dO_i, O_i>; grid (ceil(N / WARPS), B * Hq).
__global__ void __launch_bounds__(WARPS * 32) pre_kernel(const float *__restrict__ O,
                                                         const float *__restrict__ dO,
                                                         float *__restrict__ Dvec, int N, int d) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (i >= N) return;
    const size_t row = static_cast<size_t>(blockIdx.y) * N + i;
    float x[MAXE];
    load_row(dO + row * d, d, lane, x);
    const float D = dot_row(x, O + row * d, d, lane);
    if (lane == 0) Dvec[row] = D;
}

// dQ_i = scale sum_j dS_ij k_j; grid (ceil(N / WARPS), B * Hq).
__global__ void __launch_bounds__(WARPS * 32) dq_kernel(const float *__restrict__ Q,
                                                        const float *__restrict__ K,
                                                        const float *__restrict__ V,
                                                        const float *__restrict__ dO,
                                                        const float *__restrict__ LSE,
                                                        const float *__restrict__ Dvec,
                                                        float *__restrict__ dQ, int Hq, int Hkv,
                                                        int N, int d, int causal, float scale) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * WARPS + (threadIdx.x >> 5);
    const int bh = blockIdx.y;
    if (i >= N) return;
    const int b = bh / Hq, hq = bh % Hq, hk = hq / (Hq / Hkv);
    const size_t nd = static_cast<size_t>(N) * d;
    const size_t row = static_cast<size_t>(bh) * N + i;
    const float *k = K + (static_cast<size_t>(b) * Hkv + hk) * nd;
    const float *v = V + (static_cast<size_t>(b) * Hkv + hk) * nd;
    float qr[MAXE], dor[MAXE], acc[MAXE];
    load_row(Q + row * d, d, lane, qr);
    load_row(dO + row * d, d, lane, dor);
#pragma unroll
    for (int e = 0; e < MAXE; ++e) acc[e] = 0.f;
    const float lse = LSE[row], Di = Dvec[row];
    const int jend = causal ? i + 1 : N;
    for (int j = 0; j < jend; ++j) {
        const float *kj = k + static_cast<size_t>(j) * d;
        const float p = expf(scale * dot_row(qr, kj, d, lane) - lse);
        const float ds = p * (dot_row(dor, v + static_cast<size_t>(j) * d, d, lane) - Di);
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
            const int c = lane + 32 * e;
            if (c < d) acc[e] = fmaf(ds, kj[c], acc[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        if (c < d) dQ[row * d + c] = scale * acc[e];
    }
}

// dK_j, dV_j summed over the query heads of the group; grid (ceil(N / WARPS), B * Hkv).
__global__ void __launch_bounds__(WARPS * 32) dkv_kernel(const float *__restrict__ Q,
                                                         const float *__restrict__ K,
                                                         const float *__restrict__ V,
                                                         const float *__restrict__ dO,
                                                         const float *__restrict__ LSE,
                                                         const float *__restrict__ Dvec,
                                                         float *__restrict__ dK,
                                                         float *__restrict__ dV, int Hq, int Hkv,
                                                         int N, int d, int causal, float scale) {
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * WARPS + (threadIdx.x >> 5);
    const int bk = blockIdx.y;
    if (j >= N) return;
    const int b = bk / Hkv, hk = bk % Hkv, G = Hq / Hkv;
    const size_t nd = static_cast<size_t>(N) * d;
    const size_t krow = static_cast<size_t>(bk) * N + j;
    float kr[MAXE], vr[MAXE], ak[MAXE], av[MAXE];
    load_row(K + krow * d, d, lane, kr);
    load_row(V + krow * d, d, lane, vr);
#pragma unroll
    for (int e = 0; e < MAXE; ++e) ak[e] = av[e] = 0.f;
    for (int g = 0; g < G; ++g) {
        const size_t bh = static_cast<size_t>(b) * Hq + hk * G + g;
        const float *q = Q + bh * nd, *dor = dO + bh * nd;
        for (int i = causal ? j : 0; i < N; ++i) {
            const size_t row = bh * N + i;
            const float *qi = q + static_cast<size_t>(i) * d, *doi = dor + static_cast<size_t>(i) * d;
            const float p = expf(scale * dot_row(kr, qi, d, lane) - LSE[row]);
            const float ds = p * (dot_row(vr, doi, d, lane) - Dvec[row]);
#pragma unroll
            for (int e = 0; e < MAXE; ++e) {
                const int c = lane + 32 * e;
                if (c < d) {
                    av[e] = fmaf(p, doi[c], av[e]);
                    ak[e] = fmaf(ds, qi[c], ak[e]);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        if (c < d) {
            dK[krow * d + c] = scale * ak[e];
            dV[krow * d + c] = av[e];
        }
    }
}

}  // namespace simt

cudaError_t launch_fwd_fp32(const Problem &p, const float *Q, const float *K, const float *V,
                            float *O, float *LSE, cudaStream_t stream) {
    if (p.B * p.Hq > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid((p.N + simt::WARPS - 1) / simt::WARPS, p.B * p.Hq);
    simt::fwd_kernel<<<grid, simt::WARPS * 32, 0, stream>>>(Q, K, V, O, LSE, p.Hq, p.Hkv, p.N, p.d,
                                                            p.causal, p.scale);
    return cudaGetLastError();
}

cudaError_t launch_bwd_fp32(const Problem &p, const float *Q, const float *K, const float *V,
                            const float *O, const float *dO, const float *LSE, float *dQ,
                            float *dK, float *dV, float *D, cudaStream_t stream) {
    if (p.B * p.Hq > 65535) return cudaErrorInvalidConfiguration;
    const unsigned gx = (p.N + simt::WARPS - 1) / simt::WARPS;
    simt::pre_kernel<<<dim3(gx, p.B * p.Hq), simt::WARPS * 32, 0, stream>>>(O, dO, D, p.N, p.d);
    simt::dq_kernel<<<dim3(gx, p.B * p.Hq), simt::WARPS * 32, 0, stream>>>(
        Q, K, V, dO, LSE, D, dQ, p.Hq, p.Hkv, p.N, p.d, p.causal, p.scale);
    simt::dkv_kernel<<<dim3(gx, p.B * p.Hkv), simt::WARPS * 32, 0, stream>>>(
        Q, K, V, dO, LSE, D, dK, dV, p.Hq, p.Hkv, p.N, p.d, p.causal, p.scale);
    return cudaGetLastError();
}

}  // namespace fa
