// fa_fwd_tf32x3_sm103a.cu -- K9: fp32 forward on the tensor cores with three TF32 products.
//
// The same method as the bf16 forward (FlashAttention DAC'24 reading note, paper.adslab.icu,
// Methods: a query tile stays on chip while key/value blocks stream past with the running
// max / sum update; deferred normalisation as in the FlashAttention note, paweldubiel.com),
// for fp32 inputs and outputs.  Every fp32 operand x is split as x = hi + lo with hi = x with
// its 13 low mantissa bits cleared (exactly a TF32 value) and lo = x - hi (exact in fp32), and
// each product A B is formed as hi(A) hi(B) + hi(A) lo(B) + lo(A) hi(B) in fp32 accumulators
// (tcgen05 kind::tf32); the dropped lo(A) lo(B) and the 10-bit mantissa of lo leave a relative
// error near 2^-21 per product, so the result agrees with fp32 arithmetic to about 1e-6.
//
// K9a (split_kernel) writes hi / lo copies of Q and K and transposed copies of V to a workspace
// (transposed so that both operands of P V are K-major: TF32 operands are used K-major only).
// K9b: one CTA per 128-row query tile, d = 64, 32-key blocks; 192 threads:
//   warps 0-3 : softmax warps (thread = query row = TMEM lane)
//   warp 4    : TMA producer (Q hi / lo once, K and V^T hi / lo per block, 3 stages)
//   warp 5    : TMEM allocator and single-thread MMA issuer
// TMEM: S double-buffered at columns [0, 32) and [32, 64), so S of block j + 1 is computed while
// the softmax warps work on block j; P V of one block at [64, 128).  P (split into hi / lo) is
// staged in shared memory as the K-major A operand of P V.  Each block's P V starts a fresh
// accumulator and the softmax warps add it into fp32 register sums: the tensor core's
// accumulation error grows with the number of MMAs chained into one accumulator, and this keeps
// the chain at 12.  The max is rescaled lazily (threshold 8, log2 units) on the register sums;
// P is kept in three TF32 parts here, so the size of the weights does not limit its precision.
#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_tf32.cuh"

namespace fa {
namespace tf32x3 {

constexpr int D = 64;
constexpr int BM = 128, BN = 32;
constexpr int NUM_THREADS = 192;
constexpr int WARP_TMA = 4, WARP_MMA = 5;
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr float LN2 = 0.693147180559945309f;

// Shared memory (all tiles 1024-byte aligned, 128-byte swizzled rows of 32 fp32):
constexpr int Q_CHUNK = BM * 128;               // 128 rows x 32 fp32
constexpr int Q_BYTES = 2 * Q_CHUNK;            // d = 64: two chunks
constexpr int K_CHUNK = BN * 128;               // 32 rows x 32 fp32
constexpr int K_BYTES = 2 * K_CHUNK;
constexpr int VT_BYTES = D * 128;               // V^T block: 64 rows (d) x 32 keys
constexpr int P_BYTES = BM * 128;               // P block: 128 rows x 32 keys
constexpr int QH_OFF = 0, QL_OFF = Q_BYTES;
constexpr int NST = 3;                          // K / V^T ring stages
constexpr int STAGE_OFF = 2 * Q_BYTES;          // [NST stages][Kh | Kl | Vth | Vtl]
constexpr int STAGE_BYTES = 2 * K_BYTES + 2 * VT_BYTES;
constexpr int PH_OFF = STAGE_OFF + NST * STAGE_BYTES, PL_OFF = PH_OFF + P_BYTES;
constexpr int BAR_OFF = PL_OFF + P_BYTES;
// q_full, kv_full[NST], kv_empty[NST], s_full[2], p_full, o_done, mma_done
constexpr int NBARS = 1 + 2 * NST + 2 + 3;
constexpr int TMEM_OFF = BAR_OFF + NBARS * 8;
constexpr int ABORT_OFF = TMEM_OFF + 8;
constexpr int SMEM_BYTES = ABORT_OFF + 8 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
// S of block j in buffer j & 1 at T_S + 32 (j & 1); P V of one block (a fresh accumulator) at T_O
constexpr uint32_t T_S = 0, T_O = 64;

// K9a: Qh, Ql [BH, N, 64]; Kh, Kl [BHkv, N, 64]; Vth, Vtl [BHkv, 64, Np] (keys Np >= N zero).
__global__ void __launch_bounds__(256) split_kernel(const float *__restrict__ Q, const float *__restrict__ K,
                                                    const float *__restrict__ V, float *__restrict__ ws,
                                                    long long nq_el, long long nk_el, int N, int Np,
                                                    long long nvt_el) {
    float *Qh = ws, *Ql = Qh + nq_el, *Kh = Ql + nq_el, *Kl = Kh + nk_el, *Vth = Kl + nk_el,
          *Vtl = Vth + nvt_el;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < nq_el; t += stride) {
        const float x = Q[t], h = tf32_hi(x);
        Qh[t] = h;
        Ql[t] = x - h;
    }
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < nk_el; t += stride) {
        const float x = K[t], h = tf32_hi(x);
        Kh[t] = h;
        Kl[t] = x - h;
    }
    // V^T: element (bkv, c, n) of [BHkv, 64, Np] from V (bkv, n, c); n >= N is zero
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < nvt_el; t += stride) {
        const int n = static_cast<int>(t % Np);
        const long long rest = t / Np;
        const int c = static_cast<int>(rest % D);
        const long long bkv = rest / D;
        const float x = n < N ? V[(bkv * N + n) * D + c] : 0.f, h = tf32_hi(x);
        Vth[t] = h;
        Vtl[t] = x - h;
    }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmQl,
                const __grid_constant__ CUtensorMap tmKh, const __grid_constant__ CUtensorMap tmKl,
                const __grid_constant__ CUtensorMap tmVh, const __grid_constant__ CUtensorMap tmVl,
                float *__restrict__ O, float *__restrict__ LSE, int Hq, int Hkv, int N,
                float scale_log2, unsigned *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    uint64_t *q_full = bars, *kv_full = bars + 1, *kv_empty = bars + 1 + NST;
    uint64_t *s_full = bars + 1 + 2 * NST, *p_full = s_full + 2, *o_done = p_full + 1;
    uint64_t *mma_done = o_done + 1;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + TMEM_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + ABORT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = blockIdx.x * BM;
    const int bh = blockIdx.y;
    const int bkv = (bh / Hq) * Hkv + (bh % Hq) / (Hq / Hkv);
    const int nkb_all = (N + BN - 1) / BN;
    const int nb = CAUSAL ? min(nkb_all, (min(q0 + BM, N) - 1) / BN + 1) : nkb_all;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(p_full, BM);
        mbar_init(o_done, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_holder, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == WARP_TMA) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2 * Q_BYTES);
            for (int ch = 0; ch < D / 32; ++ch) {
                tma_load_3d(smem + QH_OFF + ch * Q_CHUNK, &tmQh, ch * 32, q0, bh, q_full);
                tma_load_3d(smem + QL_OFF + ch * Q_CHUNK, &tmQl, ch * 32, q0, bh, q_full);
            }
            int issued = 0;
            for (int j = 0; j < nb; ++j) {
                const int st = j % NST;
                if (j >= NST && !mbar_wait(&kv_empty[st], (j / NST - 1) & 1, abort_flag, status)) break;
                mbar_arrive_expect_tx(&kv_full[st], STAGE_BYTES);
                uint8_t *base = smem + STAGE_OFF + st * STAGE_BYTES;
                for (int ch = 0; ch < D / 32; ++ch) {
                    tma_load_3d(base + ch * K_CHUNK, &tmKh, ch * 32, j * BN, bkv, &kv_full[st]);
                    tma_load_3d(base + K_BYTES + ch * K_CHUNK, &tmKl, ch * 32, j * BN, bkv, &kv_full[st]);
                }
                tma_load_3d(base + 2 * K_BYTES, &tmVh, j * BN, 0, bkv, &kv_full[st]);
                tma_load_3d(base + 2 * K_BYTES + VT_BYTES, &tmVl, j * BN, 0, bkv, &kv_full[st]);
                issued = j + 1;
            }
            if (*abort_flag) {
                for (int j = max(0, issued - NST); j < issued; ++j) mbar_drain(&kv_full[j % NST], (j / NST) & 1);
                mbar_drain(q_full, 0);
            }
        }
        tc_fence_before();
        __syncthreads();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_tf32(BM, BN);
            constexpr uint32_t IDESC_PV = idesc_tf32(BM, D);
            const uint64_t dqh = sdesc_sw128(smem_u32(smem + QH_OFF), 16, 1024);
            const uint64_t dql = sdesc_sw128(smem_u32(smem + QL_OFF), 16, 1024);
            const uint64_t dph = sdesc_sw128(smem_u32(smem + PH_OFF), 16, 1024);
            const uint64_t dpl = sdesc_sw128(smem_u32(smem + PL_OFF), 16, 1024);
            // S = Qh Kh + Qh Kl + Ql Kh of block j into buffer j & 1, over d = 64 (8 k-steps of 8)
            auto issue_s = [&](int j) -> bool {
                const int st = j % NST;
                if (!mbar_wait(&kv_full[st], (j / NST) & 1, abort_flag, status)) return false;
                tc_fence_after();
                const uint32_t base = smem_u32(smem + STAGE_OFF + st * STAGE_BYTES);
                const uint64_t dkh = sdesc_sw128(base, 16, 1024);
                const uint64_t dkl = sdesc_sw128(base + K_BYTES, 16, 1024);
                const uint32_t ts = tmem + T_S + 32 * (j & 1);
#pragma unroll
                for (int kk = 0; kk < D / 8; ++kk) {
                    const uint32_t oq = (kk >> 2) * Q_CHUNK + (kk & 3) * 32;
                    const uint32_t ok2 = (kk >> 2) * K_CHUNK + (kk & 3) * 32;
                    mma_tf32(ts, sdesc_add(dqh, oq), sdesc_add(dkh, ok2), IDESC_S, kk > 0);
                    mma_tf32(ts, sdesc_add(dqh, oq), sdesc_add(dkl, ok2), IDESC_S, 1u);
                    mma_tf32(ts, sdesc_add(dql, oq), sdesc_add(dkh, ok2), IDESC_S, 1u);
                }
                mma_commit(&s_full[j & 1]);
                return true;
            };
            bool ok = mbar_wait(q_full, 0, abort_flag, status);
            if (ok && nb > 0) ok = issue_s(0);
            for (int j = 0; j < nb && ok; ++j) {
                // S of block j + 1 overlaps the softmax of block j; its buffer held S of block
                // j - 1, read before p_full of block j - 1
                if (j + 1 < nb && !issue_s(j + 1)) { ok = false; break; }
                if (!mbar_wait(p_full, j & 1, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                const int st = j % NST;
                const uint32_t base = smem_u32(smem + STAGE_OFF + st * STAGE_BYTES);
                const uint64_t dvh = sdesc_sw128(base + 2 * K_BYTES, 16, 1024);
                const uint64_t dvl = sdesc_sw128(base + 2 * K_BYTES + VT_BYTES, 16, 1024);
                // P V of the block = Ph Vh + Ph Vl + Pl Vh over its 32 keys (4 k-steps of 8), in
                // a fresh accumulator that the softmax warps add into their fp32 sums
#pragma unroll
                for (int kk = 0; kk < BN / 8; ++kk) {
                    const uint32_t off = kk * 32;
                    mma_tf32(tmem + T_O, sdesc_add(dph, off), sdesc_add(dvh, off), IDESC_PV, kk > 0 ? 1u : 0u);
                    mma_tf32(tmem + T_O, sdesc_add(dph, off), sdesc_add(dvl, off), IDESC_PV, 1u);
                    mma_tf32(tmem + T_O, sdesc_add(dpl, off), sdesc_add(dvh, off), IDESC_PV, 1u);
                }
                mma_commit(o_done);
                mma_commit(&kv_empty[st]);
            }
            mma_commit(mma_done);
            mbar_drain(mma_done, 0);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == WARP_MMA) {
            __syncwarp();
            tc_fence_after();
            tmem_dealloc(tmem, 128);
        }
    } else {
        // ------------------------------------------------------------------ softmax warps
        const int row = warp * 32 + lane;
        const int rq = q0 + row;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        float m = -INFINITY, l = 0.f;
        float osum[D];                 // O (unnormalised) in fp32 registers, rounded to nearest
#pragma unroll
        for (int c = 0; c < D; ++c) osum[c] = 0.f;
        // adds the finished P V of the previous block (every lane loads: .sync.aligned)
        auto add_pv = [&]() {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_x32(tmem + lane_off + T_O + c0, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) osum[c0 + i] += __uint_as_float(o[i]);
            }
        };
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, status));
            if (!ok) break;
            tc_fence_after();
            uint32_t sraw[32];
            tmem_ld_x32(tmem + lane_off + T_S + 32 * (j & 1), sraw);
            float s[32];
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int key = j * BN + c;
                s[c] = ((CAUSAL && key > rq) || key >= N) ? -INFINITY : __uint_as_float(sraw[c]);
                mx = fmaxf(mx, s[c]);
            }
            // P V of the previous block must be done before P is restaged; its result joins the
            // sums at the scale it was computed with, before any rescale
            if (j > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag, status));
                if (!ok) break;
                tc_fence_after();
                add_pv();
            }
            const float m_blk = mx * scale_log2;
            if (m_blk > m + RESCALE_THRESHOLD) {
                const float alpha = ex2_approx(m - m_blk);
                l *= alpha;
                m = m_blk;
#pragma unroll
                for (int c = 0; c < D; ++c) osum[c] *= alpha;
            }
            const float m_sub = (m == -INFINITY) ? 0.f : m;
            uint8_t *ph = smem + PH_OFF + row * 128, *pl = smem + PL_OFF + row * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                float4 h, lo;
                float pv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    pv[k] = ex2_approx(fmaf(s[4 * u + k], scale_log2, -m_sub));
                    l += pv[k];
                }
                h = make_float4(tf32_hi(pv[0]), tf32_hi(pv[1]), tf32_hi(pv[2]), tf32_hi(pv[3]));
                lo = make_float4(pv[0] - h.x, pv[1] - h.y, pv[2] - h.z, pv[3] - h.w);
                const int sw = (u ^ (row & 7)) << 4;          // 128-byte swizzle of the row
                *reinterpret_cast<float4 *>(ph + sw) = h;
                *reinterpret_cast<float4 *>(pl + sw) = lo;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        if (ok && nb > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(o_done, (nb - 1) & 1, abort_flag, status));
            if (ok) {
                tc_fence_after();
                add_pv();
                const float inv = 1.f / l;
                float *orow = O + (static_cast<size_t>(bh) * N + rq) * D;
                if (rq < N) {
#pragma unroll
                    for (int u = 0; u < D / 4; ++u)
                        reinterpret_cast<float4 *>(orow)[u] =
                            make_float4(osum[4 * u] * inv, osum[4 * u + 1] * inv, osum[4 * u + 2] * inv,
                                        osum[4 * u + 3] * inv);
                }
                if (rq < N) LSE[static_cast<size_t>(bh) * N + rq] = (m + log2f(l)) * LN2;
            }
        }
        tc_fence_before();
        __syncthreads();
    }
}

}  // namespace tf32x3

size_t tf32x3_workspace_bytes(long long BH, long long BHkv, int N, int d) {
    const long long Np = (N + 31) / 32 * 32;
    return (2ull * BH * N * d + 2ull * BHkv * N * d + 2ull * BHkv * d * Np) * sizeof(float);
}

cudaError_t launch_tf32x3_split(const Problem &p, const float *Q, const float *K, const float *V,
                                float *ws, cudaStream_t stream) {
    const long long BH = 1LL * p.B * p.Hq, BHkv = 1LL * p.B * p.Hkv;
    const int Np = (p.N + 31) / 32 * 32;
    const long long nq = BH * p.N * p.d, nk = BHkv * p.N * p.d, nvt = BHkv * p.d * Np;
    long long grid = (std::max(nq, std::max(nk, nvt)) + 255) / 256;
    grid = std::min<long long>(std::max<long long>(grid, 1), 16LL * num_sms());
    tf32x3::split_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(Q, K, V, ws, nq, nk, p.N, Np, nvt);
    return cudaGetLastError();
}

cudaError_t launch_tf32x3_attn(const Problem &p, const CUtensorMap *maps, float *O, float *LSE,
                               unsigned *status, cudaStream_t stream) {
    if (p.d != tf32x3::D) return cudaErrorInvalidValue;
    auto kern = p.causal ? tf32x3::attn_kernel<true> : tf32x3::attn_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tf32x3::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long BH = 1LL * p.B * p.Hq;
    if (BH > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((p.N + tf32x3::BM - 1) / tf32x3::BM, static_cast<unsigned>(BH));
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    kern<<<grid, tf32x3::NUM_THREADS, tf32x3::SMEM_BYTES, stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], O, LSE, p.Hq, p.Hkv, p.N, scale_log2,
        status);
    return cudaGetLastError();
}

}  // namespace fa
