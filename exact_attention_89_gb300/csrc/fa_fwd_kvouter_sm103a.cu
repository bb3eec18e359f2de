// fa_fwd_kvouter_sm103a.cu -- K8: the forward in the key/value-outer loop order (IO ablation).
//
// The FlashAttention DAC'24 reading note (paper.adslab.icu, Methods) describes the loop order
// in which every K/V element is read from HBM once: the outer loop walks key/value blocks, the
// inner loop walks query blocks, and each query block's running output O and statistics
// (m, l) go back to HBM after every key/value block to be read again by the next one.  This
// kernel computes the same O and LSE as the query-outer forward (fa_fwd) in that order, so the
// two orders' HBM traffic and time can be compared on this GPU.
//
// One CTA per (batch, query head) -- the order's only parallelism, since every key/value block
// updates every query block of its head.  192 threads:
//   warps 0-3 : softmax / update warps (thread = query row = TMEM lane)
//   warp 4    : TMA producer (K_j, V_j once per block, double-buffered; Q_i per step, 2 stages)
//   warp 5    : TMEM allocator and single-thread MMA issuer
// Step g = (key block j, query tile i), i >= j under causal masking.  TMEM: S/P of buffer
// b = g mod 2 at columns 128 b, P V of buffer b at 256 + 128 b, so S of step g+1 overlaps the
// update of step g.  The update per row: m' = max(m, rowmax), p = 2^(s c - m'),
// l' = 2^(m - m') l + sum p, O' = 2^(m - m') O + P V_j (deferred normalisation; fp32 O, m, l and
// the bf16 rounding residual lc of c16 in a workspace); the last block of a tile writes
// O = O' / (l' + lc') in bf16 and LSE = m' + ln l'.
#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace kvo {

constexpr int D = 128;
constexpr int BM = 128, BN = 128;
constexpr int NUM_THREADS = 192;
constexpr int WARP_TMA = 4, WARP_MMA = 5;
constexpr int TILE_BYTES = 128 * D * 2;       // one Q tile or one K / V block (bf16)
constexpr int CHUNK_BYTES = 128 * 128;        // 128 rows x 64 bf16
constexpr int KV_OFF = 0;                     // [2 stages][K | V]
constexpr int Q_OFF = KV_OFF + 2 * 2 * TILE_BYTES;
constexpr int BAR_OFF = Q_OFF + 2 * TILE_BYTES;
// kv_full[2], kv_empty[2], q_full[2], q_empty[2], s_full[2], p_full[2], o_full[2], t_free[2],
// mma_done
constexpr int NBARS = 8 * 2 + 1;
constexpr int TMEM_OFF = BAR_OFF + NBARS * 8;
constexpr int ABORT_OFF = TMEM_OFF + 8;
constexpr int SMEM_BYTES = ABORT_OFF + 8 + 1024;
constexpr float LN2 = 0.693147180559945309f;

// Query tiles a key block updates: [first_tile(j), nq).
template <bool CAUSAL>
__device__ __forceinline__ int first_tile(int j) {
    return CAUSAL ? j : 0;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    kvouter_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, __nv_bfloat16 *__restrict__ O,
                   float *__restrict__ LSE, float *__restrict__ Oacc, float *__restrict__ stats,
                   int Hq, int Hkv, int N, float scale_log2, unsigned *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    uint64_t *kv_full = bars, *kv_empty = bars + 2, *q_full = bars + 4, *q_empty = bars + 6;
    uint64_t *s_full = bars + 8, *p_full = bars + 10, *o_full = bars + 12, *t_free = bars + 14;
    uint64_t *mma_done = bars + 16;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + TMEM_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + ABORT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;                      // b * Hq + hq
    const int bkv = (bh / Hq) * Hkv + (bh % Hq) / (Hq / Hkv);
    const int nkb = (N + BN - 1) / BN, nq = (N + BM - 1) / BM;
    int G = 0;                                      // steps of this CTA
    for (int j = 0; j < nkb; ++j) G += nq - first_tile<CAUSAL>(j);

    if (threadIdx.x == 0) {
        for (int k = 0; k < NBARS - 1; ++k) mbar_init(&bars[k], (k >= 10 && k < 12) || k >= 14 ? 128 : 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == WARP_TMA) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int g = 0, kv_issued = 0, q_issued = 0;
            bool ok = true;
            for (int j = 0; j < nkb && ok; ++j) {
                const int ks = j & 1;
                // K/V stage ks was last used by block j-2: wait until its products are done
                if (j >= 2 && !mbar_wait(&kv_empty[ks], ((j - 2) >> 1) & 1, abort_flag, status)) { ok = false; break; }
                mbar_arrive_expect_tx(&kv_full[ks], 2 * TILE_BYTES);
                uint8_t *kd = smem + KV_OFF + ks * 2 * TILE_BYTES;
                for (int ch = 0; ch < D / 64; ++ch) {
                    tma_load_3d(kd + ch * CHUNK_BYTES, &tmK, ch * 64, j * BN, bkv, &kv_full[ks]);
                    tma_load_3d(kd + TILE_BYTES + ch * CHUNK_BYTES, &tmV, ch * 64, j * BN, bkv, &kv_full[ks]);
                }
                kv_issued = j + 1;
                for (int i = first_tile<CAUSAL>(j); i < nq; ++i, ++g) {
                    const int qs = g & 1;
                    if (!mbar_wait(&q_empty[qs], ((g >> 1) & 1) ^ 1, abort_flag, status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&q_full[qs], TILE_BYTES);
                    for (int ch = 0; ch < D / 64; ++ch)
                        tma_load_3d(smem + Q_OFF + qs * TILE_BYTES + ch * CHUNK_BYTES, &tmQ, ch * 64,
                                    i * BM, bh, &q_full[qs]);
                    q_issued = g + 1;
                }
            }
            if (!ok || *abort_flag) {
                for (int k = max(0, kv_issued - 2); k < kv_issued; ++k) mbar_drain(&kv_full[k & 1], (k >> 1) & 1);
                for (int k = max(0, q_issued - 2); k < q_issued; ++k) mbar_drain(&q_full[k & 1], (k >> 1) & 1);
            }
        }
        tc_fence_before();
        __syncthreads();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, false, true);
            // (j, i) of the step after (j, i)
            auto advance = [&](int &j, int &i) {
                if (++i == nq) {
                    ++j;
                    i = first_tile<CAUSAL>(j);
                }
            };
            bool ok = true;
            auto issue_s = [&](int g, int j, int i) -> bool {
                const int b = g & 1;
                if (i == first_tile<CAUSAL>(j) &&
                    !mbar_wait(&kv_full[j & 1], (j >> 1) & 1, abort_flag, status)) return false;
                if (!mbar_wait(&q_full[b], (g >> 1) & 1, abort_flag, status)) return false;
                // buffer b last held step g-2: the update warps must be done with it
                if (g >= 2 && !mbar_wait(&t_free[b], ((g - 2) >> 1) & 1, abort_flag, status)) return false;
                tc_fence_after();
                const uint64_t da = sdesc_sw128(smem_u32(smem + Q_OFF + b * TILE_BYTES), 16, 1024);
                const uint64_t db = sdesc_sw128(smem_u32(smem + KV_OFF + (j & 1) * 2 * TILE_BYTES), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;
                    mma_ss(tmem + b * 128, sdesc_add(da, off), sdesc_add(db, off), IDESC_S, kk > 0);
                }
                mma_commit(&s_full[b]);
                mma_commit(&q_empty[b]);
                return true;
            };
            int j = 0, i = first_tile<CAUSAL>(0);          // step g
            int jn = j, in = i;                             // step g + 1
            advance(jn, in);
            if (G > 0) ok = issue_s(0, j, i);
            for (int g = 0; g < G && ok; ++g) {
                const int b = g & 1;
                // S of the next step goes before P V of this one (its buffer is the other one)
                if (g + 1 < G && !(ok = issue_s(g + 1, jn, in))) break;
                if (!mbar_wait(&p_full[b], (g >> 1) & 1, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                const uint64_t dv = sdesc_sw128(
                    smem_u32(smem + KV_OFF + (j & 1) * 2 * TILE_BYTES + TILE_BYTES), CHUNK_BYTES, 1024);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(tmem + 256 + b * 128, tmem + b * 128 + kk * 8, sdesc_add(dv, kk * 2048),
                           IDESC_PV, kk > 0 ? 1u : 0u);
                mma_commit(&o_full[b]);
                if (i == nq - 1) mma_commit(&kv_empty[j & 1]);   // last product reading K_j / V_j
                j = jn;
                i = in;
                advance(jn, in);
            }
            mma_commit(mma_done);
            mbar_drain(mma_done, 0);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == WARP_MMA) {
            __syncwarp();
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    } else {
        // ------------------------------------------------------------------ update warps
        const int row = warp * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const size_t nstat = static_cast<size_t>(gridDim.x) * N;
        float *m_ws = stats, *l_ws = stats + nstat, *lc_ws = stats + 2 * nstat;
        bool ok = true;
        int g = 0;
        for (int j = 0; j < nkb && ok; ++j) {
            for (int i = first_tile<CAUSAL>(j); i < nq; ++i, ++g) {
                const int b = g & 1;
                const int q = i * BM + row;             // query index
                const bool first = (j == 0), last = (j == (CAUSAL ? i : nkb - 1));
                const size_t srow = static_cast<size_t>(bh) * N + q;
                float m_old = -INFINITY, l_old = 0.f, lc_old = 0.f;
                if (!first && q < N) {
                    m_old = m_ws[srow];
                    l_old = l_ws[srow];
                    lc_old = lc_ws[srow];
                }
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b], (g >> 1) & 1, abort_flag, status));
                if (!ok) break;
                tc_fence_after();
                uint32_t sraw[128];
                tmem_ld_x128(tmem + lane_off + b * 128, sraw);
                float s[128];
                const int kbase = j * BN;
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    s[c] = __uint_as_float(sraw[c]);
                    const int key = kbase + c;
                    if ((CAUSAL && key > q) || key >= N) s[c] = -INFINITY;
                    mx = fmaxf(mx, s[c]);
                }
                const float m_new = fmaxf(m_old, mx * scale_log2);
                const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = (m_old == -INFINITY) ? 0.f : ex2_approx(m_old - m_sub);
                float psum = 0.f;
                uint32_t p[64];
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const float p0 = ex2_approx(fmaf(s[2 * c], scale_log2, -m_sub));
                    const float p1 = ex2_approx(fmaf(s[2 * c + 1], scale_log2, -m_sub));
                    psum += p0 + p1;
                    p[c] = pack_bf16x2(p0, p1);
                }
                const float ptop = ex2_approx(fmaf(mx, scale_log2, -m_sub));
                const float l_new = l_old * alpha + psum;
                const float lc_new = lc_old * alpha + (__bfloat162float(__float2bfloat16_rn(ptop)) - ptop);
                tmem_st_x32(tmem + lane_off + b * 128, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                tmem_st_x32(tmem + lane_off + b * 128 + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[b]);
                // the running O of this row: read back while P V runs
                float *orow = Oacc + srow * D;
                float oo[128];
#pragma unroll
                for (int c4 = 0; c4 < 32; ++c4) {
                    const float4 v = (!first && q < N) ? reinterpret_cast<const float4 *>(orow)[c4]
                                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                    oo[4 * c4] = v.x * alpha;
                    oo[4 * c4 + 1] = v.y * alpha;
                    oo[4 * c4 + 2] = v.z * alpha;
                    oo[4 * c4 + 3] = v.w * alpha;
                }
                ok = __all_sync(0xffffffffu, mbar_wait(&o_full[b], (g >> 1) & 1, abort_flag, status));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t pv[32];
                    tmem_ld_x32(tmem + lane_off + 256 + b * 128 + c0, pv);
#pragma unroll
                    for (int c = 0; c < 32; ++c) oo[c0 + c] += __uint_as_float(pv[c]);
                }
                tc_fence_before();
                mbar_arrive(&t_free[b]);
                if (q < N) {
                    if (last) {
                        const float inv = 1.f / (l_new + lc_new);
                        uint4 *od = reinterpret_cast<uint4 *>(O + srow * D);
#pragma unroll
                        for (int u = 0; u < D / 8; ++u)
                            od[u] = make_uint4(pack_bf16x2(oo[8 * u] * inv, oo[8 * u + 1] * inv),
                                               pack_bf16x2(oo[8 * u + 2] * inv, oo[8 * u + 3] * inv),
                                               pack_bf16x2(oo[8 * u + 4] * inv, oo[8 * u + 5] * inv),
                                               pack_bf16x2(oo[8 * u + 6] * inv, oo[8 * u + 7] * inv));
                        LSE[srow] = (m_new + log2f(l_new)) * LN2;
                    } else {
#pragma unroll
                        for (int c4 = 0; c4 < 32; ++c4)
                            reinterpret_cast<float4 *>(orow)[c4] =
                                make_float4(oo[4 * c4], oo[4 * c4 + 1], oo[4 * c4 + 2], oo[4 * c4 + 3]);
                        m_ws[srow] = m_new;
                        l_ws[srow] = l_new;
                        lc_ws[srow] = lc_new;
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
    }
}

}  // namespace kvo

size_t kvouter_workspace_bytes(long long BH, int N, int d) {
    const size_t rows = static_cast<size_t>(BH) * N;
    return rows * d * sizeof(float) + 3 * rows * sizeof(float);
}

cudaError_t launch_fwd_kvouter_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                    const CUtensorMap &tmV, void *O, float *LSE, float *workspace,
                                    unsigned *status, cudaStream_t stream) {
    if (p.d != kvo::D) return cudaErrorInvalidValue;
    auto kern = p.causal ? kvo::kvouter_kernel<true> : kvo::kvouter_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kvo::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long BH = static_cast<long long>(p.B) * p.Hq;
    if (BH > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t rows = static_cast<size_t>(BH) * p.N;
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    kern<<<static_cast<unsigned>(BH), kvo::NUM_THREADS, kvo::SMEM_BYTES, stream>>>(
        tmQ, tmK, tmV, static_cast<__nv_bfloat16 *>(O), LSE, workspace, workspace + rows * p.d,
        p.Hq, p.Hkv, p.N, scale_log2, status);
    return cudaGetLastError();
}

}  // namespace fa
