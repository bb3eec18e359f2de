// fa_bwd_tf32x3_sm103a.cu -- K10: fp32 backward on the tensor cores with three TF32 products.
//
// The backward of the bf16 path ("Attention's hidden recurrence" blog by mzeromiko, "Flash
// Attention backward": P is recomputed from the stored LSE, D_i = sum_k dO_ik O_ik,
// dS = P (dP - D) with dP = dO V^T, dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K) for fp32
// inputs and outputs, every product formed from TF32 parts as in the fp32 forward
// (hi(A) hi(B) + hi(A) lo(B) + lo(A) hi(B), fa_tf32.cuh).
//
// Two passes and no atomics; dQ, dK and dV are each written once, in fp32:
//   dq pass  : one CTA per 128-row query tile of one (batch, query head).  It forms D for its
//              rows, then for every 32-key block: S = Q K^T, dP = dO V^T,
//              P = exp2(S c - LSE log2 e), dS = P (dP - D), dQ += dS K.
//   dkv pass : one CTA per 128-key block of one (batch, KV head), looping over the G query
//              heads of the group and over 32-row query blocks (under causal masking only those
//              at or below the block's diagonal): S^T = K Q^T, dP^T = V dO^T,
//              P^T = exp2(S^T c - LSE log2 e), dS^T = P^T (dP^T - D), dV += P^T dO,
//              dK += dS^T Q, so dK and dV of the block sum over the group in TMEM.
// The dq pass recomputes S and dP (seven products per tile pair instead of five); in exchange
// every product has M = 128 and dQ needs no fp32 reduction into global memory.
//
// The 128 rows a CTA owns keep both of their operands (Q and dO, or K and V), split hi / lo, in
// TMEM as the A operands of the first two products; the streamed operands come hi / lo from a
// workspace written by the split kernels (row-major copies, and transposed copies for the B
// operands of the last products, since TF32 operands are used K-major only).
//
// Accumulation: the tensor core adds every product into its fp32 accumulator with a rounding
// that does not average out (measured: the error of a sum grows with the number of MMAs
// chained into one accumulator, about half an ulp each), so the last products of each step
// start a fresh accumulator and a second warpgroup adds the step's result into fp32 register
// sums, rounded to nearest; a chain is then 12 MMAs long instead of 12 per step of the pass.
//
// Roles (320 threads): warps 0-3 gradient warps (thread = owned row = TMEM lane), warps 4-7
// accumulation warps (same rows: they own the register sums and write the gradients), warp 8
// TMA producer (two-stage ring of streamed tiles), warp 9 TMEM allocator and MMA issuer.
// TMEM (512 columns): X1 / X2 (S or S^T, dP or dP^T) double-buffered at [0,64) and [192,256),
// Y1 [64,128) (dQ or dV of the step), Y2 [128,192) (dK of the step), first resident operand hi
// [256,320) lo [320,384), second hi [384,448) lo [448,512).
#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_tf32.cuh"

namespace fa {
namespace tf32bwd {

constexpr int D = 64;
constexpr int BR = 128;                   // rows a CTA owns
constexpr int BC = 32;                    // rows of a streamed block
constexpr int NUM_THREADS = 320;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr float LOG2E = 1.4426950408889634f;

// Shared memory, every tile 1024-byte aligned, rows of 32 fp32 (128 B) with the 128-byte swizzle.
constexpr int XT_CHUNK = BC * 128;        // 32 rows x 32 fp32
constexpr int XT_BYTES = 2 * XT_CHUNK;    // 32 rows x 64 fp32 (two chunks along d)
constexpr int YT_BYTES = D * 128;         // 64 rows (d) x 32 fp32
// Operands of the first products (XA hi, XA lo, XB hi, XB lo) in a 3-slot ring; those of the last
// products (YA hi, YA lo, YB hi, YB lo) in a 2-slot ring: the first products of step s + 1 are
// issued before the last ones of step s.
constexpr int NXS = 3, NYS = 2;
constexpr int XS_BYTES = 4 * XT_BYTES, YS_BYTES = 4 * YT_BYTES;
constexpr int XS_OFF = 0, YS_OFF = NXS * XS_BYTES;
constexpr int STG_BYTES = BR * 128;       // one staged 128 x 32 fp32 operand
constexpr int STG_OFF = YS_OFF + NYS * YS_BYTES;   // P hi, P lo, dS hi, dS lo
constexpr int BAR_OFF = STG_OFF + 4 * STG_BYTES;
// xf[3], xe[3], yf[2], ye[2], r_full, x_done[2], p_full, y_full, y_empty, mma_done
constexpr int NBARS = 17;
constexpr int TMEM_OFF = BAR_OFF + NBARS * 8;
constexpr int ABORT_OFF = TMEM_OFF + 8;
constexpr int SMEM_BYTES = ABORT_OFF + 8 + 1024;
// X1 / X2 of buffer b at T_X + 192 b (+0 / +32)
constexpr uint32_t T_X = 0, T_Y1 = 64, T_Y2 = 128, T_RA = 256, T_RB = 384;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

// Streamed operands of one pass (all 3-D [inner, rows, planes] fp32, 128-byte swizzle):
//   dq pass : xa = K, xb = V (box 32 x 32), ya = K^T (box 32 x 64); yb unused
//   dkv pass: xa = Q, xb = dO (box 32 x 32), ya = dO^T, yb = Q^T (box 32 x 64)
struct Maps {
    CUtensorMap xa_h, xa_l, xb_h, xb_l, ya_h, ya_l, yb_h, yb_l;
};

// Row-major hi / lo copies: up to four tensors of n[i] elements each.
struct SplitJobs {
    const float *src[4];
    float *hi[4], *lo[4];
    long long n[4];
};

__global__ void __launch_bounds__(256) split_rows_kernel(const SplitJobs jobs) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 *src = reinterpret_cast<const float4 *>(jobs.src[j]);
        float4 *hi = reinterpret_cast<float4 *>(jobs.hi[j]), *lo = reinterpret_cast<float4 *>(jobs.lo[j]);
        for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < jobs.n[j] / 4;
             t += stride) {
            const float4 x = src[t];
            const float4 h = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
            hi[t] = h;
            lo[t] = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
        }
    }
}

// Transposed hi / lo copies [P, 64, Np] of [P, N, 64] tensors (columns n >= N are zero): one
// block per 32 rows of one plane, staged through shared memory so both sides are coalesced.
// blockIdx.z picks the tensor (Q, dO over B*Hq planes; K over B*Hkv planes).
struct TransJobs {
    const float *src[3];
    float *hi[3], *lo[3];
    int planes[3];
};

__global__ void __launch_bounds__(256) split_transpose_kernel(const TransJobs jobs, int N, int Np) {
    const int z = blockIdx.z, p = blockIdx.y;
    // (selects, not an indexed parameter array, so the job stays in registers)
    const int planes = z == 0 ? jobs.planes[0] : z == 1 ? jobs.planes[1] : jobs.planes[2];
    if (p >= planes) return;
    const float *src0 = z == 0 ? jobs.src[0] : z == 1 ? jobs.src[1] : jobs.src[2];
    float *hi0 = z == 0 ? jobs.hi[0] : z == 1 ? jobs.hi[1] : jobs.hi[2];
    float *lo0 = z == 0 ? jobs.lo[0] : z == 1 ? jobs.lo[1] : jobs.lo[2];
    __shared__ float tile[BC][D + 1];
    const int n0 = blockIdx.x * BC;
    const float *src = src0 + static_cast<size_t>(p) * N * D;
    for (int i = threadIdx.x; i < BC * D; i += blockDim.x) {
        const int r = i / D, c = i % D;
        tile[r][c] = (n0 + r < N) ? src[static_cast<size_t>(n0 + r) * D + c] : 0.f;
    }
    __syncthreads();
    float *hi = hi0 + static_cast<size_t>(p) * D * Np, *lo = lo0 + static_cast<size_t>(p) * D * Np;
    for (int i = threadIdx.x; i < BC * D; i += blockDim.x) {
        const int c = i / BC, j = i % BC;
        const float x = tile[j][c], h = tf32_hi(x);
        hi[static_cast<size_t>(c) * Np + n0 + j] = h;
        lo[static_cast<size_t>(c) * Np + n0 + j] = x - h;
    }
}

// Writes one 32-value row of a staged K-major operand, hi and lo parts, 128-byte swizzled.
__device__ __forceinline__ void stage_row(uint8_t *hi_tile, uint8_t *lo_tile, int row, const float (&v)[32]) {
    uint8_t *ph = hi_tile + row * 128, *pl = lo_tile + row * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float4 h = make_float4(tf32_hi(v[4 * u]), tf32_hi(v[4 * u + 1]), tf32_hi(v[4 * u + 2]),
                                     tf32_hi(v[4 * u + 3]));
        const float4 l = make_float4(v[4 * u] - h.x, v[4 * u + 1] - h.y, v[4 * u + 2] - h.z, v[4 * u + 3] - h.w);
        const int sw = (u ^ (row & 7)) << 4;
        *reinterpret_cast<float4 *>(ph + sw) = h;
        *reinterpret_cast<float4 *>(pl + sw) = l;
    }
}

// Loads 32 consecutive fp32 of a row (zeros when the row is past the end) and stores its hi and
// lo parts into TMEM columns [col, col + 32) and [col + 64, col + 96) of this thread's lane.
__device__ __forceinline__ void put_resident(uint32_t taddr, const float *row, bool valid, float *keep) {
    uint32_t h[32], l[32];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float4 x = valid ? reinterpret_cast<const float4 *>(row)[u] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float hh = tf32_hi(xs[k]);
            h[4 * u + k] = __float_as_uint(hh);
            l[4 * u + k] = __float_as_uint(xs[k] - hh);
            if (keep) keep[4 * u + k] = xs[k];
        }
    }
    tmem_st_x32(taddr, h);
    tmem_st_x32(taddr + 64, l);
}

template <bool DKV, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_kernel(const __grid_constant__ Maps maps, const float *__restrict__ RA,
               const float *__restrict__ RB, const float *__restrict__ O, const float *__restrict__ LSE,
               float *__restrict__ Dvec, float *__restrict__ OUT1, float *__restrict__ OUT2, int Hq,
               int Hkv, int N, float scale, float scale_log2, unsigned *status) {
    // RA, RB: the owned rows' operands (dq pass: Q, dO; dkv pass: K, V), fp32 [planes, N, 64].
    // dq pass: O is read to form D, which is written to Dvec; OUT1 = dQ.
    // dkv pass: Dvec is read; OUT1 = dV, OUT2 = dK.
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    uint64_t *xf = bars, *xe = bars + 3, *yf = bars + 6, *ye = bars + 8, *r_full = bars + 10;
    uint64_t *x_done = bars + 11, *p_full = bars + 13, *y_full = bars + 14, *y_empty = bars + 15;
    uint64_t *mma_done = bars + 16;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + TMEM_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + ABORT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = Hq / Hkv;
    const int nblk = (N + BC - 1) / BC;            // streamed blocks along N
    // owned rows and the streamed steps
    int plane_r, r0, first = 0, per = 0, T;
    int b = 0, hk = 0;
    if (DKV) {
        plane_r = blockIdx.y;                      // b * Hkv + hk
        b = plane_r / Hkv;
        hk = plane_r % Hkv;
        r0 = blockIdx.x * BR;
        first = CAUSAL ? r0 / BC : 0;              // query blocks at or below the diagonal
        per = nblk - first;
        T = G * per;
    } else {
        plane_r = blockIdx.y;                      // b * Hq + hq
        const int nt = gridDim.x;
        r0 = (CAUSAL ? nt - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x)) * BR;
        T = CAUSAL ? min(nblk, (min(r0 + BR, N) - 1) / BC + 1) : nblk;
    }
    // step s -> (plane of the streamed operands, block index)
    auto step = [&](int s, int &plane, int &blk) {
        if (DKV) {
            plane = b * Hq + hk * G + s / per;
            blk = first + s % per;
        } else {
            plane = (plane_r / Hq) * Hkv + (plane_r % Hq) / G;
            blk = s;
        }
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NXS; ++i) {
            mbar_init(&xf[i], 1);
            mbar_init(&xe[i], 1);
        }
        for (int i = 0; i < NYS; ++i) {
            mbar_init(&yf[i], 1);
            mbar_init(&ye[i], 1);
        }
        mbar_init(r_full, BR);
        mbar_init(&x_done[0], 1);
        mbar_init(&x_done[1], 1);
        mbar_init(p_full, BR);
        mbar_init(y_full, 1);
        mbar_init(y_empty, BR);
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
            const uint32_t ybytes = (DKV ? 4 : 2) * YT_BYTES;
            int xissued = 0, yissued = 0;
            for (int s = 0; s < T; ++s) {
                const int xs = s % NXS, ys = s % NYS;
                if (s >= NXS && !mbar_wait(&xe[xs], (s / NXS - 1) & 1, abort_flag, status)) break;
                int plane, blk;
                step(s, plane, blk);
                mbar_arrive_expect_tx(&xf[xs], XS_BYTES);
                uint8_t *xb = smem + XS_OFF + xs * XS_BYTES;
                for (int ch = 0; ch < D / 32; ++ch) {
                    tma_load_3d(xb + 0 * XT_BYTES + ch * XT_CHUNK, &maps.xa_h, ch * 32, blk * BC, plane, &xf[xs]);
                    tma_load_3d(xb + 1 * XT_BYTES + ch * XT_CHUNK, &maps.xa_l, ch * 32, blk * BC, plane, &xf[xs]);
                    tma_load_3d(xb + 2 * XT_BYTES + ch * XT_CHUNK, &maps.xb_h, ch * 32, blk * BC, plane, &xf[xs]);
                    tma_load_3d(xb + 3 * XT_BYTES + ch * XT_CHUNK, &maps.xb_l, ch * 32, blk * BC, plane, &xf[xs]);
                }
                xissued = s + 1;
                if (s >= NYS && !mbar_wait(&ye[ys], (s / NYS - 1) & 1, abort_flag, status)) break;
                mbar_arrive_expect_tx(&yf[ys], ybytes);
                uint8_t *yb = smem + YS_OFF + ys * YS_BYTES;
                tma_load_3d(yb, &maps.ya_h, blk * BC, 0, plane, &yf[ys]);
                tma_load_3d(yb + YT_BYTES, &maps.ya_l, blk * BC, 0, plane, &yf[ys]);
                if (DKV) {
                    tma_load_3d(yb + 2 * YT_BYTES, &maps.yb_h, blk * BC, 0, plane, &yf[ys]);
                    tma_load_3d(yb + 3 * YT_BYTES, &maps.yb_l, blk * BC, 0, plane, &yf[ys]);
                }
                yissued = s + 1;
            }
            if (*abort_flag) {
                // let copies still in flight land before the CTA's shared memory goes away
                for (int s = max(0, xissued - NXS); s < xissued; ++s) mbar_drain(&xf[s % NXS], (s / NXS) & 1);
                for (int s = max(0, yissued - NYS); s < yissued; ++s) mbar_drain(&yf[s % NYS], (s / NYS) & 1);
            }
        }
        tc_fence_before();
        __syncthreads();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_X = idesc_tf32(BR, BC);
            constexpr uint32_t IDESC_Y = idesc_tf32(BR, D);
            // staged A operands of the last products: P (dkv pass) and dS
            const uint64_t dph = sdesc_sw128(smem_u32(smem + STG_OFF), 16, 1024);
            const uint64_t dpl = sdesc_sw128(smem_u32(smem + STG_OFF + STG_BYTES), 16, 1024);
            const uint64_t dsh = sdesc_sw128(smem_u32(smem + STG_OFF + 2 * STG_BYTES), 16, 1024);
            const uint64_t dsl = sdesc_sw128(smem_u32(smem + STG_OFF + 3 * STG_BYTES), 16, 1024);
            // X1 = RA xa^T and X2 = RB xb^T of step s into buffer s & 1, over d = 64 (8 k-steps)
            auto issue_x = [&](int s) -> bool {
                const int xs = s % NXS;
                if (!mbar_wait(&xf[xs], (s / NXS) & 1, abort_flag, status)) return false;
                tc_fence_after();
                const uint32_t base = smem_u32(smem + XS_OFF + xs * XS_BYTES);
                const uint64_t dxah = sdesc_sw128(base, 16, 1024);
                const uint64_t dxal = sdesc_sw128(base + XT_BYTES, 16, 1024);
                const uint64_t dxbh = sdesc_sw128(base + 2 * XT_BYTES, 16, 1024);
                const uint64_t dxbl = sdesc_sw128(base + 3 * XT_BYTES, 16, 1024);
                const uint32_t t1 = tmem + T_X + 192 * (s & 1), t2 = t1 + 32;
#pragma unroll
                for (int kk = 0; kk < D / 8; ++kk) {
                    const uint32_t off = (kk >> 2) * XT_CHUNK + (kk & 3) * 32;
                    const uint32_t ca = tmem + T_RA + kk * 8, cb = tmem + T_RB + kk * 8;
                    mma_tf32_ts(t1, ca, sdesc_add(dxah, off), IDESC_X, kk > 0);
                    mma_tf32_ts(t1, ca, sdesc_add(dxal, off), IDESC_X, 1u);
                    mma_tf32_ts(t1, ca + 64, sdesc_add(dxah, off), IDESC_X, 1u);
                    mma_tf32_ts(t2, cb, sdesc_add(dxbh, off), IDESC_X, kk > 0);
                    mma_tf32_ts(t2, cb, sdesc_add(dxbl, off), IDESC_X, 1u);
                    mma_tf32_ts(t2, cb + 64, sdesc_add(dxbh, off), IDESC_X, 1u);
                }
                mma_commit(&x_done[s & 1]);
                mma_commit(&xe[xs]);
                return true;
            };
            bool ok = mbar_wait(r_full, 0, abort_flag, status);
            if (ok && T > 0) ok = issue_x(0);
            for (int s = 0; s < T && ok; ++s) {
                // buffer (s + 1) & 1 was read by the gradient warps before they signalled p_full
                // of step s - 1
                if (s + 1 < T && !issue_x(s + 1)) { ok = false; break; }
                if (!mbar_wait(p_full, s & 1, abort_flag, status)) { ok = false; break; }
                // the accumulation warps have read the previous step's Y
                if (s > 0 && !mbar_wait(y_empty, (s - 1) & 1, abort_flag, status)) { ok = false; break; }
                const int ys = s % NYS;
                if (!mbar_wait(&yf[ys], (s / NYS) & 1, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t base = smem_u32(smem + YS_OFF + ys * YS_BYTES);
                const uint64_t dyah = sdesc_sw128(base, 16, 1024);
                const uint64_t dyal = sdesc_sw128(base + YT_BYTES, 16, 1024);
                const uint64_t dybh = sdesc_sw128(base + 2 * YT_BYTES, 16, 1024);
                const uint64_t dybl = sdesc_sw128(base + 3 * YT_BYTES, 16, 1024);
                // Y1 = (P or dS) ya, Y2 = dS yb over the block's 32 rows (4 k-steps of 8), in a
                // fresh accumulator
#pragma unroll
                for (int kk = 0; kk < BC / 8; ++kk) {
                    const uint32_t off = kk * 32;
                    const uint32_t acc = kk > 0 ? 1u : 0u;
                    const uint64_t a1h = DKV ? dph : dsh, a1l = DKV ? dpl : dsl;
                    mma_tf32(tmem + T_Y1, sdesc_add(a1h, off), sdesc_add(dyah, off), IDESC_Y, acc);
                    mma_tf32(tmem + T_Y1, sdesc_add(a1h, off), sdesc_add(dyal, off), IDESC_Y, 1u);
                    mma_tf32(tmem + T_Y1, sdesc_add(a1l, off), sdesc_add(dyah, off), IDESC_Y, 1u);
                    if (DKV) {
                        mma_tf32(tmem + T_Y2, sdesc_add(dsh, off), sdesc_add(dybh, off), IDESC_Y, acc);
                        mma_tf32(tmem + T_Y2, sdesc_add(dsh, off), sdesc_add(dybl, off), IDESC_Y, 1u);
                        mma_tf32(tmem + T_Y2, sdesc_add(dsl, off), sdesc_add(dybh, off), IDESC_Y, 1u);
                    }
                }
                mma_commit(y_full);
                mma_commit(&ye[ys]);
            }
            // Nothing issued may still be running when TMEM is released.
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
    } else if (warp < 4) {
        // ------------------------------------------------------------------ gradient warps
        const int row = warp * 32 + lane;
        const int grow = r0 + row;
        const bool valid = grow < N;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const size_t roff = (static_cast<size_t>(plane_r) * N + (valid ? grow : 0)) * D;
        float Dr = 0.f, lse2 = -INFINITY;
        // resident operands; the dq pass forms D_r = sum_k dO_rk O_rk on the way
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            float keep[32];
            put_resident(tmem + lane_off + T_RA + h * 32, RA + roff + h * 32, valid, nullptr);
            put_resident(tmem + lane_off + T_RB + h * 32, RB + roff + h * 32, valid, DKV ? nullptr : keep);
            if (!DKV && valid) {
                const float4 *o4 = reinterpret_cast<const float4 *>(O + roff + h * 32);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 o = o4[u];
                    Dr = fmaf(keep[4 * u], o.x, Dr);
                    Dr = fmaf(keep[4 * u + 1], o.y, Dr);
                    Dr = fmaf(keep[4 * u + 2], o.z, Dr);
                    Dr = fmaf(keep[4 * u + 3], o.w, Dr);
                }
            }
        }
        tmem_wait_st();
        if (!DKV && valid) {
            Dvec[static_cast<size_t>(plane_r) * N + grow] = Dr;
            const float l = LSE[static_cast<size_t>(plane_r) * N + grow];
            lse2 = l * LOG2E;
        }
        tc_fence_before();
        mbar_arrive(r_full);

        bool ok = true;
        uint8_t *ph = smem + STG_OFF, *pl = ph + STG_BYTES, *sh = pl + STG_BYTES, *sl = sh + STG_BYTES;
        for (int s = 0; s < T; ++s) {
            ok = __all_sync(0xffffffffu, mbar_wait(&x_done[s & 1], (s >> 1) & 1, abort_flag, status));
            if (!ok) break;
            tc_fence_after();
            uint32_t x1[32], x2[32];
            tmem_ld_x32(tmem + lane_off + T_X + 192 * (s & 1), x1);
            tmem_ld_x32(tmem + lane_off + T_X + 192 * (s & 1) + 32, x2);
            int plane, blk;
            step(s, plane, blk);
            const int c0 = blk * BC;
            float p[32], ds[32];
            if (DKV) {
                // thread = key grow; column c = query c0 + c with its LSE and D
                const float *lrow = LSE + static_cast<size_t>(plane) * N;
                const float *drow = Dvec + static_cast<size_t>(plane) * N;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int q = c0 + c;
                    const bool inq = q < N;
                    const float lq = inq ? __ldg(lrow + q) * LOG2E : -INFINITY;
                    const float dq = inq ? __ldg(drow + q) : 0.f;
                    const bool allowed = valid && inq && (!CAUSAL || grow <= q) && lq != -INFINITY;
                    p[c] = allowed ? ex2_approx(fmaf(__uint_as_float(x1[c]), scale_log2, -lq)) : 0.f;
                    ds[c] = p[c] * (__uint_as_float(x2[c]) - dq);
                }
            } else {
                // thread = query grow; column c = key c0 + c
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int k = c0 + c;
                    const bool allowed = valid && k < N && (!CAUSAL || k <= grow) && lse2 != -INFINITY;
                    p[c] = allowed ? ex2_approx(fmaf(__uint_as_float(x1[c]), scale_log2, -lse2)) : 0.f;
                    ds[c] = p[c] * (__uint_as_float(x2[c]) - Dr);
                }
            }
            // the last products of step s - 1 have finished reading the staged operands
            if (s > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(y_full, (s - 1) & 1, abort_flag, status));
                if (!ok) break;
            }
            if (DKV) stage_row(ph, pl, row, p);
            stage_row(sh, sl, row, ds);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        tc_fence_before();
        __syncthreads();
    } else {
        // ------------------------------------------------------------------ accumulation warps
        // Same rows as the gradient warps (warp w and w - 4 share a TMEM lane quarter).  Each
        // step's Y (fresh accumulator) is added into fp32 register sums; the sums are written
        // out once, scaled where the method scales (dQ, dK).
        const int row = (warp - 4) * 32 + lane;
        const int grow = r0 + row;
        const bool valid = grow < N;
        const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
        const size_t roff = (static_cast<size_t>(plane_r) * N + (valid ? grow : 0)) * D;
        constexpr int NY = DKV ? 2 : 1;
        float sum[NY][D];
#pragma unroll
        for (int y = 0; y < NY; ++y)
#pragma unroll
            for (int c = 0; c < D; ++c) sum[y][c] = 0.f;
        bool ok = true;
        for (int s = 0; s < T; ++s) {
            ok = __all_sync(0xffffffffu, mbar_wait(y_full, s & 1, abort_flag, status));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int y = 0; y < NY; ++y)
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_x32(tmem + lane_off + (y ? T_Y2 : T_Y1) + c0, v);
#pragma unroll
                    for (int c = 0; c < 32; ++c) sum[y][c0 + c] += __uint_as_float(v[c]);
                }
            tc_fence_before();
            mbar_arrive(y_empty);
        }
        if (ok && valid) {
#pragma unroll
            for (int y = 0; y < NY; ++y) {
                // dkv pass: OUT1 = dV (unscaled), OUT2 = dK; dq pass: OUT1 = dQ
                const float f = (DKV && y == 0) ? 1.f : scale;
                float4 *o = reinterpret_cast<float4 *>((y ? OUT2 : OUT1) + roff);
#pragma unroll
                for (int u = 0; u < D / 4; ++u)
                    o[u] = make_float4(sum[y][4 * u] * f, sum[y][4 * u + 1] * f, sum[y][4 * u + 2] * f,
                                       sum[y][4 * u + 3] * f);
            }
        }
        tc_fence_before();
        __syncthreads();
    }
}

template <bool DKV, bool CAUSAL>
cudaError_t launch_pass(const Problem &p, const Maps &maps, const float *RA, const float *RB,
                        const float *O, const float *LSE, float *Dvec, float *OUT1, float *OUT2,
                        unsigned *status, cudaStream_t stream) {
    auto kern = bwd_kernel<DKV, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long planes = DKV ? 1LL * p.B * p.Hkv : 1LL * p.B * p.Hq;
    if (planes > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((p.N + BR - 1) / BR, static_cast<unsigned>(planes));
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    kern<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(maps, RA, RB, O, LSE, Dvec, OUT1, OUT2, p.Hq, p.Hkv,
                                                    p.N, p.scale, scale_log2, status);
    return cudaGetLastError();
}

}  // namespace tf32bwd

Tf32BwdWorkspace tf32x3_bwd_layout(long long BH, long long BHkv, int N, int d, void *workspace) {
    Tf32BwdWorkspace w{};
    w.Np = (N + 31) / 32 * 32;
    const long long nq = BH * N * d, nk = BHkv * N * d, nqt = BH * d * w.Np, nkt = BHkv * d * w.Np;
    float *f = static_cast<float *>(workspace);
    float **seq[] = {&w.Qh, &w.Ql, &w.dOh, &w.dOl, &w.Kh, &w.Kl, &w.Vh, &w.Vl,
                     &w.Qth, &w.Qtl, &w.dOth, &w.dOtl, &w.Kth, &w.Ktl, &w.D};
    const long long len[] = {nq, nq, nq, nq, nk, nk, nk, nk, nqt, nqt, nqt, nqt, nkt, nkt, BH * N};
    long long off = 0;
    for (int i = 0; i < 15; ++i) {
        *seq[i] = f ? f + off : nullptr;
        off += len[i];
    }
    w.bytes = static_cast<size_t>(off) * sizeof(float);
    return w;
}

cudaError_t launch_tf32x3_bwd_split(const Problem &p, const float *Q, const float *K, const float *V,
                                    const float *dO, const Tf32BwdWorkspace &w, cudaStream_t stream) {
    const long long BH = 1LL * p.B * p.Hq, BHkv = 1LL * p.B * p.Hkv;
    const long long nq = BH * p.N * p.d, nk = BHkv * p.N * p.d;
    tf32bwd::SplitJobs sj{{Q, dO, K, V}, {w.Qh, w.dOh, w.Kh, w.Vh}, {w.Ql, w.dOl, w.Kl, w.Vl}, {nq, nq, nk, nk}};
    long long grid = (nq / 4 + 255) / 256;
    grid = std::min<long long>(std::max<long long>(grid, 1), 16LL * num_sms());
    tf32bwd::split_rows_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(sj);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    tf32bwd::TransJobs tj{{Q, dO, K}, {w.Qth, w.dOth, w.Kth}, {w.Qtl, w.dOtl, w.Ktl},
                          {static_cast<int>(BH), static_cast<int>(BH), static_cast<int>(BHkv)}};
    const dim3 tgrid(static_cast<unsigned>(w.Np / tf32bwd::BC), static_cast<unsigned>(BH), 3);
    tf32bwd::split_transpose_kernel<<<tgrid, 256, 0, stream>>>(tj, p.N, static_cast<int>(w.Np));
    return cudaGetLastError();
}

cudaError_t launch_tf32x3_bwd(const Problem &p, const CUtensorMap *maps, const float *Q, const float *K,
                              const float *V, const float *O, const float *dO, const float *LSE,
                              float *dQ, float *dK, float *dV, float *Dvec, unsigned *status,
                              cudaStream_t stream) {
    if (p.d != tf32bwd::D) return cudaErrorInvalidValue;
    // maps: [0..5] dq pass (Kh, Kl, Vh, Vl, Kth, Ktl), [6..13] dkv pass (Qh, Ql, dOh, dOl,
    // dOth, dOtl, Qth, Qtl)
    const tf32bwd::Maps mq{maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[4], maps[5]};
    const tf32bwd::Maps mkv{maps[6], maps[7], maps[8], maps[9], maps[10], maps[11], maps[12], maps[13]};
    cudaError_t e = p.causal
                        ? tf32bwd::launch_pass<false, true>(p, mq, Q, dO, O, LSE, Dvec, dQ, nullptr, status, stream)
                        : tf32bwd::launch_pass<false, false>(p, mq, Q, dO, O, LSE, Dvec, dQ, nullptr, status, stream);
    if (e != cudaSuccess) return e;
    return p.causal ? tf32bwd::launch_pass<true, true>(p, mkv, K, V, nullptr, LSE, Dvec, dV, dK, status, stream)
                    : tf32bwd::launch_pass<true, false>(p, mkv, K, V, nullptr, LSE, Dvec, dV, dK, status, stream);
}

}  // namespace fa
