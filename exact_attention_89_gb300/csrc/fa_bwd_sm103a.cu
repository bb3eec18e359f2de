// fa_bwd_sm103a.cu -- K2 / K3 / K4: exact attention backward, bf16 in / fp32 accumulate, sm_103a.
//
// Method ("Attention's hidden recurrence" blog by mzeromiko, sections "standard attention /
// backward" and "Flash Attention backward"): nothing of P is stored by the forward pass; P is
// recomputed per tile from the stored statistics (here LSE = m + ln l, so P = exp(s - LSE)), and
//   D_i = diag(dO O^T)_i = sum_k dO_ik O_ik,   dS = P * (dP - D),  dP = dO V^T,
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
// (The blog's d(exp(QK^T) (.) M) (.) exp(QK^T) equals dS; scale enters by the chain rule.)
//
// K2 forms D and clears the fp32 dQ accumulator.  K3 gives each CTA one 128-key block of one
// (batch, KV head); it loops over the G query heads of the group and over 64-row query tiles
// (under causal masking only tiles at or below the block's diagonal), so dK and dV of the block
// accumulate in TMEM across the whole group and need no atomics.  Per query tile (step s):
//   S^T = K Q^T and dP^T = V dO^T        (SS MMAs, M = 128 keys, N = 64 queries, K = d)
//   P^T = exp2(S^T c - LSE log2 e), dS^T = P^T (dP^T - D)   (thread = key row = TMEM lane)
//   dV += P^T dO,  dK += dS^T Q          (TS MMAs: P^T / dS^T as bf16 in TMEM)
//   dQ^T = K^T dS^T                      (SS MMA, M = d = 128, dS^T staged in smem)
// and a second warpgroup reduces scale * dQ^T into the fp32 accumulator with coalesced
// fp32 reductions (thread = one column d of dQ).  K4 rounds the accumulator to bf16.
// dQ strategy: recomputing S and dP in a separate dQ kernel would cost 7 products per tile
// instead of 5 (+40% tensor work); the reduction costs L2 bandwidth instead.
//
// Software pipeline: S^T / dP^T are double-buffered in TMEM, so the products of step s+1 are
// issued before those that consume step s, and the softmax-gradient warps of one step overlap
// the tensor core's work on the other.  Inside a buffer, P^T and dS^T (bf16) are both written over
// the S^T half, which frees the dP^T half for the dQ^T product of the same step.
//
// Roles (640 threads, or 512 at head dim 64 outside the deterministic variant): warps 0-3
// softmax-gradient (queries 0-31 of each step, and the dK epilogue), warps 16-19 (12-15 at 512
// threads) the second softmax-gradient warpgroup (queries 32-63, and the dV epilogue unless the
// drain warps take it), warps 4-7 dQ drain (query columns 0-31 of each dQ^T tile; at 512 threads
// all 64, added as one bulk reduction, and the dV epilogue), warps 12-15 (640 threads) the second
// dQ drain warpgroup (columns 32-63), warp 8 TMA, warp 9 the S^T / dP^T MMAs and warp 10 the
// dQ^T / dV / dK MMAs (one elected lane each).  Warp 11 completes the third
// warpgroup for the register split; it issues the dP^T MMAs (warp 9 then only S^T), and in the
// deterministic variant it passes the dQ turns instead.
// TMEM (512 columns): dK [0,128), dV [128,256), buffer b at 256 + 128 b:
//   [+0,+64) S^T -> P^T [+0,+32) and dS^T [+32,+64) (two gradient warpgroups: P^T [+0,+16) and
//   dS^T [+16,+32) for queries 0-31, [+32,+48) and [+48,+64) for 32-63);
//   [+64,+128) dP^T -> dQ^T.
#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "fa_ptx.cuh"

namespace fa {
namespace bwd {

constexpr int BKV = 128;          // keys per CTA (= TMEM lanes)
constexpr int BQ = 64;            // query rows per step
constexpr int NSQ = 3;            // Q / dO ring stages
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;       // TMEM allocator; issues S^T (and dP^T unless warp 11 does)
constexpr int WARP_MMA2 = 10;     // issues dQ^T, dV and dK
constexpr int WARP_PASS = 11;     // issues dP^T; deterministic variant: passes the dQ turns
constexpr int NSENT = 4;          // steps the drain warps may run ahead of the turn passer
// Register split: the softmax-gradient warpgroups grow; dQ drain and TMA/MMA warpgroups shrink
// (640 threads: 144 / 56 / 80 of the 96 per thread the launch has; 512 threads: 144 / 88 / 80 of
// 128).
// Two softmax-gradient warpgroups (warps 0-3 and 16-19, or 12-15 with one drain warpgroup) take
// query columns 0-31 and 32-63 of each step.  Where dQ leaves through per-element reductions
// (head dim 128, and the deterministic variant at 64) two dQ drain warpgroups (warps 4-7 and
// 12-15) take the same columns of each dQ^T tile, so a step's element-wise work and its
// per-element reductions (and, with dropout, its keep decisions) are each split over two warps
// per scheduler; at head dim 64 otherwise dQ leaves as one bulk reduction per step from one drain
// warpgroup.  (Head dim 64: two gradient warpgroups 0.695 -> 0.633 ms; the deterministic variant
// 1.107 -> 0.933 ms with two of each kind, 1.147 with one drain warpgroup.)
template <int DR, bool DET>
struct Roles {
    static constexpr bool GRAD2 = true;                   // two softmax-gradient warpgroups
    static constexpr bool DRAIN2 = DR == 128 || DET;      // two dQ drain warpgroups
    static constexpr int GRAD1_WARP = DRAIN2 ? 16 : 12;   // first warp of the second gradient one
    static constexpr int THREADS = DRAIN2 ? 640 : 512;
    static constexpr int GRAD_THREADS = GRAD2 ? 256 : 128;
    static constexpr int DRAIN_THREADS = DRAIN2 ? 256 : 128;
    static constexpr uint32_t REGS_GRAD = GRAD2 ? 144 : 256;
    static constexpr uint32_t REGS_DRAIN = DRAIN2 ? 56 : 88;
    static constexpr uint32_t REGS_OTHER = 80;
    // registers the split needs at launch (the 640-thread launch has 96 per thread)
    static constexpr int REGS_NEEDED =
        GRAD_THREADS * REGS_GRAD + DRAIN_THREADS * REGS_DRAIN + 128 * REGS_OTHER;
};
constexpr float LOG2E = 1.4426950408889634f;
// Steps (query head of the group x query tile) a masked CTA can list in shared memory.
constexpr int MAX_MASK_STEPS = MASK_BWD_MAX_STEPS;

template <int D>
struct Layout {
    static constexpr int KV_BYTES = BKV * D * 2;          // K or V block
    static constexpr int KV_CHUNK = BKV * 128;            // 128 rows x 64 bf16
    static constexpr int Q_BYTES = BQ * D * 2;            // Q or dO tile
    static constexpr int Q_CHUNK = BQ * 128;              // 64 rows x 64 bf16
    static constexpr int DS_BYTES = BKV * BQ * 2;         // dS^T: 128 rows x 64 bf16
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + KV_BYTES;
    static constexpr int QR_OFF = V_OFF + KV_BYTES;        // ring: [stage][Q | dO]
    static constexpr int DS_OFF = QR_OFF + NSQ * 2 * Q_BYTES;  // [2][dS^T]
    static constexpr int STAT_OFF = DS_OFF + 2 * DS_BYTES;     // [2][lse2 64 | D 64] fp32
    static constexpr int BAR_OFF = STAT_OFF + 2 * 2 * BQ * 4;
    // kv_full, q_full[NSQ], q_empty[NSQ], s_full[2], p_full[2], dq_full[2], dq_empty[2],
    // acc_full, mma_done, kvd[2]
    static constexpr int NBARS = 1 + 2 * NSQ + 8 + 2 + 2;
    static constexpr int TMEM_OFF = BAR_OFF + NBARS * 8;
    static constexpr int ABORT_OFF = TMEM_OFF + 8;
    static constexpr int BYTES = ABORT_OFF + 8 + 1024;
    // General mask: the CTA's list of steps (query head, query tile) its tile mask keeps.
    static constexpr int LIST_OFF = ABORT_OFF + 16;                  // [2] step count, then entries
    static constexpr int BYTES_MASK = LIST_OFF + 4 + MAX_MASK_STEPS * 2 + 1024;
    // Dropout: keep words of the key rows for two steps [2][BKV] (bit c: query q0 + c), written
    // by the dQ drain warps one step ahead, and their km_full[2] / km_empty[2] barriers.
    static constexpr int KEEP_OFF = ABORT_OFF + 16;
    static constexpr int KM_BAR_OFF = KEEP_OFF + 2 * BKV * 8;
    static constexpr int XCH_OFF = KM_BAR_OFF + 4 * 8;   // [2 drain warpgroups][BKV] quad exchange
    static constexpr int BYTES_DROP = XCH_OFF + 2 * BKV * 8 + 1024;
    // Deterministic variant: sent_full[NSENT] / sent_empty[NSENT], the drain warps' hand-over of
    // finished steps to the turn passer.
    static constexpr int SENT_OFF = ABORT_OFF + 16;
    static constexpr int BYTES_DET = SENT_OFF + 2 * NSENT * 8 + 1024;
};

constexpr uint32_t T_DK = 0, T_DV = 128, T_BUF = 256;
constexpr uint32_t B_ST = 0, B_PT = 0, B_DST = 32, B_DPT = 64, B_DQT = 64;

// Bulk tensor reduction (add) of a shared-memory tile into global memory, and the waits on it.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *tm, const void *src, int c0, int c1,
                                                  int c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];\n\t"
        "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(tm)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------- ordered dQ reductions
// The deterministic variant adds the contributions of the key blocks to each 64-row query tile
// of dQ in one fixed order: descending key block.  A counter per query row tile in the workspace,
// zeroed by K2, says how many key blocks have added their part.  The drain warps of key block jb
// wait for their turn (the number of contributing key blocks above jb), add, and hand the step
// to the turn passer (warp 11), which moves the step's counter on with a release reduction: the
// drain warps' reductions, which it acquired through the hand-over barrier, are ordered before
// it, and the wait for them to reach L2 stays off the drain warps' loop.  CTAs of one head are launched in the same descending order,
// so a CTA only ever waits for CTAs launched before it.  All waits are bounded: a wait that runs
// out records FA_ERR_DEVICE_TIMEOUT and sets the call's abort word (after the counters), which
// ends every other CTA's waits at once.
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Warp-collective: true once counter `tile` of dq_sem equals `turn`; false after an abort (this
// CTA's or the call's, the word after the `tiles` counters) or a timeout.
__device__ __forceinline__ bool dq_turn_wait(unsigned *dq_sem, size_t tile, size_t tiles, unsigned turn,
                                             volatile int *abort_flag, unsigned *status) {
    int ok = 1;
    const unsigned *sem = dq_sem + tile * 4;
    if ((threadIdx.x & 31) == 0 && ld_acquire_gpu(sem) != turn) {
        unsigned *call_abort = dq_sem + tiles * 4;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(sem) != turn) {
            if (*abort_flag || ld_relaxed_gpu(call_abort)) {
                *abort_flag = 1;
                ok = 0;
                break;
            }
            if (globaltimer_ns() - t0 > FA_WAIT_NS) {
                *abort_flag = 1;
                atomicExch(call_abort, 1u);
                record_status(status, FA_ERR_DEVICE_TIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int W>
__device__ __forceinline__ void tmem_ld_w(uint32_t taddr, uint32_t (&r)[W]) {
    if constexpr (W == 32) tmem_ld_x32(taddr, r);
    else if constexpr (W == 64) tmem_ld_x64(taddr, r);
    else tmem_ld_x128(taddr, r);
}

// Epilogue of one fp32 accumulator (dK or dV) held in TMEM, thread = key row = TMEM lane:
// row `row` times mul -> bf16 -> the 128B-swizzled [DR / 64][128 rows][64] tile at dst (the
// layout of the K / V operand tiles, which the TMA store reads back).  W columns per TMEM load.
template <int W, int DR>
__device__ __forceinline__ void stage_acc_rows(uint32_t tsrc, float mul, uint8_t *dst, int row,
                                               bool zero) {
#pragma unroll
    for (int c0 = 0; c0 < DR; c0 += W) {
        uint32_t a[W];
        tmem_ld_w<W>(tsrc + c0, a);
        if (zero) {                                  // (a masked key block with no step)
#pragma unroll
            for (int k = 0; k < W; ++k) a[k] = 0u;
        }
#pragma unroll
        for (int c = 0; c < W; c += 8) {
            const int col = c0 + c;
            uint4 w4;
            w4.x = pack_bf16x2(__uint_as_float(a[c + 0]) * mul, __uint_as_float(a[c + 1]) * mul);
            w4.y = pack_bf16x2(__uint_as_float(a[c + 2]) * mul, __uint_as_float(a[c + 3]) * mul);
            w4.z = pack_bf16x2(__uint_as_float(a[c + 4]) * mul, __uint_as_float(a[c + 5]) * mul);
            w4.w = pack_bf16x2(__uint_as_float(a[c + 6]) * mul, __uint_as_float(a[c + 7]) * mul);
            uint8_t *rowp = dst + (col / 64) * (BKV * 128) + row * 128;
            *reinterpret_cast<uint4 *>(rowp + ((((col % 64) / 8) ^ (row & 7)) << 4)) = w4;
        }
    }
}

template <bool CAUSAL>
__device__ __forceinline__ int first_q_tile(int jb) {
    return CAUSAL ? (jb * BKV) / BQ : 0;
}

// MASK = true: the general mask mk on top of the causal rule.  The CTA lists, before the roles
// split, the steps whose tile its mask keeps (rows past the valid length and key blocks past it
// drop out); a key block with no step at all gets dK = dV = 0.
// DROP = true: dropout on P (fa_philox.cuh has the keep rule): dV takes P Z / (1 - p) and
// dS = P (Z / (1 - p) dP - D).  The dQ drain warps, idle for most of a step, generate the keep
// words one step ahead into shared memory: one Philox call gives the decisions of the four keys
// of a quad at one query, so each lane of a quad calls it for a quarter of the queries and the
// quad exchanges its four 64-bit results through shared memory (shuffles measured 4x slower).
// DET = true: the deterministic variant (ordered dQ reductions, above); dq_sem holds B * Hq *
// ceil(N / 64) * 4 counters followed by the call's abort word.
template <int D, int DR, bool CAUSAL, bool MASK, bool DROP, bool DET>
__global__ void __launch_bounds__((Roles<DR, DET>::THREADS), 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                    const __grid_constant__ CUtensorMap tmdQ,
                    const float *__restrict__ LSE, const float *__restrict__ Dvec,
                    float *__restrict__ dQacc, int Hq, int Hkv, int N, int BHkv, int HC,
                    float scale, float scale_log2, const MaskArgs mk, const DropoutArgs drop,
                    unsigned *dq_sem, unsigned *status) {
    static_assert(!(MASK && DROP), "one variant at a time");
    static_assert(!(DET && (MASK || DROP)), "the deterministic variant has no mask or dropout");
    // Laid out for d = 128.  With a real head dim DR = 64 only the first 64-column chunk of Q,
    // dO and V is loaded and S^T, dP^T (K dim), dV and dK (N) run over DR; dQ^T keeps M = 128
    // (the MMA's row count), its upper rows coming from K's second chunk, which the 64-wide
    // tensor map fills with zeros, so only the dQ reductions see DR there.
    static_assert(D == 128, "the bf16 backward main loop is laid out for d = 128");
    static_assert(DR == 64 || DR == 128, "real head dim 64 or 128");
    // At head dim 64 dQ leaves through bulk tensor reductions (see the drain warps); at 128 the
    // per-element reductions measured faster (a staged 64 x 128 tile: 0.944 ms against 0.917).
    // The deterministic variant uses the per-element reductions at both head dims, so that
    // passing a turn only has to order plain global reductions.
    constexpr bool DQ_TMA = DR == 64 && !DET;
    // The dK / dV epilogue: split between the gradient warps (dK) and the drain warps (dV) where
    // the drain warps' per-step work is the short staged reduction (DR = 64); at DR = 128 the
    // drain warps are still busy with the last step's per-element reductions then.
    constexpr bool SPLIT_EPI = DQ_TMA;
    using R = Roles<DR, DET>;
    // Outside the deterministic variant (whose warp 11 passes the dQ turns): S^T and dP^T are
    // issued by two threads (warps 9 and 11), each as soon as its own TMEM columns are free (S^T
    // after dV / dK of the step two before, dP^T after the drain's read of its dQ^T): 2-3% faster
    // than one thread issuing both at either head dim.
    constexpr bool SPLIT_A = !DET;
    // TMEM columns (within a buffer) of P^T and dS^T for the 16-query chunk kk: one warpgroup
    // writes P^T over S^T's first 32 columns and dS^T over the next 32; two write theirs over
    // their own half of S^T (queries 32 h .. 32 h + 31: P^T at 32 h, dS^T at 32 h + 16), so
    // neither overwrites S^T columns the other has not read yet.
    auto pt_col = [](int kk) -> uint32_t {
        return R::GRAD2 ? (kk >> 1) * 32 + (kk & 1) * 8 : B_PT + kk * 8;
    };
    auto dst_col = [](int kk) -> uint32_t {
        return R::GRAD2 ? (kk >> 1) * 32 + 16 + (kk & 1) * 8 : B_DST + kk * 8;
    };
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *kv_full = bars;
    uint64_t *q_full = bars + 1;
    uint64_t *q_empty = q_full + NSQ;
    uint64_t *s_full = q_empty + NSQ;      // [2]
    uint64_t *p_full = s_full + 2;         // [2]
    uint64_t *dq_full = p_full + 2;        // [2]
    uint64_t *dq_empty = dq_full + 2;      // [2]
    uint64_t *acc_full = dq_empty + 2;
    uint64_t *mma_done = acc_full + 1;
    uint64_t *kvd = mma_done + 1;          // [2] dV / dK of the buffer's last step done
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::TMEM_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ABORT_OFF);
    float *stat = reinterpret_cast<float *>(smem + L::STAT_OFF);
    uint64_t *keep_words = reinterpret_cast<uint64_t *>(smem + L::KEEP_OFF);
    uint64_t *km_full = reinterpret_cast<uint64_t *>(smem + L::KM_BAR_OFF);
    uint64_t *km_empty = km_full + 2;
    uint64_t *sent_full = reinterpret_cast<uint64_t *>(smem + L::SENT_OFF);   // [NSENT]
    uint64_t *sent_empty = sent_full + NSENT;                                // [NSENT]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = Hq / Hkv;
    const int nkb = (N + BKV - 1) / BKV;
    // rows of Q, dO, LSE, D and the dQ accumulator: the extent debug builds check accesses against
    const long long rows_total = static_cast<long long>(BHkv) * G * N;
    (void)rows_total;
    // Work item: (key block jb, batch * KV head).  KV heads go in chunks of HC (about one wave),
    // so the Q / dO / dQ accumulator rows of the heads in flight stay in L2; inside a chunk the
    // small jb (most query tiles under causal masking) go first, except in the deterministic
    // variant, whose dQ reduction order (descending jb) the launch order has to follow.
    const int chunk = blockIdx.x / (HC * nkb);
    const int in_chunk = blockIdx.x - chunk * HC * nkb;
    const int hc = min(HC, BHkv - chunk * HC);
    const int bkv = chunk * HC + in_chunk % hc;          // b * Hkv + hk
    const int jb = DET ? nkb - 1 - in_chunk / hc : in_chunk / hc;
    const int b = bkv / Hkv, hk = bkv % Hkv;
    const int nq = (N + BQ - 1) / BQ;
    const int i0 = first_q_tile<CAUSAL>(jb);
    int lq = N, lk = N;                         // valid query rows / keys of the batch
    if (MASK) {
        if (mk.q_len) lq = min(max(__ldg(mk.q_len + b), 0), N);
        if (mk.k_len) lk = min(max(__ldg(mk.k_len + b), 0), N);
    }
    const int tiles_per_head = MASK ? max(0, (lq + BQ - 1) / BQ - i0) : nq - i0;
    uint16_t *steps = reinterpret_cast<uint16_t *>(smem + L::LIST_OFF + 4);
    if (MASK && warp == 0) {
        // steps (g, i) in the unmasked order, kept if the key block is inside the valid length
        // and the tile mask lets query tile i / 2 of head g see key block jb
        const int cand = (jb * BKV < lk) ? G * tiles_per_head : 0;
        int count = 0;
        for (int c0 = 0; c0 < cand; c0 += 32) {
            const int c = c0 + lane;
            bool keep = false;
            if (c < cand) {
                keep = true;
                if (mk.block_mask) {
                    const int g = c / tiles_per_head, i = i0 + c % tiles_per_head;
                    const int hq = hk * G + g;
                    const int h = mk.mask_heads == 1 ? 0 : (mk.mask_heads == BHkv * G ? b * Hq + hq : hq);
                    keep = __ldg(mk.block_mask + (static_cast<size_t>(h) * nkb + (i * BQ) / BKV) * nkb + jb) != 0;
                }
            }
            const unsigned ball = __ballot_sync(0xffffffffu, keep);
            if (keep && count + __popc(ball & ((1u << lane) - 1u)) < MAX_MASK_STEPS)
                steps[count + __popc(ball & ((1u << lane) - 1u))] = static_cast<uint16_t>(c);
            count += __popc(ball);
        }
        if (lane == 0) *reinterpret_cast<int *>(smem + L::LIST_OFF) = min(count, MAX_MASK_STEPS);
    }

    // The loads that depend on nothing: K / V of the block and, without a general mask (the step
    // list then follows from the shape), Q / dO of the first ring stages, issued by the TMA
    // thread right after it sets up the barriers, before TMEM allocation and the block barrier.
    auto issue_kv = [&]() {
        // K: both chunks (at DR = 64 the second is zero fill, the upper rows of dQ^T's A
        // operand); V: only the real columns (its second chunk stages dQ at DR = 64)
        mbar_arrive_expect_tx(kv_full, L::KV_BYTES + (DR / 64) * L::KV_CHUNK);
        for (int ch = 0; ch < D / 64; ++ch)
            tma_load_3d(smem + L::K_OFF + ch * L::KV_CHUNK, &tmK, ch * 64, jb * BKV, bkv, kv_full);
        for (int ch = 0; ch < DR / 64; ++ch)
            tma_load_3d(smem + L::V_OFF + ch * L::KV_CHUNK, &tmV, ch * 64, jb * BKV, bkv, kv_full);
    };
    auto issue_q = [&](int s, int g, int i) {
        const int st = s % NSQ;
        const int bhq = b * Hq + hk * G + g;
        mbar_arrive_expect_tx(&q_full[st], 2 * (DR / 64) * L::Q_CHUNK);
        uint8_t *qdst = smem + L::QR_OFF + st * 2 * L::Q_BYTES;
        for (int ch = 0; ch < DR / 64; ++ch) {
            tma_load_3d(qdst + ch * L::Q_CHUNK, &tmQ, ch * 64, i * BQ, bhq, &q_full[st]);
            tma_load_3d(qdst + L::Q_BYTES + ch * L::Q_CHUNK, &tmdO, ch * 64, i * BQ, bhq, &q_full[st]);
        }
    };
    const int early_q = MASK ? 0 : min(G * tiles_per_head, NSQ);
    if (threadIdx.x == WARP_TMA * 32) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < NSQ; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s_full[k], SPLIT_A ? 2 : 1);
            mbar_init(&p_full[k], R::GRAD_THREADS);
            mbar_init(&dq_full[k], 1);
            mbar_init(&dq_empty[k], R::DRAIN_THREADS);
        }
        mbar_init(acc_full, 1);
        mbar_init(mma_done, SPLIT_A ? 3 : 2);            // one commit from each issuer
        mbar_init(&kvd[0], 1);
        mbar_init(&kvd[1], 1);
        if (DROP) {
            uint64_t *kb = reinterpret_cast<uint64_t *>(smem + L::KM_BAR_OFF);
            for (int k = 0; k < 4; ++k)                               // full, empty
                mbar_init(&kb[k], k < 2 ? R::DRAIN_THREADS : R::GRAD_THREADS);
        }
        if (DET) {
            for (int k = 0; k < NSENT; ++k) {
                mbar_init(&sent_full[k], R::DRAIN_THREADS);
                mbar_init(&sent_empty[k], 1);
            }
        }
        *abort_flag = 0;
        fence_mbar_init();
        if (!MASK) {
            issue_kv();
            for (int s = 0; s < early_q; ++s) issue_q(s, s / tiles_per_head, i0 + s % tiles_per_head);
        }
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // steps of this CTA: every (query head, tile at or below the diagonal), or the listed ones
    const int T = MASK ? *reinterpret_cast<volatile int *>(smem + L::LIST_OFF) : G * tiles_per_head;
    auto step_tile = [&](int s, int &g, int &i) {
        const int e = MASK ? static_cast<int>(steps[s]) : s;
        g = e / tiles_per_head;
        i = i0 + e % tiles_per_head;
    };
    const int qend = MASK ? lq : N, kend = MASK ? lk : N;   // rows / keys past these are masked

    // Each role branch starts with its register budget and ends with its own copy of the final
    // barrier, so no code is shared between budgets.
    if (warp >= 8 && warp < 12) {
        regs_dec<R::REGS_OTHER>();
      if (warp == WARP_TMA) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // (a masked key block may have no step; without a mask K / V and the first stages
            // are already on their way)
            if (MASK && T > 0) issue_kv();
            int issued = early_q;
            bool injected = false;
            for (int s = early_q; s < T; ++s) {
                const int st = s % NSQ, rnd = s / NSQ;
                if (!mbar_wait(&q_empty[st], (rnd & 1) ^ 1, abort_flag, status)) break;
#ifdef FA_FAULT_INJECT
                // Test builds only: CTA 0 stops delivering Q / dO after the ring's first fill, so
                // the S^T / dP^T issuer's bounded wait runs out, every role unwinds and
                // FA_ERR_DEVICE_TIMEOUT is recorded.
                if (blockIdx.x == 0 && s == NSQ) {
                    injected = true;
                    break;
                }
#endif
                int g, i;
                step_tile(s, g, i);
                issue_q(s, g, i);
                ++issued;
            }
            if (*abort_flag || injected) {
                for (int s = max(0, issued - NSQ); s < issued; ++s)
                    mbar_drain(&q_full[s % NSQ], (s / NSQ) & 1);
                if (T > 0) mbar_drain(kv_full, 0);
            }
        }
    } else if (warp == WARP_MMA || warp == WARP_MMA2 || (SPLIT_A && warp == WARP_PASS)) {
        // ------------------------------------------------------------------ MMA issuers
        // Two threads issue (three with SPLIT_A): one the S^T / dP^T products of step s + 1 as
        // soon as their buffer is free (with SPLIT_A one thread each), the other this step's
        // dQ^T, dV and dK as soon as the gradient warps are done, so neither stream queues
        // behind the other in one thread.  The reuse of a buffer that
        // one in-order stream would order by itself is ordered by barriers: S^T(s+2) waits for
        // dV / dK(s) (kvd, P^T and dS^T are their operands) and for the drain's read of dQ^T(s).
        if (lane == 0) {
            constexpr uint32_t IDESC_SP = idesc_bf16(BKV, BQ, false, false);   // S^T, dP^T
            constexpr uint32_t IDESC_KV = idesc_bf16(BKV, DR, false, true);    // dV, dK
            constexpr uint32_t IDESC_DQ = idesc_bf16(D, BQ, true, true);       // dQ^T
            // Descriptors are built once; each k-step only moves the start address.
            const uint64_t dk_k = sdesc_sw128(smem_u32(smem + L::K_OFF), 16, 1024);        // K, K-major
            const uint64_t dv_k = sdesc_sw128(smem_u32(smem + L::V_OFF), 16, 1024);        // V, K-major
            const uint64_t dk_mn = sdesc_sw128(smem_u32(smem + L::K_OFF), L::KV_CHUNK, 1024);  // K, MN-major
            const uint64_t dq_k = sdesc_sw128(smem_u32(smem + L::QR_OFF), 16, 1024);       // ring, K-major
            const uint64_t dq_mn = sdesc_sw128(smem_u32(smem + L::QR_OFF), L::Q_CHUNK, 1024);  // ring, MN-major
            const uint64_t dds = sdesc_sw128(smem_u32(smem + L::DS_OFF), L::DS_BYTES, 1024);   // dS^T
            auto ring_off = [&](int s) { return static_cast<uint32_t>((s % NSQ) * 2 * L::Q_BYTES); };
            bool ok = T > 0;
            if (warp != WARP_MMA2) {
                const bool do_s = !SPLIT_A || warp == WARP_MMA, do_dp = !SPLIT_A || warp == WARP_PASS;
                // S^T(s) and dP^T(s) into buffer s & 1
                ok = ok && mbar_wait(kv_full, 0, abort_flag, status);
                for (int s = 0; s < T && ok; ++s) {
                    const int bsel = s & 1;
                    if (!mbar_wait(&q_full[s % NSQ], (s / NSQ) & 1, abort_flag, status)) break;
                    if (s >= 2 && ((do_s && !mbar_wait(&kvd[bsel], ((s - 2) >> 1) & 1, abort_flag, status)) ||
                                   (do_dp && !mbar_wait(&dq_empty[bsel], ((s - 2) >> 1) & 1, abort_flag, status))))
                        break;
                    tc_fence_after();
                    const uint64_t dq = sdesc_add(dq_k, ring_off(s));
                    const uint64_t ddo = sdesc_add(dq, L::Q_BYTES);
                    const uint32_t buf = tmem + T_BUF + bsel * 128;
                    if (do_s) {
#pragma unroll
                        for (int kk = 0; kk < DR / 16; ++kk) {
                            const uint32_t oa = (kk >> 2) * L::KV_CHUNK + (kk & 3) * 32;
                            const uint32_t ob = (kk >> 2) * L::Q_CHUNK + (kk & 3) * 32;
                            mma_ss(buf + B_ST, sdesc_add(dk_k, oa), sdesc_add(dq, ob), IDESC_SP, kk > 0);
                        }
                    }
                    if (do_dp) {
#pragma unroll
                        for (int kk = 0; kk < DR / 16; ++kk) {
                            const uint32_t oa = (kk >> 2) * L::KV_CHUNK + (kk & 3) * 32;
                            const uint32_t ob = (kk >> 2) * L::Q_CHUNK + (kk & 3) * 32;
                            mma_ss(buf + B_DPT, sdesc_add(dv_k, oa), sdesc_add(ddo, ob), IDESC_SP, kk > 0);
                        }
                    }
                    mma_commit(&s_full[bsel]);     // (one commit from each S^T / dP^T issuer)
                }
            } else {
                for (int s = 0; s < T && ok; ++s) {
                    const int bsel = s & 1;
                    const uint32_t buf = tmem + T_BUF + bsel * 128;
                    // the gradient warps have staged P^T / dS^T (and so S^T(s), dP^T(s) are done)
                    if (!mbar_wait(&p_full[bsel], (s >> 1) & 1, abort_flag, status)) break;
                    tc_fence_after();
                    // dQ^T = K^T dS^T first (A = K MN-major, B = dS^T MN-major, K dim = 128 keys),
                    // so the drain warps read it out while dV / dK run.
                    const uint64_t dsb = sdesc_add(dds, bsel * L::DS_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BKV / 16; ++kk)
                        mma_ss(buf + B_DQT, sdesc_add(dk_mn, kk * 2048), sdesc_add(dsb, kk * 2048),
                               IDESC_DQ, kk > 0);
                    mma_commit(&dq_full[bsel]);
                    const uint64_t dqm = sdesc_add(dq_mn, ring_off(s));
                    const uint64_t dom = sdesc_add(dqm, L::Q_BYTES);
                    // dV += P^T dO ; dK += dS^T Q   (B operands MN-major: d contiguous).  The TMEM
                    // columns of P^T / dS^T for queries 16 kk .. 16 kk + 15: with two gradient
                    // warpgroups each half of the queries has its own 32 columns (P^T, then dS^T).
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + T_DV, buf + pt_col(kk), sdesc_add(dom, kk * 2048), IDESC_KV,
                               (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + T_DK, buf + dst_col(kk), sdesc_add(dqm, kk * 2048), IDESC_KV,
                               (s > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&kvd[bsel]);
                    mma_commit(&q_empty[s % NSQ]);
                }
                mma_commit(acc_full);
            }
            // Nothing either issued may still be running when TMEM is released.
            mma_commit(mma_done);
            mbar_drain(mma_done, 0);
        }
      } else if (DET && warp == WARP_PASS) {
        // ------------------------------------------------------------------ dQ turn passer
        // Takes every step the drain warps have handed over (at least one), moves those steps'
        // counters on and frees their hand-over slots.
        if (lane == 0) {
            int s = 0;
            while (s < T) {
                if (!mbar_wait(&sent_full[s % NSENT], (s / NSENT) & 1, abort_flag, status)) break;
                int e = s + 1;
                while (e < T && e - s < NSENT && mbar_try_wait(&sent_full[e % NSENT], (e / NSENT) & 1))
                    ++e;
                for (int t = s; t < e; ++t) {
                    int g, i;
                    step_tile(t, g, i);
                    unsigned *sem = dq_sem + (static_cast<size_t>(b * Hq + hk * G + g) * nq + i) * 4;
                    // a release: the drain warps' reductions, acquired through sent_full, are
                    // ordered before the counter moves (cheaper here than a fence and a relaxed add)
                    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(sem) : "memory");
                    mbar_arrive(&sent_empty[t % NSENT]);
                }
                s = e;
            }
            if (*abort_flag) atomicExch(dq_sem + static_cast<size_t>(BHkv) * G * nq * 4, 1u);
        }
      }
        tc_fence_before();
        __syncthreads();
        if (warp == WARP_MMA) {
            __syncwarp();
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    } else if (warp < 4 || (R::GRAD2 && warp >= R::GRAD1_WARP)) {
        regs_inc<R::REGS_GRAD>();
        // ------------------------------------------------------------------ P^T / dS^T warps
        const int krow = (warp & 3) * 32 + lane;    // key row within the block = TMEM lane
        const int key = jb * BKV + krow;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        // queries of each step this warp handles: NQ from qoff (two warpgroups: halves)
        constexpr int NQ = R::GRAD2 ? BQ / 2 : BQ;
        const int gh = R::GRAD2 && warp >= R::GRAD1_WARP;
        const int qoff = gh * NQ;
        const uint64_t c2 = f2_pack(scale_log2, scale_log2);
        bool ok = true;
        // Statistics of this warpgroup's NQ queries of step s: thread t < NQ holds
        // LSE_{qoff+t} * log2 e, NQ <= t < 2 NQ holds D_{qoff+t-NQ} (slot sidx of the step's stat
        // buffer; with two warpgroups each fills and reads only its own half, so they never
        // wait for each other).  They are loaded one step ahead so the global-load latency
        // overlaps a whole step instead of sitting between the MMAs and this step's work.
        const int sidx = krow < NQ ? qoff + krow : (krow < 2 * NQ ? BQ + qoff + krow - NQ : -1);
        auto load_stat = [&](int s) -> float {
            if (s >= T || sidx < 0) return 0.f;
            int g, i;
            step_tile(s, g, i);
            const int bhq = b * Hq + hk * G + g;
            const int q = i * BQ + qoff + krow % NQ;
            if (q < qend && !in_bounds(static_cast<long long>(bhq) * N + q, rows_total, status))
                return 0.f;                                  // (debug builds: reported)
            if (krow < NQ) {
                if (q >= qend) return INFINITY;
                const float lse = LSE[static_cast<size_t>(bhq) * N + q];
                // a row with no allowed key (LSE = -inf) gets P = 0 from +inf
                return (MASK && lse == -INFINITY) ? INFINITY : lse * LOG2E;
            }
            return (q < qend) ? Dvec[static_cast<size_t>(bhq) * N + q] : 0.f;
        };
        float v_next = load_stat(0);
        for (int s = 0; s < T; ++s) {
            int g, i;
            step_tile(s, g, i);
            const int q0 = i * BQ;
            const int bsel = s & 1;
            const uint32_t buf = tmem + lane_off + T_BUF + bsel * 128;
            float *sbuf = stat + bsel * 2 * BQ;
            const float v = v_next;
            v_next = load_stat(s + 1);
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&s_full[bsel], (s >> 1) & 1, abort_flag, status));
            if (sidx >= 0) sbuf[sidx] = v;
            // executed by all warps of the warpgroup every step (even after a failed wait) so the
            // counts match
            named_barrier_sync(gh ? 6 : 1, 128);
            uint64_t keep_s = ~0ull;
            if constexpr (DROP) {
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&km_full[bsel], (s >> 1) & 1, abort_flag, status));
                if (ok) {
                    keep_s = keep_words[bsel * BKV + krow];
                    mbar_arrive(&km_empty[bsel]);
                }
            }
            if (ok) {
                tc_fence_after();
                // P^T in place over the S^T registers, then dS^T with dP^T streamed in 32-query
                // pieces (this warp's queries qoff .. qoff + NQ - 1 of the step)
                uint32_t sr[NQ];
                if constexpr (NQ == 32) tmem_ld_x32(buf + B_ST + qoff, sr);
                else tmem_ld_x64(buf + B_ST, sr);
                const bool need_mask = (CAUSAL && q0 < jb * BKV + BKV) || (q0 + BQ > qend) ||
                                       (jb * BKV + BKV > kend);
                const float4 *l4 = reinterpret_cast<const float4 *>(sbuf + qoff);
                const float4 *d4 = reinterpret_cast<const float4 *>(sbuf + BQ + qoff);
                float pf[NQ];
#pragma unroll
                for (int c = 0; c < NQ; c += 4) {
                    const float4 lse = l4[c >> 2];
                    const float2 pa = f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                                       c2, f2_pack(-lse.x, -lse.y)));
                    const float2 pb = f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])),
                                                       c2, f2_pack(-lse.z, -lse.w)));
                    pf[c] = ex2_approx(pa.x);
                    pf[c + 1] = ex2_approx(pa.y);
                    pf[c + 2] = ex2_approx(pb.x);
                    pf[c + 3] = ex2_approx(pb.y);
                }
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < NQ; ++c) {
                        const int q = q0 + qoff + c;
                        if ((CAUSAL && key > q) || q >= qend || key >= kend) pf[c] = 0.f;
                    }
                }
                uint32_t pp[NQ / 2], dd[NQ / 2];
                uint64_t keep = ~0ull;                  // bit c: query q0 + c keeps this key
                if constexpr (DROP) keep = keep_s >> qoff;
                auto kept = [&](int c) -> bool { return !DROP || ((keep >> c) & 1ull); };
#pragma unroll
                for (int c = 0; c < NQ; c += 2) {
                    if constexpr (DROP)
                        pp[c >> 1] = pack_bf16x2(kept(c) ? pf[c] * drop.rscale : 0.f,
                                                 kept(c + 1) ? pf[c + 1] * drop.rscale : 0.f);
                    else
                        pp[c >> 1] = pack_bf16x2(pf[c], pf[c + 1]);
                }
#pragma unroll
                for (int h = 0; h < NQ / 32; ++h) {
                    uint32_t dr[32];
                    tmem_ld_x32(buf + B_DPT + qoff + 32 * h, dr);
                    if constexpr (DROP) {
                        // dP of a dropped pair does not reach P; a kept one is scaled by 1/(1-p)
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            dr[c] = __float_as_uint(kept(32 * h + c) ? __uint_as_float(dr[c]) * drop.rscale : 0.f);
                    }
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 dv = d4[(32 * h + c) >> 2];
                        const float2 da = f2_unpack(f2_mul(
                            f2_pack(pf[32 * h + c], pf[32 * h + c + 1]),
                            f2_add(f2_pack(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])),
                                   f2_pack(-dv.x, -dv.y))));
                        const float2 db = f2_unpack(f2_mul(
                            f2_pack(pf[32 * h + c + 2], pf[32 * h + c + 3]),
                            f2_add(f2_pack(__uint_as_float(dr[c + 2]), __uint_as_float(dr[c + 3])),
                                   f2_pack(-dv.z, -dv.w))));
                        dd[(32 * h + c) >> 1] = pack_bf16x2(da.x, da.y);
                        dd[((32 * h + c) >> 1) + 1] = pack_bf16x2(db.x, db.y);
                    }
                }
                if constexpr (NQ == 32) {
                    tmem_st_x16(buf + pt_col(2 * gh), pp);
                    tmem_st_x16(buf + dst_col(2 * gh), dd);
                } else {
                    tmem_st_x32(buf + B_PT, pp);
                    tmem_st_x32(buf + B_DST, dd);
                }
                // dS^T row -> smem buffer (128B-swizzled, MN-major B operand of the dQ^T product):
                // this warp's 16-byte chunks qoff / 8 ..
                uint8_t *ds_row = smem + L::DS_OFF + bsel * L::DS_BYTES + krow * 128;
#pragma unroll
                for (int u = 0; u < NQ / 8; ++u) {
                    uint4 w4 = make_uint4(dd[4 * u], dd[4 * u + 1], dd[4 * u + 2], dd[4 * u + 3]);
                    *reinterpret_cast<uint4 *>(ds_row + (((u + qoff / 8) ^ (krow & 7)) << 4)) = w4;
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&p_full[bsel]);
            }
        }
        // epilogue: scale * dK rows (and dV rows unless the drain warps take them) -> bf16 ->
        // smem over K (V) -> TMA store.  The barrier is passed by all four warps whatever their
        // wait returned, so its count always matches.
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, status));
        if (ok) {
            tc_fence_after();
            // two gradient warpgroups: the first stages dK, the second dV (64 columns per TMEM
            // load in their register budget)
            if constexpr (R::GRAD2) {
                if (gh == 0)
                    stage_acc_rows<64, DR>(tmem + lane_off + T_DK, scale, smem + L::K_OFF, krow, MASK && T == 0);
                else if (!SPLIT_EPI)
                    stage_acc_rows<64, DR>(tmem + lane_off + T_DV, 1.f, smem + L::V_OFF, krow, MASK && T == 0);
            } else {
                stage_acc_rows<DR, DR>(tmem + lane_off + T_DK, scale, smem + L::K_OFF, krow, MASK && T == 0);
                if constexpr (!SPLIT_EPI)
                    stage_acc_rows<DR, DR>(tmem + lane_off + T_DV, 1.f, smem + L::V_OFF, krow, MASK && T == 0);
            }
        }
        fence_proxy_async_smem();
        named_barrier_sync(R::GRAD2 ? 4 + gh : 1, 128);
        if (ok && krow == 0 && !*abort_flag) {
            const bool st_dk = !R::GRAD2 || gh == 0, st_dv = !SPLIT_EPI && (!R::GRAD2 || gh == 1);
            for (int ch = 0; ch < DR / 64; ++ch) {
                if (st_dk) tma_store_3d(&tmdK, smem + L::K_OFF + ch * L::KV_CHUNK, ch * 64, jb * BKV, bkv);
                if (st_dv) tma_store_3d(&tmdV, smem + L::V_OFF + ch * L::KV_CHUNK, ch * 64, jb * BKV, bkv);
            }
            tma_store_commit_and_wait_read();
        }
        tc_fence_before();
        __syncthreads();
    } else {
        regs_dec<R::REGS_DRAIN>();
        // ------------------------------------------------------------------ dQ drain warps
        const int wq = warp & 3;
        // with two drain warpgroups: which half of a step's 64 query columns this warp reduces
        const int half = R::DRAIN2 && warp >= 12;
        const int dcol = wq * 32 + lane;            // column of dQ = TMEM lane of dQ^T
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        // Dropout: keep words of step s for key row dcol of this block (the same lane <-> key
        // row layout as the gradient warps, so a quad of lanes is a quad of keys).
        auto make_keep = [&](int s) {
            int g, i;
            step_tile(s, g, i);
            const int bhq = b * Hq + hk * G + g;
            const int q0 = i * BQ;
            const int qd = lane & 3;                // this lane's key within its quad
            const uint32_t mkey = static_cast<uint32_t>(jb * BKV + dcol) >> 2;
            // bit 4t + k of `mine`: query q0 + 4t + qd keeps key 4 mkey + k (t over this drain
            // warpgroup's half of the queries with two of them)
            constexpr int NT = R::DRAIN2 ? BQ / 8 : BQ / 4;
            uint64_t mine = 0ull;
#pragma unroll
            for (int t = half * NT; t < (half + 1) * NT; ++t) {
                const uint4 w = dropout_words(drop, mkey, static_cast<uint32_t>(q0 + 4 * t + qd),
                                              static_cast<uint32_t>(bhq));
                mine |= (static_cast<uint64_t>(w.x < drop.thresh) << (4 * t)) |
                        (static_cast<uint64_t>(w.y < drop.thresh) << (4 * t + 1)) |
                        (static_cast<uint64_t>(w.z < drop.thresh) << (4 * t + 2)) |
                        (static_cast<uint64_t>(w.w < drop.thresh) << (4 * t + 3));
            }
            uint64_t *xch = reinterpret_cast<uint64_t *>(smem + L::XCH_OFF) + half * BKV;
            xch[dcol] = mine;
            __syncwarp();
            // from quad lane src, the bits of this lane's key (positions 4t + qd) are queries 4t + src
            uint64_t keep = 0ull;
#pragma unroll
            for (int src = 0; src < 4; ++src)
                keep |= ((xch[(dcol & ~3) + src] >> qd) & 0x1111111111111111ull) << src;
            __syncwarp();                           // the exchange words are rewritten next call
            if constexpr (R::DRAIN2)         // this warpgroup's 32 queries: one half of the word
                reinterpret_cast<uint32_t *>(keep_words + (s & 1) * BKV + dcol)[half] =
                    static_cast<uint32_t>(keep >> (32 * half));
            else
                keep_words[(s & 1) * BKV + dcol] = keep;
            mbar_arrive(&km_full[s & 1]);
        };
        if (DROP && T > 0) make_keep(0);
        if constexpr (DQ_TMA) {
            // After a failed wait a warp keeps stepping without work, so the named barriers of the
            // staged reductions always see both of their warps.
            bool dok = true;
            for (int s = 0; s < T; ++s) {
                if constexpr (DROP) {
                    // the keep words of the next step, into the buffer step s-1 has released
                    if (s + 1 < T && dok) {
                        const int sn = s + 1;
                        if (sn >= 2)
                            dok = __all_sync(0xffffffffu, mbar_wait(&km_empty[sn & 1], ((sn - 2) >> 1) & 1, abort_flag, status));
                        if (dok) make_keep(sn);
                    }
                }
                int g, i;
                step_tile(s, g, i);
                const int bhq = b * Hq + hk * G + g;
                const int q0 = i * BQ;
                const int bsel = s & 1;
                if (dok) dok = __all_sync(0xffffffffu, mbar_wait(&dq_full[bsel], (s >> 1) & 1, abort_flag, status));
                uint32_t a[64];
                if (dok) {
                    tc_fence_after();
                    tmem_ld_x64(tmem + lane_off + T_BUF + bsel * 128 + B_DQT, a);
                    tc_fence_before();
                    mbar_arrive(&dq_empty[bsel]);
                }
                // The 64 x 64 tile of dQ (query rows, d columns) goes to the accumulator as one
                // bulk reduction from shared memory, V's unused second chunk (per-element
                // reductions measured 25% of the step's time at d = 64).  Rows past the sequence
                // end are clipped by the tensor map; rows past a mask's valid length hold zeros.
                // Lanes 64-127 (K's zero-filled half of dQ^T) sit out.
                if (wq < 2) {
                    float *tile = reinterpret_cast<float *>(smem + L::V_OFF + L::KV_CHUNK);
                    // the previous tile's reductions have finished reading shared memory
                    if (threadIdx.x == 128) bulk_wait_read();
                    named_barrier_sync(2, 64);
                    float *trow = tile + dcol;
                    if (dok) {
#pragma unroll
                        for (int c = 0; c < BQ; ++c) trow[c * 64] = __uint_as_float(a[c]) * scale;
                    }
                    fence_proxy_async_smem();
                    named_barrier_sync(2, 64);
                    if (threadIdx.x == 128 && dok && !*abort_flag) tma_reduce_add_3d(&tmdQ, tile, 0, q0, bhq);
                }
            }
        } else {
            // (no named barrier inside: a warp whose wait failed just leaves)
            for (int s = 0; s < T; ++s) {
                if constexpr (DROP) {
                    // the keep words of the next step, into the buffer step s-1 has released
                    if (s + 1 < T) {
                        const int sn = s + 1;
                        if (sn >= 2 &&
                            !__all_sync(0xffffffffu, mbar_wait(&km_empty[sn & 1], ((sn - 2) >> 1) & 1, abort_flag, status)))
                            break;
                        make_keep(sn);
                    }
                }
                int g, i;
                step_tile(s, g, i);
                const int bhq = b * Hq + hk * G + g;
                const int q0 = i * BQ;
                const int bsel = s & 1;
                // (DR = 64, deterministic variant: warps 6-7 hold K's zero-filled half of dQ^T)
                if constexpr (DET) {
                    // a free hand-over slot (the passer at most NSENT steps behind), then this tile's
                    // turn: key blocks jb + 1 .. jtop add to it before this one; both waited for
                    // before the tile is read from TMEM, while the tensor core forms it
                    if (s >= NSENT &&
                        !__all_sync(0xffffffffu, mbar_wait(&sent_empty[s % NSENT], ((s / NSENT) - 1) & 1,
                                                           abort_flag, status)))
                        break;
                    const int jtop = CAUSAL ? min(nkb - 1, (i * BQ) / BKV) : nkb - 1;
                    if (dcol < DR &&
                        !dq_turn_wait(dq_sem, static_cast<size_t>(bhq) * nq + i,
                                      static_cast<size_t>(BHkv) * G * nq,
                                      static_cast<unsigned>(jtop - jb), abort_flag, status))
                        break;
                }
                if (!__all_sync(0xffffffffu, mbar_wait(&dq_full[bsel], (s >> 1) & 1, abort_flag, status))) break;
                tc_fence_after();
                constexpr int NC = R::DRAIN2 ? BQ / 2 : BQ;   // query columns per drain warp
                const int c0 = half * NC;
                uint32_t a[NC];
                if constexpr (NC == 32) tmem_ld_x32(tmem + lane_off + T_BUF + bsel * 128 + B_DQT + c0, a);
                else tmem_ld_x64(tmem + lane_off + T_BUF + bsel * 128 + B_DQT, a);
                tc_fence_before();
                mbar_arrive(&dq_empty[bsel]);
                if (dcol < DR) {
                    const long long row0 = static_cast<long long>(bhq) * N + q0 + c0;   // first row
                    float *dst = dQacc + static_cast<size_t>(row0) * DR + dcol;
                    const int nvalid = min(NC, qend - q0 - c0);   // of these rows inside the sequence
#pragma unroll
                    for (int c = 0; c < NC; ++c)
                        if (c < nvalid && in_bounds(row0 + c, rows_total, status))
                            atomicAdd(dst + static_cast<size_t>(c) * DR, __uint_as_float(a[c]) * scale);
                }
                // hand the step to the turn passer; each lane's arrival releases its own
                // reductions to it
                if constexpr (DET) mbar_arrive(&sent_full[s % NSENT]);
            }
            if (DET && *abort_flag) atomicExch(dq_sem + static_cast<size_t>(BHkv) * G * nq * 4, 1u);
        }
        if constexpr (SPLIT_EPI) {
            // epilogue, dV half: dV rows -> bf16 -> smem over V (its first DR / 64 chunks; at
            // DR = 64 the second one is the dQ staging tile) -> TMA store.  Same barrier rule as
            // the gradient warps' half.
            const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, status));
            if (acc_ok) {
                tc_fence_after();
                stage_acc_rows<32, DR>(tmem + lane_off + T_DV, 1.f, smem + L::V_OFF, dcol, MASK && T == 0);
            }
            fence_proxy_async_smem();
            named_barrier_sync(3, 128);
            if (acc_ok && threadIdx.x == 128 && !*abort_flag) {
                for (int ch = 0; ch < DR / 64; ++ch)
                    tma_store_3d(&tmdV, smem + L::V_OFF + ch * L::KV_CHUNK, ch * 64, jb * BKV, bkv);
                tma_store_commit_and_wait_read();
            }
        }
        // the last bulk reductions have finished reading shared memory (and writing)
        if (DQ_TMA && threadIdx.x == 128) bulk_wait_all();
        tc_fence_before();
        __syncthreads();
    }
}

// K2: D[row] = sum_k dO[row,k] O[row,k] (fp32) and dQacc = 0.  HBM-bound: one 16-byte vector
// per lane per tensor, 8 bf16 each.
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16 *__restrict__ O,
                                                             const __nv_bfloat16 *__restrict__ dO,
                                                             float *__restrict__ Dvec,
                                                             float4 *__restrict__ dQacc,
                                                             long long rows, int d,
                                                             long long acc_vec4) {
    const int lanes_per_row = d / 8;                 // 16 (d = 128) or 8 (d = 64)
    const int rows_per_warp = 32 / lanes_per_row;
    const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const int lane = threadIdx.x & 31, sub = lane % lanes_per_row;
    const long long warp_id = tid >> 5, nwarps = nthreads >> 5;
    // each group of lanes_per_row lanes owns one row; the loop is uniform across the warp
    for (long long wb = warp_id * rows_per_warp; wb < rows; wb += nwarps * rows_per_warp) {
        const long long row = wb + lane / lanes_per_row;
        float acc = 0.f;
        if (row < rows) {
            const uint4 a = *reinterpret_cast<const uint4 *>(O + row * d + sub * 8);
            const uint4 c = *reinterpret_cast<const uint4 *>(dO + row * d + sub * 8);
            const __nv_bfloat162 *ah = reinterpret_cast<const __nv_bfloat162 *>(&a);
            const __nv_bfloat162 *ch = reinterpret_cast<const __nv_bfloat162 *>(&c);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 x = __bfloat1622float2(ah[k]);
                const float2 y = __bfloat1622float2(ch[k]);
                acc = fmaf(x.x, y.x, acc);
                acc = fmaf(x.y, y.y, acc);
            }
        }
        for (int off = lanes_per_row / 2; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off, lanes_per_row);
        if (sub == 0 && row < rows) Dvec[row] = acc;
    }
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long k = tid; k < acc_vec4; k += nthreads) dQacc[k] = z;
}

// K4: dQ = bf16(dQacc), 8 elements per thread per step.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4 *__restrict__ acc,
                                                             uint4 *__restrict__ out,
                                                             long long n8) {
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long k = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; k < n8;
         k += nthreads) {
        const float4 a = acc[2 * k], c = acc[2 * k + 1];
        uint4 v;
        v.x = pack_bf16x2(a.x, a.y);
        v.y = pack_bf16x2(a.z, a.w);
        v.z = pack_bf16x2(c.x, c.y);
        v.w = pack_bf16x2(c.z, c.w);
        out[k] = v;
    }
}

static int grid_for(long long work, int per_block, int num_sms) {
    long long g = (work + per_block - 1) / per_block;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}


}  // namespace bwd

cudaError_t launch_bwd_preprocess_bf16(const Problem &p, const void *O, const void *dO, float *D,
                                       float *dQacc, cudaStream_t stream, size_t zero_tail_bytes) {
    const long long rows = static_cast<long long>(p.B) * p.Hq * p.N;
    const long long acc4 = rows * p.d / 4 + static_cast<long long>(zero_tail_bytes / 16);
    const int sms = num_sms();
    const int grid = bwd::grid_for(rows * (p.d / 8), 256, sms);
    bwd::bwd_preprocess_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), D,
        reinterpret_cast<float4 *>(dQacc), rows, p.d, acc4);
    return cudaGetLastError();
}

namespace bwd {
template <bool MASK, bool DROP, bool DET = false>
cudaError_t launch_main(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                        const CUtensorMap &tmV, const CUtensorMap &tmdO, const CUtensorMap &tmdK,
                        const CUtensorMap &tmdV, const CUtensorMap &tmdQ, const float *LSE,
                        const float *D, float *dQacc, const MaskArgs &mk, const DropoutArgs &dr,
                        unsigned *dq_sem, unsigned *status, cudaStream_t stream) {
    if (p.d != 128 && p.d != 64) return cudaErrorInvalidValue;
    const int BHkv = p.B * p.Hkv;
    const long long nkb = (p.N + BKV - 1) / BKV;
    // KV heads go in chunks of HC: the largest divisor of B * Hkv whose chunk is at most four
    // waves of CTAs, so the Q / dO / dQ accumulator rows a chunk's heads share stay in L2 while its
    // key blocks run (B2 H32 N4096: 16 heads, 2% faster and a fraction of the DRAM traffic), and
    // the last chunk is as full as the others (a lone last head left a long tail: +27% at
    // B1 Hkv8 N8192).
    // Under a tile mask the key blocks' step counts follow the mask and can differ by far more
    // than under causal masking (a sink block seen by every query next to window blocks seen by a
    // few), so all KV heads form one chunk and every head's longest blocks start first (chunks of
    // 4 heads left the last chunk's sink blocks as a tail: +55% at B1 H16 N16384 window + sink).
    int HC = 1;
    for (int h = 1; h <= BHkv; ++h)
        if (BHkv % h == 0 && static_cast<long long>(h) * nkb <= 4LL * num_sms()) HC = h;
    if (MASK && mk.block_mask) HC = BHkv;
    const long long grid = nkb * BHkv;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (MASK && static_cast<long long>(p.Hq / p.Hkv) * ((p.N + BQ - 1) / BQ) > MAX_MASK_STEPS)
        return cudaErrorInvalidConfiguration;
    const int smem = MASK ? Layout<128>::BYTES_MASK : DROP ? Layout<128>::BYTES_DROP
                     : DET ? Layout<128>::BYTES_DET : Layout<128>::BYTES;
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                          CUtensorMap, const float *, const float *, float *, int, int, int, int, int,
                          float, float, MaskArgs, DropoutArgs, unsigned *, unsigned *);
    Kern kern;
    if (p.d == 128)
        kern = p.causal ? bwd_main_kernel<128, 128, true, MASK, DROP, DET>
                        : bwd_main_kernel<128, 128, false, MASK, DROP, DET>;
    else
        kern = p.causal ? bwd_main_kernel<128, 64, true, MASK, DROP, DET>
                        : bwd_main_kernel<128, 64, false, MASK, DROP, DET>;
    const int threads = p.d == 128 ? Roles<128, DET>::THREADS : Roles<64, DET>::THREADS;
    const int regs_needed = p.d == 128 ? Roles<128, DET>::REGS_NEEDED : Roles<64, DET>::REGS_NEEDED;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // the in-kernel register split needs at least this many registers at launch
    cudaFuncAttributes attr{};
    if ((e = cudaFuncGetAttributes(&attr, kern)) != cudaSuccess) return e;
    if (attr.numRegs * threads < regs_needed) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(grid), threads, smem, stream>>>(
        tmQ, tmK, tmV, tmdO, tmdK, tmdV, tmdQ, LSE, D, dQacc, p.Hq, p.Hkv, p.N, BHkv, HC, p.scale,
        scale_log2, mk, dr, dq_sem, status);
    return cudaGetLastError();
}
}  // namespace bwd

cudaError_t launch_bwd_main_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                 const CUtensorMap &tmV, const CUtensorMap &tmdO,
                                 const CUtensorMap &tmdK, const CUtensorMap &tmdV,
                                 const CUtensorMap &tmdQ, const float *LSE, const float *D,
                                 float *dQacc, unsigned *status, cudaStream_t stream) {
    return bwd::launch_main<false, false>(p, tmQ, tmK, tmV, tmdO, tmdK, tmdV, tmdQ, LSE, D, dQacc,
                                          MaskArgs{}, DropoutArgs{}, nullptr, status, stream);
}

cudaError_t launch_bwd_main_deterministic_bf16(const Problem &p, const CUtensorMap &tmQ,
                                               const CUtensorMap &tmK, const CUtensorMap &tmV,
                                               const CUtensorMap &tmdO, const CUtensorMap &tmdK,
                                               const CUtensorMap &tmdV, const CUtensorMap &tmdQ,
                                               const float *LSE, const float *D, float *dQacc,
                                               unsigned *dq_sem, unsigned *status,
                                               cudaStream_t stream) {
    return bwd::launch_main<false, false, true>(p, tmQ, tmK, tmV, tmdO, tmdK, tmdV, tmdQ, LSE, D,
                                                dQacc, MaskArgs{}, DropoutArgs{}, dq_sem, status,
                                                stream);
}

cudaError_t launch_bwd_main_masked_bf16(const Problem &p, const CUtensorMap &tmQ,
                                        const CUtensorMap &tmK, const CUtensorMap &tmV,
                                        const CUtensorMap &tmdO, const CUtensorMap &tmdK,
                                        const CUtensorMap &tmdV, const CUtensorMap &tmdQ,
                                        const float *LSE, const float *D, float *dQacc,
                                        const MaskArgs &mk, unsigned *status, cudaStream_t stream) {
    return bwd::launch_main<true, false>(p, tmQ, tmK, tmV, tmdO, tmdK, tmdV, tmdQ, LSE, D, dQacc, mk,
                                         DropoutArgs{}, nullptr, status, stream);
}

cudaError_t launch_bwd_main_dropout_bf16(const Problem &p, const CUtensorMap &tmQ,
                                         const CUtensorMap &tmK, const CUtensorMap &tmV,
                                         const CUtensorMap &tmdO, const CUtensorMap &tmdK,
                                         const CUtensorMap &tmdV, const CUtensorMap &tmdQ,
                                         const float *LSE, const float *D, float *dQacc,
                                         const DropoutArgs &dr, unsigned *status, cudaStream_t stream) {
    return bwd::launch_main<false, true>(p, tmQ, tmK, tmV, tmdO, tmdK, tmdV, tmdQ, LSE, D, dQacc,
                                         MaskArgs{}, dr, nullptr, status, stream);
}

cudaError_t launch_bwd_dq_convert_bf16(const Problem &p, const float *dQacc, void *dQ,
                                       cudaStream_t stream) {
    const long long n8 = static_cast<long long>(p.B) * p.Hq * p.N * p.d / 8;
    const int grid = bwd::grid_for(n8, 256, num_sms());
    bwd::bwd_dq_convert_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const float4 *>(dQacc),
                                                         static_cast<uint4 *>(dQ), n8);
    return cudaGetLastError();
}

}  // namespace fa
