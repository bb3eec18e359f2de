// fa_fwd_sm103a.cu -- K1: exact attention forward, bf16 in / fp32 accumulate, sm_103a.
//
// Method (FlashAttention DAC'24 reading note, paper.adslab.icu, Methods): a query tile stays in
// on-chip memory while key/value blocks stream past it; per block the running row max m and
// running sum l are rescaled, l' = e^{m-m'} l + e^{m~-m'} l~, and the output accumulator is
// rescaled the same way.  Normalisation is deferred to the end (FlashAttention note,
// paweldubiel.com: keep u = sum e^{s-m} v and return u / l), which equals the per-step form of
// the reading note's O update in exact arithmetic.  The mask acts on each block's scores
// (reading note, "other operators"), here only on blocks that cross the diagonal or the end of
// the sequence.  LSE = m + ln l is stored for the backward pass (mzeromiko blog, end of the
// "blocked form with online-softmax rescaling" section: logsumexp placement).
//
// GB300 mapping: a persistent grid of one CTA per SM walks work items (two 128-row query tiles
// of one (batch, head)), longest first, carrying every pipeline phase across items; 384 threads:
//   warps 0-3 : softmax for query tile 0  (thread = query row = TMEM lane)
//   warps 4-7 : softmax for query tile 1
//   warp 8    : TMA producer (Q tiles once, then K_j / V_j through a 4-stage ring)
//   warp 9    : TMEM allocator and single-thread tcgen05.mma issuer
//   warps 10-11 complete the third warpgroup so its registers can be handed to the softmax.
// TMEM (512 columns): S/P of tile t at columns 128 t, O of tile t at 256 + 128 t.
// S = Q K_j^T runs as SS MMAs (both operands K-major in 128B-swizzled smem); P is written back
// over S as packed bf16 and O += P V_j runs as a TS MMA (P from TMEM, V MN-major in smem).
// The MMA order S0(j+1) after PV0(j) lets softmax of one tile overlap the other tile's MMAs.
// Rescaling of O is lazy: the stale max is kept until the block max exceeds it by 4 (log2
// units), so p <= 16; the shift cancels in O = u / l.  A rescale is a round trip of O through
// TMEM for the whole warp when any of its 32 rows needs one, so a tight threshold rescales most
// blocks of a warp (threshold 1: 55% of them at B2 H32 N4096); at 4 the forward is 4% faster
// there, and a kernel-faithful CPU model of the rounding over every element of the N = 32768
// workload finds the same handful of elements above 1e-2 as at 1 (15 against 13 of 537 M, all
// within the worst case of bf16 P and a bf16 output).
// O is divided by the sum of the fp32 weights plus the rounding residual of each block's largest
// bf16 weight when that weight dominates the row so far (at least half of its sum: the weights P V
// applies then sum to one); LSE uses the sum of the fp32 weights alone.  Rows that see no key
// past the first block (the first query tile of a causal head) apply that block's weights as two
// bf16 parts, hi + lo, through a second P V product (two_part_p).
#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "fa_ptx.cuh"

namespace fa {
namespace fwd {

constexpr int BM = 128;           // query rows per tile (= TMEM lanes)
constexpr int BN = 128;           // keys per block
constexpr int NS = 4;             // K/V ring stages
constexpr int NUM_THREADS = 384;   // three warpgroups
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
// Register split: softmax warpgroups 0 and 1 grow, warpgroup 2 (TMA, MMA, two idle warps) shrinks.
constexpr uint32_t REGS_SOFTMAX = 208, REGS_OTHER = 88;
constexpr int REGS_NEEDED = 2 * 128 * REGS_SOFTMAX + 128 * REGS_OTHER;
constexpr float RESCALE_THRESHOLD = 4.0f;
constexpr float LN2 = 0.693147180559945309f;

template <int D>
struct Layout {
    static constexpr int TILE_BYTES = 128 * D * 2;   // one Q tile or one K/V block, bf16
    static constexpr int CHUNK_BYTES = 128 * 128;    // 128 rows x 64 bf16 (one swizzle column)
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = 2 * TILE_BYTES;
    static constexpr int BAR_OFF = KV_OFF + NS * TILE_BYTES;
    // q_full, q_empty, kv_full[NS], kv_empty[NS], s_full[2], p_full[2], o_full[2], o_empty[2],
    // mma_done
    static constexpr int NBARS = 2 + 2 * NS + 2 + 2 + 2 + 2 + 1;
    static constexpr int TMEM_OFF = BAR_OFF + NBARS * 8;
    static constexpr int ABORT_OFF = TMEM_OFF + 8;
    static constexpr int BYTES = ABORT_OFF + 8 + 1024;   // + slack for 1024-byte alignment
};

// O row *= alpha in TMEM; the caller waits for the stores.  At head dim 128 one load and one
// store of the whole row (the caller has no other large register arrays live); at 64, in
// 32-column pieces (measured: fewer spills there).
template <int D>
__device__ __forceinline__ void rescale_o_row(uint32_t tO, float alpha) {
    if constexpr (D == 128) {
        uint32_t o[128];
        tmem_ld_x128(tO, o);
#pragma unroll
        for (int i = 0; i < 128; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st_x128(tO, o);
    } else {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld_x32(tO + c0, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_x32(tO + c0, o);
        }
    }
}

// One work item = two 128-row query tiles (a "pair") of one (batch, head) against one range of key
// blocks: all of them, or split sp of S contiguous ranges (split-KV partial results).
// Under a general mask (MASK) the valid lengths bound the range and a tile mask row decides which
// of its blocks a tile takes; the pair still shares one K/V stream (the union of both tiles').
struct Item {
    int bh, bkv, split, jb0, q0[2], nblk[2], nmax;   // nblk: key blocks of each tile in the range
    int lq, lk;                                     // valid query rows / keys of the batch (MASK)
    const uint8_t *row[2];                          // tile mask row of each tile, or null (MASK)
};

template <bool CAUSAL, bool SPLIT, bool MASK>
__device__ __forceinline__ Item decode_item(int k, int Hq, int Hkv, int N, int BH, int S,
                                            const MaskArgs &mk) {
    // Items are numbered longest-first: under causal masking the late pairs (most key blocks)
    // of every head come first.  With S ranges the ranges of one pair are adjacent, so the
    // full-length ranges of the late pairs lead and the short last ranges of the early pairs
    // come at the end.
    const int n_pairs = (N + 2 * BM - 1) / (2 * BM);
    Item it;
    it.bh = k % BH;
    const int rest = k / BH;
    it.split = SPLIT ? rest % S : 0;
    int pair = SPLIT ? rest / S : rest;
    if (CAUSAL) pair = n_pairs - 1 - pair;
    const int hq = it.bh % Hq, b = it.bh / Hq;
    it.bkv = b * Hkv + hq / (Hq / Hkv);
    const int nkb = (N + BN - 1) / BN;
    it.lq = N;
    it.lk = N;
    if (MASK) {
        if (mk.q_len) it.lq = min(max(__ldg(mk.q_len + b), 0), N);
        if (mk.k_len) it.lk = min(max(__ldg(mk.k_len + b), 0), N);
    }
    const int nkb_lim = MASK ? (it.lk + BN - 1) / BN : nkb;
    const int bps = SPLIT ? (nkb + S - 1) / S : nkb;
    it.jb0 = it.split * bps;
    const int jb1 = SPLIT ? min(nkb, it.jb0 + bps) : nkb_lim;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        it.q0[t] = pair * 2 * BM + t * BM;
        int full;
        if (it.q0[t] >= (MASK ? it.lq : N))
            full = 0;
        else if (CAUSAL)
            full = min(nkb_lim, (min(it.q0[t] + BM, N) - 1) / BN + 1);
        else
            full = nkb_lim;
        it.nblk[t] = max(0, min(full, jb1) - it.jb0);
        it.row[t] = nullptr;
        if (MASK && mk.block_mask && it.nblk[t] > 0) {
            const int h = mk.mask_heads == 1 ? 0 : (mk.mask_heads == BH ? it.bh : hq);
            it.row[t] = mk.block_mask + (static_cast<size_t>(h) * nkb + it.q0[t] / BM) * nkb;
        }
    }
    it.nmax = max(it.nblk[0], it.nblk[1]);
    return it;
}

// Rows that see no key beyond the first block (query tile 0 under causal masking, or at most BN
// valid keys) hold a few large weights, and rounding those to bf16 before P V can cost more
// accuracy than the output's own bf16 rounding leaves room for.  On that block the weights are
// applied as two bf16 parts, hi = bf16(p) and lo = bf16(p - hi), through a second P V product;
// jb is the absolute key block; dropout keeps its own rounding rule.
template <bool CAUSAL, bool MASK, bool DROP>
__device__ __forceinline__ bool two_part_p(const Item &it, int t, int jb, int N) {
    if (DROP || jb != 0) return false;
    return (CAUSAL && it.q0[t] == 0) || (MASK ? it.lk : N) <= BN;
}

// Does tile t take key block jj (relative to the item's range)?  Without MASK every block of its
// prefix; with MASK also only those its tile mask row keeps.
template <bool MASK>
__device__ __forceinline__ bool takes(const Item &it, int t, int jj) {
    if (!MASK) return jj < it.nblk[t];
    return jj < it.nblk[t] && (it.row[t] == nullptr || __ldg(it.row[t] + jj) != 0);
}

// First block >= jj that tile t takes, or it.nblk[t].
template <bool MASK>
__device__ __forceinline__ int next_of_tile(const Item &it, int t, int jj) {
    if (!MASK) return jj;
    while (jj < it.nblk[t] && !takes<MASK>(it, t, jj)) ++jj;
    return min(jj, it.nblk[t]);
}

// First block >= jj that either tile takes (the pair's K/V stream), or it.nmax.
template <bool MASK>
__device__ __forceinline__ int next_of_pair(const Item &it, int jj) {
    if (!MASK) return jj;
    while (jj < it.nmax && !takes<MASK>(it, 0, jj) && !takes<MASK>(it, 1, jj)) ++jj;
    return min(jj, it.nmax);
}

// Last block tile t takes, or -1.
template <bool MASK>
__device__ __forceinline__ int last_of_tile(const Item &it, int t) {
    int jj = it.nblk[t] - 1;
    if (MASK)
        while (jj >= 0 && !takes<MASK>(it, t, jj)) --jj;
    return jj;
}

// The r-th item of this CTA: rounds of gridDim.x items, assigned in snake order (reversed on odd
// rounds) so every CTA gets a similar share of long and short items.
__device__ __forceinline__ int item_index(int r) {
    const int G = gridDim.x;
    return r * G + ((r & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x));
}

// SPLIT = false: O (bf16) and LSE of the whole key range.  SPLIT = true: for each of S key
// ranges, the partial result over that range alone as fp32 O_parts [S, B*Hq, N, d] and
// LSE_parts [S, B*Hq, N] (LSE = -inf where a row has no allowed key in the range).
// MASK = true: the general mask mk on top of the causal rule; rows with no allowed key (and rows
// past the batch's valid length) get O = 0 and LSE = -inf.
// DROP = true: dropout on P (fa_philox.cuh has the keep rule): the weights P V applies are the
// kept ones, l sums all of them, and O is scaled by 1 / (1 - p).
template <int D, bool CAUSAL, bool SPLIT, bool MASK, bool DROP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, void *__restrict__ Out,
               float *__restrict__ LSE, int Hq, int Hkv, int N, int BH, int n_items, int S,
               float scale_log2, const MaskArgs mk, const DropoutArgs dr, unsigned *status) {
    static_assert(int(SPLIT) + int(MASK) + int(DROP) <= 1, "one variant at a time");
    constexpr bool SKIP_EMPTY = SPLIT || MASK;      // items may have no key block at all
    // rows of O (or of the partials) and of LSE: the extent debug builds check writes against
    const long long rows_total = static_cast<long long>(SPLIT ? S : 1) * BH * N;
    (void)rows_total;
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *q_full = bars;
    uint64_t *q_empty = bars + 1;
    uint64_t *kv_full = bars + 2;
    uint64_t *kv_empty = kv_full + NS;
    uint64_t *s_full = kv_empty + NS;   // [2]
    uint64_t *p_full = s_full + 2;      // [2]
    uint64_t *o_full = p_full + 2;      // [2]
    uint64_t *o_empty = o_full + 2;     // [2]
    uint64_t *mma_done = o_empty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::TMEM_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::ABORT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // number of items this CTA processes
    int n_mine = 0;
    while (item_index(n_mine) < n_items) ++n_mine;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], BM);
            mbar_init(&o_full[t], 1);
            mbar_init(&o_empty[t], BM);
        }
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

    // Each role branch starts with its register budget and ends with its own copy of the final
    // barrier, so no code is shared between budgets.
    if (warp >= 8) {
        regs_dec<REGS_OTHER>();
      if (warp == WARP_TMA) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int base = 0, issued = 0;         // K/V ring index of the current item's K_0
            int q_issued = 0;
            bool ok = true;
            for (int r = 0; r < n_mine && ok; ++r) {
                const Item it = decode_item<CAUSAL, SPLIT, MASK>(item_index(r), Hq, Hkv, N, BH, S, mk);
                const int jfirst = next_of_pair<MASK>(it, 0);
                if (SKIP_EMPTY && jfirst >= it.nmax) continue;   // no key block: no work
                // Q buffer: free once every S product of the previous item has completed
                if (q_issued > 0 && !mbar_wait(q_empty, (q_issued - 1) & 1, abort_flag, status)) { ok = false; break; }
                const int ntiles = it.nblk[1] > 0 ? 2 : 1;
                mbar_arrive_expect_tx(q_full, ntiles * L::TILE_BYTES);
                ++q_issued;
                for (int t = 0; t < ntiles; ++t)
                    for (int ch = 0; ch < D / 64; ++ch)
                        tma_load_3d(smem + L::Q_OFF + t * L::TILE_BYTES + ch * L::CHUNK_BYTES, &tmQ,
                                    ch * 64, it.q0[t], it.bh, q_full);
                int e = 0;                            // ring slots of this item so far
                for (int jj = jfirst; jj < it.nmax && ok; jj = next_of_pair<MASK>(it, jj + 1)) {
                    for (int kv = 0; kv < 2; ++kv) {
                        const int idx = base + e, j = it.jb0 + jj, st = idx % NS, rnd = idx / NS;
                        ++e;
                        if (!mbar_wait(&kv_empty[st], (rnd & 1) ^ 1, abort_flag, status)) { ok = false; break; }
#ifdef FA_FAULT_INJECT
                        // Test builds only: CTA 0 never delivers its first K block, so the MMA
                        // warp's bounded wait runs out, the CTA unwinds and FA_ERR_DEVICE_TIMEOUT
                        // is recorded.
                        if (blockIdx.x == 0 && idx == 0) continue;
#endif
                        mbar_arrive_expect_tx(&kv_full[st], L::TILE_BYTES);
                        uint8_t *dst = smem + L::KV_OFF + st * L::TILE_BYTES;
                        const CUtensorMap *tm = kv ? &tmV : &tmK;
                        for (int ch = 0; ch < D / 64; ++ch)
                            tma_load_3d(dst + ch * L::CHUNK_BYTES, tm, ch * 64, j * BN, it.bkv, &kv_full[st]);
                        issued = idx + 1;             // ring index after the last load issued
                    }
                }
                base += e;
            }
            if (!ok || *abort_flag) {
                // Unwinding: let copies still in flight land before the CTA's smem goes away.
                for (int idx = max(0, issued - NS); idx < issued; ++idx)
                    mbar_drain(&kv_full[idx % NS], (idx / NS) & 1);
                if (q_issued > 0) mbar_drain(q_full, (q_issued - 1) & 1);
            }
        }
      } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, false, true);
            // Descriptors are built once; each k-step only moves the start address.
            const uint64_t dq0 = sdesc_sw128(smem_u32(smem + L::Q_OFF), 16, 1024);
            const uint64_t dkv0 = sdesc_sw128(smem_u32(smem + L::KV_OFF), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(smem + L::KV_OFF), L::CHUNK_BYTES, 1024);
            auto issue_s = [&](int t, int st) {
                const uint64_t da = sdesc_add(dq0, t * L::TILE_BYTES);
                const uint64_t db = sdesc_add(dkv0, st * L::TILE_BYTES);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::CHUNK_BYTES + (kk & 3) * 32;
                    mma_ss(tmem + t * 128, sdesc_add(da, off), sdesc_add(db, off), IDESC_S, kk > 0);
                }
                mma_commit(&s_full[t]);
            };
            auto issue_pv = [&](int t, int st, bool accumulate) {
                const uint64_t db = sdesc_add(dv0, st * L::TILE_BYTES);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, sdesc_add(db, kk * 2048),
                           IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
            };
            // The second product of a two-part block (two_part_p): the lo parts, stored 64
            // columns after the hi parts, times the same V, added to O.
            auto issue_pv_lo = [&](int t, int st) {
#pragma unroll 1
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(tmem + 256 + t * 128, tmem + t * 128 + 64 + kk * 8,
                           sdesc_add(dv0, st * L::TILE_BYTES + kk * 2048), IDESC_PV, 1u);
            };
            int base = 0;                       // K/V ring index of the current item's K_0
            int pb[2] = {0, 0};                 // blocks consumed per tile (p_full phases)
            int of[2] = {0, 0};                 // items finished per tile (o_full / o_empty phases)
            bool ok = true;
            int qn = 0;                         // items with work so far (q_full phases)
            if constexpr (MASK) {
            // Same issue order as below, over the blocks either tile takes: S of the next block of
            // tile 0 goes between P V of tiles 0 and 1; each tile's first P V overwrites its O
            // and its last one signals o_full; the item's last S products free the Q buffer.
            for (int r = 0; r < n_mine && ok; ++r) {
                const Item it = decode_item<CAUSAL, SPLIT, MASK>(item_index(r), Hq, Hkv, N, BH, S, mk);
                int u = next_of_pair<MASK>(it, 0);
                if (u >= it.nmax) continue;
                // the tiles' two-part P blocks (only relative block 0 can be one)
                const bool two0 = two_part_p<CAUSAL, MASK, DROP>(it, 0, it.jb0, N);
                const bool two1 = two_part_p<CAUSAL, MASK, DROP>(it, 1, it.jb0, N);
                const int last0 = last_of_tile<MASK>(it, 0), last1 = last_of_tile<MASK>(it, 1);
                const int ulast = max(last0, last1);
                ok = mbar_wait(q_full, qn & 1, abort_flag, status) &&
                     mbar_wait(&kv_full[base % NS], (base / NS) & 1, abort_flag, status);
                if (!ok) break;
                tc_fence_after();
                for (int t = 0; t < 2; ++t)
                    if (takes<MASK>(it, t, u)) issue_s(t, base % NS);
                mma_commit(&kv_empty[base % NS]);
                if (u == ulast) mma_commit(q_empty);
                bool started[2] = {false, false};
                int idx = base;                 // ring index of K_u
                while (true) {
                    const int vidx = idx + 1, kidx = idx + 2;
                    const int vst = vidx % NS, kst = kidx % NS;
                    const int un = (u == ulast) ? it.nmax : next_of_pair<MASK>(it, u + 1);
                    const bool next = un < it.nmax;
                    if (!mbar_wait(&kv_full[vst], (vidx / NS) & 1, abort_flag, status)) { ok = false; break; }
                    if (takes<MASK>(it, 0, u)) {
                        if (!started[0] && of[0] > 0 &&
                            !mbar_wait(&o_empty[0], (of[0] - 1) & 1, abort_flag, status)) { ok = false; break; }
                        if (!mbar_wait(&p_full[0], pb[0] & 1, abort_flag, status)) { ok = false; break; }
                        ++pb[0];
                        tc_fence_after();
                        issue_pv(0, vst, started[0]);
                        if (two0 && u == 0) issue_pv_lo(0, vst);
                        started[0] = true;
                        if (u == last0) mma_commit(&o_full[0]);
                    }
                    if (next) {
                        if (!mbar_wait(&kv_full[kst], (kidx / NS) & 1, abort_flag, status)) { ok = false; break; }
                        tc_fence_after();
                        if (takes<MASK>(it, 0, un)) issue_s(0, kst);
                    }
                    if (takes<MASK>(it, 1, u)) {
                        if (!started[1] && of[1] > 0 &&
                            !mbar_wait(&o_empty[1], (of[1] - 1) & 1, abort_flag, status)) { ok = false; break; }
                        if (!mbar_wait(&p_full[1], pb[1] & 1, abort_flag, status)) { ok = false; break; }
                        ++pb[1];
                        tc_fence_after();
                        issue_pv(1, vst, started[1]);
                        if (two1 && u == 0) issue_pv_lo(1, vst);
                        started[1] = true;
                        if (u == last1) mma_commit(&o_full[1]);
                    }
                    mma_commit(&kv_empty[vst]);
                    if (!next) break;
                    if (takes<MASK>(it, 1, un)) issue_s(1, kst);
                    mma_commit(&kv_empty[kst]);
                    if (un == ulast) mma_commit(q_empty);
                    u = un;
                    idx += 2;
                }
                if (!ok) break;
                for (int t = 0; t < 2; ++t)
                    if (started[t]) ++of[t];
                base = idx + 2;
                ++qn;
            }
            } else {
            for (int r = 0; r < n_mine && ok; ++r) {
                const Item it = decode_item<CAUSAL, SPLIT, MASK>(item_index(r), Hq, Hkv, N, BH, S, mk);
                if (SKIP_EMPTY && it.nmax == 0) continue;
                ok = mbar_wait(q_full, qn & 1, abort_flag, status) &&
                     mbar_wait(&kv_full[base % NS], (base / NS) & 1, abort_flag, status);
                if (!ok) break;
                tc_fence_after();
                for (int t = 0; t < 2; ++t)
                    if (it.nblk[t] > 0) issue_s(t, base % NS);
                mma_commit(&kv_empty[base % NS]);
                if (it.nmax == 1) mma_commit(q_empty);     // every S product of the item issued
                const int nb0 = it.nblk[0], nb1 = it.nblk[1], nmax = it.nmax;
                // An item with a two-part block (only relative block 0 of a tile can be one: the
                // first query tile of a causal head, or a sequence of at most BN keys) takes its
                // own copy of the issue sequence with the lo products, so the sequence every
                // other item runs is unchanged.
                const bool two0 = two_part_p<CAUSAL, MASK, DROP>(it, 0, it.jb0, N);
                const bool two1 = two_part_p<CAUSAL, MASK, DROP>(it, 1, it.jb0, N);
                if (two0 || two1) {
                    for (int j = 0; j < nmax; ++j) {
                        const int vidx = base + 2 * j + 1, kidx = base + 2 * j + 2;
                        const int vst = vidx % NS, kst = kidx % NS;
                        const bool next = j + 1 < nmax;
                        if (!mbar_wait(&kv_full[vst], (vidx / NS) & 1, abort_flag, status)) { ok = false; break; }
                        if (j < nb0) {
                            if (j == 0 && of[0] > 0 &&
                                !mbar_wait(&o_empty[0], (of[0] - 1) & 1, abort_flag, status)) { ok = false; break; }
                            if (!mbar_wait(&p_full[0], pb[0] & 1, abort_flag, status)) { ok = false; break; }
                            ++pb[0];
                            tc_fence_after();
                            issue_pv(0, vst, j > 0);
                            if (two0 && j == 0) issue_pv_lo(0, vst);
                            if (j == nb0 - 1) mma_commit(&o_full[0]);
                        }
                        if (next) {
                            if (!mbar_wait(&kv_full[kst], (kidx / NS) & 1, abort_flag, status)) { ok = false; break; }
                            tc_fence_after();
                            if (j + 1 < nb0) issue_s(0, kst);
                        }
                        if (j < nb1) {
                            if (j == 0 && of[1] > 0 &&
                                !mbar_wait(&o_empty[1], (of[1] - 1) & 1, abort_flag, status)) { ok = false; break; }
                            if (!mbar_wait(&p_full[1], pb[1] & 1, abort_flag, status)) { ok = false; break; }
                            ++pb[1];
                            tc_fence_after();
                            issue_pv(1, vst, j > 0);
                            if (two1 && j == 0) issue_pv_lo(1, vst);
                            if (j == nb1 - 1) mma_commit(&o_full[1]);
                        }
                        mma_commit(&kv_empty[vst]);
                        if (next) {
                            if (j + 1 < nb1) issue_s(1, kst);
                            mma_commit(&kv_empty[kst]);
                            if (j + 1 == nmax - 1) mma_commit(q_empty);
                        }
                    }
                    if (!ok) break;
                    for (int t = 0; t < 2; ++t)
                        if (it.nblk[t] > 0) ++of[t];
                    base += 2 * it.nmax;
                    ++qn;
                    continue;
                }
                for (int j = 0; j < nmax; ++j) {
                    const int vidx = base + 2 * j + 1, kidx = base + 2 * j + 2;
                    const int vst = vidx % NS, kst = kidx % NS;
                    const bool next = j + 1 < nmax;
                    if (!mbar_wait(&kv_full[vst], (vidx / NS) & 1, abort_flag, status)) { ok = false; break; }
                    if (j < nb0) {
                        // the item's first P V overwrites O: its previous contents must be read out
                        if (j == 0 && of[0] > 0 &&
                            !mbar_wait(&o_empty[0], (of[0] - 1) & 1, abort_flag, status)) { ok = false; break; }
                        if (!mbar_wait(&p_full[0], pb[0] & 1, abort_flag, status)) { ok = false; break; }
                        ++pb[0];
                        tc_fence_after();
                        issue_pv(0, vst, j > 0);
                        if (j == nb0 - 1) mma_commit(&o_full[0]);
                    }
                    if (next) {
                        // S0 of the next block goes between PV0 and PV1 of this one
                        if (!mbar_wait(&kv_full[kst], (kidx / NS) & 1, abort_flag, status)) { ok = false; break; }
                        tc_fence_after();
                        if (j + 1 < nb0) issue_s(0, kst);
                    }
                    if (j < nb1) {
                        if (j == 0 && of[1] > 0 &&
                            !mbar_wait(&o_empty[1], (of[1] - 1) & 1, abort_flag, status)) { ok = false; break; }
                        if (!mbar_wait(&p_full[1], pb[1] & 1, abort_flag, status)) { ok = false; break; }
                        ++pb[1];
                        tc_fence_after();
                        issue_pv(1, vst, j > 0);
                        if (j == nb1 - 1) mma_commit(&o_full[1]);
                    }
                    mma_commit(&kv_empty[vst]);
                    if (next) {
                        if (j + 1 < nb1) issue_s(1, kst);
                        mma_commit(&kv_empty[kst]);
                        if (j + 1 == nmax - 1) mma_commit(q_empty);   // last S products issued
                    }
                }
                if (!ok) break;
                for (int t = 0; t < 2; ++t)
                    if (it.nblk[t] > 0) ++of[t];
                base += 2 * it.nmax;
                ++qn;
            }
            }
            // Nothing issued may still be running when TMEM is released.
            mma_commit(mma_done);
            mbar_drain(mma_done, 0);
        }
      }
        tc_fence_before();
        __syncthreads();
        if (warp == WARP_MMA) {
            __syncwarp();
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    } else {
        regs_inc<REGS_SOFTMAX>();
        // ------------------------------------------------------------------ softmax warps
        const int t = warp >> 2, wq = warp & 3;
        const int row = wq * 32 + lane;             // row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * 128;
        int sb = 0;                                 // blocks consumed by this tile (s_full phases)
        int of = 0;                                 // items finished by this tile (o_full phases)
        bool ok = true;
        for (int r = 0; r < n_mine && ok; ++r) {
            const Item it = decode_item<CAUSAL, SPLIT, MASK>(item_index(r), Hq, Hkv, N, BH, S, mk);
            const int nb = it.nblk[t];
            const int q0 = it.q0[t];
            const int rq = q0 + row;                // query index
            const int jfirst = next_of_tile<MASK>(it, t, 0);
            if (nb == 0 || (MASK && jfirst >= nb)) {
                // Split-KV: these rows have no allowed key in the range; the merge skips them.
                const long long drow = (static_cast<long long>(SPLIT ? it.split : 0) * BH + it.bh) * N + rq;
                if (SPLIT && rq < N && in_bounds(drow, rows_total, status))
                    LSE[(static_cast<size_t>(it.split) * BH + it.bh) * N + rq] = -INFINITY;
                // General mask: no allowed key at all, so O = 0 and LSE = -inf.
                if (MASK && rq < N && in_bounds(drow, rows_total, status)) {
                    uint4 *orow = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(Out) +
                                                            (static_cast<size_t>(it.bh) * N + rq) * D);
#pragma unroll
                    for (int u = 0; u < D / 8; ++u) orow[u] = make_uint4(0u, 0u, 0u, 0u);
                    LSE[static_cast<size_t>(it.bh) * N + rq] = -INFINITY;
                }
                continue;
            }
            // l: sum of the fp32 weights (gives LSE).  lc: rounding residual bf16(p) - p of each
            // block's largest weight, the dominant part of (sum of the bf16 weights that P V
            // applies) - l; O is divided by l + lc so the applied weights sum to one when one
            // weight dominates.
            float m = -INFINITY, l = 0.f, lc = 0.f;
            for (int j = jfirst, jj = 0; j < nb; j = next_of_tile<MASK>(it, t, j + 1), ++jj) {
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], sb & 1, abort_flag, status));
                if (!ok) break;
                ++sb;
                tc_fence_after();
                uint32_t sraw[128];
                tmem_ld_x128(tS, sraw);
                float s[128];
#pragma unroll
                for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sraw[c]);
                const int kbase = (it.jb0 + j) * BN;
                const int kend = MASK ? it.lk : N;    // keys past the valid length are masked
                const bool need_mask = (CAUSAL && kbase + BN - 1 > q0) || (kbase + BN > kend);
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const int key = kbase + c;
                        if ((CAUSAL && key > rq) || key >= kend) s[c] = -INFINITY;
                    }
                }
                // row max as a shallow tree of 3-input maxes (8 independent chains)
                float m8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = fmax3(s[k], s[k + 8], s[k + 16]);
#pragma unroll
                for (int i = 24; i < 120; i += 16)
#pragma unroll
                    for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], s[i + k], s[i + 8 + k]);
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], s[120 + k]);
                const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                                       fmaxf(m8[6], m8[7]));
                const float m_blk = mx * scale_log2;
                const bool need = m_blk > m + RESCALE_THRESHOLD;
                // At head dim 128, O is rescaled after this block's P is stored (below): it stays
                // untouched until p_full releases this block's P V, and by then the S and P
                // registers are free for one full-row TMEM load and store.  (At 64 that measured
                // more spills; O is rescaled here.)
                bool rescale_o = false;
                float alpha_o = 1.f;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? ex2_approx(m - m_blk) : 1.f;
                    if (need) {
                        l *= alpha;
                        lc *= alpha;
                        m = m_blk;
                    }
                    if constexpr (D == 128) {
                        rescale_o = (MASK ? jj : j) > 0;
                        alpha_o = alpha;
                    } else {
                        if ((MASK ? jj : j) > 0) {
                            rescale_o_row<D>(tO, alpha);
                            tmem_wait_st();
                        }
                    }
                }
                const float m_sub = (m == -INFINITY) ? 0.f : m;
                // P (bf16 pairs) goes over the first 64 columns of S in each branch below
                if constexpr (DROP) {
                    uint32_t p[64];
                    // p = 2^(s c - m) for four keys at a time, with the keep words of those four
                    // keys from one Philox call; l sums every weight, lc the rounding residuals
                    // of the kept ones (the weights P V applies)
                    const uint32_t m0 = static_cast<uint32_t>(kbase) >> 2;
                    float lsum = 0.f, lres = 0.f;
#pragma unroll
                    for (int c4 = 0; c4 < 32; ++c4) {
                        const uint4 w = dropout_words(dr, m0 + c4, static_cast<uint32_t>(rq),
                                                      static_cast<uint32_t>(it.bh));
                        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
                        float pk[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float pv = ex2_approx(fmaf(s[4 * c4 + q], scale_log2, -m_sub));
                            lsum += pv;
                            pk[q] = words[q] < dr.thresh ? pv : 0.f;
                            lres += __bfloat162float(__float2bfloat16_rn(pk[q])) - pk[q];
                        }
                        p[2 * c4] = pack_bf16x2(pk[0], pk[1]);
                        p[2 * c4 + 1] = pack_bf16x2(pk[2], pk[3]);
                    }
                    l += lsum;
                    lc += lres;
                    tmem_st_x32(tS, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                    tmem_st_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
                } else if (two_part_p<CAUSAL, MASK, DROP>(it, t, it.jb0 + j, N)) {
                // the row sees only this block: p = hi + lo, both bf16, stored a quarter at a time
                // (hi over the first 64 columns of S, lo over the next 64, which S no longer needs)
                // for the two P V products; the applied weights then equal p to about 2^-17
                const uint64_t c2 = f2_pack(scale_log2, scale_log2);
                const uint64_t nm2 = f2_pack(-m_sub, -m_sub);
                uint64_t acc[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = 0ull;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int e = 2 * (16 * h + c);
                        const float2 x = f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), c2, nm2));
                        const float p0 = ex2_approx(x.x);
                        const float p1 = ex2_approx(x.y);
                        acc[c & 3] = f2_add(acc[c & 3], f2_pack(p0, p1));
                        hi[c] = pack_bf16x2(p0, p1);
                        const float h0 = __uint_as_float(hi[c] << 16);
                        const float h1 = __uint_as_float(hi[c] & 0xFFFF0000u);
                        lo[c] = pack_bf16x2(p0 - h0, p1 - h1);
                    }
                    tmem_st_x16(tS + 16 * h, hi);
                    tmem_st_x16(tS + 64 + 16 * h, lo);
                }
                const float2 a = f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])));
                l += a.x + a.y;
                } else {
                uint32_t p[64];
                // p = 2^(s c - m) on pairs: one packed FMA, two ex2, packed sums in 4 chains
                const uint64_t c2 = f2_pack(scale_log2, scale_log2);
                const uint64_t nm2 = f2_pack(-m_sub, -m_sub);
                uint64_t acc[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = 0ull;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const float2 x = f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), c2, nm2));
                    const float p0 = ex2_approx(x.x);
                    const float p1 = ex2_approx(x.y);
                    acc[c & 3] = f2_add(acc[c & 3], f2_pack(p0, p1));
                    p[c] = pack_bf16x2(p0, p1);
                }
                {
                    const float2 a = f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])));
                    l += a.x + a.y;
                    // the block's largest weight, computed exactly as its element was above: its
                    // rounding residual joins the normaliser only when it dominates the row so far
                    const float ptop = ex2_approx(fmaf(mx, scale_log2, -m_sub));
                    if (ptop >= 0.5f * l) lc += __bfloat162float(__float2bfloat16_rn(ptop)) - ptop;
                }
                tmem_st_x32(tS, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                tmem_st_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
                }
                if (D == 128 && rescale_o) rescale_o_row<D>(tO, alpha_o);   // (warp-uniform)
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[t]);
            }
            if (!ok) break;
            // epilogue: O = C / (l + lc) -> bf16 -> global, LSE; then hand O's TMEM back
            ok = __all_sync(0xffffffffu, mbar_wait(&o_full[t], of & 1, abort_flag, status));
            if (!ok) break;
            ++of;
            tc_fence_after();
            // General mask: rows past the valid length, or left with no allowed key, give 0 / -inf.
            const bool dead = MASK && (rq >= it.lq || !(l > 0.f));
            const float inv_l = dead ? 0.f : (DROP ? dr.rscale : 1.f) / (l + lc);
            const size_t orow_idx = ((SPLIT ? static_cast<size_t>(it.split) * BH : 0) + it.bh) *
                                        static_cast<size_t>(N) + rq;
            // (debug builds: the row of O and LSE this thread writes lies inside them)
            const bool row_ok = rq < N && in_bounds(static_cast<long long>(orow_idx), rows_total, status);
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_x32(tO + c0, o);
                if (row_ok) {
                    if constexpr (SPLIT) {
                        float *orow = static_cast<float *>(Out) + orow_idx * D;
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            float4 v;
                            v.x = __uint_as_float(o[4 * u + 0]) * inv_l;
                            v.y = __uint_as_float(o[4 * u + 1]) * inv_l;
                            v.z = __uint_as_float(o[4 * u + 2]) * inv_l;
                            v.w = __uint_as_float(o[4 * u + 3]) * inv_l;
                            *reinterpret_cast<float4 *>(orow + c0 + 4 * u) = v;
                        }
                    } else {
                        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(Out) + orow_idx * D;
                        if (MASK && dead) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = 0u;
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(o[8 * u + 0]) * inv_l, __uint_as_float(o[8 * u + 1]) * inv_l);
                            v.y = pack_bf16x2(__uint_as_float(o[8 * u + 2]) * inv_l, __uint_as_float(o[8 * u + 3]) * inv_l);
                            v.z = pack_bf16x2(__uint_as_float(o[8 * u + 4]) * inv_l, __uint_as_float(o[8 * u + 5]) * inv_l);
                            v.w = pack_bf16x2(__uint_as_float(o[8 * u + 6]) * inv_l, __uint_as_float(o[8 * u + 7]) * inv_l);
                            *reinterpret_cast<uint4 *>(orow + c0 + 8 * u) = v;
                        }
                    }
                }
            }
            if (row_ok) LSE[orow_idx] = (MASK && dead) ? -INFINITY : (m + log2f(l)) * LN2;
            tc_fence_before();
            mbar_arrive(&o_empty[t]);
        }
        tc_fence_before();
        __syncthreads();
    }
}

template <int D, bool CAUSAL, bool SPLIT, bool MASK, bool DROP>
cudaError_t launch(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                   const CUtensorMap &tmV, void *Out, float *LSE, int S, const MaskArgs &mk,
                   const DropoutArgs &dr, unsigned *status, cudaStream_t stream) {
    auto kern = fwd_kernel<D, CAUSAL, SPLIT, MASK, DROP>;
    const int smem = Layout<D>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // The in-kernel register split needs the launch to provide at least REGS_NEEDED registers.
    cudaFuncAttributes attr{};
    e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs * NUM_THREADS < REGS_NEEDED) return cudaErrorInvalidConfiguration;
    const int BH = p.B * p.Hq;
    const long long n_pairs = (p.N + 2 * BM - 1) / (2 * BM);
    const long long n_items = n_pairs * BH * S;
    if (n_items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // persistent: one CTA per SM (TMEM and shared memory allow no second one)
    const int grid = static_cast<int>(std::min<long long>(n_items, num_sms()));
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    kern<<<grid, NUM_THREADS, smem, stream>>>(tmQ, tmK, tmV, Out, LSE, p.Hq, p.Hkv, p.N, BH,
                                              static_cast<int>(n_items), S, scale_log2, mk, dr, status);
    return cudaGetLastError();
}

template <bool SPLIT, bool MASK, bool DROP>
cudaError_t dispatch(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                     const CUtensorMap &tmV, void *Out, float *LSE, int S, const MaskArgs &mk,
                     const DropoutArgs &dr, unsigned *status, cudaStream_t stream) {
    if (p.d == 128)
        return p.causal
                   ? launch<128, true, SPLIT, MASK, DROP>(p, tmQ, tmK, tmV, Out, LSE, S, mk, dr, status, stream)
                   : launch<128, false, SPLIT, MASK, DROP>(p, tmQ, tmK, tmV, Out, LSE, S, mk, dr, status, stream);
    if (p.d == 64)
        return p.causal
                   ? launch<64, true, SPLIT, MASK, DROP>(p, tmQ, tmK, tmV, Out, LSE, S, mk, dr, status, stream)
                   : launch<64, false, SPLIT, MASK, DROP>(p, tmQ, tmK, tmV, Out, LSE, S, mk, dr, status, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fwd

cudaError_t launch_fwd_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                            const CUtensorMap &tmV, void *O, float *LSE, unsigned *status,
                            cudaStream_t stream) {
    return fwd::dispatch<false, false, false>(p, tmQ, tmK, tmV, O, LSE, 1, MaskArgs{},
                                              DropoutArgs{}, status, stream);
}

cudaError_t launch_fwd_masked_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                   const CUtensorMap &tmV, void *O, float *LSE, const MaskArgs &mk,
                                   unsigned *status, cudaStream_t stream) {
    return fwd::dispatch<false, true, false>(p, tmQ, tmK, tmV, O, LSE, 1, mk, DropoutArgs{},
                                             status, stream);
}

cudaError_t launch_fwd_split_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                  const CUtensorMap &tmV, float *O_parts, float *LSE_parts,
                                  int num_splits, unsigned *status, cudaStream_t stream) {
    return fwd::dispatch<true, false, false>(p, tmQ, tmK, tmV, O_parts, LSE_parts, num_splits,
                                             MaskArgs{}, DropoutArgs{}, status, stream);
}

cudaError_t launch_fwd_dropout_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                    const CUtensorMap &tmV, void *O, float *LSE,
                                    const DropoutArgs &dr, unsigned *status, cudaStream_t stream) {
    return fwd::dispatch<false, false, true>(p, tmQ, tmK, tmV, O, LSE, 1, MaskArgs{}, dr, status,
                                             stream);
}

}  // namespace fa
