// fa_internal.h -- host-side launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_philox.cuh"
#include "flashattn.h"

namespace fa {

// Number of SMs of the current device (cached per device).
int num_sms();

// Unique id (cuCtxGetId) of the calling thread's current CUDA context, 0 when none is current.
// Device addresses cached per device are tied to the context they were looked up in.
fa_status current_context_id(unsigned long long *id);

// Problem description after host validation.
struct Problem {
    int B, Hq, Hkv, N, d, causal;
    float scale;
};

// General mask of the masked entry points (device pointers; null members mean "no limit"):
// per-batch valid query rows and keys, and a 0/1 mask over 128 x 128 tiles [mask_heads, nb, nb].
struct MaskArgs {
    const int *q_len = nullptr;
    const int *k_len = nullptr;
    const uint8_t *block_mask = nullptr;
    int mask_heads = 0;
};

// K1: bf16 forward on tcgen05. Maps are 3-D [d, N, B*H] bf16, box [64, 128, 1], 128B swizzle;
// O is written with plain stores.
cudaError_t launch_fwd_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                            const CUtensorMap &tmV, void *O, float *LSE, unsigned *status,
                            cudaStream_t stream);

// K1 under a general mask.
cudaError_t launch_fwd_masked_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                   const CUtensorMap &tmV, void *O, float *LSE, const MaskArgs &mk,
                                   unsigned *status, cudaStream_t stream);

// K1 with dropout on P (keep rule in fa_philox.cuh).
cudaError_t launch_fwd_dropout_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                    const CUtensorMap &tmV, void *O, float *LSE,
                                    const DropoutArgs &dr, unsigned *status, cudaStream_t stream);

// Keep decisions Z [BH, N, N] bytes (1 = keep).
cudaError_t launch_dropout_mask(const DropoutArgs &dr, long long BH, int N, unsigned char *Z,
                                cudaStream_t stream);

// K1 split-KV variant: num_splits contiguous ranges of key blocks, each giving an fp32 partial
// O_parts [S, B*Hq, N, d] and LSE_parts [S, B*Hq, N] (-inf for rows with no key in the range).
cudaError_t launch_fwd_split_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                  const CUtensorMap &tmV, float *O_parts, float *LSE_parts,
                                  int num_splits, unsigned *status, cudaStream_t stream);

// K6: merge of S partials per row into O (bf16 or fp32) and LSE.
cudaError_t launch_merge(const float *O_parts, const float *LSE_parts, int S, long long rows, int d,
                         void *O, bool out_bf16, float *LSE, cudaStream_t stream);

// K8: the forward in the key/value-outer order (IO ablation); d = 128.  Workspace: fp32 running
// O [B*Hq, N, d] then m, l, lc [3][B*Hq, N].
size_t kvouter_workspace_bytes(long long BH, int N, int d);
cudaError_t launch_fwd_kvouter_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                    const CUtensorMap &tmV, void *O, float *LSE, float *workspace,
                                    unsigned *status, cudaStream_t stream);

// K9: fp32 forward with three TF32 products per product (d = 64).  Workspace: Qh, Ql
// [B*Hq, N, 64], Kh, Kl [B*Hkv, N, 64], V^T hi / lo [B*Hkv, 64, Np] fp32, Np = N rounded up to 32.
// maps: Qh, Ql (box [32, 128, 1]), Kh, Kl (box [32, 32, 1]), Vth, Vtl (box [32, 64, 1]).
size_t tf32x3_workspace_bytes(long long BH, long long BHkv, int N, int d);
cudaError_t launch_tf32x3_split(const Problem &p, const float *Q, const float *K, const float *V,
                                float *ws, cudaStream_t stream);
cudaError_t launch_tf32x3_attn(const Problem &p, const CUtensorMap *maps, float *O, float *LSE,
                               unsigned *status, cudaStream_t stream);

// K10: fp32 backward with three TF32 products per product (d = 64): the split kernels write the
// workspace below, then a dq pass (writes D and dQ) and a dkv pass (dK, dV).  Workspace, fp32:
// Qh, Ql, dOh, dOl [B*Hq, N, 64]; Kh, Kl, Vh, Vl [B*Hkv, N, 64]; transposed Qth, Qtl, dOth, dOtl
// [B*Hq, 64, Np]; Kth, Ktl [B*Hkv, 64, Np]; D [B*Hq, N]; Np = N rounded up to 32.
struct Tf32BwdWorkspace {
    float *Qh, *Ql, *dOh, *dOl, *Kh, *Kl, *Vh, *Vl, *Qth, *Qtl, *dOth, *dOtl, *Kth, *Ktl, *D;
    long long Np;
    size_t bytes;
};
// Pointers into `workspace` (null pointers when it is null) and the byte size.
Tf32BwdWorkspace tf32x3_bwd_layout(long long BH, long long BHkv, int N, int d, void *workspace);
cudaError_t launch_tf32x3_bwd_split(const Problem &p, const float *Q, const float *K, const float *V,
                                    const float *dO, const Tf32BwdWorkspace &w, cudaStream_t stream);
// maps: [0..5] Kh, Kl, Vh, Vl (box [32, 32, 1]), Kth, Ktl (box [32, 64, 1]); [6..13] Qh, Ql,
// dOh, dOl (box [32, 32, 1]), dOth, dOtl, Qth, Qtl (box [32, 64, 1]).
cudaError_t launch_tf32x3_bwd(const Problem &p, const CUtensorMap *maps, const float *Q, const float *K,
                              const float *V, const float *O, const float *dO, const float *LSE,
                              float *dQ, float *dK, float *dV, float *Dvec, unsigned *status,
                              cudaStream_t stream);

// K2: D = rowsum(dO * O) in fp32 and zeroing of the fp32 dQ accumulator, plus zero_tail_bytes
// (a multiple of 16) right after it (the deterministic variant's counters).
cudaError_t launch_bwd_preprocess_bf16(const Problem &p, const void *O, const void *dO, float *D,
                                       float *dQacc, cudaStream_t stream,
                                       size_t zero_tail_bytes = 0);

// K3: bf16 backward main loop on tcgen05.  tmQ / tmdO use a [64, 64, 1] box; tmK, tmV, tmdK,
// tmdV a [64, 128, 1] box.  Accumulates scale * dS K into dQacc with fp32 reductions: per
// element at head dim 128, per 64 x 64 tile through tmdQ (fp32 [d, N, B*Hq], box [64, 64, 1],
// no swizzle) at head dim 64; tmdQ is unused at 128.
cudaError_t launch_bwd_main_bf16(const Problem &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                                 const CUtensorMap &tmV, const CUtensorMap &tmdO,
                                 const CUtensorMap &tmdK, const CUtensorMap &tmdV,
                                 const CUtensorMap &tmdQ, const float *LSE, const float *D,
                                 float *dQacc, unsigned *status,
                                 cudaStream_t stream);

// K3 with the dQ reductions in a fixed order (bitwise reproducible dQ): dq_sem holds
// B * Hq * ceil(N / 64) * 4 zeroed turn counters and one zeroed abort word after them.
cudaError_t launch_bwd_main_deterministic_bf16(const Problem &p, const CUtensorMap &tmQ,
                                               const CUtensorMap &tmK, const CUtensorMap &tmV,
                                               const CUtensorMap &tmdO, const CUtensorMap &tmdK,
                                               const CUtensorMap &tmdV, const CUtensorMap &tmdQ,
                                               const float *LSE, const float *D, float *dQacc,
                                               unsigned *dq_sem, unsigned *status,
                                               cudaStream_t stream);

// K3 under a general mask.  Needs (Hq / Hkv) * ceil(N / 64) <= MASK_BWD_MAX_STEPS (the CTA's
// step list lives in shared memory).
constexpr int MASK_BWD_MAX_STEPS = 16384;
cudaError_t launch_bwd_main_masked_bf16(const Problem &p, const CUtensorMap &tmQ,
                                        const CUtensorMap &tmK, const CUtensorMap &tmV,
                                        const CUtensorMap &tmdO, const CUtensorMap &tmdK,
                                        const CUtensorMap &tmdV, const CUtensorMap &tmdQ,
                                        const float *LSE, const float *D,
                                        float *dQacc, const MaskArgs &mk, unsigned *status,
                                        cudaStream_t stream);

// K3 with dropout on P.
cudaError_t launch_bwd_main_dropout_bf16(const Problem &p, const CUtensorMap &tmQ,
                                         const CUtensorMap &tmK, const CUtensorMap &tmV,
                                         const CUtensorMap &tmdO, const CUtensorMap &tmdK,
                                         const CUtensorMap &tmdV, const CUtensorMap &tmdQ,
                                         const float *LSE, const float *D,
                                         float *dQacc, const DropoutArgs &dr, unsigned *status,
                                         cudaStream_t stream);

// K4: dQ = bf16(dQacc).
cudaError_t launch_bwd_dq_convert_bf16(const Problem &p, const float *dQacc, void *dQ,
                                       cudaStream_t stream);

// K5: fp32 SIMT forward / backward.
cudaError_t launch_fwd_fp32(const Problem &p, const float *Q, const float *K, const float *V,
                            float *O, float *LSE, cudaStream_t stream);
cudaError_t launch_bwd_fp32(const Problem &p, const float *Q, const float *K, const float *V,
                            const float *O, const float *dO, const float *LSE, float *dQ,
                            float *dK, float *dV, float *D, cudaStream_t stream);

}  // namespace fa
