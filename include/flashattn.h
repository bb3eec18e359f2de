/*
 * flashattn.h -- C ABI of libflashattn: exact scaled-dot-product attention on GB300 (sm_103a).
 *
 * What it computes. For every batch b and query head hq (key/value head hk = hq / (Hq / Hkv)):
 *     S = scale * Q K^T  (masked pairs excluded),  P = softmax_rows(S),  O = P V,
 *     LSE_i = ln sum_j exp(S_ij)  (natural log, over the allowed keys j).
 * The result is exact attention up to floating-point reordering: the method only reorganises
 * the computation (FlashAttention note (paweldubiel.com), section "mechanism and details").
 * The forward pass keeps one query tile on chip and streams key/value tiles past it with the
 * running row max m, running sum l and rescaled accumulator (FlashAttention DAC'24 reading note,
 * paper.adslab.icu, Methods, the l and O update equations), normalising once at the end
 * (paweldubiel.com note: result u / l).  The N x N matrices S and P never reach device memory.
 * The backward pass stores nothing but LSE from the forward and recomputes P tile by tile
 * ("Attention's hidden recurrence" blog by mzeromiko, section "Flash Attention backward"), with
 *     D_i = sum_k dO_ik O_ik,   dS = P * (dO V^T - D),
 *     dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO
 * (same blog, section "standard attention / backward"; dK and dV are summed over the query
 * heads that share a key/value head).
 *
 * Conventions shared by every entry point.
 *  - Layout: contiguous [B, H, N, d] with d fastest; Q, O, dO, dQ use H = Hq; K, V, dK, dV use
 *    H = Hkv; LSE is [B, Hq, N] fp32.  N need not be a multiple of any tile size.
 *  - causal != 0 keeps key j <= query i (top-left aligned, one N for queries and keys);
 *    causal == 0 keeps every key.
 *  - Ownership: every tensor pointer is a DEVICE pointer owned by the caller; the library keeps
 *    no reference after the call is enqueued.  The library allocates no device memory.
 *  - Execution: all work is enqueued on `stream` (0 = legacy default stream) and is
 *    asynchronous; nothing synchronises except fa_get_device_status.
 *  - Errors: arguments are validated on the host before anything is enqueued; a failed check
 *    returns its status and enqueues nothing.  A failed launch returns FA_ERR_CUDA.  Failures
 *    detected on the device (a bounded wait that ran out) are recorded in a per-device status
 *    word read by fa_get_device_status.  The library never prints, traps or exits.
 *  - Precision of the bf16 entry points: bf16 inputs and outputs, fp32 accumulation, fp32 LSE,
 *    probabilities rounded to bf16 (round-to-nearest-even) before the second product; rows that
 *    see only the first 128 keys (the first query tile of a causal head) apply them as two bf16
 *    parts, so their few large weights are not rounded.  Failures detected on the device also
 *    include FA_ERR_DEVICE_BOUNDS, reported only by debug builds (FA_DEBUG_BOUNDS), which check
 *    the kernels' computed global indices.
 */
#ifndef FLASHATTN_H
#define FLASHATTN_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,    /* a size < 1, Hq % Hkv != 0, non-finite or non-positive scale */
    FA_ERR_UNSUPPORTED = 2,    /* head dim not supported, or the device is not sm_103 */
    FA_ERR_MISALIGNED = 3,     /* a null pointer or one not aligned to 16 bytes */
    FA_ERR_WORKSPACE = 4,      /* workspace null or smaller than fa_bwd_workspace_bytes */
    FA_ERR_CUDA = 5,           /* a CUDA runtime/driver call or a launch failed */
    FA_ERR_DEVICE_TIMEOUT = 6, /* a kernel's bounded wait ran out (reported by the status word) */
    FA_ERR_DEVICE_BOUNDS = 7   /* a debug build's bounds check caught an index (reported likewise) */
} fa_status;

/*
 * Forward, bf16 on tcgen05 tensor cores.
 *   Q [B,Hq,N,d], K [B,Hkv,N,d], V [B,Hkv,N,d]: bf16 inputs.
 *   O [B,Hq,N,d] bf16 output; LSE [B,Hq,N] fp32 output (natural log, scale included).
 *   d must be 64 or 128.  scale is usually 1/sqrt(d).
 */
fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                 int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                 cudaStream_t stream);

/* Side of the square tiles a block mask of fa_fwd_masked / fa_bwd_masked covers. */
#define FA_MASK_BLOCK 128

/*
 * Forward under a general mask: valid lengths of a padded batch and a 0/1 mask over tiles, on
 * top of the causal rule.  The mask acts on whole tiles of Q K^T (FlashAttention DAC'24 reading
 * note, paper.adslab.icu, "other operators"): tiles a row may not see are skipped, not computed
 * and zeroed.  Masked pairs have weight 0.
 *   Q, K, V, O, LSE, sizes, causal, scale: as in fa_fwd (d 64 or 128).
 *   q_len, k_len: device int32 [B] or NULL.  Batch b's query rows i >= q_len[b] and keys
 *     j >= k_len[b] are padding (values clamped to [0, N]).  K and V padding rows must hold
 *     finite values (a zero weight times an infinite value would still give NaN).
 *   block_mask: device uint8 [mask_heads, nb, nb] or NULL, nb = ceil(N / FA_MASK_BLOCK);
 *     entry (h, a, c) != 0 lets query rows [a*128, a*128+128) see keys [c*128, c*128+128).
 *     mask_heads is 1 (one mask for every head), Hq (one per query head, shared by the batch)
 *     or B*Hq (one per (batch, query head), index b*Hq + hq); it is ignored when block_mask is
 *     NULL.
 *   A row with no allowed key, and every padding row, gets O = 0 and LSE = -inf.
 *   Errors as for fa_fwd, plus FA_ERR_INVALID_ARG for another mask_heads and FA_ERR_MISALIGNED
 *   for q_len / k_len not 4-byte aligned.  The mask arrays are only read, on `stream`.
 */
fa_status fa_fwd_masked(const void *Q, const void *K, const void *V, void *O, float *LSE,
                        int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                        const int *q_len, const int *k_len, const unsigned char *block_mask,
                        int mask_heads, cudaStream_t stream);

/*
 * Backward under a general mask: the gradients of fa_fwd_masked's output.  Arguments as in
 * fa_bwd, with O and LSE from fa_fwd_masked on the same mask, plus the mask of fa_fwd_masked.
 * Padding rows and rows with no allowed key get dQ = 0; padding keys (and keys no row may see)
 * get dK = dV = 0.  The padding rows of dO must hold finite values.
 * Also FA_ERR_UNSUPPORTED when (Hq / Hkv) * ceil(N / 64) > 16384 (each key block lists the
 * (query head, 64-row tile) steps its mask keeps in shared memory).
 */
fa_status fa_bwd_masked(const void *Q, const void *K, const void *V, const void *O,
                        const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                        int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                        const int *q_len, const int *k_len, const unsigned char *block_mask,
                        int mask_heads, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/*
 * Forward with dropout on the attention weights.  The FlashAttention DAC'24 reading note
 * (paper.adslab.icu, "other operators") lists dropout among the operations applied per block;
 * here it is inverted dropout on the normalised P: O = (P (.) Z / (1 - p)) V, LSE of the
 * undropped P.  Z (1 = keep) is a pure function of (seed, offset, head, query, key):
 *   element (i, j) of head b*Hq + hq is kept iff word (j mod 4) of Philox4x32-10 (Salmon et al.,
 *   "Parallel random numbers: as easy as 1, 2, 3", SC'11) with counter (j/4, i, b*Hq + hq,
 *   offset) and key (seed mod 2^32, seed / 2^32) is below floor((1 - p) 2^32).
 * The backward recomputes the same Z from the same (seed, offset); nothing is stored.
 *   Arguments as fa_fwd, plus 0 <= p_drop < 1 (0: exactly fa_fwd), seed, offset (give each
 *   call its own offset, or seed, to draw a fresh mask).  FA_ERR_INVALID_ARG for p_drop outside
 *   [0, 1) or NaN.
 */
fa_status fa_fwd_dropout(const void *Q, const void *K, const void *V, void *O, float *LSE,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         float p_drop, unsigned long long seed, unsigned offset,
                         cudaStream_t stream);

/*
 * Backward of fa_fwd_dropout (same p_drop, seed, offset; O and LSE from it):
 * dV = (P (.) Z / (1 - p))^T dO, dS = P (.) (Z / (1 - p) (.) dO V^T - D) with D = rowsum(dO (.) O),
 * dQ = scale dS K, dK = scale dS^T Q.  Arguments and errors as fa_bwd plus those of
 * fa_fwd_dropout.
 */
fa_status fa_bwd_dropout(const void *Q, const void *K, const void *V, const void *O,
                         const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         float p_drop, unsigned long long seed, unsigned offset,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The keep decisions Z of fa_fwd_dropout written out: Z [BH, N, N] device bytes (1 = keep) for
 * heads bh = 0 .. BH-1, computed by the same device code the kernels use.  For checking and
 * debugging; p_drop = 0 writes all ones.  Errors: FA_ERR_INVALID_ARG (sizes, p_drop),
 * FA_ERR_MISALIGNED (Z NULL), FA_ERR_CUDA.
 */
fa_status fa_dropout_mask(int BH, int N, float p_drop, unsigned long long seed, unsigned offset,
                          unsigned char *Z, cudaStream_t stream);

/*
 * Forward in the key/value-outer loop order, for measuring the IO cost of that order: the
 * FlashAttention DAC'24 reading note (paper.adslab.icu, Methods) reads every K/V element from
 * HBM once, with the outer loop over key/value blocks and the inner one over query blocks, and
 * each query block's running O, m and l written back and re-read per key/value block.  Same
 * result as fa_fwd (O bf16, LSE); one CTA per (batch, query head).
 *   Arguments as fa_fwd; d must be 128.  workspace: caller-owned device scratch of at least
 *   fa_fwd_kvouter_workspace_bytes(B, Hq, N, d) bytes, 16-byte aligned (fp32 running O and the
 *   per-row statistics); contents on entry do not matter.  Errors as fa_fwd plus
 *   FA_ERR_WORKSPACE.
 */
size_t fa_fwd_kvouter_workspace_bytes(int B, int Hq, int N, int d);
fa_status fa_fwd_kvouter(const void *Q, const void *K, const void *V, void *O, float *LSE,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Largest number of key ranges fa_fwd_split and fa_merge accept. */
#define FA_MAX_SPLITS 256

/*
 * Split-KV forward: the keys are cut into num_splits contiguous ranges and each range gives a
 * partial result on its own, to be combined by fa_merge.  Defined by the update of m, l and O
 * after each key block (FlashAttention DAC'24 reading note, paper.adslab.icu, Methods), applied
 * once more across ranges; a plain average of the range results would be wrong (FlashAttention
 * note, paweldubiel.com, on why each block's output needs its normaliser).  It spreads a
 * problem with few (batch, head, 256-query) items over more SMs.
 *   Q, K, V: bf16 as in fa_fwd; d must be 64 or 128; 1 <= num_splits <= FA_MAX_SPLITS.
 *   The N keys are cut in 128-key blocks; range s covers blocks [s*c, min((s+1)*c, nb)) with
 *   nb = ceil(N/128) and c = ceil(nb/num_splits) (ranges past the end are empty).
 *   O_parts [num_splits, B*Hq, N, d] fp32: range s's attention output over its keys alone,
 *     normalised over that range; unspecified for rows whose LSE_parts entry is -inf.
 *   LSE_parts [num_splits, B*Hq, N] fp32: natural-log log-sum-exp of the scaled scores over the
 *     range's allowed keys; -inf where a row has none (a range wholly after the row under the
 *     causal mask, or an empty range).
 *   Both caller-owned, 16-byte aligned, written entirely (O_parts only where LSE is finite).
 *   Errors as for fa_fwd, plus FA_ERR_INVALID_ARG for num_splits out of range.
 */
fa_status fa_fwd_split(const void *Q, const void *K, const void *V, float *O_parts,
                       float *LSE_parts, int B, int Hq, int Hkv, int N, int d, int causal,
                       float scale, int num_splits, cudaStream_t stream);

/*
 * Merge of partial attention results over disjoint key sets, row by row:
 *     LSE = ln sum_s e^{LSE_s},   O = sum_s e^{LSE_s - LSE} O_s
 * (the same reading-note update of m, l and O, in log-sum-exp form).  Parts with LSE_s = -inf
 * are skipped (their O_s is not read); a row whose parts are all -inf gets O = 0, LSE = -inf.
 *   O_parts [num_parts, rows, d] fp32 and LSE_parts [num_parts, rows] fp32 (the layout
 *   fa_fwd_split writes, with rows = B*Hq*N); 1 <= num_parts <= FA_MAX_SPLITS.
 *   O [rows, d]: bf16 when o_bf16 != 0 (the dtype fa_fwd writes), else fp32.  LSE [rows] fp32.
 *   d a multiple of 4, 4 <= d <= 1024.  All pointers 16-byte aligned device memory.
 *   Runs on the CUDA cores in fp32; computes in place of nothing (outputs must not alias inputs).
 */
fa_status fa_merge(const float *O_parts, const float *LSE_parts, int num_parts, long long rows,
                   int d, void *O, int o_bf16, float *LSE, cudaStream_t stream);

/*
 * Bytes of device workspace fa_bwd and fa_bwd_fp32 need: D [B,Hq,N] fp32 followed (at a
 * 256-byte boundary) by the fp32 dQ accumulator [B,Hq,N,d].  Returns 0 for invalid sizes and
 * SIZE_MAX when the size does not fit in size_t (no workspace can then pass the size checks).
 */
size_t fa_bwd_workspace_bytes(int B, int Hq, int N, int d);

/*
 * Backward, bf16 on tcgen05 tensor cores, recomputing P from LSE.
 *   Q, K, V, O, dO: bf16 inputs as in fa_fwd (O is the forward output; D is formed from it).
 *   LSE: the fp32 LSE fa_fwd wrote for these inputs.
 *   dQ [B,Hq,N,d], dK [B,Hkv,N,d], dV [B,Hkv,N,d]: bf16 outputs (dK, dV summed over the group).
 *   d must be 64 or 128 (at d = 64 the dQ^T product keeps the 128-row tiling over a zero-filled
 *   half of K; the other products run over the 64 real columns).
 *   workspace: caller-owned device scratch of at least fa_bwd_workspace_bytes(B,Hq,N,d) bytes,
 *   16-byte aligned; its contents on entry do not matter and are clobbered.
 *   Calls that share one workspace must not overlap on the GPU.
 */
fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                 const float *LSE, void *dQ, void *dK, void *dV,
                 int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                 void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Bytes of device workspace fa_bwd_deterministic needs: fa_bwd_workspace_bytes(B,Hq,N,d), then
 * 16 bytes per 64-row query tile of every (batch, query head) for the turn counters, then 16
 * bytes for an abort word.  Returns 0 for invalid sizes and SIZE_MAX on overflow.
 */
size_t fa_bwd_deterministic_workspace_bytes(int B, int Hq, int N, int d);

/*
 * fa_bwd with a dQ that is bitwise the same on every call with the same inputs (same GPU model
 * and library build).  Gradients by recompute as in the "Flash Attention backward" section of
 * the mzeromiko blog ("Attention's hidden recurrence"); fa_bwd adds the key blocks' shares of
 * dQ into its fp32 accumulator in whatever order the CTAs reach it, so its dQ can differ in the
 * last bits from call to call.  Here the shares of each 64-row query tile are added in one fixed
 * order (descending key block), each CTA waiting on a counter in the workspace for its turn;
 * dK and dV are computed as in fa_bwd (they need no cross-CTA sum and are reproducible there
 * too).  The results agree with fa_bwd's to the rounding of the fp32 sums.
 *   Arguments, layouts, results and errors are those of fa_bwd, except that the workspace must
 *   hold fa_bwd_deterministic_workspace_bytes(B,Hq,N,d) bytes.  Slower than fa_bwd: the CTAs of
 *   a head are launched in the reduction order (the longest last), a CTA can wait for its turn,
 *   and at d = 64 dQ goes out through per-element reductions instead of bulk tile reductions.
 *   Every wait for a turn is bounded; one that runs out reports FA_ERR_DEVICE_TIMEOUT through
 *   fa_get_device_status and ends the other CTAs' waits at once (dQ is then not valid).
 */
fa_status fa_bwd_deterministic(const void *Q, const void *K, const void *V, const void *O,
                               const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                               int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Size of the fixed device scratch that fa_bwd_noalloc uses: 64 MiB.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate device memory where
 * they run the backward (for example a plugin whose host framework owns every allocation and
 * only passes in the input and output buffers, or a runtime that plans all memory up front and
 * forbids allocation once it is serving).  The paper has no counterpart to this entry point;
 * it exists only for those callers.
 *   Arguments, layouts, results and errors are those of fa_bwd.  Instead of a workspace the
 *   call uses a fixed array of FA_NOALLOC_SCRATCH_BYTES compiled into the library, which every
 *   GPU that loads the library holds until the library is unloaded or the process exits.
 *   Returns FA_ERR_WORKSPACE, before touching the GPU, when fa_bwd_workspace_bytes(B,Hq,N,d)
 *   exceeds FA_NOALLOC_SCRATCH_BYTES (with d = 128 that is B*Hq*N above about 130,000 rows).
 *   It calls no allocation routine.  The first call on a device looks up the array's device
 *   address (cudaGetSymbolAddress, on the current device); make that first call before any
 *   stream capture.  The lookup is repeated in the first call after the device's context has
 *   changed (cudaDeviceReset, or the primary context released and created again), so the
 *   address never outlives its context; the array's contents do not survive such a reset.
 *   All calls on one device share the array.  Each call rewrites what it needs at its start,
 *   so what an earlier call left there does not matter, but calls that overlap on the GPU
 *   (other streams, other host threads) race on the array and give wrong results: order them.
 */
fa_status fa_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O,
                         const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         cudaStream_t stream);

/*
 * Forward in fp32 on the CUDA cores (no tensor cores), for checks that need fp32 accuracy.
 * Same shapes and semantics as fa_fwd with every tensor fp32; 1 <= d <= 128.
 */
fa_status fa_fwd_fp32(const float *Q, const float *K, const float *V, float *O, float *LSE,
                      int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                      cudaStream_t stream);

/*
 * Backward in fp32 on the CUDA cores.  Same shapes and semantics as fa_bwd with every tensor
 * fp32; 1 <= d <= 128; workspace as for fa_bwd (only its D part is used).
 */
fa_status fa_bwd_fp32(const float *Q, const float *K, const float *V, const float *O,
                      const float *dO, const float *LSE, float *dQ, float *dK, float *dV,
                      int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                      void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fp32 forward on the tensor cores: every product (Q K^T and P V) is formed from TF32 parts as
 * hi(A) hi(B) + hi(A) lo(B) + lo(A) hi(B) with fp32 accumulation, hi(x) being x with its 13 low
 * mantissa bits cleared and lo(x) = x - hi(x); the result agrees with the fp32 path to about
 * 1e-6.  Same method, shapes and semantics as fa_fwd_fp32 (FlashAttention DAC'24 reading note,
 * Methods); d must be 64 and B*Hq <= 65535.
 *   workspace: caller-owned device scratch of at least fa_fwd_fp32_tc_workspace_bytes(...)
 *   bytes, 16-byte aligned (the TF32 parts of Q, K and of V transposed); contents on entry do not
 *   matter.  Errors as fa_fwd_fp32 plus FA_ERR_WORKSPACE.
 */
size_t fa_fwd_fp32_tc_workspace_bytes(int B, int Hq, int Hkv, int N, int d);
fa_status fa_fwd_fp32_tc(const float *Q, const float *K, const float *V, float *O, float *LSE,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fp32 backward on the tensor cores, the counterpart of fa_fwd_fp32_tc: same shapes and
 * semantics as fa_bwd_fp32 (P recomputed from LSE, D = rowsum(dO O), dS = P (dP - D),
 * dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K; "Attention's hidden recurrence" blog,
 * "Flash Attention backward"), every product formed from TF32 parts as in fa_fwd_fp32_tc.
 * Two passes: one over query tiles (forms D and dQ) and one over key blocks (dK and dV, summed
 * over the G query heads of each KV head); each gradient is written once, no atomics.
 * d must be 64, B*Hq <= 65535; every pointer 16-byte aligned.
 *   workspace: caller-owned device scratch of at least fa_bwd_fp32_tc_workspace_bytes(...) bytes,
 *   16-byte aligned (TF32 parts of Q, dO, K, V, transposed copies of Q, dO, K, and D); contents
 *   on entry do not matter.  Errors as fa_bwd_fp32 plus FA_ERR_UNSUPPORTED for d != 64.
 */
size_t fa_bwd_fp32_tc_workspace_bytes(int B, int Hq, int Hkv, int N, int d);
fa_status fa_bwd_fp32_tc(const float *Q, const float *K, const float *V, const float *O,
                         const float *dO, const float *LSE, float *dQ, float *dK, float *dV,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status word.
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT or FA_ERR_DEVICE_BOUNDS (first failure recorded since the
 * last read), or FA_ERR_CUDA if the synchronisation itself failed.
 */
fa_status fa_get_device_status(cudaStream_t stream);

/* Static, human-readable name of a status code ("FA_OK", ...); never NULL. */
const char *fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FLASHATTN_H */
