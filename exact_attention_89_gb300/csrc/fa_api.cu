// fa_api.cu -- the C ABI of libflashattn (declared in include/flashattn.h).
//
// Host-side validation, TMA tensor-map encoding, the per-device status word and the launch
// sequence of each entry point.  No device memory is allocated here: the status word is a
// static __device__ variable, every tensor and the backward workspace belong to the caller.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "flashattn.h"

namespace fa {

__device__ unsigned g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool probed = false;
    bool sm103 = false;
    unsigned *status = nullptr;
    unsigned long long ctx_id = 0;   // context the status address belongs to
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Driver entry points behind current_context_id (looked up once through the runtime, so the
// library needs no link against libcuda).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::mutex g_ctx_mutex;

void *driver_entry(const char *name) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return fn;
}

}  // namespace

fa_status current_context_id(unsigned long long *id) {
    {
        std::lock_guard<std::mutex> lock(g_ctx_mutex);
        if (!g_ctx_get_current || !g_ctx_get_id) {
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(driver_entry("cuCtxGetCurrent"));
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(driver_entry("cuCtxGetId"));
            if (!g_ctx_get_current || !g_ctx_get_id) return FA_ERR_CUDA;
        }
    }
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return FA_ERR_CUDA;
    *id = 0;
    if (ctx != nullptr && g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return FA_ERR_CUDA;
    return FA_OK;
}

namespace {

// Current device's entry, probed once per context.  Returns FA_OK or the reason it cannot run.
fa_status current_device(DeviceInfo **out, bool need_sm103) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &di = g_dev[dev];
    // A device reset (or the primary context being released and created again) invalidates the
    // cached status address: look it up again in the new context.
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != FA_OK) return FA_ERR_CUDA;
    if (di.probed && (ctx == 0 || ctx != di.ctx_id)) di.probed = false;
    if (!di.probed) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return FA_ERR_CUDA;
        di.status = static_cast<unsigned *>(p);
        di.sm103 = (major == 10 && minor == 3);
        // the symbol lookup made the device's context current: remember which one it was
        if (current_context_id(&di.ctx_id) != FA_OK || di.ctx_id == 0) return FA_ERR_CUDA;
        di.probed = true;
    }
    if (need_sm103 && !di.sm103) return FA_ERR_UNSUPPORTED;
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return FA_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = &di;
    return FA_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_sizes(int B, int Hq, int Hkv, int N, int d, float scale) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    // index arithmetic is 64-bit; keep the TMA coordinate ranges (int32) and grid sizes sane
    if (static_cast<long long>(B) * Hq > (1LL << 31) - 1) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int g_sms[kMaxDevices] = {0};

// 3-D bf16 view [d, N, BH] of a contiguous [BH, N, d] tensor, box [64, rows, 1], 128B swizzle.
bool encode_bf16(CUtensorMap *m, const void *base, int d, int N, long long BH, int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// The backward's fp32 dQ accumulator [B*Hq, N, d] as a target of TMA reductions: box
// [64, 64, 1] (64 columns of one 64-query step of one head), no swizzle.
bool encode_dq(CUtensorMap *m, float *dQacc, int d, int N, long long BH) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dQacc, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f32(CUtensorMap *m, const void *base, long long inner, long long rows, long long planes,
                int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(planes)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 4,
                             static_cast<cuuint64_t>(inner) * static_cast<cuuint64_t>(rows) * 4};
    cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

}  // namespace fa

using fa::Problem;

extern "C" {

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
        case FA_ERR_DEVICE_BOUNDS: return "FA_ERR_DEVICE_BOUNDS";
    }
    return "FA_ERR_UNKNOWN";
}

size_t fa_bwd_workspace_bytes(int B, int Hq, int N, int d) {
    if (B < 1 || Hq < 1 || N < 1 || d < 1) return 0;
    // rows * (d + 1) * 4 + 255 must fit in size_t, or no workspace check could be trusted
    const size_t rows = static_cast<size_t>(B) * Hq;   // < 2^62: both factors are below 2^31
    const size_t limit = (SIZE_MAX - 256) / 4 / (static_cast<size_t>(d) + 1);
    if (rows > limit / static_cast<size_t>(N)) return SIZE_MAX;
    const size_t r = rows * static_cast<size_t>(N);
    return fa::align256(r * sizeof(float)) + r * static_cast<size_t>(d) * sizeof(float);
}

size_t fa_bwd_deterministic_workspace_bytes(int B, int Hq, int N, int d) {
    const size_t base = fa_bwd_workspace_bytes(B, Hq, N, d);
    if (base == 0 || base == SIZE_MAX) return base;
    // four turn counters per 64-row query tile, then the abort word (padded to 16 bytes)
    const size_t tiles = static_cast<size_t>(B) * Hq * ((static_cast<size_t>(N) + 63) / 64);
    if (tiles > (SIZE_MAX - 16) / 16) return SIZE_MAX;
    const size_t extra = tiles * 16 + 16;
    if (base > SIZE_MAX - extra) return SIZE_MAX;
    return base + extra;
}

fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int Hq,
                 int Hkv, int N, int d, int causal, float scale, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(LSE))
        return FA_ERR_MISALIGNED;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    CUtensorMap tq, tk, tv;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 128) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    return fa::from_cuda(fa::launch_fwd_bf16(p, tq, tk, tv, O, LSE, di->status, stream));
}

}  // extern "C"

namespace fa {
namespace {
// Host checks of a general mask; fills the kernel's MaskArgs.
fa_status check_mask(int B, int Hq, const int *q_len, const int *k_len,
                     const unsigned char *block_mask, int mask_heads, MaskArgs *mk) {
    if ((q_len && (reinterpret_cast<uintptr_t>(q_len) & 3u)) ||
        (k_len && (reinterpret_cast<uintptr_t>(k_len) & 3u)))
        return FA_ERR_MISALIGNED;
    if (block_mask && mask_heads != 1 && mask_heads != Hq && mask_heads != B * Hq)
        return FA_ERR_INVALID_ARG;
    mk->q_len = q_len;
    mk->k_len = k_len;
    mk->block_mask = block_mask;
    mk->mask_heads = block_mask ? mask_heads : 0;
    return FA_OK;
}
// Host checks of a dropout probability; fills the kernels' DropoutArgs (p = 0: no dropout).
fa_status make_dropout(float p, unsigned long long seed, unsigned offset, DropoutArgs *dr,
                       bool *active) {
    if (!(p >= 0.f) || !(p < 1.f)) return FA_ERR_INVALID_ARG;   // also rejects NaN
    *active = p > 0.f;
    const double t = std::floor((1.0 - static_cast<double>(p)) * 4294967296.0);
    set_round_keys(dr, seed);
    dr->offset = offset;
    dr->thresh = t >= 4294967295.0 ? 0xFFFFFFFFu : static_cast<uint32_t>(t);
    dr->rscale = static_cast<float>(1.0 / (1.0 - static_cast<double>(p)));
    return FA_OK;
}
}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_fwd_dropout(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                         int Hq, int Hkv, int N, int d, int causal, float scale, float p_drop,
                         unsigned long long seed, unsigned offset, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    fa::DropoutArgs dr;
    bool active = false;
    if ((st = fa::make_dropout(p_drop, seed, offset, &dr, &active)) != FA_OK) return st;
    if (!active) return fa_fwd(Q, K, V, O, LSE, B, Hq, Hkv, N, d, causal, scale, stream);
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(LSE))
        return FA_ERR_MISALIGNED;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    CUtensorMap tq, tk, tv;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 128) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    return fa::from_cuda(fa::launch_fwd_dropout_bf16(p, tq, tk, tv, O, LSE, dr, di->status, stream));
}

fa_status fa_bwd_dropout(const void *Q, const void *K, const void *V, const void *O,
                         const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                         int Hq, int Hkv, int N, int d, int causal, float scale, float p_drop,
                         unsigned long long seed, unsigned offset, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    fa::DropoutArgs dr;
    bool active = false;
    if ((st = fa::make_dropout(p_drop, seed, offset, &dr, &active)) != FA_OK) return st;
    if (!active)
        return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, N, d, causal, scale, workspace,
                      workspace_bytes, stream);
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(dO) || !fa::aligned16(LSE) || !fa::aligned16(dQ) || !fa::aligned16(dK) ||
        !fa::aligned16(dV))
        return FA_ERR_MISALIGNED;
    if (!fa::aligned16(workspace) || workspace_bytes < fa_bwd_workspace_bytes(B, Hq, N, d))
        return FA_ERR_WORKSPACE;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    const size_t rows = static_cast<size_t>(B) * Hq * N;
    float *Dvec = static_cast<float *>(workspace);
    float *dQacc = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                             fa::align256(rows * sizeof(float)));
    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 64) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tdo, dO, d, N, 1LL * B * Hq, 64) ||
        !fa::encode_bf16(&tdk, dK, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tdv, dV, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    if (!fa::encode_dq(&tdq, dQacc, d, N, 1LL * B * Hq)) return FA_ERR_CUDA;
    cudaError_t e = fa::launch_bwd_preprocess_bf16(p, O, dO, Dvec, dQacc, stream);
    if (e == cudaSuccess)
        e = fa::launch_bwd_main_dropout_bf16(p, tq, tk, tv, tdo, tdk, tdv, tdq, LSE, Dvec, dQacc, dr,
                                             di->status, stream);
    if (e == cudaSuccess) e = fa::launch_bwd_dq_convert_bf16(p, dQacc, dQ, stream);
    return fa::from_cuda(e);
}

fa_status fa_dropout_mask(int BH, int N, float p_drop, unsigned long long seed, unsigned offset,
                          unsigned char *Z, cudaStream_t stream) {
    if (BH < 1 || N < 1) return FA_ERR_INVALID_ARG;
    fa::DropoutArgs dr;
    bool active = false;
    fa_status st = fa::make_dropout(p_drop, seed, offset, &dr, &active);
    if (st != FA_OK) return st;
    if (Z == nullptr) return FA_ERR_MISALIGNED;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const size_t bytes = static_cast<size_t>(BH) * N * N;
    if (!active) return fa::from_cuda(cudaMemsetAsync(Z, 1, bytes, stream));
    return fa::from_cuda(fa::launch_dropout_mask(dr, BH, N, Z, stream));
}

fa_status fa_fwd_masked(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                        int Hq, int Hkv, int N, int d, int causal, float scale, const int *q_len,
                        const int *k_len, const unsigned char *block_mask, int mask_heads,
                        cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(LSE))
        return FA_ERR_MISALIGNED;
    fa::MaskArgs mk;
    if ((st = fa::check_mask(B, Hq, q_len, k_len, block_mask, mask_heads, &mk)) != FA_OK) return st;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    CUtensorMap tq, tk, tv;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 128) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    return fa::from_cuda(fa::launch_fwd_masked_bf16(p, tq, tk, tv, O, LSE, mk, di->status, stream));
}

fa_status fa_bwd_masked(const void *Q, const void *K, const void *V, const void *O,
                        const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                        int Hq, int Hkv, int N, int d, int causal, float scale, const int *q_len,
                        const int *k_len, const unsigned char *block_mask, int mask_heads,
                        void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(Hq / Hkv) * ((N + 63) / 64) > fa::MASK_BWD_MAX_STEPS)
        return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(dO) || !fa::aligned16(LSE) || !fa::aligned16(dQ) || !fa::aligned16(dK) ||
        !fa::aligned16(dV))
        return FA_ERR_MISALIGNED;
    fa::MaskArgs mk;
    if ((st = fa::check_mask(B, Hq, q_len, k_len, block_mask, mask_heads, &mk)) != FA_OK) return st;
    if (!fa::aligned16(workspace) || workspace_bytes < fa_bwd_workspace_bytes(B, Hq, N, d))
        return FA_ERR_WORKSPACE;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    const size_t rows = static_cast<size_t>(B) * Hq * N;
    float *Dvec = static_cast<float *>(workspace);
    float *dQacc = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                             fa::align256(rows * sizeof(float)));
    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 64) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tdo, dO, d, N, 1LL * B * Hq, 64) ||
        !fa::encode_bf16(&tdk, dK, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tdv, dV, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    if (!fa::encode_dq(&tdq, dQacc, d, N, 1LL * B * Hq)) return FA_ERR_CUDA;
    cudaError_t e = fa::launch_bwd_preprocess_bf16(p, O, dO, Dvec, dQacc, stream);
    if (e == cudaSuccess)
        e = fa::launch_bwd_main_masked_bf16(p, tq, tk, tv, tdo, tdk, tdv, tdq, LSE, Dvec, dQacc, mk,
                                            di->status, stream);
    if (e == cudaSuccess) e = fa::launch_bwd_dq_convert_bf16(p, dQacc, dQ, stream);
    return fa::from_cuda(e);
}

size_t fa_fwd_kvouter_workspace_bytes(int B, int Hq, int N, int d) {
    if (B < 1 || Hq < 1 || N < 1 || d < 1) return 0;
    return fa::kvouter_workspace_bytes(static_cast<long long>(B) * Hq, N, d);
}

fa_status fa_fwd_kvouter(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                         int Hq, int Hkv, int N, int d, int causal, float scale, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(LSE))
        return FA_ERR_MISALIGNED;
    if (!fa::aligned16(workspace) || workspace_bytes < fa_fwd_kvouter_workspace_bytes(B, Hq, N, d))
        return FA_ERR_WORKSPACE;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    CUtensorMap tq, tk, tv;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 128) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    return fa::from_cuda(fa::launch_fwd_kvouter_bf16(p, tq, tk, tv, O, LSE,
                                                     static_cast<float *>(workspace), di->status,
                                                     stream));
}

size_t fa_fwd_fp32_tc_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return 0;
    return fa::tf32x3_workspace_bytes(1LL * B * Hq, 1LL * B * Hkv, N, d);
}

fa_status fa_fwd_fp32_tc(const float *Q, const float *K, const float *V, float *O, float *LSE,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 64) return FA_ERR_UNSUPPORTED;
    if (1LL * B * Hq > 65535) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(LSE))
        return FA_ERR_MISALIGNED;
    if (!fa::aligned16(workspace) ||
        workspace_bytes < fa_fwd_fp32_tc_workspace_bytes(B, Hq, Hkv, N, d))
        return FA_ERR_WORKSPACE;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    const long long BH = 1LL * B * Hq, BHkv = 1LL * B * Hkv;
    const long long Np = (N + 31) / 32 * 32;
    float *ws = static_cast<float *>(workspace);
    float *Qh = ws, *Ql = Qh + BH * N * d, *Kh = Ql + BH * N * d, *Kl = Kh + BHkv * N * d;
    float *Vth = Kl + BHkv * N * d, *Vtl = Vth + BHkv * d * Np;
    CUtensorMap maps[6];
    if (!fa::encode_f32(&maps[0], Qh, d, N, BH, 128) || !fa::encode_f32(&maps[1], Ql, d, N, BH, 128) ||
        !fa::encode_f32(&maps[2], Kh, d, N, BHkv, 32) || !fa::encode_f32(&maps[3], Kl, d, N, BHkv, 32) ||
        !fa::encode_f32(&maps[4], Vth, Np, d, BHkv, 64) || !fa::encode_f32(&maps[5], Vtl, Np, d, BHkv, 64))
        return FA_ERR_CUDA;
    cudaError_t e = fa::launch_tf32x3_split(p, Q, K, V, ws, stream);
    if (e == cudaSuccess) e = fa::launch_tf32x3_attn(p, maps, O, LSE, di->status, stream);
    return fa::from_cuda(e);
}

size_t fa_bwd_fp32_tc_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return 0;
    return fa::tf32x3_bwd_layout(1LL * B * Hq, 1LL * B * Hkv, N, d, nullptr).bytes;
}

fa_status fa_bwd_fp32_tc(const float *Q, const float *K, const float *V, const float *O,
                         const float *dO, const float *LSE, float *dQ, float *dK, float *dV,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 64) return FA_ERR_UNSUPPORTED;
    if (1LL * B * Hq > 65535) return FA_ERR_UNSUPPORTED;
    const void *ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
    for (const void *q : ptrs)
        if (!fa::aligned16(q)) return FA_ERR_MISALIGNED;
    if (!fa::aligned16(workspace) ||
        workspace_bytes < fa_bwd_fp32_tc_workspace_bytes(B, Hq, Hkv, N, d))
        return FA_ERR_WORKSPACE;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    const long long BH = 1LL * B * Hq, BHkv = 1LL * B * Hkv;
    const fa::Tf32BwdWorkspace w = fa::tf32x3_bwd_layout(BH, BHkv, N, d, workspace);
    CUtensorMap maps[14];
    const bool enc =
        fa::encode_f32(&maps[0], w.Kh, d, N, BHkv, 32) && fa::encode_f32(&maps[1], w.Kl, d, N, BHkv, 32) &&
        fa::encode_f32(&maps[2], w.Vh, d, N, BHkv, 32) && fa::encode_f32(&maps[3], w.Vl, d, N, BHkv, 32) &&
        fa::encode_f32(&maps[4], w.Kth, w.Np, d, BHkv, 64) && fa::encode_f32(&maps[5], w.Ktl, w.Np, d, BHkv, 64) &&
        fa::encode_f32(&maps[6], w.Qh, d, N, BH, 32) && fa::encode_f32(&maps[7], w.Ql, d, N, BH, 32) &&
        fa::encode_f32(&maps[8], w.dOh, d, N, BH, 32) && fa::encode_f32(&maps[9], w.dOl, d, N, BH, 32) &&
        fa::encode_f32(&maps[10], w.dOth, w.Np, d, BH, 64) && fa::encode_f32(&maps[11], w.dOtl, w.Np, d, BH, 64) &&
        fa::encode_f32(&maps[12], w.Qth, w.Np, d, BH, 64) && fa::encode_f32(&maps[13], w.Qtl, w.Np, d, BH, 64);
    if (!enc) return FA_ERR_CUDA;
    cudaError_t e = fa::launch_tf32x3_bwd_split(p, Q, K, V, dO, w, stream);
    if (e == cudaSuccess)
        e = fa::launch_tf32x3_bwd(p, maps, Q, K, V, O, dO, LSE, dQ, dK, dV, w.D, di->status, stream);
    return fa::from_cuda(e);
}

fa_status fa_fwd_split(const void *Q, const void *K, const void *V, float *O_parts,
                       float *LSE_parts, int B, int Hq, int Hkv, int N, int d, int causal,
                       float scale, int num_splits, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O_parts) ||
        !fa::aligned16(LSE_parts))
        return FA_ERR_MISALIGNED;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    CUtensorMap tq, tk, tv;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 128) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    return fa::from_cuda(fa::launch_fwd_split_bf16(p, tq, tk, tv, O_parts, LSE_parts, num_splits,
                                                   di->status, stream));
}

fa_status fa_merge(const float *O_parts, const float *LSE_parts, int num_parts, long long rows,
                   int d, void *O, int o_bf16, float *LSE, cudaStream_t stream) {
    if (num_parts < 1 || num_parts > FA_MAX_SPLITS || rows < 1 || d < 4 || d % 4 != 0 || d > 1024)
        return FA_ERR_INVALID_ARG;
    if (!fa::aligned16(O_parts) || !fa::aligned16(LSE_parts) || !fa::aligned16(O) ||
        !fa::aligned16(LSE))
        return FA_ERR_MISALIGNED;
    fa::DeviceInfo *di = nullptr;
    fa_status st = fa::current_device(&di, true);
    if (st != FA_OK) return st;
    return fa::from_cuda(
        fa::launch_merge(O_parts, LSE_parts, num_parts, rows, d, O, o_bf16 != 0, LSE, stream));
}

fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                 const float *LSE, void *dQ, void *dK, void *dV, int B, int Hq, int Hkv, int N,
                 int d, int causal, float scale, void *workspace, size_t workspace_bytes,
                 cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(dO) || !fa::aligned16(LSE) || !fa::aligned16(dQ) || !fa::aligned16(dK) ||
        !fa::aligned16(dV))
        return FA_ERR_MISALIGNED;
    if (!fa::aligned16(workspace) || workspace_bytes < fa_bwd_workspace_bytes(B, Hq, N, d))
        return FA_ERR_WORKSPACE;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    const size_t rows = static_cast<size_t>(B) * Hq * N;
    float *Dvec = static_cast<float *>(workspace);
    float *dQacc = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                             fa::align256(rows * sizeof(float)));
    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 64) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tdo, dO, d, N, 1LL * B * Hq, 64) ||
        !fa::encode_bf16(&tdk, dK, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tdv, dV, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    if (!fa::encode_dq(&tdq, dQacc, d, N, 1LL * B * Hq)) return FA_ERR_CUDA;
    cudaError_t e = fa::launch_bwd_preprocess_bf16(p, O, dO, Dvec, dQacc, stream);
    if (e == cudaSuccess)
        e = fa::launch_bwd_main_bf16(p, tq, tk, tv, tdo, tdk, tdv, tdq, LSE, Dvec, dQacc, di->status,
                                     stream);
    if (e == cudaSuccess) e = fa::launch_bwd_dq_convert_bf16(p, dQacc, dQ, stream);
    return fa::from_cuda(e);
}

fa_status fa_bwd_deterministic(const void *Q, const void *K, const void *V, const void *O,
                               const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                               int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(dO) || !fa::aligned16(LSE) || !fa::aligned16(dQ) || !fa::aligned16(dK) ||
        !fa::aligned16(dV))
        return FA_ERR_MISALIGNED;
    if (!fa::aligned16(workspace) ||
        workspace_bytes < fa_bwd_deterministic_workspace_bytes(B, Hq, N, d))
        return FA_ERR_WORKSPACE;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    const size_t rows = static_cast<size_t>(B) * Hq * N;
    const size_t base = fa_bwd_workspace_bytes(B, Hq, N, d);
    float *Dvec = static_cast<float *>(workspace);
    float *dQacc = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                             fa::align256(rows * sizeof(float)));
    // the counters follow the accumulator directly (base is a multiple of 16 for d = 64, 128), so
    // K2 clears both in one pass
    unsigned *dq_sem = reinterpret_cast<unsigned *>(static_cast<char *>(workspace) + base);
    const size_t sem_bytes = fa_bwd_deterministic_workspace_bytes(B, Hq, N, d) - base;
    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
    if (!fa::encode_bf16(&tq, Q, d, N, 1LL * B * Hq, 64) ||
        !fa::encode_bf16(&tk, K, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tv, V, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tdo, dO, d, N, 1LL * B * Hq, 64) ||
        !fa::encode_bf16(&tdk, dK, d, N, 1LL * B * Hkv, 128) ||
        !fa::encode_bf16(&tdv, dV, d, N, 1LL * B * Hkv, 128))
        return FA_ERR_CUDA;
    if (!fa::encode_dq(&tdq, dQacc, d, N, 1LL * B * Hq)) return FA_ERR_CUDA;
    cudaError_t e = fa::launch_bwd_preprocess_bf16(p, O, dO, Dvec, dQacc, stream, sem_bytes);
    if (e == cudaSuccess)
        e = fa::launch_bwd_main_deterministic_bf16(p, tq, tk, tv, tdo, tdk, tdv, tdq, LSE, Dvec,
                                                   dQacc, dq_sem, di->status, stream);
    if (e == cudaSuccess) e = fa::launch_bwd_dq_convert_bf16(p, dQacc, dQ, stream);
    return fa::from_cuda(e);
}

fa_status fa_fwd_fp32(const float *Q, const float *K, const float *V, float *O, float *LSE, int B,
                      int Hq, int Hkv, int N, int d, int causal, float scale, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d > 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(LSE))
        return FA_ERR_MISALIGNED;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    return fa::from_cuda(fa::launch_fwd_fp32(p, Q, K, V, O, LSE, stream));
}

fa_status fa_bwd_fp32(const float *Q, const float *K, const float *V, const float *O,
                      const float *dO, const float *LSE, float *dQ, float *dK, float *dV, int B,
                      int Hq, int Hkv, int N, int d, int causal, float scale, void *workspace,
                      size_t workspace_bytes, cudaStream_t stream) {
    fa_status st = fa::check_sizes(B, Hq, Hkv, N, d, scale);
    if (st != FA_OK) return st;
    if (d > 128) return FA_ERR_UNSUPPORTED;
    if (!fa::aligned16(Q) || !fa::aligned16(K) || !fa::aligned16(V) || !fa::aligned16(O) ||
        !fa::aligned16(dO) || !fa::aligned16(LSE) || !fa::aligned16(dQ) || !fa::aligned16(dK) ||
        !fa::aligned16(dV))
        return FA_ERR_MISALIGNED;
    if (!fa::aligned16(workspace) || workspace_bytes < fa_bwd_workspace_bytes(B, Hq, N, d))
        return FA_ERR_WORKSPACE;
    fa::DeviceInfo *di = nullptr;
    if ((st = fa::current_device(&di, true)) != FA_OK) return st;
    const Problem p{B, Hq, Hkv, N, d, causal ? 1 : 0, scale};
    return fa::from_cuda(fa::launch_bwd_fp32(p, Q, K, V, O, dO, LSE, dQ, dK, dV,
                                             static_cast<float *>(workspace), stream));
}

fa_status fa_get_device_status(cudaStream_t stream) {
    fa::DeviceInfo *di = nullptr;
    fa_status st = fa::current_device(&di, false);
    if (st != FA_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, fa::g_status_word, sizeof(word)) != cudaSuccess)
        return FA_ERR_CUDA;
    if (word != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(fa::g_status_word, &zero, sizeof(zero)) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return static_cast<fa_status>(word);
}

}  // extern "C"
