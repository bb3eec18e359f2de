// fa_noalloc.cu -- fa_bwd_noalloc: the bf16 backward without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the backward pass:
// a plugin inside a host framework that owns every allocation and only hands the plugin its
// input and output buffers, or a runtime that plans all memory up front and forbids allocation
// (and its latency and fragmentation) once serving has started.  For them this entry point
// takes its scratch (D and the fp32 dQ accumulator) from a fixed array compiled into the
// library instead of from a workspace argument.  The array costs FA_NOALLOC_SCRATCH_BYTES of
// device memory on every GPU that loads the library, for as long as the library stays loaded.
//
// Host code must not use the array's name as a device address: on the host it names a
// stand-in object.  The device address is looked up with cudaGetSymbolAddress (with the device
// current) on the first call on each device and cached; it is looked up again when the device's
// context has changed since (after cudaDeviceReset, the array lives in a new context).
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa_internal.h"
#include "flashattn.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {nullptr};
unsigned long long g_noalloc_ctx[kMaxDevices] = {0};   // context each cached address belongs to

// Device address of the scratch array on the current device (looked up on first use, and again
// in a new context).
fa_status noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    unsigned long long ctx = 0;
    if (fa::current_context_id(&ctx) != FA_OK) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return FA_ERR_CUDA;
        // the lookup made the device's context current: remember which one it was
        if (fa::current_context_id(&ctx) != FA_OK || ctx == 0) return FA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O,
                                    const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                                    int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                                    cudaStream_t stream) {
    // Reject problems whose scratch does not fit before touching the GPU.
    if (fa_bwd_workspace_bytes(B, Hq, N, d) > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES))
        return FA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const fa_status st = noalloc_scratch(&scratch);
    if (st != FA_OK) return st;
    // The backward's first kernel rewrites all of D and zeroes the dQ accumulator on every call,
    // so whatever an earlier call left in the array does not matter.
    return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, N, d, causal, scale, scratch,
                  static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES), stream);
}
