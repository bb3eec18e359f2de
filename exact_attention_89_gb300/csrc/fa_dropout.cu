// fa_dropout.cu -- fa_dropout_mask: the dropout keep decisions the kernels use, written out.
//
// One thread per (head, query, group of four keys): one Philox4x32-10 call gives the keep
// words of four consecutive keys (fa_philox.cuh has the rule).  Z is [BH, N, N] bytes.
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_philox.cuh"

namespace fa {
namespace drop {

__global__ void __launch_bounds__(256) mask_kernel(DropoutArgs dr, long long BH, int N,
                                                   unsigned char *__restrict__ Z) {
    const int quads = (N + 3) / 4;
    const long long total = BH * N * static_cast<long long>(quads);
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int m = static_cast<int>(t % quads);
        const long long row = t / quads;                  // bh * N + i
        const int i = static_cast<int>(row % N);
        const long long bh = row / N;
        const uint4 w = dropout_words(dr, static_cast<uint32_t>(m), static_cast<uint32_t>(i),
                                      static_cast<uint32_t>(bh));
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = 4 * m + q;
            if (j < N) Z[row * N + j] = words[q] < dr.thresh ? 1 : 0;
        }
    }
}

}  // namespace drop

cudaError_t launch_dropout_mask(const DropoutArgs &dr, long long BH, int N, unsigned char *Z,
                                cudaStream_t stream) {
    const long long total = BH * N * ((N + 3) / 4);
    long long grid = (total + 255) / 256;
    const long long cap = 16LL * num_sms();
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    drop::mask_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(dr, BH, N, Z);
    return cudaGetLastError();
}

}  // namespace fa
