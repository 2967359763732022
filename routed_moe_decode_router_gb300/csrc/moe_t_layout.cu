// moe_t_layout.cu -- conversion of NVFP4 matrices into the t layout
// (input-major: packed [K][N/2], scales [K/16][N]), the layout in which the
// fused one-row form reads the down projections.  A load-time step: one
// thread per output byte, plain gathers.
#include <cuda_runtime.h>

#include "moe_layout.h"

namespace moe {

__global__ void t_layout_kernel(const uint8_t *__restrict__ packed,
                                const uint8_t *__restrict__ scales, int count, int n_out,
                                int k_in, uint8_t *__restrict__ packed_t,
                                uint8_t *__restrict__ scales_t) {
    const size_t N = (size_t)n_out, K = (size_t)k_in;
    const size_t pk = N * K / 2, sc = N * K / 16;
    const size_t total = (size_t)count * (pk + sc);
    for (size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (size_t)gridDim.x * blockDim.x) {
        if (t < (size_t)count * pk) {
            // byte (k, n/2) of matrix m: codes (n, k) low, (n + 1, k) high
            const size_t m = t / pk, r = t % pk;
            const size_t k = r / (N / 2), n = 2 * (r % (N / 2));
            const uint8_t *src = packed + m * pk;
            const int sh = (int)(k & 1) * 4;
            const uint32_t lo = (src[n * (K / 2) + k / 2] >> sh) & 0xFu;
            const uint32_t hi = (src[(n + 1) * (K / 2) + k / 2] >> sh) & 0xFu;
            packed_t[t] = (uint8_t)(lo | (hi << 4));
        } else {
            // scale (n, block b) of matrix m to byte (b, n)
            const size_t u = t - (size_t)count * pk;
            const size_t m = u / sc, r = u % sc;
            const size_t bl = r / N, n = r % N;
            scales_t[u] = scales[m * sc + n * (K / 16) + bl];
        }
    }
}

cudaError_t launch_t_layout(const uint8_t *packed, const uint8_t *scales, int count, int n_out,
                            int k_in, uint8_t *packed_t, uint8_t *scales_t, cudaStream_t stream) {
    const size_t total = (size_t)count * ((size_t)n_out * k_in / 2 + (size_t)n_out * k_in / 16);
    const size_t blocks = (total + 255) / 256;
    const unsigned grid = (unsigned)(blocks < 65536 ? blocks : 65536);
    t_layout_kernel<<<grid, 256, 0, stream>>>(packed, scales, count, n_out, k_in, packed_t,
                                              scales_t);
    return cudaGetLastError();
}

}  // namespace moe
