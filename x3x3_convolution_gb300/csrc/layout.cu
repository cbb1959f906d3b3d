// Layout conversion used by the stack driver: a 2D NCHW activation to channels-last, with the
// channel count rounded up to a multiple of 8 (zero channels) so that every position row is a whole
// number of 16-byte units for the channels-last engine's TMA boxes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace x3 {

namespace {

// One thread per position: the position's C values (one per channel plane; consecutive threads
// read consecutive positions, so each channel's reads are coalesced) are written as C8 contiguous
// channels in 16-byte pieces, zero past C.
__global__ void __launch_bounds__(256) nchw_to_nhwc_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                                                           int C, int C8, size_t plane, size_t positions) {
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < positions;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t n = idx / plane, pix = idx % plane;
        const uint16_t* xs = x + n * C * plane + pix;
        uint4* yd = reinterpret_cast<uint4*>(y + idx * C8);
        for (int c0 = 0; c0 < C8; c0 += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = c0 + 2 * e;
                const uint32_t lo = c < C ? __ldg(xs + (size_t)c * plane) : 0u;
                const uint32_t hi = c + 1 < C ? __ldg(xs + (size_t)(c + 1) * plane) : 0u;
                w[e] = lo | (hi << 16);
            }
            yd[c0 / 8] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

}  // namespace

x3_status launch_nchw_to_nhwc(const void* x, void* y, int N, int C, int C8, int H, int W, cudaStream_t s) {
    if (N < 1 || C < 1 || C8 < C || C8 % 8 != 0 || H < 1 || W < 1)
        return fail(X3_ERR_UNSUPPORTED, "layout conversion: shape out of range");
    const size_t plane = (size_t)H * W, positions = (size_t)N * plane;
    size_t blocks = (positions + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    nchw_to_nhwc_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)x, (uint16_t*)y, C, C8, plane, positions);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "layout conversion launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

}  // namespace x3
