// Layout conversion used by the stack driver: a 2D NCHW activation to channels-last, with the
// channel count rounded up to a multiple of 8 (zero channels) so that every position row is a whole
// number of 16-byte units for the channels-last engine's TMA boxes.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "internal.h"

namespace x3 {

namespace {

// One thread per position: the position's C values (one per channel plane; consecutive threads
// read consecutive positions, so each channel's reads are coalesced) are written as C8 contiguous
// channels in 16-byte pieces, zero past C. Position indices fit in 32 bits (checked by the
// launcher), so the image/pixel split is a 32-bit division.
__global__ void __launch_bounds__(256) nchw_to_nhwc_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                                                           int C, int C8, uint32_t plane, uint32_t positions) {
    for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < positions; idx += gridDim.x * blockDim.x) {
        const uint32_t n = idx / plane, pix = idx - n * plane;
        const uint16_t* xs = x + (size_t)n * C * plane + pix;
        uint4* yd = reinterpret_cast<uint4*>(y + (size_t)idx * C8);
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

// The history of a causal channels-last layer after a pass: carry row n (2 frames of `unit` 16-byte
// pieces) becomes the last two frames of the sequence [history, input row n (D frames)]. Launched as
// a programmatic dependent of the layer's kernel, which signals once all of its reads of the old
// history are done, so the copy runs beside the rest of that kernel; every thread then waits for
// that kernel to complete before it exits, which keeps the stream's order for whatever follows.
// Its loads go to L2 only (ld.global.cg): the kernel overlaps others, so no L1 line of an earlier
// pass may serve them.
__global__ void __launch_bounds__(256) carry_update_kernel(const uint4* __restrict__ in, uint4* __restrict__ carry,
                                                           int rows, uint32_t unit, int D, int history_valid) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t per_row = D >= 2 ? 2 * unit : unit;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (int r = 0; r < rows; ++r) {
        uint4* c = carry + (size_t)r * 2 * unit;
        const uint4* x = in + (size_t)r * D * unit;
        if (D >= 2) {
            const uint4* src = x + (size_t)(D - 2) * unit;
            uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
            // four independent 16-byte copies in flight per thread
            for (; e + 3 * stride < per_row; e += 4 * stride) {
                const uint4 v0 = __ldcg(src + e), v1 = __ldcg(src + e + stride), v2 = __ldcg(src + e + 2 * stride),
                            v3 = __ldcg(src + e + 3 * stride);
                c[e] = v0; c[e + stride] = v1; c[e + 2 * stride] = v2; c[e + 3 * stride] = v3;
            }
            for (; e < per_row; e += stride) c[e] = __ldcg(src + e);
        } else {
            // one frame: the older history frame is the previous newer one (or zero), the newer one
            // the input; each thread moves both frames of its own pieces
            for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < per_row; e += stride) {
                const uint4 h = history_valid ? __ldcg(c + unit + e) : make_uint4(0u, 0u, 0u, 0u);
                c[e] = h;
                c[unit + e] = __ldcg(x + e);
            }
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

// Carry update of a channels-last (NDHWC) causal layer by carry_update_kernel, as a programmatic
// dependent of the kernel just enqueued on s (that kernel must signal only after its last read of
// the carry). `frame_bytes` = H*W*C*2, a multiple of 16; `input` and `carry` 16-byte aligned.
x3_status launch_carry_update(const void* input, void* carry, int N, int D, size_t frame_bytes, int history_valid,
                              int num_sms, cudaStream_t s) {
    if (N < 1 || D < 1 || frame_bytes == 0 || frame_bytes % 16 != 0 || frame_bytes / 16 > 0x3FFFFFFFu ||
        ((uintptr_t)input & 15u) || ((uintptr_t)carry & 15u))
        return fail(X3_ERR_INVALID, "carry update: unaligned or empty frames");
    // the same shared-memory carve-out as the convolution kernels, and one CTA per SM: that fits
    // beside a persistent convolution CTA (measured: the stack stage of two 128->128 layers at
    // 4 x 352x624 takes 1.003 ms with the copies, 1.005 without them, 1.044 with cudaMemcpy2DAsync on
    // a side stream; with two copy CTAs per SM the second waits for the convolution and 1.14 ms)
    static const cudaError_t carve = cudaFuncSetAttribute(
        carry_update_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (carve != cudaSuccess) return fail(X3_ERR_CUDA, "carry update carve-out: %s", cudaGetErrorString(carve));
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(num_sms > 0 ? num_sms : 148));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, carry_update_kernel, (const uint4*)input, (uint4*)carry, N,
                                       (uint32_t)(frame_bytes / 16), D, history_valid);
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "carry update launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

x3_status launch_nchw_to_nhwc(const void* x, void* y, int N, int C, int C8, int H, int W, cudaStream_t s) {
    if (N < 1 || C < 1 || C8 < C || C8 % 8 != 0 || H < 1 || W < 1)
        return fail(X3_ERR_UNSUPPORTED, "layout conversion: shape out of range");
    const size_t plane = (size_t)H * W, positions = (size_t)N * plane;
    if (positions + 8192ull * 256ull >= (1ull << 32))
        return fail(X3_ERR_UNSUPPORTED, "layout conversion: more than 2^32 - 2^21 positions");
    size_t blocks = (positions + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    nchw_to_nhwc_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)x, (uint16_t*)y, C, C8, (uint32_t)plane,
                                                          (uint32_t)positions);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "layout conversion launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

}  // namespace x3
