// Generic direct convolution (SIMT, fp32 accumulation) and the weight-packing kernels.
//
// The direct kernel is the library's total fallback: it handles every descriptor the ABI accepts
// (2D/3D, either layout, f16/bf16, stride 1/2, any channel count, the unpatchify store). One
// thread computes one output value with the summation of musetalk-bench
// patches/taesd_conv.cuh.new, taesd_conv3x3_impl (accumulator starts at the bias, loops over
// input channel and the 3x3 window with zero padding, ReLU, round-to-nearest store), widened to
// the causal 3x3x3 window of FastVideo wan22_vae_decode/solution/head.cu (two carried frames
// before the current ones, clamp to [-1,1] for the head).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace x3 {

struct DirectArgs {
    int dims, N, C_in, C_out, D, H, W, H_out, W_out, stride, act, unpatch, channels_last, has_carry;
    int row_shift;  // banded mode: the input's first row is the band's upper halo row
};

__device__ __forceinline__ float ld_val(const __half* p, size_t i) { return __half2float(p[i]); }
__device__ __forceinline__ float ld_val(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_val(__half* p, size_t i, float v) { p[i] = __float2half_rn(v); }
__device__ __forceinline__ void st_val(__nv_bfloat16* p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(256) direct_conv_kernel(const T* __restrict__ x, const T* __restrict__ carry,
                                                          const T* __restrict__ w, const T* __restrict__ bias,
                                                          T* __restrict__ y, DirectArgs a) {
    const int KT = a.dims == 3 ? 3 : 1;
    const int Dout = a.dims == 3 ? a.D : 1;
    const size_t total = (size_t)a.N * a.C_out * Dout * a.H_out * a.W_out;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        int n, co, t, oh, ow;
        size_t r = idx;
        if (a.channels_last) {
            co = (int)(r % a.C_out); r /= a.C_out;
            ow = (int)(r % a.W_out); r /= a.W_out;
            oh = (int)(r % a.H_out); r /= a.H_out;
            t = (int)(r % Dout); r /= Dout;
            n = (int)r;
        } else {
            ow = (int)(r % a.W_out); r /= a.W_out;
            oh = (int)(r % a.H_out); r /= a.H_out;
            t = (int)(r % Dout); r /= Dout;
            co = (int)(r % a.C_out); r /= a.C_out;
            n = (int)r;
        }
        float acc = bias ? ld_val(bias, co) : 0.0f;
        for (int ci = 0; ci < a.C_in; ++ci) {
            for (int kt = 0; kt < KT; ++kt) {
                // frame kt of the window: 3D reads [carry0, carry1, x0..] at t+kt; 2D reads x itself
                const T* src;
                int F, f;
                if (a.dims == 3) {
                    const int fr = t + kt;
                    if (fr < 2) {
                        if (!a.has_carry) continue;
                        src = carry; F = 2; f = fr;
                    } else {
                        src = x; F = a.D; f = fr - 2;
                    }
                } else {
                    src = x; F = 1; f = 0;
                }
                for (int kh = 0; kh < 3; ++kh) {
                    const int ih = a.stride * oh + kh - 1 + a.row_shift;
                    if (ih < 0 || ih >= a.H) continue;
                    for (int kw = 0; kw < 3; ++kw) {
                        const int iw = a.stride * ow + kw - 1;
                        if (iw < 0 || iw >= a.W) continue;
                        size_t xi;
                        if (a.channels_last)
                            xi = ((((size_t)n * F + f) * a.H + ih) * a.W + iw) * a.C_in + ci;
                        else
                            xi = (((size_t)n * a.C_in + ci) * F + f) * (size_t)a.H * a.W + (size_t)ih * a.W + iw;
                        const size_t wi = (((size_t)co * a.C_in + ci) * KT + kt) * 9 + kh * 3 + kw;
                        acc += ld_val(w, wi) * ld_val(src, xi);
                    }
                }
            }
        }
        if (a.act == X3_ACT_RELU) acc = acc < 0.0f ? 0.0f : acc;
        else if (a.act == X3_ACT_CLAMP1) acc = fminf(1.0f, fmaxf(-1.0f, acc));
        size_t yi;
        if (a.unpatch) {
            const int rgb = co / 4, dy = (co / 2) % 2, dx = co % 2;
            const size_t H2 = 2 * (size_t)a.H_out, W2 = 2 * (size_t)a.W_out;
            const size_t hh = 2 * (size_t)oh + dy, ww = 2 * (size_t)ow + dx;
            if (a.channels_last)
                yi = ((((size_t)n * Dout + t) * H2 + hh) * W2 + ww) * 3 + rgb;
            else
                yi = ((((size_t)n * 3 + rgb) * Dout + t) * H2 + hh) * W2 + ww;
        } else if (a.channels_last) {
            yi = ((((size_t)n * Dout + t) * a.H_out + oh) * a.W_out + ow) * a.C_out + co;
        } else {
            yi = ((((size_t)n * a.C_out + co) * Dout + t) * a.H_out + oh) * (size_t)a.W_out + ow;
        }
        st_val(y, yi, acc);
    }
}

x3_status launch_direct(const x3_conv_plan* p, const void* x, const void* carry, const void* w_packed,
                        const void* bias, void* y, cudaStream_t s) {
    const x3_conv_desc& d = p->d;
    DirectArgs a;
    a.dims = d.dims; a.N = d.N; a.C_in = d.C_in; a.C_out = d.C_out; a.D = d.D; a.H = d.H; a.W = d.W;
    a.H_out = p->H_out; a.W_out = p->W_out; a.stride = d.stride; a.act = d.act; a.unpatch = d.unpatchify2x2;
    a.channels_last = (d.layout == X3_NHWC || d.layout == X3_NDHWC);
    a.has_carry = carry != nullptr;
    a.row_shift = p->row_shift;
    const size_t total = out_elems(p);
    const int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    const size_t cap = (size_t)p->num_sms * 64;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (d.dtype == X3_F16)
        direct_conv_kernel<__half><<<(unsigned)blocks, threads, 0, s>>>((const __half*)x, (const __half*)carry,
                                                                        (const __half*)w_packed, (const __half*)bias,
                                                                        (__half*)y, a);
    else
        direct_conv_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, s>>>(
            (const __nv_bfloat16*)x, (const __nv_bfloat16*)carry, (const __nv_bfloat16*)w_packed,
            (const __nv_bfloat16*)bias, (__nv_bfloat16*)y, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "direct kernel launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

// ------------------------------------------------------------------ weight packing

// Packed layout of the implicit-GEMM weights: blocks ordered [n-tile][kt][chunk][kh*3+kw]; one
// block is the K-major no-swizzle canonical tile of BN output channels x CK input channels:
// [CK/8 planes][BN rows][8 consecutive input channels]. Channels past C_out / C_in are zero.
struct PackArgs {
    int C_in, C_out, KT, BN, CK, n_chunks, n_tiles;
};

__global__ void __launch_bounds__(256) pack_igemm_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ out,
                                                         PackArgs a, size_t total) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        size_t r = i;
        const int e = (int)(r % 8); r /= 8;
        const int nrow = (int)(r % a.BN); r /= a.BN;
        const int j = (int)(r % (a.CK / 8)); r /= (a.CK / 8);
        const int tap = (int)(r % 9); r /= 9;
        const int cc = (int)(r % a.n_chunks); r /= a.n_chunks;
        const int kt = (int)(r % a.KT); r /= a.KT;
        const int nt = (int)r;
        const int co = nt * a.BN + nrow;
        const int ci = cc * a.CK + j * 8 + e;
        uint16_t v = 0;
        if (co < a.C_out && ci < a.C_in) v = w[(((size_t)co * a.C_in + ci) * a.KT + kt) * 9 + tap];
        out[i] = v;
    }
}

// Packed layout of the TN form of the channels-last engine (positions as M, horizontal taps in N):
// blocks ordered [kt][chunk][kh], each the K-major canonical B tile of N = 3 * cp rows x 64 input
// channels, [8 planes][N rows][8 channels], where row kw * cp + co carries tap (kt, kh, kw) of output
// channel co (zero for co >= C_out and for input channels >= C_in).
__global__ void __launch_bounds__(256) pack_tn_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ out,
                                                      int C_in, int C_out, int KT, int n_chunks, int cp, size_t total) {
    const int N = 3 * cp;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        size_t r = i;
        const int e = (int)(r % 8); r /= 8;
        const int row = (int)(r % N); r /= N;
        const int j = (int)(r % 8); r /= 8;
        const int kh = (int)(r % 3); r /= 3;
        const int cc = (int)(r % n_chunks); r /= n_chunks;
        const int kt = (int)r;
        const int kw = row / cp, co = row - kw * cp;
        const int ci = cc * 64 + j * 8 + e;
        uint16_t v = 0;
        if (co < C_out && ci < C_in) v = w[(((size_t)co * C_in + ci) * KT + kt) * 9 + kh * 3 + kw];
        out[i] = v;
    }
}

// Packed layout of the TK form (8 input channels, two taps per K step): five blocks (K steps), each the
// K-major canonical B tile [2 halves][cp rows][8 channels], half h of block s carrying tap 2s + h (zero for
// the tenth tap, for co >= C_out and for channels >= C_in).
__global__ void __launch_bounds__(256) pack_tk_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ out,
                                                      int C_in, int C_out, int cp, size_t total) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        size_t r = i;
        const int ci = (int)(r % 8); r /= 8;
        const int co = (int)(r % cp); r /= cp;
        const int h = (int)(r % 2); r /= 2;
        const int tap = 2 * (int)r + h;
        uint16_t v = 0;
        if (tap < 9 && co < C_out && ci < C_in) v = w[((size_t)co * C_in + ci) * 9 + tap];
        out[i] = v;
    }
}

static x3_status launch_pack_tn(const x3_conv_plan* p, const ClGeom& g, const void* w, void* out, cudaStream_t s) {
    const size_t total = cl_packed_bytes(g) / 2;
    if (g.tk) {
        pack_tk_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>((const uint16_t*)w, (uint16_t*)out, p->d.C_in,
                                                                       p->d.C_out, g.tn_cp, total);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "pack kernel launch: %s", cudaGetErrorString(e));
        return X3_OK;
    }
    size_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    pack_tn_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)w, (uint16_t*)out, p->d.C_in, p->d.C_out, g.KT,
                                                   g.n_chunks, g.tn_cp, total);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "pack kernel launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

// Packed layout of the head form of the channels-last engine: blocks ordered [kt][chunk][kh], each
// the K-major canonical A tile of 128 rows x 64 input channels, [8 planes][128 rows][8 channels],
// where row 32*g + kw*10 + r carries tap (kt, kh, kw) of output channel 10*g + r (zero elsewhere).
__global__ void __launch_bounds__(256) pack_kwm_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ out,
                                                       int C_in, int C_out, int KT, int n_chunks, size_t total) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        size_t r = i;
        const int e = (int)(r % 8); r /= 8;
        const int row = (int)(r % 128); r /= 128;
        const int j = (int)(r % 8); r /= 8;
        const int kh = (int)(r % 3); r /= 3;
        const int cc = (int)(r % n_chunks); r /= n_chunks;
        const int kt = (int)r;
        const int g = row / 32, within = row % 32;
        const int kw = within / 10, co = g * 10 + within % 10;
        const int ci = cc * 64 + j * 8 + e;
        uint16_t v = 0;
        if (within < 30 && co < C_out && ci < C_in) v = w[(((size_t)co * C_in + ci) * KT + kt) * 9 + kh * 3 + kw];
        out[i] = v;
    }
}

// Packed weights of the temporal pass of the two-pass head: blocks ordered [kt][chunk], each the
// canonical A tile [8 planes][128 rows][8 channels] where row (i*3+j)*12 + c (< 108) carries
// w[c][ci][kt][i][j] and rows 108..127 are zero.
__global__ void __launch_bounds__(256) pack_ctr_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ out,
                                                       int C_in, int n_chunks, size_t total) {
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        size_t r = idx;
        const int e = (int)(r % 8); r /= 8;
        const int row = (int)(r % 128); r /= 128;
        const int j8 = (int)(r % 8); r /= 8;
        const int cc = (int)(r % n_chunks); r /= n_chunks;
        const int kt = (int)r;
        const int ci = cc * 64 + j8 * 8 + e;
        uint16_t v = 0;
        if (row < 108 && ci < C_in) {
            const int i = row / 36, j = (row / 12) % 3, c = row % 12;
            v = w[(((size_t)c * C_in + ci) * 3 + kt) * 9 + i * 3 + j];
        }
        out[idx] = v;
    }
}

// Packed weights of the stencil head: blocks ordered [kt][chunk] like the centre-tap form, but row
// 32q + 9*cl + (i*3+j) (the last 5 rows of each 32-row quarter zero) carries w[c][ci][kt][i][j] for
// channel c = 3q + cl, so that each epilogue warp holds all nine taps of its three channels.
__global__ void __launch_bounds__(256) pack_stn_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ out,
                                                       int C_in, int n_chunks, size_t total) {
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        size_t r = idx;
        const int e = (int)(r % 8); r /= 8;
        const int row = (int)(r % 128); r /= 128;
        const int j8 = (int)(r % 8); r /= 8;
        const int cc = (int)(r % n_chunks); r /= n_chunks;
        const int kt = (int)r;
        const int ci = cc * 64 + j8 * 8 + e;
        const int q = row / 32, rr = row % 32;
        uint16_t v = 0;
        if (rr < 27 && ci < C_in) {
            const int c = 3 * q + rr / 9, tap = rr % 9;
            v = w[(((size_t)c * C_in + ci) * 3 + kt) * 9 + tap];
        }
        out[idx] = v;
    }
}

// The nine spatial taps of the two-pass head, one thread per output position: bias-initialised fp32
// accumulators for the 12 channels, the 12 values of tap plane i*3+j at each neighbour inside the
// image added in (i, j) order, clamp to [-1,1], one rounding to bf16, written as the 2x2-unpatchified
// RGB pixels (channel c = rgb*4 + dy*2 + dx goes to pixel (2h+dy, 2w+dx)), channels-last. Consecutive
// threads read consecutive positions of a plane, so every tap's loads are contiguous across a warp.
__device__ __forceinline__ void head_add12(float (&acc)[12], const float* p) {
    const float4* v = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        const float4 f = __ldg(v + q);
        acc[4 * q + 0] += f.x; acc[4 * q + 1] += f.y; acc[4 * q + 2] += f.z; acc[4 * q + 3] += f.w;
    }
}
__device__ __forceinline__ void head_add12(float (&acc)[12], const uint16_t* p) {
    const uint2* v = reinterpret_cast<const uint2*>(p);
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        const uint2 u = __ldg(v + q);
        acc[4 * q + 0] += __uint_as_float(u.x << 16);
        acc[4 * q + 1] += __uint_as_float(u.x & 0xffff0000u);
        acc[4 * q + 2] += __uint_as_float(u.y << 16);
        acc[4 * q + 3] += __uint_as_float(u.y & 0xffff0000u);
    }
}

template <typename T>
__global__ void __launch_bounds__(256) head_stencil_kernel(const T* __restrict__ g, const uint16_t* __restrict__ bias,
                                                           uint16_t* __restrict__ rgb, int frames, int H, int W) {
    const size_t hw = (size_t)H * W;
    const size_t total = (size_t)frames * hw;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int w = (int)(idx % W);
        const size_t fh = idx / W;
        const int h = (int)(fh % H);
        const size_t f = fh / H;
        float acc[12];
#pragma unroll
        for (int c = 0; c < 12; ++c) acc[c] = bias ? __bfloat162float(__ushort_as_bfloat16(__ldg(bias + c))) : 0.0f;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int hh = h + i - 1;
            if (hh < 0 || hh >= H) continue;
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int ww = w + j - 1;
                if (ww < 0 || ww >= W) continue;
                head_add12(acc, g + ((f * 9 + (size_t)(i * 3 + j)) * hw + (size_t)hh * W + ww) * 12);
            }
        }
        uint16_t o[12];
#pragma unroll
        for (int c = 0; c < 12; ++c) {
            const __nv_bfloat16 r = __float2bfloat16_rn(fminf(1.0f, fmaxf(-1.0f, acc[c])));
            o[c] = *reinterpret_cast<const uint16_t*>(&r);
        }
        const size_t W2 = 2 * (size_t)W;
#pragma unroll
        for (int dy = 0; dy < 2; ++dy) {
            uint32_t* row = reinterpret_cast<uint32_t*>(rgb + ((f * 2 * H + 2 * (size_t)h + dy) * W2 + 2 * (size_t)w) * 3);
            // pixels dx = 0, 1 x rgb: channel rgb*4 + dy*2 + dx
            const uint16_t px[6] = {o[dy * 2], o[4 + dy * 2], o[8 + dy * 2], o[dy * 2 + 1], o[4 + dy * 2 + 1], o[8 + dy * 2 + 1]};
            row[0] = (uint32_t)px[0] | ((uint32_t)px[1] << 16);
            row[1] = (uint32_t)px[2] | ((uint32_t)px[3] << 16);
            row[2] = (uint32_t)px[4] | ((uint32_t)px[5] << 16);
        }
    }
}

x3_status launch_head_stencil(const x3_conv_plan* p, const void* g, const void* bias, void* y, cudaStream_t s) {
    const int frames = p->d.N * p->d.D;
    const size_t total = (size_t)frames * p->d.H * p->d.W;
    size_t blocks = (total + 255) / 256;
    const size_t cap = (size_t)p->num_sms * 16;
    if (blocks > cap) blocks = cap;
    if (p->d.kernel == X3_KERNEL_HEAD_SPLIT)
        head_stencil_kernel<float><<<(unsigned)blocks, 256, 0, s>>>((const float*)g, (const uint16_t*)bias,
                                                                   (uint16_t*)y, frames, p->d.H, p->d.W);
    else
        head_stencil_kernel<uint16_t><<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)g, (const uint16_t*)bias,
                                                                      (uint16_t*)y, frames, p->d.H, p->d.W);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "head stencil launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

static x3_status pack_primary(const x3_conv_plan* p, const void* w, void* w_packed, cudaStream_t s);

x3_status launch_pack_weights(const x3_conv_plan* p, const void* w, void* w_packed, cudaStream_t s) {
    x3_status st = pack_primary(p, w, w_packed, s);
    if (st != X3_OK || !p->has_shadow || p->shadow_w_off == 0) return st;
    // the channels-last form's weight blocks (128, or 64 in the M = 64 form, output channels x 64
    // input channels per tap)
    const ClGeom& g = p->cl_shadow;
    if (g.tn) return launch_pack_tn(p, g, w, (uint8_t*)w_packed + p->shadow_w_off, s);
    const int rows = g.m64 ? 64 : 128;
    PackArgs a{p->d.C_in, p->d.C_out, 1, rows, 64, g.n_chunks, g.n_tiles};
    const size_t total = (size_t)g.n_tiles * g.n_chunks * 9 * rows * 64;
    size_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    pack_igemm_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)w,
                                                      (uint16_t*)((uint8_t*)w_packed + p->shadow_w_off), a, total);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "pack kernel launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

static x3_status pack_primary(const x3_conv_plan* p, const void* w, void* w_packed, cudaStream_t s) {
    if (p->kind == K_HEAD_TWO_PASS) {
        const size_t total = p->packed_bytes / 2;
        size_t blocks = (total + 255) / 256;
        if (blocks > 4096) blocks = 4096;
        pack_ctr_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)w, (uint16_t*)w_packed, p->d.C_in,
                                                        p->cl.n_chunks, total);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "pack kernel launch: %s", cudaGetErrorString(e));
        return X3_OK;
    }
    if (p->kind == K_IGEMM_CL && p->cl.tn) return launch_pack_tn(p, p->cl, w, w_packed, s);
    if (p->kind == K_IGEMM_CL && p->cl.stn) {
        const size_t total = p->packed_bytes / 2;
        size_t blocks = (total + 255) / 256;
        if (blocks > 4096) blocks = 4096;
        pack_stn_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)w, (uint16_t*)w_packed, p->d.C_in,
                                                        p->cl.n_chunks, total);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "pack kernel launch: %s", cudaGetErrorString(e));
        return X3_OK;
    }
    if (p->kind == K_IGEMM_CL && p->cl.kwm) {
        const size_t total = p->packed_bytes / 2;
        size_t blocks = (total + 255) / 256;
        if (blocks > 4096) blocks = 4096;
        pack_kwm_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)w, (uint16_t*)w_packed, p->d.C_in,
                                                        p->d.C_out, p->cl.KT, p->cl.n_chunks, total);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "pack kernel launch: %s", cudaGetErrorString(e));
        return X3_OK;
    }
    if (p->kind == K_DIRECT) {
        const size_t bytes = (size_t)p->d.C_out * p->d.C_in * (p->d.dims == 3 ? 27 : 9) * 2;
        cudaError_t e = cudaMemcpyAsync(w_packed, w, bytes, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "weight copy: %s", cudaGetErrorString(e));
        return X3_OK;
    }
    const IgemmGeom& g = p->g;
    PackArgs a{p->d.C_in, p->d.C_out, g.KT, g.BN, g.CK, g.n_chunks, g.n_tiles};
    const size_t total = (size_t)g.n_tiles * g.KT * g.n_chunks * 9 * g.BN * g.CK;
    size_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    pack_igemm_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)w, (uint16_t*)w_packed, a, total);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "pack kernel launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

}  // namespace x3
