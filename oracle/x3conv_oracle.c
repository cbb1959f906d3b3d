/*
 * x3conv oracle: a plain, slow, CPU reference of the 3x3 / causal 3x3x3 convolution hot path.
 *
 * TEST INFRASTRUCTURE. Only the test suite, __graft_entry__.smoke() and bench.py's CPU-baseline
 * and reference legs may build, load or call this file. The product (the CUDA library and its
 * Python binding) never links or imports it, and shares no code, header, table or helper with it.
 *
 * Everything here is the plain definition, written out as nested loops with one fp32 accumulator
 * per output. Sources of each definition:
 *
 *  - 2D pad-1 3x3 convolution, stride 1 or 2, NCHW, fp32 accumulation, bias as the accumulator's
 *    initial value, optional ReLU, one rounding at the store:
 *      musetalk-bench, patches/taesd_conv.cuh.new, header comment ("NCHW in/out, f16 storage with
 *      f32 accumulation. 3x3 kernel, pad 1, stride 1 or 2") and taesd_conv3x3_impl (receptive
 *      field origin stride*out - 1, zero outside the image, the c / ky / kx accumulation loop,
 *      bias-initialised accumulator, ReLU, __float2half store). The operation is a
 *      cross-correlation: weight tap (ky,kx) multiplies input (s*oh+ky-1, s*ow+kx-1).
 *  - causal 3x3x3 convolution over a frame window t..t+2 of [two carried frames, current frames],
 *    spatial zero padding, all 27 taps in one fp32 accumulator, clamp to [-1,1] for the head:
 *      FastVideo, fastvideo-kernel/wan22_vae_decode/solution/head.cu, header comment (the
 *      reference accumulates all 27 taps in one fp32 accumulator; bf16 storage with fp32
 *      accumulation; 4 latent frames per pass with a carry) and head_stencil_kernel
 *      (accumulators initialised to the bias, zero padding in the plane and across the row,
 *      clamp to [-1,1] with fminf/fmaxf, one round-to-nearest store).
 *  - f32 -> f16 / bf16 conversion: IEEE 754-2008 roundTiesToEven, written from the definition
 *    (binary16: 1 sign, 5 exponent bits with bias 15, 10 fraction bits; bfloat16: the top 16 bits
 *    of binary32).
 *
 * Readings where the pages are silent: the first pass's carried frames are zeros (the same
 * zero padding conv3d applies in the plane); the 12 head channels map to RGB by c = rgb*4+dy*2+dx.
 */
#include <math.h>
#include <stdlib.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_CLAMP1 = 2 };

static float apply_act(float v, int act)
{
    if (act == ORACLE_ACT_RELU) return v < 0.0f ? 0.0f : v;
    if (act == ORACLE_ACT_CLAMP1) return fminf(1.0f, fmaxf(-1.0f, v));
    return v;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads the next parallel region will use. */
int oracle_max_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* ---------------------------------------------------------------- IEEE 754 conversions */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* binary32 -> binary16, roundTiesToEven. */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t u = f32_bits(f);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);            /* NaN -> quiet NaN */
    /* 65520 = 65504 + half an ulp: from there on the nearest even neighbour is 2^16 -> inf */
    if (a >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);
    uint32_t e = a >> 23;                                               /* biased f32 exponent */
    if (e >= 113u) {                                                    /* |f| >= 2^-14: normal */
        uint32_t r = a - (112u << 23);                                  /* rebias 127 -> 15 */
        uint32_t keep = r >> 13, rem = r & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (keep & 1u))) keep += 1u;
        return (uint16_t)(sign | keep);
    }
    /* subnormal or zero: value in units of 2^-24 is M * 2^(e-126), M the 24-bit significand */
    if (e < 90u) return (uint16_t)sign;                                 /* far below 2^-25 */
    uint32_t M = (a & 0x7fffffu) | 0x800000u;
    uint32_t shift = 126u - e;                                          /* 14 .. 36 */
    if (shift >= 32u) return (uint16_t)sign;
    uint32_t keep = M >> shift;
    uint32_t rem = M & ((1u << shift) - 1u), half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (keep & 1u))) keep += 1u;
    return (uint16_t)(sign | keep);                                     /* 1024 is the first normal */
}

float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t e = ((uint32_t)h >> 10) & 0x1fu, m = (uint32_t)h & 0x3ffu;
    float mag;
    if (e == 0u) mag = ldexpf((float)m, -24);
    else if (e == 31u) mag = m ? NAN : INFINITY;
    else mag = ldexpf((float)(m | 0x400u), (int)e - 25);
    return bits_f32(f32_bits(mag) | sign);
}

/* binary32 -> bfloat16, roundTiesToEven on the low 16 bits. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t keep = u >> 16, rem = u & 0xffffu;
    if (rem > 0x8000u || (rem == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

float oracle_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Round each value to the storage type (0 = f16, 1 = bf16) and return the rounded value as f32. */
void oracle_round_to(const float* in, float* out, size_t n, int dtype, uint16_t* bits_out)
{
    for (size_t i = 0; i < n; ++i) {
        uint16_t h = dtype == 0 ? oracle_f32_to_f16(in[i]) : oracle_f32_to_bf16(in[i]);
        if (bits_out) bits_out[i] = h;
        out[i] = dtype == 0 ? oracle_f16_to_f32(h) : oracle_bf16_to_f32(h);
    }
}

/* ---------------------------------------------------------------- 2D convolution */

/*
 * y[n,co,oh,ow] = act( b[co] + sum_{ci,kh,kw} w[co,ci,kh,kw] * x[n,ci, s*oh+kh-1, s*ow+kw-1] )
 * x: [N][C_in][H][W]; w: [C_out][C_in][3][3]; b: [C_out] or NULL (zero);
 * y: [N][C_out][H_out][W_out], H_out = (H-1)/s + 1, W_out = (W-1)/s + 1. x is zero outside the
 * image. Returns 0, or -1 on a bad argument.
 */
int oracle_conv2d(const float* x, const float* w, const float* b, float* y,
                  int N, int C_in, int C_out, int H, int W, int stride, int act, int nthreads)
{
    if (N < 0 || C_in <= 0 || C_out <= 0 || H <= 0 || W <= 0 || (stride != 1 && stride != 2)) return -1;
    const int H_out = (H - 1) / stride + 1, W_out = (W - 1) / stride + 1;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < N; ++n)
        for (int co = 0; co < C_out; ++co)
            for (int oh = 0; oh < H_out; ++oh)
                for (int ow = 0; ow < W_out; ++ow) {
                    float acc = b ? b[co] : 0.0f;
                    for (int ci = 0; ci < C_in; ++ci)
                        for (int kh = 0; kh < 3; ++kh) {
                            const int ih = stride * oh + kh - 1;
                            if (ih < 0 || ih >= H) continue;
                            for (int kw = 0; kw < 3; ++kw) {
                                const int iw = stride * ow + kw - 1;
                                if (iw < 0 || iw >= W) continue;
                                acc += w[(((size_t)co * C_in + ci) * 3 + kh) * 3 + kw] *
                                       x[(((size_t)n * C_in + ci) * H + ih) * W + iw];
                            }
                        }
                    y[(((size_t)n * C_out + co) * H_out + oh) * W_out + ow] = apply_act(acc, act);
                }
    return 0;
}

/* ---------------------------------------------------------------- causal 3D convolution */

/*
 * The frame sequence is xt = [carry[0], carry[1], x[0], ..., x[D-1]] (carry NULL = two zero
 * frames) and, for t in [0, D):
 * y[n,co,t,h,w] = act( b[co] + sum_{ci,kt,kh,kw} w[co,ci,kt,kh,kw] * xt[n,ci,t+kt,h+kh-1,w+kw-1] )
 * with spatial zero padding and no temporal padding besides the carry.
 * x: [N][C_in][D][H][W]; carry: [N][C_in][2][H][W] or NULL; w: [C_out][C_in][3][3][3];
 * b: [C_out] or NULL; y: [N][C_out][D][H][W]. Returns 0, or -1 on a bad argument.
 */
int oracle_conv3d_causal(const float* x, const float* carry, const float* w, const float* b, float* y,
                         int N, int C_in, int C_out, int D, int H, int W, int act, int nthreads)
{
    if (N < 0 || C_in <= 0 || C_out <= 0 || D <= 0 || H <= 0 || W <= 0) return -1;
    const size_t plane = (size_t)H * W;
    set_threads(nthreads);
#pragma omp parallel for collapse(3) schedule(dynamic)
    for (int n = 0; n < N; ++n)
        for (int co = 0; co < C_out; ++co)
            for (int t = 0; t < D; ++t)
                for (int h = 0; h < H; ++h)
                    for (int wo = 0; wo < W; ++wo) {
                        float acc = b ? b[co] : 0.0f;
                        for (int ci = 0; ci < C_in; ++ci)
                            for (int kt = 0; kt < 3; ++kt) {
                                const int f = t + kt;            /* frame of xt */
                                const float* src;
                                if (f < 2) {
                                    if (!carry) continue;        /* zero carried frames */
                                    src = carry + (((size_t)n * C_in + ci) * 2 + f) * plane;
                                } else {
                                    src = x + (((size_t)n * C_in + ci) * D + (f - 2)) * plane;
                                }
                                for (int kh = 0; kh < 3; ++kh) {
                                    const int ih = h + kh - 1;
                                    if (ih < 0 || ih >= H) continue;
                                    for (int kw = 0; kw < 3; ++kw) {
                                        const int iw = wo + kw - 1;
                                        if (iw < 0 || iw >= W) continue;
                                        acc += w[((((size_t)co * C_in + ci) * 3 + kt) * 3 + kh) * 3 + kw] *
                                               src[(size_t)ih * W + iw];
                                    }
                                }
                            }
                        y[((((size_t)n * C_out + co) * D + t) * H + h) * W + wo] = apply_act(acc, act);
                    }
    return 0;
}

/* ---------------------------------------------------------------- 2x2 unpatchify */

/*
 * rgb[n,c,t,2h+dy,2w+dx] = y12[n, c*4 + dy*2 + dx, t, h, w] for c in 0..2, dy, dx in 0..1.
 * y12: [N][12][D][H][W]; rgb: [N][3][D][2H][2W]. The channel order is a reading: the pages only
 * say that a 12-channel plane is handed to the video writer.
 */
void oracle_unpatchify2x2(const float* y12, float* rgb, int N, int D, int H, int W)
{
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < 3; ++c)
            for (int dy = 0; dy < 2; ++dy)
                for (int dx = 0; dx < 2; ++dx)
                    for (int t = 0; t < D; ++t)
                        for (int h = 0; h < H; ++h)
                            for (int w = 0; w < W; ++w)
                                rgb[((((size_t)n * 3 + c) * D + t) * (2 * H) + 2 * h + dy) * (2 * (size_t)W) + 2 * w + dx] =
                                    y12[((((size_t)n * 12 + c * 4 + dy * 2 + dx) * D + t) * H + h) * W + w];
}

/* ---------------------------------------------------------------- two-pass head (the page's split) */

/*
 * The conv_out head computed in two passes, following the value path the FastVideo
 * wan22_vae_decode/solution/head.cu header comment describes:
 *   pass 1, temporal-only 3x1x1 convolution into the plane g with 9*12 channels:
 *     g[n,t,h,w,(i*3+j)*12+c] = R16( sum_{ci,kt} w[c,ci,kt,i,j] * xt[n,ci,t+kt,h,w] )
 *     (one fp32 accumulator over the 3 temporal taps and all input channels, then one rounding to
 *     bf16 when round_g != 0; kept in fp32 when round_g == 0);
 *   pass 2, the nine spatial taps, as head_stencil_kernel sums them: an fp32 accumulator starting at
 *   the bias, adding g of the neighbour (h+i-1, w+j-1) for i, j = 0..2 in that order, skipping
 *   neighbours outside the plane (the zero padding), then clamp to [-1,1] (the caller rounds once).
 * x: [N][C_in][D][H][W]; carry: [N][C_in][2][H][W] or NULL; w: [12][C_in][3][3][3]; b: [12] or NULL;
 * y: [N][12][D][H][W]. Returns 0, or -1 on a bad argument.
 */
int oracle_head_two_pass(const float* x, const float* carry, const float* w, const float* b, float* y,
                         int N, int C_in, int D, int H, int W, int round_g, int nthreads)
{
    if (N < 0 || C_in <= 0 || D <= 0 || H <= 0 || W <= 0) return -1;
    const size_t plane = (size_t)H * W;
    const size_t gsize = (size_t)N * D * plane * 108;
    float* g = (float*)malloc(gsize * sizeof(float));
    if (!g) return -1;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < N; ++n)
        for (int t = 0; t < D; ++t)
            for (int h = 0; h < H; ++h)
                for (int wo = 0; wo < W; ++wo)
                    for (int k = 0; k < 108; ++k) {
                        const int i = k / 36, j = (k / 12) % 3, c = k % 12;
                        float acc = 0.0f;
                        for (int ci = 0; ci < C_in; ++ci)
                            for (int kt = 0; kt < 3; ++kt) {
                                const int f = t + kt;
                                float v;
                                if (f < 2) {
                                    if (!carry) continue;
                                    v = carry[(((size_t)n * C_in + ci) * 2 + f) * plane + (size_t)h * W + wo];
                                } else {
                                    v = x[(((size_t)n * C_in + ci) * D + (f - 2)) * plane + (size_t)h * W + wo];
                                }
                                acc += w[((((size_t)c * C_in + ci) * 3 + kt) * 3 + i) * 3 + j] * v;
                            }
                        if (round_g) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));
                        g[((((size_t)n * D + t) * H + h) * W + wo) * 108 + k] = acc;
                    }
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < 12; ++c)
            for (int t = 0; t < D; ++t)
                for (int h = 0; h < H; ++h)
                    for (int wo = 0; wo < W; ++wo) {
                        float acc = b ? b[c] : 0.0f;
                        for (int i = 0; i < 3; ++i) {
                            const int hh = h + i - 1;
                            if (hh < 0 || hh >= H) continue;
                            for (int j = 0; j < 3; ++j) {
                                const int ww = wo + j - 1;
                                if (ww < 0 || ww >= W) continue;
                                acc += g[((((size_t)n * D + t) * H + hh) * W + ww) * 108 + (i * 3 + j) * 12 + c];
                            }
                        }
                        y[((((size_t)n * 12 + c) * D + t) * H + h) * W + wo] = apply_act(acc, ORACLE_ACT_CLAMP1);
                    }
    free(g);
    return 0;
}
