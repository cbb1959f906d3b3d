// tcgen05 / TMEM implicit-GEMM convolution engine for sm_103a.
//
// The convolution of FastVideo wan22_vae_decode/solution/head.cu (causal 3x3x3, bf16 storage,
// fp32 accumulation of all 27 taps, bias, clamp, one rounding at the store) and of musetalk-bench
// patches/taesd_conv.cuh.new (2D pad-1 3x3 over an input halo staged once in shared memory and
// reused by every tap and output channel, bias, ReLU) computed as a GEMM on the tensor cores:
//   M = output positions, N = output channels, K = taps x input channels, D accumulated in TMEM.
//
// Per tile (Rt output rows x Wt output columns of one output frame, BN output channels):
//   * the zero-padded input halo (Rt+2 rows x P = Wt+2 columns) of one temporal tap and CK input
//     channels is staged ONCE in shared memory as K-major no-swizzle planes (16 bytes = 8 channels
//     per position). Every spatial tap (kh, kw) then reads it through an MMA descriptor whose start
//     is offset by (kh*P + kw) positions, so the 9 taps reuse one staged halo;
//   * channels-last inputs are staged by TMA straight into that layout (one box of 8 channels per
//     plane, out-of-image boxes zero-filled by the TMA unit = the pad-1 zero padding; missing
//     carried frames are read at an out-of-range frame coordinate, which also fills zeros);
//   * NCHW inputs are loaded by TMA as a raw [C][rows][cols] tile and transposed into the planes
//     by ldmatrix.trans / stmatrix (the transposer warps), which also applies the one-column shift
//     of the halo;
//   * weights are pre-packed per (tap, channel chunk) into the canonical B tile and copied with a
//     plain bulk copy;
//   * one thread issues tcgen05.mma (M=128, N=BN, K=16) for NSUB subtiles of 128 positions into
//     fp32 TMEM accumulators; tcgen05.commit frees shared-memory stages as soon as the MMAs that
//     read them complete;
//   * four epilogue warps read TMEM (tcgen05.ld), add the bias, apply ReLU / clamp, round once to
//     f16/bf16 and store (channels-last vectors, NCHW rows, or the 2x2 unpatchify to RGB).
// The kernel is persistent (one CTA per SM) and warp-specialised. Every mbarrier wait is bounded
// by a 1 s limit; a wait that runs out records X3_ERR_TIMEOUT in the device status word, makes
// the other roles give up, drains outstanding copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace x3 {

__device__ unsigned int g_x3_status;  // bit 0: a bounded wait ran out

enum OutKind { OUT_CL = 0, OUT_NCHW = 1, OUT_UNPATCH_CL = 2 };

constexpr int kSmemLimit = 232448;     // 227 KB of dynamic shared memory per CTA
constexpr int kSmemFloor = 120 * 1024; // ask for at least this much: one CTA (and one TMEM owner) per SM
constexpr uint64_t kWaitNs = 1000000000ull;

struct IgemmArgs {
    int C_in, C_out, N, D, H, W, H_out, W_out, dout;
    int act, out_kind, has_carry;
    int BN, n_tiles, CK, n_chunks, KT, NSUB, Rt, Wt, P, spr, halo_rows, plane_stride, a_bytes, a_tx_bytes;
    int raw_w, raw_bytes, raw_tx_bytes, b_bytes, n_a, n_b, n_raw, acc_bufs, tmem_cols;
    int stride, raw_rows, phase_stride;  // NCHW: input stride, raw tile rows, bytes between phase planes
    int row_shift;  // banded mode: the input's first row is the band's upper halo row
    int col_tiles, row_tiles, frames;
    int scr_pitch;  // epilogue scratch row pitch in bytes (0 = direct stores)
    long long tiles;
    uint32_t idesc;
    const uint8_t* w;
    const void* bias;
    void* y;
};

struct TileCoord {
    int nt, ow0, oh0, fr;
};

__device__ __forceinline__ TileCoord decode_tile(const IgemmArgs& a, long long t) {
    TileCoord c;
    c.nt = (int)(t % a.n_tiles);
    t /= a.n_tiles;
    c.ow0 = (int)(t % a.col_tiles) * a.Wt;
    t /= a.col_tiles;
    c.oh0 = (int)(t % a.row_tiles) * a.Rt;
    t /= a.row_tiles;
    c.fr = (int)t;
    return c;
}

// Raster offset (in positions) of subtile s within the tile's output raster of pitch P.
__device__ __forceinline__ int sub_off(const IgemmArgs& a, int s) {
    return a.spr ? (s / a.spr) * a.P + (s % a.spr) * 128 : s * 128;
}

// Bounded wait. Returns false when the wait ran out or another role gave up.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((++spins & 63u) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > kWaitNs) {
                *abort_flag = 1;
                atomicOr(&g_x3_status, 1u);
                return false;
            }
        }
    }
}

__device__ __forceinline__ float act_apply(float v, int act) {
    if (act == X3_ACT_RELU) return fmaxf(v, 0.0f);
    if (act == X3_ACT_CLAMP1) return fminf(1.0f, fmaxf(-1.0f, v));
    return v;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <bool BF16>
__device__ __forceinline__ uint16_t pack1(float v) {
    if (BF16) {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        return *reinterpret_cast<uint16_t*>(&h);
    } else {
        __half h = __float2half_rn(v);
        return *reinterpret_cast<uint16_t*>(&h);
    }
}

template <bool BF16>
__device__ __forceinline__ float bias_at(const void* bias, int co) {
    if (!bias) return 0.0f;
    const uint16_t raw = __ldg(reinterpret_cast<const unsigned short*>(bias) + co);
    if (BF16) return __uint_as_float((uint32_t)raw << 16);
    return __half2float(__ushort_as_half(raw));
}

// Store 16 accumulator columns [co0, co0+16) of one output position.
template <bool BF16>
__device__ __forceinline__ void store_chunk(const IgemmArgs& a, const uint32_t (&v)[16], const float* bias16, int co0,
                                            int n, int t, int oh, int ow) {
    float f[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = act_apply(__uint_as_float(v[i]) + bias16[i], a.act);
    if (a.out_kind == OUT_CL) {
        uint16_t* y = reinterpret_cast<uint16_t*>(a.y) +
                      ((((size_t)n * a.dout + t) * a.H_out + oh) * a.W_out + ow) * (size_t)a.C_out + co0;
        if (co0 + 16 <= a.C_out && (a.C_out & 7) == 0) {
            uint4 q0, q1;
            q0.x = pack2<BF16>(f[0], f[1]);   q0.y = pack2<BF16>(f[2], f[3]);
            q0.z = pack2<BF16>(f[4], f[5]);   q0.w = pack2<BF16>(f[6], f[7]);
            q1.x = pack2<BF16>(f[8], f[9]);   q1.y = pack2<BF16>(f[10], f[11]);
            q1.z = pack2<BF16>(f[12], f[13]); q1.w = pack2<BF16>(f[14], f[15]);
            reinterpret_cast<uint4*>(y)[0] = q0;
            reinterpret_cast<uint4*>(y)[1] = q1;
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (co0 + i < a.C_out) y[i] = pack1<BF16>(f[i]);
        }
    } else if (a.out_kind == OUT_NCHW) {
        uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
        const size_t plane = (size_t)a.H_out * a.W_out;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (co0 + i < a.C_out)
                y[(((size_t)n * a.C_out + co0 + i) * a.dout + t) * plane + (size_t)oh * a.W_out + ow] = pack1<BF16>(f[i]);
    } else {  // 2x2 unpatchify of 12 channels: c = rgb*4 + dy*2 + dx -> pixel (2oh+dy, 2ow+dx), channels-last RGB
        uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
        const size_t W2 = 2 * (size_t)a.W_out, H2 = 2 * (size_t)a.H_out;
        const size_t base = ((size_t)n * a.dout + t) * H2;
#pragma unroll
        for (int dy = 0; dy < 2; ++dy) {
            uint16_t* row = y + ((base + 2 * (size_t)oh + dy) * W2 + 2 * (size_t)ow) * 3;
            // pixels (dx=0, dx=1) x rgb: 6 consecutive values
            uint16_t px[6];
#pragma unroll
            for (int dx = 0; dx < 2; ++dx)
#pragma unroll
                for (int c = 0; c < 3; ++c) px[dx * 3 + c] = pack1<BF16>(f[c * 4 + dy * 2 + dx]);
            uint32_t* r32 = reinterpret_cast<uint32_t*>(row);  // 12-byte aligned run: 3 words
            r32[0] = (uint32_t)px[0] | ((uint32_t)px[1] << 16);
            r32[1] = (uint32_t)px[2] | ((uint32_t)px[3] << 16);
            r32[2] = (uint32_t)px[4] | ((uint32_t)px[5] << 16);
        }
    }
}

template <int MODE, bool BF16>
__global__ void __launch_bounds__(MODE == STAGE_NCHW ? 320 : 192, 1)
    igemm_conv_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c,
                      const __grid_constant__ IgemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // carve shared memory (base rounded up to 128 bytes)
    const uint32_t raw_base = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_base + 127u) & ~127u;
    uint8_t* sbase = smem_raw + (base - raw_base);
    const uint32_t sA = base;
    const uint32_t sRaw = sA + (uint32_t)(a.n_a * a.a_bytes);
    const uint32_t sB = sRaw + (uint32_t)(a.n_raw * a.raw_bytes);
    const uint32_t sBar = sB + (uint32_t)(a.n_b * a.b_bytes);
    const uint32_t bar_a_full = sBar;
    const uint32_t bar_a_empty = bar_a_full + 8u * a.n_a;
    const uint32_t bar_r_full = bar_a_empty + 8u * a.n_a;
    const uint32_t bar_r_empty = bar_r_full + 8u * a.n_raw;
    const uint32_t bar_b_full = bar_r_empty + 8u * a.n_raw;
    const uint32_t bar_b_empty = bar_b_full + 8u * a.n_b;
    const uint32_t bar_acc_full = bar_b_empty + 8u * a.n_b;
    const uint32_t bar_acc_empty = bar_acc_full + 16u;
    const uint32_t bar_drain = bar_acc_empty + 16u;
    const uint32_t s_tmem = bar_drain + 8u;
    const uint32_t s_abort = s_tmem + 4u;
    const uint32_t s_junk = (s_abort + 4u + 127u) & ~127u;  // NCHW: 16 bytes per transposer lane
    const uint32_t s_bias = s_junk + (MODE == STAGE_NCHW ? 4u * 32u * 16u : 0u);  // 4 warps x BN floats
    const uint32_t s_scr = (s_bias + 16u * (uint32_t)a.BN + 127u) & ~127u;     // 4 warps x 32 rows x scr_pitch
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + (s_abort - base));
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sbase + (s_tmem - base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.n_a; ++i) {
            ptx::mbar_init(bar_a_full + 8 * i, MODE == STAGE_NCHW ? 4 : 1);
            ptx::mbar_init(bar_a_empty + 8 * i, 1);
        }
        for (int i = 0; i < a.n_raw; ++i) {
            ptx::mbar_init(bar_r_full + 8 * i, 1);
            ptx::mbar_init(bar_r_empty + 8 * i, 4);
        }
        for (int i = 0; i < a.n_b; ++i) {
            ptx::mbar_init(bar_b_full + 8 * i, 1);
            ptx::mbar_init(bar_b_empty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar_acc_full + 8 * i, 1);
            ptx::mbar_init(bar_acc_empty + 8 * i, 4);
        }
        ptx::mbar_init(bar_drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_x);
        if (MODE == STAGE_CL) ptx::prefetch_tmap(&tm_c);
    }
    if (warp == 1) {
        ptx::tmem_alloc(s_tmem, (uint32_t)a.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int kpl = a.CK / 8;  // K-major planes per chunk

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t a_cnt = 0, r_cnt = 0, b_cnt = 0;
            bool ok = true;
            for (long long tile = blockIdx.x; tile < a.tiles && ok; tile += gridDim.x) {
                const TileCoord tc = decode_tile(a, tile);
                const int n = tc.fr / a.dout, t = tc.fr % a.dout;
                for (int kt = 0; kt < a.KT && ok; ++kt) {
                    for (int cc = 0; cc < a.n_chunks && ok; ++cc) {
                        if (MODE == STAGE_CL) {
                            const uint32_t st = a_cnt % a.n_a;
                            if (!wait_bar(bar_a_empty + 8 * st, ((a_cnt / a.n_a) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                            ptx::mbar_arrive_expect_tx(bar_a_full + 8 * st, (uint32_t)a.a_tx_bytes);
                            // frame of the window: 3D reads [carry0, carry1, x0, ...] at t + kt
                            const void* map = &tm_x;
                            int fcoord;
                            if (a.KT == 3) {
                                const int f = t + kt;
                                if (f >= 2) fcoord = n * a.D + (f - 2);
                                else if (a.has_carry) { map = &tm_c; fcoord = n * 2 + f; }
                                else fcoord = -1;  // out of range: the TMA unit fills zeros
                            } else {
                                fcoord = n;
                            }
                            for (int j = 0; j < kpl; ++j)
                                ptx::tma_load_4d(sA + st * a.a_bytes + j * a.plane_stride, map, bar_a_full + 8 * st,
                                                 cc * a.CK + 8 * j, tc.ow0 - 1, tc.oh0 - 1 + a.row_shift, fcoord);
                            ++a_cnt;
                        } else {
                            const uint32_t st = r_cnt % a.n_raw;
                            if (!wait_bar(bar_r_empty + 8 * st, ((r_cnt / a.n_raw) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                            ptx::mbar_arrive_expect_tx(bar_r_full + 8 * st, (uint32_t)a.raw_tx_bytes);
                            ptx::tma_load_4d(sRaw + st * a.raw_bytes, &tm_x, bar_r_full + 8 * st,
                                             a.stride * tc.ow0 - 8, a.stride * tc.oh0 - 1 + a.row_shift, cc * a.CK, n);
                            ++r_cnt;
                        }
                        const uint8_t* wblk = a.w + ((((size_t)tc.nt * a.KT + kt) * a.n_chunks + cc) * 9) * a.b_bytes;
                        for (int tap = 0; tap < 9; ++tap) {
                            const uint32_t st = b_cnt % a.n_b;
                            if (!wait_bar(bar_b_empty + 8 * st, ((b_cnt / a.n_b) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                            ptx::mbar_arrive_expect_tx(bar_b_full + 8 * st, (uint32_t)a.b_bytes);
                            ptx::bulk_load(sB + st * a.b_bytes, wblk + (size_t)tap * a.b_bytes, (uint32_t)a.b_bytes,
                                           bar_b_full + 8 * st);
                            ++b_cnt;
                        }
                    }
                }
            }
            if (!ok) {
                // drain: wait (bounded) for the copies this thread issued into each stage
                volatile int dummy = 0;
                for (int i = 0; i < a.n_a && MODE == STAGE_CL; ++i) {
                    const uint32_t cnt = a_cnt;  // stages issued: last issue of stage i
                    if (cnt == 0) break;
                    const uint32_t last = (cnt - 1 - ((cnt - 1 + a.n_a - i) % a.n_a));
                    if (last < cnt && (last % a.n_a) == (uint32_t)i) wait_bar(bar_a_full + 8 * i, (last / a.n_a) & 1u, &dummy);
                }
                for (int i = 0; i < a.n_raw; ++i) {
                    const uint32_t cnt = r_cnt;
                    if (cnt == 0) break;
                    const uint32_t last = (cnt - 1 - ((cnt - 1 + a.n_raw - i) % a.n_raw));
                    if (last < cnt && (last % a.n_raw) == (uint32_t)i) wait_bar(bar_r_full + 8 * i, (last / a.n_raw) & 1u, &dummy);
                }
                for (int i = 0; i < a.n_b; ++i) {
                    const uint32_t cnt = b_cnt;
                    if (cnt == 0) break;
                    const uint32_t last = (cnt - 1 - ((cnt - 1 + a.n_b - i) % a.n_b));
                    if (last < cnt && (last % a.n_b) == (uint32_t)i) wait_bar(bar_b_full + 8 * i, (last / a.n_b) & 1u, &dummy);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (one thread)
        if (lane == 0) {
            uint32_t a_cnt = 0, b_cnt = 0, it = 0;
            bool ok = true;
            // Descriptor words: the high word (SBO = 128 bytes between 8-row core-matrix groups,
            // version 1) never changes; the low word is (start address >> 4) | (LBO >> 4) << 16, so
            // every offset below is added in 16-byte units to the low word only.
            const uint32_t hi = (128u >> 4) | (1u << 14);
            const uint32_t a_lo0 = ((sA >> 4) & 0x3FFFu) | ((uint32_t)(a.plane_stride >> 4) << 16);
            const uint32_t b_lo0 = ((sB >> 4) & 0x3FFFu) | ((uint32_t)((a.BN * 16) >> 4) << 16);
            const uint32_t a_stage16 = (uint32_t)a.a_bytes >> 4, b_stage16 = (uint32_t)a.b_bytes >> 4;
            const uint32_t a_ks16 = (uint32_t)(2 * a.plane_stride) >> 4, b_ks16 = (uint32_t)(2 * a.BN * 16) >> 4;
            const int ksteps = a.CK / 16;
            const int nsub = a.NSUB;
            uint32_t soff[8], dcol[8], toff[9];
            for (int tap = 0; tap < 9; ++tap) {
                const int kh = tap / 3, kw = tap % 3;
                toff[tap] = a.stride == 1
                                ? (uint32_t)(kh * a.P + kw)
                                : (uint32_t)((((kh & 1) * 2 + (kw & 1)) * a.phase_stride) >> 4) +
                                      (uint32_t)((kh >> 1) * a.P + (kw >> 1));
            }
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                soff[s] = s < nsub ? (uint32_t)sub_off(a, s) : 0u;  // raster offset = 16-byte units
                dcol[s] = (uint32_t)(s * a.BN);
            }
            for (long long tile = blockIdx.x; tile < a.tiles && ok; tile += gridDim.x, ++it) {
                const uint32_t ab = it % a.acc_bufs;
                if (!wait_bar(bar_acc_empty + 8 * ab, ((it / a.acc_bufs) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d0 = tmem_base + ab * (uint32_t)(nsub * a.BN);
                uint32_t acc = 0;
                for (int kt = 0; kt < a.KT && ok; ++kt) {
                    for (int cc = 0; cc < a.n_chunks && ok; ++cc) {
                        const uint32_t sa = a_cnt % a.n_a;
                        if (!wait_bar(bar_a_full + 8 * sa, (a_cnt / a.n_a) & 1u, abort_flag)) { ok = false; break; }
                        ptx::tc_fence_after();
                        const uint32_t a_lo_stage = a_lo0 + sa * a_stage16;
                        for (int kh = 0; kh < 3 && ok; ++kh) {
                            for (int kw = 0; kw < 3; ++kw) {
                                const uint32_t sb = b_cnt % a.n_b;
                                if (!wait_bar(bar_b_full + 8 * sb, (b_cnt / a.n_b) & 1u, abort_flag)) { ok = false; break; }
                                ptx::tc_fence_after();
                                const uint32_t b_lo = b_lo0 + sb * b_stage16;
                                const uint32_t a_lo = a_lo_stage + toff[kh * 3 + kw];
#pragma unroll
                                for (int ks = 0; ks < 2; ++ks) {
                                    if (ks < ksteps) {
                                        const uint64_t bdesc = ((uint64_t)hi << 32) | (uint64_t)(b_lo + ks * b_ks16);
                                        const uint32_t a_lo_k = a_lo + ks * a_ks16;
#pragma unroll
                                        for (int s = 0; s < 8; ++s) {
                                            if (s < nsub) {
                                                const uint64_t adesc = ((uint64_t)hi << 32) | (uint64_t)(a_lo_k + soff[s]);
                                                ptx::mma_f16(d0 + dcol[s], adesc, bdesc, a.idesc, acc);
                                            }
                                        }
                                        acc = 1;
                                    }
                                }
                                ptx::mma_commit(bar_b_empty + 8 * sb);
                                ++b_cnt;
                            }
                        }
                        if (!ok) break;
                        ptx::mma_commit(bar_a_empty + 8 * sa);
                        ++a_cnt;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(bar_acc_full + 8 * ab);
            }
            // drain: every MMA issued by this thread has completed before TMEM is released
            ptx::mma_commit(bar_drain);
            volatile int dummy = 0;
            wait_bar(bar_drain, 0, &dummy);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue (TMEM -> global)
        const int quarter = warp & 3;
        const int ew = warp - 2;
        float* s_bias_f = reinterpret_cast<float*>(sbase + (s_bias - base)) + ew * a.BN;
        uint8_t* scr = sbase + (s_scr - base) + (size_t)ew * 32 * a.scr_pitch;
        const bool staged = a.scr_pitch > 0;
        int cur_nt = -1;
        uint32_t it = 0;
        for (long long tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, ++it) {
            const uint32_t ab = it % a.acc_bufs;
            if (!wait_bar(bar_acc_full + 8 * ab, (it / a.acc_bufs) & 1u, abort_flag)) break;
            ptx::tc_fence_after();
            const TileCoord tc = decode_tile(a, tile);
            const int n = tc.fr / a.dout, t = tc.fr % a.dout;
            if (tc.nt != cur_nt) {  // this warp's copy of the N tile's bias (fp32); no cross-warp barrier
                __syncwarp();
                for (int i = lane; i < a.BN; i += 32) {
                    const int co = tc.nt * a.BN + i;
                    s_bias_f[i] = co < a.C_out ? bias_at<BF16>(a.bias, co) : 0.0f;
                }
                __syncwarp();
                cur_nt = tc.nt;
            }
            for (int s = 0; s < a.NSUB; ++s) {
                const int m = sub_off(a, s) + quarter * 32 + lane;
                const int r = m / a.P, c = m % a.P;
                const int oh = tc.oh0 + r, ow = tc.ow0 + c;
                const bool valid = (c < a.Wt) && (r < a.Rt) && (oh < a.H_out) && (ow < a.W_out);
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + ab * (uint32_t)(a.NSUB * a.BN) +
                                       (uint32_t)(s * a.BN);
                if (staged) {
                    // channels-last: this thread's position row (BN values, rounded) goes to the warp's
                    // scratch, then the warp writes whole rows of BN*2 contiguous bytes per position.
                    uint8_t* row = scr + (size_t)lane * a.scr_pitch;
                    for (int ch = 0; ch < a.BN; ch += 32) {
                        uint32_t v[32];
                        ptx::tmem_ld32(taddr + (uint32_t)ch, v);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 w4;
                            const float* bb = s_bias_f + ch + q * 8;
                            w4.x = pack2<BF16>(act_apply(__uint_as_float(v[q * 8 + 0]) + bb[0], a.act),
                                               act_apply(__uint_as_float(v[q * 8 + 1]) + bb[1], a.act));
                            w4.y = pack2<BF16>(act_apply(__uint_as_float(v[q * 8 + 2]) + bb[2], a.act),
                                               act_apply(__uint_as_float(v[q * 8 + 3]) + bb[3], a.act));
                            w4.z = pack2<BF16>(act_apply(__uint_as_float(v[q * 8 + 4]) + bb[4], a.act),
                                               act_apply(__uint_as_float(v[q * 8 + 5]) + bb[5], a.act));
                            w4.w = pack2<BF16>(act_apply(__uint_as_float(v[q * 8 + 6]) + bb[6], a.act),
                                               act_apply(__uint_as_float(v[q * 8 + 7]) + bb[7], a.act));
                            *reinterpret_cast<uint4*>(row + (ch + q * 8) * 2) = w4;
                        }
                    }
                    const unsigned long long my_off =
                        valid ? ((((unsigned long long)n * a.dout + t) * a.H_out + oh) * a.W_out + ow) * (unsigned long long)a.C_out
                              : ~0ull;
                    __syncwarp();
                    const int lpr = a.BN / 8;  // lanes per row: 16 bytes = 8 channels each
                    const int rpi = 32 / lpr;  // rows per store instruction
                    const int seg = lane % lpr;
                    const int co = tc.nt * a.BN + seg * 8;
                    uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
                    for (int r0 = 0; r0 < 32; r0 += rpi) {
                        const int rr = r0 + lane / lpr;
                        const unsigned long long off = __shfl_sync(0xffffffffu, my_off, rr);
                        if (off != ~0ull && co < a.C_out) {
                            const uint4 q = *reinterpret_cast<const uint4*>(scr + (size_t)rr * a.scr_pitch + seg * 16);
                            *reinterpret_cast<uint4*>(y + off + co) = q;
                        }
                    }
                    __syncwarp();
                } else {
                    for (int ch = 0; ch < a.BN; ch += 16) {
                        uint32_t v[16];
                        ptx::tmem_ld16(taddr + (uint32_t)ch, v);
                        ptx::tmem_ld_wait();
                        const int co0 = tc.nt * a.BN + ch;
                        if (valid && co0 < a.C_out) store_chunk<BF16>(a, v, s_bias_f + ch, co0, n, t, oh, ow);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_acc_empty + 8 * ab);
        }
    } else if (MODE == STAGE_NCHW) {
        // ------------------------------------------------------------ transposers (NCHW -> K-major planes)
        const int tw = warp - 6;  // 0..3
        uint32_t a_cnt = 0, r_cnt = 0;
        const int kb_n = a.raw_w / 8;                       // 8-column blocks per raw row
        const int nblk = kpl * a.raw_rows * kb_n;           // 8x8 blocks per stage
        const uint32_t junk = s_junk + (uint32_t)(tw * 32 + lane) * 16u;
        bool ok = true;
        for (long long tile = blockIdx.x; tile < a.tiles && ok; tile += gridDim.x) {
            for (int cc = 0; cc < a.n_chunks; ++cc) {
                const uint32_t sr = r_cnt % a.n_raw;
                const uint32_t sa = a_cnt % a.n_a;
                if (!wait_bar(bar_r_full + 8 * sr, (r_cnt / a.n_raw) & 1u, abort_flag)) { ok = false; break; }
                if (!wait_bar(bar_a_empty + 8 * sa, ((a_cnt / a.n_a) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                const uint32_t raw = sRaw + sr * a.raw_bytes;
                const uint32_t A = sA + sa * a.a_bytes;
                for (int g = tw; g * 4 < nblk; g += 4) {
                    const int blk = g * 4 + (lane >> 3);
                    const int i = lane & 7;
                    uint32_t lds_addr, sts_addr = junk;
                    if (blk < nblk) {
                        const int kb = blk % kb_n;
                        const int rest = blk / kb_n;
                        const int hr = rest % a.raw_rows;
                        const int j = rest / a.raw_rows;
                        // source row i: channel 8j+i, halo row hr, raw columns 8kb..8kb+7
                        lds_addr = raw + (uint32_t)(((8 * j + i) * a.raw_rows + hr) * a.raw_w + 8 * kb) * 2u;
                        // destination row i: raw column 8kb+i = halo position 8kb+i-7 of row hr
                        const int q = 8 * kb + i - 7;
                        if (a.stride == 1) {
                            if (q >= 0 && q < a.P)
                                sts_addr = A + (uint32_t)j * a.plane_stride + (uint32_t)(hr * a.P + q) * 16u;
                        } else if (q >= 0 && q <= 2 * a.Wt) {
                            // stride 2: de-interleave into the (row parity, column parity) phase planes
                            const uint32_t ph = (uint32_t)((hr & 1) * 2 + (q & 1));
                            sts_addr = A + ph * (uint32_t)a.phase_stride + (uint32_t)j * a.plane_stride +
                                       (uint32_t)((hr >> 1) * a.P + (q >> 1)) * 16u;
                        }
                    } else {
                        lds_addr = raw;
                    }
                    uint32_t r0, r1, r2, r3;
                    ptx::ldsm_x4_trans(lds_addr, r0, r1, r2, r3);
                    ptx::stsm_x4(sts_addr, r0, r1, r2, r3);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(bar_r_empty + 8 * sr);
                    ptx::mbar_arrive(bar_a_full + 8 * sa);
                }
                ++r_cnt;
                ++a_cnt;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, (uint32_t)a.tmem_cols);
}

// ------------------------------------------------------------------ planning

static int round_up(int v, int m) { return (v + m - 1) / m * m; }

static bool fill_smem(IgemmGeom& g, int max_read_pos) {
    const int kpl = g.CK / 8;
    g.plane_pos = g.halo_rows * g.P;
    g.plane_stride = round_up(g.plane_pos * 16, 128);
    const int phases = g.stride == 1 ? 1 : 4;
    g.phase_stride = kpl * g.plane_stride;
    const int last_plane_pos = max_read_pos + 1 > g.plane_pos ? max_read_pos + 1 : g.plane_pos;
    g.a_bytes = round_up((phases * kpl - 1) * g.plane_stride + last_plane_pos * 16, 128);
    g.a_tx_bytes = kpl * g.plane_pos * 16;
    g.b_bytes = g.BN * g.CK * 2;
    if (g.mode == STAGE_NCHW) {
        g.raw_w = g.stride * g.Wt + 16;
        g.raw_bytes = round_up(g.CK * g.raw_rows * g.raw_w * 2, 128);
    } else {
        g.raw_w = 0;
        g.raw_bytes = 0;
    }
    const int fixed = 128 /*align*/ + 512 /*barriers*/ + (g.mode == STAGE_NCHW ? 4 * 32 * 16 + 128 : 0) +
                      16 * g.BN + 128 /*bias*/ + 4 * 32 * g.scr_pitch /*epilogue scratch*/;
    // preferred depths, shrunk until the stages fit
    const int a_opts[2] = {2, 1};
    const int r_opts[2] = {2, 1};
    for (int ia = 0; ia < 2; ++ia) {
        for (int ir = 0; ir < (g.mode == STAGE_NCHW ? 2 : 1); ++ir) {
            g.n_a = a_opts[ia];
            g.n_raw = g.mode == STAGE_NCHW ? r_opts[ir] : 0;
            const int used = fixed + g.n_a * g.a_bytes + g.n_raw * g.raw_bytes;
            int nb = (kSmemLimit - used) / g.b_bytes;
            if (nb > 12) nb = 12;
            if (nb >= 3) {
                g.n_b = nb;
                g.smem_bytes = used + nb * g.b_bytes;
                if (g.smem_bytes < kSmemFloor) g.smem_bytes = kSmemFloor;
                return true;
            }
        }
    }
    return false;
}

// Cycle estimate of one tile on one SM, used only to rank tilings: the MMAs are bound by tensor
// throughput or by the shared-memory reads of their operands, the staging by L2->SM bytes; the
// epilogue is exposed unless a second TMEM accumulator buffer hides it.
static double tile_cycles(const IgemmGeom& c, int C_out) {
    const double kFlopPerClk = 8192.0, kSmemBPerClk = 128.0, kL2BPerClk = 40.0, kStoreBPerClk = 32.0;
    const double ksteps = (double)c.KT * 9.0 * c.n_chunks * (c.CK / 16);
    const double mma_flop = c.NSUB * ksteps * 128.0 * c.BN * 16.0 * 2.0 / kFlopPerClk;
    const double mma_smem = c.NSUB * ksteps * (128.0 * 16 * 2 + c.BN * 16.0 * 2) / kSmemBPerClk;
    const double mma = mma_flop > mma_smem ? mma_flop : mma_smem;
    const double load = (double)c.KT * c.n_chunks * (c.a_tx_bytes + 9.0 * c.b_bytes) / kL2BPerClk;
    const int bn_used = C_out < c.BN ? C_out : c.BN;
    const double epi = c.NSUB * 128.0 * bn_used * 2.0 / kStoreBPerClk + 600.0;
    return (mma > load ? mma : load) + (c.acc_bufs == 1 ? epi : 0.15 * epi) + 800.0;
}

bool igemm_plan(x3_conv_plan* p, int num_sms) {
    const x3_conv_desc& d = p->d;
    IgemmGeom g;
    memset(&g, 0, sizeof g);
    g.stride = d.stride;
    if (d.stride != 1 && !(d.dims == 2 && d.layout == X3_NCHW)) return false;
    if (d.dims == 3) {
        if (d.layout != X3_NDHWC) return false;
        g.mode = STAGE_CL;
        g.KT = 3;
    } else if (d.layout == X3_NHWC) {
        g.mode = STAGE_CL;
        g.KT = 1;
    } else {
        g.mode = STAGE_NCHW;
        g.KT = 1;
        if (d.W % 8 != 0 || d.unpatchify2x2) return false;
    }
    if (g.mode == STAGE_CL && d.C_in % 8 != 0) return false;
    g.BN = d.C_out <= 16 ? 16 : d.C_out <= 32 ? 32 : d.C_out <= 64 ? 64 : 128;
    g.n_tiles = (d.C_out + g.BN - 1) / g.BN;
    g.CK = d.C_in <= 16 ? 16 : 32;
    // channels-last outputs with whole 16-byte channel groups go through the epilogue's smem transpose
    g.scr_pitch = (g.mode == STAGE_CL && !d.unpatchify2x2 && d.C_out % 8 == 0 && g.BN >= 32) ? 2 * g.BN + 16 : 0;
    g.n_chunks = (d.C_in + g.CK - 1) / g.CK;
    const int H_out = p->H_out, W_out = p->W_out;
    const int frames = d.N * (d.dims == 3 ? d.D : 1);

    double best_score = 1e300;
    IgemmGeom best;
    bool found = false;
    // candidate column tilings: row-aligned 128-wide subtiles, or a flat raster of width Wt
    int wt_cands[40], spr_cands[40], nc = 0;
    wt_cands[nc] = 128; spr_cands[nc++] = 1;
    for (int k = 1; k <= 16 && nc < 40; ++k) {
        int wt = (W_out + k - 1) / k;
        if (g.mode == STAGE_NCHW) wt = round_up(wt, 8);
        wt_cands[nc] = wt; spr_cands[nc++] = 0;
    }
    for (int ci = 0; ci < nc; ++ci) {
        const int Wt = wt_cands[ci], spr = spr_cands[ci];
        const int P = Wt + 2;
        if (Wt < 1 || P > 256) continue;
        if (g.mode == STAGE_NCHW && (Wt % 8 != 0 || g.stride * Wt + 16 > 256)) continue;
        for (int bufs = 2; bufs >= 1; --bufs) {
            int nsub_cap = 512 / (g.BN * bufs);
            if (nsub_cap > 8) nsub_cap = 8;
            for (int Rt = 1; Rt <= 64; ++Rt) {
                IgemmGeom c = g;
                c.Wt = Wt; c.P = P; c.spr = spr; c.Rt = Rt;
                // stride 2 stages Rt+1 rows per phase plane (even rows: 0,2,..,2Rt; odd: 1,..,2Rt-1)
                c.halo_rows = c.stride == 1 ? Rt + 2 : Rt + 1;
                c.raw_rows = c.stride == 1 ? Rt + 2 : 2 * Rt + 1;
                c.acc_bufs = bufs;
                c.NSUB = spr ? Rt * spr : (Rt * P + 127) / 128;
                if (c.NSUB > nsub_cap || c.halo_rows > 256) break;
                int max_read;
                const int tap_reach = c.stride == 1 ? 2 * P + 2 : P + 1;  // furthest tap offset
                if (spr) max_read = (Rt - 1) * P + (spr - 1) * 128 + 127 + tap_reach;
                else max_read = c.NSUB * 128 - 1 + tap_reach;
                if (!fill_smem(c, max_read)) break;
                int cols = c.NSUB * c.BN * bufs, tc = 32;
                while (tc < cols) tc *= 2;
                if (tc > 512) break;
                c.tmem_cols = tc;
                c.col_tiles = (W_out + Wt - 1) / Wt;
                c.row_tiles = (H_out + Rt - 1) / Rt;
                c.frames = frames;
                c.tiles = (long long)c.col_tiles * c.row_tiles * frames * c.n_tiles;
                const long long waves = (c.tiles + num_sms - 1) / num_sms;
                const double score = (double)waves * tile_cycles(c, d.C_out);
                if (score < best_score - 1e-9) {
                    best_score = score;
                    best = c;
                    found = true;
                }
            }
        }
    }
    if (!found) return false;
    best.grid = (int)(best.tiles < num_sms ? best.tiles : num_sms);
    p->g = best;
    return true;
}

// ------------------------------------------------------------------ launch

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)f;
        else
            cudaGetLastError();
    });
    return fn;
}

static x3_status encode4d(CUtensorMap* m, bool bf16, const void* ptr, const uint64_t dims[4], const uint64_t strides[3],
                          const uint32_t box[4]) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return fail(X3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
    cuuint32_t bd[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                     const_cast<void*>(ptr), gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(X3_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return X3_OK;
}

template <int MODE, bool BF16>
static x3_status launch_t(const CUtensorMap& mx, const CUtensorMap& mc, const IgemmArgs& a, const IgemmGeom& g,
                          cudaStream_t s) {
    auto k = igemm_conv_kernel<MODE, BF16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "igemm smem attribute: %s", cudaGetErrorString(e));
    k<<<g.grid, MODE == STAGE_NCHW ? 320 : 192, g.smem_bytes, s>>>(mx, mc, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "igemm launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

x3_status launch_igemm(const x3_conv_plan* p, const void* x, const void* carry, const void* w_packed,
                       const void* bias, void* y, cudaStream_t s) {
    const x3_conv_desc& d = p->d;
    const IgemmGeom& g = p->g;
    const bool bf16 = d.dtype == X3_BF16;
    IgemmArgs a;
    memset(&a, 0, sizeof a);
    a.C_in = d.C_in; a.C_out = d.C_out; a.N = d.N; a.D = d.D; a.H = d.H; a.W = d.W;
    a.H_out = p->H_out; a.W_out = p->W_out; a.dout = d.dims == 3 ? d.D : 1;
    a.act = d.act;
    a.out_kind = d.unpatchify2x2 ? OUT_UNPATCH_CL : (g.mode == STAGE_NCHW ? OUT_NCHW : OUT_CL);
    a.has_carry = carry != nullptr;
    a.BN = g.BN; a.n_tiles = g.n_tiles; a.CK = g.CK; a.n_chunks = g.n_chunks; a.KT = g.KT; a.NSUB = g.NSUB;
    a.Rt = g.Rt; a.Wt = g.Wt; a.P = g.P; a.spr = g.spr; a.halo_rows = g.halo_rows; a.plane_stride = g.plane_stride;
    a.a_bytes = g.a_bytes; a.a_tx_bytes = g.a_tx_bytes; a.raw_w = g.raw_w; a.raw_bytes = g.raw_bytes;
    a.raw_tx_bytes = g.CK * g.raw_rows * g.raw_w * 2; a.b_bytes = g.b_bytes; a.n_a = g.n_a; a.n_b = g.n_b;
    a.stride = g.stride; a.raw_rows = g.raw_rows; a.phase_stride = g.phase_stride;
    a.row_shift = p->row_shift;
    a.n_raw = g.n_raw; a.acc_bufs = g.acc_bufs; a.tmem_cols = g.tmem_cols;
    a.col_tiles = g.col_tiles; a.row_tiles = g.row_tiles; a.frames = g.frames; a.tiles = g.tiles;
    a.scr_pitch = g.scr_pitch;
    a.idesc = ptx::idesc_f16(128, g.BN, bf16);
    a.w = (const uint8_t*)w_packed; a.bias = bias; a.y = y;

    CUtensorMap mx, mc;
    memset(&mx, 0, sizeof mx);
    memset(&mc, 0, sizeof mc);
    x3_status st;
    if (g.mode == STAGE_CL) {
        const uint64_t C = (uint64_t)d.C_in;
        const uint64_t frames_x = (uint64_t)d.N * (d.dims == 3 ? d.D : 1);
        const uint64_t dims[4] = {C, (uint64_t)d.W, (uint64_t)d.H, frames_x};
        const uint64_t strides[3] = {C * 2, C * 2 * d.W, C * 2 * d.W * d.H};
        const uint32_t box[4] = {8, (uint32_t)g.P, (uint32_t)g.halo_rows, 1};
        st = encode4d(&mx, bf16, x, dims, strides, box);
        if (st != X3_OK) return st;
        if (carry) {
            const uint64_t dc[4] = {C, (uint64_t)d.W, (uint64_t)d.H, (uint64_t)d.N * 2};
            st = encode4d(&mc, bf16, carry, dc, strides, box);
            if (st != X3_OK) return st;
        } else {
            mc = mx;
        }
        return bf16 ? launch_t<STAGE_CL, true>(mx, mc, a, g, s) : launch_t<STAGE_CL, false>(mx, mc, a, g, s);
    }
    const uint64_t dims[4] = {(uint64_t)d.W, (uint64_t)d.H, (uint64_t)d.C_in, (uint64_t)d.N};
    const uint64_t strides[3] = {(uint64_t)d.W * 2, (uint64_t)d.W * d.H * 2, (uint64_t)d.W * d.H * d.C_in * 2};
    const uint32_t box[4] = {(uint32_t)g.raw_w, (uint32_t)g.raw_rows, (uint32_t)g.CK, 1};
    st = encode4d(&mx, bf16, x, dims, strides, box);
    if (st != X3_OK) return st;
    mc = mx;
    return bf16 ? launch_t<STAGE_NCHW, true>(mx, mc, a, g, s) : launch_t<STAGE_NCHW, false>(mx, mc, a, g, s);
}

// One thread waits, bounded, on an mbarrier nobody arrives at; the wait runs out after limit_ns and
// the status word records the timeout, exactly as in the convolution kernels.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(b, 0)) {
        if (ptx::globaltimer() - t0 > limit_ns) {
            atomicOr(&g_x3_status, 1u);
            break;
        }
    }
}

// Device address of the status word on the current device, for kernels compiled in other files.
x3_status device_status_word(unsigned int** out) {
    static unsigned int* ptrs[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return fail(X3_ERR_CUDA, "status word: no current device");
    if (!ptrs[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_x3_status);
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "status word address: %s", cudaGetErrorString(e));
        ptrs[dev] = (unsigned int*)p;
    }
    *out = ptrs[dev];
    return X3_OK;
}

x3_status selftest_wait_timeout(int limit_ms, cudaStream_t s) {
    if (limit_ms < 1 || limit_ms > 2000) return fail(X3_ERR_INVALID, "limit_ms must be in 1..2000");
    selftest_wait_kernel<<<1, 32, 0, s>>>((uint64_t)limit_ms * 1000000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

x3_status read_device_status(int reset) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "device synchronize: %s", cudaGetErrorString(e));
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_x3_status, sizeof v);
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (reset) {
        const unsigned int z = 0;
        e = cudaMemcpyToSymbol(g_x3_status, &z, sizeof z);
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "status reset: %s", cudaGetErrorString(e));
    }
    if (v & 1u) return fail(X3_ERR_TIMEOUT, "a bounded device wait ran out");
    return X3_OK;
}

}  // namespace x3
