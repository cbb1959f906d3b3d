// Host side of libx3conv: descriptor validation, plans, dispatch and the causal stack driver.
//
// Shape checks mirror the host wrapper of FastVideo wan22_vae_decode/solution/head.cu
// (head_stencil: layout and size checks before any launch, device of the caller, launch on the
// caller's stream, launch check afterwards), extended to close the hazard that wrapper's own
// comment names: a tensor whose depth or height disagrees with the plan is rejected here rather
// than read out of bounds.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "internal.h"

namespace x3 {

static thread_local char g_err[512] = "";

x3_status fail(x3_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

static void clear_err() { g_err[0] = 0; }

size_t in_elems(const x3_conv_plan* p) {
    const x3_conv_desc& d = p->d;
    return (size_t)d.N * d.C_in * (d.dims == 3 ? d.D : 1) * d.H * d.W;
}

size_t out_elems(const x3_conv_plan* p) {
    const x3_conv_desc& d = p->d;
    return (size_t)d.N * d.C_out * (d.dims == 3 ? d.D : 1) * p->H_out * p->W_out;
}

static bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

static x3_status validate(const x3_conv_desc* d) {
    if (!d) return fail(X3_ERR_INVALID, "descriptor is NULL");
    if (d->dims != 2 && d->dims != 3) return fail(X3_ERR_INVALID, "dims must be 2 or 3 (got %d)", d->dims);
    if (d->N < 1 || d->C_in < 1 || d->C_out < 1 || d->H < 1 || d->W < 1)
        return fail(X3_ERR_INVALID, "N, C_in, C_out, H, W must be >= 1");
    if (d->dims == 2) {
        if (d->D != 1 && d->D != 0) return fail(X3_ERR_INVALID, "2D descriptors have D = 1");
        if (d->stride != 1 && d->stride != 2) return fail(X3_ERR_INVALID, "stride must be 1 or 2");
        if (d->layout != X3_NCHW && d->layout != X3_NHWC)
            return fail(X3_ERR_INVALID, "2D layout must be X3_NCHW or X3_NHWC");
    } else {
        if (d->D < 1) return fail(X3_ERR_INVALID, "3D descriptors need D >= 1");
        if (d->stride != 1) return fail(X3_ERR_INVALID, "causal 3D convolution has stride 1");
        if (d->layout != X3_NCDHW && d->layout != X3_NDHWC)
            return fail(X3_ERR_INVALID, "3D layout must be X3_NCDHW or X3_NDHWC");
    }
    if (d->dtype != X3_F16 && d->dtype != X3_BF16) return fail(X3_ERR_INVALID, "dtype must be f16 or bf16");
    if (d->act < X3_ACT_NONE || d->act > X3_ACT_CLAMP1) return fail(X3_ERR_INVALID, "bad activation");
    if (d->has_bias != 0 && d->has_bias != 1) return fail(X3_ERR_INVALID, "has_bias must be 0 or 1");
    if (d->unpatchify2x2 != 0 && d->unpatchify2x2 != 1) return fail(X3_ERR_INVALID, "unpatchify2x2 must be 0 or 1");
    if (d->unpatchify2x2 && d->C_out != 12) return fail(X3_ERR_INVALID, "unpatchify2x2 needs C_out == 12");
    if (d->kernel < X3_KERNEL_AUTO || d->kernel > X3_KERNEL_HEAD_STENCIL) return fail(X3_ERR_INVALID, "bad kernel choice");
    if (d->H_global != 0) {
        // banded mode (reading of the head.cu page's band parameters: a band must hold its halo rows
        // wherever the global row exists)
        if (d->stride != 1) return fail(X3_ERR_INVALID, "banded mode needs stride 1");
        if (d->H_global < 1 || d->band_rows < 1 || d->band_lo < 0 || d->band_lo + d->band_rows > d->H_global)
            return fail(X3_ERR_INVALID, "band [%d, %d) is not inside the %d-row image", d->band_lo,
                        d->band_lo + d->band_rows, d->H_global);
        const int lo = d->band_lo > 0 ? d->band_lo - 1 : 0;
        const int hi = d->band_lo + d->band_rows + 1 < d->H_global ? d->band_lo + d->band_rows + 1 : d->H_global;
        if (d->H != hi - lo)
            return fail(X3_ERR_INVALID,
                        "a band needs its halo rows wherever the global row exists: output rows [%d, %d) of %d "
                        "read input rows [%d, %d), so H must be %d (got %d)",
                        d->band_lo, d->band_lo + d->band_rows, d->H_global, lo, hi, hi - lo, d->H);
        if (d->kernel == X3_KERNEL_HEAD_TWO_PASS || d->kernel == X3_KERNEL_HEAD_SPLIT)
            return fail(X3_ERR_INVALID, "the two-pass head kernels have no banded mode");
    } else if (d->band_lo != 0 || d->band_rows != 0) {
        return fail(X3_ERR_INVALID, "band_lo and band_rows need H_global (0 = the whole plane)");
    }
    // Every tensor must be indexable with 63-bit offsets and every per-image plane with 31 bits.
    const long long frames = (long long)d->N * (d->dims == 3 ? d->D + 2 : 1);
    const long long plane = (long long)d->H * d->W;
    if (plane > (1LL << 30) || frames > (1LL << 30) || (long long)d->C_in > 65536 || (long long)d->C_out > 65536)
        return fail(X3_ERR_INVALID, "tensor too large");
    if ((double)frames * plane * (d->C_in > d->C_out ? d->C_in : d->C_out) > 9.0e18)
        return fail(X3_ERR_INVALID, "tensor too large");
    return X3_OK;
}

static int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        return 148;
    }
    return sms;
}

static size_t direct_packed_bytes(const x3_conv_desc& d) {
    return (size_t)d.C_out * d.C_in * (d.dims == 3 ? 27 : 9) * 2;
}

}  // namespace x3

using namespace x3;

extern "C" {

x3_status conv_plan_create(const x3_conv_desc* desc, x3_conv_plan** plan) {
    clear_err();
    if (!plan) return fail(X3_ERR_INVALID, "plan output pointer is NULL");
    *plan = nullptr;
    x3_status st = validate(desc);
    if (st != X3_OK) return st;
    x3_conv_plan* p = new (std::nothrow) x3_conv_plan();
    if (!p) return fail(X3_ERR_OOM, "out of host memory");
    p->d = *desc;
    if (p->d.dims == 2) p->d.D = 1;
    p->H_out = p->d.H_global ? p->d.band_rows : (p->d.H - 1) / p->d.stride + 1;
    p->row_shift = (p->d.H_global && p->d.band_lo > 0) ? 1 : 0;
    p->W_out = (p->d.W - 1) / p->d.stride + 1;
    p->num_sms = device_sms();
    bool igemm_ok = false;
    const char* force = getenv("X3CONV_FORCE_KERNEL");
    x3_kernel choice = p->d.kernel;
    if (choice == X3_KERNEL_AUTO && force) {
        if (!strcmp(force, "direct")) choice = X3_KERNEL_DIRECT;
        else if (!strcmp(force, "igemm")) choice = X3_KERNEL_IGEMM;
    }
    bool cl_ok = false;
    if (choice == X3_KERNEL_HEAD_TWO_PASS || choice == X3_KERNEL_HEAD_SPLIT) {
        if (!igemm_cl_plan(p, p->num_sms)) {
            delete p;
            return fail(X3_ERR_UNSUPPORTED, "the two-pass head needs unpatchify2x2, 3D, X3_NDHWC and bf16");
        }
        p->kind = K_HEAD_TWO_PASS;
        p->packed_bytes = (size_t)p->cl.KT * p->cl.n_chunks * (128 * 64 * 2);
        *plan = p;
        return X3_OK;
    }
    // the conv_out head (bf16 channels-last, unpatchified) runs by default as the stencil head
    const bool auto_head = choice == X3_KERNEL_AUTO && !force && p->d.unpatchify2x2 && p->d.dims == 3 &&
                           p->d.layout == X3_NDHWC && p->d.dtype == X3_BF16;
    if (choice == X3_KERNEL_HEAD_STENCIL || auto_head) {
        p->d.kernel = X3_KERNEL_HEAD_STENCIL;
        if (igemm_cl_plan(p, p->num_sms)) {
            p->kind = K_IGEMM_CL;
            p->packed_bytes = (size_t)p->cl.KT * p->cl.n_chunks * (128 * 64 * 2);
            *plan = p;
            return X3_OK;
        }
        if (!auto_head) {
            delete p;
            return fail(X3_ERR_UNSUPPORTED, "the stencil head needs unpatchify2x2, 3D, X3_NDHWC and bf16");
        }
        p->d.kernel = X3_KERNEL_AUTO;  // no stencil plan: the other forms below
    }
    if (choice != X3_KERNEL_DIRECT && !(force && !strcmp(force, "igemm_nsub"))) {
        // 2D channels-last layers of any width run on the swapped engine (the M = 64 form for at most
        // 64 output channels); stride 2 from the four input phases, else as the stride-1 raster with
        // even positions kept
        const bool nhwc2d = p->d.dims == 2 && p->d.layout == X3_NHWC;
        if (nhwc2d && p->d.stride == 2 && igemm_cl_plan(p, p->num_sms, true)) {
            cl_ok = true;
        } else if (nhwc2d && p->d.stride == 2) {
            x3_conv_plan q = *p;
            q.d.stride = 1;
            q.H_out = q.d.H;
            q.W_out = q.d.W;
            if (igemm_cl_plan(&q, p->num_sms, true)) {
                p->cl = q.cl;
                p->cl.sub2 = 1;
                p->g = q.g;
                cl_ok = true;
            }
        } else {
            cl_ok = igemm_cl_plan(p, p->num_sms, nhwc2d);
        }
    }
    if (choice != X3_KERNEL_DIRECT && !cl_ok) igemm_ok = igemm_plan(p, p->num_sms);
    if (choice == X3_KERNEL_IGEMM && !igemm_ok && !cl_ok) {
        delete p;
        return fail(X3_ERR_UNSUPPORTED, "the tcgen05 implicit-GEMM kernels do not handle this descriptor");
    }
    if (cl_ok) {
        p->kind = K_IGEMM_CL;
        p->packed_bytes = cl_packed_bytes(p->cl);
    } else if (igemm_ok) {
        p->kind = K_IGEMM;
        const IgemmGeom& g = p->g;
        p->packed_bytes = (size_t)g.n_tiles * g.KT * g.n_chunks * 9 * g.b_bytes;
    } else {
        p->kind = K_DIRECT;
        p->packed_bytes = direct_packed_bytes(p->d);
    }
    // A 2D NCHW layer on the tensor-core engines also gets a channels-last form for the stack driver,
    // which keeps the activations between layers channels-last; unless forced to one engine.
    if (p->d.dims == 2 && p->d.layout == X3_NCHW && choice != X3_KERNEL_DIRECT && !force && p->d.stride <= 2 &&
        p->d.C_out % 8 == 0) {
        x3_conv_plan q = *p;
        q.d.layout = X3_NHWC;
        q.d.C_in = (q.d.C_in + 7) / 8 * 8;
        // stride 2 from the four input phases when the engine takes it, else as the stride-1 raster
        bool q_ok = p->d.stride == 2 && igemm_cl_plan(&q, p->num_sms, true);
        if (!q_ok) {
            q.d.stride = 1;
            q.H_out = q.d.H;
            q.W_out = q.d.W;
            q_ok = igemm_cl_plan(&q, p->num_sms, true);
            q.cl.sub2 = p->d.stride == 2 ? 1 : 0;
        }
        if (q_ok) {
            p->has_shadow = 1;
            p->cl_shadow = q.cl;
            // the channels-last engine's weight blocks; the NCHW form of the same engine uses the
            // same blocks (n_chunks agree: C_in and its round-up to 8 need the same 64-channel chunks)
            if (p->kind == K_IGEMM_CL && !p->cl.kwm && !p->cl.ctr && !q.cl.m64 && !q.cl.tn && !p->cl.m64 && !p->cl.tn &&
                p->cl.n_chunks == q.cl.n_chunks && p->cl.n_tiles == q.cl.n_tiles) {
                p->shadow_w_off = 0;
            } else {
                p->shadow_w_off = (p->packed_bytes + 255) & ~(size_t)255;
                p->packed_bytes = p->shadow_w_off + cl_packed_bytes(q.cl);
            }
        }
    }
    *plan = p;
    return X3_OK;
}

void conv_plan_destroy(x3_conv_plan* plan) { delete plan; }

const char* conv_plan_kernel_name(const x3_conv_plan* plan) {
    if (!plan) return "";
    if (plan->kind == K_HEAD_TWO_PASS) return plan->d.kernel == X3_KERNEL_HEAD_SPLIT ? "head_split" : "head_two_pass";
    if (plan->kind == K_IGEMM_CL && plan->cl.kwm) return "igemm_tcgen05_sw128_head";
    if (plan->kind == K_IGEMM_CL && plan->cl.stn) return "igemm_tcgen05_sw128_head_stencil";
    if (plan->kind == K_IGEMM_CL && plan->cl.nchw) return "igemm_tcgen05_sw128_nchw";
    return plan->kind == K_IGEMM_CL ? "igemm_tcgen05_sw128" : plan->kind == K_IGEMM ? "igemm_tcgen05" : "direct_simt";
}

int conv_plan_launches(const x3_conv_plan* plan) { return plan ? 1 : 0; }

static int describe_main(const x3_conv_plan* plan, char* buf, size_t len) {
    if (!plan) return snprintf(buf, len, "{}");
    const IgemmGeom& g = plan->g;
    if (plan->kind == K_IGEMM_CL || plan->kind == K_HEAD_TWO_PASS) {
        const ClGeom& c = plan->cl;
        return snprintf(buf, len,
                        "{\"kernel\": \"igemm_tcgen05_sw128\", \"mode\": \"channels_last_sw128_swapped\", "
                        "\"BM\": 128, \"BN\": 256, \"CK\": 64, \"n_tiles\": %d, \"n_chunks\": %d, \"KT\": %d, "
                        "\"Wt\": %d, \"P\": %d, \"HR\": %d, \"strips\": %d, \"windows\": %d, \"frames\": %d, "
                        "\"h_bytes\": %d, \"n_h\": %d, \"n_w\": %d, \"kwm\": %d, \"nchw\": %d, \"win_adv\": %d, \"tiles\": %lld, "
                        "\"smem_bytes\": %d, \"grid\": %d, \"H_out\": %d, \"W_out\": %d, \"sms\": %d, "
                        "\"m64\": %d, \"sub2\": %d, \"s2\": %d, \"ctr\": %d, \"w2\": %d, \"stn\": %d, \"tn\": %d, "
                        "\"tk\": %d, \"row_shift\": %d}",
                        c.n_tiles, c.n_chunks, c.KT, c.Wt, c.P, c.HR, c.strips, c.windows, c.frames, c.h_bytes, c.n_h,
                        c.n_w, c.kwm, c.nchw, c.win_adv, c.tiles, c.smem_bytes, c.grid, plan->H_out, plan->W_out, plan->num_sms,
                        c.m64, c.sub2, c.s2, c.ctr, c.w2, c.stn, c.tn, c.tk, plan->row_shift);
    }
    if (plan->kind != K_IGEMM)
        return snprintf(buf, len, "{\"kernel\": \"direct_simt\", \"H_out\": %d, \"W_out\": %d, \"sms\": %d}",
                        plan->H_out, plan->W_out, plan->num_sms);
    return snprintf(buf, len,
                    "{\"kernel\": \"igemm_tcgen05\", \"mode\": \"%s\", \"BN\": %d, \"n_tiles\": %d, \"CK\": %d, "
                    "\"n_chunks\": %d, \"KT\": %d, \"NSUB\": %d, \"Rt\": %d, \"Wt\": %d, \"P\": %d, \"spr\": %d, "
                    "\"plane_stride\": %d, \"a_bytes\": %d, \"raw_bytes\": %d, \"b_bytes\": %d, \"n_a\": %d, "
                    "\"n_b\": %d, \"n_raw\": %d, \"acc_bufs\": %d, \"tmem_cols\": %d, \"col_tiles\": %d, "
                    "\"row_tiles\": %d, \"frames\": %d, \"tiles\": %lld, \"smem_bytes\": %d, \"grid\": %d, "
                    "\"H_out\": %d, \"W_out\": %d, \"sms\": %d}",
                    g.mode == STAGE_CL ? "channels_last_tma" : "nchw_tma_transpose", g.BN, g.n_tiles, g.CK,
                    g.n_chunks, g.KT, g.NSUB, g.Rt, g.Wt, g.P, g.spr, g.plane_stride, g.a_bytes, g.raw_bytes,
                    g.b_bytes, g.n_a, g.n_b, g.n_raw, g.acc_bufs, g.tmem_cols, g.col_tiles, g.row_tiles, g.frames,
                    g.tiles, g.smem_bytes, g.grid, plan->H_out, plan->W_out, plan->num_sms);
}

int conv_plan_describe(const x3_conv_plan* plan, char* buf, size_t len) {
    char tmp[2048];
    int n = describe_main(plan, tmp, sizeof tmp);
    if (plan && plan->has_shadow && n > 0 && (size_t)n < sizeof tmp) {
        // the channels-last form used inside stacks: appended as "shadow" before the closing brace
        const ClGeom& c = plan->cl_shadow;
        const int m = snprintf(tmp + n - 1, sizeof tmp - (size_t)(n - 1),
                               ", \"shadow\": {\"Wt\": %d, \"P\": %d, \"HR\": %d, \"strips\": %d, \"windows\": %d, "
                               "\"n_chunks\": %d, \"n_tiles\": %d, \"n_w\": %d, \"n_h\": %d, \"sub2\": %d, \"s2\": %d, \"tiles\": %lld, "
                               "\"smem_bytes\": %d, \"grid\": %d, \"w_off\": %zu, \"m64\": %d, \"tn\": %d, \"tk\": %d}}",
                               c.Wt, c.P, c.HR, c.strips, c.windows, c.n_chunks, c.n_tiles, c.n_w, c.n_h, c.sub2, c.s2, c.tiles,
                               c.smem_bytes, c.grid, plan->shadow_w_off, c.m64, c.tn, c.tk);
        n = n - 1 + m;
    }
    return snprintf(buf, len, "%s", tmp);
}

size_t conv_packed_weight_bytes(const x3_conv_plan* plan) { return plan ? plan->packed_bytes : 0; }

x3_status conv_pack_weights(const x3_conv_plan* plan, const void* w, void* w_packed, x3_stream_t stream) {
    clear_err();
    if (!plan || !w || !w_packed) return fail(X3_ERR_INVALID, "conv_pack_weights: NULL argument");
    if (!aligned(w, 2) || !aligned(w_packed, 256))
        return fail(X3_ERR_INVALID, "conv_pack_weights: w must be 2-byte and w_packed 256-byte aligned");
    return launch_pack_weights(plan, w, w_packed, (cudaStream_t)stream);
}

x3_status conv_forward(const x3_conv_plan* plan, const void* x, const void* carry, const void* w_packed,
                       const void* bias, void* y, x3_stream_t stream) {
    clear_err();
    if (!plan || !x || !w_packed || !y) return fail(X3_ERR_INVALID, "conv_forward: NULL argument");
    if (plan->d.has_bias && !bias) return fail(X3_ERR_INVALID, "conv_forward: plan has a bias but bias is NULL");
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(w_packed, 256) || (carry && !aligned(carry, 16)) ||
        (bias && !aligned(bias, 2)))
        return fail(X3_ERR_INVALID, "conv_forward: x, y, carry need 16-byte alignment, w_packed 256-byte");
    const void* c = plan->d.dims == 3 ? carry : nullptr;
    const char* lo_y = (const char*)y;
    const char* hi_y = lo_y + out_elems(plan) * 2;
    const char* lo_x = (const char*)x;
    const char* hi_x = lo_x + in_elems(plan) * 2;
    if (lo_y < hi_x && lo_x < hi_y) return fail(X3_ERR_INVALID, "conv_forward: y overlaps x");
    if (plan->kind == K_HEAD_TWO_PASS)
        return fail(X3_ERR_INVALID, "conv_forward: a two-pass head plan runs with conv_head_two_pass");
    if (plan->kind == K_IGEMM_CL)
        return launch_igemm_cl(plan, x, c, w_packed, plan->d.has_bias ? bias : nullptr, y, (cudaStream_t)stream);
    if (plan->kind == K_IGEMM) return launch_igemm(plan, x, c, w_packed, plan->d.has_bias ? bias : nullptr, y, (cudaStream_t)stream);
    return launch_direct(plan, x, c, w_packed, plan->d.has_bias ? bias : nullptr, y, (cudaStream_t)stream);
}

size_t conv_head_g_bytes(const x3_conv_plan* plan) {
    if (!plan || plan->kind != K_HEAD_TWO_PASS) return 0;
    // [N][D][9][H][W][12] of bf16 or fp32
    return (size_t)plan->d.N * plan->d.D * 9 * plan->d.H * plan->d.W * 12 * (plan->d.kernel == X3_KERNEL_HEAD_SPLIT ? 4 : 2);
}

x3_status conv_head_two_pass(const x3_conv_plan* plan, const void* x, const void* carry, const void* w_packed,
                             const void* bias, void* g, void* y, x3_stream_t stream) {
    clear_err();
    if (!plan || plan->kind != K_HEAD_TWO_PASS) return fail(X3_ERR_INVALID, "conv_head_two_pass: needs a two-pass head plan");
    if (!x || !w_packed || !g || !y || (plan->d.has_bias && !bias))
        return fail(X3_ERR_INVALID, "conv_head_two_pass: NULL argument");
    if (!aligned(x, 16) || !aligned(g, 16) || !aligned(y, 16) || !aligned(w_packed, 256) || (carry && !aligned(carry, 16)))
        return fail(X3_ERR_INVALID, "conv_head_two_pass: x, g, y, carry need 16-byte alignment, w_packed 256-byte");
    {
        // g is written by pass 1 while x is read, and read by pass 2 while y is written
        const char* lo_x = (const char*)x;
        const char* hi_x = lo_x + in_elems(plan) * 2;
        const char* lo_g = (const char*)g;
        const char* hi_g = lo_g + conv_head_g_bytes(plan);
        const char* lo_y = (const char*)y;
        const char* hi_y = lo_y + out_elems(plan) * 2;
        if ((lo_g < hi_x && lo_x < hi_g) || (lo_g < hi_y && lo_y < hi_g) || (lo_y < hi_x && lo_x < hi_y))
            return fail(X3_ERR_INVALID, "conv_head_two_pass: x, g and y must not overlap");
    }
    // pass 1: the temporal convolution into g (108 accumulator rows, no bias, no activation), written
    // one plane per spatial tap
    x3_conv_plan p1 = *plan;
    p1.kind = K_IGEMM_CL;
    p1.d.C_out = 112;
    p1.d.unpatchify2x2 = 0;
    p1.d.act = X3_ACT_NONE;
    p1.d.has_bias = 0;
    x3_status st = launch_igemm_cl(&p1, x, carry, w_packed, nullptr, g, (cudaStream_t)stream);
    if (st != X3_OK) return st;
    // pass 2: nine spatial taps, bias, clamp, one rounding, unpatchify
    return launch_head_stencil(plan, g, plan->d.has_bias ? bias : nullptr, y, (cudaStream_t)stream);
}

}  // extern "C"

namespace x3 {

// A stack of 2D NCHW layers that all have a channels-last form, the last one stride 1, runs with its
// activations channels-last between the layers: the input is converted once, each layer reads and
// writes NHWC, and the last layer's epilogue writes the NCHW result. X3CONV_STACK_LAYOUT=nchw turns
// this off (each layer then runs its own NCHW form).
static bool stack_channels_last(const x3_conv_plan* const* plans, int n_layers) {
    if (n_layers < 2) return false;
    const char* env = getenv("X3CONV_STACK_LAYOUT");
    if (env && !strcmp(env, "nchw")) return false;
    for (int i = 0; i < n_layers; ++i)
        if (!plans[i] || plans[i]->d.dims != 2 || plans[i]->d.layout != X3_NCHW || !plans[i]->has_shadow) return false;
    return plans[n_layers - 1]->d.stride == 1;
}

// Bytes of the channels-last copy of the first layer's input (C_in rounded up to 8).
static size_t stack_input_cl_bytes(const x3_conv_plan* p) {
    return (size_t)p->d.N * p->d.H * p->d.W * ((p->d.C_in + 7) / 8 * 8) * 2;
}

}  // namespace x3

extern "C" {

size_t conv_stack_workspace_bytes(const x3_conv_plan* const* plans, int n_layers) {
    if (!plans || n_layers < 1) return 0;
    size_t biggest = 0;
    for (int i = 0; i + 1 < n_layers; ++i) {
        if (!plans[i]) return 0;
        size_t b = out_elems(plans[i]) * 2;
        b = (b + 255) & ~(size_t)255;
        if (b > biggest) biggest = b;
    }
    if (n_layers > 1 && plans[n_layers - 1] && stack_channels_last(plans, n_layers)) {
        // two buffers: the converted input and the odd layers' outputs / the even layers' outputs
        size_t b = (stack_input_cl_bytes(plans[0]) + 255) & ~(size_t)255;
        if (b > biggest) biggest = b;
        return 2 * biggest;
    }
    return n_layers > 1 ? (n_layers > 2 ? 2 * biggest : biggest) : 0;
}

// The stack driver's side stream for carry copies, one per thread and device: calls from different
// threads never share its events. Created on first use and kept until the process exits.
struct SideStream {
    static constexpr int kEvents = 4;  // a wait always names one of the last two layers' copies
    cudaStream_t s = nullptr;
    cudaEvent_t fork[kEvents] = {};
    cudaEvent_t done[kEvents] = {};
};

static x3_status side_stream(SideStream** out) {
    constexpr int kMaxDevices = 64;
    static thread_local SideStream per_dev[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "side stream: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(X3_ERR_UNSUPPORTED, "side stream: device %d out of range", dev);
    SideStream& ss = per_dev[dev];
    if (!ss.s) {
        e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking);
        for (int k = 0; k < SideStream::kEvents && e == cudaSuccess; ++k) {
            e = cudaEventCreateWithFlags(&ss.fork[k], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.done[k], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) {
            ss = SideStream{};  // leaks what was made; the next call retries
            return fail(X3_ERR_CUDA, "side stream: %s", cudaGetErrorString(e));
        }
    }
    *out = &ss;
    return X3_OK;
}

// Copy the last two frames of the sequence [history, input] of a layer into its carry buffer.
static x3_status update_carry(const x3_conv_plan* p, const void* input, void* carry, int history_valid,
                              cudaStream_t s) {
    const x3_conv_desc& d = p->d;
    const size_t plane = (size_t)d.H * d.W * 2;  // bytes of one channel plane of one frame
    const int D = d.D;
    cudaError_t e = cudaSuccess;
    if (d.layout == X3_NDHWC) {
        const size_t frame = plane * d.C_in;
        if (D >= 2) {
            e = cudaMemcpy2DAsync(carry, 2 * frame, (const char*)input + (size_t)(D - 2) * frame, (size_t)D * frame,
                                  2 * frame, d.N, cudaMemcpyDeviceToDevice, s);
        } else {
            if (history_valid)
                e = cudaMemcpy2DAsync(carry, 2 * frame, (const char*)carry + frame, 2 * frame, frame, d.N,
                                      cudaMemcpyDeviceToDevice, s);
            else
                e = cudaMemset2DAsync(carry, 2 * frame, 0, frame, d.N, s);
            if (e == cudaSuccess)
                e = cudaMemcpy2DAsync((char*)carry + frame, 2 * frame, input, frame, frame, d.N,
                                      cudaMemcpyDeviceToDevice, s);
        }
    } else {  // NCDHW: rows are (n, c) with D or 2 frames each
        const size_t rows = (size_t)d.N * d.C_in;
        if (D >= 2) {
            e = cudaMemcpy2DAsync(carry, 2 * plane, (const char*)input + (size_t)(D - 2) * plane, (size_t)D * plane,
                                  2 * plane, rows, cudaMemcpyDeviceToDevice, s);
        } else {
            if (history_valid)
                e = cudaMemcpy2DAsync(carry, 2 * plane, (const char*)carry + plane, 2 * plane, plane, rows,
                                      cudaMemcpyDeviceToDevice, s);
            else
                e = cudaMemset2DAsync(carry, 2 * plane, 0, plane, rows, s);
            if (e == cudaSuccess)
                e = cudaMemcpy2DAsync((char*)carry + plane, 2 * plane, input, plane, plane, rows,
                                      cudaMemcpyDeviceToDevice, s);
        }
    }
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "carry update: %s", cudaGetErrorString(e));
    return X3_OK;
}

x3_status conv_stack_forward(const x3_conv_plan* const* plans, int n_layers, const void* x, void* const* carries,
                             int carry_valid, const void* const* w_packed, const void* const* bias, void* y,
                             void* workspace, size_t workspace_bytes, x3_stream_t stream) {
    clear_err();
    if (n_layers < 1) return fail(X3_ERR_INVALID, "conv_stack_forward: n_layers must be at least 1 (got %d)", n_layers);
    if (!plans || !x || !y || !w_packed || (!bias && plans[0] && plans[0]->d.has_bias))
        return fail(X3_ERR_INVALID, "conv_stack_forward: NULL argument");
    for (int i = 0; i < n_layers; ++i) {
        if (!plans[i] || !w_packed[i]) return fail(X3_ERR_INVALID, "conv_stack_forward: layer %d plan or weights NULL", i);
        if (plans[i]->d.has_bias && (!bias || !bias[i])) return fail(X3_ERR_INVALID, "conv_stack_forward: layer %d bias NULL", i);
        if (i + 1 < n_layers) {
            const x3_conv_desc& a = plans[i]->d;
            const x3_conv_desc& b = plans[i + 1]->d;
            if (a.dims != b.dims || a.N != b.N || a.D != b.D || a.layout != b.layout || a.dtype != b.dtype ||
                a.C_out != b.C_in || plans[i]->H_out != b.H || plans[i]->W_out != b.W || a.unpatchify2x2)
                return fail(X3_ERR_INVALID, "conv_stack_forward: layer %d output does not match layer %d input", i, i + 1);
        }
    }
    const size_t need = conv_stack_workspace_bytes(plans, n_layers);
    if (need && (!workspace || workspace_bytes < need))
        return fail(X3_ERR_OOM, "conv_stack_forward: workspace needs %zu bytes, got %zu", need, workspace_bytes);
    if (workspace && !aligned(workspace, 256)) return fail(X3_ERR_INVALID, "conv_stack_forward: workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    if (stack_channels_last(plans, n_layers)) {
        const size_t half = need / 2;
        void* buf[2] = {workspace, (char*)workspace + half};
        const x3_conv_desc& d0 = plans[0]->d;
        x3_status st = launch_nchw_to_nhwc(x, buf[0], d0.N, d0.C_in, (d0.C_in + 7) / 8 * 8, d0.H, d0.W, s);
        if (st != X3_OK) return st;
        const void* in = buf[0];
        for (int i = 0; i < n_layers; ++i) {
            const bool last = i == n_layers - 1;
            void* out = last ? y : buf[(i + 1) % 2];
            const x3_conv_plan* p = plans[i];
            st = launch_igemm_cl_shadow(p, in, w_packed[i], p->d.has_bias ? bias[i] : nullptr, out, last ? 1 : 0, s);
            if (st != X3_OK) return st;
            in = out;
        }
        return X3_OK;
    }
    const size_t half = n_layers > 2 ? need / 2 : need;
    // Layer i's carry copy reads its input and overwrites carries[i], which layer i's kernel reads.
    // On the channels-last tensor-core engine it is a kernel of its own, launched as a programmatic
    // dependent of layer i's kernel: that kernel signals once its reads of the carry are done, the
    // copy runs beside the rest of it and waits for it before finishing, and layer i+1 (which may
    // overwrite the copy's source) waits for the copy in turn. Otherwise the copy is a
    // cudaMemcpy2DAsync on a side stream, forked after layer i's kernel, that runs beside the next
    // layers until a kernel is about to overwrite the buffer it reads (the ping-pong buffer layer i+1
    // writes when i >= 1); the caller's stream waits for every such copy before the call's work ends.
    auto dep_copy = [&](int i, const void* in, const void* carry) {
        const x3_conv_desc& d = plans[i]->d;
        return pdl_enabled() && plans[i]->kind == K_IGEMM_CL && d.layout == X3_NDHWC && aligned(in, 16) &&
               aligned(carry, 16);
    };
    SideStream* side = nullptr;
    bool any_side = false;
    {
        const void* in_i = x;
        for (int i = 0; i < n_layers; ++i) {
            const bool c = plans[i]->d.dims == 3 && carries && carries[i];
            any_side |= c && !dep_copy(i, in_i, carries[i]);
            in_i = (i == n_layers - 1) ? y : (char*)workspace + (size_t)(i % 2) * half;
        }
    }
    if (any_side) {
        x3_status st = side_stream(&side);
        if (st != X3_OK) return st;
    }
    int pending[2] = {-1, -1};  // per workspace half: the layer whose carry copy reads it, or -1
    int last_copy = -1;
    const void* in = x;
    for (int i = 0; i < n_layers; ++i) {
        const int ob = i % 2;
        void* out = (i == n_layers - 1) ? y : (char*)workspace + (size_t)ob * half;
        cudaError_t e = cudaSuccess;
        if (i < n_layers - 1 && pending[ob] >= 0) {
            e = cudaStreamWaitEvent(s, side->done[pending[ob] % SideStream::kEvents], 0);
            pending[ob] = -1;
        }
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "conv_stack_forward: %s", cudaGetErrorString(e));
        void* carry = (plans[i]->d.dims == 3 && carries) ? carries[i] : nullptr;
        x3_status st = conv_forward(plans[i], in, (carry && carry_valid) ? carry : nullptr, w_packed[i],
                                    bias ? bias[i] : nullptr, out, stream);
        if (st != X3_OK) return st;
        if (carry && dep_copy(i, in, carry)) {
            const x3_conv_desc& d = plans[i]->d;
            st = launch_carry_update(in, carry, d.N, d.D, (size_t)d.H * d.W * d.C_in * 2, carry_valid,
                                     plans[i]->num_sms, s);
            if (st != X3_OK) return st;
        } else if (carry) {
            const int k = i % SideStream::kEvents;
            e = cudaEventRecord(side->fork[k], s);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork[k], 0);
            if (e != cudaSuccess) return fail(X3_ERR_CUDA, "conv_stack_forward: %s", cudaGetErrorString(e));
            st = update_carry(plans[i], in, carry, carry_valid, side->s);
            if (st != X3_OK) return st;
            e = cudaEventRecord(side->done[k], side->s);
            if (e != cudaSuccess) return fail(X3_ERR_CUDA, "conv_stack_forward: %s", cudaGetErrorString(e));
            if (i >= 1) pending[(i - 1) % 2] = i;  // layer i's input is the half layer i-1 wrote
            last_copy = i;
        }
        in = out;
    }
    if (last_copy >= 0) {
        // copies run in order on the side stream: waiting for the last one covers all of them
        cudaError_t e = cudaStreamWaitEvent(s, side->done[last_copy % SideStream::kEvents], 0);
        if (e != cudaSuccess) return fail(X3_ERR_CUDA, "conv_stack_forward: %s", cudaGetErrorString(e));
    }
    return X3_OK;
}

x3_status conv_device_status(int reset) {
    clear_err();
    return read_device_status(reset);
}

x3_status conv_selftest_wait_timeout(int limit_ms, x3_stream_t stream) {
    clear_err();
    return selftest_wait_timeout(limit_ms, (cudaStream_t)stream);
}

const char* conv_last_error(void) { return g_err; }

const char* conv_version(void) { return "x3conv 0.1 (sm_103a)"; }

}  // extern "C"
