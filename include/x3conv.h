/*
 * x3conv.h - C ABI of the GB300 (sm_103a) 3x3 / causal 3x3x3 convolution library.
 *
 * The operation (what every entry point below computes):
 *
 *   2D, stride s in {1,2}, pad 1 (musetalk-bench patches/taesd_conv.cuh.new, header comment and
 *   taesd_conv3x3_impl):
 *     y[n,co,oh,ow] = R( act( b[co] + sum_{ci,kh,kw} w[co,ci,kh,kw] * x[n,ci,s*oh+kh-1,s*ow+kw-1] ) )
 *     with x = 0 outside the image, H_out = (H-1)/s + 1, W_out = (W-1)/s + 1.
 *
 *   3D causal, stride 1 (FastVideo fastvideo-kernel/wan22_vae_decode/solution/head.cu, header
 *   comment and head_stencil_kernel; the decoder's causal convolutions with two carried frames):
 *     xt = [carry[0], carry[1], x[0], ..., x[D-1]]   (carry absent = two zero frames)
 *     y[n,co,t,h,w] = R( act( b[co] + sum_{ci,kt,kh,kw} w[co,ci,kt,kh,kw] * xt[n,ci,t+kt,h+kh-1,w+kw-1] ) )
 *     for t in [0, D), spatial zero padding, no temporal padding besides the carry.
 *
 *   All products are accumulated in one fp32 accumulator per output, which starts at the bias;
 *   act is none, ReLU, or clamp to [-1,1]; R is one round-to-nearest-even to the storage type
 *   (f16 or bf16) at the store. Inputs, weights and biases are stored in the same 16-bit type.
 *
 * Conventions shared by every entry point:
 *   - Device pointers are plain CUDA device (or managed) addresses owned by the caller. The
 *     library never allocates, frees or retains device memory, except for one internal 4-byte
 *     device status word per device and the scratch array built in for
 *     conv_stack_forward_noalloc (X3_NOALLOC_SCRATCH_BYTES per device).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). All work is enqueued on it;
 *     nothing synchronises. Pointers must stay valid until the enqueued work has finished.
 *   - Functions return x3_status. On failure nothing was enqueued (for X3_ERR_INVALID and
 *     X3_ERR_UNSUPPORTED) and conv_last_error() describes the problem. The library never aborts
 *     the process and never traps on the device.
 *   - Every device-side wait in the library's kernels is bounded. A wait that runs out records
 *     X3_ERR_TIMEOUT in the device status word (read with conv_device_status) and the kernel
 *     returns early, leaving the context usable.
 *   - conv_stack_forward updates each layer's carry inside the call's work on `stream`. For layers
 *     on the channels-last tensor-core engine it is a small kernel launched as a programmatic
 *     dependent of the layer's kernel, which runs beside the layer once the layer has read the old
 *     carry and finishes after it. Otherwise it is a copy on a side stream of the library's own (one
 *     per calling thread and device, created on first use with eight events and kept until the
 *     process exits), joined back into `stream` with events before the call's work ends. Either
 *     way all of a call's work is ordered as work on `stream`, including under stream capture.
 *   - The tensor-core kernels launch as programmatic dependents of the previous kernel in `stream`:
 *     they set up shared memory and TMEM while that kernel drains and wait for it to finish before
 *     touching global memory. A kernel that reads a carry lets the next kernel start only after
 *     its last read of the carry.
 *
 * Environment switches (read when a plan is created; X3CONV_STACK_LAYOUT at each
 * conv_stack_forward call, X3CONV_PDL once per process). The results are the same under every
 * setting; only the kernels that compute them change:
 *   X3CONV_FORCE_KERNEL=direct|igemm  plans made with X3_KERNEL_AUTO use that engine
 *   X3CONV_FORCE_KERNEL=igemm_nsub    plans made with X3_KERNEL_AUTO skip the swapped-operand engine and
 *                                     use the positions-as-M tcgen05 engine ("igemm_tcgen05") where it
 *                                     applies, else the direct kernel
 *   X3CONV_TN=0                       2D channels-last layers with at most 64 output channels use the
 *                                     M = 64 form instead of the positions-as-M / horizontal-taps-in-N
 *                                     form (and X3CONV_TK=0 keeps 8-channel inputs off the taps-in-K form)
 *   X3CONV_STACK_LAYOUT=nchw          2D NCHW stacks run every layer in NCHW (no channels-last pass)
 *   X3CONV_S2=0                       stride 2 as the stride-1 raster with even positions kept,
 *                                     instead of the four input phases
 *   X3CONV_W2=1                       two-window tiles for causal channels-last layers
 *   X3CONV_FRAME_PAIRS=0              causal channels-last layers compute their output frames one after
 *                                     another instead of in adjacent pairs (the pairs read each shared
 *                                     input frame from DRAM once)
 *   X3CONV_PDL=0                      launches fully serialised (no programmatic dependent launch)
 */
#ifndef X3CONV_H
#define X3CONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* x3_stream_t; /* identical to cudaStream_t */

typedef enum {
    X3_OK = 0,
    X3_ERR_INVALID = 1,     /* bad argument: shape, pointer, alignment or combination */
    X3_ERR_UNSUPPORTED = 2, /* valid, but no kernel of the library handles it (caller falls back) */
    X3_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
    X3_ERR_OOM = 4,         /* a caller-provided buffer is too small */
    X3_ERR_TIMEOUT = 5      /* a bounded device wait ran out (see conv_device_status) */
} x3_status;

typedef enum {
    X3_NCHW = 0,   /* 2D: [N][C][H][W] */
    X3_NHWC = 1,   /* 2D: [N][H][W][C] */
    X3_NCDHW = 2,  /* 3D: [N][C][D][H][W] */
    X3_NDHWC = 3   /* 3D: [N][D][H][W][C] (channels-last) */
} x3_layout;

typedef enum { X3_F16 = 0, X3_BF16 = 1 } x3_dtype;

typedef enum { X3_ACT_NONE = 0, X3_ACT_RELU = 1, X3_ACT_CLAMP1 = 2 } x3_act;

typedef enum {
    X3_KERNEL_AUTO = 0,   /* pick the fastest kernel that handles the descriptor */
    X3_KERNEL_IGEMM = 1,  /* tcgen05/TMEM implicit GEMM (fails with X3_ERR_UNSUPPORTED if it can't) */
    X3_KERNEL_DIRECT = 2, /* plain SIMT direct convolution; handles every valid descriptor */
    X3_KERNEL_HEAD_TWO_PASS = 3, /* conv_out head as two passes (run with conv_head_two_pass): a temporal-
                                    only 3x1x1 convolution into a 108-channel bf16 plane g, then the nine
                                    spatial taps with bias and clamp (FastVideo wan22_vae_decode/solution/
                                    head.cu, header comment and head_stencil_kernel); needs
                                    unpatchify2x2, 3D, X3_NDHWC, bf16 */
    X3_KERNEL_HEAD_SPLIT = 4,    /* the same two passes with g kept in fp32: every product and partial sum
                                    is carried in fp32 as in the single-pass head, so integer-valued data
                                    give the exact result; same requirements */
    X3_KERNEL_HEAD_STENCIL = 5   /* the same arithmetic as HEAD_SPLIT in one kernel run by conv_forward:
                                    the temporal sums of all nine taps stay in fp32 in TMEM and the
                                    epilogue adds the nine spatial taps; same requirements. AUTO picks it
                                    for such heads; X3_KERNEL_IGEMM gives the single-pass form (kw
                                    folded into M, one accumulator over all 27 taps) */
} x3_kernel;

/* Descriptor of one convolution layer. */
typedef struct {
    int dims;          /* 2 or 3 */
    int N;             /* batch, >= 1 */
    int C_in, C_out;   /* >= 1 each; C_out == 12 when unpatchify2x2 is set */
    int D;             /* 3D: output frames per call (input has D frames plus 2 carried); 2D: 1 */
    int H, W;          /* input height and width, >= 1 */
    int stride;        /* 1 or 2 (2D); 1 (3D) */
    x3_layout layout;  /* input and output layout: X3_NCHW/X3_NHWC for 2D, X3_NCDHW/X3_NDHWC for 3D */
    x3_dtype dtype;    /* storage type of x, carry, weights, bias and y */
    x3_act act;        /* epilogue activation */
    int has_bias;      /* 1: bias pointer required; 0: no bias */
    int unpatchify2x2; /* head only (C_out == 12): write y as RGB at twice the resolution, channel
                          c = rgb*4 + dy*2 + dx going to pixel (2h+dy, 2w+dx); the output is then
                          [N][D][2H][2W][3] for X3_NDHWC and [N][3][D][2H][2W] for X3_NCDHW
                          (2D: [N][2H][2W][3] / [N][3][2H][2W]) */
    x3_kernel kernel;  /* kernel choice (X3_KERNEL_AUTO normally) */
    /* Banded (row-band) mode, stride 1 only; all three 0 = the whole plane. The layer computes output
       rows [band_lo, band_lo + band_rows) of an image H_global rows high (FastVideo head.cu page,
       head_stencil_kernel and its wrapper: a band of the output plane with its own row offset and the
       global height). The input (and each carried frame) then holds the global rows
       [max(band_lo - 1, 0), min(band_lo + band_rows + 1, H_global)): the band's rows plus the halo
       row above and below wherever that global row exists, so H must equal that count; zero padding
       applies only at the global edges (rows -1 and H_global). The output holds band_rows rows.
       A descriptor whose H misses a halo row that exists globally is rejected with X3_ERR_INVALID
       (the page's kernel silently skips such rows instead). Bands of one plane, each with its halo,
       give, concatenated, the whole plane's output bit for bit. Not for conv_stack_forward (each
       layer's band needs its neighbours' rows: exchange them between layers) nor for the two-pass
       head kernels. */
    int band_lo, band_rows, H_global;
} x3_conv_desc;

typedef struct x3_conv_plan x3_conv_plan; /* opaque; host memory only */

/*
 * Validate a descriptor and build a plan (tiling, kernel choice, launch shapes).
 * Host only: launches nothing and touches no device memory. The caller owns *plan and releases
 * it with conv_plan_destroy. Errors: X3_ERR_INVALID (bad descriptor or NULL pointer),
 * X3_ERR_UNSUPPORTED (a forced kernel that can't handle it).
 */
x3_status conv_plan_create(const x3_conv_desc* desc, x3_conv_plan** plan);

/* Release a plan (NULL is ignored). */
void conv_plan_destroy(x3_conv_plan* plan);

/* Name of the kernel the plan runs, for logs and tests: "igemm_tcgen05_sw128" (swapped-operand
 * tcgen05 engine, channels-last, including its positions-as-M forms for low-channel 2D layers),
 * "igemm_tcgen05_sw128_head" (its single-pass conv_out head form), "igemm_tcgen05_sw128_head_stencil"
 * (the one-kernel stencil head), "igemm_tcgen05_sw128_nchw" (its NCHW form), "igemm_tcgen05"
 * (positions-as-M tcgen05 engine), "direct_simt", "head_two_pass" / "head_split" (run with
 * conv_head_two_pass). */
const char* conv_plan_kernel_name(const x3_conv_plan* plan);

/*
 * Write a one-line JSON description of the plan (kernel, tiling, pipeline depths, shared memory,
 * grid) into buf (at most len bytes including the terminating NUL). Returns the length the full
 * description needs (excluding the NUL), like snprintf.
 */
int conv_plan_describe(const x3_conv_plan* plan, char* buf, size_t len);

/* Number of kernel launches one conv_forward with this plan enqueues (a two-pass head plan runs
 * with conv_head_two_pass, which enqueues two). */
int conv_plan_launches(const x3_conv_plan* plan);

/* Bytes of the packed-weight buffer conv_pack_weights fills for this plan. */
size_t conv_packed_weight_bytes(const x3_conv_plan* plan);

/*
 * Repack canonical weights w[C_out][C_in][(3)][3][3] (PyTorch's Conv2d/Conv3d layout, storage
 * dtype) into the plan's kernel layout in w_packed (conv_packed_weight_bytes bytes, 256-byte
 * aligned, caller-owned). Done once per set of weights; conv_forward then reads only w_packed.
 * Errors: X3_ERR_INVALID (NULL or misaligned pointer), X3_ERR_CUDA.
 */
x3_status conv_pack_weights(const x3_conv_plan* plan, const void* w, void* w_packed,
                            x3_stream_t stream);

/*
 * One convolution: y = conv(x [, carry]) with the fused bias / activation / rounding epilogue.
 *   x:        input, layout and dtype of the plan; 16-byte aligned.
 *   carry:    3D only: the two frames that precede x in time, same layout as x with 2 frames
 *             ([N][2][H][W][C] or [N][C][2][H][W]); NULL = two zero frames. Ignored in 2D.
 *   w_packed: from conv_pack_weights with the same plan.
 *   bias:     C_out values (storage dtype) when has_bias, else ignored.
 *   y:        output (D frames); must not overlap x, carry or w_packed; 16-byte aligned.
 * Errors: X3_ERR_INVALID (NULL or misaligned pointer), X3_ERR_CUDA (launch failure).
 */
x3_status conv_forward(const x3_conv_plan* plan, const void* x, const void* carry,
                       const void* w_packed, const void* bias, void* y, x3_stream_t stream);

/*
 * The conv_out head computed as the head.cu page's two passes, for a plan made with
 * kernel = X3_KERNEL_HEAD_TWO_PASS or X3_KERNEL_HEAD_SPLIT (weights packed by conv_pack_weights with
 * that plan):
 *   pass 1: G[n,t,p,h,w,c] = sum_{ci,kt} w[c,ci,kt,i,j] * xt[n,ci,t+kt,h,w] for the nine spatial taps
 *           p = i*3+j: a temporal-only convolution on the tensor cores, one fp32 accumulator per value,
 *           stored as bf16 (HEAD_TWO_PASS, rounded once) or fp32 (HEAD_SPLIT);
 *   pass 2: y = bf16( clamp( b[c] + sum_{i,j} G[n,t,i*3+j,h+i-1,w+j-1,c] ) ) with the zero padding,
 *           summed in fp32 in (i, j) order, written as unpatchified RGB like conv_forward's head output.
 * The early bf16 rounding of G is the page's value path; it differs from conv_forward's single
 * accumulator over all 27 taps by a few bf16 ulps of the partial sums (max|d| moves, rms does not).
 * With fp32 G the two passes differ from the single pass only in the order of the fp32 additions.
 *   g: caller buffer of conv_head_g_bytes(plan) bytes, 16-byte aligned, layout [N][D][9][H][W][12] of
 *      bf16 or fp32 (each tap's 12 channels contiguous per position, one plane per tap).
 * Errors: X3_ERR_INVALID (wrong plan kind, NULL or misaligned pointers), X3_ERR_CUDA.
 */
size_t conv_head_g_bytes(const x3_conv_plan* plan);
x3_status conv_head_two_pass(const x3_conv_plan* plan, const void* x, const void* carry, const void* w_packed,
                             const void* bias, void* g, void* y, x3_stream_t stream);

/*
 * Workspace bytes conv_stack_forward needs for these layers: two ping-pong buffers, each the size
 * of the largest intermediate activation (every intermediate is dead as soon as the next layer
 * has read it), or, for a stack of 2D NCHW layers run channels-last between the layers, of the
 * largest of those and of the first layer's input converted to channels-last (C_in rounded up to
 * a multiple of 8). Returns 0 for an invalid stack.
 */
size_t conv_stack_workspace_bytes(const x3_conv_plan* const* plans, int n_layers);

/*
 * Run n_layers chained layers: layer i reads layer i-1's output (layer 0 reads x), the last layer
 * writes y. Consecutive plans must agree: C_out[i] == C_in[i+1], output size of i == input size of
 * i+1, same dims, N, D, layout and dtype, and no unpatchify except on the last layer. A stack of
 * 2D NCHW layers (each with C_out a multiple of 8, the last of stride 1) keeps its activations
 * channels-last between the layers (x and y stay NCHW; X3CONV_STACK_LAYOUT=nchw in the environment
 * runs every layer in NCHW instead); the values are the same.
 *   carries:     3D only; carries[i] is layer i's two-frame history buffer (layout of its input,
 *                2 frames). It is read as the frames preceding this pass (as zeros when
 *                carry_valid is 0) and then overwritten with the last two frames of the layer's
 *                input sequence [history, input], i.e. the history of the next pass. NULL
 *                (the array or an entry) = zero history and no carry written.
 *   carry_valid: 0 on the first pass of a sequence, 1 afterwards.
 *   w_packed[i], bias[i]: as for conv_forward with plans[i].
 *   workspace:   >= conv_stack_workspace_bytes(plans, n_layers) bytes, 256-byte aligned.
 * Errors: X3_ERR_INVALID (n_layers < 1, mismatched layers, NULL pointers), X3_ERR_OOM (workspace
 * too small), X3_ERR_CUDA.
 */
x3_status conv_stack_forward(const x3_conv_plan* const* plans, int n_layers, const void* x,
                             void* const* carries, int carry_valid, const void* const* w_packed,
                             const void* const* bias, void* y, void* workspace,
                             size_t workspace_bytes, x3_stream_t stream);

/*
 * Size of the scratch buffer built into the library for conv_stack_forward_noalloc: 32 MiB of
 * device memory, held on every GPU that loads the library until the process exits.
 */
#define X3_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * conv_stack_forward without a workspace argument, for callers that must not allocate device
 * memory (a plug-in inside a framework that owns every allocation, a pipeline that forbids
 * allocation after start-up, a caller whose memory is fully reserved by its own pool). The
 * pages have no counterpart of this entry point; it is an addition of this library.
 *
 * Arguments and results are those of conv_stack_forward; the caller still provides inputs,
 * outputs, carries and packed weights. The intermediate activations live in the library's own
 * X3_NOALLOC_SCRATCH_BYTES device buffer instead of a caller workspace, and this function calls
 * no device-memory allocator (no cudaMalloc, cudaFree or allocating library routine).
 *   - Stacks whose conv_stack_workspace_bytes exceeds X3_NOALLOC_SCRATCH_BYTES are rejected with
 *     X3_ERR_OOM before anything is enqueued.
 *   - The first call on a device (with that device current) looks up the buffer's device address,
 *     and so does the first call after the device's context changed (a cudaDeviceReset, or another
 *     context made current); make such a first call before capturing any stream.
 *   - Like conv_stack_forward, the first call on a calling thread and device whose stack needs the
 *     side stream for carry copies (3D NCDHW layers, or X3CONV_PDL=0) creates that stream and its
 *     eight events, which reserves driver resources but no device memory of the caller's; make it
 *     before any capture or allocation-free phase as well.
 *   - All calls on a device share the one buffer and it keeps the last call's contents (each
 *     layer overwrites every intermediate value it produces, so nothing needs clearing). Calls
 *     whose work overlaps on the GPU - on different streams, or from different threads - race on
 *     it: serialise them.
 */
x3_status conv_stack_forward_noalloc(const x3_conv_plan* const* plans, int n_layers, const void* x,
                                     void* const* carries, int carry_valid, const void* const* w_packed,
                                     const void* const* bias, void* y, x3_stream_t stream);

/*
 * Read (and with reset != 0, clear) the current device's status word: X3_OK, or X3_ERR_TIMEOUT
 * when a bounded device wait ran out since the last reset. Synchronises the device.
 */
x3_status conv_device_status(int reset);

/*
 * Self-test of the bounded-wait path: launches one small kernel whose single thread waits on a
 * shared-memory mbarrier that nothing ever arrives at, with a limit of `limit_ms` milliseconds
 * (1..2000), using the same bounded wait as the convolution kernels. When the limit runs out the
 * kernel records X3_ERR_TIMEOUT in the device status word and returns; conv_device_status then
 * reports it and the context stays usable. Errors: X3_ERR_INVALID (limit out of range),
 * X3_ERR_CUDA (launch failure).
 */
x3_status conv_selftest_wait_timeout(int limit_ms, x3_stream_t stream);

/* Thread-local description of the last error returned on this thread ("" if none). */
const char* conv_last_error(void);

/* Library version string. */
const char* conv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* X3CONV_H */
