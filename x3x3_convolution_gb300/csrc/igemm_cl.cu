// Channels-last tcgen05 implicit-GEMM engine with output channels as M and positions as N.
//
// The causal 3x3x3 convolution of FastVideo wan22_vae_decode/solution/head.cu (bf16 storage, fp32
// accumulation of all 27 taps, bias, one rounding at the store) and the 2D 3x3 convolution of the
// TAESD conv page, for channels-last layers (and, in the NCHW form, NCHW 2D layers). Each MMA is
// tcgen05.mma kind::f16 with
//   A = packed weights  (M = 128 output channels x K = 16 input channels, K-major, no swizzle;
//                        M = 64 in the form for at most 64 output channels),
//   B = input halo      (N = 256 output positions x K = 16 input channels, K-major, 128-byte swizzle),
//   D = fp32 accumulator in TMEM (128 lanes = channels x 256 columns = positions).
// Why this arrangement: with N = 256 each MMA reads 12 KB of operands for 1 MFLOP instead of the
// 8 KB per 0.5 MFLOP of a 128x128 tile, which keeps the tensor core's shared-memory operand reads
// below the SM's shared-memory bandwidth and leaves room for the TMA writes of the next stages.
// Measured on GB300: ~165 cycles per MMA when consecutive taps re-read shifted rows of one staged
// halo, ~270 when both operands are fresh (the centre-tap form), ~104 for a second MMA on the same A.
//
// Tiling. The output plane is cut into vertical strips Wt columns wide; each strip is walked as a
// raster of pitch P = Wt + 2 (two junk columns per row), and a tile is a window of 256 consecutive
// raster positions of one frame. Its halo (the rows the window touches plus one above and below,
// P positions each, 64 channels per stage) is staged once per (temporal tap, 64-channel chunk) by
// one TMA box with the 128-byte swizzle: every position is one 128-byte row, so the nine spatial
// taps are nine row offsets (kh*P + kw) of the same staged halo and every such offset reads
// conflict-free. Out-of-image boxes are zero-filled by the TMA unit (the zero padding); missing
// carried frames are read at an out-of-range frame coordinate (zeros).
//
// Roles (one persistent CTA per SM): warp 0 issues the TMA loads (halo) and bulk copies (weights),
// warp 1 owns TMEM and one thread issues the MMAs, warps 2-5 drain TMEM (two accumulator buffers,
// so the epilogue of one tile overlaps the MMAs of the next), add the bias, apply the activation,
// round once and write channels-last rows through a shared-memory transpose (the NCHW form adds
// four transposer warps). Every wait is bounded (1 s); a wait that runs out sets the device status
// word and every role gives up cleanly. The MMA issuer is a single thread whose own instruction
// stream measurably gates the tensor pipe, so its loop keeps ring positions as wrapping counters
// (no division per weight block) and issues a full block's four K steps as one group. The forms
// (head, NCHW, centre tap, stencil head, M = 64, stride-2 phases, two windows) are
// described at the kernel template below.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace x3 {

namespace {

constexpr int kSmemLimit = 232448;
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr int kBM = 128;        // output channels per tile (MMA M)
constexpr int kBNP = 256;       // positions per tile (MMA N)
constexpr int kCK = 64;         // input channels per staged chunk (one 128-byte swizzle row)
constexpr int kWBlock = kBM * kCK * 2;  // bytes of one packed weight block (one tap, one chunk)
constexpr int kWBlock64 = 64 * kCK * 2; // the same for the M = 64 form
constexpr int kCtrW = kBNP * kCK * 2;    // centre-tap form: offset of the weight block in a stage
// generic epilogue staging row: 32 channels (64 B), no pad: a store of one row spans 64 contiguous
// bytes and a 16-byte load phase reads 8 whole rows (512 contiguous bytes), both free of conflicts
constexpr int kStagePitch = 64;
constexpr int kStageGenericBytes = 32 * kStagePitch;  // per-warp staging block of the generic epilogue
constexpr int kSPitch = 35;       // head form: fp32 staging row (34 columns + pad) per TMEM lane
constexpr int kGPitch = 36;       // centre-tap form: fp32 staging row (32 accumulator rows + pad) per position
constexpr int kStageWarpBytes = 32 * kGPitch * 4;  // per-warp staging block (every form but STN)
constexpr int kStnRows = 8;       // STN: rows of a window (32 positions each: 30 output columns and 2 halo)
constexpr int kStnPitch = 33;     // STN: fp32 staging row (one 32-position window row + pad) per tap row
constexpr int kStnStageBytes = 27 * kStnPitch * 4;  // 27 rows: 9 taps x 3 channels
constexpr int kStnCarryBytes = 2 * 3 * 32 * 4;      // STN: per warp and output frame, two pending rows of 3 channels

// Division by a run-time constant d without a division instruction: for 0 <= x < 2^31,
// x / d == (x * m) >> s with l = ceil(log2 d), s = 31 + l and m = ceil(2^s / d) < 2^32 (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994: the error of m is below d,
// so x * (m * d - 2^s) < 2^s and the floor is exact). Every role of the kernel decodes every tile, and
// on the MMA issuer's single thread a run-time integer division costs hundreds of cycles.
struct FastDiv {
    uint32_t d, m, s;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    uint32_t l = 0;
    while (l < 31 && (1u << l) < d) ++l;
    f.d = d;
    f.s = 31 + l;
    f.m = (uint32_t)(((1ull << f.s) + d - 1) / d);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t x, const FastDiv& f) {
    return (uint32_t)(((uint64_t)x * f.m) >> f.s);
}

struct ClArgs {
    int C_in, C_out, N, D, H, W, H_out, W_out, dout, act, has_carry;
    int KT, n_chunks, n_tiles, Wt, P, HR, strips, windows, frames;
    int h_bytes, h_tx_bytes, n_h, n_w;
    int win_adv;     // raster positions between consecutive windows (256, or 254 when kw is folded into M)
    int raw_w, raw_bytes, raw_tx_bytes, n_raw;  // NCHW: raw tile columns, stage bytes, TMA bytes, stages
    int ngroups;     // kw folded into M: channel groups (10 channels x 3 kw per TMEM lane quarter)
    int sub2;        // 1: stride 2 as the stride-1 raster with only even (oh, ow) stored at (oh/2, ow/2)
    int out_nchw;    // 1: channels-last input, NCHW output (the NCHW epilogue)
    int yH, yW;      // stored output plane (H_out x W_out, or halved when sub2)
    int w_smem;      // bytes of shared memory for weight blocks (n_w stages, or all blocks when resident)
    int frame_inner; // tile order: 1 = output frame fastest; 2 = frame pairs (frame within a pair fastest)
    int g_f32;       // centre-tap form: the tap planes of G in fp32 (else bf16)
    int stage_warp;  // epilogue staging bytes per warp
    int tn_cp, tn_n; // TN: output channels padded to 16, MMA N (3 horizontal taps x tn_cp)
    int x_bytes;     // TN: bytes after the staging blocks (the epilogue warps' bias copies)
    int tn_tma;      // TN: each warp writes its raster row (64 channels) with one TMA store (tm_y)
    int row_shift;   // banded mode: the input's first row is the band's upper halo row
    int stn_n;       // STN: windows per run (run blockIdx.x / stn_groups starts at stn_start[run])
    int stn_fpc;     // STN: output frames per CTA (frame group blockIdx.x % stn_groups)
    int stn_full;    // STN: whole segments per run before its share of the rest (run r: r, r + runs, ...)
    int stn_runs;    // STN: runs side by side in the rounds of whole segments
    int stn_nseg, stn_seg_rows;  // STN: segments (strip-fastest: part p of strip s is p * strips + s), rows each
    long long tiles;
    FastDiv fd_frames, fd_ntiles, fd_windows, fd_strips, fd_dout, fd_P, fd_chunks;
    FastDiv fd_fpc, fd_groups;  // STN
    uint32_t idesc;
    const uint8_t* w;
    const void* bias;
    void* y;
    unsigned int* status;  // the library's device status word
    uint32_t stn_start[kStnMaxCtas];
};

struct ClTile {
    int nt, win, strip, fr;
    int grow;   // STN: input row of the window's first row
    int fslot;  // STN: the frame's place in this CTA's frame group
    int rend;   // STN: end of the window's row segment (its last window computes rows past it: not stored)
};

// The planner keeps tile counts below 2^31, so the decode runs in 32-bit unsigned arithmetic (a 64-bit
// division is a long software sequence, and every role of the kernel decodes every tile).
__device__ __forceinline__ ClTile cl_decode(const ClArgs& a, long long tile) {
    ClTile c;
    uint32_t t = (uint32_t)tile;
    uint32_t q;
    if (a.frame_inner == 2) {
        // output frames in adjacent pairs (0,1), (2,3), ... of a pass: the two frames of a pair are
        // computed together, so the two input frames they share are read from DRAM once and then
        // hit in L2, while every tile that reads the carried frames (frames 0 and 1) still comes in
        // the first pairs
        const uint32_t fi = t & 1u;
        t >>= 1;
        q = fdiv(t, a.fd_ntiles);
        c.nt = (int)(t - q * a.fd_ntiles.d);
        t = q;
        q = fdiv(t, a.fd_windows);
        c.win = (int)(t - q * a.fd_windows.d);
        t = q;
        q = fdiv(t, a.fd_strips);
        c.strip = (int)(t - q * a.fd_strips.d);
        c.fr = (int)(2 * q + fi);
        return c;
    }
    if (a.frame_inner) {
        // frames fastest: the output frames of one window are in flight together, so the input frames
        // they share (three temporal taps each) are read from DRAM once and then hit in L2
        q = fdiv(t, a.fd_frames);
        c.fr = (int)(t - q * a.fd_frames.d);
        t = q;
        q = fdiv(t, a.fd_ntiles);
        c.nt = (int)(t - q * a.fd_ntiles.d);
        t = q;
        q = fdiv(t, a.fd_windows);
        c.win = (int)(t - q * a.fd_windows.d);
        c.strip = (int)q;
        return c;
    }
    q = fdiv(t, a.fd_ntiles);
    c.nt = (int)(t - q * a.fd_ntiles.d);
    t = q;
    q = fdiv(t, a.fd_windows);
    c.win = (int)(t - q * a.fd_windows.d);
    t = q;
    q = fdiv(t, a.fd_strips);
    c.strip = (int)(t - q * a.fd_strips.d);
    c.fr = (int)q;
    return c;
}

// Stencil head: the k-th tile of this CTA, false past its last. The output frames are split into
// groups of stn_fpc frames, and the CTAs c of one run (c / groups the same) take the groups c % groups
// side by side, so that the frames reading the same input frames are computed at the same time and
// share them through L2. Each strip is cut into row segments (part p of strip s is segment
// p * strips + s, stn_seg_rows output rows). A CTA runs its windows one after another, the frames of
// its group fastest, first through stn_full whole segments (run r takes segments r, r + runs, ..., so
// that at any moment the runs are on the same rows of neighbouring strips and the halo columns two
// strips share are read from DRAM once), then from its start in the remaining segments (segment,
// first output row o0) down that segment and on through the following ones. The windows of one
// segment in one run do not overlap: window b covers input rows o0 - 1 + 8 b to o0 + 6 + 8 b, and the
// two output rows centred on the seam between windows b and b + 1 take their first kernel rows from
// sums the epilogue carries over from window b. A piece of nb windows so yields output rows
// o0 .. o0 + 8 nb - 3 (the next piece starts at o0 + 8 nb - 2 and re-reads the two rows above).
__device__ __forceinline__ void stn_segment(const ClArgs& a, int sg, int& strip, int& lo, int& hi) {
    const int part = (int)fdiv((uint32_t)sg, a.fd_strips);
    strip = sg - part * a.strips;
    lo = part * a.stn_seg_rows;
    hi = lo + a.stn_seg_rows < a.H_out ? lo + a.stn_seg_rows : a.H_out;
}

__device__ __forceinline__ bool stn_decode(const ClArgs& a, long long k, ClTile& c) {
    const uint32_t kk = (uint32_t)k;
    const uint32_t w = fdiv(kk, a.fd_fpc);
    if ((int)w >= a.stn_n) return false;
    const uint32_t run = fdiv(blockIdx.x, a.fd_groups);
    const uint32_t grp = blockIdx.x - run * a.fd_groups.d;
    int s = 0, lo = 0, hi = 0, b = (int)w, o = -1;
    for (int j = 0; j < a.stn_full; ++j) {
        stn_segment(a, (int)run + j * a.stn_runs, s, lo, hi);
        const int nwin = (hi - lo + 9) >> 3;
        if (b < nwin) {
            o = lo;
            break;
        }
        b -= nwin;
    }
    if (o < 0) {
        const uint32_t st = a.stn_start[run];
        int sg = (int)(st >> 16);
        o = (int)(st & 0xFFFFu);
        for (;;) {
            if (sg >= a.stn_nseg) return false;
            stn_segment(a, sg, s, lo, hi);
            if (o < lo) o = lo;
            const int need = (hi - o + 9) >> 3;  // windows that finish the segment from row o
            if (b < need) break;
            b -= need;
            ++sg;
            o = 0;
        }
    }
    c.nt = 0;
    c.fslot = (int)(kk - w * a.fd_fpc.d);
    c.fr = (int)(grp * a.fd_fpc.d) + c.fslot;
    c.strip = s;
    c.win = b;
    c.grow = o - 1 + kStnRows * b;
    c.rend = hi;
    return true;
}

// Position in a ring of n stages: the stage index and the parity of its current phase, advanced
// without a division (the MMA issuer takes one per weight block).
struct RingPos {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void next(uint32_t n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// Tile of this (persistent) CTA at iteration k.
__device__ __forceinline__ long long cl_tile_of(long long k) { return (long long)blockIdx.x + k * gridDim.x; }

__device__ __forceinline__ bool cl_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned int* status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((++spins & 63u) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > kWaitNs) {
                *abort_flag = 1;
                atomicOr(status, 1u);
                return false;
            }
        }
    }
}

// Stride 2: the taps that read input phase ph = 2a + b (a: odd input rows, b: odd input columns) and
// their shifts in the phase's raster. Output row oh reads input rows 2oh - 1 + kh: kh = 0 and 2 are
// odd rows (phase rows oh - 1 and oh), kh = 1 the even row oh; the phase raster starts one row and
// one column before the output window, so the shift is 0 for kh = 0 and 1 otherwise (same for kw).
__device__ __forceinline__ int s2_ntaps(int ph) { return ((ph >> 1) ? 2 : 1) * ((ph & 1) ? 2 : 1); }
__device__ __forceinline__ void s2_tap(int ph, int i, int& kh, int& kw) {
    const int ih = (ph & 1) ? i >> 1 : i, iw = (ph & 1) ? i & 1 : 0;  // two column taps when b = 1
    kh = (ph >> 1) ? 2 * ih : 1;
    kw = (ph & 1) ? 2 * iw : 1;
}

__device__ __forceinline__ float cl_act(float v, int act) {
    if (act == X3_ACT_RELU) return fmaxf(v, 0.0f);
    if (act == X3_ACT_CLAMP1) return fminf(1.0f, fmaxf(-1.0f, v));
    return v;
}

template <bool BF16>
__device__ __forceinline__ uint16_t cl_round(float v) {
    if (BF16) {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        return *reinterpret_cast<uint16_t*>(&h);
    } else {
        __half h = __float2half_rn(v);
        return *reinterpret_cast<uint16_t*>(&h);
    }
}

// Two values rounded to the storage type and packed, the first in the low half.
template <bool BF16>
__device__ __forceinline__ uint32_t cl_pack2(float lo, float hi) {
    if (BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// A packed pair of storage-type values clamped to [lo, hi] (packed bounds). Applied after rounding it
// gives what the clamp before rounding gives: the rounding is monotonic and the bounds in use (0, -1,
// 1, -inf, inf) are representable.
template <bool BF16>
__device__ __forceinline__ uint32_t cl_clamp2(uint32_t v, uint32_t lo, uint32_t hi) {
    if (BF16) {
        const __nv_bfloat162 r = __hmin2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v),
                                                 *reinterpret_cast<const __nv_bfloat162*>(&lo)),
                                         *reinterpret_cast<const __nv_bfloat162*>(&hi));
        return *reinterpret_cast<const uint32_t*>(&r);
    } else {
        const __half2 r = __hmin2(__hmax2(*reinterpret_cast<const __half2*>(&v), *reinterpret_cast<const __half2*>(&lo)),
                                  *reinterpret_cast<const __half2*>(&hi));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
}

// KWM (the conv_out head form): the MMA's M rows are (kw, output channel) triples, quarter g of the
// 128 TMEM lanes holding kw*10 + r for channel 10g + r, so one MMA covers the three horizontal taps
// of a row of the window and the K loop runs over (kt, kh, channel) only; the epilogue adds the three
// kw partial sums with their one- and two-column shifts, all inside one warp's lane quarter.
// NC (NCHW 2D input and output): the producer loads raw [16 channels][HR rows][Wt+16 columns] tiles,
// four transposer warps (6-9) turn them into the swizzled position rows with ldmatrix.trans /
// stmatrix (shifting the halo by one column on the way), and the epilogue writes NCHW planes.
// CTR (the temporal pass of the two-pass head): only the centre spatial tap, one weight block per
// (kt, chunk). Each form is its own instantiation so the MMA issuer's loops keep constant bounds.
// M64 (layers with at most 64 output channels): MMAs of M = 64, whose accumulator rows 16q..16q+15
// sit in TMEM lanes 32q..32q+15; every weight block of the layer stays resident in shared memory
// (loaded once per CTA), so a tile only streams its halo.
// W2 (channels-last, one output tile; opt-in): a tile is two consecutive 256-position windows whose
// halo is staged by one box; each weight K slice feeds an MMA for the first window and then one for
// the second, which re-uses the A operand it just fetched, the two accumulators filling all 512 TMEM
// columns (so the epilogue no longer overlaps the MMAs).
// STN (with CTR; the conv_out head in one pass): the centre-tap MMAs over 32 x 8 raster windows (one
// halo column on each side of 30 output columns) that abut down a strip segment (stn_decode), M rows
// 32q + 9cl + tap for channel 3q + cl, so each epilogue warp holds all nine taps of its three channels;
// the epilogue streams the window's rows through shared memory and adds, in fp32, the bias and the
// nine taps' values at the shifted positions into the output rows pending in registers, then clamps,
// rounds once and writes the unpatchified RGB pixels.
// S2 (2D channels-last, stride 2): the raster is the output plane (pitch Wt + 1) and the input is
// staged as its four phases, even or odd rows by even or odd columns, each box loaded by the TMA
// unit with element strides of 2. A phase is one pipeline group that feeds only the taps reading it
// (one, two, two and four of the nine), each at a shift of 0 or 1 row and column (s2_tap).
// TN (2D channels-last, stride 1, at most 80 output channels): the operands the other way round, with
// the three horizontal taps in N. A = 128 consecutive raster positions of the staged halo (M = 128,
// 128-byte swizzle), B = the weights of one kernel row kh for all three kw, N = 3 x C_out rows
// (kw, output channel), resident in shared memory. One MMA per (kh, K step) leaves in TMEM
// D[i][(kw, co)] = sum_kh w[co, kh, kw] . x[halo position i + kh P], i.e. the kw tap's contribution to
// output position i - kw, so the epilogue forms out[j] = D[j][(0,co)] + D[j+1][(1,co)] + D[j+2][(2,co)].
// The raster pitch is 32 (30 output columns and the two junk columns per strip row) and a tile is four
// whole raster rows, so TMEM lane quarter q (epilogue warp q) holds exactly raster row q of the tile:
// the j+1 and j+2 terms are shuffles down by one and two lanes inside the warp, and the two lanes that
// would reach into the next row are the junk columns. Every MMA row is an output position (or one of
// the two junk columns), where the M = 64 form leaves half of the tensor core's rows empty; three MMAs
// per 16 input channels instead of nine.
// TK (with TN; 2D channels-last layers with 8 input channels, the first layer of an NCHW stack): the
// taps go into K instead, two per 16-wide K step. The halo is staged unswizzled with 16 bytes (8
// channels) per position, and the A descriptor of K step s starts at tap 2s's rows with its
// leading-dimension byte offset (the K-half stride) set to the distance to tap 2s+1's rows, so one MMA
// reads both taps' channels for 128 positions; five MMAs (the ninth tap paired with zero weights) of
// N = C_out leave out[j] directly in TMEM, and the epilogue needs no shifts.
template <bool BF16, bool KWM, bool NC, bool CTR = false, bool M64 = false, bool W2 = false,
          bool STN = false, bool S2 = false, bool TN = false, bool TK = false>
__global__ void __launch_bounds__((NC || TN) ? 320 : 192, 1)
    igemm_cl_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c,
                    const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ ClArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 bytes
    uint8_t* sbase = smem_raw + (base - raw_base);
    const uint32_t sH = base;                                      // halo stages (1024-aligned)
    const uint32_t sW = sH + (uint32_t)(a.n_h * a.h_bytes);        // weight blocks
    const uint32_t sStage = sW + (uint32_t)a.w_smem;               // epilogue transpose tile
    constexpr int kEpiWarps = TN ? 8 : 4;  // TN: two groups of four epilogue warps, taking alternate tiles
    const uint32_t sBiasT = sStage + (uint32_t)kEpiWarps * (uint32_t)a.stage_warp;  // TN: each epilogue warp's bias copy
    const uint32_t sRaw = sBiasT + (uint32_t)a.x_bytes;                      // NCHW raw tiles (128-aligned)
    const uint32_t sJunk = sRaw + (uint32_t)(a.n_raw * a.raw_bytes);         // NCHW: 16 B per transposer lane
    const uint32_t sBar = sJunk + (NC ? 4u * 32u * 16u : 0u);
    const uint32_t bar_h_full = sBar;
    const uint32_t bar_h_empty = bar_h_full + 8u * a.n_h;
    const uint32_t bar_w_full = bar_h_empty + 8u * a.n_h;
    const uint32_t bar_w_empty = bar_w_full + 8u * a.n_w;
    const uint32_t bar_acc_full = bar_w_empty + 8u * a.n_w;
    const uint32_t bar_acc_empty = bar_acc_full + 16u;
    const uint32_t bar_drain = bar_acc_empty + 16u;
    const uint32_t bar_r_full = bar_drain + 8u;
    const uint32_t bar_r_empty = bar_r_full + 8u * a.n_raw;
    const uint32_t s_tmem = bar_r_empty + 8u * a.n_raw;
    const uint32_t s_abort = s_tmem + 4u;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + (s_abort - base));
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sbase + (s_tmem - base));
    uint8_t* stage_ptr = sbase + (sStage - base);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.n_h; ++i) {
            ptx::mbar_init(bar_h_full + 8 * i, NC ? 4 : 1);  // NCHW: one arrival per transposer warp
            ptx::mbar_init(bar_h_empty + 8 * i, 1);
        }
        for (int i = 0; i < a.n_raw; ++i) {
            ptx::mbar_init(bar_r_full + 8 * i, 1);
            ptx::mbar_init(bar_r_empty + 8 * i, 4);
        }
        for (int i = 0; i < a.n_w; ++i) {
            ptx::mbar_init(bar_w_full + 8 * i, 1);
            ptx::mbar_init(bar_w_empty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar_acc_full + 8 * i, 1);
            ptx::mbar_init(bar_acc_empty + 8 * i, 4);  // the four warps that drain the buffer
        }
        ptx::mbar_init(bar_drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_x);
        ptx::prefetch_tmap(&tm_c);
        if (TN && a.tn_tma) ptx::prefetch_tmap(&tm_y);
    }
    if (warp == 1) {
        ptx::tmem_alloc(s_tmem, 512u);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // Launched as a programmatic dependent, this grid may start while the previous kernel of the
    // stream is still running: the set-up above (barriers, TMEM) overlaps its tail, and nothing of
    // global memory is read or written before the wait. The next kernel may then be scheduled; it
    // waits in the same way before it touches this one's output. With a carry, the next kernel may
    // be the copy that overwrites it, so the MMA issuer signals only once every read of the carry
    // by this CTA has landed in shared memory (one signal per CTA counts; the first one).
    // Resident weights (M = 64, TN and TK forms) are loaded before that wait: the packed weights are
    // written by the packing kernel, never by the kernel this one may overlap (that kernel passed its
    // own wait, so every kernel before it, the packing included, has completed), and the copy then
    // overlaps the previous kernel's tail.
    if ((M64 || TN) && warp == 0 && lane == 0) {
        const int nblk = TK ? 5 : a.KT * a.n_chunks * (TN ? 3 : 9);
        const uint32_t bb = TK ? (uint32_t)a.tn_n * 32u : (TN ? (uint32_t)a.tn_n * 128u : (uint32_t)kWBlock64);
        ptx::mbar_arrive_expect_tx(bar_w_full, (uint32_t)nblk * bb);
        for (int b = 0; b < nblk; ++b)
            ptx::bulk_load(sW + (uint32_t)b * bb, a.w + (size_t)b * bb, bb, bar_w_full);
    }
    ptx::grid_dep_wait();
    if (!a.has_carry) ptx::grid_dep_launch();
    const uint32_t tmem_base = *tmem_slot;
    // K order of this CTA. In the head form (kw folded into M: few, small weight blocks per tile) each
    // CTA walks its (kt, chunk) groups and the kh taps inside a group from a CTA-dependent starting
    // point, so the CTAs, which run in near lockstep, fetch different weight blocks at any moment
    // instead of all asking L2 for the same one (measured: 15 % faster there; the other forms run
    // slower with it, so they keep the natural order). Only
    // the fp32 summation order depends on it.
    constexpr int kTapsK = KWM ? 3 : (CTR ? 1 : 9);
    const int n_groups = (S2 ? 4 : a.KT) * a.n_chunks;  // S2: (phase, chunk) groups
    const int k_id = KWM ? (int)blockIdx.x : 0;
    const int rot_g = k_id % n_groups, rot_t = (k_id / n_groups) % kTapsK;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t h_cnt = 0, w_cnt = 0, r_cnt = 0;
            RingPos hr, wr;  // halo and weight ring positions of h_cnt and w_cnt
            bool ok = true;
            if (M64 || TN) {  // every weight block of the layer, loaded once before the grid dependency wait
                w_cnt = 1;
                wr.next(a.n_w);
            }
            for (long long k = 0; ok; ++k) {
                ClTile tc;
                if (STN) {
                    if (!stn_decode(a, k, tc)) break;
                } else {
                    const long long tile = cl_tile_of(k);
                    if (tile >= a.tiles) break;
                    tc = cl_decode(a, tile);
                }
                const int n = (int)fdiv((uint32_t)tc.fr, a.fd_dout), t = tc.fr - n * a.dout;
                const int r0 = (int)fdiv((uint32_t)(tc.win * a.win_adv), a.fd_P);
                const int ow0 = tc.strip * a.Wt;
                for (int gi = 0; gi < n_groups && ok; ++gi) {
                    int kt, cc;
                    if (KWM) {
                        const int gg = gi + rot_g < n_groups ? gi + rot_g : gi + rot_g - n_groups;
                        kt = (int)fdiv((uint32_t)gg, a.fd_chunks);
                        cc = gg - kt * a.n_chunks;
                    } else {
                        kt = (int)fdiv((uint32_t)gi, a.fd_chunks);
                        cc = gi - kt * a.n_chunks;
                        // centre-tap forms: the temporal taps in the order 1, 2, 0 (measured on the
                        // stencil head at 4 + 2 frames: 0.1476 ms against 0.1511 in the order 0, 1, 2, the
                        // order 2, 0, 1 as fast; same box). The stencil head and the split head's temporal
                        // pass take the same order, so that their fp32 sums stay bit for bit equal.
                        if (CTR && a.KT == 3) kt = kt == 2 ? 0 : kt + 1;
                    }
                    const void* map = &tm_x;
                    int fcoord;
                    if (a.KT == 3) {
                        const int f = t + kt;  // frame of [carry0, carry1, x0, ...] read by tap kt
                        if (f >= 2) fcoord = n * a.D + (f - 2);
                        else if (a.has_carry) { map = &tm_c; fcoord = n * 2 + f; }
                        else fcoord = -1;  // out of range: zeros
                    } else {
                        fcoord = n;
                    }
                    {
                        if (NC) {
                            // raw NCHW slices of 16 channels for the transposers (aligned 8 columns left)
                            const int nsc = (min(a.C_in - cc * kCK, kCK) + 15) / 16;
                            for (int sc = 0; sc < nsc; ++sc) {
                                const uint32_t sr = r_cnt % a.n_raw;
                                if (!cl_wait(bar_r_empty + 8 * sr, ((r_cnt / a.n_raw) & 1u) ^ 1u, abort_flag, a.status)) { ok = false; break; }
                                ptx::mbar_arrive_expect_tx(bar_r_full + 8 * sr, (uint32_t)a.raw_tx_bytes);
                                ptx::tma_load_4d(sRaw + sr * a.raw_bytes, &tm_x, bar_r_full + 8 * sr, ow0 - 8, r0 - 1 + a.row_shift,
                                                 cc * kCK + 16 * sc, n);
                                ++r_cnt;
                            }
                            if (!ok) break;
                        } else {
                            const uint32_t sh = hr.slot;
                            if (!cl_wait(bar_h_empty + 8 * sh, hr.phase ^ 1u, abort_flag, a.status)) { ok = false; break; }
                            ptx::mbar_arrive_expect_tx(bar_h_full + 8 * sh, (uint32_t)a.h_tx_bytes);
                            if (CTR) {
                                // 256 consecutive positions of the frame's flattened plane (STN: the
                                // 32 x 8 raster window) and the (kt, chunk) weight block, one stage
                                // and one barrier for both
                                if (STN)
                                    ptx::tma_load_4d(sH + sh * a.h_bytes, map, bar_h_full + 8 * sh, cc * kCK, ow0 - 1,
                                                     tc.grow + a.row_shift, fcoord);
                                else
                                    ptx::tma_load_4d(sH + sh * a.h_bytes, map, bar_h_full + 8 * sh, cc * kCK, tc.win * kBNP, 0, fcoord);
                                ptx::bulk_load(sH + sh * a.h_bytes + (uint32_t)kCtrW,
                                               a.w + ((size_t)kt * a.n_chunks + cc) * (size_t)kWBlock, (uint32_t)kWBlock,
                                               bar_h_full + 8 * sh);
                            } else if (S2)  // phase kt = 2a + b: input rows 2(r0 - 1 + v) + a, columns 2(ow0 - 1 + u) + b
                                ptx::tma_load_4d(sH + sh * a.h_bytes, map, bar_h_full + 8 * sh, cc * kCK,
                                                 2 * (ow0 - 1) + (kt & 1), 2 * (r0 - 1) + (kt >> 1), fcoord);
                            else
                                ptx::tma_load_4d(sH + sh * a.h_bytes, map, bar_h_full + 8 * sh, cc * kCK, ow0 - 1,
                                                 r0 - 1 + a.row_shift, fcoord);
                            ++h_cnt;
                            hr.next(a.n_h);
                        }
                        const uint8_t* wblk =
                            a.w + ((((size_t)tc.nt * a.KT + (S2 ? 0 : kt)) * a.n_chunks + cc) * kTapsK) * (size_t)kWBlock;
                        for (int ti = 0; ti < ((M64 || CTR || TN) ? 0 : (S2 ? s2_ntaps(kt) : kTapsK)); ++ti) {
                            int tap = KWM ? (ti + rot_t < kTapsK ? ti + rot_t : ti + rot_t - kTapsK) : ti;
                            if (S2) {  // the phase's taps, in the MMA issuer's order
                                int kh, kw;
                                s2_tap(kt, ti, kh, kw);
                                tap = kh * 3 + kw;
                            }
                            const uint32_t sw = wr.slot;
                            if (!cl_wait(bar_w_empty + 8 * sw, wr.phase ^ 1u, abort_flag, a.status)) { ok = false; break; }
                            ptx::mbar_arrive_expect_tx(bar_w_full + 8 * sw, (uint32_t)kWBlock);
                            ptx::bulk_load(sW + sw * kWBlock, wblk + (size_t)tap * kWBlock, (uint32_t)kWBlock,
                                           bar_w_full + 8 * sw);
                            ++w_cnt;
                            wr.next(a.n_w);
                        }
                    }
                }
            }
            if (!ok) {  // wait (bounded) for the copies already issued into each stage
                volatile int dummy = 0;
                for (uint32_t i = 0; i < (uint32_t)a.n_h && i < h_cnt; ++i) {
                    const uint32_t last = i + ((h_cnt - 1 - i) / a.n_h) * a.n_h;
                    cl_wait(bar_h_full + 8 * i, (last / a.n_h) & 1u, &dummy, a.status);
                }
                for (uint32_t i = 0; i < (uint32_t)a.n_w && i < w_cnt; ++i) {
                    const uint32_t last = i + ((w_cnt - 1 - i) / a.n_w) * a.n_w;
                    cl_wait(bar_w_full + 8 * i, (last / a.n_w) & 1u, &dummy, a.status);
                }
                for (uint32_t i = 0; i < (uint32_t)a.n_raw && i < r_cnt; ++i) {
                    const uint32_t last = i + ((r_cnt - 1 - i) / a.n_raw) * a.n_raw;
                    cl_wait(bar_r_full + 8 * i, (last / a.n_raw) & 1u, &dummy, a.status);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (one thread)
        if (lane == 0) {
            uint32_t h_cnt = 0, w_cnt = 0, it = 0;
            RingPos hr, wr;  // halo and weight ring positions of h_cnt and w_cnt
            bool ok = true;
            // A (weights), no swizzle: SBO = 128 B between 8-row groups, LBO = 2 KB between the two
            // 8-channel halves of a 16-channel K step; version 1 in bits 46-47.
            constexpr int kRows = M64 ? 64 : kBM;  // rows of a weight block (MMA M)
            const uint32_t a_hi = (128u >> 4) | (1u << 14);
            const uint32_t a_lo0 = ((sW >> 4) & 0x3FFFu) | ((uint32_t)((kRows * 16) >> 4) << 16);
            if (M64 || TN) {  // resident weights
                if (!cl_wait(bar_w_full, 0, abort_flag, a.status)) ok = false;
                ptx::tc_fence_after();
            }
            // B (halo), 128-byte swizzle: SBO = 1024 B between 8-row groups, LBO encoded 1 (unused by
            // the swizzled K-major layout), version 1, layout type 2 (128-byte swizzle) in bits 61-63,
            // base offset 0. The tensor core applies the swizzle to the absolute shared-memory address
            // bits, exactly as the TMA unit wrote them, so a start shifted by any whole number of
            // 128-byte rows (a spatial tap) or by 32-byte K steps needs no base-offset correction;
            // the integer-exact parity tests pin this.
            const uint32_t b_hi_fixed = (1024u >> 4) | (1u << 14) | (2u << 29);
            // TN: descriptor of the first resident weight block (SBO 128 B, LBO N x 16 B, version 1), the
            // descriptor step between blocks and between the K steps of a block (N x 32 B)
            const uint64_t tn_wdesc0 = TN ? (((uint64_t)((128u >> 4) | (1u << 14)) << 32) |
                                             (uint64_t)(((sW >> 4) & 0x3FFFu) | ((uint32_t)((a.tn_n * 16) >> 4) << 16)))
                                          : 0;
            const uint32_t tn_wstep = TN ? (uint32_t)a.tn_n * 8u : 0u;   // N x 128 B / 16
            const uint32_t tn_kstep = TN ? (uint32_t)a.tn_n * 2u : 0u;   // N x 32 B / 16
            // with a carry: the last of this CTA's tiles that reads it (output frame 0 or 1 of the
            // pass); the launch signal follows that tile's halo waits
            long long last_carry_k = -1;
            if (a.has_carry) {
                for (long long k = 0;; ++k) {
                    int fr;
                    if (STN) {
                        ClTile tc;
                        if (!stn_decode(a, k, tc)) break;
                        fr = tc.fr;
                    } else {
                        const long long tile = cl_tile_of(k);
                        if (tile >= a.tiles) break;
                        fr = a.KT == 3 ? cl_decode(a, tile).fr : 2;
                    }
                    if (a.KT == 3 && fr - (int)fdiv((uint32_t)fr, a.fd_dout) * a.dout < 2) last_carry_k = k;
                }
                if (last_carry_k < 0) ptx::grid_dep_launch();
            }
            for (long long k = 0; ok; ++k) {
                long long tile = 0;
                ClTile tcs;
                if (STN) {
                    if (!stn_decode(a, k, tcs)) break;
                } else {
                    tile = cl_tile_of(k);
                    if (tile >= a.tiles) break;
                }
                if constexpr (TN) {
                    // positions as M: per (kt, chunk) halo and kernel row kh, A = the 128 positions from
                    // halo position kh P (swizzled K-major rows; windows start at a raster row), B = the
                    // resident (kw, co) rows of weight block (kt, chunk, kh) (no swizzle: LBO = N x 16 B
                    // between the two 8-channel halves of a K step, SBO = 128 B between 8-row groups).
                    // Descriptors are a base descriptor plus the byte offset / 16 (the 14-bit address
                    // field cannot carry: shared memory is below 256 KB). The tile needs no decode here;
                    // its first halo is awaited before the accumulator, so that the MMAs follow the
                    // accumulator wait directly.
                    const uint32_t ab = it & 1u, use = it >> 1;
                    const uint32_t d = tmem_base + ab * (uint32_t)kBNP;
                    uint32_t acc = 0;
                    for (int g = 0; g < a.KT * a.n_chunks && ok; ++g) {
                        const int kt = (int)fdiv((uint32_t)g, a.fd_chunks), cc = g - kt * a.n_chunks;
                        const uint32_t sh = hr.slot;
                        if (!cl_wait(bar_h_full + 8 * sh, hr.phase, abort_flag, a.status)) { ok = false; break; }
                        if (g == 0 && !cl_wait(bar_acc_empty + 8 * ab, (use & 1u) ^ 1u, abort_flag, a.status)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t hbase = sH + sh * (uint32_t)a.h_bytes;
                        if constexpr (TK) {
                            // K step s: taps 2s and 2s+1 (tap t = kh * 3 + kw at halo offset kh P + kw,
                            // 16 bytes per position); no swizzle, SBO = 128 B (8 positions), LBO = the
                            // second tap's offset; the ninth tap pairs with zero weights
                            const uint32_t tk_hi = (128u >> 4) | (1u << 14);
#pragma unroll
                            for (int ks = 0; ks < 5; ++ks) {
                                const int t0 = 2 * ks, t1 = 2 * ks + 1;
                                const int o0 = (t0 / 3) * a.P + t0 % 3;
                                const int o1 = t1 < 9 ? (t1 / 3) * a.P + t1 % 3 : o0 + 1;
                                const uint32_t lo = (((hbase + (uint32_t)o0 * 16u) >> 4) & 0x3FFFu) |
                                                    ((uint32_t)(o1 - o0) << 16);   // (o1 - o0) x 16 B / 16
                                const uint64_t adesc = ((uint64_t)tk_hi << 32) | (uint64_t)lo;
                                const uint64_t bdesc = tn_wdesc0 + (uint64_t)((uint32_t)ks * tn_kstep);
                                ptx::mma_f16(d, adesc, bdesc, a.idesc, ks > 0 ? 1u : 0u);
                            }
                            acc = 1;
                            ptx::mma_commit(bar_h_empty + 8 * sh);
                            ++h_cnt;
                            hr.next(a.n_h);
                            continue;
                        }
                        const uint64_t a0 = ((uint64_t)b_hi_fixed << 32) | (uint64_t)(((hbase >> 4) & 0x3FFFu) | (1u << 16));
                        const uint64_t w0 = tn_wdesc0 + (uint64_t)((uint32_t)((kt * a.n_chunks + cc) * 3) * tn_wstep);
                        const int rem = a.C_in - cc * kCK;
#pragma unroll
                        for (int kh = 0; kh < 3; ++kh) {
                            const uint64_t ak = a0 + (uint64_t)((uint32_t)(kh * a.P) * 8u);  // kh P rows x 128 B / 16
                            const uint64_t bk = w0 + (uint64_t)((uint32_t)kh * tn_wstep);
                            if (rem >= kCK) {
                                ptx::mma4_f16(d, ak, ak + 2, ak + 4, ak + 6, bk, bk + tn_kstep, bk + 2 * tn_kstep,
                                              bk + 3 * tn_kstep, a.idesc, acc);
                            } else {
                                for (int ks = 0; ks * 16 < rem; ++ks)
                                    ptx::mma_f16(d, ak + 2 * ks, bk + (uint64_t)(ks * tn_kstep), a.idesc, ks > 0 ? 1u : acc);
                            }
                            acc = 1;
                        }
                        ptx::mma_commit(bar_h_empty + 8 * sh);
                        ++h_cnt;
                        hr.next(a.n_h);
                    }
                    if (!ok) break;
                    ptx::mma_commit(bar_acc_full + 8 * ab);
                    ++it;
                    continue;
                }
                const ClTile tc = STN ? tcs : cl_decode(a, tile);
                const int pos_off = STN ? 0 : tc.win * a.win_adv - (int)fdiv((uint32_t)(tc.win * a.win_adv), a.fd_P) * a.P;
                // two accumulator buffers used alternately, or (W2) one pair of them per tile
                const uint32_t ab = W2 ? 0u : (it & 1u);
                const uint32_t use = W2 ? it : (it >> 1);
                if (!cl_wait(bar_acc_empty + 8 * ab, (use & 1u) ^ 1u, abort_flag, a.status)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + ab * (uint32_t)kBNP;
                uint32_t acc = 0;
                // the MMAs of one tap: four K steps of 16 channels into the tile's accumulator
                auto tap_mmas = [&](int cc, int kt, int kh, int kw, uint32_t hbase) -> bool {
                    const uint32_t sw = wr.slot;
                    uint32_t a_lo;
                    if (M64) {
                        a_lo = a_lo0 + (uint32_t)(((kt * a.n_chunks + cc) * 9 + kh * 3 + kw) * (kWBlock64 >> 4));
                    } else if (CTR) {  // the weight block shares the stage (and its barrier) with the window
                        a_lo = (((hbase + (uint32_t)kCtrW) >> 4) & 0x3FFFu) | ((uint32_t)((kBM * 16) >> 4) << 16);
                    } else {
                        if (!cl_wait(bar_w_full + 8 * sw, wr.phase, abort_flag, a.status)) return false;
                        ptx::tc_fence_after();
                        a_lo = a_lo0 + sw * (uint32_t)(kWBlock >> 4);
                    }
                    const uint32_t row_addr =
                        CTR ? hbase
                            : (S2 ? hbase + (uint32_t)(pos_off + (kh ? a.P : 0) + (kw ? 1 : 0)) * 128u
                                  : hbase + (uint32_t)(pos_off + kh * a.P + kw) * 128u);
                    if (!W2 && !M64 && a.C_in - cc * kCK >= kCK) {
                        // a full 64-channel block: its four K steps as one issue group (the M = 64
                        // form measured slower this way: 0.151 -> 0.160 ms for the TAESD chain)
                        uint64_t ad[4], bd[4];
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            ad[ks] = ((uint64_t)a_hi << 32) | (uint64_t)(a_lo + (uint32_t)ks * (uint32_t)((2 * kRows * 16) >> 4));
                            bd[ks] = ((uint64_t)b_hi_fixed << 32) |
                                     (uint64_t)((((row_addr + (uint32_t)ks * 32u) >> 4) & 0x3FFFu) | (1u << 16));
                        }
                        ptx::mma4_f16(d, ad[0], ad[1], ad[2], ad[3], bd[0], bd[1], bd[2], bd[3], a.idesc, acc);
                        acc = 1;
                    } else
#pragma unroll
                    for (int ks = 0; ks < kCK / 16; ++ks) {
                        if (ks * 16 >= a.C_in - cc * kCK) break;  // channels past C_in: nothing to add
                        const uint64_t adesc = ((uint64_t)a_hi << 32) |
                                               (uint64_t)(a_lo + (uint32_t)ks * (uint32_t)((2 * kRows * 16) >> 4));
                        const uint32_t baddr = row_addr + (uint32_t)ks * 32u;
                        const uint64_t bdesc = ((uint64_t)b_hi_fixed << 32) |
                                               (uint64_t)(((baddr >> 4) & 0x3FFFu) | (1u << 16));
                        ptx::mma_f16(d, adesc, bdesc, a.idesc, acc);
                        if (W2)  // the second window: 256 positions further on in the same staged halo
                            ptx::mma_f16(d + (uint32_t)kBNP, adesc, bdesc + (uint64_t)((kBNP * 128u) >> 4), a.idesc, acc);
                        acc = 1;
                    }
                    if (!M64 && !CTR) {
                        ptx::mma_commit(bar_w_empty + 8 * sw);
                        ++w_cnt;
                        wr.next(a.n_w);
                    }
                    return true;
                };
                auto group_begin = [&](uint32_t& sh, uint32_t& hbase) -> bool {
                    sh = hr.slot;
                    if (!cl_wait(bar_h_full + 8 * sh, hr.phase, abort_flag, a.status)) return false;
                    ptx::tc_fence_after();
                    hbase = sH + sh * (uint32_t)a.h_bytes;
                    return true;
                };
                if constexpr (KWM) {
                    // head form: rotated (kt, chunk) groups, rotated kh taps (kw is folded into M)
                    for (int gi = 0; gi < n_groups && ok; ++gi) {
                        const int gg = gi + rot_g < n_groups ? gi + rot_g : gi + rot_g - n_groups;
                        const int kt = gg / a.n_chunks, cc = gg - kt * a.n_chunks;
                        uint32_t sh, hbase;
                        if (!group_begin(sh, hbase)) { ok = false; break; }
#pragma unroll
                        for (int ti = 0; ti < 3; ++ti) {
                            const int kh = ti + rot_t < 3 ? ti + rot_t : ti + rot_t - 3;
                            if (ok && !tap_mmas(cc, kt, kh, 0, hbase)) ok = false;
                        }
                        if (!ok) break;
                        ptx::mma_commit(bar_h_empty + 8 * sh);
                        ++h_cnt;
                        hr.next(a.n_h);
                    }
                } else if constexpr (S2) {
                    // stride 2: (phase, chunk) groups, each with the taps that read the phase
                    for (int ph = 0; ph < 4 && ok; ++ph) {
                        for (int cc = 0; cc < a.n_chunks && ok; ++cc) {
                            uint32_t sh, hbase;
                            if (!group_begin(sh, hbase)) { ok = false; break; }
                            for (int i = 0; i < s2_ntaps(ph); ++i) {
                                int kh, kw;
                                s2_tap(ph, i, kh, kw);
                                if (!tap_mmas(cc, 0, kh, kw, hbase)) { ok = false; break; }
                            }
                            if (!ok) break;
                            ptx::mma_commit(bar_h_empty + 8 * sh);
                            ++h_cnt;
                            hr.next(a.n_h);
                        }
                    }
                } else {
                    for (int kt = 0; kt < a.KT && ok; ++kt) {
                        for (int cc = 0; cc < a.n_chunks && ok; ++cc) {
                            uint32_t sh, hbase;
                            if (!group_begin(sh, hbase)) { ok = false; break; }
                            for (int kh = (CTR ? 1 : 0); kh < (CTR ? 2 : 3) && ok; ++kh) {
                                for (int kw = (CTR ? 1 : 0); kw < (CTR ? 2 : 3); ++kw) {
                                    if (!tap_mmas(cc, kt, kh, kw, hbase)) { ok = false; break; }
                                }
                            }
                            if (!ok) break;
                            ptx::mma_commit(bar_h_empty + 8 * sh);
                            ++h_cnt;
                            hr.next(a.n_h);
                        }
                    }
                }
                if (!ok) break;
                if (k == last_carry_k) ptx::grid_dep_launch();  // this CTA's carry reads have landed
                ptx::mma_commit(bar_acc_full + 8 * ab);
                ++it;
            }
            ptx::mma_commit(bar_drain);
            volatile int dummy = 0;
            cl_wait(bar_drain, 0, &dummy, a.status);
        }
        __syncwarp();
    } else if (warp < 2 + kEpiWarps) {
        // ------------------------------------------------------------ epilogue: TMEM -> channels-last rows
        const int q = warp & 3;            // TMEM lane quarter = output channels 32q .. 32q+31
        const int ew = warp - 2;           // 0..3 (TN: 0..7): this warp's staging block
        uint32_t it = 0;
        int cur_nt = -1;
        float bias_r = 0.0f;
        float bias_g[10];
#pragma unroll
        for (int r = 0; r < 10; ++r) {
            const int co = q * 10 + r;
            bias_g[r] = 0.0f;
            if (KWM && a.bias && co < a.C_out) {
                const uint16_t raw = __ldg(reinterpret_cast<const unsigned short*>(a.bias) + co);
                bias_g[r] = BF16 ? __uint_as_float((uint32_t)raw << 16) : __half2float(__ushort_as_half(raw));
            }
        }
        uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
        // M = 64 form: one output tile, so this thread's two bias values are loaded once; the
        // activation as a clamp to [act_lo, act_hi]
        float m64_b0 = 0.0f, m64_b1 = 0.0f;
        if (M64 && a.bias) {
            const unsigned short* bp = reinterpret_cast<const unsigned short*>(a.bias);
            const int co0 = q * 16 + (lane >> 2), co1 = co0 + 8;
            if (co0 < a.C_out) m64_b0 = BF16 ? __uint_as_float((uint32_t)__ldg(bp + co0) << 16) : __half2float(__ushort_as_half(__ldg(bp + co0)));
            if (co1 < a.C_out) m64_b1 = BF16 ? __uint_as_float((uint32_t)__ldg(bp + co1) << 16) : __half2float(__ushort_as_half(__ldg(bp + co1)));
        }
        float stn_bias[3] = {0.0f, 0.0f, 0.0f};  // STN: this warp's three channels 3q..3q+2
        if (STN && a.bias) {
            const unsigned short* bp = reinterpret_cast<const unsigned short*>(a.bias);
#pragma unroll
            for (int cl = 0; cl < 3; ++cl)
                if (3 * q + cl < a.C_out) stn_bias[cl] = __uint_as_float((uint32_t)__ldg(bp + 3 * q + cl) << 16);
        }
        const float act_lo = a.act == X3_ACT_RELU ? 0.0f : (a.act == X3_ACT_CLAMP1 ? -1.0f : -INFINITY);
        const float act_hi = a.act == X3_ACT_CLAMP1 ? 1.0f : INFINITY;
        const uint32_t act2_lo = cl_pack2<BF16>(act_lo, act_lo), act2_hi = cl_pack2<BF16>(act_hi, act_hi);  // TN
        const float inv_p = 1.0f / (float)a.P;
        if (TN) {  // this warp's copy of the bias (zero past C_out)
            float* sb = reinterpret_cast<float*>(sbase + (sBiasT - base)) + ew * a.tn_cp;
            for (int co = lane; co < a.tn_cp; co += 32) {
                float b = 0.0f;
                if (a.bias && co < a.C_out) {
                    const uint16_t raw = __ldg(reinterpret_cast<const unsigned short*>(a.bias) + co);
                    b = BF16 ? __uint_as_float((uint32_t)raw << 16) : __half2float(__ushort_as_half(raw));
                }
                sb[co] = b;
            }
            __syncwarp();
        }
        for (long long k = 0;; ++k, ++it) {
            long long tile = 0;
            ClTile tcs;
            if (STN) {
                if (!stn_decode(a, k, tcs)) break;
            } else {
                tile = cl_tile_of(k);
                if (tile >= a.tiles) break;
            }
            // TN: warps 2-5 drain the even tiles (TMEM buffer 0), warps 6-9 the odd ones (buffer 1)
            if (TN && (int)(it & 1u) != (ew >> 2)) continue;
            if constexpr (TN) {
                // everything that does not depend on the accumulator is set up before waiting for it
                const uint32_t ab = it & 1u;
                const ClTile tc = cl_decode(a, tile);
                const int n = (int)fdiv((uint32_t)tc.fr, a.fd_dout), t = tc.fr - n * a.dout;
                const int m0 = tc.win * a.win_adv;
                const int ow0 = tc.strip * a.Wt;
                // Lane l of quarter q holds raster position (row q of the tile, column l): D[(kw, co)] in
                // TMEM columns kw * cp + co of this accumulator buffer. out = D(l)[(0,co)] +
                // D(l+1)[(1,co)] + D(l+2)[(2,co)] + bias: shuffles down by one and two lanes (lanes 30
                // and 31 are the raster's junk columns). Two 16-channel chunks at a time: their six TMEM
                // loads are issued before one wait; each lane stores its position's channels as 16-byte
                // pieces.
                const int cp = a.tn_cp, nck = cp >> 4;
                const float* sb = reinterpret_cast<const float*>(sbase + (sBiasT - base)) + ew * cp;
                const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBNP;
                const int m = m0 + q * 32 + lane;
                const int oh = (int)fdiv((uint32_t)m, a.fd_P), cc0 = m - oh * a.P;
                const int ow = ow0 + cc0;
                const bool valid = cc0 < a.Wt && ow < a.W_out && oh < a.H_out && !(a.sub2 && ((oh | ow) & 1));
                const int yh = a.sub2 ? oh >> 1 : oh, yw = a.sub2 ? ow >> 1 : ow;
                const size_t plane = (size_t)a.yH * a.yW;
                uint16_t* yp = a.out_nchw ? y + (size_t)n * a.C_out * plane + (size_t)yh * a.yW + yw
                                          : y + (((size_t)n * a.dout + t) * plane + (size_t)yh * a.yW + yw) * a.C_out;
                // TMA-store form (64 channels, channels-last, stride 1): this lane's position is row `lane`
                // of the warp's 4 KB buffer, 128 bytes, its 16-byte pieces placed by the 128-byte swizzle
                // (piece u at u ^ (row & 7)), which is also conflict-free for these writes; the warp's
                // 30 outputs then leave as one box {64 channels, 30 columns, 1 row, 1 frame}, clipped at
                // the image edge by the TMA unit
                const bool tma = a.tn_tma != 0;
                const uint32_t ob = sStage + (uint32_t)(ew * a.stage_warp);
                const int row_h = (int)fdiv((uint32_t)(m0 + q * 32), a.fd_P);
                if (tma) {
                    if (lane == 0) ptx::bulk_wait_group_read0();  // the previous store from this buffer has read it
                    __syncwarp();
                }
                if (!cl_wait(bar_acc_full + 8 * ab, (it >> 1) & 1u, abort_flag, a.status)) break;
                ptx::tc_fence_after();
                auto load = [&](int c, uint32_t (&v0)[16], uint32_t (&v1)[16], uint32_t (&v2)[16]) {
                    ptx::tmem_ld16(tq + (uint32_t)(16 * c), v0);
                    if (!TK) {
                        ptx::tmem_ld16(tq + (uint32_t)(cp + 16 * c), v1);
                        ptx::tmem_ld16(tq + (uint32_t)(2 * cp + 16 * c), v2);
                    }
                };
                auto sum = [&](int c, const uint32_t (&v0)[16], const uint32_t (&v1)[16], const uint32_t (&v2)[16]) {
                    // two channels at a time: ((D0 + D1 shifted) + D2 shifted) + bias with packed fp32
                    // adds (each half is the scalar add, in the same order), one rounding of the pair,
                    // then the activation's clamp on the rounded pair (measured on the TAESD-like chain:
                    // 0.114 ms with scalar adds and the clamp before rounding, 0.106 with the packed
                    // pairs, 0.119 when the clamp branches on the activation kind)
                    uint32_t h[8];
#pragma unroll
                    for (int k = 0; k < 16; k += 2) {
                        uint64_t s = ptx::f32x2(__uint_as_float(v0[k]), __uint_as_float(v0[k + 1]));
                        if (!TK) {
                            const float s1a = __shfl_down_sync(0xffffffffu, __uint_as_float(v1[k]), 1);
                            const float s1b = __shfl_down_sync(0xffffffffu, __uint_as_float(v1[k + 1]), 1);
                            const float s2a = __shfl_down_sync(0xffffffffu, __uint_as_float(v2[k]), 2);
                            const float s2b = __shfl_down_sync(0xffffffffu, __uint_as_float(v2[k + 1]), 2);
                            s = ptx::add_f32x2(s, ptx::f32x2(s1a, s1b));
                            s = ptx::add_f32x2(s, ptx::f32x2(s2a, s2b));
                        }
                        s = ptx::add_f32x2(s, *reinterpret_cast<const uint64_t*>(sb + 16 * c + k));
                        float lo, hi;
                        ptx::f32x2_split(s, lo, hi);
                        h[k >> 1] = cl_clamp2<BF16>(cl_pack2<BF16>(lo, hi), act2_lo, act2_hi);
                    }
                    if (tma) {
                        const uint4 w0 = make_uint4(h[0], h[1], h[2], h[3]), w1 = make_uint4(h[4], h[5], h[6], h[7]);
                        uint8_t* rowp = sbase + (ob - base) + lane * 128;
                        *reinterpret_cast<uint4*>(rowp + (((2 * c) ^ (lane & 7)) << 4)) = w0;
                        *reinterpret_cast<uint4*>(rowp + (((2 * c + 1) ^ (lane & 7)) << 4)) = w1;
                        return;
                    }
                    if (!valid) return;
                    if (a.out_nchw) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (16 * c + k < a.C_out) yp[(size_t)(16 * c + k) * plane] = (uint16_t)(h[k >> 1] >> (16 * (k & 1)));
                    } else {
                        const uint4 w0 = make_uint4(h[0], h[1], h[2], h[3]), w1 = make_uint4(h[4], h[5], h[6], h[7]);
                        *reinterpret_cast<uint4*>(yp + 16 * c) = w0;
                        if (16 * c + 8 < a.C_out) *reinterpret_cast<uint4*>(yp + 16 * c + 8) = w1;
                    }
                };
                {
                    uint32_t a0[16], a1[16], a2[16], b0[16], b1[16], b2[16];
                    if constexpr (TK) {
                        // one TMEM value per output: every chunk's load (at most five: 80 channels) goes
                        // out before a single wait, and the buffer goes back before any sum
                        ptx::tmem_ld16(tq, a0);
                        if (nck > 1) ptx::tmem_ld16(tq + 16u, b0);
                        if (nck > 2) ptx::tmem_ld16(tq + 32u, a1);
                        if (nck > 3) ptx::tmem_ld16(tq + 48u, b1);
                        if (nck > 4) ptx::tmem_ld16(tq + 64u, a2);
                        ptx::tmem_ld_wait();
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar_acc_empty + 8 * ab);
                        sum(0, a0, a1, a2);
                        if (nck > 1) sum(1, b0, b1, b2);
                        if (nck > 2) sum(2, a1, a1, a2);
                        if (nck > 3) sum(3, b1, b1, b2);
                        if (nck > 4) sum(4, a2, a1, a2);
                    } else
                    for (int c = 0; c < nck; c += 2) {
                        load(c, a0, a1, a2);
                        if (c + 1 < nck) load(c + 1, b0, b1, b2);
                        ptx::tmem_ld_wait();
                        if (c + 2 >= nck) {
                            // the accumulator is in registers: hand the TMEM buffer back to the MMA issuer
                            // before the last sums and stores
                            ptx::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) ptx::mbar_arrive(bar_acc_empty + 8 * ab);
                        }
                        sum(c, a0, a1, a2);
                        if (c + 1 < nck) sum(c + 1, b0, b1, b2);
                    }
                }
                if (tma) {
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && row_h < a.H_out) {
                        ptx::tma_store_4d(&tm_y, ob, 0, ow0, row_h, n * a.dout + t);
                        ptx::bulk_commit_group();
                    }
                }
                continue;
            }
            const uint32_t ab = W2 ? 0u : (it & 1u);
            if (!cl_wait(bar_acc_full + 8 * ab, (W2 ? it : (it >> 1)) & 1u, abort_flag, a.status)) break;
            ptx::tc_fence_after();
            const ClTile tc = STN ? tcs : cl_decode(a, tile);
            const int n = (int)fdiv((uint32_t)tc.fr, a.fd_dout), t = tc.fr - n * a.dout;
            constexpr int kCpw = M64 ? 16 : 32;  // accumulator rows per TMEM lane quarter
            const int co_lane = (M64 && lane >= 16) ? a.C_out : tc.nt * (M64 ? 64 : kBM) + q * kCpw + lane;
            if (tc.nt != cur_nt) {
                bias_r = 0.0f;
                if (a.bias && co_lane < a.C_out) {
                    const uint16_t raw = __ldg(reinterpret_cast<const unsigned short*>(a.bias) + co_lane);
                    bias_r = BF16 ? __uint_as_float((uint32_t)raw << 16) : __half2float(__ushort_as_half(raw));
                }
                cur_nt = tc.nt;
            }
            const int m0 = tc.win * a.win_adv;
            const int ow0 = tc.strip * a.Wt;
            if (KWM) {
                // Lane kw*10 + r of quarter q holds the partial sums of channel 10q + r over the taps
                // with that kw, at every window column; output column j adds kw = 0, 1, 2 at columns
                // j, j+1, j+2 (its left, centre and right input columns).
                if (q < a.ngroups) {
                    float* S = reinterpret_cast<float*>(stage_ptr + ew * a.stage_warp);
                    for (int chunk = 0; chunk < kBNP / 32; ++chunk) {
                        uint32_t v[32], e2[2] = {0u, 0u};
                        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBNP +
                                               (uint32_t)(chunk * 32);
                        ptx::tmem_ld32(taddr, v);
                        if (chunk + 1 < kBNP / 32) ptx::tmem_ld2(taddr + 32u, e2);
                        ptx::tmem_ld_wait();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 32; ++j) S[lane * kSPitch + j] = __uint_as_float(v[j]);
                        S[lane * kSPitch + 32] = __uint_as_float(e2[0]);
                        S[lane * kSPitch + 33] = __uint_as_float(e2[1]);
                        __syncwarp();
                        const int jw = chunk * 32 + lane;  // column of the window
                        const int m = m0 + jw;
                        const int oh = (int)fdiv((uint32_t)m, a.fd_P), c = m - oh * a.P;
                        const int ow = ow0 + c;
                        if (jw < a.win_adv && c < a.Wt && ow < a.W_out && oh < a.H_out) {
                            const size_t W2o = 2 * (size_t)a.W_out;
                            const size_t row0 = (((size_t)n * a.dout + t) * 2 * (size_t)a.H_out + 2 * (size_t)oh);
#pragma unroll
                            for (int r = 0; r < 10; ++r) {
                                const int co = q * 10 + r;
                                if (co < a.C_out) {
                                    const float acc = S[r * kSPitch + lane] + S[(10 + r) * kSPitch + lane + 1] +
                                                      S[(20 + r) * kSPitch + lane + 2] + bias_g[r];
                                    // unpatchify: channel co = rgb*4 + dy*2 + dx -> pixel (2oh+dy, 2ow+dx)
                                    const int rgb = co >> 2, dy = (co >> 1) & 1, dx = co & 1;
                                    y[((row0 + dy) * W2o + 2 * (size_t)ow + dx) * 3 + rgb] =
                                        cl_round<BF16>(cl_act(acc, a.act));
                                }
                            }
                        }
                    }
                }
            } else {
                if (NC || a.out_nchw) {
                    // NCHW: this warp's 32 channels x 32 positions are transposed through its staging
                    // block so that each store instruction writes 32 consecutive positions of a channel.
                    uint16_t* T = reinterpret_cast<uint16_t*>(stage_ptr + ew * a.stage_warp);  // [32][34]
                    const int co_base = tc.nt * (M64 ? 64 : kBM) + q * kCpw;
                    if (co_base < a.C_out) {
                        for (int chunk = 0; chunk < kBNP / 32; ++chunk) {
                            uint32_t v[32];
                            ptx::tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBNP +
                                               (uint32_t)(chunk * 32), v);
                            ptx::tmem_ld_wait();
                            __syncwarp();
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                T[lane * 34 + j] = cl_round<BF16>(cl_act(__uint_as_float(v[j]) + bias_r, a.act));
                            __syncwarp();
                            const int m = m0 + chunk * 32 + lane;
                            const int oh = (int)fdiv((uint32_t)m, a.fd_P), c = m - oh * a.P;
                            const int ow = ow0 + c;
                            const bool keep = c < a.Wt && ow < a.W_out && oh < a.H_out && !(a.sub2 && ((oh | ow) & 1));
                            if (keep) {
                                const int yh = a.sub2 ? oh >> 1 : oh, yw = a.sub2 ? ow >> 1 : ow;
                                const size_t plane = (size_t)a.yH * a.yW;
                                uint16_t* yp = y + ((size_t)n * a.C_out + co_base) * plane + (size_t)yh * a.yW + yw;
                                const int nco = min(kCpw, a.C_out - co_base);
                                for (int r = 0; r < nco; ++r) yp[(size_t)r * plane] = T[r * 34 + lane];
                            }
                        }
                    }
                } else if (M64) {
                    // M = 64: this quarter's 16 channels x 32 positions per chunk come in the MMA
                    // fragment layout (16 lanes x 256 bits, four column groups); each thread rounds its
                    // pairs of positions into packed 32-bit words and stmatrix.trans writes them as
                    // [position][16 channels] rows, four chunks into four 1 KB slots of the warp's
                    // staging block before one warp barrier; then each position's 32 bytes go out as
                    // two 16-byte stores, the sixteen loads and stores of the four chunks in flight
                    // together. The second half's TMEM load is in flight while the first is processed.
                    const uint32_t wst = sStage + (uint32_t)(ew * a.stage_warp);  // [4][32][16] x 2 B
                    const uint8_t* wstp = stage_ptr + ew * a.stage_warp;
                    const float b0 = m64_b0, b1 = m64_b1;
                    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBNP;
                    // stmatrix row address of this thread: matrix mi = lane / 8 (column group i = mi / 2,
                    // channel half mi % 2), row j = lane % 8 = position 8i + j of the pair of groups
                    const int mi = lane >> 3, jr = lane & 7;
                    const uint32_t st_addr = wst + (uint32_t)((8 * (mi >> 1) + jr) * 32 + (mi & 1) * 16);
                    // the window's first raster row and column; a position's row and column follow from
                    // its offset by a float reciprocal (exact: offsets < 512, pitch <= 256)
                    const int oh0 = (int)fdiv((uint32_t)m0, a.fd_P), c00 = m0 - oh0 * a.P;
                    uint16_t* yf = y + ((size_t)n * a.dout + t) * (size_t)a.yH * a.yW * a.C_out;
                    auto stage = [&](int slot, const uint32_t (&v)[16]) {
                        uint32_t h[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            h[2 * i] = cl_pack2<BF16>(fminf(fmaxf(__uint_as_float(v[4 * i]) + b0, act_lo), act_hi),
                                                      fminf(fmaxf(__uint_as_float(v[4 * i + 1]) + b0, act_lo), act_hi));
                            h[2 * i + 1] = cl_pack2<BF16>(fminf(fmaxf(__uint_as_float(v[4 * i + 2]) + b1, act_lo), act_hi),
                                                          fminf(fmaxf(__uint_as_float(v[4 * i + 3]) + b1, act_lo), act_hi));
                        }
                        const uint32_t sa = st_addr + (uint32_t)slot * 1024u;
                        ptx::stsm_x4_trans(sa, h[0], h[1], h[2], h[3]);            // positions 0..15
                        ptx::stsm_x4_trans(sa + 16u * 32u, h[4], h[5], h[6], h[7]);  // positions 16..31
                    };
                    auto drain = [&](int chunk0) {
#pragma unroll
                        for (int slot = 0; slot < 4; ++slot) {
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const int piece = k * 32 + lane;
                                const int pos = piece >> 1, half = piece & 1;
                                const int cc = c00 + (chunk0 + slot) * 32 + pos;
                                const int dr = __float2int_rz(((float)cc + 0.5f) * inv_p);
                                const int oh = oh0 + dr, c = cc - dr * a.P;
                                const int ow = ow0 + c;
                                const int co = q * 16 + half * 8;
                                if (c < a.Wt && ow < a.W_out && oh < a.H_out && co < a.C_out &&
                                    !(a.sub2 && ((oh | ow) & 1))) {
                                    const int yh = a.sub2 ? oh >> 1 : oh, yw = a.sub2 ? ow >> 1 : ow;
                                    const uint4 val =
                                        *reinterpret_cast<const uint4*>(wstp + slot * 1024 + pos * 32 + half * 16);
                                    *reinterpret_cast<uint4*>(yf + ((size_t)yh * a.yW + yw) * a.C_out + co) = val;
                                }
                            }
                        }
                    };
                    uint32_t ra[4][16], rb[4][16];
#pragma unroll
                    for (int c = 0; c < 4; ++c) ptx::tmem_ld16x256b_x4(tq + (uint32_t)(c * 32), ra[c]);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c) ptx::tmem_ld16x256b_x4(tq + (uint32_t)((4 + c) * 32), rb[c]);
                    __syncwarp();  // the previous tile's loads from the slots are done
#pragma unroll
                    for (int c = 0; c < 4; ++c) stage(c, ra[c]);
                    __syncwarp();
                    drain(0);
                    ptx::tmem_ld_wait();
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 4; ++c) stage(c, rb[c]);
                    __syncwarp();
                    drain(4);
                } else if (STN) {
                    // Window position m = 32 r + c holds G at window row r (input row grow + r) and column
                    // c (input column ow0 - 1 + c; columns 0 and 31 are halo). The warp takes the rows in
                    // order: it stages row r's 27 TMEM rows (9 taps x 3 channels) in shared memory,
                    // S[tap row][c], and thread c adds row r's taps of kernel row i at columns c - 1 ..
                    // c + 1 (j = 0, 1, 2) to the sums of three output rows pending in registers: i = 2 to
                    // output row grow + r - 1, which is then complete, i = 1 to grow + r, and i = 0, after
                    // the bias, to grow + r + 1. Every output so sums bias and the nine taps in (i, j)
                    // order. The two sums still pending after the last row stay in shared memory (per
                    // output frame) for the next window of the run; the first window of a run piece
                    // starts them afresh and stores from its third row on.
                    float* S = reinterpret_cast<float*>(stage_ptr + ew * a.stage_warp);  // [27][kStnPitch]
                    float* Cw = reinterpret_cast<float*>(sbase + (sBiasT - base)) +
                                (size_t)(ew * a.stn_fpc + tc.fslot) * (kStnCarryBytes / 4);  // [2][3][32]
                    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBNP;
                    const int ow = ow0 - 1 + lane;
                    const bool col_ok = lane >= 1 && lane <= 30 && ow < a.W_out;
                    const size_t W2o = 2 * (size_t)a.W_out;
                    const size_t row0 = ((size_t)n * a.dout + t) * 2 * (size_t)a.H_out;
                    const bool first = tc.win == 0;
                    float pa[3], pb[3];  // pending sums of output rows grow + r - 1 and grow + r
#pragma unroll
                    for (int cl = 0; cl < 3; ++cl) {
                        pa[cl] = (!first && col_ok) ? Cw[cl * 32 + lane] : 0.0f;
                        pb[cl] = (!first && col_ok) ? Cw[(3 + cl) * 32 + lane] : 0.0f;
                    }
                    uint32_t vn[32];
                    ptx::tmem_ld32(tq, vn);  // window row 0
                    for (int r = 0; r < kStnRows; ++r) {
                        ptx::tmem_ld_wait();
                        if (lane < 27) {
#pragma unroll
                            for (int x = 0; x < 32; ++x) S[lane * kStnPitch + x] = __uint_as_float(vn[x]);
                        }
                        if (r + 1 < kStnRows) ptx::tmem_ld32(tq + (uint32_t)(32 * (r + 1)), vn);  // in flight meanwhile
                        __syncwarp();
                        if (col_ok) {
                            const int orow = tc.grow + r - 1;  // the output row completed by window row r
                            const bool store = !(first && r < 2) && orow < tc.rend;
#pragma unroll
                            for (int cl = 0; cl < 3; ++cl) {
                                const float* sp = S + (cl * 9) * kStnPitch + lane - 1;
                                float sa = pa[cl], sb = pb[cl], sc = stn_bias[cl];
#pragma unroll
                                for (int j = 0; j < 3; ++j) sa += sp[(6 + j) * kStnPitch + j];
#pragma unroll
                                for (int j = 0; j < 3; ++j) sb += sp[(3 + j) * kStnPitch + j];
#pragma unroll
                                for (int j = 0; j < 3; ++j) sc += sp[j * kStnPitch + j];
                                if (store) {
                                    const int c = 3 * q + cl;
                                    const int rgb = c >> 2, dy = (c >> 1) & 1, dx = c & 1;
                                    y[((row0 + 2 * (size_t)orow + dy) * W2o + 2 * (size_t)ow + dx) * 3 + rgb] =
                                        cl_round<BF16>(fminf(act_hi, fmaxf(act_lo, sa)));
                                }
                                pa[cl] = sb;
                                pb[cl] = sc;
                            }
                        }
                        __syncwarp();
                    }
                    if (col_ok) {
#pragma unroll
                        for (int cl = 0; cl < 3; ++cl) {
                            Cw[cl * 32 + lane] = pa[cl];
                            Cw[(3 + cl) * 32 + lane] = pb[cl];
                        }
                    }
                } else if (CTR) {
                    // Temporal pass of the split head: accumulator row r = (i*3+j)*12 + c goes to plane
                    // p = i*3+j of G at channel c. Each warp stages its 32 rows x 32 positions as
                    // [position][row] fp32, then writes 4-row groups (16 bytes of fp32 or 8 of bf16;
                    // quarter boundaries fall on 4-channel steps of a plane) for 32 positions at a time.
                    float* S = reinterpret_cast<float*>(stage_ptr + ew * a.stage_warp);  // [32][kGPitch]
                    const long long hw = (long long)a.H_out * a.W_out;
                    for (int chunk = 0; chunk < kBNP / 32; ++chunk) {
                        uint32_t v[32];
                        ptx::tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBNP + (uint32_t)(chunk * 32), v);
                        ptx::tmem_ld_wait();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 32; ++j) S[j * kGPitch + lane] = __uint_as_float(v[j]);
                        __syncwarp();
                        const long long pos = (long long)m0 + chunk * 32 + lane;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int r0 = q * 32 + 4 * k;
                            if (r0 < 108 && pos < hw) {
                                const float4 f = *reinterpret_cast<const float4*>(S + lane * kGPitch + 4 * k);
                                const long long e = (((long long)tc.fr * 9 + r0 / 12) * hw + pos) * 12 + r0 % 12;
                                if (a.g_f32) {
                                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.y) + e) = f;
                                } else {
                                    uint2 b;
                                    b.x = cl_pack2<true>(f.x, f.y);
                                    b.y = cl_pack2<true>(f.z, f.w);
                                    *reinterpret_cast<uint2*>(y + e) = b;
                                }
                            }
                        }
                    }
                } else {
                    // Each warp transposes its own 32 channels x 32 positions through a private staging
                    // block (no barrier across warps), then writes 64 contiguous bytes per position row.
                    uint8_t* wst = stage_ptr + ew * a.stage_warp;
                    // W2: the two windows of the tile, accumulators in TMEM columns 0-255 and 256-511.
                    // A chunk's TMEM load goes out as soon as the previous chunk is staged, so it lands
                    // while that chunk's rows are written out.
                    constexpr int n_ck = (W2 ? 2 : 1) * (kBNP / 32);
                    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + ab * (uint32_t)kBNP;
                    uint32_t v[32];
                    ptx::tmem_ld32(tq, v);
                    for (int chunk = 0; chunk < n_ck; ++chunk) {
                        ptx::tmem_ld_wait();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            *reinterpret_cast<uint16_t*>(wst + j * kStagePitch + lane * 2) =
                                cl_round<BF16>(cl_act(__uint_as_float(v[j]) + bias_r, a.act));
                        if (chunk + 1 < n_ck) ptx::tmem_ld32(tq + (uint32_t)((chunk + 1) * 32), v);
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < (M64 ? 2 : 4); ++k) {
                            // 32 positions x (kCpw / 8) 16-byte channel segments per chunk
                            const int row = M64 ? k * 16 + (lane >> 1) : k * 8 + (lane >> 2);
                            const int seg = M64 ? (lane & 1) : (lane & 3);
                            const int m = m0 + chunk * 32 + row;
                            const int oh = (int)fdiv((uint32_t)m, a.fd_P), c = m - oh * a.P;
                            const int ow = ow0 + c;
                            const int co = tc.nt * (M64 ? 64 : kBM) + q * kCpw + seg * 8;
                            if (c < a.Wt && ow < a.W_out && oh < a.H_out && co < a.C_out &&
                                !(a.sub2 && ((oh | ow) & 1))) {
                                const int yh = a.sub2 ? oh >> 1 : oh, yw = a.sub2 ? ow >> 1 : ow;
                                const uint4 val = *reinterpret_cast<const uint4*>(wst + row * kStagePitch + seg * 16);
                                const size_t off =
                                    ((((size_t)n * a.dout + t) * a.yH + yh) * a.yW + yw) * (size_t)a.C_out + co;
                                *reinterpret_cast<uint4*>(y + off) = val;
                            }
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_acc_empty + 8 * ab);
        }
    } else if (NC) {
        // ------------------------------------------------------------ transposers (NCHW -> swizzled rows)
        const int tw = warp - 6;
        const int kb_n = a.raw_w / 8;      // 8-column blocks per raw row
        const uint32_t junk = sJunk + (uint32_t)(tw * 32 + lane) * 16u;
        uint32_t h_cnt = 0, r_cnt = 0;
        bool ok = true;
        for (long long tile = blockIdx.x; tile < a.tiles && ok; tile += gridDim.x) {
            for (int gi = 0; gi < n_groups && ok; ++gi) {
                // the producer's chunk order (2D: one temporal tap, so a group is a chunk)
                const int cc = gi + rot_g < n_groups ? gi + rot_g : gi + rot_g - n_groups;
                const uint32_t sh = h_cnt % a.n_h;
                if (!cl_wait(bar_h_empty + 8 * sh, ((h_cnt / a.n_h) & 1u) ^ 1u, abort_flag, a.status)) { ok = false; break; }
                const uint32_t hst = sH + sh * (uint32_t)a.h_bytes;
                const int nsc = (min(a.C_in - cc * kCK, kCK) + 15) / 16;
                for (int sc = 0; sc < nsc; ++sc) {
                    const uint32_t sr = r_cnt % a.n_raw;
                    if (!cl_wait(bar_r_full + 8 * sr, (r_cnt / a.n_raw) & 1u, abort_flag, a.status)) { ok = false; break; }
                    const uint32_t raw = sRaw + sr * (uint32_t)a.raw_bytes;
                    // rows of 8x8 blocks: item = (8-channel group j, halo row hr); each ldmatrix.x4 /
                    // stmatrix.x4 pair moves four consecutive 8-column blocks of one item
                    const int i = lane & 7;
                    for (int item = tw; item < 2 * a.HR; item += 4) {
                        const int j = item >= a.HR ? 1 : 0;
                        const int hr = item - j * a.HR;
                        const uint32_t src_row = raw + (uint32_t)(((8 * j + i) * a.HR + hr) * a.raw_w) * 2u;
                        const uint32_t dst_row = hst + (uint32_t)(hr * a.P) * 128u + (uint32_t)(2 * sc + j) * 16u;
                        for (int kb0 = 0; kb0 < kb_n; kb0 += 4) {
                            const int kb = kb0 + (lane >> 3);
                            uint32_t lds_addr = raw, sts_addr = junk;
                            if (kb < kb_n) {
                                // source row i: channel 8j+i, raw columns 8kb..8kb+7; destination row i:
                                // raw column 8kb+i = halo column 8kb+i-7 of row hr, 16-byte chunk 2sc+j of
                                // the position's 128-byte row, swizzled on the absolute address
                                lds_addr = src_row + (uint32_t)kb * 16u;
                                const int col = 8 * kb + i - 7;
                                if (col >= 0 && col < a.P) {
                                    const uint32_t addr = dst_row + (uint32_t)col * 128u;
                                    sts_addr = addr ^ (((addr >> 7) & 7u) << 4);
                                }
                            }
                            uint32_t r0v, r1v, r2v, r3v;
                            ptx::ldsm_x4_trans(lds_addr, r0v, r1v, r2v, r3v);
                            ptx::stsm_x4(sts_addr, r0v, r1v, r2v, r3v);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar_r_empty + 8 * sr);
                    ++r_cnt;
                }
                if (!ok) break;
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar_h_full + 8 * sh);
                ++h_cnt;
            }
        }
    }

    if (TN && a.tn_tma && warp >= 2 && lane == 0) ptx::bulk_wait_group0();  // this warp's row stores are done
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, 512u);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// es = 2: every second position along W and H (the box spans 2 box_w x 2 box_h positions of the
// tensor and lands box_w x box_h rows in shared memory); box_w and box_h are the landed counts.
// inner8: a box of 8 channels (16 bytes per position), no swizzle (the TK form's halo).
x3_status encode_sw128(CUtensorMap* m, bool bf16, const void* ptr, uint64_t C, uint64_t W, uint64_t H,
                       uint64_t F, uint32_t box_w, uint32_t box_h, uint32_t es_wh = 1, bool inner8 = false) {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return fail(X3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
        }
        fn = (EncodeTiledFn)f;
    }
    cuuint64_t gd[4] = {C, W, H, F};
    cuuint64_t gs[3] = {C * 2, C * 2 * W, C * 2 * W * H};
    cuuint32_t bd[4] = {inner8 ? 8u : (cuuint32_t)kCK, box_w * es_wh, box_h * es_wh, 1};
    cuuint32_t es[4] = {1, es_wh, es_wh, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(ptr), gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    inner8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(X3_ERR_CUDA, "cuTensorMapEncodeTiled (128-byte swizzle) failed (%d)", (int)r);
    return X3_OK;
}

// Plain (unswizzled) tensor map of an NCHW tensor for the raw 16-channel slices.
x3_status encode_nchw_raw(CUtensorMap* m, bool bf16, const void* ptr, uint64_t W, uint64_t H, uint64_t C, uint64_t N,
                          uint32_t box_w, uint32_t box_h) {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return fail(X3_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
        }
        fn = (EncodeTiledFn)f;
    }
    cuuint64_t gd[4] = {W, H, C, N};
    cuuint64_t gs[3] = {W * 2, W * H * 2, W * H * C * 2};
    cuuint32_t bd[4] = {box_w, box_h, 16, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(ptr), gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(X3_ERR_CUDA, "cuTensorMapEncodeTiled (NCHW raw) failed (%d)", (int)r);
    return X3_OK;
}

}  // namespace

// Programmatic dependent launches, unless X3CONV_PDL=0 in the environment (read once per process).
bool pdl_enabled() {
    static const bool on = [] {
        const char* v = getenv("X3CONV_PDL");
        return !(v && !strcmp(v, "0"));
    }();
    return on;
}

size_t cl_packed_bytes(const ClGeom& g) {
    if (g.tk) return (size_t)5 * g.tn_n * 32;
    if (g.tn) return (size_t)g.KT * g.n_chunks * 3 * g.tn_n * 128;
    return (size_t)g.n_tiles * g.KT * g.n_chunks * (g.kwm ? 3 : 9) * ((g.m64 ? 64 : kBM) * kCK * 2);
}

bool igemm_cl_plan(x3_conv_plan* p, int num_sms, bool small_cout) {
    const x3_conv_desc& d = p->d;
    ClGeom g;
    memset(&g, 0, sizeof g);
    // stride 2: 2D channels-last layers only, from their four input phases (X3CONV_S2=0 in the
    // environment declines it, so that the caller computes them as the stride-1 raster instead)
    if (d.stride == 2) {
        const char* s2_env = getenv("X3CONV_S2");
        if (d.dims != 2 || d.layout != X3_NHWC || d.unpatchify2x2 || d.kernel == X3_KERNEL_HEAD_STENCIL ||
            (s2_env && !strcmp(s2_env, "0")))
            return false;
        g.s2 = 1;
    } else if (d.stride != 1) {
        return false;
    }
    // NCHW 2D input (raw tiles transposed in shared memory) or channels-last input (swizzled TMA boxes)
    g.nchw = (d.dims == 2 && d.layout == X3_NCHW) ? 1 : 0;
    if (g.nchw) {
        if (d.W % 8 != 0 || d.unpatchify2x2) return false;  // 16-byte aligned rows for the raw TMA boxes
    } else {
        if (!(d.dims == 3 ? d.layout == X3_NDHWC : d.layout == X3_NHWC)) return false;
        if (d.C_in % 8 != 0) return false;
    }
    // the conv_out head (12 channels to unpatchified RGB) runs in the kw-folded form
    g.kwm = d.unpatchify2x2 ? 1 : 0;
    g.stn = (d.kernel == X3_KERNEL_HEAD_STENCIL) ? 1 : 0;
    g.ctr = (d.kernel == X3_KERNEL_HEAD_TWO_PASS || d.kernel == X3_KERNEL_HEAD_SPLIT || g.stn) ? 1 : 0;
    if (g.ctr) {
        // temporal pass of the two-pass head: 12 output channels x 9 spatial taps = 108 (112) channels
        if (!d.unpatchify2x2 || d.dims != 3 || d.layout != X3_NDHWC || d.dtype != X3_BF16) return false;
        g.kwm = 0;
    }
    if (!g.kwm && !g.nchw && !g.ctr && (d.C_out % 8 != 0 || (d.C_out < 96 && !small_cout))) return false;
    g.win_adv = g.kwm ? kBNP - 2 : kBNP;
    g.ngroups = g.kwm ? (d.C_out + 9) / 10 : 0;
    if (g.kwm && g.ngroups > 4) return false;
    g.KT = d.dims == 3 ? 3 : 1;
    g.n_chunks = (d.C_in + kCK - 1) / kCK;
    g.n_tiles = g.ctr ? 1 : (d.C_out + kBM - 1) / kBM;
    g.frames = d.N * (d.dims == 3 ? d.D : 1);
    const int H_out = p->H_out, W_out = p->W_out;
    // the generic channels-last epilogue (3D layers, C_out >= 96) stages 2 KB per warp, which leaves
    // room for a seventh weight-ring stage in the dominant layers; the other epilogues (and NCHW
    // output, possible for the 2D plans) stage up to 4.5 KB
    g.stage_warp = g.stn ? kStnStageBytes
                         : ((!small_cout && !g.kwm && !g.ctr && !g.nchw) ? kStageGenericBytes : kStageWarpBytes);
    const int fixed = 1024 + 4 * g.stage_warp + 512 + (g.nchw ? 4 * 32 * 16 : 0);
    bool found = false;
    long long best_cost = -1;
    int cands[80], nc = 0;
    for (int k = 1; k <= 64; ++k) cands[nc++] = (W_out + k - 1) / k;
    if (g.s2) {  // P = Wt + 1 divides 256
        cands[nc++] = 31; cands[nc++] = 63; cands[nc++] = 127;
    } else {     // P = Wt + 2 divides 256
        cands[nc++] = 30; cands[nc++] = 62; cands[nc++] = 126; cands[nc++] = 254;
    }
    // layers with at most 64 output channels (when asked for): the M = 64 form with every weight block
    // resident in shared memory; if no tiling leaves room for them, the 128-row form
    g.m64 = (small_cout && d.C_out <= 64 && !g.nchw && !g.kwm && !g.ctr) ? 1 : 0;
    if (g.m64) g.n_tiles = 1;
    constexpr int HR_TN = 6;
    // 2D layers with at most 80 output channels (when asked for), stride 1: positions as M with the
    // horizontal taps in N (TN), unless X3CONV_TN=0; falls back to the M = 64 form when no tiling fits
    {
        const char* tn_env = getenv("X3CONV_TN");
        const int cp = (d.C_out + 15) / 16 * 16;
        if (small_cout && d.dims == 2 && !g.s2 && !g.nchw && !g.kwm && !g.ctr && d.C_out <= 80 &&
            !(tn_env && !strcmp(tn_env, "0"))) {
            // eight input channels: the taps in K (TK), N = the output channels
            const bool tk = d.C_in == 8 && !(getenv("X3CONV_TK") && !strcmp(getenv("X3CONV_TK"), "0"));
            const int tn_n = tk ? cp : 3 * cp;
            // eight epilogue warps, each holding a copy of the bias; with 64 channels each also stages its
            // raster row (32 positions x 128 B, 1024-aligned) for a TMA store, other widths store straight
            // from registers
            const int x_bytes = 32 * cp;
            const int wres = tk ? 5 * tn_n * 32 : g.KT * g.n_chunks * 3 * tn_n * 128;
            int stage_warp = cp == 64 ? 4096 : 0;
            if (stage_warp && 1024 + 8 * stage_warp + 512 + x_bytes + wres + 2 * (HR_TN + 1) * 32 * 128 > kSmemLimit)
                stage_warp = 0;  // no room for the row buffers next to two halo stages: direct stores
            const int tfixed = 1024 + 8 * stage_warp + 512 + x_bytes;
            // pitch 32: a tile (128 positions) is four whole raster rows of 30 output columns and two
            // junk columns, one row per TMEM lane quarter; the halo is those rows plus one above and
            // one below (six rows of 32 positions)
            // TK: 16 bytes per position, and one more row: the pairs' second taps read up to two
            // positions past the 192 (junk outputs only)
            const int P = 32, Wt = 30, HR = tk ? HR_TN + 1 : HR_TN;
            const int h_bytes = tk ? (HR * P * 16 + 1023) / 1024 * 1024 : HR * P * 128;
            int n_h = (kSmemLimit - tfixed - wres) / h_bytes;
            if (n_h > 4) n_h = 4;
            long long best = -1;
            if (n_h >= 2) {
                best = 0;
                g.Wt = Wt; g.P = P; g.HR = HR; g.h_bytes = h_bytes; g.h_tx_bytes = (tk ? 8 : kCK) * 2 * P * HR;
                g.n_h = n_h; g.n_w = 1; g.strips = (W_out + Wt - 1) / Wt; g.windows = (H_out + 3) / 4;
                g.tiles = (long long)g.strips * g.windows * g.frames;
                g.w_smem = wres; g.n_raw = 0; g.raw_w = g.raw_bytes = g.raw_tx_bytes = 0;
                g.stage_warp = stage_warp; g.x_bytes = x_bytes;
                g.smem_bytes = tfixed + n_h * h_bytes + wres;
            }
            if (best >= 0) {
                g.tn = 1; g.tk = tk ? 1 : 0; g.tn_cp = cp; g.tn_n = tn_n; g.m64 = 0; g.n_tiles = 1; g.win_adv = 128;
                found = true;
            }
        }
    }
    int stn_ctas = 0;
    if (g.stn) {
        // stencil head: 32 x 8 raster windows (pitch 32: one halo column on each side of 30 output
        // columns). Each CTA runs a stretch of consecutive windows down the strips, every window for
        // the output frames of its group, the windows of one strip abutting (the seams are joined by
        // row sums the epilogue carries, one set per output frame)
        g.Wt = 30; g.P = 32; g.HR = kStnRows;
        g.strips = (W_out + 29) / 30;
        g.win_adv = kBNP;
        g.h_bytes = g.h_tx_bytes = kCtrW + kWBlock;
        // frame groups: the fewest frames per CTA (a divisor of the frame count) that leave no more
        // groups than CTAs
        const int ctas = num_sms < kStnMaxCtas ? num_sms : kStnMaxCtas;
        int fpc = 1;
        while (g.frames % fpc != 0 || g.frames / fpc > ctas) ++fpc;
        g.stn_fpc = fpc;
        g.stn_groups = g.frames / fpc;
        g.x_bytes = 4 * fpc * kStnCarryBytes;
        const int room = kSmemLimit - fixed - g.x_bytes;
        g.n_h = room / g.h_bytes < 4 ? room / g.h_bytes : 4;
        g.n_w = 1;
        g.w_smem = 0;
        g.smem_bytes = fixed + g.x_bytes + g.n_h * g.h_bytes;
        if (g.n_h < 2 || H_out > 0xFFFF || g.strips > 0xFFFF) return false;
        // Segments: with fewer strips than runs, each strip is cut into k row segments so that there
        // are about as many segments as runs (segments at least 16 rows). Runs: with at least as many
        // segments as runs, round j of whole segments gives segment r + j R to run r (R runs side by
        // side: neighbouring strips, same rows); the segments left after the whole rounds (or all of
        // them) are cut greedily into the fewest windows per run with which the runs cover them: a run
        // takes whole segment remainders while its windows last ((rows + 2) / 8 rounded up), else the
        // 8 n - 2 rows its last n windows yield, and the next run starts below them
        const int runs_max = ctas / g.stn_groups;
        int k = g.strips < runs_max ? (runs_max + g.strips - 1) / g.strips : 1;
        int seg_rows = (H_out + k - 1) / k;
        // a segment of rows + 2 = 8 n input rows fills its windows exactly
        if (k > 1) seg_rows += (6 - seg_rows % 8 + 8) % 8;
        if (seg_rows < 16) seg_rows = H_out < 16 ? H_out : 16;
        k = (H_out + seg_rows - 1) / seg_rows;
        const int nseg = g.strips * k;
        if (nseg > 0xFFFF) return false;
        auto seg_bounds = [&](int sg, int& lo, int& hi) {
            lo = (sg / g.strips) * seg_rows;
            hi = lo + seg_rows < H_out ? lo + seg_rows : H_out;
        };
        const bool rounds = nseg >= runs_max;
        const int R = rounds ? runs_max : 0;
        g.stn_full = rounds ? nseg / runs_max : 0;
        const int left0 = g.stn_full * R;  // first segment of the greedy part
        long long windows = 0;
        std::vector<int> per_run(runs_max, 0);
        for (int r = 0; r < R; ++r)
            for (int j = 0; j < g.stn_full; ++j) {
                int lo, hi;
                seg_bounds(r + j * R, lo, hi);
                per_run[r] += (hi - lo + 9) >> 3;
            }
        for (int r = 0; r < R; ++r) windows += per_run[r];
        // the segments left after the whole rounds: the smallest window count T per run with which
        // the runs, each taking up to T minus its whole-segment windows, cover them greedily
        int runs = R;
        int T = 0;
        for (int r = 0; r < runs_max; ++r) T = per_run[r] > T ? per_run[r] : T;
        if (left0 < nseg) {
            for (;; ++T) {
                int sg = left0, o = 0, used = 0;
                long long wsum = 0;
                {
                    int lo, hi;
                    seg_bounds(sg, lo, hi);
                    o = lo;
                }
                std::vector<int> add(runs_max, 0);
                for (int c = 0; c < runs_max && sg < nseg; ++c) {
                    const int cap = T - per_run[c];
                    if (cap <= 0) {
                        g.stn_start[c] = (uint32_t)nseg << 16;
                        continue;
                    }
                    g.stn_start[c] = ((uint32_t)sg << 16) | (uint32_t)o;
                    used = c + 1;
                    for (int rem = cap; rem > 0 && sg < nseg;) {
                        int lo, hi;
                        seg_bounds(sg, lo, hi);
                        const int need = (hi - o + 9) >> 3;
                        if (need <= rem) {
                            rem -= need;
                            wsum += need;
                            add[c] += need;
                            ++sg;
                            if (sg < nseg) {
                                seg_bounds(sg, lo, hi);
                                o = lo;
                            }
                        } else {
                            o += kStnRows * rem - 2;
                            wsum += rem;
                            add[c] += rem;
                            rem = 0;
                        }
                    }
                }
                if (sg >= nseg) {
                    windows += wsum;
                    for (int c = 0; c < runs_max; ++c) per_run[c] += add[c];
                    for (int c = used; c < runs_max; ++c) g.stn_start[c] = (uint32_t)nseg << 16;
                    if (!rounds) runs = used;
                    break;
                }
            }
        } else {
            for (int c = 0; c < runs_max; ++c) g.stn_start[c] = (uint32_t)nseg << 16;
        }
        g.stn_runs = R;
        g.stn_nseg = nseg;
        g.stn_seg_rows = seg_rows;
        g.stn_n = 0;
        for (int r = 0; r < runs_max; ++r) g.stn_n = per_run[r] > g.stn_n ? per_run[r] : g.stn_n;
        stn_ctas = runs * g.stn_groups;
        g.windows = g.stn_n;
        g.tiles = windows * g.frames;
        found = true;
    } else if (g.ctr) {
        // the centre tap needs no halo: a window is 256 consecutive positions of a frame's flattened
        // H x W plane (one strip as wide as the image, rows of pitch W), staged by one 32 KB box
        g.Wt = g.P = W_out; g.HR = 1; g.strips = 1;
        g.windows = (int)(((long long)H_out * W_out + kBNP - 1) / kBNP);
        // each stage holds the window (32 KB) and the (kt, chunk) weight block (16 KB) behind one barrier
        g.h_bytes = g.h_tx_bytes = kCtrW + kWBlock;
        g.n_h = 4; g.n_w = 1;
        g.w_smem = 0;
        g.smem_bytes = fixed + g.n_h * g.h_bytes + g.w_smem;
        if (g.smem_bytes > kSmemLimit) return false;
        g.tiles = (long long)g.windows * g.frames;
        found = true;
    }
  for (int attempt = 0; attempt < 2 && !found && !g.ctr && !g.tn; ++attempt) {
    if (attempt == 1) {
        if (!g.m64) break;
        g.m64 = 0;
        g.n_tiles = (d.C_out + kBM - 1) / kBM;
    }
    const int wres = g.m64 ? g.KT * g.n_chunks * 9 * kWBlock64 : 0;
    const bool light = g.m64 && d.C_in <= 16;
    for (int ci = 0; ci < nc; ++ci) {
        const int Wt = g.nchw ? (cands[ci] + 7) / 8 * 8 : cands[ci];  // NCHW: strips start 16-byte aligned
        // stride 2: tap shifts of 0 or 1 in each phase raster, and the phase boxes span 2P x 2HR
        // input positions (a box side is at most 256)
        const int P = g.s2 ? Wt + 1 : Wt + 2;
        if (P > (g.s2 ? 128 : 256) || (g.nchw && Wt + 16 > 256)) continue;
        // halo rows of a 256-position window starting anywhere in a row, plus one above and below
        // furthest B row read: window start offset within its row (0 when windows of 256 tile the
        // rows exactly), the window's last column, kh = 2 (+2P) and, unless folded into M, kw = 2 (+2)
        const int pos_off_max = (g.win_adv == 256 && (256 % P) == 0) ? 0 : P - 1;
        const int need_pos = g.s2 ? pos_off_max + 255 + P + 1 + 1 : pos_off_max + 255 + 2 * P + (g.kwm ? 0 : 2) + 1;
        const int HR = (need_pos + P - 1) / P;
        if (HR > (g.s2 ? 128 : 256)) continue;
        const int pos = HR * P > need_pos ? HR * P : need_pos;
        const int h_bytes = (pos * 128 + 1023) / 1024 * 1024;
        // NCHW raw slices: 16 channels x HR rows x (Wt + 16) columns, two stages
        const int raw_w = Wt + 16;
        const int raw_bytes = g.nchw ? (16 * HR * raw_w * 2 + 127) / 128 * 128 : 0;
        int n_raw = 0;
        if (g.nchw) {
            n_raw = 2;
            while (n_raw < 4 && fixed + 2 * h_bytes + (n_raw + 1) * raw_bytes + 3 * kWBlock <= kSmemLimit) ++n_raw;
        }
        int n_w = (kSmemLimit - fixed - 2 * h_bytes - n_raw * raw_bytes) / kWBlock;
        if (n_w > 7) n_w = 7;
        int n_h = 2;
        if (g.m64) {
            if (fixed + 2 * h_bytes + wres > kSmemLimit) continue;
            n_w = 7;  // no weight ring: rank as the deepest one
            // at most 16 input channels: one K step per tap, so a tile's MMAs take less time than a
            // halo load's latency; stage as many halos ahead as fit
            if (light) n_h = (int)((kSmemLimit - fixed - wres) / h_bytes) < 4 ? (int)((kSmemLimit - fixed - wres) / h_bytes) : 4;
        }
        if (n_w < 3) continue;
        const int strips = (W_out + Wt - 1) / Wt;
        const int windows = (int)(((long long)H_out * P + g.win_adv - 1) / g.win_adv);
        const long long tiles = (long long)strips * windows * g.frames * g.n_tiles;
        const long long waves = (tiles + num_sms - 1) / num_sms;
        // every tile costs the same MMA work: rank by waves, then by weight-ring depth and halo size
        // (light M = 64 layers: by halo pipeline depth first)
        const long long cost = (light ? (4 - n_h) * 10000000LL : 0) + waves * 100000 + (7 - n_w) * 10000 +
                               (g.nchw ? (4 - n_raw) * 20000 : 0) + (long long)HR * P;
        if (!found || cost < best_cost) {
            found = true;
            best_cost = cost;
            g.Wt = Wt; g.P = P; g.HR = HR; g.h_bytes = h_bytes; g.h_tx_bytes = kCK * 2 * P * HR;
            g.n_h = n_h; g.n_w = g.m64 ? 1 : n_w; g.strips = strips; g.windows = windows; g.tiles = tiles;
            g.raw_w = g.nchw ? raw_w : 0; g.raw_bytes = raw_bytes; g.n_raw = n_raw;
            g.raw_tx_bytes = g.nchw ? 16 * HR * raw_w * 2 : 0;
            g.w_smem = g.m64 ? wres : n_w * kWBlock;
            g.smem_bytes = fixed + n_h * h_bytes + g.w_smem + n_raw * raw_bytes;
        }
    }
  }
    if (!found) return false;
    // Causal channels-last layers with one output tile can run in the two-window form (W2), taken
    // only with X3CONV_W2=1. A probe had put a second MMA on the same A operand at ~104 cycles
    // against ~200, but the form measured slower on the 352x624 128->128 layer (1.151 against 1.089
    // ms per two launches): its weight ring is three blocks deep, a tile is twice as long, and the
    // epilogue no longer overlaps the MMAs.
    const char* w2_env = getenv("X3CONV_W2");
    if (!g.kwm && !g.nchw && !g.ctr && !g.m64 && g.n_tiles == 1 && d.dims == 3 && !small_cout &&
        w2_env && !strcmp(w2_env, "1")) {
        double best = 1e30;
        for (int ci = 0; ci < nc; ++ci) {
            const int Wt = cands[ci];
            const int P = Wt + 2;
            if (P > 256) continue;
            const int pos_off_max = (512 % P) == 0 ? 0 : P - 1;
            const int need_pos = pos_off_max + 511 + 2 * P + 2 + 1;
            const int HR = (need_pos + P - 1) / P;
            if (HR > 256) continue;
            const int pos = HR * P > need_pos ? HR * P : need_pos;
            const int h_bytes = (pos * 128 + 1023) / 1024 * 1024;
            int n_w = (kSmemLimit - fixed - 2 * h_bytes) / kWBlock;
            if (n_w > 6) n_w = 6;
            if (n_w < 3) continue;
            const int strips = (W_out + Wt - 1) / Wt;
            const int windows = (int)(((long long)H_out * P + 511) / 512);
            const long long tiles = (long long)strips * windows * g.frames;
            const double est = (double)((tiles + num_sms - 1) / num_sms) + 0.001 * (6 - n_w);
            if (est < best) {
                best = est;
                g.w2 = 1; g.win_adv = 512;
                g.Wt = Wt; g.P = P; g.HR = HR; g.h_bytes = h_bytes; g.h_tx_bytes = kCK * 2 * P * HR;
                g.n_h = 2; g.n_w = n_w; g.strips = strips; g.windows = windows; g.tiles = tiles;
                g.w_smem = n_w * kWBlock;
                g.smem_bytes = fixed + 2 * h_bytes + g.w_smem;
            }
        }
    }
    if (g.tiles >= (1LL << 31)) return false;  // the kernel decodes tile indices in 32 bits
    g.grid = g.stn ? stn_ctas : (int)(g.tiles < num_sms ? g.tiles : num_sms);
    p->cl = g;
    // the packed weight blocks are the generic packer's layout with BN = 128, CK = 64 (the head form
    // has its own packer: 3 kh blocks per chunk with (kw, channel) rows)
    p->g.BN = g.m64 ? 64 : kBM; p->g.CK = kCK; p->g.n_chunks = g.n_chunks; p->g.n_tiles = g.n_tiles; p->g.KT = g.KT;
    p->g.b_bytes = g.tn ? g.tn_n * 128 : (g.m64 ? kWBlock64 : kWBlock);
    return true;
}

namespace {

// One launch of the engine for descriptor d (its layout, C_in and stride as the kernel sees them)
// with tiling g over an H_out x W_out raster; the stored plane is yH x yW.
x3_status launch_cl(const x3_conv_desc& d, const ClGeom& g, int H_out, int W_out, int yH, int yW, int out_nchw, int row_shift,
                    const void* x, const void* carry, const void* w_packed, const void* bias, void* y, cudaStream_t s) {
    const bool bf16 = d.dtype == X3_BF16;
    ClArgs a;
    memset(&a, 0, sizeof a);
    a.C_in = d.C_in; a.C_out = d.C_out; a.N = d.N; a.D = d.D; a.H = d.H; a.W = d.W;
    a.H_out = H_out; a.W_out = W_out; a.dout = d.dims == 3 ? d.D : 1; a.act = d.act;
    a.sub2 = g.sub2; a.out_nchw = out_nchw; a.yH = yH; a.yW = yW; a.w_smem = g.w_smem;
    a.stage_warp = g.stage_warp;
    a.tn_cp = g.tn_cp; a.tn_n = g.tn_n; a.x_bytes = g.x_bytes;
    a.row_shift = row_shift;
    if (g.stn) {
        a.stn_n = g.stn_n;
        a.stn_fpc = g.stn_fpc;
        a.stn_full = g.stn_full;
        a.stn_runs = g.stn_runs;
        a.stn_nseg = g.stn_nseg;
        a.stn_seg_rows = g.stn_seg_rows;
        a.fd_fpc = make_fastdiv((uint32_t)g.stn_fpc);
        a.fd_groups = make_fastdiv((uint32_t)g.stn_groups);
        memcpy(a.stn_start, g.stn_start, sizeof a.stn_start);
    }
    a.frame_inner = g.ctr ? 1 : 0;
    // causal channels-last layers whose passes have an even number of frames: frame pairs, unless
    // X3CONV_FRAME_PAIRS=0 (the tiles and their sums are the same; only the order changes)
    {
        const char* fp = getenv("X3CONV_FRAME_PAIRS");
        if (!g.ctr && !g.tn && !g.nchw && !g.w2 && g.KT == 3 && d.dims == 3 && (d.D % 2) == 0 &&
            !(fp && !strcmp(fp, "0")))
            a.frame_inner = 2;
    }
    a.g_f32 = d.kernel == X3_KERNEL_HEAD_SPLIT ? 1 : 0;
    a.has_carry = carry != nullptr;
    a.KT = g.KT; a.n_chunks = g.n_chunks; a.n_tiles = g.n_tiles; a.Wt = g.Wt; a.P = g.P; a.HR = g.HR;
    a.strips = g.strips; a.windows = g.windows; a.frames = g.frames; a.h_bytes = g.h_bytes;
    a.h_tx_bytes = g.h_tx_bytes; a.n_h = g.n_h; a.n_w = g.n_w; a.tiles = g.tiles;
    a.win_adv = g.win_adv; a.ngroups = g.ngroups;
    a.raw_w = g.raw_w; a.raw_bytes = g.raw_bytes; a.raw_tx_bytes = g.raw_tx_bytes; a.n_raw = g.n_raw;
    a.idesc = g.tn ? ptx::idesc_f16(kBM, g.tn_n, bf16) : ptx::idesc_f16(g.m64 ? 64 : kBM, kBNP, bf16);
    a.fd_frames = make_fastdiv((uint32_t)g.frames);
    a.fd_ntiles = make_fastdiv((uint32_t)g.n_tiles);
    a.fd_windows = make_fastdiv((uint32_t)g.windows);
    a.fd_strips = make_fastdiv((uint32_t)g.strips);
    a.fd_dout = make_fastdiv((uint32_t)a.dout);
    a.fd_P = make_fastdiv((uint32_t)g.P);
    a.fd_chunks = make_fastdiv((uint32_t)g.n_chunks);
    a.w = (const uint8_t*)w_packed; a.bias = bias; a.y = y;
    x3_status st0 = device_status_word(&a.status);
    if (st0 != X3_OK) return st0;
    CUtensorMap mx, mc;
    x3_status st;
    if (g.nchw) {
        st = encode_nchw_raw(&mx, bf16, x, d.W, d.H, d.C_in, d.N, (uint32_t)g.raw_w, (uint32_t)g.HR);
        if (st != X3_OK) return st;
        mc = mx;
    } else {
        const uint64_t frames_x = (uint64_t)d.N * (d.dims == 3 ? d.D : 1);
        // the flat form views each frame as one row of H*W positions
        const bool flat = g.ctr && !g.stn;
        const uint64_t mw = flat ? (uint64_t)d.H * d.W : (uint64_t)d.W, mh = flat ? 1 : (uint64_t)d.H;
        const uint32_t bw = flat ? (uint32_t)kBNP : (uint32_t)g.P, bh = flat ? 1u : (uint32_t)g.HR;
        st = encode_sw128(&mx, bf16, x, d.C_in, mw, mh, frames_x, bw, bh, g.s2 ? 2u : 1u, g.tk != 0);
        if (st != X3_OK) return st;
        if (carry) {
            st = encode_sw128(&mc, bf16, carry, d.C_in, mw, mh, (uint64_t)d.N * 2, bw, bh, 1u, g.tk != 0);
            if (st != X3_OK) return st;
        } else {
            mc = mx;
        }
    }
    // TN, 64 output channels, channels-last output, stride 1: the output's tensor map for the row stores
    CUtensorMap my;
    memcpy(&my, &mx, sizeof my);
    if (g.tn && g.stage_warp >= 4096 && d.C_out == 64 && !out_nchw && !g.sub2 &&
        (d.dims == 2 ? d.layout == X3_NHWC : d.layout == X3_NDHWC)) {
        const uint64_t frames_y = (uint64_t)d.N * (d.dims == 3 ? d.D : 1);
        st = encode_sw128(&my, bf16, y, 64, (uint64_t)yW, (uint64_t)yH, frames_y, 30u, 1u);
        if (st != X3_OK) return st;
        a.tn_tma = 1;
    }
    void (*k)(CUtensorMap, CUtensorMap, CUtensorMap, ClArgs);
    if (g.tk) k = bf16 ? igemm_cl_kernel<true, false, false, false, false, false, false, false, true, true>
                       : igemm_cl_kernel<false, false, false, false, false, false, false, false, true, true>;
    else if (g.tn) k = bf16 ? igemm_cl_kernel<true, false, false, false, false, false, false, false, true>
                       : igemm_cl_kernel<false, false, false, false, false, false, false, false, true>;
    else if (g.w2) k = bf16 ? igemm_cl_kernel<true, false, false, false, false, true>
                       : igemm_cl_kernel<false, false, false, false, false, true>;
    else if (g.stn) k = igemm_cl_kernel<true, false, false, true, false, false, true>;
    else if (g.ctr) k = igemm_cl_kernel<true, false, false, true>;  // bf16 only (checked by the planner)
    else if (g.s2 && g.m64) k = bf16 ? igemm_cl_kernel<true, false, false, false, true, false, false, true>
                                     : igemm_cl_kernel<false, false, false, false, true, false, false, true>;
    else if (g.s2) k = bf16 ? igemm_cl_kernel<true, false, false, false, false, false, false, true>
                            : igemm_cl_kernel<false, false, false, false, false, false, false, true>;
    else if (g.m64) k = bf16 ? igemm_cl_kernel<true, false, false, false, true> : igemm_cl_kernel<false, false, false, false, true>;
    else if (g.nchw) k = bf16 ? igemm_cl_kernel<true, false, true> : igemm_cl_kernel<false, false, true>;
    else if (g.kwm) k = bf16 ? igemm_cl_kernel<true, true, false> : igemm_cl_kernel<false, true, false>;
    else k = bf16 ? igemm_cl_kernel<true, false, false> : igemm_cl_kernel<false, false, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "igemm_cl smem attribute: %s", cudaGetErrorString(e));
    // a programmatic dependent of the previous kernel in the stream (the kernel waits for it before
    // touching global memory)
    const bool pdl = pdl_enabled();
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)g.grid);
    cfg.blockDim = dim3((g.nchw || g.tn) ? 320u : 192u);
    cfg.dynamicSmemBytes = (size_t)g.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, k, mx, mc, my, a);
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "igemm_cl launch: %s", cudaGetErrorString(e));
    return X3_OK;
}

}  // namespace

x3_status launch_igemm_cl(const x3_conv_plan* p, const void* x, const void* carry, const void* w_packed,
                          const void* bias, void* y, cudaStream_t s) {
    // stride 2 as sub2: the raster covers the input plane, the stored plane is the output
    const int rh = p->cl.sub2 ? p->d.H : p->H_out, rw = p->cl.sub2 ? p->d.W : p->W_out;
    return launch_cl(p->d, p->cl, rh, rw, p->H_out, p->W_out, 0, p->row_shift, x, carry, w_packed, bias, y, s);
}

x3_status launch_igemm_cl_shadow(const x3_conv_plan* p, const void* x, const void* w_packed, const void* bias,
                                 void* y, int out_nchw, cudaStream_t s) {
    if (!p->has_shadow) return fail(X3_ERR_UNSUPPORTED, "layer has no channels-last form");
    x3_conv_desc d = p->d;
    d.layout = X3_NHWC;
    d.C_in = (d.C_in + 7) / 8 * 8;
    // S2: the raster is the output plane; sub2: the stride-1 raster over the input plane
    const int rh = p->cl_shadow.s2 ? p->H_out : d.H, rw = p->cl_shadow.s2 ? p->W_out : d.W;
    return launch_cl(d, p->cl_shadow, rh, rw, p->H_out, p->W_out, out_nchw, 0, x, nullptr,
                     (const uint8_t*)w_packed + p->shadow_w_off, bias, y, s);
}

}  // namespace x3
