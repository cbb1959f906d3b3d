// Internal definitions shared by the host API and the kernels of libx3conv.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "x3conv.h"

namespace x3 {

enum KernelKind { K_DIRECT = 0, K_IGEMM = 1, K_IGEMM_CL = 2, K_HEAD_TWO_PASS = 3 };

// A-operand staging modes of the implicit-GEMM engine.
enum StageMode {
    STAGE_CL = 0,    // channels-last input: TMA writes the halo straight into K-major planes
    STAGE_NCHW = 1   // channels-first 2D input: TMA loads a raw tile, warps transpose it
};

// Tiling of the tcgen05 implicit GEMM. A tile is Rt output rows x Wt output columns of one output
// frame and BN output channels. Its halo (Rt+2 rows x P columns, P = Wt + 2) sits in shared
// memory as a raster of positions; output raster position m = r*P + c (c < Wt valid) reads halo
// position m + kh*P + kw for tap (kh, kw). The tile's M rows are NSUB subtiles of 128 raster
// positions starting at sub_off(s).
struct IgemmGeom {
    int mode;          // StageMode
    int BN;            // output channels per tile (16, 64 or 128)
    int n_tiles;       // ceil(C_out / BN)
    int CK;            // input channels per staged chunk (16 or 32)
    int n_chunks;      // ceil(C_in / CK)
    int KT;            // temporal taps: 3 (causal 3D) or 1 (2D)
    int NSUB;          // 128-row MMA subtiles per tile
    int Rt, Wt, P;     // output rows / columns per tile, halo raster pitch in positions
    int spr;           // row-aligned subtile mapping: subtiles per output row; 0 = flat (128*s)
    int halo_rows;     // rows per staged plane: Rt + 2 (stride 1) or Rt + 1 per phase plane (stride 2)
    int stride;        // 1, or 2 (NCHW only: four phase planes)
    int raw_rows;      // NCHW: rows of the raw tile (Rt + 2, or 2 Rt + 1 for stride 2)
    int phase_stride;  // bytes between the phase planes of a stride-2 stage
    int plane_pos;     // positions per K-major plane (halo_rows * P)
    int plane_stride;  // bytes between planes (plane_pos * 16)
    int a_bytes;       // bytes of one A stage (CK/8 planes + read slack)
    int a_tx_bytes;    // bytes the TMA writes into one A stage
    int raw_w;         // NCHW: columns of the raw tile (Wt + 16)
    int raw_bytes;     // NCHW: bytes of one raw stage
    int b_bytes;       // bytes of one packed weight block (BN x CK)
    int n_a, n_b, n_raw; // pipeline depths
    int tmem_cols;     // TMEM columns allocated (power of two >= 32)
    int scr_pitch;     // epilogue scratch row pitch (bytes) for coalesced channels-last stores; 0 = none
    int acc_bufs;      // accumulator buffers in TMEM (1 or 2)
    int col_tiles, row_tiles, frames;
    long long tiles;   // col_tiles * row_tiles * frames * n_tiles
    int smem_bytes;    // dynamic shared memory per CTA
    int grid;          // persistent CTAs
};

// Tiling of the channels-last engine with output channels as M (128 per tile) and 256 output
// positions as N: vertical strips Wt columns wide walked as rasters of pitch P = Wt + 2, a tile being
// a window of 256 consecutive raster positions of one frame; the halo of a window (HR rows of P
// positions, 64 channels, 128-byte swizzle) is staged once per temporal tap and channel chunk.
constexpr int kStnMaxCtas = 256;  // stencil head: most CTAs of one launch (one run of windows each)

struct ClGeom {
    int KT, n_chunks, n_tiles;   // temporal taps, 64-channel chunks, 128-channel output tiles
    int Wt, P, HR;               // strip width, raster pitch, halo rows staged per window
    int strips, windows, frames; // tiles = strips * windows * frames * n_tiles
    int h_bytes, h_tx_bytes;     // bytes of one halo stage (1024-aligned) / written by its TMA box
    int n_h, n_w;                // halo stages, weight-block stages
    int kwm;                     // 1: kw folded into M (the conv_out head form, unpatchify epilogue)
    int nchw;                    // 1: NCHW 2D input/output (raw slices transposed in shared memory)
    int raw_w, raw_bytes, raw_tx_bytes, n_raw;  // NCHW raw-slice staging
    int win_adv;                 // raster positions between consecutive windows (256, or 254 when kwm)
    int ngroups;                 // kwm: groups of 10 output channels (one TMEM lane quarter each)
    int ctr;                     // 1: centre spatial tap only (temporal pass of the two-pass head)
    int sub2;                    // 1: stride 2 computed as the stride-1 raster, even positions kept
    int s2;                      // 1: stride 2 from the four input phases (element-strided TMA boxes)
    int m64;                     // 1: M = 64 MMAs (at most 64 output channels), weights resident
    int w_smem;                  // shared-memory bytes for weights (the ring, or all blocks when m64)
    int w2;                      // 1: a tile is two consecutive windows sharing every weight K slice
    int stn;                     // 1: head with the spatial stencil in the epilogue (centre-tap MMAs)
    int stage_warp;              // epilogue staging bytes per warp
    int tn;                      // 1: positions as M (128 per tile), the three horizontal taps in N
    int tn_cp, tn_n;             // tn: output channels padded to 16; MMA N = 3 * tn_cp (tk: tn_cp)
    int tk;                      // 1 (with tn): 8 input channels, two taps per 16-wide K step
    int x_bytes;                 // tn: the epilogue warps' bias copies; stn: their row carries
    long long tiles;
    int smem_bytes, grid;
    // stn: the output frames are split into stn_groups groups of stn_fpc; CTA c runs group c % groups
    // over run c / groups: at most stn_n consecutive windows, first stn_full whole row segments (run,
    // run + stn_runs, ...), then from segment stn_start[run] >> 16, output row stn_start[run] & 0xFFFF,
    // down that segment and on through the next ones
    int stn_n, stn_fpc, stn_groups;
    int stn_full, stn_runs;  // stn: rounds of whole segments per run, and the runs side by side in them
    int stn_nseg, stn_seg_rows;  // stn: row segments (part p of strip s is p * strips + s) and rows each
    uint32_t stn_start[kStnMaxCtas];
};

}  // namespace x3

struct x3_conv_plan {
    x3_conv_desc d;
    int H_out, W_out;
    x3::KernelKind kind;
    x3::IgemmGeom g;
    x3::ClGeom cl;
    size_t packed_bytes;
    int num_sms;
    // Banded mode: 1 when the input's first row is the halo row above the band (band_lo > 0), so
    // output row r reads input rows r + kh (instead of r + kh - 1, whose -1 is the zero padding)
    int row_shift;
    // Channels-last form of a 2D NCHW layer, used by the stack driver for the layers between the
    // first input and the last output: input NHWC with C_in rounded up to 8, stride 1 (stride 2 as
    // sub2). Its packed weights start at shadow_w_off bytes into the layer's packed buffer.
    int has_shadow;
    x3::ClGeom cl_shadow;
    size_t shadow_w_off;
};

namespace x3 {

// Set the thread-local error string and return the status.
x3_status fail(x3_status s, const char* fmt, ...);

// Bytes per element of the storage types.
inline int elem_bytes(x3_dtype) { return 2; }

// Elements of one activation tensor / frame.
size_t in_elems(const x3_conv_plan* p);
size_t out_elems(const x3_conv_plan* p);

// Kernel launchers (return X3_OK or an error with the message set).
x3_status launch_pack_weights(const x3_conv_plan* p, const void* w, void* w_packed, cudaStream_t s);
x3_status launch_direct(const x3_conv_plan* p, const void* x, const void* carry, const void* w_packed,
                        const void* bias, void* y, cudaStream_t s);
x3_status launch_igemm(const x3_conv_plan* p, const void* x, const void* carry, const void* w_packed,
                       const void* bias, void* y, cudaStream_t s);
bool igemm_plan(x3_conv_plan* p, int num_sms);  // fills p->g; false if the engine can't run it
// Fills p->cl (+ packing fields of p->g); small_cout also accepts channels-last layers with fewer
// than 96 output channels (the M tile is then partly empty).
bool igemm_cl_plan(x3_conv_plan* p, int num_sms, bool small_cout = false);
// Bytes of the packed weights of the channels-last engine with tiling g (all its forms but the head
// forms, which pack their own layouts).
size_t cl_packed_bytes(const ClGeom& g);
x3_status launch_igemm_cl(const x3_conv_plan* p, const void* x, const void* carry, const void* w_packed,
                          const void* bias, void* y, cudaStream_t s);
// The channels-last form (cl_shadow) of a 2D NCHW layer: x is NHWC with C_in rounded up to 8
// channels; y is NHWC, or NCHW when out_nchw. w_packed is the layer's packed buffer.
x3_status launch_igemm_cl_shadow(const x3_conv_plan* p, const void* x, const void* w_packed, const void* bias,
                                 void* y, int out_nchw, cudaStream_t s);
// NCHW [N][C][H][W] -> NHWC [N][H][W][C8], channels C..C8-1 zero.
x3_status launch_nchw_to_nhwc(const void* x, void* y, int N, int C, int C8, int H, int W, cudaStream_t s);
// Carry update of a channels-last causal layer, launched as a programmatic dependent of the layer's
// kernel (layout.cu); requires that kernel to signal only after its reads of the carry.
x3_status launch_carry_update(const void* input, void* carry, int N, int D, size_t frame_bytes, int history_valid,
                              int num_sms, cudaStream_t s);
// Programmatic dependent launches on (X3CONV_PDL unset or not "0").
bool pdl_enabled();
// Two-pass head: temporal pass into the 112-channel g plane, then the spatial stencil.
x3_status launch_head_stencil(const x3_conv_plan* p, const void* g, const void* bias, void* y, cudaStream_t s);
x3_status read_device_status(int reset);
x3_status selftest_wait_timeout(int limit_ms, cudaStream_t s);
x3_status device_status_word(unsigned int** out);  // device address of the timeout status word

}  // namespace x3
