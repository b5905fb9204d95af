// conv_internal.h -- host-side plan and launch interfaces between the C ABI
// (conv_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "conv.h"
#include "conv_common.cuh"

namespace conv {

// CUDA-core implicit GEMM tiles: output channels (BM) x pixels (BN) per block,
// TM x TN outputs per thread.
struct FfmaCfg {
  int bm, bn, tm, tn;
  int threads() const { return (bm / tm) * (bn / tn); }
};
constexpr int kFfmaBK = 16;         // k terms per pipeline stage
constexpr int kFfmaBKU = 16;        // k terms per stage with unfolded B (16-byte copies only)
constexpr int kFfmaStages = 4;      // pipeline depth
constexpr int kFfmaKTab = 2304;     // k entries of the window table per segment
constexpr int kNumFfmaCfgs = 9;
constexpr FfmaCfg kFfmaCfgs[kNumFfmaCfgs] = {
    {128, 128, 8, 8}, {64, 128, 8, 8}, {128, 64, 8, 8}, {64, 64, 4, 4}, {32, 256, 4, 8},
    {16, 256, 4, 8},  {40, 128, 8, 4}, {16, 64, 4, 4},  {40, 64, 8, 4}};
// Registers a thread of a config is planned with (the kernel's cap).
constexpr int ffma_cfg_regs(const FfmaCfg& c) {
  return c.tm * c.tn + 64 > 255 ? 255 : c.tm * c.tn + 64;
}

size_t ffma_smem_bytes(int cfg, int k_per_block, bool unfolded);  // k_per_block: terms one block sums
int ffma_ktab_entries(int k_per_block);

// The B operand of the CUDA-core kernel.
constexpr int kBGather = 0;    // per-k gather from x with 4-byte copies and bounds tests
constexpr int kBPointwise = 1; // 1x1 / stride 1 / no pad: 16-byte copies straight from x
constexpr int kBUnfolded = 2;  // 16-byte copies from a column-unfolded copy of x (below)

// Unfolded B: a pre-pass writes, in float32,
//   xw[n][c][v][r][ow] = x[n][c][r - pad_top][ow*sw - pad_left + v*dw]  (0 outside x)
// for every kernel column v, padded input row r < hu and output column ow,
// and the weights transposed to wt[g][k][m] (m padded to mg4 with zeros).
// The B value of output (n, oh, ow) and term (c, u, v) is then
// xw[n][c][v][oh*sh + u*dh][ow]: a pixel part plus a term part, so four
// consecutive output columns of one row are 16 contiguous bytes (Wo a
// multiple of 4) and need no bounds test.
struct UnfPlan {
  int hu;              // padded input rows: (Ho-1)*sh + (kh-1)*dh + 1
  int mg4;             // output channels per group, rounded up to 4
  long long xw_elems;  // N * Cin * kw * hu * Wo
  long long wt_elems;  // groups * K * mg4
  size_t xw_off, wt_off;  // byte offsets of xw and wt in scratch (after any split planes)
  // The last, partly filled round of tiles split in k: tiles [tail_first,
  // tiles) run as tail_split ranges of tail_len terms each, writing raw float32
  // tiles to scratch at tail_off; a second kernel adds the ranges in order and
  // applies the epilogue.  tail_split = 0: no tail split.
  int tail_split, tail_len;
  long long tiles, tail_first;
  size_t tail_off;
};

// Depthwise (one input channel per group) halo-tiled direct kernel.
struct DwPlan {
  int th;        // output rows per work item
  int in_rows;   // input rows staged per work item
  int lm;        // left margin (columns before input column 0), 16-byte aligned
  int row;       // staged row length in elements (>= lm + needed columns)
  int vec;       // bytes per cp.async copy of input rows (16/8/4; 0: element copies)
  int sm;        // SMs of the device (blocks loop over the work items)
  int narrow;    // one warp per plane (stride 1, dilation 1, square 3/5/7, Wo <= 32)
  int cols4_r;   // narrow planes, four columns per lane: output rows per lane (2, 4, 7, 8), 0: not used
  int mma;       // 16-bit planes on the tensor cores (band-matrix mma.sync), one warp per plane
  int mma_pitch, mma_rows;  // its staged plane: row length (elements) and rows
};
size_t depthwise_smem_bytes(const DwPlan& d, int mg, int kh, int kw, int dtype);

// tcgen05 implicit GEMM: 128 pixels (of one image) x BN channels per tile.
constexpr int kModeCh8 = 0;   // k = (tap, channel), units of 8 channels
constexpr int kModeRow8 = 1;  // k = (channel, kernel row, 8 taps), 4-byte loads
constexpr int kModeNat = 2;   // k = (channel, tap), one value at a time
constexpr size_t kTcMaxSmem = 232448;  // 227 KB of dynamic shared memory per block
struct TcPlan {
  int bn;             // N tile (output channels), a multiple of 16
  int mode;           // k order (kMode*)
  int k_pad;          // k padded to a multiple of 64
  int stages;         // A-operand pipeline depth
  int co_tiles;       // output-channel tiles per group
  int tiles_per_img;  // 128-pixel tiles per image
  int pix_tiles;      // all pixel tiles (images x tiles per image)
  int ctas;           // persistent blocks
  size_t smem;        // dynamic shared memory bytes
};
bool tc_plan(const ConvArgs& a, int sm, TcPlan* t);

// tcgen05 implicit GEMM over shifted windows of a padded input band: 128
// positions of the padded plane x nt channels per tile.
struct WinPlan {
  int ph;          // phase split: 1 (stride 1) or 2 (stride 2 as 2x2 phases)
  int vh, vw;      // input rows and columns as read (a 1x1 layer's planes cut into rows of vw)
  int ho, wo;      // output rows and columns in the same view
  int khp, kwp;    // taps per axis after the phase split
  int hp, wp;      // padded positions per image: ho + (khp-1)*dh rows of wo + (kwp-1)*dw
  int c16;         // phase channels (cg * ph * ph) rounded up to 16
  int kblocks;     // k blocks of 8: khp * kwp * c16 / 8
  int hq;          // largest tap shift, in positions
  int nt;          // output channels per tile (MMA N): a multiple of 16, at most 256
  int co_tiles;    // channel tiles
  int ring;        // ring depth R in positions
  int mirror;      // slots written twice past the ring end (128, or 0 when no window straddles it)
  int lookahead;   // tiles the producers may run ahead of the MMAs (1 or 2)
  int band;        // padded rows per TMA band (one box: vw x ph*band rows x cg channels)
  int stages;      // bands in flight
  int band_bytes;  // bytes of one band
  int rt;          // padded rows per tile (128 / wp): a tile is rt whole rows of one image
  int tpi;         // tiles per image: ceil(ho / rt)
  int out_bytes;   // one output staging buffer: nt x rt x wo elements
  int ostages;     // output staging buffers (1 or 2)
  int tiles;       // tiles over all images
  int parts;       // position ranges (blocks per channel tile)
  int tq, tr;      // tiles per range: tq, and one more for the first tr ranges
  int ctas;        // blocks
  size_t smem;     // dynamic shared memory bytes
  size_t w_bytes;  // scratch: the repacked weights
};
bool tcw_plan(const ConvArgs& a, int sm, WinPlan* w);

// Grouped layers with few channels per group on CUDA cores (float32, stride
// 1, square 3x3 or 5x5 kernel, output rows a multiple of 4, Cout/groups a
// multiple of 8): per work item (image, group, kGdRows output rows) the
// group's input rows and weights are staged once and every k term (channel,
// tap) reads its B values from the staged rows at the tap's offset.
constexpr int kGdThreads = 128;
constexpr int kGdRows = 8;
struct GdPlan {
  int ok;           // the path applies
  int k;            // kernel size (3 or 5)
  int rows_in;      // staged input rows per item: kGdRows + (k - 1) * dh
  int pitch;        // floats per staged row (a multiple of 4)
  int cofs;         // staged column of input column 0 (a multiple of 4, >= the left pad)
  int row_tiles;    // ceil(Ho / kGdRows)
  long long items;  // n * groups * row_tiles
  size_t smem;      // two buffers of (input rows + weights)
};
bool gd_plan(const conv_problem* p, long long ho, long long wo, GdPlan* g);

// 16-bit 1x1 convolutions on the tensor cores (conv_pointwise.cu): one block
// per tile of BM = 16 * cfg output channels (cfg 1-4, eight warps across the
// pixels; cfg 5: 128 channels, 2 x 4 warps) x 128 pixels of one image, all of
// k in shared memory.
struct PwPlan {
  int ok;
  int cfg;
  int kp;  // Cin rounded up to 16
};
struct PwGeo {
  int kp, wpitch, xpitch;  // k rows staged; row lengths (elements) of the weight and pixel tiles
  int pblocks;             // 128-pixel blocks per image
  int vec_w, vec_x;        // 16-byte copies of weight rows / pixel rows
  int pair_io;             // two outputs (and residual values) per access
  int vec_r;               // the residual tile staged in shared memory by 16-byte copies
};
size_t pw_smem_bytes(const PwPlan& pp, bool residual_tile);  // shared memory of a block
cudaError_t launch_pointwise(const PwPlan& pp, const ConvArgs& a, int dtype, cudaStream_t s);

struct Plan {
  conv_plan_info info;
  GdPlan gd;
  int ffma_cfg;
  int ffma_vec;     // pointwise fp32 with whole 16-byte pixel groups: vector B loads
  int ffma_unf;     // the unfolded-B pre-pass and 16-byte copies (UnfPlan)
  UnfPlan unf;
  int k_per_split;  // terms per k range of the split variant
  int cluster_k;    // split k reduced within a cluster of the k ranges' blocks (else planes + split_reduce)
  DwPlan dw;
  TcPlan tc;
  WinPlan tcw;
  int tcw_ok;       // tcw holds a plan (the variant may still fall back to tc at launch)
  PwPlan pw;
};

// Opt `func` in to `bytes` of dynamic shared memory on the current device.
// The opted-in size only grows and is remembered per (kernel, device); the
// check and the update hold one lock, so concurrent host threads never lower
// it under another thread's launch.
cudaError_t opt_in_smem(const void* func, size_t bytes);

// Whether `func` can run as clusters of `cluster` blocks (cluster dims 1 x 1 x
// cluster) of `threads` threads and `smem` bytes of dynamic shared memory on
// the current device: at least one such cluster fits.  Clusters of more than 8
// blocks are allowed for `func` first.  The answer is remembered per (kernel,
// device, cluster, threads, smem).
bool cluster_fits(const void* func, int cluster, int threads, size_t smem);

// ConvInteger (conv_integer.cu): the unfolded byte matrix cols[g][q][p]
// (k words of 4 terms x pixels), per-pixel byte sums sx[g][p], the weight
// words wq[g][q][m] and per-channel byte sums sw[co], all in scratch.
struct CiPlan {
  int kq;            // k words: ceil(K / 4)
  long long p4;      // pixels (N*Ho*Wo) rounded up to 4
  int mg4;           // channels per group rounded up to 4
  size_t cols_off, sx_off, wq_off, sw_off, scratch_bytes;
};
struct CiArgs {
  int x_signed, w_signed;      // int8 (1) or uint8 (0)
  const uint8_t* x_zero;       // one element of x's type (device)
  const uint8_t* w_zero;       // one, or c_out, elements of w's type (device)
  int wz_per_channel;
  int kq;
  long long p4;
  int mg4;
  uint32_t* cols;
  int32_t* sx;
  uint32_t* wq;
  int32_t* sw;
};
CiPlan ci_plan(const ConvArgs& a);
cudaError_t launch_conv_integer(const ConvArgs& a, const CiPlan& plan, const CiArgs& c, cudaStream_t s);

cudaError_t launch_ffma(const Plan& plan, const ConvArgs& a, int dtype, cudaStream_t s);

// The transposed convolution (conv_transpose.cu): the Gemm as a planned 1x1
// convolution (raw float32 sums into scratch) and the gathering col2im.
struct TransposeGeo {
  int ho, wo;        // output size
};
struct TransposePlan {
  int dtype;
  Plan gemm_plan;        // the CUDA-core plan of the 1x1 Gemm
  ConvArgs gemm_args;    // its geometry (addresses filled at launch)
  size_t wt_off;          // transposed weights: float32, or 16-bit for the tensor-core Gemm
  size_t xf_off;          // 16-bit types on the CUDA-core Gemm: x widened to float32
  size_t cols_off, scratch_bytes;
  int mma;                // 16-bit, one group: the Gemm on the pointwise tensor-core kernel
  PwPlan pw;
};
cudaError_t launch_conv_transpose(const TransposePlan& tp, const ConvArgs& a, const TransposeGeo& t,
                                  const void* w, void* scratch, cudaStream_t s);

// Winograd F(2x2, 3x3) (conv_winograd.cu): transformed weights U[16][K][C],
// transformed input tiles V[16][C][p4], the sixteen products M[16][K][p4]
// (a 16-group 1x1 convolution on the CUDA-core kernel), all in scratch.
struct WinoGeo {
  int th, tw;          // tiles per image: ceil(Ho/2) x ceil(Wo/2)
  long long tiles;     // over all images
  long long p4;        // tiles rounded up to 4 (the product's pixel rows)
};
struct WinoPlan {
  WinoGeo geo;
  Plan gemm_plan;      // the CUDA-core plan of the 16-group 1x1 product
  ConvArgs gemm_args;
  size_t u_off, v_off, m_off, scratch_bytes;
};
cudaError_t launch_winograd(const WinoPlan& wp, const ConvArgs& a, void* scratch, cudaStream_t s);
// Kernels one conv_forward of the CUDA-core variant launches for `plan`.
int ffma_launch_count(const Plan& plan);
// Whether the unfolded-B layout applies to the shape (element type aside),
// and its sizes; false when a size is past the kernel's 32-bit offsets.
bool unf_plan(const conv_problem* p, long long ho, long long wo, UnfPlan* u);
cudaError_t launch_split_reduce(const ConvArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_depthwise(const Plan& plan, const ConvArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_tc(const Plan& plan, const ConvArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_tcw(const Plan& plan, const ConvArgs& a, int dtype, void* scratch, cudaStream_t s);
cudaError_t tc_error_word(uint32_t* word, int reset);
cudaError_t tcw_error_word(uint32_t* word, int reset);
cudaError_t tcw_wait_selftest_run(unsigned long long limit_ns, uint32_t* report_host);

}  // namespace conv
