// conv_common.cuh -- types and device helpers shared by the convolution kernels.
//
// The fused epilogue follows "Convolution, pooling and resize", Layout and
// operands: sum, bias, residual addition, activation, in that order, each step
// rounded to float32.  The adds and multiplies below use the _rn intrinsics so
// that the compiler cannot contract them into fused multiply-adds: every step
// is rounded as written.  The activations are the ONNX operator definitions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace conv {

// Everything a kernel needs to know about one launch.  Per-image sizes are
// validated on the host to fit int32; batch-level offsets use int64.
struct ConvArgs {
  int n, c_in, h, w, c_out, kh, kw;
  int pt, pl, sh, sw, dh, dw;
  int groups, cg, mg;      // input / output channels per group
  int ho, wo;
  int K;                   // terms per output: cg * kh * kw
  long long hw, howo;      // h*w, ho*wo
  long long npix;          // n * ho * wo (GEMM columns across the batch)
  int act;
  float alpha, beta;
  const void* x;
  const void* wt;
  const void* bias;        // nullptr when absent
  const void* residual;    // nullptr when absent
  void* y;
  float* partial;          // split k: [split][n][c_out][ho][wo] float32 planes
  int split;               // ranges of k (1 = whole)
  int k_per_split;         // terms per range (a multiple of the k chunk)
  int vec_out;             // y (and scratch) 16-byte aligned: vector stores allowed
  float* xw;               // unfolded B: the column-unfolded x (float32), or nullptr
  float* wtt;              // unfolded B: the transposed weights [g][k][mg4]
  int hu, mg4;             // unfolded B: padded input rows, channels per group rounded to 4
  // tail split (unfolded B): 1-D grid of tail_first whole tiles, then
  // tail_tiles x tail_split k ranges of tail_len terms into tailbuf
  int tail_split, tail_len, tiles_gy;
  long long tail_first, tail_tiles;
  float* tailbuf;
  // CUDA-core kernel, a chunk of whole images: only output pixels in
  // [pix_lo, pix_hi) are loaded (unfolded B) and stored; the unfolded copy and
  // the split planes hold the chunk's images only, from image img0 on (planes
  // of part_total elements).  The launch keeps the whole problem's tiles.
  long long pix_lo, pix_hi, part_total;
  int img0;
  // grid offsets of a chunk: the first pixel tile (3-D grid) or, with a tail
  // split, the whole tiles [blk_whole_lo, + blk_whole_n) and the tail blocks
  // from blk_tail_lo on (1-D grid)
  long long px_tile0, blk_whole_lo, blk_whole_n, blk_tail_lo;
  int raw_out;             // CUDA-core kernel: write the raw float32 sums to `partial` (no epilogue)
  int cluster_k;           // split k: the k ranges of a tile are one thread-block cluster and are
                           // added through distributed shared memory (no planes, no second kernel)
};

enum Act {
  ACT_IDENTITY = 0, ACT_RELU = 1, ACT_SILU = 2, ACT_SIGMOID = 3, ACT_TANH = 4,
  ACT_HARD_SWISH = 5, ACT_HARD_SIGMOID = 6, ACT_CLIP = 7, ACT_LEAKY_RELU = 8
};

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float sigmoid_f32(float t) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-t)));
}

template <int ACT>
__device__ __forceinline__ float act_fn(float t, float alpha, float beta) {
  if constexpr (ACT == ACT_RELU) return t > 0.0f ? t : 0.0f;
  else if constexpr (ACT == ACT_SILU) return __fmul_rn(t, sigmoid_f32(t));
  else if constexpr (ACT == ACT_SIGMOID) return sigmoid_f32(t);
  else if constexpr (ACT == ACT_TANH) return tanhf(t);
  else if constexpr (ACT == ACT_HARD_SWISH) {
    const float s = __fadd_rn(__fmul_rn(t, 1.0f / 6.0f), 0.5f);
    return __fmul_rn(t, fmaxf(0.0f, fminf(1.0f, s)));
  } else if constexpr (ACT == ACT_HARD_SIGMOID) {
    const float s = __fadd_rn(__fmul_rn(alpha, t), beta);
    return fmaxf(0.0f, fminf(1.0f, s));
  } else if constexpr (ACT == ACT_CLIP) return fminf(fmaxf(t, alpha), beta);
  else if constexpr (ACT == ACT_LEAKY_RELU) return t >= 0.0f ? t : __fmul_rn(alpha, t);
  else return t;
}

// One activation, chosen at run time, applied to N register values: one
// branch per call, each case a straight-line loop (a switch inside a per-value
// loop would be if-converted into evaluating every activation for every value).
template <int N>
__device__ __forceinline__ void activate_n(float (&v)[N], int act, float alpha, float beta) {
#define CONV_ACT_CASE(A)                                                    \
  case A: {                                                                 \
    _Pragma("unroll") for (int i = 0; i < N; ++i) v[i] = act_fn<A>(v[i], alpha, beta); \
    break;                                                                  \
  }
  switch (act) {
    CONV_ACT_CASE(ACT_RELU)
    CONV_ACT_CASE(ACT_SILU)
    CONV_ACT_CASE(ACT_SIGMOID)
    CONV_ACT_CASE(ACT_TANH)
    CONV_ACT_CASE(ACT_HARD_SWISH)
    CONV_ACT_CASE(ACT_HARD_SIGMOID)
    CONV_ACT_CASE(ACT_CLIP)
    CONV_ACT_CASE(ACT_LEAKY_RELU)
    default: break;
  }
#undef CONV_ACT_CASE
}

__device__ __forceinline__ float activate(float t, int act, float alpha, float beta) {
  float v[1] = {t};
  activate_n<1>(v, act, alpha, beta);
  return v[0];
}

// Bias, residual, then the compiled-in activation ACT, for N values (each
// step rounded in float32).
template <int ACT, int N>
__device__ __forceinline__ void epilogue_t(float (&v)[N], const float (&bias)[N], const float (&res)[N],
                                           bool has_bias, bool has_res, float alpha, float beta) {
  if (has_bias) {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __fadd_rn(v[i], bias[i]);
  }
  if (has_res) {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __fadd_rn(v[i], res[i]);
  }
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = act_fn<ACT>(v[i], alpha, beta);
}

// Sum, bias, residual for N values of one output channel or of N channels
// (bias per value), then the activation: the float32 steps of the epilogue.
template <int N>
__device__ __forceinline__ void epilogue_n(float (&v)[N], const float (&bias)[N], const float (&res)[N],
                                           bool has_bias, bool has_res, int act, float alpha, float beta) {
  if (has_bias) {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __fadd_rn(v[i], bias[i]);
  }
  if (has_res) {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __fadd_rn(v[i], res[i]);
  }
  activate_n<N>(v, act, alpha, beta);
}

}  // namespace conv
