// conv_depthwise.cu -- direct depthwise convolution with halo tiles in shared
// memory (one input channel per group, any channel multiplier m = Cout/G).
//
// The method: "Convolution, pooling and resize", Variants (depthwise: a direct
// kernel with the window order fixed, each output summed in one chain of at
// most kernel-area terms) and "Convolutions en compute" (the halo tile: a T x T
// output tile needs its (T + 2R) x (T + 2R) input neighbourhood, loaded by the
// whole block with a strided loop, then a barrier, then each window sum reads
// shared memory).  Border taps read zeros -- ONNX Conv pads with zeros -- where
// that page clamps to the edge.
//
// A block stages TH output rows' worth of one input plane (the rows the
// windows reach, zero rows above / below the image, zero columns left /
// right), converted to float32, then computes the m output channels that read
// that plane.  Each thread computes QW adjacent outputs of a row and sums each
// one's window in (kernel row, kernel column) order in a single float32 chain;
// for stride-1, dilation-1 layers with a compiled kernel width the row
// segment is held in registers and reused across the QW outputs.  Bias,
// residual and activation are applied at the store.
#include "conv_internal.h"

namespace conv {
namespace {

constexpr int kDwThreads = 256;
constexpr int kDwQW = 4;

template <typename T, int KW>
__global__ void __launch_bounds__(kDwThreads) depthwise(const ConvArgs a, const DwPlan d, int row_tiles) {
  extern __shared__ __align__(16) float dsm[];
  const int m = a.mg;
  float* wsm = dsm;                              // [m][kh][kw]
  float* tile = dsm + ((m * a.kh * a.kw + 3) & ~3);  // [in_rows][row]
  const int tid = threadIdx.x;
  const long long plane = blockIdx.x / row_tiles;
  const int rt = static_cast<int>(blockIdx.x - plane * row_tiles);
  const int n = static_cast<int>(plane / a.groups);
  const int g = static_cast<int>(plane - static_cast<long long>(n) * a.groups);
  const int oh0 = rt * d.th;
  const int rows_out = min(d.th, a.ho - oh0);
  const int ih_start = oh0 * a.sh - a.pt;
  const T* __restrict__ x = static_cast<const T*>(a.x) + (static_cast<long long>(n) * a.c_in + g) * a.hw;
  const T* __restrict__ wt = static_cast<const T*>(a.wt);

  // weights of the m output channels of this group
  const int nw = m * a.kh * a.kw;
  for (int i = tid; i < nw; i += kDwThreads) wsm[i] = to_f32(wt[static_cast<long long>(g) * nw + i]);

  // stage the input rows [ih_start, ih_start + in_rows): zero outside the image
  const int total = d.in_rows * d.row;
  const int r_lo = max(0, ih_start), r_hi = min(a.h, ih_start + d.in_rows);
  if (d.vec) {
    // zero everything that is not image, then copy the image rows with vectors
    for (int i = tid; i < total; i += kDwThreads) {
      const int r = i / d.row, c = i - (i / d.row) * d.row;
      const int ih = ih_start + r, iw = c - d.lm;
      if (!(ih >= 0 && ih < a.h && iw >= 0 && iw < a.w)) tile[i] = 0.0f;
    }
    constexpr int VE = 16 / sizeof(T);
    const long long f0 = static_cast<long long>(r_lo) * a.w;
    const int count = (r_hi - r_lo) * a.w;
    const int nvec = count / VE;
    const uint4* src = reinterpret_cast<const uint4*>(x + f0);
    for (int i = tid; i < nvec; i += kDwThreads) {
      const uint4 v = src[i];
      const T* e = reinterpret_cast<const T*>(&v);
      const int f = i * VE;
      int r = f / a.w, c = f - (f / a.w) * a.w;
#pragma unroll
      for (int q = 0; q < VE; ++q) {
        tile[(r_lo - ih_start + r) * d.row + d.lm + c] = to_f32(e[q]);
        if (++c == a.w) { c = 0; ++r; }
      }
    }
    for (int f = nvec * VE + tid; f < count; f += kDwThreads) {
      const int r = f / a.w, c = f - (f / a.w) * a.w;
      tile[(r_lo - ih_start + r) * d.row + d.lm + c] = to_f32(x[f0 + f]);
    }
  } else {
    for (int i = tid; i < total; i += kDwThreads) {
      const int r = i / d.row, c = i - (i / d.row) * d.row;
      const int ih = ih_start + r, iw = c - d.lm;
      tile[i] = (ih >= 0 && ih < a.h && iw >= 0 && iw < a.w)
                    ? to_f32(x[static_cast<long long>(ih) * a.w + iw]) : 0.0f;
    }
  }
  __syncthreads();

  const int strips = (a.wo + kDwQW - 1) / kDwQW;
  const int items = rows_out * strips * m;
  T* y = static_cast<T*>(a.y);
  const bool fast = (KW != 0) && a.sw == 1 && a.dw == 1 && a.kw == KW;
  for (int it = tid; it < items; it += kDwThreads) {
    const int j = it / (rows_out * strips);
    const int rem = it - j * (rows_out * strips);
    const int ohl = rem / strips;
    const int ow0 = (rem - ohl * strips) * kDwQW;
    const float* wj = wsm + j * a.kh * a.kw;
    float acc[kDwQW];
#pragma unroll
    for (int q = 0; q < kDwQW; ++q) acc[q] = 0.0f;
    if (fast) {
      constexpr int KWc = KW > 0 ? KW : 1;
      for (int u = 0; u < a.kh; ++u) {
        const float* srow = tile + (ohl * a.sh + u * a.dh) * d.row + d.lm - a.pl + ow0;
        float seg[kDwQW + KWc - 1];
#pragma unroll
        for (int i = 0; i < kDwQW + KWc - 1; ++i) seg[i] = srow[i];
#pragma unroll
        for (int v = 0; v < KWc; ++v) {
          const float wv = wj[u * KWc + v];
#pragma unroll
          for (int q = 0; q < kDwQW; ++q) acc[q] = fmaf(seg[q + v], wv, acc[q]);
        }
      }
    } else {
      for (int u = 0; u < a.kh; ++u) {
        const float* srow = tile + (ohl * a.sh + u * a.dh) * d.row + d.lm - a.pl + ow0 * a.sw;
        for (int v = 0; v < a.kw; ++v) {
          const float wv = wj[u * a.kw + v];
#pragma unroll
          for (int q = 0; q < kDwQW; ++q) acc[q] = fmaf(srow[q * a.sw + v * a.dw], wv, acc[q]);
        }
      }
    }
    const int co = g * m + j;
    const int oh = oh0 + ohl;
    const long long out = ((static_cast<long long>(n) * a.c_out + co) * a.ho + oh) * a.wo + ow0;
#pragma unroll
    for (int q = 0; q < kDwQW; ++q)
      if (ow0 + q < a.wo) y[out + q] = epilogue<T>(acc[q], co, out + q, a);
  }
}

template <typename T, int KW>
cudaError_t launch_kw(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  const int row_tiles = (a.ho + d.th - 1) / d.th;
  const long long blocks = static_cast<long long>(a.n) * a.groups * row_tiles;
  const size_t smem = (static_cast<size_t>((a.mg * a.kh * a.kw + 3) & ~3) +
                       static_cast<size_t>(d.in_rows) * d.row) * sizeof(float);
  auto kern = depthwise<T, KW>;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  kern<<<static_cast<unsigned>(blocks), kDwThreads, smem, s>>>(a, d, row_tiles);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  if (a.sw == 1 && a.dw == 1) {
    if (a.kw == 3) return launch_kw<T, 3>(d, a, s);
    if (a.kw == 5) return launch_kw<T, 5>(d, a, s);
    if (a.kw == 7) return launch_kw<T, 7>(d, a, s);
  }
  return launch_kw<T, 0>(d, a, s);
}

}  // namespace

cudaError_t launch_depthwise(const Plan& plan, const ConvArgs& a, int dtype, cudaStream_t s) {
  switch (dtype) {
    case CONV_F32: return launch_typed<float>(plan.dw, a, s);
    case CONV_F16: return launch_typed<__half>(plan.dw, a, s);
    case CONV_BF16: return launch_typed<__nv_bfloat16>(plan.dw, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace conv
