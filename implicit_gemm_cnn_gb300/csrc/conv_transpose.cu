// conv_transpose.cu -- the transposed convolution (ONNX ConvTranspose).
//
// "Convolution, pooling and resize", Variants: a transposed convolution is a
// Gemm of the transposed weights with the input, then a gathering col2im --
// one thread per output element, no atomics -- with the same epilogue.
//
// The Gemm: for every image and group, cols[(co, u, v)][ih*W + iw] =
// sum_c w[c][co][u][v] * x[c][ih][iw] -- a 1x1 convolution of x whose
// weights are w transposed to [group][(co, u, v)][c], with its raw float32
// sums written to scratch (no epilogue).  16-bit layers with one group run it
// on the tensor cores (the pointwise tile kernel: products exact, float32
// accumulation); the others in float32 on the CUDA-core implicit-GEMM kernel
// (a 16-bit x and w widened first, exactly).  The col2im:
// output (n, co, oh, ow) gathers the taps (u, v)
// whose input position (oh + pt - u*dh)/sh, (ow + pl - v*dw)/sw is exact and
// inside the input, adds them in (u, v) order in float32, then bias,
// residual and activation, rounded once.  Every sum has a fixed order.
#include <algorithm>
#include <type_traits>

#include "conv_internal.h"

namespace conv {
namespace {

// w [Cin][Cout/G][kh][kw] -> wt [G][(co_l, u, v)][c_l] (float32, or the
// element type for the tensor-core Gemm), the 1x1 weights of the Gemm.  Block row r of the grid is one row (g, co_l, tap) of
// wt; its threads cover the c_l of that row.
template <typename T, typename U>
__global__ void __launch_bounds__(256) transpose_weights(const T* __restrict__ w, U* __restrict__ wt, int cg,
                                                         int mg, int khw, long long rows) {
  const int c = blockIdx.x * 256 + threadIdx.x;
  for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
    const int tap = static_cast<int>(r % khw);
    const long long gc = r / khw;
    const int col = static_cast<int>(gc % mg);
    const long long g = gc / mg;
    if (c < cg) {
      const T v = w[((g * cg + c) * mg + col) * khw + tap];
      if constexpr (std::is_same<T, U>::value) wt[r * cg + c] = v;
      else wt[r * cg + c] = to_f32(v);
    }
  }
}

// A 16-bit x widened to float32 (exact); four elements per thread step when
// x is 8-byte aligned and the count a multiple of 4.
template <typename T>
__global__ void __launch_bounds__(256) widen_x(const T* __restrict__ x, float* __restrict__ xf, long long count,
                                               int vec4) {
  const long long stride = static_cast<long long>(gridDim.x) * 256;
  if (vec4) {
    for (long long q = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; q < count / 4; q += stride) {
      const uint2 t = reinterpret_cast<const uint2*>(x)[q];
      const T* h = reinterpret_cast<const T*>(&t);
      reinterpret_cast<float4*>(xf)[q] = make_float4(to_f32(h[0]), to_f32(h[1]), to_f32(h[2]), to_f32(h[3]));
    }
  } else {
    for (long long e = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; e < count; e += stride)
      xf[e] = to_f32(x[e]);
  }
}

// The col2im: one warp per output row (n, co, oh), lanes over ow.  The taps
// whose input position is exact are found without a division per tap: with
// th = oh + pt - u*dh written as qh*sh + rh (0 <= rh < sh), stepping u to u+1
// subtracts dh = dhq*sh + dhr from it (one borrow at most), and the same for
// the columns; tap u is used when rh == 0 and 0 <= qh < H (input row qh).
// The taps are added in (u, v) order in float32, then bias, residual and
// activation, one rounding.
template <typename T, int ACT>
__global__ void __launch_bounds__(256) col2im_rows(const ConvArgs a, const TransposeGeo t,
                                                   const float* __restrict__ cols) {
  const T* __restrict__ bp = static_cast<const T*>(a.bias);
  const T* __restrict__ rp = static_cast<const T*>(a.residual);
  T* __restrict__ y = static_cast<T*>(a.y);
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(a.n) * a.c_out * t.ho;
  const int khw = a.kh * a.kw;
  const int dhq = a.dh / a.sh, dhr = a.dh - (a.dh / a.sh) * a.sh;
  const int dwq = a.dw / a.sw, dwr = a.dw - (a.dw / a.sw) * a.sw;
  for (long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5); r < rows;
       r += static_cast<long long>(gridDim.x) * 8) {
    const long long nc = r / t.ho;  // n * Cout + co
    const int oh = static_cast<int>(r - nc * t.ho);
    const int co = static_cast<int>(nc % a.c_out);
    // the Gemm's output channel (g, co_l, u, v) of image n is co * khw + u * kw + v
    const float* base = cols + nc * khw * a.hw;
    const float bv = bp ? to_f32(bp[co]) : 0.0f;
    const long long yrow = r * t.wo;
    const int th0 = oh + a.pt;
    const int qh0 = th0 / a.sh, rh0 = th0 - (th0 / a.sh) * a.sh;
    for (int ow = lane; ow < t.wo; ow += 32) {
      const int tw0 = ow + a.pl;
      const int qw0 = tw0 / a.sw, rw0 = tw0 - (tw0 / a.sw) * a.sw;
      float acc = 0.0f;
      if (a.dh == 1 && a.dw == 1) {
        // dilation 1: the taps used are u = rh0, rh0 + sh, ... (input rows qh0,
        // qh0 - 1, ...) and v = rw0, rw0 + sw, ... -- visited directly, in (u, v) order
        for (int u = rh0, ih = qh0; u < a.kh; u += a.sh, --ih) {
          if (ih < 0) break;
          if (ih >= a.h) continue;
          const float* brow = base + static_cast<long long>(u) * a.kw * a.hw + static_cast<long long>(ih) * a.w;
          for (int v = rw0, iw = qw0; v < a.kw; v += a.sw, --iw) {
            if (iw < 0) break;
            if (iw < a.w) acc = __fadd_rn(acc, brow[static_cast<long long>(v) * a.hw + iw]);
          }
        }
      } else {
        int qh = qh0, rh = rh0;
        for (int u = 0; u < a.kh; ++u) {
          if (rh == 0 && qh >= 0 && qh < a.h) {
            const float* brow = base + static_cast<long long>(u) * a.kw * a.hw + static_cast<long long>(qh) * a.w;
            int qw = qw0, rw = rw0;
            for (int v = 0; v < a.kw; ++v) {
              if (rw == 0 && qw >= 0 && qw < a.w) acc = __fadd_rn(acc, brow[static_cast<long long>(v) * a.hw + qw]);
              rw -= dwr;
              qw -= dwq;
              if (rw < 0) { rw += a.sw; qw -= 1; }
            }
          }
          rh -= dhr;
          qh -= dhq;
          if (rh < 0) { rh += a.sh; qh -= 1; }
        }
      }
      float v = acc;
      if (bp) v = __fadd_rn(v, bv);
      if (rp) v = __fadd_rn(v, to_f32(rp[yrow + ow]));
      y[yrow + ow] = from_f32<T>(act_fn<ACT>(v, a.alpha, a.beta));
    }
  }
}

template <typename T>
cudaError_t launch_col2im(const ConvArgs& a, const TransposeGeo& t, const float* cols, cudaStream_t s);

template <typename T>
cudaError_t launch_typed(const TransposePlan& tp, const ConvArgs& a, const TransposeGeo& t, const void* w,
                         void* scratch, cudaStream_t s) {
  char* sc = static_cast<char*>(scratch);
  float* cols = reinterpret_cast<float*>(sc + tp.cols_off);
  const int khw = a.kh * a.kw;
  const long long wrows = static_cast<long long>(a.groups) * a.mg * khw;
  const dim3 wgrid(static_cast<unsigned>((a.cg + 255) / 256), static_cast<unsigned>(std::min<long long>(wrows, 65535)));
  cudaError_t err = cudaSuccess;
  if constexpr (!std::is_same<T, float>::value) {
    if (tp.mma) {  // the Gemm on the tensor cores: weights in the element type, raw float32 sums
      T* wt16 = reinterpret_cast<T*>(sc + tp.wt_off);
      transpose_weights<T, T><<<wgrid, 256, 0, s>>>(static_cast<const T*>(w), wt16, a.cg, a.mg, khw, wrows);
      err = cudaGetLastError();
      if (err != cudaSuccess) return err;
      ConvArgs g = tp.gemm_args;
      g.x = a.x;
      g.wt = wt16;
      g.y = cols;
      g.bias = nullptr;
      g.residual = nullptr;
      g.raw_out = 1;
      g.act = ACT_IDENTITY;
      err = launch_pointwise(tp.pw, g, tp.dtype, s);
      if (err != cudaSuccess) return err;
      return launch_col2im<T>(a, t, cols, s);
    }
  }
  float* wt = reinterpret_cast<float*>(sc + tp.wt_off);
  transpose_weights<T, float><<<wgrid, 256, 0, s>>>(static_cast<const T*>(w), wt, a.cg, a.mg, khw, wrows);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // the Gemm: a 1x1 convolution of x (widened to float32 for 16-bit types)
  // with wt, raw float32 sums into cols
  ConvArgs g = tp.gemm_args;
  g.x = a.x;
  if constexpr (!std::is_same<T, float>::value) {
    float* xf = reinterpret_cast<float*>(sc + tp.xf_off);
    const long long count = static_cast<long long>(a.n) * a.c_in * a.hw;
    const int vec4 = reinterpret_cast<uintptr_t>(a.x) % 8 == 0 && count % 4 == 0;
    const long long work = vec4 ? count / 4 : count;
    widen_x<T><<<static_cast<unsigned>(std::max<long long>(1, std::min<long long>((work + 255) / 256, 152LL * 16))),
                 256, 0, s>>>(static_cast<const T*>(a.x), xf, count, vec4);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    g.x = xf;
  }
  g.wt = wt;
  g.y = cols;
  g.partial = cols;
  g.raw_out = 1;
  g.split = 1;
  g.k_per_split = g.K;
  err = launch_ffma(tp.gemm_plan, g, CONV_F32, s);
  if (err != cudaSuccess) return err;
  return launch_col2im<T>(a, t, cols, s);
}

template <typename T>
cudaError_t launch_col2im(const ConvArgs& a, const TransposeGeo& t, const float* cols, cudaStream_t s) {
  const long long rows = static_cast<long long>(a.n) * a.c_out * t.ho;
  const unsigned blocks = static_cast<unsigned>(std::max<long long>(1, std::min<long long>((rows + 7) / 8, 152LL * 16)));
  switch (a.act) {
#define CONV_T_CASE(A) \
  case A: col2im_rows<T, A><<<blocks, 256, 0, s>>>(a, t, cols); break;
    CONV_T_CASE(ACT_RELU)
    CONV_T_CASE(ACT_SILU)
    CONV_T_CASE(ACT_SIGMOID)
    CONV_T_CASE(ACT_TANH)
    CONV_T_CASE(ACT_HARD_SWISH)
    CONV_T_CASE(ACT_HARD_SIGMOID)
    CONV_T_CASE(ACT_CLIP)
    CONV_T_CASE(ACT_LEAKY_RELU)
#undef CONV_T_CASE
    default: col2im_rows<T, ACT_IDENTITY><<<blocks, 256, 0, s>>>(a, t, cols); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_transpose(const TransposePlan& tp, const ConvArgs& a, const TransposeGeo& t,
                                  const void* w, void* scratch, cudaStream_t s) {
  switch (tp.dtype) {
    case CONV_F32: return launch_typed<float>(tp, a, t, w, scratch, s);
    case CONV_F16: return launch_typed<__half>(tp, a, t, w, scratch, s);
    case CONV_BF16: return launch_typed<__nv_bfloat16>(tp, a, t, w, scratch, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace conv
