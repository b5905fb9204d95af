// conv_transpose.cu -- the transposed convolution (ONNX ConvTranspose).
//
// "Convolution, pooling and resize", Variants: a transposed convolution is a
// Gemm of the transposed weights with the input, then a gathering col2im --
// one thread per output element, no atomics -- with the same epilogue.
//
// The Gemm: for every image and group, cols[(co, u, v)][ih*W + iw] =
// sum_c w[c][co][u][v] * x[c][ih][iw] -- a 1x1 convolution of x whose
// weights are w transposed to [group][(co, u, v)][c]; it runs on the
// CUDA-core implicit-GEMM kernel with its raw float32 sums written to scratch
// (no epilogue).  The col2im: output (n, co, oh, ow) gathers the taps (u, v)
// whose input position (oh + pt - u*dh)/sh, (ow + pl - v*dw)/sw is exact and
// inside the input, adds them in (u, v) order in float32, then bias,
// residual and activation, rounded once.  Every sum has a fixed order.
#include <algorithm>

#include "conv_internal.h"

namespace conv {
namespace {

// w [Cin][Cout/G][kh][kw] -> wt [G][(co_l, u, v)][c_l], the 1x1 weights of the Gemm.
template <typename T>
__global__ void __launch_bounds__(256) transpose_weights(const T* __restrict__ w, T* __restrict__ wt, int groups,
                                                         int cg, int mg, int khw) {
  const long long total = static_cast<long long>(groups) * mg * khw * cg;
  for (long long e = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * 256) {
    const int c = static_cast<int>(e % cg);
    const long long r = e / cg;  // (g, co_l, tap)
    const int tap = static_cast<int>(r % khw);
    const long long gc = r / khw;
    const int col = static_cast<int>(gc % mg), g = static_cast<int>(gc / mg);
    wt[e] = w[((static_cast<long long>(g) * cg + c) * mg + col) * khw + tap];
  }
}

template <typename T, int ACT>
__global__ void __launch_bounds__(256) col2im_gather(const ConvArgs a, const TransposeGeo t, const float* cols) {
  const long long total = static_cast<long long>(a.n) * a.c_out * t.ho * t.wo;
  const T* __restrict__ bp = static_cast<const T*>(a.bias);
  const T* __restrict__ rp = static_cast<const T*>(a.residual);
  T* __restrict__ y = static_cast<T*>(a.y);
  const int khw = a.kh * a.kw;
  for (long long o = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; o < total;
       o += static_cast<long long>(gridDim.x) * 256) {
    const int ow = static_cast<int>(o % t.wo);
    const long long r1 = o / t.wo;
    const int oh = static_cast<int>(r1 % t.ho);
    const long long r2 = r1 / t.ho;
    const int co = static_cast<int>(r2 % a.c_out);
    const long long n = r2 / a.c_out;
    // the Gemm's output channel (g, co_l, u, v) is co * khw + u * kw + v
    const float* base = cols + (n * a.c_out + co) * khw * a.hw;
    float acc = 0.0f;
    for (int u = 0; u < a.kh; ++u) {
      const int th = oh + a.pt - u * a.dh;
      if (th < 0 || th % a.sh) continue;
      const int ih = th / a.sh;
      if (ih >= a.h) continue;
      for (int v = 0; v < a.kw; ++v) {
        const int tw = ow + a.pl - v * a.dw;
        if (tw < 0 || tw % a.sw) continue;
        const int iw = tw / a.sw;
        if (iw >= a.w) continue;
        acc = __fadd_rn(acc, base[static_cast<long long>(u * a.kw + v) * a.hw + static_cast<long long>(ih) * a.w + iw]);
      }
    }
    float v1[1] = {acc}, b1[1] = {bp ? to_f32(bp[co]) : 0.0f}, r1v[1] = {rp ? to_f32(rp[o]) : 0.0f};
    if (bp) v1[0] = __fadd_rn(v1[0], b1[0]);
    if (rp) v1[0] = __fadd_rn(v1[0], r1v[0]);
    y[o] = from_f32<T>(act_fn<ACT>(v1[0], a.alpha, a.beta));
  }
}

template <typename T>
cudaError_t launch_typed(const TransposePlan& tp, const ConvArgs& a, const TransposeGeo& t, const void* w,
                         void* scratch, cudaStream_t s) {
  T* wt = reinterpret_cast<T*>(static_cast<char*>(scratch) + tp.wt_off);
  float* cols = reinterpret_cast<float*>(static_cast<char*>(scratch) + tp.cols_off);
  const int khw = a.kh * a.kw;
  const long long wel = static_cast<long long>(a.groups) * a.mg * khw * a.cg;
  transpose_weights<T><<<static_cast<unsigned>(std::min<long long>((wel + 255) / 256, 4096)), 256, 0, s>>>(
      static_cast<const T*>(w), wt, a.groups, a.cg, a.mg, khw);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // the Gemm: a 1x1 convolution of x with wt, raw float32 sums into cols
  ConvArgs g = tp.gemm_args;
  g.x = a.x;
  g.wt = wt;
  g.y = cols;
  g.partial = cols;
  g.raw_out = 1;
  g.split = 1;
  g.k_per_split = g.K;
  err = launch_ffma(tp.gemm_plan, g, tp.dtype, s);
  if (err != cudaSuccess) return err;
  const long long total = static_cast<long long>(a.n) * a.c_out * t.ho * t.wo;
  const unsigned blocks = static_cast<unsigned>(std::min<long long>((total + 255) / 256, 152LL * 16));
  switch (a.act) {
#define CONV_T_CASE(A) \
  case A: col2im_gather<T, A><<<blocks, 256, 0, s>>>(a, t, cols); break;
    CONV_T_CASE(ACT_RELU)
    CONV_T_CASE(ACT_SILU)
    CONV_T_CASE(ACT_SIGMOID)
    CONV_T_CASE(ACT_TANH)
    CONV_T_CASE(ACT_HARD_SWISH)
    CONV_T_CASE(ACT_HARD_SIGMOID)
    CONV_T_CASE(ACT_CLIP)
    CONV_T_CASE(ACT_LEAKY_RELU)
#undef CONV_T_CASE
    default: col2im_gather<T, ACT_IDENTITY><<<blocks, 256, 0, s>>>(a, t, cols); break;
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
