// conv_winograd.cu -- Winograd F(2x2, 3x3) for float32 3x3 stride-1 layers.
//
// "Convolutions", section 2.6: F(m, r) computes m outputs of an r-tap filter
// with m + r - 1 multiplies; F(2x2, 3x3) needs 16 instead of 36 (2.25x
// fewer), at the cost of transforming the input tiles and the weights
// ("Convolution, pooling and resize", Not built, with the numbers: sixteen
// batched products plus the transforms' passes).  With the minimal-filtering
// matrices of that construction,
//
//   B^T = [1 0 -1 0; 0 1 1 0; 0 -1 1 0; 0 1 0 -1]
//   G   = [1 0 0; 1/2 1/2 1/2; 1/2 -1/2 1/2; 0 0 1]
//   A^T = [1 1 1 0; 0 1 -1 -1]
//
// a 2x2 output tile is Y = A^T [ sum_c (G g_c G^T) .* (B^T d_c B) ] A for the
// 4x4 input tile d_c of each channel.  Here:
//   * wino_weights: U[xi][k][c] = (G g G^T)[xi] (16 values per (k, c));
//   * wino_input:   V[xi][c][p] = (B^T d B)[xi] for every tile p (tiles of
//     2x2 outputs over all images, their 4x4 inputs overlapping by 2; zeros
//     outside the image);
//   * the sixteen products M[xi] = U[xi] V[xi], summed over c, as one grouped
//     1x1 convolution (16 groups) on the CUDA-core kernel with its raw float32
//     sums kept (no epilogue);
//   * wino_output:  Y = A^T M A per (k, tile), then bias, residual,
//     activation, rounded once.
// Every sum has a fixed order; the transforms are additions and exact
// halvings, so the float32 result differs from the direct sum by a few
// roundings of the transformed terms.
#include <algorithm>

#include "conv_internal.h"

namespace conv {
namespace {

__global__ void __launch_bounds__(256) wino_weights(const float* __restrict__ w, float* __restrict__ u, int kout,
                                                    int cin) {
  const long long total = static_cast<long long>(kout) * cin;
  for (long long e = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * 256) {
    const float* g = w + e * 9;  // OIHW: (k, c) row of 3x3
    float gg[4][3];               // G g (4 x 3)
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const float g0 = g[j], g1 = g[3 + j], g2 = g[6 + j];
      gg[0][j] = g0;
      gg[1][j] = __fmul_rn(__fadd_rn(__fadd_rn(g0, g1), g2), 0.5f);
      gg[2][j] = __fmul_rn(__fadd_rn(__fsub_rn(g0, g1), g2), 0.5f);
      gg[3][j] = g2;
    }
    const long long plane = total;  // U[xi] holds kout x cin values
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // (G g) G^T
      const float a0 = gg[i][0], a1 = gg[i][1], a2 = gg[i][2];
      const float r[4] = {a0, __fmul_rn(__fadd_rn(__fadd_rn(a0, a1), a2), 0.5f),
                          __fmul_rn(__fadd_rn(__fsub_rn(a0, a1), a2), 0.5f), a2};
#pragma unroll
      for (int j = 0; j < 4; ++j) u[(i * 4 + j) * plane + e] = r[j];
    }
  }
}

// One thread per (channel, tile): V[xi][c][p] = (B^T d B)[xi].
__global__ void __launch_bounds__(256) wino_input(const ConvArgs a, const WinoGeo wg, float* __restrict__ v) {
  const float* __restrict__ x = static_cast<const float*>(a.x);
  const long long total = static_cast<long long>(a.c_in) * wg.p4;
  for (long long e = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * 256) {
    const long long p = e % wg.p4;
    const int c = static_cast<int>(e / wg.p4);
    float d[4][4];
    if (p < wg.tiles) {
      const long long tpi = static_cast<long long>(wg.th) * wg.tw;
      const long long n = p / tpi;
      const int t = static_cast<int>(p - n * tpi);
      const int ti = t / wg.tw, tj = t - (t / wg.tw) * wg.tw;
      const int r0 = 2 * ti - a.pt, c0 = 2 * tj - a.pl;
      const float* xp = x + (n * a.c_in + c) * a.hw;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = r0 + i, cc = c0 + j;
          d[i][j] = (static_cast<unsigned>(r) < static_cast<unsigned>(a.h) &&
                     static_cast<unsigned>(cc) < static_cast<unsigned>(a.w))
                        ? xp[static_cast<long long>(r) * a.w + cc]
                        : 0.0f;
        }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) d[i][j] = 0.0f;  // padding tiles of the last group of 4
    }
    float t[4][4];  // B^T d
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      t[0][j] = __fsub_rn(d[0][j], d[2][j]);
      t[1][j] = __fadd_rn(d[1][j], d[2][j]);
      t[2][j] = __fsub_rn(d[2][j], d[1][j]);
      t[3][j] = __fsub_rn(d[1][j], d[3][j]);
    }
    const long long plane = static_cast<long long>(a.c_in) * wg.p4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // (B^T d) B
      const float r[4] = {__fsub_rn(t[i][0], t[i][2]), __fadd_rn(t[i][1], t[i][2]), __fsub_rn(t[i][2], t[i][1]),
                          __fsub_rn(t[i][1], t[i][3])};
#pragma unroll
      for (int j = 0; j < 4; ++j) v[(i * 4 + j) * plane + e] = r[j];
    }
  }
}

// One thread per (output channel, tile): Y = A^T M A, then the epilogue.
template <int ACT>
__global__ void __launch_bounds__(256) wino_output(const ConvArgs a, const WinoGeo wg, const float* __restrict__ m) {
  const float* __restrict__ bp = static_cast<const float*>(a.bias);
  const float* __restrict__ rp = static_cast<const float*>(a.residual);
  float* __restrict__ y = static_cast<float*>(a.y);
  const long long total = static_cast<long long>(a.c_out) * wg.tiles;
  const long long plane = static_cast<long long>(a.c_out) * wg.p4;
  for (long long e = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * 256) {
    const long long p = e % wg.tiles;
    const int k = static_cast<int>(e / wg.tiles);
    const float* mk = m + static_cast<long long>(k) * wg.p4 + p;
    float mm[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) mm[i][j] = mk[(i * 4 + j) * plane];
    float s[2][4];  // A^T M
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s[0][j] = __fadd_rn(__fadd_rn(mm[0][j], mm[1][j]), mm[2][j]);
      s[1][j] = __fsub_rn(__fsub_rn(mm[1][j], mm[2][j]), mm[3][j]);
    }
    const long long tpi = static_cast<long long>(wg.th) * wg.tw;
    const long long n = p / tpi;
    const int t = static_cast<int>(p - n * tpi);
    const int ti = t / wg.tw, tj = t - (t / wg.tw) * wg.tw;
    const float bv = bp ? bp[k] : 0.0f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {  // (A^T M) A
      const float yv[2] = {__fadd_rn(__fadd_rn(s[i][0], s[i][1]), s[i][2]),
                           __fsub_rn(__fsub_rn(s[i][1], s[i][2]), s[i][3])};
      const int oh = 2 * ti + i;
      if (oh >= a.ho) continue;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int ow = 2 * tj + j;
        if (ow >= a.wo) continue;
        const long long o = ((n * a.c_out + k) * a.ho + oh) * a.wo + ow;
        float v = yv[j];
        if (bp) v = __fadd_rn(v, bv);
        if (rp) v = __fadd_rn(v, rp[o]);
        y[o] = act_fn<ACT>(v, a.alpha, a.beta);
      }
    }
  }
}

unsigned grid_for(long long work) {
  return static_cast<unsigned>(std::max<long long>(1, std::min<long long>((work + 255) / 256, 152LL * 32)));
}

}  // namespace

cudaError_t launch_winograd(const WinoPlan& wp, const ConvArgs& a, void* scratch, cudaStream_t s) {
  char* sc = static_cast<char*>(scratch);
  float* u = reinterpret_cast<float*>(sc + wp.u_off);
  float* v = reinterpret_cast<float*>(sc + wp.v_off);
  float* m = reinterpret_cast<float*>(sc + wp.m_off);
  wino_weights<<<grid_for(static_cast<long long>(a.c_out) * a.c_in), 256, 0, s>>>(static_cast<const float*>(a.wt),
                                                                                  u, a.c_out, a.c_in);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  wino_input<<<grid_for(static_cast<long long>(a.c_in) * wp.geo.p4), 256, 0, s>>>(a, wp.geo, v);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // the sixteen products: a 16-group 1x1 convolution of V (16*Cin channels
  // of p4 pixels) with U, raw float32 sums into M
  ConvArgs g = wp.gemm_args;
  g.x = v;
  g.wt = u;
  g.y = m;
  g.partial = m;
  g.raw_out = 1;
  g.split = 1;
  g.k_per_split = g.K;
  err = launch_ffma(wp.gemm_plan, g, CONV_F32, s);
  if (err != cudaSuccess) return err;
  const unsigned blocks = grid_for(static_cast<long long>(a.c_out) * wp.geo.tiles);
  switch (a.act) {
#define CONV_W_CASE(A) \
  case A: wino_output<A><<<blocks, 256, 0, s>>>(a, wp.geo, m); break;
    CONV_W_CASE(ACT_RELU)
    CONV_W_CASE(ACT_SILU)
    CONV_W_CASE(ACT_SIGMOID)
    CONV_W_CASE(ACT_TANH)
    CONV_W_CASE(ACT_HARD_SWISH)
    CONV_W_CASE(ACT_HARD_SIGMOID)
    CONV_W_CASE(ACT_CLIP)
    CONV_W_CASE(ACT_LEAKY_RELU)
#undef CONV_W_CASE
    default: wino_output<ACT_IDENTITY><<<blocks, 256, 0, s>>>(a, wp.geo, m); break;
  }
  return cudaGetLastError();
}

}  // namespace conv
