// conv_integer.cu -- ConvInteger (ONNX): uint8 / int8 operands in any mix,
// zero points, exact int32 sums with wrap-around.
//
// "Convolution, pooling and resize", ConvInteger: y = sum (x - xZero) *
// (w - wZero[m]) in int32 with wrap-around; a padded tap is the quantized
// value xZero and adds nothing; lowered as the float convolution is -- one
// pass unfolds the windows of each image and group into a byte matrix (rows
// of k padded to whole 4-byte words), then the weights multiply it.
//
// Here the byte matrix is laid out k-word-major, cols[g][q][p] (the 4 bytes
// of terms 4q .. 4q+3 of output pixel p, padded pixels hold xZero, padded
// terms 0), and the product runs on CUDA cores with dp4a: 4 byte products
// added into an int32 per instruction, 8 x 8 outputs per thread.  dp4a
// multiplies the raw bytes, so the zero points enter through the exact
// expansion
//   sum (x - xz)(w - wz) = sum x w - wz * sum x - xz * sum w + K * xz * wz,
// whose terms the unfold pass (sum x per pixel) and the weight pass (sum w
// per channel) provide; all of it in 32-bit arithmetic modulo 2^32, which is
// the wrap-around the operator defines (the sum modulo 2^32 does not depend
// on the order).  Sums are exact integers: every order gives the same bits.
#include <string.h>

#include <algorithm>

#include "conv_internal.h"

namespace conv {
namespace {

constexpr int kCiBM = 128, kCiBN = 128, kCiTM = 8, kCiTN = 8;
constexpr int kCiThreads = (kCiBM / kCiTM) * (kCiBN / kCiTN);  // 256
constexpr int kCiBQ = 8;      // k words (32 terms) per stage
constexpr int kCiStages = 4;

__device__ __forceinline__ int32_t load_byte(const uint8_t* p, long long i, bool is_signed) {
  const uint8_t b = p[i];
  return is_signed ? static_cast<int32_t>(static_cast<int8_t>(b)) : static_cast<int32_t>(b);
}

template <bool XS, bool WS>
__device__ __forceinline__ int32_t dp4a_t(uint32_t xw, uint32_t ww, int32_t c) {
  int32_t d;
  if constexpr (XS && WS) asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(xw), "r"(ww), "r"(c));
  else if constexpr (XS && !WS) asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(xw), "r"(ww), "r"(c));
  else if constexpr (!XS && WS) asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(xw), "r"(ww), "r"(c));
  else asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(xw), "r"(ww), "r"(c));
  return d;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Unfold: block (32 pixels, group); thread (pixel lane, row ty of 8): the
// words q in [ty*qc, (ty+1)*qc) of its pixel into cols[g][q][p] (a warp
// writes 32 consecutive words per q), the terms' (channel, tap) walked
// without divisions, and the pixel's byte sum reduced over the 8 rows into
// sx[g][p].
__global__ void __launch_bounds__(256) ci_unfold(const ConvArgs a, const CiArgs c) {
  __shared__ int32_t part[8][32];
  const int lane = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const long long p = static_cast<long long>(blockIdx.x) * 32 + lane;
  const int g = blockIdx.y;
  const uint8_t* __restrict__ x = static_cast<const uint8_t*>(a.x);
  const int32_t xz = load_byte(c.x_zero, 0, c.x_signed);
  int32_t sum = 0;
  const int qc = (c.kq + 7) / 8;
  const int q0 = ty * qc, q1 = min(c.kq, q0 + qc);
  if (p < a.npix && q0 < q1) {
    const long long n = p / a.howo;
    const int rem = static_cast<int>(p - n * a.howo);
    const int oh = rem / a.wo, ow = rem - (rem / a.wo) * a.wo;
    const int ih0 = oh * a.sh - a.pt, iw0 = ow * a.sw - a.pl;
    const uint8_t* xg = x + (n * a.c_in + static_cast<long long>(g) * a.cg) * a.hw;
    // term k = 4*q0 as (channel, kernel row, kernel column)
    const int khw = a.kh * a.kw;
    int k = 4 * q0;
    int ch = k / khw;
    int u = (k - ch * khw) / a.kw;
    int v = k - ch * khw - u * a.kw;
    for (int q = q0; q < q1; ++q) {
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        int32_t val = 0;  // terms past K: 0 (their weight bytes are 0 too)
        if (k < a.K) {
          const int ih = ih0 + u * a.dh, iw = iw0 + v * a.dw;
          const bool in = static_cast<unsigned>(ih) < static_cast<unsigned>(a.h) &&
                          static_cast<unsigned>(iw) < static_cast<unsigned>(a.w);
          val = in ? load_byte(xg, static_cast<long long>(ch) * a.hw + static_cast<long long>(ih) * a.w + iw,
                               c.x_signed)
                   : xz;
          sum += val;
        }
        word |= (static_cast<uint32_t>(val) & 0xffu) << (8 * b);
        ++k;  // the next term: kernel column, then row, then channel
        if (++v == a.kw) {
          v = 0;
          if (++u == a.kh) { u = 0; ++ch; }
        }
      }
      c.cols[(static_cast<long long>(g) * c.kq + q) * c.p4 + p] = word;
    }
  }
  part[ty][lane] = sum;
  __syncthreads();
  if (ty == 0 && p < a.npix) {
    int32_t s = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) s += part[r][lane];
    c.sx[static_cast<long long>(g) * c.p4 + p] = s;
  }
}

// Weights.  Blocks [0, word_blocks): one thread per word wq[g][q][m]
// (channels padded to mg4 with zero words; a warp writes 32 consecutive
// channels).  The blocks after them: one warp per output channel, the
// channel's K bytes read by consecutive lanes and summed into sw[co].
__global__ void __launch_bounds__(256) ci_weights(const ConvArgs a, const CiArgs c, long long word_blocks) {
  const uint8_t* __restrict__ w = static_cast<const uint8_t*>(a.wt);
  if (blockIdx.x < word_blocks) {
    const long long t = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
    const long long words = static_cast<long long>(a.groups) * c.kq * c.mg4;
    if (t >= words) return;
    const int m = static_cast<int>(t % c.mg4);
    const long long gq = t / c.mg4;
    const int q = static_cast<int>(gq % c.kq), g = static_cast<int>(gq / c.kq);
    uint32_t word = 0;
    if (m < a.mg) {
      const long long row = (static_cast<long long>(g) * a.mg + m) * a.K;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int k = 4 * q + b;
        const int32_t v = k < a.K ? load_byte(w, row + k, c.w_signed) : 0;
        word |= (static_cast<uint32_t>(v) & 0xffu) << (8 * b);
      }
    }
    c.wq[t] = word;
    return;
  }
  const long long co = (static_cast<long long>(blockIdx.x) - word_blocks) * 8 + (threadIdx.x >> 5);
  if (co >= a.c_out) return;
  const int lane = threadIdx.x & 31;
  int32_t s = 0;
  for (int k = lane; k < a.K; k += 32) s += load_byte(w, co * a.K + k, c.w_signed);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) c.sw[co] = s;
}

// The product: block = 128 channels x 128 pixels of one group, k in stages of
// 8 words by 16-byte cp.async, 8 x 8 int32 accumulators per thread; then
// y = acc - wz*sx - xz*sw + K*xz*wz (modulo 2^32).
template <bool XS, bool WS>
__global__ void __launch_bounds__(kCiThreads, 2) ci_gemm(const ConvArgs a, const CiArgs c) {
  __shared__ __align__(16) uint32_t As[kCiStages][kCiBQ][kCiBM];
  __shared__ __align__(16) uint32_t Bs[kCiStages][kCiBQ][kCiBN];
  const int tid = threadIdx.x;
  const long long p0 = static_cast<long long>(blockIdx.x) * kCiBN;
  const int co_tiles = (a.mg + kCiBM - 1) / kCiBM;
  const int g = blockIdx.y / co_tiles;
  const int m0 = (blockIdx.y % co_tiles) * kCiBM;
  const uint32_t* __restrict__ wq = c.wq + static_cast<long long>(g) * c.kq * c.mg4;
  const uint32_t* __restrict__ cols = c.cols + static_cast<long long>(g) * c.kq * c.p4;
  // copies of a stage: 8 words x 128 = 256 16-byte units each for A and B, one per thread
  const int cq = tid / (kCiBN / 4), c4 = tid % (kCiBN / 4);
  const bool a_ok = m0 + 4 * c4 < c.mg4;
  const bool b_ok = p0 + 4 * c4 < c.p4;
  auto load = [&](int st, int q0) {
    const int q = q0 + cq;
    const bool qa = q < c.kq;
    cp_async16(&As[st][cq][4 * c4], qa && a_ok ? wq + static_cast<long long>(q) * c.mg4 + m0 + 4 * c4 : wq,
               qa && a_ok);
    cp_async16(&Bs[st][cq][4 * c4], qa && b_ok ? cols + static_cast<long long>(q) * c.p4 + p0 + 4 * c4 : cols,
               qa && b_ok);
  };
  int32_t acc[kCiTM][kCiTN];
#pragma unroll
  for (int i = 0; i < kCiTM; ++i)
#pragma unroll
    for (int j = 0; j < kCiTN; ++j) acc[i][j] = 0;
  const int tx = tid % (kCiBN / kCiTN), ty = tid / (kCiBN / kCiTN);
  const int nst = (c.kq + kCiBQ - 1) / kCiBQ;
#pragma unroll
  for (int st = 0; st < kCiStages - 1; ++st) {
    if (st < nst) load(st, st * kCiBQ);
    cp_commit();
  }
  for (int s = 0; s < nst; ++s) {
    cp_wait<kCiStages - 2>();
    __syncthreads();
    const int nxt = s + kCiStages - 1;
    if (nxt < nst) load(nxt % kCiStages, nxt * kCiBQ);
    cp_commit();
    const int st = s % kCiStages;
#pragma unroll
    for (int kk = 0; kk < kCiBQ; ++kk) {
      uint32_t ra[kCiTM], rb[kCiTN];
      const uint4 a0 = *reinterpret_cast<const uint4*>(&As[st][kk][ty * 4]);
      const uint4 a1 = *reinterpret_cast<const uint4*>(&As[st][kk][kCiBM / 2 + ty * 4]);
      const uint4 b0 = *reinterpret_cast<const uint4*>(&Bs[st][kk][tx * 4]);
      const uint4 b1 = *reinterpret_cast<const uint4*>(&Bs[st][kk][kCiBN / 2 + tx * 4]);
      ra[0] = a0.x; ra[1] = a0.y; ra[2] = a0.z; ra[3] = a0.w;
      ra[4] = a1.x; ra[5] = a1.y; ra[6] = a1.z; ra[7] = a1.w;
      rb[0] = b0.x; rb[1] = b0.y; rb[2] = b0.z; rb[3] = b0.w;
      rb[4] = b1.x; rb[5] = b1.y; rb[6] = b1.z; rb[7] = b1.w;
#pragma unroll
      for (int i = 0; i < kCiTM; ++i)
#pragma unroll
        for (int j = 0; j < kCiTN; ++j) acc[i][j] = dp4a_t<XS, WS>(rb[j], ra[i], acc[i][j]);
    }
  }
  cp_wait<0>();
  // epilogue, modulo 2^32 (unsigned arithmetic wraps by definition)
  const uint32_t xz = static_cast<uint32_t>(load_byte(c.x_zero, 0, XS));
  int32_t* y = static_cast<int32_t*>(a.y);
#pragma unroll
  for (int i = 0; i < kCiTM; ++i) {
    const int m = m0 + (i < 4 ? ty * 4 + i : kCiBM / 2 + ty * 4 + (i - 4));
    if (m >= a.mg) continue;
    const int co = g * a.mg + m;
    const uint32_t wz = static_cast<uint32_t>(load_byte(c.w_zero, c.wz_per_channel ? co : 0, WS));
    const uint32_t base = static_cast<uint32_t>(a.K) * xz * wz - xz * static_cast<uint32_t>(c.sw[co]);
#pragma unroll
    for (int j = 0; j < kCiTN; ++j) {
      const long long p = p0 + (j < 4 ? tx * 4 + j : kCiBN / 2 + tx * 4 + (j - 4));
      if (p >= a.npix) continue;
      const uint32_t sx = static_cast<uint32_t>(c.sx[static_cast<long long>(g) * c.p4 + p]);
      const uint32_t v = static_cast<uint32_t>(acc[i][j]) - wz * sx + base;
      const long long n = p / a.howo;
      y[(n * a.c_out + co) * a.howo + (p - n * a.howo)] = static_cast<int32_t>(v);
    }
  }
}

}  // namespace

CiPlan ci_plan(const ConvArgs& a) {
  CiPlan pl;
  pl.kq = (a.K + 3) / 4;
  pl.p4 = (a.npix + 3) / 4 * 4;
  pl.mg4 = (a.mg + 3) / 4 * 4;
  auto align = [](size_t v) { return (v + 255) / 256 * 256; };
  size_t off = 0;
  pl.cols_off = off;
  off = align(off + static_cast<size_t>(a.groups) * pl.kq * pl.p4 * 4);
  pl.sx_off = off;
  off = align(off + static_cast<size_t>(a.groups) * pl.p4 * 4);
  pl.wq_off = off;
  off = align(off + static_cast<size_t>(a.groups) * pl.kq * pl.mg4 * 4);
  pl.sw_off = off;
  off += static_cast<size_t>(a.c_out) * 4;
  pl.scratch_bytes = off;
  return pl;
}

cudaError_t launch_conv_integer(const ConvArgs& a, const CiPlan& pl, const CiArgs& c, cudaStream_t s) {
  const dim3 ug(static_cast<unsigned>((a.npix + 31) / 32), static_cast<unsigned>(a.groups));
  ci_unfold<<<ug, 256, 0, s>>>(a, c);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long words = static_cast<long long>(a.groups) * pl.kq * pl.mg4;
  const long long word_blocks = (words + 255) / 256;
  const long long sum_blocks = (static_cast<long long>(a.c_out) + 7) / 8;
  if (word_blocks + sum_blocks > 2147483647LL) return cudaErrorInvalidConfiguration;
  ci_weights<<<static_cast<unsigned>(word_blocks + sum_blocks), 256, 0, s>>>(a, c, word_blocks);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int co_tiles = (a.mg + kCiBM - 1) / kCiBM;
  const dim3 gg(static_cast<unsigned>((a.npix + kCiBN - 1) / kCiBN), static_cast<unsigned>(co_tiles * a.groups));
  if (c.x_signed && c.w_signed) ci_gemm<true, true><<<gg, kCiThreads, 0, s>>>(a, c);
  else if (c.x_signed) ci_gemm<true, false><<<gg, kCiThreads, 0, s>>>(a, c);
  else if (c.w_signed) ci_gemm<false, true><<<gg, kCiThreads, 0, s>>>(a, c);
  else ci_gemm<false, false><<<gg, kCiThreads, 0, s>>>(a, c);
  return cudaGetLastError();
}

}  // namespace conv
