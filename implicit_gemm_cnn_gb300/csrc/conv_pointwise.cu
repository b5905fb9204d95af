// conv_pointwise.cu -- 16-bit 1x1 convolutions (stride 1, no padding,
// ungrouped) as tiled matrix products on the tensor cores.
//
// A 1x1 convolution is the GEMM of "Convolutions en compute" with no im2col
// at all: per image, Y[co][p] = sum_c W[co][c] X[c][p], where X is the image's
// NCHW planes read as a Cin x (H*W) matrix (pixels contiguous) and W the
// Cout x Cin weights.  A block computes one BM x 128 tile (BM = Cout rounded
// up to 16, at most 64, by 128 pixels of one image) over the whole of k
// (Cin <= 256): both operand tiles
// arrive in shared memory by 16-byte cp.async (rows padded by 16 bytes, so the
// fragment loads are conflict-free), then each warp runs mma.sync m16n8k16
// (float32 accumulation) over its sub-tile: A fragments by ldmatrix from the
// weight rows, B fragments by ldmatrix.trans from the pixel rows.  Products
// of 16-bit values are exact in float32; the sums run in the MMA's float32
// order.  The epilogue adds bias and residual, applies the activation in
// float32 and rounds once, two pixels per store; or (raw_out, the Gemm of a
// transposed convolution) writes the float32 sums as they are.
#include <algorithm>
#include <type_traits>

#include "conv_internal.h"

namespace conv {
namespace {

constexpr int kPwBN = 128;  // pixels per tile
constexpr int kPwThreads = 256;

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void pw_commit_wait_all() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
template <typename T>
__device__ __forceinline__ void pw_mma(float (&d)[4], const uint32_t (&aq)[4], uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same<T, __half>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(aq[0]), "r"(aq[1]), "r"(aq[2]), "r"(aq[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(aq[0]), "r"(aq[1]), "r"(aq[2]), "r"(aq[3]), "r"(b0), "r"(b1));
  }
}
template <typename T>
__device__ __forceinline__ uint32_t pw_pack(float lo, float hi) {
  const T l = from_f32<T>(lo), h = from_f32<T>(hi);
  return static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&l)) |
         (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&h)) << 16);
}

// TMW 16-row blocks per warp; WM x WN warps; BM = 16 * TMW * WM output
// channels, 128 pixels.
template <typename T, int TMW, int WM, int WN>
__global__ void __launch_bounds__(kPwThreads, 2) pointwise_mma(const ConvArgs a, const PwGeo g) {
  constexpr int BM = 16 * TMW * WM;
  constexpr int TNW = kPwBN / 8 / WN;  // 8-pixel blocks per warp (even)
  static_assert(WM * WN * 32 == kPwThreads && TNW % 2 == 0, "warp layout");
  extern __shared__ __align__(16) unsigned char psm[];
  T* ws = reinterpret_cast<T*>(psm);                                           // [BM][wpitch]
  T* xs = reinterpret_cast<T*>(psm + static_cast<size_t>(BM) * g.wpitch * sizeof(T));  // [kp][xpitch]
  T* rs = xs + static_cast<size_t>(g.kp) * g.xpitch;  // [BM][xpitch]: the residual tile (vec_r)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x / g.pblocks;
  const int p0 = (blockIdx.x - n * g.pblocks) * kPwBN;
  const int m0 = blockIdx.y * BM;
  const T* __restrict__ xg = static_cast<const T*>(a.x);
  const T* __restrict__ wg = static_cast<const T*>(a.wt);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  const T* __restrict__ rg = static_cast<const T*>(a.residual);
  T* __restrict__ y = static_cast<T*>(a.y);
  const int K = a.c_in, hw = static_cast<int>(a.hw);
  // ---- operand tiles; rows and columns past the problem are zero ----------
  // weights: BM rows of kp values (16-byte units when K is whole units)
  const int wunits = g.kp / 8;
  for (int e = tid; e < BM * wunits; e += kPwThreads) {
    const int r = e / wunits, q = e - (e / wunits) * wunits;
    const int m = m0 + r;
    T* dst = ws + r * g.wpitch + 8 * q;
    if (g.vec_w) {
      const bool ok = m < a.c_out && 8 * q < K;
      cp_async16_zfill(static_cast<uint32_t>(__cvta_generic_to_shared(dst)),
                       ok ? wg + static_cast<long long>(m) * K + 8 * q : wg, ok);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = 8 * q + j;
        dst[j] = (m < a.c_out && k < K) ? wg[static_cast<long long>(m) * K + k] : from_f32<T>(0.0f);
      }
    }
  }
  // pixels: kp rows (input channels) of 128 pixels of image n
  const T* ximg = xg + static_cast<long long>(n) * K * hw;
  constexpr int xunits = kPwBN / 8;
  for (int e = tid; e < g.kp * xunits; e += kPwThreads) {
    const int c = e / xunits, q = e - (e / xunits) * xunits;
    const int p = p0 + 8 * q;
    T* dst = xs + c * g.xpitch + 8 * q;
    if (g.vec_x) {  // H*W a multiple of 8: a unit is all in or all out
      const bool ok = c < K && p < hw;
      cp_async16_zfill(static_cast<uint32_t>(__cvta_generic_to_shared(dst)),
                       ok ? ximg + static_cast<long long>(c) * hw + p : xg, ok);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = (c < K && p + j < hw) ? ximg[static_cast<long long>(c) * hw + p + j] : from_f32<T>(0.0f);
    }
  }
  // the residual tile, when it is read by 16-byte copies: in flight with the operands
  if (g.vec_r) {
    const T* rimg = rg + static_cast<long long>(n) * a.c_out * hw;
    for (int e = tid; e < BM * xunits; e += kPwThreads) {
      const int r = e / xunits, q = e - (e / xunits) * xunits;
      const int m = m0 + r, p = p0 + 8 * q;
      const bool ok = m < a.c_out && p < hw;
      cp_async16_zfill(static_cast<uint32_t>(__cvta_generic_to_shared(rs + r * g.xpitch + 8 * q)),
                       ok ? rimg + static_cast<long long>(m) * hw + p : rg, ok);
    }
  }
  pw_commit_wait_all();
  __syncthreads();
  // ---- the warp's sub-tile: TMW x 16 channels by TNW x 8 pixels -----------
  const int wm = warp / WN, wn = warp - (warp / WN) * WN;
  const int row_l = lane & 15, col_l = (lane >> 4) * 8;
  const uint32_t wbase = static_cast<uint32_t>(__cvta_generic_to_shared(ws)) +
                         static_cast<uint32_t>(((wm * TMW * 16 + row_l) * g.wpitch + col_l) * sizeof(T));
  const uint32_t xbase = static_cast<uint32_t>(__cvta_generic_to_shared(xs)) +
                         static_cast<uint32_t>((row_l * g.xpitch + wn * TNW * 8 + col_l) * sizeof(T));
  float acc[TMW][TNW][4];
#pragma unroll
  for (int i = 0; i < TMW; ++i)
#pragma unroll
    for (int j = 0; j < TNW; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.0f;
  for (int k0 = 0; k0 < g.kp; k0 += 16) {
    uint32_t af[TMW][4], bf[TNW / 2][4];
#pragma unroll
    for (int i = 0; i < TMW; ++i)
      ldsm_x4(af[i], wbase + static_cast<uint32_t>((i * 16 * g.wpitch + k0) * sizeof(T)));
#pragma unroll
    for (int j = 0; j < TNW / 2; ++j)
      ldsm_x4_trans(bf[j], xbase + static_cast<uint32_t>((k0 * g.xpitch + j * 16) * sizeof(T)));
#pragma unroll
    for (int i = 0; i < TMW; ++i)
#pragma unroll
      for (int j = 0; j < TNW; ++j)
        pw_mma<T>(acc[i][j], af[i], bf[j >> 1][2 * (j & 1)], bf[j >> 1][2 * (j & 1) + 1]);
  }
  // ---- epilogue: accumulator (i, j, q) is channel m0 + 16 (wm TMW + i) +
  // lane / 4 (+ 8 for q >= 2) and pixel p0 + 8 (wn TNW + j) + 2 (lane % 4) + (q & 1).
  const long long img = static_cast<long long>(n) * a.c_out;
  if (a.raw_out) {  // the raw float32 sums into the float32 array y (no epilogue)
    float* __restrict__ yf = static_cast<float*>(a.y);
#pragma unroll
    for (int i = 0; i < TMW; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int co = m0 + (wm * TMW + i) * 16 + (lane >> 2) + 8 * h;
        if (co >= a.c_out) continue;
        const long long rowo = (img + co) * hw;
#pragma unroll
        for (int j = 0; j < TNW; ++j) {
          const int p = p0 + (wn * TNW + j) * 8 + 2 * (lane & 3);
          if (p >= hw) continue;
          if (p + 1 < hw && g.pair_io) {
            *reinterpret_cast<float2*>(yf + rowo + p) = make_float2(acc[i][j][2 * h], acc[i][j][2 * h + 1]);
          } else {
            yf[rowo + p] = acc[i][j][2 * h];
            if (p + 1 < hw) yf[rowo + p + 1] = acc[i][j][2 * h + 1];
          }
        }
      }
    }
    return;
  }
  // Bias and residual per value, then the activation over all of the thread's
  // values in one dispatch (a dispatch per pair would be if-converted into
  // evaluating every activation), then the stores.
  float* v = &acc[0][0][0];
  constexpr int NV = TMW * TNW * 4;
  if (bg || rg) {
#pragma unroll
    for (int i = 0; i < TMW; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rl = (wm * TMW + i) * 16 + (lane >> 2) + 8 * h;
        const int co = m0 + rl;
        if (co >= a.c_out) continue;
        const float bv = bg ? to_f32(bg[co]) : 0.0f;
        const long long rowo = (img + co) * hw;
#pragma unroll
        for (int j = 0; j < TNW; ++j) {
          const int cl = (wn * TNW + j) * 8 + 2 * (lane & 3);
          const int p = p0 + cl;
          if (p >= hw) continue;
          float& v0 = acc[i][j][2 * h];
          float& v1 = acc[i][j][2 * h + 1];
          if (bg) {
            v0 = __fadd_rn(v0, bv);
            v1 = __fadd_rn(v1, bv);
          }
          if (g.vec_r) {  // from the staged tile (pairs: H*W is a multiple of 8)
            const uint32_t rw = *reinterpret_cast<const uint32_t*>(rs + rl * g.xpitch + cl);
            const uint16_t lo = static_cast<uint16_t>(rw & 0xffffu), hi = static_cast<uint16_t>(rw >> 16);
            v0 = __fadd_rn(v0, to_f32(*reinterpret_cast<const T*>(&lo)));
            v1 = __fadd_rn(v1, to_f32(*reinterpret_cast<const T*>(&hi)));
          } else if (rg) {
            v0 = __fadd_rn(v0, to_f32(rg[rowo + p]));
            if (p + 1 < hw) v1 = __fadd_rn(v1, to_f32(rg[rowo + p + 1]));
          }
        }
      }
    }
  }
  activate_n<NV>(*reinterpret_cast<float(*)[NV]>(v), a.act, a.alpha, a.beta);
#pragma unroll
  for (int i = 0; i < TMW; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int co = m0 + (wm * TMW + i) * 16 + (lane >> 2) + 8 * h;
      if (co >= a.c_out) continue;
      const long long rowo = (img + co) * hw;
#pragma unroll
      for (int j = 0; j < TNW; ++j) {
        const int p = p0 + (wn * TNW + j) * 8 + 2 * (lane & 3);
        if (p >= hw) continue;
        const long long o = rowo + p;
        const bool two = p + 1 < hw;
        if (two && g.pair_io) {
          *reinterpret_cast<uint32_t*>(y + o) = pw_pack<T>(acc[i][j][2 * h], acc[i][j][2 * h + 1]);
        } else {
          y[o] = from_f32<T>(acc[i][j][2 * h]);
          if (two) y[o + 1] = from_f32<T>(acc[i][j][2 * h + 1]);
        }
      }
    }
  }
}

template <typename T, int TMW, int WM, int WN>
cudaError_t launch_pw_cfg(const PwPlan& pp, const ConvArgs& a, cudaStream_t s) {
  constexpr int BM = 16 * TMW * WM;
  PwGeo g;
  g.kp = pp.kp;
  g.wpitch = pp.kp + 8;
  g.xpitch = kPwBN + 8;
  g.pblocks = static_cast<int>((a.hw + kPwBN - 1) / kPwBN);
  g.vec_w = (a.c_in % 8 == 0) && reinterpret_cast<uintptr_t>(a.wt) % 16 == 0;
  g.vec_x = (a.hw % 8 == 0) && reinterpret_cast<uintptr_t>(a.x) % 16 == 0;
  g.pair_io = (a.hw % 2 == 0) && reinterpret_cast<uintptr_t>(a.y) % (a.raw_out ? 8 : 4) == 0 &&
              (!a.residual || reinterpret_cast<uintptr_t>(a.residual) % 4 == 0);
  g.vec_r = a.residual && (a.hw % 8 == 0) && reinterpret_cast<uintptr_t>(a.residual) % 16 == 0;
  const size_t smem = (static_cast<size_t>(BM) * g.wpitch + static_cast<size_t>(g.kp) * g.xpitch +
                       (g.vec_r ? static_cast<size_t>(BM) * g.xpitch : 0)) * sizeof(T);
  auto kern = pointwise_mma<T, TMW, WM, WN>;
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  const dim3 grid(static_cast<unsigned>(static_cast<long long>(a.n) * g.pblocks),
                  static_cast<unsigned>((a.c_out + BM - 1) / BM));
  kern<<<grid, kPwThreads, smem, s>>>(a, g);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_pw_typed(const PwPlan& pp, const ConvArgs& a, cudaStream_t s) {
  switch (pp.cfg) {
    case 1: return launch_pw_cfg<T, 1, 1, 8>(pp, a, s);
    case 2: return launch_pw_cfg<T, 2, 1, 8>(pp, a, s);
    case 3: return launch_pw_cfg<T, 3, 1, 8>(pp, a, s);
    case 4: return launch_pw_cfg<T, 4, 1, 8>(pp, a, s);
    case 5: return launch_pw_cfg<T, 4, 2, 4>(pp, a, s);  // 128 channels: the raw-sum Gemm of ConvTranspose
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t pw_smem_bytes(const PwPlan& pp, bool residual_tile) {
  const int bm = pp.cfg == 5 ? 128 : 16 * pp.cfg;
  return (static_cast<size_t>(bm) * (pp.kp + 8) +
          static_cast<size_t>(pp.kp + (residual_tile ? bm : 0)) * (kPwBN + 8)) * 2;
}

cudaError_t launch_pointwise(const PwPlan& pp, const ConvArgs& a, int dtype, cudaStream_t s) {
  if (dtype == CONV_F16) return launch_pw_typed<__half>(pp, a, s);
  if (dtype == CONV_BF16) return launch_pw_typed<__nv_bfloat16>(pp, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace conv
