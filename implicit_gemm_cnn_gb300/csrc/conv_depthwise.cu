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
// Work item = (image, group, block of output rows).  A block loops over items
// and stages the next item's input rows with cp.async (16/8/4-byte copies
// straight from the NCHW plane) while it computes the current one, so loads
// and arithmetic overlap; shared-memory columns left and right of the image
// are zeroed once and never written again, rows above / below the image are
// zeroed per item.  16-bit tiles are converted to float32 once on chip.  Each
// thread computes kQW adjacent outputs of a row for one of the m channels and
// sums each window in (kernel row, kernel column) order in one float32
// chain; for stride-1 / dilation-1 columns with a compiled kernel width the
// row segment sits in registers and is reused across the kQW outputs.  Bias,
// residual and activation are applied at the store.
#include <algorithm>

#include "conv_internal.h"

namespace conv {
namespace {

constexpr int kDwThreads = 128;
constexpr int kQW = 8;
constexpr int kBlocksPerSm = 12;

template <int BYTES>
__device__ __forceinline__ void cp_async_n(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(s), "l"(gmem), "n"(BYTES) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Store n (1..4) consecutive outputs of one row starting at o.
template <typename T>
__device__ __forceinline__ void store_run(T* __restrict__ y, long long o, float v0, float v1, float v2,
                                          float v3, int n, bool vec) {
  if (vec && n == 4) {
    if constexpr (sizeof(T) == 4) {
      *reinterpret_cast<float4*>(y + o) = make_float4(v0, v1, v2, v3);
    } else {
      T h[4] = {from_f32<T>(v0), from_f32<T>(v1), from_f32<T>(v2), from_f32<T>(v3)};
      *reinterpret_cast<uint2*>(y + o) = *reinterpret_cast<const uint2*>(h);
    }
  } else {
    const float v[4] = {v0, v1, v2, v3};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < n) y[o + q] = from_f32<T>(v[q]);
  }
}

template <typename T, int KW>
__global__ void __launch_bounds__(kDwThreads)
    depthwise(const ConvArgs a, const DwPlan d, int row_tiles, long long items) {
  extern __shared__ __align__(16) unsigned char dsm[];
  const int m = a.mg;
  const int nw = m * a.kh * a.kw;
  const int nw_pad = (nw + 3) & ~3;
  const int tile_elems = d.in_rows * d.row;
  float* wsm = reinterpret_cast<float*>(dsm);                  // [2][nw_pad]
  float* ftile = wsm + 2 * nw_pad;                             // [tile] (16-bit inputs)
  T* raw = reinterpret_cast<T*>(ftile + (sizeof(T) == 4 ? 0 : tile_elems));  // [2][tile]
  const int tid = threadIdx.x;
  const T* __restrict__ xg = static_cast<const T*>(a.x);
  const T* __restrict__ wg = static_cast<const T*>(a.wt);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  const T* __restrict__ rg = static_cast<const T*>(a.residual);
  T* __restrict__ y = static_cast<T*>(a.y);

  for (int i = tid; i < 2 * tile_elems; i += kDwThreads) raw[i] = from_f32<T>(0.0f);
  __syncthreads();

  // Stage item `it` into buffer st: zero its out-of-image rows, copy its image
  // rows, convert its weights.
  auto prefetch = [&](long long it, int st) {
    const long long plane = it / row_tiles;
    const int rt = static_cast<int>(it - plane * row_tiles);
    const int n = static_cast<int>(plane / a.groups);
    const int g = static_cast<int>(plane - static_cast<long long>(n) * a.groups);
    const int ih_start = rt * d.th * a.sh - a.pt;
    const int r_lo = max(0, ih_start), r_hi = min(a.h, ih_start + d.in_rows);
    T* buf = raw + st * tile_elems;
    const int zr_top = min(d.in_rows, r_lo - ih_start);        // staged rows above the image
    const int zr_bot = d.in_rows - zr_top - max(0, r_hi - r_lo);  // staged rows below it
    const int zrows = zr_top + zr_bot;
    for (int i = tid; i < zrows * a.w; i += kDwThreads) {
      const int zr = i / a.w, c = i - (i / a.w) * a.w;
      const int r = zr < zr_top ? zr : d.in_rows - zr_bot + (zr - zr_top);
      buf[r * d.row + d.lm + c] = from_f32<T>(0.0f);
    }
    const int count = max(0, r_hi - r_lo) * a.w;
    if (count > 0) {
      const T* src = xg + (static_cast<long long>(n) * a.c_in + g) * a.hw + static_cast<long long>(r_lo) * a.w;
      T* dst0 = buf + zr_top * d.row + d.lm;
      if (d.vec > 0) {
        const int ve = d.vec / static_cast<int>(sizeof(T));  // elements per copy
        const int nchunk = count / ve;
        for (int q = tid; q < nchunk; q += kDwThreads) {
          const int f = q * ve;
          const int r = f / a.w, c = f - (f / a.w) * a.w;
          T* dst = dst0 + r * d.row + c;
          if (d.vec == 16) cp_async_n<16>(dst, src + f);
          else if (d.vec == 8) cp_async_n<8>(dst, src + f);
          else cp_async_n<4>(dst, src + f);
        }
      } else {
        for (int f = tid; f < count; f += kDwThreads) {
          const int r = f / a.w, c = f - (f / a.w) * a.w;
          dst0[r * d.row + c] = src[f];
        }
      }
    }
    float* wd = wsm + st * nw_pad;
    for (int i = tid; i < nw; i += kDwThreads) wd[i] = to_f32(wg[static_cast<long long>(g) * nw + i]);
  };

  const bool fast = (KW != 0) && a.sw == 1 && a.dw == 1 && a.kw == KW;
  const bool pair_ok = ((d.lm - a.pl) & 1) == 0 && (d.row & 1) == 0;
  const bool vec_out = a.vec_out && (a.wo & 3) == 0;

  long long it = blockIdx.x;
  if (it < items) prefetch(it, 0);
  cp_async_commit();
  for (int i = 0; it < items; it += gridDim.x, ++i) {
    const int st = i & 1;
    const long long nx = it + gridDim.x;
    if (nx < items) prefetch(nx, st ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const float* tile;
    if constexpr (sizeof(T) == 4) {
      tile = reinterpret_cast<const float*>(raw + st * tile_elems);
    } else {
      const T* rb = raw + st * tile_elems;
      for (int e = tid; e < tile_elems; e += kDwThreads) ftile[e] = to_f32(rb[e]);
      __syncthreads();
      tile = ftile;
    }
    const float* wts = wsm + st * nw_pad;

    const long long plane = it / row_tiles;
    const int rt = static_cast<int>(it - plane * row_tiles);
    const int n = static_cast<int>(plane / a.groups);
    const int g = static_cast<int>(plane - static_cast<long long>(n) * a.groups);
    const int oh0 = rt * d.th;
    const int rows_out = min(d.th, a.ho - oh0);
    const int strips = (a.wo + kQW - 1) / kQW;
    const int work = rows_out * strips * m;
    for (int wi = tid; wi < work; wi += kDwThreads) {
      const int j = wi / (rows_out * strips);
      const int rem = wi - j * (rows_out * strips);
      const int ohl = rem / strips;
      const int ow0 = (rem - ohl * strips) * kQW;
      const float* wj = wts + j * a.kh * a.kw;
      float acc[kQW];
#pragma unroll
      for (int q = 0; q < kQW; ++q) acc[q] = 0.0f;
      if (fast) {
        constexpr int KWc = KW > 0 ? KW : 1;
        constexpr int SEG = kQW + KWc - 1;
        for (int u = 0; u < a.kh; ++u) {
          const float* srow = tile + (ohl * a.sh + u * a.dh) * d.row + d.lm - a.pl + ow0;
          float seg[SEG + 1];
          if (pair_ok) {
#pragma unroll
            for (int e = 0; e < (SEG + 1) / 2; ++e) {
              const float2 v = *reinterpret_cast<const float2*>(srow + 2 * e);
              seg[2 * e] = v.x;
              seg[2 * e + 1] = v.y;
            }
          } else {
#pragma unroll
            for (int e = 0; e < SEG; ++e) seg[e] = srow[e];
          }
#pragma unroll
          for (int v = 0; v < KWc; ++v) {
            const float wv = wj[u * KWc + v];
#pragma unroll
            for (int q = 0; q < kQW; ++q) acc[q] = fmaf(seg[q + v], wv, acc[q]);
          }
        }
      } else {
        for (int u = 0; u < a.kh; ++u) {
          const float* srow = tile + (ohl * a.sh + u * a.dh) * d.row + d.lm - a.pl + ow0 * a.sw;
          for (int v = 0; v < a.kw; ++v) {
            const float wv = wj[u * a.kw + v];
#pragma unroll
            for (int q = 0; q < kQW; ++q) acc[q] = fmaf(srow[q * a.sw + v * a.dw], wv, acc[q]);
          }
        }
      }
      const int co = g * m + j;
      const long long out = ((static_cast<long long>(n) * a.c_out + co) * a.ho + oh0 + ohl) * a.wo + ow0;
      const float bv = bg ? to_f32(__ldg(bg + co)) : 0.0f;
      const int nvalid = min(kQW, a.wo - ow0);
      float rv[kQW];
#pragma unroll
      for (int q = 0; q < kQW; ++q) rv[q] = (rg && q < nvalid) ? to_f32(__ldg(rg + out + q)) : 0.0f;
      float v[kQW];
#pragma unroll
      for (int q = 0; q < kQW; ++q)
        v[q] = to_f32(epilogue_vals<T>(acc[q], bv, rv[q], bg != nullptr, rg != nullptr, a.act, a.alpha, a.beta));
      store_run<T>(y, out, v[0], v[1], v[2], v[3], min(4, nvalid), vec_out);
      if (nvalid > 4) store_run<T>(y, out + 4, v[4], v[5], v[6], v[7], nvalid - 4, vec_out);
    }
    __syncthreads();  // this buffer is refilled two items from now
  }
  cp_async_wait<0>();
}

template <typename T, int KW>
cudaError_t launch_kw(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  const int row_tiles = (a.ho + d.th - 1) / d.th;
  const long long items = static_cast<long long>(a.n) * a.groups * row_tiles;
  const long long blocks = std::min<long long>(items, static_cast<long long>(d.sm) * kBlocksPerSm);
  const size_t smem = depthwise_smem_bytes(d, a.mg, a.kh, a.kw, sizeof(T) == 4 ? CONV_F32 : CONV_F16);
  auto kern = depthwise<T, KW>;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  kern<<<static_cast<unsigned>(blocks), kDwThreads, smem, s>>>(a, d, row_tiles, items);
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

size_t depthwise_smem_bytes(const DwPlan& d, int mg, int kh, int kw, int dtype) {
  const size_t tile = static_cast<size_t>(d.in_rows) * d.row;
  const size_t es = dtype == CONV_F32 ? 4 : 2;
  return 2 * static_cast<size_t>((mg * kh * kw + 3) & ~3) * 4 + (es == 4 ? 0 : tile * 4) + 2 * tile * es;
}

cudaError_t launch_depthwise(const Plan& plan, const ConvArgs& a, int dtype, cudaStream_t s) {
  switch (dtype) {
    case CONV_F32: return launch_typed<float>(plan.dw, a, s);
    case CONV_F16: return launch_typed<__half>(plan.dw, a, s);
    case CONV_BF16: return launch_typed<__nv_bfloat16>(plan.dw, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace conv
