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
// zeroed per item.  16-bit tiles are converted to float32 once on chip.  The
// next item's weights and bias travel in registers while the current item is
// computed.
//
// Each thread computes kQH outputs of one output column (consecutive lanes,
// consecutive columns: conflict-free shared-memory reads).  For stride-1 /
// dilation-1 rows with a compiled kernel height, the kQH + kh - 1 window
// values of one kernel column sit in registers and serve all kQH outputs;
// each output is summed in one float32 chain in (kernel column, kernel row)
// order.  Bias, residual and activation are applied at the store.
//
// Planes at most 32 output columns wide at stride 1 take leaner paths (one
// warp per plane, below): no work-item arithmetic per output, the next plane
// copied while the current one is computed -- four output columns per lane
// where the plane's rows divide among the lanes, else one column per lane.
#include <algorithm>
#include <type_traits>

#include "conv_internal.h"

namespace conv {
namespace {

constexpr int kDwThreads = 128;
constexpr int kQH = 8;
constexpr int kBlocksPerSm = 12;
constexpr int kRegW = 4;  // weights per thread carried in registers (m*kh*kw <= 512)

template <int BYTES>
__device__ __forceinline__ void cp_async_n(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(s), "l"(gmem), "n"(BYTES) : "memory");
}
// n copies of BYTES each, the k-th from s + k * sstep to shared address d + k * dstep.
template <int BYTES>
__device__ __forceinline__ void cp_async_run(uint32_t d, const char* s, int n, uint32_t dstep, long long sstep) {
  for (int k = 0; k < n; ++k) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(d), "l"(s), "n"(BYTES) : "memory");
    d += dstep;
    s += sstep;
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <typename T, int KH>
__global__ void __launch_bounds__(kDwThreads)
    depthwise(const ConvArgs a, const DwPlan d, int row_tiles, long long items) {
  extern __shared__ __align__(16) unsigned char dsm[];
  const int m = a.mg;
  const int nw = m * a.kh * a.kw;
  const int nw_pad = (nw + 3) & ~3;
  const int mb_pad = (m + 3) & ~3;
  const int tile_elems = d.in_rows * d.row;
  float* wsm = reinterpret_cast<float*>(dsm);                  // [2][nw_pad]
  float* bsm = wsm + 2 * nw_pad;                               // [2][mb_pad]
  float* ftile = bsm + 2 * mb_pad;                             // [tile] (16-bit inputs)
  T* raw = reinterpret_cast<T*>(ftile + (sizeof(T) == 4 ? 0 : tile_elems));  // [2][tile]
  const int tid = threadIdx.x;
  const T* __restrict__ xg = static_cast<const T*>(a.x);
  const T* __restrict__ wg = static_cast<const T*>(a.wt);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  const T* __restrict__ rg = static_cast<const T*>(a.residual);
  T* __restrict__ y = static_cast<T*>(a.y);
  const bool wregs = nw <= kRegW * kDwThreads && m <= kDwThreads;

  for (int i = tid; i < 2 * tile_elems; i += kDwThreads) raw[i] = from_f32<T>(0.0f);

  auto decode = [&](long long it, int* n, int* g, int* rt) {
    const long long plane = it / row_tiles;
    *rt = static_cast<int>(it - plane * row_tiles);
    *n = static_cast<int>(plane / a.groups);
    *g = static_cast<int>(plane - static_cast<long long>(*n) * a.groups);
  };
  // Stage item `it`'s input rows into buffer st (zero rows outside the image,
  // cp.async copies of the image rows).
  auto stage_rows = [&](long long it, int st) {
    int n, g, rt;
    decode(it, &n, &g, &rt);
    const int ih_start = rt * d.th * a.sh - a.pt;
    const int r_lo = max(0, ih_start), r_hi = min(a.h, ih_start + d.in_rows);
    T* buf = raw + st * tile_elems;
    const int zr_top = min(d.in_rows, r_lo - ih_start);           // staged rows above the image
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
  };
  // Weights and bias of item `it`: into registers now, into shared memory
  // (buffer st) when the current item's compute is done.
  float wreg[kRegW], breg = 0.0f;
  auto load_params = [&](long long it) {
    int n, g, rt;
    decode(it, &n, &g, &rt);
#pragma unroll
    for (int k = 0; k < kRegW; ++k) {
      const int i = tid + k * kDwThreads;
      wreg[k] = i < nw ? to_f32(wg[static_cast<long long>(g) * nw + i]) : 0.0f;
    }
    breg = (bg && tid < m) ? to_f32(bg[g * m + tid]) : 0.0f;
  };
  auto store_params = [&](int st) {
#pragma unroll
    for (int k = 0; k < kRegW; ++k) {
      const int i = tid + k * kDwThreads;
      if (i < nw) wsm[st * nw_pad + i] = wreg[k];
    }
    if (tid < m) bsm[st * mb_pad + tid] = breg;
  };
  auto load_params_direct = [&](long long it, int st) {  // multipliers too large for registers
    int n, g, rt;
    decode(it, &n, &g, &rt);
    for (int i = tid; i < nw; i += kDwThreads) wsm[st * nw_pad + i] = to_f32(wg[static_cast<long long>(g) * nw + i]);
    for (int i = tid; i < m; i += kDwThreads) bsm[st * mb_pad + i] = bg ? to_f32(bg[g * m + i]) : 0.0f;
  };

  const bool fast = (KH != 0) && a.sh == 1 && a.dh == 1 && a.kh == KH;

  long long it = blockIdx.x;
  if (it < items) {
    stage_rows(it, 0);
    if (wregs) { load_params(it); store_params(0); } else { load_params_direct(it, 0); }
  }
  cp_async_commit();
  for (int i = 0; it < items; it += gridDim.x, ++i) {
    const int st = i & 1;
    const long long nx = it + gridDim.x;
    if (nx < items) {
      stage_rows(nx, st ^ 1);
      if (wregs) load_params(nx);
      else load_params_direct(nx, st ^ 1);
    }
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
    const float* bia = bsm + st * mb_pad;

    int n, g, rt;
    decode(it, &n, &g, &rt);
    const int oh0 = rt * d.th;
    const int rows_out = min(d.th, a.ho - oh0);
    const int vstrips = (rows_out + kQH - 1) / kQH;
    const int cols32 = (a.wo + 31) / 32 * 32;
    const int work = m * vstrips * cols32;
    for (int wi = tid; wi < work; wi += kDwThreads) {
      const int ow = wi % cols32;
      const int rest = wi / cols32;
      const int vs = rest % vstrips;
      const int j = rest / vstrips;
      if (ow >= a.wo) continue;
      const int ohl0 = vs * kQH;
      const int nq = min(kQH, rows_out - ohl0);
      const int co = g * m + j;
      const long long out0 = ((static_cast<long long>(n) * a.c_out + co) * a.ho + oh0 + ohl0) * a.wo + ow;
      float rv[kQH];
#pragma unroll
      for (int q = 0; q < kQH; ++q)
        rv[q] = (rg && q < nq) ? to_f32(__ldg(rg + out0 + static_cast<long long>(q) * a.wo)) : 0.0f;
      const float* wj = wts + j * a.kh * a.kw;
      const float* scol = tile + ohl0 * a.sh * d.row + d.lm - a.pl + ow * a.sw;
      float acc[kQH];
#pragma unroll
      for (int q = 0; q < kQH; ++q) acc[q] = 0.0f;
      if (fast) {
        constexpr int KHc = KH > 0 ? KH : 1;
        for (int v = 0; v < a.kw; ++v) {
          const float* sc = scol + v * a.dw;
          float col[kQH + KHc - 1];
#pragma unroll
          for (int r = 0; r < kQH + KHc - 1; ++r) col[r] = sc[r * d.row];
#pragma unroll
          for (int u = 0; u < KHc; ++u) {
            const float wv = wj[u * a.kw + v];
#pragma unroll
            for (int q = 0; q < kQH; ++q) acc[q] = fmaf(col[q + u], wv, acc[q]);
          }
        }
      } else {
        for (int v = 0; v < a.kw; ++v) {
          for (int u = 0; u < a.kh; ++u) {
            const float wv = wj[u * a.kw + v];
            const float* sc = scol + u * a.dh * d.row + v * a.dw;
#pragma unroll
            for (int q = 0; q < kQH; ++q)
              if (q < nq) acc[q] = fmaf(sc[q * a.sh * d.row], wv, acc[q]);
          }
        }
      }
      float bv[kQH];
#pragma unroll
      for (int q = 0; q < kQH; ++q) bv[q] = bia[j];
      epilogue_n<kQH>(acc, bv, rv, bg != nullptr, rg != nullptr, a.act, a.alpha, a.beta);
#pragma unroll
      for (int q = 0; q < kQH; ++q)
        if (q < nq) y[out0 + static_cast<long long>(q) * a.wo] = from_f32<T>(acc[q]);
    }
    if (wregs && nx < items) store_params(st ^ 1);
    __syncthreads();  // this buffer is refilled two items from now
  }
  cp_async_wait<0>();
}

// ---- narrow planes: one warp per (image, output channel) plane -------------
// For stride 1, dilation 1, square 3/5/7 kernels and planes at most 32 output
// columns wide (the late layers of MobileNet-style networks): lane = output
// column.  Each warp owns two shared-memory buffers of (Ho + K - 1) rows of
// `pitch` elements holding a zero-bordered input plane (the border is written
// once); while it computes one plane, cp.async copies of the next plane's rows
// fill the other buffer.  Each lane walks down its column with the K x K input
// window in registers, loading one new row segment (K values) per output row,
// and sums each output in one float32 chain in (kernel row, kernel column)
// order.  The activation is a template parameter, so the value loop holds no
// switch.
constexpr int kNwWarps = 8;  // warps per block (one plane each at a time)

struct NarrowGeo {
  int pitch;  // elements per staged row (even)
  int rows;   // staged rows: Ho + K - 1
  int cofs;   // buffer column of image column 0 (even for 16-bit elements)
  int async;  // rows copied with 4-byte cp.async (else element loads)
};

template <typename T, int K, int ACT>
__device__ __forceinline__ void narrow_planes(const ConvArgs& a, const NarrowGeo& g, T* buf0, long long planes,
                                              long long first, long long stride) {
  const int lane = threadIdx.x & 31;
  const T* __restrict__ xg = static_cast<const T*>(a.x);
  const T* __restrict__ wg = static_cast<const T*>(a.wt);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  const T* __restrict__ rg = static_cast<const T*>(a.residual);
  T* __restrict__ y = static_cast<T*>(a.y);
  const int m = a.mg;  // output channels per input channel
  const int bufsz = g.pitch * g.rows;
  // image rows / columns land at (pt + r, cofs + c); clip what no window reads
  const int r_hi = min(a.h, g.rows - a.pt), c_hi = min(a.w, g.pitch - g.cofs);
  constexpr int kPer = 4 / sizeof(T);  // elements per 4-byte copy
  auto stage = [&](long long pl, T* buf) {
    const int n = static_cast<int>(pl / a.c_out);
    const int co = static_cast<int>(pl - static_cast<long long>(n) * a.c_out);
    const T* src = xg + (static_cast<long long>(n) * a.c_in + co / m) * a.hw;
    if (g.async) {
      const int units = (c_hi + kPer - 1) / kPer;  // 4-byte units per row
      for (int r = 0; r < r_hi; ++r) {
        T* drow = buf + (a.pt + r) * g.pitch + g.cofs;
        const T* srow = src + static_cast<long long>(r) * a.w;
        for (int q = lane; q < units; q += 32) cp_async_n<4>(drow + q * kPer, srow + q * kPer);
      }
    } else {
      for (int r = 0; r < r_hi; ++r) {
        T* drow = buf + (a.pt + r) * g.pitch + g.cofs;
        const T* srow = src + static_cast<long long>(r) * a.w;
        for (int c = lane; c < c_hi; c += 32) drow[c] = srow[c];
      }
    }
  };
  int k = 0;
  if (first < planes) stage(first, buf0);
  cp_async_commit();
  for (long long pl = first; pl < planes; pl += stride, ++k) {
    T* buf = buf0 + (k & 1) * bufsz;
    if (pl + stride < planes) stage(pl + stride, buf0 + ((k + 1) & 1) * bufsz);
    cp_async_commit();
    const int n = static_cast<int>(pl / a.c_out);
    const int co = static_cast<int>(pl - static_cast<long long>(n) * a.c_out);
    float wv[K][K];
#pragma unroll
    for (int u = 0; u < K; ++u)
#pragma unroll
      for (int v = 0; v < K; ++v) wv[u][v] = to_f32(wg[static_cast<long long>(co) * K * K + u * K + v]);
    const float bv = bg ? to_f32(bg[co]) : 0.0f;
    cp_async_wait<1>();  // this plane's copies (the next plane's may still fly)
    __syncwarp();
    if (lane < a.wo) {
      const T* col = buf + g.cofs - a.pl + lane;
      float win[K][K];  // slot (row % K) holds an input row of the window
#pragma unroll
      for (int i = 0; i < K - 1; ++i)
#pragma unroll
        for (int v = 0; v < K; ++v) win[i][v] = to_f32(col[i * g.pitch + v]);
      T* yo = y + (static_cast<long long>(n) * a.c_out + co) * a.howo + lane;
      const T* ro = rg ? rg + (static_cast<long long>(n) * a.c_out + co) * a.howo + lane : nullptr;
      for (int oh0 = 0; oh0 < a.ho; oh0 += K) {
#pragma unroll
        for (int s = 0; s < K; ++s) {
          const int oh = oh0 + s;
          if (oh >= a.ho) break;
          // the window's newest row: input row oh + K - 1 into slot (s + K - 1) % K
#pragma unroll
          for (int v = 0; v < K; ++v) win[(s + K - 1) % K][v] = to_f32(col[(oh + K - 1) * g.pitch + v]);
          float acc = 0.0f;
#pragma unroll
          for (int u = 0; u < K; ++u)
#pragma unroll
            for (int v = 0; v < K; ++v) acc = fmaf(win[(s + u) % K][v], wv[u][v], acc);
          float t = acc;
          if (bg) t = __fadd_rn(t, bv);
          if (ro) t = __fadd_rn(t, to_f32(ro[oh * a.wo]));
          yo[oh * a.wo] = from_f32<T>(act_fn<ACT>(t, a.alpha, a.beta));
        }
      }
    }
    __syncwarp();  // this buffer's reads are done before it is refilled
  }
  cp_async_wait<0>();
}

template <typename T, int K>
__global__ void __launch_bounds__(kNwWarps * 32, K == 7 ? 2 : 3) depthwise_narrow(const ConvArgs a, const NarrowGeo g) {
  extern __shared__ __align__(16) unsigned char dsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  T* buf = reinterpret_cast<T*>(dsm) + static_cast<size_t>(warp) * 2 * g.pitch * g.rows;
  for (int i = lane; i < 2 * g.pitch * g.rows; i += 32) buf[i] = from_f32<T>(0.0f);  // the border stays zero
  __syncwarp();
  const long long planes = static_cast<long long>(a.n) * a.c_out;
  const long long first = static_cast<long long>(blockIdx.x) * kNwWarps + warp;
  const long long stride = static_cast<long long>(gridDim.x) * kNwWarps;
  switch (a.act) {
#define CONV_NW_CASE(A) \
  case A: narrow_planes<T, K, A>(a, g, buf, planes, first, stride); break;
    CONV_NW_CASE(ACT_RELU)
    CONV_NW_CASE(ACT_SILU)
    CONV_NW_CASE(ACT_SIGMOID)
    CONV_NW_CASE(ACT_TANH)
    CONV_NW_CASE(ACT_HARD_SWISH)
    CONV_NW_CASE(ACT_HARD_SIGMOID)
    CONV_NW_CASE(ACT_CLIP)
    CONV_NW_CASE(ACT_LEAKY_RELU)
#undef CONV_NW_CASE
    default: narrow_planes<T, K, ACT_IDENTITY>(a, g, buf, planes, first, stride);
  }
}

// ---- narrow planes, four output columns per lane -----------------------------
// One warp per plane (image, output channel) at a time; lane = (group of 4
// output columns, block of R output rows).  The zero-bordered plane sits in
// shared memory, two buffers per warp: the next plane arrives by cp.async
// (16-, 8- or 4-byte copies; each lane keeps one copy column and strides down
// the rows) while this one is computed.  A lane streams the R + K - 1 input
// rows its outputs read, each as K + 3 consecutive values fetched with vector
// shared loads, and adds the row's taps to the 4 x R accumulators it feeds:
// input row i serves output row i - u with kernel row u, so each output is
// summed in one float32 chain in (u, v) order, the order of every other
// kernel here.  Weights sit in registers; bias, residual and activation are
// applied at the store, four outputs per vector store where aligned.
struct Cols4Geo {
  int pitch;       // elements per staged row (a multiple of 16 bytes)
  int rows;        // staged rows: rblocks * R + K - 1 (rows past the plane stay zero)
  int copy;        // bytes per cp.async copy of an image row (16, 8, 4), 0: element loads
  int groups;      // column groups: ceil(Wo / 4)
  int rblocks;     // row blocks: 32 / groups
  int vec_io;      // Ho*Wo and Wo multiples of 4, y (and the residual) 16-byte aligned
  int out_stride;  // floats of one warp's staged sums (Ho*Wo rounded up to 4)
};

template <typename T, int N>
__device__ __forceinline__ void load_row_vals(const T* src, float (&v)[N]) {
  // N consecutive elements starting at a 4-element boundary of shared memory
  static_assert(N % 4 == 0, "whole quads");
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
      const float4 t = reinterpret_cast<const float4*>(src)[q];
      v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
      const uint2 t = reinterpret_cast<const uint2*>(src)[q];
      const T* h = reinterpret_cast<const T*>(&t);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[4 * q + e] = to_f32(h[e]);
    }
  }
}

// The epilogue of one plane, after its sums are in `out` (float32, the plane's
// Ho x Wo outputs in order): bias, residual, activation, one rounding, stores
// of 4 consecutive outputs by consecutive lanes (coalesced).
template <typename T, int ACT>
__device__ __forceinline__ void cols4_store_plane(const ConvArgs& a, const float* out, long long pbase, float bv,
                                                  bool has_bias, int vec_io) {
  const int lane = threadIdx.x & 31;
  const T* __restrict__ rg = static_cast<const T*>(a.residual);
  T* __restrict__ y = static_cast<T*>(a.y);
  const int hw = a.ho * a.wo;
  if (vec_io) {  // Ho*Wo a multiple of 4, y (and the residual) 16-byte aligned
#pragma unroll 2
    for (int e = 4 * lane; e < hw; e += 128) {
      float v[4];
      const float4 t = *reinterpret_cast<const float4*>(out + e);
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (has_bias) v[c] = __fadd_rn(v[c], bv);
        if (rg) v[c] = __fadd_rn(v[c], to_f32(rg[pbase + e + c]));
        v[c] = act_fn<ACT>(v[c], a.alpha, a.beta);
      }
      if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4*>(y + pbase + e) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
        T h[4] = {from_f32<T>(v[0]), from_f32<T>(v[1]), from_f32<T>(v[2]), from_f32<T>(v[3])};
        *reinterpret_cast<uint2*>(y + pbase + e) = *reinterpret_cast<const uint2*>(h);
      }
    }
  } else {
    for (int e = lane; e < hw; e += 32) {
      float v = out[e];
      if (has_bias) v = __fadd_rn(v, bv);
      if (rg) v = __fadd_rn(v, to_f32(rg[pbase + e]));
      y[pbase + e] = from_f32<T>(act_fn<ACT>(v, a.alpha, a.beta));
    }
  }
}

constexpr int kC4Warps = 4;  // warps per block of the four-column kernel (five blocks per SM)

template <typename T, int K, int R>
__global__ void __launch_bounds__(kC4Warps * 32, 5) depthwise_cols4(const ConvArgs a, const Cols4Geo g) {
  constexpr int NV = (K + 3 + 3) / 4 * 4;  // values read per input row (K + 3, rounded to quads)
  extern __shared__ __align__(16) unsigned char dsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bufsz = g.pitch * g.rows;
  T* buf0 = reinterpret_cast<T*>(dsm) + static_cast<size_t>(warp) * 2 * bufsz;
  // the plane's float32 sums (Ho x Wo), staged for the coalesced epilogue
  float* outs = reinterpret_cast<float*>(dsm + static_cast<size_t>(kC4Warps) * 2 * bufsz * sizeof(T)) +
                static_cast<size_t>(warp) * g.out_stride;
  {  // the border stays zero (a buffer is a whole number of 16-byte units)
    uint4* z = reinterpret_cast<uint4*>(buf0);
    const int units16 = 2 * bufsz * static_cast<int>(sizeof(T)) / 16;
    for (int i = lane; i < units16; i += 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncwarp();
  const T* __restrict__ xg = static_cast<const T*>(a.x);
  const T* __restrict__ wg = static_cast<const T*>(a.wt);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  const int planes = a.n * a.c_out;  // fits int32 (checked by the planner)
  // planes are dealt round-robin over the blocks first, so the last, partly
  // filled round of planes spreads over all SMs
  const int first = warp * gridDim.x + blockIdx.x;
  const int stride = gridDim.x * kC4Warps;
  const int m = a.mg;
  // staging: image rows land at buffer row pt + r, column pl + c; a lane keeps
  // one copy column and strides down the rows
  const int rows_s = min(a.h, g.rows - a.pt);
  const int ce = g.copy ? g.copy / static_cast<int>(sizeof(T)) : 1;  // elements per copy
  const int units = (a.w + ce - 1) / ce;                            // copies per image row
  const int rpp = units <= 32 ? 32 / units : 1;                      // rows per pass of the warp
  const int my_r0 = units <= 32 ? lane / units : 0;
  const int my_q = units <= 32 ? lane - my_r0 * units : lane;
  const int q_step = units <= 32 ? units : 32;
  const bool stager = units <= 32 ? my_r0 < rpp : true;
  // with at most 32 copies per image row a lane's copies are one column q and
  // the rows my_r0, my_r0 + rpp, ...: the same shared and global offsets for
  // every plane, stepped by constants (no per-copy index arithmetic)
  const bool prog = units <= 32 && g.copy != 0;
  const int ncp = prog && stager && rows_s > my_r0 ? (rows_s - my_r0 + rpp - 1) / rpp : 0;
  const uint32_t dst_first =
      static_cast<uint32_t>(((a.pt + my_r0) * g.pitch + a.pl + my_q * ce) * static_cast<int>(sizeof(T)));
  const uint32_t dst_step = static_cast<uint32_t>(rpp * g.pitch * static_cast<int>(sizeof(T)));
  const long long src_first = (static_cast<long long>(my_r0) * a.w + my_q * ce) * static_cast<long long>(sizeof(T));
  const long long src_step = static_cast<long long>(rpp) * a.w * static_cast<long long>(sizeof(T));
  auto stage = [&](int n, int co, T* buf) {
    if (!stager) return;
    const T* src = xg + (static_cast<long long>(n) * a.c_in + (m == 1 ? co : co / m)) * a.hw;
    if (prog) {
      const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(buf)) + dst_first;
      const char* sp = reinterpret_cast<const char*>(src) + src_first;
      if (g.copy == 16) cp_async_run<16>(d, sp, ncp, dst_step, src_step);
      else if (g.copy == 8) cp_async_run<8>(d, sp, ncp, dst_step, src_step);
      else cp_async_run<4>(d, sp, ncp, dst_step, src_step);
      return;
    }
    T* dst = buf + a.pt * g.pitch + a.pl;
    if (g.copy == 16) {
      for (int r = my_r0; r < rows_s; r += rpp)
        for (int q = my_q; q < units; q += q_step) cp_async_n<16>(dst + r * g.pitch + q * ce, src + r * a.w + q * ce);
    } else if (g.copy == 8) {
      for (int r = my_r0; r < rows_s; r += rpp)
        for (int q = my_q; q < units; q += q_step) cp_async_n<8>(dst + r * g.pitch + q * ce, src + r * a.w + q * ce);
    } else if (g.copy == 4) {
      for (int r = my_r0; r < rows_s; r += rpp)
        for (int q = my_q; q < units; q += q_step) cp_async_n<4>(dst + r * g.pitch + q * ce, src + r * a.w + q * ce);
    } else {
      for (int r = my_r0; r < rows_s; r += rpp)
        for (int q = my_q; q < units; q += q_step) dst[r * g.pitch + q] = src[r * a.w + q];
    }
  };
  // this lane's outputs: columns 4j .. 4j+3, rows rb*R .. rb*R + R - 1
  const int j = lane % g.groups, rb = lane / g.groups;
  const bool worker = rb < g.rblocks && 4 * j < a.wo;
  int k = 0;
  // (image, channel) of plane pl, stepped by `stride` planes without a division
  const int step_n = stride / a.c_out, step_c = stride - (stride / a.c_out) * a.c_out;
  int n = first / a.c_out, co = first - (first / a.c_out) * a.c_out;
  auto next_plane = [&](int& pn, int& pc) {
    pn += step_n;
    pc += step_c;
    if (pc >= a.c_out) { pc -= a.c_out; ++pn; }
  };
  if (first < planes) stage(n, co, buf0);
  cp_async_commit();
  for (int pl = first; pl < planes; pl += stride, ++k) {
    T* buf = buf0 + (k & 1) * bufsz;
    int n_next = n, co_next = co;
    next_plane(n_next, co_next);
    if (pl + stride < planes) stage(n_next, co_next, buf0 + ((k + 1) & 1) * bufsz);
    cp_async_commit();
    float wv[K][K];
#pragma unroll
    for (int u = 0; u < K; ++u)
#pragma unroll
      for (int v = 0; v < K; ++v) wv[u][v] = to_f32(wg[static_cast<long long>(co) * K * K + u * K + v]);
    const float bv = bg ? to_f32(bg[co]) : 0.0f;
    cp_async_wait<1>();  // this plane's copies (the next plane's may still fly)
    __syncwarp();
    if (worker) {
      float acc[R][4];
#pragma unroll
      for (int o = 0; o < R; ++o)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[o][c] = 0.0f;
      const T* base = buf + (rb * R) * g.pitch + 4 * j;  // buffer row rb*R, the group's first window column
#pragma unroll
      for (int i = 0; i < R + K - 1; ++i) {
        float xv[NV];
        load_row_vals<T, NV>(base + i * g.pitch, xv);
        // input row i feeds output row i - u with kernel row u; v outermost
        // interleaves the independent output rows (each output's terms still
        // arrive in (u, v) order: one u per input row, v ascending)
#pragma unroll
        for (int v = 0; v < K; ++v)
#pragma unroll
          for (int u = 0; u < K; ++u) {
            const int o = i - u;
            if (o < 0 || o >= R) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[o][c] = fmaf(xv[c + v], wv[u][v], acc[o][c]);
          }
      }
      // the sums into the plane's staging area (rows past Ho, columns past Wo dropped)
#pragma unroll
      for (int o = 0; o < R; ++o) {
        const int oh = rb * R + o;
        if (oh >= a.ho) break;
        float* dst = outs + oh * a.wo + 4 * j;
        if (g.vec_io && 4 * j + 3 < a.wo) {
          *reinterpret_cast<float4*>(dst) = make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (4 * j + c < a.wo) dst[c] = acc[o][c];
        }
      }
    }
    __syncwarp();  // this plane's sums are staged and its input buffer is read
    const long long pbase = (static_cast<long long>(n) * a.c_out + co) * a.howo;
    switch (a.act) {
#define CONV_C4_CASE(A) \
  case A: cols4_store_plane<T, A>(a, outs, pbase, bv, bg != nullptr, g.vec_io); break;
      CONV_C4_CASE(ACT_RELU)
      CONV_C4_CASE(ACT_SILU)
      CONV_C4_CASE(ACT_SIGMOID)
      CONV_C4_CASE(ACT_TANH)
      CONV_C4_CASE(ACT_HARD_SWISH)
      CONV_C4_CASE(ACT_HARD_SIGMOID)
      CONV_C4_CASE(ACT_CLIP)
      CONV_C4_CASE(ACT_LEAKY_RELU)
#undef CONV_C4_CASE
      default: cols4_store_plane<T, ACT_IDENTITY>(a, outs, pbase, bv, bg != nullptr, g.vec_io);
    }
    __syncwarp();  // the staging area is free for the next plane
    n = n_next;
    co = co_next;
  }
  cp_async_wait<0>();
}

// ---- 16-bit depthwise planes on the tensor cores ---------------------------
// With Xp the zero-padded input plane (stride 1, dilation 1), output row oh of
// a depthwise plane is sum_u Xp[oh + u][:] . T_u, where T_u[j][ow] =
// w[u][j - ow] (zero outside 0 .. K-1): K products with band matrices.  The
// plane sits in shared memory with padded column j at staged column
// j + delta (delta = 0 or 1, so image column 0 starts on a 4-byte boundary).
// A block of 8 output columns 8nt .. 8nt+7 reads staged columns
// 8nt .. 8nt + 7 + K - 1 + delta < 8nt + 16, so each (kernel row u, block of
// 16 output rows mt, block of 8 output columns nt) is one
// mma.sync.m16n8k16 with float32 accumulation: A = staged rows
// 16mt + u .. 16mt + u + 15, columns 8nt .. 8nt + 15 (ldmatrix), and B_u[k][n]
// = w[u][k - n - delta], the same for every column block, held in registers
// per channel (two per kernel row).  Products of 16-bit values are exact in
// float32; the sums run in the MMA's float32 order.  Then bias, residual and
// activation in float32, one rounding.  One warp per plane at a time, planes
// in channel-major order (a warp's planes share their band matrices), the
// next plane staged by cp.async while this one is computed.
struct DwMmaGeo {
  int pitch;   // staged row length in elements: a multiple of 8 with pitch / 8 odd (conflict-free ldmatrix)
  int rows;    // staged rows: mtiles * 16 + K - 1
  int mtiles;  // blocks of 16 output rows
  int ntiles;  // blocks of 8 output columns computed: 1, 2, 4 or 8 (those past Wo are dropped)
  int delta;   // staged column of padded column j: j + delta
  int copy4;   // 4-byte cp.async copies of image rows (else element copies)
  int pair_out;  // two outputs per store (Wo even, y and the residual 4-byte aligned)
  long long warps;  // warps sharing the planes (contiguous runs in channel-major order)
};
constexpr int kDmWarps = 8;

template <typename T>
__device__ __forceinline__ uint32_t pack_t2(T lo, T hi) {
  return static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&lo)) |
         (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
}

template <typename T>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&aq)[4], uint32_t b0, uint32_t b1) {
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

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <typename T, int K, int NT>
__global__ void __launch_bounds__(kDmWarps * 32, NT >= 2 ? 2 : 3) depthwise_mma(const ConvArgs a, const DwMmaGeo g) {
  extern __shared__ __align__(16) unsigned char dsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bufsz = g.pitch * g.rows;  // elements of one staged plane
  T* buf0 = reinterpret_cast<T*>(dsm) + static_cast<size_t>(warp) * 2 * bufsz;
  {  // the border stays zero (two buffers: a whole number of 16-byte units, pitch a multiple of 8)
    uint4* z = reinterpret_cast<uint4*>(buf0);
    const int units16 = 2 * bufsz * static_cast<int>(sizeof(T)) / 16;
    for (int i = lane; i < units16; i += 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncwarp();
  const T* __restrict__ xg = static_cast<const T*>(a.x);
  const T* __restrict__ wg = static_cast<const T*>(a.wt);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  const T* __restrict__ rg = static_cast<const T*>(a.residual);
  T* __restrict__ y = static_cast<T*>(a.y);
  // this warp's planes: an even share of the planes in channel-major order
  const long long planes = static_cast<long long>(a.n) * a.c_out;
  const long long gw = static_cast<long long>(blockIdx.x) * kDmWarps + warp;
  const long long p_begin = gw * planes / g.warps;
  const long long p_end = (gw + 1) * planes / g.warps;
  if (gw >= g.warps || p_begin >= p_end) return;
  const int m = a.mg;  // channel multiplier: output channel co reads input channel co / m
  // staging: image row r lands at staged row pt + r, image column c at staged
  // column pl + delta + c
  const int rows_s = min(a.h, g.rows - a.pt);
  const int col0 = a.pl + g.delta;
  const int wq = a.w / 2;  // 4-byte copies per image row
  // with at most 32 copies per image row a lane's copies are one column pair
  // and rows r0, r0 + rpp, ...: constant shared and global strides
  const bool prog = g.copy4 && wq <= 32;
  const int rpp = prog ? 32 / wq : 1, r0 = prog ? lane / wq : 0, q0 = prog ? lane - (lane / wq) * wq : 0;
  const int ncp = prog && r0 < rpp && rows_s > r0 ? (rows_s - r0 + rpp - 1) / rpp : 0;
  const uint32_t dst_first = static_cast<uint32_t>(((a.pt + r0) * g.pitch + col0 + 2 * q0) * sizeof(T));
  const uint32_t dst_step = static_cast<uint32_t>(rpp * g.pitch * sizeof(T));
  const long long src_first = (static_cast<long long>(r0) * a.w + 2 * q0) * static_cast<long long>(sizeof(T));
  const long long src_step = static_cast<long long>(rpp) * a.w * static_cast<long long>(sizeof(T));
  auto stage = [&](int n, int co, T* buf) {
    const T* src = xg + (static_cast<long long>(n) * a.c_in + (m == 1 ? co : co / m)) * a.hw;
    if (prog) {
      cp_async_run<4>(static_cast<uint32_t>(__cvta_generic_to_shared(buf)) + dst_first,
                      reinterpret_cast<const char*>(src) + src_first, ncp, dst_step, src_step);
      return;
    }
    T* dst = buf + a.pt * g.pitch + col0;
    if (g.copy4) {
      {
        for (int r = 0; r < rows_s; ++r)
          for (int q = lane; q < wq; q += 32) cp_async_n<4>(dst + r * g.pitch + 2 * q, src + r * a.w + 2 * q);
      }
    } else {
      for (int r = 0; r < rows_s; ++r)
        for (int c = lane; c < a.w; c += 32) dst[r * g.pitch + c] = src[r * a.w + c];
    }
  };
  // band matrices of channel co: thread t holds B_u[k][n] for n = t / 4 and
  // k = 2(t % 4) + {0, 1} (bq[u][0]) and + 8 (bq[u][1])
  uint32_t bq[K][2];
  int bq_co = -1;
  auto build_b = [&](int co) {
    const T* wc = wg + static_cast<long long>(co) * K * K;
    const int nn = lane >> 2, k0 = 2 * (lane & 3);
#pragma unroll
    for (int u = 0; u < K; ++u) {
      T e[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = k0 + (i & 1) + (i >> 1) * 8;
        const int d = k - nn - g.delta;
        e[i] = (d >= 0 && d < K) ? wc[u * K + d] : from_f32<T>(0.0f);
      }
      bq[u][0] = pack_t2<T>(e[0], e[1]);
      bq[u][1] = pack_t2<T>(e[2], e[3]);
    }
    bq_co = co;
  };
  // plane pl = co * N + n
  int co = static_cast<int>(p_begin / a.n), n = static_cast<int>(p_begin - static_cast<long long>(co) * a.n);
  stage(n, co, buf0);
  cp_async_commit();
  // accumulator (t, q): output row 16 mt + lane / 4 (+ 8 for q >= 2), column
  // 8 t + 2 (lane % 4) + (q & 1)
  const int ow_l = 2 * (lane & 3);
  int k = 0;
  for (long long pl = p_begin; pl < p_end; ++pl, ++k) {
    T* buf = buf0 + (k & 1) * bufsz;
    int n_next = n + 1, co_next = co;
    if (n_next == a.n) { n_next = 0; ++co_next; }
    if (pl + 1 < p_end) stage(n_next, co_next, buf0 + ((k + 1) & 1) * bufsz);
    cp_async_commit();
    if (co != bq_co) build_b(co);
    cp_async_wait<1>();  // this plane's copies (the next plane's may still fly)
    __syncwarp();
    const float bv = bg ? to_f32(bg[co]) : 0.0f;
    const long long pbase = (static_cast<long long>(n) * a.c_out + co) * a.howo;
    // ldmatrix row address of this lane: staged row (lane & 15) of the block,
    // columns 8 (lane >> 4) ..
    const uint32_t lane_addr = static_cast<uint32_t>(__cvta_generic_to_shared(buf)) +
                               static_cast<uint32_t>(((lane & 15) * g.pitch + (lane >> 4) * 8) * sizeof(T));
    // two blocks of 16 rows at a time: 2 * NT independent accumulators
    for (int mt0 = 0; mt0 < g.mtiles; mt0 += 2) {
      const bool second = mt0 + 1 < g.mtiles;
      float acc[2][NT][4];
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[b][t][q] = 0.0f;
      // per kernel row: the fragment loads first, then the MMAs (the asm
      // statements keep their order, so this is the order they issue in)
#pragma unroll
      for (int u = 0; u < K; ++u) {
        const uint32_t rowa = lane_addr + static_cast<uint32_t>((mt0 * 16 + u) * g.pitch * sizeof(T));
        uint32_t aq[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) ldmatrix_x4(aq[t], rowa + static_cast<uint32_t>(t * 8 * sizeof(T)));
        if (second) {
          const uint32_t rowb = rowa + static_cast<uint32_t>(16 * g.pitch * sizeof(T));
          uint32_t aq2[NT][4];
#pragma unroll
          for (int t = 0; t < NT; ++t) ldmatrix_x4(aq2[t], rowb + static_cast<uint32_t>(t * 8 * sizeof(T)));
#pragma unroll
          for (int t = 0; t < NT; ++t) mma_16816<T>(acc[0][t], aq[t], bq[u][0], bq[u][1]);
#pragma unroll
          for (int t = 0; t < NT; ++t) mma_16816<T>(acc[1][t], aq2[t], bq[u][0], bq[u][1]);
        } else {
#pragma unroll
          for (int t = 0; t < NT; ++t) mma_16816<T>(acc[0][t], aq[t], bq[u][0], bq[u][1]);
        }
      }
      // the epilogue: bias, residual, activation over a block's outputs at
      // once (one dispatch), then the stores
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        if (b == 1 && !second) break;
        const int oh0 = (mt0 + b) * 16 + (lane >> 2);
        float* v = &acc[b][0][0];
        float bb[NT * 4], rr[NT * 4];
#pragma unroll
        for (int i = 0; i < NT * 4; ++i) { bb[i] = bv; rr[i] = 0.0f; }
        if (rg) {
#pragma unroll
          for (int i = 0; i < NT * 4; ++i) {
            const int oh = oh0 + 8 * ((i & 3) >> 1), ow = 8 * (i >> 2) + ow_l + (i & 1);
            if (oh < a.ho && ow < a.wo) rr[i] = to_f32(rg[pbase + static_cast<long long>(oh) * a.wo + ow]);
          }
        }
        epilogue_n<NT * 4>(*reinterpret_cast<float(*)[NT * 4]>(v), bb, rr, bg != nullptr, rg != nullptr, a.act,
                           a.alpha, a.beta);
        T* yrow = y + pbase + static_cast<long long>(oh0) * a.wo + ow_l;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (oh0 + 8 * h >= a.ho) continue;
          T* yr = yrow + 8 * h * a.wo;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int ow = 8 * t + ow_l;
            if (ow >= a.wo) continue;
            const float v0 = acc[b][t][2 * h], v1 = acc[b][t][2 * h + 1];
            if (g.pair_out) {  // Wo even: ow + 1 < Wo too
              *reinterpret_cast<uint32_t*>(yr + 8 * t) = pack_t2<T>(from_f32<T>(v0), from_f32<T>(v1));
            } else {
              yr[8 * t] = from_f32<T>(v0);
              if (ow + 1 < a.wo) yr[8 * t + 1] = from_f32<T>(v1);
            }
          }
        }
      }
    }
    __syncwarp();  // this buffer is read; it is refilled two planes on
    n = n_next;
    co = co_next;
  }
  cp_async_wait<0>();
}

template <typename T, int K, int NT>
cudaError_t launch_mma_nt(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  DwMmaGeo g;
  g.pitch = d.mma_pitch;
  g.rows = d.mma_rows;
  g.mtiles = (a.ho + 15) / 16;
  g.ntiles = NT;
  g.delta = a.pl & 1;
  g.copy4 = (a.w % 2 == 0) && (a.hw % 2 == 0) && reinterpret_cast<uintptr_t>(a.x) % 4 == 0;
  g.pair_out = (a.wo % 2 == 0) && reinterpret_cast<uintptr_t>(a.y) % 4 == 0 &&
               (!a.residual || reinterpret_cast<uintptr_t>(a.residual) % 4 == 0);
  const size_t smem = static_cast<size_t>(kDmWarps) * 2 * g.pitch * g.rows * sizeof(T);
  auto kern = depthwise_mma<T, K, NT>;
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDmWarps * 32, smem);
  if (err != cudaSuccess) return err;
  const long long planes = static_cast<long long>(a.n) * a.c_out;
  // every resident warp slot of the device, or one warp per plane
  const long long slots = static_cast<long long>(d.sm) * std::max(per_sm, 1);
  const long long blocks = std::min<long long>(slots, (planes + kDmWarps - 1) / kDmWarps);
  g.warps = std::min<long long>(planes, blocks * kDmWarps);
  kern<<<static_cast<unsigned>(blocks), kDmWarps * 32, smem, s>>>(a, g);
  return cudaGetLastError();
}

template <typename T, int K>
cudaError_t launch_mma_k(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  const int nt = (a.wo + 7) / 8;  // compiled for 1, 2, 4 or 8 column blocks (extra blocks are masked)
  if (nt <= 1) return launch_mma_nt<T, K, 1>(d, a, s);
  if (nt <= 2) return launch_mma_nt<T, K, 2>(d, a, s);
  if (nt <= 4) return launch_mma_nt<T, K, 4>(d, a, s);
  return launch_mma_nt<T, K, 8>(d, a, s);
}

template <typename T>
cudaError_t launch_mma(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  if constexpr (std::is_same<T, float>::value) {
    return cudaErrorInvalidValue;  // 16-bit operands only
  } else {
    if (a.kh == 3) return launch_mma_k<T, 3>(d, a, s);
    if (a.kh == 5) return launch_mma_k<T, 5>(d, a, s);
    if (a.kh == 7) return launch_mma_k<T, 7>(d, a, s);
    return cudaErrorInvalidValue;
  }
}

// Rows per lane the four-column kernel is compiled for.
constexpr int kCols4Rows[] = {2, 4, 7, 8};

template <typename T, int K, int R>
cudaError_t launch_cols4_r(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  Cols4Geo g;
  constexpr int es = static_cast<int>(sizeof(T));
  constexpr int NV = (K + 3 + 3) / 4 * 4;
  g.groups = (a.wo + 3) / 4;
  g.rblocks = 32 / g.groups;
  g.rows = g.rblocks * R + K - 1;
  // rows of whole 16-byte units: every row (and every warp's buffer) starts on
  // 16 bytes, as 16-byte copies and the vector reads need
  constexpr int unit = 16 / es;
  g.pitch = (std::max(a.pl + a.w, 4 * (g.groups - 1) + NV) + unit - 1) / unit * unit;
  // the widest copy that keeps every row start and the buffer column aligned
  g.copy = 0;
  for (int cb = 16; cb >= 4; cb /= 2) {
    if (reinterpret_cast<uintptr_t>(a.x) % cb == 0 && (static_cast<long long>(a.w) * es) % cb == 0 &&
        (a.hw * es) % cb == 0 && (a.pl * es) % cb == 0) {
      g.copy = cb;
      break;
    }
  }
  g.vec_io = reinterpret_cast<uintptr_t>(a.y) % 16 == 0 && (a.wo % 4) == 0 &&
             (!a.residual || reinterpret_cast<uintptr_t>(a.residual) % 16 == 0);
  g.out_stride = (a.ho * a.wo + 3) / 4 * 4;
  const size_t smem = static_cast<size_t>(kC4Warps) * (2 * g.pitch * g.rows * es + g.out_stride * 4);
  auto kern = depthwise_cols4<T, K, R>;
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  const long long planes = static_cast<long long>(a.n) * a.c_out;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kC4Warps * 32, smem);
  if (err != cudaSuccess) return err;
  const long long blocks = std::min<long long>((planes + kC4Warps - 1) / kC4Warps,
                                               static_cast<long long>(d.sm) * std::max(per_sm, 1));
  kern<<<static_cast<unsigned>(blocks), kC4Warps * 32, smem, s>>>(a, g);
  return cudaGetLastError();
}

template <typename T, int K>
cudaError_t launch_cols4(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  switch (d.cols4_r) {
    case 2: return launch_cols4_r<T, K, 2>(d, a, s);
    case 4: return launch_cols4_r<T, K, 4>(d, a, s);
    case 7: return launch_cols4_r<T, K, 7>(d, a, s);
    case 8: return launch_cols4_r<T, K, 8>(d, a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int K>
cudaError_t launch_narrow(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  NarrowGeo g;
  constexpr int es = static_cast<int>(sizeof(T));
  g.cofs = es == 4 ? a.pl : (a.pl + 1) / 2 * 2;
  g.pitch = (g.cofs - a.pl + a.wo + K - 1 + 1) / 2 * 2;
  g.rows = a.ho + K - 1;
  // 4-byte copies: x 4-byte aligned, every image row starting on 4 bytes
  g.async = reinterpret_cast<uintptr_t>(a.x) % 4 == 0 && (static_cast<long long>(a.w) * es) % 4 == 0 &&
            (a.hw * es) % 4 == 0;
  const size_t smem = static_cast<size_t>(kNwWarps) * 2 * g.pitch * g.rows * es;
  auto kern = depthwise_narrow<T, K>;
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  const long long planes = static_cast<long long>(a.n) * a.c_out;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kNwWarps * 32, smem);
  if (err != cudaSuccess) return err;
  const long long blocks = std::min<long long>((planes + kNwWarps - 1) / kNwWarps,
                                               static_cast<long long>(d.sm) * std::max(per_sm, 1));
  kern<<<static_cast<unsigned>(blocks), kNwWarps * 32, smem, s>>>(a, g);
  return cudaGetLastError();
}

template <typename T, int KH>
cudaError_t launch_kh(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  const int row_tiles = (a.ho + d.th - 1) / d.th;
  const long long items = static_cast<long long>(a.n) * a.groups * row_tiles;
  const long long blocks = std::min<long long>(items, static_cast<long long>(d.sm) * kBlocksPerSm);
  const size_t smem = depthwise_smem_bytes(d, a.mg, a.kh, a.kw, sizeof(T) == 4 ? CONV_F32 : CONV_F16);
  auto kern = depthwise<T, KH>;
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  kern<<<static_cast<unsigned>(blocks), kDwThreads, smem, s>>>(a, d, row_tiles, items);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const DwPlan& d, const ConvArgs& a, cudaStream_t s) {
  if (d.mma) return launch_mma<T>(d, a, s);
  if (d.cols4_r) {
    if (a.kh == 3) return launch_cols4<T, 3>(d, a, s);
    if (a.kh == 5) return launch_cols4<T, 5>(d, a, s);
    if (a.kh == 7) return launch_cols4<T, 7>(d, a, s);
  }
  if (d.narrow) {
    if (a.kh == 3) return launch_narrow<T, 3>(d, a, s);
    if (a.kh == 5) return launch_narrow<T, 5>(d, a, s);
    if (a.kh == 7) return launch_narrow<T, 7>(d, a, s);
  }
  if (a.sh == 1 && a.dh == 1) {
    if (a.kh == 3) return launch_kh<T, 3>(d, a, s);
    if (a.kh == 5) return launch_kh<T, 5>(d, a, s);
    if (a.kh == 7) return launch_kh<T, 7>(d, a, s);
  }
  return launch_kh<T, 0>(d, a, s);
}

}  // namespace

size_t depthwise_smem_bytes(const DwPlan& d, int mg, int kh, int kw, int dtype) {
  const size_t tile = static_cast<size_t>(d.in_rows) * d.row;
  const size_t es = dtype == CONV_F32 ? 4 : 2;
  return 2 * static_cast<size_t>((mg * kh * kw + 3) & ~3) * 4 + 2 * static_cast<size_t>((mg + 3) & ~3) * 4 +
         (es == 4 ? 0 : tile * 4) + 2 * tile * es;
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
