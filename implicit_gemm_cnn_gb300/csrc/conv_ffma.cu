// conv_ffma.cu -- implicit-GEMM convolution on CUDA cores (float32 FFMA), with
// an optional split of k into ranges and the ordered reduction that finishes it.
//
// The method ("Convolution, pooling and resize", Variants: the implicit GEMM
// tile kernel that gathers the input window while it loads the tile, and
// "Convolutions", section 2.4: Y = W cols per group).  Per group g the output
// is the product of W_g (Cout/G x K) and the column matrix (K x N*Ho*Wo), with
// K = Cin/G * kh * kw ordered (channel, kernel row, kernel column) as OIHW
// weights lie.  The column matrix is never written: each k row of a pixel tile
// is gathered from x while the tile is staged into shared memory, with a
// zero for every tap outside the image.  A block computes BM output channels
// x BN pixels (pixels of several images may share a tile: batch is part of the
// GEMM's N).  Bias, residual and activation are applied as the tile is stored,
// so y is written once.
//
// Split k ("Convolution, pooling and resize", RTX 4070 split k): when the grid
// is too small to fill the device, k is cut into ranges.  Normally the ranges
// of a tile are the blocks of one thread-block cluster: each keeps its raw
// float32 sums in its shared memory and, after a cluster barrier, every block
// adds a share of the tile's outputs over the ranges in range order (reading
// the other blocks' shared memory) and applies the epilogue.  Otherwise (more
// than 16 ranges, the 128 x 128 tile, or no such cluster fits) each range's
// block writes its sums into its own plane of scratch and split_reduce adds
// the planes in range order, then applies the epilogue.  Both give the same
// bits; no atomics: every output's sum has an order fixed by the shape.
//
// Pipeline: fp32 tiles arrive by cp.async (4-byte copies with zero fill for
// padded taps) kFfmaStages deep; 16-bit operands (the fallback for shapes the
// tensor-core kernel does not take) are converted to fp32 as they are staged.
// The window offsets of the block's k range are decoded once into a table in
// shared memory (offset in the input plane set, row and column displacement).
//
// Two special cases skip the per-k gather: a pointwise layer whose planes
// hold whole 4-pixel groups copies its B tile with 16-byte cp.async, and a
// grouped layer with few channels per group (grouped_direct) stages each
// group's input rows once per work item and reads every k term from them at
// the tap's offset.
#include <string.h>

#include <algorithm>

#include "conv_internal.h"

namespace conv {
namespace {

__device__ __forceinline__ void cp_async4(float* smem, const void* gmem, bool pred) {
  unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  int n = pred ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async16(float* smem, const void* gmem, bool pred) {
  unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <typename T>
__device__ __forceinline__ void stage_elem(float* dst, const T* src, bool ok) {
  if constexpr (sizeof(T) == 4) {
    cp_async4(dst, src, ok);
  } else {
    *dst = ok ? to_f32(*src) : 0.0f;
  }
}

// Store 4 consecutive outputs (same image, same channel) starting at out.
template <typename T>
__device__ __forceinline__ void store4(T* y, long long out, const float v[4]) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(y + out) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
    T h[4] = {from_f32<T>(v[0]), from_f32<T>(v[1]), from_f32<T>(v[2]), from_f32<T>(v[3])};
    *reinterpret_cast<uint2*>(y + out) = *reinterpret_cast<const uint2*>(h);
  }
}

__host__ __device__ constexpr int pow2_floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

// The B operand (BMODE):
//  * kBGather: each k row of a pixel tile is gathered from x with 4-byte
//    copies, a window-table lookup and bounds tests per element;
//  * kBPointwise: a pointwise layer (1x1, stride 1, no pad, plane length a
//    multiple of 4, x 16-byte aligned) whose k rows of 4 consecutive pixels are
//    16 contiguous bytes of one channel plane: 16-byte copies, each thread's
//    pixel offsets computed once, the table holding k * plane length;
//  * kBUnfolded: 16-byte copies from the column-unfolded copy xw of x (see
//    UnfPlan): a thread's pixel offsets are computed once, the table holds
//    each term's offset, no bounds tests; the weights come transposed (wtt), so
//    the A tile arrives by 16-byte copies too.
// TN = 12 (three 4-pixel groups per thread) is used with unfolded B only.
// The block index, read again where it is used (an asm volatile read cannot be
// merged with an earlier one): the tile decode below is recomputed for the
// epilogue instead of keeping its results in registers through the k loop.
__device__ __forceinline__ unsigned ctaid_x() {
  unsigned v;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(v));
  return v;
}
__device__ __forceinline__ unsigned ctaid_y() {
  unsigned v;
  asm volatile("mov.u32 %0, %%ctaid.y;" : "=r"(v));
  return v;
}

// Split k within a thread-block cluster: the blocks of one tile's k ranges
// form one cluster (cluster dims 1 x 1 x split, rank = k range) and read each
// other's shared memory.
constexpr int kMaxClusterK = 16;
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned v;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(v));
  return v;
}
// All threads of all blocks of the cluster: shared-memory writes before it are
// seen by reads after it from any block of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;\n" ::: "memory");
}
// The float at this block's shared address `saddr`, read from block `rank`'s
// shared memory.
__device__ __forceinline__ float ld_cluster_f32(unsigned saddr, unsigned rank) {
  unsigned r;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}

// A block's tile: a 3-D grid (pixel tile, group x channel tile, k range), or
// with a tail split a 1-D grid: tiles [0, tail_first) whole, then tail_split
// k ranges of each remaining tile (tile = pixel tile x tiles_gy + channel tile).
struct FfmaTile {
  long long px_tile;
  int gy;
  int part;            // tail k range (-1: not a tail block)
  long long tail_tile; // tile - tail_first for tail blocks
};
template <int BMODE>
__device__ __forceinline__ FfmaTile ffma_tile(const ConvArgs& a, unsigned bx, unsigned by) {
  FfmaTile r;
  r.part = -1;
  r.tail_tile = 0;
  if (BMODE == kBUnfolded && a.tail_split > 0) {
    long long t;
    if (bx < a.blk_whole_n) {
      t = a.blk_whole_lo + bx;
    } else {
      const long long u = (a.blk_tail_lo - a.tail_first) * a.tail_split + (bx - a.blk_whole_n);
      t = a.tail_first + u / a.tail_split;
      r.part = static_cast<int>(u % a.tail_split);
      r.tail_tile = t - a.tail_first;
    }
    r.px_tile = t / a.tiles_gy;
    r.gy = static_cast<int>(t % a.tiles_gy);
  } else {
    r.px_tile = a.px_tile0 + bx;
    r.gy = static_cast<int>(by);
  }
  return r;
}

// Registers per thread for a block of nt threads: two blocks per SM from 192
// threads on, three from 128 (multiples of 8, the allocation unit).
__host__ __device__ constexpr int ffma_maxreg(int nt) {
  return nt >= 192 ? (65536 / (2 * nt)) / 8 * 8 : (nt >= 128 ? (65536 / (3 * nt)) / 8 * 8 : 255);
}

template <typename T, int BM, int BN, int TM, int TN, int BMODE>
__global__ void __launch_bounds__((BM / TM) * (BN / TN)) __maxnreg__(ffma_maxreg((BM / TM) * (BN / TN)))
    igemm_ffma(const ConvArgs a, const int ktab_cap) {
  constexpr int NT = (BM / TM) * (BN / TN);
  constexpr int BK = BMODE == kBUnfolded ? kFfmaBKU : kFfmaBK;
  constexpr int S = kFfmaStages;
  constexpr int AS = BM + 4;  // padded weight-tile row: conflict-free transposed stores
  constexpr bool VEC = BMODE != kBGather;
  constexpr int GN = BN * 4 / TN;  // distance between a thread's 4-pixel groups
  static_assert(TM == 4 || TM == 8, "TM");
  static_assert(TN == 4 || TN == 8 || TN == 12, "TN");
  static_assert(BN % TN == 0 && (BN / TN) * 4 * (TN / 4) == BN, "pixel groups");
  extern __shared__ __align__(16) float smem[];
  float* As = smem;                                       // [S][BK][AS]
  float* Bs = As + S * BK * AS;                           // [S][BK][BN]
  int2* ktab = reinterpret_cast<int2*>(Bs + S * BK * BN);  // [ktab_cap]

  const T* __restrict__ x = static_cast<const T*>(a.x);
  const T* __restrict__ wt = static_cast<const T*>(a.wt);
  const int tid = threadIdx.x;
  // ---- the block's tile and k range ------------------------------------------
  int k_begin, k_end;
  long long pix0;
  int g, m0;
  const int co_tiles = (a.mg + BM - 1) / BM;
  {
    const FfmaTile t = ffma_tile<BMODE>(a, blockIdx.x, blockIdx.y);
    if (BMODE == kBUnfolded && a.tail_split > 0) {
      k_begin = t.part < 0 ? 0 : t.part * a.tail_len;
      k_end = t.part < 0 ? a.K : min(a.K, k_begin + a.tail_len);
    } else {
      k_begin = blockIdx.z * a.k_per_split;
      k_end = min(a.K, k_begin + a.k_per_split);
    }
    pix0 = t.px_tile * BN;
    g = t.gy / co_tiles;
    m0 = (t.gy % co_tiles) * BM;
  }
  const int khw = a.kh * a.kw;

  // ---- the pixel columns this thread stages (gathered B) -------------------
  // LB threads gather the input tile: RSTEP rows at a time of BN pixels each
  // (LB >= BN), or PCOLS pixel columns each over all BK rows (LB < BN).
  constexpr int LB = NT >= BN ? pow2_floor(NT / BN < BK ? NT / BN : BK) * BN : pow2_floor(NT);
  constexpr int PCOLS = VEC ? 1 : (LB >= BN ? 1 : BN / LB);
  constexpr int RSTEP = LB >= BN ? LB / BN : 1;
  constexpr int BROWS = BK / RSTEP;
  static_assert(VEC || (BK % RSTEP == 0 && (LB >= BN ? LB % BN == 0 : BN % LB == 0)), "loader mapping");
  const bool bloader = tid < LB;
  const int r0 = LB >= BN ? tid / BN : 0;
  const int cbase = LB >= BN ? tid % BN : tid;
  long long pbase[PCOLS];
  int ih0[PCOLS], iw0[PCOLS];
  bool pval[PCOLS];
  if constexpr (!VEC) {
#pragma unroll
    for (int j = 0; j < PCOLS; ++j) {
      const int col = cbase + j * LB;
      const long long p = pix0 + col;
      pval[j] = bloader && p < a.npix;
      const long long pp = pval[j] ? p : 0;
      const int n = static_cast<int>(pp / a.howo);
      const int rem = static_cast<int>(pp - static_cast<long long>(n) * a.howo);
      const int oh = rem / a.wo, ow = rem - (rem / a.wo) * a.wo;
      ih0[j] = oh * a.sh - a.pt;
      iw0[j] = ow * a.sw - a.pl;
      pbase[j] = (static_cast<long long>(n) * a.c_in + static_cast<long long>(g) * a.cg) * a.hw +
                 static_cast<long long>(ih0[j]) * a.w + iw0[j];
    }
  }

  // vector B: the thread's 16-byte copies of a stage: q = tid + i*NT -> k row
  // q / (BN/4), pixels pix0 + 4*(q % (BN/4)) .. +3, all in one image row (the
  // plane length, or the output row, is a multiple of 4)
  constexpr int QV = VEC ? (BK * BN / 4 + NT - 1) / NT : 1;
  // when the block's threads cover whole k rows (NT a multiple of BN/4) and
  // every copy is used, a thread's copies share its 4 pixels: one pixel
  // offset and one validity flag serve all of them
  constexpr bool VSAME = VEC && NT % (BN / 4) == 0 && (BK * BN / 4) % NT == 0;
  constexpr int QVS = VSAME ? 1 : QV;
  long long vbase[BMODE == kBPointwise ? QVS : 1];
  int uoff[BMODE == kBUnfolded ? QVS : 1];  // unfolded: 32-bit element offsets into xw
  bool vok[QVS];
  if constexpr (VEC) {
    const long long unf_img = static_cast<long long>(a.c_in) * a.kw * a.hu * a.wo;  // xw per image
#pragma unroll
    for (int i = 0; i < QVS; ++i) {
      const int q = tid + i * NT;
      const long long p = pix0 + 4 * (q % (BN / 4));
      vok[i] = q < BK * BN / 4 && p < a.npix && (BMODE != kBUnfolded || (p >= a.pix_lo && p < a.pix_hi));
      const long long pp = vok[i] ? p : (BMODE == kBUnfolded ? a.pix_lo : 0);
      const long long n = pp / a.howo;
      const long long rem = pp - n * a.howo;
      if constexpr (BMODE == kBPointwise) {
        vbase[i] = (n * a.c_in + static_cast<long long>(g) * a.cg) * a.hw + rem;
      } else {
        const long long oh = rem / a.wo, ow = rem - oh * a.wo;
        uoff[i] = static_cast<int>((n - a.img0) * unf_img + static_cast<long long>(g) * a.cg * a.kw * a.hu * a.wo +
                                   oh * a.sh * a.wo + ow);
      }
    }
  }
  // unfolded A: 16-byte copies of the transposed weights.  Unfolded copies
  // address xw and wtt with 32-bit element offsets (both hold fewer than 2^31
  // elements): the pixel part of each B copy (uoff) and the group's first
  // weight of the block's channel tile (aoff) are fixed for the whole k loop.
  constexpr int QA = BMODE == kBUnfolded ? (BK * BM / 4 + NT - 1) / NT : 1;
  constexpr bool ASAME = NT % (BM / 4) == 0;  // a thread's copies share their 4 channels
  constexpr int QAS = ASAME ? 1 : QA;
  const int aoff = BMODE == kBUnfolded ? g * a.K * a.mg4 + m0 : 0;
  bool aok[QAS];  // unfolded A: the copy's four channels are real (else zeros)
#pragma unroll
  for (int i = 0; i < QAS; ++i) aok[i] = m0 + 4 * ((tid + i * NT) % (BM / 4)) < a.mg4;

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

  const int tx = tid % (BN / TN);
  const int ty = tid / (BN / TN);

  for (int kseg = k_begin; kseg < k_end; kseg += ktab_cap) {
    const int seg_end = min(k_end, kseg + ktab_cap);
    __syncthreads();  // the previous segment's table and stages are free
    for (int k = kseg + tid; k < seg_end; k += NT) {
      const int c = k / khw;
      const int tap = k - c * khw;
      const int u = tap / a.kw, v = tap - (tap / a.kw) * a.kw;
      const int dy = u * a.dh, dx = v * a.dw;
      if constexpr (BMODE == kBGather)
        ktab[k - kseg] = make_int2(c * static_cast<int>(a.hw) + dy * a.w + dx, (dy << 16) | dx);
      else if constexpr (BMODE == kBPointwise)
        ktab[k - kseg] = make_int2(k * static_cast<int>(a.hw), 0);
      else
        ktab[k - kseg] = make_int2(((c * a.kw + v) * a.hu + dy) * a.wo, 0);
    }
    __syncthreads();

    auto load_stage = [&](int st, int k0) {
      float* as = As + st * BK * AS;
      float* bs = Bs + st * BK * BN;
      if constexpr (BMODE == kBUnfolded) {
#pragma unroll
        for (int i = 0; i < QA; ++i) {
          const int q = tid + i * NT;
          const int kk = q / (BM / 4), m4 = q % (BM / 4);
          const int k = k0 + kk;
          const bool ok = k < seg_end && aok[ASAME ? 0 : i];
          const float* src = a.wtt + (ok ? aoff + k * a.mg4 + 4 * m4 : 0);
          if ((BK * BM / 4) % NT == 0 || q < BK * BM / 4) cp_async16(as + kk * AS + 4 * m4, src, ok);
        }
      } else {
        constexpr int AE = (BM * BK + NT - 1) / NT;
#pragma unroll
        for (int i = 0; i < AE; ++i) {
          const int e = tid + i * NT;
          if (e < BM * BK) {
            const int kk = e % BK, m = e / BK;
            const int k = k0 + kk;
            const bool ok = (m0 + m < a.mg) && (k < seg_end);
            const T* src = ok ? wt + static_cast<long long>(g * a.mg + m0 + m) * a.K + k : wt;
            stage_elem<T>(as + kk * AS + m, src, ok);
          }
        }
      }
      if constexpr (BMODE == kBUnfolded) {
#pragma unroll
        for (int i = 0; i < QV; ++i) {
          const int q = tid + i * NT;
          const int kk = q / (BN / 4), c4 = q % (BN / 4);
          const int k = k0 + kk;
          const bool ok = vok[VSAME ? 0 : i] && k < seg_end;
          const float* src = a.xw + (ok ? uoff[VSAME ? 0 : i] + ktab[k - kseg].x : 0);
          if ((BK * BN / 4) % NT == 0 || q < BK * BN / 4) cp_async16(bs + kk * BN + 4 * c4, src, ok);
        }
      } else if constexpr (BMODE == kBPointwise) {
        const float* xb = reinterpret_cast<const float*>(x);
#pragma unroll
        for (int i = 0; i < QV; ++i) {
          const int q = tid + i * NT;
          const int kk = q / (BN / 4), c4 = q % (BN / 4);
          const int k = k0 + kk;
          const bool ok = vok[VSAME ? 0 : i] && k < seg_end;
          const float* src = ok ? xb + vbase[VSAME ? 0 : i] + ktab[k - kseg].x : xb;
          if (q < BK * BN / 4) cp_async16(bs + kk * BN + 4 * c4, src, ok);
        }
      } else if (bloader) {
#pragma unroll
        for (int i = 0; i < BROWS; ++i) {
          const int kk = r0 + i * RSTEP;
          const int k = k0 + kk;
          const bool kok = k < seg_end;
          const int2 e = kok ? ktab[k - kseg] : make_int2(0, 0);
          const int dy = e.y >> 16, dx = e.y & 0xffff;
#pragma unroll
          for (int j = 0; j < PCOLS; ++j) {
            const int col = cbase + j * LB;
            const int ih = ih0[j] + dy, iw = iw0[j] + dx;
            const bool ok = kok && pval[j] && static_cast<unsigned>(ih) < static_cast<unsigned>(a.h) &&
                            static_cast<unsigned>(iw) < static_cast<unsigned>(a.w);
            const T* src = ok ? x + pbase[j] + e.x : x;
            stage_elem<T>(bs + kk * BN + col, src, ok);
          }
        }
      }
    };

    const int nch = (seg_end - kseg + BK - 1) / BK;
#pragma unroll
    for (int st = 0; st < S - 1; ++st) {
      if (st < nch) load_stage(st, kseg + st * BK);
      cp_async_commit();
    }
    for (int c = 0; c < nch; ++c) {
      cp_async_wait<S - 2>();
      __syncthreads();
      const int nxt = c + S - 1;
      if (nxt < nch) load_stage(nxt % S, kseg + nxt * BK);
      cp_async_commit();
      const float* as = As + (c % S) * BK * AS;
      const float* bs = Bs + (c % S) * BK * BN;
#pragma unroll 8
      for (int kk = 0; kk < BK; ++kk) {
        float ra[TM], rb[TN];
        const float4 a0 = *reinterpret_cast<const float4*>(as + kk * AS + ty * 4);
        ra[0] = a0.x; ra[1] = a0.y; ra[2] = a0.z; ra[3] = a0.w;
        if constexpr (TM == 8) {
          const float4 a1 = *reinterpret_cast<const float4*>(as + kk * AS + BM / 2 + ty * 4);
          ra[4] = a1.x; ra[5] = a1.y; ra[6] = a1.z; ra[7] = a1.w;
        }
#pragma unroll
        for (int jg = 0; jg < TN / 4; ++jg) {
          const float4 b = *reinterpret_cast<const float4*>(bs + kk * BN + jg * GN + tx * 4);
          rb[jg * 4] = b.x; rb[jg * 4 + 1] = b.y; rb[jg * 4 + 2] = b.z; rb[jg * 4 + 3] = b.w;
        }
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(ra[i], rb[j], acc[i][j]);
      }
    }
    cp_async_wait<0>();
  }

  // ---- store: a raw tail range, raw partial planes (split k), or the fused
  // epilogue ----------------------------------------------------------------
  const FfmaTile te = ffma_tile<BMODE>(a, ctaid_x(), ctaid_y());
  pix0 = te.px_tile * BN;
  g = te.gy / co_tiles;
  m0 = (te.gy % co_tiles) * BM;
  if (te.part >= 0) {
    float* tb = a.tailbuf + (te.tail_tile * a.tail_split + te.part) * static_cast<long long>(BM * BN);
#pragma unroll
    for (int jg = 0; jg < TN / 4; ++jg)
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const int ml = i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4);
        *reinterpret_cast<float4*>(tb + ml * BN + jg * GN + tx * 4) =
            make_float4(acc[i][jg * 4], acc[i][jg * 4 + 1], acc[i][jg * 4 + 2], acc[i][jg * 4 + 3]);
      }
    return;
  }
  if constexpr (BM * BN == 128 * 128) {
    // the 128 x 128 tiles (128 registers a thread) keep the epilogue per run
    // of 4 pixels: the two-pass form below cost the unfolded kernel 6 % (664
    // against 627 us) and made the gathered one spill
    // only pixels in [pix_lo, pix_hi) (the whole batch, or a chunk of images)
    // are stored; split planes hold the chunk's outputs from image img0 on
    const long long out0 = static_cast<long long>(a.img0) * a.c_out * a.howo;
    T* y = static_cast<T*>(a.y);
  #pragma unroll
    for (int jg = 0; jg < TN / 4; ++jg) {
      const long long p = pix0 + jg * GN + tx * 4;
      if (p >= a.pix_hi || p + 3 < a.pix_lo) continue;
      const int n = static_cast<int>(p / a.howo);
      const long long rem = p - static_cast<long long>(n) * a.howo;
      const bool whole4 = a.vec_out && p >= a.pix_lo && (p + 3 < a.pix_hi) && (rem + 3 < a.howo) && ((a.howo & 3) == 0);
      // output offset (image, position) of pixel p + q, stepped from p's
      // without a division: the 4 pixels may cross image boundaries
      long long oo[4];
      int on[4];
  #pragma unroll
      for (int q = 0; q < 4; ++q) {
        long long o = rem + q;
        int nq = n;
        while (o >= a.howo) { o -= a.howo; ++nq; }
        oo[q] = o;
        on[q] = nq;
      }
  #pragma unroll
      for (int i = 0; i < TM; ++i) {
        const int m = m0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
        if (m >= a.mg) continue;
        const int co = g * a.mg + m;
        const long long out = (static_cast<long long>(n) * a.c_out + co) * a.howo + rem;
        if (a.split > 1 || a.raw_out) {
          float* part = a.partial + static_cast<long long>(blockIdx.z) * a.part_total;  // chunk-local
          if (whole4) {
            *reinterpret_cast<float4*>(part + (out - out0)) =
                make_float4(acc[i][jg * 4], acc[i][jg * 4 + 1], acc[i][jg * 4 + 2], acc[i][jg * 4 + 3]);
          } else {
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const long long pq = p + q;
              if (pq < a.pix_lo || pq >= a.pix_hi) continue;
              part[(static_cast<long long>(on[q]) * a.c_out + co) * a.howo + oo[q] - out0] = acc[i][jg * 4 + q];
            }
          }
        } else {
          // the epilogue on this run of 4 pixels of one channel
          const T* __restrict__ resp = static_cast<const T*>(a.residual);
          const float bco = a.bias ? to_f32(static_cast<const T*>(a.bias)[co]) : 0.0f;
          float v[4], bv[4], rv[4];
          long long oq[4];
          bool in[4];
  #pragma unroll
          for (int q = 0; q < 4; ++q) {
            const long long pq = p + q;
            in[q] = pq >= a.pix_lo && pq < a.pix_hi;
            oq[q] = whole4 ? out + q : (static_cast<long long>(on[q]) * a.c_out + co) * a.howo + oo[q];
            v[q] = acc[i][jg * 4 + q];
            bv[q] = bco;
            rv[q] = (resp && in[q]) ? to_f32(resp[oq[q]]) : 0.0f;
          }
          epilogue_n<4>(v, bv, rv, a.bias != nullptr, resp != nullptr, a.act, a.alpha, a.beta);
          if (whole4) {
            store4<T>(y, out, v);
          } else {
  #pragma unroll
            for (int q = 0; q < 4; ++q)
              if (in[q]) y[oq[q]] = from_f32<T>(v[q]);
          }
        }
      }
    }
    return;
  } else {
    if (a.cluster_k) {
      // split k within the cluster: each k range's block writes its raw sums
      // to its own shared memory; after the cluster barrier, rank r finishes
      // a 1/split share of the tile: per output the ranges' sums added in rank
      // (= k) order, then the fused epilogue and one store -- the additions
      // and roundings of the planes + split_reduce path, bit for bit.
      __syncthreads();  // every warp is past its last reads of the stages
#pragma unroll
      for (int jg = 0; jg < TN / 4; ++jg)
#pragma unroll
        for (int i = 0; i < TM; ++i) {
          const int ml = i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4);
          *reinterpret_cast<float4*>(smem + ml * BN + jg * GN + tx * 4) =
              make_float4(acc[i][jg * 4], acc[i][jg * 4 + 1], acc[i][jg * 4 + 2], acc[i][jg * 4 + 3]);
        }
      cluster_sync();
      const int rank = static_cast<int>(cluster_rank());
      const int per = (BM * BN + a.split - 1) / a.split;
      const int e_end = min(BM * BN, (rank + 1) * per);
      const unsigned sbase = static_cast<unsigned>(__cvta_generic_to_shared(smem));
      const T* __restrict__ resp = static_cast<const T*>(a.residual);
      const T* __restrict__ biasp = static_cast<const T*>(a.bias);
      T* __restrict__ yo = static_cast<T*>(a.y);
      for (int e = rank * per + tid; e < e_end; e += NT) {
        const int ml = e / BN, col = e - (e / BN) * BN;
        const int m = m0 + ml;
        const long long p = pix0 + col;
        if (m >= a.mg || p < a.pix_lo || p >= a.pix_hi) continue;
        const unsigned addr = sbase + static_cast<unsigned>(e) * 4u;
        float t[kMaxClusterK];
#pragma unroll
        for (int z = 0; z < kMaxClusterK; ++z)
          if (z < a.split) t[z] = ld_cluster_f32(addr, static_cast<unsigned>(z));
        float v[1] = {t[0]};
#pragma unroll
        for (int z = 1; z < kMaxClusterK; ++z)
          if (z < a.split) v[0] = __fadd_rn(v[0], t[z]);
        const int n = static_cast<int>(p / a.howo);
        const long long rem = p - static_cast<long long>(n) * a.howo;
        const int co = g * a.mg + m;
        const long long out = (static_cast<long long>(n) * a.c_out + co) * a.howo + rem;
        float bv[1] = {biasp ? to_f32(biasp[co]) : 0.0f};
        float rv[1] = {resp ? to_f32(resp[out]) : 0.0f};
        epilogue_n<1>(v, bv, rv, biasp != nullptr, resp != nullptr, a.act, a.alpha, a.beta);
        yo[out] = from_f32<T>(v[0]);
      }
      cluster_sync();  // no block leaves while another still reads its tile
      return;
    }
    // only pixels in [pix_lo, pix_hi) (the whole batch, or a chunk of images)
    // are stored; split planes hold the chunk's outputs from image img0 on
    const long long out0 = static_cast<long long>(a.img0) * a.c_out * a.howo;
    T* y = static_cast<T*>(a.y);
    const bool raw = a.split > 1 || a.raw_out;
    // pixel group jg: its first pixel, image and position, and the (image,
    // position) of each of its 4 pixels, stepped without a division (the 4
    // pixels may cross image boundaries)
    auto group = [&](int jg, long long& p, int& n, long long& rem, long long (&oo)[4], int (&on)[4]) {
      p = pix0 + jg * GN + tx * 4;
      n = static_cast<int>(p / a.howo);
      rem = p - static_cast<long long>(n) * a.howo;
  #pragma unroll
      for (int q = 0; q < 4; ++q) {
        long long o = rem + q;
        int nq = n;
        while (o >= a.howo) { o -= a.howo; ++nq; }
        oo[q] = o;
        on[q] = nq;
      }
    };
    if (!raw) {
      // the fused epilogue in float32: bias and residual per value, then the
      // activation over all of the thread's values in one dispatch (a dispatch
      // per 4 values is if-converted into evaluating every activation)
      const T* __restrict__ resp = static_cast<const T*>(a.residual);
      const T* __restrict__ biasp = static_cast<const T*>(a.bias);
      if (biasp || resp) {
  #pragma unroll
        for (int jg = 0; jg < TN / 4; ++jg) {
          long long p, rem, oo[4];
          int n, on[4];
          group(jg, p, n, rem, oo, on);
          if (p >= a.pix_hi || p + 3 < a.pix_lo) continue;
  #pragma unroll
          for (int i = 0; i < TM; ++i) {
            const int m = m0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
            if (m >= a.mg) continue;
            const int co = g * a.mg + m;
            const float bco = biasp ? to_f32(biasp[co]) : 0.0f;
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              float& v = acc[i][jg * 4 + q];
              if (biasp) v = __fadd_rn(v, bco);
              const long long pq = p + q;
              if (resp && pq >= a.pix_lo && pq < a.pix_hi)
                v = __fadd_rn(v, to_f32(resp[(static_cast<long long>(on[q]) * a.c_out + co) * a.howo + oo[q]]));
            }
          }
        }
      }
      activate_n<TM * TN>(*reinterpret_cast<float(*)[TM * TN]>(&acc[0][0]), a.act, a.alpha, a.beta);
    }
  #pragma unroll
    for (int jg = 0; jg < TN / 4; ++jg) {
      long long p, rem, oo[4];
      int n, on[4];
      group(jg, p, n, rem, oo, on);
      if (p >= a.pix_hi || p + 3 < a.pix_lo) continue;
      const bool whole4 = a.vec_out && p >= a.pix_lo && (p + 3 < a.pix_hi) && (rem + 3 < a.howo) && ((a.howo & 3) == 0);
  #pragma unroll
      for (int i = 0; i < TM; ++i) {
        const int m = m0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
        if (m >= a.mg) continue;
        const int co = g * a.mg + m;
        const long long out = (static_cast<long long>(n) * a.c_out + co) * a.howo + rem;
        if (raw) {
          float* part = a.partial + static_cast<long long>(blockIdx.z) * a.part_total;  // chunk-local
          if (whole4) {
            *reinterpret_cast<float4*>(part + (out - out0)) =
                make_float4(acc[i][jg * 4], acc[i][jg * 4 + 1], acc[i][jg * 4 + 2], acc[i][jg * 4 + 3]);
          } else {
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const long long pq = p + q;
              if (pq < a.pix_lo || pq >= a.pix_hi) continue;
              part[(static_cast<long long>(on[q]) * a.c_out + co) * a.howo + oo[q] - out0] = acc[i][jg * 4 + q];
            }
          }
        } else if (whole4) {
          float v[4] = {acc[i][jg * 4], acc[i][jg * 4 + 1], acc[i][jg * 4 + 2], acc[i][jg * 4 + 3]};
          store4<T>(y, out, v);
        } else {
  #pragma unroll
          for (int q = 0; q < 4; ++q) {
            const long long pq = p + q;
            if (pq >= a.pix_lo && pq < a.pix_hi)
              y[(static_cast<long long>(on[q]) * a.c_out + co) * a.howo + oo[q]] = from_f32<T>(acc[i][jg * 4 + q]);
          }
        }
      }
    }
  }
}

// The unfolded-B pre-pass.  Blocks [0, planes) unfold one input plane (n, c)
// each into xw[n][c][v][r][ow] (float32, 16-byte stores, zeros outside x),
// reading the plane once, coalesced, into shared memory when it fits
// (`staged`); the blocks after them transpose the weights into wtt[g][k][m]
// (float32, channels padded to mg4 with zeros) through 32 x 32 tiles.
template <typename T>
__global__ void __launch_bounds__(256) ffma_unfold(const ConvArgs a, long long planes, int wt_tiles_k,
                                                   int wt_tiles_m, int staged) {
  __shared__ float tile[32][33];
  extern __shared__ float plane_s[];  // the input plane when staged
  const T* __restrict__ x = static_cast<const T*>(a.x);
  const T* __restrict__ w = static_cast<const T*>(a.wt);
  const int tid = threadIdx.x;
  if (blockIdx.x < planes) {
    const long long nc = blockIdx.x;  // the chunk's planes, from image img0 on
    const T* __restrict__ plane = x + (static_cast<long long>(a.img0) * a.c_in + nc) * a.hw;
    const int hw = static_cast<int>(a.hw);
    if (staged) {
      for (int e = tid; e < hw; e += 256) plane_s[e] = to_f32(plane[e]);
      __syncthreads();
    }
    const int wq = a.wo / 4;
    float* out = a.xw + nc * static_cast<long long>(a.kw) * a.hu * a.wo;
    // thread = one 4-column group of `rows_per_pass` rows at a time; the
    // output rows (v, r) are walked without divisions
    const int tpr = min(wq, 256);
    const int rows_per_pass = 256 / tpr;
    const int r0 = tid / tpr;
    if (r0 >= rows_per_pass) return;
    for (int ow4 = tid - r0 * tpr; ow4 < wq; ow4 += tpr) {
      for (int v = 0; v < a.kw; ++v) {
        const int col0 = ow4 * 4 * a.sw - a.pl + v * a.dw;
        float* ov = out + static_cast<long long>(v) * a.hu * a.wo + 4 * ow4;
        for (int r = r0; r < a.hu; r += rows_per_pass) {
          const int ih = r - a.pt;
          const bool rok = static_cast<unsigned>(ih) < static_cast<unsigned>(a.h);
          const int row = (rok ? ih : 0) * a.w;
          float o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int iw = col0 + j * a.sw;
            const bool ok = rok && static_cast<unsigned>(iw) < static_cast<unsigned>(a.w);
            o[j] = ok ? (staged ? plane_s[row + iw] : to_f32(plane[row + iw])) : 0.0f;
          }
          *reinterpret_cast<float4*>(ov + static_cast<long long>(r) * a.wo) = make_float4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    return;
  }
  // weights: tile (g, k block, m block) of 32 x 32
  const long long b = blockIdx.x - planes;
  const int mb = static_cast<int>(b % wt_tiles_m);
  const long long rest = b / wt_tiles_m;
  const int kb = static_cast<int>(rest % wt_tiles_k);
  const int g = static_cast<int>(rest / wt_tiles_k);
  const int tx = tid % 32, ty = tid / 32;  // 8 rows of 32
  for (int i = ty; i < 32; i += 8) {       // read along k (OIHW rows are contiguous in k)
    const int m = mb * 32 + i, k = kb * 32 + tx;
    tile[i][tx] = (m < a.mg && k < a.K) ? to_f32(w[(static_cast<long long>(g) * a.mg + m) * a.K + k]) : 0.0f;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {       // write along m
    const int k = kb * 32 + i, m = mb * 32 + tx;
    if (k < a.K && m < a.mg4) a.wtt[(static_cast<long long>(g) * a.K + k) * a.mg4 + m] = tile[tx][i];
  }
}

// The tail of a tail-split launch: for every tile of the last round, the
// float32 sums of its tail_split k ranges added in range order, then the fused
// epilogue, four pixels of one channel at a time (the output width is a
// multiple of 4, so four consecutive tile pixels share an image row).
template <typename T, int BM, int BN>
__global__ void __launch_bounds__(256) ffma_tail_reduce(const ConvArgs a) {
  constexpr int Q = BN / 4;
  const long long units = a.tail_tiles * BM * Q;
  const int co_tiles = (a.mg + BM - 1) / BM;
  T* y = static_cast<T*>(a.y);
  const T* __restrict__ bp = static_cast<const T*>(a.bias);
  const T* __restrict__ rp = static_cast<const T*>(a.residual);
  for (long long u = blockIdx.x * 256LL + threadIdx.x; u < units; u += static_cast<long long>(gridDim.x) * 256) {
    const long long tt = u / (BM * Q);
    const int rem = static_cast<int>(u - tt * (BM * Q));
    const int ml = rem / Q, c4 = rem - (rem / Q) * Q;
    const long long t = a.tail_first + tt;
    const long long px_tile = t / a.tiles_gy;
    const int gy = static_cast<int>(t % a.tiles_gy);
    const int g = gy / co_tiles;
    const int m = (gy % co_tiles) * BM + ml;
    const long long p = px_tile * BN + 4 * c4;
    if (m >= a.mg || p < a.pix_lo || p >= a.pix_hi) continue;
    const float* src = a.tailbuf + tt * a.tail_split * static_cast<long long>(BM * BN) + ml * BN + 4 * c4;
    float4 sum = *reinterpret_cast<const float4*>(src);
    for (int r = 1; r < a.tail_split; ++r) {
      const float4 t4 = *reinterpret_cast<const float4*>(src + r * static_cast<long long>(BM * BN));
      sum.x = __fadd_rn(sum.x, t4.x); sum.y = __fadd_rn(sum.y, t4.y);
      sum.z = __fadd_rn(sum.z, t4.z); sum.w = __fadd_rn(sum.w, t4.w);
    }
    const int co = g * a.mg + m;
    const long long n = p / a.howo;
    const long long out = (n * a.c_out + co) * a.howo + (p - n * a.howo);
    float v[4] = {sum.x, sum.y, sum.z, sum.w}, bv[4], rv[4];
    const float bco = bp ? to_f32(bp[co]) : 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      bv[q] = bco;
      rv[q] = rp ? to_f32(rp[out + q]) : 0.0f;
    }
    epilogue_n<4>(v, bv, rv, bp != nullptr, rp != nullptr, a.act, a.alpha, a.beta);
    if (a.vec_out) {
      store4<T>(y, out, v);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) y[out + q] = from_f32<T>(v[q]);
    }
  }
}

// Sum the split planes in range order, then the fused epilogue.  Four
// consecutive outputs per thread when the plane length allows vector loads.
template <typename T, int ACT>
__global__ void __launch_bounds__(256) split_reduce(const ConvArgs a) {
  // the planes hold the outputs of images [img0, img0 + chunk): part_total
  // elements each, output out0 + i at element i
  const long long total = a.part_total;
  const long long out0 = static_cast<long long>(a.img0) * a.c_out * a.howo;
  T* y = static_cast<T*>(a.y) + out0;
  const T* __restrict__ rbase = a.residual ? static_cast<const T*>(a.residual) + out0 : nullptr;
  const float* part = a.partial;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  if ((total & 3) == 0 && (out0 & 3) == 0) {
    const long long q = total >> 2;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < q; i += stride) {
      const float4* p4 = reinterpret_cast<const float4*>(part) + i;
      const long long zs = q;  // float4s per plane
      float4 s = p4[0];
      int z = 1;
      // four planes' loads in flight at a time; the adds stay in range order
      for (; z + 3 < a.split; z += 4) {
        float4 t[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) t[j] = p4[(z + j) * zs];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s.x = __fadd_rn(s.x, t[j].x); s.y = __fadd_rn(s.y, t[j].y);
          s.z = __fadd_rn(s.z, t[j].z); s.w = __fadd_rn(s.w, t[j].w);
        }
      }
      for (; z < a.split; ++z) {
        const float4 t = p4[z * zs];
        s.x = __fadd_rn(s.x, t.x); s.y = __fadd_rn(s.y, t.y);
        s.z = __fadd_rn(s.z, t.z); s.w = __fadd_rn(s.w, t.w);
      }
      const long long o = i * 4;
      const T* __restrict__ bp = static_cast<const T*>(a.bias);
      const T* __restrict__ rp = rbase;
      float v[4] = {s.x, s.y, s.z, s.w}, bv[4], rv[4];
      // the channel of output out0 + o, then stepped (4 outputs may cross planes)
      const long long plane = (out0 + o) / a.howo;
      long long pos = out0 + o - plane * a.howo;
      int ck = static_cast<int>(plane % a.c_out);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (k > 0 && ++pos >= a.howo) {
          pos = 0;
          if (++ck == a.c_out) ck = 0;
        }
        bv[k] = bp ? to_f32(bp[ck]) : 0.0f;
        rv[k] = rp ? to_f32(rp[o + k]) : 0.0f;
      }
      epilogue_t<ACT, 4>(v, bv, rv, bp != nullptr, rp != nullptr, a.alpha, a.beta);
      if (a.vec_out) {
        store4<T>(y, o, v);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) y[o + k] = from_f32<T>(v[k]);
      }
    }
  } else {
    const T* __restrict__ bp = static_cast<const T*>(a.bias);
    const T* __restrict__ rp = rbase;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total; i += stride) {
      float v[1] = {part[i]};
      for (int z = 1; z < a.split; ++z) v[0] = __fadd_rn(v[0], part[z * total + i]);
      const int co = static_cast<int>(((out0 + i) / a.howo) % a.c_out);
      float bv[1] = {bp ? to_f32(bp[co]) : 0.0f}, rv[1] = {rp ? to_f32(rp[i]) : 0.0f};
      epilogue_t<ACT, 1>(v, bv, rv, bp != nullptr, rp != nullptr, a.alpha, a.beta);
      y[i] = from_f32<T>(v[0]);
    }
  }
}

// ---- grouped layers, input rows staged once per item ------------------------
// The implicit GEMM of one group (M = Cout/groups, K = (Cin/groups)*k*k,
// N = pixels) with its B operand read in place: item = (group, image, kGdRows
// output rows); the group's input rows (zero rows above and below the image,
// zero columns left and right, written once) and its weights, transposed to
// [channel][tap][output channel], arrive in shared memory by cp.async, the
// next item's while this one is computed.  A thread holds 8 output channels
// x 4 pixels of one row, Wo/4 columns apart; each k term (channel c, tap u, v)
// is 4 staged inputs at the tap's offset, two broadcast float4 weight loads and 32
// FMAs, k in (c, u, v) order into one float32 chain per output, then the fused
// epilogue.
template <int K, int ACT>
__global__ void __launch_bounds__(kGdThreads, 3) grouped_direct(const ConvArgs a, const GdPlan g) {
  extern __shared__ __align__(16) float gsm[];
  const int tid = threadIdx.x;
  const int xs_floats = a.cg * g.rows_in * g.pitch;
  const int buf_floats = xs_floats + a.cg * K * K * a.mg;
  for (int i = tid; i < 2 * buf_floats; i += kGdThreads) gsm[i] = 0.0f;  // borders stay zero
  __syncthreads();
  const float* __restrict__ x = static_cast<const float*>(a.x);
  const float* __restrict__ wt = static_cast<const float*>(a.wt);
  const float* __restrict__ bias = static_cast<const float*>(a.bias);
  const float* __restrict__ res = static_cast<const float*>(a.residual);
  float* __restrict__ y = static_cast<float*>(a.y);
  const bool vec16 = (a.w & 3) == 0 && (a.hw & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  const int q_per_row = vec16 ? a.w / 4 : a.w;  // copies per staged row
  const int taps = K * K;
  auto decode = [&](long long item, int* n, int* gi, int* oh0) {
    const int rt = static_cast<int>(item % g.row_tiles);
    const long long rest = item / g.row_tiles;
    *n = static_cast<int>(rest % a.n);
    *gi = static_cast<int>(rest / a.n);
    *oh0 = rt * kGdRows;
  };
  auto stage = [&](long long item, float* buf) {
    int n, gi, oh0;
    decode(item, &n, &gi, &oh0);
    const float* xg = x + (static_cast<long long>(n) * a.c_in + static_cast<long long>(gi) * a.cg) * a.hw;
    const int copies = a.cg * g.rows_in * q_per_row;
    for (int e = tid; e < copies; e += kGdThreads) {
      const int c = e / (g.rows_in * q_per_row);
      const int rem = e - c * (g.rows_in * q_per_row);
      const int rr = rem / q_per_row, qq = rem - (rem / q_per_row) * q_per_row;
      const int ih = oh0 - a.pt + rr;
      const bool ok = static_cast<unsigned>(ih) < static_cast<unsigned>(a.h);  // else zeros
      float* dst = buf + (c * g.rows_in + rr) * g.pitch + g.cofs + (vec16 ? 4 * qq : qq);
      const float* src = ok ? xg + static_cast<long long>(c) * a.hw + static_cast<long long>(ih) * a.w +
                                  (vec16 ? 4 * qq : qq)
                            : x;
      if (vec16) cp_async16(dst, src, ok);
      else cp_async4(dst, src, ok);
    }
    // weights of the group: OIHW rows (contiguous over channel and tap) into
    // [channel * taps + tap][output channel]
    float* ws = buf + xs_floats;
    const int ck = a.cg * taps;
    const float* wg = wt + static_cast<long long>(gi) * a.mg * ck;
    for (int e = tid; e < a.mg * ck; e += kGdThreads) {
      const int m = e / ck, r = e - (e / ck) * ck;
      cp_async4(ws + r * a.mg + m, wg + e, true);
    }
  };
  const long long first = blockIdx.x, step = gridDim.x;
  if (first < g.items) stage(first, gsm);
  cp_async_commit();
  const int groups4 = a.wo / 4, halves = a.mg / 8;
  const int units = kGdRows * groups4 * halves;
  int k = 0;
  for (long long item = first; item < g.items; item += step, ++k) {
    float* buf = gsm + (k & 1) * buf_floats;
    if (item + step < g.items) stage(item + step, gsm + ((k + 1) & 1) * buf_floats);
    cp_async_commit();
    cp_async_wait<1>();  // this item's copies (the next item's may still fly)
    __syncthreads();
    int n, gi, oh0;
    decode(item, &n, &gi, &oh0);
    const float* xs = buf;
    const float* ws = buf + xs_floats;
    for (int u_ = tid; u_ < units; u_ += kGdThreads) {
      // a thread's 4 pixels are columns cb, cb + Wo/4, cb + 2 Wo/4, cb + 3 Wo/4
      // of its row: consecutive threads take consecutive cb, so each of the 4
      // staged-input reads of a tap (and each store) is consecutive across them
      const int h8 = u_ % halves, pg = u_ / halves;
      const int r = pg / groups4, cb = pg - (pg / groups4) * groups4;
      if (oh0 + r >= a.ho) continue;
      float acc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = 0.0f;
      const float* xb = xs + r * g.pitch + g.cofs - a.pl + cb;
      const float* wb = ws + 8 * h8;
      for (int c = 0; c < a.cg; ++c) {
        const float* xc = xb + c * g.rows_in * g.pitch;
        const float* wc = wb + c * taps * a.mg;
#pragma unroll
        for (int u = 0; u < K; ++u)
#pragma unroll
          for (int v = 0; v < K; ++v) {
            const float* xp = xc + u * a.dh * g.pitch + v * a.dw;
            const float xv[4] = {xp[0], xp[groups4], xp[2 * groups4], xp[3 * groups4]};
            const float4 w0 = *reinterpret_cast<const float4*>(wc + (u * K + v) * a.mg);
            const float4 w1 = *reinterpret_cast<const float4*>(wc + (u * K + v) * a.mg + 4);
            const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[j][q] = fmaf(wv[j], xv[q], acc[j][q]);
          }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int co = gi * a.mg + 8 * h8 + j;
        const long long out = (static_cast<long long>(n) * a.c_out + co) * a.howo +
                              static_cast<long long>(oh0 + r) * a.wo + cb;
        const float b = bias ? bias[co] : 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float t = acc[j][q];
          if (bias) t = __fadd_rn(t, b);
          if (res) t = __fadd_rn(t, res[out + q * groups4]);
          y[out + q * groups4] = act_fn<ACT>(t, a.alpha, a.beta);
        }
      }
    }
    __syncthreads();  // this buffer is refilled two items from now
  }
  cp_async_wait<0>();
}

template <int K>
cudaError_t launch_gd_k(const Plan& plan, const ConvArgs& a, cudaStream_t s) {
  auto kern = grouped_direct<K, ACT_IDENTITY>;
  switch (a.act) {
#define CONV_GD_CASE(A)             \
  case A:                           \
    kern = grouped_direct<K, A>;    \
    break;
    CONV_GD_CASE(ACT_RELU)
    CONV_GD_CASE(ACT_SILU)
    CONV_GD_CASE(ACT_SIGMOID)
    CONV_GD_CASE(ACT_TANH)
    CONV_GD_CASE(ACT_HARD_SWISH)
    CONV_GD_CASE(ACT_HARD_SIGMOID)
    CONV_GD_CASE(ACT_CLIP)
    CONV_GD_CASE(ACT_LEAKY_RELU)
#undef CONV_GD_CASE
    default:
      break;
  }
  const GdPlan& g = plan.gd;
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), g.smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0, dev = 0, sms = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGdThreads, g.smem);
  if (err != cudaSuccess) return err;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const long long blocks = std::min<long long>(g.items, static_cast<long long>(sms) * std::max(per_sm, 1));
  kern<<<static_cast<unsigned>(blocks), kGdThreads, g.smem, s>>>(a, g);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_reduce_typed(const ConvArgs& a, cudaStream_t s);

template <typename T, int CFG, int BMODE>
cudaError_t launch_cfg_vb(const Plan& plan, const ConvArgs& args, cudaStream_t s) {
  constexpr FfmaCfg c = kFfmaCfgs[CFG];
  auto kern = igemm_ffma<T, c.bm, c.bn, c.tm, c.tn, BMODE>;
  ConvArgs a = args;
  const int ktab_cap = ffma_ktab_entries(a.k_per_split);
  const size_t smem = ffma_smem_bytes(CFG, a.k_per_split, BMODE == kBUnfolded);
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  // the tiles that hold pixels of [pix_lo, pix_hi)
  const int co_tiles = (a.mg + c.bm - 1) / c.bm;
  const long long px_lo = a.pix_lo / c.bn, px_hi = (a.pix_hi + c.bn - 1) / c.bn;
  const long long gx = px_hi - px_lo;
  a.px_tile0 = px_lo;
  if constexpr (BMODE == kBUnfolded) {
    if (a.tail_split > 0) {
      // tiles are pixel-tile major: the chunk's tiles are [t_lo, t_hi); whole
      // tiles below tail_first, the rest as tail_split blocks each
      const long long gyn = static_cast<long long>(a.tiles_gy);
      const long long t_lo = px_lo * gyn, t_hi = px_hi * gyn;
      a.blk_whole_lo = t_lo;
      a.blk_whole_n = std::max(0LL, std::min(t_hi, a.tail_first) - t_lo);
      const long long tail_lo = std::max(t_lo, a.tail_first);
      const long long tail_n = std::max(0LL, t_hi - tail_lo);
      a.blk_tail_lo = tail_lo;
      const long long blocks = a.blk_whole_n + tail_n * a.tail_split;
      if (blocks < 1 || blocks > 2147483647LL) return cudaErrorInvalidConfiguration;
      kern<<<static_cast<unsigned>(blocks), c.threads(), smem, s>>>(a, ktab_cap);
      err = cudaGetLastError();
      if (err != cudaSuccess) return err;
      if (tail_n == 0) return cudaSuccess;
      const long long units = a.tail_tiles * c.bm * (c.bn / 4);
      const long long rblocks = std::min<long long>((units + 255) / 256, 65535LL * 8);
      ffma_tail_reduce<T, c.bm, c.bn><<<static_cast<unsigned>(rblocks), 256, 0, s>>>(a);
      return cudaGetLastError();
    }
  }
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(co_tiles * a.groups),
            static_cast<unsigned>(a.split));
  if (a.cluster_k) {
    // the k ranges of a tile as one cluster; its shared memory also holds the
    // block's BM x BN float32 sums
    const size_t csmem = std::max(smem, static_cast<size_t>(c.bm) * c.bn * sizeof(float));
    const void* fn = reinterpret_cast<const void*>(kern);
    err = opt_in_smem(fn, csmem);
    if (err != cudaSuccess) return err;
    if (c.bm * c.bn != 128 * 128 && a.split >= 2 && a.split <= kMaxClusterK &&
        cluster_fits(fn, a.split, c.threads(), csmem)) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = grid;
      cfg.blockDim = dim3(static_cast<unsigned>(c.threads()), 1, 1);
      cfg.dynamicSmemBytes = csmem;
      cfg.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = static_cast<unsigned>(a.split);
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, kern, static_cast<const ConvArgs&>(a), ktab_cap);
    }
    // no such cluster fits this device: the planes and the reduction kernel
    a.cluster_k = 0;
    kern<<<grid, c.threads(), smem, s>>>(a, ktab_cap);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_reduce_typed<T>(a, s);
  }
  kern<<<grid, c.threads(), smem, s>>>(a, ktab_cap);
  (void)plan;
  return cudaGetLastError();
}

template <typename T, int CFG>
cudaError_t launch_cfg(const Plan& plan, const ConvArgs& a, cudaStream_t s) {
  if (a.xw) return launch_cfg_vb<T, CFG, kBUnfolded>(plan, a, s);
  if constexpr (sizeof(T) == 4) {
    if (plan.ffma_vec && reinterpret_cast<uintptr_t>(a.x) % 16 == 0)
      return launch_cfg_vb<T, CFG, kBPointwise>(plan, a, s);
  }
  return launch_cfg_vb<T, CFG, kBGather>(plan, a, s);
}

constexpr long long kUnfoldStageMax = 11000;  // plane elements staged in shared memory (with the
                                              // 4.2 KB transpose tile, under 48 KB)

template <typename T>
cudaError_t launch_unfold(const UnfPlan& u, const ConvArgs& a, cudaStream_t s) {
  const long long planes = (a.pix_hi - a.pix_lo) / a.howo * a.c_in;  // the chunk's images
  const int tk = (a.K + 31) / 32, tm = (u.mg4 + 31) / 32;
  const long long blocks = planes + static_cast<long long>(a.groups) * tk * tm;
  if (blocks > 2147483647LL) return cudaErrorInvalidConfiguration;
  const int staged = a.hw <= kUnfoldStageMax ? 1 : 0;
  const size_t smem = staged ? static_cast<size_t>(a.hw) * sizeof(float) : 0;
  ffma_unfold<T><<<static_cast<unsigned>(blocks), 256, smem, s>>>(a, planes, tk, tm, staged);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const Plan& plan, const ConvArgs& a, cudaStream_t s) {
  switch (plan.ffma_cfg) {
    case 0: return launch_cfg<T, 0>(plan, a, s);
    case 1: return launch_cfg<T, 1>(plan, a, s);
    case 2: return launch_cfg<T, 2>(plan, a, s);
    case 3: return launch_cfg<T, 3>(plan, a, s);
    case 4: return launch_cfg<T, 4>(plan, a, s);
    case 5: return launch_cfg<T, 5>(plan, a, s);
    case 6: return launch_cfg<T, 6>(plan, a, s);
    case 7: return launch_cfg<T, 7>(plan, a, s);
    case 8: return launch_cfg<T, 8>(plan, a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_reduce_typed(const ConvArgs& a, cudaStream_t s) {
  const long long total = a.part_total;
  const long long work = (total & 3) == 0 ? total / 4 : total;
  // small reductions in 64-thread blocks, so that they spread over more SMs
  const int threads = work < 152LL * 256 ? 64 : 256;
  long long blocks = (work + threads - 1) / threads;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  switch (a.act) {  // the activation compiled in: one code path per kernel
#define CONV_SR_CASE(A) \
  case A: split_reduce<T, A><<<static_cast<unsigned>(blocks), threads, 0, s>>>(a); break;
    CONV_SR_CASE(ACT_RELU)
    CONV_SR_CASE(ACT_SILU)
    CONV_SR_CASE(ACT_SIGMOID)
    CONV_SR_CASE(ACT_TANH)
    CONV_SR_CASE(ACT_HARD_SWISH)
    CONV_SR_CASE(ACT_HARD_SIGMOID)
    CONV_SR_CASE(ACT_CLIP)
    CONV_SR_CASE(ACT_LEAKY_RELU)
#undef CONV_SR_CASE
    default: split_reduce<T, ACT_IDENTITY><<<static_cast<unsigned>(blocks), threads, 0, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

int ffma_ktab_entries(int k_per_block) {
  return k_per_block < kFfmaKTab ? (k_per_block + 7) / 8 * 8 : kFfmaKTab;
}

size_t ffma_smem_bytes(int cfg, int k_per_block, bool unfolded) {
  const FfmaCfg c = kFfmaCfgs[cfg];
  return static_cast<size_t>(kFfmaStages) * (unfolded ? kFfmaBKU : kFfmaBK) * (c.bm + 4 + c.bn) * sizeof(float) +
         static_cast<size_t>(ffma_ktab_entries(k_per_block)) * sizeof(int2);
}

int ffma_launch_count(const Plan& plan) {
  if (plan.gd.ok) return 1;
  int n = 1;
  if (plan.ffma_unf) n += 1 + (plan.unf.tail_split > 0 ? 1 : 0);
  if (plan.info.split_k > 1 && !plan.cluster_k) n += 1;
  return n;
}

bool unf_plan(const conv_problem* p, long long ho, long long wo, UnfPlan* u) {
  memset(u, 0, sizeof(*u));
  if (wo % 4 != 0) return false;  // 4-pixel groups within one output row
  const long long hu = (ho - 1) * p->stride_h + (p->kh - 1) * p->dil_h + 1;
  const long long cg = p->c_in / p->groups, mg = p->c_out / p->groups;
  const long long per_group = cg * p->kw * hu * wo;  // the largest term offset (int32)
  if (hu > 2147483647LL || per_group > 2147483647LL) return false;
  u->hu = static_cast<int>(hu);
  u->mg4 = static_cast<int>((mg + 3) / 4 * 4);
  u->xw_elems = p->n * p->c_in * p->kw * hu * wo;
  u->wt_elems = p->groups * cg * p->kh * p->kw * u->mg4;
  // the kernel addresses both with 32-bit element offsets
  if (u->xw_elems >= 2147483647LL || u->wt_elems >= 2147483647LL) return false;
  return true;
}

bool gd_plan(const conv_problem* p, long long ho, long long wo, GdPlan* g) {
  memset(g, 0, sizeof(*g));
  if (p->dtype != CONV_F32 || p->groups < 2 || p->stride_h != 1 || p->stride_w != 1) return false;
  if (p->kh != p->kw || (p->kh != 3 && p->kh != 5) || wo % 4 != 0) return false;
  const long long cg = p->c_in / p->groups, mg = p->c_out / p->groups;
  if (mg % 8 != 0 || mg > 64 || cg > 64) return false;
  g->k = static_cast<int>(p->kh);
  g->rows_in = static_cast<int>(kGdRows + (p->kh - 1) * p->dil_h);
  g->cofs = static_cast<int>((p->pad_left + 3) / 4 * 4);
  const long long reach = g->cofs - p->pad_left + wo + (p->kw - 1) * p->dil_w;  // columns a tap reads
  const long long pitch = std::max<long long>(reach, g->cofs + p->w);
  g->pitch = static_cast<int>((pitch + 3) / 4 * 4);
  g->row_tiles = static_cast<int>((ho + kGdRows - 1) / kGdRows);
  g->items = p->n * p->groups * g->row_tiles;
  const long long buf = cg * g->rows_in * g->pitch + cg * p->kh * p->kw * mg;
  g->smem = static_cast<size_t>(2 * buf * 4);
  if (g->smem > 100 * 1024) return false;  // at least two blocks per SM
  g->ok = 1;
  return true;
}

cudaError_t launch_ffma(const Plan& plan, const ConvArgs& a, int dtype, cudaStream_t s) {
  // grouped layers with staged input rows (any alignment of y and the residual;
  // x rows are copied 16 bytes at a time when x allows it)
  if (plan.gd.ok && dtype == CONV_F32)
    return plan.gd.k == 3 ? launch_gd_k<3>(plan, a, s) : launch_gd_k<5>(plan, a, s);
  if (a.xw) {
    cudaError_t err = cudaErrorInvalidValue;
    switch (dtype) {
      case CONV_F32: err = launch_unfold<float>(plan.unf, a, s); break;
      case CONV_F16: err = launch_unfold<__half>(plan.unf, a, s); break;
      case CONV_BF16: err = launch_unfold<__nv_bfloat16>(plan.unf, a, s); break;
      default: break;
    }
    if (err != cudaSuccess) return err;
  }
  switch (dtype) {
    case CONV_F32: return launch_typed<float>(plan, a, s);
    case CONV_F16: return launch_typed<__half>(plan, a, s);
    case CONV_BF16: return launch_typed<__nv_bfloat16>(plan, a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_split_reduce(const ConvArgs& a, int dtype, cudaStream_t s) {
  switch (dtype) {
    case CONV_F32: return launch_reduce_typed<float>(a, s);
    case CONV_F16: return launch_reduce_typed<__half>(a, s);
    case CONV_BF16: return launch_reduce_typed<__nv_bfloat16>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace conv
