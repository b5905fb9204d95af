// conv_tc.cu -- implicit-GEMM convolution on the tcgen05 tensor cores
// (half / bfloat16 operands, float32 accumulation in tensor memory).
//
// The method is the implicit GEMM of "Convolution, pooling and resize",
// Variants (a tile kernel that gathers the input window while it stages the
// tile: no column matrix; bias, residual and activation applied as the result
// is stored, so the output is written once) and "Convolutions en compute",
// implicit im2col (the GEMM computes the window indices inside its tile-load
// loop).  Per group g:  Y_g^T (pixels x Cout/G) = cols_g^T (pixels x K) .
// W_g^T (K x Cout/G), K = Cin/G * kh * kw.
//
// Tiles and roles (one persistent block per SM, 13 warps):
//   * a tile is 128 consecutive output pixels of one image (MMA M = 128) x BN
//     output channels (MMA N); its float32 accumulator lives in tensor memory,
//     double buffered so the epilogue of one tile overlaps the next;
//   * warps 4-11 gather the A operand into 128-byte-swizzled K-major stages
//     that tcgen05.mma reads directly, 16 bytes (8 k values) per store, zero
//     for taps outside the image.  Three k orders: (tap, channel) with units
//     of 8 channels when the channels per group are a multiple of 8 -- one
//     window test per unit, as "Convolution, pooling and resize" (Apple M2,
//     taps innermost) orders its staging; (channel, kernel row, 8 taps) for
//     rows of 5..8 taps at dilation 1 -- one row test and five 4-byte loads
//     plus byte permutes per unit, taps past the kernel width or the image
//     masked per pixel; (channel, tap) otherwise.  Window offsets come from a
//     table decoded once per block;
//   * warps 0-3 first copy the block's weight rows into shared memory (one
//     bulk copy of the OIHW rows, then a permutation into the swizzled K-major
//     layout in the same k order -- the weight re-layout that "Convolution,
//     pooling and resize" measured at 1.27x on 3x3 layers, done on chip), then
//     run the epilogue: tcgen05.ld of the accumulator (thread = pixel), bias,
//     residual, activation in float32, one rounding to the element type.  The
//     tile is staged in shared memory as one 256-byte row per channel and
//     written with bulk copies (each row is contiguous in NCHW y); the
//     residual tile arrives the same way ahead of its use.  Shapes or
//     addresses that do not allow that (Ho*Wo not a multiple of 8, unaligned
//     y) store from registers instead;
//   * warp 12 allocates tensor memory and one lane issues the MMAs
//     (kind::f16, M=128, N=BN, K=16 per instruction) and the commits that
//     release stages and accumulators.
// Every mbarrier wait is bounded: after kWaitNs the waiting thread flags the
// block and the device error word, every role drains out, outstanding copies
// and MMAs are waited for (bounded again) and tensor memory is freed before
// exit.
#include <algorithm>
#include <type_traits>

#include "conv_internal.h"
#include "tc_ptx.cuh"

namespace conv {

__device__ uint32_t g_tc_error;  // nonzero once a bounded wait gave up

namespace {

constexpr int kM = 128;              // pixels per tile (MMA M)
constexpr int kBK = 64;              // k terms per stage: one 128-byte swizzle row
constexpr int kStageBytes = kM * kBK * 2;
constexpr int kEpiWarps = 4;         // warps 0-3 (tensor-memory lanes 32w .. 32w+31)
constexpr int kProdWarps = 8;        // warps 4-11
constexpr int kMmaWarp = 12;
constexpr int kThreads = 13 * 32;
constexpr int kProd = kProdWarps * 32;

using namespace tcx;

// The bounded wait of tc_ptx.cuh, reporting into this kernel's error word.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t code,
                                           bool ignore_abort = false) {
  return tcx::wait_phase(&g_tc_error, bar, parity, abort_flag, code, ignore_abort);
}

// Byte offset of the 16-byte unit j (k = 8j .. 8j+7) of row r in a 128-byte
// swizzled K-major tile: 8-row groups of 1024 bytes, unit index XOR row%8.
__device__ __forceinline__ uint32_t swz(int r, int j) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

__device__ __forceinline__ void epi_sync() {  // the four epilogue warps only
  asm volatile("bar.sync 1, %0;\n" ::"n"(kEpiWarps * 32) : "memory");
}

// Launch-time choices that depend on the operands' addresses.
struct TcLaunch {
  int mode;             // kModeCh8 / kModeRow8 / kModeNat
  int k_pad;
  int stages;
  int epi_bulk;         // stage the tile in shared memory, bulk-copy rows in/out
  int nio;              // staging buffers (1 or 2)
  int bulk_w;           // weights arrive by one bulk copy
  long long stg_bytes;  // bytes of that copy
  int halo_bufs;        // input halo buffers in shared memory (0: gather from global)
  int halo_slot;        // elements per input channel in a halo buffer (a multiple of 8)
  int halo_cg;          // input channels per group (channels per halo buffer)
};

struct TcLayout {
  uint32_t b_off, a_off, sio_off, halo_off, tab_off, bias_off, bar_off, slot_off, end;
};

__host__ __device__ inline int tc_ntab(int mode, int k_pad) {
  return mode == kModeNat ? k_pad : k_pad / 8;
}

__host__ __device__ inline TcLayout tc_layout(int bn, const TcLaunch& c) {
  TcLayout L;
  L.b_off = 0;
  L.a_off = static_cast<uint32_t>(c.k_pad / kBK) * bn * 128;  // multiple of 1024
  L.sio_off = L.a_off + static_cast<uint32_t>(c.stages) * kStageBytes;
  // the weight staging copy is dead once the weights are laid out: the
  // epilogue's tile buffers reuse its space
  const long long stg = c.bulk_w ? (c.stg_bytes + 127) / 128 * 128 : 0;
  const long long io = c.epi_bulk ? static_cast<long long>(c.nio) * bn * kM * 2 : 0;
  const long long halo = static_cast<long long>(c.halo_bufs) * c.halo_cg * c.halo_slot * 2;
  L.halo_off = L.sio_off + static_cast<uint32_t>((io + 127) / 128 * 128);  // after the tile buffers
  const long long r1 = (io + 127) / 128 * 128 + halo;
  L.tab_off = L.sio_off + static_cast<uint32_t>(stg > r1 ? stg : r1);
  L.bias_off = L.tab_off + static_cast<uint32_t>(tc_ntab(c.mode, c.k_pad)) * 16;
  L.bar_off = L.bias_off + static_cast<uint32_t>(bn) * 4;
  L.slot_off = L.bar_off + static_cast<uint32_t>(2 * c.stages + 13) * 8;
  L.end = L.slot_off + 16;
  return L;
}

template <typename T, int BN>
__global__ void __launch_bounds__(kThreads, 1) igemm_tc(const ConvArgs a, const TcPlan p, const TcLaunch c) {
  extern __shared__ uint8_t tsm_raw[];
  // 1024-byte alignment for the swizzled tiles (the launch adds 1 KB of slack)
  uint8_t* tsm = tsm_raw + ((1024 - (smem_u32(tsm_raw) & 1023)) & 1023);
  const int S = c.stages;
  const TcLayout L = tc_layout(BN, c);
  uint8_t* sB = tsm + L.b_off;
  uint8_t* sA = tsm + L.a_off;
  uint8_t* sio = tsm + L.sio_off;
  const uint16_t* stg = reinterpret_cast<const uint16_t*>(sio);
  int4* tab = reinterpret_cast<int4*>(tsm + L.tab_off);
  float* sbias = reinterpret_cast<float*>(tsm + L.bias_off);
  const uint32_t bar0 = smem_u32(tsm + L.bar_off);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t stg_bar = bar0 + 8u * (2 * S + 5);
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 6);
  auto res_bar = [&](int i) { return bar0 + 8u * (2 * S + 7 + i); };
  auto hfull_bar = [&](int i) { return bar0 + 8u * (2 * S + 9 + i); };   // halo buffer filled
  auto hempty_bar = [&](int i) { return bar0 + 8u * (2 * S + 11 + i); };  // halo buffer consumed
  volatile int* halo_a0 = reinterpret_cast<volatile int*>(tsm + L.slot_off + 8);  // [2] first element copied
  uint16_t* halo = reinterpret_cast<uint16_t*>(tsm + L.halo_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tsm + L.slot_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tsm + L.slot_off + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int kchunks = c.k_pad / kBK;
  const int khw = a.kh * a.kw;
  constexpr uint32_t kCols = BN * 2 <= 32 ? 32 : (BN * 2 <= 64 ? 64 : (BN * 2 <= 128 ? 128 : (BN * 2 <= 256 ? 256 : 512)));

  // ---- set-up: barriers, window table, tensor memory ------------------------
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), kProd);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps * 32);
      mbar_init(res_bar(b), 1);
      mbar_init(hfull_bar(b), 1);
      mbar_init(hempty_bar(b), kProd);
    }
    mbar_init(stg_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  // window table: per 8-value unit (ch8: 8 channels of one tap; row8: 8 taps
  // of one kernel row of one channel) or per value (nat)
  const int ntab = tc_ntab(c.mode, c.k_pad);
  for (int e = tid; e < ntab; e += kThreads) {
    int coff, dy, dx, ok;
    if (c.mode == kModeRow8) {
      const int ch = e / a.kh, u = e - (e / a.kh) * a.kh;
      dy = u * a.dh;
      dx = 0;
      coff = ch * (c.halo_bufs ? c.halo_slot : static_cast<int>(a.hw)) + dy * a.w;
      ok = ch < a.cg;
    } else {
      const int k = c.mode == kModeCh8 ? e * 8 : e;
      int tap, ch;
      if (c.mode == kModeCh8) { tap = k / a.cg; ch = k - tap * a.cg; }
      else { ch = k / khw; tap = k - ch * khw; }
      const int u = tap / a.kw, v = tap - (tap / a.kw) * a.kw;
      dy = u * a.dh;
      dx = v * a.dw;
      coff = ch * (c.halo_bufs ? c.halo_slot : static_cast<int>(a.hw)) + dy * a.w + dx;
      ok = k < a.K;
    }
    tab[e] = make_int4(coff, dy, dx, ok);
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // ---- this block's tiles: one (group, channel tile), strided pixel tiles.
  // A pixel tile is 128 consecutive output pixels of one image.
  const int combos = a.groups * p.co_tiles;
  const int cpc = gridDim.x / combos;  // blocks per combination
  const int combo = blockIdx.x / cpc;
  const int local = blockIdx.x - combo * cpc;
  const int g = combo / p.co_tiles;
  const int co0 = (combo - g * p.co_tiles) * BN;
  const int ntiles = local < p.pix_tiles ? (p.pix_tiles - local + cpc - 1) / cpc : 0;
  const int rows_valid = min(BN, a.mg - co0);
  const uint16_t* __restrict__ xs = static_cast<const uint16_t*>(a.x);
  const uint16_t* __restrict__ ws = static_cast<const uint16_t*>(a.wt);
  auto tile_origin = [&](int t, int* n, int* p0) {
    const int pt = local + t * cpc;
    *n = pt / p.tiles_per_img;
    *p0 = (pt - *n * p.tiles_per_img) * kM;
  };

  // ---- the block's weight rows: one bulk copy of the OIHW rows, then every
  // thread lays them out as swizzled K-major tiles in the block's k order,
  // four 16-byte units at a time with their loads issued first
  {
    const long long wrow0 = static_cast<long long>(g) * a.mg + co0;  // first OIHW row
    bool okw = true;
    if (c.bulk_w) {
      if (tid == 0) {
        const uint32_t bytes = static_cast<uint32_t>(c.stg_bytes);
        mbar_arrive_expect_tx(stg_bar, bytes);
        const char* src = reinterpret_cast<const char*>(ws + wrow0 * a.K);
        for (uint32_t off = 0; off < bytes; off += 32768u)
          bulk_load(smem_u32(sio) + off, src + off, min(32768u, bytes - off), stg_bar);
      }
      okw = wait_phase(stg_bar, 0, abort_flag, 1u);
    }
    if (okw) {
      const int units = BN * kchunks * 8;
      for (int base = tid; base < units; base += 4 * kThreads) {
        uint16_t v[4][8];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int q = base + b * kThreads;
          const int j = q & 7;
          const int r = (q >> 3) % BN;
          const int kc = (q >> 3) / BN;
          const int k0 = kc * kBK + j * 8;
          int tap0 = 0, c0 = 0, ch = 0, u = 0;
          if (c.mode == kModeCh8 && k0 < a.K) { tap0 = k0 / a.cg; c0 = k0 - tap0 * a.cg; }
          if (c.mode == kModeRow8) { ch = (k0 / 8) / a.kh; u = (k0 / 8) - ch * a.kh; }
          int idx[8];  // positions in the OIHW row, -1: zero padding
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            idx[e] = -1;
            if (q < units && r < rows_valid) {
              if (c.mode == kModeCh8) idx[e] = (k0 + e < a.K) ? (c0 + e) * khw + tap0 : -1;
              else if (c.mode == kModeRow8) idx[e] = (ch < a.cg && e < a.kw) ? ch * khw + u * a.kw + e : -1;
              else idx[e] = (k0 + e < a.K) ? k0 + e : -1;
            }
          }
          // one source per launch (a uniform branch, not a select of two loads)
          if (c.bulk_w) {
            const uint16_t* src = stg + static_cast<long long>(min(r, rows_valid - 1)) * a.K;  // a real row
#pragma unroll
            for (int e = 0; e < 8; ++e) v[b][e] = idx[e] < 0 ? 0 : src[idx[e] < 0 ? 0 : idx[e]];
          } else {
            const uint16_t* src = ws + (wrow0 + min(r, rows_valid - 1)) * a.K;  // a real row
#pragma unroll
            for (int e = 0; e < 8; ++e) v[b][e] = idx[e] < 0 ? 0 : src[idx[e] < 0 ? 0 : idx[e]];
          }
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int q = base + b * kThreads;
          if (q < units) {
            const int j = q & 7, r = (q >> 3) % BN, kc = (q >> 3) / BN;
            *reinterpret_cast<uint4*>(sB + kc * (BN * 128) + swz(r, j)) =
                make_uint4(pack2(v[b][0], v[b][1]), pack2(v[b][2], v[b][3]), pack2(v[b][4], v[b][5]),
                           pack2(v[b][6], v[b][7]));
          }
        }
      }
      for (int cc = tid; cc < BN; cc += kThreads)
        sbias[cc] = (a.bias && cc < rows_valid) ? to_f32(static_cast<const T*>(a.bias)[g * a.mg + co0 + cc]) : 0.0f;
    }
    fence_proxy_async();  // the generic-proxy stores above, visible to tcgen05.mma
  }
  __syncthreads();  // weights laid out; the staging space becomes the tile buffers

  if (warp < kEpiWarps) {
    // ================================ epilogue ================================
    bool ok = !*abort_flag;
    const int row = warp * 32 + lane;
    T* __restrict__ y = static_cast<T*>(a.y);
    const T* __restrict__ res = static_cast<const T*>(a.residual);
    const bool has_bias = a.bias != nullptr, has_res = res != nullptr;
    const long long cbase = static_cast<long long>(g) * a.mg + co0;  // first output channel

    // residual rows of tile t into buffer i: one bulk copy per channel row
    auto issue_res = [&](int t, int i) {
      int n, p0;
      tile_origin(t, &n, &p0);
      const int vpx = min(kM, static_cast<int>(a.howo) - p0);
      if (tid == 0) mbar_arrive_expect_tx(res_bar(i), static_cast<uint32_t>(rows_valid * vpx * 2));
      for (int cc = tid; cc < rows_valid; cc += kEpiWarps * 32) {
        const T* src = res + ((static_cast<long long>(n) * a.c_out + cbase + cc) * a.howo + p0);
        bulk_load(smem_u32(sio + (i * BN + cc) * (kM * 2)), src, static_cast<uint32_t>(vpx * 2), res_bar(i));
      }
    };
    int res_pending = -1;  // tile whose residual copy is in flight and not yet waited for
    if (c.epi_bulk && has_res && ok && ntiles > 0) { issue_res(0, 0); res_pending = 0; }

    for (int t = 0; ok && t < ntiles; ++t) {
      const int b = t & 1;
      const uint32_t u = static_cast<uint32_t>(t >> 1);
      // warp-uniform: the tensor-memory loads below are .sync.aligned
      if (!__all_sync(0xffffffffu, wait_phase(tfull_bar(b), u & 1u, abort_flag, 2u))) break;
      tc_fence_after();
      int n, p0;
      tile_origin(t, &n, &p0);
      const int vpx = min(kM, static_cast<int>(a.howo) - p0);
      const bool valid = row < vpx;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + b * BN;
      if (c.epi_bulk) {
        const int i = c.nio == 2 ? (t & 1) : 0;
        T* io = reinterpret_cast<T*>(sio) + static_cast<long long>(i) * BN * kM;
        if (has_res) {
          const uint32_t rphase = static_cast<uint32_t>((c.nio == 2 ? t >> 1 : t) & 1);
          if (!__all_sync(0xffffffffu, wait_phase(res_bar(i), rphase, abort_flag, 128u))) break;
          res_pending = -1;
        }
#pragma unroll 1
        for (int cc = 0; cc < BN; cc += 16) {
          uint32_t r[16];
          tmem_ld16(tbase + cc, r);
          float v[16], bv[16], rv[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            v[jj] = __uint_as_float(r[jj]);
            bv[jj] = sbias[cc + jj];
            rv[jj] = has_res ? to_f32(io[(cc + jj) * kM + row]) : 0.0f;
          }
          epilogue_n<16>(v, bv, rv, has_bias, has_res, a.act, a.alpha, a.beta);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) io[(cc + jj) * kM + row] = from_f32<T>(v[jj]);
        }
        tc_fence_before();
        mbar_arrive(tempty_bar(b));  // the accumulator buffer is free for the tile after next
        fence_proxy_async();         // this thread's tile values, visible to the bulk copies
        epi_sync();
        for (int cc = tid; cc < rows_valid; cc += kEpiWarps * 32) {
          T* dst = y + ((static_cast<long long>(n) * a.c_out + cbase + cc) * a.howo + p0);
          bulk_store(dst, smem_u32(io + cc * kM), static_cast<uint32_t>(vpx * 2));
        }
        bulk_commit();
        // the buffer of the next tile was last stored from a tile ago (two
        // buffers) or just now (one): its reads must be done before reuse
        if (c.nio == 2) bulk_wait_read<1>();
        else bulk_wait_read<0>();
        epi_sync();
        if (has_res && t + 1 < ntiles) { issue_res(t + 1, c.nio == 2 ? ((t + 1) & 1) : 0); res_pending = t + 1; }
      } else {
        long long obase = 0;
        if (valid) obase = (static_cast<long long>(n) * a.c_out + cbase) * a.howo + p0 + row;
        // residual values of the next 16 channels are requested before this
        // chunk's stores, so their latency overlaps the chunk's work
        float rnext[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          rnext[jj] = (has_res && valid && jj < rows_valid)
                          ? to_f32(__ldg(res + obase + static_cast<long long>(jj) * a.howo)) : 0.0f;
#pragma unroll 1
        for (int cc = 0; cc < BN; cc += 16) {
          float rcur[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) rcur[jj] = rnext[jj];
          if (has_res && valid && cc + 16 < BN) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int col = cc + 16 + jj;
              rnext[jj] = col < rows_valid ? to_f32(__ldg(res + obase + static_cast<long long>(col) * a.howo)) : 0.0f;
            }
          }
          uint32_t r[16];
          tmem_ld16(tbase + cc, r);
          float v[16], bv[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            v[jj] = __uint_as_float(r[jj]);
            bv[jj] = sbias[cc + jj];
          }
          epilogue_n<16>(v, bv, rcur, has_bias, has_res, a.act, a.alpha, a.beta);
          if (valid) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              if (cc + jj < rows_valid) y[obase + static_cast<long long>(cc + jj) * a.howo] = from_f32<T>(v[jj]);
          }
        }
        tc_fence_before();
        mbar_arrive(tempty_bar(b));
      }
    }
    if (res_pending >= 0) {  // aborted with a residual copy in flight: let it land first
      const int i = c.nio == 2 ? (res_pending & 1) : 0;
      const uint32_t rphase = static_cast<uint32_t>((c.nio == 2 ? res_pending >> 1 : res_pending) & 1);
      wait_phase(res_bar(i), rphase, abort_flag, 128u, true);
    }
    if (c.epi_bulk) bulk_wait_all();  // the output rows have landed before the block retires
  } else if (warp < kEpiWarps + kProdWarps) {
    // ============================ A-operand gather ============================
    // Stage jobs (tile, k chunk) run as a software pipeline: the loads of the
    // next job are issued into registers before the current job's values are
    // packed into its stage, so two jobs' loads are in flight per thread.
    const int ptid = tid - kEpiWarps * 32;
    const int row = ptid & (kM - 1);
    const int part = ptid >> 7;  // 0 or 1: 16-byte units 4*part .. 4*part+3 of each row
    int stage = 0;
    uint32_t phase = 0;
    bool ok = !*abort_flag;
    const int HB = c.halo_bufs;
    struct Pix {
      bool valid;
      int ih0, iw0;
      long long pb;          // element of tap (0,0), channel 0, in src
      const uint16_t* src;   // x, or the tile's halo buffer in shared memory
      long long cs;          // elements from one input channel to the next in src
      uint32_t em[4];  // row8: valid taps of a kernel row as 16-bit lane masks
      uint32_t wv0, wv1;  // row8: 4-byte words worth loading, for an even / odd first tap
    };
    auto pix_of = [&](int t) {
      Pix ps;
      int n, p0;
      tile_origin(t, &n, &p0);
      const int pix = p0 + row;
      ps.valid = pix < a.howo;
      ps.ih0 = 0; ps.iw0 = 0; ps.pb = 0;
      ps.src = HB ? halo + static_cast<long long>(t % HB) * c.halo_cg * c.halo_slot : xs;
      ps.cs = HB ? c.halo_slot : a.hw;
      ps.em[0] = ps.em[1] = ps.em[2] = ps.em[3] = 0;
      ps.wv0 = ps.wv1 = 0;
      if (ps.valid) {
        const int oh = pix / a.wo, ow = pix - (pix / a.wo) * a.wo;
        ps.ih0 = oh * a.sh - a.pt;
        ps.iw0 = ow * a.sw - a.pl;
        if (HB) {  // the halo slot holds the plane from element halo_a0 on, 8 elements in
          ps.pb = 8 + static_cast<long long>(ps.ih0) * a.w + ps.iw0 - halo_a0[t % HB];
        } else {
          ps.pb = (static_cast<long long>(n) * a.c_in + static_cast<long long>(g) * a.cg) * a.hw +
                  static_cast<long long>(ps.ih0) * a.w + ps.iw0;
        }
        if (c.mode == kModeRow8) {
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const int iw = ps.iw0 + v;
            if (v < a.kw && iw >= 0 && iw < a.w) ps.em[v >> 1] |= (v & 1) ? 0xFFFF0000u : 0x0000FFFFu;
          }
#pragma unroll
          for (int sp = 0; sp < 2; ++sp)
#pragma unroll
            for (int k = 0; k < 5; ++k) {
              const int c0 = ps.iw0 - sp + 2 * k;  // columns c0, c0 + 1 of word k
              const bool any = (c0 >= 0 && c0 < a.w) || (c0 + 1 >= 0 && c0 + 1 < a.w);
              if (any && c0 < ps.iw0 + a.kw && c0 + 1 >= ps.iw0) {
                if (sp) ps.wv1 |= 1u << k;
                else ps.wv0 |= 1u << k;
              }
            }
          if (HB) ps.wv0 = ps.wv1 = 0x1Fu;  // shared memory around the slot: every word is readable
        }
      }
      return ps;
    };
    // raw values of one job's 4 units: row8 keeps 5 words + selector + flag,
    // the others 8 zero-extended 16-bit values
    auto load_job = [&](const Pix& ps, int kc, uint32_t (&raw)[4][8]) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = part * 4 + jj;
        if (c.mode == kModeRow8) {
          const int4 e = tab[kc * 8 + j];
          const int ih = ps.ih0 + e.y;
          const bool in = ps.valid && e.w && static_cast<unsigned>(ih) < static_cast<unsigned>(a.h);
          const long long e0 = ps.pb + e.x;  // first tap's element
          const int sp = static_cast<int>(e0 & 1);
          const uint32_t* wp = reinterpret_cast<const uint32_t*>(ps.src + (in ? e0 - sp : 0));
          const uint32_t m = in ? (sp ? ps.wv1 : ps.wv0) : 0u;
          if (HB) {  // shared memory: generic loads (ld.global.nc is for global addresses only)
#pragma unroll
            for (int k = 0; k < 5; ++k) raw[jj][k] = (m >> k & 1u) ? wp[k] : 0u;
          } else {
#pragma unroll
            for (int k = 0; k < 5; ++k) raw[jj][k] = (m >> k & 1u) ? __ldg(wp + k) : 0u;
          }
          raw[jj][5] = sp ? 0x5432u : 0x3210u;
          raw[jj][6] = in ? 1u : 0u;
          raw[jj][7] = 0u;
        } else if (c.mode == kModeCh8) {
          const int4 e = tab[kc * 8 + j];
          const int ih = ps.ih0 + e.y, iw = ps.iw0 + e.z;
          const bool in = ps.valid && e.w && static_cast<unsigned>(ih) < static_cast<unsigned>(a.h) &&
                          static_cast<unsigned>(iw) < static_cast<unsigned>(a.w);
          const uint16_t* src = ps.src + (in ? ps.pb + e.x : 0);
#pragma unroll
          for (int q = 0; q < 8; ++q) raw[jj][q] = in ? src[static_cast<long long>(q) * ps.cs] : 0u;
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int4 e = tab[kc * kBK + j * 8 + q];
            const int ih = ps.ih0 + e.y, iw = ps.iw0 + e.z;
            const bool in = ps.valid && e.w && static_cast<unsigned>(ih) < static_cast<unsigned>(a.h) &&
                            static_cast<unsigned>(iw) < static_cast<unsigned>(a.w);
            raw[jj][q] = in ? ps.src[in ? ps.pb + e.x : 0] : 0u;
          }
        }
      }
    };
    auto emit_job = [&](const Pix& ps, const uint32_t (&raw)[4][8], uint8_t* As) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = part * 4 + jj;
        uint4 o;
        if (c.mode == kModeRow8) {
          const uint32_t sel = raw[jj][5];
          const uint32_t keep = raw[jj][6] ? 0xFFFFFFFFu : 0u;
          o.x = __byte_perm(raw[jj][0], raw[jj][1], sel) & ps.em[0] & keep;
          o.y = __byte_perm(raw[jj][1], raw[jj][2], sel) & ps.em[1] & keep;
          o.z = __byte_perm(raw[jj][2], raw[jj][3], sel) & ps.em[2] & keep;
          o.w = __byte_perm(raw[jj][3], raw[jj][4], sel) & ps.em[3] & keep;
        } else {
          o = make_uint4(raw[jj][0] | (raw[jj][1] << 16), raw[jj][2] | (raw[jj][3] << 16),
                         raw[jj][4] | (raw[jj][5] << 16), raw[jj][6] | (raw[jj][7] << 16));
        }
        *reinterpret_cast<uint4*>(As + swz(row, j)) = o;
      }
    };
    const int njobs = ntiles * kchunks;
    // two raw buffers used in turn (no copy between them, so nothing waits on
    // the loads just issued until their job is emitted)
    uint32_t ra[4][8], rb[4][8];
    // the halo of tile tt is in its buffer / this thread is done reading it
    auto halo_in = [&](int tt) -> bool {
      return !HB || wait_phase(hfull_bar(tt % HB), static_cast<uint32_t>((tt / HB) & 1), abort_flag, 512u);
    };
    auto halo_out = [&](int tt) {
      if (HB) mbar_arrive(hempty_bar(tt % HB));
    };
    Pix pa, pb;
    if (ok && njobs > 0) {
      ok = halo_in(0);
      if (ok) {
        pa = pix_of(0);
        load_job(pa, 0, ra);
        if (kchunks == 1) halo_out(0);
      }
    }
    int t = 0, kc = 0;
    // one pipeline step: issue the next job's loads into `nxt`, then emit `cur`
    auto step = [&](int jb, const Pix& pc, uint32_t (&cur)[4][8], Pix& pn, uint32_t (&nxt)[4][8]) {
      int tn = t, kcn = kc + 1;
      if (kcn == kchunks) { kcn = 0; tn = t + 1; }
      if (jb + 1 < njobs) {
        if (tn != t) {
          if (!halo_in(tn)) return false;
          pn = pix_of(tn);
        } else {
          pn = pc;
        }
        load_job(pn, kcn, nxt);
        if (kcn == kchunks - 1) halo_out(tn);
      }
      if (!wait_phase(empty_bar(stage), phase ^ 1u, abort_flag, 4u)) return false;
      emit_job(pc, cur, sA + stage * kStageBytes);
      fence_proxy_async();
      mbar_arrive(full_bar(stage));
      if (++stage == S) { stage = 0; phase ^= 1u; }
      t = tn;
      kc = kcn;
      return true;
    };
    if (HB) {
      // gathering from shared memory: short latency, no register pipeline
      for (int jb = 0; ok && jb < njobs; ++jb) {
        if (jb > 0) {
          int tn = t, kcn = kc + 1;
          if (kcn == kchunks) { kcn = 0; tn = t + 1; }
          if (tn != t) {
            if (!halo_in(tn)) { ok = false; break; }
            pa = pix_of(tn);
          }
          load_job(pa, kcn, ra);
          if (kcn == kchunks - 1) halo_out(tn);
          t = tn;
          kc = kcn;
        }
        if (!wait_phase(empty_bar(stage), phase ^ 1u, abort_flag, 4u)) { ok = false; break; }
        emit_job(pa, ra, sA + stage * kStageBytes);
        fence_proxy_async();
        mbar_arrive(full_bar(stage));
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    } else {
      for (int jb = 0; ok && jb < njobs; jb += 2) {
        ok = step(jb, pa, ra, pb, rb);
        if (ok && jb + 1 < njobs) ok = step(jb + 1, pb, rb, pa, ra);
      }
    }
  } else {
    // ============ halo copies (lanes 1-31) and MMA issue (lane 0) ==============
    const int HB = c.halo_bufs;
    if (lane != 0 && HB > 0) {
      // per tile: the input rows its windows reach, one contiguous span of each
      // input channel's plane, rounded out to 16 bytes, into the tile's buffer
      bool okl = !*abort_flag;
      int issued = 0;
      for (int t = 0; okl && t < ntiles; ++t) {
        const int hb = t % HB;
        okl = __all_sync(0xFFFFFFFEu, wait_phase(hempty_bar(hb), static_cast<uint32_t>(((t / HB) & 1) ^ 1),
                                                 abort_flag, 256u));
        if (!okl) break;
        int n, p0;
        tile_origin(t, &n, &p0);
        const int vpx = min(kM, static_cast<int>(a.howo) - p0);
        const int oh_f = p0 / a.wo, oh_l = (p0 + vpx - 1) / a.wo;
        const int r_lo = max(0, oh_f * a.sh - a.pt);
        const int r_hi = min(a.h, oh_l * a.sh - a.pt + (a.kh - 1) * a.dh + 1);
        long long a0 = 0, a1 = 0;
        if (r_hi > r_lo) {
          a0 = (static_cast<long long>(r_lo) * a.w) & ~7LL;
          a1 = (static_cast<long long>(r_hi) * a.w + 7) & ~7LL;
        }
        const uint32_t bytes = static_cast<uint32_t>((a1 - a0) * 2);
        if (lane == 1) {
          halo_a0[hb] = static_cast<int>(a0);
          mbar_arrive_expect_tx(hfull_bar(hb), bytes * static_cast<uint32_t>(a.cg));
        }
        __syncwarp(0xFFFFFFFEu);
        if (bytes) {
          const uint16_t* plane0 = xs + (static_cast<long long>(n) * a.c_in + static_cast<long long>(g) * a.cg) * a.hw;
          for (int ch = lane - 1; ch < a.cg; ch += 31)
            bulk_load(smem_u32(halo + (static_cast<long long>(hb) * a.cg + ch) * c.halo_slot + 8),
                      plane0 + static_cast<long long>(ch) * a.hw + a0, bytes, hfull_bar(hb));
        }
        issued = t + 1;
      }
      if (!okl) {  // aborted: copies still in flight must land before the block retires
        for (int t = max(0, issued - HB); t < issued; ++t)
          wait_phase(hfull_bar(t % HB), static_cast<uint32_t>((t / HB) & 1), abort_flag, 512u, true);
      }
    }
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc = make_idesc(sizeof(T) == 2 && !std::is_same<T, __half>::value, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = !*abort_flag;
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int b = t & 1;
        const uint32_t u = static_cast<uint32_t>(t >> 1);
        if (!wait_phase(tempty_bar(b), (u & 1u) ^ 1u, abort_flag, 16u)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + b * BN;
        for (int kc = 0; kc < kchunks; ++kc) {
          if (!wait_phase(full_bar(stage), phase, abort_flag, 32u)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = sw128_desc(a0 + stage * kStageBytes + kk * 32);
            const uint64_t bd = sw128_desc(b0 + kc * (BN * 128) + kk * 32);
            mma_f16(d, ad, bd, idesc, (kc | kk) != 0 ? 1u : 0u);
          }
          mma_commit(empty_bar(stage));
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull_bar(b));
      }
    }
  }

  // ---- teardown ----------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    if (lane == 0 && *abort_flag) {
      // outstanding MMAs must finish before their tensor memory is freed
      mma_commit(drain_bar);
      wait_phase(drain_bar, 0, abort_flag, 64u, true);
    }
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem_base), "r"(kCols)
                 : "memory");
  }
}

// Shared-memory bytes of a launch configuration (with the 1 KB alignment slack).
size_t tc_bytes(int bn, const TcLaunch& c) { return tc_layout(bn, c).end + 1024; }

template <typename T, int BN>
cudaError_t launch_bn(const TcPlan& p, const TcLaunch& c, const ConvArgs& a, cudaStream_t s) {
  auto kern = igemm_tc<T, BN>;
  const size_t smem = tc_bytes(BN, c);
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  kern<<<p.ctas, kThreads, smem, s>>>(a, p, c);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const TcPlan& p, const TcLaunch& c, const ConvArgs& a, cudaStream_t s) {
  switch (p.bn) {
    case 32: return launch_bn<T, 32>(p, c, a, s);
    case 48: return launch_bn<T, 48>(p, c, a, s);
    case 64: return launch_bn<T, 64>(p, c, a, s);
    case 128: return launch_bn<T, 128>(p, c, a, s);
    case 256: return launch_bn<T, 256>(p, c, a, s);
    default: return cudaErrorInvalidValue;
  }
}

int kpad_of(int mode, const ConvArgs& a) {
  const long long k = mode == kModeRow8 ? static_cast<long long>(a.cg) * a.kh * 8 : a.K;
  return static_cast<int>((k + kBK - 1) / kBK * kBK);
}

// Fill the address-dependent part of a launch; false if nothing fits.
bool configure(const TcPlan& p, const ConvArgs& a, bool addresses_known, TcLaunch* c) {
  c->mode = p.mode;
  if (c->mode == kModeRow8 && addresses_known) {
    // 4-byte word loads: x 4-byte aligned and an even element count (so no
    // word straddles the end of x)
    const long long xe = static_cast<long long>(a.n) * a.c_in * a.hw;
    if (reinterpret_cast<uintptr_t>(a.x) % 4 != 0 || (xe & 1)) c->mode = kModeNat;
  }
  c->k_pad = kpad_of(c->mode, a);
  const int rows_first = min(p.bn, a.mg);  // rows of the first channel tile
  c->stg_bytes = static_cast<long long>(rows_first) * a.K * 2;
  c->bulk_w = (!addresses_known || reinterpret_cast<uintptr_t>(a.wt) % 16 == 0) &&
              (static_cast<long long>(p.bn) * a.K * 2) % 16 == 0 &&
              (static_cast<long long>(a.mg) * a.K * 2) % 16 == 0 &&
              ((a.mg % p.bn) == 0 || a.groups * p.co_tiles == 1) && c->stg_bytes % 16 == 0 &&
              c->stg_bytes < (1 << 20);
  c->epi_bulk = (a.howo % 8 == 0) &&
                (!addresses_known || (reinterpret_cast<uintptr_t>(a.y) % 16 == 0 &&
                                      (!a.residual || reinterpret_cast<uintptr_t>(a.residual) % 16 == 0)));
  // input halo: the rows a tile's windows reach, per input channel of the
  // group, copied whole into shared memory (planes must start on 16 bytes)
  const int r_out = min(a.ho, (a.wo - 1 + kM - 1) / a.wo + 1);  // output rows a tile can touch
  const long long r_in = static_cast<long long>(r_out - 1) * a.sh + static_cast<long long>(a.kh - 1) * a.dh + 1;
  const long long slot = (r_in * a.w + 7) / 8 * 8 + 24;       // 8 elements of slack on each side
  const bool halo_ok = (a.hw % 8 == 0) && slot * a.cg * 2 < (1 << 20) &&
                       (!addresses_known || reinterpret_cast<uintptr_t>(a.x) % 16 == 0);
  c->halo_cg = a.cg;
  c->halo_slot = static_cast<int>(halo_ok ? slot : 0);
  for (int hb = halo_ok ? 2 : 0; hb >= 0; --hb) {
    for (int epi = c->epi_bulk; epi >= 0; --epi) {
      for (int nio = epi ? 2 : 1; nio >= 1; --nio) {
        for (int st = 4; st >= 2; --st) {
          TcLaunch t = *c;
          t.halo_bufs = hb;
          t.epi_bulk = epi;
          t.nio = nio;
          t.stages = st;
          if (tc_bytes(p.bn, t) <= kTcMaxSmem) {
            *c = t;
            return true;
          }
        }
      }
    }
  }
  return false;
}

}  // namespace

// Planner entry (host): channel tile, k order, tiles and blocks for a shape
// (addresses unknown: assumed aligned).  The channel tile is the one with
// the fewest padded channels (ties: the wider) whose weights fit in shared
// memory; false when not even the narrowest fits.
bool tc_plan(const ConvArgs& a, int sm, TcPlan* t) {
  static const int bns[] = {256, 128, 64, 48, 32};
  constexpr int kNb = sizeof(bns) / sizeof(bns[0]);
  int order[kNb];
  for (int i = 0; i < kNb; ++i) order[i] = i;
  auto padded = [&](int i) { return (static_cast<long long>(a.mg) + bns[i] - 1) / bns[i] * bns[i]; };
  std::stable_sort(order, order + kNb, [&](int x, int y) { return padded(x) < padded(y); });
  if (a.cg % 8 == 0) t->mode = kModeCh8;
  else if (a.dw == 1 && a.kw <= 8 && a.kw >= 5) t->mode = kModeRow8;  // rows of 5..8 taps: few padded
  else t->mode = kModeNat;
  t->tiles_per_img = static_cast<int>((a.howo + kM - 1) / kM);
  const long long pix_tiles = static_cast<long long>(a.n) * t->tiles_per_img;
  if (pix_tiles > 2147483647LL) return false;
  t->pix_tiles = static_cast<int>(pix_tiles);
  TcLaunch c;
  bool fits = false;
  for (int i = 0; i < kNb && !fits; ++i) {
    t->bn = bns[order[i]];
    t->co_tiles = (a.mg + t->bn - 1) / t->bn;
    fits = configure(*t, a, false, &c);
  }
  if (!fits) return false;
  const int bn = t->bn;
  t->k_pad = c.k_pad;
  t->stages = c.stages;
  t->smem = tc_bytes(bn, c);
  const long long combos = static_cast<long long>(a.groups) * t->co_tiles;
  long long cpc = combos >= sm ? 1 : std::min<long long>(pix_tiles, sm / combos);
  if (cpc < 1) cpc = 1;
  if (combos * cpc > 2147483647LL) return false;
  t->ctas = static_cast<int>(combos * cpc);
  return true;
}

cudaError_t launch_tc(const Plan& plan, const ConvArgs& a, int dtype, cudaStream_t s) {
  TcLaunch c;
  if (!configure(plan.tc, a, true, &c)) return cudaErrorInvalidConfiguration;
  switch (dtype) {
    case CONV_F16: return launch_typed<__half>(plan.tc, c, a, s);
    case CONV_BF16: return launch_typed<__nv_bfloat16>(plan.tc, c, a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t tc_error_word(uint32_t* word, int reset) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  err = cudaMemcpyFromSymbol(word, g_tc_error, sizeof(uint32_t));
  if (err != cudaSuccess || !reset) return err;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(uint32_t));
}

}  // namespace conv
