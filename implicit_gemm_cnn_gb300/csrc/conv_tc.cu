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
//   * a tile is 128 output pixels (flattened over the batch: MMA M = 128) x
//     BN output channels (MMA N); its float32 accumulator lives in tensor
//     memory, double buffered so the epilogue of one tile overlaps the next;
//   * warps 4-11 gather the A operand: for each pixel row and each k chunk of
//     64 terms they load 8 x 16-bit values per 16-byte unit from x, zero for
//     taps outside the image, and store them into a 128-byte-swizzled K-major
//     stage that tcgen05.mma reads directly.  k is ordered (tap, channel) when
//     the channels per group are a multiple of 8 -- one window test per 8
//     values, the channels one input plane apart, as "Convolution, pooling and
//     resize" (Apple M2, taps innermost) orders its staging -- and (channel,
//     tap) otherwise.  The window offsets come from a table decoded once per
//     block;
//   * warps 0-3 first copy the block's weight rows into shared memory (one
//     bulk copy of the OIHW rows, then a permutation into the swizzled K-major
//     layout in the same k order -- the weight re-layout that "Convolution,
//     pooling and resize" measured at 1.27x on 3x3 layers, done on chip), then
//     run the epilogue: tcgen05.ld of the accumulator (thread = pixel, so each
//     warp's stores of one channel are 32 consecutive pixels of NCHW y),
//     bias, residual, activation in float32, one rounding to the element type;
//   * warp 12 allocates tensor memory and one lane issues the MMAs
//     (kind::f16, M=128, N=BN, K=16 per instruction) and the commits that
//     release stages and accumulators.
// Every mbarrier wait is bounded: after kWaitNs the waiting thread flags the
// block and the device error word, every role drains out, outstanding MMAs are
// waited for (bounded again) and tensor memory is freed before exit.
#include <type_traits>

#include "conv_internal.h"

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
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s
constexpr unsigned kMaxSpins = 1u << 28;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}

// Wait until the phase of `bar` with parity `parity` has completed.  Gives up
// (returns false) after kWaitNs or kMaxSpins polls -- then it raises the
// block's abort flag and the device error word -- or as soon as another
// thread of the block raised the abort flag (unless `ignore_abort`).
__device__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t code,
                           bool ignore_abort = false) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (unsigned i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (!ignore_abort && *abort_flag) return false;
      if (globaltimer() - t0 > kWaitNs || i > kMaxSpins) {
        *abort_flag = 1;
        atomicOr(&g_tc_error, code);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (SBO); the leading offset is unused for this layout.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;   // descriptor version of tcgen05
  d |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: D float32, A and B half or bfloat16, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc(bool bf16, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Byte offset of the 16-byte unit j (k = 8j .. 8j+7) of row r in a 128-byte
// swizzled K-major tile: 8-row groups of 1024 bytes, unit index XOR row%8.
__device__ __forceinline__ uint32_t swz(int r, int j) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi) {
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

struct TcLayout {
  uint32_t b_off, stg_off, a_off, tab_off, bias_off, bar_off, slot_off, end;
};

__host__ __device__ inline TcLayout tc_layout(int bn, int k_pad, int stages, int tap_major,
                                              long long stg_bytes) {
  TcLayout L;
  L.b_off = 0;
  L.a_off = static_cast<uint32_t>(k_pad / kBK) * bn * 128;           // multiple of 1024
  L.stg_off = L.a_off + static_cast<uint32_t>(stages) * kStageBytes;
  L.tab_off = L.stg_off + static_cast<uint32_t>((stg_bytes + 15) / 16 * 16);
  const int ntab = tap_major ? k_pad / 8 : k_pad;
  L.bias_off = L.tab_off + static_cast<uint32_t>(ntab) * 16;
  L.bar_off = L.bias_off + static_cast<uint32_t>(bn) * 4;
  L.slot_off = L.bar_off + static_cast<uint32_t>(2 * stages + 7) * 8;
  L.end = L.slot_off + 16;
  return L;
}

template <typename T, int BN>
__global__ void __launch_bounds__(kThreads, 1) igemm_tc(const ConvArgs a, const TcPlan p,
                                                        long long stg_bytes, int bulk_ok) {
  extern __shared__ uint8_t tsm_raw[];
  // 1024-byte alignment for the swizzled tiles (the launch adds 1 KB of slack)
  uint8_t* tsm = tsm_raw + ((1024 - (smem_u32(tsm_raw) & 1023)) & 1023);
  const int S = p.stages;
  const TcLayout L = tc_layout(BN, p.k_pad, S, p.tap_major, stg_bytes);
  uint8_t* sB = tsm + L.b_off;
  uint8_t* sA = tsm + L.a_off;
  uint16_t* stg = reinterpret_cast<uint16_t*>(tsm + L.stg_off);
  int4* tab = reinterpret_cast<int4*>(tsm + L.tab_off);
  float* sbias = reinterpret_cast<float*>(tsm + L.bias_off);
  const uint32_t bar0 = smem_u32(tsm + L.bar_off);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t wready_bar = bar0 + 8u * (2 * S + 4);
  const uint32_t stg_bar = bar0 + 8u * (2 * S + 5);
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 6);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tsm + L.slot_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tsm + L.slot_off + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int kchunks = p.k_pad / kBK;
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
    }
    mbar_init(wready_bar, kEpiWarps * 32);
    mbar_init(stg_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  const int ntab = p.tap_major ? p.k_pad / 8 : p.k_pad;
  for (int e = tid; e < ntab; e += kThreads) {
    const int k = p.tap_major ? e * 8 : e;
    int tap, c;
    if (p.tap_major) { tap = k / a.cg; c = k - tap * a.cg; }
    else { c = k / khw; tap = k - c * khw; }
    const int u = tap / a.kw, v = tap - (tap / a.kw) * a.kw;
    const int dy = u * a.dh, dx = v * a.dw;
    tab[e] = make_int4(c * static_cast<int>(a.hw) + dy * a.w + dx, dy, dx, k < a.K ? 1 : 0);
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

  // ---- this block's tiles: one (group, channel tile), strided pixel tiles ---
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

  if (warp < kEpiWarps) {
    // ======================= weights, then the epilogue ======================
    const long long wrow0 = static_cast<long long>(g) * a.mg + co0;  // first OIHW row
    bool ok = true;
    if (bulk_ok) {
      if (tid == 0) {
        const uint32_t bytes = static_cast<uint32_t>(stg_bytes);
        mbar_arrive_expect_tx(stg_bar, bytes);
        const char* src = reinterpret_cast<const char*>(ws + wrow0 * a.K);
        for (uint32_t off = 0; off < bytes; off += 32768u) {
          const uint32_t n = min(32768u, bytes - off);
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                  smem_u32(stg) + off),
              "l"(src + off), "r"(n), "r"(stg_bar)
              : "memory");
        }
      }
      ok = wait_phase(stg_bar, 0, abort_flag, 1u);
    }
    ok = __all_sync(0xffffffffu, ok);  // warp-uniform before the loop below
    if (ok) {
      const int units = BN * kchunks * 8;
      for (int q = tid; q < units; q += kEpiWarps * 32) {
        const int j = q & 7;
        const int r = (q >> 3) % BN;
        const int kc = (q >> 3) / BN;
        const int k0 = kc * kBK + j * 8;
        uint16_t v[8];
        int tap0 = 0, c0 = 0;
        if (p.tap_major && k0 < a.K) { tap0 = k0 / a.cg; c0 = k0 - tap0 * a.cg; }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int k = k0 + e;
          uint16_t val = 0;
          if (r < rows_valid && k < a.K) {
            const int idx = p.tap_major ? (c0 + e) * khw + tap0 : k;  // OIHW order within the row
            val = bulk_ok ? stg[static_cast<long long>(r) * a.K + idx]
                          : ws[(wrow0 + r) * a.K + idx];
          }
          v[e] = val;
        }
        *reinterpret_cast<uint4*>(sB + kc * (BN * 128) + swz(r, j)) =
            make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
      }
      fence_proxy_async();
      mbar_arrive(wready_bar);
    }
    // epilogue: bias of the block's channel tile staged once in shared memory
    for (int c = tid; c < BN; c += kEpiWarps * 32)
      sbias[c] = (a.bias && c < rows_valid) ? to_f32(static_cast<const T*>(a.bias)[g * a.mg + co0 + c]) : 0.0f;
    asm volatile("bar.sync 1, %0;\n" ::"n"(kEpiWarps * 32) : "memory");  // epilogue warps only
    const int row = warp * 32 + lane;
    T* __restrict__ y = static_cast<T*>(a.y);
    const T* __restrict__ res = static_cast<const T*>(a.residual);
    const bool has_bias = a.bias != nullptr, has_res = res != nullptr;
    for (int t = 0; ok && t < ntiles; ++t) {
      const int b = t & 1;
      const uint32_t u = static_cast<uint32_t>(t >> 1);
      // warp-uniform: the tensor-memory loads below are .sync.aligned
      if (!__all_sync(0xffffffffu, wait_phase(tfull_bar(b), u & 1u, abort_flag, 2u))) break;
      tc_fence_after();
      const long long pix = static_cast<long long>(local + t * cpc) * kM + row;
      const bool valid = pix < a.npix;
      long long obase = 0;
      if (valid) {
        const long long n = pix / a.howo;
        obase = (n * a.c_out + static_cast<long long>(g) * a.mg + co0) * a.howo + (pix - n * a.howo);
      }
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + b * BN;
      // residual values of the next 16 channels are requested before this
      // chunk's stores, so their latency overlaps the chunk's work
      float rnext[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        rnext[jj] = (has_res && valid && jj < rows_valid)
                        ? to_f32(__ldg(res + obase + static_cast<long long>(jj) * a.howo)) : 0.0f;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float rcur[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) rcur[jj] = rnext[jj];
        if (has_res && valid && c + 16 < BN) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int col = c + 16 + jj;
            rnext[jj] = col < rows_valid ? to_f32(__ldg(res + obase + static_cast<long long>(col) * a.howo)) : 0.0f;
          }
        }
        uint32_t r[16];
        tmem_ld16(tbase + c, r);
        if (valid) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int col = c + jj;
            if (col < rows_valid)
              y[obase + static_cast<long long>(col) * a.howo] = epilogue_vals<T>(
                  __uint_as_float(r[jj]), sbias[col], rcur[jj], has_bias, has_res, a.act, a.alpha, a.beta);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(b));
    }
  } else if (warp < kEpiWarps + kProdWarps) {
    // ============================ A-operand gather ============================
    const int ptid = tid - kEpiWarps * 32;
    const int row = ptid & (kM - 1);
    const int part = ptid >> 7;  // 0 or 1: 16-byte units 4*part .. 4*part+3 of each row
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = 0; ok && t < ntiles; ++t) {
      const long long pix = static_cast<long long>(local + t * cpc) * kM + row;
      const bool valid = pix < a.npix;
      int ih0 = 0, iw0 = 0;
      long long pb = 0;
      if (valid) {
        const int n = static_cast<int>(pix / a.howo);
        const int rem = static_cast<int>(pix - static_cast<long long>(n) * a.howo);
        const int oh = rem / a.wo, ow = rem - (rem / a.wo) * a.wo;
        ih0 = oh * a.sh - a.pt;
        iw0 = ow * a.sw - a.pl;
        pb = (static_cast<long long>(n) * a.c_in + static_cast<long long>(g) * a.cg) * a.hw +
             static_cast<long long>(ih0) * a.w + iw0;
      }
      for (int kc = 0; kc < kchunks; ++kc) {
        if (!wait_phase(empty_bar(stage), phase ^ 1u, abort_flag, 4u)) { ok = false; break; }
        uint8_t* As = sA + stage * kStageBytes;
        if (p.tap_major) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = part * 4 + jj;
            const int4 e = tab[kc * 8 + j];
            const int ih = ih0 + e.y, iw = iw0 + e.z;
            const bool in = valid && e.w && static_cast<unsigned>(ih) < static_cast<unsigned>(a.h) &&
                            static_cast<unsigned>(iw) < static_cast<unsigned>(a.w);
            uint16_t v[8];
            const uint16_t* src = xs + (in ? pb + e.x : 0);
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = in ? src[static_cast<long long>(q) * a.hw] : 0;
            *reinterpret_cast<uint4*>(As + swz(row, j)) =
                make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = part * 4 + jj;
            uint16_t v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int4 e = tab[kc * kBK + j * 8 + q];
              const int ih = ih0 + e.y, iw = iw0 + e.z;
              const bool in = valid && e.w && static_cast<unsigned>(ih) < static_cast<unsigned>(a.h) &&
                              static_cast<unsigned>(iw) < static_cast<unsigned>(a.w);
              v[q] = in ? xs[pb + e.x] : 0;
            }
            *reinterpret_cast<uint4*>(As + swz(row, j)) =
                make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
          }
        }
        fence_proxy_async();
        mbar_arrive(full_bar(stage));
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // ============================ MMA issue (one lane) ========================
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc = make_idesc(sizeof(T) == 2 && !std::is_same<T, __half>::value, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = wait_phase(wready_bar, 0, abort_flag, 8u);
      if (ok) tc_fence_after();
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

template <typename T, int BN>
cudaError_t launch_bn(const TcPlan& p, const ConvArgs& a, cudaStream_t s) {
  auto kern = igemm_tc<T, BN>;
  const int rows_valid = min(BN, a.mg);  // rows copied per block (co tile 0 is the widest)
  const long long stg_bytes = static_cast<long long>(rows_valid) * a.K * 2;
  // the bulk copy needs 16-byte aligned source rows of every block's tile
  const bool bulk_ok = (reinterpret_cast<uintptr_t>(a.wt) % 16 == 0) &&
                       ((static_cast<long long>(BN) * a.K * 2) % 16 == 0) &&
                       ((static_cast<long long>(a.mg) * a.K * 2) % 16 == 0) &&
                       ((a.mg % BN) == 0 || a.groups * p.co_tiles == 1) && stg_bytes % 16 == 0 &&
                       stg_bytes < (1 << 20);
  const TcLayout L = tc_layout(BN, p.k_pad, p.stages, p.tap_major, bulk_ok ? stg_bytes : 0);
  const size_t smem = L.end + 1024;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && configured[dev] < static_cast<int>(smem)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    configured[dev] = static_cast<int>(smem);
  }
  kern<<<p.ctas, kThreads, smem, s>>>(a, p, bulk_ok ? stg_bytes : 0, bulk_ok ? 1 : 0);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const TcPlan& p, const ConvArgs& a, cudaStream_t s) {
  switch (p.bn) {
    case 32: return launch_bn<T, 32>(p, a, s);
    case 48: return launch_bn<T, 48>(p, a, s);
    case 64: return launch_bn<T, 64>(p, a, s);
    case 128: return launch_bn<T, 128>(p, a, s);
    case 256: return launch_bn<T, 256>(p, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Shared-memory bytes of a plan (host): the planner keeps only plans that fit.
size_t tc_smem_bytes(int bn, int k_pad, int stages, int tap_major, long long stg_bytes) {
  return tc_layout(bn, k_pad, stages, tap_major, stg_bytes).end + 1024;
}

cudaError_t launch_tc(const Plan& plan, const ConvArgs& a, int dtype, cudaStream_t s) {
  switch (dtype) {
    case CONV_F16: return launch_typed<__half>(plan.tc, a, s);
    case CONV_BF16: return launch_typed<__nv_bfloat16>(plan.tc, a, s);
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
