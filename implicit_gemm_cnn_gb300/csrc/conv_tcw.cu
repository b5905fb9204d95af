// conv_tcw.cu -- implicit-GEMM convolution on the tcgen05 tensor cores over
// shifted windows of a zero-padded input band held in shared memory
// (half / bfloat16 operands, float32 accumulation in tensor memory).
//
// The GEMM is the one of "Convolutions en compute" (implicit im2col: Y^T =
// cols^T . W^T per image, K = Cin * kh * kw) with the column matrix never
// formed, not even per tile.  Positions are counted in the zero-padded input
// plane of each image, hp x wp with hp = Ho + (kh-1)*dh and wp = Wo + (kw-1)*dw,
// images one after another: output (n, oh, ow) is position
// q = (n*hp + oh)*wp + ow, and the input it reads through tap (u, v) is
// position q + u*dh*wp + v*dw.  Every tap is therefore a shift of one
// position sequence: if shared memory holds the padded input with the
// channels of a position side by side (16 bytes = 8 channels per position
// and channel block), the A operand of tap (u, v) for the tile of positions
// q0 .. q0+127 is the same buffer read from position q0 + u*dh*wp + v*dw, and
// the MMA descriptor's start address does the im2col.  Positions with
// ow >= Wo or oh >= Ho are computed and dropped (a few percent of the tile).
//
// Stride 2 (dilation 1) becomes stride 1 by splitting the input into its
// 2 x 2 phases: channel (c, a, b) of phase position (i, j) is input pixel
// (2i + a - pad_top, 2j + b - pad_left), and the kernel becomes
// ceil(kh/2) x ceil(kw/2) taps over Cin*4 channels (taps past kh or kw get
// zero weights).  The ResNet-50 stem (7x7 / 2, 3 channels) becomes a 4x4 /1
// convolution over 12 (padded to 16) channels.
//
// Roles (one persistent block per SM, 24 warps):
//   * warps 16-21 (producers) stream the block's band of padded input rows:
//     the rows of x each padded row needs arrive in shared memory by bulk
//     copies, several rows in flight; the producers then interleave each row's
//     channels into the ring (16 bytes per position and 8-channel block; zero
//     for padding, phantom channels and rows outside the image).  The ring is
//     R positions deep; positions at ring slots below 128 are also written
//     R slots further on, so that every 128-position window is contiguous;
//   * warps 22 and 23 issue the MMAs, warp 22 of the even tiles and warp 23 of
//     the odd ones (one warp issues an MMA every 80-140 cycles, slower than
//     the tensor pipe runs a 128 x 64 x 16 MMA, so two warps keep it busy):
//     per tile kh*kw*C/16 MMAs (kind::f16, M = 128 positions, N = the channel
//     tile, K = 16) whose A descriptors point at the shifted windows; a commit
//     releases the ring for the producers and another hands the accumulator
//     to the epilogue.  Warp 22 also loads the repacked weights of its
//     channel tile once (one bulk copy) and owns the tensor memory;
//   * warps 0-15 (epilogue): tcgen05.ld of the float32 accumulator (thread =
//     position; warps split over the 32-lane quarters and 8-column chunks),
//     bias, residual, activation in float32, one rounding, and a store of each
//     valid position's value to NCHW y -- the output is written once.  With
//     two output staging buffers the epilogue works as two groups of eight
//     warps, one per accumulator, so two tiles are read out at once.
// Accumulators live in tensor memory, four of them when four channel tiles fit
// the 512 columns, else two (tile i in accumulator i % that), so a tile's
// epilogue overlaps the MMAs of the next ones; the producers run up to four
// tiles ahead (as deep as shared memory holds the ring).
// Every wait is bounded: after the limit the waiting thread flags the block
// and the device error word, every role drains out, outstanding copies and
// MMAs are waited for (bounded) and tensor memory is freed before exit.
//
// The weights reach shared memory in the layout the MMA reads ([k block of
// 8][output channel][8 k values], k in (tap, phase channel) order): the
// weight re-layout "Convolution, pooling and resize" measured at 1.27x on 3x3
// layers, done once per call by a small kernel into scratch; the conv kernel
// is launched as its programmatic dependent, so everything up to the first
// MMA overlaps it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "conv_internal.h"
#include "tc_ptx.cuh"

namespace conv {

__device__ uint32_t g_tcw_error;  // nonzero once a bounded wait gave up

namespace {

using namespace tcx;

constexpr int kEpiWarps = 16;  // warps 0-15: one or two groups, see epilogue_role
constexpr int kProdWarps = 6;  // warps 16-21
constexpr int kMmaWarp = kEpiWarps + kProdWarps;  // warps 22, 23 issue the MMAs of even, odd tiles
constexpr int kMmaWarps = 2;
constexpr int kThreads = (kMmaWarp + kMmaWarps) * 32;
constexpr int kEpi = kEpiWarps * 32;
constexpr int kProd = kProdWarps * 32;
constexpr uint32_t kProdBar = 2;  // named barrier of the producer warps
constexpr size_t kOneBlockPerSm = 116 * 1024;  // shared memory that keeps a second block off the SM

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t code,
                                           bool ignore_abort = false, uint32_t sleep_ns = 0) {
  return tcx::wait_phase(&g_tcw_error, bar, parity, abort_flag, code, ignore_abort, sleep_ns);
}

// True on every thread of named barrier `id` (`count` threads) iff `pred`
// holds on all of them; a barrier for those threads.
__device__ __forceinline__ bool group_all(uint32_t id, uint32_t count, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ bool producers_all(bool pred) { return group_all(kProdBar, kProd, pred); }
// named barriers of the epilogue groups: 1 and 3 (0 is __syncthreads, 2 the producers')
__device__ __forceinline__ uint32_t epi_bar(int g) { return g ? 3u : 1u; }

struct WinLayout {
  uint32_t w_off, ring_off, stg_off, out_off, bias_off, tab_off, bar_off, slot_off, end;
};

__host__ __device__ inline uint32_t align128(uint32_t v) { return (v + 127u) / 128u * 128u; }

// Barriers (8 bytes each, from bar_off): weights, full[4], rel[4], tfull[4],
// tempty[4], drain, res[2], then one per band stage.  Tile i uses full and
// rel i % max(lookahead, 2) (lookahead 1, 2 or 4) and accumulator, tfull and
// tempty i % (2 or 4): the tiles of one barrier belong to one MMA warp and
// one epilogue group, in order.
constexpr int kMaxLookahead = 4;
constexpr int kMaxAcc = 4;  // accumulators in tensor memory: four when 4 x N columns fit, else two
constexpr int kBarFull = 1, kBarRel = kBarFull + kMaxLookahead, kBarTfull = kBarRel + kMaxLookahead;
constexpr int kBarTempty = kBarTfull + kMaxAcc, kBarDrain = kBarTempty + kMaxAcc, kBarRes = kBarDrain + 1;
__host__ __device__ inline int tmem_accs(int nt) { return kMaxAcc * nt <= 512 ? kMaxAcc : 2; }
constexpr int kBarFixed = kBarRes + 2;

__host__ __device__ inline WinLayout win_layout(const WinPlan& p) {
  WinLayout L;
  L.w_off = 0;
  L.ring_off = align128(static_cast<uint32_t>(p.kblocks) * p.nt * 16u);
  L.stg_off = L.ring_off + align128(static_cast<uint32_t>(p.c16 / 8) * (p.ring + p.mirror) * 16u);
  L.out_off = L.stg_off + align128(static_cast<uint32_t>(p.stages) * p.band_bytes);
  L.bias_off = L.out_off + align128(static_cast<uint32_t>(p.ostages) * p.out_bytes);
  L.tab_off = L.bias_off + align128(static_cast<uint32_t>(p.nt) * 8u);  // bias: one copy per epilogue group
  L.bar_off = L.tab_off + align128(static_cast<uint32_t>(p.kblocks / 2) * 16u);  // one int4 per MMA
  L.slot_off = L.bar_off + static_cast<uint32_t>(kBarFixed + p.stages) * 8u;
  L.end = L.slot_off + 16u;
  return L;
}

// What the epilogue warps need besides the element type and the activation
// (copied from the launch arguments and the plan into registers).
struct EpiCtx {
  uint32_t tmem_base, bar0, out_s;  // tensor memory; barriers and output staging (shared addresses)
  uint8_t* out;                     // output staging and bias (shared memory)
  int t0, ntiles, co0;
  int tpi, rt, wp, wo, ho, nt, out_bytes, ostages;
  int groups;  // epilogue groups: 2 (group g reads out tiles g, g+2, ... into staging buffer g) or 1
  int accs;    // accumulators in tensor memory (tile i in accumulator i % accs)
  bool has_b, has_r;
  float alpha, beta;
  const void* bias;  // the layer's bias (has_b), staged into sbias first
  float* sbias_w;
  int c_out;
  volatile int* abort_flag;
  const CUtensorMap* ymap;
  const CUtensorMap* rmap;
};

// The epilogue warps' loop over the block's tiles, for activation ACT.  The
// sixteen warps form e.groups groups; group g reads out tiles g, g + groups,
// ... (with two groups, group g always meets accumulator g and staging buffer
// g).  Within a group, warp w reads tensor-memory lanes 32*(w%4) .. +31
// (thread = position of the tile) and every (warps per quarter)-th 8-column
// chunk, up to four chunks per tensor-memory wait; bias, residual and
// activation in float32, one rounding into the tile's staging buffer
// [channel][row][column]; then one TMA store of the box (wo x rows x channels)
// to y -- rows past Ho and channels past Cout fall outside y and are not
// written.  The residual tile arrives in the same buffer by TMA ahead of its
// tile.  Dropped positions (columns past Wo) are computed and not staged.
template <typename T, int ACT>
__device__ __forceinline__ void epilogue_role(const EpiCtx e) {
  const int gw = kEpiWarps / e.groups;  // warps per group
  const int gthreads = gw * 32;
  const int g = static_cast<int>(threadIdx.x) / gthreads;
  const int tid = static_cast<int>(threadIdx.x) - g * gthreads;  // thread within the group
  const int warp = tid >> 5, lane = tid & 31;
  const int nq = gw / 4;                    // warps per lane quarter
  const int qd = warp & 3, hf = warp >> 2;  // lane quarter, column group
  const uint32_t gbar = epi_bar(g);
  const int nchunks = e.nt / 8;
  const int plane = e.rt * e.wo;  // elements per channel in a staging buffer
  const int OS = e.ostages;
  float* sbias = e.sbias_w + g * e.nt;  // the group's copy of the bias
  auto res_bar = [&](int k) { return e.bar0 + 8u * (kBarRes + k); };
  auto issue_res = [&](int i) {  // group leader: the residual box of tile t0+i into buffer i % OS
    const int t = e.t0 + i, n = t / e.tpi, j = t - (t / e.tpi) * e.tpi;
    const int ob = i % OS;
    mbar_arrive_expect_tx(res_bar(ob), static_cast<uint32_t>(e.out_bytes));
    tma_load_4d(e.out_s + static_cast<uint32_t>(ob * e.out_bytes), e.rmap, 0, j * e.rt, e.co0, n, res_bar(ob));
  };
  if (e.has_r && tid == 0 && g < e.ntiles) issue_res(g);
  if (e.has_b) {  // ordered before its first use by the group's first tile barrier
    const T* bias = static_cast<const T*>(e.bias);
    for (int j = tid; j < e.nt; j += gthreads) sbias[j] = e.co0 + j < e.c_out ? to_f32<T>(bias[e.co0 + j]) : 0.0f;
  }
  // the thread's position in every tile
  const int qq = qd * 32 + lane;
  const int rr = qq / e.wp, c = qq - (qq / e.wp) * e.wp;
  const int soff2 = (rr * e.wo + c) * 2;
  for (int i = g; i < e.ntiles; i += e.groups) {
    const int t = e.t0 + i, n = t / e.tpi, j = t - (t / e.tpi) * e.tpi;
    const int b = i % e.accs, ob = i % OS;
    const uint32_t tfull = e.bar0 + 8u * (kBarTfull + b), tempty = e.bar0 + 8u * (kBarTempty + b);
    // accumulator ready, residual landed; the barrier also orders the staging
    // writes after the leader's wait for the store that last read the buffer
    // (without a residual that wait comes here, in the shadow of the MMAs,
    // rather than straight after the store)
    if (!e.has_r && tid == 0) {
      if (OS > e.groups) bulk_wait_read<1>();  // one group, two buffers: the store of tile i-2
      else bulk_wait_read<0>();                // the group's one buffer
    }
    bool okw = wait_phase(tfull, static_cast<uint32_t>(i / e.accs) & 1u, e.abort_flag, 2u, false, 64u);
    if (okw && e.has_r) okw = wait_phase(res_bar(ob), static_cast<uint32_t>(i / OS) & 1u, e.abort_flag, 128u);
    if (!group_all(gbar, gthreads, okw)) break;
    tc_fence_after();
    const int rows_here = min(e.rt, e.ho - j * e.rt);
    const bool valid = rr < rows_here && c < e.wo;
    T* st = reinterpret_cast<T*>(e.out + ob * e.out_bytes + soff2);
    const uint32_t tb = e.tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + static_cast<uint32_t>(b * e.nt);
    for (int k0 = hf; k0 < nchunks; k0 += 4 * nq) {
      uint32_t v[4][8];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (k0 + nq * q < nchunks) tmem_ld8_nowait(tb + (k0 + nq * q) * 8, v[q]);
      tmem_wait_ld();
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int k = k0 + nq * q;
          if (k >= nchunks) break;
          // the chunk's bias values are loaded before any of its stores: the
          // compiler cannot tell the staging stores from the bias copy
          T* dst = st + k * 8 * plane;
          float add[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) add[jj] = -0.0f;  // x + -0 == x for every x
          if (e.has_b) {
            const float4 b0 = *reinterpret_cast<const float4*>(sbias + k * 8);
            const float4 b1 = *reinterpret_cast<const float4*>(sbias + k * 8 + 4);
            add[0] = b0.x, add[1] = b0.y, add[2] = b0.z, add[3] = b0.w;
            add[4] = b1.x, add[5] = b1.y, add[6] = b1.z, add[7] = b1.w;
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            float x = __uint_as_float(v[q][jj]);
            x = __fadd_rn(x, add[jj]);
            if (e.has_r) x = __fadd_rn(x, to_f32<T>(dst[jj * plane]));
            dst[jj * plane] = from_f32<T>(act_fn<ACT>(x, e.alpha, e.beta));
          }
        }
      }
    }
    tc_fence_before();
    mbar_arrive(tempty);
    fence_proxy_async();  // the staged tile is visible to the TMA store
    named_sync(gbar, gthreads);
    if (tid == 0) {
      tma_store_4d(e.ymap, e.out_s + static_cast<uint32_t>(ob * e.out_bytes), 0, j * e.rt, e.co0, n);
      bulk_commit();
      if (e.has_r) {  // the next residual tile of this buffer goes in as soon as the store has read it
        if (OS > e.groups) bulk_wait_read<1>();
        else bulk_wait_read<0>();
        if (i + e.groups < e.ntiles) issue_res(i + e.groups);
      }
    }
  }
  if (tid == 0) bulk_wait_all();  // the stores have landed before the block retires
}

// One kernel per (element type, phase split, activation): each carries only
// its own epilogue, which keeps the code the warps run close together.
template <typename T, int PH, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    igemm_tcw(const ConvArgs a, const WinPlan p, const uint8_t* __restrict__ wpack,
              const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
              const __grid_constant__ CUtensorMap rmap) {
  extern __shared__ uint8_t sm_raw[];
  if (threadIdx.x == kEpi)  // the input's tensor map is fetched while every warp runs its prologue
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
  uint8_t* sm = sm_raw + ((128u - (smem_u32(sm_raw) & 127u)) & 127u);  // the launch adds 128 bytes of slack
  const WinLayout L = win_layout(p);
  const uint32_t bar0 = smem_u32(sm + L.bar_off);
  auto full_bar = [&](int k) { return bar0 + 8u * (kBarFull + k); };     // tile's input rows are in the ring
  auto rel_bar = [&](int k) { return bar0 + 8u * (kBarRel + k); };       // tile's MMAs done: ring reusable
  auto tfull_bar = [&](int b) { return bar0 + 8u * (kBarTfull + b); };   // accumulator b ready
  auto tempty_bar = [&](int b) { return bar0 + 8u * (kBarTempty + b); }; // accumulator b read out
  const uint32_t wbar = bar0;  // the raw weight copy landed
  const uint32_t drain_bar = bar0 + 8u * kBarDrain;
  auto res_bar = [&](int k) { return bar0 + 8u * (kBarRes + k); };       // residual tile k landed
  auto sfull_bar = [&](int s) { return bar0 + 8u * (kBarFixed + s); };  // staged band s landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L.slot_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L.slot_off + 4);
  float* sbias = reinterpret_cast<float*>(sm + L.bias_off);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int ct = static_cast<int>(blockIdx.x) % p.co_tiles;
  const int part = static_cast<int>(blockIdx.x) / p.co_tiles;
  // the block's tiles: tq each, one more for the first tr blocks (no division
  // here: every warp runs this before its role)
  const int t0 = part * p.tq + min(part, p.tr);
  const int ntiles = p.tq + (part < p.tr ? 1 : 0);
  const int co0 = ct * p.nt;
  const int TA = tmem_accs(p.nt);
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(TA * p.nt)) cols <<= 1;
  // tile t: rows j*rt .. of image n (t = n*tpi + j); its first position
  auto tile_q0 = [&](int t) {
    const int n = t / p.tpi, j = t - (t / p.tpi) * p.tpi;
    return (n * p.hp + j * p.rt) * p.wp;
  };

  // ---- producers' band state.  Their first bands are requested first thing,
  // before the rest of the set-up and the weights, so the input's trip from
  // memory overlaps all of it: lane 0 of the first producer warp sets up the
  // band barriers itself and issues the copies.
  const int ptid = tid - kEpi;
  const int pw = ptid >> 5;
  const int DS = p.stages, SB = p.band, LA = p.lookahead, NB = LA < 2 ? 2 : LA;
  auto row_end = [&](int i) {  // padded rows (exclusive) the valid outputs of tile t0+i read
    const int t = t0 + i, n = t / p.tpi, j = t - (t / p.tpi) * p.tpi;
    return n * p.hp + min((j + 1) * p.rt, p.ho) + (p.khp - 1) * a.dh;
  };
  // (the divisions below run on the producer warps only)
  const bool producer = warp >= kEpiWarps && warp < kMmaWarp;
  int rho0 = 0, rho_end = 0;
  const uint32_t stg_s = smem_u32(sm + L.stg_off);
  // bands: rows [b*SB, min((b+1)*SB, hp)) of one image; the next band to
  // load is (ni, bi), the band being consumed is (nf, bf)
  int ni = 0, bi = 0;
  if (producer) {
    const int n0 = t0 / p.tpi, j0 = t0 - n0 * p.tpi;  // first tile: image n0, rows j0*rt ..
    rho0 = n0 * p.hp + j0 * p.rt;
    rho_end = ntiles > 0 ? row_end(ntiles - 1) : rho0;
    ni = n0;
    bi = j0 * p.rt / SB;
  }
  int nf = ni, bf = bi;
  int k_issue = 0, k_fill = 0;
  auto band_row0 = [&](int n, int b) { return n * p.hp + b * SB; };
  // one TMA box per band: vw columns x PH*SB input rows x cg channels of image n
  auto issue = [&]() {
    const int s = k_issue % DS;
    if (lane == 0) {
      mbar_arrive_expect_tx(sfull_bar(s), static_cast<uint32_t>(p.band_bytes));
      tma_load_4d(stg_s + static_cast<uint32_t>(s) * p.band_bytes, &xmap, 0, PH * bi * SB - a.pt, 0, ni,
                  sfull_bar(s));
    }
    __syncwarp();
    if (++bi * SB >= p.hp) { bi = 0; ++ni; }
    ++k_issue;
  };
  if (warp == kEpiWarps) {
    if (lane == 0) {
      for (int st = 0; st < DS; ++st) mbar_init(sfull_bar(st), 1);
      asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncwarp();
    for (int k = 0; k < DS && band_row0(ni, bi) < rho_end; ++k) issue();
  }

  // ---- set-up: barriers, bias, MMA table, tensor memory --------------------
  const int epi_groups = p.ostages == 2 ? 2 : 1;
  if (tid == 0) {
    for (int k = 0; k < kMaxLookahead; ++k) {
      mbar_init(full_bar(k), kProd);
      mbar_init(rel_bar(k), 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), kEpi / epi_groups);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(res_bar(i), 1);
    }
    mbar_init(drain_bar, kMmaWarps);
    mbar_init(wbar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), cols);
    // per MMA of a tile: the window shift of its tap, the k-block offset of
    // its channel pair in the ring, and its weights' offset (16-byte units)
    int4* tab = reinterpret_cast<int4*>(sm + L.tab_off);
    const int pairs = p.c16 / 16, nmma = p.kblocks / 2;
    for (int e = lane; e < nmma; e += 32) {
      const int tap = e / pairs, m = e - (e / pairs) * pairs;
      const int u = tap / p.kwp, v = tap - (tap / p.kwp) * p.kwp;
      tab[e] = make_int4(u * a.dh * p.wp + v * a.dw, 2 * m * (p.ring + p.mirror), (2 * e) * p.nt, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < kEpiWarps) {
    // ---- epilogue
    EpiCtx e;
    e.tmem_base = tmem_base;
    e.bar0 = bar0;
    e.out_s = smem_u32(sm + L.out_off);
    e.out = sm + L.out_off;
    e.t0 = t0;
    e.ntiles = ntiles;
    e.co0 = co0;
    e.tpi = p.tpi;
    e.rt = p.rt;
    e.wp = p.wp;
    e.wo = p.wo;
    e.ho = p.ho;
    e.nt = p.nt;
    e.out_bytes = p.out_bytes;
    e.ostages = p.ostages;
    e.groups = epi_groups;
    e.accs = TA;
    e.has_b = a.bias != nullptr;
    e.has_r = a.residual != nullptr;
    e.alpha = a.alpha;
    e.beta = a.beta;
    e.bias = a.bias;
    e.sbias_w = sbias;
    e.c_out = a.c_out;
    e.abort_flag = abort_flag;
    e.ymap = &ymap;
    e.rmap = &rmap;
    epilogue_role<T, ACT>(e);
  } else if (warp < kEpiWarps + kProdWarps) {
    // ---- producers: bands of input rows by TMA, channels interleaved into the ring
    const int nb = p.c16 / 8;
    const int R = p.ring, RM = p.ring + p.mirror;
    uint8_t* ring = sm + L.ring_off;
    int filled = rho0;  // rows below this are in the ring
    // the thread's next unit is kProd units on: step_br rows, step_cb blocks, step_c columns
    const int cstride = PH * SB * p.vw;  // one staged channel
    const int step_br = kProd / (p.wp * nb);
    const int step_cb = (kProd % (p.wp * nb)) / p.wp, step_c = kProd % p.wp;
    bool ok = true;
    for (int i = 0; ok && i < ntiles; ++i) {
      if (i >= LA) {
        const int j = i - LA;
        ok = producers_all(wait_phase(rel_bar(j % NB), static_cast<uint32_t>(j / NB) & 1u, abort_flag, 4u));
        if (!ok) break;
      }
      const int re = row_end(i);
      while (filled < re) {
        // the whole band (nf, bf) from row `filled` on
        const int s = k_fill % DS;
        ok = producers_all(wait_phase(sfull_bar(s), static_cast<uint32_t>(k_fill / DS) & 1u, abort_flag, 8u));
        if (!ok) break;
        const int brow0 = band_row0(nf, bf);
        const int blen = min(SB, p.hp - bf * SB);
        const int first = filled - brow0;  // rows of the band already in the ring (first band only)
        const uint16_t* sg = reinterpret_cast<const uint16_t*>(sm + L.stg_off + static_cast<uint32_t>(s) * p.band_bytes);
        const int rows = blen - first;
        const int units = rows * p.wp * nb;  // (row, channel block, column)
        const int per_row = p.wp * nb;
        const int base_slot = static_cast<int>((static_cast<long long>(brow0) * p.wp) % R);
        bool vec_done = false;
        if constexpr (PH == 1) {
          if ((a.cg & 7) == 0) {
            // whole 8-channel blocks: 4 staged columns of 8 channels at a time
            // (eight 8-byte reads, a register transpose, four 16-byte
            // writes), then the padding columns as zeros
            vec_done = true;
            const int nq = p.vw / 4;  // 4-column chunks of a staged row
            const int vunits = rows * nb * nq;
            for (int e = ptid; e < vunits; e += kProd) {
              const int q4 = e % nq, t1 = e / nq;
              const int cbv = t1 % nb, brv = first + t1 / nb;
              uint32_t o[4][4];  // o[i]: column i's channels (0,1) (2,3) (4,5) (6,7), low half the even one
              if (cbv * 8 < a.cg) {
                const uint16_t* src = sg + (static_cast<size_t>(cbv) * 8 * SB + brv) * p.vw + 4 * q4;
                uint2 r[8];  // r[j]: channel j, columns (0,1) and (2,3)
#pragma unroll
                for (int j = 0; j < 8; ++j) r[j] = *reinterpret_cast<const uint2*>(src + static_cast<size_t>(j) * cstride);
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {
                  o[0][pr] = __byte_perm(r[2 * pr].x, r[2 * pr + 1].x, 0x5410);
                  o[1][pr] = __byte_perm(r[2 * pr].x, r[2 * pr + 1].x, 0x7632);
                  o[2][pr] = __byte_perm(r[2 * pr].y, r[2 * pr + 1].y, 0x5410);
                  o[3][pr] = __byte_perm(r[2 * pr].y, r[2 * pr + 1].y, 0x7632);
                }
              } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                  for (int pr = 0; pr < 4; ++pr) o[i][pr] = 0u;
              }
              int slot = base_slot + brv * p.wp + a.pl + 4 * q4;  // < 2R: R exceeds a band's positions
              if (slot >= R) slot -= R;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint4 u4 = make_uint4(o[i][0], o[i][1], o[i][2], o[i][3]);
                uint8_t* dst = ring + (static_cast<size_t>(cbv) * RM + slot) * 16u;
                *reinterpret_cast<uint4*>(dst) = u4;
                if (slot < p.mirror) *reinterpret_cast<uint4*>(dst + static_cast<size_t>(R) * 16u) = u4;
                if (++slot == R) slot = 0;
              }
            }
            const int pc = p.wp - p.vw;  // padding columns: [0, pl) and [pl + vw, wp)
            for (int e = ptid; e < rows * nb * pc; e += kProd) {
              const int q = e % pc, t1 = e / pc;
              const int cbv = t1 % nb, brv = first + t1 / nb;
              int slot = base_slot + brv * p.wp + (q < a.pl ? q : q + p.vw);
              if (slot >= R) slot -= R;
              uint8_t* dst = ring + (static_cast<size_t>(cbv) * RM + slot) * 16u;
              *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
              if (slot < p.mirror) *reinterpret_cast<uint4*>(dst + static_cast<size_t>(R) * 16u) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        int br = first + ptid / per_row, cb = (ptid % per_row) / p.wp, c = ptid % p.wp;
        for (int e = ptid; !vec_done && e < units; e += kProd) {
          // value j of the unit: channel cb*8 + j (PH 1), or channel
          // cb*2 + j/4, phase row (j/2)%2, phase column j%2 (PH 2); staged at
          // [channel][PH*SB rows][vw columns]
          uint16_t v[8];
          if constexpr (PH == 1) {
            const int wc = c - a.pl;
            const uint16_t* src = sg + (cb * 8 * SB + br) * p.vw + wc;
            const int nv = static_cast<unsigned>(wc) < static_cast<unsigned>(p.vw) ? min(8, a.cg - cb * 8) : 0;
            if (nv == 8) {
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = src[j * cstride];
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = j < nv ? src[j * cstride] : static_cast<uint16_t>(0);
            }
          } else {
            const int wc = 2 * c - a.pl;
            const uint16_t* src = sg + (cb * 2 * 2 * SB + 2 * br) * p.vw + wc;
            const bool ok0 = static_cast<unsigned>(wc) < static_cast<unsigned>(p.vw);
            const bool ok1 = static_cast<unsigned>(wc + 1) < static_cast<unsigned>(p.vw);
            const int nch = min(2, a.cg - cb * 2);  // real channels of the unit
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const bool okv = ((j & 1) ? ok1 : ok0) && (j >> 2) < nch;
              v[j] = okv ? src[(j >> 2) * cstride + ((j >> 1) & 1) * p.vw + (j & 1)] : static_cast<uint16_t>(0);
            }
          }
          int slot = base_slot + br * p.wp + c;  // < 2R: R exceeds a band's positions
          if (slot >= R) slot -= R;
          const uint4 u4 = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
          uint8_t* dst = ring + (static_cast<size_t>(cb) * RM + slot) * 16u;
          *reinterpret_cast<uint4*>(dst) = u4;
          if (slot < p.mirror) *reinterpret_cast<uint4*>(dst + static_cast<size_t>(R) * 16u) = u4;
          c += step_c;
          cb += step_cb;
          br += step_br;
          if (c >= p.wp) { c -= p.wp; ++cb; }
          if (cb >= nb) { cb -= nb; ++br; }
        }
        named_sync(kProdBar, kProd);  // the staged band is consumed: its slot may be refilled
        if (pw == 0 && band_row0(ni, bi) < rho_end) {
          fence_proxy_async();
          issue();
        }
        filled = brow0 + blen;
        if (++bf * SB >= p.hp) { bf = 0; ++nf; }
        ++k_fill;
      }
      if (!ok) break;
      fence_proxy_async();  // ring writes visible to the tensor cores
      mbar_arrive(full_bar(i % NB));
    }
    if (pw == 0) {  // copies still in flight land before the block retires
      for (int k = k_fill; k < k_issue; ++k)
        wait_phase(sfull_bar(k % DS), static_cast<uint32_t>(k / DS) & 1u, abort_flag, 8u, true);
    }
  } else if (ntiles > 0) {
    // ---- MMA issuers: warp kMmaWarp + mw takes tiles mw, mw + 2, ...; the whole
    // warp runs the loop, one elected lane issues
    const int mw = warp - kMmaWarp;
    if (mw == 0) {
      // the packed weights come from the repack kernel launched just before
      // this one (programmatic dependent launch: everything above overlapped it)
      asm volatile("griddepcontrol.wait;\n" ::: "memory");
      const uint32_t wbytes = static_cast<uint32_t>(p.kblocks) * p.nt * 16u;
      if (lane == 0) {
        mbar_arrive_expect_tx(wbar, wbytes);
        bulk_load(smem_u32(sm + L.w_off), wpack + static_cast<size_t>(ct) * wbytes, wbytes, wbar);
      }
      __syncwarp();
    }
    bool ok = __all_sync(0xffffffffu, wait_phase(wbar, 0, abort_flag, 1u));
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t idesc = make_idesc(kBf16, p.nt);
    const int R = p.ring, RM = p.ring + p.mirror;
    // descriptors of the ring's and the weights' first core matrices; every
    // operand is one of them advanced by a whole number of 16-byte units
    // (the start-address field holds addr >> 4 and never carries out)
    const uint64_t ad0 = kmajor_desc(smem_u32(sm + L.ring_off), static_cast<uint32_t>(RM) * 16u, 128u);
    const uint64_t bd0 = kmajor_desc(smem_u32(sm + L.w_off), static_cast<uint32_t>(p.nt) * 16u, 128u);
    const int4* tab = reinterpret_cast<const int4*>(sm + L.tab_off);
    const int nmma = p.kblocks / 2;
    for (int i = mw; ok && i < ntiles; i += kMmaWarps) {
      const int b = i % TA;
      ok = __all_sync(0xffffffffu, wait_phase(tempty_bar(b), (static_cast<uint32_t>(i / TA) & 1u) ^ 1u, abort_flag, 16u));
      if (!ok) break;
      ok = __all_sync(0xffffffffu, wait_phase(full_bar(i % NB), static_cast<uint32_t>(i / NB) & 1u, abort_flag, 32u));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tmem_base + static_cast<uint32_t>(b * p.nt);
      const int pbase = tile_q0(t0 + i) % R;
#pragma unroll 4
      for (int e = 0; e < nmma; ++e) {
        const int4 tv = tab[e];
        int pos = pbase + tv.x;
        if (pos >= R) pos -= R;
        mma_f16_elect(d, ad0 + static_cast<uint64_t>(pos + tv.y), bd0 + static_cast<uint64_t>(tv.z), idesc,
                      e > 0 ? 1u : 0u);
      }
      mma_commit_elect(rel_bar(i % NB));
      mma_commit_elect(tfull_bar(b));
    }
  }

  // ---- teardown ----------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp >= kMmaWarp) {
    if (*abort_flag) {
      // outstanding MMAs of both issuing warps finish before their tensor
      // memory is freed
      mma_commit_elect(drain_bar);
      if (warp == kMmaWarp) {
        wait_phase(drain_bar, 0, abort_flag, 64u, true);
        if (ntiles > 0) wait_phase(wbar, 0, abort_flag, 1u, true);  // the weight copy has landed
      }
    }
    __syncwarp();
    if (warp == kMmaWarp) tmem_dealloc(tmem_base, cols);
  }
}

// Weights OIHW -> [channel tile][k block][output channel][8 k values], k in
// (tap, phase channel) order, zero for phantom channels, taps past the kernel
// and output channels past c_out.
template <int PH>
__global__ void tcw_repack(const ConvArgs a, const WinPlan p, uint4* __restrict__ out) {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");  // the conv kernel may start now
  const uint16_t* w = static_cast<const uint16_t*>(a.wt);
  const int nb = p.c16 / 8;
  const long long units = static_cast<long long>(p.co_tiles) * p.kblocks * p.nt;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < units;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int col = static_cast<int>(e % p.nt);
    const long long rest = e / p.nt;
    const int kb = static_cast<int>(rest % p.kblocks);
    const int ct = static_cast<int>(rest / p.kblocks);
    const int co = ct * p.nt + col;
    const int tap = kb / nb, cb = kb - (kb / nb) * nb;
    const int u0 = tap / p.kwp, v0 = tap - (tap / p.kwp) * p.kwp;
    uint16_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = cb * 8 + j;
      const int ch = k / (PH * PH), ph = (k / PH) % PH, pb = k % PH;
      const int u = u0 * PH + ph, vv = v0 * PH + pb;
      const bool ok = co < a.c_out && ch < a.cg && u < a.kh && vv < a.kw;
      v[j] = ok ? w[((static_cast<long long>(co) * a.cg + ch) * a.kh + u) * a.kw + vv] : static_cast<uint16_t>(0);
    }
    out[e] = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
  }
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// A 4-d tensor map over an NCHW array viewed as (cols, rows, channels, n),
// boxes of (box_cols, box_rows, box_ch, 1), zeros outside.
template <typename T>
bool encode_nchw(CUtensorMap* map, const void* base, int cols, int rows, int ch, int n, int box_cols, int box_rows,
                 int box_ch) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(ch), static_cast<cuuint64_t>(n)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(cols) * 2, static_cast<cuuint64_t>(cols) * rows * 2,
                                 static_cast<cuuint64_t>(cols) * rows * ch * 2};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_ch), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      std::is_same<T, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return encode(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int PH>
cudaError_t launch_win(const WinPlan& p, const ConvArgs& a, void* scratch, cudaStream_t s) {
  // x: one box = a band of every channel; y and the residual: one box = a tile
  CUtensorMap xmap, ymap, rmap;
  if (!encode_nchw<T>(&xmap, a.x, p.vw, p.vh, a.c_in, a.n, p.vw, PH * p.band, a.cg) ||
      !encode_nchw<T>(&ymap, a.y, p.wo, p.ho, a.c_out, a.n, p.wo, p.rt, p.nt))
    return cudaErrorInvalidValue;
  rmap = ymap;
  if (a.residual && !encode_nchw<T>(&rmap, a.residual, p.wo, p.ho, a.c_out, a.n, p.wo, p.rt, p.nt))
    return cudaErrorInvalidValue;
  auto kern = igemm_tcw<T, PH, ACT_IDENTITY>;
  switch (a.act) {
#define CONV_TCW_CASE(A)           \
  case A:                          \
    kern = igemm_tcw<T, PH, A>;    \
    break;
    CONV_TCW_CASE(ACT_RELU)
    CONV_TCW_CASE(ACT_SILU)
    CONV_TCW_CASE(ACT_SIGMOID)
    CONV_TCW_CASE(ACT_TANH)
    CONV_TCW_CASE(ACT_HARD_SWISH)
    CONV_TCW_CASE(ACT_HARD_SIGMOID)
    CONV_TCW_CASE(ACT_CLIP)
    CONV_TCW_CASE(ACT_LEAKY_RELU)
#undef CONV_TCW_CASE
    default:
      break;
  }
  auto repack = tcw_repack<PH>;
  cudaError_t err = opt_in_smem(reinterpret_cast<const void*>(kern), p.smem);
  if (err != cudaSuccess) return err;
  const long long units = static_cast<long long>(p.co_tiles) * p.kblocks * p.nt;
  const int rblocks = static_cast<int>(std::min<long long>((units + 255) / 256, 1024));
  repack<<<rblocks, 256, 0, s>>>(a, p, static_cast<uint4*>(scratch));
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // programmatic dependent launch: the conv kernel's set-up and input staging
  // overlap the repack; its MMA warp waits for the repack's completion
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, p, static_cast<const uint8_t*>(scratch), xmap, ymap, rmap);
}

// Channel tile, lookahead, output buffers, band height and band stages that
// fit shared memory for the geometry already in `p` (two output buffers
// first -- the epilogue's two groups are worth more than lookahead or the
// widest tile -- then the widest tile, deepest lookahead, bands of about
// 8 KB, most bands in flight), with the ring depth each choice needs.  False
// if none fits.
bool fit_smem(const ConvArgs& a, WinPlan* p) {
  const long long row_bytes = static_cast<long long>(p->vw) * p->ph * a.cg * 2;  // one padded row's box
  const int sb_max = static_cast<int>(std::min<long long>({8, p->hp, 256 / p->ph}));
  int sb_pref = 1;
  while (sb_pref < sb_max && row_bytes * sb_pref < 8192) ++sb_pref;
  const int nt0 = static_cast<int>(std::min<long long>((a.c_out + 15) / 16 * 16, 256));
  // first pass: two output buffers (two epilogue groups) with a channel tile
  // of 64 or more, at any lookahead; then anything that fits
  for (int pass = 0; pass < 2; ++pass) {
    for (int nt = nt0; nt >= 16; nt = nt > 16 ? std::max(16, (nt / 2 + 15) / 16 * 16) : 0) {
      p->nt = nt;
      p->co_tiles = (a.c_out + nt - 1) / nt;
      p->out_bytes = nt * p->rt * p->wo * 2;
      // (lookahead, output buffers): deeper lookahead first, but two output
      // buffers (two epilogue groups) before a lookahead past two, and a
      // lookahead past two only with full bands and stages
      static const int kChoice[][2] = {{4, 2}, {2, 2}, {2, 1}, {1, 2}, {1, 1}};
      for (const auto& choice : kChoice) {
        const int la = choice[0], os = choice[1];
        if (pass == 0 && (os != 2 || nt < 64)) continue;
        for (int sb = sb_pref; sb >= 1; --sb) {
          if (row_bytes * sb >= (1 << 20)) continue;  // transaction count of one mbarrier phase
          for (int ds = 4; ds >= 2; --ds) {
            if (la > 2 && (sb != sb_pref || ds != 4)) continue;
            // rows the producers may write beyond the oldest window still in
            // use: la tiles of rt rows (one of them across an image's dropped
            // rows), the kernel's reach and a band
            const long long rows = static_cast<long long>(la - 1) * (p->rt + p->hp - p->ho) + p->rt +
                                   static_cast<long long>(p->khp - 1) * a.dh + sb;
            const long long ring = (rows * p->wp + 7) / 8 * 8;
            if (ring + 128 > 16000) continue;  // the descriptors' 14-bit offsets
            p->ring = static_cast<int>(ring);
            p->mirror = 128;  // windows start anywhere: 128 slots written twice
            p->lookahead = la;
            p->ostages = os;
            p->band = sb;
            p->band_bytes = static_cast<int>(row_bytes * sb);
            p->stages = ds;
            if (win_layout(*p).end + 128 <= kTcMaxSmem) return true;
          }
        }
      }
    }
  }
  return false;
}

// Everything of the plan that follows from the view (vh, vw, ho, wo) and the
// phase split: padded plane, rows per tile, channels, shifts, tiles.  False
// if a size is past the kernel's limits or nothing fits shared memory.
bool plan_view(const ConvArgs& a, WinPlan* p) {
  if (p->vw > 256 || a.cg > 256 || p->wo % 8 != 0) return false;  // TMA boxes: rows of 16-byte multiples
  p->khp = (a.kh + p->ph - 1) / p->ph;
  p->kwp = (a.kw + p->ph - 1) / p->ph;
  const long long hp = p->ho + static_cast<long long>(p->khp - 1) * a.dh;
  const long long wp = p->wo + static_cast<long long>(p->kwp - 1) * a.dw;
  if (wp > 128 || hp > 65535) return false;  // a tile holds whole padded rows
  p->hp = static_cast<int>(hp);
  p->wp = static_cast<int>(wp);
  p->rt = 128 / p->wp;
  if (p->rt > 256) p->rt = 256;
  p->tpi = (p->ho + p->rt - 1) / p->rt;
  const long long cgp = static_cast<long long>(a.cg) * p->ph * p->ph;
  if (cgp > 512) return false;
  p->c16 = static_cast<int>((cgp + 15) / 16 * 16);
  p->hq = static_cast<int>(static_cast<long long>(p->khp - 1) * a.dh * wp + static_cast<long long>(p->kwp - 1) * a.dw);
  const long long npos = static_cast<long long>(a.n) * hp * wp;
  if (npos + 1024 + p->hq + 16 * wp > (1LL << 30)) return false;
  const long long tiles = static_cast<long long>(a.n) * p->tpi;
  if (tiles > (1LL << 30)) return false;
  p->tiles = static_cast<int>(tiles);
  p->kblocks = p->khp * p->kwp * p->c16 / 8;
  return fit_smem(a, p);
}

}  // namespace

// Planner (host): whether the shifted-window kernel takes the shape, and its
// geometry, channel tile, ring and staging depth.  Addresses are not known
// here; the launch checks them.
bool tcw_plan(const ConvArgs& a, int sm, WinPlan* out) {
  if (a.groups != 1) return false;
  WinPlan p;
  memset(&p, 0, sizeof(p));
  if (a.sh == 1 && a.sw == 1) p.ph = 1;
  else if (a.sh == 2 && a.sw == 2 && a.dh == 1 && a.dw == 1) p.ph = 2;
  else return false;
  const bool pointwise = a.kh == 1 && a.kw == 1 && p.ph == 1 && a.pt == 0 && a.pl == 0 && a.ho == a.h &&
                         a.wo == a.w;
  bool ok = false;
  if (pointwise) {
    // a 1x1 layer reads each plane as it lies: view it as rows of vw
    // positions (a multiple of 8 dividing h*w, for 16-byte rows), the view
    // whose tiles use most of the 128 MMA rows, longer rows first
    int best = 0;
    double best_eff = 0.0;
    for (long long l = std::min<long long>(128, a.hw) / 8 * 8; l >= 8; l -= 8) {
      if (a.hw % l) continue;
      const double eff = static_cast<double>((128 / l) * l) / 128.0;
      if (eff > best_eff + 1e-9) { best_eff = eff; best = static_cast<int>(l); }
    }
    for (int pass = 0; pass < 2 && !ok && best; ++pass) {
      for (long long l = best; l >= 8 && !ok; l -= 8) {
        if (a.hw % l) continue;
        if (pass == 0 && l != best) continue;
        p.vw = static_cast<int>(l);
        p.vh = static_cast<int>(a.hw / l);
        p.ho = p.vh;
        p.wo = p.vw;
        ok = plan_view(a, &p);
      }
    }
  } else if (a.w % 8 == 0) {  // x rows start on 16 bytes
    p.vh = a.h;
    p.vw = a.w;
    p.ho = a.ho;
    p.wo = a.wo;
    ok = plan_view(a, &p);
  }
  if (!ok) return false;
  p.parts = static_cast<int>(std::min<long long>(p.tiles, std::max(1, sm / p.co_tiles)));
  p.tq = p.tiles / p.parts;
  p.tr = p.tiles % p.parts;
  p.ctas = p.parts * p.co_tiles;
  p.w_bytes = static_cast<size_t>(p.co_tiles) * p.kblocks * p.nt * 16;
  p.smem = std::max<size_t>(win_layout(p).end + 128, kOneBlockPerSm);
  *out = p;
  return true;
}

cudaError_t launch_tcw(const Plan& plan, const ConvArgs& a, int dtype, void* scratch, cudaStream_t s) {
  const WinPlan& p = plan.tcw;
  if (dtype == CONV_F16)
    return p.ph == 2 ? launch_win<__half, 2>(p, a, scratch, s) : launch_win<__half, 1>(p, a, scratch, s);
  if (dtype == CONV_BF16)
    return p.ph == 2 ? launch_win<__nv_bfloat16, 2>(p, a, scratch, s)
                     : launch_win<__nv_bfloat16, 1>(p, a, scratch, s);
  return cudaErrorInvalidValue;
}

// ---- the bounded-wait abort path, run on its own --------------------------
//
// The shifted-window kernel's give-up path (a wait that runs out raises the
// block's abort flag and ORs its code into g_tcw_error; the other roles see the
// flag and stop; the copies still in flight are waited for; tensor memory is
// freed) only runs when a partner role stops, which never happens in a correct
// launch.  This kernel walks the same steps with the same wait helper on a
// block where nothing else can be outstanding: warp 0 allocates 32 columns of
// tensor memory; thread 0 starts one 256-byte bulk copy into shared memory;
// all 64 threads wait, with a short limit, on an mbarrier nothing arrives on;
// the copy is then drained (its own wait ignores the abort flag, with the
// usual limit), written back out, and the tensor memory freed.
constexpr uint32_t kSelftestWaitCode = 256u;   // the withheld arrival's wait ran out
constexpr uint32_t kSelftestDrainCode = 512u;  // the drain of the copy ran out

__global__ void __launch_bounds__(64) tcw_wait_selftest(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                        unsigned long long limit_ns, uint32_t* __restrict__ report) {
  __shared__ __align__(128) uint4 buf[16];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x / 32;
  const uint32_t never = smem_u32(&bars[0]), copied = smem_u32(&bars[1]);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(never, 1);
    mbar_init(copied, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(copied, sizeof(buf));
    bulk_load(smem_u32(buf), src, sizeof(buf), copied);
  }
  const bool got = tcx::wait_phase(&g_tcw_error, never, 0, &abort_flag, kSelftestWaitCode, false, 0, limit_ns);
  if (got) atomicAdd(&report[0], 1u);
  const bool drained = tcx::wait_phase(&g_tcw_error, copied, 0, &abort_flag, kSelftestDrainCode, true);
  if (drained) atomicAdd(&report[1], 1u);
  __syncthreads();
  if (threadIdx.x == 0) report[2] = static_cast<uint32_t>(abort_flag);
  if (drained && threadIdx.x < 16) dst[threadIdx.x] = buf[threadIdx.x];
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_base, 32);
  if (threadIdx.x == 0) report[3] = 1;  // reached the end
}

cudaError_t tcw_wait_selftest_run(unsigned long long limit_ns, uint32_t* report_host) {
  // device: 256 bytes source, 256 bytes destination, 4 report words
  void* mem = nullptr;
  cudaError_t err = cudaMalloc(&mem, 512 + 4 * sizeof(uint32_t));
  if (err != cudaSuccess) return err;
  uint4* src = static_cast<uint4*>(mem);
  uint4* dst = src + 16;
  uint32_t* report = reinterpret_cast<uint32_t*>(dst + 16);
  uint32_t pattern[64];
  for (uint32_t i = 0; i < 64; ++i) pattern[i] = 0x9e3779b9u * (i + 1);
  err = cudaMemcpy(src, pattern, sizeof(pattern), cudaMemcpyHostToDevice);
  if (err == cudaSuccess) err = cudaMemset(dst, 0, 256 + 4 * sizeof(uint32_t));
  if (err == cudaSuccess) {
    tcw_wait_selftest<<<1, 64>>>(src, dst, limit_ns, report);
    err = cudaGetLastError();
  }
  if (err == cudaSuccess) err = cudaDeviceSynchronize();
  uint32_t back[64 + 4];
  if (err == cudaSuccess) err = cudaMemcpy(back, dst, sizeof(back), cudaMemcpyDeviceToHost);
  if (err == cudaSuccess) {
    for (int i = 0; i < 4; ++i) report_host[i] = back[64 + i];
    report_host[4] = memcmp(back, pattern, sizeof(pattern)) == 0 ? 1u : 0u;
  }
  const cudaError_t ferr = cudaFree(mem);
  return err != cudaSuccess ? err : ferr;
}

cudaError_t tcw_error_word(uint32_t* word, int reset) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  err = cudaMemcpyFromSymbol(word, g_tcw_error, sizeof(uint32_t));
  if (err != cudaSuccess || !reset) return err;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_tcw_error, &zero, sizeof(uint32_t));
}

}  // namespace conv
