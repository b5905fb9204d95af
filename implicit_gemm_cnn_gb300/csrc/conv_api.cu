// conv_api.cu -- the C ABI of libconv: validation, planning and dispatch.
//
// "Convolution, pooling and resize" (Layout and operands; Variants; split k)
// describes the host side this follows: a problem struct carrying the shape,
// explicit pads, dilation, groups and the fused activation; sizes checked with
// checked arithmetic and the device's limits before anything is recorded; a
// scratch query; a variant chosen from the problem and the device; a k split
// that depends only on the shape; an error for scratch that overlaps an
// operand.  Everything here runs on the host; conv_forward only enqueues.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "conv_internal.h"


using namespace conv;

namespace {

constexpr long long kI32 = 2147483647LL;
constexpr int kMaxDevices = 64;
constexpr size_t kMaxDynSmem = 232448;  // 227 KB per block on sm_100-class devices

bool mul_ok(long long a, long long b, long long* out) {
  return !__builtin_mul_overflow(a, b, out);
}

struct Shape {
  long long ho, wo, cg, mg, K, npix, x_elems, w_elems, y_elems;
};

conv_status validate(const conv_problem* p, Shape* s) {
  if (!p) return CONV_ERR_NULL;
  if (p->dtype < CONV_F32 || p->dtype > CONV_BF16) return CONV_ERR_DTYPE;
  if (p->act < CONV_ACT_IDENTITY || p->act > CONV_ACT_LEAKY_RELU) return CONV_ERR_ACT;
  const long long pos[] = {p->n, p->c_in, p->h, p->w, p->c_out, p->kh, p->kw,
                           p->stride_h, p->stride_w, p->dil_h, p->dil_w, p->groups};
  for (long long v : pos)
    if (v < 1) return CONV_ERR_SHAPE;
  if (p->pad_top < 0 || p->pad_left < 0 || p->pad_bottom < 0 || p->pad_right < 0) return CONV_ERR_SHAPE;
  if (p->c_in % p->groups || p->c_out % p->groups) return CONV_ERR_SHAPE;
  long long span_h, span_w, ext_h, ext_w;
  if (!mul_ok(p->dil_h, p->kh - 1, &span_h) || !mul_ok(p->dil_w, p->kw - 1, &span_w))
    return CONV_ERR_OVERFLOW;
  if (__builtin_add_overflow(p->h, p->pad_top, &ext_h) || __builtin_add_overflow(ext_h, p->pad_bottom, &ext_h) ||
      __builtin_add_overflow(p->w, p->pad_left, &ext_w) || __builtin_add_overflow(ext_w, p->pad_right, &ext_w))
    return CONV_ERR_OVERFLOW;
  if (ext_h - 1 < span_h || ext_w - 1 < span_w) return CONV_ERR_SHAPE;  // no output position
  s->ho = (ext_h - span_h - 1) / p->stride_h + 1;
  s->wo = (ext_w - span_w - 1) / p->stride_w + 1;
  s->cg = p->c_in / p->groups;
  s->mg = p->c_out / p->groups;
  long long t;
  if (!mul_ok(s->cg, p->kh, &t) || !mul_ok(t, p->kw, &s->K)) return CONV_ERR_OVERFLOW;
  if (!mul_ok(p->n, s->ho, &t) || !mul_ok(t, s->wo, &s->npix)) return CONV_ERR_OVERFLOW;
  if (!mul_ok(p->n, p->c_in, &t) || !mul_ok(t, p->h, &t) || !mul_ok(t, p->w, &s->x_elems))
    return CONV_ERR_OVERFLOW;
  if (!mul_ok(p->c_out, s->K, &s->w_elems)) return CONV_ERR_OVERFLOW;
  if (!mul_ok(s->npix, p->c_out, &s->y_elems)) return CONV_ERR_OVERFLOW;
  if (!mul_ok(s->x_elems, 4, &t) || !mul_ok(s->y_elems, 4 * 64, &t) || !mul_ok(s->w_elems, 4, &t))
    return CONV_ERR_OVERFLOW;  // byte counts (and split planes) fit int64
  // kernel limits: per-image sizes and window offsets fit their 32-bit fields
  long long per_img_in, per_img_out;
  if (!mul_ok(p->c_in, p->h * p->w, &per_img_in) || per_img_in > kI32) return CONV_ERR_SHAPE;
  if (!mul_ok(p->c_out, s->ho * s->wo, &per_img_out) || per_img_out > kI32) return CONV_ERR_SHAPE;
  if (s->K > kI32 || p->h > kI32 || p->w > kI32 || p->pad_top > kI32 || p->pad_left > kI32 ||
      p->stride_h > kI32 || p->stride_w > kI32 || p->n > kI32 || p->c_out > kI32)
    return CONV_ERR_SHAPE;
  if (span_h > 32767 || span_w > 32767) return CONV_ERR_SHAPE;  // packed window table fields
  if (s->ho > kI32 || s->wo > kI32) return CONV_ERR_SHAPE;
  return CONV_OK;
}

// Resident blocks of a CUDA-core config per SM: threads (2048), shared memory,
// and registers -- each of the SM's four schedulers has a 16K-register file,
// allocated per warp in units of 256, and a block's warps are spread over the
// four, so a block of w warps fits as long as every scheduler can hold its
// share.
int occupancy_estimate(const FfmaCfg& c, size_t smem) {
  const int t = c.threads();
  const int warps = (t + 31) / 32;
  const int per_warp = (ffma_cfg_regs(c) * 32 + 255) / 256 * 256;
  const int warps_per_quarter = 16384 / per_warp;
  int occ = 2048 / t;
  occ = std::min(occ, static_cast<int>(kMaxDynSmem / std::max<size_t>(smem, 1)));
  occ = std::min(occ, 4 * warps_per_quarter / warps);
  return std::max(occ, 1);
}

// Scratch of the CUDA-core variant for a chunk of `images` whole images:
// split planes, then (256-byte aligned) the unfolded input, the transposed
// weights and the raw tiles of a tail split.  Only the planes and the
// unfolded input grow with the images; images = n gives the whole batch.
struct FfmaLayout {
  uint64_t xw_off, wt_off, tail_off, total;
};
FfmaLayout ffma_layout(const Plan& plan, const Shape& s, long long n, long long images) {
  auto align = [](uint64_t v) { return (v + 255) / 256 * 256; };
  FfmaLayout L{};
  uint64_t off = plan.info.split_k > 1
                     ? static_cast<uint64_t>(plan.info.split_k) * (s.y_elems / n) * images * sizeof(float)
                     : 0;
  if (plan.ffma_unf) {
    const UnfPlan& u = plan.unf;
    L.xw_off = align(off);
    off = L.xw_off + static_cast<uint64_t>(u.xw_elems / n) * images * sizeof(float);
    L.wt_off = align(off);
    off = L.wt_off + static_cast<uint64_t>(u.wt_elems) * sizeof(float);
    if (u.tail_split > 0) {
      const FfmaCfg& c = kFfmaCfgs[plan.ffma_cfg];
      L.tail_off = align(off);
      off = L.tail_off + static_cast<uint64_t>(u.tiles - u.tail_first) * u.tail_split * c.bm * c.bn * sizeof(float);
    }
  }
  L.total = off;
  return L;
}

// Whether the unfolded-B pre-pass pays for a CUDA-core layer: it moves x once
// and writes and reads the unfolded copy once, so it is taken when the
// layer's arithmetic is at least 64 FLOP per byte of that traffic (the
// multiply-adds then take several times the pre-pass) and k is long enough
// for 16-byte staging to matter.
bool unf_worth(const conv_problem* p, const Shape& s, const UnfPlan& u) {
  const double es = p->dtype == CONV_F32 ? 4.0 : 2.0;
  const double traffic = static_cast<double>(s.x_elems) * es + 2.0 * 4.0 * static_cast<double>(u.xw_elems);
  const double flops = 2.0 * static_cast<double>(s.y_elems) * static_cast<double>(s.K);
  return s.K >= 64 && flops >= 64.0 * traffic;
}

void plan_ffma(const conv_problem* p, const Shape& s, int sm, Plan* out) {
  // the B operand: 16-byte copies from an unfolded copy of x where that
  // applies and pays (or is forced), else the per-k gather
  const bool pointwise = p->kh == 1 && p->kw == 1 && p->stride_h == 1 && p->stride_w == 1 &&
                         p->pad_top == 0 && p->pad_left == 0 && p->pad_bottom == 0 && p->pad_right == 0;
  UnfPlan u;
  const bool unf_ok = !(p->flags & CONV_FLAG_NO_UNFOLD) && !(pointwise && p->dtype == CONV_F32) &&
                      unf_plan(p, s.ho, s.wo, &u);
  const bool unf = unf_ok && ((p->flags & CONV_FLAG_FORCE_UNFOLD) || unf_worth(p, s, u));
  // Per-SM time model: an SM runs ceil(blocks / SMs) tiles of bm x bn outputs
  // (padding included) at a rate set by the register tile, slowed when fewer
  // than 8 warps are resident to hide latency.  Lowest time wins; ties go to
  // the earlier (larger) tile.  With unfolded B the model follows the rounds
  // of resident blocks (`occupancy` per SM) and prices the tail split below:
  // the tiles of a last round that would fill at most half the device run as
  // s k ranges each, s = min(8, slots / tail tiles, k / 128).
  double best = 0.0;
  int bi = -1, best_tail = 0;
  for (int i = 0; i < kNumFfmaCfgs; ++i) {
    const FfmaCfg& c = kFfmaCfgs[i];
    const long long tm = (s.mg + c.bm - 1) / c.bm, tn = (s.npix + c.bn - 1) / c.bn;
    const long long ctas = tm * tn * p->groups;
    if (tm * p->groups > 65535) continue;
    const long long per_sm = (ctas + sm - 1) / sm;
    const int occ = occupancy_estimate(c, ffma_smem_bytes(i, static_cast<int>(s.K), unf));
    const double base = c.tm * c.tn >= 64 ? 1.0 : (c.tm * c.tn == 32 ? 0.85 : 0.6);
    double t;
    int tail = 0;
    if (!unf) {
      const double warps = static_cast<double>(std::min<long long>(per_sm, occ)) * c.threads() / 32.0;
      const double speed = base * std::min(1.0, warps / 8.0);
      t = static_cast<double>(per_sm) * c.bm * c.bn / speed;
    } else {
      auto speed = [&](long long blocks) {
        return base * std::min(1.0, static_cast<double>(blocks) * c.threads() / 32.0 / 12.0);
      };
      const double work = static_cast<double>(c.bm) * c.bn;
      const long long slots = static_cast<long long>(sm) * occ;
      const double t_round = occ * work / speed(occ);
      const long long full = ctas / slots, rest = ctas % slots;
      // whole rounds plus the last one as it is ...
      const long long last_per_sm = (rest + sm - 1) / sm;
      t = full * t_round + (rest ? last_per_sm * work / speed(last_per_sm) : 0.0);
      // ... or its tiles split in k
      if (full >= 1 && rest > 0 && 2 * rest <= slots && s.K >= 256 && p->groups == 1) {
        const long long ts = std::min<long long>({8, slots / rest, s.K / 128});
        if (ts >= 2) {
          const long long units_per_sm = (rest * ts + sm - 1) / sm;
          const double t_tail = full * t_round + units_per_sm * (work / ts) / speed(units_per_sm);
          if (t_tail < t) {
            t = t_tail;
            tail = static_cast<int>(ts);
          }
        }
      }
    }
    if (bi < 0 || t < best * (1.0 - 1e-9)) { best = t; bi = i; best_tail = tail; }
  }
  if (bi < 0) bi = 0;
  const FfmaCfg& c = kFfmaCfgs[bi];
  const long long ctas = ((s.mg + c.bm - 1) / c.bm) * ((s.npix + c.bn - 1) / c.bn) * p->groups;
  // split k ("Convolution, pooling and resize", split k for small grids): a
  // grid smaller than the device whose k has at least 256 terms runs k in at
  // most 16 ranges of at least 128 terms, each a whole number of stages,
  // aiming at about two blocks per SM; the cut is a function of (shape, SM
  // count) only.
  int split = 1;
  const int forced = static_cast<int>((p->flags & CONV_FLAG_SPLIT_K_MASK) >> CONV_FLAG_SPLIT_K_SHIFT);
  if (!(p->flags & CONV_FLAG_NO_SPLIT_K)) {
    if (forced > 0) {
      split = forced;
    } else if (ctas < sm && s.K >= 256) {
      const long long want = (2LL * sm + ctas - 1) / ctas;  // about two blocks per SM
      split = static_cast<int>(std::min<long long>({16, s.K / 128, want}));
    }
  }
  long long len = s.K;
  if (split > 1) {
    const int bk = unf ? kFfmaBKU : kFfmaBK;  // ranges of whole stages
    len = ((s.K + split - 1) / split + bk - 1) / bk * bk;
    split = static_cast<int>((s.K + len - 1) / len);
  }
  if (split <= 1) { split = 1; len = s.K; }
  // grouped layers with few channels per group: input rows staged once per
  // item instead of a per-k gather (no split k there)
  if (split == 1 && !unf) gd_plan(p, s.ho, s.wo, &out->gd);
  out->ffma_cfg = bi;
  out->ffma_unf = unf ? 1 : 0;
  // pointwise fp32 (1x1, stride 1, no pad, dilation 1) whose planes hold whole
  // groups of 4 pixels: 16-byte B copies (x's alignment is checked at launch)
  const long long hw = p->h * p->w;
  out->ffma_vec = p->dtype == CONV_F32 && p->kh == 1 && p->kw == 1 && p->stride_h == 1 && p->stride_w == 1 &&
                  p->pad_top == 0 && p->pad_left == 0 && p->pad_bottom == 0 && p->pad_right == 0 &&
                  hw % 4 == 0 && kFfmaCfgs[bi].bn % 4 == 0;
  out->info.variant = split > 1 ? CONV_VARIANT_IGEMM_FFMA_SPLIT : CONV_VARIANT_IGEMM_FFMA;
  out->info.split_k = split;
  out->info.tile_m = c.bm;
  out->info.tile_n = c.bn;
  out->info.ctas = ctas * split;
  if (unf) {
    u.tiles = ctas;
    if (split == 1 && best_tail > 0) {
      const int occ = occupancy_estimate(c, ffma_smem_bytes(bi, static_cast<int>(s.K), true));
      const long long slots = static_cast<long long>(sm) * occ;
      const long long rest = ctas % slots;
      u.tail_split = best_tail;
      u.tail_len = static_cast<int>(((s.K + best_tail - 1) / best_tail + kFfmaBKU - 1) / kFfmaBKU * kFfmaBKU);
      u.tail_split = static_cast<int>((s.K + u.tail_len - 1) / u.tail_len);  // ranges that hold terms
      u.tail_first = ctas - rest;
      out->info.ctas = u.tail_first + rest * u.tail_split;
    }
    out->unf = u;
  }
  const FfmaLayout L = ffma_layout(*out, s, p->n, p->n);
  out->unf.xw_off = L.xw_off;
  out->unf.wt_off = L.wt_off;
  out->unf.tail_off = L.tail_off;
  out->info.scratch_bytes = L.total;
  out->k_per_split = static_cast<int>(len);
  // the k ranges of a tile reduced within a thread-block cluster (at most 16
  // blocks; the 128 x 128 tile keeps the planes); the planes stay in the
  // scratch figure, for a device where no such cluster fits
  out->cluster_k = split >= 2 && split <= 16 && bi != 0 && !(p->flags & CONV_FLAG_NO_CLUSTER_K) ? 1 : 0;
  if (out->gd.ok) {
    out->info.tile_m = static_cast<int>(s.mg);
    out->info.tile_n = static_cast<int>(kGdRows * s.wo);
    out->info.ctas = std::min<long long>(out->gd.items, 3LL * sm);
  }
}

// 16-bit 1x1 layers (stride 1, no padding, dilation 1, one group, Cin <=
// 256, Cout <= 64) as channel x pixel tiles on the tensor cores, BM = the
// channels rounded up to 16.  Wider layers stay on the shifted-window kernel
// (its 1x1 view), which streams them better: a 64 -> 256 layer with a
// residual measured 84 us here against 39 us there.
bool plan_pointwise(const conv_problem* p, const Shape& s, int sm, Plan* out) {
  (void)sm;
  if (p->dtype == CONV_F32 || (p->flags & CONV_FLAG_NO_PW_MMA)) return false;
  if (p->kh != 1 || p->kw != 1 || p->stride_h != 1 || p->stride_w != 1 || p->groups != 1) return false;
  if (p->pad_top || p->pad_left || p->pad_bottom || p->pad_right) return false;
  if (p->c_in > 256 || p->c_out > 64 || s.ho * s.wo > (1LL << 30)) return false;
  const long long pblocks = (s.ho * s.wo + 127) / 128;
  if (p->n * pblocks > 2000000000LL) return false;
  PwPlan pp;
  pp.ok = 1;
  pp.kp = static_cast<int>((p->c_in + 15) / 16 * 16);
  pp.cfg = static_cast<int>((p->c_out + 15) / 16);
  const int bm = 16 * pp.cfg;
  if ((p->c_out + bm - 1) / bm > 65535) return false;
  if (pw_smem_bytes(pp, true) > 110 * 1024) return false;  // two blocks per SM
  out->pw = pp;
  out->info.variant = CONV_VARIANT_POINTWISE_MMA;
  out->info.split_k = 1;
  out->info.tile_m = bm;
  out->info.tile_n = 128;
  out->info.ctas = p->n * pblocks * ((p->c_out + bm - 1) / bm);
  out->info.scratch_bytes = 0;
  return true;
}

bool plan_depthwise(const conv_problem* p, const Shape& s, int sm, Plan* out) {
  constexpr int QH = 8;                       // output rows per thread (one column)
  const int es = p->dtype == CONV_F32 ? 4 : 2;
  const int al = 16 / es;                     // elements per 16 bytes
  DwPlan d;
  d.lm = static_cast<int>((p->pad_left + al - 1) / al * al);  // image column 0 on a 16-byte boundary
  // columns the windows of the last output column reach
  const long long need = d.lm - p->pad_left + (s.wo - 1) * p->stride_w + (p->kw - 1) * p->dil_w + 1;
  long long row = std::max<long long>(d.lm + p->w, need);
  row = (row + al - 1) / al * al;
  const long long wbytes = 2 * ((s.mg * p->kh * p->kw + 3) / 4 * 4) * 4 + 2 * ((s.mg + 3) / 4 * 4) * 4;
  const long long per_elem = 2LL * es + (es == 4 ? 0 : 4);  // two staging buffers (+ fp32 tile)
  const long long budget = 16 * 1024 - wbytes;              // bytes: ~12 blocks per SM
  if (row > (1 << 20) || wbytes > 64 * 1024) return false;
  // staged rows: a thread's 8-row strip may run past the block's last output
  // row, so stage whole strips
  auto in_rows = [&](long long t) {
    return ((t + QH - 1) / QH * QH - 1) * p->stride_h + (p->kh - 1) * p->dil_h + 1;
  };
  long long th = s.ho;
  while (th > QH && in_rows(th) * row * per_elem > budget) th = (th / 2 + QH - 1) / QH * QH;
  if (in_rows(th) * row * per_elem + wbytes > 200 * 1024) return false;
  d.th = static_cast<int>(th);
  d.in_rows = static_cast<int>(in_rows(th));
  d.row = static_cast<int>(row);
  d.vec = 0;
  d.sm = sm;
  // narrow planes: one warp per plane, two (Ho + k - 1)-row buffers of the
  // plane in shared memory per warp (8 warps per block)
  const long long nw_bytes = 8LL * 2 * (s.ho + p->kh - 1) * (s.wo + p->kw + 2) * es;
  d.narrow = p->stride_h == 1 && p->stride_w == 1 && p->dil_h == 1 && p->dil_w == 1 && p->kh == p->kw &&
             (p->kh == 3 || p->kh == 5 || p->kh == 7) && s.wo <= 32 && nw_bytes <= 96 * 1024;
  // four output columns per lane: the column groups x row blocks of a plane
  // fill one warp, with at most 8 rows per lane (the compiled row counts
  // 2, 4, 7, 8: the smallest that covers the plane)
  d.cols4_r = 0;
  if (d.narrow) {
    const long long groups = (s.wo + 3) / 4, rblocks = 32 / groups;
    const long long r = (s.ho + rblocks - 1) / rblocks;
    for (int rt : {2, 4, 7, 8}) {
      if (rt >= r) { d.cols4_r = rt; break; }
    }
    const long long nv = (p->kw + 6) / 4 * 4;
    const long long unit = 16 / es;
    const long long pitch = (std::max<long long>(p->pad_left + p->w, 4 * (groups - 1) + nv) + unit - 1) / unit * unit;
    const long long rows = rblocks * d.cols4_r + p->kh - 1;
    const long long outs = (s.ho * s.wo + 3) / 4 * 4 * 4;  // one warp's staged sums
    if (d.cols4_r && 4LL * (2 * pitch * rows * es + outs) > 45 * 1024) d.cols4_r = 0;  // five blocks per SM
    if (p->n * p->c_out > 2000000000LL) d.cols4_r = 0;  // plane indices (and the stride past them) in 32 bits
  }
  // 16-bit planes up to 64 columns wide on the tensor cores (band matrices,
  // mma.sync): the staged plane per warp, 16-byte rows with an odd number of
  // 16-byte units per row (conflict-free ldmatrix), eight warps, two buffers
  d.mma = 0;
  d.mma_pitch = d.mma_rows = 0;
  if (p->dtype != CONV_F32 && !(p->flags & CONV_FLAG_NO_DW_MMA) && p->stride_h == 1 && p->stride_w == 1 &&
      p->dil_h == 1 && p->dil_w == 1 && p->kh == p->kw && (p->kh == 3 || p->kh == 5 || p->kh == 7) &&
      s.wo <= 64 && p->n * p->c_out < 2000000000LL && p->n < 2000000000LL) {
    long long ntiles = (s.wo + 7) / 8;  // compiled for 1, 2, 4 or 8 column blocks
    ntiles = ntiles <= 1 ? 1 : ntiles <= 2 ? 2 : ntiles <= 4 ? 4 : 8;
    const long long mtiles = (s.ho + 15) / 16;
    const long long delta = p->pad_left & 1;
    long long pitch = std::max<long long>(8 * ntiles + 8, p->pad_left + delta + p->w);
    pitch = (pitch + 7) / 8 * 8;
    if ((pitch / 8) % 2 == 0) pitch += 8;
    const long long rows = 16 * mtiles + p->kh - 1;
    if (8LL * 2 * pitch * rows * 2 <= 110 * 1024) {
      d.mma = 1;
      d.mma_pitch = static_cast<int>(pitch);
      d.mma_rows = static_cast<int>(rows);
    }
  }
  out->dw = d;
  out->info.variant = CONV_VARIANT_DEPTHWISE;
  out->info.split_k = 1;
  out->info.tile_m = static_cast<int>(s.mg);
  out->info.tile_n = static_cast<int>(th * s.wo);
  const long long items = p->n * p->groups * ((s.ho + th - 1) / th);
  out->info.ctas = std::min<long long>(items, 12LL * sm);
  out->info.scratch_bytes = 0;
  return true;
}

// Geometry part of the kernel arguments (no addresses).
void shape_args(const conv_problem* p, const Shape& s, ConvArgs* a) {
  memset(a, 0, sizeof(*a));
  a->n = static_cast<int>(p->n); a->c_in = static_cast<int>(p->c_in);
  a->h = static_cast<int>(p->h); a->w = static_cast<int>(p->w);
  a->c_out = static_cast<int>(p->c_out); a->kh = static_cast<int>(p->kh); a->kw = static_cast<int>(p->kw);
  a->pt = static_cast<int>(p->pad_top); a->pl = static_cast<int>(p->pad_left);
  a->sh = static_cast<int>(p->stride_h); a->sw = static_cast<int>(p->stride_w);
  a->dh = static_cast<int>(p->dil_h); a->dw = static_cast<int>(p->dil_w);
  a->groups = static_cast<int>(p->groups); a->cg = static_cast<int>(s.cg); a->mg = static_cast<int>(s.mg);
  a->ho = static_cast<int>(s.ho); a->wo = static_cast<int>(s.wo);
  a->K = static_cast<int>(s.K);
  a->hw = p->h * p->w; a->howo = s.ho * s.wo; a->npix = s.npix;
  a->pix_lo = 0; a->pix_hi = s.npix; a->img0 = 0; a->part_total = s.y_elems;  // the whole batch
  a->act = p->act; a->alpha = p->act_alpha; a->beta = p->act_beta;
}

bool plan_tc(const conv_problem* p, const Shape& s, int sm, Plan* out) {
  if (p->dtype == CONV_F32) return false;
  ConvArgs a;
  shape_args(p, s, &a);
  a.residual = p->has_residual ? reinterpret_cast<const void*>(16) : nullptr;  // presence only
  TcPlan t;
  if (!tc_plan(a, sm, &t)) return false;
  out->tc = t;
  out->info.variant = CONV_VARIANT_IGEMM_TC;
  out->info.split_k = 1;
  out->info.tile_m = t.bn;
  out->info.tile_n = 128;
  out->info.ctas = t.ctas;
  out->info.scratch_bytes = 0;
  // the shifted-window kernel where it takes the shape (the gather kernel
  // above stays planned: the launch falls back to it when x is not 16-byte
  // aligned)
  WinPlan w;
  if (!(p->flags & CONV_FLAG_NO_WINDOW) && tcw_plan(a, sm, &w)) {
    out->tcw = w;
    out->tcw_ok = 1;
    out->info.variant = CONV_VARIANT_IGEMM_TC_WINDOW;
    out->info.tile_m = w.nt;
    out->info.ctas = w.ctas;
    out->info.scratch_bytes = w.w_bytes;
  }
  return true;
}

// Winograd F(2x2, 3x3): the shapes it covers, and whether it is taken.
bool wino_applies(const conv_problem* p) {
  return p->dtype == CONV_F32 && p->kh == 3 && p->kw == 3 && p->stride_h == 1 && p->stride_w == 1 &&
         p->dil_h == 1 && p->dil_w == 1 && p->groups == 1 && !(p->flags & CONV_FLAG_NO_WINOGRAD) &&
         !(p->flags & CONV_FLAG_FORCE_FFMA);
}

conv_status make_plan(const conv_problem* p, int sm, Plan* out, Shape* shape);

// The Winograd plan: tiles, the 16-group 1x1 product's plan and the scratch.
conv_status wino_prepare(const conv_problem* p, const Shape& s, int sm, WinoPlan* wp) {
  memset(wp, 0, sizeof(*wp));
  wp->geo.th = static_cast<int>((s.ho + 1) / 2);
  wp->geo.tw = static_cast<int>((s.wo + 1) / 2);
  wp->geo.tiles = p->n * wp->geo.th * wp->geo.tw;
  wp->geo.p4 = (wp->geo.tiles + 3) / 4 * 4;
  conv_problem q;
  memset(&q, 0, sizeof(q));
  q.n = 1; q.c_in = 16 * p->c_in; q.h = 1; q.w = wp->geo.p4;
  q.c_out = 16 * p->c_out; q.kh = q.kw = 1; q.stride_h = q.stride_w = 1; q.dil_h = q.dil_w = 1;
  q.groups = 16; q.act = CONV_ACT_IDENTITY; q.dtype = CONV_F32;
  q.flags = CONV_FLAG_FORCE_FFMA | CONV_FLAG_NO_SPLIT_K | CONV_FLAG_NO_UNFOLD;
  Shape sq;
  conv_status st = make_plan(&q, sm, &wp->gemm_plan, &sq);
  if (st != CONV_OK) return st;
  if (wp->gemm_plan.info.scratch_bytes != 0) return CONV_ERR_SHAPE;
  shape_args(&q, sq, &wp->gemm_args);
  auto align = [](uint64_t v) { return (v + 255) / 256 * 256; };
  uint64_t off = 0;
  wp->u_off = off;
  off = align(off + 16ull * p->c_out * p->c_in * 4);
  wp->v_off = off;
  off = align(off + 16ull * p->c_in * wp->geo.p4 * 4);
  wp->m_off = off;
  off += 16ull * p->c_out * wp->geo.p4 * 4;
  wp->scratch_bytes = off;
  return CONV_OK;
}

conv_status make_plan(const conv_problem* p, int sm, Plan* out, Shape* shape) {
  if (sm < 1) return CONV_ERR_ARG;
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  memset(out, 0, sizeof(*out));
  out->info.ho = s.ho;
  out->info.wo = s.wo;
  out->info.gemm_m = s.mg;
  out->info.gemm_n = s.npix;
  out->info.gemm_k = s.K;
  const bool force_ffma = (p->flags & CONV_FLAG_FORCE_FFMA) != 0;
  bool done = false;
  // Winograd where it is forced, or for 3x3 stride-1 float32 layers with 64 or
  // more channels each way (the sixteen products then dominate the transforms)
  if (wino_applies(p) && ((p->flags & CONV_FLAG_WINOGRAD) || (p->c_in >= 64 && p->c_out >= 64))) {
    WinoPlan wp;
    if (wino_prepare(p, s, sm, &wp) == CONV_OK) {
      out->info.variant = CONV_VARIANT_WINOGRAD;
      out->info.split_k = 1;
      out->info.tile_m = 2;
      out->info.tile_n = 2;
      out->info.ctas = wp.gemm_plan.info.ctas;
      out->info.scratch_bytes = wp.scratch_bytes;
      done = true;
    }
  }
  if (!done && !force_ffma && s.cg == 1) done = plan_depthwise(p, s, sm, out);
  if (!done && !force_ffma) done = plan_pointwise(p, s, sm, out);
  if (!done && !force_ffma) done = plan_tc(p, s, sm, out);
  if (!done) plan_ffma(p, s, sm, out);
  if (shape) *shape = s;
  return CONV_OK;
}

struct DevInfo {
  int sm = 0;
  int ok = 0;  // 1 usable, -1 not an sm_103 device
};
std::mutex g_dev_mu;
DevInfo g_dev[kMaxDevices];

conv_status device_info(int* dev_out, int* sm_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CONV_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.ok == 0) {
    int major = 0, minor = 0, sm = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return CONV_ERR_DEVICE;
    }
    d.sm = sm;
    d.ok = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (d.ok != 1) return CONV_ERR_DEVICE;
  *dev_out = dev;
  *sm_out = d.sm;
  return CONV_OK;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || !na || !nb) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

const char* variant_name(int v) {
  switch (v) {
    case CONV_VARIANT_IGEMM_FFMA: return "igemm_ffma";
    case CONV_VARIANT_IGEMM_FFMA_SPLIT: return "igemm_ffma_split_k";
    case CONV_VARIANT_DEPTHWISE: return "depthwise_halo";
    case CONV_VARIANT_IGEMM_TC: return "igemm_tcgen05";
    case CONV_VARIANT_IGEMM_TC_WINDOW: return "igemm_tcgen05_window";
    case CONV_VARIANT_WINOGRAD: return "winograd_f2x2_3x3";
    case CONV_VARIANT_POINTWISE_MMA: return "pointwise_mma";
    default: return "unknown";
  }
}

std::mutex g_smem_mu;
std::map<std::pair<const void*, int>, size_t> g_smem_optin;  // (kernel, device) -> bytes

struct ClusterKey {
  const void* func;
  int dev, cluster, threads;
  size_t smem;
  bool operator<(const ClusterKey& o) const {
    if (func != o.func) return func < o.func;
    if (dev != o.dev) return dev < o.dev;
    if (cluster != o.cluster) return cluster < o.cluster;
    if (threads != o.threads) return threads < o.threads;
    return smem < o.smem;
  }
};
std::mutex g_cluster_mu;
std::map<ClusterKey, bool> g_cluster_fits;

}  // namespace

bool conv::cluster_fits(const void* func, int cluster, int threads, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  const ClusterKey key{func, dev, cluster, threads, smem};
  auto it = g_cluster_fits.find(key);
  if (it != g_cluster_fits.end()) return it->second;
  bool ok = true;
  if (cluster > 8 && cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();  // a refused attribute leaves no error behind for the next launch check
    ok = false;
  }
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, static_cast<unsigned>(cluster));
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = static_cast<unsigned>(cluster);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) {
      cudaGetLastError();  // likewise for a refused query
      n = 0;
    }
    ok = n >= 1;
  }
  g_cluster_fits[key] = ok;
  return ok;
}

cudaError_t conv::opt_in_smem(const void* func, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;  // no opt-in needed
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_smem_mu);
  size_t& cur = g_smem_optin[std::make_pair(func, dev)];
  if (cur >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (err == cudaSuccess) cur = bytes;
  return err;
}

extern "C" {

int32_t conv_abi_version(void) { return CONV_ABI_VERSION; }

const char* conv_status_string(conv_status s) {
  switch (s) {
    case CONV_OK: return "ok";
    case CONV_ERR_SHAPE: return "invalid shape";
    case CONV_ERR_OVERFLOW: return "size overflow";
    case CONV_ERR_DTYPE: return "unknown element type";
    case CONV_ERR_ACT: return "unknown activation";
    case CONV_ERR_NULL: return "required pointer is NULL";
    case CONV_ERR_SCRATCH: return "scratch too small or misaligned";
    case CONV_ERR_ALIAS: return "overlapping operands";
    case CONV_ERR_DEVICE: return "no usable sm_103 device";
    case CONV_ERR_CUDA: return "CUDA launch failed";
    case CONV_ERR_ARG: return "invalid argument";
    default: return "unknown status";
  }
}

conv_status conv_output_shape(const conv_problem* p, int64_t* ho, int64_t* wo) {
  if (!ho || !wo) return CONV_ERR_NULL;
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  *ho = s.ho;
  *wo = s.wo;
  return CONV_OK;
}

conv_status conv_apply_auto_pad(conv_problem* p, int32_t mode) {
  if (!p) return CONV_ERR_NULL;
  if (mode < CONV_AUTO_PAD_NOTSET || mode > CONV_AUTO_PAD_VALID) return CONV_ERR_ARG;
  conv_problem q = *p;
  if (mode == CONV_AUTO_PAD_VALID) {
    q.pad_top = q.pad_left = q.pad_bottom = q.pad_right = 0;
  } else if (mode != CONV_AUTO_PAD_NOTSET) {
    // one axis: (input, kernel, stride, dilation) -> (begin, end)
    auto axis = [mode](long long in, long long k, long long s, long long d, int64_t* b, int64_t* e) {
      if (in < 1 || k < 1 || s < 1 || d < 1 || k > (1LL << 40) || d > (1LL << 20)) return false;
      const long long out = (in + s - 1) / s;
      long long total = 0;
      if (__builtin_mul_overflow(out - 1, s, &total) || __builtin_add_overflow(total, d * (k - 1) + 1 - in, &total))
        return false;
      if (total < 0) total = 0;
      const long long small = total / 2, large = total - total / 2;
      *b = mode == CONV_AUTO_PAD_SAME_UPPER ? small : large;
      *e = mode == CONV_AUTO_PAD_SAME_UPPER ? large : small;
      return true;
    };
    if (!axis(q.h, q.kh, q.stride_h, q.dil_h, &q.pad_top, &q.pad_bottom) ||
        !axis(q.w, q.kw, q.stride_w, q.dil_w, &q.pad_left, &q.pad_right))
      return CONV_ERR_SHAPE;
  }
  Shape s;
  const conv_status st = validate(&q, &s);
  if (st != CONV_OK) return st;
  *p = q;
  return CONV_OK;
}

conv_status conv_plan(const conv_problem* p, int32_t sm_count, conv_plan_info* out) {
  if (!out) return CONV_ERR_NULL;
  Plan plan;
  conv_status st = make_plan(p, sm_count, &plan, nullptr);
  if (st == CONV_OK) *out = plan.info;
  return st;
}

conv_status conv_scratch_bytes(const conv_problem* p, size_t* bytes) {
  if (!bytes) return CONV_ERR_NULL;
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  int dev, sm;
  st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  Plan plan;
  st = make_plan(p, sm, &plan, nullptr);
  if (st == CONV_OK) *bytes = static_cast<size_t>(plan.info.scratch_bytes);
  return st;
}

conv_status conv_scratch_bytes_per_image(const conv_problem* p, size_t* bytes) {
  if (!bytes) return CONV_ERR_NULL;
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  int dev, sm;
  st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  Plan plan;
  st = make_plan(p, sm, &plan, nullptr);
  if (st != CONV_OK) return st;
  const bool ffma = plan.info.variant == CONV_VARIANT_IGEMM_FFMA || plan.info.variant == CONV_VARIANT_IGEMM_FFMA_SPLIT;
  *bytes = static_cast<size_t>(ffma ? ffma_layout(plan, s, p->n, 1).total : plan.info.scratch_bytes);
  return CONV_OK;
}

conv_status conv_describe_variant(const conv_problem* p, char* buf, size_t len) {
  if (!buf || !len) return CONV_ERR_NULL;
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  int dev, sm;
  st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  return conv_describe_plan(p, sm, buf, len);
}

conv_status conv_describe_plan(const conv_problem* p, int32_t sm_count, char* buf, size_t len) {
  if (!buf || !len) return CONV_ERR_NULL;
  const int sm = sm_count;
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  Plan plan;
  st = make_plan(p, sm, &plan, nullptr);
  if (st != CONV_OK) return st;
  const conv_plan_info& i = plan.info;
  const int launches = (i.variant == CONV_VARIANT_IGEMM_FFMA || i.variant == CONV_VARIANT_IGEMM_FFMA_SPLIT)
                           ? ffma_launch_count(plan)
                           : (i.variant == CONV_VARIANT_IGEMM_TC_WINDOW ? 2 : (i.variant == CONV_VARIANT_WINOGRAD ? 4 : 1));
  if (i.variant == CONV_VARIANT_WINOGRAD) {
    WinoPlan wp;
    if (wino_prepare(p, s, sm, &wp) != CONV_OK) return CONV_ERR_SHAPE;
    const FfmaCfg& c = kFfmaCfgs[wp.gemm_plan.ffma_cfg];
    snprintf(buf, len, "%s tiles=%dx%d per image (%lld in all) products=16 x %lldco x %lldci on CUDA cores "
             "tile=%dco x %dpx scratch=%llu sms=%d", variant_name(i.variant), wp.geo.th, wp.geo.tw,
             static_cast<long long>(wp.geo.tiles), static_cast<long long>(p->c_out), static_cast<long long>(p->c_in),
             c.bm, c.bn, static_cast<unsigned long long>(i.scratch_bytes), sm);
  } else if (i.variant == CONV_VARIANT_IGEMM_TC) {
    static const char* orders[] = {"tap/8-channel", "channel/row/8-tap", "channel/tap"};
    snprintf(buf, len, "%s tile=128px x %dco k=%lld (padded %d, %s order) stages=%d blocks=%lld sms=%d",
             variant_name(i.variant), plan.tc.bn, static_cast<long long>(i.gemm_k), plan.tc.k_pad,
             orders[plan.tc.mode], plan.tc.stages, static_cast<long long>(i.ctas), sm);
  } else if (i.variant == CONV_VARIANT_IGEMM_TC_WINDOW) {
    const WinPlan& w = plan.tcw;
    snprintf(buf, len,
             "%s tile=128pos x %dco phases=%dx%d taps=%dx%d k=%lld (padded %d) padded plane=%dx%d "
             "ring=%d+%d bands of %d rows, %d in flight, lookahead=%d blocks=%lld sms=%d",
             variant_name(i.variant), w.nt, w.ph, w.ph, w.khp, w.kwp, static_cast<long long>(i.gemm_k),
             w.kblocks * 8, w.hp, w.wp, w.ring, w.mirror, w.band, w.stages, w.lookahead,
             static_cast<long long>(i.ctas), sm);
  } else if (i.variant == CONV_VARIANT_IGEMM_FFMA && plan.gd.ok) {
    snprintf(buf, len,
             "%s grouped: input rows staged once per (group, image, %d output rows), %d staged rows of %d, "
             "8co x 4px per thread, items=%lld sms=%d",
             variant_name(i.variant), kGdRows, plan.gd.rows_in, plan.gd.pitch, static_cast<long long>(plan.gd.items), sm);
  } else if (i.variant == CONV_VARIANT_POINTWISE_MMA) {
    snprintf(buf, len,
             "%s tile=%dco x 128px (one image), k=%d in shared memory, mma.sync m16n8k16, blocks=%lld sms=%d",
             variant_name(i.variant), i.tile_m, plan.pw.kp, static_cast<long long>(i.ctas), sm);
  } else if (i.variant == CONV_VARIANT_DEPTHWISE && plan.dw.mma) {
    snprintf(buf, len,
             "%s tensor cores: per channel %d band matrices, mma.sync m16n8k16 over 16 x 8 output blocks, "
             "one warp per plane, staged plane %dx%d sms=%d",
             variant_name(i.variant), static_cast<int>(p->kh), plan.dw.mma_rows, plan.dw.mma_pitch, sm);
  } else if (i.variant == CONV_VARIANT_DEPTHWISE && plan.dw.cols4_r) {
    snprintf(buf, len, "%s one warp per plane, 4 columns x %d rows per lane, double-buffered planes sms=%d",
             variant_name(i.variant), plan.dw.cols4_r, sm);
  } else if (i.variant == CONV_VARIANT_DEPTHWISE && plan.dw.narrow) {
    snprintf(buf, len, "%s one warp per plane, window in registers, double-buffered planes sms=%d",
             variant_name(i.variant), sm);
  } else if (i.variant == CONV_VARIANT_DEPTHWISE) {
    snprintf(buf, len, "%s rows/block=%d staged=%dx%d blocks=%lld sms=%d", variant_name(i.variant),
             plan.dw.th, plan.dw.in_rows, plan.dw.row, static_cast<long long>(i.ctas), sm);
  } else {
    const FfmaCfg& c = kFfmaCfgs[plan.ffma_cfg];
    char tail[64] = "";
    if (plan.ffma_unf && plan.unf.tail_split > 0)
      snprintf(tail, sizeof(tail), " tail=%lld tiles x %d k ranges", static_cast<long long>(plan.unf.tiles - plan.unf.tail_first),
               plan.unf.tail_split);
    const char* reduce = i.split_k < 2 ? "" : (plan.cluster_k ? " reduce=cluster" : " reduce=planes");
    snprintf(buf, len, "%s tile=%dco x %dpx (%dx%d per thread) B=%s split_k=%d%s%s blocks=%lld scratch=%llu sms=%d",
             variant_name(i.variant), i.tile_m, i.tile_n, c.tm, c.tn,
             plan.ffma_unf ? "unfolded" : (plan.ffma_vec ? "pointwise" : "gathered"), i.split_k, reduce, tail,
             static_cast<long long>(i.ctas), static_cast<unsigned long long>(i.scratch_bytes), sm);
  }
  // the number of kernels one call launches, last
  const size_t used = strlen(buf);
  if (used + 1 < len) snprintf(buf + used, len - used, " launches=%d", launches);
  return CONV_OK;
}

conv_status conv_forward(const conv_problem* p, const void* x, const void* w, const void* bias,
                         const void* residual, void* y, void* scratch, size_t scratch_bytes,
                         void* stream) {
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  if (!x || !w || !y) return CONV_ERR_NULL;
  if (p->has_bias && !bias) return CONV_ERR_NULL;
  if (p->has_residual && !residual) return CONV_ERR_NULL;
  const size_t es = p->dtype == CONV_F32 ? 4 : 2;
  const size_t xb = s.x_elems * es, wb = s.w_elems * es, yb = s.y_elems * es;
  const size_t bb = p->has_bias ? p->c_out * es : 0, rb = p->has_residual ? yb : 0;
  const void* in_ptr[] = {x, w, p->has_bias ? bias : nullptr, p->has_residual ? residual : nullptr};
  const size_t in_len[] = {xb, wb, bb, rb};
  for (int i = 0; i < 4; ++i)
    if (overlap(y, yb, in_ptr[i], in_len[i])) return CONV_ERR_ALIAS;
  int dev, sm;
  st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  Plan plan;
  st = make_plan(p, sm, &plan, nullptr);
  if (st != CONV_OK) return st;
  size_t need = plan.info.scratch_bytes;
  // chunks of whole images when the CUDA-core variant's scratch is smaller
  // than the whole batch needs ("Convolution, pooling and resize", Layout and
  // operands: a smaller buffer makes the batch run in chunks of whole
  // images, which changes no bit of the result)
  const bool ffma = plan.info.variant == CONV_VARIANT_IGEMM_FFMA || plan.info.variant == CONV_VARIANT_IGEMM_FFMA_SPLIT;
  long long chunk = p->n;
  if (need && ffma && scratch && scratch_bytes < need) {
    chunk = 0;
    for (long long lo = 1, hi = p->n - 1; lo <= hi;) {  // the most images whose scratch fits
      const long long mid = lo + (hi - lo) / 2;
      if (ffma_layout(plan, s, p->n, mid).total <= scratch_bytes) { chunk = mid; lo = mid + 1; }
      else hi = mid - 1;
    }
    if (chunk == 0) return CONV_ERR_SCRATCH;
    need = ffma_layout(plan, s, p->n, chunk).total;
  }
  if (need) {
    if (!scratch || scratch_bytes < need || reinterpret_cast<uintptr_t>(scratch) % 16) return CONV_ERR_SCRATCH;
    for (int i = 0; i < 4; ++i)
      if (overlap(scratch, need, in_ptr[i], in_len[i])) return CONV_ERR_ALIAS;
    if (overlap(scratch, need, y, yb)) return CONV_ERR_ALIAS;
  }

  ConvArgs a;
  shape_args(p, s, &a);
  a.x = x; a.wt = w; a.y = y;
  a.bias = p->has_bias ? bias : nullptr;
  a.residual = p->has_residual ? residual : nullptr;
  a.vec_out = (reinterpret_cast<uintptr_t>(y) % 16 == 0) ? 1 : 0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaSuccess;
  switch (plan.info.variant) {
    case CONV_VARIANT_DEPTHWISE: {
      // widest cp.async copy that keeps every plane and row start aligned
      plan.dw.vec = 0;
      for (int cb = 16; cb >= 4; cb /= 2) {
        if (reinterpret_cast<uintptr_t>(x) % cb == 0 && (a.hw * es) % cb == 0 && (p->w * es) % cb == 0) {
          plan.dw.vec = cb;
          break;
        }
      }
      err = launch_depthwise(plan, a, p->dtype, cs);
      break;
    }
    case CONV_VARIANT_IGEMM_TC_WINDOW:
      // bulk copies of x rows need a 16-byte-aligned x; otherwise the gather kernel
      // TMA boxes of x, y (and the residual) want 16-byte-aligned arrays;
      // otherwise the gather kernel
      if (reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
          (!residual || reinterpret_cast<uintptr_t>(residual) % 16 == 0))
        err = launch_tcw(plan, a, p->dtype, scratch, cs);
      else err = launch_tc(plan, a, p->dtype, cs);
      break;
    case CONV_VARIANT_IGEMM_TC:
      err = launch_tc(plan, a, p->dtype, cs);
      break;
    case CONV_VARIANT_POINTWISE_MMA:
      err = launch_pointwise(plan.pw, a, p->dtype, cs);
      break;
    case CONV_VARIANT_WINOGRAD: {
      WinoPlan wp;
      if (wino_prepare(p, s, sm, &wp) != CONV_OK) return CONV_ERR_SHAPE;
      err = launch_winograd(wp, a, scratch, cs);
      break;
    }
    default: {
      a.split = plan.info.split_k;
      a.k_per_split = plan.k_per_split;
      a.cluster_k = plan.cluster_k;
      a.partial = static_cast<float*>(scratch);
      const FfmaLayout L = ffma_layout(plan, s, p->n, chunk);
      if (plan.ffma_unf) {
        a.xw = reinterpret_cast<float*>(static_cast<char*>(scratch) + L.xw_off);
        a.wtt = reinterpret_cast<float*>(static_cast<char*>(scratch) + L.wt_off);
        a.hu = plan.unf.hu;
        a.mg4 = plan.unf.mg4;
        if (plan.unf.tail_split > 0) {
          const FfmaCfg& c = kFfmaCfgs[plan.ffma_cfg];
          a.tail_split = plan.unf.tail_split;
          a.tail_len = plan.unf.tail_len;
          a.tiles_gy = static_cast<int>((s.mg + c.bm - 1) / c.bm * p->groups);
          a.tail_first = plan.unf.tail_first;
          a.tail_tiles = plan.unf.tiles - plan.unf.tail_first;
          a.tailbuf = reinterpret_cast<float*>(static_cast<char*>(scratch) + L.tail_off);
        }
      }
      // the whole batch, or chunks of whole images: every output is computed
      // by the whole problem's tile, k ranges and order either way
      for (long long n0 = 0; n0 < p->n && err == cudaSuccess; n0 += chunk) {
        const long long n1 = std::min<long long>(p->n, n0 + chunk);
        a.pix_lo = n0 * a.howo;
        a.pix_hi = n1 * a.howo;
        a.img0 = static_cast<int>(n0);
        a.part_total = (n1 - n0) * a.c_out * a.howo;
        err = launch_ffma(plan, a, p->dtype, cs);
        if (err == cudaSuccess && a.split > 1 && !a.cluster_k) err = launch_split_reduce(a, p->dtype, cs);
      }
      break;
    }
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return CONV_ERR_CUDA;
  }
  return CONV_OK;
}

// ---- ConvTranspose -------------------------------------------------------------
// The transposed problem: its output size, the 1x1 Gemm problem and its plan,
// the kernel arguments (addresses left empty) and the scratch layout.
static conv_status t_prepare(const conv_transpose_problem* tp, int sm, TransposePlan* out, ConvArgs* a,
                             TransposeGeo* geo, Shape* shape) {
  if (!tp) return CONV_ERR_NULL;
  const conv_problem* p = &tp->conv;
  if (p->dtype < CONV_F32 || p->dtype > CONV_BF16) return CONV_ERR_DTYPE;
  if (p->act < CONV_ACT_IDENTITY || p->act > CONV_ACT_LEAKY_RELU) return CONV_ERR_ACT;
  const long long pos[] = {p->n, p->c_in, p->h, p->w, p->c_out, p->kh, p->kw,
                           p->stride_h, p->stride_w, p->dil_h, p->dil_w, p->groups};
  for (long long v : pos)
    if (v < 1) return CONV_ERR_SHAPE;
  if (p->pad_top < 0 || p->pad_left < 0 || p->pad_bottom < 0 || p->pad_right < 0) return CONV_ERR_SHAPE;
  if (p->c_in % p->groups || p->c_out % p->groups) return CONV_ERR_SHAPE;
  // ONNX: output_padding below the stride or the dilation of its axis
  if (tp->out_pad_h < 0 || tp->out_pad_w < 0 || tp->out_pad_h >= std::max(p->stride_h, p->dil_h) ||
      tp->out_pad_w >= std::max(p->stride_w, p->dil_w))
    return CONV_ERR_SHAPE;
  const long long big = 1LL << 31;
  const long long dims[] = {p->n, p->c_in, p->h, p->w, p->c_out, p->kh, p->kw, p->stride_h, p->stride_w,
                            p->dil_h, p->dil_w, p->pad_top, p->pad_left, p->pad_bottom, p->pad_right};
  for (long long v : dims)
    if (v >= big) return CONV_ERR_SHAPE;
  const long long ho = p->stride_h * (p->h - 1) + tp->out_pad_h + p->dil_h * (p->kh - 1) + 1 - p->pad_top - p->pad_bottom;
  const long long wo = p->stride_w * (p->w - 1) + tp->out_pad_w + p->dil_w * (p->kw - 1) + 1 - p->pad_left - p->pad_right;
  if (ho < 1 || wo < 1) return CONV_ERR_SHAPE;
  if (ho >= big || wo >= big) return CONV_ERR_SHAPE;
  long long per_img_out, y_elems, t;
  if (!mul_ok(p->c_out, ho, &t) || !mul_ok(t, wo, &per_img_out) || per_img_out > kI32) return CONV_ERR_SHAPE;
  if (!mul_ok(per_img_out, p->n, &y_elems)) return CONV_ERR_OVERFLOW;
  // the Gemm: a 1x1 convolution of x to Cout*kh*kw channels (groups kept)
  conv_problem q;
  memset(&q, 0, sizeof(q));
  q.n = p->n; q.c_in = p->c_in; q.h = p->h; q.w = p->w;
  long long cout_k;
  if (!mul_ok(p->c_out, p->kh * p->kw, &cout_k)) return CONV_ERR_OVERFLOW;
  q.c_out = cout_k;
  q.kh = q.kw = 1; q.stride_h = q.stride_w = 1; q.dil_h = q.dil_w = 1; q.groups = p->groups;
  // The Gemm runs in float32 for every element type: 16-bit x is widened
  // into scratch first (exact), so the pointwise kernel's 16-byte copies apply;
  // its products and sums are those of the 16-bit kernel, which widens each
  // element as it stages it.
  q.act = CONV_ACT_IDENTITY; q.dtype = CONV_F32;
  q.flags = CONV_FLAG_FORCE_FFMA | CONV_FLAG_NO_SPLIT_K | CONV_FLAG_NO_UNFOLD;
  Shape sq;
  conv_status st = make_plan(&q, sm, &out->gemm_plan, &sq);
  if (st != CONV_OK) return st;
  if (out->gemm_plan.info.scratch_bytes != 0) return CONV_ERR_SHAPE;  // a plain one-pass Gemm
  shape_args(&q, sq, &out->gemm_args);
  out->dtype = p->dtype;
  auto up256 = [](size_t v) { return (v + 255) / 256 * 256; };
  // 16-bit, one group, Cin <= 256: the Gemm on the pointwise tensor-core
  // kernel with raw float32 sums (x read as it is, the weights transposed in
  // their own type); else the float32 CUDA-core Gemm above
  out->mma = 0;
  memset(&out->pw, 0, sizeof(out->pw));
  if (p->dtype != CONV_F32 && p->groups == 1 && p->c_in <= 256 && !(p->flags & CONV_FLAG_NO_PW_MMA) &&
      p->n * ((p->h * p->w + 127) / 128) <= 2000000000LL && (cout_k + 127) / 128 <= 65535) {
    PwPlan pp;
    pp.ok = 1;
    pp.kp = static_cast<int>((p->c_in + 15) / 16 * 16);
    pp.cfg = cout_k <= 64 ? static_cast<int>((cout_k + 15) / 16) : 5;
    if (pp.cfg == 5 && pw_smem_bytes(pp, false) > 110 * 1024) pp.cfg = 4;  // 64-channel tiles when k is long
    if (pw_smem_bytes(pp, false) <= 110 * 1024) {  // two blocks per SM
      out->mma = 1;
      out->pw = pp;
    }
  }
  out->wt_off = 0;
  if (out->mma) {
    out->xf_off = 0;
    out->cols_off = up256(static_cast<size_t>(sq.w_elems) * 2);
  } else {
    out->xf_off = up256(static_cast<size_t>(sq.w_elems) * 4);
    out->cols_off = out->xf_off + (p->dtype == CONV_F32 ? 0 : up256(static_cast<size_t>(sq.x_elems) * 4));
  }
  long long cols_bytes;
  if (!mul_ok(sq.y_elems, 4, &cols_bytes)) return CONV_ERR_OVERFLOW;
  out->scratch_bytes = out->cols_off + static_cast<size_t>(cols_bytes);
  // the col2im's arguments: the transposed problem's geometry
  memset(a, 0, sizeof(*a));
  a->n = static_cast<int>(p->n); a->c_in = static_cast<int>(p->c_in);
  a->h = static_cast<int>(p->h); a->w = static_cast<int>(p->w);
  a->c_out = static_cast<int>(p->c_out); a->kh = static_cast<int>(p->kh); a->kw = static_cast<int>(p->kw);
  a->pt = static_cast<int>(p->pad_top); a->pl = static_cast<int>(p->pad_left);
  a->sh = static_cast<int>(p->stride_h); a->sw = static_cast<int>(p->stride_w);
  a->dh = static_cast<int>(p->dil_h); a->dw = static_cast<int>(p->dil_w);
  a->groups = static_cast<int>(p->groups);
  a->cg = static_cast<int>(p->c_in / p->groups); a->mg = static_cast<int>(p->c_out / p->groups);
  a->hw = p->h * p->w;
  a->act = p->act; a->alpha = p->act_alpha; a->beta = p->act_beta;
  geo->ho = static_cast<int>(ho);
  geo->wo = static_cast<int>(wo);
  if (shape) {
    memset(shape, 0, sizeof(*shape));
    shape->ho = ho; shape->wo = wo;
    shape->x_elems = p->n * p->c_in * p->h * p->w;
    shape->w_elems = p->c_in * (p->c_out / p->groups) * p->kh * p->kw;
    shape->y_elems = y_elems;
  }
  return CONV_OK;
}

conv_status conv_transpose_output_shape(const conv_transpose_problem* tp, int64_t* ho, int64_t* wo) {
  if (!ho || !wo) return CONV_ERR_NULL;
  TransposePlan pl;
  ConvArgs a;
  TransposeGeo g;
  const conv_status st = t_prepare(tp, 152, &pl, &a, &g, nullptr);
  if (st != CONV_OK) return st;
  *ho = g.ho;
  *wo = g.wo;
  return CONV_OK;
}

conv_status conv_transpose_scratch_bytes(const conv_transpose_problem* tp, size_t* bytes) {
  if (!bytes) return CONV_ERR_NULL;
  int dev, sm;
  conv_status st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  TransposePlan pl;
  ConvArgs a;
  TransposeGeo g;
  st = t_prepare(tp, sm, &pl, &a, &g, nullptr);
  if (st == CONV_OK) *bytes = pl.scratch_bytes;
  return st;
}

conv_status conv_transpose_forward(const conv_transpose_problem* tp, const void* x, const void* w,
                                   const void* bias, const void* residual, void* y, void* scratch,
                                   size_t scratch_bytes, void* stream) {
  if (!tp) return CONV_ERR_NULL;
  const conv_problem* p = &tp->conv;
  int dev, sm;
  conv_status st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  TransposePlan pl;
  ConvArgs a;
  TransposeGeo g;
  Shape s;
  st = t_prepare(tp, sm, &pl, &a, &g, &s);
  if (st != CONV_OK) return st;
  if (!x || !w || !y) return CONV_ERR_NULL;
  if (p->has_bias && !bias) return CONV_ERR_NULL;
  if (p->has_residual && !residual) return CONV_ERR_NULL;
  const size_t es = p->dtype == CONV_F32 ? 4 : 2;
  const size_t xb = s.x_elems * es, wb = s.w_elems * es, yb = s.y_elems * es;
  const size_t bb = p->has_bias ? p->c_out * es : 0, rb = p->has_residual ? yb : 0;
  const void* in_ptr[] = {x, w, p->has_bias ? bias : nullptr, p->has_residual ? residual : nullptr};
  const size_t in_len[] = {xb, wb, bb, rb};
  for (int i = 0; i < 4; ++i)
    if (overlap(y, yb, in_ptr[i], in_len[i])) return CONV_ERR_ALIAS;
  if (!scratch || scratch_bytes < pl.scratch_bytes || reinterpret_cast<uintptr_t>(scratch) % 256)
    return CONV_ERR_SCRATCH;
  for (int i = 0; i < 4; ++i)
    if (overlap(scratch, pl.scratch_bytes, in_ptr[i], in_len[i])) return CONV_ERR_ALIAS;
  if (overlap(scratch, pl.scratch_bytes, y, yb)) return CONV_ERR_ALIAS;
  a.x = x; a.wt = w; a.y = y;
  a.bias = p->has_bias ? bias : nullptr;
  a.residual = p->has_residual ? residual : nullptr;
  if (launch_conv_transpose(pl, a, g, w, scratch, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return CONV_ERR_CUDA;
  }
  return CONV_OK;
}

// ---- ConvInteger -------------------------------------------------------------
// The geometry of conv_problem; no bias, residual or activation.
static conv_status ci_validate(const conv_problem* p, int32_t x_type, int32_t w_type, Shape* s) {
  conv_status st = validate(p, s);
  if (st != CONV_OK) return st;
  if (x_type < CONV_U8 || x_type > CONV_I8 || w_type < CONV_U8 || w_type > CONV_I8) return CONV_ERR_DTYPE;
  if (p->act != CONV_ACT_IDENTITY || p->has_bias || p->has_residual) return CONV_ERR_ARG;
  if ((s->mg + 127) / 128 * p->groups > 65535 || p->groups > 65535) return CONV_ERR_SHAPE;  // grid limits
  return CONV_OK;
}

conv_status conv_integer_scratch_bytes(const conv_problem* p, int32_t x_type, int32_t w_type, size_t* bytes) {
  if (!bytes) return CONV_ERR_NULL;
  Shape s;
  conv_status st = ci_validate(p, x_type, w_type, &s);
  if (st != CONV_OK) return st;
  ConvArgs a;
  shape_args(p, s, &a);
  *bytes = ci_plan(a).scratch_bytes;
  return CONV_OK;
}

conv_status conv_integer_forward(const conv_problem* p, int32_t x_type, int32_t w_type, const void* x,
                                 const void* w, const void* x_zero, const void* w_zero, int32_t w_zero_count,
                                 int32_t* y, void* scratch, size_t scratch_bytes, void* stream) {
  Shape s;
  conv_status st = ci_validate(p, x_type, w_type, &s);
  if (st != CONV_OK) return st;
  if (!x || !w || !x_zero || !w_zero || !y) return CONV_ERR_NULL;
  if (w_zero_count != 1 && w_zero_count != p->c_out) return CONV_ERR_ARG;
  int dev, sm;
  st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  ConvArgs a;
  shape_args(p, s, &a);
  const CiPlan pl = ci_plan(a);
  const size_t yb = s.y_elems * 4;
  const void* in_ptr[] = {x, w, x_zero, w_zero};
  const size_t in_len[] = {static_cast<size_t>(s.x_elems), static_cast<size_t>(s.w_elems), 1,
                           static_cast<size_t>(w_zero_count)};
  for (int i = 0; i < 4; ++i)
    if (overlap(y, yb, in_ptr[i], in_len[i])) return CONV_ERR_ALIAS;
  if (!scratch || scratch_bytes < pl.scratch_bytes || reinterpret_cast<uintptr_t>(scratch) % 256)
    return CONV_ERR_SCRATCH;
  for (int i = 0; i < 4; ++i)
    if (overlap(scratch, pl.scratch_bytes, in_ptr[i], in_len[i])) return CONV_ERR_ALIAS;
  if (overlap(scratch, pl.scratch_bytes, y, yb)) return CONV_ERR_ALIAS;
  a.x = x; a.wt = w; a.y = y;
  CiArgs c;
  memset(&c, 0, sizeof(c));
  c.x_signed = x_type == CONV_I8;
  c.w_signed = w_type == CONV_I8;
  c.x_zero = static_cast<const uint8_t*>(x_zero);
  c.w_zero = static_cast<const uint8_t*>(w_zero);
  c.wz_per_channel = w_zero_count > 1;
  c.kq = pl.kq;
  c.p4 = pl.p4;
  c.mg4 = pl.mg4;
  char* sc = static_cast<char*>(scratch);
  c.cols = reinterpret_cast<uint32_t*>(sc + pl.cols_off);
  c.sx = reinterpret_cast<int32_t*>(sc + pl.sx_off);
  c.wq = reinterpret_cast<uint32_t*>(sc + pl.wq_off);
  c.sw = reinterpret_cast<int32_t*>(sc + pl.sw_off);
  if (launch_conv_integer(a, pl, c, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return CONV_ERR_CUDA;
  }
  return CONV_OK;
}

conv_status conv_device_error(uint32_t* word, int32_t reset) {
  if (!word) return CONV_ERR_NULL;
  int dev, sm;
  conv_status st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  uint32_t w1 = 0, w2 = 0;
  if (tc_error_word(&w1, reset) != cudaSuccess || tcw_error_word(&w2, reset) != cudaSuccess) return CONV_ERR_CUDA;
  *word = w1 | (w2 << 16);
  return CONV_OK;
}

conv_status conv_selftest_bounded_wait(uint32_t limit_us, uint32_t* report) {
  if (!report) return CONV_ERR_NULL;
  if (limit_us < 1 || limit_us > 100000) return CONV_ERR_ARG;
  int dev, sm;
  conv_status st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  if (tcw_wait_selftest_run(1000ull * limit_us, report) != cudaSuccess) {
    cudaGetLastError();
    return CONV_ERR_CUDA;
  }
  return CONV_OK;
}

}  // extern "C"

// ---- a forward call for callers that cannot allocate device memory ---------
//
// Some callers cannot call cudaMalloc: code running where allocation is not
// permitted (a plug-in of a host framework that owns every allocation, a
// real-time path that must not touch the allocator, a caller with no CUDA
// runtime of its own beyond this library).  For them the scratch -- the
// split-k planes, or the shifted-window variant's repacked weights -- lives
// in one fixed device array that the library owns.  It is reserved on every
// GPU that loads this library and kept until the process exits.
static __device__ __align__(256) unsigned char g_fixed_scratch[CONV_FIXED_SCRATCH_BYTES];

namespace {
std::mutex g_fixed_mu;
void* g_fixed_addr[kMaxDevices];  // device address of g_fixed_scratch, per device
}  // namespace

extern "C" conv_status conv_forward_fixed_scratch(const conv_problem* p, const void* x, const void* w,
                                                  const void* bias, const void* residual, void* y,
                                                  void* stream) {
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  int dev, sm;
  st = device_info(&dev, &sm);
  if (st != CONV_OK) return st;
  Plan plan;
  st = make_plan(p, sm, &plan, nullptr);
  if (st != CONV_OK) return st;
  // When the plan's scratch does not fit the array, a variant that needs none
  // may still run the problem: the gather tensor-core kernel instead of the
  // shifted-window one (no repacked weights), or k unsplit (no partial
  // planes), unless the caller forced the split.
  conv_problem q = *p;
  const int forced_split = static_cast<int>((p->flags & CONV_FLAG_SPLIT_K_MASK) >> CONV_FLAG_SPLIT_K_SHIFT);
  const uint32_t fallbacks[] = {CONV_FLAG_NO_WINDOW, CONV_FLAG_NO_WINOGRAD, CONV_FLAG_NO_UNFOLD,
                                forced_split ? 0u : CONV_FLAG_NO_SPLIT_K};
  for (uint32_t f : fallbacks) {
    if (plan.info.scratch_bytes <= CONV_FIXED_SCRATCH_BYTES) break;
    if (!f || (q.flags & f)) continue;
    if (f == CONV_FLAG_NO_UNFOLD && (q.flags & CONV_FLAG_FORCE_UNFOLD)) continue;
    if (f == CONV_FLAG_NO_WINOGRAD && (q.flags & CONV_FLAG_WINOGRAD)) continue;
    q.flags |= f;
    st = make_plan(&q, sm, &plan, nullptr);
    if (st != CONV_OK) return st;
  }
  if (plan.info.scratch_bytes > CONV_FIXED_SCRATCH_BYTES) return CONV_ERR_SCRATCH;
  void* addr = nullptr;
  {
    // set-up, once per device, with that device current: the array's name is
    // a host-side stand-in, the kernels need its device address
    std::lock_guard<std::mutex> lock(g_fixed_mu);
    if (!g_fixed_addr[dev]) {
      void* a = nullptr;
      if (cudaGetSymbolAddress(&a, g_fixed_scratch) != cudaSuccess || !a) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
      }
      g_fixed_addr[dev] = a;
    }
    addr = g_fixed_addr[dev];
  }
  return conv_forward(&q, x, w, bias, residual, y, addr, CONV_FIXED_SCRATCH_BYTES, stream);
}
