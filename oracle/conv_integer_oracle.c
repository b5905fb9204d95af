/*
 * conv_integer_oracle.c -- the CPU oracle of ConvInteger.
 *
 * TEST INFRASTRUCTURE ONLY, like conv_oracle.c beside it: nothing in the
 * product path may link, load or call this file, and it shares no code,
 * header or constant with the CUDA library.
 *
 * What it computes ("Convolution, pooling and resize", ConvInteger; ONNX
 * ConvInteger):
 *
 *   y[n,co,oh,ow] = sum_{c < Cin/g} sum_{u < kh} sum_{v < kw}
 *                     (X(n, g(co)*Cin/g + c, oh*sh - pt + u*dh, ow*sw - pl + v*dw) - xz)
 *                   * (W[co, c, u, v] - wz(co))
 *
 *   in int32 with wrap-around.  x and w are each uint8 or int8 (any mix); xz
 *   is one value of x's type, wz one value of w's type or one per output
 *   channel.  A tap outside the image is the real value zero, which is the
 *   quantized value xz, so it adds nothing: X(...) = xz there.
 *
 * Each output is summed exactly in int64 (a term is at most 255 * 255 in
 * magnitude), in the fixed order c, u, v, and the exact sum is reduced
 * modulo 2^32 to a two's-complement int32 -- the value an int32 accumulator
 * that wraps around on overflow ends with, in any summation order.
 *
 * The geometry arrives as the same flat int64 array as conv_oracle.c's
 * (n, cin, h, w, cout, kh, kw, pt, pl, pb, pr, sh, sw, dh, dw, groups).
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum {
  I_N, I_CIN, I_H, I_W, I_COUT, I_KH, I_KW,
  I_PT, I_PL, I_PB, I_PR,
  I_SH, I_SW, I_DH, I_DW, I_GROUPS,
  I_COUNT
};

/* An element of a uint8 (is_signed = 0) or int8 (is_signed = 1) array. */
static int32_t byte_at(const void* p, int64_t i, int is_signed) {
#if ORACLE_MUTANT == 23
  (void)is_signed;
  return (int32_t)((const uint8_t*)p)[i]; /* mutant: int8 read as uint8 */
#else
  return is_signed ? (int32_t)((const int8_t*)p)[i] : (int32_t)((const uint8_t*)p)[i];
#endif
}

/* Reduce an exact integer modulo 2^32 to two's-complement int32. */
static int32_t wrap32(int64_t v) {
#if ORACLE_MUTANT == 24
  if (v > INT32_MAX) return INT32_MAX; /* mutant: saturation instead of wrap-around */
  if (v < INT32_MIN) return INT32_MIN;
  return (int32_t)v;
#else
  uint64_t u = (uint64_t)v & 0xffffffffull;
  return u >= 0x80000000ull ? (int32_t)((int64_t)u - 0x100000000ll) : (int32_t)u;
#endif
}

static int64_t extent(int64_t size, int64_t k, int64_t pb, int64_t pe, int64_t s, int64_t d) {
  int64_t span = d * (k - 1) + 1;
  int64_t padded = size + pb + pe;
  if (padded < span) return 0;
  return (padded - span) / s + 1;
}

typedef struct {
  const int64_t* g;
  int x_signed, w_signed;
  const void* x;
  const void* w;
  int32_t xz;
  const int32_t* wz;  /* decoded zero points: one per output channel, or one */
  int wz_per_channel;
  const int64_t* index;
  int64_t begin, end;
  int64_t ho, wo;
  int32_t* y;
} ijob;

static void* run_ijob(void* arg) {
  const ijob* J = (const ijob*)arg;
  const int64_t* g = J->g;
  const int64_t cg = g[I_CIN] / g[I_GROUPS], mg = g[I_COUT] / g[I_GROUPS];
  for (int64_t e = J->begin; e < J->end; ++e) {
    const int64_t o = J->index ? J->index[e] : e;
    const int64_t ow = o % J->wo;
    const int64_t oh = (o / J->wo) % J->ho;
    const int64_t co = (o / (J->wo * J->ho)) % g[I_COUT];
    const int64_t n = o / (J->wo * J->ho * g[I_COUT]);
#if ORACLE_MUTANT == 22
    const int32_t wz = J->wz[0]; /* mutant: the first channel's zero point for every channel */
#else
    const int32_t wz = J->wz_per_channel ? J->wz[co] : J->wz[0];
#endif
    const int64_t grp = co / mg;
    int64_t acc = 0;
    for (int64_t c = 0; c < cg; ++c) {
      for (int64_t u = 0; u < g[I_KH]; ++u) {
        const int64_t ih = oh * g[I_SH] - g[I_PT] + u * g[I_DH];
        for (int64_t v = 0; v < g[I_KW]; ++v) {
          const int64_t iw = ow * g[I_SW] - g[I_PL] + v * g[I_DW];
          int32_t xv;
          if (ih >= 0 && ih < g[I_H] && iw >= 0 && iw < g[I_W]) {
            xv = byte_at(J->x, ((n * g[I_CIN] + grp * cg + c) * g[I_H] + ih) * g[I_W] + iw, J->x_signed);
          } else {
#if ORACLE_MUTANT == 21
            xv = 0; /* mutant: padded taps as the quantized value 0, not the zero point */
#else
            xv = J->xz;
#endif
          }
          const int32_t wv = byte_at(J->w, ((co * cg + c) * g[I_KH] + u) * g[I_KW] + v, J->w_signed);
#if ORACLE_MUTANT == 25
          acc += (int64_t)xv * (int64_t)(wv - wz); /* mutant: x's zero point ignored */
#else
          acc += (int64_t)(xv - J->xz) * (int64_t)(wv - wz);
#endif
        }
      }
    }
    J->y[e] = wrap32(acc);
  }
  return NULL;
}

/*
 * x_signed / w_signed: 0 uint8, 1 int8.  xz: x's zero point (already
 * decoded); wz: count 1 or Cout decoded zero points.  index (optional): NCHW
 * linear output indices, count of them; without it every output, count =
 * N*Cout*Ho*Wo.  Returns 0, or -1 for a geometry outside the definition.
 */
int oracle_conv_integer(const int64_t* geom, int x_signed, int w_signed, const void* x, const void* w,
                        int32_t xz, const int32_t* wz, int wz_per_channel, const int64_t* index,
                        int64_t count, int32_t* y, int nthreads) {
  for (int i = 0; i < I_COUNT; ++i) {
    if (i >= I_PT && i <= I_PR) { if (geom[i] < 0) return -1; }
    else if (geom[i] < 1) return -1;
  }
  if (geom[I_CIN] % geom[I_GROUPS] || geom[I_COUT] % geom[I_GROUPS]) return -1;
  const int64_t ho = extent(geom[I_H], geom[I_KH], geom[I_PT], geom[I_PB], geom[I_SH], geom[I_DH]);
  const int64_t wo = extent(geom[I_W], geom[I_KW], geom[I_PL], geom[I_PR], geom[I_SW], geom[I_DW]);
  if (ho < 1 || wo < 1) return -1;
  const int64_t total = geom[I_N] * geom[I_COUT] * ho * wo;
  if (index) {
    for (int64_t i = 0; i < count; ++i)
      if (index[i] < 0 || index[i] >= total) return -1;
  } else {
    count = total;
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  ijob jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    ijob* J = &jobs[t];
    memset(J, 0, sizeof *J);
    J->g = geom; J->x_signed = x_signed; J->w_signed = w_signed; J->x = x; J->w = w;
    J->xz = xz; J->wz = wz; J->wz_per_channel = wz_per_channel; J->index = index;
    J->ho = ho; J->wo = wo; J->y = y;
    J->begin = count * t / nthreads;
    J->end = count * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, run_ijob, &jobs[t]) != 0) break;
    started = t;
  }
  run_ijob(&jobs[0]);
  for (int t = started + 1; t < nthreads; ++t) run_ijob(&jobs[t]); /* not started */
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  return 0;
}
