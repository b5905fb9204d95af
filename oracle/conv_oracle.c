/*
 * conv_oracle.c -- the CPU oracle for the forward 2-D convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header or constant with the CUDA
 * library: the geometry arrives as a flat array of integers and every
 * conversion, index computation and activation below is written out here.
 *
 * What it computes (one output element at a time, by plain nested loops):
 *
 *   Ho = floor((H + pad_top + pad_bottom - dil_h*(kh-1) - 1) / stride_h) + 1
 *     "Convolutions", section 2.1 (output size, boxed equation), with the two
 *     pads of an axis added separately as ONNX Conv allows ("Convolution,
 *     pooling and resize", Layout and operands: explicit pads).
 *
 *   acc[n,co,oh,ow] = sum_{c < Cin/g} sum_{u < kh} sum_{v < kw}
 *                      X(n, g(co)*Cin/g + c, oh*sh - pt + u*dh, ow*sw - pl + v*dw)
 *                      * W[co, c, u, v]
 *     "Convolutions", section 3, the naive loop definition
 *     (out[b,o,i,j] = sum of patch * w[o]), extended to groups as its
 *     exercise 4 describes and to per-axis stride / dilation / pads.
 *     X(...) is zero outside the image (zero padding, as np.pad does there).
 *     The sum runs in double, in the fixed order c, u, v.
 *
 *   S[n,co,oh,ow]   = the same sum of |X * W|  (the per-output error scale of
 *                      the parity bar |err| <= tol * sum |w x|).
 *
 *   t = (float)acc; t = t + bias[co]; t = t + residual[n,co,oh,ow]; t = act(t)
 *     "Convolution, pooling and resize", Layout and operands: sum, bias,
 *     residual addition, activation, in that order, each step rounded to
 *     float32.  The activations are the ONNX operator definitions.
 *
 *   y = t rounded to the element type (round to nearest, ties to even).
 *
 * Element types: 0 = float32, 1 = IEEE binary16, 2 = bfloat16.  Half and
 * bfloat16 operands are decoded exactly to double here.
 *
 * Built with -ffp-contract=off so that no multiply-add is fused: the float32
 * epilogue then rounds each step as written on every host.
 *
 * The transposed convolution (ONNX ConvTranspose; "Convolution, pooling and
 * resize", Layout and operands: weights [Cin][Cout/groups][kh][kw]; output
 * size from "Convolutions", section 2.1, (H - 1)s - pads + d(kh - 1) + 1 +
 * output_padding) is the same loop read the other way round:
 *
 *   acc[n,co,oh,ow] = sum_{c < Cin/g} sum_{u < kh} sum_{v < kw}
 *                      X(n, g(co)*Cin/g + c, (oh + pt - u*dh)/sh, (ow + pl - v*dw)/sw)
 *                      * W[g(co)*Cin/g + c, co - g(co)*Cout/g, u, v]
 *
 * where a term exists only when both divisions are exact and land inside the
 * image (each input pixel spreads the kernel over the output at s-strided
 * positions; each output gathers the taps that reach it).  The same double
 * sum, error scale and float32 epilogue as the forward convolution.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0 /* >0 plants one deliberate mistake (pin self-test) */
#endif

/* ---- geometry: a flat array, index names ------------------------------ */
enum {
  G_N, G_CIN, G_H, G_W, G_COUT, G_KH, G_KW,
  G_PT, G_PL, G_PB, G_PR,
  G_SH, G_SW, G_DH, G_DW, G_GROUPS,
  G_COUNT
};

/* activation codes of this file (the Python wrapper maps names to these) */
enum {
  A_IDENTITY = 0, A_RELU = 1, A_SILU = 2, A_SIGMOID = 3, A_TANH = 4,
  A_HARD_SWISH = 5, A_HARD_SIGMOID = 6, A_CLIP = 7, A_LEAKY_RELU = 8
};

/* ---- number formats ---------------------------------------------------- */

/* binary16 -> double, exact: sign, 5-bit exponent (bias 15), 10-bit fraction. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 -> double, exact: the upper 16 bits of a float32. */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round the integer q * 2^-shift to the nearest integer, ties to even. */
static uint32_t rne_shift(uint64_t q, int shift) {
  if (shift <= 0) return (uint32_t)q;
  if (shift > 40) return 0;
  uint64_t keep = q >> shift;
  uint64_t rem = q & ((1ull << shift) - 1);
  uint64_t half = 1ull << (shift - 1);
#if ORACLE_MUTANT == 9
  (void)rem; (void)half; /* mutant: truncation instead of round-to-even */
#else
  if (rem > half || (rem == half && (keep & 1))) keep += 1;
#endif
  return (uint32_t)keep;
}

/* float32 -> binary16, round to nearest even; overflow to infinity. */
uint16_t oracle_float_to_half(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
  uint32_t a = u & 0x7fffffffu;
  if (a > 0x7f800000u) return sign | 0x7e00; /* NaN */
  if (a >= 0x477ff000u) return sign | 0x7c00; /* >= 65520 rounds to inf */
  int e = (int)(a >> 23);
  uint64_t m = (a & 0x7fffffu) | (e ? 0x800000u : 0);
  if (e == 0) e = 1; /* float32 subnormal: exponent -126 */
  /* value = m * 2^(e - 150).  Half units: subnormal step 2^-24. */
  if (e < 113) { /* below 2^-14: a half subnormal (or zero) */
    int shift = 126 - e; /* m * 2^(e-150) / 2^-24 = m * 2^(e-126) */
    return sign | (uint16_t)rne_shift(m, shift);
  }
  /* normal: 10 fraction bits kept of 23; the carry may bump the exponent */
  uint32_t r = rne_shift(m, 13); /* 1024 .. 2048 */
  uint32_t eh = (uint32_t)(e - 127 + 15);
  return sign | (uint16_t)((eh << 10) + (r - 1024));
}

/* float32 -> bfloat16, round to nearest even. */
uint16_t oracle_float_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);
  uint32_t keep = u >> 16;
  uint32_t rem = u & 0xffffu;
  if (rem > 0x8000u || (rem == 0x8000u && (keep & 1))) keep += 1;
  return (uint16_t)keep;
}

static double load_elem(const void* p, int64_t i, int dtype) {
  if (dtype == 0) return (double)((const float*)p)[i];
  if (dtype == 1) return oracle_half_to_double(((const uint16_t*)p)[i]);
  return oracle_bf16_to_double(((const uint16_t*)p)[i]);
}

/* ---- activations (ONNX definitions, evaluated in float32) -------------- */
float oracle_activation(int act, float t, float alpha, float beta) {
  switch (act) {
    case A_IDENTITY: return t;
    case A_RELU: return t > 0.0f ? t : 0.0f;
    case A_SIGMOID: return 1.0f / (1.0f + expf(-t));
    case A_TANH: return tanhf(t);
    case A_SILU: return t * (1.0f / (1.0f + expf(-t)));
    case A_HARD_SIGMOID: {
      float s = alpha * t;
      s = s + beta;
      return fmaxf(0.0f, fminf(1.0f, s));
    }
    case A_HARD_SWISH: { /* HardSwish: alpha = 1/6, beta = 0.5 */
      float s = t * (1.0f / 6.0f);
      s = s + 0.5f;
      return t * fmaxf(0.0f, fminf(1.0f, s));
    }
    case A_CLIP: return fminf(fmaxf(t, alpha), beta); /* alpha=min, beta=max */
    case A_LEAKY_RELU: return t >= 0.0f ? t : alpha * t;
    default: return NAN;
  }
}

/* ---- output size -------------------------------------------------------- */
int64_t oracle_output_extent(int64_t in, int64_t k, int64_t pad_begin,
                             int64_t pad_end, int64_t stride, int64_t dil) {
  int64_t span = dil * (k - 1) + 1; /* the dilated kernel's extent */
  int64_t room = in + pad_begin + pad_end - span;
  if (room < 0 || stride < 1) return 0;
#if ORACLE_MUTANT == 6
  return room / stride; /* mutant: the +1 dropped */
#else
  return room / stride + 1;
#endif
}

/* ---- one output element -------------------------------------------------- */
typedef struct {
  const int64_t* g;
  int act;
  float alpha, beta;
  int dtype;
  const void *x, *w, *b, *r;
  void* y;
  float* t_out;
  double *acc_out, *scale_out;
  const int64_t* index; /* NULL: outputs [begin, end) in order */
  int64_t begin, end;
  int64_t ho, wo;
  int transpose; /* 1: the transposed convolution */
} job;

/* The transposed sum of one output: see the header. */
static void transposed_sum(const job* J, int64_t n, int64_t co, int64_t oh, int64_t ow, double* acc_out,
                           double* scale_out) {
  const int64_t* g = J->g;
  const int64_t cg = g[G_CIN] / g[G_GROUPS], mg = g[G_COUT] / g[G_GROUPS];
  const int64_t grp = co / mg, col = co - grp * mg;
  double acc = 0.0, scale = 0.0;
  for (int64_t c = 0; c < cg; ++c) {
    const int64_t ci = grp * cg + c;
    for (int64_t u = 0; u < g[G_KH]; ++u) {
      const int64_t th = oh + g[G_PT] - u * g[G_DH];
#if ORACLE_MUTANT == 11
      if (th < 0) continue; /* mutant: the stride's divisibility is not checked */
      const int64_t ih = th / g[G_SH];
#else
      if (th < 0 || th % g[G_SH]) continue;
      const int64_t ih = th / g[G_SH];
#endif
      if (ih >= g[G_H]) continue;
      for (int64_t v = 0; v < g[G_KW]; ++v) {
        const int64_t tw = ow + g[G_PL] - v * g[G_DW];
        if (tw < 0 || tw % g[G_SW]) continue;
        const int64_t iw = tw / g[G_SW];
        if (iw >= g[G_W]) continue;
        const double xv = load_elem(J->x, ((n * g[G_CIN] + ci) * g[G_H] + ih) * g[G_W] + iw, J->dtype);
#if ORACLE_MUTANT == 12
        const double wv = load_elem(J->w, ((ci * mg + col) * g[G_KH] + (g[G_KH] - 1 - u)) * g[G_KW] +
                                           (g[G_KW] - 1 - v), J->dtype); /* mutant: kernel flipped */
#else
        const double wv = load_elem(J->w, ((ci * mg + col) * g[G_KH] + u) * g[G_KW] + v, J->dtype);
#endif
        acc += xv * wv;
        scale += fabs(xv * wv);
      }
    }
  }
  *acc_out = acc;
  *scale_out = scale;
}

static void one_output(const job* J, int64_t lin, int64_t slot) {
  const int64_t* g = J->g;
  int64_t ho = J->ho, wo = J->wo;
  int64_t ow = lin % wo;
  int64_t oh = (lin / wo) % ho;
  int64_t co = (lin / (wo * ho)) % g[G_COUT];
  int64_t n = lin / (wo * ho * g[G_COUT]);
  int64_t cg = g[G_CIN] / g[G_GROUPS];
  int64_t mg = g[G_COUT] / g[G_GROUPS];
  int64_t grp = co / mg;
#if ORACLE_MUTANT == 3
  grp = 0; /* mutant: every group reads the first channel slice */
#endif
  double acc = 0.0, scale = 0.0;
  if (J->transpose) transposed_sum(J, n, co, oh, ow, &acc, &scale);
  for (int64_t c = 0; c < cg && !J->transpose; ++c) {
    for (int64_t u = 0; u < g[G_KH]; ++u) {
      for (int64_t v = 0; v < g[G_KW]; ++v) {
#if ORACLE_MUTANT == 5
        int64_t ih = oh * g[G_SH] * g[G_DH] - g[G_PT] + u; /* mutant */
        int64_t iw = ow * g[G_SW] * g[G_DW] - g[G_PL] + v;
#elif ORACLE_MUTANT == 2
        int64_t ih = oh * g[G_SH] - g[G_PT] + u * g[G_DH];
        int64_t iw = ow * g[G_SW] - g[G_PT] + v * g[G_DW]; /* mutant: pad */
#else
        int64_t ih = oh * g[G_SH] - g[G_PT] + u * g[G_DH];
        int64_t iw = ow * g[G_SW] - g[G_PL] + v * g[G_DW];
#endif
        double xv = 0.0;
#if ORACLE_MUTANT == 10
        /* mutant: clamp-to-edge border instead of zeros */
        int64_t ihc = ih < 0 ? 0 : (ih >= g[G_H] ? g[G_H] - 1 : ih);
        int64_t iwc = iw < 0 ? 0 : (iw >= g[G_W] ? g[G_W] - 1 : iw);
        xv = load_elem(J->x, ((n * g[G_CIN] + grp * cg + c) * g[G_H] + ihc) * g[G_W] + iwc, J->dtype);
#else
        if (ih >= 0 && ih < g[G_H] && iw >= 0 && iw < g[G_W])
          xv = load_elem(J->x, ((n * g[G_CIN] + grp * cg + c) * g[G_H] + ih) * g[G_W] + iw,
                         J->dtype);
#endif
#if ORACLE_MUTANT == 1
        double wv = load_elem(J->w, ((co * cg + c) * g[G_KH] + v) * g[G_KW] + u, J->dtype);
#else
        double wv = load_elem(J->w, ((co * cg + c) * g[G_KH] + u) * g[G_KW] + v, J->dtype);
#endif
#if ORACLE_MUTANT == 7
        acc -= xv * wv; /* mutant: sign */
#else
        acc += xv * wv;
#endif
        scale += fabs(xv * wv);
      }
    }
  }
  float t = (float)acc;
#if ORACLE_MUTANT == 4
  if (J->r) t = t + (float)load_elem(J->r, lin, J->dtype);
  if (J->b) t = t + (float)load_elem(J->b, co, J->dtype);
  t = oracle_activation(J->act, t, J->alpha, J->beta);
#elif ORACLE_MUTANT == 8
  if (J->b) t = t + (float)load_elem(J->b, co, J->dtype);
  t = oracle_activation(J->act, t, J->alpha, J->beta); /* mutant: act first */
  if (J->r) t = t + (float)load_elem(J->r, lin, J->dtype);
#else
  if (J->b) t = t + (float)load_elem(J->b, co, J->dtype);
  if (J->r) t = t + (float)load_elem(J->r, lin, J->dtype);
  t = oracle_activation(J->act, t, J->alpha, J->beta);
#endif
  if (J->dtype == 0) ((float*)J->y)[slot] = t;
  else if (J->dtype == 1) ((uint16_t*)J->y)[slot] = oracle_float_to_half(t);
  else ((uint16_t*)J->y)[slot] = oracle_float_to_bf16(t);
  if (J->t_out) J->t_out[slot] = t;
  if (J->acc_out) J->acc_out[slot] = acc;
  if (J->scale_out) J->scale_out[slot] = scale;
}

static void* run_job(void* p) {
  const job* J = (const job*)p;
  for (int64_t s = J->begin; s < J->end; ++s)
    one_output(J, J->index ? J->index[s] : s, s);
  return NULL;
}

static int run(job base, int64_t count, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > count) nthreads = count > 0 ? (int)count : 1;
  pthread_t th[256];
  job jobs[256];
  for (int i = 0; i < nthreads; ++i) {
    jobs[i] = base;
    jobs[i].begin = count * i / nthreads;
    jobs[i].end = count * (i + 1) / nthreads;
  }
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, run_job, &jobs[i]) != 0) break;
    started = i;
  }
  run_job(&jobs[0]);
  for (int i = started + 1; i < nthreads; ++i) run_job(&jobs[i]); /* not started */
  for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
  return 0;
}

static int check_geom(const int64_t* g, int64_t* ho, int64_t* wo) {
  for (int i = 0; i < G_COUNT; ++i) {
    if (i >= G_PT && i <= G_PR) { if (g[i] < 0) return -1; }
    else if (g[i] < 1) return -1;
  }
  if (g[G_CIN] % g[G_GROUPS] || g[G_COUT] % g[G_GROUPS]) return -1;
  *ho = oracle_output_extent(g[G_H], g[G_KH], g[G_PT], g[G_PB], g[G_SH], g[G_DH]);
  *wo = oracle_output_extent(g[G_W], g[G_KW], g[G_PL], g[G_PR], g[G_SW], g[G_DW]);
  return (*ho >= 1 && *wo >= 1) ? 0 : -1;
}

/*
 * Every output of the problem, in NCHW order.  y has N*Cout*Ho*Wo elements
 * of the element type; t_out / acc_out / scale_out (each optional) receive
 * the float32 epilogue result, the double sum and the error scale.
 * Returns 0, or -1 for a geometry the definition does not cover.
 */
int oracle_conv2d(const int64_t* geom, int act, float alpha, float beta, int dtype,
                  const void* x, const void* w, const void* b, const void* r,
                  void* y, float* t_out, double* acc_out, double* scale_out,
                  int nthreads) {
  int64_t ho, wo;
  if (check_geom(geom, &ho, &wo)) return -1;
  job J;
  memset(&J, 0, sizeof J);
  J.g = geom; J.act = act; J.alpha = alpha; J.beta = beta; J.dtype = dtype;
  J.x = x; J.w = w; J.b = b; J.r = r; J.y = y;
  J.t_out = t_out; J.acc_out = acc_out; J.scale_out = scale_out;
  J.ho = ho; J.wo = wo;
  return run(J, geom[G_N] * geom[G_COUT] * ho * wo, nthreads);
}

/* The outputs whose NCHW linear indices are listed in index[0..count). */
int oracle_conv2d_at(const int64_t* geom, int act, float alpha, float beta, int dtype,
                     const void* x, const void* w, const void* b, const void* r,
                     const int64_t* index, int64_t count,
                     void* y, float* t_out, double* acc_out, double* scale_out,
                     int nthreads) {
  int64_t ho, wo;
  if (check_geom(geom, &ho, &wo)) return -1;
  int64_t total = geom[G_N] * geom[G_COUT] * ho * wo;
  for (int64_t i = 0; i < count; ++i)
    if (index[i] < 0 || index[i] >= total) return -1;
  job J;
  memset(&J, 0, sizeof J);
  J.g = geom; J.act = act; J.alpha = alpha; J.beta = beta; J.dtype = dtype;
  J.x = x; J.w = w; J.b = b; J.r = r; J.y = y; J.index = index;
  J.t_out = t_out; J.acc_out = acc_out; J.scale_out = scale_out;
  J.ho = ho; J.wo = wo;
  return run(J, count, nthreads);
}

/* ---- the transposed convolution --------------------------------------------- */
/* Output extent: s*(in - 1) + output_padding + d*(k - 1) + 1 - pad_begin - pad_end. */
int64_t oracle_transpose_extent(int64_t in, int64_t k, int64_t pad_begin, int64_t pad_end, int64_t stride,
                                int64_t dil, int64_t out_pad) {
  if (in < 1 || k < 1 || stride < 1 || dil < 1 || out_pad < 0 || pad_begin < 0 || pad_end < 0) return 0;
  int64_t e = stride * (in - 1) + out_pad + dil * (k - 1) + 1 - pad_begin - pad_end;
  return e > 0 ? e : 0;
}

static int check_tgeom(const int64_t* g, int64_t oph, int64_t opw, int64_t* ho, int64_t* wo) {
  for (int i = 0; i < G_COUNT; ++i) {
    if (i >= G_PT && i <= G_PR) { if (g[i] < 0) return -1; }
    else if (g[i] < 1) return -1;
  }
  if (g[G_CIN] % g[G_GROUPS] || g[G_COUT] % g[G_GROUPS]) return -1;
  *ho = oracle_transpose_extent(g[G_H], g[G_KH], g[G_PT], g[G_PB], g[G_SH], g[G_DH], oph);
  *wo = oracle_transpose_extent(g[G_W], g[G_KW], g[G_PL], g[G_PR], g[G_SW], g[G_DW], opw);
  return (*ho >= 1 && *wo >= 1) ? 0 : -1;
}

/* Every output (index NULL) or the listed NCHW outputs of the transposed
 * convolution; geom as for oracle_conv2d with G_COUT the output channels,
 * w laid out [Cin][Cout/groups][kh][kw]. */
int oracle_conv_transpose2d(const int64_t* geom, int64_t out_pad_h, int64_t out_pad_w, int act, float alpha,
                            float beta, int dtype, const void* x, const void* w, const void* b, const void* r,
                            const int64_t* index, int64_t count, void* y, float* t_out, double* acc_out,
                            double* scale_out, int nthreads) {
  int64_t ho, wo;
  if (check_tgeom(geom, out_pad_h, out_pad_w, &ho, &wo)) return -1;
  const int64_t total = geom[G_N] * geom[G_COUT] * ho * wo;
  if (index) {
    for (int64_t i = 0; i < count; ++i)
      if (index[i] < 0 || index[i] >= total) return -1;
  } else {
    count = total;
  }
  job J;
  memset(&J, 0, sizeof J);
  J.g = geom; J.act = act; J.alpha = alpha; J.beta = beta; J.dtype = dtype;
  J.x = x; J.w = w; J.b = b; J.r = r; J.y = y; J.index = index;
  J.t_out = t_out; J.acc_out = acc_out; J.scale_out = scale_out;
  J.ho = ho; J.wo = wo; J.transpose = 1;
  return run(J, count, nthreads);
}

int oracle_mutant(void) { return ORACLE_MUTANT; }
