/*
 * dsc_oracle.c -- fp64 CPU oracle for Dynamic Short Convolutions (DSC).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the only thing both sides share is the seeded input generator.
 *
 * What it computes (each function below names the passage it follows):
 *
 *   Dynamic short convolution ("Technische Samenvatting: Dynamische Korte
 *   Convoluties Verbeteren Transformers", section Methodologie / Mechanisme;
 *   and "Dynamic Short Convolutions: The 'Locality Bias' Transformers Were
 *   Missing", section 1 "Mathematical Intuition"):
 *
 *       y_t = sum_{k=0}^{W-1} w(t)_k (.) x_{t-k}        (.) = per channel
 *
 *   with x_{t-k} = 0 before the first token of each sequence, and the
 *   optional residual X + DSC(X) (same summary, Methodologie / Plaatsing).
 *
 *   Head-wise tying (same summary, Parametrisatie item 2): one filter is
 *   shared by H consecutive channels, so channel c reads filter g = c / H and
 *   w has shape [B, T, C/H, W], tap index fastest.
 *
 *   Low-rank factorisation (same summary, Parametrisatie item 1, and section
 *   Efficiente Trainingsimplementatie / Fused Low-Rank Kernel): the filter of
 *   token t is w(t) = z_t U with z of shape [B, T, R] and U of shape
 *   [R, (C/H) W]; column j of U is filter element (g, k) with j = g W + k.
 *   Here the product z U is formed explicitly, one token row at a time, in
 *   fp64 -- the naive path the fused kernel exists to avoid.
 *
 *   The backward pass is not written on the pages; it is the chain rule of
 *   the forward definition, written out term by term:
 *       dx[s,c]  = res*dy[s,c] + sum_{k: s+k<T} w[s+k, g(c), k] * dy[s+k, c]
 *       dw[t,g,k]= sum_{c in g, t-k>=0} dy[t,c] * x[t-k,c]
 *       dz[t,r]  = sum_j dw[t,j] * U[r,j]
 *       dU[r,j]  = sum_{b,t} z[b,t,r] * dw[b,t,j]
 *
 * Inputs may be fp64, fp32 or bf16 (decoded exactly to fp64 before use), so
 * the oracle sees the very values the GPU sees.  Every output is fp64.
 * Tensors are dense row-major: x, y, dy, dx [B,T,C]; w, dw [B,T,G,W];
 * z, dz [B,T,R]; U, dU [R, G*W].  A "row" is one token (b, t), numbered
 * b*T + t.
 *
 * Reductions run in a fixed order (taps k = 0..W-1, channels in increasing
 * order, tokens in increasing (b, t) order) whatever the thread count.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

/* Element i of a tensor stored as fp64, fp32 or bf16 (bf16 = top half of an
 * IEEE binary32, decoded exactly). */
static double ld(const void* p, int dt, int64_t i) {
  if (dt == ORC_F64) return ((const double*)p)[i];
  if (dt == ORC_F32) return (double)((const float*)p)[i];
  uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Where the filter of a token comes from: a materialised w (head-wise
 * parameterisation) or the product z_t U (low-rank parameterisation). */
typedef struct {
  const void* w; int wdt;            /* head-wise: w [B,T,G,W]            */
  const void* z; int zdt;            /* low-rank:  z [B,T,R]              */
  const double* U;                   /* low-rank:  U [R,G*W], decoded     */
  int64_t R;
  int lowrank;
} filters_t;

typedef struct {
  int64_t B, T, C, H, W, G;
  int residual;
} shape_t;

/* out[g*W + k] = w(row)[g, k] for every filter element of token `row`. */
static void filter_row(const filters_t* f, const shape_t* s, int64_t row,
                       double* out) {
  const int64_t GW = s->G * s->W;
  if (!f->lowrank) {
    for (int64_t j = 0; j < GW; ++j) out[j] = ld(f->w, f->wdt, row * GW + j);
    return;
  }
  /* w(t) = z_t U: a [1,R] x [R,G*W] product. */
  for (int64_t j = 0; j < GW; ++j) out[j] = 0.0;
  for (int64_t r = 0; r < f->R; ++r) {
    const double zr = ld(f->z, f->zdt, row * f->R + r);
    const double* Ur = f->U + r * GW;
    for (int64_t j = 0; j < GW; ++j) out[j] += zr * Ur[j];
  }
}

/* Forward, one token: y[b,t,:] = res*x[b,t,:] + sum_k w(t)[g(c),k] x[b,t-k,:]. */
static void fwd_row(const void* x, int xdt, const filters_t* f,
                    const shape_t* s, int64_t row, double* wt, double* yrow) {
  const int64_t t = row % s->T;
  filter_row(f, s, row, wt);
  for (int64_t c = 0; c < s->C; ++c) {
    const int64_t g = c / s->H;
    double acc = s->residual ? ld(x, xdt, row * s->C + c) : 0.0;
    for (int64_t k = 0; k < s->W; ++k) {
      if (t - k < 0) break;                 /* zero before the sequence start */
      acc += wt[g * s->W + k] * ld(x, xdt, (row - k) * s->C + c);
    }
    yrow[c] = acc;
  }
}

/* Backward w.r.t. x, one token s:
 * dx[b,s,c] = res*dy[b,s,c] + sum_{k: s+k<T} w(s+k)[g(c),k] dy[b,s+k,c].
 * wbuf holds W filter rows. */
static void dx_row(const void* dy, int dydt, const filters_t* f,
                   const shape_t* s, int64_t row, double* wbuf,
                   double* dxrow) {
  const int64_t t = row % s->T;
  const int64_t GW = s->G * s->W;
  for (int64_t k = 0; k < s->W; ++k)
    if (t + k < s->T) filter_row(f, s, row + k, wbuf + k * GW);
  for (int64_t c = 0; c < s->C; ++c) {
    const int64_t g = c / s->H;
    double acc = s->residual ? ld(dy, dydt, row * s->C + c) : 0.0;
    for (int64_t k = 0; k < s->W; ++k) {
      if (t + k >= s->T) break;             /* no output past the sequence end */
      acc += wbuf[k * GW + g * s->W + k] * ld(dy, dydt, (row + k) * s->C + c);
    }
    dxrow[c] = acc;
  }
}

/* Backward w.r.t. the filter, one token t:
 * dw[b,t,g,k] = sum_{c = gH}^{gH+H-1} dy[b,t,c] x[b,t-k,c]  (0 when t-k < 0). */
static void dw_row(const void* x, int xdt, const void* dy, int dydt,
                   const shape_t* s, int64_t row, double* dwrow) {
  const int64_t t = row % s->T;
  for (int64_t g = 0; g < s->G; ++g)
    for (int64_t k = 0; k < s->W; ++k) {
      double acc = 0.0;
      if (t - k >= 0)
        for (int64_t c = g * s->H; c < (g + 1) * s->H; ++c)
          acc += ld(dy, dydt, row * s->C + c) * ld(x, xdt, (row - k) * s->C + c);
      dwrow[g * s->W + k] = acc;
    }
}

/* Low-rank backward w.r.t. z, one token: dz[t,r] = sum_j dw[t,j] U[r,j]. */
static void dz_row(const double* dwrow, const double* U, int64_t R,
                   int64_t GW, double* dzrow) {
  for (int64_t r = 0; r < R; ++r) {
    double acc = 0.0;
    for (int64_t j = 0; j < GW; ++j) acc += dwrow[j] * U[r * GW + j];
    dzrow[r] = acc;
  }
}

static double* decode_all(const void* p, int dt, int64_t n) {
  double* out = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
  if (!out) return NULL;
  for (int64_t i = 0; i < n; ++i) out[i] = ld(p, dt, i);
  return out;
}

static int shape_ok(const shape_t* s) {
  return s->B >= 0 && s->T >= 0 && s->C >= 1 && s->H >= 1 && s->W >= 1 &&
         s->C % s->H == 0;
}

static shape_t mkshape(int64_t B, int64_t T, int64_t C, int64_t H, int64_t W,
                       int residual) {
  shape_t s = {B, T, C, H, W, H > 0 ? C / H : 0, residual};
  return s;
}

/* ------------------------------------------------------------------------ */
/* Exported entry points.  `rows` (optional) lists the tokens b*T+t to      */
/* evaluate; output row i then belongs to rows[i].  rows == NULL means all  */
/* B*T tokens in order.  Returns 0 on success, -1 on a bad argument or an   */
/* allocation failure.                                                      */
/* ------------------------------------------------------------------------ */

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

static int run_fwd(const void* x, int xdt, const filters_t* f,
                   const shape_t* s, const int64_t* rows, int64_t nrows,
                   double* y) {
  const int64_t GW = s->G * s->W;
  int fail = 0;
#pragma omp parallel
  {
    double* wt = (double*)malloc((size_t)GW * sizeof(double));
    if (!wt) {
#pragma omp atomic write
      fail = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t i = 0; i < nrows; ++i) {
        const int64_t row = rows ? rows[i] : i;
        fwd_row(x, xdt, f, s, row, wt, y + i * s->C);
      }
    }
    free(wt);
  }
  return fail ? -1 : 0;
}

/* Head-wise forward (Mechanisme + Parametrisatie item 2 + Plaatsing). */
int orc_headwise_fwd(const void* x, int xdt, const void* w, int wdt,
                     double* y, int64_t B, int64_t T, int64_t C, int64_t H,
                     int64_t W, int residual, const int64_t* rows,
                     int64_t nrows) {
  shape_t s = mkshape(B, T, C, H, W, residual);
  if (!shape_ok(&s)) return -1;
  filters_t f = {w, wdt, NULL, 0, NULL, 0, 0};
  return run_fwd(x, xdt, &f, &s, rows, rows ? nrows : B * T, y);
}

/* Low-rank forward: materialise each token's filter z_t U, then the
 * head-wise forward (Parametrisatie item 1; Fused Low-Rank Kernel). */
int orc_lowrank_fwd(const void* x, int xdt, const void* z, int zdt,
                    const void* U, int Udt, double* y, int64_t B, int64_t T,
                    int64_t C, int64_t H, int64_t W, int64_t R, int residual,
                    const int64_t* rows, int64_t nrows) {
  shape_t s = mkshape(B, T, C, H, W, residual);
  if (!shape_ok(&s) || R < 1) return -1;
  double* Ud = decode_all(U, Udt, R * s.G * W);
  if (!Ud) return -1;
  filters_t f = {NULL, 0, z, zdt, Ud, R, 1};
  int rc = run_fwd(x, xdt, &f, &s, rows, rows ? nrows : B * T, y);
  free(Ud);
  return rc;
}

/* Materialised low-rank filter w[b,t,g,k] = sum_r z[b,t,r] U[r, g*W+k]. */
int orc_lowrank_filters(const void* z, int zdt, const void* U, int Udt,
                        double* w, int64_t B, int64_t T, int64_t C, int64_t H,
                        int64_t W, int64_t R) {
  shape_t s = mkshape(B, T, C, H, W, 0);
  if (!shape_ok(&s) || R < 1) return -1;
  double* Ud = decode_all(U, Udt, R * s.G * W);
  if (!Ud) return -1;
  filters_t f = {NULL, 0, z, zdt, Ud, R, 1};
#pragma omp parallel for schedule(static)
  for (int64_t row = 0; row < B * T; ++row)
    filter_row(&f, &s, row, w + row * s.G * W);
  free(Ud);
  return 0;
}

/* Row-local backward outputs: dx (if dx != NULL), dw (if dw != NULL), and
 * for the low-rank parameterisation dz (if dz != NULL). */
static int run_bwd_rows(const void* x, int xdt, const void* dy, int dydt,
                        const filters_t* f, const shape_t* s,
                        const int64_t* rows, int64_t nrows, double* dx,
                        double* dw, double* dz) {
  const int64_t GW = s->G * s->W;
  int fail = 0;
#pragma omp parallel
  {
    double* wbuf = (double*)malloc((size_t)(s->W * GW) * sizeof(double));
    double* dwrow = (double*)malloc((size_t)GW * sizeof(double));
    if (!wbuf || !dwrow) {
#pragma omp atomic write
      fail = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t i = 0; i < nrows; ++i) {
        const int64_t row = rows ? rows[i] : i;
        if (dx) dx_row(dy, dydt, f, s, row, wbuf, dx + i * s->C);
        if (dw || dz) {
          double* d = dw ? dw + i * GW : dwrow;
          dw_row(x, xdt, dy, dydt, s, row, d);
          if (dz) dz_row(d, f->U, f->R, GW, dz + i * f->R);
        }
      }
    }
    free(wbuf);
    free(dwrow);
  }
  return fail ? -1 : 0;
}

/* Head-wise backward: dx [rows,C] and dw [rows,G,W]. */
int orc_headwise_bwd(const void* x, int xdt, const void* w, int wdt,
                     const void* dy, int dydt, double* dx, double* dw,
                     int64_t B, int64_t T, int64_t C, int64_t H, int64_t W,
                     int residual, const int64_t* rows, int64_t nrows) {
  shape_t s = mkshape(B, T, C, H, W, residual);
  if (!shape_ok(&s)) return -1;
  filters_t f = {w, wdt, NULL, 0, NULL, 0, 0};
  return run_bwd_rows(x, xdt, dy, dydt, &f, &s, rows, rows ? nrows : B * T,
                      dx, dw, NULL);
}

/* Low-rank backward, row-local part: dx [rows,C] (if dx != NULL), dz
 * [rows,R] (if dz != NULL), and (if dw != NULL) the intermediate dw
 * [rows,G,W]. */
int orc_lowrank_bwd_rows(const void* x, int xdt, const void* z, int zdt,
                         const void* U, int Udt, const void* dy, int dydt,
                         double* dx, double* dz, double* dw, int64_t B,
                         int64_t T, int64_t C, int64_t H, int64_t W, int64_t R,
                         int residual, const int64_t* rows, int64_t nrows) {
  shape_t s = mkshape(B, T, C, H, W, residual);
  if (!shape_ok(&s) || R < 1) return -1;
  double* Ud = decode_all(U, Udt, R * s.G * W);
  if (!Ud) return -1;
  filters_t f = {NULL, 0, z, zdt, Ud, R, 1};
  int rc = run_bwd_rows(x, xdt, dy, dydt, &f, &s, rows, rows ? nrows : B * T,
                        dx, dw, dz);
  free(Ud);
  return rc;
}

/* Low-rank backward w.r.t. U: dU[r,j] = sum over all tokens (b,t), in
 * increasing order, of z[b,t,r] dw[b,t,j].  Threads split the filter groups
 * g into blocks, so every element is summed in the same token order whatever
 * the thread count. */
int orc_lowrank_dU(const void* x, int xdt, const void* z, int zdt,
                   const void* dy, int dydt, double* dU, int64_t B, int64_t T,
                   int64_t C, int64_t H, int64_t W, int64_t R) {
  shape_t s = mkshape(B, T, C, H, W, 0);
  if (!shape_ok(&s) || R < 1) return -1;
  const int64_t G = s.G, GW = G * W, N = B * T;
  const int64_t GB = 32;                    /* groups per work block */
  const int64_t nblk = (G + GB - 1) / GB;
  for (int64_t i = 0; i < R * GW; ++i) dU[i] = 0.0;
  int fail = 0;
#pragma omp parallel
  {
    double* zrow = (double*)malloc((size_t)R * sizeof(double));
    double* dwb = (double*)malloc((size_t)(GB * W) * sizeof(double));
    if (!zrow || !dwb) {
#pragma omp atomic write
      fail = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t blk = 0; blk < nblk; ++blk) {
        const int64_t g0 = blk * GB;
        const int64_t g1 = g0 + GB < G ? g0 + GB : G;
        for (int64_t row = 0; row < N; ++row) {
          const int64_t t = row % T;
          /* dw[row, g, :] for the groups of this block, by definition */
          for (int64_t g = g0; g < g1; ++g)
            for (int64_t k = 0; k < W; ++k) {
              double acc = 0.0;
              if (t - k >= 0)
                for (int64_t c = g * H; c < (g + 1) * H; ++c)
                  acc += ld(dy, dydt, row * C + c) *
                         ld(x, xdt, (row - k) * C + c);
              dwb[(g - g0) * W + k] = acc;
            }
          for (int64_t r = 0; r < R; ++r) zrow[r] = ld(z, zdt, row * R + r);
          for (int64_t r = 0; r < R; ++r)
            for (int64_t g = g0; g < g1; ++g)
              for (int64_t k = 0; k < W; ++k)
                dU[r * GW + g * W + k] += zrow[r] * dwb[(g - g0) * W + k];
        }
      }
    }
    free(zrow);
    free(dwb);
  }
  return fail ? -1 : 0;
}
