/*
 * exact_oracle.c -- plain, slow CPU oracle for the exact residue GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's compute path may link,
 * load or call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * What it computes is the plain definition of each result, not the residue
 * method:
 *   - oracle_matmul_i64 / oracle_matmul_limbs: C = A * B over the integers by
 *     schoolbook summation in a wide two's-complement accumulator.  This is the
 *     integer the residue engine reconstructs ("exact-solve" and
 *     "enclosure-gemm" pages, Method: an exact integer matrix product recovered
 *     from residues modulo the primes below 256).
 *   - oracle_enclose_f64: the exact real inner product of binary64 operands,
 *     summed as an integer on a fixed binary grid, then the largest double <= it
 *     and the smallest double >= it, found by stepping with nextafter() and
 *     comparing exactly ("enclosure-gemm" page, Correctness: the reference is
 *     exact rational arithmetic; lo/hi must bracket the exact product and, when
 *     scaling is lossless, equal its floor and ceiling in the format).
 *   - oracle_enclose_f32: the same for binary32 operands, whose floor and
 *     ceiling are taken in binary32 ("enclosure-gemm" page, Usage: operands
 *     are float32 or float64; every binary32 value is also a binary64 value,
 *     so the exact sum is formed the same way).
 *   - oracle_interval_f64 / _f32: Rump's midpoint-radius product of interval
 *     matrices <Am, Ar> and <Bm, Br> (radii >= 0): the exact midpoint
 *     S = Am * Bm and the exact radius R = |Am| * Br + Ar * |Bm| + Ar * Br,
 *     then the largest value of the format <= S - R and the smallest >= S + R
 *     ("enclosure-gemm" page, Method: Rump's bound with its products and
 *     radius formed exactly, so the only overestimation is the bound's).
 *
 * Parallelism: OpenMP over output rows only; every entry is computed by the
 * same sequential loop over k.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef unsigned __int128 u128;
typedef __int128 i128;

#define MAXW 24 /* largest accumulator, in 64-bit words */

/* ------------------------------------------------------------------------ */
/* Integer product                                                          */
/* ------------------------------------------------------------------------ */

/* acc (nw words, two's complement) += p (np words, two's complement), mod 2^(64 nw). */
static void acc_add(uint64_t *acc, int nw, const uint64_t *p, int np) {
  uint64_t ext = (p[np - 1] >> 63) ? ~(uint64_t)0 : 0;
  uint64_t carry = 0;
  for (int i = 0; i < nw; i++) {
    uint64_t w = i < np ? p[i] : ext;
    u128 s = (u128)acc[i] + w + carry;
    acc[i] = (uint64_t)s;
    carry = (uint64_t)(s >> 64);
  }
}

/* Two's-complement negation of an n-word number, in place. */
static void negate(uint64_t *x, int n) {
  uint64_t carry = 1;
  for (int i = 0; i < n; i++) {
    u128 s = (u128)(~x[i]) + carry;
    x[i] = (uint64_t)s;
    carry = (uint64_t)(s >> 64);
  }
}

/* out (la+lb words, two's complement) = a (la limbs) * b (lb limbs), exactly.
 * Sign and magnitude are separated, the magnitudes multiplied by schoolbook,
 * and the sign applied at the end. */
static void mul_signed(const int64_t *a, int la, const int64_t *b, int lb, uint64_t *out) {
  uint64_t ma[8], mb[8];
  int sa = a[la - 1] < 0, sb = b[lb - 1] < 0;
  for (int i = 0; i < la; i++) ma[i] = (uint64_t)a[i];
  for (int i = 0; i < lb; i++) mb[i] = (uint64_t)b[i];
  if (sa) negate(ma, la);
  if (sb) negate(mb, lb);
  memset(out, 0, sizeof(uint64_t) * (size_t)(la + lb));
  for (int i = 0; i < la; i++) {
    uint64_t carry = 0;
    for (int j = 0; j < lb; j++) {
      u128 t = (u128)ma[i] * mb[j] + out[i + j] + carry;
      out[i + j] = (uint64_t)t;
      carry = (uint64_t)(t >> 64);
    }
    out[i + lb] = carry;
  }
  if (sa ^ sb) negate(out, la + lb);
}

/* Copy the low lc words of acc (nw words) to C; return 1 if the value does not
 * fit in lc two's-complement words. */
static int store_limbs(const uint64_t *acc, int nw, int64_t *C, int lc) {
  for (int i = 0; i < lc; i++) C[i] = (int64_t)(i < nw ? acc[i] : ((acc[nw - 1] >> 63) ? ~(uint64_t)0 : 0));
  uint64_t ext = ((uint64_t)C[lc - 1] >> 63) ? ~(uint64_t)0 : 0;
  for (int i = lc; i < nw; i++)
    if (acc[i] != ext) return 1;
  return 0;
}

static void set_threads(int threads) {
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
}

/*
 * C[r][j] (lc limbs) = sum_k A[row][k] * B[k][j] for int64 operands, exactly.
 * rows: the output rows to compute (NULL = all M rows, in order); C has nrows
 * rows.  Each product fits a signed 128-bit integer; the sum is held in 192
 * bits (a signed high word over an unsigned 128-bit low part).
 * Returns the number of entries that do not fit in lc limbs.
 */
long oracle_matmul_i64(const int64_t *A, const int64_t *B, int64_t *C, int M, int N, int K, int lc,
                       const int64_t *rows, int nrows, int threads) {
  if (!rows) nrows = M;
  set_threads(threads);
  long bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
  for (int r = 0; r < nrows; r++) {
    int64_t i = rows ? rows[r] : r;
    for (int j = 0; j < N; j++) {
      u128 lo = 0;
      int64_t hi = 0;
      for (int k = 0; k < K; k++) {
        i128 p = (i128)A[(size_t)i * K + k] * (i128)B[(size_t)k * N + j];
        u128 nlo = lo + (u128)p;
        hi += (p < 0 ? -1 : 0) + (nlo < lo ? 1 : 0);
        lo = nlo;
      }
      uint64_t acc[3] = {(uint64_t)lo, (uint64_t)(lo >> 64), (uint64_t)hi};
      bad += store_limbs(acc, 3, C + ((size_t)r * N + j) * lc, lc);
    }
  }
  return bad;
}

/*
 * Multi-limb operands: A[M][K][la], B[K][N][lb], little-endian 64-bit limbs,
 * two's complement with a signed top limb.  C[r][j] gets lc limbs.
 * Returns the number of entries that do not fit in lc limbs, or -1 on bad
 * arguments.
 */
long oracle_matmul_limbs(const int64_t *A, int la, const int64_t *B, int lb, int64_t *C, int lc, int M, int N,
                         int K, const int64_t *rows, int nrows, int threads) {
  if (la < 1 || lb < 1 || la > 8 || lb > 8 || lc < 1 || la + lb + 1 > MAXW) return -1;
  if (!rows) nrows = M;
  set_threads(threads);
  int nw = la + lb + 1;
  long bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
  for (int r = 0; r < nrows; r++) {
    int64_t i = rows ? rows[r] : r;
    uint64_t acc[MAXW], prod[16];
    for (int j = 0; j < N; j++) {
      memset(acc, 0, sizeof(acc));
      for (int k = 0; k < K; k++) {
        mul_signed(A + ((size_t)i * K + k) * la, la, B + ((size_t)k * N + j) * lb, lb, prod);
        acc_add(acc, nw, prod, la + lb);
      }
      bad += store_limbs(acc, nw, C + ((size_t)r * N + j) * lc, lc);
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* Exact fp64 inner product and outward rounding                             */
/* ------------------------------------------------------------------------ */

/* Every product of two binary64 values is m * 2^e with e >= -2148 and
 * m < 2^106; every such sum of fewer than 2^31 terms is below 2^2079.  A grid
 * with its least bit at 2^GRID_LSB and GRID_W words holds all of them, and
 * every finite double, exactly. */
#define GRID_LSB (-2200)
#define GRID_W 70

typedef struct {
  uint64_t w[GRID_W];
} grid_t; /* non-negative integer, least significant word first */

/* Decompose a finite double into (-1)^s * m * 2^e, m < 2^53, e >= -1074. */
static int decompose(double x, int *s, uint64_t *m, int *e) {
  uint64_t bits;
  memcpy(&bits, &x, 8);
  int be = (int)((bits >> 52) & 0x7FF);
  uint64_t frac = bits & (((uint64_t)1 << 52) - 1);
  if (be == 0x7FF) return -1;
  *s = (int)(bits >> 63);
  if (be == 0) {
    *m = frac;
    *e = -1074;
  } else {
    *m = frac | ((uint64_t)1 << 52);
    *e = be - 1075;
  }
  return 0;
}

/* g += v * 2^(sh - GRID_LSB) for v < 2^128, sh >= GRID_LSB. */
static void grid_add(grid_t *g, u128 v, int sh) {
  int off = sh - GRID_LSB;
  int wi = off / 64, b = off % 64;
  uint64_t parts[3];
  parts[0] = (uint64_t)v << b;
  parts[1] = b ? (uint64_t)(v >> (64 - b)) : (uint64_t)(v >> 64);
  parts[2] = b ? (uint64_t)((v >> 64) >> (64 - b)) : 0;
  uint64_t carry = 0;
  for (int i = wi; i < GRID_W; i++) {
    uint64_t add = (i - wi < 3) ? parts[i - wi] : 0;
    u128 s = (u128)g->w[i] + add + carry;
    g->w[i] = (uint64_t)s;
    carry = (uint64_t)(s >> 64);
    if (i - wi >= 2 && !carry) break;
  }
}

static int grid_cmp(const grid_t *a, const grid_t *b) {
  for (int i = GRID_W - 1; i >= 0; i--)
    if (a->w[i] != b->w[i]) return a->w[i] > b->w[i] ? 1 : -1;
  return 0;
}

static int grid_is_zero(const grid_t *a) {
  for (int i = 0; i < GRID_W; i++)
    if (a->w[i]) return 0;
  return 1;
}

/* r = a - b, assuming a >= b. */
static void grid_sub(const grid_t *a, const grid_t *b, grid_t *r) {
  uint64_t borrow = 0;
  for (int i = 0; i < GRID_W; i++) {
    u128 t = (u128)a->w[i] - b->w[i] - borrow;
    r->w[i] = (uint64_t)t;
    borrow = (uint64_t)((t >> 64) & 1);
  }
}

/* The exact value V = sgn * mag * 2^GRID_LSB, sgn in {-1, 0, 1}. */
typedef struct {
  int sgn;
  grid_t mag;
} exact_t;

/* Sign of (V - d) for a double d that may be infinite. */
static int cmp_exact_double(const exact_t *V, double d) {
  if (isinf(d)) return d > 0 ? -1 : 1;
  int s, e;
  uint64_t m;
  decompose(d, &s, &m, &e);
  int sd = m == 0 ? 0 : (s ? -1 : 1);
  if (V->sgn != sd) return V->sgn > sd ? 1 : -1;
  if (sd == 0) return 0;
  grid_t D;
  memset(&D, 0, sizeof(D));
  grid_add(&D, (u128)m, e);
  int c = grid_cmp(&V->mag, &D);
  return sd > 0 ? c : -c;
}

/* A double near V (any nearby value will do: it only starts the search). */
static double rough_value(const exact_t *V) {
  if (V->sgn == 0) return 0.0;
  int hw = GRID_W - 1;
  while (hw > 0 && V->mag.w[hw] == 0) hw--;
  double c = ldexp((double)V->mag.w[hw], 64 * hw + GRID_LSB);
  if (hw > 0) c += ldexp((double)V->mag.w[hw - 1], 64 * (hw - 1) + GRID_LSB);
  return V->sgn < 0 ? -c : c;
}

/* lo = the largest double (or -inf) <= V; hi = the smallest double (or +inf)
 * >= V.  V == 0 gives lo = hi = +0.0.  The starting guess is within a few
 * steps of V, so a walk longer than MAX_STEPS means the comparison is broken:
 * return -1 rather than loop. */
#define MAX_STEPS 64
static int outward(const exact_t *V, double *lo, double *hi) {
  if (V->sgn == 0) {
    *lo = 0.0;
    *hi = 0.0;
    return 0;
  }
  double c = rough_value(V);
  int steps = 0;
  while (cmp_exact_double(V, c) < 0) {
    c = nextafter(c, -INFINITY);
    if (++steps > MAX_STEPS) return -1;
  }
  for (;;) {
    if (c == INFINITY) break;
    double n = nextafter(c, INFINITY);
    if (cmp_exact_double(V, n) >= 0)
      c = n;
    else
      break;
    if (++steps > MAX_STEPS) return -1;
  }
  *lo = c;
  *hi = cmp_exact_double(V, c) == 0 ? c : nextafter(c, INFINITY);
  return 0;
}

/* The same search over the binary32 values: lo = the largest float (or -inf)
 * <= V, hi = the smallest float (or +inf) >= V.  Every float is a double, so
 * the comparison is the exact one above. */
static int outward_f32(const exact_t *V, float *lo, float *hi) {
  if (V->sgn == 0) {
    *lo = 0.0f;
    *hi = 0.0f;
    return 0;
  }
  double r = rough_value(V);
  float c = fabs(r) > FLT_MAX ? (r > 0 ? INFINITY : -INFINITY) : (float)r;
  int steps = 0;
  while (cmp_exact_double(V, (double)c) < 0) {
    c = nextafterf(c, -INFINITY);
    if (++steps > MAX_STEPS) return -1;
  }
  for (;;) {
    if (c == INFINITY) break;
    float n = nextafterf(c, INFINITY);
    if (cmp_exact_double(V, (double)n) >= 0)
      c = n;
    else
      break;
    if (++steps > MAX_STEPS) return -1;
  }
  *lo = c;
  *hi = cmp_exact_double(V, (double)c) == 0 ? c : nextafterf(c, INFINITY);
  return 0;
}

/* The exact value of row i of A[M][K] times column j of B[K][N]. */
static void exact_entry(const double *A, const double *B, int64_t i, int j, int N, int K, exact_t *V) {
  grid_t pos, neg;
  memset(&pos, 0, sizeof(pos));
  memset(&neg, 0, sizeof(neg));
  for (int k = 0; k < K; k++) {
    int sa, sb, ea, eb;
    uint64_t ma, mb;
    decompose(A[(size_t)i * K + k], &sa, &ma, &ea);
    decompose(B[(size_t)k * N + j], &sb, &mb, &eb);
    if (ma == 0 || mb == 0) continue;
    grid_add((sa ^ sb) ? &neg : &pos, (u128)ma * mb, ea + eb);
  }
  int c = grid_cmp(&pos, &neg);
  if (c >= 0)
    grid_sub(&pos, &neg, &V->mag);
  else
    grid_sub(&neg, &pos, &V->mag);
  V->sgn = grid_is_zero(&V->mag) ? 0 : c;
}

/* Rows of the bracket; lo/hi are double (f32 = 0) or float (f32 = 1). */
static int enclose_rows(const double *A, const double *B, void *lo, void *hi, int f32, int M, int N, int K,
                        const int64_t *rows, int nrows, int threads) {
  int broken = 0;
  (void)M;
  set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : broken)
  for (int r = 0; r < nrows; r++) {
    int64_t i = rows ? rows[r] : r;
    for (int j = 0; j < N; j++) {
      exact_t V;
      exact_entry(A, B, i, j, N, K, &V);
      size_t o = (size_t)r * N + j;
      if (f32)
        broken |= outward_f32(&V, (float *)lo + o, (float *)hi + o) != 0;
      else
        broken |= outward(&V, (double *)lo + o, (double *)hi + o) != 0;
    }
  }
  return broken ? -2 : 0;
}

/*
 * lo[r][j], hi[r][j] for row rows[r] (NULL = all rows) of the exact product
 * A[M][K] * B[K][N] of binary64 matrices.  Returns 0, -1 if an operand entry
 * is not finite, or -2 if the outward search did not converge (a defect).
 */
int oracle_enclose_f64(const double *A, const double *B, double *lo, double *hi, int M, int N, int K,
                       const int64_t *rows, int nrows, int threads) {
  if (!rows) nrows = M;
  for (size_t t = 0; t < (size_t)M * K; t++)
    if (!isfinite(A[t])) return -1;
  for (size_t t = 0; t < (size_t)K * N; t++)
    if (!isfinite(B[t])) return -1;
  return enclose_rows(A, B, lo, hi, 0, M, N, K, rows, nrows, threads);
}

/* The same for binary32 matrices and binary32 bounds.  Returns -3 if the
 * double copies of the operands cannot be allocated. */
int oracle_enclose_f32(const float *A, const float *B, float *lo, float *hi, int M, int N, int K,
                       const int64_t *rows, int nrows, int threads) {
  if (!rows) nrows = M;
  for (size_t t = 0; t < (size_t)M * K; t++)
    if (!isfinite(A[t])) return -1;
  for (size_t t = 0; t < (size_t)K * N; t++)
    if (!isfinite(B[t])) return -1;
  double *Ad = malloc(((size_t)M * K + 1) * sizeof(double));
  double *Bd = malloc(((size_t)K * N + 1) * sizeof(double));
  int rc = -3;
  if (Ad && Bd) {
    for (size_t t = 0; t < (size_t)M * K; t++) Ad[t] = (double)A[t]; /* exact */
    for (size_t t = 0; t < (size_t)K * N; t++) Bd[t] = (double)B[t];
    rc = enclose_rows(Ad, Bd, lo, hi, 1, M, N, K, rows, nrows, threads);
  }
  free(Ad);
  free(Bd);
  return rc;
}

/* acc += sign * v, exactly (sign-magnitude). */
static void exact_add(exact_t *acc, const exact_t *v, int sign) {
  int vs = v->sgn * sign;
  if (vs == 0) return;
  if (acc->sgn == 0) {
    acc->mag = v->mag;
    acc->sgn = vs;
    return;
  }
  if (acc->sgn == vs) {
    uint64_t carry = 0;
    for (int i = 0; i < GRID_W; i++) {
      u128 t = (u128)acc->mag.w[i] + v->mag.w[i] + carry;
      acc->mag.w[i] = (uint64_t)t;
      carry = (uint64_t)(t >> 64);
    }
    return;
  }
  int c = grid_cmp(&acc->mag, &v->mag);
  if (c == 0) {
    memset(&acc->mag, 0, sizeof(acc->mag));
    acc->sgn = 0;
  } else if (c > 0) {
    grid_sub(&acc->mag, &v->mag, &acc->mag);
  } else {
    grid_t r;
    grid_sub(&v->mag, &acc->mag, &r);
    acc->mag = r;
    acc->sgn = vs;
  }
}

/* Interval rows from double copies of the operands (radii already checked). */
static int interval_rows(const double *Am, const double *Ar, const double *Bm, const double *Br, void *lo, void *hi,
                         int f32, int M, int N, int K, const int64_t *rows, int nrows, int threads) {
  double *aAm = malloc(((size_t)M * K + 1) * sizeof(double));
  double *aBm = malloc(((size_t)K * N + 1) * sizeof(double));
  if (!aAm || !aBm) {
    free(aAm);
    free(aBm);
    return -3;
  }
  for (size_t t = 0; t < (size_t)M * K; t++) aAm[t] = fabs(Am[t]);
  for (size_t t = 0; t < (size_t)K * N; t++) aBm[t] = fabs(Bm[t]);
  int broken = 0;
  set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : broken)
  for (int r = 0; r < nrows; r++) {
    int64_t i = rows ? rows[r] : r;
    for (int j = 0; j < N; j++) {
      exact_t S, R, t, L, H;
      exact_entry(Am, Bm, i, j, N, K, &S);
      exact_entry(aAm, Br, i, j, N, K, &R);
      exact_entry(Ar, aBm, i, j, N, K, &t);
      exact_add(&R, &t, 1);
      exact_entry(Ar, Br, i, j, N, K, &t);
      exact_add(&R, &t, 1);
      L = S;
      exact_add(&L, &R, -1);
      H = S;
      exact_add(&H, &R, 1);
      size_t o = (size_t)r * N + j;
      if (f32) {
        float unused;
        broken |= outward_f32(&L, (float *)lo + o, &unused) != 0;
        broken |= outward_f32(&H, &unused, (float *)hi + o) != 0;
      } else {
        double unused;
        broken |= outward(&L, (double *)lo + o, &unused) != 0;
        broken |= outward(&H, &unused, (double *)hi + o) != 0;
      }
    }
  }
  free(aAm);
  free(aBm);
  return broken ? -2 : 0;
}

/* Checks for the interval operands: -1 for a non-finite entry, -4 for a
 * negative radius (a sign bit on a nonzero radius), else 0. */
static int check_interval(const double *Am, const double *Ar, size_t n) {
  for (size_t t = 0; t < n; t++) {
    if (!isfinite(Am[t]) || !isfinite(Ar[t])) return -1;
    if (Ar[t] < 0) return -4;
  }
  return 0;
}

/*
 * lo, hi [nrows][N] of the interval product <Am, Ar> * <Bm, Br> for binary64
 * operands (A [M][K], B [K][N]).  Returns 0, -1 (non-finite entry), -2 (the
 * outward search did not converge: a defect), -3 (no memory), -4 (negative
 * radius).
 */
int oracle_interval_f64(const double *Am, const double *Ar, const double *Bm, const double *Br, double *lo,
                        double *hi, int M, int N, int K, const int64_t *rows, int nrows, int threads) {
  if (!rows) nrows = M;
  int c = check_interval(Am, Ar, (size_t)M * K);
  if (!c) c = check_interval(Bm, Br, (size_t)K * N);
  if (c) return c;
  return interval_rows(Am, Ar, Bm, Br, lo, hi, 0, M, N, K, rows, nrows, threads);
}

/* The same for binary32 operands and binary32 bounds. */
int oracle_interval_f32(const float *Am, const float *Ar, const float *Bm, const float *Br, float *lo, float *hi,
                        int M, int N, int K, const int64_t *rows, int nrows, int threads) {
  if (!rows) nrows = M;
  size_t na = (size_t)M * K, nb = (size_t)K * N;
  double *d = malloc((2 * na + 2 * nb + 1) * sizeof(double));
  if (!d) return -3;
  double *dAm = d, *dAr = d + na, *dBm = d + 2 * na, *dBr = d + 2 * na + nb;
  for (size_t t = 0; t < na; t++) {
    dAm[t] = (double)Am[t]; /* exact */
    dAr[t] = (double)Ar[t];
  }
  for (size_t t = 0; t < nb; t++) {
    dBm[t] = (double)Bm[t];
    dBr[t] = (double)Br[t];
  }
  int c = check_interval(dAm, dAr, na);
  if (!c) c = check_interval(dBm, dBr, nb);
  if (!c) c = interval_rows(dAm, dAr, dBm, dBr, lo, hi, 1, M, N, K, rows, nrows, threads);
  free(d);
  return c;
}

/* Number of OpenMP threads a parallel region will use. */
int oracle_threads(int threads) {
  set_threads(threads);
#ifdef _OPENMP
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
  return n;
#else
  return 1;
#endif
}
