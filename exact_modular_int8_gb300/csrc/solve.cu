// solve.cu -- exact rational solution of an integer system A X = B on the
// residue engine ("exact-solve" page, Method):
//   1. A^-1 mod q for every prime q < 256 at once, by Gauss-Jordan
//      elimination over all primes, blocked: per block of pivots, one panel
//      factorisation in shared memory and one tensor-core update;
//   2. Dixon's p-adic lift with the modulus P = the product of the primes that
//      do not divide det(A): X_i = A^-1 R_i mod P (per prime, then balanced
//      Garner into the wide base-P digit), R_{i+1} = (R_i - A X_i) / P formed
//      in one 64-bit limb as (R_i - A X_i) P^-1 mod 2^64 (P odd);
//   3. rational reconstruction of a few components on host threads for the
//      common denominator, then every component's value and numerator on the
//      GPU (recon.cu).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "bigint.h"
#include "recon.h"
#include "rg_garner.cuh"
#include "rg_kernels.h"

namespace rg {
namespace {

// Tables of the prime sequence a solve lifts with (a subset of the residue
// base), uploaded once the inverse shows which primes divide det(A).
__constant__ Tables c_sol;
// The same tables in global memory, for reads whose index differs between the
// lanes of a warp (divergent constant-memory reads are serialised).
__device__ Tables g_sol;
__constant__ Tables c_all;  // the full base, for the inverse

struct SolTab {
  __device__ static __forceinline__ const Tables& t() { return c_sol; }
};

constexpr int kMaxSolveN = 8192;
constexpr int kW = 11;  // 32-bit words of a base-P digit (|x| < P / 2 < 2^333)

// ---------------------------------------------------------------------------
// Norms and range: row and column sums of squares of A, column sums of
// squares of B (fp64, for the Hadamard bounds) and max |A|.
// ---------------------------------------------------------------------------
// One warp per row of A (its sum of squares and max |A|), then one thread per
// column of B.
__global__ void __launch_bounds__(256) norms_kernel(const int64_t* __restrict__ A, const int64_t* __restrict__ B,
                                                    int n, int c, double* rows, double* bcols,
                                                    unsigned long long* maxabs) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp < n) {
    double s = 0.0;
    unsigned long long m = 0;
    for (int k = lane; k < n; k += 32) {
      const long long v = A[(long long)warp * n + k];
      const double d = (double)v;
      s = fma(d, d, s);
      const unsigned long long a = v < 0 ? 0ull - (unsigned long long)v : (unsigned long long)v;
      m = a > m ? a : m;
    }
    for (int o = 16; o; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      const unsigned long long t = __shfl_xor_sync(0xffffffffu, m, o);
      m = t > m ? t : m;
    }
    if (lane == 0) {
      rows[warp] = s;
      atomicMax(maxabs, m);
    }
  }
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < c) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) {
      const double d = (double)B[(long long)i * c + t];
      s = fma(d, d, s);
    }
    bcols[t] = s;
  }
}

// Column sums of squares of A over the rows [y * rows_per, (y + 1) * rows_per)
// of chunk y = blockIdx.y, one thread per column (a row of A is read by
// consecutive threads): part[y][t].
__global__ void __launch_bounds__(256) col_norms_part_kernel(const int64_t* __restrict__ A, int n, int rows_per,
                                                             double* __restrict__ part) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  const int i0 = blockIdx.y * rows_per, i1 = min(n, i0 + rows_per);
  double s = 0.0;
  for (int i = i0; i < i1; ++i) {
    const double d = (double)A[(long long)i * n + t];
    s = fma(d, d, s);
  }
  part[(size_t)blockIdx.y * n + t] = s;
}

// cols[t] = the chunks' partial sums of column t, added in chunk order.
__global__ void __launch_bounds__(256) col_norms_sum_kernel(const double* __restrict__ part, int n, int chunks,
                                                            double* __restrict__ cols) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  double s = 0.0;
  for (int y = 0; y < chunks; ++y) s += part[(size_t)y * n + t];
  cols[t] = s;
}

// ---------------------------------------------------------------------------
// Batched modular inverse ("exact-solve", Method: A^-1 mod q for every prime
// by Gauss-Jordan, each launch spanning all primes; here blocked, below).
// M[p] is A mod q_p in [0, q), n x n bytes, inverted in place: at step k the
// pivot row is the first row >= k with a nonzero in column k; it is swapped
// up, scaled by the pivot's inverse (its own column entry becoming that
// inverse), and every other row i subtracts f_i times it, f_i its old column
// entry (the column entry itself becoming -f_i times the inverse).  The row
// swaps become column swaps of the result, undone at the end.  A prime with
// no pivot at some step divides det(A) and is marked singular.
// ---------------------------------------------------------------------------

// x mod q in [0, q) for an int64 x, by the split's byte weights (wbyte,
// wword of the full base, prime index p).
__device__ __forceinline__ int residue_i64(long long x, int p) {
  const unsigned long long u = (unsigned long long)x;
  int acc = x < 0 ? -c_all.wword[p][2] : 0;
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"((uint32_t)u), "r"(c_all.wbyte[p][0]));
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"((uint32_t)(u >> 32)), "r"(c_all.wbyte[p][1]));
  const float q = c_all.qf[p];
  float r = bal_mod_small(int_to_float_exact(acc), q, c_all.invq[p]);  // |acc| < 2^20
  return (int)(r < 0.0f ? r + q : r);
}

// M[p] = diag(A, I) mod q_p, of order nE = n rounded up to 16 (the padding
// keeps every row a whole number of 16-byte vectors; the inverse of diag(A, I)
// is diag(A^-1, I), and the same primes divide both determinants).
__global__ void __launch_bounds__(256) gj_init_kernel(const int64_t* __restrict__ A, int n, int nE,
                                                      uint8_t* __restrict__ M, int* __restrict__ rowsrc) {
  const long long nn = (long long)nE * nE;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < (long long)kNumPrimes * nE;
       e += (long long)gridDim.x * blockDim.x)
    rowsrc[e] = (int)(e % nE);
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < nn; e += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(e / nE), j = (int)(e - (long long)i * nE);
    const long long x = (i < n && j < n) ? A[(long long)i * n + j] : (i == j ? 1 : 0);
    for (int p = 0; p < kNumPrimes; ++p) M[p * nn + e] = (uint8_t)residue_i64(x, p);
  }
}

// (a * b) mod q for a, b in [0, q), q < 256.
__device__ __forceinline__ int mulmod(int a, int b, float q, float iq) {
  float r = bal_mod_small((float)(a * b), q, iq);
  return (int)(r < 0.0f ? r + q : r);
}

__device__ __forceinline__ int invmod(int a, int q) {  // a^(q-2) mod q, a != 0
  int r = 1, b = a, e = q - 2;
  while (e) {
    if (e & 1) r = r * b % q;
    b = b * b % q;
    e >>= 1;
  }
  return r;
}

// ---------------------------------------------------------------------------
// Blocked Gauss-Jordan.  The pivots are taken in blocks J = [k0, k0 + b).  The
// steps of the in-place elimination for one pivot k are: the first nonzero at
// or below the diagonal of column k is the pivot, its row is swapped with row
// k, row k is scaled by the pivot's inverse (its entry in column k becoming
// that inverse), and every other row loses its multiple f of row k (its
// entry in column k becoming -f / pivot).  For a column outside J, the b steps
// of a block compose to one linear map: with Xs the column after the block's
// row swaps, Xs_J its entries in the pivot rows, and W the panel (the columns
// of J, all rows) after the b steps,
//     X <- Xs with the pivot rows zeroed + W Xs_J.
// W differs from the identity only in J's columns, so the map is a product of
// inner dimension b per prime.  The panel kernel runs the b steps on the
// panel alone, in shared memory; the update kernel forms the product with
// the INT8 tensor-core MMA on balanced residues.  Both keep the unblocked
// elimination's pivots, so the result and the recorded swaps are the same.
// ---------------------------------------------------------------------------

constexpr int kPanelThreads = 1024;
constexpr int kSwapCols = 256;                // columns per chunk of the panel kernel's row-permutation pass
constexpr int kSwapStride = kSwapCols + 4;    // an odd number of words: column reads across rows hit distinct banks
constexpr size_t kPanelSmemLimit = 200u << 10;

// Dynamic shared memory of the panel kernel for order nE and width b: the
// panel (rows of b + 4 bytes, an odd number of words, so that one thread per
// row reads without bank conflicts), then the source-row index of every row.
size_t panel_smem(int nE, int b) { return (size_t)nE * (b + 4) + (size_t)nE * 2; }

// The panel kernel's shape for order nE: the block width B (its panel of
// nE x (B + 4) bytes within kPanelSmemLimit), the sub-block S and the rows
// per thread RPT = nE / 1024 rounded up, with RPT x S <= 32 entries held in
// registers.
struct PanelCfg {
  int B, S, RPT;
};
PanelCfg panel_cfg(int nE) {
  if (nE <= kPanelThreads) return {64, 16, 1};
  if (nE <= 2 * kPanelThreads) return {64, 8, 2};
  if (nE <= 4 * kPanelThreads) return {32, 8, 4};
  return {16, 4, 8};
}

// Reduction of |x| <= 2^23 into [0, q).
__device__ __forceinline__ int red_q(int x, float qf, float iq) {
  const float v = bal_mod_small((float)x, qf, iq);
  return (int)(v < 0.0f ? v + qf : v);
}

// One block per prime.  Factors the panel of block [k0, k0 + b), b <= B a
// multiple of 16 (the steps above, on J's columns only), writes it back
// (uint8 in [0, q)) and as balanced fp16 rows of kb entries, Wb[p][i][t]
// (zero for t >= b), then applies the block's row swaps to the columns outside J:
// the rows the swaps move out of J get their final contents, and the pivot
// rows' contents go, balanced and transposed, to RT[p][j][t] (zero in J's
// columns and for t >= b).  rowsrc[p][i] follows the original row that row i
// holds.  A prime without a pivot sets sing[p].
//
// The panel itself is factored in sub-blocks of S pivots by the same
// composition: each thread holds the S sub-block entries of its RPT rows in
// registers, unreduced during the sub-block's steps (each step adds at most
// 250^2 in magnitude: |x| < 2^20 after 16), reducing only the entry that
// decides the multiplier and the next pivot; then the other panel columns
// take X <- Xs with the sub-block's pivot rows zeroed + W_S Xs_S by dp4a.
template <int B, int S, int RPT>
__global__ void __launch_bounds__(kPanelThreads) gj_panel_kernel(uint8_t* __restrict__ M, int nE, int k0, int b,
                                                                 int kb, __half* __restrict__ Wb,
                                                                 uint16_t* __restrict__ gsrc, int* __restrict__ sing) {
  static_assert(S % 4 == 0 && B % S == 0 && 16 % S == 0, "sub-blocks of whole words dividing every panel width");
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ uint8_t invtab[256];
  __shared__ __align__(16) int spiv[S];
  __shared__ __align__(16) uint8_t Rt[B * S];  // [panel column][t]: a sub-block's pivot rows, transposed
  __shared__ int s_piv[2];
  constexpr int PS = B + 4;  // panel row stride: an odd number of words
  constexpr int SW = S / 4;
  const int p = blockIdx.x, tid = threadIdx.x;
  const int q = c_all.q[p], h = (q - 1) / 2;
  const float qf = c_all.qf[p], iq = c_all.invq[p];
  uint8_t* pan = sm;
  const size_t body = (size_t)nE * PS;  // nE is a multiple of 16: src stays 2-byte aligned
  uint16_t* src = reinterpret_cast<uint16_t*>(sm + body);  // row i holds original row src[i]
  for (int a = tid; a < 256; a += kPanelThreads) invtab[a] = (a > 0 && a < q) ? (uint8_t)invmod(a, q) : 0;
  for (int i = tid; i < nE; i += kPanelThreads) src[i] = (uint16_t)i;
  if (tid == 0) {
    s_piv[0] = s_piv[1] = nE;
  }
  wait_for_predecessor();
  if (sing[p]) return;
  uint8_t* Mp = M + (size_t)p * nE * nE;
  const int vpr = b / 16;  // 16-byte vectors per panel row in M
  for (int e = tid; e < nE * vpr; e += kPanelThreads) {
    const int i = e / vpr, v = e - i * vpr;
    const uint4 w = *reinterpret_cast<const uint4*>(Mp + (size_t)i * nE + k0 + v * 16);
    uint32_t* d = reinterpret_cast<uint32_t*>(pan + (size_t)i * PS + v * 16);
    d[0] = w.x;
    d[1] = w.y;
    d[2] = w.z;
    d[3] = w.w;
  }
  __syncthreads();
  for (int c0 = 0; c0 < b; c0 += S) {  // sub-block: panel columns [c0, c0 + S), pivots k0 + c0 + tt
    const int kc0 = k0 + c0;
    int a[RPT][S];
    int rid[RPT];  // the panel row each register slot holds; a row swap exchanges two slots' ids
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int row = tid + k * kPanelThreads;
      rid[k] = row;
#pragma unroll
      for (int w = 0; w < SW; ++w) {
        const uint32_t x = row < nE ? reinterpret_cast<const uint32_t*>(pan + (size_t)row * PS + c0)[w] : 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) a[k][4 * w + e] = (int)((x >> (8 * e)) & 255u);
      }
      if (row >= kc0 && row < nE && a[k][0] != 0) atomicMin(&s_piv[c0 & 1], row);
    }
    __syncthreads();
#pragma unroll
    for (int tt = 0; tt < S; ++tt) {
      const int tg = c0 + tt, kc = k0 + tg;
      const int r = s_piv[tg & 1];
      if (r >= nE) {  // no pivot: q_p divides det(A) (the same value in every thread)
        if (tid == 0) sing[p] = 1;
        return;
      }
#pragma unroll
      for (int k = 0; k < RPT; ++k) {
        rid[k] = rid[k] == kc ? r : (rid[k] == r ? kc : rid[k]);
        if (rid[k] == kc) {  // the pivot row: reduced, scaled by the pivot's inverse
          const int inv = invtab[red_q(a[k][tt], qf, iq)];
#pragma unroll
          for (int j = 0; j < S; ++j) {
            const int v = j == tt ? inv : mulmod(red_q(a[k][j], qf, iq), inv, qf, iq);
            a[k][j] = v;
            spiv[j] = v;
          }
        }
      }
      if (r != kc) {
        if (tid < b / 4 && (tid < c0 / 4 || tid >= c0 / 4 + SW)) {  // the panel's other columns
          uint32_t* x = reinterpret_cast<uint32_t*>(pan + (size_t)kc * PS) + tid;
          uint32_t* y = reinterpret_cast<uint32_t*>(pan + (size_t)r * PS) + tid;
          const uint32_t t0 = *x;
          *x = *y;
          *y = t0;
        } else if (tid == kPanelThreads - 1) {
          const uint16_t t0 = src[kc];
          src[kc] = src[r];
          src[r] = t0;
        }
      }
      if (tid == 0) s_piv[(tg + 1) & 1] = nE;  // read last before the previous step's end
      __syncthreads();
      // every other row loses f times the pivot row (its entry tt becoming -f * inverse); the
      // next column's reduced entry names a pivot candidate for the next step
#pragma unroll
      for (int k = 0; k < RPT; ++k) {
        const int row = rid[k];
        if (row >= nE || row == kc) continue;
        const int f = red_q(a[k][tt], qf, iq);
        if (f) {
          a[k][tt] = 0;
#pragma unroll
          for (int j = 0; j < S; ++j) a[k][j] -= f * spiv[j];
        }
        if (tt + 1 < S && row > kc && red_q(a[k][tt + 1], qf, iq) != 0) atomicMin(&s_piv[(tg + 1) & 1], row);
      }
      __syncthreads();
    }
    // the sub-block back into the panel, reduced, each slot into the row it holds
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int row = rid[k];
      if (row >= nE) continue;
#pragma unroll
      for (int w = 0; w < SW; ++w) {
        uint32_t x = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) x |= (uint32_t)red_q(a[k][4 * w + e], qf, iq) << (8 * e);
        reinterpret_cast<uint32_t*>(pan + (size_t)row * PS + c0)[w] = x;
      }
    }
    if (b == S) break;  // no other panel columns
    __syncthreads();
    for (int e = tid; e < b * S; e += kPanelThreads) {
      const int j = e / S, t = e - j * S;
      Rt[e] = pan[(size_t)(kc0 + t) * PS + j];
    }
    __syncthreads();
    // the other panel columns: X <- (0 in the sub-block's pivot rows, else X) + W_S Rt (sums < 16 * 250^2)
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int row = tid + k * kPanelThreads;
      if (row >= nE) continue;
      uint32_t* prow = reinterpret_cast<uint32_t*>(pan + (size_t)row * PS);
      uint32_t wv[SW];
#pragma unroll
      for (int u = 0; u < SW; ++u) wv[u] = prow[c0 / 4 + u];
      const bool pivot_row = row >= kc0 && row < kc0 + S;
      for (int w = 0; w < b / 4; ++w) {
        if (w >= c0 / 4 && w < c0 / 4 + SW) continue;
        const uint32_t base = pivot_row ? 0u : prow[w];
        uint32_t out = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t* rt = reinterpret_cast<const uint32_t*>(Rt + (4 * w + e) * S);
          int x = (int)((base >> (8 * e)) & 255u);
#pragma unroll
          for (int u = 0; u < SW; ++u) asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(x) : "r"(wv[u]), "r"(rt[u]));
          out |= (uint32_t)red_q(x, qf, iq) << (8 * e);
        }
        prow[w] = out;
      }
    }
    __syncthreads();
  }
  __syncthreads();
  // the panel back into M, and balanced into Wb
  for (int e = tid; e < nE * vpr; e += kPanelThreads) {
    const int i = e / vpr, v = e - i * vpr;
    const uint32_t* s = reinterpret_cast<const uint32_t*>(pan + (size_t)i * PS + v * 16);
    *reinterpret_cast<uint4*>(Mp + (size_t)i * nE + k0 + v * 16) = make_uint4(s[0], s[1], s[2], s[3]);
  }
  __half* Wp = Wb + (size_t)p * nE * kb;
  const int kp = kb / 2;  // pairs of fp16 per row
  for (int e = tid; e < nE * kp; e += kPanelThreads) {
    const int i = e / kp, t = 2 * (e - i * kp);
    __half2 out = __floats2half2_rn(0.0f, 0.0f);
    if (t < b) {
      int v0 = pan[(size_t)i * PS + t], v1 = pan[(size_t)i * PS + t + 1];
      v0 = v0 > h ? v0 - q : v0;
      v1 = v1 > h ? v1 - q : v1;
      out = __floats2half2_rn((float)v0, (float)v1);  // |v| <= 125: exact
    }
    *reinterpret_cast<__half2*>(Wp + (size_t)i * kb + t) = out;
  }
  // the original row each row of the panel holds, for the swap pass
  for (int x = tid; x < nE; x += kPanelThreads) gsrc[(size_t)p * nE + x] = src[x];
  allow_dependents();
}

// After a block's panel: its row swaps (gsrc[p][i], the original row that row
// i holds after them) applied to the columns outside J.  The rows the swaps
// move out of J get their final contents, the pivot rows' contents go,
// balanced, transposed and as fp16, to RT[p][j][t] (zero in J's columns and
// for t >= b), and rowsrc[p][i] follows the original row that row i of M
// holds.  One block per prime (blockIdx.x) and chunk of kSwapCols columns
// (blockIdx.y); it must run after every update of the previous block.
constexpr int kMaxPanel = 64;
size_t swap_smem(int nE) { return (size_t)2 * kMaxPanel * kSwapStride + (size_t)nE * 2; }

__global__ void __launch_bounds__(kPanelThreads) gj_swap_kernel(uint8_t* __restrict__ M, int nE, int k0, int b, int kb,
                                                                const uint16_t* __restrict__ gsrc,
                                                                __half* __restrict__ RT, int* __restrict__ rowsrc,
                                                                const int* __restrict__ sing) {
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ int s_nd;
  __shared__ int s_disp[kMaxPanel];
  __shared__ int s_rs[2 * kMaxPanel];
  const int p = blockIdx.x, tid = threadIdx.x;
  const int q = c_all.q[p], h = (q - 1) / 2;
  uint8_t* buf = sm;  // row chunks: slot s < b the pivot row k0 + s, slot b + u the displaced row s_disp[u]
  uint16_t* src = reinterpret_cast<uint16_t*>(sm + (size_t)2 * kMaxPanel * kSwapStride);
  if (tid == 0) s_nd = 0;
  wait_for_predecessor();
  if (sing[p]) return;
  for (int x = tid; x < nE; x += kPanelThreads) src[x] = gsrc[(size_t)p * nE + x];
  __syncthreads();
  uint8_t* Mp = M + (size_t)p * nE * nE;
  const int kp = kb / 2;  // pairs of fp16 per RT row
  // rows outside J that the swaps changed (at most one per swap)
  for (int i = tid; i < nE; i += kPanelThreads)
    if ((i < k0 || i >= k0 + b) && src[i] != i) {
      const int u = atomicAdd(&s_nd, 1);
      if (u < b) s_disp[u] = i;  // always: each swap moves at most one row outside J
    }
  __syncthreads();
  const int nd = min(s_nd, b);
  const int slots = b + nd;  // slot s < b: pivot row k0 + s; slot b + u: displaced row s_disp[u]
  // the original row each row of M holds: rowsrc[i] <- rowsrc[src[i]] for the rows the swaps changed
  if (blockIdx.y == 0) {
    int* rs = rowsrc + (size_t)p * nE;
    for (int s = tid; s < slots; s += kPanelThreads) s_rs[s] = rs[src[s < b ? k0 + s : s_disp[s - b]]];
    __syncthreads();
    for (int s = tid; s < slots; s += kPanelThreads) rs[s < b ? k0 + s : s_disp[s - b]] = s_rs[s];
  }
  __half* Rp = RT + (size_t)p * nE * kb;
  {
    const int c0 = blockIdx.y * kSwapCols;
    const int cw = min(kSwapCols, nE - c0), cwords = cw / 4;  // cw is a multiple of 16
    for (int e = tid; e < slots * cwords; e += kPanelThreads) {
      const int s = e / cwords, w = e - s * cwords;
      const int from = src[s < b ? k0 + s : s_disp[s - b]];
      reinterpret_cast<uint32_t*>(buf + (size_t)s * kSwapStride)[w] =
          reinterpret_cast<const uint32_t*>(Mp + (size_t)from * nE + c0)[w];
    }
    __syncthreads();
    for (int e = tid; e < nd * cwords; e += kPanelThreads) {
      const int u = e / cwords, w = e - u * cwords;
      const int col = c0 + 4 * w;
      if (col >= k0 && col < k0 + b) continue;  // the panel's columns already hold W
      reinterpret_cast<uint32_t*>(Mp + (size_t)s_disp[u] * nE + c0)[w] =
          reinterpret_cast<const uint32_t*>(buf + (size_t)(b + u) * kSwapStride)[w];
    }
    for (int e = tid; e < cw * kp; e += kPanelThreads) {
      const int c = e / kp, t = 2 * (e - c * kp);
      const int col = c0 + c;
      __half2 out = __floats2half2_rn(0.0f, 0.0f);
      if (t < b && (col < k0 || col >= k0 + b)) {
        int v0 = buf[(size_t)t * kSwapStride + c], v1 = buf[(size_t)(t + 1) * kSwapStride + c];
        v0 = v0 > h ? v0 - q : v0;
        v1 = v1 > h ? v1 - q : v1;
        out = __floats2half2_rn((float)v0, (float)v1);
      }
      *reinterpret_cast<__half2*>(Rp + (size_t)col * kb + t) = out;
    }
    __syncthreads();
  }
  allow_dependents();
}

constexpr int kUpdTile = 128;                 // rows and columns of one update tile
constexpr int kUpdThreads = 256;              // 8 warps, each 32 rows x 64 columns of the tile
constexpr int kUpdOutStride = kUpdTile + 16;  // bytes per staged result row (36 words: the 2-byte stores of
                                              // a warp's eight rows fall in distinct banks)

// Operand rows of kb fp16 plus 16 bytes: kb / 2 + 4 words, so that the eight rows of a fragment load (four
// words each) fall in distinct banks.
size_t update_smem(int kb) { return (size_t)2 * kUpdTile * (kb * 2 + 16) + (size_t)kUpdTile * kUpdOutStride; }

// d += a b for one m16n8k16 tile: fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (a + b) mod q for four byte lanes, a and b in [0, q).
__device__ __forceinline__ uint32_t add_mod4(uint32_t a, uint32_t b, uint32_t q4) {
  const uint32_t c = __vsub4(q4, b);      // q - b, in [1, q]
  const uint32_t ge = __vcmpgeu4(a, c);   // a + b >= q
  return (ge & __vsub4(a, c)) | (~ge & __vadd4(a, b));
}

// One 128 x 128 tile of one prime's matrix (grid.z = prime, column tile jt0 +
// blockIdx.x): X[i][j] <- base + sum_t W[i][t] RT[j][t] mod q for the columns
// j in [cb, ce) outside [x0, x1) (which covers J), base = 0 in the pivot rows
// and X[i][j] elsewhere (the swap pass has already permuted the rows the
// swaps moved).  The product runs on the warp-level fp16 tensor
// MMA with fp32 accumulation, exact here: the balanced residues (|r| <= 125)
// are fp16 integers and |sum| <= 64 125^2 < 2^24.  One reduction into
// [0, q), then one modular addition folds in the base.
__global__ void __launch_bounds__(kUpdThreads, 2) gj_update_kernel(uint8_t* __restrict__ M, int nE, int k0, int b,
                                                                   int kb, const __half* __restrict__ Wb,
                                                                   const __half* __restrict__ RT,
                                                                   const int* __restrict__ sing, int cb, int ce,
                                                                   int x0, int x1, int jt0) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int p = blockIdx.z;
  const int i0 = blockIdx.y * kUpdTile, j0 = (jt0 + blockIdx.x) * kUpdTile;
  const int lw = kb / 2 + 4;  // operand row stride in 32-bit words
  uint32_t* Ws = reinterpret_cast<uint32_t*>(sm);
  uint32_t* Rs = Ws + kUpdTile * lw;
  uint8_t* Cs = reinterpret_cast<uint8_t*>(Rs + kUpdTile * lw);
  wait_for_predecessor();
  const int wlo = max(j0, cb), whi = min(j0 + kUpdTile, ce);  // the tile's columns in range
  if (sing[p] || wlo >= whi || (wlo >= x0 && whi <= x1)) return;
  const __half* Wp = Wb + (size_t)p * nE * kb;
  const __half* Rp = RT + (size_t)p * nE * kb;
  const int vr = kb / 8;  // 16-byte vectors per operand row
  for (int e = threadIdx.x; e < kUpdTile * vr; e += kUpdThreads) {
    const int r = e / vr, v = e - r * vr;
    uint4 a = make_uint4(0u, 0u, 0u, 0u), c = a;
    if (i0 + r < nE) a = *reinterpret_cast<const uint4*>(Wp + (size_t)(i0 + r) * kb + v * 8);
    if (j0 + r < nE) c = *reinterpret_cast<const uint4*>(Rp + (size_t)(j0 + r) * kb + v * 8);
    *reinterpret_cast<uint4*>(Ws + r * lw + v * 4) = a;
    *reinterpret_cast<uint4*>(Rs + r * lw + v * 4) = c;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c4 = lane & 3;
  const int wr = (warp & 3) * 32, wc = (warp >> 2) * 64;
  float acc[2][8][4] = {};
  for (int ks = 0; ks < kb / 2; ks += 8) {  // 16 fp16 of K = 8 words
    uint32_t a[2][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      const uint32_t* ap = Ws + (wr + mi * 16 + g) * lw + ks + c4;
      a[mi][0] = ap[0];
      a[mi][1] = ap[8 * lw];
      a[mi][2] = ap[4];
      a[mi][3] = ap[8 * lw + 4];
    }
#pragma unroll
    for (int ni = 0; ni < 8; ++ni) {
      const uint32_t* bp = Rs + (wc + ni * 8 + g) * lw + ks + c4;
      const uint32_t b0 = bp[0], b1 = bp[4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) mma_f16(acc[mi][ni], a[mi], b0, b1);
    }
  }
  const int q = c_all.q[p];
  const float qf = c_all.qf[p], iq = c_all.invq[p];
  auto red = [&](float x) {
    const float v = bal_mod_small(x, qf, iq);
    return (uint32_t)(int)(v < 0.0f ? v + qf : v);
  };
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 8; ++ni) {
      const int row = wr + mi * 16 + g, col = wc + ni * 8 + c4 * 2;
      *reinterpret_cast<uint16_t*>(Cs + row * kUpdOutStride + col) =
          (uint16_t)(red(acc[mi][ni][0]) | red(acc[mi][ni][1]) << 8);
      *reinterpret_cast<uint16_t*>(Cs + (row + 8) * kUpdOutStride + col) =
          (uint16_t)(red(acc[mi][ni][2]) | red(acc[mi][ni][3]) << 8);
    }
  __syncthreads();
  uint8_t* Mp = M + (size_t)p * nE * nE;
  const uint32_t q4 = (uint32_t)q * 0x01010101u;
  for (int e = threadIdx.x; e < kUpdTile * (kUpdTile / 16); e += kUpdThreads) {
    const int r = e >> 3, v = e & 7;
    const int i = i0 + r, j = j0 + v * 16;
    if (i >= nE || j >= nE || j < cb || j >= ce || (j >= x0 && j < x1)) continue;
    uint4 o = *reinterpret_cast<const uint4*>(Cs + r * kUpdOutStride + v * 16);
    uint8_t* dst = Mp + (size_t)i * nE + j;
    if (i < k0 || i >= k0 + b) {
      const uint4 x = *reinterpret_cast<const uint4*>(dst);
      o = make_uint4(add_mod4(o.x, x.x, q4), add_mod4(o.y, x.y, q4), add_mod4(o.z, x.z, q4), add_mod4(o.w, x.w, q4));
    }
    *reinterpret_cast<uint4*>(dst) = o;
  }
  allow_dependents();
}

// The lift's primes, in order: map[s] = index of the s-th prime kept.
struct PrimeMap {
  int idx[kNumPrimes];
};

// Undoes the row swaps, which act on the in-place result as column swaps,
// and writes the balanced int8 inverse planes of the lift's primes: column c
// of M[map[s]] is column rowsrc[c] of the inverse, Binv[s][i][rowsrc[c]] =
// bal(M[map[s]][i][c]) for i < n, in rows of nE bytes (zero past n).  The
// padded block keeps its identity rows in place, so rowsrc maps the first n
// columns among themselves.  Each block stages whole rows in shared memory.
__global__ void __launch_bounds__(256) gj_finish_kernel(const uint8_t* __restrict__ M, const int* __restrict__ rowsrc,
                                                        int n, int nE, PrimeMap map, int8_t* __restrict__ Binv) {
  __shared__ __align__(16) int8_t out[kMaxSolveN];
  const int s = blockIdx.y, p = map.idx[s];
  const int q = c_all.q[p], h = (q - 1) / 2;
  const int* rs = rowsrc + (size_t)p * nE;
  for (int j = n + threadIdx.x; j < nE; j += blockDim.x) out[j] = 0;
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const uint8_t* row = M + ((size_t)p * nE + i) * nE;
    for (int c = threadIdx.x; c < n; c += blockDim.x) {
      const int v = row[c];
      out[rs[c]] = (int8_t)(v > h ? v - q : v);
    }
    __syncthreads();
    int8_t* dst = Binv + ((size_t)s * n + i) * nE;
    for (int v = threadIdx.x; v < nE / 16; v += blockDim.x)
      reinterpret_cast<uint4*>(dst)[v] = reinterpret_cast<const uint4*>(out)[v];
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// The lift ("exact-solve", Method: Dixon's lift on the residue engine).
// ---------------------------------------------------------------------------

// Rr[s][t][k] = bal(R[k][t] mod q_s) (int8), rows of length ld (zero
// padded); one thread per (entry, prime), the prime index s = blockIdx.y
// uniform across the block.
__global__ void __launch_bounds__(256) lift_residue_kernel(const int64_t* __restrict__ R, int n, int c, int ld,
                                                           int8_t* __restrict__ Rr) {
  wait_for_predecessor();
  const int s = blockIdx.y;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < (long long)c * ld;
       e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / ld), k = (int)(e - (long long)t * ld);
    const long long x = k < n ? R[(long long)k * c + t] : 0;
    const unsigned long long u = (unsigned long long)x;
    int acc = x < 0 ? -c_sol.wword[s][2] : 0;
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"((uint32_t)u), "r"(c_sol.wbyte[s][0]));
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"((uint32_t)(u >> 32)), "r"(c_sol.wbyte[s][1]));
    Rr[((long long)s * c + t) * ld + k] = (int8_t)bal_mod_small(int_to_float_exact(acc), c_sol.qf[s], c_sol.invq[s]);
  }
  allow_dependents();
}

// RC[s][i][t] = (Binv[s][i][:] . Rr[s][t][:]) mod q_s in [0, q): one warp per
// (prime, row), 16 int8 per lane and step, dp4a; |sum| <= n 125^2 < 2^31.
__global__ void __launch_bounds__(256) lift_gemv_kernel(const int8_t* __restrict__ Binv, const int8_t* __restrict__ Rr,
                                                        int n, int c, int ld, int E, uint8_t* __restrict__ RC) {
  wait_for_predecessor();
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (long long)E * n) return;
  const int s = (int)(warp / n), i = (int)(warp - (long long)s * n);
  const int8_t* brow = Binv + ((long long)s * n + i) * ld;
  const int q = c_sol.q[s];
  for (int t = 0; t < c; ++t) {
    const int8_t* rv = Rr + ((long long)s * c + t) * ld;
    int acc = 0;
    for (int k = lane * 16; k < ld; k += 32 * 16) {
      const int4 a = *reinterpret_cast<const int4*>(brow + k);
      const int4 b = *reinterpret_cast<const int4*>(rv + k);
      acc = __dp4a(a.x, b.x, acc);
      acc = __dp4a(a.y, b.y, acc);
      acc = __dp4a(a.z, b.z, acc);
      acc = __dp4a(a.w, b.w, acc);
    }
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      int r = acc % q;
      RC[((long long)s * n + i) * c + t] = (uint8_t)(r < 0 ? r + q : r);
    }
  }
  allow_dependents();
}

// The base-P digit X_i of every component (balanced Garner over the lift's
// primes), kept for the reconstruction, and its low 64 bits for the update.
__global__ void __launch_bounds__(128) lift_digit_kernel(const uint8_t* __restrict__ RC, int n, int c, int E,
                                                         uint32_t* __restrict__ digit,
                                                         unsigned long long* __restrict__ xlow) {
  wait_for_predecessor();
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e < (long long)n * c) {
    uint32_t x[1][kW];
    garner_reconstruct<kW, 1, SolTab>(RC + e, (long long)n * c, E, x);
#pragma unroll
    for (int w = 0; w < kW; ++w) digit[e * kW + w] = x[0][w];
    xlow[e] = ((unsigned long long)x[0][1] << 32) | x[0][0];
  }
  allow_dependents();
}

// R[i][t] = (R[i][t] - sum_k A[i][k] Xlow[k][t]) * P^-1 mod 2^64: the exact
// quotient (R - A X) / P, which fits one signed limb.  One warp per row.
__global__ void __launch_bounds__(256) lift_update_kernel(const int64_t* __restrict__ A, int n, int c,
                                                          const unsigned long long* __restrict__ xlow,
                                                          unsigned long long pinv64, int64_t* __restrict__ R) {
  wait_for_predecessor();
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp < n) {
    const int64_t* arow = A + warp * n;
    for (int t = 0; t < c; ++t) {
      unsigned long long acc = 0;
      for (int k = lane; k < n; k += 32) acc += (unsigned long long)arow[k] * xlow[(long long)k * c + t];
      for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) {
        const unsigned long long r = (unsigned long long)R[warp * c + t];
        R[warp * c + t] = (int64_t)((r - acc) * pinv64);
      }
    }
  }
  allow_dependents();
}

// The lift's step in two kernels when B has few columns (c <= kFusedLiftCols):
// one block per row i of the inverse planes forms the E GEMV results of
// its c components in shared memory and reconstructs their digits there; one
// warp per row then updates the residual and writes its residues for the
// next step's GEMV.
constexpr int kFusedLiftCols = 16;
static_assert(kW == kQWords, "a digit has as many words as the mixed-radix weights");

// Digits (balanced Garner) and low 64 bits of components i * c + t, t < c.
// First RC[t][s] = (Binv[s][i][:] . Rr[s][t][:]) mod q_s, for every (s, t)
// by a group of 4 or 16 threads (16 int8 per thread and step, dp4a; |sum|
// <= n 125^2 < 2^31), all groups' loads independent.  Then one warp per column:
// lane l owns primes l and l + 32; for each prime i in order its owner forms
// v_i = bal(acc_i mod q_i) and every later prime p adds gd[p][i] v_i to its
// acc_p (acc_p = ginv[p] r_p + sum_{j<p} gd[p][j] v_j, |acc| < 2^20); lane w
// then sums column w of x = sum_i v_i Q_i (|.| < 2^45) and lane 0 carries the
// columns into kW two's complement words.
template <int G>  // threads per dot product
__global__ void __launch_bounds__(256) lift_row_kernel(const int8_t* __restrict__ Binv, const int8_t* __restrict__ Rr,
                                                       int n, int c, int ld, int E, uint32_t* __restrict__ digit,
                                                       unsigned long long* __restrict__ xlow) {
  __shared__ uint8_t rc[kFusedLiftCols][kNumPrimes];
  __shared__ int gd[kNumPrimes][kGarnerWords];
  __shared__ uint32_t Qw[kNumPrimes][kQWords];
  __shared__ int vs[8][kNumPrimes];
  __shared__ long long cols[8][kW];
  for (int x = threadIdx.x; x < kNumPrimes * kGarnerWords; x += blockDim.x) (&gd[0][0])[x] = (&g_sol.gd_packed[0][0])[x];
  for (int x = threadIdx.x; x < kNumPrimes * kQWords; x += blockDim.x) (&Qw[0][0])[x] = (&g_sol.Qw[0][0])[x];
  wait_for_predecessor();
  const int i = blockIdx.x, vpr = ld / 16;
  const int grp = threadIdx.x / G, gl = threadIdx.x % G;
  // every thread runs the same number of rounds, so that the whole warp
  // reaches each shuffle (a group past the last task adds zeros)
  for (int base = 0; base < E * c; base += blockDim.x / G) {
    const int task = base + grp;
    const bool active = task < E * c;
    const int s = active ? task / c : 0, t = active ? task - s * c : 0;
    const int8_t* brow = Binv + ((long long)s * n + i) * ld;
    const int8_t* rv = Rr + ((long long)s * c + t) * ld;
    int acc = 0;
#pragma unroll 4
    for (int v = gl; active && v < vpr; v += G) {
      const int4 a = *reinterpret_cast<const int4*>(brow + 16 * v);
      const int4 b = *reinterpret_cast<const int4*>(rv + 16 * v);
      acc = __dp4a(a.x, b.x, acc);
      acc = __dp4a(a.y, b.y, acc);
      acc = __dp4a(a.z, b.z, acc);
      acc = __dp4a(a.w, b.w, acc);
    }
    for (int o = G / 2; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);  // within the group
    if (active && gl == 0) {
      const int q = c_sol.q[s];
      const int r = acc % q;
      rc[t][s] = (uint8_t)(r < 0 ? r + q : r);
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = warp; t < c; t += blockDim.x / 32) {
    const int p0 = lane, p1 = lane + 32;
    int acc0 = p0 < E ? g_sol.ginv[p0] * (int)rc[t][p0] : 0;
    int acc1 = p1 < E ? g_sol.ginv[p1] * (int)rc[t][p1] : 0;
    for (int pi = 0; pi < E; ++pi) {
      const int own = pi & 31;
      int v = 0;
      if (lane == own) {
        const int a = pi < 32 ? acc0 : acc1;
        v = (int)bal_mod_small((float)a, c_sol.qf[pi], c_sol.invq[pi]);
        vs[warp][pi] = v;
      }
      v = __shfl_sync(0xffffffffu, v, own);
      const int sh = 8 * (pi & 3);
      if (p0 > pi && p0 < E) acc0 += (int)(int8_t)(gd[p0][pi >> 2] >> sh) * v;
      if (p1 > pi && p1 < E) acc1 += (int)(int8_t)(gd[p1][pi >> 2] >> sh) * v;
    }
    __syncwarp();
    if (lane < kW) {
      long long col = 0;
      for (int pi = 0; pi < E; ++pi) col += (long long)vs[warp][pi] * Qw[pi][lane];
      cols[warp][lane] = col;
    }
    __syncwarp();
    if (lane == 0) {
      const long long e = (long long)i * c + t;
      long long carry = 0;
      uint32_t w[kW];
#pragma unroll
      for (int k = 0; k < kW; ++k) {
        const long long v = cols[warp][k] + carry;
        w[k] = (uint32_t)v;
        carry = v >> 32;  // arithmetic: the columns are signed
      }
#pragma unroll
      for (int k = 0; k < kW; ++k) digit[e * kW + k] = w[k];
      xlow[e] = ((unsigned long long)w[1] << 32) | w[0];
    }
    __syncwarp();
  }
  allow_dependents();
}

// R[i][t] = (R[i][t] - sum_k A[i][k] Xlow[k][t]) * P^-1 mod 2^64 (the exact
// quotient (R - A X) / P, which fits one signed limb), then its balanced
// residues Rr[s][t][i] for every lift prime.  One warp per row.
__global__ void __launch_bounds__(256) lift_update_residue_kernel(const int64_t* __restrict__ A, int n, int c,
                                                                  int ld, int E,
                                                                  const unsigned long long* __restrict__ xlow,
                                                                  unsigned long long pinv64, int64_t* __restrict__ R,
                                                                  int8_t* __restrict__ Rr) {
  wait_for_predecessor();
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp < n) {
    const int64_t* arow = A + warp * n;
    for (int t = 0; t < c; ++t) {
      unsigned long long acc = 0;
      for (int k = lane; k < n; k += 32) acc += (unsigned long long)arow[k] * xlow[(long long)k * c + t];
      for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      const unsigned long long r = (unsigned long long)R[warp * c + t];
      const long long x = (long long)((r - acc) * pinv64);  // the same in every lane
      if (lane == 0) R[warp * c + t] = x;
      const unsigned long long u = (unsigned long long)x;
      for (int s = lane; s < E; s += 32) {  // one prime per lane: the tables from global memory
        int v = x < 0 ? -g_sol.wword[s][2] : 0;
        asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(v) : "r"((uint32_t)u), "r"(g_sol.wbyte[s][0]));
        asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(v) : "r"((uint32_t)(u >> 32)), "r"(g_sol.wbyte[s][1]));
        Rr[((long long)s * c + t) * ld + warp] = (int8_t)bal_mod_small(int_to_float_exact(v), g_sol.qf[s], g_sol.invq[s]);
      }
    }
  }
  allow_dependents();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// The little-endian 32-bit words of a (no leading zero word; at least
// min_words, zero-padded).
std::vector<uint32_t> words_of(const big::Nat& a, size_t min_words = 0) {
  std::vector<uint32_t> w(a.v.size() * 2);
  for (size_t i = 0; i < a.v.size(); ++i) {
    w[2 * i] = (uint32_t)a.v[i];
    w[2 * i + 1] = (uint32_t)(a.v[i] >> 32);
  }
  while (!w.empty() && w.back() == 0) w.pop_back();
  if (w.size() < min_words) w.resize(min_words, 0);
  return w;
}

struct DevBuf {  // stream-ordered device allocation
  void* p = nullptr;
  cudaStream_t s = nullptr;
  cudaError_t alloc(size_t bytes, cudaStream_t st) {
    s = st;
    return cudaMallocAsync(&p, bytes ? bytes : 16, st);
  }
  ~DevBuf() {
    if (p) cudaFreeAsync(p, s);
  }
};

// A high- and a low-priority stream and an event for each, joined to the
// caller's stream: open() makes both wait for the caller's stream, join() (and
// the destructor, on an early return) makes the caller's stream wait for both.
struct SideStreams {
  cudaStream_t hi = nullptr, lo = nullptr, caller = nullptr;
  cudaEvent_t ev_hi = nullptr, ev_lo = nullptr;
  bool joined = true;
  cudaError_t open(cudaStream_t st) {
    caller = st;
    int least = 0, greatest = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&hi, cudaStreamNonBlocking, greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&lo, cudaStreamNonBlocking, least);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_hi, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_lo, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ev_hi, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hi, ev_hi, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(lo, ev_hi, 0);
    joined = e != cudaSuccess;
    return e;
  }
  cudaError_t join() {
    joined = true;
    cudaError_t e = cudaEventRecord(ev_hi, hi);
    if (e == cudaSuccess) e = cudaEventRecord(ev_lo, lo);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(caller, ev_hi, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(caller, ev_lo, 0);
    return e;
  }
  ~SideStreams() {
    if (!joined && hi && lo) join();
    if (ev_hi) cudaEventDestroy(ev_hi);
    if (ev_lo) cudaEventDestroy(ev_lo);
    if (hi) cudaStreamDestroy(hi);
    if (lo) cudaStreamDestroy(lo);
  }
};

#define SOLVE_TRY(x)                             \
  do {                                           \
    cudaError_t e_ = (x);                        \
    if (e_ != cudaSuccess) return RG_ERR_CUDA;   \
  } while (0)

unsigned long long inverse_mod_2_64(unsigned long long a) {  // a odd; Newton iteration
  unsigned long long x = a;  // correct to 3 bits
  for (int i = 0; i < 6; ++i) x *= 2 - a * x;
  return x;
}

int sm_count_host() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

unsigned grid_for(long long items, int per_block = 256) {
  long long b = (items + per_block - 1) / per_block;
  const long long cap = 8LL * sm_count_host();
  return (unsigned)std::max(1LL, std::min(b, cap));
}

// The panel and update kernels' dynamic shared memory above the default
// 48 KB, set once per device.
cudaError_t allow_panel_smem() {
  static std::mutex mu;
  static bool done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  const int bytes = (int)kPanelSmemLimit;
  const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  e = cudaFuncSetAttribute(gj_panel_kernel<64, 16, 1>, attr, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gj_panel_kernel<64, 8, 2>, attr, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gj_panel_kernel<32, 8, 4>, attr, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gj_panel_kernel<16, 4, 8>, attr, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gj_update_kernel, attr, (int)update_smem(64));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gj_swap_kernel, attr, (int)swap_smem(kMaxSolveN));
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

}  // namespace
}  // namespace rg

using namespace rg;

extern "C" void rg_solution_free(rg_solution* s) {
  if (!s) return;
  delete[] s->values;
  s->values = nullptr;
}

extern "C" int rg_solve_i64(const int64_t* A_in, const int64_t* B_in, int64_t n64, int64_t c64, unsigned flags,
                            void* stream, rg_solution* out) {
  if (!A_in || !B_in || !out) return RG_ERR_ARG;
  std::memset(out, 0, sizeof(*out));
  if (n64 < 1 || c64 < 1 || c64 > (1 << 20)) return RG_ERR_ARG;
  if (n64 > kMaxSolveN) return RG_ERR_RANGE;
  const int n = (int)n64, c = (int)c64;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  using clock = std::chrono::steady_clock;
  const auto t0 = clock::now();
  auto ms_since = [](clock::time_point a) {
    return std::chrono::duration<double, std::milli>(clock::now() - a).count();
  };
  SOLVE_TRY(upload_tables());
  {
    static std::mutex mu;
    static bool uploaded[64];
    int dev = 0;
    SOLVE_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return RG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!uploaded[dev]) {
      SOLVE_TRY(cudaMemcpyToSymbol(c_all, &host_tables(), sizeof(Tables)));
      uploaded[dev] = true;
    }
  }
  const size_t nn = (size_t)n * n;
  DevBuf dA, dB;
  const int64_t* A = A_in;
  const int64_t* B = B_in;
  if (flags & RG_FLAG_HOST) {
    SOLVE_TRY(dA.alloc(nn * 8, st));
    SOLVE_TRY(dB.alloc((size_t)n * c * 8, st));
    SOLVE_TRY(cudaMemcpyAsync(dA.p, A_in, nn * 8, cudaMemcpyHostToDevice, st));
    SOLVE_TRY(cudaMemcpyAsync(dB.p, B_in, (size_t)n * c * 8, cudaMemcpyHostToDevice, st));
    A = static_cast<const int64_t*>(dA.p);
    B = static_cast<const int64_t*>(dB.p);
  }

  // 1. norms and the range check (one host synchronisation)
  DevBuf dn;
  SOLVE_TRY(dn.alloc(((size_t)2 * n + c) * 8 + 8, st));
  double* rows = static_cast<double*>(dn.p);
  double* cols = rows + n;
  double* bcols = cols + n;
  unsigned long long* maxabs = reinterpret_cast<unsigned long long*>(bcols + c);
  SOLVE_TRY(cudaMemsetAsync(maxabs, 0, 8, st));
  const int rows_per = std::max(32, (n + 63) / 64), chunks = (n + rows_per - 1) / rows_per;
  DevBuf dpart;
  SOLVE_TRY(dpart.alloc((size_t)chunks * n * 8, st));
  norms_kernel<<<(unsigned)((std::max((long long)n * 32, (long long)c) + 255) / 256), 256, 0, st>>>(A, B, n, c, rows,
                                                                                                     bcols, maxabs);
  SOLVE_TRY(cudaGetLastError());
  col_norms_part_kernel<<<dim3((unsigned)((n + 255) / 256), (unsigned)chunks), 256, 0, st>>>(
      A, n, rows_per, static_cast<double*>(dpart.p));
  SOLVE_TRY(cudaGetLastError());
  col_norms_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(static_cast<const double*>(dpart.p), n, chunks,
                                                                     cols);
  SOLVE_TRY(cudaGetLastError());
  std::vector<double> hn((size_t)2 * n + c + 1);
  SOLVE_TRY(cudaMemcpyAsync(hn.data(), dn.p, hn.size() * 8, cudaMemcpyDeviceToHost, st));
  SOLVE_TRY(cudaStreamSynchronize(st));
  unsigned long long amax;
  std::memcpy(&amax, &hn[2 * n + c], 8);
  if (amax == 0) return RG_ERR_SINGULAR;
  if ((unsigned __int128)amax * (unsigned __int128)n >= ((unsigned __int128)1 << 63)) return RG_ERR_RANGE;
  // Hadamard bounds (in bits, rounded up with a margin for the fp64 sums):
  // |det A| <= prod of row (or column) norms; by Cramer's rule each numerator
  // is the determinant of A with one column replaced by a column of B.
  double row_bits = 0.0, col_bits = 0.0, min_col = 1e300, bmax = 0.0;
  bool zero_line = false;
  for (int i = 0; i < n; ++i) {
    if (hn[i] <= 0.0 || hn[n + i] <= 0.0) zero_line = true;
    row_bits += 0.5 * std::log2(std::max(hn[i], 1.0));
    col_bits += 0.5 * std::log2(std::max(hn[n + i], 1.0));
    min_col = std::min(min_col, 0.5 * std::log2(std::max(hn[n + i], 1.0)));
  }
  if (zero_line) return RG_ERR_SINGULAR;
  for (int t = 0; t < c; ++t) bmax = std::max(bmax, 0.5 * std::log2(std::max(hn[2 * n + t], 1.0)));
  const double margin = 4.0 + 1e-9 * n;
  const double dbits = std::min(row_bits, col_bits) + margin;
  double nbits_rows = 0.0;  // replacing column t: row norms grow to sqrt(|a_i|^2 + b_i^2) <= |a_i| + |b|
  for (int i = 0; i < n; ++i) nbits_rows += 0.5 * std::log2(std::max(hn[i], 1.0) + std::exp2(2.0 * bmax));
  const double nbits = std::min(nbits_rows, col_bits - min_col + bmax) + margin;

  // 2. batched inverse, on diag(A, I) of order nE = n rounded up to 16
  const int nE = (n + 15) / 16 * 16, ld = nE;
  const size_t nnE = (size_t)nE * nE;
  const PanelCfg pc = panel_cfg(nE);
  const int bw = pc.B, kbw = (bw + 31) / 32 * 32;
  DevBuf dM, dW, dRT, drowsrc, dsing, dgsrc;
  const size_t wplane = (size_t)kNumPrimes * nE * kbw;  // fp16 entries of one block's W for every prime
  SOLVE_TRY(dM.alloc((size_t)kNumPrimes * nnE, st));
  SOLVE_TRY(dW.alloc(2 * wplane * 2, st));  // two blocks' W: one factored while the other is applied
  SOLVE_TRY(dRT.alloc(wplane * 2, st));
  SOLVE_TRY(drowsrc.alloc((size_t)kNumPrimes * nE * 4, st));
  SOLVE_TRY(dsing.alloc(kNumPrimes * 4, st));
  SOLVE_TRY(dgsrc.alloc((size_t)kNumPrimes * nE * 2, st));
  uint8_t* M = static_cast<uint8_t*>(dM.p);
  __half* Wbuf = static_cast<__half*>(dW.p);
  __half* RT = static_cast<__half*>(dRT.p);
  int* rowsrc = static_cast<int*>(drowsrc.p);
  int* sing = static_cast<int*>(dsing.p);
  uint16_t* gsrc = static_cast<uint16_t*>(dgsrc.p);
  SOLVE_TRY(cudaMemsetAsync(sing, 0, kNumPrimes * 4, st));
  gj_init_kernel<<<grid_for((long long)nnE), 256, 0, st>>>(A, n, nE, M, rowsrc);
  SOLVE_TRY(cudaGetLastError());
  SOLVE_TRY(allow_panel_smem());
  // Look-ahead: the chain panel -> swap -> update of the next panel's columns
  // runs on a high-priority stream, and the update of the other columns on a
  // low-priority one, so that each block's bulk update overlaps the next
  // block's panel.  Both streams join the call's stream on every exit.
  SideStreams ss;
  SOLVE_TRY(ss.open(st));
  cudaStream_t sA = ss.hi, sB = ss.lo;
  auto W_of = [&](int blk) { return Wbuf + (size_t)(blk & 1) * wplane; };
  // a kernel that follows a cross-stream wait is launched plainly (programmatic
  // dependent launch relaxes only the dependency on the stream's previous kernel)
  auto go = [&](auto kern, bool dependent, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                auto... args) -> cudaError_t {
    if (dependent) return launch_dependent(kern, grid, block, smem, s, args...);
    kern<<<grid, block, smem, s>>>(args...);
    return cudaGetLastError();
  };
  auto panel = [&](bool dependent, int k0, int b, int kb, __half* W) -> cudaError_t {
    const size_t smem = panel_smem(nE, bw);
    const dim3 pg(kNumPrimes), pt(kPanelThreads);
    if (pc.RPT == 1) return go(gj_panel_kernel<64, 16, 1>, dependent, pg, pt, smem, sA, M, nE, k0, b, kb, W, gsrc, sing);
    if (pc.RPT == 2) return go(gj_panel_kernel<64, 8, 2>, dependent, pg, pt, smem, sA, M, nE, k0, b, kb, W, gsrc, sing);
    if (pc.RPT == 4) return go(gj_panel_kernel<32, 8, 4>, dependent, pg, pt, smem, sA, M, nE, k0, b, kb, W, gsrc, sing);
    return go(gj_panel_kernel<16, 4, 8>, dependent, pg, pt, smem, sA, M, nE, k0, b, kb, W, gsrc, sing);
  };
  auto swap = [&](int k0, int b, int kb) -> cudaError_t {  // follows a cross-stream wait: a plain launch
    gj_swap_kernel<<<dim3(kNumPrimes, (unsigned)((nE + kSwapCols - 1) / kSwapCols)), kPanelThreads, swap_smem(nE), sA>>>(
        M, nE, k0, b, kb, gsrc, RT, rowsrc, sing);
    return cudaGetLastError();
  };
  auto update = [&](cudaStream_t s, bool dependent, int k0, int b, int kb, const __half* W, int cb, int ce, int x0,
                    int x1) -> cudaError_t {
    const int jt0 = cb / kUpdTile, jt1 = (ce + kUpdTile - 1) / kUpdTile;
    const dim3 grid((unsigned)(jt1 - jt0), (unsigned)((nE + kUpdTile - 1) / kUpdTile), kNumPrimes);
    return go(gj_update_kernel, dependent, grid, dim3(kUpdThreads), update_smem(kb), s, M, nE, k0, b, kb, W,
              (const __half*)RT, (const int*)sing, cb, ce, x0, x1, jt0);
  };
  {
    const int b0 = std::min(bw, nE), kb0 = (b0 + 31) / 32 * 32;
    SOLVE_TRY(panel(false, 0, b0, kb0, W_of(0)));
    SOLVE_TRY(swap(0, b0, kb0));
  }
  for (int blk = 0, k0 = 0; k0 < nE; ++blk, k0 += bw) {
    const int b = std::min(bw, nE - k0), kb = (b + 31) / 32 * 32;  // b: a multiple of 16
    const int k1 = k0 + b;
    if (k1 >= nE) {  // the last block: the other columns at once
      if (b < nE) SOLVE_TRY(update(sA, true, k0, b, kb, W_of(blk), 0, nE, k0, k1));
      break;
    }
    const int b1 = std::min(bw, nE - k1), kb1 = (b1 + 31) / 32 * 32;
    SOLVE_TRY(update(sA, true, k0, b, kb, W_of(blk), k1, k1 + b1, k0, k1));  // the next panel's columns
    SOLVE_TRY(cudaEventRecord(ss.ev_hi, sA));
    SOLVE_TRY(panel(true, k1, b1, kb1, W_of(blk + 1)));
    SOLVE_TRY(cudaStreamWaitEvent(sB, ss.ev_hi, 0));
    SOLVE_TRY(update(sB, false, k0, b, kb, W_of(blk), 0, nE, k0, k1 + b1));  // the rest, beside the panel
    SOLVE_TRY(cudaEventRecord(ss.ev_lo, sB));
    SOLVE_TRY(cudaStreamWaitEvent(sA, ss.ev_lo, 0));
    SOLVE_TRY(swap(k1, b1, kb1));
  }
  SOLVE_TRY(ss.join());
  int hsing[kNumPrimes];
  SOLVE_TRY(cudaMemcpyAsync(hsing, sing, sizeof(hsing), cudaMemcpyDeviceToHost, st));
  SOLVE_TRY(cudaStreamSynchronize(st));
  const Tables& T = host_tables();
  std::vector<int> qs;
  PrimeMap map{};
  for (int p = 0; p < kNumPrimes; ++p)
    if (!hsing[p]) {
      map.idx[qs.size()] = p;
      qs.push_back(T.q[p]);
    }
  const int E = (int)qs.size();
  if (E == 0) return RG_ERR_SINGULAR;  // singular modulo every prime below 256
  Tables sol;
  build_tables_for(qs.data(), E, &sol);
  SOLVE_TRY(cudaMemcpyToSymbolAsync(c_sol, &sol, sizeof(Tables), 0, cudaMemcpyHostToDevice, st));
  SOLVE_TRY(cudaMemcpyToSymbolAsync(g_sol, &sol, sizeof(Tables), 0, cudaMemcpyHostToDevice, st));
  DevBuf dBinv;
  SOLVE_TRY(dBinv.alloc((size_t)E * n * ld, st));
  int8_t* Binv = static_cast<int8_t*>(dBinv.p);
  gj_finish_kernel<<<dim3((unsigned)std::min(n, 128), E), 256, 0, st>>>(M, rowsrc, n, nE, map, Binv);
  SOLVE_TRY(cudaGetLastError());

  // 3. the lift
  SOLVE_TRY(cudaStreamSynchronize(st));
  const double ms_inverse = ms_since(t0);
  const auto t1 = clock::now();
  double log2P = 0.0;
  big::Nat Pn = big::from_u64(1);
  for (int q : qs) {
    log2P += std::log2((double)q);
    Pn = big::mul(Pn, big::from_u64((uint64_t)q));
  }
  const int steps = std::max(1, (int)std::ceil((1.0 + nbits + dbits) / log2P));
  unsigned long long P64 = 1;
  for (int q : qs) P64 *= (unsigned long long)q;  // P mod 2^64
  const unsigned long long pinv64 = inverse_mod_2_64(P64);
  // P^m, the powers P^i (i < m) and Barrett's constant for P^m, as 32-bit
  // words, built on a host thread while the GPU lifts.
  std::vector<uint32_t> pow_words, PMw, MUw;
  std::vector<int> pow_idx(2 * (size_t)steps);  // offsets, then lengths
  big::Nat Pm;
  std::thread tables([&] {
    Pm = big::from_u64(1);
    for (int i = 0; i < steps; ++i) {
      const std::vector<uint32_t> w = words_of(Pm);
      pow_idx[i] = (int)pow_words.size();
      pow_idx[steps + i] = (int)w.size();
      pow_words.insert(pow_words.end(), w.begin(), w.end());
      Pm = big::mul(Pm, Pn);
    }
    PMw = words_of(Pm);
    big::Nat mu;
    big::divmod(big::pow2((size_t)64 * PMw.size()), Pm, &mu, nullptr);
    MUw = words_of(mu, PMw.size() + 1);
  });
  struct Joiner {  // the thread is joined on every return path
    std::thread& t;
    ~Joiner() {
      if (t.joinable()) t.join();
    }
  } joiner{tables};
  DevBuf dR, dRr, dRC, dX, dlow;
  SOLVE_TRY(dR.alloc((size_t)n * c * 8, st));
  SOLVE_TRY(dRr.alloc((size_t)E * c * ld, st));
  SOLVE_TRY(dRC.alloc((size_t)E * n * c, st));
  SOLVE_TRY(dX.alloc((size_t)steps * n * c * kW * 4, st));
  SOLVE_TRY(dlow.alloc((size_t)n * c * 8, st));
  int64_t* R = static_cast<int64_t*>(dR.p);
  SOLVE_TRY(cudaMemcpyAsync(R, B, (size_t)n * c * 8, cudaMemcpyDeviceToDevice, st));
  uint32_t* X = static_cast<uint32_t*>(dX.p);
  const bool fused = c <= kFusedLiftCols;
  if (fused)  // the residues of R = B; each step's update writes the next ones
    SOLVE_TRY(launch_dependent(lift_residue_kernel,
                               dim3(std::max(1u, std::min((unsigned)(((long long)c * ld + 255) / 256), 64u)), E),
                               dim3(256), 0, st, (const int64_t*)R, n, c, ld, static_cast<int8_t*>(dRr.p)));
  for (int i = 0; fused && i < steps; ++i) {
    // 4 threads per dot product up to rows of 1 KiB (every prime of one right-hand side at once), 16 for
    // longer rows (more loads in flight per row; measured at n = 1024 and 2048)
    SOLVE_TRY(launch_dependent(ld <= 1024 ? lift_row_kernel<4> : lift_row_kernel<16>, dim3((unsigned)n), dim3(256), 0,
                               st, (const int8_t*)Binv, (const int8_t*)dRr.p, n, c, ld, E, X + (size_t)i * n * c * kW,
                               static_cast<unsigned long long*>(dlow.p)));
    SOLVE_TRY(launch_dependent(lift_update_residue_kernel, dim3((unsigned)(((long long)n * 32 + 255) / 256)),
                               dim3(256), 0, st, A, n, c, ld, E, (const unsigned long long*)dlow.p, pinv64, R,
                               static_cast<int8_t*>(dRr.p)));
  }
  for (int i = 0; !fused && i < steps; ++i) {
    SOLVE_TRY(launch_dependent(lift_residue_kernel,
                               dim3(std::max(1u, std::min((unsigned)(((long long)c * ld + 255) / 256), 64u)), E),
                               dim3(256), 0, st, (const int64_t*)R, n, c, ld, static_cast<int8_t*>(dRr.p)));
    SOLVE_TRY(launch_dependent(lift_gemv_kernel, dim3((unsigned)(((long long)E * n * 32 + 255) / 256)), dim3(256), 0,
                               st, (const int8_t*)Binv, (const int8_t*)dRr.p, n, c, ld, E,
                               static_cast<uint8_t*>(dRC.p)));
    SOLVE_TRY(launch_dependent(lift_digit_kernel, dim3((unsigned)(((long long)n * c + 127) / 128)), dim3(128), 0, st,
                               (const uint8_t*)dRC.p, n, c, E, X + (size_t)i * n * c * kW,
                               static_cast<unsigned long long*>(dlow.p)));
    SOLVE_TRY(launch_dependent(lift_update_kernel, dim3((unsigned)(((long long)n * 32 + 255) / 256)), dim3(256), 0, st,
                               A, n, c, (const unsigned long long*)dlow.p, pinv64, R));
  }
  // 4. Reconstruction (exact-solve, Method).  The components' values and
  // numerators are formed on the GPU; the common denominator D comes from a
  // few components' rational reconstructions on host threads.  The tables
  // of P^m were built by a host thread while the lift ran.
  const long long comps = (long long)n * c;
  // the digits to the host, for the sampled components
  std::vector<uint32_t> hX((size_t)steps * n * c * kW);
  SOLVE_TRY(cudaMemcpyAsync(hX.data(), X, hX.size() * 4, cudaMemcpyDeviceToHost, st));
  SOLVE_TRY(cudaStreamSynchronize(st));
  const double ms_lift = ms_since(t1);
  const auto t2 = clock::now();
  tables.join();
  const int kP = (int)PMw.size();
  const std::vector<uint32_t> Pw = words_of(Pn, kW);
  const big::Nat nbound = big::pow2((size_t)std::ceil(nbits));
  const big::Nat dbound = big::pow2((size_t)std::ceil(dbits));
  const int bound_bits = (int)std::ceil(nbits);
  const int wDmax = (int)(words_of(dbound).size());
  const int blocks = recon_blocks(comps);
  DevBuf dtab, dtabi, dY, dN, dD, dinfo, dscr;
  const size_t ntab = pow_words.size() + Pw.size() + PMw.size() + MUw.size();
  SOLVE_TRY(dtab.alloc(ntab * 4, st));
  SOLVE_TRY(dtabi.alloc(pow_idx.size() * 4, st));
  uint32_t* tabp = static_cast<uint32_t*>(dtab.p);
  int* tabi = static_cast<int*>(dtabi.p);
  ReconTables tab;
  tab.pow = tabp;
  tab.P = tabp + pow_words.size();
  tab.PM = tab.P + Pw.size();
  tab.MU = tab.PM + PMw.size();
  tab.pow_off = tabi;
  tab.pow_len = tabi + steps;
  tab.pw = kW;
  tab.m = steps;
  tab.k = kP;
  SOLVE_TRY(cudaMemcpyAsync(tabp, pow_words.data(), pow_words.size() * 4, cudaMemcpyHostToDevice, st));
  SOLVE_TRY(cudaMemcpyAsync(const_cast<uint32_t*>(tab.P), Pw.data(), Pw.size() * 4, cudaMemcpyHostToDevice, st));
  SOLVE_TRY(cudaMemcpyAsync(const_cast<uint32_t*>(tab.PM), PMw.data(), PMw.size() * 4, cudaMemcpyHostToDevice, st));
  SOLVE_TRY(cudaMemcpyAsync(const_cast<uint32_t*>(tab.MU), MUw.data(), MUw.size() * 4, cudaMemcpyHostToDevice, st));
  SOLVE_TRY(cudaMemcpyAsync(tabi, pow_idx.data(), pow_idx.size() * 4, cudaMemcpyHostToDevice, st));
  SOLVE_TRY(dY.alloc((size_t)comps * kP * 4, st));
  SOLVE_TRY(dN.alloc((size_t)comps * (kP + 2) * 4, st));
  SOLVE_TRY(dD.alloc((size_t)wDmax * 4, st));
  SOLVE_TRY(dinfo.alloc((size_t)comps * 4, st));
  SOLVE_TRY(dscr.alloc(recon_scratch_bytes(tab, wDmax, blocks), st));
  uint32_t* Yv = static_cast<uint32_t*>(dY.p);
  uint32_t* Nw = static_cast<uint32_t*>(dN.p);
  int* info = static_cast<int*>(dinfo.p);
  uint32_t* scr = static_cast<uint32_t*>(dscr.p);
  SOLVE_TRY(recon_values(X, comps, tab, Yv, scr, st));

  // X_k = sum_i x_i P^i mod P^m on the host, for the sampled components and
  // any whose denominator D misses: the balanced digits normalised to [0, P)
  // by borrow propagation (a final borrow is a multiple of P^m), then
  // converted by halves with the powers P^(2^j) (big::radix_value).
  const size_t pl = Pn.v.size();  // limbs of P (<= 6)
  struct Scratch {
    std::vector<big::Limb> acc;
    std::vector<big::Limb> z;  // normalised digits, m x pl limbs
  };
  std::vector<big::Nat> pw(1, Pn);  // P^(2^j) for every 2^j below the step count
  while (((size_t)1 << pw.size()) < (size_t)steps) pw.push_back(big::mul(pw.back(), pw.back()));
  auto value_of = [&](long long k, Scratch& S) {
    S.z.assign((size_t)steps * pl, 0);
    int borrow = 0;
    for (int i = 0; i < steps; ++i) {
      big::Int x = big::from_words(&hX[((size_t)i * comps + k) * kW], kW);
      if (borrow) x = big::sub(x, big::Int{false, big::from_u64(1)});
      borrow = x.neg ? 1 : 0;
      const big::Nat zi = x.neg ? big::sub(Pn, x.mag) : x.mag;
      std::copy(zi.v.begin(), zi.v.end(), S.z.begin() + (size_t)i * pl);
    }
    big::radix_value(S.z.data(), (size_t)steps, pl, pw, S.acc);
    big::Nat Xk;
    Xk.v = S.acc;
    big::trim(Xk);
    return Xk;
  };
  // The denominators of a few components, one host thread each while the
  // GPU forms the values, give the common denominator D: their lcm divides
  // det A, and a factor cancelled in one component's fraction rarely cancels
  // in all of them.
  const int nthreads = std::max(1, std::min((int)std::thread::hardware_concurrency(), 64));
  const long long sample = std::min<long long>(comps, std::max(1, std::min(4, nthreads / 2)));
  std::vector<big::Nat> Ds(sample);
  std::vector<char> rec_ok(sample, 0);
  {
    std::vector<std::thread> th;
    for (long long k = 0; k < sample; ++k)
      th.emplace_back([&, k] {
        Scratch S;
        const big::Nat Xk = value_of(k, S);
        big::Int Nk;
        rec_ok[k] = big::rational_reconstruct(Xk, Pm, nbound, dbound, &Nk, &Ds[k]);
      });
    for (auto& t : th) t.join();
  }
  big::Nat D = big::from_u64(1);
  for (long long k = 0; k < sample; ++k) {
    if (!rec_ok[k]) return RG_ERR_RANGE;
    big::Nat t;
    big::divmod(Ds[k], big::gcd(D, Ds[k]), &t, nullptr);
    D = big::mul(D, t);
  }
  // N_k = D X_k mod P^m, balanced, for every k, on the GPU.  A component
  // whose N_k exceeds the numerator bound has a denominator not dividing D:
  // its own reconstruction extends D by the missing factor, and the
  // numerators are formed again (each stays <= |det A_k|, since D still
  // divides det A).
  std::vector<int> hinfo(comps);
  auto numerators = [&]() -> int {
    const std::vector<uint32_t> Dw = words_of(D);
    if ((int)Dw.size() > wDmax) return RG_ERR_RANGE;  // not reached: D <= dbound
    SOLVE_TRY(cudaMemcpyAsync(dD.p, Dw.data(), Dw.size() * 4, cudaMemcpyHostToDevice, st));
    SOLVE_TRY(recon_numerators(Yv, comps, tab, static_cast<const uint32_t*>(dD.p), (int)Dw.size(), bound_bits, Nw,
                               info, scr, st));
    SOLVE_TRY(cudaMemcpyAsync(hinfo.data(), info, (size_t)comps * 4, cudaMemcpyDeviceToHost, st));
    SOLVE_TRY(cudaStreamSynchronize(st));
    return RG_OK;
  };
  int rc = numerators();
  if (rc != RG_OK) return rc;
  for (long long k = 0; k < comps; ++k) {
    if (hinfo[k] >= 0) continue;
    Scratch S;
    const big::Nat Xk = value_of(k, S);
    big::Int Nk;
    big::Nat Dk;
    if (!big::rational_reconstruct(Xk, Pm, nbound, dbound, &Nk, &Dk)) return RG_ERR_RANGE;
    big::Nat t;
    big::divmod(Dk, big::gcd(D, Dk), &t, nullptr);
    D = big::mul(D, t);
    rc = numerators();
    if (rc != RG_OK) return rc;
    if (hinfo[k] < 0) return RG_ERR_RANGE;
  }
  // the numerators and the denominator as limbs: the low limbs of each
  // numerator's two's complement words
  size_t maxbits = big::bit_length(D);
  for (long long k = 0; k < comps; ++k) maxbits = std::max(maxbits, (size_t)hinfo[k]);
  const int limbs = (int)(maxbits / 64 + 1);  // <= (kP + 2) / 2: |N|, D < P^m < 2^(32 kP)
  out->n = n;
  out->c = c;
  out->limbs = limbs;
  out->steps = steps;
  out->primes = E;
  out->ms_inverse = ms_inverse;
  out->ms_lift = ms_lift;
  out->values = new int64_t[(size_t)(comps + 1) * limbs];
  if (cudaMemcpy2DAsync(out->values, (size_t)limbs * 8, Nw, (size_t)(kP + 2) * 4, (size_t)limbs * 8, (size_t)comps,
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    rg_solution_free(out);
    return RG_ERR_CUDA;
  }
  big::Int Di;
  Di.mag = D;
  if (!big::to_limbs(Di, out->values + (size_t)comps * limbs, limbs)) {
    rg_solution_free(out);
    return RG_ERR_RANGE;
  }
  out->ms_reconstruct = ms_since(t2);
  return RG_OK;
}

extern "C" int rg_rational_reconstruct(const int64_t* x, int xl, const int64_t* m, int ml, int nbits, int dbits,
                                       int64_t* num, int64_t* den, int limbs) {
  if (!x || !m || !num || !den || xl < 1 || ml < 1 || limbs < 1 || nbits < 0 || dbits < 0) return RG_ERR_ARG;
  big::Nat X, M;
  X.v.assign((const uint64_t*)x, (const uint64_t*)x + xl);
  M.v.assign((const uint64_t*)m, (const uint64_t*)m + ml);
  big::trim(X);
  big::trim(M);
  if (big::is_zero(M) || big::cmp(X, M) >= 0) return RG_ERR_ARG;
  big::Int N;
  big::Nat D;
  if (!big::rational_reconstruct(X, M, big::pow2(nbits), big::pow2(dbits), &N, &D)) return RG_ERR_RANGE;
  big::Int Di;
  Di.mag = D;
  if (!big::to_limbs(N, num, limbs) || !big::to_limbs(Di, den, limbs)) return RG_ERR_RANGE;
  return RG_OK;
}

extern "C" int rg_big_mulmod(const uint64_t* a, int al, const uint64_t* b, int bl, const uint64_t* m, int ml,
                             uint64_t* r, int rl) {
  if (!a || !b || !m || !r || al < 1 || bl < 1 || ml < 1 || rl < 1) return RG_ERR_ARG;
  big::Nat A, B, M;
  A.v.assign(a, a + al);
  B.v.assign(b, b + bl);
  M.v.assign(m, m + ml);
  big::trim(A);
  big::trim(B);
  big::trim(M);
  if (big::is_zero(M) || big::cmp(A, M) >= 0 || big::cmp(B, M) >= 0) return RG_ERR_ARG;
  const big::Barrett bar = big::make_barrett(M);
  std::vector<big::Limb> prod, s1, s2;
  big::kmul_into(A.v.data(), A.v.size(), B.v.data(), B.v.size(), prod);
  big::Nat R;
  if (!big::reduce_barrett(bar, prod.data(), prod.size(), s1, s2, &R)) return RG_ERR_RANGE;
  if ((int)R.v.size() > rl) return RG_ERR_RANGE;
  for (int i = 0; i < rl; ++i) r[i] = i < (int)R.v.size() ? R.v[i] : 0;
  return RG_OK;
}

extern "C" int rg_big_gcd(const uint64_t* a, int al, const uint64_t* b, int bl, uint64_t* g, int gl) {
  if (!a || !b || !g || al < 1 || bl < 1 || gl < 1) return RG_ERR_ARG;
  big::Nat A, B;
  A.v.assign(a, a + al);
  B.v.assign(b, b + bl);
  big::trim(A);
  big::trim(B);
  const big::Nat G = big::gcd(A, B);
  if ((int)G.v.size() > gl) return RG_ERR_RANGE;
  for (int i = 0; i < gl; ++i) g[i] = i < (int)G.v.size() ? G.v[i] : 0;
  return RG_OK;
}
