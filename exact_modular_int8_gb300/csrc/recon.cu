// recon.cu -- the exact solve's per-component big-integer work on the GPU
// ("exact-solve", Method: rational reconstruction of the lifted solution).
// Once the lift has produced the base-P digits of every component, two
// kernels, one block per component, form
//   the value  X = sum_i z_i P^i mod P^m (digits normalised into [0, P)), and
//   the numerator  N = D X mod P^m, balanced, by Barrett's reduction,
// with D the common denominator the host derives from a few components.
// Products are schoolbook by columns: each thread sums its columns' 32 x 32
// bit products in a 96-bit accumulator, then one thread carries them into
// words.  Little-endian 32-bit words throughout.
#include <cuda_runtime.h>

#include <algorithm>

#include "recon.h"
#include "rg_common.cuh"

namespace rg {
namespace {

constexpr int kReconThreads = 256;

// (s2:s1:s0) += a * b.
__device__ __forceinline__ void mad96(uint32_t& s0, uint32_t& s1, uint32_t& s2, uint32_t a, uint32_t b) {
  asm("mad.lo.cc.u32 %0, %3, %4, %0;\n\t"
      "madc.hi.cc.u32 %1, %3, %4, %1;\n\t"
      "addc.u32 %2, %2, 0;"
      : "+r"(s0), "+r"(s1), "+r"(s2)
      : "r"(a), "r"(b));
}

// Per-block scratch: three column-sum arrays and the intermediate products.
struct Scratch {
  uint32_t *c0, *c1, *c2;  // column sums, low to high word
  uint32_t* T;             // D X
  uint32_t* Q2;            // q1 MU
  uint32_t* R2;            // q3 PM mod 2^(32 (k + 1))
};

__host__ __device__ inline size_t scratch_words(int k, int wD) {
  const size_t cols = (size_t)wD + k + 4;  // the longest product: q1 MU has (wD + 1) + (k + 1) words
  return 3 * cols + ((size_t)wD + k) + cols + ((size_t)k + 1);
}

__device__ Scratch scratch_of(uint32_t* base, int k, int wD) {
  const size_t cols = (size_t)wD + k + 4;
  uint32_t* p = base + (size_t)blockIdx.x * scratch_words(k, wD);
  Scratch s;
  s.c0 = p;
  s.c1 = p + cols;
  s.c2 = p + 2 * cols;
  s.T = p + 3 * cols;
  s.Q2 = s.T + (size_t)wD + k;
  s.R2 = s.Q2 + cols;
  return s;
}

// Block-parallel word arithmetic.  Each thread owns one contiguous chunk of
// the word positions; a carry or borrow leaving a chunk is passed to the next
// chunk and rippled in, round after round, until none is left (a round moves
// it one chunk: rounds beyond the first are rare, since a carry crosses a
// chunk only through words that are all ones).  Every thread of the block
// calls these functions.
__device__ __forceinline__ void chunk_of(int n, int& a, int& b) {
  const int per = (n + kReconThreads - 1) / kReconThreads;
  a = min(n, (int)threadIdx.x * per);
  b = min(n, a + per);
}

// Ripples the chunks' outgoing carries (cout, +1 per unit) or borrows (-1)
// through out[0, n), modulo 2^(32 n).
__device__ void ripple(uint32_t* __restrict__ out, int n, uint32_t cout, bool borrow) {
  __shared__ uint32_t s_c[kReconThreads];
  int a, b;
  chunk_of(n, a, b);
  for (;;) {
    s_c[threadIdx.x] = cout;
    __syncthreads();
    uint32_t c = threadIdx.x > 0 ? s_c[threadIdx.x - 1] : 0u;
    __syncthreads();
    for (int j = a; j < b && c; ++j) {
      const uint32_t v = out[j];
      if (borrow) {
        out[j] = v - c;
        c = v < c ? 1u : 0u;
      } else {
        const unsigned long long t = (unsigned long long)v + c;
        out[j] = (uint32_t)t;
        c = (uint32_t)(t >> 32);
      }
    }
    cout = c;
    if (!__syncthreads_or(cout != 0u)) break;
  }
}

// out[0, n) = the words of sum_j (c0[j] + c1[j] 2^32 + c2[j] 2^64) 2^(32 j),
// modulo 2^(32 n).
__device__ void block_carry(const uint32_t* __restrict__ c0, const uint32_t* __restrict__ c1,
                            const uint32_t* __restrict__ c2, uint32_t* __restrict__ out, int n) {
  int a, b;
  chunk_of(n, a, b);
  unsigned long long carry = 0;
  for (int j = a; j < b; ++j) {
    const unsigned long long v =
        carry + c0[j] + (j >= 1 ? (unsigned long long)c1[j - 1] : 0ull) + (j >= 2 ? (unsigned long long)c2[j - 2] : 0ull);
    out[j] = (uint32_t)v;
    carry = v >> 32;  // < 4
  }
  ripple(out, n, (uint32_t)carry, false);
}

// a[0, n) -= b[0, nb) (nb <= n), modulo 2^(32 n).
__device__ void block_sub(uint32_t* __restrict__ a, int n, const uint32_t* __restrict__ b, int nb) {
  int lo, hi;
  chunk_of(n, lo, hi);
  uint32_t borrow = 0;
  for (int j = lo; j < hi; ++j) {
    const unsigned long long d = (unsigned long long)a[j] - (j < nb ? b[j] : 0u) - borrow;
    a[j] = (uint32_t)d;
    borrow = (uint32_t)((d >> 32) & 1ull);
  }
  __syncthreads();
  ripple(a, n, borrow, true);
}

// -1, 0, 1 as a[0, na) <, ==, > b[0, nb) (as naturals).
__device__ int block_cmp(const uint32_t* __restrict__ a, int na, const uint32_t* __restrict__ b, int nb) {
  __shared__ int s_top;
  const int n = max(na, nb);
  if (threadIdx.x == 0) s_top = -1;
  __syncthreads();
  int lo, hi;
  chunk_of(n, lo, hi);
  for (int j = hi - 1; j >= lo; --j)
    if ((j < na ? a[j] : 0u) != (j < nb ? b[j] : 0u)) {
      atomicMax(&s_top, j);
      break;
    }
  __syncthreads();
  const int t = s_top;
  __syncthreads();
  if (t < 0) return 0;
  return (t < na ? a[t] : 0u) < (t < nb ? b[t] : 0u) ? -1 : 1;
}

// The bit length of a[0, n), and whether a is a power of two.
__device__ int block_bits(const uint32_t* __restrict__ a, int n, bool& pow2) {
  __shared__ int s_bits, s_pop;
  if (threadIdx.x == 0) s_bits = s_pop = 0;
  __syncthreads();
  int lo, hi;
  chunk_of(n, lo, hi);
  int top = 0, pop = 0;
  for (int j = lo; j < hi; ++j)
    if (a[j]) {
      top = 32 * j + 32 - __clz(a[j]);
      pop += __popc(a[j]);
    }
  if (top) atomicMax(&s_bits, top);
  if (pop) atomicAdd(&s_pop, pop);
  __syncthreads();
  const int bits = s_bits;
  pow2 = s_pop == 1;
  __syncthreads();
  return bits;
}

// out[0, nout) = (a[0, na) * b[0, nb)) mod 2^(32 nout); a, b in shared or
// global memory, out anywhere but a, b or the scratch.
__device__ void block_mul(const uint32_t* a, int na, const uint32_t* b, int nb, uint32_t* out, int nout,
                          const Scratch& s) {
  for (int j = threadIdx.x; j < nout; j += blockDim.x) {
    uint32_t s0 = 0, s1 = 0, s2 = 0;
    const int lo = max(0, j - nb + 1), hi = min(j, na - 1);
    for (int l = lo; l <= hi; ++l) mad96(s0, s1, s2, a[l], b[j - l]);
    s.c0[j] = s0;
    s.c1[j] = s1;
    s.c2[j] = s2;
  }
  __syncthreads();
  block_carry(s.c0, s.c1, s.c2, out, nout);
  __syncthreads();
}

// X_e from its digits.  Shared memory: the m digits (pw words each) and
// their signs.
__global__ void __launch_bounds__(kReconThreads) recon_values_kernel(const uint32_t* __restrict__ digits,
                                                                     long long comps, ReconTables t,
                                                                     uint32_t* __restrict__ Y,
                                                                     uint32_t* __restrict__ scratch) {
  extern __shared__ __align__(16) uint32_t sm[];
  const int pw = t.pw, m = t.m, k = t.k;
  uint32_t* z = sm;                                       // m x pw
  int* cls = reinterpret_cast<int*>(z + (size_t)m * pw);  // -1, 0, +1: the digit's sign
  const Scratch s = scratch_of(scratch, k, 0);
  for (long long e = blockIdx.x; e < comps; e += gridDim.x) {
    for (int x = threadIdx.x; x < m * pw; x += blockDim.x) {
      const int i = x / pw, w = x - i * pw;
      z[x] = digits[((size_t)i * comps + e) * pw + w];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
      const uint32_t* d = z + (size_t)i * pw;
      uint32_t any = 0;
      for (int w = 0; w < pw; ++w) any |= d[w];
      cls[i] = (d[pw - 1] >> 31) ? -1 : (any ? 1 : 0);
    }
    __syncthreads();
    // z_i = x_i - b_{i-1}, plus P if that is negative; the borrow b_i is 1
    // when x_i < 0, 0 when x_i > 0, and b_{i-1} when x_i = 0 (|x_i| < P/2),
    // so it is the sign of the last nonzero digit at or below i.
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
      int b = 0;
      for (int j = i - 1; j >= 0; --j)
        if (cls[j] != 0) {
          b = cls[j] < 0;
          break;
        }
      uint32_t* d = z + (size_t)i * pw;
      uint32_t borrow = (uint32_t)b;
      for (int w = 0; w < pw; ++w) {
        const uint32_t v = d[w];
        d[w] = v - borrow;
        borrow = borrow && v == 0u;
      }
      if (d[pw - 1] >> 31) {  // negative: add P (the result lies in [0, P))
        unsigned long long c = 0;
        for (int w = 0; w < pw; ++w) {
          c += (unsigned long long)d[w] + t.P[w];
          d[w] = (uint32_t)c;
          c >>= 32;
        }
      }
    }
    __syncthreads();
    // column j of sum_i z_i P^i: the products z_i[l] P^i[j - l]
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      uint32_t s0 = 0, s1 = 0, s2 = 0;
      for (int i = 0; i < m; ++i) {
        const int len = t.pow_len[i];
        if (j - (pw - 1) >= len) continue;  // P^i too short to reach column j
        const uint32_t* p = t.pow + t.pow_off[i];
        const uint32_t* d = z + (size_t)i * pw;
        const int l0 = max(0, j - len + 1), l1 = min(pw - 1, j);
        for (int l = l0; l <= l1; ++l) mad96(s0, s1, s2, d[l], p[j - l]);
      }
      s.c0[j] = s0;
      s.c1[j] = s1;
      s.c2[j] = s2;
    }
    __syncthreads();
    block_carry(s.c0, s.c1, s.c2, Y + (size_t)e * k, k);
    __syncthreads();
  }
}

// N = D Y mod PM, balanced.  Shared memory: D (wD words), Y (k words) and q
// (wD + 1 words).  Barrett (B = 2^32, PM of k words, T = D Y < PM^2 <
// B^(2k)): q1 = floor(T / B^(k-1)), q3 = floor(q1 MU / B^(k+1)) is at most 2
// below floor(T / PM), so r = T - q3 PM lies in [0, 3 PM) and is found
// modulo B^(k+1), then brought below PM by at most two subtractions.
__global__ void __launch_bounds__(kReconThreads) recon_numerators_kernel(
    const uint32_t* __restrict__ Y, long long comps, ReconTables t, const uint32_t* __restrict__ D, int wD,
    int bound_bits, uint32_t* __restrict__ N, int* __restrict__ info, uint32_t* __restrict__ scratch) {
  extern __shared__ __align__(16) uint32_t sm[];
  const int k = t.k;
  const int nT = wD + k, nq = wD + 1, nN = k + 2;
  uint32_t* Ds = sm;
  uint32_t* Ys = Ds + wD;
  uint32_t* q = Ys + k;
  const Scratch s = scratch_of(scratch, k, wD);
  for (int w = threadIdx.x; w < wD; w += blockDim.x) Ds[w] = D[w];
  for (long long e = blockIdx.x; e < comps; e += gridDim.x) {
    for (int w = threadIdx.x; w < k; w += blockDim.x) Ys[w] = Y[(size_t)e * k + w];
    __syncthreads();
    block_mul(Ds, wD, Ys, k, s.T, nT, s);  // T = D Y, exactly
    for (int w = threadIdx.x; w < nq; w += blockDim.x) q[w] = s.T[k - 1 + w];
    __syncthreads();
    block_mul(q, nq, t.MU, k + 1, s.Q2, nq + k + 1, s);  // q1 MU
    for (int w = threadIdx.x; w < nq; w += blockDim.x) q[w] = s.Q2[k + 1 + w];  // q3 (< B^(wD + 1))
    __syncthreads();
    block_mul(q, nq, t.PM, k, s.R2, k + 1, s);  // q3 PM mod B^(k + 1)
    uint32_t* out = N + (size_t)e * nN;
    // r = T - q3 PM modulo B^(k + 1), then at most two subtractions of PM
    for (int w = threadIdx.x; w <= k; w += blockDim.x) out[w] = s.T[w];
    __syncthreads();
    block_sub(out, k + 1, s.R2, k + 1);
    __syncthreads();
    for (int it = 0; it < 2 && block_cmp(out, k + 1, t.PM, k) >= 0; ++it) {
      block_sub(out, k + 1, t.PM, k);
      __syncthreads();
    }
    int bits = -1;
    if (block_cmp(out, k + 1, t.PM, k) < 0) {  // always (else reported as not fitting)
      // balanced: with h = PM - r, N = -h when r > h (2 r > PM), else N = r
      uint32_t* h = s.R2;
      for (int w = threadIdx.x; w <= k; w += blockDim.x) h[w] = w < k ? t.PM[w] : 0u;
      __syncthreads();
      block_sub(h, k + 1, out, k + 1);
      __syncthreads();
      const bool negative = block_cmp(out, k + 1, h, k + 1) > 0;
      if (negative) {
        block_sub(out, k + 1, t.PM, k);  // r - PM: the two's complement of -h
      }
      if (threadIdx.x == 0) out[k + 1] = negative ? 0xFFFFFFFFu : 0u;
      __syncthreads();
      bool pow2;
      bits = block_bits(negative ? h : out, k + 1, pow2);
      if (!(bits <= bound_bits || (bits == bound_bits + 1 && pow2))) bits = -1;
    }
    if (threadIdx.x == 0) info[e] = bits;
    __syncthreads();
  }
}

}  // namespace

size_t recon_scratch_bytes(const ReconTables& t, int wD, int blocks) {
  return scratch_words(t.k, wD) * 4 * (size_t)blocks;
}

int recon_blocks(long long comps) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  return (int)std::max(1LL, std::min(comps, 8LL * sms));
}

static cudaError_t allow_smem(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t recon_values(const uint32_t* digits, long long comps, const ReconTables& t, uint32_t* Y,
                         uint32_t* scratch, cudaStream_t st) {
  const size_t smem = (size_t)t.m * t.pw * 4 + (size_t)t.m * 4;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(recon_values_kernel), smem);
  if (e != cudaSuccess) return e;
  recon_values_kernel<<<recon_blocks(comps), kReconThreads, smem, st>>>(digits, comps, t, Y, scratch);
  return cudaGetLastError();
}

cudaError_t recon_numerators(const uint32_t* Y, long long comps, const ReconTables& t, const uint32_t* D, int wD,
                             int bound_bits, uint32_t* N, int* info, uint32_t* scratch, cudaStream_t st) {
  const size_t smem = ((size_t)wD + t.k + wD + 1) * 4;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(recon_numerators_kernel), smem);
  if (e != cudaSuccess) return e;
  recon_numerators_kernel<<<recon_blocks(comps), kReconThreads, smem, st>>>(Y, comps, t, D, wD, bound_bits, N, info,
                                                                            scratch);
  return cudaGetLastError();
}

}  // namespace rg
