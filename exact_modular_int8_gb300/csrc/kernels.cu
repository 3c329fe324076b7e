// kernels.cu -- planner, residue-split and balanced-Garner kernels.
//
// Pages: "exact-solve" (Method: residues modulo a squarefree product of primes
// below 256, Barrett-style reduction instead of hardware modulo, balanced-Garner
// reconstruction of the wide digit) and "enclosure-gemm" (Method: power-of-two
// fixed-point scaling planned from exponent-field reductions; the exact integer
// S and exponent Q turned into an outward IEEE pair by bit manipulation).
#include <cuda_fp16.h>

#include <cstdint>
#include <mutex>

#include "rg_common.cuh"
#include "rg_kernels.h"

namespace rg {

__constant__ Tables c_tab;

namespace {

// ---------------------------------------------------------------------------
// small device utilities
// ---------------------------------------------------------------------------

__device__ __forceinline__ int bitlen64(unsigned long long v) { return v ? 64 - __clzll(v) : 0; }

__device__ __forceinline__ int ceil_log2_i64(long long k) {  // k >= 1
  return k <= 1 ? 0 : 64 - __clzll((unsigned long long)(k - 1));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__device__ __forceinline__ int warp_max_i32(int v) { return __reduce_max_sync(0xffffffffu, v); }

// Block-wide max of a 64-bit value; result valid in thread 0.
__device__ unsigned long long block_max_u64(unsigned long long v) {
  __shared__ unsigned long long s[32];
  v = warp_max_u64(v);
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? s[lane] : 0ull;
    v = warp_max_u64(v);
  }
  __syncthreads();
  return v;
}

__device__ int block_max_i32(int v) {
  __shared__ int s[32];
  v = warp_max_i32(v);
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? s[lane] : 0;
    v = warp_max_i32(v);
  }
  __syncthreads();
  return v;
}

// ---------------------------------------------------------------------------
// Planner reductions ("enclosure-gemm", Method: three reductions over the
// exponent field, stacked and read together; for integer operands the bound
// K * max|A| * max|B| fixes the prime count)
// ---------------------------------------------------------------------------

// max |x| of A and of B (int64), one launch: blocks [0, nbA) read A.
__global__ void plan_i64_kernel(const int64_t* __restrict__ A, long long nA, const int64_t* __restrict__ B,
                                long long nB, int nbA, DevPlan* plan) {
  bool isA = (int)blockIdx.x < nbA;
  const int64_t* X = isA ? A : B;
  long long n = isA ? nA : nB;
  long long b0 = isA ? blockIdx.x : blockIdx.x - nbA;
  long long nb = isA ? nbA : gridDim.x - nbA;
  unsigned long long m = 0;
  for (long long i = b0 * blockDim.x + threadIdx.x; i < n; i += nb * blockDim.x) {
    long long x = X[i];
    unsigned long long a = x < 0 ? 0ull - (unsigned long long)x : (unsigned long long)x;
    m = a > m ? a : m;
  }
  m = block_max_u64(m);
  if (threadIdx.x == 0 && m) atomicMax(isA ? &plan->maxmag_a : &plan->maxmag_b, m);
}

// Bit length of |x| for multi-limb x (two's complement, signed top limb).
__device__ __forceinline__ int limb_magnitude_bits(const int64_t* x, int L) {
  unsigned long long w[RG_MAX_LIMBS_IN];
  bool neg = x[L - 1] < 0;
  unsigned long long carry = 1;
#pragma unroll
  for (int i = 0; i < RG_MAX_LIMBS_IN; ++i) {
    if (i < L) {
      unsigned long long v = (unsigned long long)x[i];
      if (neg) {
        v = ~v + carry;
        carry = (v == 0 && carry) ? 1 : 0;
      }
      w[i] = v;
    }
  }
  for (int i = L - 1; i >= 0; --i)
    if (w[i]) return 64 * i + bitlen64(w[i]);
  return 0;
}

__global__ void plan_limbs_kernel(const int64_t* __restrict__ A, long long nA, int la, const int64_t* __restrict__ B,
                                  long long nB, int lb, int nbA, DevPlan* plan) {
  bool isA = (int)blockIdx.x < nbA;
  const int64_t* X = isA ? A : B;
  long long n = isA ? nA : nB;
  int L = isA ? la : lb;
  long long b0 = isA ? blockIdx.x : blockIdx.x - nbA;
  long long nb = isA ? nbA : gridDim.x - nbA;
  int m = 0;
  for (long long i = b0 * blockDim.x + threadIdx.x; i < n; i += nb * blockDim.x) {
    int b = limb_magnitude_bits(X + i * L, L);
    m = b > m ? b : m;
  }
  m = block_max_i32(m);
  if (threadIdx.x == 0 && m) atomicMax(isA ? &plan->maxbits_a : &plan->maxbits_b, m);
}

// fp64: max and min of max(biased exponent, 1) over nonzero entries, and a
// non-finite flag.  Reads only the bit patterns.
__global__ void plan_f64_kernel(const unsigned long long* __restrict__ A, long long nA,
                                const unsigned long long* __restrict__ B, long long nB, int nbA, DevPlan* plan) {
  bool isA = (int)blockIdx.x < nbA;
  const unsigned long long* X = isA ? A : B;
  long long n = isA ? nA : nB;
  long long b0 = isA ? blockIdx.x : blockIdx.x - nbA;
  long long nb = isA ? nbA : gridDim.x - nbA;
  int emax = 0, einv = 0, bad = 0;
  for (long long i = b0 * blockDim.x + threadIdx.x; i < n; i += nb * blockDim.x) {
    unsigned long long v = X[i];
    int be = (int)((v >> 52) & 0x7FF);
    if (be == 0x7FF) {
      bad = 1;
      continue;
    }
    if ((v << 1) == 0) continue;  // +-0
    int e = be > 1 ? be : 1;
    emax = e > emax ? e : emax;
    einv = (4096 - e) > einv ? (4096 - e) : einv;
  }
  emax = block_max_i32(emax);
  einv = block_max_i32(einv);
  bad = block_max_i32(bad);
  if (threadIdx.x == 0) {
    if (emax) atomicMax(isA ? &plan->maxe_a : &plan->maxe_b, emax);
    if (einv) atomicMax(isA ? &plan->inv_mine_a : &plan->inv_mine_b, einv);
    if (bad) atomicMax(&plan->nonfinite, 1);
  }
}

// ---------------------------------------------------------------------------
// Plan finalisation, evaluated identically by every block of the split kernel
// ---------------------------------------------------------------------------

struct LocalPlan {
  int status, P, bits_a, bits_b, T, f_a, f_b, lossless, nchunk_a, nchunk_b;
};

__device__ int primes_for_bound(int T) {  // fewest primes with P > 2^(T+1); 0 if none
  for (int n = 1; n <= kNumPrimes; ++n)
    if (c_tab.log2P[n] >= T + 1) return n;
  return 0;
}

__device__ LocalPlan finalize_plan(const DevPlan* plan, int op, long long K, int nprimes_fixed, int la, int lb,
                                   int lc) {
  LocalPlan p = {};
  int ck = ceil_log2_i64(K);
  auto full_chunks = [](int L) { return (64 * L + kChunkBits - 1) / kChunkBits; };
  if (op == RG_OP_I64) {
    unsigned long long ma = plan->maxmag_a, mb = plan->maxmag_b;
    p.bits_a = bitlen64(ma);
    p.bits_b = bitlen64(mb);
    p.T = p.bits_a + p.bits_b + ck;
    if (nprimes_fixed) {
      p.nchunk_a = p.nchunk_b = full_chunks(1);
    } else {
      p.nchunk_a = (p.bits_a + 1 + kChunkBits - 1) / kChunkBits;
      p.nchunk_b = (p.bits_b + 1 + kChunkBits - 1) / kChunkBits;
      unsigned __int128 prod = (unsigned __int128)ma * mb;
      unsigned __int128 lim = (unsigned __int128)0x7FFFFFFFFFFFFFFFull / (unsigned long long)K;
      if (prod > lim) p.status = RG_ERR_RANGE;
    }
  } else if (op == RG_OP_LIMBS) {
    p.bits_a = plan->maxbits_a;
    p.bits_b = plan->maxbits_b;
    p.T = p.bits_a + p.bits_b + ck;
    if (nprimes_fixed) {
      p.nchunk_a = full_chunks(la);
      p.nchunk_b = full_chunks(lb);
    } else {
      p.nchunk_a = min((p.bits_a + 1 + kChunkBits - 1) / kChunkBits, full_chunks(la));
      p.nchunk_b = min((p.bits_b + 1 + kChunkBits - 1) / kChunkBits, full_chunks(lb));
      if (p.T > RG_MAX_BOUND_BITS || p.T > 64 * lc - 1) p.status = RG_ERR_RANGE;
    }
  } else {  // RG_OP_ENCLOSE
    if (plan->nonfinite) {
      p.status = RG_ERR_NONFINITE;
      return p;
    }
    int ea = plan->maxe_a, eb = plan->maxe_b;
    int mina = 4096 - plan->inv_mine_a, minb = 4096 - plan->inv_mine_b;
    p.bits_a = ea ? ea - mina + 53 : 0;  // |A * 2^f_a| < 2^bits_a
    p.bits_b = eb ? eb - minb + 53 : 0;
    p.f_a = ea ? 1075 - mina : 0;        // finest binary point of A: 2^-f_a
    p.f_b = eb ? 1075 - minb : 0;
    p.T = p.bits_a + p.bits_b + ck;
    p.lossless = p.bits_a <= 255 && p.bits_b <= 255 && p.T <= RG_MAX_BOUND_BITS;
    if (!p.lossless) p.status = RG_ERR_LOSSY;
  }
  if (p.status) return p;
  p.P = nprimes_fixed ? nprimes_fixed : primes_for_bound(p.T);
  if (p.P == 0) p.status = RG_ERR_RANGE;
  return p;
}

// ---------------------------------------------------------------------------
// Residue split ("exact-solve", Method: residues for every prime at once,
// reduction by a precomputed reciprocal instead of hardware modulo)
//
// Every entry x is written as sum_c a_c 2^(12c) with 12-bit chunks a_c (the
// top chunk signed), so x mod q == sum_c a_c w_{q,c} (mod q) with the
// balanced weights w_{q,c} = 2^(12c) mod q.  With |a_c| < 2^12, |w| <= 125 and
// at most 22 chunks the sum stays below 2^24 and is formed exactly in fp32;
// one reciprocal-based reduction then yields the balanced residue, written as
// fp16 (exact for |r| <= 125).  Columns from C up to the padded row length
// are written as zeros.
// ---------------------------------------------------------------------------

struct SplitSide {
  const void* X;   // int64 [R][C], limbs [R][C][L] or binary64 [R][C]
  __half* Y;       // [pmax][R][ldy]
  long long R, C, ldy, plane;  // plane = R * ldy
  int L;           // limbs per entry (integer kinds)
  long long items; // R * ldy / VEC
};

// 12 bits starting at bit `pos` of the sign-extended two's-complement value x[0..L).
__device__ __forceinline__ unsigned chunk_bits(const int64_t* x, int L, int pos) {
  int w = pos >> 6, off = pos & 63;
  unsigned long long sign = (unsigned long long)(x[L - 1] >> 63);
  unsigned long long lo = w < L ? (unsigned long long)x[w] : sign;
  unsigned long long v = lo >> off;
  if (off > 64 - kChunkBits) {
    unsigned long long hi = (w + 1) < L ? (unsigned long long)x[w + 1] : sign;
    v |= hi << (64 - off);
  }
  return (unsigned)(v & 0xFFFu);
}

template <int VEC, int NCH>
__device__ __forceinline__ void emit_residues(const float (&cf)[VEC][NCH], int nch, int P, __half* y,
                                              long long plane) {
  for (int p = 0; p < P; ++p) {
    const float q = c_tab.qf[p], iq = c_tab.invq[p];
    __half h[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      float s = 0.0f;
#pragma unroll
      for (int c = 0; c < NCH; ++c)
        if (c < nch) s = __fmaf_rn(cf[e][c], c_tab.chunk_w[p][c], s);
      h[e] = __float2half_rn(bal_mod(s, q, iq));
    }
    __half* dst = y + (long long)p * plane;
    if constexpr (VEC == 8) {
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(h);
    } else if constexpr (VEC == 4) {
      *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(h);
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) dst[e] = h[e];
    }
  }
}

// Integer operands (int64 when L == 1, or limbs).  VEC consecutive columns per thread.
template <int VEC, int NCH>
__global__ void __launch_bounds__(256) split_int_kernel(SplitSide sa, SplitSide sb, long long nbA, DevPlan* plan,
                                                        int op, long long K, int nprimes_fixed, int la, int lb,
                                                        int lc) {
  LocalPlan lp = finalize_plan(plan, op, K, nprimes_fixed, la, lb, lc);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    plan->P = lp.P;
    plan->bits_a = lp.bits_a;
    plan->bits_b = lp.bits_b;
    plan->bound_bits = lp.T;
    plan->nchunk_a = lp.nchunk_a;
    plan->nchunk_b = lp.nchunk_b;
    if (lp.status) set_status(&plan->status, lp.status);
  }
  if (lp.status) return;
  bool isA = (long long)blockIdx.x < nbA;
  const SplitSide& s = isA ? sa : sb;
  int nch = isA ? lp.nchunk_a : lp.nchunk_b;
  long long item = (isA ? (long long)blockIdx.x : (long long)blockIdx.x - nbA) * blockDim.x + threadIdx.x;
  if (item >= s.items) return;
  long long per_row = s.ldy / VEC;
  long long row = item / per_row;
  long long col0 = (item - row * per_row) * VEC;
  const int64_t* X = static_cast<const int64_t*>(s.X);
  float cf[VEC][NCH];
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    long long col = col0 + e;
    if (col < s.C) {
      const int64_t* x = X + (row * s.C + col) * s.L;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        if (c < nch) {
          unsigned a = chunk_bits(x, s.L, c * kChunkBits);
          int v = (c == nch - 1) ? (int)((a ^ 0x800u) - 0x800u) : (int)a;  // top chunk signed
          cf[e][c] = (float)v;
        } else {
          cf[e][c] = 0.0f;
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < NCH; ++c) cf[e][c] = 0.0f;
    }
  }
  emit_residues<VEC, NCH>(cf, nch, lp.P, s.Y + row * s.ldy + col0, s.plane);
}

// Binary64 operands: X' = x * 2^f = +-m * 2^sh with sh = max(be,1) - min(be',1)
// >= 0; the 53-bit significand shifted by sh % 12 is cut into six chunks
// starting at chunk index sh / 12.  No floating-point instruction reads x.
template <int VEC>
__global__ void __launch_bounds__(256) split_f64_kernel(SplitSide sa, SplitSide sb, long long nbA, DevPlan* plan,
                                                        long long K) {
  __shared__ float w_s[kNumPrimes][kMaxChunks];
  LocalPlan lp = finalize_plan(plan, RG_OP_ENCLOSE, K, 0, 1, 1, 1);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    plan->P = lp.P;
    plan->bits_a = lp.bits_a;
    plan->bits_b = lp.bits_b;
    plan->bound_bits = lp.T;
    plan->f_a = lp.f_a;
    plan->f_b = lp.f_b;
    plan->lossless = lp.lossless;
    if (lp.status) set_status(&plan->status, lp.status);
  }
  if (lp.status) return;
  for (int i = threadIdx.x; i < lp.P * kMaxChunks; i += blockDim.x)
    w_s[i / kMaxChunks][i % kMaxChunks] = c_tab.chunk_w[i / kMaxChunks][i % kMaxChunks];
  __syncthreads();
  bool isA = (long long)blockIdx.x < nbA;
  const SplitSide& s = isA ? sa : sb;
  int emin = isA ? 4096 - plan->inv_mine_a : 4096 - plan->inv_mine_b;
  long long item = (isA ? (long long)blockIdx.x : (long long)blockIdx.x - nbA) * blockDim.x + threadIdx.x;
  if (item >= s.items) return;
  long long per_row = s.ldy / VEC;
  long long row = item / per_row;
  long long col0 = (item - row * per_row) * VEC;
  const unsigned long long* X = static_cast<const unsigned long long*>(s.X);
  constexpr int NC = 6;
  float cf[VEC][NC];
  int c0[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    long long col = col0 + e;
    unsigned long long v = col < s.C ? X[row * s.C + col] : 0ull;
    int be = (int)((v >> 52) & 0x7FF);
    unsigned long long m = (v & 0xFFFFFFFFFFFFFull) | (be ? (1ull << 52) : 0ull);
    int sh = (be > 1 ? be : 1) - emin;
    if (m == 0) sh = 0;
    c0[e] = sh / kChunkBits;
    unsigned long long t = m << (sh % kChunkBits);
    float sg = (v >> 63) ? -1.0f : 1.0f;
#pragma unroll
    for (int c = 0; c < NC; ++c) cf[e][c] = sg * (float)(unsigned)((t >> (kChunkBits * c)) & 0xFFFu);
  }
  __half* y = s.Y + row * s.ldy + col0;
  for (int p = 0; p < lp.P; ++p) {
    const float q = c_tab.qf[p], iq = c_tab.invq[p];
    __half h[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      float acc = 0.0f;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc = __fmaf_rn(cf[e][c], w_s[p][c0[e] + c], acc);
      h[e] = __float2half_rn(bal_mod(acc, q, iq));
    }
    *reinterpret_cast<uint4*>(y + (long long)p * s.plane) = *reinterpret_cast<const uint4*>(h);
  }
}

// ---------------------------------------------------------------------------
// Balanced Garner ("exact-solve" and "enclosure-gemm", Method: balanced-Garner
// mixed-radix digits).  With Q_i = q_0 ... q_{i-1} the digits
//   v_i = bal( (r_i - sum_{j<i} v_j Q_j) Q_i^-1  mod q_i ),  |v_i| <= (q_i-1)/2,
// give x = sum_i v_i Q_i, the unique representative with |x| <= (P-1)/2.
// Each digit costs one int8x4 dot product per four earlier digits and one
// reciprocal reduction; x is then evaluated by Horner from the top digit.
// ---------------------------------------------------------------------------

constexpr int kGE = 4;  // output elements per thread (one 32-bit residue load per prime)

__device__ __forceinline__ void garner_digits(const uint8_t* __restrict__ rc, long long plane, int P,
                                              uint32_t (&V)[kGE][kGarnerWords]) {
#pragma unroll
  for (int e = 0; e < kGE; ++e)
#pragma unroll
    for (int w = 0; w < kGarnerWords; ++w) V[e][w] = 0u;
#pragma unroll
  for (int i = 0; i < kNumPrimes; ++i) {
    if (i < P) {
      uint32_t rw = __ldg(reinterpret_cast<const uint32_t*>(rc + (long long)i * plane));
      const float q = c_tab.qf[i], iq = c_tab.invq[i];
      const int gi = c_tab.ginv[i];
#pragma unroll
      for (int e = 0; e < kGE; ++e) {
        int s = gi * (int)((rw >> (8 * e)) & 0xFFu);
        int acc = 0;
#pragma unroll
        for (int w = 0; w < kGarnerWords; ++w)
          if (4 * w < i) acc = __dp4a((int)V[e][w], c_tab.gd_packed[i][w], acc);
        s -= acc;
        int v = (int)bal_mod((float)s, q, iq);
        V[e][i / 4] |= ((uint32_t)v & 0xFFu) << (8 * (i % 4));
      }
    }
  }
}

__device__ __forceinline__ int digit(const uint32_t (&V)[kGarnerWords], int i) {
  return (int)(int8_t)((V[i / 4] >> (8 * (i % 4))) & 0xFFu);
}

// x (W 32-bit words, two's complement, mod 2^(32W)) = sum_i v_i Q_i by Horner.
template <int W>
__device__ __forceinline__ void horner_words(const uint32_t (&V)[kGarnerWords], int P, uint32_t (&x)[W]) {
#pragma unroll
  for (int k = 0; k < W; ++k) x[k] = 0u;
#pragma unroll
  for (int i = kNumPrimes - 1; i >= 0; --i) {
    if (i < P) {
      // x = x * q_i + v_i
      // The digit is added sign-extended to W words; all arithmetic is mod 2^(32W).
      const uint32_t q = (uint32_t)c_tab.q[i];
      const int v = digit(V, i);
      const uint32_t ext = v < 0 ? 0xFFFFFFFFu : 0u;
      unsigned long long carry = 0ull;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const unsigned long long t =
            (unsigned long long)x[k] * q + (k == 0 ? (unsigned long long)(uint32_t)v : (unsigned long long)ext) + carry;
        x[k] = (uint32_t)t;
        carry = t >> 32;
      }
    }
  }
}

template <int LC>
__global__ void __launch_bounds__(128) garner_int_kernel(const uint8_t* __restrict__ RC, long long ldc,
                                                         long long plane, long long M, long long N, DevPlan* plan,
                                                         int64_t* __restrict__ C) {
  if (plan->status) return;
  int P = plan->P;
  long long per_row = (N + kGE - 1) / kGE;
  long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= M * per_row) return;
  long long m = item / per_row;
  long long n0 = (item - m * per_row) * kGE;
  uint32_t V[kGE][kGarnerWords];
  garner_digits(RC + m * ldc + n0, plane, P, V);
#pragma unroll
  for (int e = 0; e < kGE; ++e) {
    if (n0 + e >= N) break;
    uint32_t x[2 * LC];
    horner_words<2 * LC>(V[e], P, x);
    int64_t* out = C + ((m * N) + n0 + e) * LC;
#pragma unroll
    for (int l = 0; l < LC; ++l) out[l] = (int64_t)(((unsigned long long)x[2 * l + 1] << 32) | x[2 * l]);
  }
}

// Outward bit-pattern epilogue ("enclosure-gemm", Method): S (W words, two's
// complement) times 2^-Q -> (lo, hi) IEEE binary64 bit patterns.
constexpr int kEncW = 11;  // 352 bits hold |S| < 2^333 with its sign

__device__ __forceinline__ void outward_bits(const uint32_t (&x)[kEncW], int Q, unsigned long long& lo,
                                             unsigned long long& hi) {
  const unsigned long long kMaxFinite = 0x7FEFFFFFFFFFFFFFull, kInf = 0x7FF0000000000000ull,
                           kSign = 0x8000000000000000ull;
  bool neg = (x[kEncW - 1] >> 31) != 0;
  uint32_t mag[kEncW];
  unsigned long long carry = neg ? 1ull : 0ull;
#pragma unroll
  for (int k = 0; k < kEncW; ++k) {
    unsigned long long t = (unsigned long long)(neg ? ~x[k] : x[k]) + carry;
    mag[k] = (uint32_t)t;
    carry = t >> 32;
  }
  int L = -1;  // index of the leading bit
#pragma unroll
  for (int k = kEncW - 1; k >= 0; --k)
    if (L < 0 && mag[k]) L = 32 * k + 31 - __clz(mag[k]);
  if (L < 0) {  // S == 0
    lo = hi = 0ull;
    return;
  }
  int E = L - Q;  // floor(log2 |S 2^-Q|)
  if (E > 1023) {
    lo = neg ? (kSign | kInf) : kMaxFinite;
    hi = neg ? (kSign | kMaxFinite) : kInf;
    return;
  }
  int u = E - 52 > -1074 ? E - 52 : -1074;  // exponent of one ulp at this magnitude
  int sh = u + Q;                            // bit of |S| holding that ulp
  unsigned long long T = 0ull;
  bool rem = false;
  if (sh <= 0) {
    // exact: |S| < 2^53 after the shift, since L - sh <= 52
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      int b = 32 * k - sh;  // destination bit of word k
      if (b < 64 && k < kEncW) T |= (unsigned long long)mag[k] << b;
    }
  } else {
    // T = bits [sh, sh + 53) of |S|; rem = any bit below sh
#pragma unroll
    for (int k = 0; k < kEncW; ++k) {
      int lo_bit = 32 * k, hi_bit = 32 * k + 32;
      unsigned long long w = mag[k];
      if (hi_bit <= sh) {
        rem |= w != 0;
      } else if (lo_bit < sh) {
        int cut = sh - lo_bit;
        rem |= (w & ((1ull << cut) - 1ull)) != 0;
        T |= w >> cut;
      } else if (lo_bit - sh < 64) {
        T |= w << (lo_bit - sh);
      }
    }
    T &= (1ull << 53) - 1ull;
  }
  unsigned long long enc = (E >= -1022 ? (unsigned long long)(E + 1022) << 52 : 0ull) + T;
  if (!rem) {
    lo = hi = (neg ? kSign : 0ull) | enc;
  } else if (!neg) {
    lo = enc;
    hi = enc + 1ull;
  } else {
    lo = kSign | (enc + 1ull);
    hi = kSign | enc;
  }
}

__global__ void __launch_bounds__(128) garner_enclose_kernel(const uint8_t* __restrict__ RC, long long ldc,
                                                             long long plane, long long M, long long N,
                                                             DevPlan* plan, unsigned long long* __restrict__ lo,
                                                             unsigned long long* __restrict__ hi) {
  if (plan->status) return;
  int P = plan->P;
  int Q = plan->f_a + plan->f_b;
  long long per_row = (N + kGE - 1) / kGE;
  long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= M * per_row) return;
  long long m = item / per_row;
  long long n0 = (item - m * per_row) * kGE;
  uint32_t V[kGE][kGarnerWords];
  garner_digits(RC + m * ldc + n0, plane, P, V);
#pragma unroll
  for (int e = 0; e < kGE; ++e) {
    if (n0 + e >= N) break;
    uint32_t x[kEncW];
    horner_words<kEncW>(V[e], P, x);
    unsigned long long l, h;
    outward_bits(x, Q, l, h);
    lo[m * N + n0 + e] = l;
    hi[m * N + n0 + e] = h;
  }
}

int g_sm_count[64];

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!g_sm_count[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = n > 0 ? n : 148;
  }
  return g_sm_count[dev];
}

}  // namespace

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

cudaError_t upload_tables() {
  static std::mutex mu;
  static bool done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaMemcpyToSymbol(c_tab, &host_tables(), sizeof(Tables));
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

static int planner_blocks(long long n) {
  long long b = (n + 256LL * 8 - 1) / (256LL * 8);
  long long cap = 2LL * sm_count();
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

cudaError_t launch_plan_i64(const int64_t* A, long long nA, const int64_t* B, long long nB, DevPlan* plan,
                            cudaStream_t s) {
  int ba = planner_blocks(nA), bb = planner_blocks(nB);
  plan_i64_kernel<<<ba + bb, 256, 0, s>>>(A, nA, B, nB, ba, plan);
  return cudaGetLastError();
}

cudaError_t launch_plan_limbs(const int64_t* A, long long nA, int la, const int64_t* B, long long nB, int lb,
                              DevPlan* plan, cudaStream_t s) {
  int ba = planner_blocks(nA), bb = planner_blocks(nB);
  plan_limbs_kernel<<<ba + bb, 256, 0, s>>>(A, nA, la, B, nB, lb, ba, plan);
  return cudaGetLastError();
}

cudaError_t launch_plan_f64(const double* A, long long nA, const double* B, long long nB, DevPlan* plan,
                            cudaStream_t s) {
  int ba = planner_blocks(nA), bb = planner_blocks(nB);
  plan_f64_kernel<<<ba + bb, 256, 0, s>>>(reinterpret_cast<const unsigned long long*>(A), nA,
                                          reinterpret_cast<const unsigned long long*>(B), nB, ba, plan);
  return cudaGetLastError();
}

static SplitSide make_side(const void* X, __half* Y, long long R, long long C, long long ldy, int L, int vec) {
  SplitSide s;
  s.X = X;
  s.Y = Y;
  s.R = R;
  s.C = C;
  s.ldy = ldy;
  s.plane = R * ldy;
  s.L = L;
  s.items = R * (ldy / vec);
  return s;
}

cudaError_t launch_split(int op, const void* A, const void* B, int la, int lb, int lc, long long M, long long N,
                         long long K, long long lda, long long ldb, void* RA, void* RB, int nprimes_fixed,
                         DevPlan* plan, cudaStream_t st) {
  __half* ra = static_cast<__half*>(RA);
  __half* rb = static_cast<__half*>(RB);
  if (op == RG_OP_ENCLOSE) {
    constexpr int V = 8;
    SplitSide sa = make_side(A, ra, M, K, lda, 1, V), sb = make_side(B, rb, K, N, ldb, 1, V);
    long long nbA = (sa.items + 255) / 256, nbB = (sb.items + 255) / 256;
    split_f64_kernel<V><<<(unsigned)(nbA + nbB), 256, 0, st>>>(sa, sb, nbA, plan, K);
    return cudaGetLastError();
  }
  int L = la > lb ? la : lb;
  if (L <= 1) {
    constexpr int V = 8;
    SplitSide sa = make_side(A, ra, M, K, lda, la, V), sb = make_side(B, rb, K, N, ldb, lb, V);
    long long nbA = (sa.items + 255) / 256, nbB = (sb.items + 255) / 256;
    split_int_kernel<V, 6><<<(unsigned)(nbA + nbB), 256, 0, st>>>(sa, sb, nbA, plan, op, K, nprimes_fixed, la, lb,
                                                                  lc);
  } else if (L <= 2) {
    constexpr int V = 4;
    SplitSide sa = make_side(A, ra, M, K, lda, la, V), sb = make_side(B, rb, K, N, ldb, lb, V);
    long long nbA = (sa.items + 255) / 256, nbB = (sb.items + 255) / 256;
    split_int_kernel<V, 11><<<(unsigned)(nbA + nbB), 256, 0, st>>>(sa, sb, nbA, plan, op, K, nprimes_fixed, la, lb,
                                                                   lc);
  } else {
    constexpr int V = 2;
    SplitSide sa = make_side(A, ra, M, K, lda, la, V), sb = make_side(B, rb, K, N, ldb, lb, V);
    long long nbA = (sa.items + 255) / 256, nbB = (sb.items + 255) / 256;
    split_int_kernel<V, 22><<<(unsigned)(nbA + nbB), 256, 0, st>>>(sa, sb, nbA, plan, op, K, nprimes_fixed, la, lb,
                                                                   lc);
  }
  return cudaGetLastError();
}

cudaError_t launch_garner(int op, const void* RC, long long ldc, long long plane, long long M, long long N, int lc,
                          DevPlan* plan, void* out0, void* out1, cudaStream_t st) {
  long long items = M * ((N + kGE - 1) / kGE);
  unsigned blocks = (unsigned)((items + 127) / 128);
  const uint8_t* rc = static_cast<const uint8_t*>(RC);
  if (op == RG_OP_ENCLOSE) {
    garner_enclose_kernel<<<blocks, 128, 0, st>>>(rc, ldc, plane, M, N, plan,
                                                  static_cast<unsigned long long*>(out0),
                                                  static_cast<unsigned long long*>(out1));
    return cudaGetLastError();
  }
  int64_t* C = static_cast<int64_t*>(out0);
  switch (lc) {
    case 1: garner_int_kernel<1><<<blocks, 128, 0, st>>>(rc, ldc, plane, M, N, plan, C); break;
    case 2: garner_int_kernel<2><<<blocks, 128, 0, st>>>(rc, ldc, plane, M, N, plan, C); break;
    case 3: garner_int_kernel<3><<<blocks, 128, 0, st>>>(rc, ldc, plane, M, N, plan, C); break;
    case 4: garner_int_kernel<4><<<blocks, 128, 0, st>>>(rc, ldc, plane, M, N, plan, C); break;
    case 5: garner_int_kernel<5><<<blocks, 128, 0, st>>>(rc, ldc, plane, M, N, plan, C); break;
    case 6: garner_int_kernel<6><<<blocks, 128, 0, st>>>(rc, ldc, plane, M, N, plan, C); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace rg
