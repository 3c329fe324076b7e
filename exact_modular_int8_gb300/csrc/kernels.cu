// kernels.cu -- planner, residue-split and balanced-Garner kernels.
//
// Pages: "exact-solve" (Method: residues modulo a squarefree product of primes
// below 256, Barrett-style reduction instead of hardware modulo, balanced-Garner
// reconstruction of the wide digit) and "enclosure-gemm" (Method: power-of-two
// fixed-point scaling planned from exponent-field reductions; the exact integer
// S and exponent Q turned into an outward IEEE pair by bit manipulation).
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>
#include <atomic>
#include <mutex>

#include "rg_common.cuh"
#include "rg_garner.cuh"
#include "rg_kernels.h"

namespace rg {

__constant__ Tables c_tab;

// Garner reads the library's own prime tables.
struct MainTab {
  __device__ static __forceinline__ const Tables& t() { return c_tab; }
};

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

// Block-wide max; result valid in thread 0.
__device__ unsigned long long block_max_u64(unsigned long long v) {
  __shared__ unsigned long long s[32];
  v = warp_max_u64(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? s[lane] : 0;
    v = warp_max_i32(v);
  }
  __syncthreads();
  return v;
}

__device__ __forceinline__ unsigned long long abs_u64(unsigned long long v) {
  return (long long)v < 0 ? 0ull - v : v;
}

// ---------------------------------------------------------------------------
// IEEE binary formats of the enclosure's operands and bounds ("enclosure-gemm",
// Usage: operands are float32 or float64), read and written as bit patterns.
// A finite nonzero x is (-1)^s * m * 2^(max(be, 1) - kLsbBias), with m the
// significand including its hidden bit (kFracBits + 1 bits).
// ---------------------------------------------------------------------------
template <typename Bits>
struct FloatFormat;
template <>
struct FloatFormat<unsigned long long> {  // binary64
  static constexpr int kFracBits = 52, kExpMask = 0x7FF, kLsbBias = 1075, kEmax = 1023, kEminNormal = -1022,
                       kUlpMin = -1074;
  static constexpr unsigned long long kMaxFinite = 0x7FEFFFFFFFFFFFFFull, kInf = 0x7FF0000000000000ull,
                                      kSign = 0x8000000000000000ull;
};
template <>
struct FloatFormat<uint32_t> {  // binary32
  static constexpr int kFracBits = 23, kExpMask = 0xFF, kLsbBias = 150, kEmax = 127, kEminNormal = -126,
                       kUlpMin = -149;
  static constexpr uint32_t kMaxFinite = 0x7F7FFFFFu, kInf = 0x7F800000u, kSign = 0x80000000u;
};

// ---------------------------------------------------------------------------
// The plan ("enclosure-gemm", Method: three reductions over the exponent
// field, stacked and read together; Requirements: K <= 2^17 and
// bits_a + bits_b + ceil(log2 K) <= 332).  The planner kernels reduce into the
// plan block with atomics; the last block to finish derives the prime count,
// the chunk counts and the fp64 scales once, for all later kernels.
// ---------------------------------------------------------------------------

struct PlanArgs {
  int op;
  long long K;
  int nprimes_fixed, la, lb, lc;
  int allow_rn;  // the wide outputs may use round-to-nearest CRT
  int pcap;      // floating point: the most primes the workspace's planes hold
};

struct LocalPlan {
  int status, P, bits_a, bits_b, T, f_a, f_b, lossless, nword_a, nword_b, crt_rn;
};

__device__ int primes_for_bound(int T) {  // fewest primes with P > 2^(T+1); 0 if none
  for (int n = 1; n <= kNumPrimes; ++n)
    if (c_tab.log2P[n] >= T + 1) return n;
  return 0;
}

// Reads the reductions through L2 (they were written with device atomics).
__device__ LocalPlan finalize_plan(DevPlan* plan, const PlanArgs& a) {
  LocalPlan p = {};
  const int ck = ceil_log2_i64(a.K);
  // 32-bit words holding an entry of `bits` magnitude bits with its sign, at most the limbs' 2L
  auto words_for = [](int bits, int L) { return min((bits + 1 + 31) / 32, 2 * L); };
  if (a.op == RG_OP_LIMBS) {
    p.bits_a = __ldcg(&plan->maxbits_a);
    p.bits_b = __ldcg(&plan->maxbits_b);
    p.T = p.bits_a + p.bits_b + ck;
    if (a.nprimes_fixed) {
      p.nword_a = 2 * a.la;
      p.nword_b = 2 * a.lb;
    } else {
      p.nword_a = p.bits_a <= 23 ? 0 : words_for(p.bits_a, a.la);
      p.nword_b = p.bits_b <= 23 ? 0 : words_for(p.bits_b, a.lb);
      if (p.T > RG_MAX_BOUND_BITS || p.T > 64 * a.lc - 1) p.status = RG_ERR_RANGE;
    }
  } else {  // RG_OP_ENCLOSE[_F32], RG_OP_INTERVAL[_F32]
    if (__ldcg(&plan->nonfinite)) {
      p.status = RG_ERR_NONFINITE;
      return p;
    }
    if (__ldcg(&plan->neg_radius)) {
      p.status = RG_ERR_RADIUS;
      return p;
    }
    const bool f32 = a.op == RG_OP_ENCLOSE_F32 || a.op == RG_OP_INTERVAL_F32;
    // intervals: the midpoint and the two radius products add up to at most
    // 4 K 2^(bits_a + bits_b), two bits above a point product
    const int extra = (a.op == RG_OP_INTERVAL || a.op == RG_OP_INTERVAL_F32) ? 2 : 0;
    const int sig = f32 ? FloatFormat<uint32_t>::kFracBits + 1 : FloatFormat<unsigned long long>::kFracBits + 1;
    const int bias = f32 ? FloatFormat<uint32_t>::kLsbBias : FloatFormat<unsigned long long>::kLsbBias;
    const int ea = __ldcg(&plan->maxe_a), eb = __ldcg(&plan->maxe_b);
    const int mina = 4096 - __ldcg(&plan->inv_mine_a), minb = 4096 - __ldcg(&plan->inv_mine_b);
    // finest binary point holding every entry exactly: |A * 2^f_a| < 2^bits_a
    const int bits_a0 = ea ? ea - mina + sig : 0, bits_b0 = eb ? eb - minb + sig : 0;
    // coarsened until each operand fits 256-bit two's complement and the
    // product fits the residue range (enclosure-gemm, Method), here the range
    // of the primes the workspace holds: the larger operand gives up bits first
    const int cap_bits = min(RG_MAX_BOUND_BITS, c_tab.log2P[a.pcap] - 1);
    if (cap_bits - ck - extra < 2) {  // not one bit per operand
      p.status = RG_ERR_WORKSPACE;
      return p;
    }
    int ba = min(bits_a0, 255), bb = min(bits_b0, 255);
    int excess = ba + bb + ck + extra - cap_bits;
    if (excess > 0) {
      const int d = min(excess, abs(ba - bb));
      if (ba >= bb) ba -= d; else bb -= d;
      excess -= d;
      ba -= (excess + 1) / 2;
      bb -= excess / 2;
    }
    p.bits_a = ba;
    p.bits_b = bb;
    p.f_a = ea ? bias - mina - (bits_a0 - ba) : 0;
    p.f_b = eb ? bias - minb - (bits_b0 - bb) : 0;
    p.T = ba + bb + ck + extra;
    p.lossless = ba == bits_a0 && bb == bits_b0;
  }
  if (p.status) return p;
  if (a.nprimes_fixed) {
    p.P = a.nprimes_fixed;
  } else {
    p.P = primes_for_bound(p.T);
    // on request the wide outputs reconstruct by round-to-nearest CRT, which
    // wants one more bit of headroom (P > 4 |x|); where 53 primes cannot give
    // it, balanced Garner reconstructs from the usual prime count
    if (a.allow_rn) {
      const int prn = primes_for_bound(p.T + 1);
      if (prn && prn <= a.pcap) {  // within the workspace's planes
        p.P = prn;
        p.crt_rn = 1;
      }
    }
  }
  if (p.P == 0) p.status = RG_ERR_RANGE;
  return p;
}

// Called at the end of every planner block: the last block writes the plan.
__device__ void planner_finish(DevPlan* plan, const PlanArgs& a) {
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned done = atomicAdd(&plan->blocks_done, 1u);
    s_last = done == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    const LocalPlan lp = finalize_plan(plan, a);
    plan->P = lp.P;
    plan->bits_a = lp.bits_a;
    plan->bits_b = lp.bits_b;
    plan->bound_bits = lp.T;
    plan->f_a = lp.f_a;
    plan->f_b = lp.f_b;
    plan->lossless = lp.lossless;
    plan->nword_a = lp.nword_a;
    plan->nword_b = lp.nword_b;
    plan->crt_rn = lp.crt_rn;
    if (lp.status) set_status(&plan->status, lp.status);
  }
  __syncthreads();
  allow_dependents();
}

// Blocks [0, nbA) read A, the others read B.
struct PlannerSide {
  long long b0, nb, stride;
  bool isA;
};
__device__ __forceinline__ PlannerSide planner_side(int nbA) {
  PlannerSide s;
  s.isA = (int)blockIdx.x < nbA;
  s.b0 = s.isA ? blockIdx.x : blockIdx.x - nbA;
  s.nb = s.isA ? nbA : gridDim.x - nbA;
  s.stride = s.nb * blockDim.x;
  return s;
}

// Bit length of |x| for an L-limb two's-complement integer held in w.
template <int L>
__device__ __forceinline__ int limb_magnitude_bits(const unsigned long long (&w)[L]) {
  const bool neg = (long long)w[L - 1] < 0;
  unsigned long long carry = 1, m[L];
#pragma unroll
  for (int i = 0; i < L; ++i) {
    unsigned long long v = w[i];
    if (neg) {
      v = ~v + carry;
      carry = (v == 0 && carry) ? 1 : 0;
    }
    m[i] = v;
  }
  int b = 0;
#pragma unroll
  for (int i = 0; i < L; ++i)
    if (m[i]) b = 64 * i + bitlen64(m[i]);
  return b;
}

// VEC: 16-byte loads (L even and the base 16-byte aligned, which the caller checks).
template <int L, bool VEC>
__device__ __forceinline__ void load_limbs(const int64_t* __restrict__ x, unsigned long long (&w)[L]) {
  if constexpr (VEC) {
    static_assert(L % 2 == 0, "pairs of limbs");
#pragma unroll
    for (int i = 0; i < L; i += 2) {
      const ulonglong2 v = __ldg(reinterpret_cast<const ulonglong2*>(x) + i / 2);
      w[i] = v.x;
      w[i + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < L; ++i) w[i] = (unsigned long long)__ldg(x + i);
  }
}

// max bit length over n L-limb entries of X, strided as the planner side says;
// four entries' limbs are loaded before any is examined.
template <int L, bool VEC>
__device__ __forceinline__ int scan_limbs(const int64_t* __restrict__ X, long long n, const PlannerSide& sd) {
  int m = 0;
  long long i = sd.b0 * blockDim.x + threadIdx.x;
  for (; i + 3 * sd.stride < n; i += 4 * sd.stride) {
    unsigned long long w0[L], w1[L], w2[L], w3[L];
    load_limbs<L, VEC>(X + i * L, w0);
    load_limbs<L, VEC>(X + (i + sd.stride) * L, w1);
    load_limbs<L, VEC>(X + (i + 2 * sd.stride) * L, w2);
    load_limbs<L, VEC>(X + (i + 3 * sd.stride) * L, w3);
    m = max(m, max(max(limb_magnitude_bits<L>(w0), limb_magnitude_bits<L>(w1)),
                   max(limb_magnitude_bits<L>(w2), limb_magnitude_bits<L>(w3))));
  }
  for (; i < n; i += sd.stride) {
    unsigned long long w[L];
    load_limbs<L, VEC>(X + i * L, w);
    m = max(m, limb_magnitude_bits<L>(w));
  }
  return m;
}

__global__ void __launch_bounds__(256) plan_limbs_kernel(const int64_t* __restrict__ A, long long nA, int la,
                                                         const int64_t* __restrict__ B, long long nB, int lb, int nbA,
                                                         DevPlan* plan, PlanArgs pa) {
  const PlannerSide sd = planner_side(nbA);
  const int64_t* X = sd.isA ? A : B;
  const long long n = sd.isA ? nA : nB;
  const int L = sd.isA ? la : lb;
  // even limb counts read 16 bytes at a time when the base is 16-byte aligned
  const bool aligned = (reinterpret_cast<uintptr_t>(X) & 15u) == 0;
  int m = 0;
  switch (L) {
    case 1: m = scan_limbs<1, false>(X, n, sd); break;
    case 2: m = aligned ? scan_limbs<2, true>(X, n, sd) : scan_limbs<2, false>(X, n, sd); break;
    case 3: m = scan_limbs<3, false>(X, n, sd); break;
    default: m = aligned ? scan_limbs<4, true>(X, n, sd) : scan_limbs<4, false>(X, n, sd); break;
  }
  m = block_max_i32(m);
  if (threadIdx.x == 0 && m) atomicMax(sd.isA ? &plan->maxbits_a : &plan->maxbits_b, m);
  planner_finish(plan, pa);
}

// Floating-point operands: max and min of max(biased exponent, 1) over nonzero
// entries and a non-finite flag, from the bit patterns only.
template <typename Bits>
__device__ __forceinline__ void exponent_stats(Bits v, int& emax, int& einv, int& bad) {
  using F = FloatFormat<Bits>;
  const int be = (int)((v >> F::kFracBits) & F::kExpMask);
  const int e = be > 1 ? be : 1;
  const bool nonzero = (Bits)(v << 1) != 0;
  const bool finite = be != F::kExpMask;
  bad |= finite ? 0 : 1;
  if (finite && nonzero) {
    emax = e > emax ? e : emax;
    einv = (4096 - e) > einv ? (4096 - e) : einv;
  }
}

// One array's share of the exponent reductions (16-byte loads when aligned);
// a radius array also flags negative entries (a set sign bit on a nonzero).
template <typename Bits>
__device__ __forceinline__ void scan_float(const Bits* __restrict__ X, long long n, const PlannerSide& sd,
                                           bool radius, int& emax, int& einv, int& bad, int& negr) {
  using F = FloatFormat<Bits>;
  constexpr int PER = 16 / sizeof(Bits);  // entries per 16-byte load
  const long long nv = (reinterpret_cast<uintptr_t>(X) & 15u) == 0 ? n / PER : 0;
  const uint4* X4 = reinterpret_cast<const uint4*>(X);
  auto one = [&](Bits v) {
    exponent_stats<Bits>(v, emax, einv, bad);
    if (radius && (v & F::kSign) && (Bits)(v << 1) != 0) negr = 1;
  };
  auto chunk = [&](const uint4& v) {
    if constexpr (PER == 4) {
      one(v.x);
      one(v.y);
      one(v.z);
      one(v.w);
    } else {
      one(((unsigned long long)v.y << 32) | v.x);
      one(((unsigned long long)v.w << 32) | v.z);
    }
  };
  long long i = sd.b0 * blockDim.x + threadIdx.x;
  for (; i + 3 * sd.stride < nv; i += 4 * sd.stride) {  // four 16-byte loads in flight before any work
    const uint4 v0 = __ldg(X4 + i), v1 = __ldg(X4 + i + sd.stride), v2 = __ldg(X4 + i + 2 * sd.stride),
                v3 = __ldg(X4 + i + 3 * sd.stride);
    chunk(v0);
    chunk(v1);
    chunk(v2);
    chunk(v3);
  }
  for (; i < nv; i += sd.stride) chunk(__ldg(X4 + i));
  for (long long i = PER * nv + sd.b0 * blockDim.x + threadIdx.x; i < n; i += sd.stride) one(__ldg(X + i));
}

// A and B, each with an optional radius array of the same size (intervals:
// one scale covers an operand's midpoints and radii).
template <typename Bits>
__global__ void __launch_bounds__(256) plan_float_kernel(const Bits* __restrict__ A, const Bits* __restrict__ A2,
                                                         long long nA, const Bits* __restrict__ B,
                                                         const Bits* __restrict__ B2, long long nB, int nbA,
                                                         DevPlan* plan, PlanArgs pa) {
  const PlannerSide sd = planner_side(nbA);
  const long long n = sd.isA ? nA : nB;
  const Bits* X2 = sd.isA ? A2 : B2;
  int emax = 0, einv = 0, bad = 0, negr = 0;
  scan_float<Bits>(sd.isA ? A : B, n, sd, false, emax, einv, bad, negr);
  if (X2) scan_float<Bits>(X2, n, sd, true, emax, einv, bad, negr);
  emax = block_max_i32(emax);
  einv = block_max_i32(einv);
  bad = block_max_i32(bad);
  negr = block_max_i32(negr);
  if (threadIdx.x == 0) {
    if (emax) atomicMax(sd.isA ? &plan->maxe_a : &plan->maxe_b, emax);
    if (einv) atomicMax(sd.isA ? &plan->inv_mine_a : &plan->inv_mine_b, einv);
    if (bad) atomicMax(&plan->nonfinite, 1);
    if (negr) atomicMax(&plan->neg_radius, 1);
  }
  planner_finish(plan, pa);
}

// ---------------------------------------------------------------------------
// Residue split ("exact-solve", Method: residues for every prime at once,
// reduction by a precomputed reciprocal instead of hardware modulo)
//
// Integers: an entry x whose two's complement fits nw little-endian 32-bit
// words equals U - [x < 0] 2^(32 nw), U those words read as unsigned, so over
// the bytes b_j of U
//   x mod q == sum_j b_j (2^(8j) mod q) - [x < 0] (2^(32 nw) mod q)   (mod q).
// The byte weights are balanced (|w| <= 125) and packed four to a word, so a
// word costs one dp4a (unsigned data bytes times signed weights).  At most 8
// words keep the sum below 2^20, an exact fp32, and one reciprocal reduction
// gives the balanced residue.  Entries with |x| <= 2^23 skip the bytes: x is
// itself an exact fp32.
//
// Floating point: |x| 2^f = t 2^sh, t the significand (or, at a coarsened
// point, the floored scaled magnitude with sh = 0), so
//   x 2^f mod q == +-(t 2^sh mod q)   (mod q),
// and t 2^sh mod q is the dot product of t's bytes with the byte weights
// bal(2^(8k + sh) mod q) of its shift (ShiftWeights), reduced once.
//
// Residues are written as fp16 (exact for |r| <= 125).  Columns from C up to
// the padded row length are written as zeros.  Grid-stride over the items
// (VEC consecutive entries of one row) of A, then of B.
// ---------------------------------------------------------------------------

struct SplitSide {
  const void* X;   // int64 [R][C], limbs [R][C][L] or floating point [R][C]
  __half* Y;       // [pmax][R][ldy]
  long long R, C, ldy, plane;  // plane = R * ldy
  int L;           // limbs per entry (integer kinds)
  long long items; // R * ldy / VEC
  RowDiv rd;       // division by the items per row, ldy / VEC
};

// c + the four bytes of a (unsigned) dotted with the four bytes of b (signed).
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Per-prime constants of a split block, read with 16-byte shared loads.
struct alignas(16) PrimeRec {
  int w[kMaxWords];  // packed byte weights of words 0..7
  float q, iq;       // q and fl(1/q)
  int pad[2];
};

// The records of every prime, built on the host and uploaded with the
// constant tables; kept in global memory so that a block copies them to
// shared memory with coalesced 16-byte loads (the constant bank serialises
// loads whose addresses differ across a warp).
struct SplitTables {
  PrimeRec rec[kNumPrimes];
  int ws[kNumPrimes][kMaxWords + 1];
};
__device__ SplitTables g_split;

// Every prime's record (and, if ws is given, its word-string weights); none
// of it depends on the predecessor kernel, so it is read before waiting.
__device__ __forceinline__ void load_prime_recs(PrimeRec* rec, int (*ws)[kMaxWords + 1]) {
  constexpr int kRecVec = (int)(sizeof(PrimeRec) * kNumPrimes / 16);
  for (int i = threadIdx.x; i < kRecVec; i += blockDim.x)
    reinterpret_cast<uint4*>(rec)[i] = reinterpret_cast<const uint4*>(g_split.rec)[i];
  if (ws)
    for (int i = threadIdx.x; i < kNumPrimes * (kMaxWords + 1); i += blockDim.x)
      (&ws[0][0])[i] = (&g_split.ws[0][0])[i];
}

// The first NW packed byte weights of a record (NW = 1, 2, 4 or 8).
template <int NW>
__device__ __forceinline__ void load_weights(const PrimeRec& r, int (&wv)[NW]) {
  if constexpr (NW == 1) {
    wv[0] = r.w[0];
  } else if constexpr (NW == 2) {
    const int2 v = *reinterpret_cast<const int2*>(r.w);
    wv[0] = v.x;
    wv[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < NW; k += 4) {
      const int4 v = *reinterpret_cast<const int4*>(r.w + k);
      wv[k] = v.x;
      wv[k + 1] = v.y;
      wv[k + 2] = v.z;
      wv[k + 3] = v.w;
    }
  }
}

template <int VEC>
__device__ __forceinline__ void store_residues(const float (&r)[VEC], __half* dst) {
  static_assert(VEC == 2 || VEC == 4 || VEC == 8, "residues are written as half2 pairs");
  __half2 h[VEC / 2];
#pragma unroll
  for (int e = 0; e < VEC / 2; ++e) h[e] = __floats2half2_rn(r[2 * e], r[2 * e + 1]);
  if constexpr (VEC == 8)
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(h);
  else if constexpr (VEC == 4)
    *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(h);
  else
    *reinterpret_cast<__half2*>(dst) = h[0];
}

// Residues of VEC integer entries for every prime: nw == 0 takes the exact
// fp32 values xf, otherwise the first nw words wd with the signs neg.
template <int VEC, int NW>
__device__ __forceinline__ void emit_int_residues(const uint32_t (&wd)[VEC][NW], const bool (&neg)[VEC],
                                                  const float (&xf)[VEC], int nw, int P, const PrimeRec* rec,
                                                  const int (*ws)[kMaxWords + 1], __half* y, long long plane,
                                                  int p0 = 0) {
  for (int p = p0; p < P; ++p) {
    const PrimeRec& R = rec[p];
    const float q = R.q, iq = R.iq;
    float r[VEC];
    if (nw == 0) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) r[e] = bal_mod_small(xf[e], q, iq);
    } else {
      int wv[NW];
      load_weights<NW>(R, wv);
#pragma unroll
      for (int w = 0; w < NW; ++w) wv[w] = w < nw ? wv[w] : 0;  // words past nw weigh nothing
      const int sg = ws[p][nw];
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        int acc = neg[e] ? -sg : 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) acc = dp4a_us(wd[e][w], wv[w], acc);
        r[e] = bal_mod_small(int_to_float_exact(acc), q, iq);  // |acc| < 2^20
      }
    }
    store_residues<VEC>(r, y + (long long)p * plane);
  }
}

// Integer operands: int64 (L = 1) or limbs (L <= LMAX).  VEC consecutive
// columns per item; their VEC * L words are contiguous and are read with
// 16-byte loads when they lie fully inside the row and are aligned.
template <int VEC, int LMAX>
__global__ void __launch_bounds__(256) split_int_kernel(SplitSide sa, SplitSide sb, const DevPlan* plan) {
  constexpr int NW = 2 * LMAX;
  __shared__ PrimeRec rec[kNumPrimes];
  __shared__ int ws[kNumPrimes][kMaxWords + 1];
  load_prime_recs(rec, ws);
  __syncthreads();
  wait_for_predecessor();
  if (plan->status) return;
  const int P = plan->P;
  const int nw_a = plan->nword_a, nw_b = plan->nword_b;
  const long long total = sa.items + sb.items;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const bool isA = it < sa.items;
    const SplitSide& s = isA ? sa : sb;
    const int nw = isA ? nw_a : nw_b;
    const long long item = isA ? it : it - sa.items;
    const long long per_row = s.ldy / VEC;
    const long long row = div_row(item, s.rd);
    const long long col0 = (item - row * per_row) * VEC;
    const int L = s.L;
    const unsigned long long* X = static_cast<const unsigned long long*>(s.X) + (row * s.C + col0) * L;
    unsigned long long xw[VEC][LMAX];
    if (col0 + VEC <= s.C && L == LMAX && ((reinterpret_cast<uintptr_t>(X) & 15u) == 0) &&
        (VEC * LMAX) % 2 == 0) {
#pragma unroll
      for (int t = 0; t < VEC * LMAX / 2; ++t) {
        const ulonglong2 v = __ldg(reinterpret_cast<const ulonglong2*>(X) + t);
        xw[(2 * t) / LMAX][(2 * t) % LMAX] = v.x;
        xw[(2 * t + 1) / LMAX][(2 * t + 1) % LMAX] = v.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e)
#pragma unroll
        for (int k = 0; k < LMAX; ++k) xw[e][k] = (col0 + e < s.C && k < L) ? __ldg(X + e * L + k) : 0ull;
    }
    uint32_t wd[VEC][NW];
    bool neg[VEC];
    float xf[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      unsigned long long top = 0ull;  // the top limb, selected with masks (no dynamic register index)
#pragma unroll
      for (int k = 0; k < LMAX; ++k) top |= xw[e][k] & (0ull - (unsigned long long)(k == L - 1));
      neg[e] = (long long)top < 0;
      xf[e] = (float)(int)(long long)xw[e][0];  // used only when |x| <= 2^23
#pragma unroll
      for (int k = 0; k < LMAX; ++k) {
        wd[e][2 * k] = (uint32_t)xw[e][k];
        wd[e][2 * k + 1] = (uint32_t)(xw[e][k] >> 32);
      }
    }
    emit_int_residues<VEC, NW>(wd, neg, xf, nw, P, rec, ws, s.Y + row * s.ldy + col0, s.plane);
  }
  allow_dependents();
}

// int64 operands without a planner pass: every entry's residues are written
// for `P` primes (the most the bound can need, or the caller's count), the
// word count is decided per warp from the warp's largest |x|, and max |A|,
// max |B| are reduced on the side for the GEMM kernel to derive the prime count
// and check the range.  Saves one read of A and B and one kernel launch.
template <int VEC>
struct I64Item {
  unsigned long long x[VEC];
};

// The VEC int64 entries of item `it` (zeros past the row's end or the last item).
template <int VEC>
__device__ __forceinline__ I64Item<VEC> load_i64_item(const SplitSide& sa, const SplitSide& sb, long long it,
                                                      long long total) {
  I64Item<VEC> v;
  const bool valid = it < total;
  const bool isA = it < sa.items;
  const SplitSide& s = isA ? sa : sb;
  const long long item = isA ? it : it - sa.items;
  const long long per_row = s.ldy / VEC;
  const long long row = div_row(item, s.rd);
  const long long col0 = (item - row * per_row) * VEC;
  const unsigned long long* X = static_cast<const unsigned long long*>(s.X) + row * s.C + col0;
  if (valid && col0 + VEC <= s.C && ((reinterpret_cast<uintptr_t>(X) & 15u) == 0)) {
#pragma unroll
    for (int t = 0; t < VEC / 2; ++t) {
      const ulonglong2 w = __ldg(reinterpret_cast<const ulonglong2*>(X) + t);
      v.x[2 * t] = w.x;
      v.x[2 * t + 1] = w.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) v.x[e] = (valid && col0 + e < s.C) ? __ldg(X + e) : 0ull;
  }
  return v;
}

// The residue-plane count a planner-free int64 split writes: `pmax`, or the
// prime count the previous call on this workspace used (its GEMM records it,
// tagged, in the plan block beyond the part each call clears) when that is
// smaller.  A later fix-up pass writes whatever planes the call turns out to
// need beyond it, so the count only saves writes and never decides a result.
__device__ __forceinline__ int i64_planes_written(const uint32_t* hint, int pmax) {
  if (!hint) return pmax;
  const uint32_t h = __ldcg(hint);
  const int p = (int)(h & 0xFFFFu);
  return (h & 0xFFFF0000u) == kPlaneHintTag && p >= 1 && p < pmax ? p : pmax;
}

// Residues of the VEC int64 entries of `cur` (item `it`) for the primes
// [p0, p1); the word count is decided per warp from the warp's largest |x|
// (none when every |x| <= 2^23), m receives this item's largest |x|.
template <int VEC>
__device__ __forceinline__ void emit_i64_item(const SplitSide& sa, const SplitSide& sb, const I64Item<VEC>& cur,
                                              long long it, long long total, int p0, int p1, const PrimeRec* rec,
                                              const int (*ws)[kMaxWords + 1], unsigned long long& m, bool& isA) {
  const bool valid = it < total;
  isA = it < sa.items;
  const SplitSide& s = isA ? sa : sb;
  const long long item = isA ? it : it - sa.items;
  const long long per_row = s.ldy / VEC;
  const long long row = div_row(item, s.rd);
  const long long col0 = (item - row * per_row) * VEC;
  m = 0;
#pragma unroll
  for (int e = 0; e < VEC; ++e) m = max(m, abs_u64(cur.x[e]));
  // words for the whole warp: none when every |x| <= 2^23, else the fewest
  // holding every entry's two's complement
  const int bits = __reduce_max_sync(0xffffffffu, (unsigned)bitlen64(m));
  const int nw = (bits <= 23 || (bits == 24 && __all_sync(0xffffffffu, m <= (1ull << 23)))) ? 0
                 : bits + 1 <= 32 ? 1 : 2;
  if (!valid) return;
  uint32_t wd[VEC][2];
  bool neg[VEC];
  float xf[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    neg[e] = (long long)cur.x[e] < 0;
    xf[e] = (float)(int)(long long)cur.x[e];
    wd[e][0] = (uint32_t)cur.x[e];
    wd[e][1] = (uint32_t)(cur.x[e] >> 32);
  }
  emit_int_residues<VEC, 2>(wd, neg, xf, nw, p1, rec, ws, s.Y + row * s.ldy + col0, s.plane, p0);
}

template <int VEC>
__global__ void __launch_bounds__(256) split_i64_kernel(SplitSide sa, SplitSide sb, DevPlan* plan, int P,
                                                        const uint32_t* hint) {
  __shared__ PrimeRec rec[kNumPrimes];
  __shared__ int ws[kNumPrimes][kMaxWords + 1];
  load_prime_recs(rec, ws);
  __syncthreads();
  wait_for_predecessor();
  const int planes = i64_planes_written(hint, P);
  const int lane = threadIdx.x & 31;
  const long long total = sa.items + sb.items;
  const long long stride = (long long)gridDim.x * blockDim.x;
  unsigned long long max_a = 0, max_b = 0;
  // grid-stride over warp-aligned items; the next item's words are loaded
  // while the current one is reduced, so reads, arithmetic and residue
  // stores overlap
  long long base = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31);
  I64Item<VEC> next = load_i64_item<VEC>(sa, sb, base + lane, total);
  for (; base < total; base += stride) {
    const I64Item<VEC> cur = next;
    if (base + stride < total) next = load_i64_item<VEC>(sa, sb, base + stride + lane, total);
    unsigned long long m;
    bool isA;
    emit_i64_item<VEC>(sa, sb, cur, base + lane, total, 0, planes, rec, ws, m, isA);
    if (isA) max_a = max(max_a, m);
    else max_b = max(max_b, m);
  }
  max_a = block_max_u64(max_a);
  max_b = block_max_u64(max_b);
  if (threadIdx.x == 0) {
    if (max_a) atomicMax(&plan->maxmag_a, max_a);
    if (max_b) atomicMax(&plan->maxmag_b, max_b);
  }
  allow_dependents();
}

// After a split that wrote fewer than pmax planes: derives the call's prime
// count from the split's reductions, as the GEMM will (fewest primes with
// product > 2^(T+1), T = bits(max|A|) + bits(max|B|) + ceil(log2 K), within
// the int64 range), and writes the planes from the split's count up to it.
// Returns at once when the split's planes suffice, or when the range check
// fails (the GEMM records the error).
template <int VEC>
__global__ void __launch_bounds__(256) split_i64_fixup_kernel(SplitSide sa, SplitSide sb, DevPlan* plan, int pmax,
                                                              const uint32_t* hint, long long K, int ceil_log2_k) {
  __shared__ PrimeRec rec[kNumPrimes];
  __shared__ int ws[kNumPrimes][kMaxWords + 1];
  wait_for_predecessor();
  if (plan->status) return;
  const int planes = i64_planes_written(hint, pmax);
  const unsigned long long ma = __ldcg(&plan->maxmag_a), mb = __ldcg(&plan->maxmag_b);
  const int T = bitlen64(ma) + bitlen64(mb) + ceil_log2_k;
  const unsigned long long ab = ma * mb;
  if (__umul64hi(ma, mb) != 0 || __umul64hi(ab, (unsigned long long)K) != 0 ||
      ab * (unsigned long long)K > 0x7FFFFFFFFFFFFFFFull)
    return;
  const int P = min(primes_for_bound(T), pmax);
  if (P <= planes) {  // the usual case: every block leaves at once (the decision is the same in all)
    allow_dependents();
    return;
  }
  load_prime_recs(rec, ws);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long total = sa.items + sb.items;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < total; base += stride) {
    const I64Item<VEC> cur = load_i64_item<VEC>(sa, sb, base + lane, total);
    unsigned long long m;
    bool isA;
    emit_i64_item<VEC>(sa, sb, cur, base + lane, total, planes, P, rec, ws, m, isA);
  }
  allow_dependents();
}

// |x| * 2^f for a floating-point x, from its bit pattern, as t * 2^sh: at a
// lossless point t is the significand and sh >= 0 (lost = false); at a
// coarsened point t = floor(|x| 2^f), sh = 0, and lost tells whether any bit
// was dropped.
template <typename Bits>
__device__ __forceinline__ void scaled_magnitude(Bits v, int f, bool& neg, unsigned long long& t, bool& lost,
                                                 int& sh) {
  using F = FloatFormat<Bits>;
  const int be = (int)((v >> F::kFracBits) & F::kExpMask);
  neg = (v & F::kSign) != 0;
  const unsigned long long hidden = 1ull << F::kFracBits;
  const unsigned long long m = ((unsigned long long)v & (hidden - 1ull)) | (be ? hidden : 0ull);
  sh = (be > 1 ? be : 1) - F::kLsbBias + f;  // |x| * 2^f = m * 2^sh
  if (m == 0 || sh >= 0) {
    if (m == 0) sh = 0;
    t = m;
    lost = false;
  } else {
    const int r = -sh;
    t = r >= 64 ? 0ull : m >> r;
    lost = r >= 64 ? true : (m & ((1ull << r) - 1ull)) != 0ull;
    sh = 0;
  }
}

// Byte weights of 2^(8k + s) mod q (ShiftWeights), uploaded with the tables.
__device__ uint2 g_wsh[kNumPrimes][kPow2Span];

// Dynamic shared memory of the floating-point splits: the shifted byte
// weights of P primes and `cols` shifts, [P][cols], when they fit in
// kWshEntries (a plan's usual size: tens of primes, tens of shifts);
// larger plans read the global table through L1 instead.  The plan is only
// known on the device, so the launch reserves the fixed kWshBytes.
constexpr int kWshEntries = 2048;
constexpr size_t kWshBytes = sizeof(uint2) * kWshEntries;

// Stages the table for P primes and `cols` shifts in shared memory if it
// fits; false if the block must read the global table.
__device__ __forceinline__ bool stage_wsh(uint2* wsh, int P, int cols) {
  if (P * cols > kWshEntries) return false;
  for (int i = threadIdx.x; i < P * cols; i += blockDim.x) {
    const int p = i / cols, c = i - p * cols;
    wsh[i] = g_wsh[p][c];
  }
  return true;
}

// The weights of prime p and shift sh: staged ([P][cols]) or global.
template <bool STAGED>
__device__ __forceinline__ uint2 wsh_get(const uint2* wsh, int cols, int p, int sh) {
  if constexpr (STAGED) return wsh[p * cols + sh];
  else return __ldg(&g_wsh[p][sh]);
}

// Balanced residue of t * 2^s from the bytes of t and the shifted byte weights
// w of s: one dot product per word, one reduction (|acc| <= 8 * 255 * 125 < 2^21).
template <int NWF>
__device__ __forceinline__ float shifted_residue(unsigned long long t, uint2 w, float q, float iq) {
  int acc = dp4a_us((uint32_t)t, (int)w.x, 0);
  if constexpr (NWF == 2) acc = dp4a_us((uint32_t)(t >> 32), (int)w.y, acc);
  return bal_mod_small(int_to_float_exact(acc), q, iq);
}

// Shifts a floating-point split can meet: sh < max(bits_a, bits_b) <= 255.
__device__ __forceinline__ int pow2_cols(const DevPlan* plan) {
  const int b = max(plan->bits_a, plan->bits_b);
  return b < 1 ? 1 : (b > kPow2Span ? kPow2Span : b);
}

// The split's main loop (weights staged in shared memory or read from the
// global table).
template <typename Bits, int VEC, bool STAGED>
__device__ __forceinline__ void split_float_loop(const SplitSide& sa, const SplitSide& sb, int P, int fa, int fb,
                                                 const PrimeRec* rec, const uint2* wsh, int cols) {
  using F = FloatFormat<Bits>;
  constexpr int NWF = F::kFracBits + 2 > 32 ? 2 : 1;  // words of t (the floored magnitude may gain a bit)
  constexpr int PER = 16 / sizeof(Bits);
  const long long total = sa.items + sb.items;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const bool isA = it < sa.items;
    const SplitSide& s = isA ? sa : sb;
    const int f = isA ? fa : fb;
    const long long item = isA ? it : it - sa.items;
    const long long per_row = s.ldy / VEC;
    const long long row = div_row(item, s.rd);
    const long long col0 = (item - row * per_row) * VEC;
    const Bits* X = static_cast<const Bits*>(s.X) + row * s.C + col0;
    Bits xv[VEC];
    if (col0 + VEC <= s.C && ((reinterpret_cast<uintptr_t>(X) & 15u) == 0)) {
#pragma unroll
      for (int t = 0; t < VEC / PER; ++t) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(X) + t);
        memcpy(xv + PER * t, &v, 16);
      }
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) xv[e] = col0 + e < s.C ? __ldg(X + e) : (Bits)0;
    }
    unsigned long long tv[VEC];
    int shv[VEC];
    bool negv[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      bool lost;
      scaled_magnitude<Bits>(xv[e], f, negv[e], tv[e], lost, shv[e]);
      if (negv[e] && lost) ++tv[e];  // floor of a negative value rounds away from zero
    }
    __half* y = s.Y + row * s.ldy + col0;
    for (int p = 0; p < P; ++p) {
      const PrimeRec& R = rec[p];
      const float q = R.q, iq = R.iq;
      float r[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float rr = shifted_residue<NWF>(tv[e], wsh_get<STAGED>(wsh, cols, p, shv[e]), q, iq);
        r[e] = negv[e] ? -rr : rr;
      }
      store_residues<VEC>(r, y + (long long)p * s.plane);
    }
  }
}

// Floating-point operands.  No floating-point instruction reads x.
template <typename Bits, int VEC>
__global__ void __launch_bounds__(256) split_float_kernel(SplitSide sa, SplitSide sb, const DevPlan* plan) {
  __shared__ PrimeRec rec[kNumPrimes];
  extern __shared__ uint2 wsh[];
  load_prime_recs(rec, nullptr);
  wait_for_predecessor();
  if (plan->status) return;
  const int P = plan->P;
  const int fa = plan->f_a, fb = plan->f_b;
  const int cols = pow2_cols(plan);
  const bool staged = stage_wsh(wsh, P, cols);
  __syncthreads();
  if (staged)
    split_float_loop<Bits, VEC, true>(sa, sb, P, fa, fb, rec, wsh, cols);
  else
    split_float_loop<Bits, VEC, false>(sa, sb, P, fa, fb, rec, wsh, cols);
  allow_dependents();
}

// Interval operands ("enclosure-gemm", Method: Rump's midpoint-radius bound,
// its three products formed exactly): mid(C) = Am Bm and
// rad(C) = |Am| Br + Ar (|Bm| + Br).  The split writes three residue planes per
// prime for each operand, A -> (Am, |Am|, Ar) and B -> (Bm, Br, |Bm| + Br), so
// the per-prime GEMM over the three planes forms the three products in one
// launch.  At a coarsened point midpoints are floored (their error is bounded
// in the epilogue) and every magnitude in the radius is rounded up, so the
// radius products stay upper bounds.  The residue of |Am| comes from that of
// floor(Am): ceil(|x| 2^f) is -floor(x 2^f) for x < 0 and floor(x 2^f) + lost
// otherwise.
struct IvSide {
  const void* Xm;   // midpoints [R][C]
  const void* Xr;   // radii [R][C]
  __half* Y;        // [pmax][3][R][ldy]
  long long R, C, ldy, sub, plane;  // sub = R * ldy (plane to plane), plane = 3 * sub (prime to prime)
  long long items;  // R * ldy / VEC
  RowDiv rd;        // division by the items per row, ldy / VEC
};

template <typename Bits, int VEC, bool STAGED>
__device__ __forceinline__ void split_interval_loop(const IvSide& sa, const IvSide& sb, int P, int fa, int fb,
                                                    const PrimeRec* rec, const uint2* wsh, int cols) {
  using F = FloatFormat<Bits>;
  constexpr int NWF = F::kFracBits + 2 > 32 ? 2 : 1;
  constexpr int PER = 16 / sizeof(Bits);
  static_assert((VEC * sizeof(Bits)) % 16 == 0, "whole 16-byte loads");
  const long long total = sa.items + sb.items;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const bool isA = it < sa.items;
    const IvSide& s = isA ? sa : sb;
    const int f = isA ? fa : fb;
    const long long item = isA ? it : it - sa.items;
    const long long per_row = s.ldy / VEC;
    const long long row = div_row(item, s.rd);
    const long long col0 = (item - row * per_row) * VEC;
    Bits xm[VEC], xr[VEC];
    {
      const Bits* Xm = static_cast<const Bits*>(s.Xm) + row * s.C + col0;
      const Bits* Xr = static_cast<const Bits*>(s.Xr) + row * s.C + col0;
      if (col0 + VEC <= s.C && (((reinterpret_cast<uintptr_t>(Xm) | reinterpret_cast<uintptr_t>(Xr)) & 15u) == 0)) {
#pragma unroll
        for (int t = 0; t < VEC / PER; ++t) {
          const uint4 a = __ldg(reinterpret_cast<const uint4*>(Xm) + t);
          const uint4 b = __ldg(reinterpret_cast<const uint4*>(Xr) + t);
          memcpy(xm + PER * t, &a, 16);
          memcpy(xr + PER * t, &b, 16);
        }
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          xm[e] = col0 + e < s.C ? __ldg(Xm + e) : (Bits)0;
          xr[e] = col0 + e < s.C ? __ldg(Xr + e) : (Bits)0;
        }
      }
    }
    unsigned long long tm[VEC], tr[VEC];
    int shm[VEC], shr[VEC];
    bool negm[VEC], lostm[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      bool neg, lost;
      scaled_magnitude<Bits>(xm[e], f, negm[e], tm[e], lostm[e], shm[e]);
      if (negm[e] && lostm[e]) ++tm[e];  // |floor(x 2^f)|
      scaled_magnitude<Bits>(xr[e], f, neg, tr[e], lost, shr[e]);  // radii are >= 0 (the planner checked)
      if (lost) ++tr[e];                                            // ceil(r 2^f)
    }
    __half* y = s.Y + row * s.ldy + col0;
    // A writes (Am, |Am|, Ar), B writes (Bm, Br, |Bm| + Br); the side is
    // uniform over an item, so each side has its own loop
    auto planes = [&](auto side_a) {
      constexpr bool IS_A = decltype(side_a)::value;
      for (int p = 0; p < P; ++p) {
        const PrimeRec& R = rec[p];
        const float q = R.q, iq = R.iq;
        float r0[VEC], r1[VEC], r2[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float am = shifted_residue<NWF>(tm[e], wsh_get<STAGED>(wsh, cols, p, shm[e]), q, iq);
          const float rr = shifted_residue<NWF>(tr[e], wsh_get<STAGED>(wsh, cols, p, shr[e]), q, iq);
          const float rabs = negm[e] ? am : bal_mod_small(am + (lostm[e] ? 1.0f : 0.0f), q, iq);  // ceil |x| 2^f
          r0[e] = negm[e] ? -am : am;  // floor(x 2^f)
          if constexpr (IS_A) {
            r1[e] = rabs;
            r2[e] = rr;
          } else {
            r1[e] = rr;
            r2[e] = bal_mod_small(rabs + rr, q, iq);
          }
        }
        __half* yp = y + (long long)p * s.plane;
        store_residues<VEC>(r0, yp);
        store_residues<VEC>(r1, yp + s.sub);
        store_residues<VEC>(r2, yp + 2 * s.sub);
      }
    };
    if (isA)
      planes(std::true_type{});
    else
      planes(std::false_type{});
  }
}

template <typename Bits, int VEC>
__global__ void __launch_bounds__(256) split_interval_kernel(IvSide sa, IvSide sb, const DevPlan* plan) {
  __shared__ PrimeRec rec[kNumPrimes];
  extern __shared__ uint2 wsh[];
  load_prime_recs(rec, nullptr);
  wait_for_predecessor();
  if (plan->status) return;
  const int P = plan->P;
  const int fa = plan->f_a, fb = plan->f_b;
  const int cols = pow2_cols(plan);
  const bool staged = stage_wsh(wsh, P, cols);
  __syncthreads();
  if (staged)
    split_interval_loop<Bits, VEC, true>(sa, sb, P, fa, fb, rec, wsh, cols);
  else
    split_interval_loop<Bits, VEC, false>(sa, sb, P, fa, fb, rec, wsh, cols);
  allow_dependents();
}

// ---------------------------------------------------------------------------
// Garner kernels ("exact-solve" and "enclosure-gemm", Method: balanced-Garner
// mixed-radix digits); the reconstruction itself is garner_reconstruct in
// rg_garner.cuh.
// ---------------------------------------------------------------------------

__device__ CrtTables g_crt;  // round-to-nearest CRT tables of every prime count
__constant__ IdemTables c_idem;  // idempotent-sum CRT tables, prime counts 1..kIdemMaxP

// x[e] = the int64 results of four adjacent entries from their residues r_i
// in [0, q_i) (one 32-bit word per prime, `plane` bytes apart), for exactly PP
// primes, by the idempotent sum S = sum_i r_i E_i and the rounded quotient
// k = round(S / P) (tables in IdemTables); S and k P are formed modulo 2^64,
// which holds the result x = S - k P.  The quotient is estimated as
// sum_i r_i f_i with f_i = round(2^20 E_i / P), within PP * 250 * 2^-21 <
// 0.0015 of S / P (and below 2^32 - 2^19).  S / P lies within |x| / P of the
// true quotient, and |x| <= (P - 1) / 2, so the estimate rounds to the true
// quotient or to a neighbour:
//  - PP >= 9: P > 2^70 and |x| < 2^63, so |x| / P < 2^-7 and it is the true one;
//  - PP <= 8: P < 2^63, so the three candidates are told apart exactly: the
//    result is the one in [-(P - 1) / 2, (P - 1) / 2] (a wrong one lies at
//    least P / 2 + 1/2 from zero, also after wrapping modulo 2^64).
// Four integer multiply-adds per prime and entry, no modular reduction.
template <int PP, int G>
__device__ __forceinline__ void idem_reconstruct(const uint8_t* __restrict__ rc, long long plane,
                                                 unsigned long long (&x)[G]) {
  static_assert(G == 4 || G == 8, "four or eight adjacent entries");
  constexpr int NW = G / 4;  // residue words per plane
  uint32_t rw[PP][NW];
#pragma unroll
  for (int i = 0; i < PP; ++i) {
    if constexpr (NW == 2) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(rc + (long long)i * plane));
      rw[i][0] = w.x;
      rw[i][1] = w.y;
    } else {
      rw[i][0] = __ldg(reinterpret_cast<const uint32_t*>(rc + (long long)i * plane));
    }
  }
  unsigned long long lo[G];
  uint32_t hi[G], kq[G];
#pragma unroll
  for (int e = 0; e < G; ++e) {
    lo[e] = 0ull;
    hi[e] = kq[e] = 0u;
  }
#pragma unroll
  for (int i = 0; i < PP; ++i) {
    const uint32_t elo = c_idem.elo[PP][i], ehi = c_idem.ehi[PP][i], f = c_idem.f[PP][i];
#pragma unroll
    for (int e = 0; e < G; ++e) {
      const uint32_t r = __byte_perm(rw[i][e / 4], 0u, 0x4440u + (uint32_t)(e % 4));  // byte e, zero-extended
      lo[e] += (unsigned long long)r * elo;                                           // < 12 * 250 * 2^32 < 2^44
      hi[e] += r * ehi;                                                               // modulo 2^32
      kq[e] += r * f;                                                                 // < 12 * 250 * 2^20
    }
  }
  const unsigned long long P64 = ((unsigned long long)c_idem.phi[PP] << 32) | c_idem.plo[PP];
#pragma unroll
  for (int e = 0; e < G; ++e) {
    const uint32_t k = (kq[e] + (1u << (kIdemFracBits - 1))) >> kIdemFracBits;
    unsigned long long v = lo[e] + ((unsigned long long)hi[e] << 32) - (unsigned long long)k * P64;
    if constexpr (PP <= 8) {
      const unsigned long long h = P64 >> 1;  // (P - 1) / 2, P odd
      if (v + h > 2 * h) {                    // v outside [-h, h]: the quotient was off by one
        const unsigned long long up = v - P64;  // quotient + 1
        v = (up + h <= 2 * h) ? up : v + P64;
      }
    }
    x[e] = v;
  }
}

// Int64 results (one limb) of up to kIdemMaxP primes by idempotent sums
// (idem_reconstruct), G adjacent entries per thread (G bytes of every
// residue plane in one load); the prime count is dispatched to a
// compile-time constant, so every table entry is an immediate constant
// operand.  Exact for every int64 result the plan (or the caller's prime
// count) allows; rg_get_plan reports crt_rn = 2.
template <int G>
__global__ void __launch_bounds__(128) crt_idem_kernel(const uint8_t* __restrict__ RC, long long ldc, long long plane,
                                                       long long M, long long N, RowDiv rd, DevPlan* plan,
                                                       int64_t* __restrict__ C) {
  wait_for_predecessor();
  if (plan->status) return;
  const int P = plan->P;
  if (P < 1 || P > kIdemMaxP) {  // the launch is chosen for pmax <= kIdemMaxP
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(&plan->status, RG_ERR_RANGE);
    return;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) plan->crt_rn = 2;
  const long long per_row = (N + G - 1) / G;
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= M * per_row) return;
  const long long m = div_row(item, rd);  // item / per_row
  const long long n0 = (item - m * per_row) * G;
  const uint8_t* rc = RC + m * ldc + n0;  // G bytes within the row's ldc (a multiple of 16)
  unsigned long long v[G];
  switch (P) {
    case 1: idem_reconstruct<1, G>(rc, plane, v); break;
    case 2: idem_reconstruct<2, G>(rc, plane, v); break;
    case 3: idem_reconstruct<3, G>(rc, plane, v); break;
    case 4: idem_reconstruct<4, G>(rc, plane, v); break;
    case 5: idem_reconstruct<5, G>(rc, plane, v); break;
    case 6: idem_reconstruct<6, G>(rc, plane, v); break;
    case 7: idem_reconstruct<7, G>(rc, plane, v); break;
    case 8: idem_reconstruct<8, G>(rc, plane, v); break;
    case 9: idem_reconstruct<9, G>(rc, plane, v); break;
    case 10: idem_reconstruct<10, G>(rc, plane, v); break;
    case 11: idem_reconstruct<11, G>(rc, plane, v); break;
    default: idem_reconstruct<12, G>(rc, plane, v); break;
  }
  int64_t* out = C + m * N + n0;
  if (n0 + G <= N && ((reinterpret_cast<uintptr_t>(out) & 15u) == 0)) {
#pragma unroll
    for (int t = 0; t < G / 2; ++t) *reinterpret_cast<ulonglong2*>(out + 2 * t) = make_ulonglong2(v[2 * t], v[2 * t + 1]);
  } else {
#pragma unroll
    for (int e = 0; e < G; ++e)
      if (n0 + e < N) out[e] = (int64_t)v[e];
  }
}
static_assert(kIdemMaxP == 12, "crt_idem_kernel dispatches prime counts 1..12");
// Entries per thread of the int64 reconstruction (ldc is a multiple of 16, so
// every group's bytes lie within its row's padded planes).
constexpr int kIdemGroup = 8;

__device__ __forceinline__ CrtView crt_view(int P) { return CrtView{g_crt.M[P], g_crt.Pw[P], g_crt.Cw[P], g_crt.y[P]}; }

// MAXP: a compile-time bound on the prime count (the workspace's pmax).
// rn_free: reconstruct by round-to-nearest CRT whenever the planned primes
// already exceed 4 |result| (the bound's prime count for one more bit is no
// larger than P), at no extra prime; otherwise as the plan says.
template <int LC, int MAXP>
__global__ void __launch_bounds__(128) garner_int_kernel(const uint8_t* __restrict__ RC, long long ldc,
                                                         long long plane, long long M, long long N, RowDiv rd,
                                                         DevPlan* plan, int64_t* __restrict__ C, int rn_free) {
  constexpr int W = 2 * LC, GE = GarnerGE<W>::value;
  wait_for_predecessor();
  if (plan->status) return;
  const int P = plan->P;
  if (P > MAXP) {  // the planner keeps P within the workspace's planes
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(&plan->status, RG_ERR_RANGE);
    return;
  }
  const bool plan_rn = plan->crt_rn != 0;
  bool rn = plan_rn;
  if (!rn && rn_free) {
    const int prn = primes_for_bound(plan->bound_bits + 1);
    rn = prn != 0 && prn <= P;
  }
  // recorded for rg_get_plan; every block takes the same decision from the
  // same plan fields, so a block that reads the flag already set agrees
  if (rn && !plan_rn && blockIdx.x == 0 && threadIdx.x == 0) plan->crt_rn = 1;
  const CrtView crt = crt_view(P);
  const long long per_row = (N + GE - 1) / GE;
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= M * per_row) return;
  const long long m = div_row(item, rd);  // item / per_row
  const long long n0 = (item - m * per_row) * GE;
  uint32_t x[GE][W];
  if (rn)
    crt_rn_reconstruct<W, GE, MainTab>(RC + m * ldc + n0, plane, P, crt, x);
  else
    garner_reconstruct<W, GE, MainTab, MAXP>(RC + m * ldc + n0, plane, P, x);
  int64_t* out = C + (m * N + n0) * LC;
  if (n0 + GE <= N && ((reinterpret_cast<uintptr_t>(out) & 15u) == 0)) {
    // GE * LC consecutive int64: 16-byte stores
#pragma unroll
    for (int t = 0; t < GE * LC / 2; ++t) {
      const int e0 = (2 * t) / LC, l0 = (2 * t) % LC, e1 = (2 * t + 1) / LC, l1 = (2 * t + 1) % LC;
      *reinterpret_cast<uint4*>(out + 2 * t) =
          make_uint4(x[e0][2 * l0], x[e0][2 * l0 + 1], x[e1][2 * l1], x[e1][2 * l1 + 1]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < GE; ++e) {
      if (n0 + e >= N) break;
#pragma unroll
      for (int l = 0; l < LC; ++l)
        out[e * LC + l] = (int64_t)(((unsigned long long)x[e][2 * l + 1] << 32) | x[e][2 * l]);
    }
  }
}

// Outward bit-pattern epilogue ("enclosure-gemm", Method): S (W words, two's
// complement) times 2^-Q -> (lo, hi) IEEE bit patterns of the format of Bits
// (binary64 or binary32).
constexpr int kEncW = 11;  // 352 bits hold |S| < 2^333 with its sign

template <typename Bits>
__device__ __forceinline__ void outward_bits(const uint32_t (&x)[kEncW], int Q, Bits& lo, Bits& hi) {
  using F = FloatFormat<Bits>;
  constexpr Bits kMaxFinite = F::kMaxFinite, kInf = F::kInf, kSign = F::kSign;
  constexpr int kFrac = F::kFracBits;
  const bool neg = (x[kEncW - 1] >> 31) != 0;
  uint32_t mag[kEncW];
  unsigned long long carry = neg ? 1ull : 0ull;
#pragma unroll
  for (int k = 0; k < kEncW; ++k) {
    const unsigned long long t = (unsigned long long)(neg ? ~x[k] : x[k]) + carry;
    mag[k] = (uint32_t)t;
    carry = t >> 32;
  }
  int L = -1;  // index of the leading bit
#pragma unroll
  for (int k = kEncW - 1; k >= 0; --k)
    if (L < 0 && mag[k]) L = 32 * k + 31 - __clz(mag[k]);
  if (L < 0) {  // S == 0
    lo = hi = 0;
    return;
  }
  const int E = L - Q;  // floor(log2 |S 2^-Q|)
  if (E > F::kEmax) {
    lo = neg ? (kSign | kInf) : kMaxFinite;
    hi = neg ? (kSign | kMaxFinite) : kInf;
    return;
  }
  const int u = E - kFrac > F::kUlpMin ? E - kFrac : F::kUlpMin;  // exponent of one ulp at this magnitude
  const int sh = u + Q;                                            // bit of |S| holding that ulp
  unsigned long long T = 0ull;
  bool rem = false;
  if (sh <= 0) {
    // exact: |S| < 2^(kFrac+1) after the shift, since L - sh <= kFrac
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int b = 32 * k - sh;  // destination bit of word k
      if (b < 64 && k < kEncW) T |= (unsigned long long)mag[k] << b;
    }
  } else {
    // T = bits [sh, sh + kFrac + 1) of |S|; rem = any bit below sh
#pragma unroll
    for (int k = 0; k < kEncW; ++k) {
      const int lo_bit = 32 * k, hi_bit = 32 * k + 32;
      const unsigned long long w = mag[k];
      if (hi_bit <= sh) {
        rem |= w != 0;
      } else if (lo_bit < sh) {
        const int cut = sh - lo_bit;
        rem |= (w & ((1ull << cut) - 1ull)) != 0;
        T |= w >> cut;
      } else if (lo_bit - sh < 64) {
        T |= w << (lo_bit - sh);
      }
    }
    T &= (1ull << (kFrac + 1)) - 1ull;
  }
  // the hidden bit of T carries into the exponent field: biased exponent E + bias
  const Bits enc = (Bits)((E >= F::kEminNormal ? (unsigned long long)(E - F::kEminNormal) << kFrac : 0ull) + T);
  if (!rem) {
    lo = hi = (neg ? kSign : (Bits)0) | enc;
  } else if (!neg) {
    lo = enc;
    hi = (Bits)(enc + 1);
  } else {
    lo = kSign | (Bits)(enc + 1);
    hi = kSign | enc;
  }
}

// x (kEncW words, two's complement) += sign * (v << shift), v < 2^31, shift >= 0.
__device__ __forceinline__ void add_shifted(uint32_t (&x)[kEncW], long long v, int shift, int sign) {
  const int w0 = shift >> 5, b = shift & 31;
  const unsigned long long part = (unsigned long long)v << b;  // < 2^63: two words
  long long carry = 0;
#pragma unroll
  for (int k = 0; k < kEncW; ++k) {
    long long add = 0;
    if (k == w0) add = (long long)(part & 0xFFFFFFFFull);
    if (k == w0 + 1) add = (long long)(part >> 32);
    const long long t = (long long)x[k] + sign * add + carry;
    x[k] = (uint32_t)t;
    carry = t >> 32;
  }
}

template <typename Bits>
__global__ void __launch_bounds__(128) garner_enclose_kernel(const uint8_t* __restrict__ RC, long long ldc,
                                                             long long plane, long long M, long long N,
                                                             long long K, RowDiv rd, DevPlan* plan,
                                                             Bits* __restrict__ lo, Bits* __restrict__ hi) {
  constexpr int GE = GarnerGE<kEncW>::value;
  static_assert(GE == 2, "the bound stores below write GE entries as one vector");
  wait_for_predecessor();
  if (plan->status) return;
  const int P = plan->P;
  const int Q = plan->f_a + plan->f_b;
  const bool rn = plan->crt_rn != 0;
  const CrtView crt = crt_view(P);
  const long long per_row = (N + GE - 1) / GE;
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= M * per_row) return;
  const long long m = div_row(item, rd);  // item / per_row
  const long long n0 = (item - m * per_row) * GE;
  uint32_t x[GE][kEncW];
  if (rn)
    crt_rn_reconstruct<kEncW, GE, MainTab>(RC + m * ldc + n0, plane, P, crt, x);
  else
    garner_reconstruct<kEncW, GE, MainTab>(RC + m * ldc + n0, plane, P, x);
  Bits l[GE], h[GE];
  if (plan->lossless) {
#pragma unroll
    for (int e = 0; e < GE; ++e) outward_bits(x[e], Q, l[e], h[e]);
  } else {
    // Coarsened operands A' = floor(A 2^f_a), B' = floor(B 2^f_b) leave
    // remainders in [0, 1) per entry; with |A'| <= 2^bits_a, |B'| <= 2^bits_b
    // the exact (A 2^f_a)(B 2^f_b) lies in S + (-K(2^a + 2^b), K(2^a + 2^b) + K)
    // ("enclosure-gemm", Method: the termwise bound added back outward).
    const int ba = plan->bits_a, bb = plan->bits_b;
#pragma unroll
    for (int e = 0; e < GE; ++e) {
      uint32_t xl[kEncW], xh[kEncW];
#pragma unroll
      for (int k = 0; k < kEncW; ++k) xl[k] = xh[k] = x[e][k];
      add_shifted(xl, K, ba, -1);
      add_shifted(xl, K, bb, -1);
      add_shifted(xh, K, ba, 1);
      add_shifted(xh, K, bb, 1);
      add_shifted(xh, K, 0, 1);
      Bits unused;
      outward_bits(xl, Q, l[e], unused);
      outward_bits(xh, Q, unused, h[e]);
    }
  }
  Bits* plo = lo + m * N + n0;
  Bits* phi = hi + m * N + n0;
  constexpr unsigned kRowBytes = GE * sizeof(Bits);  // 16 (binary64) or 8 (binary32)
  if (n0 + GE <= N && ((reinterpret_cast<uintptr_t>(plo) & (kRowBytes - 1)) == 0)) {
    if constexpr (kRowBytes == 16) {
      uint4 vl, vh;
      memcpy(&vl, l, 16);
      memcpy(&vh, h, 16);
      *reinterpret_cast<uint4*>(plo) = vl;
      *reinterpret_cast<uint4*>(phi) = vh;
    } else {
      uint2 vl, vh;
      memcpy(&vl, l, 8);
      memcpy(&vh, h, 8);
      *reinterpret_cast<uint2*>(plo) = vl;
      *reinterpret_cast<uint2*>(phi) = vh;
    }
  } else {
#pragma unroll
    for (int e = 0; e < GE; ++e) {
      if (n0 + e >= N) break;
      plo[e] = l[e];
      phi[e] = h[e];
    }
  }
}

// x += sign * y, kEncW-word two's complement (sign = +1 or -1).
__device__ __forceinline__ void add_words(uint32_t (&x)[kEncW], const uint32_t (&y)[kEncW], int sign) {
  unsigned long long carry = sign < 0 ? 1ull : 0ull;  // x - y = x + ~y + 1
#pragma unroll
  for (int k = 0; k < kEncW; ++k) {
    const unsigned long long t = (unsigned long long)x[k] + (sign < 0 ? ~y[k] : y[k]) + carry;
    x[k] = (uint32_t)t;
    carry = t >> 32;
  }
}

// Interval epilogue ("enclosure-gemm", Method: Rump's bound with the
// midpoint and radius as exact integers, rounded outward once): from the
// three product planes S1 = Am Bm, S2 = |Am| Br, S3 = Ar (|Bm| + Br) at rows
// `sub` bytes apart, lo = down(S1 - S2 - S3) and hi = up(S1 + S2 + S3), with
// the midpoint's flooring bound widened outward at a coarsened point.
template <typename Bits>
__global__ void __launch_bounds__(128) garner_interval_kernel(const uint8_t* __restrict__ RC, long long ldc,
                                                              long long plane, long long sub, long long M,
                                                              long long N, long long K, RowDiv rd, DevPlan* plan,
                                                              Bits* __restrict__ lo, Bits* __restrict__ hi) {
  constexpr int GE = 1;
  wait_for_predecessor();
  if (plan->status) return;
  const int P = plan->P;
  const int Q = plan->f_a + plan->f_b;
  const bool rn = plan->crt_rn != 0;
  const CrtView crt = crt_view(P);
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= M * N) return;
  const long long m = div_row(item, rd), n = item - m * N;  // item / N
  const uint8_t* base = RC + m * ldc + n;
  auto reconstruct = [&](const uint8_t* at, uint32_t (&v)[GE][kEncW]) {
    if (rn)
      crt_rn_reconstruct<kEncW, GE, MainTab>(at, plane, P, crt, v);
    else
      garner_reconstruct<kEncW, GE, MainTab>(at, plane, P, v);
  };
  uint32_t x[GE][kEncW], xl[kEncW], xh[kEncW];
  reconstruct(base, x);
#pragma unroll
  for (int k = 0; k < kEncW; ++k) xl[k] = xh[k] = x[0][k];
  reconstruct(base + sub, x);
  add_words(xl, x[0], -1);
  add_words(xh, x[0], 1);
  reconstruct(base + 2 * sub, x);
  add_words(xl, x[0], -1);
  add_words(xh, x[0], 1);
  if (!plan->lossless) {
    // floored midpoints: (A 2^f_a)(B 2^f_b) - S1 lies in (-K(2^a + 2^b), K(2^a + 2^b) + K)
    const int ba = plan->bits_a, bb = plan->bits_b;
    add_shifted(xl, K, ba, -1);
    add_shifted(xl, K, bb, -1);
    add_shifted(xh, K, ba, 1);
    add_shifted(xh, K, bb, 1);
    add_shifted(xh, K, 0, 1);
  }
  Bits l, h, unused;
  outward_bits(xl, Q, l, unused);
  outward_bits(xh, Q, unused, h);
  lo[m * N + n] = l;
  hi[m * N + n] = h;
}

std::atomic<int> g_sm_count[64];  // per device, 0 until read
// 0: balanced Garner; 1: round-to-nearest CRT for the wide outputs where the
// plan can keep P > 4 |x|, and for int64 where its primes already do
std::atomic<int> g_crt_mode{0};

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (!n) {  // threads that race here all store the same count
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
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
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(c_idem, &host_idem_tables(), sizeof(IdemTables));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_wsh, host_shift_weights().w, sizeof(ShiftWeights));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_crt, &host_crt_tables(), sizeof(CrtTables));
  if (e == cudaSuccess) {
    static SplitTables st;  // built from the host tables
    const Tables& t = host_tables();
    for (int p = 0; p < kNumPrimes; ++p) {
      for (int w = 0; w < kMaxWords; ++w) st.rec[p].w[w] = t.wbyte[p][w];
      st.rec[p].q = t.qf[p];
      st.rec[p].iq = t.invq[p];
      st.rec[p].pad[0] = st.rec[p].pad[1] = 0;
      for (int k = 0; k <= kMaxWords; ++k) st.ws[p][k] = t.wword[p][k];
    }
    e = cudaMemcpyToSymbol(g_split, &st, sizeof(SplitTables));
  }
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

static int planner_blocks(long long n) {
  long long b = (n + 256LL * 8 - 1) / (256LL * 8);
  // two blocks per SM and side: with four 16-byte loads in flight per thread
  // that covers HBM latency, and every block ends with atomics on the plan
  long long cap = 2LL * sm_count();
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

cudaError_t launch_plan(int op, const void* A, const void* A2, long long nA, int la, const void* B, const void* B2,
                        long long nB, int lb, int lc, long long K, int nprimes_fixed, int pcap, DevPlan* plan,
                        cudaStream_t s) {
  if (pcap < 1 || pcap > kNumPrimes) return cudaErrorInvalidValue;
  PlanArgs pa{op, K, nprimes_fixed, la, lb, lc, g_crt_mode.load() == 1 ? 1 : 0, pcap};
  if (nprimes_fixed) nA = nB = 0;  // only the finalisation is needed
  const int ba = planner_blocks(nA), bb = planner_blocks(nB);
  if (op == RG_OP_I64)
    return cudaErrorInvalidValue;  // int64 plans in its split and GEMM kernels, with no planner pass
  if (op == RG_OP_LIMBS)
    plan_limbs_kernel<<<ba + bb, 256, 0, s>>>(static_cast<const int64_t*>(A), nA, la,
                                              static_cast<const int64_t*>(B), nB, lb, ba, plan, pa);
  else if (op == RG_OP_ENCLOSE || op == RG_OP_INTERVAL) {
    using U = unsigned long long;
    plan_float_kernel<U><<<ba + bb, 256, 0, s>>>(static_cast<const U*>(A), static_cast<const U*>(A2), nA,
                                                 static_cast<const U*>(B), static_cast<const U*>(B2), nB, ba, plan, pa);
  } else {
    plan_float_kernel<uint32_t><<<ba + bb, 256, 0, s>>>(static_cast<const uint32_t*>(A), static_cast<const uint32_t*>(A2),
                                                        nA, static_cast<const uint32_t*>(B),
                                                        static_cast<const uint32_t*>(B2), nB, ba, plan, pa);
  }
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
  s.rd = make_rowdiv(ldy / vec);
  return s;
}

static unsigned split_grid(long long items, int blocks_per_sm = 8) {
  long long b = (items + 255) / 256;
  const long long cap = (long long)blocks_per_sm * sm_count();
  return (unsigned)(b < 1 ? 1 : (b > cap ? cap : b));
}

// Blocks per SM of the int64 split: few enough that each thread walks several
// items and its prefetch overlaps the reduction of the current one; at 2^21
// items and more, enough for full occupancy (GB300: 1024^3 43.0 us per call
// with 3 and 45.1 with 8; 4096^3 826 us with 3 and 819 with 8).
constexpr int kSplitI64BlocksPerSm = 3;
constexpr int kSplitI64BlocksPerSmLarge = 8;
constexpr long long kSplitI64LargeItems = 1LL << 21;

static IvSide make_iv_side(const void* Xm, const void* Xr, __half* Y, long long R, long long C, long long ldy,
                           int vec) {
  IvSide s;
  s.Xm = Xm;
  s.Xr = Xr;
  s.Y = Y;
  s.R = R;
  s.C = C;
  s.ldy = ldy;
  s.sub = R * ldy;
  s.plane = 3 * s.sub;
  s.items = R * (ldy / vec);
  s.rd = make_rowdiv(ldy / vec);
  return s;
}

// The floating-point splits' dynamic shared memory (kWshBytes) exceeds the
// default 48 KB limit; raised once per device.
static cudaError_t allow_wsh_smem() {
  static std::mutex mu;
  static bool done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  const int bytes = (int)kWshBytes;
  e = cudaFuncSetAttribute(split_interval_kernel<unsigned long long, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(split_interval_kernel<uint32_t, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(split_float_kernel<unsigned long long, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(split_float_kernel<uint32_t, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

cudaError_t launch_split(int op, const void* A, const void* A2, const void* B, const void* B2, int la, int lb,
                         long long batch, long long Mb, long long N, long long K, long long lda, long long ldb,
                         void* RA, void* RB, DevPlan* plan, int i64_planes, bool transb, cudaStream_t st,
                         const uint32_t* plane_hint) {
  __half* ra = static_cast<__half*>(RA);
  __half* rb = static_cast<__half*>(RB);
  // The products of a batch lie back to back, so each side is one matrix of
  // batch * rows rows.  B [K][N] -> RB [P][K][ldb]; a transposed B [N][K] ->
  // RB [P][N][ldb], laid out like A.
  const long long M = batch * Mb;
  const long long brows = batch * (transb ? N : K), bcols = transb ? K : N;
  if (op == RG_OP_INTERVAL || op == RG_OP_INTERVAL_F32 || op == RG_OP_ENCLOSE || op == RG_OP_ENCLOSE_F32) {
    cudaError_t e = allow_wsh_smem();
    if (e != cudaSuccess) return e;
  }
  if (op == RG_OP_INTERVAL || op == RG_OP_INTERVAL_F32) {
    constexpr int V = 4;
    const IvSide sa = make_iv_side(A, A2, ra, M, K, lda, V), sb = make_iv_side(B, B2, rb, brows, bcols, ldb, V);
    if (op == RG_OP_INTERVAL)
      return launch_dependent(split_interval_kernel<unsigned long long, V>, split_grid(sa.items + sb.items), 256,
                              kWshBytes, st, sa, sb, (const DevPlan*)plan);
    return launch_dependent(split_interval_kernel<uint32_t, V>, split_grid(sa.items + sb.items), 256, kWshBytes, st,
                            sa, sb, (const DevPlan*)plan);
  }
  if (op == RG_OP_ENCLOSE || op == RG_OP_ENCLOSE_F32) {
    constexpr int V = 8;
    const SplitSide sa = make_side(A, ra, M, K, lda, 1, V), sb = make_side(B, rb, brows, bcols, ldb, 1, V);
    if (op == RG_OP_ENCLOSE)
      return launch_dependent(split_float_kernel<unsigned long long, V>, split_grid(sa.items + sb.items), 256,
                              kWshBytes, st, sa, sb, (const DevPlan*)plan);
    return launch_dependent(split_float_kernel<uint32_t, V>, split_grid(sa.items + sb.items), 256, kWshBytes, st, sa, sb,
                            (const DevPlan*)plan);
  }
  const int L = la > lb ? la : lb;
  if (op == RG_OP_I64) {
    constexpr int V = 8;
    const SplitSide sa = make_side(A, ra, M, K, lda, 1, V);
    SplitSide sb = make_side(B, rb, brows, bcols, ldb, 1, V);
    if (!B) sb.items = 0;  // A alone: B's residues are already in RB
    const long long items = sa.items + sb.items;
    const unsigned grid =
        split_grid(items, items >= kSplitI64LargeItems ? kSplitI64BlocksPerSmLarge : kSplitI64BlocksPerSm);
    cudaError_t e = launch_dependent(split_i64_kernel<V>, grid, 256, 0, st, sa, sb, plan, i64_planes, plane_hint);
    if (e != cudaSuccess || !plane_hint) return e;
    int ck = 0;
    while ((1LL << ck) < K) ++ck;
    return launch_dependent(split_i64_fixup_kernel<V>, grid, 256, 0, st, sa, sb, plan, i64_planes,
                            (const uint32_t*)plane_hint, K, ck);
  }
  if (L <= 1) {
    constexpr int V = 8;
    const SplitSide sa = make_side(A, ra, M, K, lda, la, V), sb = make_side(B, rb, brows, bcols, ldb, lb, V);
    return launch_dependent(split_int_kernel<V, 1>, split_grid(sa.items + sb.items), 256, 0, st, sa, sb,
                            (const DevPlan*)plan);
  } else if (L <= 2) {
    constexpr int V = 8;
    const SplitSide sa = make_side(A, ra, M, K, lda, la, V), sb = make_side(B, rb, brows, bcols, ldb, lb, V);
    return launch_dependent(split_int_kernel<V, 2>, split_grid(sa.items + sb.items), 256, 0, st, sa, sb,
                            (const DevPlan*)plan);
  } else {
    constexpr int V = 4;
    const SplitSide sa = make_side(A, ra, M, K, lda, la, V), sb = make_side(B, rb, brows, bcols, ldb, lb, V);
    return launch_dependent(split_int_kernel<V, 4>, split_grid(sa.items + sb.items), 256, 0, st, sa, sb,
                            (const DevPlan*)plan);
  }
  return cudaGetLastError();
}

// Prime bound of the register-lean integer Garner kernels.
constexpr int kGarnerSmallP = 12;

cudaError_t launch_garner(int op, const void* RC, long long ldc, long long plane, long long sub, long long M,
                          long long N, long long K, int lc, int pmax, DevPlan* plan, void* out0, void* out1,
                          cudaStream_t st) {
  const uint8_t* rc = static_cast<const uint8_t*>(RC);
  auto blocks_for = [&](int ge) { return dim3((unsigned)((M * ((N + ge - 1) / ge) + 127) / 128)); };
  if (op == RG_OP_INTERVAL)
    return launch_dependent(garner_interval_kernel<unsigned long long>, blocks_for(1), 128, 0, st, rc, ldc, plane, sub,
                            M, N, K, make_rowdiv(N), plan, static_cast<unsigned long long*>(out0),
                            static_cast<unsigned long long*>(out1));
  if (op == RG_OP_INTERVAL_F32)
    return launch_dependent(garner_interval_kernel<uint32_t>, blocks_for(1), 128, 0, st, rc, ldc, plane, sub, M, N, K,
                            make_rowdiv(N), plan, static_cast<uint32_t*>(out0), static_cast<uint32_t*>(out1));
  const RowDiv rd_enc = make_rowdiv((N + GarnerGE<kEncW>::value - 1) / GarnerGE<kEncW>::value);
  if (op == RG_OP_ENCLOSE)
    return launch_dependent(garner_enclose_kernel<unsigned long long>, blocks_for(GarnerGE<kEncW>::value), 128, 0, st,
                            rc, ldc, plane, M, N, K, rd_enc, plan, static_cast<unsigned long long*>(out0),
                            static_cast<unsigned long long*>(out1));
  if (op == RG_OP_ENCLOSE_F32)
    return launch_dependent(garner_enclose_kernel<uint32_t>, blocks_for(GarnerGE<kEncW>::value), 128, 0, st, rc, ldc,
                            plane, M, N, K, rd_enc, plan, static_cast<uint32_t*>(out0), static_cast<uint32_t*>(out1));
  int64_t* C = static_cast<int64_t*>(out0);
  auto rowdiv_for = [&](int ge) { return make_rowdiv((N + ge - 1) / ge); };
  // the packed digits of at most kGarnerSmallP primes fit in 3 registers per
  // entry, against 14 for all 53
  const bool small = pmax <= kGarnerSmallP;
  const int mode = g_crt_mode.load();
  // mode 0: one-limb results of at most kIdemMaxP primes by idempotent sums
  if (mode == 0 && lc == 1 && pmax >= 1 && pmax <= kIdemMaxP)
    return launch_dependent(crt_idem_kernel<kIdemGroup>, blocks_for(kIdemGroup), 128, 0, st, rc, ldc, plane, M, N,
                            rowdiv_for(kIdemGroup), plan, C);
  // mode 1: int64 by round-to-nearest CRT on balanced digits when its primes allow it
  const int rn_free = op == RG_OP_I64 && mode == 1 ? 1 : 0;
  auto go = [&](auto k_small, auto k_all, int ge) {
    return launch_dependent(small ? k_small : k_all, blocks_for(ge), 128, 0, st, rc, ldc, plane, M, N, rowdiv_for(ge),
                            plan, C, rn_free);
  };
  switch (lc) {
    case 1: return go(garner_int_kernel<1, kGarnerSmallP>, garner_int_kernel<1, kNumPrimes>, GarnerGE<2>::value);
    case 2: return go(garner_int_kernel<2, kGarnerSmallP>, garner_int_kernel<2, kNumPrimes>, GarnerGE<4>::value);
    case 3: return go(garner_int_kernel<3, kGarnerSmallP>, garner_int_kernel<3, kNumPrimes>, GarnerGE<6>::value);
    case 4: return go(garner_int_kernel<4, kGarnerSmallP>, garner_int_kernel<4, kNumPrimes>, GarnerGE<8>::value);
    case 5: return go(garner_int_kernel<5, kGarnerSmallP>, garner_int_kernel<5, kNumPrimes>, GarnerGE<10>::value);
    case 6: return go(garner_int_kernel<6, kGarnerSmallP>, garner_int_kernel<6, kNumPrimes>, GarnerGE<12>::value);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rg

extern "C" int rg_set_crt_mode(int mode) {
  if (mode < 0 || mode > 2) return -1;
  return rg::g_crt_mode.exchange(mode);
}
