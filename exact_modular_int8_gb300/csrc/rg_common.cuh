// rg_common.cuh -- types, tables and device helpers shared by the library's
// translation units (never by the oracle).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/resgemm.h"

namespace rg {

constexpr int kNumPrimes = RG_NUM_PRIMES;  // odd primes 3..251, largest first
constexpr int kMaxWords = 8;               // 32-bit words of a 256-bit operand
constexpr int kPow2Span = 256;             // shifts s < 256 are tabulated
constexpr int kGarnerWords = 14;           // ceil(53 / 4) int8x4 words per Garner row
constexpr int kQWords = 11;                // 32-bit words of the mixed-radix weights Q_i
constexpr int kMaxLimbsOut = RG_MAX_LIMBS_OUT;

// Plan of one call, kept in the first bytes of the workspace.  The planner
// kernels fill the reduction fields with atomics (so the host zeroes the block
// first); the split kernel derives the rest identically in every block and
// block 0 writes it back for the later kernels.
struct DevPlan {
  int status;             // RG_OK or the first device-side error (atomicCAS from 0)
  int P;                  // primes used
  int bits_a, bits_b;     // bit length of max |entry| (scaled entries for fp64)
  int bound_bits;         // bits_a + bits_b + ceil(log2 K)
  int f_a, f_b;           // fp64 scale exponents
  int lossless;           // fp64: 1 if the scaling is exact
  int nword_a, nword_b;   // 32-bit words the split reads per integer entry (0: the entry is an exact fp32)
  unsigned blocks_done;   // planner blocks finished (the last one derives the plan)
  int splits;             // K slices the GEMM used (1: none)
  int crt_rn;             // 1: reconstruct by round-to-nearest CRT (P > 4 |x| guaranteed), 0: balanced Garner
  int pad0[3];
  // reductions written by the planner kernels
  unsigned long long maxmag_a, maxmag_b;  // int64 operands: max |x|
  int maxbits_a, maxbits_b;               // limb operands: max bit length of |x|
  int maxe_a, maxe_b;                     // fp64: max of max(biased exponent, 1) over nonzero entries
  int inv_mine_a, inv_mine_b;             // fp64: 4096 - min of that exponent (0 = no nonzero entry)
  int nonfinite;                          // floating point: an inf or nan entry was seen
  int neg_radius;                         // intervals: a radius entry below zero was seen
  int pad1[6];
  // diagnostics of a bounded wait that expired (which role, which wait)
  int timeout_where;
  int pad2[15];
};
static_assert(sizeof(DevPlan) <= 256, "plan block");

// A word of the workspace's plan block beyond the DevPlan that each call
// clears: the planner-free int64 path's GEMM records there the prime count
// it used (tagged), and the next call's split writes only that many residue
// planes when it is below the most an int64 product can need (a fix-up pass
// adds any planes the call then needs).
constexpr size_t kPlaneHintOffset = 256;
constexpr uint32_t kPlaneHintTag = 0x52470000u;

// Constant tables for the split and Garner kernels, computed on the host once.
struct Tables {
  int q[kNumPrimes];                          // q_0 = 251 > q_1 > ... > q_52 = 3
  float qf[kNumPrimes];                       // q as float
  float invq[kNumPrimes];                     // fl(1/q)
  // Residue split: byte j of a little-endian word string weighs 2^(8j) mod q
  // (balanced), packed four to an int32 (byte 4w + b in bits 8b..8b+7 of
  // wbyte[.][w]); a string of k words as a whole weighs 2^(32k) mod q.
  int wbyte[kNumPrimes][kMaxWords];
  int wword[kNumPrimes][kMaxWords + 1];
  int log2P[kNumPrimes + 1];                  // floor(log2(q_0 * ... * q_{n-1})), n = 0..53
  // Balanced Garner: v_i = bal( ginv[i] * r_i + sum_{j<i} gd[i][j] * v_j  mod q_i )
  // with ginv[i] = bal(Q_i^-1 mod q_i), gd[i][j] = bal(-(Q_j mod q_i) * Q_i^-1 mod q_i),
  // Q_i = q_0 * ... * q_{i-1}.  gd rows are packed 4 per int32 for dp4a.
  int ginv[kNumPrimes];
  int gd_packed[kNumPrimes][kGarnerWords];
  // Q_i = q_0 * ... * q_{i-1} as little-endian 32-bit words (Q_52 < 2^330).
  uint32_t Qw[kNumPrimes][kQWords];
};

// Host side: the tables (built once) and the primes.
const Tables& host_tables();
// The same tables for another sequence of distinct odd primes below 256
// (count <= 53), e.g. the subset a solve can use.
void build_tables_for(const int* qs, int count, Tables* out);

// Byte weights of shifted words: for every prime q, shift s < 256 and byte
// position k < 8, bal(2^(8k + s) mod q) as an int8, four to a word (word 0:
// k = 0..3, word 1: k = 4..7).  A dot product of an integer's bytes with the
// words of shift s gives its residue times 2^s.  Kept in global memory.
struct ShiftWeights {
  uint32_t w[kNumPrimes][kPow2Span][2];
};
const ShiftWeights& host_shift_weights();

// CRT with a round-to-nearest quotient, for the first P primes of the
// library's order and every P = 1..53: M[P][i] = (q_0 ... q_{P-1}) / q_i and
// Pw[P] = q_0 ... q_{P-1} as little-endian 32-bit words (kCrtWords significant,
// rows padded to kCrtStride), Cw[P] = 128 * sum_i M[P][i], and
// y[P][i] = bal(M[P][i]^-1 mod q_i).  Built once on the host, read from global
// memory by the kernels.
constexpr int kCrtWords = 11;   // q_0 ... q_52 < 2^334
constexpr int kCrtStride = 12;  // words per row (16-byte aligned rows)
struct CrtTables {
  uint32_t M[kNumPrimes + 1][kNumPrimes][kCrtStride];
  uint32_t Pw[kNumPrimes + 1][kCrtStride];
  uint32_t Cw[kNumPrimes + 1][kCrtStride];
  float y[kNumPrimes + 1][kNumPrimes];
};
const CrtTables& host_crt_tables();

// CRT by idempotent sums, for results that fit in int64 ("Accelerating
// Multiple-Precision LU Decomposition with Ozaki Scheme II", CRT with a
// round-to-nearest quotient, taken here on the unreduced residues): for the
// first P primes (P <= kIdemMaxP) and their product P, E_i = (P / q_i) *
// ((P / q_i)^-1 mod q_i) mod P is 1 modulo q_i and 0 modulo every other
// prime, so S = sum_i r_i E_i == x (mod P) for residues r_i in [0, q_i), and
// x = S - round(S / P) P when |x| < P / 4.  Rows hold E_i mod 2^64 (two
// words), f_i = round(2^20 E_i / P) and P mod 2^64.
constexpr int kIdemMaxP = 12;
constexpr int kIdemFracBits = 20;
struct IdemTables {
  uint32_t elo[kIdemMaxP + 1][kIdemMaxP];
  uint32_t ehi[kIdemMaxP + 1][kIdemMaxP];
  uint32_t f[kIdemMaxP + 1][kIdemMaxP];
  uint32_t plo[kIdemMaxP + 1];
  uint32_t phi[kIdemMaxP + 1];
};
const IdemTables& host_idem_tables();

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Balanced residue of an integer-valued float s, |s| < 2^24, modulo odd q:
// the unique r == s (mod q) with |r| <= (q-1)/2.  The quotient estimate
// rint(s * fl(1/q)) is within one of round(s/q), so one correction on each
// side suffices; every operation is exact on these integers.
__device__ __forceinline__ float bal_mod(float s, float q, float invq) {
  const float magic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer
  float t = __fadd_rn(__fmaf_rn(s, invq, magic), -magic);
  float r = __fmaf_rn(-t, q, s);
  float h = 0.5f * (q - 1.0f);
  r = r > h ? r - q : r;
  r = r < -h ? r + q : r;
  return r;
}

// The same for |s| <= 2^23, without corrections: |s * fl(1/q) - s/q| <
// |s/q| 2^-24 <= 1/(2q), while s/q (s an integer, q odd) lies at least 1/(2q)
// from every half-integer, so rint(s * fl(1/q)) == round(s/q) exactly and
// s - q * round(s/q) is already the balanced residue.
__device__ __forceinline__ float bal_mod_small(float s, float q, float invq) {
  const float magic = 12582912.0f;
  const float t = __fadd_rn(__fmaf_rn(s, invq, magic), -magic);
  return __fmaf_rn(-t, q, s);
}

__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23
constexpr int kMagicBits = 0x4B400000;  // its bit pattern

// Exact int -> float for |v| < 2^22 (and back) without the conversion unit:
// the integer sits in the low mantissa bits of kMagic + v.
__device__ __forceinline__ float int_to_float_exact(int v) { return __int_as_float(kMagicBits + v) - kMagic; }
__device__ __forceinline__ int float_bits_offset(float v) { return __float_as_int(v + kMagic); }  // = kMagicBits + v

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while its predecessor finishes; it must wait here
// before reading anything the predecessor wrote.  Without that launch
// attribute both instructions are no-ops.
__device__ __forceinline__ void wait_for_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream be scheduled (called after a block's
// main work, so an early dependent never competes with unfinished work).
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Division by a row length fixed for a launch, n / d for 0 <= n, by one
// multiply-high and shifts (Granlund and Montgomery, "Division by invariant
// integers using multiplication", unsigned N-bit division with a rounded-up
// 33-bit multiplier): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// t = mulhi(m, n) gives n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0) for
// every n < 2^32.  Larger n, or d >= 2^31, divide in 64 bits.
struct RowDiv {
  long long d;
  uint32_t magic;
  uint32_t sh1, sh2;
  int fast;
};

inline RowDiv make_rowdiv(long long d) {
  RowDiv r{d > 0 ? d : 1, 0u, 0u, 0u, 0};
  if (d <= 0 || d >= (1LL << 31)) return r;
  int l = 0;
  while ((1LL << l) < d) ++l;
  r.magic = (uint32_t)(((1ULL << 32) * ((1ULL << l) - (unsigned long long)d)) / (unsigned long long)d + 1ULL);
  r.sh1 = l > 0 ? 1u : 0u;
  r.sh2 = l > 0 ? (uint32_t)(l - 1) : 0u;
  r.fast = 1;
  return r;
}

__device__ __forceinline__ long long div_row(long long n, const RowDiv& r) {
  if (r.fast && (unsigned long long)n < (1ULL << 32)) {
    const uint32_t nn = (uint32_t)n, t = __umulhi(r.magic, nn);
    return (long long)((t + ((nn - t) >> r.sh1)) >> r.sh2);
  }
  return n / r.d;
}

// Launches `kernel` with programmatic stream serialisation.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace rg
