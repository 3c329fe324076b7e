// rg_garner.cuh -- balanced Garner reconstruction, shared by the GEMM path
// and the exact solve (internal).
//
// Balanced Garner ("exact-solve" and "enclosure-gemm", Method: balanced-Garner
// mixed-radix digits).  With Q_i = q_0 ... q_{i-1} the digits
//   v_i = bal( (r_i - sum_{j<i} v_j Q_j) Q_i^-1  mod q_i ),  |v_i| <= (q_i-1)/2,
// give x = sum_i v_i Q_i, the unique representative with |x| <= (P-1)/2.
// Each digit costs one int8x4 dot product per four earlier digits and one
// reciprocal reduction, and is added into x at once: after digit i,
// |x| < Q_{i+1} / 2 < 2^(8(i+1) - 1) (every q_i < 2^8), so only the low
// i/4 + 2 words of x can differ from its sign extension and only those are
// updated.  Residues are fetched eight primes at a time, so the loads of a
// batch are in flight together; the loop stops at the prime count.
//
// TAB::t() names the constant tables of the prime sequence q_0, q_1, ...:
// the library's own order for the GEMM path, or the sequence a solve uses.
#pragma once
#include <cstdint>

#include "rg_common.cuh"

namespace rg {
namespace {

// Output elements per thread: four (one 32-bit residue load per prime) for
// narrow results, two for wide ones to bound register use.
template <int W>
struct GarnerGE {
  static constexpr int value = W <= 4 ? 4 : 2;
};

constexpr int kGarnerBatch = 8;

// x (W 32-bit words, two's complement, mod 2^(32W)) += D * Q_i, for the words
// that can be significant once digits up to `last` are in (|x| < 2^(8(last+1)-1)).
template <int W, typename TAB>
__device__ __forceinline__ void add_scaled_weight(uint32_t (&x)[W], int D, int i, int last) {
  if constexpr (W == 2) {
    const unsigned long long Qi = ((unsigned long long)TAB::t().Qw[i][1] << 32) | TAB::t().Qw[i][0];
    const unsigned long long x64 = (((unsigned long long)x[1] << 32) | x[0]) + (unsigned long long)(long long)D * Qi;
    x[0] = (uint32_t)x64;
    x[1] = (uint32_t)(x64 >> 32);
  } else {
    long long carry = 0;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      if (k < last / 4 + 2) {
        const long long qk = k < kQWords ? (long long)TAB::t().Qw[i][k < kQWords ? k : 0] : 0ll;
        const long long t = (long long)x[k] + qk * D + carry;
        x[k] = (uint32_t)t;
        carry = t >> 32;
      }
    }
  }
}

// x[e] (W 32-bit words, two's complement) = the reconstructed integers of the
// GE residue vectors starting at rc (plane = distance between primes).
// Digits are combined in pairs, D = v_i + q_i v_{i+1} (|D| < 2^15, exact in
// fp32), so the wide accumulation runs once per two primes.
template <int W, int GE, typename TAB>
__device__ __forceinline__ void garner_reconstruct(const uint8_t* __restrict__ rc, long long plane, int P,
                                                   uint32_t (&x)[GE][W]) {
  uint32_t V[GE][kGarnerWords];
  float pend[GE];  // the even digit of the current pair, as float
#pragma unroll
  for (int e = 0; e < GE; ++e) {
#pragma unroll
    for (int w = 0; w < kGarnerWords; ++w) V[e][w] = 0u;
#pragma unroll
    for (int k = 0; k < W; ++k) x[e][k] = 0u;
    pend[e] = 0.0f;
  }
#pragma unroll
  for (int i0 = 0; i0 < kNumPrimes; i0 += kGarnerBatch) {
    if (i0 >= P) break;
    uint32_t rw[kGarnerBatch];
#pragma unroll
    for (int j = 0; j < kGarnerBatch; ++j) {
      const int i = i0 + j;
      static_assert(GE == 1 || GE == 2 || GE == 4, "one, two or four adjacent entries");
      if constexpr (GE == 4)
        rw[j] = (i < P) ? __ldg(reinterpret_cast<const uint32_t*>(rc + (long long)i * plane)) : 0u;
      else if constexpr (GE == 2)
        rw[j] = (i < P) ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(rc + (long long)i * plane)) : 0u;
      else
        rw[j] = (i < P) ? (uint32_t)__ldg(rc + (long long)i * plane) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kGarnerBatch; ++j) {
      const int i = i0 + j;
      if (i >= kNumPrimes || i >= P) break;
      const float q = TAB::t().qf[i], iq = TAB::t().invq[i];
      const int gi = TAB::t().ginv[i];
      // byte selector that inserts a new low byte at position i % 4
      constexpr unsigned kSel[4] = {0x3214u, 0x3240u, 0x3410u, 0x4210u};
#pragma unroll
      for (int e = 0; e < GE; ++e) {
        // s = Q_i^-1 r_i - sum_{j<i} (Q_j Q_i^-1 mod q_i) v_j, |s| < 2^20
        int acc = gi * (int)((rw[j] >> (8 * e)) & 0xFFu);
#pragma unroll
        for (int w = 0; w < kGarnerWords; ++w)
          if (4 * w < i) acc = __dp4a((int)V[e][w], TAB::t().gd_packed[i][w], acc);
        const float vf = bal_mod_small(int_to_float_exact(acc), q, iq);
        const int vb = float_bits_offset(vf);
        V[e][i / 4] = __byte_perm(V[e][i / 4], (uint32_t)vb, kSel[i % 4]);
        if ((i & 1) == 0) {
          pend[e] = vf;
          if (i + 1 >= P) {  // unpaired last digit
            if (W > 2 && (i % 4) == 0 && i > 0 && i / 4 + 1 < W)
              x[e][i / 4 + 1] = (uint32_t)((int)x[e][i / 4] >> 31);
            add_scaled_weight<W, TAB>(x[e], vb - kMagicBits, i, i);
          }
        } else {
          const float D = __fmaf_rn(vf, TAB::t().qf[i - 1], pend[e]);  // v_{i-1} + q_{i-1} v_i
          if (W > 2 && ((i - 1) % 4) == 0 && i > 1 && (i - 1) / 4 + 1 < W)
            x[e][(i - 1) / 4 + 1] = (uint32_t)((int)x[e][(i - 1) / 4] >> 31);
          add_scaled_weight<W, TAB>(x[e], float_bits_offset(D) - kMagicBits, i - 1, i);
        }
      }
    }
  }
  if constexpr (W == 2) return;  // the 64-bit form is complete
  // sign-extend from the last significant word (branch-free, so x stays in
  // registers: every index is a compile-time constant)
  const int top = (P - 1) / 4 + 2;
#pragma unroll
  for (int e = 0; e < GE; ++e) {
    uint32_t sign = 0u;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const uint32_t at_top = 0u - (uint32_t)(k == top - 1);
      const uint32_t above = 0u - (uint32_t)(k >= top);
      sign = (sign & ~at_top) | ((uint32_t)((int)x[e][k] >> 31) & at_top);
      x[e][k] = (x[e][k] & ~above) | (sign & above);
    }
  }
}


}  // namespace
}  // namespace rg
