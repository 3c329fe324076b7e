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
// Digits are combined four at a time, D = v_i + q_i v_{i+1} + q_i q_{i+1}
// (v_{i+2} + q_{i+2} v_{i+3}), |D| <= (q_i q_{i+1} q_{i+2} q_{i+3} - 1) / 2 < 2^31:
// the pairs in fp32 (|pair| < 2^15), the quad in int32, so the wide
// accumulation runs once per four primes.  MAXP bounds P at compile time (the
// packed digits take (MAXP + 3) / 4 registers per entry).  SHARED: rc points
// into shared memory (one entry; plain loads instead of read-only cache loads).
template <int W, int GE, typename TAB, int MAXP = kNumPrimes, bool SHARED = false>
__device__ __forceinline__ void garner_reconstruct(const uint8_t* __restrict__ rc, long long plane, int P,
                                                   uint32_t (&x)[GE][W]) {
  static_assert(!SHARED || GE == 1, "one entry from shared memory");
  static_assert(MAXP >= 1 && MAXP <= kNumPrimes, "prime bound");
  constexpr int kWords = (MAXP + 3) / 4;
  uint32_t V[GE][kWords];
  float pend[GE];  // the even digit of the current pair, as float
  int dq[GE];      // the first pair of the current quad
#pragma unroll
  for (int e = 0; e < GE; ++e) {
#pragma unroll
    for (int w = 0; w < kWords; ++w) V[e][w] = 0u;
#pragma unroll
    for (int k = 0; k < W; ++k) x[e][k] = 0u;
    pend[e] = 0.0f;
    dq[e] = 0;
  }
#pragma unroll
  for (int i0 = 0; i0 < MAXP; i0 += kGarnerBatch) {
    if (i0 >= P) break;
    uint32_t rw[kGarnerBatch];
#pragma unroll
    for (int j = 0; j < kGarnerBatch; ++j) {
      const int i = i0 + j;
      static_assert(GE == 1 || GE == 2 || GE == 4, "one, two or four adjacent entries");
      const bool in = i < P && i < MAXP;
      if constexpr (SHARED)
        rw[j] = in ? (uint32_t)rc[(long long)i * plane] : 0u;
      else if constexpr (GE == 4)
        rw[j] = in ? __ldg(reinterpret_cast<const uint32_t*>(rc + (long long)i * plane)) : 0u;
      else if constexpr (GE == 2)
        rw[j] = in ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(rc + (long long)i * plane)) : 0u;
      else
        rw[j] = in ? (uint32_t)__ldg(rc + (long long)i * plane) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kGarnerBatch; ++j) {
      const int i = i0 + j;
      if (i >= MAXP || i >= P) break;
      const float q = TAB::t().qf[i], iq = TAB::t().invq[i];
      const int gi = TAB::t().ginv[i];
      // byte selector that inserts a new low byte at position i % 4
      constexpr unsigned kSel[4] = {0x3214u, 0x3240u, 0x3410u, 0x4210u};
#pragma unroll
      for (int e = 0; e < GE; ++e) {
        // s = Q_i^-1 r_i - sum_{j<i} (Q_j Q_i^-1 mod q_i) v_j, |s| < 2^20
        int acc = gi * (int)((rw[j] >> (8 * e)) & 0xFFu);
#pragma unroll
        for (int w = 0; w < kWords; ++w)
          if (4 * w < i) acc = __dp4a((int)V[e][w], TAB::t().gd_packed[i][w], acc);
        const float vf = bal_mod_small(int_to_float_exact(acc), q, iq);
        const int vb = float_bits_offset(vf);
        V[e][i / 4] = __byte_perm(V[e][i / 4], (uint32_t)vb, kSel[i % 4]);
        const int s0 = i & ~3;  // the quad's first prime
        int d = 0;              // the quad's value, when it is added now
        bool add = false;
        if ((i & 1) == 0) {
          pend[e] = vf;
          if (i + 1 >= P) {  // the last digit opens a pair: v_i, or the first pair plus q_{i-2} q_{i-1} v_i
            d = (i & 2) ? dq[e] + TAB::t().q[i - 2] * TAB::t().q[i - 1] * (vb - kMagicBits) : vb - kMagicBits;
            add = true;
          }
        } else {
          const int pair = float_bits_offset(__fmaf_rn(vf, TAB::t().qf[i - 1], pend[e])) - kMagicBits;
          if ((i & 2) == 0) {  // the quad's first pair
            dq[e] = pair;
            if (i + 1 >= P) {
              d = pair;
              add = true;
            }
          } else {
            d = dq[e] + TAB::t().q[i - 3] * TAB::t().q[i - 2] * pair;
            add = true;
          }
        }
        if (add) {
          if (W > 2 && s0 > 0 && s0 / 4 + 1 < W) x[e][s0 / 4 + 1] = (uint32_t)((int)x[e][s0 / 4] >> 31);
          add_scaled_weight<W, TAB>(x[e], d, s0, i);
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

namespace rg {
namespace {

// ---------------------------------------------------------------------------
// CRT with a round-to-nearest quotient ("Accelerating Multiple-Precision LU
// Decomposition with Ozaki Scheme II", CRT reconstruction of the centred
// representative by round-to-nearest).  With M_i = P / q_i and
// y_i = bal(M_i^-1 mod q_i), the digits s_i = bal(r_i y_i mod q_i) give
// S = sum_i s_i M_i == x (mod P), and S / P = sum_i s_i / q_i = k + x / P.
// When |x| < P / 4 the quotient k is the nearest integer to the fp32 sum of
// s_i / q_i (|s_i / q_i| <= 1/2, so 53 terms carry an error far below 1/4),
// and x = S - k P exactly.  O(P W) work per output instead of Garner's O(P^2);
// S and k P are formed modulo 2^(32 W), which holds x.
// ---------------------------------------------------------------------------
// The tables of one prime count P (CrtTables rows in global memory).
struct CrtView {
  const uint32_t (*M)[kCrtStride];  // M[i] = P / q_i
  const uint32_t* Pw;               // P
  const uint32_t* Cw;               // 128 * sum_i M_i (the digits are summed offset by +128)
  const float* y;                   // bal(M_i^-1 mod q_i)
};

// x[e] (W words, two's complement) = the centred integers of the GE residue
// vectors (residues in [0, q)) starting at rc, plane bytes apart.
template <int W, int GE, typename TAB>
__device__ __forceinline__ void crt_rn_reconstruct(const uint8_t* __restrict__ rc, long long plane, int P,
                                                   const CrtView& T, uint32_t (&x)[GE][W]) {
  constexpr int NW = W < kCrtWords ? W : kCrtWords;  // words that can differ from the sign
  static_assert(GE == 1 || GE == 2 || GE == 4, "one, two or four adjacent entries");
  unsigned long long acc[GE][NW];  // sum_i (s_i + 128) M_i, words not yet normalised (< 2^46)
  float kf[GE];
#pragma unroll
  for (int e = 0; e < GE; ++e) {
    kf[e] = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) acc[e][w] = 0;
  }
#pragma unroll 1
  for (int i0 = 0; i0 < P; i0 += kGarnerBatch) {
    uint32_t rw[kGarnerBatch];
#pragma unroll
    for (int j = 0; j < kGarnerBatch; ++j) {
      const int i = i0 + j;
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
      if (i >= P) break;
      const float q = TAB::t().qf[i], iq = TAB::t().invq[i], y = __ldg(T.y + i);
      uint32_t m[NW];
#pragma unroll
      for (int w = 0; w < NW; ++w) m[w] = __ldg(&T.M[i][w]);
#pragma unroll
      for (int e = 0; e < GE; ++e) {
        const float r = int_to_float_exact((int)((rw[j] >> (8 * e)) & 0xFFu));
        const float s = bal_mod_small(r * y, q, iq);  // |r y| <= 250 * 125
        kf[e] = __fmaf_rn(s, iq, kf[e]);
        const uint32_t sp = (uint32_t)(float_bits_offset(s) - kMagicBits + 128);  // s + 128 in [3, 253]
#pragma unroll
        for (int w = 0; w < NW; ++w) acc[e][w] += (unsigned long long)sp * m[w];
      }
    }
  }
#pragma unroll
  for (int e = 0; e < GE; ++e) {
    const long long k = (long long)(float_bits_offset(kf[e]) - kMagicBits);  // nearest integer (|k| <= 27)
    long long carry = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const long long t = (long long)acc[e][w] - (long long)__ldg(T.Cw + w) - k * (long long)__ldg(T.Pw + w) + carry;
      x[e][w] = (uint32_t)t;
      carry = t >> 32;  // arithmetic shift: the next word's borrow or carry
    }
    const uint32_t sign = (uint32_t)((int)x[e][NW - 1] >> 31);
#pragma unroll
    for (int w = NW; w < W; ++w) x[e][w] = sign;
  }
}

}  // namespace
}  // namespace rg
