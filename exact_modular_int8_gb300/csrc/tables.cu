// tables.cpp -- host computation of the residue base and its constants.
//
// The residue base is the 53 odd primes below 256, largest first.  The pages
// ("exact-solve" and "enclosure-gemm", Method) use the primes below 256 and
// need an odd modulus; their capacity gate bits_a + bits_b + ceil(log2 K) <= 332
// is exactly floor(log2((P - 1) / 2)) for the product P of the 53 odd primes.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "rg_common.cuh"

namespace rg {
namespace {

int mod_pow(int a, int e, int q) {
  long long r = 1, b = a % q;
  while (e > 0) {
    if (e & 1) r = r * b % q;
    b = b * b % q;
    e >>= 1;
  }
  return (int)r;
}

int balanced(int r, int q) {  // r in [0, q) -> [-(q-1)/2, (q-1)/2]
  return r > (q - 1) / 2 ? r - q : r;
}

// Tables for the prime sequence qs[0..E) (distinct odd primes below 256, in
// the order the residues are combined); entries past E stay zero.
void build_for(const int* qs, int E, Tables& t) {
  std::memset(&t, 0, sizeof(t));
  for (int i = 0; i < E; ++i) t.q[i] = qs[i];

  for (int i = 0; i < E; ++i) {
    int q = t.q[i];
    t.qf[i] = (float)q;
    t.invq[i] = 1.0f / (float)q;
    for (int w = 0; w < kMaxWords; ++w) {
      uint32_t packed = 0;
      for (int b = 0; b < 4; ++b)
        packed |= (uint32_t)(uint8_t)(int8_t)balanced(mod_pow(2, 8 * (4 * w + b), q), q) << (8 * b);
      t.wbyte[i][w] = (int)packed;
    }
    for (int k = 0; k <= kMaxWords; ++k) t.wword[i][k] = balanced(mod_pow(2, 32 * k, q), q);
  }

  // floor(log2) of the running product, with an exact multi-word product.
  uint32_t big[16] = {1};
  t.log2P[0] = 0;
  for (int n2 = 1; n2 <= E; ++n2) {
    uint64_t carry = 0;
    for (int w = 0; w < 16; ++w) {
      uint64_t v = (uint64_t)big[w] * (uint64_t)t.q[n2 - 1] + carry;
      big[w] = (uint32_t)v;
      carry = v >> 32;
    }
    int top = 15;
    while (top > 0 && big[top] == 0) --top;
    int b = 31;
    while (!((big[top] >> b) & 1)) --b;
    t.log2P[n2] = 32 * top + b;
  }

  // Mixed-radix weights Q_i as words.
  {
    uint32_t q_words[kQWords] = {1};
    for (int i = 0; i < E; ++i) {
      for (int w = 0; w < kQWords; ++w) t.Qw[i][w] = q_words[w];
      uint64_t carry = 0;
      for (int w = 0; w < kQWords; ++w) {
        uint64_t v = (uint64_t)q_words[w] * (uint64_t)t.q[i] + carry;
        q_words[w] = (uint32_t)v;
        carry = v >> 32;
      }
    }
  }

  // Garner constants.
  for (int i = 0; i < E; ++i) {
    int q = t.q[i];
    long long Qi = 1;  // Q_i mod q
    for (int j = 0; j < i; ++j) Qi = Qi * t.q[j] % q;
    int inv = mod_pow((int)Qi, q - 2, q);  // q prime
    t.ginv[i] = balanced(inv, q);
    long long Qj = 1;  // Q_j mod q, j = 0..i-1
    for (int j = 0; j < i; ++j) {
      // negated, so that the digit is Q_i^-1 r_i + sum_j gd[i][j] v_j
      int d = balanced((int)((q - Qj * inv % q) % q), q);
      uint32_t byte = (uint32_t)(uint8_t)(int8_t)d;
      t.gd_packed[i][j / 4] |= (int)(byte << (8 * (j % 4)));
      Qj = Qj * t.q[j] % q;
    }
  }
}

// The residue base: the odd primes below 256, largest first.
void canonical_primes(int (&qs)[kNumPrimes]) {
  bool composite[256] = {};
  int n = 0;
  int asc[kNumPrimes];
  for (int i = 2; i < 256; ++i) {
    if (composite[i]) continue;
    for (int j = i * i; j < 256; j += i) composite[j] = true;
    if (i != 2) asc[n++] = i;
  }
  for (int i = 0; i < kNumPrimes; ++i) qs[i] = asc[kNumPrimes - 1 - i];
}

}  // namespace

const Tables& host_tables() {
  static Tables t;
  static std::once_flag once;
  std::call_once(once, [] {
    int qs[kNumPrimes];
    canonical_primes(qs);
    build_for(qs, kNumPrimes, t);
  });
  return t;
}

void build_tables_for(const int* qs, int count, Tables* out) { build_for(qs, count, *out); }

const ShiftWeights& host_shift_weights() {
  static ShiftWeights t;
  static std::once_flag once;
  std::call_once(once, [] {
    const Tables& b = host_tables();
    for (int i = 0; i < kNumPrimes; ++i)
      for (int s = 0; s < kPow2Span; ++s)
        for (int word = 0; word < 2; ++word) {
          uint32_t packed = 0;
          for (int j = 0; j < 4; ++j) {
            const int k = 4 * word + j;
            const int v = balanced(mod_pow(2, 8 * k + s, b.q[i]), b.q[i]);  // |v| <= 125
            packed |= (uint32_t)(uint8_t)(int8_t)v << (8 * j);
          }
          t.w[i][s][word] = packed;
        }
  });
  return t;
}

const CrtTables& host_crt_tables() {
  static CrtTables t;
  static std::once_flag once;
  std::call_once(once, [] {
    const Tables& b = host_tables();
    // w (kCrtWords little-endian words) *= f, for f < 2^32
    auto mul_small = [](uint32_t (&w)[kCrtWords], uint32_t f) {
      unsigned long long carry = 0;
      for (int k = 0; k < kCrtWords; ++k) {
        const unsigned long long v = (unsigned long long)w[k] * f + carry;
        w[k] = (uint32_t)v;
        carry = v >> 32;
      }
    };
    for (int P = 1; P <= kNumPrimes; ++P) {
      unsigned long long csum[kCrtWords] = {};  // 128 * sum_i M_i, word by word before the carries
      for (int i = 0; i <= P; ++i) {  // i = P: the whole product
        uint32_t w[kCrtWords] = {1u};
        int mmod = 1;  // M_i mod q_i
        for (int j = 0; j < P; ++j) {
          if (j == i) continue;
          mul_small(w, (uint32_t)b.q[j]);
          if (i < P) mmod = mmod * (b.q[j] % b.q[i]) % b.q[i];
        }
        uint32_t* dst = i < P ? t.M[P][i] : t.Pw[P];
        for (int k = 0; k < kCrtStride; ++k) dst[k] = k < kCrtWords ? w[k] : 0u;
        if (i < P) {
          t.y[P][i] = (float)balanced(mod_pow(mmod, b.q[i] - 2, b.q[i]), b.q[i]);  // Fermat: q_i prime
          for (int k = 0; k < kCrtWords; ++k) csum[k] += (unsigned long long)w[k] << 7;
        }
      }
      unsigned long long carry = 0;
      for (int k = 0; k < kCrtWords; ++k) {
        const unsigned long long v = csum[k] + carry;  // csum[k] < 53 * 2^39
        t.Cw[P][k] = (uint32_t)v;
        carry = v >> 32;
      }
      t.Cw[P][kCrtWords] = 0;
    }
  });
  return t;
}

const IdemTables& host_idem_tables() {
  static IdemTables t;
  static std::once_flag once;
  std::call_once(once, [] {
    const Tables& b = host_tables();
    typedef unsigned __int128 u128;  // the product of 12 primes below 256 is below 2^96
    std::memset(&t, 0, sizeof(t));
    for (int P = 1; P <= kIdemMaxP; ++P) {
      u128 prod = 1;
      for (int j = 0; j < P; ++j) prod *= (u128)b.q[j];
      for (int i = 0; i < P; ++i) {
        const int q = b.q[i];
        const u128 m = prod / (u128)q;
        const int inv = mod_pow((int)(m % (u128)q), q - 2, q);  // Fermat: q prime
        const u128 e = m * (u128)inv % prod;                     // m * inv < 2^104
        t.elo[P][i] = (uint32_t)e;
        t.ehi[P][i] = (uint32_t)(e >> 32);
        t.f[P][i] = (uint32_t)(((e << kIdemFracBits) + prod / 2) / prod);  // e * 2^20 < 2^116
      }
      t.plo[P] = (uint32_t)prod;
      t.phi[P] = (uint32_t)(prod >> 32);
    }
  });
  return t;
}

}  // namespace rg

extern "C" int rg_prime(int i) {
  if (i < 0 || i >= rg::kNumPrimes) return 0;
  return rg::host_tables().q[i];
}
