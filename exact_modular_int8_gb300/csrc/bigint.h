// bigint.h -- host multi-precision integers for the exact solve's rational
// reconstruction (internal).  Little-endian 64-bit limbs; naturals carry no
// leading zero limb (zero is the empty vector).
#pragma once
#include <cstdint>
#include <vector>

namespace rg {
namespace big {

using Limb = uint64_t;

struct Nat {
  std::vector<Limb> v;
};

struct Int {  // sign and magnitude; zero is never negative
  bool neg = false;
  Nat mag;
};

void trim(Nat& a);
bool is_zero(const Nat& a);
int cmp(const Nat& a, const Nat& b);
size_t bit_length(const Nat& a);
Nat from_u64(uint64_t x);
Nat pow2(size_t e);

Nat add(const Nat& a, const Nat& b);
Nat sub(const Nat& a, const Nat& b);  // requires a >= b
Nat mul(const Nat& a, const Nat& b);
// q = a / b, r = a % b (b != 0).
void divmod(const Nat& a, const Nat& b, Nat* q, Nat* r);
Nat mod(const Nat& a, const Nat& b);
Nat gcd(Nat a, Nat b);

Int add(const Int& a, const Int& b);
Int sub(const Int& a, const Int& b);
Int mul(const Int& a, const Nat& b);

// Two's-complement words (little-endian 32-bit) -> Int.
Int from_words(const uint32_t* w, int nw);
// Int -> `limbs` little-endian two's-complement int64 limbs; false if it does not fit.
bool to_limbs(const Int& a, int64_t* out, int limbs);

// Repeated reduction modulo one fixed M > 0 (normalised once for long
// division), with caller-owned scratch so that no call allocates once the
// buffers have grown.
struct Reducer {
  Nat M;
  std::vector<Limb> vn;  // M shifted so its top limb has its top bit set
  int shift = 0;
};
Reducer make_reducer(const Nat& M);
// out = (a[0..na) * b[0..nb)) as limbs (length na + nb, not trimmed).
void mul_into(const Limb* a, size_t na, const Limb* b, size_t nb, std::vector<Limb>& out);
// r = a mod R.M for a given as na limbs; un is scratch.
void reduce(const Reducer& R, const Limb* a, size_t na, std::vector<Limb>& un, Nat* r);
// out = a * b by Karatsuba's method above kKaratsubaLimbs limbs per factor
// (schoolbook below), out of length na + nb, not trimmed.
constexpr size_t kKaratsubaLimbs = 32;
void kmul_into(const Limb* a, size_t na, const Limb* b, size_t nb, std::vector<Limb>& out);

// Repeated reduction modulo one fixed M > 0 by Barrett's method: with n the
// limbs of M and mu = floor(B^(2n) / M) (B = 2^64), the quotient of any
// x < B^(2n) is floor(floor(x / B^(n-1)) mu / B^(n+1)) minus at most 2, so
// the remainder takes two products and at most two subtractions.
struct Barrett {
  Nat M;
  Nat mu;
  size_t n = 0;
};
Barrett make_barrett(const Nat& M);
// r = a mod R.M for a of na limbs, a < B^(2n) (else false); s1, s2 are scratch.
bool reduce_barrett(const Barrett& R, const Limb* a, size_t na, std::vector<Limb>& s1, std::vector<Limb>& s2, Nat* r);

// out = sum_{i < cnt} z_i R^i for digits z_i of pl limbs each (z = cnt x pl
// limbs) and R = pw[0], with pw[k] = R^(2^k) for every 2^k < cnt: the lower
// and upper halves (at the largest power of two below cnt) recursively, then
// one Karatsuba product by a power of R; Horner's rule below 16 digits.
void radix_value(const Limb* z, size_t cnt, size_t pl, const std::vector<Nat>& pw, std::vector<Limb>& out);

// acc = acc * m + z in place (m and z as limb arrays; acc grows as needed).
void mul_add_into(std::vector<Limb>& acc, const Limb* m, size_t nm, const Limb* z, size_t nz,
                  std::vector<Limb>& scratch);

// Rational reconstruction: the N, D with D X == N (mod M), |N| <= nbound,
// 0 < D <= dbound, for 0 <= X < M and 2 nbound dbound < M (then unique, in
// lowest terms).  False if there is none.
bool rational_reconstruct(const Nat& X, const Nat& M, const Nat& nbound, const Nat& dbound, Int* N, Nat* D);

}  // namespace big
}  // namespace rg
