// bigint.cpp -- host multi-precision arithmetic for the exact solve's
// rational reconstruction: schoolbook and Karatsuba products, long division
// (Knuth's algorithm D on 64-bit limbs), Barrett's reduction by a fixed
// modulus, radix conversion by halves, and Lehmer's gcd and extended-Euclid
// rational reconstruction, each batch of leading-digit quotients applied to
// the full numbers in one in-place pass.
#include "bigint.h"

#include <algorithm>

namespace rg {
namespace big {

using u128 = unsigned __int128;

void trim(Nat& a) {
  while (!a.v.empty() && a.v.back() == 0) a.v.pop_back();
}

bool is_zero(const Nat& a) { return a.v.empty(); }

int cmp(const Nat& a, const Nat& b) {
  if (a.v.size() != b.v.size()) return a.v.size() < b.v.size() ? -1 : 1;
  for (size_t i = a.v.size(); i-- > 0;)
    if (a.v[i] != b.v[i]) return a.v[i] < b.v[i] ? -1 : 1;
  return 0;
}

size_t bit_length(const Nat& a) {
  if (a.v.empty()) return 0;
  return 64 * (a.v.size() - 1) + (64 - __builtin_clzll(a.v.back()));
}

Nat from_u64(uint64_t x) {
  Nat r;
  if (x) r.v.push_back(x);
  return r;
}

Nat pow2(size_t e) {
  Nat r;
  r.v.assign(e / 64 + 1, 0);
  r.v[e / 64] = 1ull << (e % 64);
  return r;
}

Nat add(const Nat& a, const Nat& b) {
  const Nat& x = a.v.size() >= b.v.size() ? a : b;
  const Nat& y = a.v.size() >= b.v.size() ? b : a;
  Nat r;
  r.v.resize(x.v.size() + 1);
  Limb carry = 0;
  for (size_t i = 0; i < x.v.size(); ++i) {
    const u128 t = (u128)x.v[i] + (i < y.v.size() ? y.v[i] : 0) + carry;
    r.v[i] = (Limb)t;
    carry = (Limb)(t >> 64);
  }
  r.v[x.v.size()] = carry;
  trim(r);
  return r;
}

Nat sub(const Nat& a, const Nat& b) {
  Nat r;
  r.v.resize(a.v.size());
  Limb borrow = 0;
  for (size_t i = 0; i < a.v.size(); ++i) {
    const Limb y = i < b.v.size() ? b.v[i] : 0;
    const Limb t = a.v[i] - y - borrow;
    borrow = (a.v[i] < y || (a.v[i] == y && borrow)) ? 1 : 0;
    r.v[i] = t;
  }
  trim(r);
  return r;
}

Nat mul(const Nat& a, const Nat& b) {
  Nat r;
  if (a.v.empty() || b.v.empty()) return r;
  r.v.assign(a.v.size() + b.v.size(), 0);
  for (size_t i = 0; i < a.v.size(); ++i) {
    Limb carry = 0;
    const Limb ai = a.v[i];
    for (size_t j = 0; j < b.v.size(); ++j) {
      const u128 t = (u128)ai * b.v[j] + r.v[i + j] + carry;
      r.v[i + j] = (Limb)t;
      carry = (Limb)(t >> 64);
    }
    r.v[i + b.v.size()] = carry;
  }
  trim(r);
  return r;
}

void divmod(const Nat& a, const Nat& b, Nat* q, Nat* r) {
  if (cmp(a, b) < 0) {
    if (q) q->v.clear();
    if (r) *r = a;
    return;
  }
  const size_t n = b.v.size(), m = a.v.size() - n;
  if (n == 1) {  // one-limb divisor
    Nat qq;
    qq.v.assign(a.v.size(), 0);
    u128 rem = 0;
    for (size_t i = a.v.size(); i-- > 0;) {
      const u128 cur = (rem << 64) | a.v[i];
      qq.v[i] = (Limb)(cur / b.v[0]);
      rem = cur % b.v[0];
    }
    trim(qq);
    if (q) *q = qq;
    if (r) *r = from_u64((uint64_t)rem);
    return;
  }
  // Knuth, The Art of Computer Programming vol. 2, 4.3.1, algorithm D.
  const int s = __builtin_clzll(b.v[n - 1]);
  std::vector<Limb> vn(n), un(a.v.size() + 1);
  for (size_t i = n; i-- > 1;) vn[i] = (b.v[i] << s) | (s ? b.v[i - 1] >> (64 - s) : 0);
  vn[0] = b.v[0] << s;
  un[a.v.size()] = s ? a.v[a.v.size() - 1] >> (64 - s) : 0;
  for (size_t i = a.v.size(); i-- > 1;) un[i] = (a.v[i] << s) | (s ? a.v[i - 1] >> (64 - s) : 0);
  un[0] = a.v[0] << s;
  Nat qq;
  qq.v.assign(m + 1, 0);
  for (size_t j = m + 1; j-- > 0;) {
    const u128 num = ((u128)un[j + n] << 64) | un[j + n - 1];
    u128 qhat = num / vn[n - 1], rhat = num % vn[n - 1];
    while (qhat >> 64 || qhat * vn[n - 2] > ((rhat << 64) | un[j + n - 2])) {
      --qhat;
      rhat += vn[n - 1];
      if (rhat >> 64) break;
    }
    // un[j .. j+n] -= qhat * vn
    Limb borrow = 0, carry = 0;
    for (size_t i = 0; i < n; ++i) {
      const u128 p = qhat * vn[i] + carry;
      carry = (Limb)(p >> 64);
      const Limb lo = (Limb)p;
      const Limb t = un[i + j] - lo - borrow;
      borrow = (un[i + j] < lo || (un[i + j] == lo && borrow)) ? 1 : 0;
      un[i + j] = t;
    }
    const Limb top = un[j + n];
    const Limb t = top - carry - borrow;
    const bool negative = top < carry || (top == carry && borrow);
    un[j + n] = t;
    if (negative) {  // qhat was one too large: add vn back
      --qhat;
      Limb c = 0;
      for (size_t i = 0; i < n; ++i) {
        const u128 sum = (u128)un[i + j] + vn[i] + c;
        un[i + j] = (Limb)sum;
        c = (Limb)(sum >> 64);
      }
      un[j + n] += c;
    }
    qq.v[j] = (Limb)qhat;
  }
  trim(qq);
  if (q) *q = qq;
  if (r) {
    Nat rr;
    rr.v.resize(n);
    for (size_t i = 0; i < n; ++i) rr.v[i] = (un[i] >> s) | (s ? un[i + 1] << (64 - s) : 0);
    trim(rr);
    *r = rr;
  }
}

Nat mod(const Nat& a, const Nat& b) {
  Nat r;
  divmod(a, b, nullptr, &r);
  return r;
}

Int add(const Int& a, const Int& b) {
  Int r;
  if (a.neg == b.neg) {
    r.mag = add(a.mag, b.mag);
    r.neg = a.neg && !is_zero(r.mag);
    return r;
  }
  const int c = cmp(a.mag, b.mag);
  if (c == 0) return r;
  if (c > 0) {
    r.mag = sub(a.mag, b.mag);
    r.neg = a.neg;
  } else {
    r.mag = sub(b.mag, a.mag);
    r.neg = b.neg;
  }
  return r;
}

Int sub(const Int& a, const Int& b) {
  Int nb = b;
  nb.neg = !b.neg && !is_zero(b.mag);
  return add(a, nb);
}

Int mul(const Int& a, const Nat& b) {
  Int r;
  r.mag = mul(a.mag, b);
  r.neg = a.neg && !is_zero(r.mag);
  return r;
}

Int from_words(const uint32_t* w, int nw) {
  Int r;
  const bool neg = nw > 0 && (w[nw - 1] >> 31) != 0;
  // magnitude = two's complement negation when negative
  std::vector<uint32_t> m(w, w + nw);
  if (neg) {
    uint64_t carry = 1;
    for (int i = 0; i < nw; ++i) {
      const uint64_t t = (uint64_t)(uint32_t)~m[i] + carry;
      m[i] = (uint32_t)t;
      carry = t >> 32;
    }
  }
  r.mag.v.assign((nw + 1) / 2, 0);
  for (int i = 0; i < nw; ++i) r.mag.v[i / 2] |= (Limb)m[i] << (32 * (i % 2));
  trim(r.mag);
  r.neg = neg && !is_zero(r.mag);
  return r;
}

bool to_limbs(const Int& a, int64_t* out, int limbs) {
  // the magnitude must leave the sign bit free: |a| < 2^(64 limbs - 1), or
  // a == -2^(64 limbs - 1)
  const size_t bl = bit_length(a.mag);
  if (bl > (size_t)64 * limbs) return false;
  std::vector<Limb> v(limbs, 0);
  for (size_t i = 0; i < a.mag.v.size(); ++i) v[i] = a.mag.v[i];
  if (!a.neg) {
    if (bl == (size_t)64 * limbs) return false;
  } else {
    Limb carry = 1;
    for (int i = 0; i < limbs; ++i) {
      const u128 t = (u128)(Limb)~v[i] + carry;
      v[i] = (Limb)t;
      carry = (Limb)(t >> 64);
    }
    if (!((v[limbs - 1] >> 63) & 1)) return false;
  }
  for (int i = 0; i < limbs; ++i) out[i] = (int64_t)v[i];
  return true;
}

Reducer make_reducer(const Nat& M) {
  Reducer R;
  R.M = M;
  const size_t n = M.v.size();
  R.shift = __builtin_clzll(M.v[n - 1]);
  R.vn.resize(n);
  for (size_t i = n; i-- > 1;) R.vn[i] = (M.v[i] << R.shift) | (R.shift ? M.v[i - 1] >> (64 - R.shift) : 0);
  R.vn[0] = M.v[0] << R.shift;
  return R;
}

void mul_into(const Limb* a, size_t na, const Limb* b, size_t nb, std::vector<Limb>& out) {
  out.assign(na + nb, 0);
  for (size_t i = 0; i < na; ++i) {
    Limb carry = 0;
    const Limb ai = a[i];
    Limb* o = out.data() + i;
    for (size_t j = 0; j < nb; ++j) {
      const u128 t = (u128)ai * b[j] + o[j] + carry;
      o[j] = (Limb)t;
      carry = (Limb)(t >> 64);
    }
    o[nb] = carry;
  }
}

void reduce(const Reducer& R, const Limb* a, size_t na, std::vector<Limb>& un, Nat* r) {
  while (na > 0 && a[na - 1] == 0) --na;
  const size_t n = R.vn.size();
  if (na < n || (na == n && [&] {
        for (size_t i = n; i-- > 0;)
          if (a[i] != R.M.v[i]) return a[i] < R.M.v[i];
        return false;
      }())) {
    r->v.assign(a, a + na);
    return;
  }
  const int s = R.shift;
  const std::vector<Limb>& vn = R.vn;
  un.assign(na + 1, 0);
  un[na] = s ? a[na - 1] >> (64 - s) : 0;
  for (size_t i = na; i-- > 1;) un[i] = (a[i] << s) | (s ? a[i - 1] >> (64 - s) : 0);
  un[0] = a[0] << s;
  if (n == 1) {
    u128 rem = 0;
    for (size_t i = na + 1; i-- > 0;) rem = ((rem << 64) | un[i]) % vn[0];
    r->v.assign(1, (Limb)(rem >> s));
    trim(*r);
    return;
  }
  for (size_t j = na - n + 1; j-- > 0;) {  // Knuth's algorithm D, remainder only
    const u128 num = ((u128)un[j + n] << 64) | un[j + n - 1];
    u128 qhat = num / vn[n - 1], rhat = num % vn[n - 1];
    while (qhat >> 64 || qhat * vn[n - 2] > ((rhat << 64) | un[j + n - 2])) {
      --qhat;
      rhat += vn[n - 1];
      if (rhat >> 64) break;
    }
    Limb borrow = 0, carry = 0;
    for (size_t i = 0; i < n; ++i) {
      const u128 p = qhat * vn[i] + carry;
      carry = (Limb)(p >> 64);
      const Limb lo = (Limb)p;
      const Limb t = un[i + j] - lo - borrow;
      borrow = (un[i + j] < lo || (un[i + j] == lo && borrow)) ? 1 : 0;
      un[i + j] = t;
    }
    const Limb top = un[j + n];
    const bool negative = top < carry || (top == carry && borrow);
    un[j + n] = top - carry - borrow;
    if (negative) {
      Limb c = 0;
      for (size_t i = 0; i < n; ++i) {
        const u128 sum = (u128)un[i + j] + vn[i] + c;
        un[i + j] = (Limb)sum;
        c = (Limb)(sum >> 64);
      }
      un[j + n] += c;
    }
  }
  r->v.resize(n);
  for (size_t i = 0; i < n; ++i) r->v[i] = (un[i] >> s) | (s ? un[i + 1] << (64 - s) : 0);
  trim(*r);
}

namespace {

// out[0 .. na + nb) = a * b, schoolbook (out need not be cleared).
void school_mul(const Limb* a, size_t na, const Limb* b, size_t nb, Limb* out) {
  std::fill(out, out + na + nb, Limb(0));
  for (size_t i = 0; i < na; ++i) {
    Limb carry = 0;
    const Limb ai = a[i];
    Limb* o = out + i;
    for (size_t j = 0; j < nb; ++j) {
      const u128 t = (u128)ai * b[j] + o[j] + carry;
      o[j] = (Limb)t;
      carry = (Limb)(t >> 64);
    }
    o[nb] = carry;
  }
}

// r[0 .. n) += a[0 .. na) (na <= n); returns the carry out of r[n - 1].
Limb add_to(Limb* r, size_t n, const Limb* a, size_t na) {
  Limb carry = 0;
  size_t i = 0;
  for (; i < na; ++i) {
    const u128 t = (u128)r[i] + a[i] + carry;
    r[i] = (Limb)t;
    carry = (Limb)(t >> 64);
  }
  for (; carry && i < n; ++i) {
    const u128 t = (u128)r[i] + carry;
    r[i] = (Limb)t;
    carry = (Limb)(t >> 64);
  }
  return carry;
}

// r[0 .. n) -= a[0 .. na) (na <= n); returns the borrow out of r[n - 1].
Limb sub_from(Limb* r, size_t n, const Limb* a, size_t na) {
  Limb borrow = 0;
  size_t i = 0;
  for (; i < na; ++i) {
    const Limb x = r[i], y = a[i];
    const Limb d = x - y - borrow;
    borrow = (x < y || (x == y && borrow)) ? 1 : 0;
    r[i] = d;
  }
  for (; borrow && i < n; ++i) {
    borrow = r[i] == 0 ? 1 : 0;
    r[i] -= 1;
  }
  return borrow;
}

// out[0 .. na + nb) = a * b with na >= nb (Karatsuba on halves of the longer
// factor when both are long; the longer split into nb-limb pieces when the
// factors are far apart in length).
void kmul(const Limb* a, size_t na, const Limb* b, size_t nb, Limb* out) {
  if (na < nb) {
    std::swap(a, b);
    std::swap(na, nb);
  }
  if (nb < kKaratsubaLimbs) {
    school_mul(a, na, b, nb, out);
    return;
  }
  if (na >= 2 * nb) {  // pieces of nb limbs of a, each a balanced product
    std::fill(out, out + na + nb, Limb(0));
    std::vector<Limb> piece(2 * nb);
    for (size_t off = 0; off < na; off += nb) {
      const size_t len = std::min(nb, na - off);
      kmul(a + off, len, b, nb, piece.data());
      add_to(out + off, na + nb - off, piece.data(), len + nb);
    }
    return;
  }
  // a = a0 + a1 B^h, b = b0 + b1 B^h, h = ceil(na / 2) (so nb > h as na < 2 nb)
  const size_t h = (na + 1) / 2, na1 = na - h, nb1 = nb - h;
  // z0 = a0 b0 in out[0 .. 2h), z2 = a1 b1 in out[2h .. na + nb)
  kmul(a, h, b, h, out);
  kmul(a + h, na1, b + h, nb1, out + 2 * h);
  // sa = a0 + a1, sb = b0 + b1 (h + 1 limbs each), z1 = sa sb - z0 - z2
  std::vector<Limb> sa(h + 1, 0), sb(h + 1, 0), z1(2 * h + 2);
  std::copy(a, a + h, sa.begin());
  sa[h] = add_to(sa.data(), h, a + h, na1);
  std::copy(b, b + h, sb.begin());
  sb[h] = add_to(sb.data(), h, b + h, nb1);
  kmul(sa.data(), h + 1, sb.data(), h + 1, z1.data());
  sub_from(z1.data(), 2 * h + 2, out, 2 * h);
  sub_from(z1.data(), 2 * h + 2, out + 2 * h, na1 + nb1);
  size_t nz1 = 2 * h + 2;
  while (nz1 > 0 && z1[nz1 - 1] == 0) --nz1;
  add_to(out + h, na + nb - h, z1.data(), nz1);
}

}  // namespace

void kmul_into(const Limb* a, size_t na, const Limb* b, size_t nb, std::vector<Limb>& out) {
  out.assign(na + nb, 0);
  if (!na || !nb) return;
  kmul(a, na, b, nb, out.data());
}

void radix_value(const Limb* z, size_t cnt, size_t pl, const std::vector<Nat>& pw, std::vector<Limb>& out) {
  if (cnt <= 16) {
    out.clear();
    std::vector<Limb> scratch;
    for (size_t i = cnt; i-- > 0;) mul_add_into(out, pw[0].v.data(), pw[0].v.size(), z + i * pl, pl, scratch);
    return;
  }
  size_t h = 1, k = 0;
  while (2 * h < cnt) {
    h *= 2;
    ++k;
  }
  std::vector<Limb> lo, hi;
  radix_value(z, h, pl, pw, lo);
  radix_value(z + h * pl, cnt - h, pl, pw, hi);
  size_t nh = hi.size(), nl = lo.size();
  while (nh > 0 && hi[nh - 1] == 0) --nh;
  while (nl > 0 && lo[nl - 1] == 0) --nl;
  if (nh == 0) {
    out.assign(lo.begin(), lo.begin() + nl);
    return;
  }
  kmul_into(hi.data(), nh, pw[k].v.data(), pw[k].v.size(), out);
  if (out.size() < nl + 1) out.resize(nl + 1, 0);
  out.push_back(0);
  add_to(out.data(), out.size(), lo.data(), nl);
}

Barrett make_barrett(const Nat& M) {
  Barrett R;
  R.M = M;
  R.n = M.v.size();
  Nat b2n;
  b2n.v.assign(2 * R.n + 1, 0);
  b2n.v[2 * R.n] = 1;
  divmod(b2n, M, &R.mu, nullptr);
  return R;
}

bool reduce_barrett(const Barrett& R, const Limb* a, size_t na, std::vector<Limb>& s1, std::vector<Limb>& s2,
                    Nat* r) {
  while (na > 0 && a[na - 1] == 0) --na;
  const size_t n = R.n;
  if (na > 2 * n) return false;
  if (na < n) {
    r->v.assign(a, a + na);
    return true;
  }
  // q3 = floor(floor(a / B^(n-1)) mu / B^(n+1))
  kmul_into(a + (n - 1), na - (n - 1), R.mu.v.data(), R.mu.v.size(), s1);
  const size_t q3 = s1.size() > n + 1 ? s1.size() - (n + 1) : 0;
  // r = (a - q3 M) mod B^(n+1)
  if (q3)
    kmul_into(s1.data() + (n + 1), q3, R.M.v.data(), n, s2);
  else
    s2.clear();
  std::vector<Limb> rr(a, a + std::min(na, n + 1));
  rr.resize(n + 1, 0);
  sub_from(rr.data(), n + 1, s2.data(), std::min(s2.size(), n + 1));  // a borrow out of limb n is the wrap mod B^(n+1)
  // at most two more subtractions of M
  auto ge_m = [&]() {
    if (rr[n] != 0) return true;
    for (size_t i = n; i-- > 0;)
      if (rr[i] != R.M.v[i]) return rr[i] > R.M.v[i];
    return true;
  };
  for (int k = 0; k < 3 && ge_m(); ++k) sub_from(rr.data(), n + 1, R.M.v.data(), n);
  if (ge_m()) return false;  // cannot happen for a < B^(2n)
  r->v.assign(rr.begin(), rr.begin() + n);
  trim(*r);
  return true;
}

void mul_add_into(std::vector<Limb>& acc, const Limb* m, size_t nm, const Limb* z, size_t nz,
                  std::vector<Limb>& scratch) {
  size_t na = acc.size();
  while (na > 0 && acc[na - 1] == 0) --na;
  scratch.assign(std::max(na + nm, nz) + 1, 0);
  for (size_t i = 0; i < na; ++i) {
    Limb carry = 0;
    const Limb ai = acc[i];
    Limb* o = scratch.data() + i;
    for (size_t j = 0; j < nm; ++j) {
      const u128 t = (u128)ai * m[j] + o[j] + carry;
      o[j] = (Limb)t;
      carry = (Limb)(t >> 64);
    }
    o[nm] = carry;
  }
  Limb carry = 0;
  for (size_t i = 0; i < scratch.size(); ++i) {
    const u128 t = (u128)scratch[i] + (i < nz ? z[i] : 0) + carry;
    scratch[i] = (Limb)t;
    carry = (Limb)(t >> 64);
  }
  acc.swap(scratch);
}

namespace {

// The 62 bits of x starting at bit s (x < 2^(s + 62)).
uint64_t bits_at(const Nat& x, size_t s) {
  const size_t w = s / 64, o = s % 64;
  uint64_t lo = w < x.v.size() ? x.v[w] >> o : 0;
  if (o && w + 1 < x.v.size()) lo |= x.v[w + 1] << (64 - o);
  return lo & ((1ull << 62) - 1);
}

// Lehmer's method (Knuth, TAOCP vol. 2, 4.5.2, algorithm L) for x >= y: the
// quotient sequence of the leading 62 bits (x's top 62 and y's bits at the
// same place), accepted while the bracketing quotients (u + A) / (v + C) and
// (u + B) / (v + D) agree, is the full numbers' sequence.  Returns the 2x2
// matrix of those steps: (A x + B y, C x + D y) are the remainders they reach.
// B == 0 when not even the first quotient is certain (y far below x).
struct Lehmer {
  long long A, B, C, D;
};
Lehmer lehmer_matrix(const Nat& x, const Nat& y) {
  const size_t b0 = bit_length(x);
  const size_t sh = b0 > 62 ? b0 - 62 : 0;
  long long u = (long long)bits_at(x, sh), v = (long long)bits_at(y, sh);
  long long A = 1, B = 0, C = 0, D = 1;
  while (true) {
    const __int128 d1 = (__int128)v + C, d2 = (__int128)v + D;
    if (d1 <= 0 || d2 <= 0) break;
    const __int128 q1 = ((__int128)u + A) / d1, q2 = ((__int128)u + B) / d2;
    if (q1 != q2) break;
    const long long q = (long long)q1;
    long long T = A - q * C;
    A = C;
    C = T;
    T = B - q * D;
    B = D;
    D = T;
    T = u - q * v;
    u = v;
    v = T;
  }
  return Lehmer{A, B, C, D};
}

// (x, y) <- (A x + B y, C x + D y) in one pass and in place, for a Lehmer
// matrix applied to two remainders: each row's entries have opposite signs
// (or one is zero) and magnitudes below 2^62, so every limb's A x_i + B y_i
// lies below 2^126 and, with its carry, fits a signed 128-bit accumulator;
// the images are the next two remainders, nonnegative and no longer than x.
void apply_matrix(Nat& x, Nat& y, long long A, long long B, long long C, long long D) {
  const size_t n = std::max(x.v.size(), y.v.size());
  x.v.resize(n, 0);
  y.v.resize(n, 0);
  __int128 c1 = 0, c2 = 0;
  for (size_t i = 0; i < n; ++i) {
    const __int128 xi = (__int128)x.v[i], yi = (__int128)y.v[i];
    const __int128 t1 = (__int128)A * xi + (__int128)B * yi + c1;
    const __int128 t2 = (__int128)C * xi + (__int128)D * yi + c2;
    x.v[i] = (Limb)t1;
    y.v[i] = (Limb)t2;
    c1 = t1 >> 64;  // arithmetic: a borrow carries as -1
    c2 = t2 >> 64;
  }
  trim(x);
  trim(y);
}

// The same matrix on the cofactors of those remainders, (t0, t1) <- (A t0 +
// B t1, C t0 + D t1), in one pass and in place.  Consecutive cofactors of
// Euclid's sequence alternate in sign, as do the entries of each row, so
// A t0 and B t1 never have opposite signs: the new magnitude is
// |A| |t0| + |B| |t1| (below 2^127 per limb with its carry) and the sign is
// that of either nonzero term.
void apply_matrix_cofactors(Int& t0, Int& t1, long long A, long long B, long long C, long long D) {
  auto mag = [](long long v) { return (unsigned long long)(v < 0 ? -(unsigned long long)v : (unsigned long long)v); };
  auto sign_of = [](long long a, const Int& x, long long b, const Int& y) {
    if (a != 0 && !is_zero(x.mag)) return (a < 0) != x.neg;
    return (b < 0) != y.neg;
  };
  const bool n0 = sign_of(A, t0, B, t1), n1 = sign_of(C, t0, D, t1);
  const unsigned __int128 a = mag(A), b = mag(B), c = mag(C), d = mag(D);
  const size_t n = std::max(t0.mag.v.size(), t1.mag.v.size());
  t0.mag.v.resize(n + 1, 0);
  t1.mag.v.resize(n + 1, 0);
  unsigned __int128 c0 = 0, c1 = 0;
  for (size_t i = 0; i <= n; ++i) {
    const unsigned __int128 x = t0.mag.v[i], y = t1.mag.v[i];
    const unsigned __int128 u0 = a * x + b * y + c0, u1 = c * x + d * y + c1;
    t0.mag.v[i] = (Limb)u0;
    t1.mag.v[i] = (Limb)u1;
    c0 = u0 >> 64;
    c1 = u1 >> 64;
  }
  if (c0) t0.mag.v.push_back((Limb)c0);
  if (c1) t1.mag.v.push_back((Limb)c1);
  trim(t0.mag);
  trim(t1.mag);
  t0.neg = n0 && !is_zero(t0.mag);
  t1.neg = n1 && !is_zero(t1.mag);
}

}  // namespace

Nat gcd(Nat a, Nat b) {
  if (cmp(a, b) < 0) std::swap(a, b);
  // Lehmer batches while b is wider than two limbs (each replaces about 30
  // single steps by one pass over the numbers), then Euclid's single steps
  while (b.v.size() > 2) {
    const Lehmer m = lehmer_matrix(a, b);
    if (m.B == 0) {
      Nat r = mod(a, b);
      a = std::move(b);
      b = std::move(r);
    } else {
      apply_matrix(a, b, m.A, m.B, m.C, m.D);
    }
  }
  while (!is_zero(b)) {
    Nat r = mod(a, b);
    a = std::move(b);
    b = std::move(r);
  }
  return a;
}

bool rational_reconstruct(const Nat& X, const Nat& M, const Nat& nbound, const Nat& dbound, Int* N, Nat* D) {
  // Extended Euclid on (M, X) with the cofactor of X, stopped at the first
  // remainder <= nbound (Wang's reconstruction).
  Nat r0 = M, r1 = X;
  Int t0, t1;
  t1.mag = from_u64(1);
  // Lehmer batches (lehmer_matrix), each applied once to the remainders and
  // the cofactors.  Run only while r1 stays more than 64 bits above the
  // bound: one batch shrinks r1 by less than 2^63, so no remainder of a batch
  // reaches the stopping point.
  const size_t stop_bits = bit_length(nbound) + 64;
  while (bit_length(r1) > stop_bits) {
    const Lehmer lm = lehmer_matrix(r0, r1);
    const long long A = lm.A, B = lm.B, C = lm.C, Dc = lm.D;
    if (B == 0) {  // no usable leading quotient: one full-precision step
      Nat q, r;
      divmod(r0, r1, &q, &r);
      Int t = sub(t0, mul(t1, q));
      r0 = std::move(r1);
      r1 = std::move(r);
      t0 = std::move(t1);
      t1 = std::move(t);
    } else {
      apply_matrix(r0, r1, A, B, C, Dc);
      apply_matrix_cofactors(t0, t1, A, B, C, Dc);
    }
  }
  while (cmp(r1, nbound) > 0) {
    Nat q, r;
    divmod(r0, r1, &q, &r);
    Int t = sub(t0, mul(t1, q));
    r0 = std::move(r1);
    r1 = std::move(r);
    t0 = std::move(t1);
    t1 = std::move(t);
  }
  if (is_zero(t1.mag) || cmp(t1.mag, dbound) > 0) return false;
  Int n;
  n.mag = r1;
  n.neg = t1.neg && !is_zero(r1);  // N / D with D = |t1|
  const Nat g = gcd(r1, t1.mag);
  if (cmp(g, from_u64(1)) != 0) return false;
  *N = n;
  *D = t1.mag;
  return true;
}

}  // namespace big
}  // namespace rg
