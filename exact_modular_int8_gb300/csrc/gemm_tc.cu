// gemm_tc.cu -- the per-prime residue product on the sm_103a tensor cores.
//
// Page "exact-solve", Method: each step's per-prime product is one batched
// tensor-core GEMM on balanced residues; page "enclosure-gemm", Requirements:
// K <= 2^17, set by the accumulator.
//
// sm_103a has no integer tcgen05 MMA, so the residues (|r| <= 125) go through
// tcgen05.mma kind::f16 as exactly representable fp16 values, accumulating in
// fp32 in tensor memory.  Every product is an integer below 2^14 in magnitude;
// a chunk of Kc = 1024 products therefore sums to less than 1024 * 15625 <
// 2^24 and stays an exact fp32 integer.  After each chunk the accumulator is
// reduced modulo q in place (|remainder| <= 2.2 q), so the next chunk adds
// onto a small value and never reaches 2^24.  Two accumulators alternate
// chunks, so the reduction of one overlaps the products of the other; the
// last two chunks of a tile are reduced to [0, q), summed, and written as
// uint8 residues through shared memory and a TMA store.  (The in-place
// remainder is at most 2.2 q, so a chunk ends below 1024 * 125^2 + 553 < 2^24.)
//
// Warp roles (one CTA per SM, persistent over tiles of (prime, m, n)):
//   warp 0      TMA producer: A tile 128x64 (K-major) and B tile 64x256
//               (N-major) per pipeline stage, 128-byte swizzle.
//   warp 1      owns the tensor memory and issues the MMAs (one thread).
//   warps 2..9  epilogue, two warpgroups of four (each warp may only reach
//               the tensor-memory lanes of its warp index mod 4; each
//               warpgroup drains 128 of the 256 columns): tcgen05.ld,
//               reduction mod q, tcgen05.st / output.
// Every wait is bounded; on expiry the kernel records RG_ERR_TIMEOUT, lets
// in-flight copies and MMAs finish, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <atomic>
#include <mutex>

#include "rg_common.cuh"
#include "rg_kernels.h"

namespace rg {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // fp16 per k-block: one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int KC_BLOCKS = 16;  // k-blocks per exact fp32 chunk: Kc = 1024
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_SLAB = 64 * BK * 2;  // one 64-column slab of B
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int OUT_HALF = 128 * 128;  // uint8 staging: two 128x128 halves
constexpr int OUT_BYTES = 2 * OUT_HALF;
constexpr int TMEM_COLS = 2 * BN;
constexpr int EPI_WARPS = 8;  // two warpgroups, each draining 128 of the 256 columns
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + OUT_BYTES + BAR_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory");

// Instruction descriptor, kind::f16: D f32, A and B f16, A K-major, B MN-major,
// N = 256, M = 128.
constexpr uint32_t IDESC = (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (1u << 16) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

struct GemmParams {
  int M, N, K;
  int mt, nt;
  int kb_total;
  int batch;       // independent products per prime; plane = prime * batch + product
  int planes;      // residue planes of one K slice of RC (pmax * batch)
  int max_splits;  // K slices the output buffer has room for (1: no split-K)
  int P_fixed;     // 0: read (or derive) the prime count from the plan
  int derive_i64;  // derive the int64 plan from max |A|, max |B|
  int ceil_log2_k;
  int fault;
  unsigned long long wait_ns;
  uint32_t* plane_hint;  // derive_i64: where to record the prime count for the next call's split (or null)
  float qf[kNumPrimes];
  float invq[kNumPrimes];
  int log2P[kNumPrimes + 1];  // floor(log2(q_0 ... q_{n-1}))
};

// The prime count of this launch, or 0 if the call has already failed.  For
// the int64 path without a planner pass every CTA derives the same plan from
// the split's reductions (fewest primes with product > 2^(T+1),
// T = bits(max|A|) + bits(max|B|) + ceil(log2 K), and the exact check
// K * max|A| * max|B| <= 2^63 - 1); CTA 0 records it for the Garner kernel.
__device__ int launch_primes(const GemmParams& gp, DevPlan* plan) {
  if (!gp.derive_i64) {
    if (plan->status) return 0;
    return gp.P_fixed ? gp.P_fixed : plan->P;
  }
  const unsigned long long ma = __ldcg(&plan->maxmag_a), mb = __ldcg(&plan->maxmag_b);
  const int bits_a = ma ? 64 - __clzll(ma) : 0, bits_b = mb ? 64 - __clzll(mb) : 0;
  const int T = bits_a + bits_b + gp.ceil_log2_k;
  int P = gp.P_fixed;
  bool range = false;
  if (!P) {
    const unsigned long long k = (unsigned long long)gp.K, ab = ma * mb;
    range = __umul64hi(ma, mb) != 0 || __umul64hi(ab, k) != 0 || ab * k > 0x7FFFFFFFFFFFFFFFull;
    for (int n = 1; n <= kNumPrimes && !P; ++n)
      if (gp.log2P[n] >= T + 1) P = n;
    if (!P) range = true;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    plan->P = range ? 0 : P;
    plan->bits_a = bits_a;
    plan->bits_b = bits_b;
    plan->bound_bits = T;
    if (range) atomicCAS(&plan->status, 0, RG_ERR_RANGE);
    else if (gp.plane_hint && !gp.P_fixed) *gp.plane_hint = kPlaneHintTag | (uint32_t)P;
  }
  return range ? 0 : P;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

struct Ctl {
  volatile int* abort;
  int* status;
  int* where;
  unsigned long long limit_ns;
};

// Wait for the phase of `parity` to complete, for at most ctl.limit_ns.
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, const Ctl& ctl, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*ctl.abort) return false;
      if (globaltimer() - t0 > ctl.limit_ns) {
        *ctl.abort = 1;
        atomicCAS(ctl.status, 0, RG_ERR_TIMEOUT);
        atomicCAS(ctl.where, 0, where);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void umma_f16(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle.  lbo/sbo in bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

#define RG_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define RG_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : RG_R8(0), RG_R8(8), RG_R8(16), RG_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      RG_W8(0), RG_W8(8), RG_W8(16), RG_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// x - q * t with t an integer within 1.7 of x/q, for any |x| < 2^24: y + 2^24
// rounds to an integer (spacing 1 or 2) for |y| <= 2^23.  The result is an
// integer with |r| <= 2.2 q, small enough to carry into the next chunk
// (1024 * 125^2 + 2.2 * 251 < 2^24).
__device__ __forceinline__ float partial_residue(float x, float q, float iq) {
  const float two24 = 16777216.0f;
  const float t = __fadd_rn(__fmaf_rn(x, iq, two24), -two24);
  return __fmaf_rn(-t, q, x);
}

// Final residues of 32 accumulator values (|x| < 2^24) plus an optional byte
// carry, packed four per word, using only FMA-pipe and byte-permute
// instructions.  The first reduction leaves |r| <= 2.2 q; the second is exact
// (|r| < 2^23, see the split kernel's reduction), giving the balanced residue,
// moved to [0, q).  Bytes enter and leave the float domain through
// the low mantissa bits of 2^23.
// Residue bytes of 32 accumulator values (|x| < 2^24, exact integers in
// fp32), in [0, q), packed four to a word; with CARRY the bytes in `carry`
// are added mod q.  ONE_ROUND: one rounding suffices when |x / q| < 2^22,
// true for every |x| < 2^24 once q >= 5: t = rint(x fl(1/q)) is within
// 1/2 + 1/q of x / q, so |x - t q| < q and one conditional add gives [0, q).
// For q = 3 (large unreduced residues from the stage entry point) the
// partial reduction runs first.  Straight-line code over the 32 values, so
// that their dependency chains interleave.
template <bool ONE_ROUND, bool CARRY>
__device__ __forceinline__ void final_residues_t(const uint32_t (&r)[32], const uint32_t (&carry)[8], float q,
                                                 float iq, uint32_t (&packed)[8]) {
  const float magic = 12582912.0f, two23 = 8388608.0f;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(r[i]);
    if constexpr (!ONE_ROUND) v[i] = partial_residue(v[i], q, iq);
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float t = __fadd_rn(__fmaf_rn(v[i], iq, magic), -magic);
    v[i] = __fmaf_rn(-t, q, v[i]);
    v[i] = v[i] < 0.0f ? v[i] + q : v[i];
  }
  if constexpr (CARRY) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      // 0x4B0000cc is the float 2^23 + c for the carry byte c
      const float c = __uint_as_float(__byte_perm(carry[i >> 2], 0x4B000000u, 0x7540u + (uint32_t)(i & 3))) - two23;
      v[i] = v[i] + c;
      v[i] = v[i] >= q ? v[i] - q : v[i];
    }
  }
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t b[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) b[k] = __float_as_uint(v[4 * w + k] + two23);  // low byte = v
    packed[w] = __byte_perm(__byte_perm(b[0], b[1], 0x0040u), __byte_perm(b[2], b[3], 0x0040u), 0x5410u);
  }
}

__device__ __forceinline__ void final_residues(const uint32_t (&r)[32], const uint32_t (&carry)[8], bool add_carry,
                                               float q, float iq, uint32_t (&packed)[8]) {
  const bool one_round = q > 4.0f;  // uniform: one prime per tile
  if (one_round) {
    if (add_carry) final_residues_t<true, true>(r, carry, q, iq, packed);
    else final_residues_t<true, false>(r, carry, q, iq, packed);
  } else {
    if (add_carry) final_residues_t<false, true>(r, carry, q, iq, packed);
    else final_residues_t<false, false>(r, carry, q, iq, packed);
  }
}

// Byte offset of (row, 16-byte chunk j) in a 128-row x 128-byte swizzled half.
__device__ __forceinline__ uint32_t sw128_off(int row, int j) { return (uint32_t)(row * 128 + ((j ^ (row & 7)) << 4)); }

// p: the residue plane (prime-major, then product of the batch); pr: its prime.
struct TileCoord {
  int p, pr, m, n;
};
__device__ __forceinline__ TileCoord tile_coord(int t, int mt, int nt, int batch) {
  int per = mt * nt;
  TileCoord c;
  c.p = t / per;
  c.pr = c.p / batch;
  int r = t - c.p * per;
  c.n = r / mt;  // consecutive CTAs share a B column block
  c.m = r - c.n * mt;
  return c;
}

// After tcgen05.wait::ld: ties the loaded registers to this point, so that no
// use of them is scheduled before the wait.
__device__ __forceinline__ void pin32(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}


// 32 accumulator columns (from col) of this thread's row: mode 0 writes the
// partial residues back to tensor memory for the next chunk; modes 1 and 2
// write residue bytes to the staging halves, mode 2 adding the bytes the
// carry chunk left there when add_carry is set.
__device__ __forceinline__ void reduce32(uint32_t (&r)[32], uint32_t taddr_col, int col, int row, int mode,
                                         bool add_carry, float q, float iq, uint8_t* out_base) {
  if (mode == 0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(partial_residue(__uint_as_float(r[i]), q, iq));
    tmem_st32(taddr_col, r);
    return;
  }
  const int half = col >> 7;
  const int j0 = (col & 127) >> 4;
  uint8_t* hbase = out_base + half * OUT_HALF;
  uint4* p0 = reinterpret_cast<uint4*>(hbase + sw128_off(row, j0));
  uint4* p1 = reinterpret_cast<uint4*>(hbase + sw128_off(row, j0 + 1));
  uint32_t carry[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (add_carry) {
    const uint4 c0 = *p0, c1 = *p1;
    carry[0] = c0.x; carry[1] = c0.y; carry[2] = c0.z; carry[3] = c0.w;
    carry[4] = c1.x; carry[5] = c1.y; carry[6] = c1.z; carry[7] = c1.w;
  }
  uint32_t packed[8];
  final_residues(r, carry, add_carry, q, iq, packed);
  *p0 = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  *p1 = make_uint4(packed[4], packed[5], packed[6], packed[7]);
}

// This thread's 128 accumulator columns from col_begin, 32 at a time.
__device__ __forceinline__ void drain128(uint32_t taddr, int col_begin, int row, int mode, bool add_carry, float q,
                                         float iq, uint8_t* out_base) {
#pragma unroll 1
  for (int col = col_begin; col < col_begin + 128; col += 32) {
    uint32_t r[32];
    tmem_ld32(taddr + col, r);
    tmem_wait_ld();
    pin32(r);
    reduce32(r, taddr + col, col, row, mode, add_carry, q, iq, out_base);
  }
}

// Split-K: when there are too few tiles for the persistent CTAs, K is cut
// into S slices of whole 1024-K chunks; a unit is one tile of one slice, and
// each unit's residues go to its slice's planes of RC (summed mod q by
// slice_sum_kernel afterwards).  S minimises the time in chunk units:
// (waves of units) x (chunks per unit), plus, for S > 1, the summing pass (a
// launch, about half a chunk, and S slices of one byte per output, about
// tiles / 512 chunks per slice at HBM rate).  Every CTA derives the same S,
// the smallest on ties, and CTA 0 records it in the plan.
struct Unit {
  TileCoord tc;
  int s, kb_lo, kb_hi, nc;  // slice, k-block range, 1024-K chunks
};

struct Splits {
  int S, kbs;  // slices and k-blocks per slice
};

__device__ __forceinline__ Splits choose_splits(const GemmParams& gp, int tiles, int workers, DevPlan* plan) {
  const int nkc = (gp.kb_total + KC_BLOCKS - 1) / KC_BLOCKS;
  int best = 1;
  long long best_cost = -1;
  for (int S = 1; S <= gp.max_splits && S <= nkc; ++S) {
    const int cps = (nkc + S - 1) / S;
    if ((nkc + cps - 1) / cps != S) continue;  // a slice would be empty
    const long long waves = ((long long)tiles * S + workers - 1) / workers;
    const long long cost = waves * cps * 512 + (S > 1 ? 256 + (long long)S * tiles : 0);  // in 1/512 chunk
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) plan->splits = best;
  return Splits{best, (nkc + best - 1) / best * KC_BLOCKS};
}

// The launch's prime count and K slicing, read from the plan by thread 0 and
// passed on through shared memory (sh, three ints): all threads of every CTA
// reading the plan's line at once would queue thousands of L2 requests on it.
// Ends with a block barrier.
__device__ __forceinline__ void read_plan_once(const GemmParams& gp, DevPlan* plan, int tiles_per_prime, int workers,
                                               int* sh, int& P, Splits& sp) {
  if (threadIdx.x == 0) {
    const int p = launch_primes(gp, plan);
    const Splits s = p ? choose_splits(gp, p * tiles_per_prime, workers, plan) : Splits{1, gp.kb_total};
    sh[0] = p;
    sh[1] = s.S;
    sh[2] = s.kbs;
  }
  __syncthreads();
  P = sh[0];
  sp = Splits{sh[1], sh[2]};
}

__device__ __forceinline__ Unit unit_of(int u, int tiles, int mt, int nt, int batch, const Splits& sp, int kb_total) {
  Unit r;
  r.s = u / tiles;
  r.tc = tile_coord(u - r.s * tiles, mt, nt, batch);
  r.kb_lo = r.s * sp.kbs;
  r.kb_hi = min(r.kb_lo + sp.kbs, kb_total);
  r.nc = (r.kb_hi - r.kb_lo + KC_BLOCKS - 1) / KC_BLOCKS;
  return r;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// B_KMAJOR: residues of B arrive as [N][K] (a transposed operand) instead of
// [K][N]; the tiles are then staged like A's and read as a K-major operand.
template <bool B_KMAJOR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    residue_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ GemmParams gp,
                        DevPlan* plan) {
  extern __shared__ uint8_t smem_raw[];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* out_base = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_base + OUT_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* ep_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);  // two ints

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl ctl{abort_flag, &plan->status, &plan->timeout_where, gp.wait_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), EPI_WARPS);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"((uint32_t)TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Everything above uses only this CTA's shared and tensor memory and so
  // overlaps the predecessor's tail; the plan is read after the wait.  A call
  // that has already failed (P = 0) gets no units and goes to the teardown.
  wait_for_predecessor();
  __shared__ int s_plan[3];
  int P;
  Splits sp;
  read_plan_once(gp, plan, gp.batch * gp.mt * gp.nt, (int)gridDim.x, s_plan, P, sp);
  const int tiles = P * gp.batch * gp.mt * gp.nt;
  const int total = P ? tiles * sp.S : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool issued[STAGES] = {};
      uint32_t issued_phase[STAGES] = {};
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Unit u = unit_of(t, tiles, gp.mt, gp.nt, gp.batch, sp, gp.kb_total);
        const TileCoord& tc = u.tc;
        for (int kb = u.kb_lo; kb < u.kb_hi; ++kb) {
          if (!wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, ctl, 1)) {
            ok = false;
            break;
          }
          uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          uint32_t a_dst = smem_u32(stage_base + stage * STAGE_BYTES);
          uint32_t b_dst = a_dst + A_BYTES;
          tma_load_3d(a_dst, &tmA, fb, kb * BK, tc.m * BM, tc.p);
          if constexpr (B_KMAJOR) {
            tma_load_3d(b_dst, &tmB, fb, kb * BK, tc.n * BN, tc.p);  // BN rows of 64 K
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_3d(b_dst + j * B_SLAB, &tmB, fb, tc.n * BN + 64 * j, kb * BK, tc.p);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let issued copies land before the block exits
        Ctl drain_ctl = ctl;
        volatile int never = 0;
        drain_ctl.abort = &never;
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) wait_bounded(smem_u32(&full[s]), issued_phase[s], drain_ctl, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_iter = 0;
      bool ok = true, any = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Unit u = unit_of(t, tiles, gp.mt, gp.nt, gp.batch, sp, gp.kb_total);
        for (int c = 0; c < u.nc && ok; ++c) {
          const uint32_t b = acc_iter & 1u, aph = (acc_iter >> 1) & 1u;
          if (!wait_bounded(smem_u32(&tempty[b]), aph ^ 1u, ctl, 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + b * BN;
          const int kb0 = u.kb_lo + c * KC_BLOCKS;
          const int kb1 = min(kb0 + KC_BLOCKS, u.kb_hi);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_bounded(smem_u32(&full[stage]), phase, ctl, 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(stage_base + stage * STAGE_BYTES);
            const uint64_t adesc = sw128_desc(a_addr, 16, 1024);
            const uint64_t bdesc = B_KMAJOR ? sw128_desc(a_addr + A_BYTES, 16, 1024)
                                            : sw128_desc(a_addr + A_BYTES, B_SLAB, 1024);
            constexpr uint32_t b_step = B_KMAJOR ? 2 : 128;  // 16 K: 32 bytes along a row, or 16 rows of 128 bytes
            constexpr uint32_t idesc = B_KMAJOR ? (IDESC & ~(1u << 16)) : IDESC;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint32_t acc = (c >= 2 || kb > kb0 || kk > 0) ? 1u : 0u;
              umma_f16(d, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(b_step * kk), idesc, acc);
            }
            any = true;
            umma_commit(smem_u32(&empty[stage]));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (!(gp.fault == 1 && acc_iter == 0)) umma_commit(smem_u32(&tfull[b]));
          ++acc_iter;
        }
      }
      if (!ok && any) {  // all issued MMAs must finish before the memory is freed
        Ctl drain_ctl = ctl;
        volatile int never = 0;
        drain_ctl.abort = &never;
        umma_commit(smem_u32(drain));
        wait_bounded(smem_u32(drain), 0, drain_ctl, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;  // tensor-memory lane quarter this warp may access
    const int row = q4 * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..255
    const int col_begin = (et >> 7) * (BN / 2);  // this warpgroup's half of the columns
    uint32_t acc_iter = 0;
    bool ok = true;
    const uint32_t out_s = smem_u32(out_base);
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Unit u = unit_of(t, tiles, gp.mt, gp.nt, gp.batch, sp, gp.kb_total);
      const TileCoord& tc = u.tc;
      const int nc_tile = u.nc;
      const int out_plane = u.s * gp.planes + tc.p;
      const float q = gp.qf[tc.pr], iq = gp.invq[tc.pr];
      bool first_write = true;
      for (int c = 0; c < nc_tile; ++c) {
        const uint32_t b = acc_iter & 1u, aph = (acc_iter >> 1) & 1u;
        // One thread waits (bounded) and publishes the outcome, so all 128
        // threads take the same branch; the flag is double-buffered because a
        // thread can reach the next chunk's wait before the others read it.
        if (et == 0) ep_flag[acc_iter & 1u] = wait_bounded(smem_u32(&tfull[b]), aph, ctl, 4) ? 1 : 0;
        epilogue_bar();
        if (!ep_flag[acc_iter & 1u]) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q4 * 32) << 16) + b * BN;
        const int mode = (c + 2 < nc_tile) ? 0 : (c + 2 == nc_tile ? 1 : 2);  // partial, carry, final
        if (mode != 0 && first_write) {
          if (et == 0) bulk_wait_read0();  // the previous tile's store has read the staging
          epilogue_bar();
          first_write = false;
        }
        drain128(taddr, col_begin, row, mode, mode == 2 && nc_tile >= 2, q, iq, out_base);
        if (mode == 0) tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty[b]));
        if (mode == 2) {
          fence_proxy_async_smem();
          epilogue_bar();
          if (et == 0) {
            tma_store_3d(&tmC, out_s, tc.n * BN, tc.m * BM, out_plane);
            if (tc.n * BN + 128 < gp.N) tma_store_3d(&tmC, out_s + OUT_HALF, tc.n * BN + 128, tc.m * BM, out_plane);
            bulk_commit();
          }
        }
        ++acc_iter;
      }
    }
    if (et == 0) bulk_wait0();
  }

  // the role branches leave single lanes working while the rest of their warp
  // runs ahead: reconverge every warp, so that the block barrier below sees
  // whole warps and the memory is freed only after the last tensor-memory read
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  allow_dependents();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)TMEM_COLS));
  }
}

// ---------------------------------------------------------------------------
// The CTA-pair kernel (tcgen05 cta_group::2)
//
// Two CTAs of a cluster share one 256 x 256 tile: each holds 128 rows of A and
// 128 columns of B per stage (32 KB, six stages), the first CTA of the pair
// issues M = 256, N = 256 MMAs that read both CTAs' shared memory, and each
// CTA's tensor memory receives its own 128 rows of the accumulator.  Per
// multiply-add the pair moves a third fewer operand bytes from L2 than two
// single-CTA tiles, and the deeper pipeline hides more load latency.
// Protocol: both CTAs' TMA loads complete on the first CTA's "full" barrier
// (64 KB per stage); the first CTA's MMA commits multicast to both CTAs'
// "empty" and "tfull" barriers; both epilogues arrive on the first CTA's
// "tempty" barrier (8 warps).  The epilogue is the single-CTA one.
// ---------------------------------------------------------------------------
constexpr int STAGES2 = 6;
constexpr int B2_BYTES = 128 * BK * 2;  // this CTA's 128 columns of B
constexpr int STAGE2_BYTES = A_BYTES + B2_BYTES;
constexpr int SMEM2_BYTES = 1024 + STAGES2 * STAGE2_BYTES + OUT_BYTES + BAR_BYTES;
static_assert(SMEM2_BYTES <= 232448, "shared memory");
// M = 256, N = 256, otherwise as IDESC.
constexpr uint32_t IDESC2 = (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (1u << 16) | ((uint32_t)(256 >> 3) << 17) |
                            ((uint32_t)(256 >> 4) << 24);

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster_addr,
                                                 int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void umma_f16_pair(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive on the barrier at this shared offset in both CTAs of the pair once
// all earlier MMAs of this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Bounded wait with cluster-scope acquire (barriers that receive arrivals from
// the peer CTA or from its copies).
__device__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, const Ctl& ctl, int where) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*ctl.abort) return false;
      if (globaltimer() - t0 > ctl.limit_ns) {
        *ctl.abort = 1;
        atomicCAS(ctl.status, 0, RG_ERR_TIMEOUT);
        atomicCAS(ctl.where, 0, where);
        return false;
      }
    }
  }
}

template <bool B_KMAJOR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    residue_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const __grid_constant__ GemmParams gp,
                             DevPlan* plan) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t rank = cluster_rank();
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* out_base = smem + STAGES2 * STAGE2_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_base + OUT_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES2;
  uint64_t* tfull = bars + 2 * STAGES2;
  uint64_t* tempty = bars + 2 * STAGES2 + 2;
  uint64_t* drain = bars + 2 * STAGES2 + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES2 + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* ep_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);  // two ints

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl ctl{abort_flag, &plan->status, &plan->timeout_where, gp.wait_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 2 * EPI_WARPS);  // the epilogue warps of both CTAs
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
  }
  if (warp == 1) {  // one warp in each CTA allocates for the pair
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"((uint32_t)TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // As in the single-CTA kernel: the setup above overlaps the predecessor's
  // tail, and a failed call (P = 0, the same in both CTAs) gets no units.
  wait_for_predecessor();
  const int mt2 = (gp.M + 255) / 256;
  __shared__ int s_plan[3];
  int P;
  Splits sp;
  read_plan_once(gp, plan, gp.batch * mt2 * gp.nt, (int)(gridDim.x >> 1), s_plan, P, sp);
  const int tiles = P * gp.batch * mt2 * gp.nt;
  const int total = P ? tiles * sp.S : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        const Unit u = unit_of(t, tiles, mt2, gp.nt, gp.batch, sp, gp.kb_total);
        const TileCoord& tc = u.tc;
        for (int kb = u.kb_lo; kb < u.kb_hi; ++kb) {
          if (!wait_bounded_cluster(smem_u32(&empty[stage]), phase ^ 1u, ctl, 11)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = smem_u32(&full[stage]);
          if (rank == 0) mbar_arrive_expect_tx(fb_local, 2 * STAGE2_BYTES);
          const uint32_t fb = mapa_shared(fb_local, 0);
          const uint32_t a_dst = smem_u32(stage_base + stage * STAGE2_BYTES);
          const uint32_t b_dst = a_dst + A_BYTES;
          tma_load_3d_pair(a_dst, &tmA, fb, kb * BK, tc.m * 256 + (int)rank * 128, tc.p);
          if constexpr (B_KMAJOR) {
            tma_load_3d_pair(b_dst, &tmB, fb, kb * BK, tc.n * BN + (int)rank * 128, tc.p);  // 128 rows of 64 K
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_3d_pair(b_dst + j * B_SLAB, &tmB, fb, tc.n * BN + (int)rank * 128 + 64 * j, kb * BK, tc.p);
          }
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (first CTA)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_iter = 0;
      bool ok = true, any = false;
      for (int t = cid; t < total && ok; t += ncl) {
        const Unit u = unit_of(t, tiles, mt2, gp.nt, gp.batch, sp, gp.kb_total);
        for (int c = 0; c < u.nc && ok; ++c) {
          const uint32_t b = acc_iter & 1u, aph = (acc_iter >> 1) & 1u;
          if (!wait_bounded_cluster(smem_u32(&tempty[b]), aph ^ 1u, ctl, 12)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + b * BN;
          const int kb0 = u.kb_lo + c * KC_BLOCKS;
          const int kb1 = min(kb0 + KC_BLOCKS, u.kb_hi);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_bounded_cluster(smem_u32(&full[stage]), phase, ctl, 13)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(stage_base + stage * STAGE2_BYTES);
            const uint64_t adesc = sw128_desc(a_addr, 16, 1024);
            const uint64_t bdesc = B_KMAJOR ? sw128_desc(a_addr + A_BYTES, 16, 1024)
                                            : sw128_desc(a_addr + A_BYTES, B_SLAB, 1024);
            constexpr uint32_t b_step = B_KMAJOR ? 2 : 128;
            constexpr uint32_t idesc = B_KMAJOR ? (IDESC2 & ~(1u << 16)) : IDESC2;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint32_t acc = (c >= 2 || kb > kb0 || kk > 0) ? 1u : 0u;
              umma_f16_pair(d, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(b_step * kk), idesc, acc);
            }
            any = true;
            umma_commit_pair(smem_u32(&empty[stage]));
            if (++stage == STAGES2) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (!(gp.fault == 1 && acc_iter == 0)) umma_commit_pair(smem_u32(&tfull[b]));
          ++acc_iter;
        }
      }
      if (!ok && any) {  // all issued MMAs must finish before the memory is freed
        Ctl drain_ctl = ctl;
        volatile int never = 0;
        drain_ctl.abort = &never;
        umma_commit_pair_local(smem_u32(drain));
        wait_bounded(smem_u32(drain), 0, drain_ctl, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..255
    const int col_begin = (et >> 7) * (BN / 2);  // this warpgroup's half of the columns
    uint32_t acc_iter = 0;
    bool ok = true;
    const uint32_t out_s = smem_u32(out_base);
    const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty[0]), 0), mapa_shared(smem_u32(&tempty[1]), 0)};
    for (int t = cid; t < total && ok; t += ncl) {
      const Unit u = unit_of(t, tiles, mt2, gp.nt, gp.batch, sp, gp.kb_total);
      const TileCoord& tc = u.tc;
      const int nc_tile = u.nc;
      const int out_plane = u.s * gp.planes + tc.p;
      const float q = gp.qf[tc.pr], iq = gp.invq[tc.pr];
      const int row0 = tc.m * 256 + (int)rank * 128;
      bool first_write = true;
      for (int c = 0; c < nc_tile; ++c) {
        const uint32_t b = acc_iter & 1u, aph = (acc_iter >> 1) & 1u;
        if (et == 0) ep_flag[acc_iter & 1u] = wait_bounded_cluster(smem_u32(&tfull[b]), aph, ctl, 14) ? 1 : 0;
        epilogue_bar();
        if (!ep_flag[acc_iter & 1u]) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q4 * 32) << 16) + b * BN;
        const int mode = (c + 2 < nc_tile) ? 0 : (c + 2 == nc_tile ? 1 : 2);  // partial, carry, final
        if (mode != 0 && first_write) {
          if (et == 0) bulk_wait_read0();
          epilogue_bar();
          first_write = false;
        }
        drain128(taddr, col_begin, row, mode, mode == 2 && nc_tile >= 2, q, iq, out_base);
        if (mode == 0) tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader[b]);
        if (mode == 2) {
          fence_proxy_async_smem();
          epilogue_bar();
          if (et == 0 && row0 < gp.M) {
            tma_store_3d(&tmC, out_s, tc.n * BN, row0, out_plane);
            if (tc.n * BN + 128 < gp.N) tma_store_3d(&tmC, out_s + OUT_HALF, tc.n * BN + 128, row0, out_plane);
            bulk_commit();
          }
        }
        ++acc_iter;
      }
    }
    if (et == 0) bulk_wait0();
  }

  __syncwarp();  // whole warps again before the abort check and the barriers below
  if (*abort_flag) {
    // an aborted role may leave copies in flight that signal either CTA:
    // give them time to land before the pair leaves
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 200000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  allow_dependents();
  cluster_sync();  // neither CTA frees the pair's memory while the other still uses it
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)TMEM_COLS));
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult qr;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  (void)esize;
  CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Sums the K slices of the product residues into slice 0:
// RC[0][p] = (RC[0][p] + ... + RC[S-1][p]) mod q, q the prime of plane p, for
// the planes of the primes in use.  16 bytes per thread and slice; the bytes
// are summed in 16-bit lanes (S <= 16 residues of at most 250 each).
struct PrimeQ {
  int q[kNumPrimes];
};

__global__ void __launch_bounds__(256) slice_sum_kernel(uint8_t* __restrict__ RC, long long slice_bytes,
                                                        long long plane_bytes, int batch, PrimeQ qs,
                                                        const DevPlan* plan) {
  wait_for_predecessor();
  if (plan->status) return;
  const int S = plan->splits;
  if (S <= 1) return;
  const long long n16 = (long long)plan->P * batch * plane_bytes / 16;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x) {
    const long long off = i * 16;
    const int q = qs.q[(int)(off / plane_bytes) / batch];
    uint32_t even[4] = {0, 0, 0, 0}, odd[4] = {0, 0, 0, 0};
    for (int sl = 0; sl < S; ++sl) {
      const uint4 v = *reinterpret_cast<const uint4*>(RC + sl * slice_bytes + off);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        even[k] += w[k] & 0x00FF00FFu;
        odd[k] += (w[k] >> 8) & 0x00FF00FFu;
      }
    }
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t b0 = (even[k] & 0xFFFFu) % q, b2 = (even[k] >> 16) % q;
      const uint32_t b1 = (odd[k] & 0xFFFFu) % q, b3 = (odd[k] >> 16) % q;
      out[k] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
    *reinterpret_cast<uint4*>(RC + off) = make_uint4(out[0], out[1], out[2], out[3]);
  }
  allow_dependents();
}

std::atomic<int> g_gemm_variant{0};  // 0 automatic, 1 single-CTA, 2 CTA pair

// Per device, set up once under a lock: the kernels' shared-memory limits, the
// SM count and how many CTA pairs can be resident at once.
struct GemmDevice {
  int sms = 0, max_pairs = 0;
};

cudaError_t gemm_device(int dev, GemmDevice& out) {
  static std::mutex mu;
  static GemmDevice devs[64];
  std::lock_guard<std::mutex> lock(mu);
  GemmDevice& d = devs[dev];
  if (!d.sms) {
    for (auto k : {residue_gemm_kernel<false>, residue_gemm_kernel<true>}) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (e != cudaSuccess) return e;
    }
    for (auto k : {residue_gemm_pair_kernel<false>, residue_gemm_pair_kernel<true>}) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM2_BYTES);
      if (e != cudaSuccess) return e;
    }
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (sms < 2) return cudaErrorInvalidDevice;
    // not every SM can be paired within its GPC
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM2_BYTES;
    cfg.gridDim = dim3((unsigned)(sms & ~1));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, residue_gemm_pair_kernel<false>, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();  // the query's own failure is not the call's
      n = sms / 2;
    }
    d.max_pairs = n;
    d.sms = sms;
  }
  out = d;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm(const void* RA, long long lda, const void* RB, long long ldb, void* RC, long long ldc,
                        int pmax, int batch, int P_fixed, long long M, long long N, long long K, DevPlan* plan,
                        cudaStream_t st, int fault, unsigned long long wait_ns, bool derive_i64, bool b_kmajor,
                        int max_splits, uint32_t* plane_hint) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  GemmDevice gd;
  e = gemm_device(dev, gd);
  if (e != cudaSuccess) return e;
  // the pair kernel loads A in 128-row halves of a 256-row tile
  const int variant = g_gemm_variant.load();
  const bool pair = variant == 2 || (variant == 0 && M > BM);
  CUtensorMap ma, mb, mc;
  const uint64_t planes = (uint64_t)pmax * (uint64_t)batch;
  if (!make_map_3d(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, RA, (uint64_t)K, (uint64_t)M, planes,
                   (uint64_t)lda * 2, (uint64_t)M * lda * 2, BK, BM) ||
      !(b_kmajor ? make_map_3d(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, RB, (uint64_t)K, (uint64_t)N, planes,
                               (uint64_t)ldb * 2, (uint64_t)N * ldb * 2, BK, pair ? 128 : BN)
                 : make_map_3d(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, RB, (uint64_t)N, (uint64_t)K, planes,
                               (uint64_t)ldb * 2, (uint64_t)K * ldb * 2, 64, BK)) ||
      !make_map_3d(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, RC, (uint64_t)N, (uint64_t)M,
                   planes * (uint64_t)max_splits, (uint64_t)ldc,
                   (uint64_t)M * ldc, 128, 128))
    return cudaErrorInvalidValue;
  GemmParams gp;
  gp.M = (int)M;
  gp.N = (int)N;
  gp.K = (int)K;
  gp.mt = (int)((M + BM - 1) / BM);
  gp.nt = (int)((N + BN - 1) / BN);
  gp.kb_total = (int)((K + BK - 1) / BK);
  gp.batch = batch;
  gp.planes = (int)planes;
  gp.max_splits = max_splits;
  gp.P_fixed = P_fixed;
  gp.derive_i64 = derive_i64 ? 1 : 0;
  gp.ceil_log2_k = 0;
  while ((1LL << gp.ceil_log2_k) < K) ++gp.ceil_log2_k;
  gp.fault = fault;
  gp.wait_ns = wait_ns;
  gp.plane_hint = derive_i64 ? plane_hint : nullptr;
  const Tables& t = host_tables();
  for (int i = 0; i < kNumPrimes; ++i) {
    gp.qf[i] = t.qf[i];
    gp.invq[i] = t.invq[i];
  }
  for (int i = 0; i <= kNumPrimes; ++i) gp.log2P[i] = t.log2P[i];
  auto slice_sum = [&]() -> cudaError_t {
    if (max_splits <= 1) return cudaSuccess;
    PrimeQ qs;
    for (int i = 0; i < kNumPrimes; ++i) qs.q[i] = t.q[i];
    const long long plane_bytes = M * ldc, n16 = (long long)planes * plane_bytes / 16;
    long long blocks = (n16 + 255) / 256;
    if (blocks > 4LL * gd.sms) blocks = 4LL * gd.sms;
    return launch_dependent(slice_sum_kernel, dim3((unsigned)(blocks < 1 ? 1 : blocks)), dim3(256), 0, st,
                            static_cast<uint8_t*>(RC), (long long)planes * plane_bytes, plane_bytes, batch, qs,
                            (const DevPlan*)plan);
  };
  if (!pair) {
    const long long tiles = (long long)planes * gp.mt * gp.nt * max_splits;
    int grid = (int)(tiles < gd.sms ? tiles : gd.sms);
    if (grid < 1) grid = 1;
    e = b_kmajor ? launch_dependent(residue_gemm_kernel<true>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, st, ma, mb,
                                    mc, gp, plan)
                 : launch_dependent(residue_gemm_kernel<false>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, st, ma, mb,
                                    mc, gp, plan);
    return e != cudaSuccess ? e : slice_sum();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM2_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // persistent: as many pairs as can be resident at once, never more than
  // there are tiles
  const long long tiles2 = (long long)planes * ((M + 255) / 256) * gp.nt * max_splits;
  long long clusters = gd.max_pairs;
  if (tiles2 < clusters) clusters = tiles2;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  e = b_kmajor ? cudaLaunchKernelEx(&cfg, residue_gemm_pair_kernel<true>, ma, mb, mc, gp, plan)
               : cudaLaunchKernelEx(&cfg, residue_gemm_pair_kernel<false>, ma, mb, mc, gp, plan);
  return e != cudaSuccess ? e : slice_sum();
}

int gemm_max_splits(long long gemm_batch, long long M, long long N, long long K) {
  const long long nkc = (K + (long long)KC_BLOCKS * BK - 1) / ((long long)KC_BLOCKS * BK);
  // tiles with a single prime, of the larger (CTA-pair) kind; 160 bounds the
  // persistent workers of any launch on this part
  const long long tiles = gemm_batch * ((M + 255) / 256) * ((N + BN - 1) / BN);
  long long want = (160 + tiles - 1) / tiles;
  if (want > kMaxSplits) want = kMaxSplits;
  if (want > nkc) want = nkc;
  return (int)(want < 1 ? 1 : want);
}

}  // namespace rg

extern "C" int rg_set_gemm_variant(int variant) {
  if (variant < 0 || variant > 2) return -1;
  return rg::g_gemm_variant.exchange(variant);
}
