// rg_kernels.h -- launchers of the library's kernels (internal, C++ linkage).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "rg_common.cuh"

namespace rg {

// Copies the constant tables to the current device once.
cudaError_t upload_tables();

// Planner: reductions over A and B into the plan block (the host zeroes it
// first); the last block derives the prime count, chunk counts and
// floating-point scales.  With nprimes_fixed > 0 only that derivation runs.
// A2, B2: the radii of interval operands (same sizes as A, B), else null.
// pcap: the most primes the workspace holds planes for; the floating-point
// plans coarsen their scaling to fit them (RG_ERR_WORKSPACE if not one bit per
// operand is left).
cudaError_t launch_plan(int op, const void* A, const void* A2, long long nA, int la, const void* B, const void* B2,
                        long long nB, int lb, int lc, long long K, int nprimes_fixed, int pcap, DevPlan* plan,
                        cudaStream_t s);

// Residue split of A [M][K] into RA [pmax][M][lda] and of B [K][N] into
// RB [pmax][K][ldb] (fp16 balanced residues), for the plan's prime count.
// For op I64 no planner runs first: the split writes i64_planes planes and
// reduces max |A|, max |B| into the plan; the GEMM derives the rest.
// transb: B is given transposed, [N][K], and RB becomes [pmax][N][ldb].
// batch: A and B hold `batch` products back to back ([batch][M][K] and
// [batch][K][N]); the residue planes become [pmax][batch][..][..].
// int64 only: B == nullptr splits A alone (B's residues already in RB; max |B|
// already in the plan).
// Intervals (A2, B2 the radii): three planes per prime and operand,
// RA [pmax][3][batch * M][lda] holding (Am, |Am|, Ar) and RB likewise
// (Bm, Br, |Bm| + Br).
// plane_hint (int64 only, may be null): the workspace's plane-count word; the
// split then writes only as many planes as the previous call used and a
// fix-up pass adds the planes this call needs beyond them.
cudaError_t launch_split(int op, const void* A, const void* A2, const void* B, const void* B2, int la, int lb,
                         long long batch, long long M, long long N, long long K, long long lda, long long ldb,
                         void* RA, void* RB, DevPlan* plan, int i64_planes, bool transb, cudaStream_t st,
                         const uint32_t* plane_hint = nullptr);

// Per-prime tensor-core product RC[p] = RA[p] * RB[p] mod q_p (uint8).
// derive_i64: the prime count is derived here from max |A|, max |B| (or
// taken from P_fixed), with the int64 range check, and written to the plan.
// b_kmajor: RB is [pmax][N][ldb] (K contiguous) instead of [pmax][K][ldb].
// batch: every prime's planes hold `batch` independent products
// (RA [pmax][batch][M][lda], RB and RC likewise).
// max_splits: RC has room for that many K slices ([max_splits][pmax * batch]
// [M][ldc]); the kernel may split K across them when there are too few tiles,
// and a second kernel then sums the slices into slice 0.
cudaError_t launch_gemm(const void* RA, long long lda, const void* RB, long long ldb, void* RC, long long ldc,
                        int pmax, int batch, int P_fixed, long long M, long long N, long long K, DevPlan* plan,
                        cudaStream_t st, int fault, unsigned long long wait_ns, bool derive_i64, bool b_kmajor,
                        int max_splits, uint32_t* plane_hint = nullptr);

// plane_hint (derive_i64 only, may be null): receives the prime count used,
// tagged, for the next call's split.
// K slices worth room in RC for a product of this shape (1: never split).
constexpr int kMaxSplits = 16;
int gemm_max_splits(long long gemm_batch, long long M, long long N, long long K);

// Balanced Garner: RC [P][M][ldc] -> int64 limbs C [M][N][lc] (op I64/LIMBS),
// or the outward pair (lo, hi) as IEEE bit patterns (ops ENCLOSE[_F32]).  For
// the interval ops RC holds three planes per prime, `sub` bytes apart: the
// midpoint and the two radius products.  pmax bounds the plan's prime count
// (the planes the workspace holds).
cudaError_t launch_garner(int op, const void* RC, long long ldc, long long plane, long long sub, long long M,
                          long long N, long long K, int lc, int pmax, DevPlan* plan, void* out0, void* out1,
                          cudaStream_t st);

}  // namespace rg
