// rg_kernels.h -- launchers of the library's kernels (internal, C++ linkage).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "rg_common.cuh"

namespace rg {

// Copies the constant tables to the current device once.
cudaError_t upload_tables();

// Planner reductions into plan (the host zeroes the plan block first).
cudaError_t launch_plan_i64(const int64_t* A, long long nA, const int64_t* B, long long nB, DevPlan* plan,
                            cudaStream_t s);
cudaError_t launch_plan_limbs(const int64_t* A, long long nA, int la, const int64_t* B, long long nB, int lb,
                              DevPlan* plan, cudaStream_t s);
cudaError_t launch_plan_f64(const double* A, long long nA, const double* B, long long nB, DevPlan* plan,
                            cudaStream_t s);

// Residue split of A [M][K] into RA [pmax][M][lda] and of B [K][N] into
// RB [pmax][K][ldb] (fp16 balanced residues); also finalises the plan.
cudaError_t launch_split(int op, const void* A, const void* B, int la, int lb, int lc, long long M, long long N,
                         long long K, long long lda, long long ldb, void* RA, void* RB, int nprimes_fixed,
                         DevPlan* plan, cudaStream_t st);

// Per-prime tensor-core product RC[p] = RA[p] * RB[p] mod q_p (uint8).
cudaError_t launch_gemm(const void* RA, long long lda, const void* RB, long long ldb, void* RC, long long ldc,
                        int pmax, int P_fixed, long long M, long long N, long long K, DevPlan* plan, cudaStream_t st,
                        int fault, unsigned long long wait_ns);

// Balanced Garner: RC [P][M][ldc] -> int64 limbs C [M][N][lc] (op I64/LIMBS),
// or the outward pair (lo, hi) as binary64 bit patterns (op ENCLOSE).
cudaError_t launch_garner(int op, const void* RC, long long ldc, long long plane, long long M, long long N, int lc,
                          DevPlan* plan, void* out0, void* out1, cudaStream_t st);

}  // namespace rg
