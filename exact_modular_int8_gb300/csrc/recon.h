// recon.h -- the exact solve's per-component big-integer stage on the GPU
// (internal, C++ linkage).  Little-endian 32-bit words throughout.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace rg {

// Tables shared by every component, on the device: the lift's modulus P
// (pw words), its powers P^i for i < m (P^i at pow_off[i], pow_len[i] words),
// PM = P^m (k words, its top word nonzero) and Barrett's constant
// MU = floor(2^(64 k) / PM) (k + 1 words).
struct ReconTables {
  const uint32_t* P;
  int pw;
  const uint32_t* pow;
  const int* pow_off;
  const int* pow_len;
  int m;
  const uint32_t* PM;
  const uint32_t* MU;
  int k;
};

// Device scratch (bytes) for `blocks` blocks of either kernel with a
// denominator of at most wD words.
size_t recon_scratch_bytes(const ReconTables& t, int wD, int blocks);

// The blocks both kernels launch with for `comps` components.
int recon_blocks(long long comps);

// Y[e] (k words) = sum_i z_i P^i for component e, where z_i are the balanced
// base-P digits digits[i][e][0..pw) (two's complement words, |x| < P/2)
// normalised into [0, P) by borrow propagation: Y[e] = X_e mod P^m in [0, P^m).
cudaError_t recon_values(const uint32_t* digits, long long comps, const ReconTables& t, uint32_t* Y,
                         uint32_t* scratch, cudaStream_t st);

// For every component: N = D Y[e] mod PM, balanced into (-PM/2, PM/2], as
// k + 2 two's complement words at N[e]; info[e] = the bit length of |N|
// when |N| <= 2^bound_bits, else -1.  D: wD words, 0 < D < PM.
cudaError_t recon_numerators(const uint32_t* Y, long long comps, const ReconTables& t, const uint32_t* D, int wD,
                             int bound_bits, uint32_t* N, int* info, uint32_t* scratch, cudaStream_t st);

}  // namespace rg
