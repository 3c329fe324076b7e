// rate_probe.cu -- peak-rate probes of the tensor-core instructions this GPU
// offers for the per-prime residue product.
//
//   RG_PROBE_MMA_S8        mma.sync.aligned.m16n8k32 s8 x s8 -> s32, the
//                          warp-level INT8 MMA: the only integer tensor-core
//                          instruction sm_103a accepts (tcgen05.mma has no
//                          integer kind on this target).
//   RG_PROBE_TCGEN05_F16   tcgen05.mma kind::f16 (fp16 operands, fp32
//                          accumulator in tensor memory): the instruction the
//                          residue GEMM runs on.
//   RG_PROBE_TCGEN05_E4M3  tcgen05.mma kind::f8f6f4 with E4M3 operands: the
//                          instruction an FP8 digit split of the residues
//                          would use (page "Accelerating Multiple-Precision LU
//                          Decomposition with Ozaki Scheme II", FP8 balanced
//                          base-17 encoding).
//   RG_PROBE_MMA_F16       mma.sync.aligned.m16n8k16 f16 x f16 -> f32, the
//                          warp-level fp16 MMA (the exact solve's elimination
//                          update could hold its residues in either type).
//   RG_PROBE_TCGEN05_F16_BMN, _PAIR, _PAIR_BMN, _PAIR_BMN_SYNC: kind::f16 in
//                          the forms the residue GEMM uses: B MN-major, the
//                          CTA-pair instruction (cta_group::2, M = 256), and
//                          the pair's issue loop (a wait on a completed
//                          barrier and a commit every four MMAs).
//
// Not part of the product path.  The INT8 rate is the denominator of the
// "% of INT8 tensor-core roofline" reported for the per-prime GEMM; the
// f16/E4M3 pair decides whether the digit split could beat one fp16 product.
// Each launch runs a fixed number of independent MMAs on operands held in
// registers or shared memory, with no global-memory traffic; the caller times
// it with events on its stream.  Operand values are arbitrary finite numbers;
// the results are folded into one word so that no MMA is optimised away.
#include <cuda_runtime.h>

#include <cstdint>

#include "rg_common.cuh"

namespace {
using rg::DevPlan;

constexpr int kProbeThreadsSync = 256;  // eight warps per block
constexpr int kSyncChains = 8;          // independent accumulators per warp

__global__ void __launch_bounds__(kProbeThreadsSync) probe_mma_s8_kernel(int iters, int* sink) {
  const uint32_t h = (blockIdx.x * kProbeThreadsSync + threadIdx.x) * 2654435761u;
  uint32_t a[4], b[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = h ^ (0x9E3779B9u * (uint32_t)(i + 1));
#pragma unroll
  for (int i = 0; i < 2; ++i) b[i] = h ^ (0x85EBCA6Bu * (uint32_t)(i + 5));
  int c[kSyncChains][4];
#pragma unroll
  for (int j = 0; j < kSyncChains; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < kSyncChains; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < kSyncChains; ++j) s ^= c[j][0] ^ c[j][1] ^ c[j][2] ^ c[j][3];
  atomicXor(sink, s);
}

// The same loop with mma.sync m16n8k16 fp16 x fp16 -> fp32 (operands 1.0).
__global__ void __launch_bounds__(kProbeThreadsSync) probe_mma_f16_kernel(int iters, int* sink) {
  const uint32_t one2 = 0x3C003C00u;  // two fp16 ones
  float c[kSyncChains][4];
#pragma unroll
  for (int j = 0; j < kSyncChains; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.0f;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < kSyncChains; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
          : "r"(one2), "r"(one2), "r"(one2), "r"(one2), "r"(one2), "r"(one2));
  }
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < kSyncChains; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  atomicXor(sink, __float_as_int(s) + (int)(blockIdx.x * kProbeThreadsSync + threadIdx.x));
}

// ---------------------------------------------------------------------------
// tcgen05: one CTA per SM, A 128 x 128 bytes and B 256 x 128 bytes in shared
// memory (both K-major, 128-byte swizzle), D 128 x 256 fp32 in tensor memory.
// One thread issues `iters` rounds of four MMAs (each consumes 32 bytes of K
// per row: 16 fp16 or 32 E4M3 values), then waits for them (bounded).
// ---------------------------------------------------------------------------
constexpr int kTcM = 128, kTcN = 256;
constexpr int kTcA = kTcM * 128, kTcB = kTcN * 128;
constexpr int kTcSmem = 120 * 1024;  // more than half the SM's shared memory: one CTA per SM
// instruction descriptor: D fp32, A and B format 0 (fp16 for kind::f16, E4M3
// for kind::f8f6f4), both K-major, N and M
constexpr uint32_t kTcIdesc = (1u << 4) | ((uint32_t)(kTcN >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t probe_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused with a 128-byte swizzle, K-major)
  d |= (uint64_t)((1024 >> 4) & 0x3FFFu) << 32;  // eight rows of 128 bytes
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ bool probe_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long probe_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ bool probe_wait(uint32_t bar, unsigned long long limit_ns) {
  const unsigned long long t0 = probe_now();
  for (uint32_t i = 0;; ++i) {
    if (probe_try_wait(bar, 0)) return true;
    if ((i & 63u) == 63u && probe_now() - t0 > limit_ns) return false;
  }
}

template <int KIND>
__device__ __forceinline__ void probe_umma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
  if constexpr (KIND == 0)
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d),
        "l"(a), "l"(b), "r"(kTcIdesc), "r"(acc)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d),
        "l"(a), "l"(b), "r"(kTcIdesc), "r"(acc)
        : "memory");
}

template <int KIND>
__device__ __forceinline__ void probe_umma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  static_assert(KIND == 0, "the pair probe runs kind::f16");
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void probe_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// KIND 0: kind::f16, 1: kind::f8f6f4 (E4M3).  BMN: B is read MN-major (64-column
// slabs 8 KB apart, as the residue GEMM stages an N-major B).  PAIR: clusters
// of two CTAs, the first issuing cta_group::2 MMAs with M = 256 (each CTA
// holds 128 rows of A and 128 columns of B).  SYNC: every round also waits on
// an already completed barrier and commits to another, as the GEMM's issue
// loop does per k-block.
template <int KIND, bool BMN = false, bool PAIR = false, bool SYNC = false>
__global__ void __launch_bounds__(128, 1) probe_tcgen05_kernel(int iters, unsigned long long limit_ns, DevPlan* plan) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* words = reinterpret_cast<uint32_t*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kTcA + kTcB);
  uint64_t* bar_ready = bar + 1;  // SYNC: completed once at set-up
  uint64_t* bar_commit = bar + 2;  // SYNC: receives a commit every round
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 3);
  uint32_t rank = 0;
  if constexpr (PAIR) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  // finite operand values: fp16 pairs in +-[1, 2), or E4M3 bytes with the
  // exponent's low bit clear (never the all-ones exponent and mantissa of NaN)
  for (int i = threadIdx.x; i < (kTcA + kTcB) / 4; i += blockDim.x) {
    const uint32_t h = (uint32_t)(i + 1) * 2654435761u ^ blockIdx.x;
    words[i] = KIND == 0 ? ((h & 0x83FF83FFu) | 0x3C003C00u) : (h & 0xF7F7F7F7u);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(bar)) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(bar_ready)) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(bar_commit)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar_ready)) : "memory");  // phase 0 done
  }
  if (threadIdx.x < 32) {  // one warp of each CTA allocates (for the pair, jointly)
    if constexpr (PAIR) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                   "r"((uint32_t)kTcN));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                   "r"((uint32_t)kTcN));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if constexpr (PAIR) probe_cluster_sync();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0 && rank == 0) {
    const uint64_t a = probe_desc(su32(smem));
    // B: K-major rows (32 bytes per K step), or MN-major 64-column slabs 8 KB
    // apart (16 K rows = 2048 bytes per K step)
    const uint64_t b = BMN ? ((probe_desc(su32(smem + kTcA)) & ~(0x3FFFull << 16)) | ((uint64_t)(8192 >> 4) << 16))
                           : probe_desc(su32(smem + kTcA));
    constexpr uint32_t b_step = BMN ? 128 : 2;
    constexpr uint32_t idesc =
        (kTcIdesc & ~(0x1Fu << 24)) | ((uint32_t)((PAIR ? 2 * kTcM : kTcM) >> 4) << 24) | (BMN ? (1u << 16) : 0u);
    for (int it = 0; it < iters; ++it) {
      if constexpr (SYNC) {
        if (!probe_try_wait(su32(bar_ready), 0)) atomicCAS(&plan->status, 0, RG_ERR_TIMEOUT);  // never: phase 0 done
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if constexpr (PAIR)
          probe_umma_pair<KIND>(tmem, a + 2 * kk, b + b_step * kk, idesc, (it | kk) ? 1u : 0u);
        else
          probe_umma<KIND>(tmem, a + 2 * kk, b + b_step * kk, (it | kk) ? 1u : 0u);
      }
      if constexpr (SYNC) {
        if constexpr (PAIR)
          asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           su32(bar_commit))
                       : "memory");
        else
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           su32(bar_commit))
                       : "memory");
      }
    }
    if constexpr (PAIR)
      asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                   : "memory");
    else
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                   : "memory");
    if (!probe_wait(su32(bar), limit_ns)) {
      atomicCAS(&plan->status, 0, RG_ERR_TIMEOUT);
      probe_wait(su32(bar), limit_ns);  // the issued MMAs must end before the memory is freed
    }
  }
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if constexpr (PAIR) probe_cluster_sync();  // the first CTA's MMAs read both CTAs' memory
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)kTcN));
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)kTcN));
  }
}

template <typename K>
cudaError_t launch_probe(K kernel, int blocks, bool pair, cudaStream_t s, int iters, unsigned long long limit_ns,
                         DevPlan* plan) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, iters, limit_ns, plan);
}

}  // namespace

extern "C" int rg_probe_mma_rate(int kind, int blocks, int iters, void* ws, size_t ws_bytes, void* stream,
                                 double* ops_per_launch) {
  if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u) || iters < 1 || iters > (1 << 24) ||
      blocks < 0 || blocks > 65536 || !ops_per_launch)
    return RG_ERR_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return RG_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevPlan* plan = static_cast<DevPlan*>(ws);
  if (cudaMemsetAsync(plan, 0, 256, s) != cudaSuccess) return RG_ERR_CUDA;
  const unsigned long long limit_ns = 5000000000ull;
  switch (kind) {
    case RG_PROBE_MMA_S8: {
      const int nb = blocks ? blocks : 4 * sms;
      probe_mma_s8_kernel<<<nb, kProbeThreadsSync, 0, s>>>(iters, &plan->pad0[0]);
      *ops_per_launch = 2.0 * nb * (kProbeThreadsSync / 32) * (double)iters * kSyncChains * (16.0 * 8.0 * 32.0);
      break;
    }
    case RG_PROBE_MMA_F16: {
      const int nb = blocks ? blocks : 4 * sms;
      probe_mma_f16_kernel<<<nb, kProbeThreadsSync, 0, s>>>(iters, &plan->pad0[0]);
      *ops_per_launch = 2.0 * nb * (kProbeThreadsSync / 32) * (double)iters * kSyncChains * (16.0 * 8.0 * 16.0);
      break;
    }
    case RG_PROBE_TCGEN05_F16:
    case RG_PROBE_TCGEN05_E4M3:
    case RG_PROBE_TCGEN05_F16_BMN:
    case RG_PROBE_TCGEN05_F16_PAIR:
    case RG_PROBE_TCGEN05_F16_PAIR_BMN:
    case RG_PROBE_TCGEN05_F16_PAIR_BMN_SYNC: {
      const bool pair = kind >= RG_PROBE_TCGEN05_F16_PAIR;
      const int nb = blocks ? blocks : (pair ? (sms & ~1) : sms);
      if (pair && (nb & 1)) return RG_ERR_ARG;
      cudaError_t e;
      switch (kind) {
        case RG_PROBE_TCGEN05_F16: e = launch_probe(probe_tcgen05_kernel<0>, nb, false, s, iters, limit_ns, plan); break;
        case RG_PROBE_TCGEN05_E4M3: e = launch_probe(probe_tcgen05_kernel<1>, nb, false, s, iters, limit_ns, plan); break;
        case RG_PROBE_TCGEN05_F16_BMN:
          e = launch_probe(probe_tcgen05_kernel<0, true>, nb, false, s, iters, limit_ns, plan);
          break;
        case RG_PROBE_TCGEN05_F16_PAIR:
          e = launch_probe(probe_tcgen05_kernel<0, false, true>, nb, true, s, iters, limit_ns, plan);
          break;
        case RG_PROBE_TCGEN05_F16_PAIR_BMN:
          e = launch_probe(probe_tcgen05_kernel<0, true, true>, nb, true, s, iters, limit_ns, plan);
          break;
        default:
          e = launch_probe(probe_tcgen05_kernel<0, true, true, true>, nb, true, s, iters, limit_ns, plan);
          break;
      }
      if (e != cudaSuccess) return RG_ERR_CUDA;
      // per CTA and round: four MMAs of 128 rows (a pair's M = 256 instruction covers both CTAs' rows)
      *ops_per_launch = 2.0 * nb * (double)iters * 4 * kTcM * kTcN * (kind == RG_PROBE_TCGEN05_E4M3 ? 32.0 : 16.0);
      break;
    }
    default:
      return RG_ERR_ARG;
  }
  return cudaGetLastError() == cudaSuccess ? RG_OK : RG_ERR_CUDA;
}
