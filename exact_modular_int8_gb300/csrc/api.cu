// api.cu -- the C ABI (include/resgemm.h): validation, workspace layout and
// the launch sequence planner -> split -> per-prime GEMM -> Garner.
//
// The sequence keeps the data path free of host synchronisation: the planner
// reductions, the prime count and the scale exponents all live in the
// workspace's plan block, and every kernel reads them there.  Only
// RG_FLAG_SYNC / RG_FLAG_HOST calls, rg_status() and rg_get_plan() wait for the
// device.
#include <atomic>
#include <climits>
#include <mutex>
#include <cstdint>
#include <cstring>

#include "rg_kernels.h"

namespace {
using namespace rg;

constexpr size_t kPlanBytes = 4096;
// One residue plane of A and B (fp16) from which the int64 split writes the
// previous call's plane count instead of the most an int64 product can need:
// below it the saved writes are worth less than the fix-up pass's launch.
constexpr size_t kPlaneHintMinBytes = size_t(16) << 20;
constexpr size_t kAlign = 4096;

std::atomic<unsigned long long> g_wait_ns{1000000000ull};
std::atomic<int> g_fault{0};
// Stage timing events (rg_set_stage_events): recorded on the call's stream
// before the first kernel, before the GEMM, after the GEMM and after Garner.
std::mutex g_ev_mu;
cudaEvent_t g_ev[4] = {nullptr, nullptr, nullptr, nullptr};
bool g_ev_on = false;

cudaError_t record_stage(int i, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_ev_mu);
  return g_ev_on ? cudaEventRecord(g_ev[i], s) : cudaSuccess;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }

int ceil_log2(long long k) {
  int c = 0;
  while ((1LL << c) < k) ++c;
  return c;
}

int primes_for_bound_host(int T) {
  const Tables& t = host_tables();
  for (int n = 1; n <= kNumPrimes; ++n)
    if (t.log2P[n] >= T + 1) return n;
  return kNumPrimes;
}

// Largest prime count a call can need when it plans on the device.
int pmax_for(int op, long long K, int la, int lb, int nprimes) {
  if (nprimes > 0) return nprimes;
  int ck = ceil_log2(K);
  switch (op) {
    case RG_OP_I64:
      // K * max|A| * max|B| <= 2^63 - 1 bounds bits_a + bits_b + ceil(log2 K) by 65.
      return primes_for_bound_host(65);
    case RG_OP_LIMBS: {
      int T = 64 * la + 64 * lb + ck;
      return primes_for_bound_host(T < RG_MAX_BOUND_BITS ? T : RG_MAX_BOUND_BITS);
    }
    default:
      return kNumPrimes;
  }
}

struct Layout {
  size_t plan, ra, rb, rc, a, b, c, c2, total;
  long long lda, ldb, ldc;
  int pmax, splits;  // splits: K slices RC has room for
};

bool is_interval(int op) { return op == RG_OP_INTERVAL || op == RG_OP_INTERVAL_F32; }
// operations with two outputs (lo, hi)
bool is_enclose(int op) { return op == RG_OP_ENCLOSE || op == RG_OP_ENCLOSE_F32 || is_interval(op); }
// residue planes per product and prime: intervals need three products
int planes_per_product(int op) { return is_interval(op) ? 3 : 1; }
// arrays per operand: an interval operand is a midpoint and a radius array
int arrays_per_operand(int op) { return is_interval(op) ? 2 : 1; }

// Bytes of one operand or output entry: limbs of int64, one int64, one double or one float.
size_t elem_bytes(int op, int limbs) {
  return op == RG_OP_LIMBS ? 8 * (size_t)limbs : (op == RG_OP_ENCLOSE_F32 || op == RG_OP_INTERVAL_F32) ? 4 : 8;
}

// An empty problem (batch, M, N or K zero) needs only the plan block.
bool is_empty(long long batch, long long M, long long N, long long K) { return !batch || !M || !N || !K; }

bool make_layout(int op, long long batch, long long M, long long N, long long K, int la, int lb, int lc, int nprimes,
                 unsigned flags, Layout* L) {
  if (batch < 0 || M < 0 || N < 0 || K < 0) return false;
  if (nprimes < 0 || nprimes > kNumPrimes) return false;
  if (op == RG_OP_LIMBS && (la < 1 || la > RG_MAX_LIMBS_IN || lb < 1 || lb > RG_MAX_LIMBS_IN || lc < 1 ||
                            lc > RG_MAX_LIMBS_OUT))
    return false;
  if (op != RG_OP_LIMBS) la = lb = lc = 1;
  // shapes the kernels index in 32 bits (rows, columns, products) and the
  // longest exact-sum K; with these and the tile bound below, every size in
  // the layout stays below 2^61
  if (M > INT32_MAX || N > INT32_MAX || batch > INT32_MAX || K > RG_MAX_K) return false;
  std::memset(L, 0, sizeof(*L));
  const bool transb = (flags & RG_FLAG_TRANS_B) != 0;
  L->lda = round_up(K, 8);
  L->ldb = transb ? round_up(K, 8) : round_up(N, 64);
  L->ldc = round_up(N, 16);
  L->plan = 0;
  size_t off = kPlanBytes;
  if (op == RG_OP_STAGE || is_empty(batch, M, N, K)) {
    L->total = off;
    L->pmax = nprimes;
    return true;
  }
  int pmax = pmax_for(op, K, la, lb, nprimes);
  // the persistent GEMM numbers its tiles (plane, row block, column block)
  // in int: at most 2^31 - 1 of the single-CTA kind (the larger count)
  const __int128 tiles = (__int128)pmax * planes_per_product(op) * batch * ((M + 127) / 128) * ((N + 255) / 256);
  if (tiles > INT32_MAX) return false;
  L->pmax = pmax;
  const size_t planes = (size_t)pmax * planes_per_product(op) * batch;
  L->splits = gemm_max_splits((long long)planes_per_product(op) * batch, M, N, K);
  L->ra = off;
  off = align_up(off + planes * M * L->lda * 2, kAlign);
  L->rb = off;
  off = align_up(off + planes * (transb ? N : K) * L->ldb * 2, kAlign);
  L->rc = off;
  off = align_up(off + planes * M * L->ldc * L->splits, kAlign);
  if (flags & RG_FLAG_HOST) {
    size_t ea = elem_bytes(op, la), eb = elem_bytes(op, lb), ec = elem_bytes(op, lc);
    const size_t arrays = arrays_per_operand(op);
    L->a = off;
    off = align_up(off + arrays * batch * M * K * ea, kAlign);
    L->b = off;
    off = align_up(off + arrays * batch * K * N * eb, kAlign);
    L->c = off;
    off = align_up(off + (size_t)batch * M * N * ec, kAlign);
    if (is_enclose(op)) {
      L->c2 = off;
      off = align_up(off + (size_t)batch * M * N * ec, kAlign);
    }
  }
  L->total = off;
  return true;
}

// A pinned host word per thread and device for the final status read (a
// copy into pageable memory is staged by the driver and takes longer).
int* status_word() {
  thread_local int* words[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!words[dev]) {
    void* p = nullptr;
    if (cudaHostAlloc(&p, sizeof(int), cudaHostAllocDefault) != cudaSuccess) return nullptr;
    words[dev] = static_cast<int*>(p);
  }
  return words[dev];
}

// The status word of the call: read into `host_word` when the caller gives
// one (any host int, pinned or not), else into this thread's pinned word.
int finish(void* ws, cudaStream_t s, unsigned flags, int* host_word = nullptr) {
  if (!(flags & (RG_FLAG_SYNC | RG_FLAG_HOST))) return RG_OK;
  int fallback = 0;
  int* st = host_word ? host_word : status_word();
  if (!st) st = &fallback;
  DevPlan* plan = static_cast<DevPlan*>(ws);
  if (cudaMemcpyAsync(st, &plan->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return RG_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RG_ERR_CUDA;
  return *st;
}

#define RG_TRY(x)                          \
  do {                                     \
    cudaError_t e_ = (x);                  \
    if (e_ != cudaSuccess) return RG_ERR_CUDA; \
  } while (0)

// ---------------------------------------------------------------------------
// Host-buffer int64 products large enough for the CPU-GPU link to dominate:
// A is copied in row blocks on a copy stream while the blocks already on the
// device are split, multiplied and reconstructed on the call's stream, and
// every block of C goes back on a second copy stream as soon as it is done
// (copies in opposite directions share the link).  B is copied and split
// once; each A block reuses one block-sized region of residue planes.
// ---------------------------------------------------------------------------
constexpr int kPipeMaxBlocks = 8;
constexpr size_t kPipeMinBytes = size_t(32) << 20;  // operands and result; below this one block wins

struct HostPipe {
  std::mutex mu;  // one pipelined call per device at a time (the copy streams and events are shared)
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, b = nullptr, done = nullptr, a[kPipeMaxBlocks] = {}, c[kPipeMaxBlocks] = {};
};
HostPipe g_pipe[64];
std::mutex g_pipe_init_mu;

// The copy streams and events of the current device, created on first use.
HostPipe* host_pipe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  HostPipe& p = g_pipe[dev];
  std::lock_guard<std::mutex> lk(g_pipe_init_mu);
  if (!p.ready) {
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.b, ef) == cudaSuccess && cudaEventCreateWithFlags(&p.done, ef) == cudaSuccess;
    for (int j = 0; ok && j < kPipeMaxBlocks; ++j)
      ok = cudaEventCreateWithFlags(&p.a[j], ef) == cudaSuccess && cudaEventCreateWithFlags(&p.c[j], ef) == cudaSuccess;
    if (!ok) return nullptr;  // the call fails; a later call retries the creation
    p.ready = true;
  }
  return &p;
}

// Row blocks of a pipelined host-buffer int64 call: at least two, one per
// 1024 rows up to kPipeMaxBlocks, whole 256-row pair tiles each; false when
// the problem is too small to gain from the overlap.
bool pipeline_shape(long long M, long long N, long long K, int* nb, long long* mb) {
  const unsigned __int128 bytes = ((unsigned __int128)M * K + (unsigned __int128)K * N + (unsigned __int128)M * N) * 8;
  if (M < 512 || bytes < kPipeMinBytes) return false;
  long long n = M / 1024;
  n = n < 2 ? 2 : (n > kPipeMaxBlocks ? kPipeMaxBlocks : n);
  const long long rows = ((M + n - 1) / n + 255) / 256 * 256;
  if (rows >= M) return false;
  *mb = rows;
  *nb = (int)((M + rows - 1) / rows);
  return *nb >= 2 && *nb <= kPipeMaxBlocks;
}

// The pipelined host-buffer int64 call (see HostPipe); the workspace is the
// host layout `L` (staging for A, B and C, residue planes for all M rows, of
// which one block's rows are used).
int run_i64_host_pipelined(const void* A, const void* B, void* C, long long M, long long N, long long K, int nprimes,
                           unsigned flags, const Layout& L, uint8_t* w, cudaStream_t s, int nb, long long mb) {
  HostPipe* hp = host_pipe();
  if (!hp) return RG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(hp->mu);
  const bool transb = (flags & RG_FLAG_TRANS_B) != 0;
  DevPlan* plan = reinterpret_cast<DevPlan*>(w + L.plan);
  int64_t* dA = reinterpret_cast<int64_t*>(w + L.a);
  int64_t* dB = reinterpret_cast<int64_t*>(w + L.b);
  int64_t* dC = reinterpret_cast<int64_t*>(w + L.c);
  const int64_t* hA = static_cast<const int64_t*>(A);
  int64_t* hC = static_cast<int64_t*>(C);
  RG_TRY(upload_tables());
  RG_TRY(cudaMemsetAsync(plan, 0, sizeof(DevPlan), s));
  // the copies start once the call's stream has reached this call
  RG_TRY(cudaEventRecord(hp->start, s));
  RG_TRY(cudaStreamWaitEvent(hp->h2d, hp->start, 0));
  RG_TRY(cudaStreamWaitEvent(hp->d2h, hp->start, 0));
  RG_TRY(cudaMemcpyAsync(dB, B, (size_t)K * N * 8, cudaMemcpyHostToDevice, hp->h2d));
  RG_TRY(cudaEventRecord(hp->b, hp->h2d));
  for (int j = 0; j < nb; ++j) {
    const long long m0 = j * mb, mj = M - m0 < mb ? M - m0 : mb;
    RG_TRY(cudaMemcpyAsync(dA + m0 * K, hA + m0 * K, (size_t)mj * K * 8, cudaMemcpyHostToDevice, hp->h2d));
    RG_TRY(cudaEventRecord(hp->a[j], hp->h2d));
  }
  RG_TRY(cudaStreamWaitEvent(s, hp->b, 0));
  int fault = g_fault.exchange(0);
  for (int j = 0; j < nb; ++j) {
    const long long m0 = j * mb, mj = M - m0 < mb ? M - m0 : mb;
    RG_TRY(cudaStreamWaitEvent(s, hp->a[j], 0));
    // the first block's split also takes B (and max |B|); the GEMM of every
    // block derives its prime count from the reductions so far, and Garner
    // reads that count, so each block is exact on its own
    RG_TRY(launch_split(RG_OP_I64, dA + m0 * K, nullptr, j == 0 ? dB : nullptr, nullptr, 1, 1, 1, mj, N, K, L.lda,
                        L.ldb, w + L.ra, w + L.rb, plan, L.pmax, transb, s));
    RG_TRY(launch_gemm(w + L.ra, L.lda, w + L.rb, L.ldb, w + L.rc, L.ldc, L.pmax, 1, nprimes, mj, N, K, plan, s,
                       j == 0 ? fault : 0, g_wait_ns.load(), true, transb, L.splits));
    RG_TRY(launch_garner(RG_OP_I64, w + L.rc, L.ldc, mj * L.ldc, mj * L.ldc, mj, N, K, 1, L.pmax, plan, dC + m0 * N,
                         nullptr, s));
    RG_TRY(cudaEventRecord(hp->c[j], s));
  }
  // results go back after all the work is enqueued (a copy into pageable
  // memory returns only when it is done)
  for (int j = 0; j < nb; ++j) {
    const long long m0 = j * mb, mj = M - m0 < mb ? M - m0 : mb;
    RG_TRY(cudaStreamWaitEvent(hp->d2h, hp->c[j], 0));
    RG_TRY(cudaMemcpyAsync(hC + m0 * N, dC + m0 * N, (size_t)mj * N * 8, cudaMemcpyDeviceToHost, hp->d2h));
  }
  RG_TRY(cudaEventRecord(hp->done, hp->d2h));
  RG_TRY(cudaStreamWaitEvent(s, hp->done, 0));
  return finish(w, s, flags);
}

bool stage_events_on() {
  std::lock_guard<std::mutex> lk(g_ev_mu);
  return g_ev_on;
}

// Shared driver for every entry point; `batch` products of the same shape
// share one plan (one prime count, one pair of scale exponents).  A2 and B2
// are the radii of interval operands (null otherwise).  `status_host`, if
// given, is the host int the final status read lands in (see finish()).
// `pipeline`: large host-buffer int64 products may take the pipelined path
// (which creates copy streams and events on first use).
int run(int op, const void* A, const void* A2, int la, const void* B, const void* B2, int lb, void* C, void* C2,
        int lc, long long batch, long long M, long long N, long long K, int nprimes, unsigned flags, void* ws,
        size_t ws_bytes, void* stream, int* status_host = nullptr, bool pipeline = true) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return RG_ERR_ARG;
  if (batch < 0 || M < 0 || N < 0 || K < 0 || nprimes < 0 || nprimes > kNumPrimes) return RG_ERR_ARG;
  // an empty problem reads no operand, and writes outputs only if it has entries
  const bool empty = is_empty(batch, M, N, K), has_out = batch && M && N;
  if ((!empty && (!A || !B || (is_interval(op) && (!A2 || !B2)))) || (has_out && (!C || (is_enclose(op) && !C2))))
    return RG_ERR_ARG;
  if (op == RG_OP_LIMBS &&
      (la < 1 || la > RG_MAX_LIMBS_IN || lb < 1 || lb > RG_MAX_LIMBS_IN || lc < 1 || lc > RG_MAX_LIMBS_OUT))
    return RG_ERR_ARG;
  if (K > RG_MAX_K) return RG_ERR_RANGE;
  if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || batch > (1LL << 31) - 1) return RG_ERR_ARG;
  Layout L;
  if (!make_layout(op, batch, M, N, K, la, lb, lc, nprimes, flags, &L)) return RG_ERR_ARG;
  if (ws_bytes < L.total) {
    // floating point: a smaller workspace holds planes for fewer primes, and
    // the plan coarsens the scaling to fit them (reported as not lossless)
    if (!is_enclose(op) || empty) return RG_ERR_WORKSPACE;
    int p = L.pmax - 1;
    for (; p >= 1; --p) {
      Layout Lp;
      if (make_layout(op, batch, M, N, K, la, lb, lc, p, flags, &Lp) && Lp.total <= ws_bytes) {
        L = Lp;
        break;
      }
    }
    if (p < 1) return RG_ERR_WORKSPACE;
  }
  const long long gemm_batch = batch * planes_per_product(op);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  DevPlan* plan = reinterpret_cast<DevPlan*>(w + L.plan);
  const size_t ea = elem_bytes(op, la), eb = elem_bytes(op, lb), ec = elem_bytes(op, lc);
  const size_t out_bytes = (size_t)batch * M * N * ec;
  if (empty) {
    // Nothing to multiply; an empty sum is exactly zero (lo = hi = +0).
    RG_TRY(cudaMemsetAsync(plan, 0, sizeof(DevPlan), s));
    if (out_bytes) {
      if (flags & RG_FLAG_HOST) {
        std::memset(C, 0, out_bytes);
        if (is_enclose(op)) std::memset(C2, 0, out_bytes);
      } else {
        RG_TRY(cudaMemsetAsync(C, 0, out_bytes, s));
        if (is_enclose(op)) RG_TRY(cudaMemsetAsync(C2, 0, out_bytes, s));
      }
    }
    return finish(ws, s, flags, status_host);
  }
  if (pipeline && op == RG_OP_I64 && batch == 1 && (flags & RG_FLAG_HOST) && !stage_events_on()) {
    int nb = 0;
    long long mb = 0;
    if (pipeline_shape(M, N, K, &nb, &mb))
      return run_i64_host_pipelined(A, B, C, M, N, K, nprimes, flags, L, w, s, nb, mb);
  }
  RG_TRY(upload_tables());
  const void* dA = A;
  const void* dA2 = A2;
  const void* dB = B;
  const void* dB2 = B2;
  void* dC = C;
  void* dC2 = C2;
  // Host buffers are copied through the workspace.  (Kernels reading and
  // writing pinned host memory in place over the CPU-GPU link were measured
  // slower than these copies plus HBM-resident kernels.)
  if (flags & RG_FLAG_HOST) {
    const size_t na = (size_t)batch * M * K * ea, nb = (size_t)batch * K * N * eb;
    dA = w + L.a;
    dB = w + L.b;
    dC = w + L.c;
    dC2 = is_enclose(op) ? static_cast<void*>(w + L.c2) : nullptr;
    RG_TRY(cudaMemcpyAsync(const_cast<void*>(dA), A, na, cudaMemcpyHostToDevice, s));
    RG_TRY(cudaMemcpyAsync(const_cast<void*>(dB), B, nb, cudaMemcpyHostToDevice, s));
    if (is_interval(op)) {  // radii right after the midpoints
      dA2 = w + L.a + na;
      dB2 = w + L.b + nb;
      RG_TRY(cudaMemcpyAsync(const_cast<void*>(dA2), A2, na, cudaMemcpyHostToDevice, s));
      RG_TRY(cudaMemcpyAsync(const_cast<void*>(dB2), B2, nb, cudaMemcpyHostToDevice, s));
    }
  }
  RG_TRY(cudaMemsetAsync(plan, 0, sizeof(DevPlan), s));
  const int la1 = op == RG_OP_LIMBS ? la : 1, lb1 = op == RG_OP_LIMBS ? lb : 1, lc1 = op == RG_OP_LIMBS ? lc : 1;
  // int64: the split reduces max |A|, max |B| itself and the GEMM derives the
  // plan; the other operations run the planner kernel first
  const bool i64 = op == RG_OP_I64;
  RG_TRY(record_stage(0, s));
  if (!i64)
    RG_TRY(launch_plan(op, dA, dA2, batch * M * K, la1, dB, dB2, batch * K * N, lb1, lc1, K,
                       is_enclose(op) ? 0 : nprimes, L.pmax, plan, s));
  const bool transb = (flags & RG_FLAG_TRANS_B) != 0;
  // planner-free int64 with large planes: the split writes as many planes as
  // the previous call on this workspace used, and a fix-up pass adds any that
  // this call needs beyond them (see kPlaneHintOffset)
  uint32_t* plane_hint = reinterpret_cast<uint32_t*>(w + L.plan + kPlaneHintOffset);
  const bool use_hint =
      i64 && nprimes == 0 && (unsigned __int128)batch * (M + N) * K * 2 >= (unsigned __int128)kPlaneHintMinBytes;
  RG_TRY(launch_split(op, dA, dA2, dB, dB2, la1, lb1, batch, M, N, K, L.lda, L.ldb, w + L.ra, w + L.rb, plan, L.pmax,
                      transb, s, use_hint ? plane_hint : nullptr));
  int fault = g_fault.exchange(0);
  RG_TRY(record_stage(1, s));
  RG_TRY(launch_gemm(w + L.ra, L.lda, w + L.rb, L.ldb, w + L.rc, L.ldc, L.pmax, (int)gemm_batch, i64 ? nprimes : 0,
                     M, N, K, plan, s, fault, g_wait_ns.load(), i64, transb, L.splits, i64 ? plane_hint : nullptr));
  // Garner sees the batch as batch * M rows of each plane; an interval's
  // three product planes lie batch * M rows apart
  const long long sub = batch * M * L.ldc;
  RG_TRY(record_stage(2, s));
  RG_TRY(launch_garner(op, w + L.rc, L.ldc, planes_per_product(op) * sub, sub, batch * M, N, K,
                       op == RG_OP_LIMBS ? lc : 1, L.pmax, plan, dC, dC2, s));
  RG_TRY(record_stage(3, s));
  if (flags & RG_FLAG_HOST) {
    RG_TRY(cudaMemcpyAsync(C, dC, out_bytes, cudaMemcpyDeviceToHost, s));
    if (is_enclose(op)) RG_TRY(cudaMemcpyAsync(C2, dC2, out_bytes, cudaMemcpyDeviceToHost, s));
  }
  return finish(ws, s, flags, status_host);
}

}  // namespace

extern "C" {

int res_gemm_i64(const int64_t* A, const int64_t* B, int64_t* C, int64_t M, int64_t N, int64_t K, int nprimes,
                 unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return run(RG_OP_I64, A, nullptr, 1, B, nullptr, 1, C, nullptr, 1, 1, M, N, K, nprimes, flags, ws, ws_bytes, stream);
}

int res_gemm_limbs(const int64_t* A, int la, const int64_t* B, int lb, int64_t* C, int lc, int64_t M, int64_t N,
                   int64_t K, int nprimes, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return run(RG_OP_LIMBS, A, nullptr, la, B, nullptr, lb, C, nullptr, lc, 1, M, N, K, nprimes,
             flags, ws, ws_bytes, stream);
}

int enclose_gemm_f64(const double* A, const double* B, double* lo, double* hi, int64_t M, int64_t N, int64_t K,
                     unsigned flags, int* info, void* ws, size_t ws_bytes, void* stream) {
  if (info) flags |= RG_FLAG_SYNC;  // the regime is known once the call has run
  const int rc = run(RG_OP_ENCLOSE, A, nullptr, 1, B, nullptr, 1, lo, hi, 1, 1, M, N, K, 0, flags, ws, ws_bytes, stream);
  if (rc != RG_OK || !info) return rc;
  int lossless = 1;
  if (M && N && K) {  // an empty product is exactly zero: lossless
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const DevPlan* plan = static_cast<const DevPlan*>(ws);
    if (cudaMemcpyAsync(&lossless, &plan->lossless, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return RG_ERR_CUDA;
  }
  *info = lossless ? 0 : 1;
  return RG_OK;
}

int enclose_gemm_f32(const float* A, const float* B, float* lo, float* hi, int64_t M, int64_t N, int64_t K,
                     unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return run(RG_OP_ENCLOSE_F32, A, nullptr, 1, B, nullptr, 1, lo, hi, 1, 1, M, N, K, 0, flags, ws, ws_bytes, stream);
}

int enclose_gemm_f32_batched(const float* A, const float* B, float* lo, float* hi, int64_t batch, int64_t M,
                             int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return run(RG_OP_ENCLOSE_F32, A, nullptr, 1, B, nullptr, 1, lo, hi, 1, batch, M, N, K, 0,
             flags, ws, ws_bytes, stream);
}

int interval_gemm_f64_batched(const double* Am, const double* Ar, const double* Bm, const double* Br, double* lo,
                              double* hi, int64_t batch, int64_t M, int64_t N, int64_t K, unsigned flags, void* ws,
                              size_t ws_bytes, void* stream) {
  return run(RG_OP_INTERVAL, Am, Ar, 1, Bm, Br, 1, lo, hi, 1, batch, M, N, K, 0, flags, ws, ws_bytes, stream);
}

int interval_gemm_f64(const double* Am, const double* Ar, const double* Bm, const double* Br, double* lo, double* hi,
                      int64_t M, int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return run(RG_OP_INTERVAL, Am, Ar, 1, Bm, Br, 1, lo, hi, 1, 1, M, N, K, 0, flags, ws, ws_bytes, stream);
}

int interval_gemm_f32_batched(const float* Am, const float* Ar, const float* Bm, const float* Br, float* lo,
                              float* hi, int64_t batch, int64_t M, int64_t N, int64_t K, unsigned flags, void* ws,
                              size_t ws_bytes, void* stream) {
  return run(RG_OP_INTERVAL_F32, Am, Ar, 1, Bm, Br, 1, lo, hi, 1, batch, M, N, K, 0, flags, ws, ws_bytes, stream);
}

int interval_gemm_f32(const float* Am, const float* Ar, const float* Bm, const float* Br, float* lo, float* hi,
                      int64_t M, int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return run(RG_OP_INTERVAL_F32, Am, Ar, 1, Bm, Br, 1, lo, hi, 1, 1, M, N, K, 0, flags, ws, ws_bytes, stream);
}

int res_gemm_i64_batched(const int64_t* A, const int64_t* B, int64_t* C, int64_t batch, int64_t M, int64_t N,
                         int64_t K, int nprimes, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return run(RG_OP_I64, A, nullptr, 1, B, nullptr, 1, C, nullptr, 1, batch, M, N, K, nprimes,
             flags, ws, ws_bytes, stream);
}

int res_gemm_limbs_batched(const int64_t* A, int la, const int64_t* B, int lb, int64_t* C, int lc, int64_t batch,
                           int64_t M, int64_t N, int64_t K, int nprimes, unsigned flags, void* ws, size_t ws_bytes,
                           void* stream) {
  return run(RG_OP_LIMBS, A, nullptr, la, B, nullptr, lb, C, nullptr, lc, batch, M, N, K, nprimes,
             flags, ws, ws_bytes, stream);
}

int enclose_gemm_f64_batched(const double* A, const double* B, double* lo, double* hi, int64_t batch, int64_t M,
                             int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return run(RG_OP_ENCLOSE, A, nullptr, 1, B, nullptr, 1, lo, hi, 1, batch, M, N, K, 0, flags, ws, ws_bytes, stream);
}

int res_gemm_stage(const uint16_t* RA, int64_t lda, const uint16_t* RB, int64_t ldb, uint8_t* RC, int64_t ldc,
                   int nprimes, int64_t M, int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!RA || !RB || !RC || !ws || (flags & RG_FLAG_HOST)) return RG_ERR_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || nprimes < 1 || nprimes > kNumPrimes) return RG_ERR_ARG;
  if (M > INT32_MAX || N > INT32_MAX) return RG_ERR_ARG;
  if ((__int128)nprimes * ((M + 127) / 128) * ((N + 255) / 256) > INT32_MAX) return RG_ERR_ARG;  // int tile numbers
  const bool transb = (flags & RG_FLAG_TRANS_B) != 0;
  if (lda < K || lda % 8 || ldc < N || ldc % 16) return RG_ERR_ARG;
  if (transb ? (ldb < K || ldb % 8) : (ldb < N || ldb % 64)) return RG_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(RA) | reinterpret_cast<uintptr_t>(RB) | reinterpret_cast<uintptr_t>(RC)) & 15u)
    return RG_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return RG_ERR_ARG;
  if (K > RG_MAX_K) return RG_ERR_RANGE;
  if (ws_bytes < kPlanBytes) return RG_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevPlan* plan = static_cast<DevPlan*>(ws);
  RG_TRY(cudaMemsetAsync(plan, 0, sizeof(DevPlan), s));
  int fault = g_fault.exchange(0);
  RG_TRY(launch_gemm(RA, lda, RB, ldb, RC, ldc, nprimes, 1, nprimes, M, N, K, plan, s, fault, g_wait_ns.load(), false,
                     transb, 1));
  return finish(ws, s, flags);
}

size_t rg_workspace_bytes_batched(int op, int64_t batch, int64_t M, int64_t N, int64_t K, int la, int lb, int lc,
                                  int nprimes, unsigned flags) {
  Layout L;
  if (op < RG_OP_I64 || op > RG_OP_INTERVAL_F32) return 0;
  if (!make_layout(op, batch, M, N, K, la, lb, lc, nprimes, flags, &L)) return 0;
  return L.total;
}

size_t rg_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int la, int lb, int lc, int nprimes,
                          unsigned flags) {
  return rg_workspace_bytes_batched(op, 1, M, N, K, la, lb, lc, nprimes, flags);
}

int rg_workspace_layout_batched(int op, int64_t batch, int64_t M, int64_t N, int64_t K, int la, int lb, int lc,
                                int nprimes, unsigned flags, rg_layout* out) {
  Layout L;
  if (!out || op < RG_OP_I64 || op > RG_OP_INTERVAL_F32) return RG_ERR_ARG;
  if (!make_layout(op, batch, M, N, K, la, lb, lc, nprimes, flags, &L)) return RG_ERR_ARG;
  out->ra = L.ra;
  out->rb = L.rb;
  out->rc = L.rc;
  out->lda = L.lda;
  out->ldb = L.ldb;
  out->ldc = L.ldc;
  out->pmax = L.pmax;
  out->splits = L.splits > 0 ? L.splits : 1;
  return RG_OK;
}

int rg_workspace_layout(int op, int64_t M, int64_t N, int64_t K, int la, int lb, int lc, int nprimes,
                        unsigned flags, rg_layout* out) {
  return rg_workspace_layout_batched(op, 1, M, N, K, la, lb, lc, nprimes, flags, out);
}

int rg_get_plan(const void* ws, void* stream, rg_plan_info* out) {
  if (!ws || !out) return RG_ERR_ARG;
  DevPlan p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&p, ws, sizeof(p), cudaMemcpyDeviceToHost, s) != cudaSuccess) return RG_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RG_ERR_CUDA;
  out->status = p.status;
  out->nprimes = p.P;
  out->bits_a = p.bits_a;
  out->bits_b = p.bits_b;
  out->bound_bits = p.bound_bits;
  out->f_a = p.f_a;
  out->f_b = p.f_b;
  out->lossless = p.lossless;
  out->splits = p.splits > 0 ? p.splits : 1;
  out->crt_rn = p.crt_rn;
  return RG_OK;
}

int rg_status(const void* ws, void* stream) {
  if (!ws) return RG_ERR_ARG;
  return finish(const_cast<void*>(ws), static_cast<cudaStream_t>(stream), RG_FLAG_SYNC);
}

const char* rg_strerror(int code) {
  switch (code) {
    case RG_OK: return "ok";
    case RG_ERR_ARG: return "invalid argument";
    case RG_ERR_RANGE: return "out of range: K > 2^17 or the product bound exceeds the primes or the output width";
    case RG_ERR_NONFINITE: return "an fp64 operand entry is inf or nan";
    case RG_ERR_LOSSY: return "fp64 operands do not scale losslessly into the 256-bit fixed point";
    case RG_ERR_WORKSPACE: return "workspace too small";
    case RG_ERR_CUDA: return "CUDA error";
    case RG_ERR_TIMEOUT: return "a bounded wait inside a kernel expired";
    case RG_ERR_RADIUS: return "an interval radius entry is negative";
    case RG_ERR_SINGULAR: return "the matrix is singular modulo every prime below 256";
    default: return "unknown status";
  }
}

uint64_t rg_set_wait_limit_ns(uint64_t ns) { return g_wait_ns.exchange(ns ? ns : 1000000000ull); }

void rg_inject_fault(int kind) { g_fault.store(kind); }

int rg_set_stage_events(void* const* events, int n) {
  if (n != 0 && (n != 4 || !events)) return RG_ERR_ARG;
  if (n == 4)
    for (int i = 0; i < 4; ++i)
      if (!events[i]) return RG_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_ev_mu);
  for (int i = 0; i < 4; ++i) g_ev[i] = n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  g_ev_on = n == 4;
  return RG_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of res_gemm_i64.
//
// Some callers cannot allocate device memory at call time: code running
// inside a host framework that owns every byte of device memory through its
// own arena, code on a latency-critical path where cudaMalloc's implicit
// device synchronisation is not allowed, and code whose only device memory
// is the buffers it was handed.  For them, res_gemm_i64_noalloc keeps its
// scratch (plan block and residue planes) in one fixed static device array.
// The array is part of this library's module: every GPU that loads the
// library holds it until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];  // device address of the array, per device

// The array's name is only a host-side stand-in; its device address is looked
// up once per device, with that device current.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return RG_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return RG_OK;
}

}  // namespace

extern "C" size_t rg_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int res_gemm_i64_noalloc(const int64_t* A, const int64_t* B, int64_t* C, int64_t M, int64_t N, int64_t K,
                                    int nprimes, unsigned flags, void* stream) {
  // the argument checks of res_gemm_i64, in its order, before the layout
  if (M < 0 || N < 0 || K < 0 || nprimes < 0 || nprimes > kNumPrimes) return RG_ERR_ARG;
  if ((M && N && K && (!A || !B)) || (M && N && !C)) return RG_ERR_ARG;
  if (K > RG_MAX_K) return RG_ERR_RANGE;
  Layout L;
  if (!make_layout(RG_OP_I64, 1, M, N, K, 1, 1, 1, nprimes, flags, &L)) return RG_ERR_ARG;
  if (L.total > kNoAllocScratchBytes) return RG_ERR_WORKSPACE;  // before any device work
  void* ws = nullptr;
  int rc = noalloc_scratch(&ws);
  if (rc != RG_OK) return rc;
  // the closing status read lands in this stack word: the pinned per-thread
  // word of the other entry points is allocated on first use
  int status = 0;
  return run(RG_OP_I64, A, nullptr, 1, B, nullptr, 1, C, nullptr, 1, 1, M, N, K, nprimes,
             flags, ws, kNoAllocScratchBytes, stream, &status, /*pipeline=*/false);
}
