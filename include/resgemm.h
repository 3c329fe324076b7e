/*
 * resgemm.h -- exact matrix products through residues modulo small primes,
 * for one GB300 (sm_103a) GPU.
 *
 * The method (pages "exact-solve" and "enclosure-gemm", section Method):
 * every integer operand entry is reduced to a balanced residue modulo each
 * of the odd primes below 256 that the bound needs; one tensor-core product
 * per prime yields the product matrix modulo that prime; balanced Garner
 * mixed-radix reconstruction then rebuilds every signed entry exactly.  For
 * binary64 operands, a power-of-two fixed-point scaling turns the operands
 * into integers first, and an integer-only epilogue rounds the exact product
 * outward once into an IEEE (lo, hi) pair.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Matrices are dense and row-major: A is [M][K], B is [K][N], outputs are
 *    [M][N].  Multi-limb integers keep their limbs innermost ([.][.][L]):
 *    little-endian 64-bit limbs, two's complement, signed top limb.
 *  - Pointers are device pointers, unless RG_FLAG_HOST is set; then A, B and
 *    the outputs are host pointers (pinned memory gives asynchronous
 *    copies) and the library stages them through the workspace.  A
 *    single (unbatched) res_gemm_i64 call with at least 512 rows and 32 MiB
 *    of operands and result moves A and C in row blocks on two copy streams
 *    of its own (created on a device's first such call), overlapping the
 *    link with the blocks' kernels; such calls on one device run one at a
 *    time.
 *  - The caller owns every buffer, including the workspace `ws` of
 *    `ws_bytes` bytes (device memory, 256-byte aligned), sized by
 *    rg_workspace_bytes().  The product entry points allocate no device
 *    memory.  Two exceptions elsewhere in the library: rg_solve_i64 takes
 *    its device buffers from cudaMallocAsync on its stream (and frees them
 *    there), and the module holds one fixed 64 MiB static device array, the
 *    scratch of res_gemm_i64_noalloc, on every GPU that loads it.
 *  - A synchronising call reads its closing status into a pinned host word
 *    that the library allocates (cudaHostAlloc) once per host thread and
 *    device, on that thread's first synchronising call;
 *    res_gemm_i64_noalloc reads it into a stack word instead.
 *  - All work is ordered on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  Without RG_FLAG_SYNC a call only enqueues work: it returns
 *    RG_OK once the arguments are accepted, and errors found on the device
 *    (range, non-finite operand, time-out) are read later with rg_status().
 *    With RG_FLAG_SYNC (implied by RG_FLAG_HOST) the call synchronises the
 *    stream and returns the device status.
 *  - On any error the outputs are unspecified.
 *  - Calls sharing one workspace must not overlap on the GPU; calls on
 *    different workspaces may run concurrently.
 */
#ifndef RESGEMM_H
#define RESGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define RG_OK 0
#define RG_ERR_ARG 1        /* null pointer, negative size, bad limb count, misaligned workspace */
#define RG_ERR_RANGE 2      /* K > 2^17, or the product bound exceeds the primes or the output width */
#define RG_ERR_NONFINITE 3  /* an fp64 operand entry is inf or nan */
#define RG_ERR_LOSSY 4      /* reserved: wide fp64 operands now get a valid, looser bracket (rg_get_plan) */
#define RG_ERR_WORKSPACE 5  /* workspace too small */
#define RG_ERR_CUDA 6       /* a CUDA runtime or driver call failed */
#define RG_ERR_TIMEOUT 7    /* a bounded wait inside a kernel expired; the kernel stopped early */
#define RG_ERR_RADIUS 8     /* an interval radius entry is negative */
#define RG_ERR_SINGULAR 9   /* rg_solve_i64: A is singular modulo every prime below 256 */

/* Flags. */
#define RG_FLAG_SYNC 1u /* synchronise the stream before returning; return the device status */
#define RG_FLAG_HOST 2u /* A, B and the outputs are host pointers; implies RG_FLAG_SYNC */
#define RG_FLAG_TRANS_B 4u /* B is given transposed: [N][K] (limbs [N][K][lb]); the product is A * B^T,
                              without a transposed copy ("enclosure-gemm", Usage: mm_enclose_nt) */

/* Operations, for rg_workspace_bytes() and rg_workspace_layout(). */
#define RG_OP_I64 0
#define RG_OP_LIMBS 1
#define RG_OP_ENCLOSE 2
#define RG_OP_STAGE 3
#define RG_OP_ENCLOSE_F32 4
#define RG_OP_INTERVAL 5
#define RG_OP_INTERVAL_F32 6

/* Limits. */
#define RG_MAX_K 131072 /* K <= 2^17 ("exact-solve" and "enclosure-gemm", Requirements and limits) */
#define RG_NUM_PRIMES 53 /* the odd primes 3..251 */
#define RG_MAX_BOUND_BITS 332 /* bits_a + bits_b + ceil(log2 K) <= 332 ("enclosure-gemm", Requirements) */
#define RG_MAX_LIMBS_IN 4 /* operands of up to 256 bits ("enclosure-gemm", Method: four int64 limbs) */
#define RG_MAX_LIMBS_OUT 6 /* results of up to 384 bits ("enclosure-gemm", Method: signed 384-bit arithmetic) */

/*
 * Exact C = A * B for int64 A [M][K] and B [K][N]; C is int64 [M][N].
 * ("exact-solve", Method: one product per prime below 256 on balanced
 * residues, balanced-Garner reconstruction.)
 *
 * nprimes = 0 plans on the device: it takes max |A|, max |B| and uses the
 * fewest primes (largest first) whose product P satisfies
 * P > 2^(bits_a + bits_b + ceil(log2 K) + 1), bits_x being the bit length of
 * max |x|.  nprimes in [1, 53] skips the planner: the caller then guarantees
 * |C| <= (P - 1) / 2 for the product P of the nprimes largest primes, and the
 * entries must fit in 64 bits, as they always do.
 * M, N or K = 0 is an empty problem: C (when it has entries) is set to 0
 * and no kernel runs; K = 0 gives the empty sum, exactly 0.
 * Errors: RG_ERR_ARG (negative sizes, null pointers, nprimes out of range),
 * RG_ERR_RANGE (K > 2^17; the exact bound K * max|A| * max|B| exceeds
 * 2^63 - 1, so C might not fit int64), RG_ERR_WORKSPACE, RG_ERR_CUDA,
 * RG_ERR_TIMEOUT.
 */
int res_gemm_i64(const int64_t* A, const int64_t* B, int64_t* C, int64_t M, int64_t N, int64_t K, int nprimes,
                 unsigned flags, void* ws, size_t ws_bytes, void* stream);

/*
 * Exact C = A * B for multi-limb operands: A [M][K][la], B [K][N][lb]
 * (1 <= la, lb <= 4), C [M][N][lc] (1 <= lc <= 6), limb layout as above.
 * ("enclosure-gemm", Method: integers of up to four int64 limbs, balanced
 * Garner digits in signed 384-bit arithmetic.)
 *
 * nprimes as for res_gemm_i64, with bits_x the bit length of the largest
 * |entry|.  Errors: RG_ERR_RANGE when K > 2^17, when
 * bits_a + bits_b + ceil(log2 K) > 332 (the 53 primes cannot hold the
 * product), or when that bound exceeds 64 * lc - 1 bits (C might not fit lc
 * limbs); otherwise as for res_gemm_i64.
 */
int res_gemm_limbs(const int64_t* A, int la, const int64_t* B, int lb, int64_t* C, int lc, int64_t M, int64_t N,
                   int64_t K, int nprimes, unsigned flags, void* ws, size_t ws_bytes, void* stream);

/*
 * Outward enclosure of the exact product of binary64 matrices:
 * lo[i][j] <= sum_k A[i][k] * B[k][j] <= hi[i][j] in exact real arithmetic.
 * ("enclosure-gemm", Method.)
 *
 * Each operand is scaled by its own power of two 2^F, F being the finest
 * binary point among its entries, so every scaled entry is an integer
 * (lossless).  The exact integer S = sum A'B' and Q = F_a + F_b are turned
 * into bit patterns: a zero remainder gives lo == hi == S * 2^-Q; otherwise
 * the truncated value is the endpoint toward zero and the next encoding the
 * endpoint away from zero; beyond the largest finite value the endpoint
 * toward zero is +-max finite and the other +-inf.  S == 0 gives +0.0 for
 * both; a negative value too small for a subnormal gives [-2^-1074, -0.0].
 * No floating-point instruction touches the result.
 * Operands wider than the fixed point (more than 255 bits, or
 * bits_a + bits_b + ceil(log2 K) > 332) are coarsened: the larger operand
 * gives up bits first, entries are floored at the coarser point (remainder in
 * [0, 1) per entry), and the interval (-K(2^bits_a + 2^bits_b),
 * K(2^bits_a + 2^bits_b) + K) bounding the induced error is added to S before
 * each endpoint is rounded outward: a valid, looser bracket, reported by
 * rg_get_plan() with lossless = 0 ("enclosure-gemm", Method).
 * info: null, or a host int that receives the regime on success: 0 when both
 * operands scaled exactly (the tightest bracket), 1 when they were coarsened
 * (return_info's "regime" in "enclosure-gemm", Usage).  A non-null info
 * implies RG_FLAG_SYNC.
 * Errors: RG_ERR_NONFINITE (an inf or nan entry), RG_ERR_RANGE (K > 2^17),
 * and the errors of res_gemm_i64.
 */
int enclose_gemm_f64(const double* A, const double* B, double* lo, double* hi, int64_t M, int64_t N, int64_t K,
                     unsigned flags, int* info, void* ws, size_t ws_bytes, void* stream);

/*
 * enclose_gemm_f64 for binary32 operands, with binary32 bounds: lo and hi are
 * the largest and smallest floats bracketing the exact product; overflow
 * gives +-max finite toward zero and +-inf away from it, and a negative value
 * too small for a subnormal gives [-2^-149, -0.0] ("enclosure-gemm", Usage:
 * operands are float32 or float64; Correctness: the floor and ceiling in the
 * format).  The scale exponents come from the binary32 exponent field and the
 * 24-bit significand, so a float32 operand needs no more bits than its values
 * span.  Regimes, workspace (RG_OP_ENCLOSE_F32) and errors as for
 * enclose_gemm_f64.
 */
int enclose_gemm_f32(const float* A, const float* B, float* lo, float* hi, int64_t M, int64_t N, int64_t K,
                     unsigned flags, void* ws, size_t ws_bytes, void* stream);

/*
 * Outward enclosure of the product of interval matrices in midpoint-radius
 * form, <Am, Ar> [M][K] times <Bm, Br> [K][N] (radii >= 0), by Rump's bound:
 * the midpoint S = Am * Bm and the radius R = |Am| * Br + Ar * (|Bm| + Br)
 * are formed as exact integers (three products on the residue engine, one
 * launch), and lo is the largest value of the format <= S - R, hi the
 * smallest >= S + R.  Every point product A * B with A in <Am, Ar>, B in
 * <Bm, Br> lies in [lo, hi]; the only overestimation is the bound's own
 * ("enclosure-gemm", Usage: mm_interval; Method: Rump's midpoint-radius bound
 * with its products and radius formed as exact integers).
 *
 * One scale covers an operand's midpoints and radii.  At a coarsened point
 * (lossless = 0 in rg_get_plan) midpoints are floored and radius magnitudes
 * rounded up, and the midpoint's flooring bound is added outward as for
 * enclose_gemm_f64.  The residue range must hold bits_a + bits_b +
 * ceil(log2 K) + 2 bits (bound_bits in rg_get_plan).  RG_FLAG_TRANS_B gives
 * Bm and Br as [N][K].  Workspace: RG_OP_INTERVAL (RG_OP_INTERVAL_F32).
 * Errors: RG_ERR_RADIUS (a negative radius: a set sign bit on a nonzero
 * entry), RG_ERR_NONFINITE, and the errors of enclose_gemm_f64.
 */
int interval_gemm_f64(const double* Am, const double* Ar, const double* Bm, const double* Br, double* lo, double* hi,
                      int64_t M, int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes, void* stream);
int interval_gemm_f32(const float* Am, const float* Ar, const float* Bm, const float* Br, float* lo, float* hi,
                      int64_t M, int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes, void* stream);

/*
 * Batched forms: `batch` independent products of one shape, each operand's
 * products stored back to back: A [batch][M][K], B [batch][K][N] (with
 * RG_FLAG_TRANS_B [batch][N][K]; limbs add a last dimension as above),
 * outputs [batch][M][N].  One plan covers the whole batch: one prime count
 * from the largest entry of all of A and of all of B and, for fp64, one pair
 * of scale exponents, so the batch pays the planning cost once ("enclosure-
 * gemm", Usage: bmm_enclose; Method: a batch shares one plan).  A shared
 * scale is the finest binary point of the whole batch, so each product's
 * bracket is the one a separate call would give when the call is lossless.
 * batch = 0 is an empty problem.  Errors as for the unbatched forms.
 */
int res_gemm_i64_batched(const int64_t* A, const int64_t* B, int64_t* C, int64_t batch, int64_t M, int64_t N,
                         int64_t K, int nprimes, unsigned flags, void* ws, size_t ws_bytes, void* stream);
int res_gemm_limbs_batched(const int64_t* A, int la, const int64_t* B, int lb, int64_t* C, int lc, int64_t batch,
                           int64_t M, int64_t N, int64_t K, int nprimes, unsigned flags, void* ws, size_t ws_bytes,
                           void* stream);
int enclose_gemm_f64_batched(const double* A, const double* B, double* lo, double* hi, int64_t batch, int64_t M,
                             int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes, void* stream);
int enclose_gemm_f32_batched(const float* A, const float* B, float* lo, float* hi, int64_t batch, int64_t M,
                             int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes, void* stream);
int interval_gemm_f64_batched(const double* Am, const double* Ar, const double* Bm, const double* Br, double* lo,
                              double* hi, int64_t batch, int64_t M, int64_t N, int64_t K, unsigned flags, void* ws,
                              size_t ws_bytes, void* stream);
int interval_gemm_f32_batched(const float* Am, const float* Ar, const float* Bm, const float* Br, float* lo,
                              float* hi, int64_t batch, int64_t M, int64_t N, int64_t K, unsigned flags, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * The per-prime tensor-core stage alone, on caller-provided residues:
 * RC[p][m][n] = (sum_k RA[p][m][k] * RB[p][k][n]) mod q_p, in [0, q_p), for
 * the nprimes largest primes q_0 = 251 > q_1 = 241 > ...
 * ("exact-solve", Method: per-prime products as one batched GEMM.)
 *
 * RA: fp16 bit patterns [nprimes][M][lda], lda >= K, lda % 8 == 0.
 * RB: fp16 bit patterns [nprimes][K][ldb], ldb >= N, ldb % 64 == 0; with
 *     RG_FLAG_TRANS_B, [nprimes][N][ldb], ldb >= K, ldb % 8 == 0.
 * RC: uint8 [nprimes][M][ldc], ldc >= N, ldc % 16 == 0.
 * Every residue must be an integer in [-125, 125]; RA columns k >= K and RB
 * columns n >= N are not read.  ws needs rg_workspace_bytes(RG_OP_STAGE, ...).
 * Errors: RG_ERR_ARG, RG_ERR_RANGE (K > 2^17), RG_ERR_CUDA, RG_ERR_TIMEOUT.
 */
int res_gemm_stage(const uint16_t* RA, int64_t lda, const uint16_t* RB, int64_t ldb, uint8_t* RC, int64_t ldc,
                   int nprimes, int64_t M, int64_t N, int64_t K, unsigned flags, void* ws, size_t ws_bytes,
                   void* stream);

/*
 * res_gemm_i64 without a caller workspace and without any allocation.  The
 * pages have no counterpart; this entry point exists for callers that cannot
 * allocate device memory when they call: code inside a host framework that
 * owns all device memory through its own arena, latency-critical code where
 * cudaMalloc's implicit synchronisation is not allowed, and code whose only
 * device memory is the buffers it was handed.
 *
 * Arguments, results and status codes are those of res_gemm_i64 (the
 * caller still passes A, B and C; K > 2^17 gives RG_ERR_RANGE).  The scratch
 * is one fixed static device array of rg_noalloc_scratch_bytes() bytes
 * (64 MiB) inside the library, which every GPU that loads the library holds
 * until the process exits.  A problem whose scratch
 * (rg_workspace_bytes(RG_OP_I64, ...)) exceeds it returns RG_ERR_WORKSPACE
 * before any device work.  No cudaMalloc, cudaFree, cudaHostAlloc or other
 * allocating routine is called: with RG_FLAG_SYNC or RG_FLAG_HOST the
 * closing status is copied into a host stack word and the stream is
 * synchronised.
 *
 * The first call on each device looks up the array's device address (and
 * copies the constant tables), so make that first call before any stream
 * capture on that device.  Every call shares the one array and its leftover
 * contents; each call clears what must start at zero.  Calls that overlap on
 * the GPU (on different streams, or from several host threads) race on the
 * array: serialise them.
 */
int res_gemm_i64_noalloc(const int64_t* A, const int64_t* B, int64_t* C, int64_t M, int64_t N, int64_t K, int nprimes,
                         unsigned flags, void* stream);

/* Size in bytes of the fixed scratch of res_gemm_i64_noalloc (64 MiB). */
size_t rg_noalloc_scratch_bytes(void);

/*
 * Workspace size in bytes for one call of `op` (RG_OP_*) with these shapes.
 * la, lb, lc are the limb counts (1 for RG_OP_I64 / RG_OP_ENCLOSE[_F32]); nprimes
 * is the value the call will pass (0 = plan on the device).  flags must
 * match the call's RG_FLAG_HOST and RG_FLAG_TRANS_B bits.  Returns 0 for
 * invalid arguments, including shapes the kernels cannot index: M, N or
 * batch above 2^31 - 1, K above 2^17, or more than 2^31 - 1 GEMM tiles
 * (primes x products x ceil(M / 128) x ceil(N / 256)); the entry points
 * return RG_ERR_ARG (RG_ERR_RANGE for K) for the same shapes.  An empty
 * problem needs the 4 KiB plan block only.
 * The floating-point operations (RG_OP_ENCLOSE[_F32], RG_OP_INTERVAL[_F32])
 * plan on the device, so with nprimes = 0 the size covers all 53 primes.
 * Their entry points also accept a smaller workspace, down to the size this
 * function gives for nprimes = 1: the call then uses the largest prime count
 * p whose size (nprimes = p) fits, and the plan coarsens the scaling to fit p
 * primes where it needs more (a valid, looser bracket; rg_get_plan reports
 * lossless = 0).  A workspace sized for the prime count a first call reports
 * (rg_get_plan's nprimes) gives later calls on operands of the same binary
 * range the same bits, as the page's working-memory model P (MK + KN) has it
 * ("enclosure-gemm", Requirements and limits).  When not one bit per operand
 * is left the call fails with RG_ERR_WORKSPACE.
 */
size_t rg_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int la, int lb, int lc, int nprimes,
                          unsigned flags);
/* The same for a batched call of `batch` products. */
size_t rg_workspace_bytes_batched(int op, int64_t batch, int64_t M, int64_t N, int64_t K, int la, int lb, int lc,
                                  int nprimes, unsigned flags);

/* Offsets (bytes from ws) of the stage buffers a call leaves in its
 * workspace, for inspection:
 *   ra: fp16 residues of A, [pmax][M][lda]   (lda = K rounded up to 8)
 *   rb: fp16 residues of B, [pmax][K][ldb]   (ldb = N rounded up to 64), or
 *       [pmax][N][ldb] with RG_FLAG_TRANS_B    (ldb = K rounded up to 8)
 *   rc: uint8 product residues, [pmax][M][ldc] (ldc = N rounded up to 16)
 * Residue planes follow the prime order q_0 = 251, q_1 = 241, ...; a batched
 * call stores each prime's planes for all products back to back
 * ([pmax][batch][M][lda] and so on).  splits: the K slices rc has room for
 * (more than one lets the GEMM split long K over idle SMs; the slices are then
 * summed mod q into the first by one extra kernel launch per call). */
typedef struct {
  size_t ra, rb, rc;
  int64_t lda, ldb, ldc;
  int pmax;
  int splits;
} rg_layout;
int rg_workspace_layout(int op, int64_t M, int64_t N, int64_t K, int la, int lb, int lc, int nprimes,
                        unsigned flags, rg_layout* out);
int rg_workspace_layout_batched(int op, int64_t batch, int64_t M, int64_t N, int64_t K, int la, int lb, int lc,
                                int nprimes, unsigned flags, rg_layout* out);

/* The plan a call chose, read back from its workspace after the stream is
 * synchronised ("enclosure-gemm", Method: return_info reports the regime). */
typedef struct {
  int status;   /* RG_OK or the first error the device recorded */
  int nprimes;  /* primes used */
  int bits_a;   /* bit length of the largest |entry| (scaled entry for fp64) */
  int bits_b;
  int bound_bits; /* bits_a + bits_b + ceil(log2 K) */
  int f_a;      /* fp64 only: A' = A * 2^f_a */
  int f_b;
  int lossless; /* fp64 only: 1 if both operands scaled exactly */
  int splits;   /* K slices the per-prime GEMM used (1: none; more when there were too few output tiles) */
  int crt_rn;   /* 0: balanced Garner; 1: round-to-nearest CRT on balanced digits; 2: CRT by idempotent
                 * sums (both with P > 4 |result|; see rg_set_crt_mode) */
} rg_plan_info;
int rg_get_plan(const void* ws, void* stream, rg_plan_info* out);

/*
 * Exact rational solution of A X = B for integer A [n][n] and B [n][c]
 * (row-major int64; device pointers, or host pointers with RG_FLAG_HOST)
 * ("exact-solve", Method).
 *  1. A^-1 mod q for all 53 primes at once by Gauss-Jordan elimination on the
 *     GPU, over all primes in each launch, blocked: per block of up to 64
 *     pivots, one panel factorisation and one fp16 tensor-core update of the
 *     other columns; the primes that divide det(A) are dropped.
 *  2. Dixon's p-adic lift with P = the product of the remaining primes:
 *     X_i = A^-1 R_i mod P per prime, then balanced Garner into the base-P
 *     digit; R_{i+1} = (R_i - A X_i) P^-1 mod 2^64, exact in one limb; as
 *     many steps as make P^m exceed twice the product of the Hadamard bounds
 *     of numerator and denominator.
 *  3. Rational reconstruction of a few components on host threads for the
 *     common denominator d; on the GPU, every component's value from its
 *     base-P digits and its numerator d X mod P^m (balanced), one block per
 *     component.
 * On success `out` holds the numerators N [n][c] and the least common
 * denominator d > 0 (X = N / d exactly), as `limbs` little-endian
 * two's-complement int64 limbs each, in a host array the library allocates
 * and rg_solution_free releases.  Requires n * max|A| < 2^63 (so the residual
 * stays one limb) and n <= 8192.  The call synchronises `stream`.  Unlike the
 * product entry points it takes no workspace: its device buffers come from
 * cudaMallocAsync on `stream` and are freed there before it returns.  It is
 * not safe to run two solves at once on one device (one constant table holds
 * the lift's primes).
 * Errors: RG_ERR_ARG, RG_ERR_RANGE (n or the entries out of range),
 * RG_ERR_SINGULAR (A is singular modulo every prime below 256: singular over
 * the rationals, unless det(A) is divisible by all 53 primes), RG_ERR_CUDA.
 */
typedef struct {
  int64_t n, c;     /* shape of the solution */
  int64_t limbs;    /* int64 limbs per value */
  int64_t* values;  /* (n * c + 1) * limbs: the numerators row-major, then d */
  int64_t steps;    /* lift steps m */
  int primes;       /* primes in the lift modulus P */
  double ms_inverse;      /* wall time of the batched inverse (incl. norms and range check) */
  double ms_lift;         /* wall time of the lift, digits copied to the host */
  double ms_reconstruct;  /* wall time of the host reconstruction */
} rg_solution;
int rg_solve_i64(const int64_t* A, const int64_t* B, int64_t n, int64_t c, unsigned flags, void* stream,
                 rg_solution* out);
void rg_solution_free(rg_solution* s);

/*
 * Rational reconstruction on the host (the solve's last step, exposed for
 * testing): N, D with D X == N (mod M), |N| <= 2^nbits, 0 < D <= 2^dbits, in
 * lowest terms, for 0 <= X < M given as xl and ml little-endian 64-bit limbs.
 * Writes `limbs` two's-complement limbs each to num and den.  Returns
 * RG_ERR_RANGE if no such pair exists or it does not fit, RG_ERR_ARG on bad
 * arguments.  Unique when 2^(nbits + dbits + 1) < M.
 */
int rg_rational_reconstruct(const int64_t* x, int xl, const int64_t* m, int ml, int nbits, int dbits, int64_t* num,
                            int64_t* den, int limbs);

/*
 * gcd(a, b) of naturals given as al and bl little-endian 64-bit limbs, by the
 * host big-integer code the solve's reconstruction uses (exposed for
 * testing; gcd(0, 0) = 0).  Writes gl limbs to g.  RG_ERR_RANGE if the gcd
 * needs more than gl limbs, RG_ERR_ARG on bad arguments.
 */
int rg_big_gcd(const uint64_t* a, int al, const uint64_t* b, int bl, uint64_t* g, int gl);

/*
 * (a * b) mod m of naturals a, b < m given as little-endian 64-bit limbs, by
 * the host big-integer code the solve's numerators use: a Karatsuba product
 * and Barrett's reduction (exposed for testing).  Writes rl limbs to r.
 * RG_ERR_RANGE if the result needs more than rl limbs, RG_ERR_ARG on bad
 * arguments (m zero, a or b not below m).
 */
int rg_big_mulmod(const uint64_t* a, int al, const uint64_t* b, int bl, const uint64_t* m, int ml, uint64_t* r,
                  int rl);

/* Reconstruction of the results.  Mode 0 (the default): one-limb results
 * (res_gemm_i64, res_gemm_limbs with lc = 1) of at most 12 primes (every
 * int64 product the library plans, and caller-fixed counts up to 12) by CRT
 * with idempotent sums: S = sum_i r_i E_i over the unreduced residues, E_i
 * the CRT idempotent of q_i, and the result S - k P formed modulo 2^64 with
 * k the rounded estimate of S / P, or a neighbour of it when that leaves the
 * symmetric range (four integer multiply-adds per prime and entry);
 * everything else by balanced Garner.  Mode 1: CRT with a round-to-nearest
 * quotient on balanced digits ("Accelerating Multiple-Precision LU
 * Decomposition with Ozaki Scheme II") for the wide outputs (limbs, enclosures, intervals) where the plan can
 * keep P > 4 |result| (one more bit of headroom, so sometimes one more
 * prime), and for int64 where its planned primes already exceed 4 |result|;
 * Garner otherwise.  Mode 2: balanced Garner for every result.  On GB300
 * Garner is faster than mode 1's digits (38 primes, 128-bit, 2048^2 outputs:
 * 264 against 317 us; 8 primes, int64, 1024^2 outputs: 12.5 against 14.3 us).
 * rg_get_plan's crt_rn reports the choice a call made (0 Garner, 1 balanced
 * digits, 2 idempotent sums).  Returns the previous mode, or -1 for an
 * invalid one. */
int rg_set_crt_mode(int mode);

/* Synchronise `stream` and return the device status of the last call that
 * used `ws` (RG_OK, RG_ERR_RANGE, RG_ERR_NONFINITE, RG_ERR_LOSSY,
 * RG_ERR_TIMEOUT) or RG_ERR_CUDA. */
int rg_status(const void* ws, void* stream);

/* The i-th prime of the residue base, largest first (251, 241, ...);
 * 0 if i is out of range. */
int rg_prime(int i);

/* A static description of a status code. */
const char* rg_strerror(int code);

/* Test hook: the time limit (nanoseconds) of every bounded wait inside the
 * library's kernels (default one second), and a fault to inject into the next
 * tensor-core stage: 1 = its producer never signals the first accumulator,
 * so the consumer's wait must expire and return RG_ERR_TIMEOUT.  Returns the
 * previous limit.  Not thread-safe; for tests only. */
uint64_t rg_set_wait_limit_ns(uint64_t ns);
void rg_inject_fault(int kind);

/* Measurement hook: with n = 4, every later GEMM call (res_gemm_i64/limbs,
 * enclose_gemm_*, interval_gemm_*, batched or not) records events[0] on its
 * stream before its first kernel, events[1] before the per-prime GEMM,
 * events[2] after it (split-K summation included) and events[3] after the
 * reconstruction kernel, so that the caller can time each stage inside a
 * real call with cudaEventElapsedTime.  events are cudaEvent_t handles the
 * caller created and keeps alive while the hook is set.  The records
 * serialise the stages (no overlap of one kernel's start with the previous
 * one's end).  n = 0 removes the hook.  Process-wide; returns RG_OK, or
 * RG_ERR_ARG for another n or a null handle. */
int rg_set_stage_events(void* const* events, int n);

/* Test hook: which tensor-core kernel runs the per-prime stage.  0 = choose
 * by shape (the CTA-pair kernel when M > 128), 1 = single-CTA kernel,
 * 2 = CTA-pair kernel.  Returns the previous choice, or -1 for an invalid
 * value.  Not thread-safe; for tests and measurements only. */
int rg_set_gemm_variant(int variant);

/* Measurement: one launch of a peak-rate probe of a tensor-core instruction,
 * enqueued on `stream` for the caller to time with events.  No page has a
 * counterpart: the probes give the denominators the per-prime GEMM is
 * reported against ("enclosure-gemm", Method: one INT8 tensor-core GEMM per
 * prime, hence a "% of INT8 tensor-core roofline"), and the rate of the FP8
 * instruction that a balanced base-17 digit split of the residues would use
 * ("Accelerating Multiple-Precision LU Decomposition with Ozaki Scheme II",
 * FP8 encoding).  Not part of the product path.
 *   kind  RG_PROBE_MMA_S8: warp-level mma.sync m16n8k32 s8 x s8 -> s32 from
 *           registers, eight independent accumulators per warp, 8 warps per
 *           block (blocks = 0: four per SM);
 *         RG_PROBE_TCGEN05_F16 / RG_PROBE_TCGEN05_E4M3: tcgen05.mma
 *           cta_group::1 kind::f16 (fp16) / kind::f8f6f4 (E4M3), M = 128,
 *           N = 256, operands in shared memory (both K-major), fp32
 *           accumulator in tensor memory, one CTA per SM (blocks = 0: the SM
 *           count);
 *         RG_PROBE_TCGEN05_F16_BMN: the same with B read MN-major;
 *         RG_PROBE_TCGEN05_F16_PAIR / _PAIR_BMN: cta_group::2 (clusters of
 *           two CTAs, M = 256, N = 256), B K-major / MN-major; blocks must
 *           be even (0: the SM count rounded down to even);
 *         RG_PROBE_TCGEN05_F16_PAIR_BMN_SYNC: the pair form with the residue
 *           GEMM's per-k-block issue loop (a barrier wait and a commit every
 *           four MMAs), without data movement;
 *         RG_PROBE_MMA_F16: warp-level mma.sync m16n8k16 f16 x f16 -> f32,
 *           otherwise as RG_PROBE_MMA_S8.
 *   iters  rounds per warp or CTA (1 .. 2^24): 8 MMAs per round for
 *          mma.sync, 4 for tcgen05 (K = 64 fp16 or 128 E4M3 per round;
 *          *ops_per_launch counts 128 rows per CTA for the pair forms too).
 *   ws     device memory of >= 256 bytes, 256-byte aligned, caller-owned;
 *          the probe's status (RG_ERR_TIMEOUT if the tcgen05 probe's bounded
 *          wait expired) is read from it with rg_status(ws, stream).
 * *ops_per_launch receives 2 x the multiply-adds one launch performs.
 * Returns RG_OK once enqueued, RG_ERR_ARG or RG_ERR_CUDA. */
#define RG_PROBE_MMA_S8 0
#define RG_PROBE_TCGEN05_F16 1
#define RG_PROBE_TCGEN05_E4M3 2
#define RG_PROBE_TCGEN05_F16_BMN 3
#define RG_PROBE_TCGEN05_F16_PAIR 4
#define RG_PROBE_TCGEN05_F16_PAIR_BMN 5
#define RG_PROBE_TCGEN05_F16_PAIR_BMN_SYNC 6
#define RG_PROBE_MMA_F16 7
int rg_probe_mma_rate(int kind, int blocks, int iters, void* ws, size_t ws_bytes, void* stream,
                      double* ops_per_launch);

#ifdef __cplusplus
}
#endif
#endif /* RESGEMM_H */
