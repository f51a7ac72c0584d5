/*
 * muon_ns.h -- C ABI of the owner-side Muon update for one NVIDIA GB300 (sm_103a).
 *
 * What the library computes (for each 2D matrix it is given):
 *
 *   M  <- beta * M + G                      momentum accumulate (heavy ball)
 *   X  =  M, or M^T when rows > cols        short side first
 *   X0 =  X / (||X||_F + 1e-7)
 *   repeat `steps` times:                   Newton-Schulz (NS) iteration
 *       X <- a X + b (X X^T) X + c (X X^T)^2 X
 *   O  =  X (un-transposed)
 *   W  <- W - lr * O                        scaled apply
 *
 * Sources: DMuon technical summary (gist.science, arXiv 2606.27153), §1
 * "Definizione del Problema" (NS on momentum-aggregated gradients, the product
 * X X^T needs the whole matrix) and §2.2 "Iterazione Gram Newton-Schulz
 * Efficiente" (run the iteration on G = X X^T of the short side, compute only
 * the lower triangle of the symmetric products, batch matrices of the same
 * shape).  MatrixFSDP technical summary (gist.science, arXiv 2607.05895),
 * "Metodologia": the owner of a matrix runs this update locally.  The pages do
 * not fix the momentum form, the normalisation or the apply; the readings
 * above are the plainest ones.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers to memory the caller owns
 *    (e.g. torch tensors).  Arrays of pointers (W, grad, mom) and `shapes`
 *    are HOST arrays.  The library allocates no device memory: scratch comes
 *    from the caller's workspace `ws` (size from muon_workspace_bytes).
 *  - Matrices are dense row-major: element (i, j) of an m x n matrix is at
 *    offset i*n + j.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns before it completes.
 *  - Argument errors are detected before anything is launched, so a failed
 *    call writes nothing.  Nothing throws across the ABI.  The message of the
 *    last error on the calling thread is returned by muon_last_error().
 *  - A kernel that waits longer than its bound (4e9 SM clock cycles: about
 *    2 s at the 2.07 GHz maximum clock, longer at lower clocks) on an
 *    internal barrier stops, records MUON_ERR_TIMEOUT in the workspace's
 *    status word and returns; muon_device_status() reports it.  The output
 *    of such a call is incomplete.
 *  - NaN and Inf in the inputs propagate; they are not checked.
 *  - Calls that share a workspace must be ordered on one stream.
 */
#ifndef MUON_NS_H
#define MUON_NS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MUON_API __attribute__((visibility("default")))
#else
#define MUON_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MUON_OK = 0,
    MUON_ERR_ARG = 1,          /* null pointer, negative count, bad enum, bad scalar */
    MUON_ERR_SHAPE = 2,        /* a dimension <= 0 or above MUON_MAX_DIM */
    MUON_ERR_ALIGN = 3,        /* workspace not 256-byte aligned, or a tensor not aligned to its element size */
    MUON_ERR_WORKSPACE = 4,    /* ws_bytes too small for even one matrix of a bucket */
    MUON_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed (message has the CUDA error) */
    MUON_ERR_TIMEOUT = 6,      /* a kernel's bounded wait ran out (reported by muon_device_status) */
    MUON_ERR_UNSUPPORTED = 7   /* e.g. no sm_103a device for the tensor-core path */
} muon_status;

typedef enum {
    MUON_BF16 = 0,   /* grad, W (and X/out of muon_ns_batched) are bfloat16; momentum is fp32 */
    MUON_FP32 = 1,   /* all tensors fp32; NS computed with fp32 arithmetic */
    MUON_FP16 = 2    /* muon_debug_gemm only: fp16 operands and an fp16 output pair */
} muon_dtype;

typedef enum {
    MUON_SCHED_AUTO = 0,     /* cheapest schedule that meets the dtype's accuracy (see below) */
    MUON_SCHED_GRAM_X3 = 1,  /* Gram space without restarts; split-bf16 operands (hi*hi + hi*lo + lo*hi) */
    MUON_SCHED_GRAM_X1 = 2,  /* Gram space without restarts; plain bf16 operands (diverges on rank-deficient inputs) */
    MUON_SCHED_ORIG = 3,     /* original space (bf16: step 0 in bf16, later steps on fp16 operands, see below) */
    MUON_SCHED_ORIG_BF16 = 4, /* original space on bf16 operands only; split A in A*A and B in B*X in the last max(2, steps - 3) steps */
    MUON_SCHED_ORIG_F16X3 = 5, /* original space; every operand an fp16 pair (~22 bits), three tensor-core products per product */
    MUON_SCHED_GRAM_R2 = 6     /* Gram space restarted from X every two steps (bf16: fp16 operands; fp32: FFMA) */
} muon_sched;

/*
 * Schedules and precision.  Every tensor-core product accumulates in fp32.
 *  - bf16, AUTO: up to 10 steps GRAM_R2 where it executes at most 0.9x
 *    ORIG's tensor-core work (the long side at least about 1.5x the short
 *    side, and 3 or more steps), else ORIG.  Past 10 steps ORIG_F16X3: the
 *    quintic does not contract inside the band it maps singular values into,
 *    so single fp16 operands drift with the step count (at most 8.9e-3 at 10
 *    steps, 2.1e-2 at 15, up to 3.7e-2 at 20-100), where fp16 pairs stay at
 *    the bf16 output rounding.
 *  - fp32, AUTO: up to 6 steps ORIG_F16X3 (tensor cores, below); longer runs
 *    on fp32 FFMA (CUDA cores): GRAM_R2 where it saves at least a tenth of
 *    ORIG's work, else ORIG.  Explicit GRAM_X3 / GRAM_X1 on fp32 data run
 *    Gram space without restarts on FFMA, which is unstable on rank-deficient
 *    inputs over many steps: rounding leaves G with small negative
 *    eigenvalues that the recurrence grows by about a^2 per step.
 *  - ORIG (bf16).  Step 0 multiplies the packed bf16 copy of M (exact for bf16
 *    gradients from a zero momentum state) on bf16 operands.  Every later
 *    product takes fp16 operands (11 significant bits against bf16's 8).
 *    Between steps X is carried as an fp16 pair, hi + lo / 2^11 (about 22 bits).
 *    A = X X^T and B = b A + c A^2 are single fp16 values.  fp16's range is safe:
 *    the Frobenius normalisation gives sigma(X0) <= 1.  When the polynomial
 *    p(s) = a s + b s^3 + c s^5 maps [0, 1.25] into [-1.25, 1.25], every
 *    iterate keeps sigma <= 1.25 (the quintic and the cubic (1.5, -0.5, 0)
 *    do).  Coefficients that fail this check, or whose |b|, |c| could take B
 *    out of fp16's range, run as ORIG_BF16.
 *  - ORIG_BF16.  bf16 operands throughout, with X carried as a bf16 pair (about
 *    16 bits).  A*A and B*X use split operands in the last max(2, steps - 3)
 *    steps (every step from the fourth on when there are more than five).
 *  - GRAM_X3 / GRAM_X1.  The Gram recurrence for all steps, without restarts,
 *    on bf16 pairs (split products) or on plain bf16: the pages' form, kept
 *    for comparison.  Over several Gram steps the rounding of G (and the
 *    symmetric storage of products that commute only up to rounding) is
 *    amplified in the directions of small singular values.  Measured on
 *    rank-8 + noise inputs at 5 steps: GRAM_X3 reaches 2.1e-2, and GRAM_X1
 *    diverges (relative errors of 9 to 45).  On full-rank inputs GRAM_X3
 *    stays at the bf16 output rounding (1.7e-3).  Use GRAM_R2 for Gram space.
 *  - GRAM_R2 (bf16; fp32 runs the same segments with FFMA).  Step 0 is ORIG's bf16 step; the remaining steps run in
 *    segments of two (a last single step when steps - 1 is odd).  A segment
 *    forms A = X_hi X_hi^T once, runs two steps of the Gram recurrence on it
 *    (P_0 = a I + b A + c A^2, G_1 = P_0 A P_0, P_1 likewise, Q = P_1 P_0,
 *    fp16 operands) and restarts from X <- Q X_hi + a^2 X_lo.  Per two steps
 *    that is one s x l SYRK, one s x s x l update and five s x s products,
 *    against two SYRKs, two updates and two s x s products in ORIG.  Longer
 *    Gram segments on fp16 operands lose the directions of small singular
 *    values on low-rank inputs; two-step segments stay within about 1e-2 of
 *    the fp64 result on them.  With coefficients outside fp16's range it runs
 *    as ORIG_BF16.  Its workspace is ORIG's.
 *  - ORIG_F16X3 (either dtype).  X0 = M / (||M||_F + eps) is formed in fp32
 *    and split into an fp16 pair hi + lo / 2^11; every product takes pairs
 *    (A, B' and X) and runs as hi*lo + lo*hi followed by hi*hi on an
 *    accumulator the tensor core scales by 2^-11, in fp32.  About 22-bit
 *    operands at three times the tensor-core work of one product: the
 *    tensor-core form of the fp32 path, several times faster than FFMA.  Its
 *    accuracy is set by the tensor cores' fp32 accumulation (about 1e-6 of
 *    the sum of |products| per product, against 1e-7 for FFMA), so it is
 *    fp32's AUTO choice only up to 6 steps (within 3e-5 there on Gaussian
 *    and row-scaled inputs, about 9e-5 at 10 steps).
 * muon_workspace_bytes is the same for ORIG, ORIG_BF16 and GRAM_R2 (bf16).
 */

/*
 * Launch-mode flags, OR'ed into a muon_sched argument (its low 8 bits are the
 * schedule).  By default the tensor-core products of a batch chunk share
 * persistent launches (up to 16 consecutive products per launch, ordered per
 * matrix by completion counters) when the chunk is small -- at most 16
 * 256 x 256 tile pairs per CTA pair in its largest product, or at most 4 in
 * its s x s products -- and run one launch per product otherwise.  These flags force one of the two; the
 * numerics are the same either way (every tile is computed identically).
 * Measured per shape by the binding's tune_schedules.
 */
#define MUON_SCHED_SHARED_LAUNCH 0x100
#define MUON_SCHED_SEPARATE_LAUNCH 0x200
#define MUON_SCHED_MASK 0xff

#define MUON_MAX_DIM 65536   /* largest accepted m or n */
#define MUON_MAX_STEPS 100   /* largest accepted number of NS steps */
#define MUON_WS_ALIGN 256    /* required alignment of the workspace pointer */
#define MUON_PARTITION_EXACT_MAX 24           /* largest count muon_partition solves exactly */
#define MUON_PARTITION_NODE_BUDGET 4000000LL  /* search nodes before the exact solver stops */

/*
 * muon_ns_batched -- NS orthogonalisation of B same-shape matrices.
 *   X      [B, m, n] contiguous, dtype dt (device, read only).
 *   B      number of matrices (0 is a no-op).
 *   m, n   shape of each matrix.
 *   steps  NS iterations T (0 returns X0, the normalised input).
 *   coeffs host array {a, b, c}; NULL selects the quintic (3.4445, -4.7750, 2.0315).
 *   out    [B, m, n] contiguous, dtype dt (device, written; must not overlap X
 *          or the workspace).  out[i] = O_i as defined above.
 *   dt, sc dtype and schedule.
 *   ws, ws_bytes  workspace (device, 256-byte aligned) and its size.  If it
 *          is smaller than muon_workspace_bytes() for this problem, the batch
 *          is processed in smaller chunks; below one matrix it is an error.
 *   stream cudaStream_t.
 */
MUON_API muon_status muon_ns_batched(const void* X, int B, int m, int n, int steps,
                            const float* coeffs, void* out, muon_dtype dt,
                            muon_sched sc, void* ws, size_t ws_bytes, void* stream);

/*
 * muon_step -- one owner-side Muon step over `count` matrices of any shapes.
 *   W      host array of `count` device pointers to weights [m_i, n_i], dtype
 *          dt, updated in place: W <- W - lr * O.
 *   grad   host array of device pointers to gradients [m_i, n_i], dtype dt (read only).
 *   mom    host array of device pointers to fp32 momentum [m_i, n_i], updated
 *          in place: M <- beta*M + G.
 *   shapes host int64 array {m_0, n_0, m_1, n_1, ...}.
 *   Matrices are grouped by (short side, long side); each group is run as one
 *   batch (wider groups are split to fit the workspace).  W, grad and mom of
 *   different matrices must not overlap.
 *   The remaining arguments are as for muon_ns_batched.
 */
MUON_API muon_status muon_step(void* const* W, const void* const* grad, float* const* mom,
                      const int64_t* shapes, int count, float beta, float lr, int steps,
                      const float* coeffs, muon_dtype dt, muon_sched sc,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * muon_workspace_bytes -- workspace that lets every shape group of the given
 * matrices run as one batch (capped at 256 matrices per batch) with schedule
 * `sc` (AUTO resolved per group as the library would).  Returns 0 on bad
 * arguments (see muon_last_error).
 */
MUON_API size_t muon_workspace_bytes(const int64_t* shapes, int count, int steps,
                            muon_dtype dt, muon_sched sc);

/*
 * muon_resolve_schedule -- the schedule AUTO picks for one m x n group with
 * `steps` iterations and the quintic coefficients (launch-mode flags in `sc`
 * are ignored; the result has none).  Host only.
 */
MUON_API muon_sched muon_resolve_schedule(int64_t m, int64_t n, int steps, muon_dtype dt, muon_sched sc);

/*
 * muon_bucket_plan -- the grouping muon_step uses, for inspection.  Fills
 * order[count] with matrix indices (groups by increasing (short, long) key,
 * members in input order) and group_start[count+1] with the offsets of each
 * group in `order`; returns the number of groups, or -1 on bad arguments.
 * Host only, no GPU needed.
 */
MUON_API int muon_bucket_plan(const int64_t* shapes, int count, int* order, int* group_start);

/*
 * muon_device_status -- synchronise `stream`, then read and clear the status
 * word of workspace `ws`.  Returns MUON_ERR_TIMEOUT if a kernel gave up on a
 * bounded wait since the last check, MUON_ERR_CUDA on a CUDA error, else MUON_OK.
 */
MUON_API muon_status muon_device_status(void* ws, void* stream);

/*
 * muon_debug_bounded_wait -- failure-detection self-test: launches one block
 * that waits on an on-chip barrier nobody arrives at, with a bound of
 * `max_cycles` SM cycles, records MUON_ERR_TIMEOUT in the workspace status
 * word and returns.  Used by the tests to check that a timed-out wait is
 * reported and leaves the context usable.
 */
MUON_API muon_status muon_debug_bounded_wait(void* ws, long long max_cycles, void* stream);

/*
 * muon_debug_gemm -- test hook exposing one batched GEMM kernel on its own.
 *   C[b] = A[b] * op(B[b]) with A [M, K] row-major and B either [N, K]
 *   row-major (b_mn = 0, C = A B^T) or [K, N] row-major (b_mn = 1, C = A B).
 *   Batch strides are M*K, N*K (or K*N) and M*N elements.
 *   dt = MUON_BF16 runs the tcgen05 tensor-core kernel: split = 1 uses A, B;
 *   split = 2 uses (A + A_lo) B (b_mn = 1 only); split = 3 uses
 *   A B + A B_lo + A_lo B.  C is returned as a bf16 pair: out = bf16(C) and,
 *   if out_lo is not NULL, out_lo = bf16(C - out) ([batch, M, N] each).
 *   dt = MUON_FP16: the same kernel on fp16 A, B (and A_lo, B_lo); C is
 *   returned as an fp16 pair, out = fp16(C), out_lo = fp16((C - out) * 2^11).
 *   split = 4 (fp16, b_mn = 1, M == K, sym bit 0 clear): C = A B + B_lo / 2^11,
 *   the second term run on the tensor cores as a diagonal K segment (the
 *   form the original-space update takes for the low part of X); the
 *   diagonal table is written into the workspace after the header, so
 *   ws_bytes must be at least 1024 + 131072.
 *   split = 5 (fp16): A and B are fp16 pairs whose low parts are stored scaled,
 *   A_lo = fp16((A_true - A) * 2^11) and likewise B_lo; C = A B + (A B_lo +
 *   A_lo B) / 2^11, the low-part products accumulated first and the 2^-11
 *   applied by the tensor core to the accumulator (about 22-bit operands).
 *   dt = MUON_FP32 runs the FFMA kernel on fp32 A, B and writes fp32 C to out.
 *   sym bit 0 (M == N): symmetric output; the bf16 kernel computes the tiles
 *   touching the lower triangle and stores the output "block-lower" (only the
 *   256 x 256 blocks on or below the diagonal are written), the fp32 kernel
 *   writes the full matrix.  sym bits 1 / 2 (bf16 only): A / B is a symmetric
 *   matrix given in block-lower storage (its upper blocks are never read).
 *   Sizes: bf16 / fp16 need M % 256, N % 256, K % 128 == 0; fp32 needs M, N % 128 and
 *   K % 16 == 0.  The kernel is enqueued on `stream`.
 */
MUON_API muon_status muon_debug_gemm(const void* A, const void* A_lo, const void* B, const void* B_lo, int batch,
                                     int M, int N, int K, int split, int b_mn, int sym, muon_dtype dt,
                                     void* out, void* out_lo, void* ws, size_t ws_bytes, void* stream);

/*
 * Launch profiling (process-wide, not thread safe; off by default).
 * muon_profile_enable(1) clears the record list and starts recording a pair of
 * CUDA events around every kernel the library enqueues (on the caller's
 * stream); muon_profile_enable(0) stops.  muon_profile_get(i, ...) waits for
 * record i and returns its kernel kind ("pack", "tc_syrk", "tc_sym",
 * "tc_rect", ...), elapsed milliseconds, and the launch's algorithmic flops and
 * HBM bytes (symmetric products counted once).
 */
MUON_API void muon_profile_enable(int on);
MUON_API int muon_profile_count(void);
MUON_API muon_status muon_profile_get(int i, const char** kind, float* ms, double* flops, double* bytes);

/*
 * muon_ns_batched_static -- muon_ns_batched for callers that cannot allocate
 * device memory: code running where a cudaMalloc is not allowed or must not
 * happen (inside a framework that owns every byte of device memory through
 * its own pool, a latency-critical loop where an allocation would stall the
 * device, a plug-in that is handed only input and output buffers).  It takes
 * no workspace: its scratch is one fixed array of muon_static_scratch_bytes()
 * (64 MiB) compiled into the library, which every GPU that loads the library
 * holds until the process exits.  The caller still passes X and out
 * (arguments as for muon_ns_batched).  The pages have no counterpart of this
 * entry point.
 *  - Problems whose single matrix needs more scratch than the array holds
 *    (e.g. a bf16 2048 x 2048 matrix) are rejected with MUON_ERR_WORKSPACE
 *    before anything is launched; larger batches are processed in chunks.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.  Every call
 *    looks up the array's device address on the current device
 *    (cudaGetSymbolAddress, which allocates nothing); the first call on a
 *    device may load the library's device code, so make that first call
 *    before any stream capture.
 *  - All calls share the one array: calls whose work overlaps on the GPU (two
 *    streams, two threads without ordering) race and give wrong results.
 *    Order them on one stream.
 *  - A bounded-wait timeout inside one of its kernels is recorded in the
 *    array's status word, which persists across calls until
 *    muon_static_status() reads and clears it.
 */
MUON_API muon_status muon_ns_batched_static(const void* X, int B, int m, int n, int steps,
                                            const float* coeffs, void* out, muon_dtype dt,
                                            muon_sched sc, void* stream);
MUON_API size_t muon_static_scratch_bytes(void);

/*
 * muon_static_status -- muon_device_status for the static scratch: synchronise
 * `stream`, then read and clear the status word of the array that
 * muon_ns_batched_static runs in.  Returns MUON_ERR_TIMEOUT if one of its
 * kernels gave up on a bounded wait since the last check (the output of that
 * call is incomplete), MUON_ERR_CUDA on a CUDA error, else MUON_OK.
 * Allocates nothing.
 */
MUON_API muon_status muon_static_status(void* stream);

/*
 * muon_debug_bounded_wait_static -- muon_debug_bounded_wait on the static
 * scratch's status word (failure-detection self-test of muon_static_status).
 */
MUON_API muon_status muon_debug_bounded_wait_static(long long max_cycles, void* stream);

/*
 * muon_adamw_tail -- one AdamW step over the non-matrix "tail" of a model
 * (MatrixFSDP technical summary, gist.science 2607.05895, "Metodologia" §1:
 * 1-D vectors and other non-matrix tensors are packed into a tail that a
 * separate owner updates with standard AdamW).  For every element of tensor i:
 *
 *   p <- p * (1 - lr * weight_decay)                 decoupled weight decay
 *   m <- beta1 m + (1 - beta1) g
 *   v <- beta2 v + (1 - beta2) g^2
 *   p <- p - lr / (1 - beta1^step) * m / (sqrt(v) / sqrt(1 - beta2^step) + eps)
 *
 *   params, grads  host arrays of `count` device pointers, dtype dt (bf16 or
 *                  fp32; params updated in place, grads read only), any shape,
 *                  numel[i] contiguous elements each.
 *   exp_avg, exp_avg_sq  host arrays of device pointers to fp32 moments
 *                  (numel[i] each), updated in place; zero before step 1.
 *   numel  host int64 array; 0 is allowed.
 *   step   1 for the first step (bias corrections use it).
 * Arithmetic is fp32; bf16 parameters are rounded once, to nearest even.
 * All tensors go through one launch per 512 of them.  Tensors must not
 * overlap.  16-byte aligned tensors use vector accesses; others take a
 * scalar path.
 * Errors (nothing launched): MUON_ERR_ARG for count < 0, NULL arrays or NULL
 * pointers of non-empty tensors, step < 1, non-finite lr / eps / weight_decay,
 * eps < 0 or betas outside [0, 1), a bad dtype; MUON_ERR_SHAPE for a negative
 * numel; MUON_ERR_ALIGN for a pointer not aligned to its element size;
 * MUON_ERR_UNSUPPORTED without an sm_103 device.
 */
MUON_API muon_status muon_adamw_tail(void* const* params, const void* const* grads, float* const* exp_avg,
                                     float* const* exp_avg_sq, const int64_t* numel, int count, float lr,
                                     float beta1, float beta2, float eps, float weight_decay, int step,
                                     muon_dtype dt, void* stream);

/*
 * ---- owner placement (DMuon technical summary, gist.science 2606.27153,
 * §2.3 "compute-aware load balancing"): every 2-D matrix is updated by exactly
 * one owner rank, and the owners are chosen so that the largest per-owner cost
 * (the makespan) is small.  The pages profile each shape's update time at
 * start-up and minimise the predicted makespan with a MILP, falling back to a
 * greedy heuristic on large inputs.  Host only, no GPU needed.
 */

/*
 * muon_cost_estimate -- predicted device seconds of one matrix's update for
 * each matrix of `shapes` (count x 2, int64 m, n, row-major), under the
 * schedule `sc` resolves to at that shape with `steps` iterations and dtype
 * `dt`.  It counts the launches muon_step issues, with each launch's executed
 * flops (padded 256-blocks, symmetric outputs on lower blocks, split operands
 * 2x / 3x) at a nominal kernel rate and its HBM bytes at a nominal bandwidth,
 * and takes the larger of the two.  A model for placement when no measured
 * costs are at hand.  Writes seconds[count].
 * Errors (nothing written): MUON_ERR_ARG for NULL pointers with count > 0,
 * count < 0, or bad steps, dtype or schedule; MUON_ERR_SHAPE for m or n
 * outside [1, MUON_MAX_DIM].
 */
MUON_API muon_status muon_cost_estimate(const int64_t* shapes, int count, int steps, muon_dtype dt,
                                        muon_sched sc, double* seconds);

/*
 * muon_partition -- assign each of `count` matrices, with costs cost[count]
 * (finite, >= 0, any unit), to one of `world` owners: owner[i] in [0, world).
 *  - Greedy longest-processing-time (LPT): matrices in decreasing cost
 *    (equal costs: lower index first), each to the owner with the least total
 *    so far (equal totals: lower rank).  Makespan <= (4/3 - 1/(3 world)) x the
 *    optimum (Graham's bound).
 *  - If 0 < count <= exact_limit (exact_limit <= MUON_PARTITION_EXACT_MAX), a
 *    depth-first branch and bound seeded with the LPT answer then replaces it
 *    by an assignment of strictly smaller makespan if one exists.  The search
 *    stops after MUON_PARTITION_NODE_BUDGET nodes, keeping the best found, so
 *    the answer is optimal unless the budget ran out, and never worse than LPT.
 *  - Deterministic in (cost, world, exact_limit): every rank computes the same
 *    placement with no communication.
 * load[world] (may be NULL) receives each owner's total cost.
 * Errors (nothing written): MUON_ERR_ARG for count < 0, world < 1, NULL
 * cost/owner with count > 0, exact_limit out of range, or a cost that is
 * negative, NaN or infinite.
 */
MUON_API muon_status muon_partition(const double* cost, int count, int world, int exact_limit,
                                    int32_t* owner, double* load);

/* Thread-local message of the last failed call on this thread ("" if none). */
MUON_API const char* muon_last_error(void);

/* Library version string. */
MUON_API const char* muon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MUON_NS_H */
