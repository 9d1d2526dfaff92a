/*
 * flashot.h -- C ABI of the GB300 (sm_103a) streaming log-domain Sinkhorn library.
 *
 * Problem (FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract; SAI
 * replication review, "Summary"): entropic optimal transport between point clouds
 * X (n x d) and Y (m x d) with weights a (n), b (m), squared Euclidean cost
 * C_ij = |x_i - y_j|^2 and regularisation eps, solved by stabilized log-domain Sinkhorn.
 * The dual potentials are updated as row-wise log-sum-exps of biased dot-product scores
 * (the review's "Weaknesses" names the cost form c_ij = alpha_i + beta_j - Q_i^T K_j):
 *
 *   F (f-update): f_i = |x_i|^2 - eps * LSE_j[ (2<x_i,y_j> - |y_j|^2 + g_j)/eps + log b_j ]
 *   G (g-update): g_j = |y_j|^2 - eps * LSE_i[ (2<x_i,y_j> - |x_i|^2 + f_i)/eps + log a_i ]
 *   plan:         P_ij = a_i b_j exp((f_i + g_j - C_ij) / eps)     (never materialised)
 *
 * Conventions shared by every entry point below.
 *  - Pointers named X, Y, a, b, f, g, V, out, grad, h, loss and ws are CUDA DEVICE
 *    pointers owned by the caller, on the current CUDA device. Matrices are row-major
 *    and contiguous (X: n*d floats, Y: m*d floats). Vectors are contiguous.
 *  - a == NULL (b == NULL) means uniform weights 1/n (1/m). Weights are used as given:
 *    they are not renormalised; a zero weight removes its point; negative or NaN weights
 *    give undefined results unless FLASHOT_VALIDATE is set (the check synchronises).
 *  - Work is enqueued asynchronously on `stream` (NULL = legacy default stream). The
 *    library allocates no device memory: all scratch comes from the caller's workspace
 *    `ws` of `ws_bytes` bytes, at least flashot_workspace_bytes(...) for the same
 *    (n, m, d, k, flags), 256-byte aligned. A workspace must not be used by two calls
 *    that may run concurrently.
 *  - Every call returns FLASHOT_OK (0) or a negative status; no exception or abort
 *    crosses the ABI. Argument errors are detected on the host before anything is
 *    enqueued. FLASHOT_ERR_CUDA reports a failed launch; its cudaError_t is returned
 *    by flashot_last_cuda_error() on the calling thread.
 *  - Sizes: n, m >= 1, 1 <= d <= 4096, 1 <= k <= 4096, eps > 0 and finite.
 *  - Arithmetic: scores and log-sum-exps are accumulated in fp32 (exp2 on the SFU);
 *    the <x, y> contraction runs in the precision chosen by the FLASHOT_PREC_* flag.
 *    Norms |x|^2, |y|^2 are taken from the fp32 inputs. The loss is reduced in fp64.
 */
#ifndef FLASHOT_H_
#define FLASHOT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st *flashot_stream_t;

/* ---- status codes ------------------------------------------------------------------ */
#define FLASHOT_OK                        0
#define FLASHOT_ERR_INVALID_ARG          -1  /* NULL pointer, size or eps out of range   */
#define FLASHOT_ERR_ALIGNMENT            -2  /* ws not 256-byte aligned                   */
#define FLASHOT_ERR_WORKSPACE_TOO_SMALL  -3  /* ws_bytes < flashot_workspace_bytes(...)   */
#define FLASHOT_ERR_CUDA                 -4  /* a CUDA runtime call or launch failed      */
#define FLASHOT_ERR_DEVICE_TIMEOUT       -5  /* a kernel gave up a bounded wait           */
#define FLASHOT_ERR_UNSUPPORTED_DEVICE   -6  /* current device is not sm_103              */
#define FLASHOT_ERR_NOT_IMPLEMENTED      -7  /* combination of flags not available        */

/* ---- flags ------------------------------------------------------------------------- */
/* Precision of the <x_i, y_j> contraction (low 4 bits). */
#define FLASHOT_PREC_AUTO   0x0  /* FP32 for d < 32, TF32 tensor cores for d >= 32        */
#define FLASHOT_PREC_FP32   0x1  /* fp32 FMA on CUDA cores (any d)                         */
#define FLASHOT_PREC_TF32   0x2  /* tcgen05 kind::tf32, inputs rounded to tf32 (nearest)   */
#define FLASHOT_PREC_BF16   0x3  /* tcgen05 kind::f16 with bf16 operands (nearest)         */
/* tcgen05 kind::tf32 on split operands: x = hi + lo (hi = tf32(x), lo = tf32(x - hi)), packed
 * along K as X = [hi | hi | lo], Y = [hi | lo | hi], so one contraction over 3x the K
 * returns hi.hi + hi.lo + lo.hi (about fp32 accuracy for the scores; 3x the MMA work). The
 * second contraction of transport application / gradient stays single tf32. */
#define FLASHOT_PREC_TF32X3 0x4
#define FLASHOT_PREC_MASK   0xF
/* solve: start from the g passed in (warm start / resume) instead of g = 0. */
#define FLASHOT_WARM_START  0x10
/* The workspace already holds the packed X, Y, norms and log-weights written by an
 * earlier call with the same X, Y, a, b, n, m, d, flags and workspace; skip re-packing. */
#define FLASHOT_REUSE_PACK  0x20
/* solve: symmetric (averaged) schedule, f' = (f + F(g))/2 and g' = (g + G(f))/2 from the
 * same previous iterate (the review's "Strengths": symmetric-vs-alternating comparison).
 * Starts from f = g = 0, or with FLASHOT_WARM_START from the f and g passed in. When X == Y
 * and a == b (the same pointers) without a warm start, f == g at every iteration, and the
 * solve runs one pass per iteration instead of two. */
#define FLASHOT_SYMMETRIC   0x40
/* Check the inputs before any work: every coordinate of X and Y finite, every weight of a
 * and b (when given) finite and non-negative. One device pass over X, Y, a, b and a read of
 * its result, which SYNCHRONISES `stream`; a violation returns FLASHOT_ERR_INVALID_ARG with
 * nothing else enqueued. Accepted by every entry point that reads X and Y. */
#define FLASHOT_VALIDATE    0x80

/* ---- library information ------------------------------------------------------------ */
int flashot_version(void);                       /* major*10000 + minor*100 + patch      */
const char *flashot_status_string(int status);   /* static string, never NULL            */
int flashot_last_cuda_error(void);               /* cudaError_t of the last ERR_CUDA      */

/* Device-side status word kept in the workspace: synchronises `stream`, returns
 * FLASHOT_ERR_DEVICE_TIMEOUT if a kernel that used this workspace gave up a bounded
 * wait since the last call (and clears the word), else FLASHOT_OK, or ERR_CUDA. */
int flashot_workspace_status(void *ws, flashot_stream_t stream);

/* ---- diagnostics (no effect on results) ----------------------------------------------- */
/* Number of kernels this library has launched in this process (all devices, all threads). */
uint64_t flashot_launch_count(void);

/* Kernel classes for the timer below. */
#define FLASHOT_KERNEL_LSE    0  /* streaming log-sum-exp half-step pass (the hot kernel)  */
#define FLASHOT_KERNEL_WSUM   1  /* streaming weighted-sum pass (apply, Hadamard, gradient) */
#define FLASHOT_KERNEL_OTHER  2  /* packing, biases, LSE combine, loss reduction           */

/* Per-launch timing on the launching stream: flashot_timer_start(cap) creates cap CUDA event
 * pairs (host-side objects, no device memory) and from then on records one pair around each
 * kernel launch, until cap pairs are used. flashot_timer_read(cls, &launches, &ms) waits for
 * the recorded events and returns, for kernel class cls, the number of timed launches and
 * their summed duration in milliseconds. flashot_timer_stop() destroys the events. Not for
 * concurrent use from several threads. Returns a FLASHOT_* status. */
int flashot_timer_start(int cap);
int flashot_timer_read(int kernel_class, int64_t *launches, double *total_ms);
int flashot_timer_stop(void);

/* Self-test of the bounded waits the tensor-core kernels use: one CTA waits on an mbarrier
 * that nothing ever arrives on, then one thread waits, as at the grid barrier of the
 * persistent solve, for a word of ws (byte 128, zeroed first) that nothing writes; each
 * gives up after limit_ns (1e6 .. 2e9 ns) and records the timeout in the status word of ws
 * (>= 256 bytes, 256-byte aligned, device memory): bit 0 for any wait, bit 1 also for the
 * grid-barrier wait. The call returns normally; flashot_workspace_status(ws, stream) then
 * reports FLASHOT_ERR_DEVICE_TIMEOUT and the context stays usable. No fault, no trap. */
int flashot_selftest_bounded_wait(void *ws, int64_t limit_ns, flashot_stream_t stream);

/* Bytes of workspace needed for calls with these sizes and flags. k is the column count
 * of V for flashot_transport_apply (0 if that call is not used). Returns 0 on invalid
 * sizes. The same workspace serves every entry point with equal (n, m, d, k, flags). */
size_t flashot_workspace_bytes(int64_t n, int64_t m, int64_t d, int64_t k, int flags);

/* ---- the hot path ------------------------------------------------------------------- */

/*
 * Full alternating solve (FlashSinkhorn abstract: stabilized log-domain Sinkhorn; the
 * review "Summary": fused f^/g^ updates that write only the potentials back).
 * For s = 0..n_stages-1 and it = 0..iters_per_stage-1: f = F(g), then g = G(f), at
 * eps = eps_sched[s]. g starts at 0 unless FLASHOT_WARM_START is set (then the g passed
 * in is read first). eps_sched is a HOST array of n_stages floats (annealing schedule).
 * Writes f (n floats), g (m floats) and, if loss != NULL, *loss (ONE device double) =
 * sum_i a_i f_i + sum_j b_j g_j after the final g-update.
 * Launches: one LSE pass and one merge per half-step; for tensor-core precisions with a
 * short contraction (bf16 d <= 192, tf32 d <= 96, split tf32 d <= 64), at most 32 eps
 * stages and at least 1.5 tiles of 128 x 256 scores per SM and pass, every half-step runs
 * in one cooperative launch instead (all its CTAs, at most one per SM, resident together;
 * a grid-wide barrier separates the passes). Both give the same bits.
 * FLASHOT_SHORT_SOLVE=0 in the environment keeps the per-pass launches, =1 takes the
 * single launch whenever the contraction and stage count allow.
 */
int flashot_sinkhorn_solve(const float *X, const float *Y, const float *a, const float *b,
                           int64_t n, int64_t m, int64_t d, const float *eps_sched,
                           int n_stages, int iters_per_stage, int flags, float *f, float *g,
                           double *loss, void *ws, size_t ws_bytes, flashot_stream_t stream);

/*
 * Convergence-driven alternating solve at one eps (the review's "Strengths": the low-eps
 * regime run to a marginal tolerance; its "Summary": the fused f^/g^ updates). Iteration
 * k = 1, 2, ... is f = F(g), then g = G(f), from g = 0. After a g-update the column sums of
 * the plan equal b, so an iterate's error is its row-marginal L1 error
 *     err = sum_i |sum_j P_ij - a_i| = sum_i a_i |exp((f_i - F(g)_i) / eps) - 1|,
 * which the f-update of iteration k yields for iterate k-1 inside its LSE combine (no
 * extra pass over the points). On check iterations (k >= 2, k % check_every == 0) the
 * error is reduced in fp64 on the device and read back (this SYNCHRONISES `stream`), and
 * the solve stops after iteration k if err < tol; otherwise after max_iters iterations.
 * The returned iterate's error is at most the reported one (marginal errors of Sinkhorn
 * iterates do not increase).
 *   tol >= 0 (0: never stop early); max_iters >= 1; check_every >= 1.
 *   iters_done: HOST int, iterations run. err: HOST double or NULL, the last measured
 *   error (-1 if none). err_hist: HOST array of max_iters / check_every doubles or NULL;
 *   entry k / check_every - 1 receives the error measured at check iteration k.
 *   loss: device double or NULL, <a, f> + <b, g> of the returned iterate.
 * flags: a precision and optionally FLASHOT_REUSE_PACK and FLASHOT_VALIDATE; anything else
 * returns FLASHOT_ERR_NOT_IMPLEMENTED. The error is formed from fp32 potentials, so it cannot
 * resolve much below ~1e-6 * max|f| / eps (the fp32 spacing of f, relative to eps).
 * Returns FLASHOT_ERR_DEVICE_TIMEOUT (and stops) if a kernel gave up a bounded wait.
 * Launches: as flashot_sinkhorn_solve; for short tensor-core contractions with
 * check_every >= 4, the iterations up to each check run as one cooperative launch (the same
 * bits and decisions).
 */
int flashot_sinkhorn_solve_tol(const float *X, const float *Y, const float *a,
                               const float *b, int64_t n, int64_t m, int64_t d, float eps,
                               double tol, int max_iters, int check_every, int flags,
                               float *f, float *g, double *loss, int *iters_done,
                               double *err, double *err_hist, void *ws, size_t ws_bytes,
                               flashot_stream_t stream);

/* One f-update (review "Summary": the f^ update): f = F(g). Reads g (m), writes f (n). */
int flashot_sinkhorn_step_f(const float *X, const float *Y, const float *b, const float *g,
                            int64_t n, int64_t m, int64_t d, float eps, int flags, float *f,
                            void *ws, size_t ws_bytes, flashot_stream_t stream);

/* One g-update (the g^ update): g = G(f). Reads f (n), writes g (m). */
int flashot_sinkhorn_step_g(const float *X, const float *Y, const float *a, const float *f,
                            int64_t n, int64_t m, int64_t d, float eps, int flags, float *g,
                            void *ws, size_t ws_bytes, flashot_stream_t stream);

/*
 * Debiased Sinkhorn divergence S(a, b) = OT(a, b) - OT(a, a)/2 - OT(b, b)/2 (the review's
 * "Reproducibility & code": the debiased-Sinkhorn sweep of the OTDD pipeline), each OT
 * term the dual loss of a solve of X against Y, X against X and Y against Y with the same
 * eps schedule, iteration count and flags (FLASHOT_SYMMETRIC selects the schedule).
 * out: FOUR device doubles {S, OT(a,b), OT(a,a), OT(b,b)}. ws must hold at least
 * flashot_divergence_workspace_bytes(n, m, d, flags) bytes.
 */
size_t flashot_divergence_workspace_bytes(int64_t n, int64_t m, int64_t d, int flags);
int flashot_sinkhorn_divergence(const float *X, const float *Y, const float *a, const float *b,
                                int64_t n, int64_t m, int64_t d, const float *eps_sched,
                                int n_stages, int iters_per_stage, int flags, double *out,
                                void *ws, size_t ws_bytes, flashot_stream_t stream);

/* Dual loss sum_i a_i f_i + sum_j b_j g_j, reduced in fp64 into ONE device double. */
int flashot_dual_loss(const float *a, const float *b, const float *f, const float *g,
                      int64_t n, int64_t m, double *loss, void *ws, size_t ws_bytes,
                      flashot_stream_t stream);

/*
 * Matrix-free transport application (review "Summary" (ii): transport-vector and
 * transport-matrix application) with P built on the fly from (f, g):
 *   transpose == 0: out (n x k) = P V,    V is m x k row-major;
 *   transpose != 0: out (m x k) = P^T V,  V is n x k row-major.
 * out must not alias V.
 */
int flashot_transport_apply(const float *X, const float *Y, const float *a, const float *b,
                            const float *f, const float *g, int64_t n, int64_t m, int64_t d,
                            float eps, const float *V, int64_t k, int transpose, float *out,
                            int flags, void *ws, size_t ws_bytes, flashot_stream_t stream);

/* Hadamard-weighted transport with W = X Y^T (review "Summary" (ii)):
 * h_i = sum_j P_ij <x_i, y_j>, h has n floats. */
int flashot_transport_hadamard_xy(const float *X, const float *Y, const float *a,
                                  const float *b, const float *f, const float *g, int64_t n,
                                  int64_t m, int64_t d, float eps, float *h, int flags,
                                  void *ws, size_t ws_bytes, flashot_stream_t stream);

/*
 * Gradient of the OT loss w.r.t. X as a barycentric projection (review "Summary" (i):
 * the gradient as a residual "attention output"; "Weaknesses": exact for the
 * marginal-perturbed problem at early-stopped potentials). With f~ = F(g) computed
 * internally (softmax over j of the F-step scores):
 *   grad_i = 2 a_i (x_i - yhat_i),  yhat_i = sum_j softmax_j(s_ij) y_j.
 * grad has n x d floats (row-major).
 */
int flashot_ot_grad_x(const float *X, const float *Y, const float *a, const float *b,
                      const float *g, int64_t n, int64_t m, int64_t d, float eps, float *grad,
                      int flags, void *ws, size_t ws_bytes, flashot_stream_t stream);

/*
 * Hessian-vector product of the OT loss w.r.t. X (the review's "Summary" (iii): a streaming
 * HVP oracle for O((n + m) d)-memory Newton-CG, through a Schur solve with streaming P and
 * P^T products; "Strengths": parity against a dense Moore-Penrose HVP).
 * At the potentials (f, g), with P_ij = a_i b_j exp((f_i + g_j - |x_i - y_j|^2)/eps),
 * r = P 1 and c = P^T 1, the Lagrangian L = <a,f> + <b,g> - eps sum_ij (P_ij - a_i b_j) has
 *   L_XX   block i: 2 r_i I - (4/eps) sum_j P_ij (x_i - y_j)(x_i - y_j)^T,
 *   L_Xf (i, i) = (2/eps) sum_j P_ij (x_i - y_j),  L_Xg (i, j) = (2/eps) P_ij (x_i - y_j),
 *   L_phiphi = -K/eps,  K = [[diag r, P], [P^T, diag c]],
 * and out = H V = L_XX V + L_Xphi (eps K^+ L_phiX V) (the potentials' response by the
 * implicit function theorem; K^+ fixes the gauge direction, which L_Xphi annihilates). At
 * optimal potentials this is the Hessian of OT_eps(X, Y) applied to V.
 * K (u, z) = w is solved by conjugate gradients on the Schur complement
 * S = diag(c) - P^T diag(1/r) P with preconditioner diag(c), stopping when the residual
 * falls below cg_tol times the initial one (checked after every iteration, which
 * SYNCHRONISES `stream`) or after cg_max_iters iterations. Each CG iteration is two
 * streaming passes (P p and P^T t); the rest is five more passes and O((n + m) d) work.
 *   V, out: n x d device floats (out must not alias V). f (n), g (m): device floats.
 *   cg_iters, cg_rel_residual: HOST pointers or NULL (iterations run; final residual ratio).
 *   flags: FLASHOT_PREC_AUTO or FLASHOT_PREC_FP32 (the passes run on fp32 CUDA cores),
 *   optionally FLASHOT_REUSE_PACK and FLASHOT_VALIDATE; anything else returns
 *   FLASHOT_ERR_NOT_IMPLEMENTED.
 *   ws: at least flashot_hvp_workspace_bytes(n, m, d, flags) bytes.
 */
size_t flashot_hvp_workspace_bytes(int64_t n, int64_t m, int64_t d, int flags);
int flashot_ot_hvp_x(const float *X, const float *Y, const float *a, const float *b,
                     const float *f, const float *g, int64_t n, int64_t m, int64_t d,
                     float eps, const float *V, float *out, double cg_tol, int cg_max_iters,
                     int flags, int *cg_iters, double *cg_rel_residual, void *ws,
                     size_t ws_bytes, flashot_stream_t stream);

/*
 * Batched Sinkhorn-Knopp projection of tiny matrices onto the doubly stochastic matrices
 * ("Fused & Furious: Sinkhorn Triton Kernels", section II: the KL projection of M = exp(H)
 * onto the Birkhoff polytope; section III: one matrix per token, n = 4, n_iter = 20):
 *   M = exp(H_b), v = 1; n_iter times: u = 1 / (M v), v = 1 / (M^T u);
 *   P_b = diag(u) M diag(v)      (its columns sum to 1; its rows approach 1).
 *   H, P: B matrices of n x n fp32, row-major, contiguous, device memory; P may equal H
 *   (in place). 1 <= n <= 8, n_iter >= 1, B >= 0 (B = 0 does nothing). When n*n is a
 *   multiple of 4, H and P must be 16-byte aligned (else FLASHOT_ERR_ALIGNMENT).
 * Needs no workspace. Each matrix's largest logit is subtracted before exp (P does not
 * change); logits that lie more than about 87 below a matrix's largest underflow to 0 in
 * fp32, and a row or column of such zeros makes that matrix's P undefined. The scalings use
 * one SFU reciprocal (rcp.approx, about 1 ulp) per pair of sums, 1/s0 = s1 / (s0 s1), so
 * products of two row (or column) sums must stay in the fp32 range: logits of one matrix
 * should span less than about 40.
 */
int flashot_sinkhorn_knopp_batched(const float *H, int64_t B, int n, int n_iter, float *P,
                                   flashot_stream_t stream);

/*
 * Diagnostics of the plan defined by (f, g) (the review's "Summary": the dual potentials
 * define the plan P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps)), from three streaming passes
 * (P 1, P^T 1 and the Hadamard sums h_i = sum_j P_ij <x_i, y_j>) and one fp64 reduction:
 *   out[0] primal objective <C, P> + eps KL(P | a b^T)  (KL with the -sum P + sum a b terms)
 *   out[1] dual objective   <a, f> + <b, g> - eps (sum P - sum a sum b)
 *   out[2] transport cost   <C, P> = sum_i r_i |x_i|^2 + sum_j c_j |y_j|^2 - 2 sum_i h_i
 *   out[3] row-marginal L1 error    sum_i |r_i - a_i|,  r = P 1
 *   out[4] column-marginal L1 error sum_j |c_j - b_j|,  c = P^T 1
 *   out[5] mass sum P
 * At optimal potentials primal = dual and both errors vanish. out: SIX device doubles.
 * The passes run in the precision of flags (the fp32 path gives fp32-accurate sums; the
 * transport cost is a difference of larger terms). ws: at least
 * flashot_diagnostics_workspace_bytes(n, m, d, flags) bytes.
 */
size_t flashot_diagnostics_workspace_bytes(int64_t n, int64_t m, int64_t d, int flags);
int flashot_plan_diagnostics(const float *X, const float *Y, const float *a, const float *b,
                             const float *f, const float *g, int64_t n, int64_t m, int64_t d,
                             float eps, int flags, double *out, void *ws, size_t ws_bytes,
                             flashot_stream_t stream);

/* ---- allocation-free variant -------------------------------------------------------- */
/*
 * The paper has no counterpart to this entry point; it exists for callers that cannot give
 * the library a workspace: a host framework that owns all device memory through its own
 * fixed arena and forbids its plugins to call cudaMalloc, or a latency-critical loop where
 * a cudaMalloc / cudaFree (which may synchronise the device) is not acceptable.
 *
 * flashot_sinkhorn_step_f_noalloc computes the same f = F(g) as flashot_sinkhorn_step_f
 * (same arguments, minus ws / ws_bytes) and allocates nothing: its scratch is one array of
 * FLASHOT_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library as device memory. The
 * array is reserved in a context when the library's module that holds it is loaded there:
 * under CUDA's default lazy module loading that is the first call of either function below
 * in that context; with CUDA_MODULE_LOADING=EAGER it is when the context is created. It
 * stays reserved until the context is destroyed. X, Y, b, g and f are still the caller's
 * device buffers.
 *  - Sizes whose workspace (flashot_workspace_bytes(n, m, d, 0, flags)) exceeds 64 MiB are
 *    rejected with FLASHOT_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *  - flags are those of flashot_sinkhorn_step_f (precision bits, FLASHOT_VALIDATE), except
 *    that FLASHOT_REUSE_PACK is ignored: the array keeps whatever the previous call left in
 *    it, so the inputs are always packed afresh (which also clears the status word).
 *  - Every call looks up the array's device address in the current context
 *    (cudaGetSymbolAddress), after checking that the current device is sm_103. The first
 *    call in a context also loads the module; make it before any stream capture.
 *  - All calls on a device share the one array: calls whose GPU work may overlap (other
 *    streams, other host threads) race on it and give undefined results. Serialise them.
 *
 * flashot_noalloc_status(stream) is flashot_workspace_status for that array: it
 * synchronises `stream` and returns FLASHOT_ERR_DEVICE_TIMEOUT if a kernel of an earlier
 * flashot_sinkhorn_step_f_noalloc call in the current context gave up a bounded wait (and
 * clears the word), else FLASHOT_OK; FLASHOT_ERR_UNSUPPORTED_DEVICE or FLASHOT_ERR_CUDA if
 * the array cannot be reached. It allocates nothing either.
 */
#define FLASHOT_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int flashot_sinkhorn_step_f_noalloc(const float *X, const float *Y, const float *b,
                                    const float *g, int64_t n, int64_t m, int64_t d, float eps,
                                    int flags, float *f, flashot_stream_t stream);
int flashot_noalloc_status(flashot_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FLASHOT_H_ */
