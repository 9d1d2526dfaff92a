// flashot.cu -- host side of the C ABI declared in include/flashot.h.
//
// Argument validation, workspace layout, pass launchers and the alternating solve
// driver for streaming log-domain Sinkhorn (FlashSinkhorn: IO-Aware Entropic Optimal
// Transport on GPU, abstract and SAI replication review, "Summary"). Every step of the
// computation runs in the kernels of prep_kernels.cuh, fma_kernels.cuh and
// tc_kernels.cuh; this file only validates, carves the caller's workspace and enqueues.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cstdlib>

#include "flashot.h"
#include "common.cuh"
#include "fma_kernels.cuh"
#include "hvp_kernels.cuh"
#include "host_internal.h"
#include "prep_kernels.cuh"
#include "small_solve.h"
#include "tc_api.h"
#include "tc_solve_short.h"
#include "tc_wsum_pair.h"
#include "trace.h"
#include <vector>

namespace flashot {

// ---- launch accounting (diagnostics) ----------------------------------------------------
namespace {
std::atomic<uint64_t> g_launches{0};
struct EventTimer {
  bool on = false;
  int cap = 0, used = 0;
  std::vector<cudaEvent_t> ev;  // 2 per launch
  std::vector<int> cls;
};
EventTimer g_timer;
}  // namespace

void trace_before(int, cudaStream_t st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_timer.on && g_timer.used < g_timer.cap) cudaEventRecord(g_timer.ev[2 * g_timer.used], st);
}

void trace_after(int kernel_class, cudaStream_t st) {
  if (g_timer.on && g_timer.used < g_timer.cap) {
    cudaEventRecord(g_timer.ev[2 * g_timer.used + 1], st);
    g_timer.cls[g_timer.used] = kernel_class;
    ++g_timer.used;
  }
}

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kVersion = 10000;  // 1.0.0
constexpr int64_t kMaxRows = int64_t(1) << 28;
constexpr int64_t kMaxD = 4096;
constexpr int64_t kMaxK = 4096;
constexpr int kMaxSplits = 64;
constexpr int kRowPad = 256;  // the tensor-core LSE pass tiles columns by 256

inline int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }
inline int64_t ceil_div(int64_t x, int64_t q) { return (x + q - 1) / q; }

// ---- device checks -------------------------------------------------------------------
struct DeviceInfo {
  int ok = 0;  // 0 unknown, 1 sm_103, 2 other
  int sms = 0;
};
DeviceInfo g_dev[64];

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return FLASHOT_ERR_CUDA;
}

int current_device(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return FLASHOT_ERR_UNSUPPORTED_DEVICE;
  DeviceInfo& di = g_dev[dev];
  if (di.ok == 0) {
    int maj = 0, mnr = 0, sms_ = 0;
    if ((e = cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&mnr, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&sms_, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    di.sms = sms_;
    di.ok = (maj == 10 && mnr == 3) ? 1 : 2;
  }
  if (di.ok != 1) return FLASHOT_ERR_UNSUPPORTED_DEVICE;
  *sms = di.sms;
  return FLASHOT_OK;
}

// A device pointer of the current context (device or managed memory).
bool is_device_ptr(const void* p) {
  if (p == nullptr) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

bool opt_device_ptr(const void* p) { return p == nullptr || is_device_ptr(p); }

// ---- problem geometry and workspace layout ------------------------------------------
struct Geometry {
  int64_t n, m, d, k;
  int prec;          // FLASHOT_PREC_{FP32,TF32,BF16}
  bool small;        // FP32 path with d_pad <= 32 (registers hold a whole point)
  int64_t n_pad, m_pad;
  int64_t dpf;       // d_pad of the fp32 packing (FP32 path)
  int64_t dpt;       // d_pad of the tensor-core packing (TF32/BF16 path)
  int es;            // element size of the tensor-core packing
};

int resolve_prec(int flags, int64_t d) {
  const int p = flags & FLASHOT_PREC_MASK;
  if (p == FLASHOT_PREC_AUTO) return d < 32 ? FLASHOT_PREC_FP32 : FLASHOT_PREC_TF32;
  return p;
}

bool make_geometry(int64_t n, int64_t m, int64_t d, int64_t k, int flags, Geometry* g) {
  if (n < 1 || m < 1 || d < 1 || n > kMaxRows || m > kMaxRows || d > kMaxD || k < 0 ||
      k > kMaxK)
    return false;
  const int p = resolve_prec(flags, d);
  if (p != FLASHOT_PREC_FP32 && p != FLASHOT_PREC_TF32 && p != FLASHOT_PREC_BF16 &&
      p != FLASHOT_PREC_TF32X3)
    return false;
  g->n = n;
  g->m = m;
  g->d = d;
  g->k = k;
  g->prec = p;
  g->n_pad = round_up(n, kRowPad);
  g->m_pad = round_up(m, kRowPad);
  g->small = d <= 32;
  g->dpf = g->small ? round_up(d, 4) : round_up(d, 32);
  g->es = (p == FLASHOT_PREC_BF16) ? 2 : 4;
  // One 128-byte swizzle row per k-chunk. Split tf32 packs the three parts of the
  // coordinates back to back ([hi | hi | lo] against [hi | lo | hi], d elements each) and
  // pads the 3d elements once.
  g->dpt = round_up(p == FLASHOT_PREC_TF32X3 ? 3 * d : d, 128 / g->es);
  return true;
}

struct Layout {
  size_t status, xp, yp, xq, yq, vtq, wsp, tsp, alpha, beta, wa, wb, la2, lb2, biasF, biasG,
      ftilde, lse2, partial, loss, sync, total;
};

// The stream-K partials of an LSE pass: up to kMaxSplits (max, sum) pairs per row.
size_t partial_bytes(const Geometry& g) {
  return (size_t)kMaxSplits * (size_t)std::max(g.n_pad, g.m_pad) * sizeof(float2);
}

Layout make_layout(const Geometry& g) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = (off + bytes + 1023) / 1024 * 1024;
    return o;
  };
  const size_t np = (size_t)g.n_pad, mp = (size_t)g.m_pad;
  L.status = take(256);
  if (g.prec == FLASHOT_PREC_FP32) {
    L.xp = take(np * g.dpf * 4);
    L.yp = take(mp * g.dpf * 4);
  } else {
    L.xq = take(np * g.dpt * g.es);
    L.yq = take(mp * g.dpt * g.es);
  }
  L.alpha = take(np * 4);
  L.beta = take(mp * 4);
  L.wa = take(np * 4);
  L.wb = take(mp * 4);
  L.la2 = take(np * 4);
  L.lb2 = take(mp * 4);
  L.biasF = take(mp * 4);
  L.biasG = take(np * 4);
  L.ftilde = take(np * 4);
  L.lse2 = take(std::max(np, mp) * 4);
  L.partial = take(partial_bytes(g));
  L.loss = take(64);
  // Arrival counters and grid barrier of the persistent short-contraction solve.
  if (g.prec != FLASHOT_PREC_FP32) L.sync = take(tc_short_solve_sync_bytes(g.n_pad, g.m_pad));
  // Last, so that every offset above is independent of k: the transposed right operand
  // of the tensor-core weighted sums (V^T for apply, Y^T for the gradient), padded to
  // multiples of 256 output columns.
  if (g.prec != FLASHOT_PREC_FP32)
    L.vtq = take(std::max((size_t)std::max(round_up(g.k, 256), round_up(g.d, 256)) *
                              std::max(np, mp) * g.es,
                          tc_wsum_pair_vt_bytes(g.prec, (int64_t)std::max(np, mp),
                                                std::max(g.k, g.d))));
  // Partial sums of the stream-K weighted-sum passes (bf16 single-CTA, and the CTA-pair pass
  // of every tensor-core precision).
  if (g.prec != FLASHOT_PREC_FP32)
    L.wsp = take(std::max(tc_wsum2_scratch_bytes((int64_t)std::max(np, mp), std::max(g.k, g.d)),
                          tc_wsum_pair_scratch_bytes((int64_t)std::max(np, mp),
                                                     std::max(g.k, g.d))));
  // Partial sums of the tf32 weighted-sum passes' column splits.
  if (g.prec == FLASHOT_PREC_TF32 || g.prec == FLASHOT_PREC_TF32X3)
    L.tsp = take(tc_wsum_split_bytes((int64_t)std::max(np, mp), std::max(g.k, g.d)));
  L.total = off + 256;
  return L;
}

// Everything a pass needs, resolved from the caller's workspace.
struct Ctx {
  Geometry g;
  Layout L;
  char* ws;
  int sms;
  cudaStream_t st;
  template <typename T>
  T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
};

int check_ws(const Geometry& g, void* ws, size_t ws_bytes, Layout* L) {
  if (!is_device_ptr(ws)) return FLASHOT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FLASHOT_ERR_ALIGNMENT;
  *L = make_layout(g);
  if (ws_bytes < L->total) return FLASHOT_ERR_WORKSPACE_TOO_SMALL;
  return FLASHOT_OK;
}

bool eps_ok(float eps) { return std::isfinite(eps) && eps > 0.0f; }

int launch_check() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FLASHOT_OK : cuda_fail(e);
}

inline unsigned grid1(int64_t total, int threads) {
  int64_t b = ceil_div(total, threads);
  return (unsigned)std::min<int64_t>(std::max<int64_t>(b, 1), 1 << 20);
}

// ---- packing ---------------------------------------------------------------------------
int pack_inputs(const Ctx& c, const float* X, const float* Y, const float* a, const float* b) {
  const Geometry& g = c.g;
  const int T = 256;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    weights_kernel<<<grid1(g.n_pad, T), T, 0, c.st>>>(a, g.n, g.n_pad, c.at<float>(c.L.wa),
                                                      c.at<float>(c.L.la2), c.at<unsigned>(c.L.status));
  }
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    weights_kernel<<<grid1(g.m_pad, T), T, 0, c.st>>>(b, g.m, g.m_pad, c.at<float>(c.L.wb),
                                                      c.at<float>(c.L.lb2), nullptr);
  }
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    row_norms_kernel<<<grid1(g.n_pad * 32, T), T, 0, c.st>>>(X, g.n, g.d, g.n_pad,
                                                             c.at<float>(c.L.alpha));
  }
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    row_norms_kernel<<<grid1(g.m_pad * 32, T), T, 0, c.st>>>(Y, g.m, g.d, g.m_pad,
                                                             c.at<float>(c.L.beta));
  }
  const unsigned pg = (unsigned)std::min<int64_t>(ceil_div((g.n_pad + g.m_pad) * 64, T), c.sms * 8);
  if (g.prec == FLASHOT_PREC_FP32) {
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      pack_rows_kernel<PackKind::F32><<<pg, T, 0, c.st>>>(X, c.at<void>(c.L.xp), g.n, g.d, g.n_pad, g.dpf);
    }
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      pack_rows_kernel<PackKind::F32><<<pg, T, 0, c.st>>>(Y, c.at<void>(c.L.yp), g.m, g.d, g.m_pad, g.dpf);
    }
  } else {
    const int mode = g.prec == FLASHOT_PREC_BF16 ? 1 : (g.prec == FLASHOT_PREC_TF32X3 ? 2 : 0);
    int rc = tc_pack_inputs(mode, X, Y, g.n, g.m, g.d, g.n_pad, g.m_pad, g.dpt,
                            c.at<void>(c.L.xq), c.at<void>(c.L.yq), c.sms, c.st);
    if (rc != FLASHOT_OK) return rc;
  }
  return launch_check();
}

// FLASHOT_VALIDATE: X and Y finite, a and b (when given) finite and non-negative. Reads
// back one flag, so it synchronises the stream; returns FLASHOT_ERR_INVALID_ARG on a
// violation, before anything else is enqueued for the call.
int validate_inputs(const Ctx& c, int flags, const float* X, const float* Y, const float* a,
                    const float* b) {
  if (!(flags & FLASHOT_VALIDATE)) return FLASHOT_OK;
  unsigned* flag = reinterpret_cast<unsigned*>(c.at<char>(c.L.loss) + 48);
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(unsigned), c.st);
  if (e != cudaSuccess) return cuda_fail(e);
  const Geometry& g = c.g;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    validate_kernel<<<(unsigned)std::min<int64_t>(c.sms * 8, grid1(g.n * g.d + g.m * g.d, 256)),
                      256, 0, c.st>>>(X, X ? g.n * g.d : 0, Y, Y ? g.m * g.d : 0, a,
                                      a ? g.n : 0, b, b ? g.m : 0, flag);
  }
  int rc = launch_check();
  if (rc != FLASHOT_OK) return rc;
  unsigned word = 0;
  e = cudaMemcpyAsync(&word, flag, sizeof(word), cudaMemcpyDeviceToHost, c.st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c.st);
  if (e != cudaSuccess) return cuda_fail(e);
  return word ? FLASHOT_ERR_INVALID_ARG : FLASHOT_OK;
}

// bias = (pot - norms) log2e / eps + lw2 over one side (pot == NULL: pot = 0).
int launch_bias(const Ctx& c, const float* pot, bool x_side, float eps) {
  const Geometry& g = c.g;
  const int64_t rows = x_side ? g.n : g.m, rows_pad = x_side ? g.n_pad : g.m_pad;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    bias_kernel<<<grid1(rows_pad, 256), 256, 0, c.st>>>(
        pot, c.at<float>(x_side ? c.L.alpha : c.L.beta), c.at<float>(x_side ? c.L.la2 : c.L.lb2),
        rows, rows_pad, kLog2e / eps, c.at<float>(x_side ? c.L.biasG : c.L.biasF));
  }
  return launch_check();
}

// ---- one LSE half-step -----------------------------------------------------------------
// F-type (x_rows = true): rows X, columns Y, column bias biasF; writes out_pot (= f),
// the next pass's bias biasG (at eps_next), and optionally the row LSE (base 2).
// G-type: the same with X and Y exchanged.
// err_rows: see lse_combine_kernel (the convergence check; NULL otherwise).
int run_lse_pass(const Ctx& c, bool x_rows, float eps, float eps_next, float* out_pot,
                 bool write_next_bias, float* out_lse2, bool average = false,
                 float* err_rows = nullptr) {
  const Geometry& g = c.g;
  const int64_t n_rows = x_rows ? g.n : g.m;
  const int64_t rows_pad = x_rows ? g.n_pad : g.m_pad;
  const int64_t cols_pad = x_rows ? g.m_pad : g.n_pad;
  const float* colBias = c.at<float>(x_rows ? c.L.biasF : c.L.biasG);
  float2* partial = c.at<float2>(c.L.partial);
  const float kappa = 2.0f * kLog2e / eps;
  SplitInfo split{1, 1, 0, 0, 0, 128};
  int n_splits = 1;
  if (g.prec == FLASHOT_PREC_FP32) {
    const float* rowP = c.at<float>(x_rows ? c.L.xp : c.L.yp);
    const float* colP = c.at<float>(x_rows ? c.L.yp : c.L.xp);
    const int R = (g.dpf <= 16) ? 4 : 2;
    const int64_t rows_per_block = g.small ? (int64_t)kFmaThreads * R : kFmaThreads;
    const int64_t row_blocks = ceil_div(n_rows, rows_per_block);
    const int n_tiles = (int)(cols_pad / (g.small ? kFmaBN : 32));
    // CTAs to aim for: 16 per SM for the small-d kernel (several waves, 4 CTAs fit per SM at
    // d_pad = 16: the uneven finish of one wave's CTAs is evened out by the next; 20k x 80k,
    // d = 16 measured 5% faster than at 8 per SM), 8 for the generic one.
    const int64_t target = (int64_t)c.sms * (g.small ? 16 : 8);
    n_splits = (int)std::min<int64_t>({ceil_div(target, row_blocks), (int64_t)n_tiles,
                                        (int64_t)kMaxSplits});
    n_splits = std::max(n_splits, 1);
    const int tps = (int)ceil_div(n_tiles, n_splits);
    n_splits = (int)ceil_div(n_tiles, tps);
    split.n_splits = n_splits;
    dim3 grid((unsigned)row_blocks, (unsigned)n_splits);
    if (g.small) {
      TraceScope ts_(FLASHOT_KERNEL_LSE, c.st);
#define FLASHOT_LSE_SMALL(DPV, RV)                                                        \
  lse_fma_small_kernel<DPV, RV><<<grid, kFmaThreads, 0, c.st>>>(rowP, colP, colBias, n_rows, \
                                                                n_tiles, tps, kappa, partial, \
                                                                rows_pad)
      switch (g.dpf) {
        case 4: FLASHOT_LSE_SMALL(4, 4); break;
        case 8: FLASHOT_LSE_SMALL(8, 4); break;
        case 12: FLASHOT_LSE_SMALL(12, 4); break;
        case 16: FLASHOT_LSE_SMALL(16, 4); break;
        case 20: FLASHOT_LSE_SMALL(20, 2); break;
        case 24: FLASHOT_LSE_SMALL(24, 2); break;
        case 28: FLASHOT_LSE_SMALL(28, 2); break;
        case 32: FLASHOT_LSE_SMALL(32, 2); break;
        default: return FLASHOT_ERR_INVALID_ARG;
      }
#undef FLASHOT_LSE_SMALL
    } else {
      {
        TraceScope ts_(FLASHOT_KERNEL_LSE, c.st);
        lse_fma_generic_kernel<<<grid, kFmaThreads, 0, c.st>>>(rowP, colP, colBias, n_rows, g.dpf,
                                                               n_tiles, tps, kappa, partial,
                                                               rows_pad);
      }
    }
  } else {
    int rc = tc_lse_pass(g.prec == FLASHOT_PREC_BF16, c.at<void>(x_rows ? c.L.xq : c.L.yq),
                         c.at<void>(x_rows ? c.L.yq : c.L.xq), colBias, n_rows, rows_pad,
                         cols_pad, g.dpt, kappa, partial, kMaxSplits, c.sms,
                         c.at<unsigned>(c.L.status), &split, c.st);
    if (rc != FLASHOT_OK) return rc;
  }
  int rc = launch_check();
  if (rc != FLASHOT_OK) return rc;
  {
    // Programmatic dependent of the LSE pass (the kernel waits for it at entry): the launch
    // latency overlaps the pass's tail.
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid1(rows_pad, 256));
    cfg.blockDim = dim3(256);
    cfg.stream = c.st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CombineArgs args;
    args.rows = n_rows;
    args.rows_pad = rows_pad;
    args.norms = c.at<float>(x_rows ? c.L.alpha : c.L.beta);
    args.eps = eps;
    args.lw2 = c.at<float>(x_rows ? c.L.la2 : c.L.lb2);
    args.eps_ratio = eps / eps_next;
    args.out_pot = out_pot;
    args.next_bias = write_next_bias ? c.at<float>(x_rows ? c.L.biasG : c.L.biasF) : nullptr;
    args.out_lse2 = out_lse2;
    args.average = average ? 1 : 0;
    args.err_w = c.at<float>(x_rows ? c.L.wa : c.L.wb);
    args.err_rows = err_rows;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lse_combine_kernel, (const float2*)partial, split,
                                       (int64_t)rows_pad, args);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return launch_check();
}

// ---- weighted-sum passes (apply, grad, Hadamard, Hessian curvature) ----------------------
// rows on the X side unless `transpose`; rowBias / colBias as prepared by the caller.
// rowU (kWsumHessT only): the packed fp32 rows u_i (same layout as the packed row points).
int run_wsum_pass(const Ctx& c, int mode, bool transpose, float eps, const float* V, int64_t ldv,
                  int64_t k, const float* X, const float* Y, float* out, int64_t ldo,
                  const float* rowU = nullptr) {
  const Geometry& g = c.g;
  const bool x_rows = !transpose;
  const int64_t n_rows = x_rows ? g.n : g.m;
  const int64_t n_cols = x_rows ? g.m : g.n;
  const int64_t cols_pad = x_rows ? g.m_pad : g.n_pad;
  const float* colBias = c.at<float>(x_rows ? c.L.biasF : c.L.biasG);
  const float* rowBias = c.at<float>(x_rows ? c.L.biasG : c.L.biasF);
  const float* rowW = c.at<float>(x_rows ? c.L.wa : c.L.wb);
  const float kappa = 2.0f * kLog2e / eps;
  if (g.prec != FLASHOT_PREC_FP32) {
    if (mode == kWsumHessT) return FLASHOT_ERR_NOT_IMPLEMENTED;
    if (mode == kWsumGrad) {  // right operand of the second contraction: the column points
      V = x_rows ? Y : X;
      ldv = g.d;
      k = g.d;
    }
    // CTA pairs unless FLASHOT_WSUM_PAIRS=0 in the environment (single-CTA kernels, for
    // comparisons) or too few 2-CTA clusters fit.
    static const bool pairs_enabled = [] {
      const char* e = std::getenv("FLASHOT_WSUM_PAIRS");
      return !(e && e[0] == '0');
    }();
    if (pairs_enabled && tc_wsum_pair_available(c.sms))
      return tc_wsum_pair_pass(g.prec, mode, c.at<void>(x_rows ? c.L.xq : c.L.yq),
                               c.at<void>(x_rows ? c.L.yq : c.L.xq), colBias, rowBias, n_rows,
                               n_cols, x_rows ? g.n_pad : g.m_pad, cols_pad, g.d, g.dpt, kappa,
                               V, ldv, k, c.at<void>(c.L.vtq), c.at<void>(c.L.wsp), rowW, X,
                               out, ldo, c.sms, c.at<unsigned>(c.L.status), c.st);
    if (g.prec == FLASHOT_PREC_BF16)
      return tc_wsum2_pass(mode, c.at<void>(x_rows ? c.L.xq : c.L.yq),
                           c.at<void>(x_rows ? c.L.yq : c.L.xq), colBias, rowBias, n_rows, n_cols,
                           x_rows ? g.n_pad : g.m_pad, cols_pad, g.d, g.dpt, kappa, V, ldv, k,
                           c.at<void>(c.L.vtq), c.at<void>(c.L.wsp), rowW, X, out, ldo, c.sms,
                           c.at<unsigned>(c.L.status), c.st);
    return tc_wsum_pass(g.prec == FLASHOT_PREC_BF16, mode, c.at<void>(x_rows ? c.L.xq : c.L.yq),
                        c.at<void>(x_rows ? c.L.yq : c.L.xq), colBias, rowBias, n_rows, n_cols,
                        x_rows ? g.n_pad : g.m_pad, cols_pad, g.d, g.dpt, kappa, V, ldv, k,
                        c.at<void>(c.L.vtq), rowW, X, out, ldo, c.sms,
                        c.at<unsigned>(c.L.status), c.st, c.at<void>(c.L.tsp),
                        tc_wsum_split_bytes(std::max(g.n_pad, g.m_pad), std::max(g.k, g.d)));
  }
  const float* rowP = c.at<float>(x_rows ? c.L.xp : c.L.yp);
  const float* colP = c.at<float>(x_rows ? c.L.yp : c.L.xp);
  if (mode == kWsumGrad) {
    V = colP;
    ldv = g.dpf;
    k = g.d;
  }
  if (mode == kWsumHessT && rowU == nullptr) return FLASHOT_ERR_INVALID_ARG;
  const int64_t kk = (mode == kWsumHadamard) ? 1 : k;
  // One output column (a transport-vector application): a narrow accumulator.
  const bool narrow = (mode == kWsumApply && k == 1);
  // Up to 4 or 8 output columns (apply / curvature passes of small d): a 4- or 8-wide
  // accumulator.
  const bool mid = g.small && !narrow && k <= 8 && (mode == kWsumApply || mode == kWsumHessT);
  const bool quad = mid && k <= 4;
  const int KO = narrow ? 1 : (quad ? 4 : (mid ? 8 : 32));
  // Rows per thread of the small-d kernel: 4 for the narrow pass (2 when d_pad > 16), 2 for
  // the 4- and 8-wide ones.
  const int R = (g.small && narrow) ? (g.dpf <= 16 ? 4 : 2) : (mid ? 2 : 1);
  const int64_t row_blocks = ceil_div(n_rows, (int64_t)kFmaThreads * R);
  const int64_t k_groups = ceil_div(kk, KO);
  const int n_tiles = (int)(cols_pad / 32);
  // Column splits for the small-d kernel when rows x output groups give fewer than 16 CTAs
  // per SM (two waves of the 8 that fit at d_pad = 4: CTAs finish unevenly, and a second
  // wave evens the SMs' loads; measured 5% faster than one wave on 50k x 50k, d = 3); the
  // partials ([split][row][kp] floats) live in the workspace's partial region.
  int n_splits = 1, tps = n_tiles, kp = 0;
  if (g.small) {
    kp = (int)(mode == kWsumHadamard ? 1 : k_groups * KO) + 1;
    const int64_t cap_floats = (int64_t)kMaxSplits * std::max(g.n_pad, g.m_pad) * 2;
    const int64_t rows_pad_ = x_rows ? g.n_pad : g.m_pad;
    const int64_t max_splits = std::min<int64_t>(cap_floats / (rows_pad_ * kp), n_tiles);
    const int64_t want = ceil_div((int64_t)c.sms * 16, row_blocks * k_groups);
    n_splits = (int)std::max<int64_t>(1, std::min(want, max_splits));
    tps = (int)ceil_div(n_tiles, n_splits);
    n_splits = (int)ceil_div(n_tiles, tps);
  }
  float* part = n_splits > 1 ? c.at<float>(c.L.partial) : nullptr;
  const int64_t rows_pad = x_rows ? g.n_pad : g.m_pad;
  dim3 grid((unsigned)row_blocks, (unsigned)k_groups, (unsigned)n_splits);
  {
  TraceScope ts_(FLASHOT_KERNEL_WSUM, c.st);
  if (g.small) {
#define FLASHOT_WSUM_SMALL(DPV, MODEV, KOV, RV)                                              \
  wsum_fma_small_kernel<DPV, MODEV, KOV, RV><<<grid, kFmaThreads, 0, c.st>>>(                \
      rowP, colP, colBias, rowBias, n_rows, n_cols, n_tiles, kappa, V, ldv, k, rowW, X, g.d, \
      out, ldo, rowU, tps, part, rows_pad, kp)
#define FLASHOT_WSUM_PAIR_F(DPV, MODEV, KOV, RV, FOLD)                                       \
  wsum_fma_pair_kernel<DPV, MODEV, KOV, RV, FOLD><<<grid, kFmaThreads, 0, c.st>>>(           \
      rowP, colP, colBias, rowBias, n_rows, n_cols, n_tiles, kappa, V, ldv, k, rowW, X, g.d, \
      out, ldo, rowU, tps, part, rows_pad, kp)
  // the row bias rides in the first padding lane when there is one
#define FLASHOT_WSUM_PAIR(DPV, MODEV, KOV, RV)                                               \
  do {                                                                                       \
    if (g.d < (DPV)) FLASHOT_WSUM_PAIR_F(DPV, MODEV, KOV, RV, true);                         \
    else FLASHOT_WSUM_PAIR_F(DPV, MODEV, KOV, RV, false);                                    \
  } while (0)
#define FLASHOT_WSUM_MODES(DPV)                                                     \
  case DPV:                                                                         \
    if (narrow) FLASHOT_WSUM_PAIR(DPV, kWsumApply, 1, ((DPV) <= 16 ? 4 : 2));       \
    else if (quad && mode == kWsumApply) FLASHOT_WSUM_PAIR(DPV, kWsumApply, 4, 2);  \
    else if (quad) FLASHOT_WSUM_PAIR(DPV, kWsumHessT, 4, 2);                        \
    else if (mid && mode == kWsumApply) FLASHOT_WSUM_PAIR(DPV, kWsumApply, 8, 2);   \
    else if (mid) FLASHOT_WSUM_PAIR(DPV, kWsumHessT, 8, 2);                         \
    else if (mode == kWsumApply) FLASHOT_WSUM_SMALL(DPV, kWsumApply, 32, 1);        \
    else if (mode == kWsumGrad) FLASHOT_WSUM_SMALL(DPV, kWsumGrad, 32, 1);          \
    else if (mode == kWsumHessT) FLASHOT_WSUM_SMALL(DPV, kWsumHessT, 32, 1);        \
    else FLASHOT_WSUM_SMALL(DPV, kWsumHadamard, 32, 1);                             \
    break;
    switch (g.dpf) {
      FLASHOT_WSUM_MODES(4)
      FLASHOT_WSUM_MODES(8)
      FLASHOT_WSUM_MODES(12)
      FLASHOT_WSUM_MODES(16)
      FLASHOT_WSUM_MODES(20)
      FLASHOT_WSUM_MODES(24)
      FLASHOT_WSUM_MODES(28)
      FLASHOT_WSUM_MODES(32)
      default: return FLASHOT_ERR_INVALID_ARG;
    }
#undef FLASHOT_WSUM_MODES
#undef FLASHOT_WSUM_PAIR
#undef FLASHOT_WSUM_PAIR_F
#undef FLASHOT_WSUM_SMALL
  } else {
#define FLASHOT_WSUM_GENERIC(MODEV, KOV)                                                      \
  wsum_fma_generic_kernel<MODEV, KOV><<<grid, kFmaThreads, 0, c.st>>>(                        \
      rowP, colP, colBias, rowBias, n_rows, n_cols, n_tiles, g.dpf, kappa, V, ldv, k, rowW, X, \
      g.d, out, ldo, rowU)
    if (narrow) FLASHOT_WSUM_GENERIC(kWsumApply, 1);
    else if (mode == kWsumApply) FLASHOT_WSUM_GENERIC(kWsumApply, 32);
    else if (mode == kWsumGrad) FLASHOT_WSUM_GENERIC(kWsumGrad, 32);
    else if (mode == kWsumHessT) FLASHOT_WSUM_GENERIC(kWsumHessT, 32);
    else FLASHOT_WSUM_GENERIC(kWsumHadamard, 32);
#undef FLASHOT_WSUM_GENERIC
  }
  }
  if (n_splits > 1) {
    int rc = launch_check();
    if (rc != FLASHOT_OK) return rc;
    const int64_t total = n_rows * kk;
    TraceScope ts2_(FLASHOT_KERNEL_OTHER, c.st);
#define FLASHOT_WSUM_REDUCE(MODEV)                                                       \
  wsum_split_reduce_lanes_kernel<MODEV><<<grid1(total * kSplitLanes, 256), 256, 0, c.st>>>( \
      part, n_splits, rows_pad, kp, n_rows, k, rowW, X, g.d, out, ldo)
    if (mode == kWsumApply) FLASHOT_WSUM_REDUCE(kWsumApply);
    else if (mode == kWsumGrad) FLASHOT_WSUM_REDUCE(kWsumGrad);
    else if (mode == kWsumHessT) FLASHOT_WSUM_REDUCE(kWsumHessT);
    else FLASHOT_WSUM_REDUCE(kWsumHadamard);
#undef FLASHOT_WSUM_REDUCE
  }
  return launch_check();
}

// ---- Hessian-vector product scratch (after the ordinary workspace) ----------------------
struct HvpLayout {
  size_t vp, VA, OA, VB, OB, T, wf, t1, PtT, z, res, yv, p, Pp, tn, VD, OD, sc, cgp, total;
};

HvpLayout make_hvp_layout(const Geometry& g, size_t base) {
  HvpLayout H{};
  size_t off = base;
  auto take = [&](size_t floats) {
    size_t o = off;
    off = (off + floats * 4 + 255) / 256 * 256;
    return o;
  };
  const size_t n = (size_t)g.n, m = (size_t)g.m, d = (size_t)g.d;
  H.vp = take((size_t)g.n_pad * g.dpf);
  H.VA = take(m * (d + 1));
  H.OA = take(n * (d + 1));
  H.VB = take(n * (d + 2));
  H.OB = take(m * (d + 2));
  H.T = take(n * d);
  H.wf = take(n);
  H.t1 = take(n);
  H.PtT = take(m);
  H.z = take(m);
  H.res = take(m);
  H.yv = take(m);
  H.p = take(m);
  H.Pp = take(n);
  H.tn = take(n);
  H.VD = take(m * (d + 1));
  H.OD = take(n * (d + 1));
  H.sc = take(2 * kHvpScalars);
  H.cgp = take(2 * 6 * kCgMaxBlocks);  // doubles: 4 and 2 partials per CG block
  H.total = off + 256;
  return H;
}

// The Hessian-vector product runs on the fp32 CUDA-core passes; its geometry.
bool hvp_geometry(int64_t n, int64_t m, int64_t d, int flags, Geometry* g) {
  const int p = flags & FLASHOT_PREC_MASK;
  if (p != FLASHOT_PREC_AUTO && p != FLASHOT_PREC_FP32) return false;
  return make_geometry(n, m, d, d + 2, FLASHOT_PREC_FP32, g);
}

// Common prologue of every hot-path entry point.
int begin(int64_t n, int64_t m, int64_t d, int64_t k, int flags, void* ws, size_t ws_bytes,
          flashot_stream_t stream, Ctx* c) {
  if (!make_geometry(n, m, d, k, flags, &c->g)) return FLASHOT_ERR_INVALID_ARG;
  int sms = 0;
  int rc = current_device(&sms);
  if (rc != FLASHOT_OK) return rc;
  rc = check_ws(c->g, ws, ws_bytes, &c->L);
  if (rc != FLASHOT_OK) return rc;
  c->ws = static_cast<char*>(ws);
  c->sms = sms;
  c->st = reinterpret_cast<cudaStream_t>(stream);
  return FLASHOT_OK;
}

}  // namespace

int checked_current_device() {
  int sms = 0;
  return current_device(&sms);
}

int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

}  // namespace flashot

using namespace flashot;

extern "C" {

int flashot_version(void) { return kVersion; }

const char* flashot_status_string(int s) {
  switch (s) {
    case FLASHOT_OK: return "ok";
    case FLASHOT_ERR_INVALID_ARG: return "invalid argument";
    case FLASHOT_ERR_ALIGNMENT: return "workspace pointer is not 256-byte aligned";
    case FLASHOT_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FLASHOT_ERR_CUDA: return "CUDA runtime error (see flashot_last_cuda_error)";
    case FLASHOT_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case FLASHOT_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103";
    case FLASHOT_ERR_NOT_IMPLEMENTED: return "not implemented for these flags";
    default: return "unknown status";
  }
}

int flashot_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t flashot_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int flashot_timer_stop(void) {
  for (cudaEvent_t e : g_timer.ev) cudaEventDestroy(e);
  g_timer = EventTimer{};
  return FLASHOT_OK;
}

int flashot_timer_start(int cap) {
  if (cap < 1 || cap > (1 << 20)) return FLASHOT_ERR_INVALID_ARG;
  flashot_timer_stop();
  g_timer.ev.resize(2 * (size_t)cap, nullptr);
  g_timer.cls.assign((size_t)cap, -1);
  for (auto& e : g_timer.ev) {
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) {
      flashot_timer_stop();
      return cuda_fail(err);
    }
  }
  g_timer.cap = cap;
  g_timer.on = true;
  return FLASHOT_OK;
}

int flashot_timer_read(int kernel_class, int64_t* launches, double* total_ms) {
  if (!launches || !total_ms) return FLASHOT_ERR_INVALID_ARG;
  int64_t cnt = 0;
  double ms = 0.0;
  for (int i = 0; i < g_timer.used; ++i) {
    if (g_timer.cls[i] != kernel_class) continue;
    cudaError_t err = cudaEventSynchronize(g_timer.ev[2 * i + 1]);
    float t = 0.0f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&t, g_timer.ev[2 * i], g_timer.ev[2 * i + 1]);
    if (err != cudaSuccess) return cuda_fail(err);
    ++cnt;
    ms += t;
  }
  *launches = cnt;
  *total_ms = ms;
  return FLASHOT_OK;
}

size_t flashot_workspace_bytes(int64_t n, int64_t m, int64_t d, int64_t k, int flags) {
  Geometry g;
  if (!make_geometry(n, m, d, k, flags, &g)) return 0;
  return make_layout(g).total;
}

int flashot_workspace_status(void* ws, flashot_stream_t stream) {
  if (!is_device_ptr(ws)) return FLASHOT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FLASHOT_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word != 0) {
    e = cudaMemsetAsync(ws, 0, sizeof(word), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    return FLASHOT_ERR_DEVICE_TIMEOUT;
  }
  return FLASHOT_OK;
}

int flashot_selftest_bounded_wait(void* ws, int64_t limit_ns, flashot_stream_t stream) {
  if (limit_ns < 1000000 || limit_ns > 2000000000) return FLASHOT_ERR_INVALID_ARG;
  int sms = 0;
  int rc = current_device(&sms);
  if (rc != FLASHOT_OK) return rc;
  if (!is_device_ptr(ws)) return FLASHOT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FLASHOT_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned* status = static_cast<unsigned*>(ws);
  rc = tc_selftest_bounded_wait(status, limit_ns, st);
  // then the grid barrier's wait, on the word at byte 128 of ws
  if (rc == FLASHOT_OK) rc = tc_selftest_grid_wait(status, status + 32, limit_ns, st);
  return rc == FLASHOT_OK ? launch_check() : rc;
}

int flashot_sinkhorn_solve(const float* X, const float* Y, const float* a, const float* b,
                           int64_t n, int64_t m, int64_t d, const float* eps_sched, int n_stages,
                           int iters_per_stage, int flags, float* f, float* g, double* loss,
                           void* ws, size_t ws_bytes, flashot_stream_t stream) {
  if (!eps_sched || n_stages < 1 || iters_per_stage < 1) return FLASHOT_ERR_INVALID_ARG;
  for (int s = 0; s < n_stages; ++s)
    if (!eps_ok(eps_sched[s])) return FLASHOT_ERR_INVALID_ARG;
  Ctx c;
  int rc = begin(n, m, d, 0, flags, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(a) || !opt_device_ptr(b) ||
      !is_device_ptr(f) || !is_device_ptr(g) || !opt_device_ptr(loss))
    return FLASHOT_ERR_INVALID_ARG;
  const bool symmetric = (flags & FLASHOT_SYMMETRIC) != 0;
  if ((rc = validate_inputs(c, flags, X, Y, a, b)) != FLASHOT_OK) return rc;
  // Small fp32 problems: every iteration in one launch of one thread-block cluster.
  if (!symmetric && c.g.prec == FLASHOT_PREC_FP32 && c.g.small &&
      small_solve_eligible(n, m, c.g.dpf, n_stages))
    return small_solve(X, Y, a, b, n, m, d, c.g.dpf, eps_sched, n_stages, iters_per_stage,
                       (flags & FLASHOT_WARM_START) != 0, f, g, loss, c.st);
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, a, b)) != FLASHOT_OK) return rc;
  if (symmetric) {
    // Both half-steps read the previous iterate; the combines average in place.
    if (!(flags & FLASHOT_WARM_START)) {
      cudaError_t e = cudaMemsetAsync(f, 0, (size_t)n * sizeof(float), c.st);
      if (e == cudaSuccess) e = cudaMemsetAsync(g, 0, (size_t)m * sizeof(float), c.st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    // A self-transport problem (the same cloud and weights on both sides, e.g. the OT(a, a)
    // terms of the debiased divergence) started from f = g keeps f == g: the g-update is
    // the f-update's arithmetic on identical inputs. One pass per iteration then suffices,
    // and g is copied from f at the end.
    const bool self = X == Y && a == b && n == m && !(flags & FLASHOT_WARM_START);
    // Short tensor-core contractions: every iteration in one persistent launch (the same
    // passes, merges and biases as below, so the same bits), from the first iteration's
    // biases.
    bool done = false;
    if (c.g.prec != FLASHOT_PREC_FP32) {
      if ((rc = launch_bias(c, self ? f : g, false, eps_sched[0])) != FLASHOT_OK) return rc;
      if (!self && (rc = launch_bias(c, f, true, eps_sched[0])) != FLASHOT_OK) return rc;
      rc = tc_short_solve(c.g.prec == FLASHOT_PREC_BF16, c.at<void>(c.L.xq),
                          c.at<void>(c.L.yq), n, m, c.g.n_pad, c.g.m_pad, c.g.dpt,
                          c.at<float>(c.L.alpha), c.at<float>(c.L.beta), c.at<float>(c.L.la2),
                          c.at<float>(c.L.lb2), c.at<float>(c.L.biasF), c.at<float>(c.L.biasG),
                          f, g, eps_sched, n_stages, iters_per_stage, self ? 2 : 1, nullptr,
                          nullptr, -1, c.at<float2>(c.L.partial), partial_bytes(c.g), kMaxSplits,
                          c.at<void>(c.L.sync), tc_short_solve_sync_bytes(c.g.n_pad, c.g.m_pad),
                          c.sms, c.at<unsigned>(c.L.status), c.st);
      if (rc == FLASHOT_OK) done = true;
      else if (rc != FLASHOT_ERR_NOT_IMPLEMENTED) return rc;
    }
    for (int s = 0; !done && s < n_stages; ++s) {
      const float eps = eps_sched[s];
      for (int it = 0; it < iters_per_stage; ++it) {
        if ((rc = launch_bias(c, self ? f : g, false, eps)) != FLASHOT_OK) return rc;
        if (!self && (rc = launch_bias(c, f, true, eps)) != FLASHOT_OK) return rc;
        if ((rc = run_lse_pass(c, true, eps, eps, f, false, nullptr, true)) != FLASHOT_OK)
          return rc;
        if (!self && (rc = run_lse_pass(c, false, eps, eps, g, false, nullptr, true)) !=
                         FLASHOT_OK)
          return rc;
      }
    }
    if (self) {
      cudaError_t e = cudaMemcpyAsync(g, f, (size_t)m * sizeof(float), cudaMemcpyDeviceToDevice,
                                      c.st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  } else {
  // Initial F-step bias from g (warm start) or g = 0.
  if ((rc = launch_bias(c, (flags & FLASHOT_WARM_START) ? g : nullptr, false, eps_sched[0])) !=
      FLASHOT_OK)
    return rc;
  // Short tensor-core contractions: every half-step in one persistent launch (the same
  // tiles, partials and merges as the passes below, so the same bits).
  bool done = false;
  if (c.g.prec != FLASHOT_PREC_FP32) {
    rc = tc_short_solve(c.g.prec == FLASHOT_PREC_BF16, c.at<void>(c.L.xq), c.at<void>(c.L.yq), n,
                        m, c.g.n_pad, c.g.m_pad, c.g.dpt, c.at<float>(c.L.alpha),
                        c.at<float>(c.L.beta), c.at<float>(c.L.la2), c.at<float>(c.L.lb2),
                        c.at<float>(c.L.biasF), c.at<float>(c.L.biasG), f, g, eps_sched,
                        n_stages, iters_per_stage, 0, nullptr, nullptr, -1,
                        c.at<float2>(c.L.partial),
                        partial_bytes(c.g), kMaxSplits, c.at<void>(c.L.sync),
                        tc_short_solve_sync_bytes(c.g.n_pad, c.g.m_pad), c.sms,
                        c.at<unsigned>(c.L.status), c.st);
    if (rc == FLASHOT_OK) done = true;
    else if (rc != FLASHOT_ERR_NOT_IMPLEMENTED) return rc;
  }
  for (int s = 0; !done && s < n_stages; ++s) {
    const float eps = eps_sched[s];
    for (int it = 0; it < iters_per_stage; ++it) {
      const bool last_of_stage = (it == iters_per_stage - 1);
      const float eps_next = (last_of_stage && s + 1 < n_stages) ? eps_sched[s + 1] : eps;
      if ((rc = run_lse_pass(c, true, eps, eps, f, true, nullptr)) != FLASHOT_OK) return rc;
      if ((rc = run_lse_pass(c, false, eps, eps_next, g, true, nullptr)) != FLASHOT_OK) return rc;
    }
  }
  }
  if (loss) {
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      dual_loss_kernel<<<1, 1024, 0, c.st>>>(c.at<float>(c.L.wa), f, n, c.at<float>(c.L.wb), g, m,
                                             loss);
    }
    if ((rc = launch_check()) != FLASHOT_OK) return rc;
  }
  return FLASHOT_OK;
}

int flashot_sinkhorn_solve_tol(const float* X, const float* Y, const float* a, const float* b,
                               int64_t n, int64_t m, int64_t d, float eps, double tol,
                               int max_iters, int check_every, int flags, float* f, float* g,
                               double* loss, int* iters_done, double* err, double* err_hist,
                               void* ws, size_t ws_bytes, flashot_stream_t stream) {
  if (!eps_ok(eps) || !std::isfinite(tol) || tol < 0.0 || max_iters < 1 || check_every < 1 ||
      iters_done == nullptr)
    return FLASHOT_ERR_INVALID_ARG;
  if (flags & ~(FLASHOT_PREC_MASK | FLASHOT_REUSE_PACK | FLASHOT_VALIDATE))
    return FLASHOT_ERR_NOT_IMPLEMENTED;
  Ctx c;
  int rc = begin(n, m, d, 0, flags, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(a) || !opt_device_ptr(b) ||
      !is_device_ptr(f) || !is_device_ptr(g) || !opt_device_ptr(loss))
    return FLASHOT_ERR_INVALID_ARG;
  *iters_done = 0;
  if (err) *err = -1.0;
  if ((rc = validate_inputs(c, flags, X, Y, a, b)) != FLASHOT_OK) return rc;
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, a, b)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, nullptr, false, eps)) != FLASHOT_OK) return rc;
  float* err_rows = c.at<float>(c.L.lse2);
  double* err_dev = c.at<double>(c.L.loss);
  // The check of iteration kk: sum the error rows its f-update wrote, read the sum and the
  // status word, and decide.
  auto check_error = [&](int kk, bool* stop) -> int {
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      sum_rows_kernel<<<1, 1024, 0, c.st>>>(err_rows, n, err_dev);
    }
    int r = launch_check();
    if (r != FLASHOT_OK) return r;
    double e_host = 0.0;
    unsigned word = 0;
    cudaError_t e = cudaMemcpyAsync(&e_host, err_dev, sizeof(double), cudaMemcpyDeviceToHost,
                                    c.st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(&word, c.at<unsigned>(c.L.status), sizeof(word),
                          cudaMemcpyDeviceToHost, c.st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c.st);
    if (e != cudaSuccess) return cuda_fail(e);
    // A kernel that gave up a bounded wait left garbage: stop (the word stays set for
    // flashot_workspace_status).
    if (word != 0) return FLASHOT_ERR_DEVICE_TIMEOUT;
    if (err) *err = e_host;
    if (err_hist) err_hist[kk / check_every - 1] = e_host;
    *stop = e_host < tol;
    return FLASHOT_OK;
  };
  int k = 1;
  bool stop = false;
  // Short tensor-core contractions, checks at least 4 iterations apart: the iterations up to
  // each check in one persistent launch, whose check iteration's f-update writes the error
  // rows (the same bits and decisions as the per-pass loop below, which takes over from
  // iteration k when the launch does not apply).
  while (c.g.prec != FLASHOT_PREC_FP32 && check_every >= 4 && !stop && k <= max_iters) {
    const int kc = (std::max(k, 2) + check_every - 1) / check_every * check_every;
    const int last = std::min(kc, max_iters);
    const bool check = last == kc;
    rc = tc_short_solve(c.g.prec == FLASHOT_PREC_BF16, c.at<void>(c.L.xq), c.at<void>(c.L.yq),
                        n, m, c.g.n_pad, c.g.m_pad, c.g.dpt, c.at<float>(c.L.alpha),
                        c.at<float>(c.L.beta), c.at<float>(c.L.la2), c.at<float>(c.L.lb2),
                        c.at<float>(c.L.biasF), c.at<float>(c.L.biasG), f, g, &eps, 1,
                        last - k + 1, 0, check ? err_rows : nullptr, c.at<float>(c.L.wa),
                        check ? last - k : -1, c.at<float2>(c.L.partial), partial_bytes(c.g),
                        kMaxSplits, c.at<void>(c.L.sync),
                        tc_short_solve_sync_bytes(c.g.n_pad, c.g.m_pad), c.sms,
                        c.at<unsigned>(c.L.status), c.st);
    if (rc == FLASHOT_ERR_NOT_IMPLEMENTED) break;
    if (rc != FLASHOT_OK) return rc;
    if (check && (rc = check_error(last, &stop)) != FLASHOT_OK) return rc;
    k = stop ? last : last + 1;
  }
  for (; !stop && k <= max_iters; ++k) {
    // Iteration k measures, inside its f-update, the row-marginal error of iterate k-1.
    const bool check = k >= 2 && k % check_every == 0;
    if ((rc = run_lse_pass(c, true, eps, eps, f, true, nullptr, false,
                           check ? err_rows : nullptr)) != FLASHOT_OK)
      return rc;
    if ((rc = run_lse_pass(c, false, eps, eps, g, true, nullptr)) != FLASHOT_OK) return rc;
    if (check) {
      if ((rc = check_error(k, &stop)) != FLASHOT_OK) return rc;
      if (stop) break;
    }
  }
  *iters_done = std::min(k, max_iters);
  if (loss) {
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      dual_loss_kernel<<<1, 1024, 0, c.st>>>(c.at<float>(c.L.wa), f, n, c.at<float>(c.L.wb), g, m,
                                             loss);
    }
    if ((rc = launch_check()) != FLASHOT_OK) return rc;
  }
  return FLASHOT_OK;
}

size_t flashot_hvp_workspace_bytes(int64_t n, int64_t m, int64_t d, int flags) {
  Geometry g;
  if (!hvp_geometry(n, m, d, flags, &g)) return 0;
  return make_hvp_layout(g, make_layout(g).total).total;
}

int flashot_ot_hvp_x(const float* X, const float* Y, const float* a, const float* b,
                     const float* f, const float* g, int64_t n, int64_t m, int64_t d, float eps,
                     const float* V, float* out, double cg_tol, int cg_max_iters, int flags,
                     int* cg_iters, double* cg_rel_residual, void* ws, size_t ws_bytes,
                     flashot_stream_t stream) {
  if (!eps_ok(eps) || !std::isfinite(cg_tol) || cg_tol < 0.0 || cg_max_iters < 0)
    return FLASHOT_ERR_INVALID_ARG;
  if (flags & ~(FLASHOT_PREC_MASK | FLASHOT_REUSE_PACK | FLASHOT_VALIDATE))
    return FLASHOT_ERR_NOT_IMPLEMENTED;
  {
    const int p = flags & FLASHOT_PREC_MASK;
    if (p != FLASHOT_PREC_AUTO && p != FLASHOT_PREC_FP32) return FLASHOT_ERR_NOT_IMPLEMENTED;
  }
  const int fl = (flags & (FLASHOT_REUSE_PACK | FLASHOT_VALIDATE)) | FLASHOT_PREC_FP32;
  Ctx c;
  int rc = begin(n, m, d, d + 2, fl, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  const HvpLayout H = make_hvp_layout(c.g, c.L.total);
  if (ws_bytes < H.total) return FLASHOT_ERR_WORKSPACE_TOO_SMALL;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(a) || !opt_device_ptr(b) ||
      !is_device_ptr(f) || !is_device_ptr(g) || !is_device_ptr(V) || !is_device_ptr(out) ||
      (const void*)out == (const void*)V)
    return FLASHOT_ERR_INVALID_ARG;
  if (cg_iters) *cg_iters = 0;
  if (cg_rel_residual) *cg_rel_residual = 0.0;
  if ((rc = validate_inputs(c, flags, X, Y, a, b)) != FLASHOT_OK) return rc;
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, a, b)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, g, false, eps)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, f, true, eps)) != FLASHOT_OK) return rc;
  float* vp = c.at<float>(H.vp);
  float* VA = c.at<float>(H.VA);
  float* OA = c.at<float>(H.OA);
  float* VB = c.at<float>(H.VB);
  float* OB = c.at<float>(H.OB);
  float* T = c.at<float>(H.T);
  float* wf = c.at<float>(H.wf);
  float* t1 = c.at<float>(H.t1);
  float* PtT = c.at<float>(H.PtT);
  float* z = c.at<float>(H.z);
  float* res = c.at<float>(H.res);
  float* yv = c.at<float>(H.yv);
  float* pv = c.at<float>(H.p);
  float* Pp = c.at<float>(H.Pp);
  float* tn = c.at<float>(H.tn);
  float* VD = c.at<float>(H.VD);
  float* OD = c.at<float>(H.OD);
  double* sc = c.at<double>(H.sc);
  double* cgp = c.at<double>(H.cgp);
  double* cgp2 = cgp + 4 * kCgMaxBlocks;
  const int cg_blocks = (int)std::min<int64_t>(std::max<int64_t>(ceil_div(m, kCgThreads), 1),
                                               kCgMaxBlocks);
  const int T256 = 256;
  const int64_t nm = std::max(n, m);
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    pack_rows_kernel<PackKind::F32><<<grid1(c.g.n_pad * c.g.dpf, T256), T256, 0, c.st>>>(
        V, vp, n, d, c.g.n_pad, c.g.dpf);
  }
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    hvp_prep_kernel<<<grid1(nm, T256), T256, 0, c.st>>>(X, Y, V, n, m, d, VA, VB);
  }
  if ((rc = launch_check()) != FLASHOT_OK) return rc;
  // [PY | r], [P^T V | P^T s | c] and the curvature term T.
  if ((rc = run_wsum_pass(c, kWsumApply, false, eps, VA, d + 1, d + 1, X, Y, OA, d + 1)) !=
      FLASHOT_OK)
    return rc;
  if ((rc = run_wsum_pass(c, kWsumApply, true, eps, VB, d + 2, d + 2, X, Y, OB, d + 2)) !=
      FLASHOT_OK)
    return rc;
  if ((rc = run_wsum_pass(c, kWsumHessT, false, eps, Y, d, d, X, Y, T, d, vp)) != FLASHOT_OK)
    return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    hvp_rhs_kernel<<<grid1(n, T256), T256, 0, c.st>>>(OA, VB, n, d, eps, wf, t1);
  }
  if ((rc = launch_check()) != FLASHOT_OK) return rc;
  if ((rc = run_wsum_pass(c, kWsumApply, true, eps, t1, 1, 1, X, Y, PtT, 1)) != FLASHOT_OK)
    return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    hvp_cg_init_kernel<<<1, 1024, 0, c.st>>>(Y, OB, PtT, m, d, eps, z, res, yv, pv, sc);
  }
  if ((rc = launch_check()) != FLASHOT_OK) return rc;
  // Preconditioned CG on the Schur complement S = diag(c) - P^T diag(1/r) P.
  double host_sc[kHvpScalars];
  auto read_scalars = [&]() -> int {
    cudaError_t e = cudaMemcpyAsync(host_sc, sc, sizeof(host_sc), cudaMemcpyDeviceToHost, c.st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c.st);
    return e == cudaSuccess ? FLASHOT_OK : cuda_fail(e);
  };
  if ((rc = read_scalars()) != FLASHOT_OK) return rc;
  const double rr0 = host_sc[kHvpRR0];
  double rel = rr0 > 0.0 ? 1.0 : 0.0;
  int it = 0;
  while (rr0 > 0.0 && rel > cg_tol && it < cg_max_iters) {
    if ((rc = run_wsum_pass(c, kWsumApply, false, eps, pv, 1, 1, X, Y, Pp, 1)) != FLASHOT_OK)
      return rc;
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      hvp_div_kernel<<<grid1(n, T256), T256, 0, c.st>>>(Pp, OA + d, d + 1, n, tn);
    }
    if ((rc = launch_check()) != FLASHOT_OK) return rc;
    if ((rc = run_wsum_pass(c, kWsumApply, true, eps, tn, 1, 1, X, Y, PtT, 1)) != FLASHOT_OK)
      return rc;
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      hvp_cg_q_kernel<<<cg_blocks, kCgThreads, 0, c.st>>>(OB, PtT, m, d, pv, cgp);
    }
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      hvp_cg_update_kernel<<<cg_blocks, kCgThreads, 0, c.st>>>(OB, PtT, m, d, z, res, yv, pv,
                                                                cgp, cgp2, sc);
    }
    {
      TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
      hvp_cg_dir_kernel<<<cg_blocks, kCgThreads, 0, c.st>>>(m, pv, yv, cgp2, sc);
    }
    if ((rc = launch_check()) != FLASHOT_OK) return rc;
    if ((rc = read_scalars()) != FLASHOT_OK) return rc;
    ++it;
    if (host_sc[kHvpBreak] != 0.0) break;
    rel = std::sqrt(std::max(host_sc[kHvpRR], 0.0) / rr0);
  }
  unsigned word = 0;
  {
    cudaError_t e = cudaMemcpyAsync(&word, c.at<unsigned>(c.L.status), sizeof(word),
                                    cudaMemcpyDeviceToHost, c.st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c.st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (word != 0) return FLASHOT_ERR_DEVICE_TIMEOUT;
  if (cg_iters) *cg_iters = it;
  if (cg_rel_residual) *cg_rel_residual = rel;
  // [P diag(z) Y | P z], then assemble H V.
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    hvp_vd_kernel<<<grid1(m, T256), T256, 0, c.st>>>(Y, z, m, d, VD);
  }
  if ((rc = launch_check()) != FLASHOT_OK) return rc;
  if ((rc = run_wsum_pass(c, kWsumApply, false, eps, VD, d + 1, d + 1, X, Y, OD, d + 1)) !=
      FLASHOT_OK)
    return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    hvp_final_kernel<<<grid1(n, T256), T256, 0, c.st>>>(X, OA, VB, T, wf, OD, n, d, eps, out);
  }
  return launch_check();
}

size_t flashot_diagnostics_workspace_bytes(int64_t n, int64_t m, int64_t d, int flags) {
  Geometry g;
  if (!make_geometry(n, m, d, 1, flags, &g)) return 0;
  // r (n), c (m), h (n) and a vector of ones (max(n, m)), each 256-byte aligned
  const size_t mx = (size_t)std::max(g.n_pad, g.m_pad);
  return make_layout(g).total + 4 * (mx * 4 + 256);
}

int flashot_plan_diagnostics(const float* X, const float* Y, const float* a, const float* b,
                             const float* f, const float* g, int64_t n, int64_t m, int64_t d,
                             float eps, int flags, double* out, void* ws, size_t ws_bytes,
                             flashot_stream_t stream) {
  if (!eps_ok(eps)) return FLASHOT_ERR_INVALID_ARG;
  Ctx c;
  int rc = begin(n, m, d, 1, flags, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (ws_bytes < flashot_diagnostics_workspace_bytes(n, m, d, flags))
    return FLASHOT_ERR_WORKSPACE_TOO_SMALL;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(a) || !opt_device_ptr(b) ||
      !is_device_ptr(f) || !is_device_ptr(g) || !is_device_ptr(out))
    return FLASHOT_ERR_INVALID_ARG;
  if ((rc = validate_inputs(c, flags, X, Y, a, b)) != FLASHOT_OK) return rc;
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, a, b)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, g, false, eps)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, f, true, eps)) != FLASHOT_OK) return rc;
  const size_t mx = (size_t)std::max(c.g.n_pad, c.g.m_pad);
  const size_t slot = (mx * 4 + 255) / 256 * 256;
  float* r_ = reinterpret_cast<float*>(c.ws + c.L.total);
  float* c_ = reinterpret_cast<float*>(c.ws + c.L.total + slot);
  float* h_ = reinterpret_cast<float*>(c.ws + c.L.total + 2 * slot);
  float* ones = reinterpret_cast<float*>(c.ws + c.L.total + 3 * slot);
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    fill_kernel<<<grid1((int64_t)mx, 256), 256, 0, c.st>>>(ones, (int64_t)mx, 1.0f);
  }
  if ((rc = launch_check()) != FLASHOT_OK) return rc;
  if ((rc = run_wsum_pass(c, kWsumApply, false, eps, ones, 1, 1, X, Y, r_, 1)) != FLASHOT_OK)
    return rc;
  if ((rc = run_wsum_pass(c, kWsumApply, true, eps, ones, 1, 1, X, Y, c_, 1)) != FLASHOT_OK)
    return rc;
  if ((rc = run_wsum_pass(c, kWsumHadamard, false, eps, nullptr, 0, 1, X, Y, h_, 1)) !=
      FLASHOT_OK)
    return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    diagnostics_kernel<<<1, 1024, 0, c.st>>>(r_, c_, h_, c.at<float>(c.L.alpha),
                                             c.at<float>(c.L.beta), c.at<float>(c.L.wa),
                                             c.at<float>(c.L.wb), f, g, n, m, (double)eps, out);
  }
  return launch_check();
}

size_t flashot_divergence_workspace_bytes(int64_t n, int64_t m, int64_t d, int flags) {
  const size_t w1 = flashot_workspace_bytes(n, m, d, 0, flags);
  const size_t w2 = flashot_workspace_bytes(n, n, d, 0, flags);
  const size_t w3 = flashot_workspace_bytes(m, m, d, 0, flags);
  if (w1 == 0 || w2 == 0 || w3 == 0) return 0;
  // six potential vectors (f, g of the three solves), each 256-byte aligned, then the
  // largest solve workspace
  const size_t pots = 2 * ((size_t)(n + 64) * 4 / 256 + 1) * 256 * 2 +
                      2 * ((size_t)(m + 64) * 4 / 256 + 1) * 256 * 2;
  return pots + std::max(w1, std::max(w2, w3)) + 256;
}

int flashot_sinkhorn_divergence(const float* X, const float* Y, const float* a, const float* b,
                                int64_t n, int64_t m, int64_t d, const float* eps_sched,
                                int n_stages, int iters_per_stage, int flags, double* out,
                                void* ws, size_t ws_bytes, flashot_stream_t stream) {
  const size_t need = flashot_divergence_workspace_bytes(n, m, d, flags);
  if (need == 0 || !is_device_ptr(out)) return FLASHOT_ERR_INVALID_ARG;
  if (!is_device_ptr(ws)) return FLASHOT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FLASHOT_ERR_ALIGNMENT;
  if (ws_bytes < need) return FLASHOT_ERR_WORKSPACE_TOO_SMALL;
  char* p = static_cast<char*>(ws);
  auto take = [&](int64_t count) {
    float* r = reinterpret_cast<float*>(p);
    p += ((size_t)(count + 64) * 4 / 256 + 1) * 256;
    return r;
  };
  float* f_xy = take(n);
  float* g_xy = take(m);
  float* f_xx = take(n);
  float* g_xx = take(n);
  float* f_yy = take(m);
  float* g_yy = take(m);
  const size_t used = (size_t)(p - static_cast<char*>(ws));
  void* sub = p;
  const size_t sub_bytes = ws_bytes - used;
  const int sflags = flags & ~(FLASHOT_WARM_START | FLASHOT_REUSE_PACK);
  int rc = flashot_sinkhorn_solve(X, Y, a, b, n, m, d, eps_sched, n_stages, iters_per_stage,
                                  sflags, f_xy, g_xy, out + 1, sub, sub_bytes, stream);
  if (rc == FLASHOT_OK)
    rc = flashot_sinkhorn_solve(X, X, a, a, n, n, d, eps_sched, n_stages, iters_per_stage,
                                sflags, f_xx, g_xx, out + 2, sub, sub_bytes, stream);
  if (rc == FLASHOT_OK)
    rc = flashot_sinkhorn_solve(Y, Y, b, b, m, m, d, eps_sched, n_stages, iters_per_stage,
                                sflags, f_yy, g_yy, out + 3, sub, sub_bytes, stream);
  if (rc != FLASHOT_OK) return rc;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, reinterpret_cast<cudaStream_t>(stream));
    divergence_combine_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(out);
  }
  return launch_check();
}

int flashot_sinkhorn_step_f(const float* X, const float* Y, const float* b, const float* g,
                            int64_t n, int64_t m, int64_t d, float eps, int flags, float* f,
                            void* ws, size_t ws_bytes, flashot_stream_t stream) {
  if (!eps_ok(eps)) return FLASHOT_ERR_INVALID_ARG;
  Ctx c;
  int rc = begin(n, m, d, 0, flags, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(b) || !is_device_ptr(g) ||
      !is_device_ptr(f))
    return FLASHOT_ERR_INVALID_ARG;
  if ((rc = validate_inputs(c, flags, X, Y, nullptr, b)) != FLASHOT_OK) return rc;
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, nullptr, b)) != FLASHOT_OK)
    return rc;
  if ((rc = launch_bias(c, g, false, eps)) != FLASHOT_OK) return rc;
  return run_lse_pass(c, true, eps, eps, f, false, nullptr);
}

int flashot_sinkhorn_step_g(const float* X, const float* Y, const float* a, const float* f,
                            int64_t n, int64_t m, int64_t d, float eps, int flags, float* g,
                            void* ws, size_t ws_bytes, flashot_stream_t stream) {
  if (!eps_ok(eps)) return FLASHOT_ERR_INVALID_ARG;
  Ctx c;
  int rc = begin(n, m, d, 0, flags, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(a) || !is_device_ptr(f) ||
      !is_device_ptr(g))
    return FLASHOT_ERR_INVALID_ARG;
  if ((rc = validate_inputs(c, flags, X, Y, a, nullptr)) != FLASHOT_OK) return rc;
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, a, nullptr)) != FLASHOT_OK)
    return rc;
  if ((rc = launch_bias(c, f, true, eps)) != FLASHOT_OK) return rc;
  return run_lse_pass(c, false, eps, eps, g, false, nullptr);
}

int flashot_dual_loss(const float* a, const float* b, const float* f, const float* g, int64_t n,
                      int64_t m, double* loss, void* ws, size_t ws_bytes, flashot_stream_t stream) {
  Ctx c;
  int rc = begin(n, m, 1, 0, FLASHOT_PREC_FP32, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (!opt_device_ptr(a) || !opt_device_ptr(b) || !is_device_ptr(f) || !is_device_ptr(g) ||
      !is_device_ptr(loss))
    return FLASHOT_ERR_INVALID_ARG;
  const int T = 256;
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    weights_kernel<<<grid1(c.g.n_pad, T), T, 0, c.st>>>(a, n, c.g.n_pad, c.at<float>(c.L.wa),
                                                        c.at<float>(c.L.la2), nullptr);
  }
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    weights_kernel<<<grid1(c.g.m_pad, T), T, 0, c.st>>>(b, m, c.g.m_pad, c.at<float>(c.L.wb),
                                                        c.at<float>(c.L.lb2), nullptr);
  }
  {
    TraceScope ts_(FLASHOT_KERNEL_OTHER, c.st);
    dual_loss_kernel<<<1, 1024, 0, c.st>>>(c.at<float>(c.L.wa), f, n, c.at<float>(c.L.wb), g, m,
                                           loss);
  }
  return launch_check();
}

int flashot_transport_apply(const float* X, const float* Y, const float* a, const float* b,
                            const float* f, const float* g, int64_t n, int64_t m, int64_t d,
                            float eps, const float* V, int64_t k, int transpose, float* out,
                            int flags, void* ws, size_t ws_bytes, flashot_stream_t stream) {
  if (!eps_ok(eps) || k < 1) return FLASHOT_ERR_INVALID_ARG;
  Ctx c;
  int rc = begin(n, m, d, k, flags, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(a) || !opt_device_ptr(b) ||
      !is_device_ptr(f) || !is_device_ptr(g) || !is_device_ptr(V) || !is_device_ptr(out) ||
      (const void*)out == (const void*)V)
    return FLASHOT_ERR_INVALID_ARG;
  if ((rc = validate_inputs(c, flags, X, Y, a, b)) != FLASHOT_OK) return rc;
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, a, b)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, g, false, eps)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, f, true, eps)) != FLASHOT_OK) return rc;
  return run_wsum_pass(c, kWsumApply, transpose != 0, eps, V, k, k, X, Y, out, k);
}

int flashot_transport_hadamard_xy(const float* X, const float* Y, const float* a, const float* b,
                                  const float* f, const float* g, int64_t n, int64_t m, int64_t d,
                                  float eps, float* h, int flags, void* ws, size_t ws_bytes,
                                  flashot_stream_t stream) {
  if (!eps_ok(eps)) return FLASHOT_ERR_INVALID_ARG;
  Ctx c;
  int rc = begin(n, m, d, 0, flags, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(a) || !opt_device_ptr(b) ||
      !is_device_ptr(f) || !is_device_ptr(g) || !is_device_ptr(h))
    return FLASHOT_ERR_INVALID_ARG;
  if ((rc = validate_inputs(c, flags, X, Y, a, b)) != FLASHOT_OK) return rc;
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, a, b)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, g, false, eps)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, f, true, eps)) != FLASHOT_OK) return rc;
  return run_wsum_pass(c, kWsumHadamard, false, eps, nullptr, 0, 1, X, Y, h, 1);
}

int flashot_ot_grad_x(const float* X, const float* Y, const float* a, const float* b,
                      const float* g, int64_t n, int64_t m, int64_t d, float eps, float* grad,
                      int flags, void* ws, size_t ws_bytes, flashot_stream_t stream) {
  if (!eps_ok(eps)) return FLASHOT_ERR_INVALID_ARG;
  Ctx c;
  int rc = begin(n, m, d, 0, flags, ws, ws_bytes, stream, &c);
  if (rc != FLASHOT_OK) return rc;
  if (!is_device_ptr(X) || !is_device_ptr(Y) || !opt_device_ptr(a) || !opt_device_ptr(b) ||
      !is_device_ptr(g) || !is_device_ptr(grad))
    return FLASHOT_ERR_INVALID_ARG;
  if ((rc = validate_inputs(c, flags, X, Y, a, b)) != FLASHOT_OK) return rc;
  if (!(flags & FLASHOT_REUSE_PACK) && (rc = pack_inputs(c, X, Y, a, b)) != FLASHOT_OK) return rc;
  if ((rc = launch_bias(c, g, false, eps)) != FLASHOT_OK) return rc;
  // f~ = F(g); its combine writes biasG = log2 a_i - L_i, so the weighted pass below uses
  // w_ij = a_i softmax_j(s_ij); the gradient kernel renormalises by sum_j w_ij.
  if ((rc = run_lse_pass(c, true, eps, eps, c.at<float>(c.L.ftilde), true, nullptr)) != FLASHOT_OK)
    return rc;
  return run_wsum_pass(c, kWsumGrad, false, eps, nullptr, 0, d, X, Y, grad, d);
}

}  // extern "C"
