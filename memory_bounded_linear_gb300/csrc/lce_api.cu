// C ABI of the memory-bounded linear cross-entropy library (declared in include/lce.h):
// argument validation, workspace layout, the strip loop, launch counting and launch tracing.
// Every compute step runs in the kernels of lce_tc.cu / lce_simt.cu / lce_reduce.cu.
#include <cuda_runtime.h>
#include <stdint.h>

#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>

#include "lce.h"
#include "lce_internal.h"

namespace lce {
namespace {

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
// Largest dH job (in 256 x 256 tiles) whose backward step is overlapped with the next strip's
// gradient computation (a few waves of the GPU's 76 CTA pairs).
constexpr int64_t kOverlapMaxTiles = 512;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  int bn;           // logit tile width of the engine
  int64_t w;        // strip width (strip_columns): every strip but the last is w columns wide
  int64_t ldg;      // row stride of the strip gradient workspace (elements)
  int tiles;        // logit tiles per full strip
  size_t off_run, off_tgt, off_part, off_g;
  size_t g_bytes;   // one gradient strip (LCE_F32_TF32X3: its hi part; the lo part follows)
  bool overlap_bwd; // two gradient strips: each backward launch also computes the next gradient
  // LCE_F32_TF32X3 only: tf32 hi / lo parts, each at off_* with its lo part *_part bytes later
  size_t off_h, h_part;    // H [N x d]
  size_t off_w, w_part;    // one strip of W [w x d]
  size_t off_ht, ht_part;  // H^T [d x ldt]              (backward)
  size_t off_wt, wt_part;  // the W strip transposed [d x ldg]   (backward)
  size_t off_gt, gt_part;  // the gradient strip transposed [ldg x ldt] (backward)
  int64_t ldt;             // N rounded up to a multiple of 32
  size_t total;
};

// Rows of H and W are d elements: d x (element size) must be a multiple of 16 bytes (TMA row
// strides, 16-byte vector accesses), so d % 8 == 0 for bf16 and d % 4 == 0 for fp32.
bool shape_ok(int64_t N, int64_t d, int64_t V, int64_t strip_V, lce_dtype_t dt) {
  const int64_t d_mult = (dt == LCE_BF16) ? 8 : 4;
  if (N < 0 || N > kMaxDim) return false;
  if (V < 1 || V > kMaxDim) return false;
  if (d < d_mult || d % d_mult != 0 || d > kMaxDim) return false;
  if (strip_V < 128 || strip_V % 128 != 0 || strip_V > kMaxDim) return false;
  return true;
}

// Width of the strips: the vocabulary is cut into ceil(V / strip_V) strips of equal width, rounded
// up to the tile width of the engine (so that only the last strip ends inside a tile) when that
// stays within strip_V, else to 128 columns; never wider than strip_V or V.  With strips of
// strip_V columns the last one could be a sliver (4,096 of 151,552 columns at strip 16,384) whose
// launches fill the GPU poorly.
int64_t strip_columns(int64_t V, int64_t strip_V, int bn) {
  const int64_t S = (V + strip_V - 1) / strip_V;
  const int64_t even = (V + S - 1) / S;
  int64_t w = (even + bn - 1) / bn * bn;
  if (w > strip_V) w = (even + 127) / 128 * 128;
  return std::min(w, V);
}

bool make_layout(int64_t N, int64_t d, int64_t V, int64_t strip_V, lce_dtype_t dt, Layout* L) {
  if (dt != LCE_BF16 && dt != LCE_F32 && dt != LCE_F32_TF32X3) return false;
  if (!shape_ok(N, d, V, strip_V, dt)) return false;
  const bool x3 = (dt == LCE_F32_TF32X3);
  *L = Layout{};
  L->bn = (dt == LCE_F32) ? SIMT_BN : TC_BN;
  L->w = strip_columns(V, strip_V, L->bn);
  L->ldg = (L->w + L->bn - 1) / L->bn * L->bn;
  L->tiles = static_cast<int>((L->w + L->bn - 1) / L->bn);
  L->ldt = (N + 31) / 32 * 32;
  const size_t n = static_cast<size_t>(N);
  const size_t dd = static_cast<size_t>(d);
  const size_t elt = (dt == LCE_BF16) ? 2 : 4;
  size_t base = WS_HEADER_BYTES;
  if (x3) {  // split operands of both directions: H once per call, W one strip at a time
    L->h_part = align256(n * dd * 4);
    L->w_part = align256(static_cast<size_t>(L->w) * dd * 4);
    L->off_h = base;
    L->off_w = L->off_h + 2 * L->h_part;
    base = L->off_w + 2 * L->w_part;
  }
  L->off_run = base;
  L->off_tgt = L->off_run + align256(n * sizeof(float2));
  L->off_part = L->off_tgt + align256(n * sizeof(float));
  const size_t fwd_end = L->off_part + align256(static_cast<size_t>(L->tiles) * n * sizeof(float2));
  L->g_bytes = align256(n * static_cast<size_t>(L->ldg) * elt);
  size_t bwd_end;
  if (x3) {
    // transposed parts for the K-major tf32 MMAs of dH and dW, then G and G^T (hi, lo each)
    L->ht_part = align256(dd * static_cast<size_t>(L->ldt) * 4);
    L->wt_part = align256(dd * static_cast<size_t>(L->ldg) * 4);
    L->gt_part = align256(static_cast<size_t>(L->ldg) * static_cast<size_t>(L->ldt) * 4);
    L->off_ht = base;
    L->off_wt = L->off_ht + 2 * L->ht_part;
    L->off_g = L->off_wt + 2 * L->wt_part;
    L->off_gt = L->off_g + 2 * L->g_bytes;
    bwd_end = L->off_gt + 2 * L->gt_part;
  } else {
    // A small backward step (dH of one strip: few 256 x 256 tiles, a launch of a few waves) runs
    // overlapped with the next strip's gradient in one launch, which needs a second gradient
    // strip; a large one fills the GPU by itself and keeps the single strip.
    const int64_t dh_tiles = ((N + 255) / 256) * ((d + 255) / 256);
    L->overlap_bwd = (dt == LCE_BF16) && dh_tiles <= kOverlapMaxTiles;
    L->off_g = base;
    bwd_end = L->off_g + (L->overlap_bwd ? 2 : 1) * L->g_bytes;
  }
  L->total = std::max(fwd_end, bwd_end);
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device buffer of lce_forward_backward_host: the workspace, then the device copies of the inputs
// (H, W, labels, dloss) and the results (loss, n_valid, lse, dH, dW), each 256-byte aligned.
struct HostLayout {
  size_t ws, off_H, off_W, off_y, off_dloss, off_loss, off_nv, off_lse, off_dH, off_dW, total;
};

bool make_host_layout(int64_t N, int64_t d, int64_t V, int64_t strip_V, lce_dtype_t dt,
                      HostLayout* h) {
  Layout L;
  if (!make_layout(N, d, V, strip_V, dt, &L)) return false;
  const size_t n = static_cast<size_t>(N), dd = static_cast<size_t>(d), v = static_cast<size_t>(V);
  const size_t elt = (dt == LCE_BF16) ? 2 : 4;
  h->ws = L.total;
  size_t off = align256(L.total);
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  h->off_H = take(n * dd * elt);
  h->off_W = take(v * dd * elt);
  h->off_y = take(n * sizeof(int64_t));
  h->off_dloss = take(sizeof(float));
  h->off_loss = take(sizeof(float));
  h->off_nv = take(sizeof(int64_t));
  h->off_lse = take(n * sizeof(float));
  h->off_dH = take(n * dd * sizeof(float));
  h->off_dW = take(v * dd * sizeof(float));
  h->total = off;
  return true;
}

// --------------------------------------------------------------------------- device checks
thread_local char g_last_error[384] = "none";
thread_local bool g_detail_set = false;

int g_sms[kMaxDevices];
signed char g_dev_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 not sm_103

}  // namespace

// Records the CUDA error of a failed call unless the failing step already described itself.
cudaError_t note(cudaError_t e) {
  if (e != cudaSuccess && !g_detail_set)
    snprintf(g_last_error, sizeof(g_last_error), "%s", cudaGetErrorName(e));
  g_detail_set = false;
  return e;
}

lce_status_t check_device(int* num_sms) {
  int dev = 0;
  if (note(cudaGetDevice(&dev)) != cudaSuccess) return LCE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LCE_ERR_UNSUPPORTED_DEVICE;
  // Make the device's primary context current on this thread: the tensor maps are encoded with
  // the driver API, which needs a current context, and a fresh thread (e.g. autograd's backward
  // worker) has none until its first context-creating runtime call.
  if (note(cudaSetDevice(dev)) != cudaSuccess) return LCE_ERR_CUDA;
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LCE_ERR_CUDA;
    g_sms[dev] = sms;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_dev_ok[dev] < 0) return LCE_ERR_UNSUPPORTED_DEVICE;
  *num_sms = g_sms[dev];
  return LCE_OK;
}

namespace {

// --------------------------------------------------------------------------- launch bookkeeping
std::atomic<int64_t> g_launches{0};

struct Trace {
  void* const* start = nullptr;
  void* const* stop = nullptr;
  int32_t* ids = nullptr;
  int32_t cap = 0;
  int32_t n = 0;
  bool active = false;
};
Trace g_trace;

template <typename F>
cudaError_t traced(int kid, cudaStream_t stream, F&& launch) {
  const bool rec = g_trace.active && g_trace.n < g_trace.cap;
  if (rec) {
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(g_trace.start[g_trace.n]), stream);
    if (e != cudaSuccess) return e;
  }
  // Drop a stale, non-sticky error another library may have left on this thread, so that the
  // check after the launch reports only this launch (sticky errors are reported again anyway).
  (void)cudaGetLastError();
  g_detail_set = false;
  g_extra_kernels = 0;
  cudaError_t e = note(launch());
  if (e != cudaSuccess) return e;
  g_launches.fetch_add(1 + g_extra_kernels, std::memory_order_relaxed);
  g_extra_kernels = 0;
  if (rec) {
    e = cudaEventRecord(static_cast<cudaEvent_t>(g_trace.stop[g_trace.n]), stream);
    if (e != cudaSuccess) return e;
    g_trace.ids[g_trace.n] = kid;
    ++g_trace.n;
  }
  return cudaSuccess;
}

cudaError_t strip_gemm(const StripArgs& a, lce_dtype_t dt, cudaStream_t stream, int num_sms) {
  if (dt != LCE_F32)  // the tensor-core backward goes through tc_strip_jobs, never through here
    return traced(K_TC_FWD, stream, [&] { return tc_strip_gemm(a, stream, num_sms); });
  static const int kid[4] = {K_SIMT_FWD, K_SIMT_BWD_G, K_SIMT_DH, K_SIMT_DW};
  return traced(kid[a.mode], stream, [&] { return simt_strip_gemm(a, stream); });
}

lce_status_t common_checks(const void* H, const void* W, const int64_t* labels, int64_t N,
                           int64_t d, int64_t V, int64_t strip_V, lce_reduction_t red,
                           lce_dtype_t dt, const void* ws, size_t ws_bytes, Layout* L) {
  if (red != LCE_REDUCTION_MEAN && red != LCE_REDUCTION_SUM) return LCE_ERR_INVALID_ARG;
  if (dt != LCE_BF16 && dt != LCE_F32 && dt != LCE_F32_TF32X3) return LCE_ERR_INVALID_ARG;
  // H and labels may be null only when there is no token
  if (!W || !ws || (N > 0 && (!H || !labels))) return LCE_ERR_INVALID_ARG;
  if (!aligned16(H) || !aligned16(W) || !aligned16(labels) || !aligned16(ws))
    return LCE_ERR_INVALID_ARG;
  if (!make_layout(N, d, V, strip_V, dt, L)) return LCE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < L->total) return LCE_ERR_WORKSPACE_TOO_SMALL;
  return LCE_OK;
}

// LCE_F32_TF32X3: tf32 hi / lo parts of n fp32 values into the workspace at `off` (lo at
// off + part).
cudaError_t split(const void* x, size_t n, char* ws, size_t off, size_t part, cudaStream_t stream) {
  return traced(K_SPLIT, stream, [&] {
    return launch_split_tf32(static_cast<const float*>(x), reinterpret_cast<float*>(ws + off),
                             reinterpret_cast<float*>(ws + off + part), n, stream);
  });
}
// The same for x [rows x cols], written transposed with row stride ld_out.
cudaError_t split_t(const void* x, int64_t rows, int64_t cols, int64_t ld_out, char* ws,
                    size_t off, size_t part, cudaStream_t stream) {
  return traced(K_SPLIT, stream, [&] {
    return launch_split_tf32_t(static_cast<const float*>(x), rows, cols, ld_out,
                               reinterpret_cast<float*>(ws + off),
                               reinterpret_cast<float*>(ws + off + part), stream);
  });
}

// Operands of one LCE_F32_TF32X3 strip GEMM: the split parts of H and of the current W strip
// (which holds only this strip's rows), and for the backward the transposed parts and G / G^T.
void set_x3_operands(StripArgs& a, char* ws, const Layout& L) {
  a.op = OP_TF32X3;
  a.H = ws + L.off_h;   a.H2 = ws + L.off_h + L.h_part;
  a.W = ws + L.off_w;   a.W2 = ws + L.off_w + L.w_part;
  a.w_strip_local = 1;
  a.HT = ws + L.off_ht; a.HT2 = ws + L.off_ht + L.ht_part;
  a.WT = ws + L.off_wt; a.WT2 = ws + L.off_wt + L.wt_part;
  a.G = ws + L.off_g;   a.G2 = ws + L.off_g + L.g_bytes;
  a.GT = ws + L.off_gt; a.GT2 = ws + L.off_gt + L.gt_part;
  a.ldt = L.ldt;
}

}  // namespace

thread_local int g_extra_kernels = 0;

void set_error_detail(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  g_detail_set = true;
}

}  // namespace lce

using namespace lce;

extern "C" {

int64_t lce_strip_columns(int64_t V, int64_t strip_V, lce_dtype_t dtype) {
  if (dtype != LCE_BF16 && dtype != LCE_F32 && dtype != LCE_F32_TF32X3) return 0;
  if (V < 1 || V > kMaxDim || strip_V < 128 || strip_V % 128 != 0 || strip_V > kMaxDim) return 0;
  return strip_columns(V, strip_V, dtype == LCE_F32 ? SIMT_BN : TC_BN);
}

size_t lce_workspace_size(int64_t N, int64_t d, int64_t V, int64_t strip_V, lce_dtype_t dtype) {
  Layout L;
  if (!make_layout(N, d, V, strip_V, dtype, &L)) return 0;
  return L.total;
}

lce_status_t lce_forward(const void* H, const void* W, const int64_t* labels, int64_t N, int64_t d,
                         int64_t V, int64_t ignore_index, int64_t strip_V, lce_reduction_t reduction,
                         lce_dtype_t dtype, float* loss, float* lse, int64_t* n_valid,
                         void* workspace, size_t ws_bytes, void* stream_) {
  Layout L;
  lce_status_t st = common_checks(H, W, labels, N, d, V, strip_V, reduction, dtype, workspace,
                                  ws_bytes, &L);
  if (st != LCE_OK) return st;
  if (!loss || !n_valid || (N > 0 && !lse)) return LCE_ERR_INVALID_ARG;
  if (!aligned16(lse)) return LCE_ERR_INVALID_ARG;
  int num_sms = 0;
  if ((st = check_device(&num_sms)) != LCE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  char* ws = static_cast<char*>(workspace);
  unsigned* err = reinterpret_cast<unsigned*>(ws);
  float2* run = reinterpret_cast<float2*>(ws + L.off_run);
  float* tgt = reinterpret_cast<float*>(ws + L.off_tgt);
  float2* part = reinterpret_cast<float2*>(ws + L.off_part);
  if (note(cudaMemsetAsync(ws, 0, WS_HEADER_BYTES, stream)) != cudaSuccess) return LCE_ERR_CUDA;

  // The forward keeps one (max, sum-exp) partial per token and logit tile of the columns a launch
  // covers.  When the partials of the whole vocabulary fit in the workspace sized for the strip
  // width (the backward's gradient strip is larger whenever it is >= V/64), one persistent launch covers
  // every strip; otherwise there is one launch per strip.  Either way the workspace is the same.
  // LCE_F32_TF32X3 splits W one strip at a time, so it keeps one launch per strip.
  const bool x3 = (dtype == LCE_F32_TF32X3);
  const int64_t tiles_all = (V + L.bn - 1) / L.bn;
  const bool one_launch =
      !x3 && L.off_part + static_cast<size_t>(tiles_all) * static_cast<size_t>(N) * sizeof(float2) <=
                 L.total;
  const int64_t fwd_step = one_launch ? V : L.w;
  if (N > 0) {
    if (x3 && split(H, static_cast<size_t>(N) * d, ws, L.off_h, L.h_part, stream) != cudaSuccess)
      return LCE_ERR_CUDA;
    for (int64_t col0 = 0, s = 0; col0 < V; col0 += fwd_step, ++s) {
      StripArgs a{};
      a.mode = MODE_FWD_LSE;
      a.col0 = static_cast<int>(col0);
      a.strip_cols = static_cast<int>(std::min(fwd_step, V - col0));
      a.H = H; a.W = W; a.d = d; a.N = N; a.V = V;
      a.part = part; a.tgt = tgt;
      a.labels = labels; a.ignore_index = ignore_index;
      a.err = err; a.first_strip = (s == 0);
      if (x3) {
        const float* w_strip = static_cast<const float*>(W) + static_cast<size_t>(col0) * d;
        if (split(w_strip, static_cast<size_t>(a.strip_cols) * d, ws, L.off_w, L.w_part,
                  stream) != cudaSuccess)
          return LCE_ERR_CUDA;
        set_x3_operands(a, ws, L);
      }
      if (strip_gemm(a, dtype, stream, num_sms) != cudaSuccess) return LCE_ERR_CUDA;
      const int tiles = (a.strip_cols + L.bn - 1) / L.bn;
      if (traced(K_COMBINE, stream, [&] {
            return launch_combine(part, tiles, N, run, s == 0, stream);
          }) != cudaSuccess)
        return LCE_ERR_CUDA;
    }
  }
  if (traced(K_FINALIZE, stream, [&] {
        return launch_finalize(run, tgt, labels, N, V, ignore_index, reduction, loss, lse, n_valid,
                               err, stream);
      }) != cudaSuccess)
    return LCE_ERR_CUDA;
  return LCE_OK;
}

}  // extern "C"

namespace lce {
namespace {

// The backward.  keep_flags: leave the error flags (header word 0) as the forward left them, so
// that one flag word reports both passes (lce_forward_backward_host); the rest of the header (the
// tile scheduler's counters) is cleared either way.
lce_status_t backward_impl(const void* H, const void* W, const int64_t* labels, const float* lse,
                           const int64_t* n_valid, const float* dloss, int64_t N, int64_t d,
                           int64_t V, int64_t ignore_index, int64_t strip_V,
                           lce_reduction_t reduction, lce_dtype_t dtype, int32_t parts, float* dH,
                           float* dW, void* workspace, size_t ws_bytes, void* stream_,
                           bool keep_flags) {
  Layout L;
  lce_status_t st = common_checks(H, W, labels, N, d, V, strip_V, reduction, dtype, workspace,
                                  ws_bytes, &L);
  if (st != LCE_OK) return st;
  if (parts < 1 || parts > (LCE_GRAD_DH | LCE_GRAD_DW)) return LCE_ERR_INVALID_ARG;
  const bool want_dh = (parts & LCE_GRAD_DH) != 0;
  const bool want_dw = (parts & LCE_GRAD_DW) != 0;
  if (!n_valid || !dloss || (want_dw && !dW) || (N > 0 && (!lse || (want_dh && !dH))))
    return LCE_ERR_INVALID_ARG;
  if (!aligned16(lse) || !aligned16(dH) || !aligned16(dW)) return LCE_ERR_INVALID_ARG;
  int num_sms = 0;
  if ((st = check_device(&num_sms)) != LCE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  char* ws = static_cast<char*>(workspace);
  unsigned* err = reinterpret_cast<unsigned*>(ws);
  void* G = ws + L.off_g;
  // error flags and scheduler counters start from zero (the workspace may be fresh memory)
  const size_t keep = keep_flags ? sizeof(unsigned) : 0;
  if (note(cudaMemsetAsync(ws + keep, 0, WS_HEADER_BYTES - keep, stream)) != cudaSuccess)
    return LCE_ERR_CUDA;
  if (N == 0) {
    // no token: every logit-gradient row is absent, so dW = 0 (dH has no rows)
    if (want_dw &&
        note(cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * d * sizeof(float), stream)) !=
            cudaSuccess)
      return LCE_ERR_CUDA;
    return LCE_OK;
  }
  auto strip_job = [&](int64_t s, int mode, void* g) {
    StripArgs a{};
    const int64_t col0 = s * L.w;
    a.mode = mode;
    a.col0 = static_cast<int>(col0);
    a.strip_cols = static_cast<int>(std::min(L.w, V - col0));
    a.H = H; a.W = W; a.d = d; a.N = N; a.V = V;
    a.G = g; a.ldg = L.ldg;
    a.labels = labels; a.ignore_index = ignore_index;
    a.lse = lse; a.dloss = dloss; a.n_valid = n_valid; a.reduction = reduction;
    a.err = err; a.first_strip = (s == 0);
    a.ldc = d; a.c_cols = static_cast<int>(d);
    if (mode == MODE_DH) {
      a.C = dH; a.accumulate = (s > 0); a.c_rows = static_cast<int>(N);
    } else if (mode == MODE_DW) {
      a.C = dW + static_cast<size_t>(col0) * d; a.c_rows = a.strip_cols;
    }
    return a;
  };
  const int64_t S = (V + L.w - 1) / L.w;
  auto run = [&](StripArgs* jobs, int nj) {
    bool grad = false, dhdw = false;
    for (int j = 0; j < nj; ++j) (jobs[j].mode == MODE_BWD_G ? grad : dhdw) = true;
    const int kid = (grad && dhdw) ? K_TC_BWD : (grad ? K_TC_GRAD : K_TC_DHDW);
    return traced(kid, stream, [&] { return tc_strip_jobs(jobs, nj, stream, num_sms); });
  };
  if (dtype == LCE_F32_TF32X3) {
    // H split once, plain (and transposed for dW).  Per strip: the W strip split, plain (and
    // transposed for dH); one launch for its gradient (G and G^T, hi and lo parts); one launch
    // for dH and dW from it (dH's tiles first; dH accumulates strip after strip in order).
    if (split(H, static_cast<size_t>(N) * d, ws, L.off_h, L.h_part, stream) != cudaSuccess ||
        (want_dw && split_t(H, N, d, L.ldt, ws, L.off_ht, L.ht_part, stream) != cudaSuccess))
      return LCE_ERR_CUDA;
    for (int64_t s = 0; s < S; ++s) {
      StripArgs grad = strip_job(s, MODE_BWD_G, nullptr);
      set_x3_operands(grad, ws, L);
      StripArgs jobs[2];
      int nj = 0;
      if (want_dh) jobs[nj++] = strip_job(s, MODE_DH, nullptr);
      if (want_dw) jobs[nj++] = strip_job(s, MODE_DW, nullptr);
      for (int j = 0; j < nj; ++j) set_x3_operands(jobs[j], ws, L);
      const float* w_strip = static_cast<const float*>(W) + static_cast<size_t>(s * L.w) * d;
      if (split(w_strip, static_cast<size_t>(grad.strip_cols) * d, ws, L.off_w, L.w_part,
                stream) != cudaSuccess ||
          (want_dh && split_t(w_strip, grad.strip_cols, d, L.ldg, ws, L.off_wt, L.wt_part,
                              stream) != cudaSuccess))
        return LCE_ERR_CUDA;
      if (run(&grad, 1) != cudaSuccess || run(jobs, nj) != cudaSuccess) return LCE_ERR_CUDA;
    }
    return LCE_OK;
  }
  if (dtype == LCE_BF16) {
    if (L.overlap_bwd) {
      // Step s computes dH and dW of strip s-1 (from gradient buffer (s-1) % 2, the longer
      // reductions first) together with the gradient strip s (into buffer s % 2): one persistent
      // launch per step, S + 1 steps.  dH accumulates strip after strip in order.
      void* gbuf[2] = {G, static_cast<char*>(G) + L.g_bytes};
      for (int64_t s = 0; s <= S; ++s) {
        StripArgs jobs[3];
        int nj = 0;
        if (s >= 1 && want_dh) jobs[nj++] = strip_job(s - 1, MODE_DH, gbuf[(s - 1) & 1]);
        if (s >= 1 && want_dw) jobs[nj++] = strip_job(s - 1, MODE_DW, gbuf[(s - 1) & 1]);
        if (s < S) jobs[nj++] = strip_job(s, MODE_BWD_G, gbuf[s & 1]);
        if (run(jobs, nj) != cudaSuccess) return LCE_ERR_CUDA;
      }
    } else {
      // Per strip: its gradient, then dW and dH from it in one launch (the dW tiles, the longer
      // reductions, first, so the dH tiles fill the last wave) -- one gradient strip.
      for (int64_t s = 0; s < S; ++s) {
        StripArgs grad = strip_job(s, MODE_BWD_G, G);
        if (run(&grad, 1) != cudaSuccess) return LCE_ERR_CUDA;
        StripArgs jobs[2];
        int nj = 0;
        if (want_dw) jobs[nj++] = strip_job(s, MODE_DW, G);
        if (want_dh) jobs[nj++] = strip_job(s, MODE_DH, G);
        if (run(jobs, nj) != cudaSuccess) return LCE_ERR_CUDA;
      }
    }
    return LCE_OK;
  }
  for (int64_t col0 = 0, s = 0; col0 < V; col0 += L.w, ++s) {
    StripArgs a = strip_job(s, MODE_BWD_G, G);
    a.mode = MODE_BWD_G;
    if (strip_gemm(a, dtype, stream, num_sms) != cudaSuccess) return LCE_ERR_CUDA;

    a.mode = MODE_DH;
    a.C = dH; a.ldc = d; a.accumulate = (s > 0); a.c_rows = static_cast<int>(N);
    a.c_cols = static_cast<int>(d);
    if (want_dh && strip_gemm(a, dtype, stream, num_sms) != cudaSuccess) return LCE_ERR_CUDA;

    a.mode = MODE_DW;
    a.C = dW + static_cast<size_t>(col0) * d; a.ldc = d; a.accumulate = 0;
    a.c_rows = a.strip_cols; a.c_cols = static_cast<int>(d);
    if (want_dw && strip_gemm(a, dtype, stream, num_sms) != cudaSuccess) return LCE_ERR_CUDA;
  }
  return LCE_OK;
}

}  // namespace
}  // namespace lce

extern "C" {

lce_status_t lce_backward_parts(const void* H, const void* W, const int64_t* labels,
                                const float* lse, const int64_t* n_valid, const float* dloss,
                                int64_t N, int64_t d, int64_t V, int64_t ignore_index,
                                int64_t strip_V, lce_reduction_t reduction, lce_dtype_t dtype,
                                int32_t parts, float* dH, float* dW, void* workspace,
                                size_t ws_bytes, void* stream) {
  return backward_impl(H, W, labels, lse, n_valid, dloss, N, d, V, ignore_index, strip_V,
                       reduction, dtype, parts, dH, dW, workspace, ws_bytes, stream, false);
}

lce_status_t lce_backward(const void* H, const void* W, const int64_t* labels, const float* lse,
                          const int64_t* n_valid, const float* dloss, int64_t N, int64_t d, int64_t V,
                          int64_t ignore_index, int64_t strip_V, lce_reduction_t reduction,
                          lce_dtype_t dtype, float* dH, float* dW, void* workspace,
                          size_t ws_bytes, void* stream) {
  return lce_backward_parts(H, W, labels, lse, n_valid, dloss, N, d, V, ignore_index, strip_V,
                            reduction, dtype, LCE_GRAD_DH | LCE_GRAD_DW, dH, dW, workspace,
                            ws_bytes, stream);
}

size_t lce_host_buffer_size(int64_t N, int64_t d, int64_t V, int64_t strip_V, lce_dtype_t dtype) {
  HostLayout h;
  if (!make_host_layout(N, d, V, strip_V, dtype, &h)) return 0;
  return h.total;
}

lce_status_t lce_forward_backward_host(const void* H, const void* W, const int64_t* labels,
                                       const float* dloss, int64_t N, int64_t d, int64_t V,
                                       int64_t ignore_index, int64_t strip_V,
                                       lce_reduction_t reduction, lce_dtype_t dtype, float* loss,
                                       float* lse, int64_t* n_valid, float* dH, float* dW,
                                       uint32_t* device_error_flags, void* device_buffer,
                                       size_t device_bytes, void* stream_,
                                       const void* compute_after, void* compute_done) {
  // host-side validation first: nothing reaches the CUDA runtime on a bad argument
  if (reduction != LCE_REDUCTION_MEAN && reduction != LCE_REDUCTION_SUM) return LCE_ERR_INVALID_ARG;
  if (dtype != LCE_BF16 && dtype != LCE_F32 && dtype != LCE_F32_TF32X3) return LCE_ERR_INVALID_ARG;
  if (!W || !dloss || !device_buffer || (N > 0 && (!H || !labels))) return LCE_ERR_INVALID_ARG;
  if (!aligned16(device_buffer)) return LCE_ERR_INVALID_ARG;
  HostLayout h;
  if (!make_host_layout(N, d, V, strip_V, dtype, &h)) return LCE_ERR_UNSUPPORTED_SHAPE;
  if (device_bytes < h.total) return LCE_ERR_WORKSPACE_TOO_SMALL;
  int num_sms = 0;
  lce_status_t st = check_device(&num_sms);
  if (st != LCE_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  char* buf = static_cast<char*>(device_buffer);
  const size_t n = static_cast<size_t>(N), dd = static_cast<size_t>(d), v = static_cast<size_t>(V);
  const size_t elt = (dtype == LCE_BF16) ? 2 : 4;
  void* dH_in = buf + h.off_H;
  void* dW_in = buf + h.off_W;
  int64_t* d_y = reinterpret_cast<int64_t*>(buf + h.off_y);
  float* d_dloss = reinterpret_cast<float*>(buf + h.off_dloss);
  float* d_loss = reinterpret_cast<float*>(buf + h.off_loss);
  int64_t* d_nv = reinterpret_cast<int64_t*>(buf + h.off_nv);
  float* d_lse = reinterpret_cast<float*>(buf + h.off_lse);
  float* d_dH = reinterpret_cast<float*>(buf + h.off_dH);
  float* d_dW = reinterpret_cast<float*>(buf + h.off_dW);
  auto copy = [&](void* dst, const void* src, size_t bytes, cudaMemcpyKind kind) {
    return bytes == 0 || note(cudaMemcpyAsync(dst, src, bytes, kind, stream)) == cudaSuccess;
  };
  if (!copy(dH_in, H, n * dd * elt, cudaMemcpyHostToDevice) ||
      !copy(dW_in, W, v * dd * elt, cudaMemcpyHostToDevice) ||
      !copy(d_y, labels, n * sizeof(int64_t), cudaMemcpyHostToDevice) ||
      !copy(d_dloss, dloss, sizeof(float), cudaMemcpyHostToDevice))
    return LCE_ERR_CUDA;
  if (compute_after &&
      note(cudaStreamWaitEvent(stream, static_cast<cudaEvent_t>(const_cast<void*>(compute_after)),
                               0)) != cudaSuccess)
    return LCE_ERR_CUDA;
  st = lce_forward(dH_in, dW_in, d_y, N, d, V, ignore_index, strip_V, reduction, dtype, d_loss,
                   d_lse, d_nv, buf, h.ws, stream_);
  if (st != LCE_OK) return st;
  // the backward keeps the forward's error bits and adds its own
  st = backward_impl(dH_in, dW_in, d_y, d_lse, d_nv, d_dloss, N, d, V, ignore_index, strip_V,
                     reduction, dtype, LCE_GRAD_DH | LCE_GRAD_DW, d_dH, d_dW, buf, h.ws, stream_,
                     true);
  if (st != LCE_OK) return st;
  if (compute_done &&
      note(cudaEventRecord(static_cast<cudaEvent_t>(compute_done), stream)) != cudaSuccess)
    return LCE_ERR_CUDA;
  if ((loss && !copy(loss, d_loss, sizeof(float), cudaMemcpyDeviceToHost)) ||
      (n_valid && !copy(n_valid, d_nv, sizeof(int64_t), cudaMemcpyDeviceToHost)) ||
      (lse && !copy(lse, d_lse, n * sizeof(float), cudaMemcpyDeviceToHost)) ||
      (dH && !copy(dH, d_dH, n * dd * sizeof(float), cudaMemcpyDeviceToHost)) ||
      (dW && !copy(dW, d_dW, v * dd * sizeof(float), cudaMemcpyDeviceToHost)) ||
      (device_error_flags &&
       !copy(device_error_flags, buf, sizeof(uint32_t), cudaMemcpyDeviceToHost)))
    return LCE_ERR_CUDA;
  return LCE_OK;
}

lce_status_t lce_check_error(const void* workspace, void* stream_) {
  if (!workspace) return LCE_ERR_INVALID_ARG;
  unsigned flags = 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (note(cudaMemcpyAsync(&flags, workspace, sizeof(flags), cudaMemcpyDeviceToHost, stream)) !=
      cudaSuccess)
    return LCE_ERR_CUDA;
  if (note(cudaStreamSynchronize(stream)) != cudaSuccess) return LCE_ERR_CUDA;
  if (flags & ERR_TIMEOUT) return LCE_ERR_TIMEOUT;
  if (flags & ERR_LABEL) return LCE_ERR_LABEL_OUT_OF_RANGE;
  return LCE_OK;
}

const char* lce_status_string(lce_status_t s) {
  switch (s) {
    case LCE_OK: return "ok";
    case LCE_ERR_INVALID_ARG: return "invalid argument";
    case LCE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case LCE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case LCE_ERR_LABEL_OUT_OF_RANGE: return "label out of range";
    case LCE_ERR_CUDA: return "CUDA error";
    case LCE_ERR_TIMEOUT: return "kernel wait timed out";
    case LCE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
  }
  return "unknown status";
}

const char* lce_last_cuda_error(void) { return g_last_error; }

lce_status_t lce_set_tile_config(int32_t config) {
  if (config < 0 || config > 2) return LCE_ERR_INVALID_ARG;
  g_tile_config = config;
  return LCE_OK;
}

lce_status_t lce_test_inject_stall(int32_t on) {
  if (on != 0 && on != 1) return LCE_ERR_INVALID_ARG;
  g_inject_stall = on;
  return LCE_OK;
}

int64_t lce_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

lce_status_t lce_trace_begin(void* const* start_events, void* const* stop_events,
                             int32_t* kernel_ids, int32_t capacity) {
  if (capacity < 0 || (capacity > 0 && (!start_events || !stop_events || !kernel_ids)))
    return LCE_ERR_INVALID_ARG;
  g_trace.start = start_events;
  g_trace.stop = stop_events;
  g_trace.ids = kernel_ids;
  g_trace.cap = capacity;
  g_trace.n = 0;
  g_trace.active = true;
  return LCE_OK;
}

int32_t lce_trace_end(void) {
  g_trace.active = false;
  return g_trace.n;
}

const char* lce_kernel_name(int32_t id) {
  static const char* names[K_NUM] = {"tc_fwd_lse",    "tc_bwd",   "simt_fwd_lse",
                                     "simt_bwd_grad", "simt_dh",  "simt_dw",
                                     "combine",       "finalize", "split_tf32",
                                     "tc_bwd_grad",   "tc_dh_dw"};
  return (id >= 0 && id < K_NUM) ? names[id] : nullptr;
}

}  // extern "C"
