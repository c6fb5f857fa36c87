// Internal interfaces between the C-ABI host code (lce_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lce.h"

namespace lce {

// Devices a process may use with this library (ordinals 0 .. kMaxDevices-1).
constexpr int kMaxDevices = 64;

// Checks that the current device is compute capability 10.3 and makes its primary context
// current on the calling thread; fills the device's SM count.  LCE_OK, LCE_ERR_CUDA or
// LCE_ERR_UNSUPPORTED_DEVICE (lce_api.cu).
lce_status_t check_device(int* num_sms);
// Passes a CUDA status through, recording the name of a failure for lce_last_cuda_error unless
// the failing step already described itself (lce_api.cu).
cudaError_t note(cudaError_t e);

// Error-flag bits kept in the first word of the workspace header.
constexpr unsigned ERR_LABEL = 1u;     // a label outside [0, V) that is not ignore_index
constexpr unsigned ERR_TIMEOUT = 2u;   // a kernel-side wait ran out of time

// Workspace header: word 0 error flags; words 16-17 the tile scheduler's ticket counters (zero
// between launches: cleared with the header by each entry point, reset by every launch's last
// CTA).  Both entry points clear the header before their first launch.
constexpr size_t WS_HEADER_BYTES = 256;
constexpr int WS_SCHED_WORD = 16;

// The four epilogues of the strip GEMM engine.
enum Mode : int {
  MODE_FWD_LSE = 0,  // Z tile = H W_s^T; epilogue folds it into per-(row, tile) (max, sum-exp)
  MODE_BWD_G = 1,    // Z tile recomputed; epilogue writes G = scale (softmax - onehot)
  MODE_DH = 2,       // dH (+)= G_s W_s
  MODE_DW = 3,       // dW_s = G_s^T H
};

// Kernel ids reported by the launch tracer.
// K_TC_BWD is an overlapped backward step: dH and dW of one strip together with the gradient of
// the next.  K_TC_GRAD is a strip's gradient alone; K_TC_DHDW its dH and / or dW.
// K_SPLIT is the tf32 hi / lo split of an fp32 operand (plain or transposed).
enum KernelId : int {
  K_TC_FWD = 0, K_TC_BWD = 1,
  K_SIMT_FWD = 2, K_SIMT_BWD_G = 3, K_SIMT_DH = 4, K_SIMT_DW = 5,
  K_COMBINE = 6, K_FINALIZE = 7, K_SPLIT = 8, K_TC_GRAD = 9, K_TC_DHDW = 10, K_NUM = 11
};

// Operand formats of the tensor-core engine.  OP_BF16: bf16 operands.  OP_TF32X3: fp32 operands
// held as tf32 parts x = hi + lo; every product is hi*hi' + hi*lo' + lo*hi'.
constexpr int OP_BF16 = 0;
constexpr int OP_TF32X3 = 1;

// Arguments of one strip-GEMM launch (both the tensor-core and the fp32 CUDA-core engines).
// GEMM view: C[M x Ncols] = A[M x K] * B[Ncols x K]^T.
struct StripArgs {
  int mode;
  int M, Ncols, K;            // GEMM extents
  int col0;                   // first vocabulary column of the strip (W row offset)
  int strip_cols;             // columns of this strip (<= strip_V)
  // operands (device pointers)
  const void* H; const void* W; int64_t d, N, V;
  void* G; int64_t ldg;       // strip gradient workspace, row stride ldg elements
  // forward epilogue
  float2* part;               // [tiles_n][N] per-(tile, row) (max, sum-exp)
  float* tgt;                 // [N] target logit
  // backward epilogue
  const int64_t* labels; int64_t ignore_index;
  const float* lse; const float* dloss; const int64_t* n_valid; int reduction;
  // dH / dW epilogue
  float* C; int64_t ldc; int accumulate; int c_rows; int c_cols;
  unsigned* err;
  int first_strip;
  // Operand format (OP_*).  For OP_TF32X3, H, W and G point at the hi parts and H2, W2, G2 at
  // the lo parts.
  int op;
  const void* H2; const void* W2; void* G2;
  // W (and W2) hold only this strip's rows (row 0 = vocabulary column col0), not all V rows.
  int w_strip_local;
  // OP_TF32X3 only.  The tf32 MMAs read every operand K-major, so the contractions over the
  // vocabulary (dH) and over the tokens (dW) take transposed hi / lo copies:
  //   WT, WT2 [d x ldg]    this strip's rows of W, transposed (dH's B operand)
  //   HT, HT2 [d x ldt]    H transposed (dW's B operand)
  //   GT, GT2 [ldg x ldt]  the gradient strip transposed, written by the gradient epilogue
  //                        beside G (dW's A operand)
  const void* WT; const void* WT2; const void* HT; const void* HT2; void* GT; void* GT2;
  int64_t ldt;  // row stride (elements) of HT and GT: N rounded up to a multiple of 32
};

// Kernels a launcher started beyond its first one (the launch counter adds them), per thread.
extern thread_local int g_extra_kernels;

// Records a human-readable description of the last failure on the calling thread (reported by
// lce_last_cuda_error).  printf-style.
void set_error_detail(const char* fmt, ...);

// Tile widths of the two engines (columns of a logit tile).
constexpr int TC_BN = 256;
constexpr int SIMT_BN = 128;

// Tile variant of the tensor-core engine: 0 automatic, 1 single-CTA 128x256 tiles, 2 CTA-pair
// 256x256 tiles (set through lce_set_tile_config).
extern int g_tile_config;
// Test hook: when set, the next tensor-core launch withholds its first k-block (then it clears).
extern int g_inject_stall;

// Tensor-core (tcgen05) engine, bf16 or tf32-split fp32 operands: lce_tc.cu
cudaError_t tc_strip_gemm(const StripArgs& a, cudaStream_t stream, int num_sms);
// Up to three strip GEMMs in one persistent launch, their tiles scheduled together in order.
cudaError_t tc_strip_jobs(const StripArgs* jobs, int njobs, cudaStream_t stream, int num_sms);
// CUDA-core engine, fp32 operands (exact FFMA): lce_simt.cu
cudaError_t simt_strip_gemm(const StripArgs& a, cudaStream_t stream);
// Reductions and operand splits: lce_reduce.cu
// x[0..n) -> hi = nearest tf32 of x, lo = nearest tf32 of (x - hi), both in fp32 containers.
cudaError_t launch_split_tf32(const float* x, float* hi, float* lo, size_t n, cudaStream_t stream);
// The same split of x [rows x cols] (row-major), written transposed: hi / lo [cols x ld_out].
cudaError_t launch_split_tf32_t(const float* x, int64_t rows, int64_t cols, int64_t ld_out,
                                float* hi, float* lo, cudaStream_t stream);
// Folds the per-(tile, row) partials of one strip into the running state; may overwrite
// partials (they are consumed).
cudaError_t launch_combine(float2* part, int tiles, int64_t N, float2* run, int first,
                           cudaStream_t stream);
cudaError_t launch_finalize(const float2* run, const float* tgt, const int64_t* labels,
                            int64_t N, int64_t V, int64_t ignore_index, int reduction,
                            float* loss, float* lse, int64_t* n_valid, unsigned* err,
                            cudaStream_t stream);

}  // namespace lce
