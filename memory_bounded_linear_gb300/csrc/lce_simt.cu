// CUDA-core strip GEMM engine for fp32 operands (exact fp32 FFMA; TF32 tensor cores would not
// hold fp32 accuracy).  Same four epilogue modes and the same workspace contract as the
// tensor-core engine, with 64 x 64 output tiles:
//   FWD_LSE  per-(row, 64-column tile) (max, sum-exp) partial and the target logit
//   BWD_G    G = scale (softmax - onehot) into the fp32 strip workspace
//   DH       dH (+)= G_s W_s           DW   dW_s = G_s^T H
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "lce_internal.h"

namespace lce {
namespace {

constexpr int TM = 64;
constexpr int TN = SIMT_BN;  // 64
constexpr int TK = 16;
constexpr int THREADS = 256;  // 16 x 16 threads, 4 x 4 outputs each

struct SParams {
  int M, Ncols, K;
  int tiles_n;
  // element (m, k) of A is A[m * a_sm + k * a_sk]; (n, k) of B is B[n * b_sn + k * b_sk]
  const float* A;
  int64_t a_sm, a_sk;
  const float* B;
  int64_t b_sn, b_sk;
  int strip_cols, col0;
  float2* part;
  float* tgt;
  const int64_t* labels;
  int64_t V, ignore_index;
  const float* lse;
  const float* dloss;
  const int64_t* n_valid;
  int reduction;
  float* G;
  int64_t ldg;
  float* C;
  int64_t ldc;
  int accumulate, c_rows, c_cols;
  unsigned* err;
  int first_strip;
};

template <int MODE>
__global__ void __launch_bounds__(THREADS) simt_strip_kernel(const SParams p) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  __shared__ float Cs[TM][TN + 1];

  const int tm = blockIdx.y, tn = blockIdx.x;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = tm * TM, n0 = tn * TN;

  float acc[4][4] = {};
  for (int k0 = 0; k0 < p.K; k0 += TK) {
    for (int i = tid; i < TM * TK; i += THREADS) {
      // K-major operands walk k fastest, MN-major operands walk m fastest (coalesced either way)
      int mm, kk;
      if (p.a_sk == 1) { mm = i / TK; kk = i % TK; } else { mm = i % TM; kk = i / TM; }
      const int gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < p.M && gk < p.K) ? p.A[gm * p.a_sm + gk * p.a_sk] : 0.f;
      int nn, kb;
      if (p.b_sk == 1) { nn = i / TK; kb = i % TK; } else { nn = i % TN; kb = i / TN; }
      const int gn = n0 + nn, gkb = k0 + kb;
      Bs[kb][nn] = (gn < p.Ncols && gkb < p.K) ? p.B[gn * p.b_sn + gkb * p.b_sk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  if (MODE == MODE_FWD_LSE) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
    __syncthreads();
    if (tid < TM) {
      const int row = m0 + tid;
      if (row < p.M) {
        const int ncols = min(TN, p.strip_cols - n0);
        float m = -INFINITY;
        for (int j = 0; j < ncols; ++j) m = fmaxf(m, Cs[tid][j]);
        float s = 0.f;
        for (int j = 0; j < ncols; ++j) s += expf(Cs[tid][j] - m);
        p.part[static_cast<size_t>(tn) * p.M + row] = make_float2(m, s);
        const int64_t y = p.labels[row];
        const int64_t rel = y - static_cast<int64_t>(p.col0 + n0);
        if (y != p.ignore_index && y >= 0 && y < p.V && rel >= 0 && rel < ncols)
          p.tgt[row] = Cs[tid][rel];
      }
    }
  } else if (MODE == MODE_BWD_G) {
    const float dl = *p.dloss;
    const float scale_valid = (p.reduction == 0) ? dl / static_cast<float>(*p.n_valid) : dl;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = m0 + ty * 4 + i;
      if (row >= p.M) continue;
      const int64_t y = p.labels[row];
      const bool ok = (y != p.ignore_index) && (y >= 0) && (y < p.V);
      if (!ok && y != p.ignore_index && p.first_strip && tn == 0 && tx == 0)
        atomicOr(p.err, ERR_LABEL);
      const float l = ok ? p.lse[row] : 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = n0 + tx * 4 + j;  // strip-local column, < ldg by construction
        float g = 0.f;
        if (ok && col < p.strip_cols) {
          g = scale_valid * expf(acc[i][j] - l);
          if (static_cast<int64_t>(p.col0 + col) == y) g -= scale_valid;
        }
        p.G[static_cast<size_t>(row) * p.ldg + col] = g;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = m0 + ty * 4 + i;
      if (row >= p.c_rows) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = n0 + tx * 4 + j;
        if (col >= p.c_cols) continue;
        float* c = p.C + static_cast<size_t>(row) * p.ldc + col;
        *c = p.accumulate ? *c + acc[i][j] : acc[i][j];
      }
    }
  }
}

}  // namespace

cudaError_t simt_strip_gemm(const StripArgs& s, cudaStream_t stream) {
  SParams p{};
  const float* H = static_cast<const float*>(s.H);
  const float* W = static_cast<const float*>(s.W);
  const float* G = static_cast<const float*>(s.G);
  switch (s.mode) {
    case MODE_FWD_LSE:
    case MODE_BWD_G:
      p.M = static_cast<int>(s.N); p.Ncols = s.strip_cols; p.K = static_cast<int>(s.d);
      p.A = H; p.a_sm = s.d; p.a_sk = 1;
      p.B = W + static_cast<size_t>(s.col0) * s.d; p.b_sn = s.d; p.b_sk = 1;
      break;
    case MODE_DH:
      p.M = static_cast<int>(s.N); p.Ncols = static_cast<int>(s.d); p.K = s.strip_cols;
      p.A = G; p.a_sm = s.ldg; p.a_sk = 1;
      p.B = W + static_cast<size_t>(s.col0) * s.d; p.b_sn = 1; p.b_sk = s.d;
      break;
    case MODE_DW:
      p.M = s.strip_cols; p.Ncols = static_cast<int>(s.d); p.K = static_cast<int>(s.N);
      p.A = G; p.a_sm = 1; p.a_sk = s.ldg;
      p.B = H; p.b_sn = 1; p.b_sk = s.d;
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (p.M == 0 || p.Ncols == 0 || p.K == 0) return cudaSuccess;
  p.tiles_n = (p.Ncols + TN - 1) / TN;
  p.strip_cols = s.strip_cols; p.col0 = s.col0;
  p.part = s.part; p.tgt = s.tgt;
  p.labels = s.labels; p.V = s.V; p.ignore_index = s.ignore_index;
  p.lse = s.lse; p.dloss = s.dloss; p.n_valid = s.n_valid; p.reduction = s.reduction;
  p.G = static_cast<float*>(s.G); p.ldg = s.ldg;
  p.C = s.C; p.ldc = s.ldc; p.accumulate = s.accumulate; p.c_rows = s.c_rows; p.c_cols = s.c_cols;
  p.err = s.err; p.first_strip = s.first_strip;
  const dim3 grid(p.tiles_n, (p.M + TM - 1) / TM);
  switch (s.mode) {
    case MODE_FWD_LSE: simt_strip_kernel<MODE_FWD_LSE><<<grid, THREADS, 0, stream>>>(p); break;
    case MODE_BWD_G: simt_strip_kernel<MODE_BWD_G><<<grid, THREADS, 0, stream>>>(p); break;
    case MODE_DH: simt_strip_kernel<MODE_DH><<<grid, THREADS, 0, stream>>>(p); break;
    default: simt_strip_kernel<MODE_DW><<<grid, THREADS, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace lce
