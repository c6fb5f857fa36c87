// CUDA-core strip GEMM engine for fp32 operands with exact fp32 products (FFMA).  Same four
// epilogue modes and the same workspace contract as the tensor-core engine, with 128 x 128
// output tiles:
//   FWD_LSE  per-(row, 128-column tile) (max, sum-exp) partial and the target logit
//   BWD_G    G = scale (softmax - onehot) into the fp32 strip workspace
//   DH       dH (+)= G_s W_s           DW   dW_s = G_s^T H
//
// A register-tiled SGEMM: 128 threads (four warps, each owning 32 rows x 128 columns of the
// tile), each thread an 8 x 16 block of outputs: rows warp*32 + r*4 + {0..3} and the same + 16,
// columns c*4 + {0..3} + 32 q for q = 0..3, with r = lane / 8 and c = lane % 8.  A row of the tile
// therefore lives in the 8 lanes of one warp that share r.  k-blocks of 8 are staged in shared
// memory as [k][m] and [k][n] rows, so every k step is two float4 reads of A and four of B for
// 128 FMAs, issued as 64 packed fp32 FMAs (__ffma2_rn) on pairs of adjacent columns with a
// broadcast A value; the reads of step k + 1 are issued before the FMAs of step k, and the next
// k-block is loaded into registers while the current one is multiplied (one barrier per k-block).
// Operands are K-major or MN-major per mode; both are read as float4 along their contiguous
// dimension, with a scalar path at the ragged edges.  Two blocks per SM, up to 255 registers a
// thread: 128 accumulators, two sets of 24 fragment values, 16 staged operand values.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "lce_internal.h"

namespace lce {
namespace {

constexpr int TM = 128;
constexpr int TN = SIMT_BN;  // 128
constexpr int TK = 8;
constexpr int THREADS = 128;  // 4 warps x 32 lanes, 8 x 16 outputs each
constexpr int RASTER = 8;     // row tiles per rasterisation group
static_assert(TN == 128, "the epilogues assume 128-column tiles");
// Resident blocks per SM the kernel is compiled for (build-time tunable): 2 caps registers at
// 255 per thread.
#ifndef LCE_SIMT_MIN_BLOCKS
#define LCE_SIMT_MIN_BLOCKS 2
#endif

struct SParams {
  int M, Ncols, K;
  int tiles_m, tiles_n;
  // element (m, k) of A is A[m * a_sm + k * a_sk]; (n, k) of B is B[n * b_sn + k * b_sk]; one of
  // the two strides of each operand is 1
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

// Shared-memory layout of a staged operand block: [TK][128] floats, element (k, m) at column
// m ^ swz(k).  The swizzle flips bit 4 of m for k = 4..7: a warp's transposed scalar stores of a
// K-major block (16 consecutive m at k and 16 at k + 4) then land in 32 distinct banks, while
// groups of 4 consecutive m stay contiguous for the float4 reads of the multiply.
__device__ __forceinline__ int swz(int k) { return ((k >> 2) & 1) << 4; }

// A thread's two fragments of a TK x 128 operand block, four consecutive elements each along the
// operand's contiguous dimension.  Fragment f covers u = t + 128 f:
//   K-major (stride 1 along k):  m = u / 2,  k = (u % 2) * 4       (fragment 1: m + 64)
//   MN-major (stride 1 along m): k = u / 32, m = (u % 32) * 4      (fragment 1: k + 4)
// One base pointer per operand (fragment 0 of the current k-block) advances by TK along k.
template <bool KMAJ>
struct Operand {
  const float* base;
  int64_t step;  // elements between consecutive k-blocks
  int off1;      // fragment 1 relative to fragment 0 (64 rows, or TK / 2 k-rows)
  int mn0, k0;   // fragment 0's m and k offsets within the block (tile-relative m added)
  unsigned ok;   // bit f: fragment f's m range lies inside the operand

  __device__ __forceinline__ void init(const float* X, int64_t s_mn, int64_t s_k, int tile_mn,
                                       int MN, int t) {
    mn0 = tile_mn + (KMAJ ? t / 2 : (t % 32) * 4);
    k0 = KMAJ ? (t % 2) * 4 : t / 32;
    base = X + static_cast<int64_t>(mn0) * s_mn + static_cast<int64_t>(k0) * s_k;
    off1 = KMAJ ? static_cast<int>(64 * s_mn) : static_cast<int>((TK / 2) * s_k);
    step = static_cast<int64_t>(TK) * s_k;
    ok = KMAJ ? ((mn0 < MN ? 1u : 0u) | (mn0 + 64 < MN ? 2u : 0u))
              : (mn0 + 3 < MN ? 3u : 0u);
  }

  // k-block kb (base already advanced to it); `kfull`: the whole block lies inside K.  Off the
  // fast path every element is checked on its own (ragged M, N or K edges).
  __device__ __forceinline__ void load(int kb, bool kfull, int MN, int K, float (&v)[2][4]) const {
#pragma unroll
    for (int f = 0; f < 2; ++f) {
      const float* p = base + (f ? off1 : 0);
      if (kfull && ((ok >> f) & 1u)) {
        const float4 q = *reinterpret_cast<const float4*>(p);  // 16-byte aligned: see simt_strip_gemm
        v[f][0] = q.x; v[f][1] = q.y; v[f][2] = q.z; v[f][3] = q.w;
      } else {
        const int mn = mn0 + ((KMAJ && f) ? 64 : 0);
        const int k = kb * TK + k0 + ((!KMAJ && f) ? TK / 2 : 0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool in = KMAJ ? (mn < MN && k + i < K) : (k < K && mn + i < MN);
          v[f][i] = in ? p[i] : 0.f;  // stride 1 along the contiguous dimension either way
        }
      }
    }
  }

  __device__ __forceinline__ void store(float (*S)[TM], const float (&v)[2][4], int t) const {
#pragma unroll
    for (int f = 0; f < 2; ++f) {
      if (KMAJ) {
        const int m = t / 2 + 64 * f, k = (t % 2) * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) S[k + i][m ^ swz(k + i)] = v[f][i];
      } else {
        const int k = t / 32 + (TK / 2) * f, m = (t % 32) * 4;
        *reinterpret_cast<float4*>(&S[k][m ^ swz(k)]) =
            make_float4(v[f][0], v[f][1], v[f][2], v[f][3]);
      }
    }
  }

};

// Grouped rasterisation: RASTER row tiles sweep the column tiles together (operand reuse in L2).
__device__ __forceinline__ void tile_of(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int per_group = RASTER * tiles_n;
  const int g = t / per_group;
  const int first = g * RASTER;
  const int gm = min(tiles_m - first, RASTER);
  const int r = t - g * per_group;
  tm = first + r % gm;
  tn = r / gm;
}

// One k step's fragments from staged block `buf`: a = rows arow + {0..3}, arow + 16 + {0..3};
// b = columns bcol + 32 q + {0..3}, q = 0..3, as pairs of adjacent columns (element (k, m) at
// column m ^ swz(k)).
__device__ __forceinline__ void fragments(const float (*As)[TM], const float (*Bs)[TN], int kk,
                                          int arow, int bcol, float (&a)[8], float2 (&b)[8]) {
  const int z = swz(kk);
  const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][arow ^ z]);
  const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][(arow + 16) ^ z]);
  a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
  a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = *reinterpret_cast<const float4*>(&Bs[kk][(bcol + 32 * q) ^ z]);
    b[2 * q] = make_float2(v.x, v.y);
    b[2 * q + 1] = make_float2(v.z, v.w);
  }
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, LCE_SIMT_MIN_BLOCKS) simt_strip_kernel(const SParams p) {
  __shared__ __align__(16) float As[2][TK][TM];
  __shared__ __align__(16) float Bs[2][TK][TN];

  int tm, tn;
  tile_of(blockIdx.x, p.tiles_m, p.tiles_n, tm, tn);
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int r = lane >> 3, c = lane & 7;  // the 8 lanes sharing r hold one row's 128 columns
  const int arow = warp * 32 + r * 4, bcol = c * 4;
  const int m0 = tm * TM, n0 = tn * TN;

  // acc2[i][p]: outputs (row i, columns 2p and 2p + 1) of the thread's 8 x 16, updated two at a
  // time by the packed fp32 FMA (each lane an ordinary round-to-nearest fp32 FMA)
  float2 acc2[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc2[i][j] = make_float2(0.f, 0.f);

  // operand majorness per mode: A = H (K-major) or G (K-major for dH, MN-major for dW);
  // B = W strip (K-major for the logits, MN-major for dH) or H (MN-major for dW)
  Operand<MODE != MODE_DW> oa;
  Operand<MODE == MODE_FWD_LSE || MODE == MODE_BWD_G> ob;
  oa.init(p.A, p.a_sm, p.a_sk, m0, p.M, t);
  ob.init(p.B, p.b_sn, p.b_sk, n0, p.Ncols, t);
  float va[2][4], vb[2][4];
  const int nkb = (p.K + TK - 1) / TK;
  oa.load(0, TK <= p.K, p.M, p.K, va);
  ob.load(0, TK <= p.K, p.Ncols, p.K, vb);
  oa.store(As[0], va, t);
  ob.store(Bs[0], vb, t);
  __syncthreads();
  for (int kb = 0; kb < nkb; ++kb) {
    const int cur = kb & 1;
    const bool more = kb + 1 < nkb;
    if (more) {  // next k-block into registers while this one is multiplied
      const bool kfull = (kb + 2) * TK <= p.K;
      oa.base += oa.step;
      ob.base += ob.step;
      oa.load(kb + 1, kfull, p.M, p.K, va);
      ob.load(kb + 1, kfull, p.Ncols, p.K, vb);
    }
    float a[2][8];
    float2 b[2][8];
    fragments(As[cur], Bs[cur], 0, arow, bcol, a[0], b[0]);
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      if (kk + 1 < TK)  // step kk + 1's reads in flight during step kk's FMAs
        fragments(As[cur], Bs[cur], kk + 1, arow, bcol, a[(kk + 1) & 1], b[(kk + 1) & 1]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 ai = make_float2(a[kk & 1][i], a[kk & 1][i]);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc2[i][j] = __ffma2_rn(ai, b[kk & 1][j], acc2[i][j]);
      }
    }
    if (more) {  // the other buffer was last read before the previous barrier
      oa.store(As[cur ^ 1], va, t);
      ob.store(Bs[cur ^ 1], vb, t);
    }
    __syncthreads();
  }

  // this thread's rows and columns (tile-local), and output (i, j) of its 8 x 16
  auto row_of = [&](int i) { return arow + (i >> 2) * 16 + (i & 3); };
  auto col_of = [&](int j) { return bcol + (j >> 2) * 32 + (j & 3); };
  float acc[8][16];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[i][2 * j] = acc2[i][j].x;
      acc[i][2 * j + 1] = acc2[i][j].y;
    }

  if (MODE == MODE_FWD_LSE) {
    // The 8 lanes sharing a row (c = 0..7) are consecutive: reduce over them by shuffles.
    const int ncols = min(TN, p.strip_cols - n0);  // >= 1
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = m0 + row_of(i);
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (col_of(j) < ncols) mx = fmaxf(mx, acc[i][j]);
#pragma unroll
      for (int o = 4; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sm = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (col_of(j) < ncols) sm += expf(acc[i][j] - mx);
#pragma unroll
      for (int o = 4; o >= 1; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      if (row < p.M) {
        if (c == 0) p.part[static_cast<size_t>(tn) * p.M + row] = make_float2(mx, sm);
        const int64_t y = p.labels[row];
        const int64_t rel = y - static_cast<int64_t>(p.col0 + n0);
        if (y != p.ignore_index && y >= 0 && y < p.V && rel >= 0 && rel < ncols) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (col_of(j) == rel) p.tgt[row] = acc[i][j];
        }
      }
    }
  } else if (MODE == MODE_BWD_G) {
    const float dl = *p.dloss;
    const float scale_valid = (p.reduction == 0) ? dl / static_cast<float>(*p.n_valid) : dl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = m0 + row_of(i);
      if (row >= p.M) continue;
      const int64_t y = p.labels[row];
      const bool ok = (y != p.ignore_index) && (y >= 0) && (y < p.V);
      if (!ok && y != p.ignore_index && p.first_strip && tn == 0 && c == 0)
        atomicOr(p.err, ERR_LABEL);
      const float l = ok ? p.lse[row] : 0.f;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float g[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int col = n0 + col_of(h * 4 + q);  // strip-local column, < ldg by construction
          g[q] = 0.f;
          if (ok && col < p.strip_cols) {
            g[q] = scale_valid * expf(acc[i][h * 4 + q] - l);
            if (static_cast<int64_t>(p.col0 + col) == y) g[q] -= scale_valid;
          }
        }
        *reinterpret_cast<float4*>(p.G + static_cast<size_t>(row) * p.ldg + n0 + col_of(h * 4)) =
            make_float4(g[0], g[1], g[2], g[3]);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = m0 + row_of(i);
      if (row >= p.c_rows) continue;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int col = n0 + col_of(h * 4);
        if (col >= p.c_cols) continue;  // c_cols % 4 == 0: a group is all in or all out
        float4* cp = reinterpret_cast<float4*>(p.C + static_cast<size_t>(row) * p.ldc + col);
        float4 v = make_float4(acc[i][h * 4], acc[i][h * 4 + 1], acc[i][h * 4 + 2],
                               acc[i][h * 4 + 3]);
        if (p.accumulate) {
          const float4 o = *cp;
          v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
        }
        *cp = v;
      }
    }
  }
}

}  // namespace

// Alignment of the float4 accesses: every operand base is 16-byte aligned (caller pointers, the
// W strip at col0 * d with col0 % 128 == 0, workspace offsets), every row stride is a multiple of
// 4 elements (d % 4 == 0, ldg % 128 == 0), and float4 offsets along the contiguous dimension are
// multiples of 4.
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
  // 32-bit index arithmetic in the kernel: fragment offsets of 64 rows (or 4 k-rows) of the
  // largest stride, and tile-relative indices up to M + 255, N + 255, K + 31
  const int64_t max_stride = std::max(std::max(p.a_sm, p.a_sk), std::max(p.b_sn, p.b_sk));
  const int64_t kIntMax = 0x7fffffffLL;
  if (64 * max_stride > kIntMax || p.M > kIntMax - 256 || p.Ncols > kIntMax - 256 ||
      p.K > kIntMax - 64) {
    set_error_detail("fp32 strip GEMM: shape beyond the engine's 32-bit indexing (M %d, N %d, K %d,"
                     " stride %lld)", p.M, p.Ncols, p.K, static_cast<long long>(max_stride));
    return cudaErrorInvalidValue;
  }
  p.tiles_m = (p.M + TM - 1) / TM;
  p.tiles_n = (p.Ncols + TN - 1) / TN;
  if (static_cast<int64_t>(p.tiles_m) * p.tiles_n > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.strip_cols = s.strip_cols; p.col0 = s.col0;
  p.part = s.part; p.tgt = s.tgt;
  p.labels = s.labels; p.V = s.V; p.ignore_index = s.ignore_index;
  p.lse = s.lse; p.dloss = s.dloss; p.n_valid = s.n_valid; p.reduction = s.reduction;
  p.G = static_cast<float*>(s.G); p.ldg = s.ldg;
  p.C = s.C; p.ldc = s.ldc; p.accumulate = s.accumulate; p.c_rows = s.c_rows; p.c_cols = s.c_cols;
  p.err = s.err; p.first_strip = s.first_strip;
  const unsigned grid = static_cast<unsigned>(p.tiles_m * p.tiles_n);
  switch (s.mode) {
    case MODE_FWD_LSE: simt_strip_kernel<MODE_FWD_LSE><<<grid, THREADS, 0, stream>>>(p); break;
    case MODE_BWD_G: simt_strip_kernel<MODE_BWD_G><<<grid, THREADS, 0, stream>>>(p); break;
    case MODE_DH: simt_strip_kernel<MODE_DH><<<grid, THREADS, 0, stream>>>(p); break;
    default: simt_strip_kernel<MODE_DW><<<grid, THREADS, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace lce
