// Per-token state reductions of the forward pass, and the tf32 operand splits.
//
// combine:  folds the per-(tile, row) (max, sum-exp) partials of one vocabulary strip, in tile
//           order, into the running per-token state (m, s):
//             (m, s) (+) (m', s') = (M, s e^(m - M) + s' e^(m' - M)),  M = max(m, m')
//           ("Flattening Every Memory Peak in Long-Context Mixture-of-Experts Training",
//           section 3.2: each strip is folded into a running per-token state and released).
//           Eight warps share the tiles of 64 tokens; coalesced over tokens.
// finalize: lse_i = m_i + log s_i for every row; per-token loss lse_i - t_i on valid rows; the
//           sum over rows in a fixed order in fp64 (one block, fixed per-thread strides and a
//           fixed tree), n_valid, and the label-range check.
// split:    fp32 x -> tf32 parts hi = rna(x), lo = rna(x - hi) for the three-product tensor-core
//           path (x = hi + lo + r with |r| about 2^-22 |x|); plain, or transposed through 64 x 64
//           shared-memory tiles for the operands the tf32 MMAs need K-major.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "lce_internal.h"
#include "ptx.cuh"

namespace lce {
namespace {

using ptx::round_tf32;

__device__ __forceinline__ float2 fold(float2 a, float2 b) {
  const float M = fmaxf(a.x, b.x);
  if (M == -INFINITY) return make_float2(-INFINITY, 0.f);
  return make_float2(M, a.y * expf(a.x - M) + b.y * expf(b.x - M));
}

// One block folds 64 consecutive tokens over one chunk of the tiles: lane j of every warp holds
// tokens 2j and 2j + 1 (one 16-byte load per tile when N is even), warp w takes the chunk's tiles
// w, w + 8, w + 16, ... and issues the loads of COMBINE_BATCH tiles before folding them (bytes in
// flight for HBM), folding in tile order.  Then lane j of warp 0 folds the eight warp states in
// warp order.  With one chunk the result goes into the running state; with several (few tokens,
// so few blocks), each block writes its chunk's state over the chunk's first partial slot and
// combine_chunks_kernel folds the chunks in order.  Every order is fixed by N and the tile count,
// so the result is deterministic.
constexpr int COMBINE_WARPS = 8;
constexpr int COMBINE_TOKENS = 64;
constexpr int COMBINE_BATCH = 8;

__global__ void __launch_bounds__(COMBINE_WARPS * 32)
    combine_kernel(float2* __restrict__ part, int tiles, int chunk_tiles, int chunks, int64_t N,
                   float2* __restrict__ run, int first) {
  __shared__ float4 st_w[COMBINE_WARPS][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * COMBINE_TOKENS + 2 * lane;
  const int t_begin = static_cast<int>(blockIdx.y) * chunk_tiles;
  const int t_end = min(tiles, t_begin + chunk_tiles);
  const bool has0 = i0 < N, has1 = i0 + 1 < N;
  const bool vec = has1 && (N % 2 == 0);  // part + t * N + i0 is then 16-byte aligned
  const float2 none = make_float2(-INFINITY, 0.f);
  float2 a0 = none, a1 = none;
  auto load2 = [&](int t, float2& x0, float2& x1) {
    const float2* q = part + static_cast<size_t>(t) * N + i0;
    if (vec) {
      const float4 v = *reinterpret_cast<const float4*>(q);
      x0 = make_float2(v.x, v.y);
      x1 = make_float2(v.z, v.w);
    } else {
      x0 = q[0];
      x1 = has1 ? q[1] : none;
    }
  };
  if (has0) {
    int t = t_begin + warp;
    for (; t + (COMBINE_BATCH - 1) * COMBINE_WARPS < t_end; t += COMBINE_BATCH * COMBINE_WARPS) {
      float2 x[COMBINE_BATCH][2];
#pragma unroll
      for (int u = 0; u < COMBINE_BATCH; ++u) load2(t + u * COMBINE_WARPS, x[u][0], x[u][1]);
#pragma unroll
      for (int u = 0; u < COMBINE_BATCH; ++u) {
        a0 = fold(a0, x[u][0]);
        a1 = fold(a1, x[u][1]);
      }
    }
    for (; t < t_end; t += COMBINE_WARPS) {
      float2 x0, x1;
      load2(t, x0, x1);
      a0 = fold(a0, x0);
      a1 = fold(a1, x1);
    }
  }
  st_w[warp][lane] = make_float4(a0.x, a0.y, a1.x, a1.y);
  __syncthreads();  // every read of this block's partials is done before slot t_begin is reused
  if (warp == 0 && has0) {
    const bool direct = (chunks == 1);
    float2 r0 = (first || !direct) ? none : run[i0];
    float2 r1 = (first || !direct || !has1) ? none : run[i0 + 1];
#pragma unroll
    for (int w = 0; w < COMBINE_WARPS; ++w) {
      const float4 v = st_w[w][lane];
      r0 = fold(r0, make_float2(v.x, v.y));
      r1 = fold(r1, make_float2(v.z, v.w));
    }
    float2* out = direct ? run + i0 : part + static_cast<size_t>(t_begin) * N + i0;
    out[0] = r0;
    if (has1) out[1] = r1;
  }
}

// Second pass of a chunked combine: token i folds its chunk states in chunk order.
__global__ void combine_chunks_kernel(const float2* __restrict__ part, int chunk_tiles, int chunks,
                                      int64_t N, float2* __restrict__ run, int first) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  float2 acc = first ? make_float2(-INFINITY, 0.f) : run[i];
  for (int c = 0; c < chunks; ++c)
    acc = fold(acc, part[static_cast<size_t>(c) * chunk_tiles * N + i]);
  run[i] = acc;
}

constexpr int FIN_THREADS = 1024;

__global__ void __launch_bounds__(FIN_THREADS)
    finalize_kernel(const float2* __restrict__ run, const float* __restrict__ tgt,
                    const int64_t* __restrict__ labels, int64_t N, int64_t V, int64_t ignore_index,
                    int reduction, float* loss, float* lse, int64_t* n_valid, unsigned* err) {
  __shared__ double ssum[FIN_THREADS];
  __shared__ long long scnt[FIN_THREADS];
  __shared__ int sbad;
  if (threadIdx.x == 0) sbad = 0;
  __syncthreads();
  double acc = 0.0;
  long long cnt = 0;
  int bad = 0;
  for (int64_t i = threadIdx.x; i < N; i += FIN_THREADS) {
    const float2 st = run[i];
    const float l = st.x + logf(st.y);
    lse[i] = l;
    const int64_t y = labels[i];
    const bool in_range = (y >= 0) && (y < V);
    if (y != ignore_index && in_range) {
      acc += static_cast<double>(l) - static_cast<double>(tgt[i]);
      ++cnt;
    } else if (y != ignore_index) {
      bad = 1;
    }
  }
  ssum[threadIdx.x] = acc;
  scnt[threadIdx.x] = cnt;
  if (bad) sbad = 1;
  __syncthreads();
  for (int w = FIN_THREADS / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      ssum[threadIdx.x] += ssum[threadIdx.x + w];
      scnt[threadIdx.x] += scnt[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double total = ssum[0];
    const long long nv = scnt[0];
    if (reduction == 0)
      *loss = nv > 0 ? static_cast<float>(total / static_cast<double>(nv)) : nanf("");
    else
      *loss = static_cast<float>(total);
    *n_valid = nv;
    if (sbad) atomicOr(err, ERR_LABEL);
  }
}

// Elementwise split, four values per thread, grid-stride.
__global__ void split_tf32_kernel(const float4* __restrict__ x, float4* __restrict__ hi,
                                  float4* __restrict__ lo, size_t n4) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 v = x[i];
    float4 h, l;
    h.x = round_tf32(v.x); l.x = round_tf32(v.x - h.x);
    h.y = round_tf32(v.y); l.y = round_tf32(v.y - h.y);
    h.z = round_tf32(v.z); l.z = round_tf32(v.z - h.z);
    h.w = round_tf32(v.w); l.w = round_tf32(v.w - h.w);
    hi[i] = h;
    lo[i] = l;
  }
}

// Transposing split: x [rows x cols] -> hi / lo [cols x ld_out], one 64 x 64 tile at a time
// (grid-stride over tiles) through shared memory padded by one word against bank conflicts: each
// thread issues its 16 loads of a tile before the barrier, and both the reads of x and the writes
// of hi / lo are coalesced 128-byte rows.
constexpr int TT = 64;

__global__ void __launch_bounds__(32 * 8)
    split_tf32_t_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld_out,
                        float* __restrict__ hi, float* __restrict__ lo) {
  __shared__ float t[TT][TT + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  const int64_t tiles_c = (cols + TT - 1) / TT;
  const int64_t tiles = tiles_c * ((rows + TT - 1) / TT);
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t r0 = (tile / tiles_c) * TT, c0 = (tile % tiles_c) * TT;
#pragma unroll
    for (int i = 0; i < TT / 8; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t r = r0 + ty + 8 * i, c = c0 + tx + 32 * h;
        t[ty + 8 * i][tx + 32 * h] = (r < rows && c < cols) ? x[r * cols + c] : 0.f;
      }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < TT / 8; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t c = c0 + ty + 8 * i, r = r0 + tx + 32 * h;
        if (c < cols && r < rows) {
          const float v = t[tx + 32 * h][ty + 8 * i];
          const float hv = round_tf32(v);
          hi[c * ld_out + r] = hv;
          lo[c * ld_out + r] = round_tf32(v - hv);
        }
      }
    __syncthreads();
  }
}

// Grid-stride kernels run at most a few waves of blocks over the 152 SMs.
constexpr int64_t kSplitMaxBlocks = 152 * 16;

}  // namespace

cudaError_t launch_split_tf32(const float* x, float* hi, float* lo, size_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  if (n % 4 != 0) return cudaErrorInvalidValue;  // whole rows of d % 4 == 0 elements
  const size_t n4 = n / 4;
  const int threads = 256;
  const int64_t need = static_cast<int64_t>((n4 + threads - 1) / threads);
  const int64_t blocks = need < kSplitMaxBlocks ? need : kSplitMaxBlocks;
  split_tf32_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      reinterpret_cast<const float4*>(x), reinterpret_cast<float4*>(hi),
      reinterpret_cast<float4*>(lo), n4);
  return cudaGetLastError();
}

cudaError_t launch_split_tf32_t(const float* x, int64_t rows, int64_t cols, int64_t ld_out,
                                float* hi, float* lo, cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (ld_out < rows) return cudaErrorInvalidValue;
  const int64_t tiles = ((rows + TT - 1) / TT) * ((cols + TT - 1) / TT);
  const int64_t blocks = tiles < kSplitMaxBlocks ? tiles : kSplitMaxBlocks;
  split_tf32_t_kernel<<<static_cast<unsigned>(blocks), dim3(32, 8), 0, stream>>>(x, rows, cols,
                                                                                ld_out, hi, lo);
  return cudaGetLastError();
}

cudaError_t launch_combine(float2* part, int tiles, int64_t N, float2* run, int first,
                           cudaStream_t stream) {
  if (N == 0 || tiles < 1) return cudaSuccess;
  // Fewer token blocks than the 152 SMs of a GB300: the tiles are split into chunks (at least 8
  // tiles each, so every warp has one) until there are about two blocks per SM.  The chunking
  // depends on N and the tile count only.
  const int64_t token_blocks = (N + COMBINE_TOKENS - 1) / COMBINE_TOKENS;
  int64_t want = (token_blocks < 152) ? (2 * 152 + token_blocks - 1) / token_blocks : 1;
  want = std::min<int64_t>(want, std::max(1, tiles / 8));
  const int chunk_tiles = static_cast<int>((tiles + want - 1) / want);
  const int chunks = (tiles + chunk_tiles - 1) / chunk_tiles;
  combine_kernel<<<dim3(static_cast<unsigned>(token_blocks), static_cast<unsigned>(chunks)),
                   COMBINE_WARPS * 32, 0, stream>>>(part, tiles, chunk_tiles, chunks, N, run, first);
  if (chunks > 1) {
    ++g_extra_kernels;
    const int threads = 256;
    combine_chunks_kernel<<<static_cast<unsigned>((N + threads - 1) / threads), threads, 0,
                            stream>>>(part, chunk_tiles, chunks, N, run, first);
  }
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float2* run, const float* tgt, const int64_t* labels, int64_t N,
                            int64_t V, int64_t ignore_index, int reduction, float* loss, float* lse,
                            int64_t* n_valid, unsigned* err, cudaStream_t stream) {
  finalize_kernel<<<1, FIN_THREADS, 0, stream>>>(run, tgt, labels, N, V, ignore_index, reduction,
                                                 loss, lse, n_valid, err);
  return cudaGetLastError();
}

}  // namespace lce
