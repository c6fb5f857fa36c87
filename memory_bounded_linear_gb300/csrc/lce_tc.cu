// Tensor-core strip GEMM engine on sm_103a (tcgen05 + TMEM + TMA), for bf16 operands and for
// fp32 operands split into tf32 hi / lo parts (three tf32 products per fp32 product).
//
// One persistent, warp-specialised kernel.  A launch carries up to three GEMM jobs, each with its
// own epilogue mode, operands and output; its tiles are scheduled together:
//   warp 0      TMA producer: streams A and B k-blocks (one 128-byte swizzle span of K: 64 bf16
//               or 32 fp32 per part) into a shared-memory ring; it also hands out the tiles
//               (dynamic scheduler);
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and one elected
//               lane issues tcgen05.mma into the accumulator of the tile;
//   warps 2..5  epilogue: each thread owns one accumulator row (TMEM lane) and reads its 256
//               columns 32 at a time with tcgen05.ld, so every per-row reduction of the tile
//               (max, sum of exp, target gather) is thread-local -- no shuffles are needed.
// While the epilogue drains one accumulator the MMA warp fills the other.
//
// GEMM view: C[M x Ncols] = A[M x K] B[Ncols x K]^T.  Operand layouts per mode:
//   FWD_LSE, BWD_G  A = H   [N x d] K-major    B = W strip [w x d] K-major
//   DH              A = G_s [N x w] K-major    B = W strip [w x d] MN-major (d contiguous)
//   DW              A = G_s^T      MN-major    B = H [N x d]       MN-major
// For tf32 parts every operand is K-major: dH's B is the transposed strip W_s^T [d x w], dW's A
// the transposed gradient G_s^T [w x N] (written by the gradient epilogue beside G_s) and its B
// the transposed H^T [d x N].
// TMA zero-fills every box element outside the tensor, so ragged M, N and K edges contribute 0
// to the products; the epilogues mask the columns beyond the strip / vocabulary, and TMA stores
// clip the output boxes at the edges of their tensors.
//
// "Flattening Every Memory Peak in Long-Context Mixture-of-Experts Training", section 3.2 and
// appendix C: each logit strip is folded into a running per-token state and released; backward
// recomputes the strip and its gradient.  Here a strip's logits only ever live in TMEM.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <type_traits>

#include "lce_internal.h"
#include "ptx.cuh"

namespace lce {
namespace {

constexpr int BM = 128;     // accumulator rows held by one CTA (TMEM lanes)
constexpr int BN = TC_BN;  // 256 columns per tile
// bf16 MN-major operands: 64(MN) x 64(K) boxes of 8 KB
constexpr int MN_BOX_ELEMS = 64;
constexpr int MN_BOX_BYTES = 64 * 64 * 2;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int MAX_STAGES = 6;
constexpr int CTL_BYTES = 256;
// Epilogue output staging: per epilogue warp two 4 KB buffers, each a 32-row x 128-byte box
// (32 fp32 or 64 bf16 columns) in the 128-byte-swizzled layout a TMA store reads.
constexpr int STAGE_BUF_BYTES = 32 * 128;
constexpr int STAGING_BYTES = 4 * 2 * STAGE_BUF_BYTES;
constexpr float LOG2E = 1.4426950408889634f;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // a wait longer than 2 s is treated as a hang
constexpr int MAX_JOBS = 3;

// Pair tiles per rasterisation group (build-time tunable): more tiles per group re-read the
// column operand less often but keep a larger row panel live in L2.
#ifndef LCE_PAIR_RASTER_GROUP
#define LCE_PAIR_RASTER_GROUP 8
#endif

// Tile geometry.  Single: one CTA computes a 128 x 256 tile and holds all of B.  Pair: the two
// CTAs of a cluster compute a 256 x 256 tile with cta_group::2 MMAs; each holds its 128 rows of
// A and half (128 columns) of B.
// Operand formats.  OP_BF16: one bf16 part per operand, kind::f16 MMAs (K = 16); a bf16 stage
// is 32 KB in a pair, six stages.  OP_TF32X3: two tf32 parts (hi, lo) per operand, kind::tf32
// MMAs (K = 8), three MMAs per k-slice (hi*hi' + hi*lo' + lo*hi') into one fp32 accumulator; a
// stage holds both parts, so there are half as many.  A stage always covers one 128-byte
// swizzle span of K per row and part, and four MMA k-slices.
template <bool PAIR, int OP>
struct Cfg {
  static constexpr bool X3 = (OP == OP_TF32X3);
  static constexpr int ELEM = X3 ? 4 : 2;
  static constexpr int BK = 128 / ELEM;    // K elements per stage
  static constexpr int KI = X3 ? 8 : 16;   // K of one MMA instruction
  static constexpr int PARTS = X3 ? 2 : 1;
  static constexpr int TILE_M = PAIR ? 2 * BM : BM;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // tile columns whose B rows this CTA loads
  static constexpr int A_BYTES = BM * 128;           // one part of the A block
  static constexpr int B_BYTES = B_ROWS * 128;       // one part of the B block
  static constexpr int PART_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGE_BYTES = PARTS * PART_BYTES;
  static constexpr int STAGES = (PAIR ? 6 : 4) / PARTS;  // 192 KB of stages either way
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + CTL_BYTES;
  static_assert(STAGES <= MAX_STAGES, "control block sized for MAX_STAGES");
  static_assert(BK / KI == 4, "four MMA k-slices per stage");
};

// Row tiles per rasterisation group, by tile variant.
template <bool PAIR>
constexpr int RASTER_GROUP = PAIR ? LCE_PAIR_RASTER_GROUP : 16;

// Tiles handed out by the dynamic scheduler wait in a small ring until every role has read them.
constexpr int TQ = 4;

struct Ctl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t tq_full[TQ];
  uint64_t tq_empty[TQ];
  int tq[TQ];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Ctl) <= CTL_BYTES, "control block too large");

// One GEMM of a launch.
struct Job {
  int mode;                           // MODE_*
  int tiles_m, tiles_n, num_tiles, nkb;
  int b_off;       // FWD/BWD_G: W row of the strip start; DH: W row (K coordinate) of the strip
  int strip_cols;  // FWD/BWD_G: columns of the strip
  int col0;        // FWD/BWD_G: first vocabulary column of the strip
  int c_cols;      // DH/DW: columns of C
  int accumulate;  // DH: add into C instead of storing
  int first_strip; // BWD_G: the strip that reports bad labels
};

struct KParams {
  Job job[MAX_JOBS];
  int njobs, total_tiles;
  int64_t N, V, ignore_index;
  float2* part;             // FWD: [tiles_n][N] per-(tile, row) (max, sum-exp)
  float* tgt;               // FWD: [N] target logit
  const int64_t* labels;
  const float* lse;         // BWD_G
  const float* dloss;       // BWD_G (null when no job needs it)
  const int64_t* n_valid;   // BWD_G
  int reduction;
  unsigned* err;
  unsigned* sched;  // [0] next tile ticket, [1] units finished; both zero between launches
  int inject_stall;  // test hook (lce_test_inject_stall): withhold the first k-block
};

// Per job: A and B operand maps, one per operand part ([0] only for bf16), and the maps of the
// epilogue's TMA stores: C in [0]; the bf16 gradient strip in [0]; the tf32 gradient strip's
// hi and lo parts in [0] and [1], and their transposes in [2] and [3].
struct TcMaps {
  CUtensorMap a[MAX_JOBS][2];
  CUtensorMap b[MAX_JOBS][2];
  CUtensorMap c[MAX_JOBS][4];
};

// Suspend-time hint of every barrier wait (ns): a waiting thread sleeps in the try_wait until the
// phase completes, up to this long, instead of returning early and polling again.  Measured 1.0-
// 1.5% faster steps than the instruction's default, with or without the power cap.
#ifndef LCE_WAIT_HINT_NS
#define LCE_WAIT_HINT_NS 20000
#endif

// Bounded wait on an mbarrier phase.  Gives up after WAIT_LIMIT_NS (or at once when another role
// already gave up), raising the CTA's abort flag and the workspace timeout bit.
template <bool CLUSTER_ACQUIRE = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned* err) {
  auto try_once = [&]() {
    return CLUSTER_ACQUIRE ? ptx::mbar_try_wait_cluster(bar, parity, LCE_WAIT_HINT_NS)
                           : ptx::mbar_try_wait(bar, parity, LCE_WAIT_HINT_NS);
  };
  if (try_once()) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (*abort_flag) return false;
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (try_once()) return true;
    if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      atomicOr(err, ERR_TIMEOUT);
      return false;
    }
  }
}

// Wait on a barrier regardless of the abort flag, for at most `limit_ns` (used while draining).
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity, LCE_WAIT_HINT_NS))
    if (ptx::globaltimer() - t0 > limit_ns) return;
}

// Grouped rasterisation: `group` row tiles sweep the column tiles together, so the tiles
// resident at one time share a few A row-blocks and B column-blocks through L2.
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group, int& tm,
                                            int& tn) {
  const int per_group = group * tiles_n;
  const int g = tile / per_group;
  const int first_m = g * group;
  const int gm = min(tiles_m - first_m, group);
  const int r = tile - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

// A scheduler ticket resolved to its job and to the job's row / column tile.
struct TilePos {
  int job, tm, tn;
};
template <bool PAIR>
__device__ __forceinline__ TilePos locate(const KParams& p, int t) {
  int j = 0;
  while (j + 1 < p.njobs && t >= p.job[j].num_tiles) {
    t -= p.job[j].num_tiles;
    ++j;
  }
  TilePos r;
  r.job = j;
  tile_coords(t, p.job[j].tiles_m, p.job[j].tiles_n, RASTER_GROUP<PAIR>, r.tm, r.tn);
  return r;
}

// Dynamic tile scheduler.  The producer thread of the (first) CTA takes tickets from a global
// counter -- tiles come out in job and raster order, so the tiles in flight at any moment stay
// together however unevenly the SMs progress, and operands keep being shared through L2 -- and
// posts each ticket into the ring `tq` of both CTAs of a pair.  Every other role reads the
// tickets from its own CTA's ring and hands the slot back.  -1 ends the sequence.  The producer
// takes the ticket of its next tile from the counter as soon as it has posted the current one, so
// the atomic's round trip overlaps the current tile's loads instead of opening a gap in the
// operand stream at every tile boundary.
template <bool PAIR>
struct TileQueue {
  Ctl* ctl;
  volatile int* abort_flag;
  unsigned* err;
  int slot;
  uint32_t ph;
  // a reader in the second CTA of a pair: it hands slots back to the first CTA's barrier with a
  // cluster-scope release; readers in the first CTA hand back locally with a CTA-scope release,
  // which does not make them wait the way the cluster-scope one does (measured: the MMA thread
  // spent 5-14% of its time in a cluster-scope hand-back)
  bool remote;

  __device__ __forceinline__ void advance() {
    if (++slot == TQ) { slot = 0; ph ^= 1u; }
  }

  // Scheduler: posts `ticket` (taken from the counter sched[0] beforehand) to both CTAs, or -1
  // when it is past the last tile.  Returns what was posted (-1 also after a timeout); the last
  // unit to receive -1 clears the counters for the next launch.
  __device__ __forceinline__ int post(unsigned ticket, unsigned* sched, int num_tiles, int units) {
    const uint32_t empty = ptx::smem_addr(&ctl->tq_empty[slot]);
    if (!wait_bar<PAIR>(empty, ph ^ 1u, abort_flag, err)) return -1;
    const int t = (ticket < static_cast<unsigned>(num_tiles)) ? static_cast<int>(ticket) : -1;
    ctl->tq[slot] = t;
    const uint32_t full = ptx::smem_addr(&ctl->tq_full[slot]);
    if (PAIR) {
      ptx::st_shared_cluster(ptx::mapa_shared(ptx::smem_addr(&ctl->tq[slot]), 1), t);
      ptx::mbar_arrive_cluster(ptx::mapa_shared(full, 1));
    }
    ptx::mbar_arrive(full);
    advance();
    if (t < 0 && atomicAdd(&sched[1], 1u) == static_cast<unsigned>(units - 1)) {
      atomicExch(&sched[0], 0u);
      atomicExch(&sched[1], 0u);
    }
    return t;
  }

  // Reader: the next ticket of this CTA's ring.  `mask` names the lanes of the calling warp that
  // read it together; the slot is handed back (once per warp) after all of them have.
  __device__ __forceinline__ int take(unsigned mask) {
    const uint32_t full = ptx::smem_addr(&ctl->tq_full[slot]);
    int t = -1;
    if (wait_bar<PAIR>(full, ph, abort_flag, err)) t = ctl->tq[slot];
    __syncwarp(mask);
    if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(mask) - 1)) {
      const uint32_t empty = ptx::smem_addr(&ctl->tq_empty[slot]);
      if (remote) ptx::mbar_arrive_cluster(ptx::mapa_shared(empty, 0));
      else ptx::mbar_arrive(empty);
    }
    advance();
    return t;
  }
};

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_base, int k) {
  // K-major, 128B swizzle: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart; the k-th
  // MMA slice (16 bf16 or 8 tf32 elements) starts 32 bytes further into the row.
  return ptx::sw128_desc(tile_base + k * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile_base, int k16) {
  // bf16 MN-major, 128B swizzle: each 64-wide MN box holds 64 rows (one per k) of 128 bytes;
  // boxes are MN_BOX_BYTES apart (leading byte offset), groups of 8 k-rows 1024 bytes apart
  // (stride byte offset); the k-th 16-row slice starts 16 * 128 bytes further.
  return ptx::sw128_desc(tile_base + k16 * 16 * 128, MN_BOX_BYTES, 1024);
}

// Operand majorness per mode.  bf16: dW's A (G, contracted over tokens) and the B operands of dH
// (W, contracted over the vocabulary) and of dW (H, over tokens) are read MN-major straight from
// their row-major arrays.  tf32: the kind::tf32 MMAs are given K-major operands only (with an
// MN-major tf32 operand the accumulator stayed zero on sm_103a), so those operands come from
// transposed copies.
template <int MODE, int OP>
__host__ __device__ constexpr bool a_mn_major() {
  return MODE == MODE_DW && OP == OP_BF16;
}
template <int MODE, int OP>
__host__ __device__ constexpr bool b_mn_major() {
  return (MODE == MODE_DH || MODE == MODE_DW) && OP == OP_BF16;
}

// The kernel is compiled per set of modes a launch carries (a bit mask of MODE_*): the forward;
// the gradient; dW and dH; and all three backward modes (the launches that overlap dW and dH of
// one strip with the next strip's gradient).  Keeping the code of each kernel small matters: a
// kernel carrying all four epilogues ran 13% slower, and the dW + dH launches of the kernel
// carrying all three backward modes ran slower than they do alone.
constexpr int MODES_FWD = 1 << MODE_FWD_LSE;
constexpr int MODES_G = 1 << MODE_BWD_G;
constexpr int MODES_DHDW = (1 << MODE_DH) | (1 << MODE_DW);
constexpr int MODES_BWD = MODES_G | MODES_DHDW;
template <int MODES>
__host__ __device__ __forceinline__ constexpr bool has_mode(int m) {
  return ((MODES >> m) & 1) != 0;
}
// The job's mode as the compiler sees it: a constant when the kernel serves a single mode.
template <int MODES>
__device__ __forceinline__ int mode_of(const Job& jb) {
  if constexpr (MODES == MODES_FWD) return MODE_FWD_LSE;
  else if constexpr (MODES == MODES_G) return MODE_BWD_G;
  else return jb.mode;
}

// Calls f(integral_constant<int, mode>) for the job's mode, among the modes the kernel serves, so
// that the per-tile loops below are compiled once per mode with their operand layouts fixed.
template <int MODES, typename F>
__device__ __forceinline__ void dispatch_mode(int mode, F&& f) {
  if constexpr (has_mode<MODES>(MODE_FWD_LSE))
    if (mode == MODE_FWD_LSE) { f(std::integral_constant<int, MODE_FWD_LSE>{}); return; }
  if constexpr (has_mode<MODES>(MODE_BWD_G))
    if (mode == MODE_BWD_G) { f(std::integral_constant<int, MODE_BWD_G>{}); return; }
  if constexpr (has_mode<MODES>(MODE_DH))
    if (mode == MODE_DH) { f(std::integral_constant<int, MODE_DH>{}); return; }
  if constexpr (has_mode<MODES>(MODE_DW))
    if (mode == MODE_DW) { f(std::integral_constant<int, MODE_DW>{}); return; }
}

// Position in a shared-memory ring (stage index and phase parity).
struct Ring {
  int stage;
  uint32_t ph;
};

// Producer side of one tile: its k-blocks of A and B (every operand part) into the stage ring.
// False when a wait gave up.  `withhold_first` is the timeout-path test hook.  The job's fields
// come in as scalars, read once per tile: this one thread's time per k-block paces the operand
// stream, and the TMA instructions' memory clobbers would make it re-read fields of the job in
// every k-block.
template <int MODE, bool PAIR, int OP>
__device__ __forceinline__ bool produce_tile(int nkb, int b_off, const CUtensorMap* mA, const CUtensorMap* mB, int m0,
                                             int n0, uint32_t base, Ctl* ctl, Ring& r,
                                             volatile int* abort_flag, unsigned* err,
                                             uint32_t rank, bool withhold_first) {
  using Cf = Cfg<PAIR, OP>;
  constexpr bool A_MN = a_mn_major<MODE, OP>();
  constexpr bool B_MN = b_mn_major<MODE, OP>();
  for (int kb = 0; kb < nkb; ++kb) {
    const uint32_t empty = ptx::smem_addr(&ctl->empty[r.stage]);
    const uint32_t full_local = ptx::smem_addr(&ctl->full[r.stage]);
    if (!wait_bar(empty, r.ph ^ 1u, abort_flag, err)) return false;
    const bool withhold = withhold_first && kb == 0 && r.stage == 0 && r.ph == 0;
    if (!withhold) {
      // In a pair every stage's bytes (of both CTAs) are counted on the issuer's barrier.
      const uint32_t full = PAIR ? ptx::mapa_shared(full_local, 0) : full_local;
      if (rank == 0) ptx::mbar_arrive_expect_tx(full_local, (PAIR ? 2 : 1) * Cf::STAGE_BYTES);
      auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y) {
        if (PAIR) ptx::tma_load_2d_pair(dst, m, x, y, full);
        else ptx::tma_load_2d(dst, m, x, y, full);
      };
#pragma unroll
      for (int part = 0; part < Cf::PARTS; ++part) {
        const uint32_t sa = base + r.stage * Cf::STAGE_BYTES + part * Cf::PART_BYTES;
        const uint32_t sb = sa + Cf::A_BYTES;
        if (A_MN) {
#pragma unroll
          for (int c = 0; c < BM / MN_BOX_ELEMS; ++c)
            load(sa + c * MN_BOX_BYTES, &mA[part], m0 + c * MN_BOX_ELEMS, kb * Cf::BK);
        } else {
          load(sa, &mA[part], kb * Cf::BK, m0);
        }
        if (B_MN) {
          const int krow = (MODE == MODE_DH ? b_off : 0) + kb * Cf::BK;
#pragma unroll
          for (int c = 0; c < Cf::B_ROWS / MN_BOX_ELEMS; ++c)
            load(sb + c * MN_BOX_BYTES, &mB[part], n0 + c * MN_BOX_ELEMS, krow);
        } else {
          load(sb, &mB[part], kb * Cf::BK, b_off + n0);
        }
      }
    }  // else (test hook): no bytes, no arrival -- the MMA issuer's wait on this stage runs out
    if (++r.stage == Cf::STAGES) { r.stage = 0; r.ph ^= 1u; }
  }
  return true;
}

// MMA side of one tile: nkb k-blocks of 4 MMA k-slices (K = 16 bf16, or K = 8 with three tf32
// products) into the accumulator at d_tmem.
template <int MODE, bool PAIR, int OP>
__device__ __forceinline__ bool mma_tile(int nkb, uint32_t d_tmem, uint32_t base, Ctl* ctl, Ring& r,
                                         volatile int* abort_flag, unsigned* err) {
  using Cf = Cfg<PAIR, OP>;
  constexpr bool A_MN = a_mn_major<MODE, OP>();
  constexpr bool B_MN = b_mn_major<MODE, OP>();
  constexpr uint32_t IDESC = Cf::X3 ? ptx::idesc_tf32_f32(Cf::TILE_M, BN, false, false)
                                    : ptx::idesc_bf16_f32(Cf::TILE_M, BN, A_MN, B_MN);
  auto mma = [&](uint64_t ad, uint64_t bd, uint32_t accumulate) {
    if constexpr (Cf::X3) {
      if (PAIR) ptx::tc_mma_tf32_pair(d_tmem, ad, bd, IDESC, accumulate);
      else ptx::tc_mma_tf32(d_tmem, ad, bd, IDESC, accumulate);
    } else {
      if (PAIR) ptx::tc_mma_f16_pair(d_tmem, ad, bd, IDESC, accumulate);
      else ptx::tc_mma_f16(d_tmem, ad, bd, IDESC, accumulate);
    }
  };
  for (int kb = 0; kb < nkb; ++kb) {
    if (!wait_bar(ptx::smem_addr(&ctl->full[r.stage]), r.ph, abort_flag, err)) return false;
    ptx::tc_fence_after();
    const uint32_t s0 = base + r.stage * Cf::STAGE_BYTES;
#pragma unroll
    for (int k = 0; k < Cf::BK / Cf::KI; ++k) {
      const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
      auto da = [&](int part) {
        const uint32_t sa = s0 + part * Cf::PART_BYTES;
        return A_MN ? desc_mnmajor(sa, k) : desc_kmajor(sa, k);
      };
      auto db = [&](int part) {
        const uint32_t sb = s0 + part * Cf::PART_BYTES + Cf::A_BYTES;
        return B_MN ? desc_mnmajor(sb, k) : desc_kmajor(sb, k);
      };
      mma(da(0), db(0), acc);
      if constexpr (Cf::X3) {
        mma(da(0), db(1), 1u);  // hi * lo'
        mma(da(1), db(0), 1u);  // lo * hi'
      }
    }
    // frees the stage (in both CTAs of a pair) once the MMAs have read it
    if (PAIR) ptx::tc_commit_pair(ptx::smem_addr(&ctl->empty[r.stage]), 0x3);
    else ptx::tc_commit(ptx::smem_addr(&ctl->empty[r.stage]));
    if (++r.stage == Cf::STAGES) { r.stage = 0; r.ph ^= 1u; }
  }
  return true;
}

template <int MODES, bool PAIR, int OP>
__global__ void __launch_bounds__(THREADS, 1)
    tc_strip_kernel(const __grid_constant__ TcMaps maps, const KParams p) {
  using Cf = Cfg<PAIR, OP>;
  constexpr int STAGES = Cf::STAGES;
  constexpr int STAGE_BYTES = Cf::STAGE_BYTES;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;  // 128B-swizzled tiles need 1024B alignment
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t staging = base + STAGES * STAGE_BYTES;  // 1024-aligned (stage sizes are)
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + STAGES * STAGE_BYTES + STAGING_BYTES);
  volatile int* abort_flag = &ctl->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;  // 0 = the pair's MMA issuer
  const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl->full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_addr(&ctl->tfull[b]), 1);
      // one arrival per epilogue warp (of both CTAs of a pair)
      ptx::mbar_init(ptx::smem_addr(&ctl->tempty[b]), PAIR ? 8 : 4);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    for (int i = 0; i < TQ; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->tq_full[i]), 1);
      // readers: MMA issuer + 4 epilogue warps, plus the second CTA's producer and 4 epilogue warps
      ptx::mbar_init(ptx::smem_addr(&ctl->tq_empty[i]), PAIR ? 10 : 5);
    }
    ctl->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    if (PAIR) {
      ptx::tmem_alloc_pair(ptx::smem_addr(&ctl->tmem_base), TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), TMEM_COLS);
      ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
  }
  // Barriers initialised and TMEM allocated in both CTAs before either uses the other's.
  if (PAIR) ptx::cluster_sync(); else __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int j = 0; j < p.njobs; ++j)
        for (int part = 0; part < Cf::PARTS; ++part) {
          ptx::prefetch_tmap(&maps.a[j][part]);
          ptx::prefetch_tmap(&maps.b[j][part]);
        }
      bool ok = true;
      Ring ring{0, 0u};
      TileQueue<PAIR> tq{ctl, abort_flag, p.err, 0, 0u, PAIR && rank != 0};
      // The first CTA posts every tile's ticket one tile ahead: when it starts loading tile t, the
      // ticket of tile t+1 is already in the ring, so the readers (and the peer CTA's producer)
      // find it there at the tile boundary; the counter is read one more tile ahead still.
      unsigned next = 0u;
      int upcoming = -1;
      if (rank == 0) {
        next = atomicAdd(&p.sched[0], 1u);
        upcoming = tq.post(next, p.sched, p.total_tiles, units);
        if (upcoming >= 0) next = atomicAdd(&p.sched[0], 1u);
      }
      while (ok) {
        int tile;
        if (rank == 0) {
          tile = upcoming;
          if (tile < 0) break;
          upcoming = tq.post(next, p.sched, p.total_tiles, units);
          if (upcoming >= 0) next = atomicAdd(&p.sched[0], 1u);
        } else {
          tile = tq.take(1u);
        }
        if (tile < 0) break;
        const TilePos tp = locate<PAIR>(p, tile);
        const Job& jb = p.job[tp.job];
        const int m0 = tp.tm * Cf::TILE_M + static_cast<int>(rank) * BM;       // first A row here
        const int n0 = tp.tn * BN + static_cast<int>(rank) * Cf::B_ROWS * PAIR;  // first B row
        dispatch_mode<MODES>(mode_of<MODES>(jb), [&](auto m) {
          ok = produce_tile<decltype(m)::value, PAIR, OP>(
              jb.nkb, jb.b_off, maps.a[tp.job], maps.b[tp.job], m0, n0, base, ctl, ring,
              abort_flag, p.err, rank, p.inject_stall != 0);
        });
      }
      if (!ok) {
        // Let copies already in flight land before the CTA can exit.
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 2000000ull) {}
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      bool ok = true;
      Ring ring{0, 0u};
      int acc = 0;
      uint32_t aph = 0;
      TileQueue<PAIR> tq{ctl, abort_flag, p.err, 0, 0u, PAIR && rank != 0};
      while (ok) {
        const int tile = tq.take(1u);
        if (tile < 0) break;
        const TilePos tp = locate<PAIR>(p, tile);
        const Job& jb = p.job[tp.job];
        if (!wait_bar(ptx::smem_addr(&ctl->tempty[acc]), aph ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        dispatch_mode<MODES>(mode_of<MODES>(jb), [&](auto m) {
          ok = mma_tile<decltype(m)::value, PAIR, OP>(jb.nkb, d_tmem, base, ctl, ring, abort_flag,
                                                      p.err);
        });
        if (!ok) break;
        // accumulator ready for the epilogue warps (of both CTAs of a pair)
        if (PAIR) ptx::tc_commit_pair(ptx::smem_addr(&ctl->tfull[acc]), 0x3);
        else ptx::tc_commit(ptx::smem_addr(&ctl->tfull[acc]));
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      if (!ok) {
        // Make sure no MMA is still writing TMEM before it is released.
        if (PAIR) ptx::tc_commit_pair(ptx::smem_addr(&ctl->drain), 0x1);
        else ptx::tc_commit(ptx::smem_addr(&ctl->drain));
        wait_bar_drain(ptx::smem_addr(&ctl->drain), 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;          // TMEM lane quadrant this warp may access
    const int r_in = q * 32 + lane;  // accumulator row owned by this thread
    const uint32_t wbuf0 = staging + q * 2 * STAGE_BUF_BYTES;  // this warp's two staging buffers
    float scale_valid = 0.f;
    if (p.dloss != nullptr) {
      const float dl = *p.dloss;
      scale_valid = (p.reduction == 0) ? dl / static_cast<float>(*p.n_valid) : dl;
    }
    int acc = 0;
    uint32_t aph = 0;
    TileQueue<PAIR> tq{ctl, abort_flag, p.err, 0, 0u, PAIR && rank != 0};
    while (true) {
      const int tile = tq.take(0xffffffffu);
      if (tile < 0) break;
      const TilePos tp = locate<PAIR>(p, tile);
      const Job& jb = p.job[tp.job];
      const CUtensorMap* mC = maps.c[tp.job];  // C or G in [0]; tf32 gradient parts in [0..3]
      const uint32_t tfull = ptx::smem_addr(&ctl->tfull[acc]);
      const uint32_t tempty_local = ptx::smem_addr(&ctl->tempty[acc]);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const int row = tp.tm * Cf::TILE_M + static_cast<int>(rank) * BM + r_in;
      const int box_row = tp.tm * Cf::TILE_M + static_cast<int>(rank) * BM + q * 32;
      // hand the accumulator back to the MMA issuer (in the pair's first CTA)
      auto release = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_local, 0));
          else ptx::mbar_arrive(tempty_local);
        }
      };

      const int mode = mode_of<MODES>(jb);
      const bool is_fwd = has_mode<MODES>(MODE_FWD_LSE) && mode == MODE_FWD_LSE;
      const bool is_grad = has_mode<MODES>(MODE_BWD_G) && mode == MODE_BWD_G;
      if (is_fwd || is_grad) {
        const bool row_ok = row < p.N;
        const int tcol0 = tp.tn * BN;
        const int ncols = min(BN, jb.strip_cols - tcol0);  // valid columns of this tile (>= 1)
        const int64_t y = row_ok ? p.labels[row] : p.ignore_index;
        const bool label_ok = (y != p.ignore_index) && (y >= 0) && (y < p.V);
        const int64_t trel = y - static_cast<int64_t>(jb.col0 + tcol0);
        const int tloc = (label_ok && trel >= 0 && trel < ncols) ? static_cast<int>(trel) : -1;

        if (is_fwd) {
          float m = -INFINITY, s = 0.f, t = 0.f;
          if (!wait_bar(tfull, aph, abort_flag, p.err)) break;
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            if (c * 32 >= ncols) break;  // same for every thread of the CTA
            float v[32];
            ptx::tmem_load32(tbase + c * 32, v);
            const int lim = ncols - c * 32;
            if (lim < 32) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j >= lim) v[j] = -INFINITY;
            }
            if (static_cast<unsigned>(tloc - c * 32) < 32u) {
              const int jt = tloc - c * 32;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j == jt) t = v[j];
            }
            float cm = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) cm = fmaxf(cm, v[j]);
            const float mn = fmaxf(m, cm);
            const float nml = -mn * LOG2E;
            float cs = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) cs += exp2f(fmaf(v[j], LOG2E, nml));
            s = s * exp2f(fmaf(m, LOG2E, nml)) + cs;
            m = mn;
          }
          release();
          if (row_ok) {
            p.part[static_cast<size_t>(tp.tn) * p.N + row] = make_float2(m, s);
            if (tloc >= 0) p.tgt[row] = t;
          }
        } else {
          // MODE_BWD_G: G = scale * (exp(Z - lse) - onehot) -> strip workspace.  Rows that are
          // not valid (ignored, bad label, past N) get exact zeros by selection, never as
          // 0 * exp(Z): their logits are not bounded by an lse of theirs, so exp can overflow
          // to inf there (Z above about 88.7), and 0 * inf would be NaN.
          if (row_ok && !label_ok && y != p.ignore_index && jb.first_strip && tp.tn == 0)
            atomicOr(p.err, ERR_LABEL);
          const float scale = scale_valid;
          const float nl = label_ok ? -p.lse[row] * LOG2E : 0.f;
          if (!wait_bar(tfull, aph, abort_flag, p.err)) break;
          ptx::tc_fence_after();
          if constexpr (OP == OP_TF32X3) {
            // fp32 gradient as tf32 hi / lo parts.  Per 32 columns the warp writes a 32 x 32 box
            // of each part into G (rows = its tokens) and then, transposed in shared memory, into
            // G^T (rows = the columns): lane t stores its value of column j at row j, word t of
            // the box, in the 128-byte swizzle (16-byte chunk (t/4) ^ (j%8)) -- one word per bank.
            const uint32_t hbuf = wbuf0, lbuf = wbuf0 + STAGE_BUF_BYTES;
            const bool rows_live = box_row < p.N;  // the warp holds at least one real token
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
              float g[32];
              if (c * 32 < ncols) {
                float v[32];
                ptx::tmem_load32(tbase + c * 32, v);
                const int lim = label_ok ? ncols - c * 32 : 0;  // no live column on such rows
                const int jt = tloc - c * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  g[j] = (j < lim) ? scale * exp2f(fmaf(v[j], LOG2E, nl)) : 0.f;
                  if (j == jt) g[j] -= scale;
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) g[j] = 0.f;
              }
              if (!rows_live) continue;
              if (c > 0) {  // both buffers' previous boxes must have been read
                if (lane == 0) ptx::bulk_wait_read<0>();
                __syncwarp();
              }
              const uint32_t hrow = hbuf + lane * 128, lrow = lbuf + lane * 128;
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                float h[4], l[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  h[t] = ptx::round_tf32(g[4 * jj + t]);
                  l[t] = ptx::round_tf32(g[4 * jj + t] - h[t]);
                }
                const uint32_t off = (static_cast<uint32_t>(jj) ^ (lane & 7)) << 4;
                ptx::st_shared_v4(hrow + off, __float_as_uint(h[0]), __float_as_uint(h[1]),
                                  __float_as_uint(h[2]), __float_as_uint(h[3]));
                ptx::st_shared_v4(lrow + off, __float_as_uint(l[0]), __float_as_uint(l[1]),
                                  __float_as_uint(l[2]), __float_as_uint(l[3]));
              }
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::tma_store_2d(&mC[0], hbuf, tcol0 + c * 32, box_row);
                ptx::tma_store_2d(&mC[1], lbuf, tcol0 + c * 32, box_row);
                ptx::bulk_commit();
                ptx::bulk_wait_read<0>();
              }
              __syncwarp();
              const uint32_t tw = (static_cast<uint32_t>(lane) & 3u) << 2;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float h = ptx::round_tf32(g[j]);
                const uint32_t off =
                    j * 128 + (((static_cast<uint32_t>(lane) >> 2) ^ (j & 7)) << 4) + tw;
                ptx::st_shared_f32(hbuf + off, h);
                ptx::st_shared_f32(lbuf + off, ptx::round_tf32(g[j] - h));
              }
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::tma_store_2d(&mC[2], hbuf, box_row, tcol0 + c * 32);
                ptx::tma_store_2d(&mC[3], lbuf, box_row, tcol0 + c * 32);
                ptx::bulk_commit();
              }
            }
            release();
            if (lane == 0) ptx::bulk_wait_read<0>();  // both buffers free for the next tile
            __syncwarp();
          } else {
          // The warp's 32 rows go out as 32 x 64-column boxes through its two staging buffers.
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            const uint32_t sbuf = wbuf0 + ((c >> 1) & 1) * STAGE_BUF_BYTES;
            if ((c & 1) == 0 && c >= 4) {  // the buffer's previous box must have been read
              if (lane == 0) ptx::bulk_wait_read<1>();
              __syncwarp();
            }
            uint32_t packed[16];
            if (c * 32 < ncols) {
              float v[32];
              ptx::tmem_load32(tbase + c * 32, v);
              const int lim = label_ok ? ncols - c * 32 : 0;  // no live column on such rows
              const int jt = tloc - c * 32;
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float g0 = (j < lim) ? scale * exp2f(fmaf(v[j], LOG2E, nl)) : 0.f;
                float g1 = (j + 1 < lim) ? scale * exp2f(fmaf(v[j + 1], LOG2E, nl)) : 0.f;
                if (j == jt) g0 -= scale;
                if (j + 1 == jt) g1 -= scale;
                __nv_bfloat162 h2 = __floats2bfloat162_rn(g0, g1);
                packed[j / 2] = *reinterpret_cast<uint32_t*>(&h2);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) packed[j] = 0u;
            }
            // this thread's row of the box: 128 bytes, 16-byte chunk jj at (jj ^ (row % 8)) -- the
            // 128-byte swizzle the store's tensor map expects (also spreads the warp over banks)
            const uint32_t rowaddr = sbuf + lane * 128;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t jj = (c & 1) * 4 + kk;
              ptx::st_shared_v4(rowaddr + ((jj ^ (lane & 7)) << 4), packed[4 * kk],
                                packed[4 * kk + 1], packed[4 * kk + 2], packed[4 * kk + 3]);
            }
            if (c & 1) {
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::tma_store_2d(mC, sbuf, tcol0 + (c - 1) * 32, box_row);
                ptx::bulk_commit();
              }
            }
          }
          release();
          if (lane == 0) ptx::bulk_wait_read<0>();  // both buffers free for the next tile
          __syncwarp();
          }
        }
      } else {
        // MODE_DH / MODE_DW: C (+)= accumulator, fp32.  The warp's 32 rows go out as 32 x 32
        // fp32 boxes through its two staging buffers; the tensor map clips rows and columns
        // outside C.  Accumulation into dH is a TMA add (one add per element per launch, in
        // strip order: deterministic).
        if (!wait_bar(tfull, aph, abort_flag, p.err)) break;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int col = tp.tn * BN + c * 32;
          if (col >= jb.c_cols) break;  // same for every thread of the CTA
          float v[32];
          ptx::tmem_load32(tbase + c * 32, v);
          const uint32_t sbuf = wbuf0 + (c & 1) * STAGE_BUF_BYTES;
          if (c >= 2) {  // the buffer's previous box must have been read
            if (lane == 0) ptx::bulk_wait_read<1>();
            __syncwarp();
          }
          const uint32_t rowaddr = sbuf + lane * 128;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            ptx::st_shared_v4(rowaddr + ((static_cast<uint32_t>(jj) ^ (lane & 7)) << 4),
                              __float_as_uint(v[4 * jj]), __float_as_uint(v[4 * jj + 1]),
                              __float_as_uint(v[4 * jj + 2]), __float_as_uint(v[4 * jj + 3]));
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (jb.accumulate) ptx::tma_reduce_add_2d(mC, sbuf, col, box_row);
            else ptx::tma_store_2d(mC, sbuf, col, box_row);
            ptx::bulk_commit();
          }
        }
        release();
        if (lane == 0) ptx::bulk_wait_read<0>();  // both buffers free for the next tile
        __syncwarp();
      }
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    if (lane == 0) ptx::bulk_wait<0>();  // this warp's output stores have landed
    __syncwarp();
  }

  // Every role of both CTAs is done (and no remote arrival is still on its way) before TMEM is
  // released and the CTAs exit.
  if (PAIR) ptx::cluster_sync(); else __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PAIR) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// 2-D tensor map (bf16, or fp32) over a row-major [outer x inner] array with `ld` elements per
// row, box = [box_outer x box_inner], 128-byte swizzle, zero fill outside the array.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
              uint32_t box_inner, uint32_t box_outer, int mode, char operand, bool fp32 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    set_error_detail("cuTensorMapEncodeTiled entry point unavailable");
    return false;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * (fp32 ? 4 : 2)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
          const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error_detail("tensor map of operand %c, strip GEMM mode %d refused (CUresult %d; %llu x %llu"
                     " elements, row stride %llu, box %u x %u, address %p)",
                     operand, mode, static_cast<int>(r), static_cast<unsigned long long>(outer),
                     static_cast<unsigned long long>(inner), static_cast<unsigned long long>(ld),
                     box_outer, box_inner, ptr);
    return false;
  }
  return true;
}

template <int MODES, bool PAIR, int OP>
cudaError_t launch(const TcMaps& maps, const KParams& p, int grid, cudaStream_t stream) {
  using Cf = Cfg<PAIR, OP>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tc_strip_kernel<MODES, PAIR, OP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cf::SMEM_BYTES);
    if (e != cudaSuccess) {
      set_error_detail("shared-memory attribute of the strip GEMM: %s", cudaGetErrorName(e));
      return e;
    }
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, tc_strip_kernel<MODES, PAIR, OP>, maps, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess)
    set_error_detail("launch of the strip GEMM (mode %d%s%s, %d jobs, grid %d, stream %p): %s",
                     p.job[0].mode, PAIR ? ", CTA pairs" : "", Cf::X3 ? ", tf32 parts" : "",
                     p.njobs, grid,
                     static_cast<void*>(stream), cudaGetErrorName(e));
  return e;
}

// Fills job j (maps and tile counts) from one strip GEMM description; false if a map is refused.
// OP_BF16 operands are bf16 arrays; OP_TF32X3 operands are pairs of fp32 arrays (hi, lo), with
// the transposed copies the K-major tf32 MMAs need for dH and dW.
template <bool PAIR, int OP>
bool make_job(const StripArgs& s, TcMaps& maps, Job& jb, int j) {
  using Cf = Cfg<PAIR, OP>;
  constexpr bool X3 = Cf::X3;
  constexpr int BK = Cf::BK;
  // the W operand: all V rows, or just this strip's rows starting at row 0
  const int64_t w_rows = s.w_strip_local ? s.strip_cols : s.V;
  const int w_row0 = s.w_strip_local ? 0 : s.col0;
  // one map per operand part: [0] from the hi (or only) array, [1] from the lo array
  auto parts = [&](CUtensorMap* m, const void* hi, const void* lo, uint64_t inner, uint64_t outer,
                   uint64_t ld, uint32_t bi, uint32_t bo, char name) {
    if (!make_map(&m[0], hi, inner, outer, ld, bi, bo, s.mode, name, X3)) return false;
    if (X3) return make_map(&m[1], lo, inner, outer, ld, bi, bo, s.mode, name, true);
    m[1] = m[0];
    return true;
  };
  int M, Ncols, K;
  bool ok;
  jb = Job{};
  jb.mode = s.mode;
  for (int c = 0; c < 4; ++c) maps.c[j][c] = CUtensorMap{};
  switch (s.mode) {
    case MODE_FWD_LSE:
    case MODE_BWD_G:
      M = static_cast<int>(s.N);
      Ncols = s.strip_cols;
      K = static_cast<int>(s.d);
      jb.b_off = w_row0;
      ok = parts(maps.a[j], s.H, s.H2, s.d, s.N, s.d, BK, BM, 'A') &&
           parts(maps.b[j], s.W, s.W2, s.d, w_rows, s.d, BK, Cf::B_ROWS, 'B');
      if (ok && s.mode == MODE_BWD_G) {
        if (X3) {
          // gradient strip [N x ldg] hi / lo and its transpose [ldg x ldt] (N tokens per row),
          // written as 32 x 32 fp32 boxes
          ok = parts(maps.c[j], s.G, s.G2, s.ldg, s.N, s.ldg, 32, 32, 'G') &&
               parts(&maps.c[j][2], s.GT, s.GT2, s.N, s.ldg, s.ldt, 32, 32, 'T');
        } else {
          // gradient strip [N x ldg] bf16, written as 64-column x 32-row boxes
          ok = make_map(&maps.c[j][0], s.G, s.ldg, s.N, s.ldg, 64, 32, s.mode, 'G');
        }
      }
      break;
    case MODE_DH:
      M = static_cast<int>(s.N);
      Ncols = static_cast<int>(s.d);
      K = s.strip_cols;
      if (X3) {
        // B = W_s^T [d x strip_cols] (row stride ldg): the map stops at the strip's columns, so
        // the k-block past them reads zeros, not the unwritten padding
        jb.b_off = 0;
        ok = parts(maps.a[j], s.G, s.G2, s.ldg, s.N, s.ldg, BK, BM, 'A') &&
             parts(maps.b[j], s.WT, s.WT2, s.strip_cols, s.d, s.ldg, BK, Cf::B_ROWS, 'B');
      } else {
        jb.b_off = w_row0;
        ok = make_map(&maps.a[j][0], s.G, s.ldg, s.N, s.ldg, BK, BM, s.mode, 'A') &&
             make_map(&maps.b[j][0], s.W, s.d, w_rows, s.d, MN_BOX_ELEMS, BK, s.mode, 'B');
      }
      ok = ok && make_map(&maps.c[j][0], s.C, s.d, s.N, s.ldc, 32, 32, s.mode, 'C', true);
      break;
    case MODE_DW:
      M = s.strip_cols;
      Ncols = static_cast<int>(s.d);
      K = static_cast<int>(s.N);
      jb.b_off = 0;
      if (X3) {
        // A = G_s^T [strip_cols x N], B = H^T [d x N] (row stride ldt): both maps stop at N
        ok = parts(maps.a[j], s.GT, s.GT2, s.N, s.strip_cols, s.ldt, BK, BM, 'A') &&
             parts(maps.b[j], s.HT, s.HT2, s.N, s.d, s.ldt, BK, Cf::B_ROWS, 'B');
      } else {
        ok = make_map(&maps.a[j][0], s.G, s.ldg, s.N, s.ldg, MN_BOX_ELEMS, BK, s.mode, 'A') &&
             make_map(&maps.b[j][0], s.H, s.d, s.N, s.d, MN_BOX_ELEMS, BK, s.mode, 'B');
      }
      ok = ok && make_map(&maps.c[j][0], s.C, s.d, s.strip_cols, s.ldc, 32, 32, s.mode, 'C', true);
      break;
    default:
      set_error_detail("unknown strip GEMM mode %d", s.mode);
      return false;
  }
  if (!ok) return false;
  jb.tiles_m = (M + Cf::TILE_M - 1) / Cf::TILE_M;
  jb.tiles_n = (Ncols + BN - 1) / BN;
  jb.nkb = (K + BK - 1) / BK;
  // tiles are numbered with 32-bit tickets
  if (static_cast<int64_t>(jb.tiles_m) * jb.tiles_n > (int64_t(1) << 30)) {
    set_error_detail("strip GEMM of %d x %d tiles: beyond the tile scheduler's range", jb.tiles_m,
                     jb.tiles_n);
    return false;
  }
  jb.num_tiles = (jb.nkb > 0) ? jb.tiles_m * jb.tiles_n : 0;
  jb.strip_cols = s.strip_cols;
  jb.col0 = s.col0;
  jb.c_cols = s.c_cols;
  jb.accumulate = s.accumulate;
  jb.first_strip = s.first_strip;
  return true;
}

template <bool PAIR, int OP>
cudaError_t run(const StripArgs* jobs, int njobs, cudaStream_t stream, int num_sms) {
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  KParams p{};
  for (int i = 0; i < njobs; ++i) {
    Job jb;
    if (!make_job<PAIR, OP>(jobs[i], maps, jb, p.njobs)) return cudaErrorInvalidResourceHandle;
    if (jb.num_tiles == 0) continue;  // nothing to compute (e.g. an empty dimension)
    p.job[p.njobs++] = jb;
    if (p.total_tiles > (1 << 30) - jb.num_tiles) return cudaErrorInvalidValue;  // 32-bit tickets
    p.total_tiles += jb.num_tiles;
  }
  if (p.njobs == 0) return cudaSuccess;
  const StripArgs& s = jobs[0];
  p.N = s.N;
  p.V = s.V;
  p.ignore_index = s.ignore_index;
  p.part = s.part;
  p.tgt = s.tgt;
  p.labels = s.labels;
  p.reduction = s.reduction;
  p.err = s.err;
  for (int i = 0; i < njobs; ++i)
    if (jobs[i].mode == MODE_BWD_G) {
      p.lse = jobs[i].lse;
      p.dloss = jobs[i].dloss;
      p.n_valid = jobs[i].n_valid;
    }
  p.sched = s.err + WS_SCHED_WORD;
  p.inject_stall = g_inject_stall;  // one launch only
  g_inject_stall = 0;
  // persistent grid: one CTA (or CTA pair) per SM (pair of SMs), never more than there are tiles
  const int units = PAIR ? num_sms / 2 : num_sms;
  const int grid = (p.total_tiles < units ? p.total_tiles : units) * (PAIR ? 2 : 1);
  // the kernel compiled for the modes of this launch (a launch never mixes the forward with the
  // backward)
  int present = 0;
  for (int j = 0; j < p.njobs; ++j) present |= 1 << p.job[j].mode;
  if (present == MODES_FWD) return launch<MODES_FWD, PAIR, OP>(maps, p, grid, stream);
  if (present == MODES_G) return launch<MODES_G, PAIR, OP>(maps, p, grid, stream);
  if ((present & ~MODES_DHDW) == 0) return launch<MODES_DHDW, PAIR, OP>(maps, p, grid, stream);
  return launch<MODES_BWD, PAIR, OP>(maps, p, grid, stream);
}

}  // namespace

int g_tile_config = 0;
int g_inject_stall = 0;

cudaError_t tc_strip_jobs(const StripArgs* jobs, int njobs, cudaStream_t stream, int num_sms) {
  if (njobs < 1 || njobs > MAX_JOBS) return cudaErrorInvalidValue;
  // Rows of C: tokens for the logit, gradient and dH GEMMs, strip columns for dW.
  int64_t rows = 0;
  for (int i = 0; i < njobs; ++i) {
    const int64_t r = (jobs[i].mode == MODE_DW) ? jobs[i].strip_cols : jobs[i].N;
    rows = r > rows ? r : rows;
  }
  bool pair;
  if (g_tile_config == 1) pair = false;
  else if (g_tile_config == 2) pair = true;
  else pair = rows > BM;  // pairs need a second 128-row half to be worth launching
  // every job of a launch has the first job's operand format
  for (int i = 1; i < njobs; ++i)
    if (jobs[i].op != jobs[0].op) return cudaErrorInvalidValue;
  if (jobs[0].op == OP_TF32X3)
    return pair ? run<true, OP_TF32X3>(jobs, njobs, stream, num_sms)
                : run<false, OP_TF32X3>(jobs, njobs, stream, num_sms);
  return pair ? run<true, OP_BF16>(jobs, njobs, stream, num_sms)
              : run<false, OP_BF16>(jobs, njobs, stream, num_sms);
}

cudaError_t tc_strip_gemm(const StripArgs& s, cudaStream_t stream, int num_sms) {
  return tc_strip_jobs(&s, 1, stream, num_sms);
}

}  // namespace lce
