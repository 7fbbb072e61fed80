// Persistent, warp-specialised BF16 GEMM for sm_103a with a pluggable epilogue.
//
// This is the "fixed GEMM mainloop" tier of CODA (CODA note, overall framework:
// a fixed tensor-core mainloop produces accumulator tiles; a programmable
// epilogue transforms each tile on chip before the global store; light
// auxiliary kernels combine tile partial statistics). The mainloop is written
// for GB300 rather than translated from the pages' Hopper design:
//
//   warp 0 (one thread)  TMA producer: 128B-swizzled A/B tiles into a
//                        kStages-deep shared-memory ring (mbarrier full/empty).
//   warp 1 (one thread)  MMA issuer: tcgen05.mma M=128 N=256 K=16, fp32
//                        accumulators in TMEM, two accumulator buffers so the
//                        epilogue of tile t overlaps the mainloop of tile t+1.
//   warps 2-5            epilogue: tcgen05.ld 32 lanes x 32 columns (thread =
//                        accumulator row), the epilogue program in registers,
//                        bf16 results staged in 64B-swizzled shared memory and
//                        written by TMA stores; per-row / per-column partial
//                        statistics written directly.
//
// Operands: C[M,N] = op(A)[M,K] * op(B)[K,N]. A is K-major ([M,K] row-major)
// or M-major ([K,M] row-major); B is N-major ([K,N] row-major, the weight
// layout) or K-major ([N,K] row-major). Ragged M, N, K are handled by TMA
// zero fill on loads and clipping on stores.
//
// Every mbarrier wait is bounded by %globaltimer. On expiry the kernel sets a
// bit in the device status word, raises a CTA-wide abort flag so that the
// other roles stop waiting, drains its own TMA loads and MMAs, frees TMEM and
// returns. No trap, no unbounded spin.
#pragma once

#include <type_traits>

#include "ptx.cuh"
#include "../../include/coda.h"

namespace coda {

constexpr int BM = 128;       // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;       // accumulator columns per tile
constexpr int BK = 64;        // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kTmemCols = 2 * BN;  // two accumulator buffers
constexpr int kStageBoxBytes = 32 * 64;  // one epilogue TMA store box: 32 rows x 64 bytes
constexpr int kEpiBufs = 2;              // staging double buffer
// Rank-2 epilogue inputs (z, Y, h1, dres, GU) arrive by TMA in 32 x 64B
// boxes into a per-warp ring of kInWarpBytes, issued several chunks ahead.
constexpr int kInBoxBytes = 32 * 64;
constexpr int kInWarpBytes = 8192;
constexpr int kMaxInSlots = 4;

// Per-variant constants. kCG = 1: one SM computes a 128 x 256 tile. kCG = 2:
// an SM pair (cta_group::2) computes a 256 x 256 tile; each CTA holds its 128
// rows of A and half (128 columns) of B, so a stage is 32 KiB per SM instead
// of 48 KiB.
// kIn = input boxes per chunk (0, 1, 2), kInWarp = bytes of each epilogue
// warp's input ring, kSlots = store boxes per staging buffer (1-3), kBufs =
// staging buffers, kShared = bytes of an epilogue-wide table. The mainloop gets
// as many stages as the shared memory left after the epilogue's staging, input
// ring and table allows, at most 6 (pair) or 4 (single): 6 / 4 without
// inputs, 5 / 3 with an 8 KiB ring per warp or three staging boxes.
template <int kCG, int kIn, int kSlots, int kInWarp = kInWarpBytes, int kBufs = kEpiBufs, int kShared = 0>
struct Cfg {
  static_assert(kCG == 1 || kCG == 2, "single-SM or SM-pair tiles");
  static constexpr int kPair = kCG;               // CTAs per MMA (cta_group)
  static constexpr int kTileM = BM * kPair;
  static constexpr int kBLoad = BN / kPair;       // B columns loaded per CTA
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = kBLoad * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStageBufs = kBufs;  // staging buffers per warp (2, or 1 to buy a stage)
  static constexpr int kEpiWarpBytes = kStageBoxBytes * kSlots * kBufs;
  static constexpr int kInSlots = kIn ? kInWarp / (kIn * kInBoxBytes) : 0;
  static constexpr int kInBytes = kIn ? kEpiWarps * kInWarp : 0;
  static constexpr int kSharedBytes = kShared;  // epilogue-wide table, filled once per CTA
  // As many mainloop stages as the rest of shared memory leaves room for, at
  // most 6 (SM pair) or 4 (single SM).
  static constexpr int kFixedBytes = 1024 + kEpiWarps * kEpiWarpBytes + kInBytes + kShared + 16 +
                                     8 * (2 + 2 + 1 + kEpiWarps * kMaxInSlots + kEpiWarps * 8);
  static constexpr int kFitStages = (232448 - kFixedBytes) / (kStageBytes + 16);
  static constexpr int kMaxStages = kCG == 2 ? 6 : 4;
  static constexpr int kStages = kFitStages < kMaxStages ? kFitStages : kMaxStages;
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + kEpiWarps * kMaxInSlots + kEpiWarps * 8;
  static constexpr int kSmemBytes =
      1024 + kStages * kStageBytes + kEpiWarps * kEpiWarpBytes + kInBytes + kShared + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kStages >= 3, "mainloop ring");
  static_assert(kInSlots <= kMaxInSlots && (kIn == 0 || kInSlots >= 1), "input ring slots");
  static_assert(kSlots >= 1 && kSlots <= 3, "staging slots");
  static_assert(kBufs == 1 || kBufs == 2, "staging buffers");
  static_assert(kShared % 16 == 0, "epilogue table alignment");
};

// Per-epilogue staging buffers: two unless the epilogue declares kStageBufs.
template <class E, class = void>
struct StageBufsOf {
  static constexpr int value = kEpiBufs;
};
template <class E>
struct StageBufsOf<E, std::void_t<decltype(E::kStageBufs)>> {
  static constexpr int value = E::kStageBufs;
};

// Per-epilogue input-ring size: kInWarpBytes unless the epilogue declares
// kInRingBytes (a smaller ring can buy a mainloop stage).
template <class E, class = void>
struct InRingOf {
  static constexpr int value = kInWarpBytes;
};
template <class E>
struct InRingOf<E, std::void_t<decltype(E::kInRingBytes)>> {
  static constexpr int value = E::kInRingBytes;
};

// Per-epilogue shared table: none unless the epilogue declares kSharedBytes,
// in which case its init_shared() fills the table once per CTA before the
// first tile (all four epilogue warps, then a named barrier among them).
template <class E, class = void>
struct SharedOf {
  static constexpr int value = 0;
};
template <class E>
struct SharedOf<E, std::void_t<decltype(E::kSharedBytes)>> {
  static constexpr int value = E::kSharedBytes;
};

// TMA loads per chunk: kInBoxes (32 x 64-byte boxes) unless the epilogue
// declares kInLoads = 1, one 32 x 128-byte box filling the same ring bytes
// (the SwiGLU backward's 64 pre-activation columns per chunk).
template <class E, class = void>
struct InLoadsOf {
  static constexpr int value = E::kInBoxes;
};
template <class E>
struct InLoadsOf<E, std::void_t<decltype(E::kInLoads)>> {
  static constexpr int value = E::kInLoads;
};

template <class Epi, int kCG>
using CfgOf = Cfg<kCG, Epi::kInBoxes, Epi::kMaxSlots, InRingOf<Epi>::value, StageBufsOf<Epi>::value,
                  SharedOf<Epi>::value>;

constexpr int BSEG = 128;  // epilogue segment: columns per partial-statistics block

// L2 cache policy of the epilogue's input boxes and stores: they stream
// through once, and evict-first keeps them from displacing operand tiles that
// later tiles read again.
constexpr bool kEpiEvictFirst = true;

struct GemmShape {
  int M, N, K;
  int a_mn, b_mn;  // 0: K-major; 1: MN-major, 64-wide 2-D boxes; 2: MN-major, one 3-D box per stage
  int m_blocks, n_blocks, k_blocks, num_tiles, group_m;
  // Data-parallel work items, raster tiles from dp_first on: the first
  // full_items are whole tiles; each of the remaining ones up to num_items (a
  // partial last wave) is split into two 128-column halves so the last wave
  // takes half a tile's time.
  int dp_first, full_items, num_items;
  // Stream-K tiles (sk_tiles > 0; then dp_first = sk_tiles and there are no
  // half tiles): raster tiles 0 .. sk_tiles-1, one wave plus the leftover
  // tiles, are dealt out as ranges of the flattened (tile, k-block) iteration
  // space, sk_q + 1 k-blocks to each of the first sk_r clusters and sk_q to
  // the others, so every cluster's work is the same. Each cluster runs its
  // range before its data-parallel tiles, so the partials of split tiles are
  // combined while later tiles' mainloops run. sk_q is at least k_blocks, so
  // a tile is split at most once, at the boundary between two neighbouring
  // clusters' ranges (see WorkCursor for the order a range is walked in);
  // both pieces write their fp32 partial accumulator to sk_part, and the
  // piece that arrives second (counted in sk_ctr, tagged with the launch's
  // sk_epoch) adds the other's partial and runs the epilogue.
  int sk_tiles, sk_q, sk_r;
  int sk_rotate;       // 1: walk each range from its first tile boundary (see WorkCursor)
  float4* sk_part;     // [boundary][side][CTA of the pair][epilogue warp][32 x 256 fp32], see sk_slot()
  unsigned* sk_ctr;    // [boundary][CTA of the pair][epilogue warp] arrival words
  long sk_part_f4;     // extents of the two (float4s, words), for the checked build
  int sk_ctr_n;
  unsigned sk_epoch;   // 1 .. 2^30 - 1, unique per launch on the workspace
  int seg_blocks;  // ceil(N / 128): second dimension of the [M, seg_blocks] partials
  int* status;                    // device status word (CODA_DEVST_* bits)
  unsigned long long timeout_ns;  // bound on every mbarrier wait
  int inject;                     // test hook: 1 = producers skip their first stage fill
  float alpha;                    // FP8 mainloop: product of the operands' per-tensor scales
};

// One unit of a cluster's work: a tile (or a 128-column half tile) and the
// range of k-blocks it accumulates. side -1: the whole reduction; side 0: the
// first k-blocks of a tile split at the end of this cluster's stream-K range
// (boundary bnd = this cluster); side 1: the last k-blocks of a tile split at
// the start of it (bnd = the previous cluster).
struct Work {
  int m_blk, n0, ncols;
  int kb0, kb1;
  int side, bnd;
};
// Each role walks its cluster's work with its own cursor: the cluster's
// stream-K range first, then the data-parallel items (t = cluster,
// cluster + clusters, ...). With sk_rotate the range [lo, end) is walked
// from its first tile boundary [pos, end), then the piece before it [lo, hi):
// every cluster then starts at k-block 0 of some tile and all of them move
// through K in step, as in the data-parallel waves, so the operand slices
// read at one time are few. Without it the clusters' k positions are spread
// over the whole reduction, which is faster while the stream-K tiles'
// operands fit in L2 together and much slower once they do not; there each
// cluster walks the shorter of its two parts [lo, b) and [b, end) (b the first
// tile boundary) first. The longer part then covers the split epilogue of the
// shorter one: the first whole tile after the range reuses the shorter
// part's accumulator buffer, and a short second part would leave its MMAs
// waiting for that epilogue.
struct WorkCursor {
  int t, pos, end, lo, hi;
};

struct EpiCtx {
  int* status;  // device status word (CODA_DEVST_* bits)
  int M, N;
  int m0, n0;   // this segment's first row (of the CTA's 128) and first column
  int m_blk;
  int n_blk;    // n0 / 128: the column block of the segment's partial statistics
  int n_blocks; // ceil(N / 128)
  int row;    // this thread's accumulator row (global index)
  int wrow0;  // first row of this warp's 32-row slice (global index)
  int ew;     // warp quarter (TMEM lanes 32*ew .. 32*ew+31)
  int lane;
  int k_blocks;
  uint32_t shared;  // shared-memory address of the epilogue's table (kSharedBytes), 0 if none
};

// Checked build (CODA_CHECKED=1): every direct global access of an epilogue
// first tests its index against the extent of the tensor it touches; an index
// outside sets CODA_DEVST_BOUNDS in the device status word and the access is
// skipped. In the normal build the test compiles away.
#if defined(CODA_CHECKED) && CODA_CHECKED
__device__ __forceinline__ bool coda_in_extent(long idx, long extent, int* status) {
  if (idx >= 0 && idx < extent) return true;
  atomicOr(status, CODA_DEVST_BOUNDS);
  return false;
}
#define CODA_IN_ST(status, idx, extent) coda_in_extent(static_cast<long>(idx), static_cast<long>(extent), (status))
#else
#define CODA_IN_ST(status, idx, extent) true
#endif
#define CODA_IN(cx, idx, extent) CODA_IN_ST((cx).status, idx, extent)

// Tile order: groups of group_m row-blocks sweep all column blocks, so the
// A rows of a group and the B columns in flight stay L2 resident.
__device__ __forceinline__ void tile_coords(int t, const GemmShape& p, int& m_blk, int& n_blk);
// Work item t -> row block, first column and width (256 or 128 columns).
__device__ __forceinline__ void item_coords(int t, const GemmShape& p, int& m_blk, int& n0, int& ncols) {
  int n_blk;
  if (t < p.full_items) {
    tile_coords(p.dp_first + t, p, m_blk, n_blk);
    n0 = n_blk * BN;
    ncols = BN;
  } else {
    const int h = t - p.full_items;
    tile_coords(p.full_items + (h >> 1), p, m_blk, n_blk);
    n0 = n_blk * BN + (h & 1) * BSEG;
    ncols = BSEG;
  }
}
__device__ __forceinline__ void tile_coords(int t, const GemmShape& p, int& m_blk, int& n_blk) {
  const int per_group = p.group_m * p.n_blocks;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int first_m = g * p.group_m;
  int gsz = p.m_blocks - first_m;
  if (gsz > p.group_m) gsz = p.group_m;
  m_blk = first_m + r % gsz;
  n_blk = r / gsz;
}

__device__ __forceinline__ void work_begin(const GemmShape& p, int cluster, WorkCursor& w) {
  w.t = cluster;
  w.pos = w.end = w.lo = w.hi = 0;
  if (p.sk_tiles > 0) {
    w.lo = cluster * p.sk_q + (cluster < p.sk_r ? cluster : p.sk_r);
    w.end = w.lo + p.sk_q + (cluster < p.sk_r ? 1 : 0);
    const int b = (w.lo + p.k_blocks - 1) / p.k_blocks * p.k_blocks;  // < end: range >= k_blocks
    w.hi = (p.sk_rotate || w.end - b < b - w.lo) ? b : w.lo;
    w.pos = w.hi;
  }
}
// The cluster's next work unit; false when it has none left. Every role of
// the cluster calls this in the same order and gets the same sequence.
__device__ __forceinline__ bool work_next(const GemmShape& p, int cluster, int clusters, WorkCursor& w, Work& o) {
  const bool rotated = w.pos >= w.end;  // the range's head [pos, end) is done: its first piece [lo, hi)
  if (!rotated || w.lo < w.hi) {
    const int s = rotated ? w.lo : w.pos;
    const int e = rotated ? w.hi : w.end;
    const int u = s / p.k_blocks;
    const int base = u * p.k_blocks;
    int n_blk;
    tile_coords(u, p, o.m_blk, n_blk);
    o.n0 = n_blk * BN;
    o.ncols = BN;
    o.kb0 = s - base;
    o.kb1 = e - base < p.k_blocks ? e - base : p.k_blocks;
    if (o.kb0 > 0) {
      o.side = 1;
      o.bnd = cluster - 1;
    } else if (o.kb1 < p.k_blocks) {
      o.side = 0;
      o.bnd = cluster;
    } else {
      o.side = -1;
      o.bnd = 0;
    }
    if (rotated)
      w.lo = w.hi;
    else
      w.pos = base + o.kb1;
    return true;
  }
  if (w.t < p.num_items) {
    item_coords(w.t, p, o.m_blk, o.n0, o.ncols);
    o.kb0 = 0;
    o.kb1 = p.k_blocks;
    o.side = -1;
    o.bnd = 0;
    w.t += clusters;
    return true;
  }
  return false;
}
// Partial accumulator of one epilogue warp's 32 rows x 256 columns for the
// piece `side` of the tile split at boundary `bnd`: chunk c (32 columns),
// vector v (4 columns) of lane l's row at float4 index (c * 8 + v) * 32 + l,
// so each warp-wide 16-byte access covers 512 contiguous bytes.
__device__ __forceinline__ long sk_slot(int kPair, int bnd, int side, uint32_t q, int ew) {
  return static_cast<long>(((bnd * 2 + side) * kPair + static_cast<int>(q)) * 4 + ew) << 11;
}
__device__ __forceinline__ int sk_counter(int kPair, int bnd, uint32_t q, int ew) {
  return (bnd * kPair + static_cast<int>(q)) * 4 + ew;
}
// Count one piece's arrival at a split tile (lane 0 of the warp, after the
// warp's partial writes and a fence). The word holds the launch's epoch in
// its upper 30 bits and the arrivals in the lower 2; a word left by another
// launch, also one that stopped part way, restarts the count. Returns the
// number of arrivals including this one (2 = both pieces are in), or 0 if
// the word could not be updated.
__device__ __forceinline__ unsigned sk_arrive(unsigned* ctr, unsigned epoch) {
  unsigned cur = atomicAdd(ctr, 0u);
#pragma unroll 1
  for (int i = 0; i < 64; ++i) {
    const unsigned want = (cur >> 2) == epoch ? cur + 1u : ((epoch << 2) | 1u);
    const unsigned prev = atomicCAS(ctr, cur, want);
    if (prev == cur) return want & 3u;
    cur = prev;
  }
  return 0u;
}

// Bounded wait. Returns false (after flagging the status word and the CTA
// abort flag) if the phase did not complete within timeout_ns, or if another
// role of this CTA already aborted.
static __device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, const GemmShape& p,
                                               volatile int* abort_flag) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > p.timeout_ns) {
      atomicOr(p.status, CODA_DEVST_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const GemmShape& p,
                                             volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return wait_bounded_slow(bar, parity, p, abort_flag);
}
// Bounded wait for long waits off the critical path (the epilogue waiting for
// the next accumulator): the thread sleeps on the barrier between checks, so
// it does not take issue slots from the producer and MMA threads that share
// its SM sub-partition.
static __device__ __noinline__ bool wait_bounded_sleep(uint32_t bar, uint32_t parity, const GemmShape& p,
                                                       volatile int* abort_flag) {
  if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > p.timeout_ns) {
      atomicOr(p.status, CODA_DEVST_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}
// Bounded wait used while draining after an abort: ignores the abort flag.
static __device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, unsigned long long timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
  return true;
}

// Write 16 bytes of row `r` (0..31), 16-byte chunk `c16` (0..3), into a
// 32 x 64B staging box laid out with the TMA 64-byte swizzle.
__device__ __forceinline__ void stage_put(uint32_t box, int r, int c16, uint32_t a, uint32_t b, uint32_t c,
                                          uint32_t d) {
  st_shared_v4(box + r * 64 + ((c16 ^ ((r >> 1) & 3)) << 4), a, b, c, d);
}
// Pack 32 fp32 values to bf16 and write them as one full 64-byte staging row.
__device__ __forceinline__ void stage_row32(uint32_t box, int r, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    stage_put(box, r, q, pack_bf16(v[8 * q + 0], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
              pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}

// Row r (0..31) of a 32 x 128B box laid out with the TMA 128-byte swizzle
// (16-byte granule q of row r at granule q ^ (r mod 8)), as eight vectors; and
// the matching staging write. Such a box must start on a 1024-byte boundary.
__device__ __forceinline__ void box128_row(uint32_t box, int r, uint4 (&v)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) v[q] = ld_shared_v4(box + r * 128 + ((q ^ (r & 7)) << 4));
}
__device__ __forceinline__ void stage128_put(uint32_t box, int r, int q, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  st_shared_v4(box + r * 128 + ((q ^ (r & 7)) << 4), a, b, c, d);
}

// Row r (0..31) of a 32 x 64B box laid out with the TMA 64-byte swizzle, as
// four 16-byte vectors (conflict-free across the warp).
__device__ __forceinline__ void box_row(uint32_t box, int r, uint4 (&v)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = ld_shared_v4(box + r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
}

// Issue the loads of 32 consecutive bf16 of a row-major [rows, cols] tensor
// starting at (row, col0) as four 16-byte vectors; vectors past the bounds are
// zero. cols is a multiple of 8 and col0 of 32, so each vector is all-in or
// all-out. The values are consumed later (unpack32), so the load latency
// overlaps whatever runs in between.
__device__ __forceinline__ void load_raw32(const __nv_bfloat16* base, long ld, int rows, int cols, int row, int col0,
                                           uint4 (&v)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[q] = make_uint4(0, 0, 0, 0);
    if (row < rows && col0 + 8 * q < cols) v[q] = ldg_nc_v4(base + static_cast<long>(row) * ld + col0 + 8 * q);
  }
}
__device__ __forceinline__ void unpack32(const uint4 (&u)[4], float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[8 * q + 0] = bf16_lo(u[q].x);
    v[8 * q + 1] = bf16_hi(u[q].x);
    v[8 * q + 2] = bf16_lo(u[q].y);
    v[8 * q + 3] = bf16_hi(u[q].y);
    v[8 * q + 4] = bf16_lo(u[q].z);
    v[8 * q + 5] = bf16_hi(u[q].z);
    v[8 * q + 6] = bf16_lo(u[q].w);
    v[8 * q + 7] = bf16_hi(u[q].w);
  }
}

// ---------------------------------------------------------------------------
// The kernel. Epi provides:
//   struct Params; struct State; struct Pre (registers for a chunk's direct loads);
//   static constexpr int kChunksPerStore;          // 32-col chunks per store step
//   static constexpr int kInBoxes;                 // TMA input boxes per chunk (0..2)
//   static constexpr int kMaxSlots;                // staging boxes per store step (2 or 3)
//   __device__ static bool has_input(const Params&, const EpiCtx&, int c);
//   __device__ static void in_coord(const Params&, const EpiCtx&, int c, int box, int& map, int& x, int& y);
//   __device__ static int  slots(const Params&);   // TMA store boxes per step (0..kMaxSlots)
//   __device__ static void begin(State&, const Params&, const EpiCtx&);
//   __device__ static void prefetch(const Params&, const EpiCtx&, int c, Pre&);  // issue chunk c's loads
//   __device__ static void chunk(State&, const Params&, const EpiCtx&, int c, float (&acc)[32],
//                                const Pre&, uint32_t in, uint32_t box0, uint32_t box1);
//     (`in` = shared address of the chunk's input boxes, 0 if it has none)
//   __device__ static void store_coord(const Params&, const EpiCtx&, int c, int slot, int& map, int& x, int& y);
//   __device__ static void end(State&, const Params&, const EpiCtx&);
// ---------------------------------------------------------------------------
// kF8: the FP8 mainloop. A and B are E4M3, K-major; a stage holds 128 K
// elements (the same 128-byte rows, so the same shared-memory layout, boxes and
// descriptors as bf16), the MMAs are kind::f8f6f4 with K = 32, and the
// accumulator is scaled by p.alpha before the epilogue program sees it.
template <class Epi, int kCG, bool kF8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_epilogue_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
                         const __grid_constant__ CUtensorMap tmI0, const __grid_constant__ CUtensorMap tmI1,
                         const GemmShape p, const typename Epi::Params ep) {
  constexpr int kIn = Epi::kInBoxes;
  constexpr int kSlots = Epi::kMaxSlots;
  using C = CfgOf<Epi, kCG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_epi = smem + C::kStages * C::kStageBytes;
  uint8_t* s_in = s_epi + kEpiWarps * C::kEpiWarpBytes;
  uint8_t* s_tab = s_in + C::kInBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_tab + C::kSharedBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t s_base = smem_u32(smem);
  // In a pair, the even CTA (the leader) issues the MMAs for both; its full
  // and TMEM-empty barriers collect the pair's arrivals. q is this CTA's place
  // in the pair.
  constexpr int kPair = C::kPair;
  const uint32_t q = kCG == 2 ? cluster_ctarank() : 0u;
  constexpr uint32_t leader_rank = 0u;
  const bool leader = q == 0;
  const int cluster_id = blockIdx.x / kCG;
  const int num_clusters = gridDim.x / kCG;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + C::kStages + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * C::kStages + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * C::kStages + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * C::kStages + 4);
  auto in_bar = [&](int ew_, int slot) { return smem_u32(bars + 2 * C::kStages + 5 + ew_ * kMaxInSlots + slot); };
  // the last tile's input boxes, loaded all at once into the then idle mainloop
  // stages: one barrier per chunk (at most 8) and epilogue warp
  auto last_bar = [&](int ew_, int j) {
    return smem_u32(bars + 2 * C::kStages + 5 + kEpiWarps * kMaxInSlots + ew_ * 8 + j);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps * kPair);
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < kEpiWarps * kMaxInSlots; ++i) mbar_init(in_bar(i / kMaxInSlots, i % kMaxInSlots), 1);
    for (int i = 0; i < kEpiWarps * 8; ++i) mbar_init(last_bar(i / 8, i % 8), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    if constexpr (kCG == 2) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kCG == 2) cluster_sync_all();  // barriers of all CTAs initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The prologue above (barriers, TMEM, tensor-map prefetch) touches no global
  // memory, so it may overlap the previous kernel of the stream; everything
  // below reads or writes global memory and waits for that kernel first.
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer (every CTA)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // stage fills issued (for the drain)
      bool ok = true;
      if (p.inject == 1) {
        // test hook: the first fill is never issued, so the MMA's wait on it
        // must run out and take the abort path (the outputs are then undefined)
        stage = 1;
        issued = 1;
      }
      WorkCursor wc;
      work_begin(p, cluster_id, wc);
      Work w;
      while (ok && work_next(p, cluster_id, num_clusters, wc, w)) {
        const int m0 = w.m_blk * C::kTileM + static_cast<int>(q) * BM;
        const int bcols = w.ncols / kPair;  // B columns this CTA loads
        const int nb0 = w.n0 + static_cast<int>(q) * bcols;
        // N-major B arrives in 64-column boxes (b_mn 1) or as one 3-D box of
        // kBLoad columns (b_mn 2); K-major B as one box of kBLoad rows (a half
        // tile reads past its columns: harmless extra bytes)
        const int nbox = p.b_mn == 1 ? bcols / 64 : 0;
        const uint32_t tx = kPair * (C::kABytes + (p.b_mn == 1 ? static_cast<uint32_t>(bcols * BK * 2) : C::kBBytes));
        // The k-loop is the kernel's critical path: keep it to the wait, the
        // expected-bytes arrive and the copies.
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, p, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          if (leader) mbar_arrive_expect_tx(fb, tx);
          const uint32_t fb_target = kCG == 2 ? mapa_shared(fb, leader_rank) : fb;
          const uint32_t a_dst = s_base + stage * C::kStageBytes;
          const uint32_t b_dst = a_dst + C::kABytes;
          const int k0 = kb * (kF8 ? 2 * BK : BK);  // elements: one 128-byte row per stage either way
          auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y) {
            if constexpr (kCG == 2)
              tma_load_2d_pair(dst, m, fb_target, x, y);
            else
              tma_load_2d(dst, m, fb_target, x, y);
          };
          auto load3 = [&](uint32_t dst, const CUtensorMap* m, int y, int z) {
            if constexpr (kCG == 2)
              tma_load_3d_pair(dst, m, fb_target, 0, y, z);
            else
              tma_load_3d(dst, m, fb_target, 0, y, z);
          };
          if (p.a_mn == 2) {
            load3(a_dst, &tmA, k0, m0 >> 6);
          } else if (p.a_mn) {
            load(a_dst, &tmA, m0, k0);
            load(a_dst + 8192, &tmA, m0 + 64, k0);
          } else {
            load(a_dst, &tmA, k0, m0);
          }
          if (p.b_mn == 2) {
            load3(b_dst, &tmB, k0, nb0 >> 6);
          } else if (p.b_mn) {
#pragma unroll
            for (int j = 0; j < C::kBLoad / 64; ++j)
              if (j < nbox) load(b_dst + j * 8192, &tmB, nb0 + 64 * j, k0);
          } else {
            load(b_dst, &tmB, k0, nb0);
          }
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every load signalled on this CTA's full barriers has landed
      // before the CTA exits (in a pair, both CTAs' loads signal the leader's,
      // in lock step). Fill f of stage s completes phase (f / kStages) & 1 of
      // that stage's barrier.
      if (leader)
        for (int s = 0; s < C::kStages; ++s) {
          const uint32_t fills = issued / C::kStages + (static_cast<uint32_t>(s) < issued % C::kStages ? 1u : 0u);
          if (fills > 0 && !(p.inject == 1 && s == 0 && fills == 1))
            wait_drain(full_bar(s), (fills - 1) & 1u, p.timeout_ns);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (lane == 0 && leader) {
      const int amn = p.a_mn != 0, bmn = p.b_mn != 0;
      const uint32_t idesc_full = kF8 ? idesc_e4m3_f32(C::kTileM, BN) : idesc_bf16_f32(C::kTileM, BN, amn, bmn);
      const uint32_t idesc_half = kF8 ? idesc_e4m3_f32(C::kTileM, BSEG) : idesc_bf16_f32(C::kTileM, BSEG, amn, bmn);
      // Operand descriptors. K-major: 128B rows, 8-row groups 1024B apart,
      // K advances 32B (16 bf16) inside the swizzle atom. MN-major: 64-element
      // MN chunks 8192B apart (LBO), 8-row K groups 1024B apart (SBO), K
      // advances 16 rows = 2048B.
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, b_lbo = p.b_mn ? 8192u : 16u;
      const uint32_t a_kstep = p.a_mn ? 2048u : 32u, b_kstep = p.b_mn ? 2048u : 32u;
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      WorkCursor wc;
      work_begin(p, cluster_id, wc);
      Work w;
      for (; ok && work_next(p, cluster_id, num_clusters, wc, w); ++local) {
        const uint32_t idesc = w.ncols == BN ? idesc_full : idesc_half;
        const int buf = local & 1;
        const uint32_t tphase = static_cast<uint32_t>((local >> 1) & 1);
        if (!wait_bounded(tempty_bar(buf), tphase ^ 1u, p, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, p, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = s_base + stage * C::kStageBytes;
          const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = smem_desc_sw128(a_addr + k * a_kstep, a_lbo, 1024u);
            const uint64_t bd = smem_desc_sw128(b_addr + k * b_kstep, b_lbo, 1024u);
            const uint32_t acc_in = (kb > w.kb0 || k > 0) ? 1u : 0u;
            if constexpr (kF8) {
              if constexpr (kCG == 2)
                tc_mma_f8_pair(d_tmem, ad, bd, idesc, acc_in);
              else
                tc_mma_f8(d_tmem, ad, bd, idesc, acc_in);
            } else {
              if constexpr (kCG == 2)
                tc_mma_bf16_pair(d_tmem, ad, bd, idesc, acc_in);
              else
                tc_mma_bf16(d_tmem, ad, bd, idesc, acc_in);
            }
          }
          // the stage is free in both CTAs of the pair
          if constexpr (kCG == 2)
            tc_commit_pair(empty_bar(stage), 0x3);
          else
            tc_commit(empty_bar(stage));
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kCG == 2)
          tc_commit_pair(tfull_bar(buf), static_cast<uint16_t>(0x3u << leader_rank));
        else
          tc_commit(tfull_bar(buf));
      }
      // Drain: all MMAs issued here complete before TMEM is freed.
      if constexpr (kCG == 2)
        tc_commit_pair(drain_bar, static_cast<uint16_t>(1u << leader_rank));
      else
        tc_commit(drain_bar);
      wait_drain(drain_bar, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (every CTA)
    // Chunk c+1's global loads are issued before chunk c is read from TMEM, and
    // the next tile's first chunk before waiting for that tile's accumulator,
    // so load latency overlaps TMEM reads, math and the mainloop.
    const int ew = warp & 3;
    const uint32_t my_stage = smem_u32(s_epi) + ew * C::kEpiWarpBytes;
    const uint64_t pol_stream = kEpiEvictFirst ? l2_policy_evict_first() : 0ull;
    (void)pol_stream;
    if constexpr (C::kSharedBytes > 0) {
      // the 128 epilogue threads fill the table together, then wait for each other
      Epi::init_shared(ep, smem_u32(s_tab), static_cast<int>(threadIdx.x) - 64, p.status);
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    // Segment `seg` (128 columns) of work unit wk; false if it lies past N.
    auto make_ctx = [&](const Work& wk, int seg, EpiCtx& cx) {
      cx.m_blk = wk.m_blk;
      const int n0 = wk.n0;
      cx.status = p.status;
      cx.M = p.M;
      cx.N = p.N;
      cx.m0 = cx.m_blk * C::kTileM + static_cast<int>(q) * BM;
      cx.n0 = n0 + seg * BSEG;
      cx.n_blk = cx.n0 / BSEG;
      cx.n_blocks = p.seg_blocks;
      cx.ew = ew;
      cx.lane = lane;
      cx.wrow0 = cx.m0 + 32 * ew;
      cx.row = cx.wrow0 + lane;
      cx.k_blocks = p.k_blocks;
      cx.shared = C::kSharedBytes ? smem_u32(s_tab) : 0u;
      return cx.n0 < p.N;
    };
    auto item_segs = [&](const Work& wk) { return wk.ncols / BSEG; };
    constexpr int kSegChunks = BSEG / 32;
    // stage-memory bytes per epilogue warp for the last unit's inputs: 8 chunks
    constexpr int kLastWarpBytes = 2 * kSegChunks * (kIn > 0 ? kIn : 1) * kInBoxBytes;
    static_assert(kEpiWarps * kLastWarpBytes <= C::kStages * C::kStageBytes, "last unit's inputs fit the stages");
    int local = 0;
    int sbuf = 0;
    const int nslots = Epi::slots(ep);

    // Input ring: lane 0 keeps up to kInSlots chunks' input boxes in flight,
    // running ahead across segments and work items; every lane consumes them
    // in the same order.
    const uint32_t in_base = smem_u32(s_in) + ew * InRingOf<Epi>::value;
    uint32_t seq_used = 0;    // chunks consumed (all lanes)
    uint32_t seq_issued = 0;  // chunks issued (lane 0)
    int last_issued = 0;      // lane 0: chunks of the last unit loaded into the stage memory
    int it_s = 0, it_c = 0;  // issue cursor (lane 0): segment and chunk of work unit iw
    WorkCursor icur;
    work_begin(p, cluster_id, icur);
    Work iw;
    bool it_live = work_next(p, cluster_id, num_clusters, icur, iw);
    EpiCtx ic;
    bool ic_ok = it_live && make_ctx(iw, 0, ic);
    auto issue_ahead = [&]() {
      if constexpr (kIn > 0) {
        while (it_live && seq_issued < seq_used + C::kInSlots) {
          if (ic_ok && Epi::has_input(ep, ic, it_c)) {
            const int slot = static_cast<int>(seq_issued % C::kInSlots);
            const uint32_t bar = in_bar(ew, slot);
            const uint32_t dst = in_base + slot * kIn * kInBoxBytes;
            mbar_arrive_expect_tx(bar, kIn * kInBoxBytes);
#pragma unroll
            for (int b = 0; b < InLoadsOf<Epi>::value; ++b) {
              int map, x, y;
              Epi::in_coord(ep, ic, it_c, b, map, x, y);
              if constexpr (kEpiEvictFirst)
                tma_load_2d_hint(dst + b * kInBoxBytes, map ? &tmI1 : &tmI0, bar, x, y, pol_stream);
              else
                tma_load_2d(dst + b * kInBoxBytes, map ? &tmI1 : &tmI0, bar, x, y);
            }
            ++seq_issued;
          }
          if (!ic_ok || ++it_c == kSegChunks) {
            it_c = 0;
            if (++it_s == item_segs(iw)) {
              it_s = 0;
              it_live = work_next(p, cluster_id, num_clusters, icur, iw);
            }
            ic_ok = it_live && make_ctx(iw, it_s, ic);
          }
        }
      }
    };
    if (lane == 0) issue_ahead();
    bool ok = true;
    typename Epi::Pre pa, pb;
    EpiCtx cx;
    // A stream-K piece that arrives first at its tile runs no epilogue: the
    // input boxes issued ahead for the unit are waited for and dropped, in the
    // order the ring issued them.
    auto skip_inputs = [&](const Work& wk) {
      if constexpr (kIn > 0) {
        for (int seg = 0; seg < item_segs(wk); ++seg) {
          EpiCtx sx;
          if (!make_ctx(wk, seg, sx)) break;
          for (int cs = 0; cs < kSegChunks; ++cs) {
            if (!Epi::has_input(ep, sx, cs)) continue;
            const int slot = static_cast<int>(seq_used % C::kInSlots);
            if (!wait_bounded(in_bar(ew, slot), (seq_used / C::kInSlots) & 1u, p, abort_flag)) ok = false;
            __syncwarp();
            ++seq_used;
            if (lane == 0) issue_ahead();
          }
        }
      }
    };

    WorkCursor ecur;
    work_begin(p, cluster_id, ecur);
    Work w;
    for (; ok && work_next(p, cluster_id, num_clusters, ecur, w); ++local) {
      const int buf = local & 1;
      const uint32_t tphase = static_cast<uint32_t>((local >> 1) & 1);
      if (!wait_bounded_sleep(tfull_bar(buf), tphase, p, abort_flag)) break;
      tc_fence_after();
      // A piece of a split tile runs the epilogue only as the second piece to
      // arrive, on the sum of both partials (two fp32 terms: the same sum
      // whichever piece is second). If the other piece has already arrived
      // (its arrival word shows one arrival of this launch) this one is
      // second and goes straight on; otherwise it stores this warp's partial
      // accumulator and counts its arrival, which tells it which it is.
      const float4* partner = nullptr;
      bool run = true;
      const long own_slot = w.side >= 0 ? sk_slot(kPair, w.bnd, w.side, q, ew) : 0;
      const long other_slot = w.side >= 0 ? sk_slot(kPair, w.bnd, 1 - w.side, q, ew) : 0;
      const int ctr_i = w.side >= 0 ? sk_counter(kPair, w.bnd, q, ew) : 0;
      if (w.side >= 0 && !(CODA_IN_ST(p.status, own_slot + 2047, p.sk_part_f4) &&
                           CODA_IN_ST(p.status, other_slot + 2047, p.sk_part_f4) &&
                           CODA_IN_ST(p.status, ctr_i, p.sk_ctr_n))) {
        run = false;  // checked build only: the tile is left unwritten, CODA_DEVST_BOUNDS is set
        skip_inputs(w);
      } else if (w.side >= 0) {
        unsigned* ctr = p.sk_ctr + ctr_i;
        unsigned seen = 0;
        if (lane == 0) seen = atomicAdd(ctr, 0u);
        seen = __shfl_sync(0xffffffffu, seen, 0);
        unsigned arrivals = 2;
        if (seen != ((p.sk_epoch << 2) | 1u)) {
          const uint32_t tb = tmem_base + (static_cast<uint32_t>(32 * ew) << 16) + static_cast<uint32_t>(buf * BN);
          float4* mine = p.sk_part + own_slot + lane;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float a[32];
            tmem_ld32(tb + 32 * c, a);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              mine[(c * 8 + v) * 32] = make_float4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) {
            arrivals = sk_arrive(ctr, p.sk_epoch);
            if (arrivals == 0) atomicOr(p.status, CODA_DEVST_SPLIT);
          }
          arrivals = __shfl_sync(0xffffffffu, arrivals, 0);
        }
        if (arrivals == 2) {
          __threadfence();
          partner = p.sk_part + other_slot + lane;
        } else {
          run = false;
          skip_inputs(w);
        }
      }
      // One loop over the item's 8 (or 4) chunks; partial statistics close and
      // reopen at the 128-column segment boundary (chunk 4). A segment that
      // starts past N ends the item (only the last column block can).
      const int nchunks = item_segs(w) * kSegChunks;
      // This CTA's last unit runs its epilogue exposed after the final MMA, and
      // with a single input slot in the ring (the two-box epilogues at long K)
      // each chunk would wait a full memory round trip. The mainloop stages are
      // idle by then (every load has landed and every MMA completed), so the
      // unit's input boxes not yet in the ring are all issued at once into
      // them, one barrier per chunk. Measured: the SwiGLU backward at
      // 4096x14336x4096 1.1 % faster; with a two-slot ring (K <= 3072) the same
      // was 0.5 % slower, so rings of two or more slots keep the ring.
      int in_idx = 0;           // input chunks of this unit consumed so far
      int last_from = 1 << 30;  // first input chunk taken from the stage memory
      const uint32_t last_base = s_base + static_cast<uint32_t>(ew * kLastWarpBytes);
      if constexpr (kIn > 0 && C::kInSlots == 1) {
        WorkCursor pc = ecur;
        Work nx;
        if (run && !work_next(p, cluster_id, num_clusters, pc, nx)) {
          const int n_ring = __shfl_sync(0xffffffffu, static_cast<int>(seq_issued - seq_used), 0);
          int n_in = 0;
          for (int seg = 0; seg < item_segs(w); ++seg) {
            EpiCtx sx;
            if (!make_ctx(w, seg, sx)) break;
            for (int cs = 0; cs < kSegChunks; ++cs) n_in += Epi::has_input(ep, sx, cs) ? 1 : 0;
          }
          if (n_in > n_ring) {
            last_from = n_ring;
            if (lane == 0) {
              it_live = false;  // the ring issues nothing more
              last_issued = n_in - n_ring;
              int j = 0;
              for (int seg = 0; seg < item_segs(w); ++seg) {
                EpiCtx sx;
                if (!make_ctx(w, seg, sx)) break;
                for (int cs = 0; cs < kSegChunks; ++cs) {
                  if (!Epi::has_input(ep, sx, cs)) continue;
                  if (j >= n_ring) {
                    const uint32_t dst = last_base + static_cast<uint32_t>((j - n_ring) * kIn * kInBoxBytes);
                    const uint32_t bar = last_bar(ew, j - n_ring);
                    mbar_arrive_expect_tx(bar, kIn * kInBoxBytes);
#pragma unroll
                    for (int b = 0; b < InLoadsOf<Epi>::value; ++b) {
                      int map, x, y;
                      Epi::in_coord(ep, sx, cs, b, map, x, y);
                      tma_load_2d_hint(dst + b * kInBoxBytes, map ? &tmI1 : &tmI0, bar, x, y, pol_stream);
                    }
                  }
                  ++j;
                }
              }
            }
          }
        }
      }
      if (run && make_ctx(w, 0, cx)) {
        typename Epi::State st;
        Epi::begin(st, ep, cx);
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * ew) << 16) + static_cast<uint32_t>(buf * BN);
        auto do_chunk = [&](int c, const typename Epi::Pre& pre) {
          const int cs = c & (kSegChunks - 1);  // chunk index inside its segment
          uint32_t in = 0;
          bool from_ring = false;
          if constexpr (kIn > 0) {
            if (Epi::has_input(ep, cx, cs)) {
              if (in_idx >= last_from) {
                if (!wait_bounded(last_bar(ew, in_idx - last_from), 0u, p, abort_flag)) ok = false;
                in = last_base + static_cast<uint32_t>((in_idx - last_from) * kIn * kInBoxBytes);
              } else {
                const int slot = static_cast<int>(seq_used % C::kInSlots);
                if (!wait_bounded(in_bar(ew, slot), (seq_used / C::kInSlots) & 1u, p, abort_flag)) ok = false;
                in = in_base + slot * kIn * kInBoxBytes;
                from_ring = true;
              }
              ++in_idx;
            }
          }
          float acc[32];
          tmem_ld32(tbase + 32 * c, acc);
          if (partner != nullptr) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 o = __ldcg(partner + (c * 8 + v) * 32);
              acc[4 * v] += o.x;
              acc[4 * v + 1] += o.y;
              acc[4 * v + 2] += o.z;
              acc[4 * v + 3] += o.w;
            }
          }
          if (p.k_blocks == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
          }
          if constexpr (kF8) {
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] *= p.alpha;
          }
          // this store step's boxes are contiguous: box k at box0 + k * kStageBoxBytes
          const uint32_t box0 = my_stage + (sbuf * kSlots) * kStageBoxBytes;
          const uint32_t box1 = box0 + kStageBoxBytes;
          if (nslots > 0 && (cs % Epi::kChunksPerStore) == 0) {
            // the staging buffer about to be written was last read by the store
            // group kStageBufs groups back
            if (lane == 0) bulk_wait_read<C::kStageBufs - 1>();
            __syncwarp();
          }
          Epi::chunk(st, ep, cx, cs, acc, pre, in, box0, box1);
          // One proxy fence and warp sync serve both hand-offs to TMA: every
          // lane's reads of the input slot happen before the copy that refills
          // it, and every lane's staging writes before the store that reads them.
          const bool store_step = nslots > 0 && (cs % Epi::kChunksPerStore) == Epi::kChunksPerStore - 1;
          if (in != 0 || store_step) {
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (store_step) {
            if (lane == 0) {
              for (int s = 0; s < nslots; ++s) {
                int map, x, y;
                Epi::store_coord(ep, cx, cs, s, map, x, y);
                if constexpr (kEpiEvictFirst)
                  tma_store_2d_hint(map ? &tmO1 : &tmO0, box0 + s * kStageBoxBytes, x, y, pol_stream);
                else
                  tma_store_2d(map ? &tmO1 : &tmO0, box0 + s * kStageBoxBytes, x, y);
              }
              bulk_commit();
            }
            if constexpr (C::kStageBufs == 2) sbuf ^= 1;
          }
          if constexpr (kIn > 0) {
            if (from_ring) {
              ++seq_used;
              if (lane == 0) issue_ahead();
            }
          }
        };
        // vector operands: chunk c+1's loads are issued before chunk c runs
        Epi::prefetch(ep, cx, 0, pa);
#pragma unroll 1
        for (int c = 0; c < nchunks; c += 2) {
          if (c == kSegChunks) {
            Epi::end(st, ep, cx);
            if (!make_ctx(w, 1, cx)) break;
            Epi::begin(st, ep, cx);
            Epi::prefetch(ep, cx, 0, pa);
          }
          Epi::prefetch(ep, cx, (c + 1) & (kSegChunks - 1), pb);
          do_chunk(c, pa);
          if (((c + 2) & (kSegChunks - 1)) != 0) Epi::prefetch(ep, cx, (c + 2) & (kSegChunks - 1), pa);
          do_chunk(c + 1, pb);
          if (c + 2 == nchunks) Epi::end(st, ep, cx);
        }
      }
      // accumulator buffer fully read: hand it back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kCG == 2)
          mbar_arrive_remote(mapa_shared(tempty_bar(buf), leader_rank));
        else
          mbar_arrive(tempty_bar(buf));
      }
    }
    if (lane == 0) {
      bulk_wait_all<0>();
      // input boxes still in flight (only after an abort) land before exit
      if constexpr (kIn > 0) {
        for (uint32_t q = seq_used; q < seq_issued; ++q)
          wait_drain(in_bar(ew, static_cast<int>(q % C::kInSlots)), (q / C::kInSlots) & 1u, p.timeout_ns);
        for (int j = 0; j < last_issued; ++j) wait_drain(last_bar(ew, j), 0u, p.timeout_ns);  // returns at once if waited
      }
    }
    __syncwarp();
  }

  __syncthreads();
  // In a pair, neither CTA releases TMEM (or its shared memory) while the
  // leader's MMAs may still read or write it.
  if constexpr (kCG == 2) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kCG == 2)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace coda
