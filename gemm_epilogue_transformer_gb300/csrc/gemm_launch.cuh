// Launch template for the fused GEMM kernels: builds the operand tensor maps,
// the tile grid, and launches one persistent CTA per SM (or per tile when
// there are fewer tiles than SMs).
#pragma once

#include <string.h>

#include <atomic>

#include "epilogues.cuh"
#include "host.h"

namespace coda {

// Two-box input epilogues keep two chunks of inputs in flight (a larger ring,
// one mainloop stage less) when K is at most this: a mainloop that short
// cannot hide one HBM round trip per chunk.
constexpr int kDeepRingMaxK = 3072;

// Stream-K split: only with at least this many k-blocks per tile (shorter
// reductions gain little next to the partials' round trip).
constexpr int kStreamKMinKBlocks = 16;
// Whether the stream-K split is expected to beat the data-parallel schedule.
// The latter's last wave costs a full tile time, or about 0.6 of one when it
// runs as half tiles; the split costs rem / clusters of a tile time plus a
// fixed overhead (the partials' round trip through L2 and the extra epilogue
// passes of split tiles), measured on GB300 at 0.2-0.45 tile times for
// 64 k-block tiles and near zero for 128-192 k-blocks: about 28 k-blocks.
constexpr int kStreamKOverheadKBlocks = 28;
inline bool stream_k_pays(int rem, int clusters, int N, int k_blocks) {
  const double frac = static_cast<double>(rem) / clusters;
  const double dp_tail = (2 * rem <= clusters && N > BSEG) ? 0.6 : 1.0;
  return (dp_tail - frac) * k_blocks >= kStreamKOverheadKBlocks;
}

// Output map for a TMA store target: row-major bf16 [rows, cols], leading
// dimension ld (elements), 32 x 32 boxes with the 64-byte swizzle.
inline int make_out_map(CUtensorMap* m, const void* base, int rows, int cols, int ld) {
  return make_map_bf16(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                       static_cast<uint64_t>(ld) * 2u, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// A map of 32 x 64-element (128-byte) boxes with the 128-byte swizzle over a
// row-major bf16 [rows, cols] tensor: the SwiGLU backward's pre-activation
// input and its interleaved gradient output, 64 columns per chunk.
inline int make_wide_map(CUtensorMap* m, const void* base, int rows, int cols, int ld) {
  return make_map_bf16(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                       static_cast<uint64_t>(ld) * 2u, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Checks shared by the fused bf16 entry points: non-negative dims, 8-element
// granularity of N and K (16-byte rows), aligned operand pointers.
inline int check_fused(const char* fn, int M, int N, int K, const void* A, const void* B) {
  CODA_REQUIRE(M >= 0 && N >= 0 && K >= 0, CODA_ERR_INVALID, "%s: negative dimension (M=%d N=%d K=%d)", fn, M, N, K);
  CODA_REQUIRE(N % 8 == 0 && K % 8 == 0, CODA_ERR_UNSUPPORTED, "%s: N=%d and K=%d must be multiples of 8", fn, N, K);
  if (M > 0 && N > 0 && K > 0) {
    CODA_REQ_PTR16(A);
    CODA_REQ_PTR16(B);
  }
  return CODA_OK;
}

// The RoPE epilogue forms a warp's cos/sin values by angle addition from table
// rows 0..31 (kept in shared memory) and the warp's first position when S is a
// multiple of 32 (a warp's 32 rows never wrap) and a table row fits 256 bytes
// (head_dim <= 128); otherwise every row loads its own values.
inline int rope_lane_tables(int S, int head_dim) { return (S % 32 == 0 && head_dim <= 128) ? 1 : 0; }

// kF8: E4M3 operands, K-major only (A [M, K], B stored [N, K], lda / ldb in
// bytes = elements), 128-element K stages, accumulator scaled by alpha.
template <class Epi, int kCG, bool kF8 = false>
int launch_variant(const char* fn, const DeviceInfo* di, int M, int N, int K, const void* A, int lda, int a_mn,
                   const void* B, int ldb, int b_mn, const CUtensorMap& o0, const CUtensorMap& o1,
                   const CUtensorMap& i0, const CUtensorMap& i1, const typename Epi::Params& ep,
                   cudaStream_t stream, float alpha = 1.0f) {
  using C = CfgOf<Epi, kCG>;
  CUtensorMap tA, tB;
  memset(&tA, 0, sizeof(tA));
  memset(&tB, 0, sizeof(tB));
  int rc;
  // An MN-major operand whose MN extent is a multiple of 64 is read with one
  // 3-D box per stage (mode 2) instead of one 2-D box per 64 columns (mode 1).
  if (a_mn && M % 64 == 0) a_mn = 2;
  if (b_mn && N % 64 == 0) b_mn = 2;
  if (kF8 && K > 0) {
    if (a_mn || b_mn) return fail(CODA_ERR_UNSUPPORTED, "%s: FP8 operands must be K-major", fn);
    rc = make_map_u8(&tA, A, K, M, static_cast<uint64_t>(lda), 2 * BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = make_map_u8(&tB, B, K, N, static_cast<uint64_t>(ldb), 2 * BK, C::kBLoad, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  } else if (K > 0) {
    if (a_mn == 2)
      rc = make_map_bf16_mn3d(&tA, A, M, K, static_cast<uint64_t>(lda) * 2u, BM / 64);
    else if (a_mn)
      rc = make_map_bf16(&tA, A, M, K, static_cast<uint64_t>(lda) * 2u, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    else
      rc = make_map_bf16(&tA, A, K, M, static_cast<uint64_t>(lda) * 2u, 64, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    if (b_mn == 2)
      rc = make_map_bf16_mn3d(&tB, B, N, K, static_cast<uint64_t>(ldb) * 2u, C::kBLoad / 64);
    else if (b_mn)
      rc = make_map_bf16(&tB, B, N, K, static_cast<uint64_t>(ldb) * 2u, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    else
      rc = make_map_bf16(&tB, B, K, N, static_cast<uint64_t>(ldb) * 2u, 64, C::kBLoad, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  auto kernel = &gemm_epilogue_kernel<Epi, kCG, kF8>;
  static std::atomic<int> max_clusters[64] = {};  // per device; 0 = not yet queried (any thread may fill it)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return fail(CODA_ERR_INVALID, "%s: device index %d", fn, dev);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!max_clusters[dev]) {
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(max dynamic shared memory)");
    int n = 0;
    cfg.gridDim = dim3(kCG, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = di->sm_count / kCG;
    }
    max_clusters[dev] = n;
  }
  const int cmax = max_clusters[dev];

  GemmShape p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.a_mn = a_mn;
  p.b_mn = b_mn;
  p.m_blocks = (M + C::kTileM - 1) / C::kTileM;
  p.n_blocks = (N + BN - 1) / BN;
  p.k_blocks = kF8 ? (K + 2 * BK - 1) / (2 * BK) : (K + BK - 1) / BK;
  p.num_tiles = p.m_blocks * p.n_blocks;
  // Raster group: the row blocks that sweep all column blocks together (tile
  // order in tile_coords). B is read from DRAM once per group when it does not
  // fit in L2, so a group of 4096 rows halves that traffic against 2048 rows;
  // it is used when B exceeds half of L2 and the group's A rows (4096 x K)
  // still fit in a third of it.
  {
    const double eb = kF8 ? 1.0 : 2.0, l2 = static_cast<double>(di->l2_bytes);
    const bool wide = static_cast<double>(K) * N * eb > 0.5 * l2 && 4096.0 * K * eb <= l2 / 3.0;
    const int gm = (wide ? 4096 : 2048) / C::kTileM;
    p.group_m = p.m_blocks < gm ? p.m_blocks : gm;
  }
  p.seg_blocks = (N + BSEG - 1) / BSEG;
  // Wave balance. With `rem` tiles past the last full wave of the persistent
  // clusters, either one wave and those tiles run as stream-K work (their
  // k-blocks dealt out evenly, ahead of the data-parallel tiles: every
  // cluster ends together, at the cost of one partial-accumulator round trip
  // through L2 per split tile), or, without it, a last wave of at most half
  // the clusters runs as 2 * rem half tiles (256 x 128 per pair).
  const int rem = p.num_tiles % cmax;
  p.dp_first = 0;
  p.sk_tiles = p.sk_q = p.sk_r = p.sk_rotate = 0;
  p.sk_part = nullptr;
  p.sk_ctr = nullptr;
  p.sk_part_f4 = 0;
  p.sk_ctr_n = 0;
  p.sk_epoch = 0;
  const int skm = stream_k_setting();
  if (rem > 0 && cmax >= 2 && p.num_tiles >= cmax + rem && p.k_blocks >= kStreamKMinKBlocks &&
      (skm == 2 || (skm == 1 && stream_k_pays(rem, cmax, N, p.k_blocks)))) {
    SkWorkspace ws;
    if (sk_workspace(di, dev, stream, &ws)) {
      p.sk_tiles = cmax + rem;
      p.dp_first = p.sk_tiles;
      const long long total = static_cast<long long>(p.sk_tiles) * p.k_blocks;
      p.sk_q = static_cast<int>(total / cmax);
      p.sk_r = static_cast<int>(total % cmax);
      p.sk_part = static_cast<float4*>(ws.part);
      p.sk_ctr = ws.ctr;
      p.sk_part_f4 = static_cast<long>(sk_part_bytes(di->sm_count) / sizeof(float4));
      p.sk_ctr_n = sk_ctr_words(di->sm_count);
      p.sk_epoch = ws.epoch;
      // Walk the ranges in step (see WorkCursor) when the stream-K tiles'
      // operands, spread over all of K, would take more than half of L2: the
      // distinct row and column blocks of raster tiles 0 .. sk_tiles-1.
      const int gm = p.group_m;
      const int cols_b = (p.sk_tiles + gm - 1) / gm < p.n_blocks ? (p.sk_tiles + gm - 1) / gm : p.n_blocks;
      const int rows_need = (p.sk_tiles + cols_b - 1) / cols_b;
      const int rows_b = rows_need < p.m_blocks ? rows_need : p.m_blocks;
      const double ws_bytes = (static_cast<double>(rows_b) * C::kTileM + static_cast<double>(cols_b) * BN) *
                              static_cast<double>(p.k_blocks) * (kF8 ? 2 * BK : BK) * (kF8 ? 1.0 : 2.0);
      p.sk_rotate = ws_bytes > 0.5 * static_cast<double>(di->l2_bytes) ? 1 : 0;
    }
  }
  if (p.sk_tiles > 0) {
    p.full_items = p.num_items = p.num_tiles - p.sk_tiles;
  } else if (rem > 0 && 2 * rem <= cmax && N > BSEG) {
    p.full_items = p.num_tiles - rem;
    p.num_items = p.num_tiles + rem;
  } else {
    p.full_items = p.num_tiles;
    p.num_items = p.num_tiles;
  }
  p.status = di->status;
  p.timeout_ns = wait_timeout_ns();
  p.inject = take_injected_fault();
  p.alpha = alpha;

  const int clusters = p.sk_tiles > 0 ? cmax : (p.num_items < cmax ? p.num_items : cmax);
  cfg.gridDim = dim3(clusters * kCG, 1, 1);
  // Programmatic dependent launch: the grid may be scheduled while the previous
  // kernel of the stream drains; the kernel waits for it before any global
  // access (griddep_wait), so only launch latency and the prologue overlap.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tA, tB, o0, o1, i0, i1, p, ep);
  if (e != cudaSuccess) return fail_cuda(e, fn);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, fn);
  return CODA_OK;
}

// One persistent CTA (kCG = 1) or CTA pair (kCG = 2) per SM / SM pair. The
// pair variant is used once M spans more than one 128-row block, unless
// coda_set_cta_group() fixed the choice.
// o0 / o1: TMA store targets; i0 / i1: TMA sources of the epilogue's input
// boxes (unused maps may be any valid map).
template <class Epi, bool kF8 = false>
int launch_fused(const char* fn, int M, int N, int K, const void* A, int lda, int a_mn, const void* B, int ldb,
                 int b_mn, const CUtensorMap& o0, const CUtensorMap& o1, const CUtensorMap& i0,
                 const CUtensorMap& i1, const typename Epi::Params& ep, cudaStream_t stream, float alpha = 1.0f) {
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const int forced = cta_group_setting();
  const int g = forced ? forced : (M > BM ? 2 : 1);
  if (g == 2)
    return launch_variant<Epi, 2, kF8>(fn, di, M, N, K, A, lda, a_mn, B, ldb, b_mn, o0, o1, i0, i1, ep, stream,
                                       alpha);
  return launch_variant<Epi, 1, kF8>(fn, di, M, N, K, A, lda, a_mn, B, ldb, b_mn, o0, o1, i0, i1, ep, stream, alpha);
}

}  // namespace coda
