// Launch template for the fused GEMM kernels: builds the operand tensor maps,
// the tile grid, and launches one persistent CTA per SM (or per tile when
// there are fewer tiles than SMs).
#pragma once

#include <string.h>

#include "epilogues.cuh"
#include "host.h"

namespace coda {

constexpr int kGroupM = 16;  // row blocks per raster group

// Output map for a TMA store target: row-major bf16 [rows, cols], leading
// dimension ld (elements), 32 x 32 boxes with the 64-byte swizzle.
inline int make_out_map(CUtensorMap* m, const void* base, int rows, int cols, int ld) {
  return make_map_bf16(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                       static_cast<uint64_t>(ld) * 2u, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

template <class Epi>
int launch_fused(const char* fn, int M, int N, int K, const void* A, int lda, int a_mn, const void* B, int ldb,
                 int b_mn, const CUtensorMap& o0, const CUtensorMap& o1, const typename Epi::Params& ep,
                 cudaStream_t stream) {
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  CUtensorMap tA, tB;
  memset(&tA, 0, sizeof(tA));
  memset(&tB, 0, sizeof(tB));
  int rc;
  if (K > 0) {
    rc = a_mn ? make_map_bf16(&tA, A, M, K, static_cast<uint64_t>(lda) * 2u, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)
              : make_map_bf16(&tA, A, K, M, static_cast<uint64_t>(lda) * 2u, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = b_mn ? make_map_bf16(&tB, B, N, K, static_cast<uint64_t>(ldb) * 2u, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)
              : make_map_bf16(&tB, B, K, N, static_cast<uint64_t>(ldb) * 2u, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  GemmShape p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.a_mn = a_mn;
  p.b_mn = b_mn;
  p.m_blocks = (M + BM - 1) / BM;
  p.n_blocks = (N + BN - 1) / BN;
  p.k_blocks = (K + BK - 1) / BK;
  p.num_tiles = p.m_blocks * p.n_blocks;
  p.group_m = p.m_blocks < kGroupM ? p.m_blocks : kGroupM;
  p.status = di->status;
  p.timeout_ns = wait_timeout_ns();

  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&gemm_epilogue_kernel<Epi>),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(max dynamic shared memory)");
    attr_done[dev] = 1;
  }
  const int grid = p.num_tiles < di->sm_count ? p.num_tiles : di->sm_count;
  gemm_epilogue_kernel<Epi><<<grid, kThreads, kSmemBytes, stream>>>(tA, tB, o0, o1, p, ep);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, fn);
  return CODA_OK;
}

}  // namespace coda
