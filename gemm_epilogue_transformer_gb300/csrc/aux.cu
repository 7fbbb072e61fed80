// Light auxiliary kernels: combine the tile partials written by the fused
// epilogues (pith page, Figure 4 caption: a small kernel reads a few partial
// values per tile instead of the full activation), plus the RoPE tables.
// All are HBM/latency bound; one warp per row, coalesced over the partials.
// They are launched with programmatic dependent launch (light_launch.cuh), so
// their launch and block scheduling overlap the tail of the GEMM before them.
#include "host.h"
#include "light_launch.cuh"

using namespace coda;

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// r[i] = 1 / sqrt(sum_t psq[i,t] / d + eps)   (pith page, Figure 5 caption)
__global__ void rms_reduce_kernel(int M, int nb, float inv_d, const float* __restrict__ psq, float eps,
                                  float* __restrict__ r) {
  light_kernel_enter();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < M; row += warps) {
    float s = 0.f;
    for (int t = lane; t < nb; t += 32) s += psq[static_cast<long>(row) * nb + t];
    s = warp_sum(s);
    if (lane == 0) r[row] = 1.0f / sqrtf(s * inv_d + eps);
  }
}

// s[i] = sum_t pdot[i,t] / d   (CODA note, Key design 3)
__global__ void rowdot_reduce_kernel(int M, int nb, float inv_d, const float* __restrict__ pdot,
                                     float* __restrict__ s_out) {
  light_kernel_enter();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < M; row += warps) {
    float s = 0.f;
    for (int t = lane; t < nb; t += 32) s += pdot[static_cast<long>(row) * nb + t];
    s = warp_sum(s);
    if (lane == 0) s_out[row] = s * inv_d;
  }
}

// Combine per-tile online-softmax states (CODA note, Key design 4):
// LSE = Mx + ln sum_t psum_t exp(pmax_t - Mx).
__global__ void ce_reduce_kernel(int M, int nb, const float* __restrict__ pmax, const float* __restrict__ psum,
                                 const int32_t* __restrict__ parg, const float* __restrict__ tgt,
                                 float* __restrict__ lse_out, float* __restrict__ loss_row,
                                 int32_t* __restrict__ argmax_out) {
  light_kernel_enter();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < M; row += warps) {
    const float* pm = pmax + static_cast<long>(row) * nb;
    const float* ps = psum + static_cast<long>(row) * nb;
    float mx = -INFINITY;
    for (int t = lane; t < nb; t += 32) mx = fmaxf(mx, pm[t]);
    mx = warp_max(mx);
    float s = 0.f;
    int first = 0x7fffffff;
    for (int t = lane; t < nb; t += 32) {
      const float m = pm[t];
      s += ps[t] * expf(m - mx);
      if (m == mx && t < first) first = t;
    }
    s = warp_sum(s);
    first = warp_min_i(first);
    if (lane == 0) {
      const float lse = mx + logf(s);
      if (lse_out) lse_out[row] = lse;
      if (loss_row) loss_row[row] = lse - tgt[row];
      if (argmax_out && parg) argmax_out[row] = parg[static_cast<long>(row) * nb + first];
    }
  }
}

// Deterministic mean of loss_row in one block (double accumulation).
__global__ void mean_kernel(int M, const float* __restrict__ v, float* __restrict__ out) {
  light_kernel_enter();
  __shared__ double sh[32];
  double acc = 0.0;
  for (int i = threadIdx.x; i < M; i += blockDim.x) acc += static_cast<double>(v[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    acc = (threadIdx.x < (blockDim.x >> 5)) ? sh[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (threadIdx.x == 0) out[0] = static_cast<float>(acc / M);
  }
}

// dgamma[j] = sum_b pdg[b, j]. A block owns a strip of 32 columns (one
// coalesced 128-byte segment per row); its 16 warps take interleaved rows,
// 8 independent loads in flight per lane, and combine their sums in shared
// memory in a fixed order (deterministic).
constexpr int kColsumWarps = 16;
__global__ void __launch_bounds__(kColsumWarps * 32) colsum_kernel(int rows, int d, const float* __restrict__ pdg,
                                                                   float* __restrict__ out) {
  light_kernel_enter();
  __shared__ float sh[kColsumWarps][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int j0 = blockIdx.x * 32; j0 < d; j0 += gridDim.x * 32) {
    const int j = j0 + lane;
    float s = 0.f;
    if (j < d) {
      int b = w;
      for (; b + 7 * kColsumWarps < rows; b += 8 * kColsumWarps) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldg(pdg + static_cast<long>(b + u * kColsumWarps) * d + j);
#pragma unroll
        for (int u = 0; u < 8; ++u) s += v[u];
      }
      for (; b < rows; b += kColsumWarps) s += __ldg(pdg + static_cast<long>(b) * d + j);
    }
    sh[w][lane] = s;
    __syncthreads();
    if (w == 0) {
      float t = 0.f;
#pragma unroll
      for (int q = 0; q < kColsumWarps; ++q) t += sh[q][lane];
      if (j < d) out[j] = t;
    }
    __syncthreads();
  }
}

// cos/sin(p * theta^(-2i/head_dim)) in fp64, rounded to fp32.
__global__ void rope_tables_kernel(int S, int half, int head_dim, double theta, float* __restrict__ c,
                                   float* __restrict__ s) {
  light_kernel_enter();
  const long n = static_cast<long>(S) * half;
  for (long k = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<long>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(k / half);
    const int i = static_cast<int>(k % half);
    const double ang = static_cast<double>(p) * pow(theta, -2.0 * i / head_dim);
    double sv, cv;
    sincos(ang, &sv, &cv);
    c[k] = static_cast<float>(cv);
    s[k] = static_cast<float>(sv);
  }
}

int row_grid(const DeviceInfo* di, int rows, int rows_per_block) {
  long g = (static_cast<long>(rows) + rows_per_block - 1) / rows_per_block;
  const long cap = static_cast<long>(di->sm_count) * 16;
  return static_cast<int>(g < cap ? (g > 0 ? g : 1) : cap);
}

int launched(cudaError_t e, const char* fn) {
  return e == cudaSuccess ? CODA_OK : fail_cuda(e, fn);
}

}  // namespace

extern "C" {

int coda_rms_reduce(int M, int nb, int d, const float* psq, float eps, float* r_out, coda_stream_t stream) {
  const char* fn = "coda_rms_reduce";
  CODA_REQUIRE(M >= 0 && nb >= 0 && d > 0, CODA_ERR_INVALID, "%s: bad dims M=%d nb=%d d=%d", fn, M, nb, d);
  CODA_REQUIRE(eps >= 0.f, CODA_ERR_INVALID, "%s: eps must be >= 0", fn);
  if (M == 0) return CODA_OK;
  CODA_REQUIRE(nb > 0, CODA_ERR_INVALID, "%s: nb must be positive", fn);
  CODA_REQ_PTR4(psq);
  CODA_REQ_PTR4(r_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  return launched(launch_light(rms_reduce_kernel, row_grid(di, M, 8), 256, 0, as_stream(stream), M, nb, 1.0f / d, psq,
                               eps, r_out), fn);
}

int coda_rowdot_reduce(int M, int nb, int d, const float* pdot, float* s_out, coda_stream_t stream) {
  const char* fn = "coda_rowdot_reduce";
  CODA_REQUIRE(M >= 0 && nb >= 0 && d > 0, CODA_ERR_INVALID, "%s: bad dims M=%d nb=%d d=%d", fn, M, nb, d);
  if (M == 0) return CODA_OK;
  CODA_REQUIRE(nb > 0, CODA_ERR_INVALID, "%s: nb must be positive", fn);
  CODA_REQ_PTR4(pdot);
  CODA_REQ_PTR4(s_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  return launched(launch_light(rowdot_reduce_kernel, row_grid(di, M, 8), 256, 0, as_stream(stream), M, nb, 1.0f / d,
                               pdot, s_out), fn);
}

int coda_ce_reduce(int M, int nb, const float* pmax, const float* psum, const int32_t* parg, const float* tgt,
                   float* lse_out, float* loss_row_out, float* loss_mean_out, int32_t* argmax_out,
                   coda_stream_t stream) {
  const char* fn = "coda_ce_reduce";
  CODA_REQUIRE(M >= 0 && nb >= 0, CODA_ERR_INVALID, "%s: bad dims M=%d nb=%d", fn, M, nb);
  if (M == 0) return CODA_OK;
  CODA_REQUIRE(nb > 0, CODA_ERR_INVALID, "%s: nb must be positive", fn);
  CODA_REQ_PTR4(pmax);
  CODA_REQ_PTR4(psum);
  CODA_REQ_PTR4(tgt);
  CODA_REQ_PTR4(lse_out);
  CODA_REQ_PTR4(loss_row_out);
  CODA_REQ_OPT4(loss_mean_out);
  CODA_REQ_OPT4(parg);
  CODA_REQ_OPT4(argmax_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  int rc = launched(launch_light(ce_reduce_kernel, row_grid(di, M, 8), 256, 0, st, M, nb, pmax, psum, parg, tgt,
                                 lse_out, loss_row_out, argmax_out), fn);
  if (rc || !loss_mean_out) return rc;
  return launched(launch_light(mean_kernel, 1, 1024, 0, st, M, loss_row_out, loss_mean_out), fn);
}

int coda_colsum_reduce(int rows, int d, const float* pdg, float* dgamma_out, coda_stream_t stream) {
  const char* fn = "coda_colsum_reduce";
  CODA_REQUIRE(rows >= 0 && d >= 0, CODA_ERR_INVALID, "%s: bad dims rows=%d d=%d", fn, rows, d);
  if (d == 0) return CODA_OK;
  CODA_REQ_PTR4(dgamma_out);
  if (rows > 0) CODA_REQ_PTR4(pdg);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const int strips = (d + 31) / 32;
  const int grid = strips < di->sm_count * 4 ? strips : di->sm_count * 4;
  return launched(launch_light(colsum_kernel, grid, kColsumWarps * 32, 0, as_stream(stream), rows, d, pdg, dgamma_out),
                  fn);
}

int coda_rope_tables(int S, int head_dim, double theta, float* cos_out, float* sin_out, coda_stream_t stream) {
  const char* fn = "coda_rope_tables";
  CODA_REQUIRE(S >= 0 && head_dim > 0 && head_dim % 2 == 0, CODA_ERR_INVALID,
               "%s: S=%d must be >= 0 and head_dim=%d positive and even", fn, S, head_dim);
  CODA_REQUIRE(theta > 0.0, CODA_ERR_INVALID, "%s: theta must be positive", fn);
  if (S == 0) return CODA_OK;
  CODA_REQ_PTR4(cos_out);
  CODA_REQ_PTR4(sin_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const int half = head_dim / 2;
  return launched(launch_light(rope_tables_kernel, row_grid(di, S * half, 256), 256, 0, as_stream(stream), S, half,
                               head_dim, theta, cos_out, sin_out), fn);
}

}  // extern "C"
