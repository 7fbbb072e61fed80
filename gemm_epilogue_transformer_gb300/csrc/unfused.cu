// Unfused comparison path: the memory-bound operators that CODA folds into GEMM
// epilogues, as stand-alone kernels that read and write every intermediate
// through HBM (CODA note, research background). 16-byte vector accesses,
// grid-stride loops sized to the SM count, fp32 arithmetic, bf16 storage.
#include <cuda_bf16.h>

#include <atomic>

#include "host.h"

using namespace coda;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float exp_f(float x) { return exp2f(x * kLog2e); }

__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}
__device__ __forceinline__ uint4 ld16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void st16(void* p, const uint4& v) { *reinterpret_cast<uint4*>(p) = v; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Block-wide sum (blockDim multiple of 32); every thread gets the result.
__device__ float block_sum(float v, float* sh) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = (l < nw) ? sh[l] : 0.f;
  v = warp_sum(v);
  __syncthreads();
  return v;
}

// Blocks for a one-item-per-step grid-stride kernel: up to 8 per SM (2048
// threads of 256).
int grid_for(const DeviceInfo* di, long work_items, int block) {
  long g = (work_items + block - 1) / block;
  const long cap = static_cast<long>(di->sm_count) * 8;
  if (g < 1) g = 1;
  return static_cast<int>(g < cap ? g : cap);
}

// Blocks for a grid-stride kernel: as many as the SMs hold at once (the SM
// count times the kernel's occupancy, queried once per call site into
// per_sm), so every block runs from the start and the equal per-thread shares
// end together; fewer when the work is smaller.
template <class Kern>
int grid_resident(const DeviceInfo* di, Kern kernel, std::atomic<int>& per_sm, long work_items, int block) {
  int n = per_sm.load();
  if (n <= 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, 0) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 2;
    }
    per_sm.store(n);
  }
  long g = (work_items + block - 1) / block;
  const long cap = static_cast<long>(di->sm_count) * n;
  if (g < 1) g = 1;
  return static_cast<int>(g < cap ? g : cap);
}

int launched(const char* fn) {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CODA_OK : fail_cuda(e, fn);
}

#define GRID_STRIDE(i, n) \
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < (n); i += static_cast<long>(gridDim.x) * blockDim.x)

// Grid-stride over n items, kUnroll per step: a thread takes items i0 + j *
// stride (j < kUnroll) and issues the loads of all of them before it computes
// or stores any, so each thread has kUnroll 16-byte loads (per input) in
// flight instead of one. Per element the arithmetic is the same as one item
// at a time.
constexpr int kUnroll = 4;
#define GRID_STRIDE_STEP(i0, stride, n)                                 \
  const long stride = static_cast<long>(gridDim.x) * blockDim.x;        \
  for (long i0 = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i0 < (n); i0 += stride * kUnroll)

__global__ void add_kernel(long nvec, const uint4* a, const uint4* b, uint4* out) {
  GRID_STRIDE_STEP(i0, stride, nvec) {
    uint4 ra[kUnroll], rb[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const long i = i0 + j * stride;
      if (i < nvec) {
        ra[j] = __ldg(a + i);
        rb[j] = __ldg(b + i);
      }
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const long i = i0 + j * stride;
      if (i < nvec) {
        float x[8], y[8];
        unpack8(ra[j], x);
        unpack8(rb[j], y);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] += y[k];
        out[i] = pack8(x);
      }
    }
  }
}

// One block per row (grid-stride over rows): r = 1/sqrt(mean h^2 + eps),
// n = r h gamma. With kVec > 0 (d <= 8 * kVec * blockDim) a thread keeps its
// kVec vectors of the row in registers between the two passes, all loaded at
// once; with kVec = 0 it loops over the row twice (any width).
template <int kVec>
__global__ void rmsnorm_kernel(int M, int d, const __nv_bfloat16* h, const __nv_bfloat16* gamma, float eps,
                               __nv_bfloat16* n, float* r_out) {
  __shared__ float sh[32];
  const int nv = d / 8;
  for (int row = blockIdx.x; row < M; row += gridDim.x) {
    const __nv_bfloat16* hr = h + static_cast<long>(row) * d;
    __nv_bfloat16* nr = n + static_cast<long>(row) * d;
    float ss = 0.f;
    if constexpr (kVec > 0) {
      uint4 raw[kVec];
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        const int v = threadIdx.x + j * blockDim.x;
        if (v < nv) raw[j] = ld16(hr + 8 * v);
      }
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        if (threadIdx.x + j * blockDim.x < nv) {
          float x[8];
          unpack8(raw[j], x);
#pragma unroll
          for (int k = 0; k < 8; ++k) ss = fmaf(x[k], x[k], ss);
        }
      }
      ss = block_sum(ss, sh);
      const float r = 1.0f / sqrtf(ss / d + eps);
      if (threadIdx.x == 0 && r_out) r_out[row] = r;
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        const int v = threadIdx.x + j * blockDim.x;
        if (v < nv) {
          float x[8], g[8];
          unpack8(raw[j], x);
          unpack8(ld16(gamma + 8 * v), g);
#pragma unroll
          for (int k = 0; k < 8; ++k) x[k] = (x[k] * r) * g[k];
          st16(nr + 8 * v, pack8(x));
        }
      }
    } else {
      for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float x[8];
        unpack8(ld16(hr + 8 * v), x);
#pragma unroll
        for (int k = 0; k < 8; ++k) ss = fmaf(x[k], x[k], ss);
      }
      ss = block_sum(ss, sh);
      const float r = 1.0f / sqrtf(ss / d + eps);
      if (threadIdx.x == 0 && r_out) r_out[row] = r;
      for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float x[8], g[8];
        unpack8(ld16(hr + 8 * v), x);
        unpack8(ld16(gamma + 8 * v), g);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = (x[k] * r) * g[k];
        st16(nr + 8 * v, pack8(x));
      }
    }
  }
}

__global__ void rowscale_kernel(int M, int N, const __nv_bfloat16* x, const float* r, __nv_bfloat16* out) {
  const long nvr = N / 8;
  GRID_STRIDE(i, static_cast<long>(M) * nvr) {
    const float s = r[i / nvr];
    float v[8];
    unpack8(ld16(x + 8 * i), v);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] *= s;
    st16(out + 8 * i, pack8(v));
  }
}

// Each item: 8 outputs from 16 interleaved gate/up values.
__global__ void swiglu_kernel(long nitems, const __nv_bfloat16* gu, __nv_bfloat16* a) {
  GRID_STRIDE_STEP(i0, stride, nitems) {
    uint4 rp[kUnroll], rq[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const long i = i0 + j * stride;
      if (i < nitems) {
        rp[j] = ld16(gu + 16 * i);
        rq[j] = ld16(gu + 16 * i + 8);
      }
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const long i = i0 + j * stride;
      if (i < nitems) {
        float p[8], q[8], o[8];
        unpack8(rp[j], p);
        unpack8(rq[j], q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          o[k] = p[2 * k] / (1.0f + exp_f(-p[2 * k])) * p[2 * k + 1];
          o[k + 4] = q[2 * k] / (1.0f + exp_f(-q[2 * k])) * q[2 * k + 1];
        }
        st16(a + 8 * i, pack8(o));
      }
    }
  }
}

__global__ void swiglu_bwd_kernel(long nitems, const __nv_bfloat16* dA, const __nv_bfloat16* gu,
                                  __nv_bfloat16* dgu) {
  GRID_STRIDE_STEP(i0, stride, nitems) {
    uint4 rd[kUnroll], rg[kUnroll][2];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const long i = i0 + j * stride;
      if (i < nitems) {
        rd[j] = ld16(dA + 8 * i);
        rg[j][0] = ld16(gu + 16 * i);
        rg[j][1] = ld16(gu + 16 * i + 8);
      }
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const long i = i0 + j * stride;
      if (i < nitems) {
        float da[8];
        unpack8(rd[j], da);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float g[8], o[8];
          unpack8(rg[j][h], g);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float G = g[2 * k], U = g[2 * k + 1], d = da[4 * h + k];
            const float s = 1.0f / (1.0f + exp_f(-G));
            o[2 * k] = d * U * s * (1.0f + G * (1.0f - s));
            o[2 * k + 1] = d * G * s;
          }
          st16(dgu + 16 * i + 8 * h, pack8(o));
        }
      }
    }
  }
}

// In-place rotation of 4 pairs per item; kSign = +1 forward, -1 transposed.
template <int kSign>
__global__ void rope_kernel(int M, int N, const float* ct, const float* st, int S, int head_dim, int rope_cols,
                            __nv_bfloat16* x) {
  const long nvr = rope_cols / 8;
  const int half = head_dim / 2;
  GRID_STRIDE(i, static_cast<long>(M) * nvr) {
    const int row = static_cast<int>(i / nvr);
    const int c0 = static_cast<int>(i % nvr) * 8;
    const int pos = row % S;
    const int i0 = (c0 % head_dim) / 2;
    __nv_bfloat16* p = x + static_cast<long>(row) * N + c0;
    const float4 cs = __ldg(reinterpret_cast<const float4*>(ct + static_cast<long>(pos) * half + i0));
    const float4 sn = __ldg(reinterpret_cast<const float4*>(st + static_cast<long>(pos) * half + i0));
    const float c[4] = {cs.x, cs.y, cs.z, cs.w};
    const float s[4] = {sn.x, sn.y, sn.z, sn.w};
    float v[8];
    unpack8(*reinterpret_cast<const uint4*>(p), v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float e = v[2 * k], o = v[2 * k + 1], sk = kSign > 0 ? s[k] : -s[k];
      v[2 * k] = e * c[k] - o * sk;
      v[2 * k + 1] = e * sk + o * c[k];
    }
    st16(p, pack8(v));
  }
}

// One warp per row (grid-stride over rows): online max / sum-exp, argmax
// (lowest index), target. Each lane loads kCeBatch 16-byte vectors of the row
// before it uses any of them, so a warp keeps 4 KiB in flight, and rescales its
// running sum once per batch of 64 values.
constexpr int kCeBatch = 8;
__global__ void ce_fwd_kernel(int M, int V, const __nv_bfloat16* logits, const int32_t* labels, float* lse_out,
                              float* loss_row, int32_t* argmax_out, int* status) {
  const int lane = threadIdx.x & 31;
  const int nv = V / 8;
  const long nwarps = static_cast<long>(gridDim.x) * (blockDim.x >> 5);
  for (long row = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < M;
       row += nwarps) {
    const __nv_bfloat16* lr = logits + row * V;
    float m = -INFINITY, s = 0.f;
    int bi = 0x7fffffff;
    for (int v0 = lane; v0 < nv; v0 += 32 * kCeBatch) {
      uint4 raw[kCeBatch];
#pragma unroll
      for (int j = 0; j < kCeBatch; ++j) {
        const int v = v0 + 32 * j;
        raw[j] = v < nv ? ld16(lr + 8L * v) : make_uint4(0, 0, 0, 0);
      }
      // batch maximum; vectors and their elements in increasing column order,
      // so the first occurrence of the maximum is kept
      float cm = -INFINITY;
      int ci = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < kCeBatch; ++j) {
        if (v0 + 32 * j < nv) {
          float x[8];
          unpack8(raw[j], x);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (x[k] > cm) {
              cm = x[k];
              ci = 8 * (v0 + 32 * j) + k;
            }
        }
      }
      if (cm > m) bi = ci;
      const float nm = fmaxf(m, cm);
      float add = 0.f;
#pragma unroll
      for (int j = 0; j < kCeBatch; ++j) {
        if (v0 + 32 * j < nv) {
          float x[8];
          unpack8(raw[j], x);
#pragma unroll
          for (int k = 0; k < 8; ++k) add += exp_f(x[k] - nm);
        }
      }
      s = s * exp_f(m - nm) + add;
      m = nm;
    }
    // warp combine (m, s, bi); a lane that saw no column has m = -inf, s = 0
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const int b2 = __shfl_xor_sync(0xffffffffu, bi, o);
      const float nm = fmaxf(m, m2);
      const float a1 = (m == -INFINITY) ? 0.f : s * exp_f(m - nm);
      const float a2 = (m2 == -INFINITY) ? 0.f : s2 * exp_f(m2 - nm);
      if (m2 > m || (m2 == m && b2 < bi)) bi = b2;
      s = a1 + a2;
      m = nm;
    }
    if (lane == 0) {
      const float lse = m + logf(s);
      const int y = labels[row];
      float t;
      if (y < 0 || y >= V) {
        atomicOr(status, CODA_DEVST_BAD_LABEL);
        t = __uint_as_float(0x7fc00000u);
      } else {
        t = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(lr)[y]) << 16);
      }
      lse_out[row] = lse;
      loss_row[row] = lse - t;
      if (argmax_out) argmax_out[row] = bi;
    }
  }
}

__global__ void ce_mean_kernel(int M, const float* v, float* out) {
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

__global__ void ce_bwd_kernel(int M, int V, const __nv_bfloat16* logits, const int32_t* labels, const float* lse,
                              float g, __nv_bfloat16* dl) {
  const long nvr = V / 8;
  GRID_STRIDE(i, static_cast<long>(M) * nvr) {
    const int row = static_cast<int>(i / nvr);
    const int c0 = static_cast<int>(i % nvr) * 8;
    const float L = lse[row];
    const int y = labels[row];
    float x[8];
    unpack8(ld16(logits + 8 * i), x);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float p = exp_f(x[k] - L);
      if (c0 + k == y) p -= 1.0f;
      x[k] = g * p;
    }
    st16(dl + 8 * i, pack8(x));
  }
}

__global__ void rowdot_kernel(int M, int N, float inv_d, const __nv_bfloat16* dY, const __nv_bfloat16* Y,
                              float* s_out) {
  __shared__ float sh[32];
  const int nv = N / 8;
  for (int row = blockIdx.x; row < M; row += gridDim.x) {
    float acc = 0.f;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      float a[8], b[8];
      unpack8(ld16(dY + static_cast<long>(row) * N + 8 * v), a);
      unpack8(ld16(Y + static_cast<long>(row) * N + 8 * v), b);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = fmaf(a[k], b[k], acc);
    }
    acc = block_sum(acc, sh);
    if (threadIdx.x == 0) s_out[row] = acc * inv_d;
  }
}

// One block of kRbThreads per 32-row tile (the partials' row blocks), its rows
// in four groups of kRbGroup. For a group, two warps per row form
// c = (1/d) sum G gamma h with kRowBatch vectors of G and of h in flight per
// thread; then each thread takes its kOwn column vectors through the group's
// rows, kPair2 at a time (read back from L2, where phase one just brought them),
// writing dh = r gamma G - r^3 c h and accumulating the column partials of
// r G h in registers. Covers d <= 8 * kRbThreads * kOwn.
constexpr int kRbThreads = 512;
constexpr int kRbGroup = 8;
constexpr int kRowBatch = 4;
template <int kOwn, int kPair2 = (kOwn >= 4 ? 1 : 2)>
__global__ void __launch_bounds__(kRbThreads) rmsnorm_bwd_kernel(int M, int d, const __nv_bfloat16* G,
                                                                 const __nv_bfloat16* h,
                                                                 const __nv_bfloat16* gamma, const float* r,
                                                                 __nv_bfloat16* dh, float* pdg) {
  __shared__ float part[2][kRbGroup][2];
  const int nv = d / 8;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grow = w >> 1;              // the group row this warp reduces
  const int q = ((w & 1) << 5) | lane;  // this thread's place among the row's 64
  const int r0 = blockIdx.x * 32;
  float acc[kOwn][8];
#pragma unroll
  for (int o = 0; o < kOwn; ++o)
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[o][k] = 0.f;
#pragma unroll 1
  for (int g = 0; g < 32 / kRbGroup; ++g) {
    const int gr0 = r0 + g * kRbGroup;
    if (gr0 >= M) break;  // the same for every thread of the block
    // phase one: the group's row statistics
    const int row = gr0 + grow;
    float c = 0.f;
    if (row < M) {
      const long off = static_cast<long>(row) * d;
      for (int v0 = q; v0 < nv; v0 += 64 * kRowBatch) {
        uint4 ga[kRowBatch], ha[kRowBatch];
#pragma unroll
        for (int j = 0; j < kRowBatch; ++j) {
          const int v = v0 + 64 * j;
          if (v < nv) {
            ga[j] = ld16(G + off + 8L * v);
            ha[j] = ld16(h + off + 8L * v);
          }
        }
#pragma unroll
        for (int j = 0; j < kRowBatch; ++j) {
          const int v = v0 + 64 * j;
          if (v < nv) {
            float a[8], b[8], gg[8];
            unpack8(ga[j], a);
            unpack8(ha[j], b);
            unpack8(ld16(gamma + 8 * v), gg);
#pragma unroll
            for (int k = 0; k < 8; ++k) c = fmaf(a[k] * gg[k], b[k], c);
          }
        }
      }
    }
    c = warp_sum(c);
    if (lane == 0) part[g & 1][grow][w & 1] = c;
    __syncthreads();
    // phase two: gradients and column partials, kPair2 rows at a time
#pragma unroll 1
    for (int i = 0; i < kRbGroup; i += kPair2) {
      const int ra = gr0 + i;
      if (ra >= M) break;
      const int nrows = ra + kPair2 <= M ? kPair2 : M - ra;
      uint4 ga[kPair2][kOwn], ha[kPair2][kOwn];
#pragma unroll
      for (int t = 0; t < kPair2; ++t)
#pragma unroll
        for (int o = 0; o < kOwn; ++o) {
          const int v = threadIdx.x + kRbThreads * o;
          if (t < nrows && v < nv) {
            const long off = static_cast<long>(ra + t) * d + 8L * v;
            ga[t][o] = ld16(G + off);
            ha[t][o] = ld16(h + off);
          }
        }
#pragma unroll
      for (int t = 0; t < kPair2; ++t) {
        if (t >= nrows) break;
        const float cr = (part[g & 1][i + t][0] + part[g & 1][i + t][1]) / d;
        const float rv = r[ra + t];
        const float r3c = rv * rv * rv * cr;
#pragma unroll
        for (int o = 0; o < kOwn; ++o) {
          const int v = threadIdx.x + kRbThreads * o;
          if (v < nv) {
            float a[8], b[8], gg[8], out[8];
            unpack8(ga[t][o], a);
            unpack8(ha[t][o], b);
            unpack8(ld16(gamma + 8 * v), gg);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              out[k] = rv * gg[k] * a[k] - r3c * b[k];
              acc[o][k] += rv * a[k] * b[k];
            }
            st16(dh + static_cast<long>(ra + t) * d + 8L * v, pack8(out));
          }
        }
      }
    }
  }
  // scalar stores: the partials need only 4-byte alignment
#pragma unroll
  for (int o = 0; o < kOwn; ++o) {
    const int v = threadIdx.x + kRbThreads * o;
    if (v < nv) {
      float* dst = pdg + static_cast<long>(blockIdx.x) * d + 8L * v;
#pragma unroll
      for (int k = 0; k < 8; ++k) dst[k] = acc[o][k];
    }
  }
}

// Wider rows (d > 8 * kRbThreads * 4): one block per 32-row tile, one row at
// a time: per row c = (1/d) sum G gamma h (block reduce), dh = r gamma G -
// r^3 c h; column partials of r G h kept in shared memory.
__global__ void rmsnorm_bwd_wide_kernel(int M, int d, const __nv_bfloat16* G, const __nv_bfloat16* h,
                                   const __nv_bfloat16* gamma, const float* r, __nv_bfloat16* dh, float* pdg) {
  extern __shared__ float colacc[];
  __shared__ float sh[32];
  const int nv = d / 8;
  const int tiles = (M + 31) / 32;
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    for (int j = threadIdx.x; j < d; j += blockDim.x) colacc[j] = 0.f;
    const int r0 = tile * 32, r1 = min(M, r0 + 32);
    for (int row = r0; row < r1; ++row) {
      const long off = static_cast<long>(row) * d;
      float c = 0.f;
      for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float a[8], b[8], g[8];
        unpack8(ld16(G + off + 8 * v), a);
        unpack8(ld16(h + off + 8 * v), b);
        unpack8(ld16(gamma + 8 * v), g);
#pragma unroll
        for (int k = 0; k < 8; ++k) c = fmaf(a[k] * g[k], b[k], c);
      }
      c = block_sum(c, sh) / d;
      const float rv = r[row];
      const float r3c = rv * rv * rv * c;
      for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float a[8], b[8], g[8], o[8];
        unpack8(ld16(G + off + 8 * v), a);
        unpack8(ld16(h + off + 8 * v), b);
        unpack8(ld16(gamma + 8 * v), g);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          o[k] = rv * g[k] * a[k] - r3c * b[k];
          colacc[8 * v + k] += rv * a[k] * b[k];
        }
        st16(dh + off + 8 * v, pack8(o));
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < d; j += blockDim.x) pdg[static_cast<long>(tile) * d + j] = colacc[j];
    __syncthreads();
  }
}

int check_mn(const char* fn, int M, int N) {
  CODA_REQUIRE(M >= 0 && N >= 0, CODA_ERR_INVALID, "%s: negative dimension", fn);
  CODA_REQUIRE(N % 8 == 0, CODA_ERR_UNSUPPORTED, "%s: N=%d must be a multiple of 8", fn, N);
  return CODA_OK;
}

}  // namespace

extern "C" {

int coda_unfused_add(int M, int N, const coda_bf16* a, const coda_bf16* b, coda_bf16* out, coda_stream_t stream) {
  const char* fn = "coda_unfused_add";
  int rc = check_mn(fn, M, N);
  if (rc || M == 0 || N == 0) return rc;
  CODA_REQ_PTR16(a);
  CODA_REQ_PTR16(b);
  CODA_REQ_PTR16(out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const long nvec = static_cast<long>(M) * N / 8;
  static std::atomic<int> occ{0};
  add_kernel<<<grid_resident(di, add_kernel, occ, nvec, 256), 256, 0, as_stream(stream)>>>(nvec, reinterpret_cast<const uint4*>(a),
                                                                     reinterpret_cast<const uint4*>(b),
                                                                     reinterpret_cast<uint4*>(out));
  return launched(fn);
}

int coda_unfused_rmsnorm(int M, int d, const coda_bf16* h, const coda_bf16* gamma, float eps, coda_bf16* n_out,
                         float* r_out, coda_stream_t stream) {
  const char* fn = "coda_unfused_rmsnorm";
  int rc = check_mn(fn, M, d);
  if (rc || M == 0 || d == 0) return rc;
  CODA_REQUIRE(eps >= 0.f, CODA_ERR_INVALID, "%s: eps must be >= 0", fn);
  CODA_REQ_PTR16(h);
  CODA_REQ_PTR16(gamma);
  CODA_REQ_PTR16(n_out);
  CODA_REQ_OPT4(r_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const int grid = M < di->sm_count * 16 ? M : di->sm_count * 16;
  const auto* hb = reinterpret_cast<const __nv_bfloat16*>(h);
  const auto* gb = reinterpret_cast<const __nv_bfloat16*>(gamma);
  auto* nb = reinterpret_cast<__nv_bfloat16*>(n_out);
  if (d / 8 <= 4 * 256)
    rmsnorm_kernel<4><<<grid, 256, 0, as_stream(stream)>>>(M, d, hb, gb, eps, nb, r_out);
  else
    rmsnorm_kernel<0><<<grid, 256, 0, as_stream(stream)>>>(M, d, hb, gb, eps, nb, r_out);
  return launched(fn);
}

int coda_unfused_rowscale(int M, int N, const coda_bf16* x, const float* r, coda_bf16* out, coda_stream_t stream) {
  const char* fn = "coda_unfused_rowscale";
  int rc = check_mn(fn, M, N);
  if (rc || M == 0 || N == 0) return rc;
  CODA_REQ_PTR16(x);
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR16(out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  rowscale_kernel<<<grid_for(di, static_cast<long>(M) * N / 8, 256), 256, 0, as_stream(stream)>>>(
      M, N, reinterpret_cast<const __nv_bfloat16*>(x), r, reinterpret_cast<__nv_bfloat16*>(out));
  return launched(fn);
}

int coda_unfused_swiglu(int M, int F, const coda_bf16* gu, coda_bf16* A_out, coda_stream_t stream) {
  const char* fn = "coda_unfused_swiglu";
  int rc = check_mn(fn, M, F);
  if (rc || M == 0 || F == 0) return rc;
  CODA_REQ_PTR16(gu);
  CODA_REQ_PTR16(A_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const long n = static_cast<long>(M) * F / 8;
  static std::atomic<int> occ{0};
  swiglu_kernel<<<grid_resident(di, swiglu_kernel, occ, n, 256), 256, 0, as_stream(stream)>>>(n, reinterpret_cast<const __nv_bfloat16*>(gu),
                                                                     reinterpret_cast<__nv_bfloat16*>(A_out));
  return launched(fn);
}

int coda_unfused_swiglu_bwd(int M, int F, const coda_bf16* dA, const coda_bf16* gu, coda_bf16* dgu_out,
                            coda_stream_t stream) {
  const char* fn = "coda_unfused_swiglu_bwd";
  int rc = check_mn(fn, M, F);
  if (rc || M == 0 || F == 0) return rc;
  CODA_REQ_PTR16(dA);
  CODA_REQ_PTR16(gu);
  CODA_REQ_PTR16(dgu_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const long n = static_cast<long>(M) * F / 8;
  static std::atomic<int> occ{0};
  swiglu_bwd_kernel<<<grid_resident(di, swiglu_bwd_kernel, occ, n, 256), 256, 0, as_stream(stream)>>>(
      n, reinterpret_cast<const __nv_bfloat16*>(dA), reinterpret_cast<const __nv_bfloat16*>(gu),
      reinterpret_cast<__nv_bfloat16*>(dgu_out));
  return launched(fn);
}

static int rope_unfused(const char* fn, int sign, int M, int N, const float* ct, const float* st, int S, int hd,
                        int rope_cols, coda_bf16* x, coda_stream_t stream) {
  int rc = check_mn(fn, M, N);
  if (rc) return rc;
  CODA_REQUIRE(hd > 0 && hd % 8 == 0, CODA_ERR_UNSUPPORTED, "%s: head_dim=%d must be a positive multiple of 8", fn, hd);
  CODA_REQUIRE(rope_cols >= 0 && rope_cols % hd == 0 && rope_cols <= N, CODA_ERR_INVALID,
               "%s: rope_cols=%d must be a multiple of head_dim in [0, N]", fn, rope_cols);
  CODA_REQUIRE(S > 0, CODA_ERR_INVALID, "%s: S must be positive", fn);
  if (M == 0 || rope_cols == 0) return CODA_OK;
  CODA_REQ_PTR16(ct);
  CODA_REQ_PTR16(st);
  CODA_REQ_PTR16(x);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const int g = grid_for(di, static_cast<long>(M) * rope_cols / 8, 256);
  __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(x);
  if (sign > 0)
    rope_kernel<1><<<g, 256, 0, as_stream(stream)>>>(M, N, ct, st, S, hd, rope_cols, p);
  else
    rope_kernel<-1><<<g, 256, 0, as_stream(stream)>>>(M, N, ct, st, S, hd, rope_cols, p);
  return launched(fn);
}

int coda_unfused_rope(int M, int N, const float* cos_tab, const float* sin_tab, int S, int head_dim, int rope_cols,
                      coda_bf16* x, coda_stream_t stream) {
  return rope_unfused("coda_unfused_rope", 1, M, N, cos_tab, sin_tab, S, head_dim, rope_cols, x, stream);
}

int coda_unfused_rope_bwd(int M, int N, const float* cos_tab, const float* sin_tab, int S, int head_dim,
                          int rope_cols, coda_bf16* x, coda_stream_t stream) {
  return rope_unfused("coda_unfused_rope_bwd", -1, M, N, cos_tab, sin_tab, S, head_dim, rope_cols, x, stream);
}

int coda_unfused_ce_fwd(int M, int V, const coda_bf16* logits, const int32_t* labels, float* lse_out,
                        float* loss_row_out, float* loss_mean_out, int32_t* argmax_out, coda_stream_t stream) {
  const char* fn = "coda_unfused_ce_fwd";
  int rc = check_mn(fn, M, V);
  if (rc || M == 0) return rc;
  CODA_REQUIRE(V > 0, CODA_ERR_INVALID, "%s: V must be positive", fn);
  CODA_REQ_PTR16(logits);
  CODA_REQ_PTR4(labels);
  CODA_REQ_PTR4(lse_out);
  CODA_REQ_PTR4(loss_row_out);
  CODA_REQ_OPT4(loss_mean_out);
  CODA_REQ_OPT4(argmax_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  // one warp per row, 8 warps per block
  const long blocks = (static_cast<long>(M) + 7) / 8;
  const int grid = static_cast<int>(blocks < di->sm_count * 16L ? blocks : di->sm_count * 16L);
  cudaStream_t st = as_stream(stream);
  ce_fwd_kernel<<<grid, 256, 0, st>>>(M, V, reinterpret_cast<const __nv_bfloat16*>(logits), labels, lse_out,
                                      loss_row_out, argmax_out, di->status);
  rc = launched(fn);
  if (rc || !loss_mean_out) return rc;
  ce_mean_kernel<<<1, 1024, 0, st>>>(M, loss_row_out, loss_mean_out);
  return launched(fn);
}

int coda_unfused_ce_bwd(int M, int V, const coda_bf16* logits, const int32_t* labels, const float* lse,
                        float grad_scale, coda_bf16* dl_out, coda_stream_t stream) {
  const char* fn = "coda_unfused_ce_bwd";
  int rc = check_mn(fn, M, V);
  if (rc || M == 0 || V == 0) return rc;
  CODA_REQ_PTR16(logits);
  CODA_REQ_PTR4(labels);
  CODA_REQ_PTR4(lse);
  CODA_REQ_PTR16(dl_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  ce_bwd_kernel<<<grid_for(di, static_cast<long>(M) * V / 8, 256), 256, 0, as_stream(stream)>>>(
      M, V, reinterpret_cast<const __nv_bfloat16*>(logits), labels, lse, grad_scale,
      reinterpret_cast<__nv_bfloat16*>(dl_out));
  return launched(fn);
}

int coda_unfused_rowdot(int M, int N, int d, const coda_bf16* dY, const coda_bf16* Y, float* s_out,
                        coda_stream_t stream) {
  const char* fn = "coda_unfused_rowdot";
  int rc = check_mn(fn, M, N);
  if (rc || M == 0) return rc;
  CODA_REQUIRE(d > 0, CODA_ERR_INVALID, "%s: d must be positive", fn);
  CODA_REQ_PTR16(dY);
  CODA_REQ_PTR16(Y);
  CODA_REQ_PTR4(s_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const int grid = M < di->sm_count * 16 ? M : di->sm_count * 16;
  rowdot_kernel<<<grid, 256, 0, as_stream(stream)>>>(M, N, 1.0f / d, reinterpret_cast<const __nv_bfloat16*>(dY),
                                                     reinterpret_cast<const __nv_bfloat16*>(Y), s_out);
  return launched(fn);
}

int coda_unfused_rmsnorm_bwd(int M, int d, const coda_bf16* G, const coda_bf16* h, const coda_bf16* gamma,
                             const float* r, coda_bf16* dh_out, float* pdg_out, coda_stream_t stream) {
  const char* fn = "coda_unfused_rmsnorm_bwd";
  int rc = check_mn(fn, M, d);
  if (rc || M == 0 || d == 0) return rc;
  CODA_REQUIRE(d <= 49152, CODA_ERR_UNSUPPORTED, "%s: d=%d exceeds 49152", fn, d);
  CODA_REQ_PTR16(G);
  CODA_REQ_PTR16(h);
  CODA_REQ_PTR16(gamma);
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR16(dh_out);
  CODA_REQ_PTR4(pdg_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const int tiles = (M + 31) / 32;
  const auto* Gb = reinterpret_cast<const __nv_bfloat16*>(G);
  const auto* hb = reinterpret_cast<const __nv_bfloat16*>(h);
  const auto* gb = reinterpret_cast<const __nv_bfloat16*>(gamma);
  auto* db = reinterpret_cast<__nv_bfloat16*>(dh_out);
  cudaStream_t st = as_stream(stream);
  const int nv = d / 8;
  if (nv <= kRbThreads) {
    rmsnorm_bwd_kernel<1><<<tiles, kRbThreads, 0, st>>>(M, d, Gb, hb, gb, r, db, pdg_out);
  } else if (nv <= 2 * kRbThreads) {
    rmsnorm_bwd_kernel<2><<<tiles, kRbThreads, 0, st>>>(M, d, Gb, hb, gb, r, db, pdg_out);
  } else if (nv <= 4 * kRbThreads) {
    rmsnorm_bwd_kernel<4><<<tiles, kRbThreads, 0, st>>>(M, d, Gb, hb, gb, r, db, pdg_out);
  } else {
    const size_t smem = static_cast<size_t>(d) * sizeof(float);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&rmsnorm_bwd_wide_kernel),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(rmsnorm_bwd)");
    }
    rmsnorm_bwd_wide_kernel<<<tiles, 512, smem, st>>>(M, d, Gb, hb, gb, r, db, pdg_out);
  }
  return launched(fn);
}

}  // extern "C"
