// The block-level chain (CODA note, block-level ablation): one period of two
// consecutive GEMM-Residual-RMSNorm-GEMM structures, the RoPE path and then
// the SwiGLU path, forward and backward, as a fixed sequence of launches on
// one stream. The fused sequence runs the CODA kernels (residual + RMS-prep
// GEMM, aux reduction, rowscale GEMM with the pair map; SwiGLU-backward GEMM
// with the row statistic, RMSNorm-backward GEMM with the residual gradient,
// the RoPE-path glue, plain weight-gradient GEMMs). The unfused sequence runs
// plain GEMMs and the stand-alone memory-bound kernels of the comparison path.
//
// Also here: the RoPE-path glue kernel. The attention backward delivers the
// gradient of the rotated QKV; no GEMM of the chain produces it, so its
// transposed rotation, the row statistic and the row scale run as one pass
// over dQKV and the saved QKV.
#include <cuda_bf16.h>

#include <mutex>

#include "host.h"

using namespace coda;

namespace {

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
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One 256-thread block per row (grid-stride over rows). Per 8-column vector:
// dYq = RoPE^T(dQKV) on the rope columns (g_e = a_e cos + a_o sin,
// g_o = -a_e sin + a_o cos), the row dot of dQKV and the stored QKV (the
// rotation is orthogonal, so it equals rowsum(dYq (.) Yq) with Yq the
// unrotated projection), and dYqr = r dYq.
constexpr int kGlueThreads = 256;
__global__ void __launch_bounds__(kGlueThreads) rope_bwd_rowdot_kernel(
    int M, int N, const __nv_bfloat16* __restrict__ dqkv, const __nv_bfloat16* __restrict__ qkv,
    const float* __restrict__ r, const float* __restrict__ ct, const float* __restrict__ st, int S, int head_dim,
    int rope_cols, float inv_d, __nv_bfloat16* __restrict__ dqr, float* __restrict__ s_out) {
  __shared__ float sh[kGlueThreads / 32];
  const int nv = N / 8;
  const int half = head_dim / 2;
  for (int row = blockIdx.x; row < M; row += gridDim.x) {
    const long base = static_cast<long>(row) * N;
    const float rv = r[row];
    const int pos = row % S;
    float dot = 0.f;
    for (int v = threadIdx.x; v < nv; v += kGlueThreads) {
      const int c0 = 8 * v;
      float a[8], y[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(dqkv + base + c0)), a);
      unpack8(__ldg(reinterpret_cast<const uint4*>(qkv + base + c0)), y);
#pragma unroll
      for (int k = 0; k < 8; ++k) dot = fmaf(a[k], y[k], dot);
      float o[8];
      if (c0 < rope_cols) {
        const int i0 = (c0 % head_dim) >> 1;
        const float4 cv = __ldg(reinterpret_cast<const float4*>(ct + static_cast<long>(pos) * half + i0));
        const float4 sv = __ldg(reinterpret_cast<const float4*>(st + static_cast<long>(pos) * half + i0));
        const float cs[4] = {cv.x, cv.y, cv.z, cv.w};
        const float sn[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float e = a[2 * k], od = a[2 * k + 1];
          o[2 * k] = rv * (e * cs[k] + od * sn[k]);
          o[2 * k + 1] = rv * (od * cs[k] - e * sn[k]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = rv * a[k];
      }
      *reinterpret_cast<uint4*>(dqr + base + c0) =
          make_uint4(pack2(o[0], o[1]), pack2(o[2], o[3]), pack2(o[4], o[5]), pack2(o[6], o[7]));
    }
    dot = warp_sum(dot);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) sh[w] = dot;
    __syncthreads();
    if (w == 0) {
      dot = (l < kGlueThreads / 32) ? sh[l] : 0.f;
      dot = warp_sum(dot);
      if (l == 0) s_out[row] = dot * inv_d;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------ workspace
struct Ws {
  float* psq;   // [M, ceil(d/128)]
  float* pdot;  // [M, ceil(F/128)]
  float* pdg;   // [ceil(M/32), d]
  coda_bf16* t;   // unfused: [M, d] GEMM output before the residual add / RMSNorm-backward output
  coda_bf16* dA;  // unfused: [M, F]
  coda_bf16* dn;  // unfused: [M, d]
};

inline size_t up256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

size_t ws_layout(int M, int d, int F, int unfused, char* base, Ws* w) {
  const size_t m = static_cast<size_t>(M);
  const size_t nbd = static_cast<size_t>((d + 127) / 128), nbf = static_cast<size_t>((F + 127) / 128);
  const size_t rows32 = static_cast<size_t>((M + 31) / 32);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off += up256(bytes);
    return p;
  };
  Ws l;
  l.psq = reinterpret_cast<float*>(take(m * nbd * 4));
  l.pdot = reinterpret_cast<float*>(take(m * nbf * 4));
  l.pdg = reinterpret_cast<float*>(take(rows32 * static_cast<size_t>(d) * 4));
  l.t = l.dA = l.dn = nullptr;
  if (unfused) {
    l.t = reinterpret_cast<coda_bf16*>(take(m * d * 2));
    l.dA = reinterpret_cast<coda_bf16*>(take(m * static_cast<size_t>(F) * 2));
    l.dn = reinterpret_cast<coda_bf16*>(take(m * d * 2));
  }
  if (w) *w = l;
  return off;
}

int check_block(const char* fn, const coda_block_t* b) {
  CODA_REQUIRE(b != nullptr, CODA_ERR_INVALID, "%s: null block descriptor", fn);
  CODA_REQUIRE(b->M >= 0 && b->d >= 0 && b->F >= 0, CODA_ERR_INVALID, "%s: negative size", fn);
  CODA_REQUIRE(b->d % 8 == 0 && b->F % 8 == 0, CODA_ERR_UNSUPPORTED, "%s: d=%d and F=%d must be multiples of 8", fn,
               b->d, b->F);
  CODA_REQUIRE(b->workspace != nullptr && (reinterpret_cast<uintptr_t>(b->workspace) & 255u) == 0, CODA_ERR_INVALID,
               "%s: workspace must be a non-null 256-byte aligned device pointer", fn);
  return CODA_OK;
}

// Scratch of coda_block_fwd_noalloc, the forward for callers that cannot
// allocate device memory (a plugin given only its input and output buffers, a
// serving loop that may not call cudaMalloc after start-up, a process whose
// pool holds the device's memory): the forward's only scratch, the
// per-(row, 128-column block) sum-of-squares partials, in a file-scope device
// array instead of the caller's workspace. One array per device (the module
// is loaded per context), shared by every call on that device.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB: M * ceil(d/128) fp32 partials
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up by the
// first call on each device (with that device current) and cached for the
// process, which assumes one context per device (as every per-device cache of
// the library does); nullptr after fail().
void* noalloc_scratch() {
  static std::mutex mu;
  static void* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    fail(CODA_ERR_CUDA, "coda_block_fwd_noalloc: no current device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      fail_cuda(e == cudaSuccess ? cudaErrorInvalidSymbol : e, "cudaGetSymbolAddress(noalloc scratch)");
      return nullptr;
    }
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

#define CODA_TRY(call)        \
  do {                        \
    const int rc_ = (call);   \
    if (rc_) return rc_;      \
  } while (0)

}  // namespace

extern "C" {

int coda_rope_bwd_rowdot(int M, int N, const coda_bf16* dqkv, const coda_bf16* qkv, const float* r,
                         const float* cos_tab, const float* sin_tab, int S, int head_dim, int rope_cols, int d,
                         coda_bf16* dqr_out, float* s_out, coda_stream_t stream) {
  const char* fn = "coda_rope_bwd_rowdot";
  CODA_REQUIRE(M >= 0 && N >= 0, CODA_ERR_INVALID, "%s: negative dimension", fn);
  CODA_REQUIRE(N % 8 == 0, CODA_ERR_UNSUPPORTED, "%s: N=%d must be a multiple of 8", fn, N);
  CODA_REQUIRE(head_dim > 0 && head_dim % 8 == 0, CODA_ERR_UNSUPPORTED,
               "%s: head_dim=%d must be a positive multiple of 8", fn, head_dim);
  CODA_REQUIRE(rope_cols >= 0 && rope_cols % head_dim == 0 && rope_cols <= N, CODA_ERR_INVALID,
               "%s: rope_cols=%d must be a multiple of head_dim in [0, N]", fn, rope_cols);
  CODA_REQUIRE(S > 0 && d > 0, CODA_ERR_INVALID, "%s: S=%d and d=%d must be positive", fn, S, d);
  if (M == 0) return CODA_OK;
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR4(s_out);
  if (N > 0) {
    CODA_REQ_PTR16(dqkv);
    CODA_REQ_PTR16(qkv);
    CODA_REQ_PTR16(dqr_out);
    if (rope_cols > 0) {
      CODA_REQ_PTR16(cos_tab);
      CODA_REQ_PTR16(sin_tab);
    }
  }
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  const int grid = M < di->sm_count * 8 ? M : di->sm_count * 8;
  rope_bwd_rowdot_kernel<<<grid, kGlueThreads, 0, as_stream(stream)>>>(
      M, N, reinterpret_cast<const __nv_bfloat16*>(dqkv), reinterpret_cast<const __nv_bfloat16*>(qkv), r, cos_tab,
      sin_tab, S, head_dim, rope_cols, 1.0f / static_cast<float>(d), reinterpret_cast<__nv_bfloat16*>(dqr_out), s_out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CODA_OK : fail_cuda(e, fn);
}

size_t coda_block_workspace_bytes(int M, int d, int F, int unfused) {
  if (M < 0 || d < 0 || F < 0) return 0;
  return ws_layout(M, d, F, unfused, nullptr, nullptr);
}

int coda_block_fwd(const coda_block_t* b, coda_stream_t stream) {
  const char* fn = "coda_block_fwd";
  CODA_TRY(check_block(fn, b));
  const int M = b->M, d = b->d, F = b->F;
  if (M == 0) return CODA_OK;
  Ws w;
  ws_layout(M, d, F, 0, static_cast<char*>(b->workspace), &w);
  const int nbd = coda_num_col_tiles(d);
  // RoPE path: h1 = P Wd + x -> h1, h1g = h1 (.) gamma1, sum-of-squares partials; r1; QKV = RoPE(r1 (.) h1g Wqkv)
  CODA_TRY(coda_gemm_res_rmsprep(M, d, F, b->P, b->Wd, b->x, b->gamma1, b->h1, b->h1g, w.psq, stream));
  CODA_TRY(coda_rms_reduce(M, nbd, d, w.psq, b->eps, b->r1, stream));
  CODA_TRY(coda_gemm_rowscale_rope(M, 3 * d, d, b->h1g, b->Wqkv, b->r1, b->cos_tab, b->sin_tab, b->S, b->head_dim,
                                   b->rope_cols, b->qkv, stream));
  // SwiGLU path: h2 = O Wo + h1; r2; GU = r2 (.) h2g Wgu (saved), A = SwiGLU(GU)
  CODA_TRY(coda_gemm_res_rmsprep(M, d, d, b->O, b->Wo, b->h1, b->gamma2, b->h2, b->h2g, w.psq, stream));
  CODA_TRY(coda_rms_reduce(M, nbd, d, w.psq, b->eps, b->r2, stream));
  CODA_TRY(coda_gemm_rowscale_swiglu(M, F, d, b->h2g, b->Wgu, b->r2, b->a, b->gu, stream));
  return CODA_OK;
}

int coda_block_fwd_noalloc(const coda_block_t* b, coda_stream_t stream) {
  const char* fn = "coda_block_fwd_noalloc";
  CODA_REQUIRE(b != nullptr, CODA_ERR_INVALID, "%s: null block descriptor", fn);
  CODA_REQUIRE(b->M >= 0 && b->d >= 0 && b->F >= 0, CODA_ERR_INVALID, "%s: negative size", fn);
  const size_t need = static_cast<size_t>(b->M) * static_cast<size_t>((b->d + 127) / 128) * sizeof(float);
  CODA_REQUIRE(need <= kNoAllocScratchBytes, CODA_ERR_UNSUPPORTED,
               "%s: M * ceil(d/128) * 4 = %zu bytes of partials exceed the %zu-byte static scratch", fn, need,
               kNoAllocScratchBytes);
  if (b->M == 0) return CODA_OK;
  void* scratch = noalloc_scratch();
  if (!scratch) return CODA_ERR_CUDA;
  // the same launch sequence as coda_block_fwd, with the static array as its workspace (the
  // forward touches only the partials, which the workspace layout places first); the GEMMs
  // run without the stream-K tail, whose per-stream workspace would be allocated
  coda_block_t c = *b;
  c.workspace = scratch;
  NoAllocScope no_alloc;
  return coda_block_fwd(&c, stream);
}

int coda_block_bwd(const coda_block_t* b, coda_stream_t stream) {
  const char* fn = "coda_block_bwd";
  CODA_TRY(check_block(fn, b));
  const int M = b->M, d = b->d, F = b->F;
  if (M == 0) return CODA_OK;
  Ws w;
  ws_layout(M, d, F, 0, static_cast<char*>(b->workspace), &w);
  const int rows32 = coda_num_row_tiles(M);
  // SwiGLU path: dGUr = r2 (.) SwiGLU'(gh Wdn^T; GU) with the row statistic s2
  CODA_TRY(coda_gemm_swiglu_bwd_rowdot(M, F, d, b->gh, b->Wdn, b->gu, b->r2, b->dgur, w.pdot, stream));
  CODA_TRY(coda_rowdot_reduce(M, coda_num_col_tiles(F), d, w.pdot, b->s2, stream));
  // dh2 = gamma2 (.) (dGUr Wgu^T) - r2^2 s2 h2 + gh
  CODA_TRY(coda_gemm_rmsnorm_bwd_res(M, d, 2 * F, b->dgur, b->Wgu, b->h2, b->gamma2, b->r2, b->s2, b->gh, b->dh2,
                                     w.pdg, stream));
  CODA_TRY(coda_colsum_reduce(rows32, d, w.pdg, b->dgamma2, stream));
  CODA_TRY(coda_gemm(d, 2 * F, M, b->h2g, d, 1, b->dgur, 2 * F, 0, b->dWgu, 2 * F, stream));
  // attention output projection: dO = dh2 Wo^T, dWo = O^T dh2
  CODA_TRY(coda_gemm(M, d, d, b->dh2, d, 0, b->Wo, d, 1, b->dO, d, stream));
  CODA_TRY(coda_gemm(d, d, M, b->O, d, 1, b->dh2, d, 0, b->dWo, d, stream));
  // RoPE path: dYqr = r1 (.) RoPE^T(dQKV), s1; dh1 = gamma1 (.) (dYqr Wqkv^T) - r1^2 s1 h1 + dh2
  CODA_TRY(coda_rope_bwd_rowdot(M, 3 * d, b->dqkv, b->qkv, b->r1, b->cos_tab, b->sin_tab, b->S, b->head_dim,
                                b->rope_cols, d, b->dqr, b->s1, stream));
  CODA_TRY(coda_gemm_rmsnorm_bwd_res(M, d, 3 * d, b->dqr, b->Wqkv, b->h1, b->gamma1, b->r1, b->s1, b->dh2, b->dh1,
                                     w.pdg, stream));
  CODA_TRY(coda_colsum_reduce(rows32, d, w.pdg, b->dgamma1, stream));
  CODA_TRY(coda_gemm(d, 3 * d, M, b->h1g, d, 1, b->dqr, 3 * d, 0, b->dWqkv, 3 * d, stream));
  CODA_TRY(coda_gemm(F, d, M, b->P, F, 1, b->dh1, d, 0, b->dWd, d, stream));
  return CODA_OK;
}

int coda_block_fwd_unfused(const coda_block_t* b, coda_stream_t stream) {
  const char* fn = "coda_block_fwd_unfused";
  CODA_TRY(check_block(fn, b));
  const int M = b->M, d = b->d, F = b->F;
  if (M == 0) return CODA_OK;
  Ws w;
  ws_layout(M, d, F, 1, static_cast<char*>(b->workspace), &w);
  // h1 = P Wd + x; n1, r1 = RMSNorm(h1); QKV = n1 Wqkv; RoPE in place
  CODA_TRY(coda_gemm(M, d, F, b->P, F, 0, b->Wd, d, 0, w.t, d, stream));
  CODA_TRY(coda_unfused_add(M, d, w.t, b->x, b->h1, stream));
  CODA_TRY(coda_unfused_rmsnorm(M, d, b->h1, b->gamma1, b->eps, b->h1g, b->r1, stream));
  CODA_TRY(coda_gemm(M, 3 * d, d, b->h1g, d, 0, b->Wqkv, 3 * d, 0, b->qkv, 3 * d, stream));
  CODA_TRY(coda_unfused_rope(M, 3 * d, b->cos_tab, b->sin_tab, b->S, b->head_dim, b->rope_cols, b->qkv, stream));
  // h2 = O Wo + h1; n2, r2 = RMSNorm(h2); GU = n2 Wgu; A = SwiGLU(GU)
  CODA_TRY(coda_gemm(M, d, d, b->O, d, 0, b->Wo, d, 0, w.t, d, stream));
  CODA_TRY(coda_unfused_add(M, d, w.t, b->h1, b->h2, stream));
  CODA_TRY(coda_unfused_rmsnorm(M, d, b->h2, b->gamma2, b->eps, b->h2g, b->r2, stream));
  CODA_TRY(coda_gemm(M, 2 * F, d, b->h2g, d, 0, b->Wgu, 2 * F, 0, b->gu, 2 * F, stream));
  CODA_TRY(coda_unfused_swiglu(M, F, b->gu, b->a, stream));
  return CODA_OK;
}

int coda_block_bwd_unfused(const coda_block_t* b, coda_stream_t stream) {
  const char* fn = "coda_block_bwd_unfused";
  CODA_TRY(check_block(fn, b));
  const int M = b->M, d = b->d, F = b->F;
  if (M == 0) return CODA_OK;
  Ws w;
  ws_layout(M, d, F, 1, static_cast<char*>(b->workspace), &w);
  const int rows32 = coda_num_row_tiles(M);
  // SwiGLU path: dA = gh Wdn^T; dGU; dn2 = dGU Wgu^T; dh2 = RMSNorm'(dn2) + gh
  CODA_TRY(coda_gemm(M, F, d, b->gh, d, 0, b->Wdn, d, 1, w.dA, F, stream));
  CODA_TRY(coda_unfused_swiglu_bwd(M, F, w.dA, b->gu, b->dgur, stream));
  CODA_TRY(coda_gemm(M, d, 2 * F, b->dgur, 2 * F, 0, b->Wgu, 2 * F, 1, w.dn, d, stream));
  CODA_TRY(coda_unfused_rmsnorm_bwd(M, d, w.dn, b->h2, b->gamma2, b->r2, w.t, w.pdg, stream));
  CODA_TRY(coda_colsum_reduce(rows32, d, w.pdg, b->dgamma2, stream));
  CODA_TRY(coda_unfused_add(M, d, w.t, b->gh, b->dh2, stream));
  CODA_TRY(coda_gemm(d, 2 * F, M, b->h2g, d, 1, b->dgur, 2 * F, 0, b->dWgu, 2 * F, stream));
  CODA_TRY(coda_gemm(M, d, d, b->dh2, d, 0, b->Wo, d, 1, b->dO, d, stream));
  CODA_TRY(coda_gemm(d, d, M, b->O, d, 1, b->dh2, d, 0, b->dWo, d, stream));
  // RoPE path: transposed rotation in place on dQKV; dn1 = dYq Wqkv^T; dh1 = RMSNorm'(dn1) + dh2
  CODA_TRY(coda_unfused_rope_bwd(M, 3 * d, b->cos_tab, b->sin_tab, b->S, b->head_dim, b->rope_cols, b->dqkv, stream));
  CODA_TRY(coda_gemm(M, d, 3 * d, b->dqkv, 3 * d, 0, b->Wqkv, 3 * d, 1, w.dn, d, stream));
  CODA_TRY(coda_unfused_rmsnorm_bwd(M, d, w.dn, b->h1, b->gamma1, b->r1, w.t, w.pdg, stream));
  CODA_TRY(coda_colsum_reduce(rows32, d, w.pdg, b->dgamma1, stream));
  CODA_TRY(coda_unfused_add(M, d, w.t, b->dh2, b->dh1, stream));
  CODA_TRY(coda_gemm(d, 3 * d, M, b->h1g, d, 1, b->dqkv, 3 * d, 0, b->dWqkv, 3 * d, stream));
  CODA_TRY(coda_gemm(F, d, M, b->P, F, 1, b->dh1, d, 0, b->dWd, d, stream));
  return CODA_OK;
}

}  // extern "C"
