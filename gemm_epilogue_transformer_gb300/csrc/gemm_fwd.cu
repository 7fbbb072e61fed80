// Forward GEMM entry points: plain GEMM, residual + RMS-prep, delayed row
// scale, SwiGLU, RoPE.
#include "gemm_launch.cuh"

using namespace coda;

extern "C" {

int coda_gemm(int M, int N, int K, const coda_bf16* A, int lda, int transA, const coda_bf16* B, int ldb, int transB,
              coda_bf16* C, int ldc, coda_stream_t stream) {
  const char* fn = "coda_gemm";
  CODA_REQUIRE(M >= 0 && N >= 0 && K >= 0, CODA_ERR_INVALID, "%s: negative dimension", fn);
  CODA_REQUIRE(transA == 0 || transA == 1, CODA_ERR_INVALID, "%s: transA must be 0 or 1", fn);
  CODA_REQUIRE(transB == 0 || transB == 1, CODA_ERR_INVALID, "%s: transB must be 0 or 1", fn);
  if (M == 0 || N == 0) return CODA_OK;
  CODA_REQ_PTR16(C);
  CODA_REQUIRE(ldc >= N && ldc % 8 == 0, CODA_ERR_INVALID, "%s: ldc=%d must be >= N=%d and a multiple of 8", fn, ldc, N);
  if (K > 0) {
    CODA_REQ_PTR16(A);
    CODA_REQ_PTR16(B);
    const int a_inner = transA ? M : K, b_inner = transB ? K : N;
    CODA_REQUIRE(lda >= a_inner && lda % 8 == 0, CODA_ERR_INVALID,
                 "%s: lda=%d must be >= %d and a multiple of 8", fn, lda, a_inner);
    CODA_REQUIRE(ldb >= b_inner && ldb % 8 == 0, CODA_ERR_INVALID,
                 "%s: ldb=%d must be >= %d and a multiple of 8", fn, ldb, b_inner);
  }
  CUtensorMap o;
  int rc = make_out_map(&o, C, M, N, ldc);
  if (rc) return rc;
  EpiPlain::Params ep{0};
  // transA = 1: A stored [K, M] is M-major. transB = 0: B stored [K, N] is
  // N-major; transB = 1: B stored [N, K] is K-major.
  return launch_fused<EpiPlain>(fn, M, N, K, A, lda, /*a_mn=*/transA, B, ldb, /*b_mn=*/transB ? 0 : 1, o, o, o, o,
                                ep, as_stream(stream));
}

int coda_gemm_res_rmsprep(int M, int N, int K, const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                          const coda_bf16* gamma, coda_bf16* h1_out, coda_bf16* h2_out, float* psq_out,
                          coda_stream_t stream) {
  const char* fn = "coda_gemm_res_rmsprep";
  int rc = check_fused(fn, M, N, K, x, W0);
  if (rc) return rc;
  if (M == 0 || N == 0) return CODA_OK;
  CODA_REQ_PTR16(z);
  CODA_REQ_PTR16(gamma);
  CODA_REQ_PTR16(h1_out);
  CODA_REQ_PTR16(h2_out);
  CODA_REQ_PTR4(psq_out);
  CUtensorMap o0, o1;
  if ((rc = make_out_map(&o0, h1_out, M, N, N))) return rc;
  if ((rc = make_out_map(&o1, h2_out, M, N, N))) return rc;
  CUtensorMap iz;
  if ((rc = make_out_map(&iz, z, M, N, N))) return rc;
  EpiResRmsPrep::Params ep{reinterpret_cast<const __nv_bfloat16*>(z), reinterpret_cast<const __nv_bfloat16*>(gamma),
                           psq_out};
  return launch_fused<EpiResRmsPrep>(fn, M, N, K, x, K, 0, W0, N, /*b_mn=*/1, o0, o1, iz, iz, ep, as_stream(stream));
}

int coda_gemm_rowscale(int M, int N, int K, const coda_bf16* h2, const coda_bf16* W1, const float* r,
                       coda_bf16* Y_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_rowscale";
  int rc = check_fused(fn, M, N, K, h2, W1);
  if (rc) return rc;
  if (M == 0 || N == 0) return CODA_OK;
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR16(Y_out);
  CUtensorMap o;
  if ((rc = make_out_map(&o, Y_out, M, N, N))) return rc;
  EpiRowScale::Params ep{r};
  return launch_fused<EpiRowScale>(fn, M, N, K, h2, K, 0, W1, N, /*b_mn=*/1, o, o, o, o, ep, as_stream(stream));
}

int coda_gemm_swiglu(int M, int F, int K, const coda_bf16* X, const coda_bf16* Wgu, coda_bf16* A_out,
                     coda_bf16* gu_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_swiglu";
  CODA_REQUIRE(F >= 0, CODA_ERR_INVALID, "%s: negative F", fn);
  CODA_REQUIRE(F <= (1 << 30), CODA_ERR_INVALID, "%s: F too large", fn);
  int rc = check_fused(fn, M, 2 * F, K, X, Wgu);
  if (rc) return rc;
  CODA_REQUIRE(F % 8 == 0, CODA_ERR_UNSUPPORTED, "%s: F=%d must be a multiple of 8", fn, F);
  if (M == 0 || F == 0) return CODA_OK;
  CODA_REQ_PTR16(A_out);
  CODA_REQ_OPT16(gu_out);
  CUtensorMap o, og;
  if ((rc = make_out_map(&o, A_out, M, F, F))) return rc;
  og = o;
  if (gu_out && (rc = make_out_map(&og, gu_out, M, 2 * F, 2 * F))) return rc;
  if (gu_out) {
    EpiSwiGLU<true>::Params ep{0};
    return launch_fused<EpiSwiGLU<true>>(fn, M, 2 * F, K, X, K, 0, Wgu, 2 * F, /*b_mn=*/1, o, og, o, o, ep,
                                         as_stream(stream));
  }
  EpiSwiGLU<false>::Params ep{0};
  return launch_fused<EpiSwiGLU<false>>(fn, M, 2 * F, K, X, K, 0, Wgu, 2 * F, /*b_mn=*/1, o, og, o, o, ep,
                                        as_stream(stream));
}

static int rope_common(const char* fn, int M, int N, int K, const coda_bf16* X, const coda_bf16* W,
                       const float* cos_tab, const float* sin_tab, int S, int head_dim, int rope_cols, coda_bf16* out) {
  int rc = check_fused(fn, M, N, K, X, W);
  if (rc) return rc;
  CODA_REQUIRE(head_dim > 0 && head_dim % 32 == 0, CODA_ERR_UNSUPPORTED, "%s: head_dim=%d must be a positive multiple of 32",
               fn, head_dim);
  CODA_REQUIRE(rope_cols >= 0 && rope_cols % head_dim == 0 && rope_cols <= N, CODA_ERR_INVALID,
               "%s: rope_cols=%d must be a multiple of head_dim in [0, N]", fn, rope_cols);
  CODA_REQUIRE(S > 0, CODA_ERR_INVALID, "%s: S=%d must be positive", fn, S);
  if (M == 0 || N == 0) return CODA_OK;
  CODA_REQ_PTR16(cos_tab);
  CODA_REQ_PTR16(sin_tab);
  CODA_REQ_PTR16(out);
  return CODA_OK;
}

int coda_gemm_rope(int M, int N, int K, const coda_bf16* X, const coda_bf16* W, const float* cos_tab,
                   const float* sin_tab, int S, int head_dim, int rope_cols, coda_bf16* out, coda_stream_t stream) {
  const char* fn = "coda_gemm_rope";
  int rc = rope_common(fn, M, N, K, X, W, cos_tab, sin_tab, S, head_dim, rope_cols, out);
  if (rc || M == 0 || N == 0) return rc;
  CUtensorMap o;
  if ((rc = make_out_map(&o, out, M, N, N))) return rc;
  EpiRope<1>::Params ep{cos_tab, sin_tab, S, head_dim, rope_cols, rope_lane_tables(S, head_dim)};
  return launch_fused<EpiRope<1>>(fn, M, N, K, X, K, 0, W, N, /*b_mn=*/1, o, o, o, o, ep, as_stream(stream));
}

int coda_gemm_rope_bwd(int M, int N, int K, const coda_bf16* A, const coda_bf16* B, const float* cos_tab,
                       const float* sin_tab, int S, int head_dim, int rope_cols, coda_bf16* out,
                       coda_stream_t stream) {
  const char* fn = "coda_gemm_rope_bwd";
  int rc = rope_common(fn, M, N, K, A, B, cos_tab, sin_tab, S, head_dim, rope_cols, out);
  if (rc || M == 0 || N == 0) return rc;
  CUtensorMap o;
  if ((rc = make_out_map(&o, out, M, N, N))) return rc;
  EpiRope<-1>::Params ep{cos_tab, sin_tab, S, head_dim, rope_cols, rope_lane_tables(S, head_dim)};
  return launch_fused<EpiRope<-1>>(fn, M, N, K, A, K, 0, B, N, /*b_mn=*/1, o, o, o, o, ep, as_stream(stream));
}

}  // extern "C"
