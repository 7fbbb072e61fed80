// Fused GEMM entry points of the block-level chain (CODA note, block-level
// ablation: two consecutive GEMM-Residual-RMSNorm-GEMM structures, one on the
// RoPE path and one on the SwiGLU path). Each composes epilogue primitives of
// the single-operator kernels: the delayed row scale with the RoPE or SwiGLU
// pair map in the forward; the row statistic with the SwiGLU backward, and the
// residual-stream gradient with the RMSNorm backward, in the backward.
#include "gemm_launch.cuh"

using namespace coda;

extern "C" {

int coda_gemm_rowscale_rope(int M, int N, int K, const coda_bf16* X, const coda_bf16* W, const float* r,
                            const float* cos_tab, const float* sin_tab, int S, int head_dim, int rope_cols,
                            coda_bf16* out, coda_stream_t stream) {
  const char* fn = "coda_gemm_rowscale_rope";
  int rc = check_fused(fn, M, N, K, X, W);
  if (rc) return rc;
  CODA_REQUIRE(head_dim > 0 && head_dim % 32 == 0, CODA_ERR_UNSUPPORTED,
               "%s: head_dim=%d must be a positive multiple of 32", fn, head_dim);
  CODA_REQUIRE(rope_cols >= 0 && rope_cols % head_dim == 0 && rope_cols <= N, CODA_ERR_INVALID,
               "%s: rope_cols=%d must be a multiple of head_dim in [0, N]", fn, rope_cols);
  CODA_REQUIRE(S > 0, CODA_ERR_INVALID, "%s: S=%d must be positive", fn, S);
  if (M == 0 || N == 0) return CODA_OK;
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR16(cos_tab);
  CODA_REQ_PTR16(sin_tab);
  CODA_REQ_PTR16(out);
  CUtensorMap o;
  if ((rc = make_out_map(&o, out, M, N, N))) return rc;
  using E = EpiRope<1, true>;
  E::Params ep{cos_tab, sin_tab, S, head_dim, rope_cols, rope_lane_tables(S, head_dim), r};
  return launch_fused<E>(fn, M, N, K, X, K, 0, W, N, /*b_mn=*/1, o, o, o, o, ep, as_stream(stream));
}

int coda_gemm_rowscale_swiglu(int M, int F, int K, const coda_bf16* X, const coda_bf16* Wgu, const float* r,
                              coda_bf16* A_out, coda_bf16* gu_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_rowscale_swiglu";
  CODA_REQUIRE(F >= 0 && F <= (1 << 30), CODA_ERR_INVALID, "%s: F=%d out of range", fn, F);
  int rc = check_fused(fn, M, 2 * F, K, X, Wgu);
  if (rc) return rc;
  CODA_REQUIRE(F % 8 == 0, CODA_ERR_UNSUPPORTED, "%s: F=%d must be a multiple of 8", fn, F);
  if (M == 0 || F == 0) return CODA_OK;
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR16(A_out);
  CODA_REQ_OPT16(gu_out);
  CUtensorMap o, og;
  if ((rc = make_out_map(&o, A_out, M, F, F))) return rc;
  og = o;
  if (gu_out && (rc = make_out_map(&og, gu_out, M, 2 * F, 2 * F))) return rc;
  if (gu_out) {
    using E = EpiSwiGLU<true, true>;
    E::Params ep{0, r};
    return launch_fused<E>(fn, M, 2 * F, K, X, K, 0, Wgu, 2 * F, /*b_mn=*/1, o, og, o, o, ep, as_stream(stream));
  }
  using E = EpiSwiGLU<false, true>;
  E::Params ep{0, r};
  return launch_fused<E>(fn, M, 2 * F, K, X, K, 0, Wgu, 2 * F, /*b_mn=*/1, o, og, o, o, ep, as_stream(stream));
}

int coda_gemm_swiglu_bwd_rowdot(int M, int F, int K, const coda_bf16* dY, const coda_bf16* Wd, const coda_bf16* gu,
                                const float* r, coda_bf16* dgur_out, float* pdot_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_swiglu_bwd_rowdot";
  int rc = check_fused(fn, M, F, K, dY, Wd);
  if (rc) return rc;
  if (M == 0 || F == 0) return CODA_OK;
  CODA_REQ_PTR16(gu);
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR16(dgur_out);
  CODA_REQ_PTR4(pdot_out);
  CUtensorMap o, ig;
  if ((rc = make_wide_map(&o, dgur_out, M, 2 * F, 2 * F))) return rc;
  if ((rc = make_wide_map(&ig, gu, M, 2 * F, 2 * F))) return rc;
  const auto* g = reinterpret_cast<const __nv_bfloat16*>(gu);
  // dA = dY Wd^T: Wd is stored [F, K] = [N, K], a K-major B operand.
  if (K <= kDeepRingMaxK) {
    using E = EpiSwiGLUBwdRowdot<8192>;
    return launch_fused<E>(fn, M, F, K, dY, K, 0, Wd, K, /*b_mn=*/0, o, o, ig, ig, E::Params{g, r, pdot_out},
                           as_stream(stream));
  }
  using E = EpiSwiGLUBwdRowdot<>;
  return launch_fused<E>(fn, M, F, K, dY, K, 0, Wd, K, /*b_mn=*/0, o, o, ig, ig, E::Params{g, r, pdot_out},
                         as_stream(stream));
}

int coda_gemm_rmsnorm_bwd_res(int M, int d, int K, const coda_bf16* dYr, const coda_bf16* W1, const coda_bf16* h,
                              const coda_bf16* gamma, const float* r, const float* s, const coda_bf16* dres,
                              coda_bf16* dh_out, float* pdg_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_rmsnorm_bwd_res";
  int rc = check_fused(fn, M, d, K, dYr, W1);
  if (rc) return rc;
  if (M == 0 || d == 0) return CODA_OK;
  CODA_REQ_PTR16(h);
  CODA_REQ_PTR16(gamma);
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR4(s);
  CODA_REQ_PTR16(dres);
  CODA_REQ_PTR16(dh_out);
  CODA_REQ_PTR4(pdg_out);
  CUtensorMap o, ih, ir;
  if ((rc = make_out_map(&o, dh_out, M, d, d))) return rc;
  if ((rc = make_out_map(&ih, h, M, d, d))) return rc;
  if ((rc = make_out_map(&ir, dres, M, d, d))) return rc;
  const auto* hb = reinterpret_cast<const __nv_bfloat16*>(h);
  const auto* gb = reinterpret_cast<const __nv_bfloat16*>(gamma);
  // Gr = dYr W1^T: W1 is stored [d, K] = [N, K], a K-major B operand.
  if (K <= kDeepRingMaxK) {
    using E = EpiRmsNormBwdRes<8192>;
    return launch_fused<E>(fn, M, d, K, dYr, K, 0, W1, K, /*b_mn=*/0, o, o, ih, ir, E::Params{hb, gb, r, s, pdg_out},
                           as_stream(stream));
  }
  using E = EpiRmsNormBwdRes<>;
  return launch_fused<E>(fn, M, d, K, dYr, K, 0, W1, K, /*b_mn=*/0, o, o, ih, ir, E::Params{hb, gb, r, s, pdg_out},
                         as_stream(stream));
}

}  // extern "C"
