// Backward GEMM entry points: SwiGLU backward, the row statistic in the
// dY-producing GEMM, RMSNorm backward in the data-gradient GEMM, and the
// cross-entropy forward (partials) and backward (dl) GEMMs.
#include "gemm_launch.cuh"

using namespace coda;

extern "C" {

int coda_gemm_swiglu_bwd(int M, int F, int K, const coda_bf16* dY, const coda_bf16* Wd, const coda_bf16* gu,
                         coda_bf16* dgu_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_swiglu_bwd";
  int rc = check_fused(fn, M, F, K, dY, Wd);
  if (rc) return rc;
  if (M == 0 || F == 0) return CODA_OK;
  CODA_REQ_PTR16(gu);
  CODA_REQ_PTR16(dgu_out);
  CUtensorMap o;
  if ((rc = make_wide_map(&o, dgu_out, M, 2 * F, 2 * F))) return rc;
  CUtensorMap ig;
  if ((rc = make_wide_map(&ig, gu, M, 2 * F, 2 * F))) return rc;
  const auto* g = reinterpret_cast<const __nv_bfloat16*>(gu);
  // dA = dY Wd^T: Wd is stored [F, K] = [N, K], a K-major B operand.
  if (K <= kDeepRingMaxK) {
    using E = EpiSwiGLUBwd<8192>;
    return launch_fused<E>(fn, M, F, K, dY, K, 0, Wd, K, /*b_mn=*/0, o, o, ig, ig, E::Params{g}, as_stream(stream));
  }
  using E = EpiSwiGLUBwd<>;
  return launch_fused<E>(fn, M, F, K, dY, K, 0, Wd, K, /*b_mn=*/0, o, o, ig, ig, E::Params{g}, as_stream(stream));
}

int coda_gemm_rowdot(int M, int N, int K, const coda_bf16* dO, const coda_bf16* Wn, const coda_bf16* Y,
                     const float* r, coda_bf16* dY_out, coda_bf16* dYr_out, float* pdot_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_rowdot";
  int rc = check_fused(fn, M, N, K, dO, Wn);
  if (rc) return rc;
  if (M == 0 || N == 0) return CODA_OK;
  CODA_REQ_PTR16(Y);
  CODA_REQ_PTR16(dY_out);
  CODA_REQ_OPT16(dYr_out);
  CODA_REQ_PTR4(pdot_out);
  if (dYr_out) CODA_REQ_PTR4(r);
  CUtensorMap o0, o1;
  if ((rc = make_out_map(&o0, dY_out, M, N, N))) return rc;
  if (dYr_out) {
    if ((rc = make_out_map(&o1, dYr_out, M, N, N))) return rc;
  } else {
    o1 = o0;
  }
  CUtensorMap iy;
  if ((rc = make_out_map(&iy, Y, M, N, N))) return rc;
  EpiRowdot::Params ep{reinterpret_cast<const __nv_bfloat16*>(Y), r, pdot_out, dYr_out != nullptr};
  return launch_fused<EpiRowdot>(fn, M, N, K, dO, K, 0, Wn, N, /*b_mn=*/1, o0, o1, iy, iy, ep, as_stream(stream));
}

int coda_gemm_rmsnorm_bwd(int M, int d, int K, const coda_bf16* dY, const coda_bf16* W1, const coda_bf16* h1,
                          const coda_bf16* gamma, const float* r, const float* s, coda_bf16* dh1_out, float* pdg_out,
                          coda_stream_t stream) {
  const char* fn = "coda_gemm_rmsnorm_bwd";
  int rc = check_fused(fn, M, d, K, dY, W1);
  if (rc) return rc;
  if (M == 0 || d == 0) return CODA_OK;
  CODA_REQ_PTR16(h1);
  CODA_REQ_PTR16(gamma);
  CODA_REQ_PTR4(r);
  CODA_REQ_PTR4(s);
  CODA_REQ_PTR16(dh1_out);
  CODA_REQ_PTR4(pdg_out);
  CUtensorMap o;
  if ((rc = make_out_map(&o, dh1_out, M, d, d))) return rc;
  CUtensorMap ih;
  if ((rc = make_out_map(&ih, h1, M, d, d))) return rc;
  EpiRmsNormBwd::Params ep{reinterpret_cast<const __nv_bfloat16*>(h1), reinterpret_cast<const __nv_bfloat16*>(gamma),
                           r, s, pdg_out};
  // G = dY W1^T: W1 is stored [d, K] = [N, K], a K-major B operand.
  return launch_fused<EpiRmsNormBwd>(fn, M, d, K, dY, K, 0, W1, K, /*b_mn=*/0, o, o, ih, ih, ep, as_stream(stream));
}

int coda_gemm_ce_lse(int M, int V, int K, const coda_bf16* H, const coda_bf16* W, const int32_t* labels,
                     float* pmax_out, float* psum_out, int32_t* parg_out, float* tgt_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_ce_lse";
  int rc = check_fused(fn, M, V, K, H, W);
  if (rc) return rc;
  CODA_REQUIRE(M == 0 || V > 0, CODA_ERR_INVALID, "%s: V must be positive", fn);
  if (M == 0) return CODA_OK;
  CODA_REQ_PTR4(labels);
  CODA_REQ_PTR4(pmax_out);
  CODA_REQ_PTR4(psum_out);
  CODA_REQ_OPT4(parg_out);
  CODA_REQ_PTR4(tgt_out);
  const DeviceInfo* di = current_device();
  if (!di) return CODA_ERR_UNSUPPORTED;
  CUtensorMap o;
  memset(&o, 0, sizeof(o));
  EpiCeLse::Params ep{labels, pmax_out, psum_out, parg_out, tgt_out, di->status};
  return launch_fused<EpiCeLse>(fn, M, V, K, H, K, 0, W, V, /*b_mn=*/1, o, o, o, o, ep, as_stream(stream));
}

int coda_gemm_ce_bwd(int M, int V, int K, const coda_bf16* H, const coda_bf16* W, const int32_t* labels,
                     const float* lse, float grad_scale, coda_bf16* dl_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_ce_bwd";
  int rc = check_fused(fn, M, V, K, H, W);
  if (rc) return rc;
  if (M == 0 || V == 0) return CODA_OK;
  CODA_REQ_PTR4(labels);
  CODA_REQ_PTR4(lse);
  CODA_REQ_PTR16(dl_out);
  CUtensorMap o;
  if ((rc = make_out_map(&o, dl_out, M, V, V))) return rc;
  EpiCeBwd::Params ep{labels, lse, grad_scale};
  return launch_fused<EpiCeBwd>(fn, M, V, K, H, K, 0, W, V, /*b_mn=*/1, o, o, o, o, ep, as_stream(stream));
}

}  // extern "C"
