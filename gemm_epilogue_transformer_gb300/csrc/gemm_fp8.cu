// FP8 (E4M3) mainloop variants of the single-GEMM forward operators, with the
// same epilogue programs as their bf16 twins (CODA note, research background:
// as low-precision GEMMs multiply the tensor throughput, the memory-bound
// operators around them take a larger share of the time, which the fused
// epilogues remove). Operands are K-major E4M3 with per-tensor scales; the
// accumulator is scaled by alpha = scale_A * scale_B before the epilogue.
#include "gemm_launch.cuh"

using namespace coda;

namespace {

// Checks shared by the FP8 entry points: dims, 16-byte rows of the K-major
// E4M3 operands (K % 16) and of the bf16 outputs (N % 8), a finite alpha.
int check_fp8(const char* fn, int M, int N, int K, const void* A, const void* B, float alpha) {
  CODA_REQUIRE(M >= 0 && N >= 0 && K >= 0, CODA_ERR_INVALID, "%s: negative dimension (M=%d N=%d K=%d)", fn, M, N, K);
  CODA_REQUIRE(K % 16 == 0, CODA_ERR_UNSUPPORTED, "%s: K=%d must be a multiple of 16 (16-byte FP8 rows)", fn, K);
  CODA_REQUIRE(N % 8 == 0, CODA_ERR_UNSUPPORTED, "%s: N=%d must be a multiple of 8", fn, N);
  CODA_REQUIRE(alpha == alpha && alpha - alpha == 0.0f, CODA_ERR_INVALID, "%s: alpha must be finite", fn);
  if (M > 0 && N > 0 && K > 0) {
    CODA_REQ_PTR16(A);
    CODA_REQ_PTR16(B);
  }
  return CODA_OK;
}

}  // namespace

extern "C" {

int coda_gemm_fp8(int M, int N, int K, const uint8_t* A, const uint8_t* B, float alpha, coda_bf16* C,
                  coda_stream_t stream) {
  const char* fn = "coda_gemm_fp8";
  int rc = check_fp8(fn, M, N, K, A, B, alpha);
  if (rc || M == 0 || N == 0) return rc;
  CODA_REQ_PTR16(C);
  CUtensorMap o;
  if ((rc = make_out_map(&o, C, M, N, N))) return rc;
  EpiPlain::Params ep{0};
  return launch_fused<EpiPlain, true>(fn, M, N, K, A, K, 0, B, K, 0, o, o, o, o, ep, as_stream(stream), alpha);
}

int coda_gemm_rope_fp8(int M, int N, int K, const uint8_t* X, const uint8_t* W, float alpha, const float* cos_tab,
                       const float* sin_tab, int S, int head_dim, int rope_cols, coda_bf16* out, coda_stream_t stream) {
  const char* fn = "coda_gemm_rope_fp8";
  int rc = check_fp8(fn, M, N, K, X, W, alpha);
  if (rc) return rc;
  CODA_REQUIRE(head_dim > 0 && head_dim % 32 == 0, CODA_ERR_UNSUPPORTED,
               "%s: head_dim=%d must be a positive multiple of 32", fn, head_dim);
  CODA_REQUIRE(rope_cols >= 0 && rope_cols % head_dim == 0 && rope_cols <= N, CODA_ERR_INVALID,
               "%s: rope_cols=%d must be a multiple of head_dim in [0, N]", fn, rope_cols);
  CODA_REQUIRE(S > 0, CODA_ERR_INVALID, "%s: S=%d must be positive", fn, S);
  if (M == 0 || N == 0) return CODA_OK;
  CODA_REQ_PTR16(cos_tab);
  CODA_REQ_PTR16(sin_tab);
  CODA_REQ_PTR16(out);
  CUtensorMap o;
  if ((rc = make_out_map(&o, out, M, N, N))) return rc;
  EpiRope<1>::Params ep{cos_tab, sin_tab, S, head_dim, rope_cols, rope_lane_tables(S, head_dim), nullptr};
  return launch_fused<EpiRope<1>, true>(fn, M, N, K, X, K, 0, W, K, 0, o, o, o, o, ep, as_stream(stream), alpha);
}

int coda_gemm_swiglu_fp8(int M, int F, int K, const uint8_t* X, const uint8_t* Wgu, float alpha, coda_bf16* A_out,
                         coda_bf16* gu_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_swiglu_fp8";
  CODA_REQUIRE(F >= 0 && F <= (1 << 30), CODA_ERR_INVALID, "%s: F=%d out of range", fn, F);
  int rc = check_fp8(fn, M, 2 * F, K, X, Wgu, alpha);
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
    EpiSwiGLU<true>::Params ep{0, nullptr};
    return launch_fused<EpiSwiGLU<true>, true>(fn, M, 2 * F, K, X, K, 0, Wgu, K, 0, o, og, o, o, ep,
                                               as_stream(stream), alpha);
  }
  EpiSwiGLU<false>::Params ep{0, nullptr};
  return launch_fused<EpiSwiGLU<false>, true>(fn, M, 2 * F, K, X, K, 0, Wgu, K, 0, o, og, o, o, ep, as_stream(stream),
                                              alpha);
}

int coda_gemm_ce_lse_fp8(int M, int V, int K, const uint8_t* H, const uint8_t* W, float alpha, const int32_t* labels,
                         float* pmax_out, float* psum_out, int32_t* parg_out, float* tgt_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_ce_lse_fp8";
  int rc = check_fp8(fn, M, V, K, H, W, alpha);
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
  return launch_fused<EpiCeLse, true>(fn, M, V, K, H, K, 0, W, K, 0, o, o, o, o, ep, as_stream(stream), alpha);
}

int coda_gemm_ce_bwd_fp8(int M, int V, int K, const uint8_t* H, const uint8_t* W, float alpha, const int32_t* labels,
                         const float* lse, float grad_scale, coda_bf16* dl_out, coda_stream_t stream) {
  const char* fn = "coda_gemm_ce_bwd_fp8";
  int rc = check_fp8(fn, M, V, K, H, W, alpha);
  if (rc || M == 0 || V == 0) return rc;
  CODA_REQ_PTR4(labels);
  CODA_REQ_PTR4(lse);
  CODA_REQ_PTR16(dl_out);
  CUtensorMap o;
  if ((rc = make_out_map(&o, dl_out, M, V, V))) return rc;
  EpiCeBwd::Params ep{labels, lse, grad_scale};
  return launch_fused<EpiCeBwd, true>(fn, M, V, K, H, K, 0, W, K, 0, o, o, o, o, ep, as_stream(stream), alpha);
}

}  // extern "C"
