// Epilogue programs: what runs on a 128 x 256 fp32 accumulator tile after the
// mainloop and before the global store (CODA note, Key design 4: element/pair
// maps, rank-1 loads, rank-2 tile loads/stores, tile partial reductions,
// stateful transforms).
//
// Thread layout inside an epilogue warp: lane = one accumulator row, a chunk =
// 32 consecutive columns of that row in registers (acc[32]). Pairs (2i, 2i+1)
// therefore always sit in the same thread, and per-row partial reductions are
// thread-local; per-column partials use a warp transpose-reduce.
#pragma once

#include "gemm_core.cuh"

namespace coda {

constexpr float kLog2e = 1.4426950408889634f;

// e^x = 2^(x log2 e) and 1 / x from the hardware approximations of the PTX
// ISA (ex2.approx.ftz.f32, rcp.approx.ftz.f32; relative error near 2^-22,
// far below the bf16 outputs' 2^-9 and the fp32 statistics' 1e-4). Results
// below the normal range flush to zero, the correct limit for the softmax
// terms and the sigmoid.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float exp_f(float x) { return ex2_approx(x * kLog2e); }
// 1 / (1 + e^-g); for g below about -88 the denominator is +inf and the result
// 0, for g above about 88 it is 1: the correct limits.
__device__ __forceinline__ float sigmoid_f(float g) { return rcp_approx(1.0f + exp_f(-g)); }

// Two fp32 lanes per instruction (the sm_100 family's packed f32x2 forms):
// each lane rounds exactly as the scalar multiply, add or fused multiply-add.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }
// sigmoid_f on two lanes
__device__ __forceinline__ float2 sigmoid2(float2 g) {
  const float2 t = mul2(g, splat2(-kLog2e));
  const float2 den = add2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), splat2(1.0f));
  return make_float2(rcp_approx(den.x), rcp_approx(den.y));
}
// Gate and up values of features j and j+1 from their stored pair words
// (bf16 G at the even column, the lower half of the word; U the upper half).
__device__ __forceinline__ void gu_unpack2(uint32_t wj, uint32_t wj1, float2& G, float2& U) {
  G = make_float2(bf16_lo(wj), bf16_lo(wj1));
  U = make_float2(bf16_hi(wj), bf16_hi(wj1));
}
// SwiGLU backward of two features: with s = sigmoid(G),
// dG = (dA s) U (1 + G (1 - s)), dU = (dA s) G.
__device__ __forceinline__ void swiglu_bwd2(float2 dA, float2 G, float2 U, float2& dG, float2& dU) {
  const float2 s = sigmoid2(G);
  const float2 as = mul2(dA, s);
  dU = mul2(as, G);
  const float2 q = fma2(G, fma2(s, splat2(-1.0f), splat2(1.0f)), splat2(1.0f));
  dG = mul2(mul2(as, U), q);
}
// Write 16 packed words (32 bf16) as one 64-byte staging row.
__device__ __forceinline__ void stage_words16(uint32_t box, int r, const uint32_t (&w)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) stage_put(box, r, q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}
__device__ __forceinline__ void words16(const uint4 (&u)[4], uint32_t (&w)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    w[4 * q] = u[q].x;
    w[4 * q + 1] = u[q].y;
    w[4 * q + 2] = u[q].z;
    w[4 * q + 3] = u[q].w;
  }
}

// Shared-memory trade: an epilogue may declare kStageBufs = 1 (single-buffered
// store staging), kInRingBytes = 4096 (a smaller input ring) or kMaxSlots = 1
// (one store box per chunk). Each frees room for a sixth mainloop stage on SM
// pairs; measured 1.5-3.5 % faster for the one-box input epilogues and for
// SwiGLU with its GU side output than five stages with the larger buffers.
// The two-box input epilogues (SwiGLU backward, RMSNorm backward with the
// residual gradient) take the ring size as a template argument: 4096 bytes
// (one chunk of inputs in flight, six stages) or 8192 (two chunks, five
// stages). With one chunk in flight each chunk waits a full HBM round trip,
// which a short mainloop cannot hide: at K = 2048 the SwiGLU backward ran 14 %
// slower with the small ring, at K = 4096 2 % faster. The launchers pick by K
// (gemm_launch.cuh, kDeepRingMaxK).

// Epilogues without global inputs carry an empty prefetch buffer.
struct NoPre {
  uint32_t unused;
};
#define CODA_NO_PREFETCH                                                            \
  using Pre = NoPre;                                                                \
  __device__ static void prefetch(const Params&, const EpiCtx&, int, Pre&) {}
#define CODA_NO_INPUT                                                                                   \
  static constexpr int kInBoxes = 0;                                                                    \
  __device__ static bool has_input(const Params&, const EpiCtx&, int) { return false; }                 \
  __device__ static void in_coord(const Params&, const EpiCtx&, int, int, int& map, int& x, int& y) {  \
    map = 0;                                                                                            \
    x = 0;                                                                                              \
    y = 0;                                                                                              \
  }
// One bf16 input box per chunk: the 32 x 32 block of a [M, N] tensor under the
// warp's rows and the chunk's columns.
#define CODA_INPUT_SAME_TILE                                                                             \
  static constexpr int kInBoxes = 1;                                                                     \
  __device__ static bool has_input(const Params&, const EpiCtx&, int) { return true; }                   \
  __device__ static void in_coord(const Params&, const EpiCtx& cx, int c, int, int& map, int& x, int& y) { \
    map = 0;                                                                                             \
    x = cx.n0 + 32 * c;                                                                                  \
    y = cx.wrow0;                                                                                        \
  }

// Sum each of the 32 columns held by the warp's 32 rows; afterwards lane j
// holds the total of column j in v[0]. 31 shuffles per thread.
__device__ __forceinline__ float warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// Default store coordinates: one full 32-column box per chunk per slot.
#define CODA_STORE_SAME_COLS(MAP1)                                                                           \
  __device__ static void store_coord(const Params&, const EpiCtx& cx, int c, int s, int& map, int& x, int& y) { \
    map = (s == 0) ? 0 : (MAP1);                                                                             \
    x = cx.n0 + 32 * c;                                                                                      \
    y = cx.wrow0;                                                                                            \
  }

// ------------------------------------------------------------------ identity
struct EpiPlain {
  struct Params {
    int unused;
  };
  struct State {};
  CODA_NO_PREFETCH
  CODA_NO_INPUT
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 2;
  __device__ static int slots(const Params&) { return 1; }
  __device__ static void begin(State&, const Params&, const EpiCtx&) {}
  __device__ static void chunk(State&, const Params&, const EpiCtx& cx, int, float (&acc)[32], const Pre&, uint32_t,
                               uint32_t box0, uint32_t) {
    stage_row32(box0, cx.lane, acc);
  }
  CODA_STORE_SAME_COLS(0)
  __device__ static void end(State&, const Params&, const EpiCtx&) {}
};

// ------------------------------------------- residual + gamma + sum of squares
// h1 = acc + z; psq += h1^2 (fp32 h1, unscaled); h2 = h1 * gamma.
// (CODA note, Key design 1; the partial is measured on the unscaled output.)
struct EpiResRmsPrep {
  struct Params {
    const __nv_bfloat16* z;
    const __nv_bfloat16* gamma;
    float* psq;
  };
  struct State {
    float sumsq;
  };
  struct Pre {
    uint4 g[4];
  };
  __device__ static void prefetch(const Params& ep, const EpiCtx& cx, int c, Pre& pr) {
    load_raw32(ep.gamma, 0, 1, cx.N, 0, cx.n0 + 32 * c, pr.g);
  }
  CODA_INPUT_SAME_TILE  // z
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 2;
  static constexpr int kStageBufs = 1;
  static constexpr int kInRingBytes = 4096;
  __device__ static int slots(const Params&) { return 2; }
  __device__ static void begin(State& st, const Params&, const EpiCtx&) { st.sumsq = 0.f; }
  __device__ static void chunk(State& st, const Params&, const EpiCtx& cx, int, float (&acc)[32], const Pre& pr,
                               uint32_t in, uint32_t box0, uint32_t box1) {
    float v[32];
    uint4 u[4];
    box_row(in, cx.lane, u);
    unpack32(u, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      acc[i] += v[i];
      st.sumsq = fmaf(acc[i], acc[i], st.sumsq);
    }
    stage_row32(box0, cx.lane, acc);
    unpack32(pr.g, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] *= v[i];
    stage_row32(box1, cx.lane, acc);
  }
  CODA_STORE_SAME_COLS(1)
  __device__ static void end(State& st, const Params& ep, const EpiCtx& cx) {
    const long i = static_cast<long>(cx.row) * cx.n_blocks + cx.n_blk;
    if (cx.row < cx.M && CODA_IN(cx, i, static_cast<long>(cx.M) * cx.n_blocks)) ep.psq[i] = st.sumsq;
  }
};

// ------------------------------------------------------- delayed row scale
// Y[i,j] = r[i] * acc[i,j] (CODA note, Key design 1).
struct EpiRowScale {
  struct Params {
    const float* r;
  };
  struct State {
    float rv;
  };
  CODA_NO_PREFETCH
  CODA_NO_INPUT
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 2;
  __device__ static int slots(const Params&) { return 1; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    st.rv = (cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) ? ep.r[cx.row] : 0.f;
  }
  __device__ static void chunk(State& st, const Params&, const EpiCtx& cx, int, float (&acc)[32], const Pre&,
                               uint32_t, uint32_t box0, uint32_t) {
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] *= st.rv;
    stage_row32(box0, cx.lane, acc);
  }
  CODA_STORE_SAME_COLS(0)
  __device__ static void end(State&, const Params&, const EpiCtx&) {}
};

// ---------------------------------------------------------------- SwiGLU fwd
// Even column = gate G, odd = up U; out[f] = silu(G) * U; the 32 accumulator
// columns of a chunk give 16 outputs, two chunks fill one 32-column store box
// (CODA note, Key design 2: halve the width and compact before the store).
// kSaveGU: also store the pre-activation GU (bf16) for the backward, one more
// store box per chunk (a separate instantiation: the extra staging box costs
// one mainloop stage, which the plain forward keeps).
// kScale: the delayed RMSNorm row scale of the block chain, GU = r[i] * acc,
// applied before the pair map (CODA note, Key design 1 composed with Key
// design 2); the saved GU is the scaled pre-activation.
template <bool kSaveGU, bool kScale = false>
struct EpiSwiGLU {
  struct Params {
    int unused;
    const float* r;  // kScale only
  };
  struct State {
    float rv;
  };
  CODA_NO_PREFETCH
  CODA_NO_INPUT
  static constexpr int kChunksPerStore = 2;
  static constexpr int kMaxSlots = kSaveGU ? 3 : 2;
  static constexpr int kStageBufs = kSaveGU ? 1 : 2;
  // slot 0: A (32 outputs from two chunks); slots 1, 2: GU of the two chunks
  __device__ static int slots(const Params&) { return kSaveGU ? 3 : 1; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    if constexpr (kScale) st.rv = (cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) ? ep.r[cx.row] : 0.f;
  }
  __device__ static void chunk(State& st, const Params&, const EpiCtx& cx, int c, float (&acc)[32], const Pre&,
                               uint32_t, uint32_t box0, uint32_t) {
    if constexpr (kScale) {
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] *= st.rv;
    }
    if (kSaveGU) stage_row32(box0 + (1 + (c & 1)) * kStageBoxBytes, cx.lane, acc);
    float o[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float g = acc[2 * k], u = acc[2 * k + 1];
      o[k] = g * sigmoid_f(g) * u;
    }
    const int h = 2 * (c & 1);
    stage_put(box0, cx.lane, h + 0, pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]),
              pack_bf16(o[6], o[7]));
    stage_put(box0, cx.lane, h + 1, pack_bf16(o[8], o[9]), pack_bf16(o[10], o[11]), pack_bf16(o[12], o[13]),
              pack_bf16(o[14], o[15]));
  }
  __device__ static void store_coord(const Params&, const EpiCtx& cx, int c, int s, int& map, int& x, int& y) {
    y = cx.wrow0;
    if (s == 0) {
      map = 0;
      x = cx.n0 / 2 + 16 * (c - 1);
    } else {
      map = 1;
      x = cx.n0 + 32 * (c - 2 + s);
    }
  }
  __device__ static void end(State&, const Params&, const EpiCtx&) {}
};

// ---------------------------------------------------------------- SwiGLU bwd
// acc = dA[:, f0..f0+31]; loads the saved GU pairs, recomputes sigmoid(G), and
// emits interleaved (dG, dU) for 64 output columns. The chunk's 64 GU columns
// arrive as one 32 x 128-byte box and its 64 outputs leave as one, with the
// 128-byte swizzle: half the TMA requests of two 64-byte boxes.
// (pith page, Figure 7: one incoming gradient -> both paired input gradients.)
template <int kRing = 4096>
struct EpiSwiGLUBwd {
  struct Params {
    const __nv_bfloat16* gu;  // [M, 2F]
  };
  struct State {};
  CODA_NO_PREFETCH
  static constexpr int kInBoxes = 2;  // ring bytes per chunk: two 64-byte boxes' worth
  static constexpr int kInLoads = 1;  // filled by one 128-byte box
  __device__ static bool has_input(const Params&, const EpiCtx&, int) { return true; }
  __device__ static void in_coord(const Params&, const EpiCtx& cx, int c, int, int& map, int& x, int& y) {
    map = 0;
    x = 2 * (cx.n0 + 32 * c);
    y = cx.wrow0;
  }
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 2;  // staging bytes of two 64-byte boxes, stored as one 128-byte box
  static constexpr int kStageBufs = 1;
  static constexpr int kInRingBytes = kRing;  // 4096: one chunk of inputs in flight; 8192: two
  __device__ static int slots(const Params&) { return 1; }
  __device__ static void begin(State&, const Params&, const EpiCtx&) {}
  __device__ static void chunk(State&, const Params&, const EpiCtx& cx, int, float (&acc)[32], const Pre&,
                               uint32_t in, uint32_t box0, uint32_t) {
    uint4 u[8];
    box128_row(in, cx.lane, u);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        w[4 * q] = u[4 * half + q].x;
        w[4 * q + 1] = u[4 * half + q].y;
        w[4 * q + 2] = u[4 * half + q].z;
        w[4 * q + 3] = u[4 * half + q].w;
      }
      // features j, j+1 as two-lane vectors; each (dG, dU) pair packs into one word
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        float2 G, U, dG, dU;
        gu_unpack2(w[j], w[j + 1], G, U);
        swiglu_bwd2(make_float2(acc[16 * half + j], acc[16 * half + j + 1]), G, U, dG, dU);
        w[j] = pack_bf16(dG.x, dU.x);
        w[j + 1] = pack_bf16(dG.y, dU.y);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        stage128_put(box0, cx.lane, 4 * half + q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
  }
  __device__ static void store_coord(const Params&, const EpiCtx& cx, int c, int, int& map, int& x, int& y) {
    map = 0;
    x = 2 * (cx.n0 + 32 * c);
    y = cx.wrow0;
  }
  __device__ static void end(State&, const Params&, const EpiCtx&) {}
};

// ---------------------------------------------------------------- RoPE
// Adjacent pairs (2i, 2i+1) within each head of the first rope_cols columns,
// position = row mod S, cos/sin from the caller's fp32 tables [S, head_dim/2].
// kSign = +1: forward rotation; -1: transposed rotation (backward).
// kScale: the delayed RMSNorm row scale of the block chain, out = RoPE(r[i] *
// acc) (CODA note, Key design 1 composed with Key design 2; the row scale
// commutes with the per-row rotation).
//
// Table traffic. A warp's 32 rows are positions p0 + l, l = 0..31. When S is a
// multiple of 32 (no wrap inside a warp) and head_dim <= 128, the angle of
// position p0 + l is the sum of the angles of p0 and of l, so
//   cos((p0+l) w) = cos(p0 w) cos(l w) - sin(p0 w) sin(l w),
//   sin((p0+l) w) = sin(p0 w) cos(l w) + cos(p0 w) sin(l w).
// Table rows 0..31 (the l factors) are copied into shared memory once per CTA;
// per chunk a warp reads only row p0's 16 cos and 16 sin values (one broadcast
// load each). That replaces 4 KiB of table reads per warp and chunk from L2 by
// 128 bytes. Otherwise each row loads its own 16 + 16 values directly.
// Requires tables of angles linear in the position, cos_tab[p, i] =
// cos(p * w_i), as coda_rope_tables writes them.
template <int kSign, bool kScale = false>
struct EpiRope {
  struct Params {
    const float* cos_tab;
    const float* sin_tab;
    int S, head_dim, rope_cols;
    int lane_tables;  // 1: angle addition with table rows 0..31 in shared memory; 0: per-row loads
    const float* r;   // kScale only
  };
  struct State {
    float rv;
  };
  // lane_tables: row p0's values (the same for the whole warp); else the row's own
  struct Pre {
    uint4 c[4], s[4];
  };
  CODA_NO_INPUT
  // Table rows 0..31 of cos and sin, 256 bytes per row (64 frequencies at
  // most); 16-byte granule j of row l sits at granule j ^ (l & 7), so the
  // warp's 32 row reads of one granule are conflict-free.
  static constexpr int kSharedBytes = 2 * 32 * 256;
  __device__ static uint32_t lane_addr(uint32_t base, int t, int l, int j) {
    return base + t * (32 * 256) + l * 256 + ((j ^ (l & 7)) << 4);
  }
  __device__ static void init_shared(const Params& ep, uint32_t base, int tid, int* status) {
    if (!ep.lane_tables) return;
    const int g = ep.head_dim >> 3;  // 16-byte granules per table row (head_dim / 2 floats)
    const long extent = static_cast<long>(ep.S) * (ep.head_dim >> 1);
    for (int idx = tid; idx < 2 * 32 * g; idx += 128) {
      const int t = idx / (32 * g), rem = idx - t * 32 * g;
      const int l = rem / g, j = rem - l * g;
      const long off = static_cast<long>(l) * (ep.head_dim >> 1) + 4 * j;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (CODA_IN_ST(status, off + 3, extent)) v = ldg_nc_v4((t ? ep.sin_tab : ep.cos_tab) + off);
      st_shared_v4(lane_addr(base, t, l, j), v.x, v.y, v.z, v.w);
    }
  }
  __device__ static void prefetch(const Params& ep, const EpiCtx& cx, int c, Pre& pr) {
    const int col0 = cx.n0 + 32 * c;
    if (col0 < ep.rope_cols) {
      const int pos = ep.lane_tables ? (cx.wrow0 % ep.S) : ((cx.row < cx.M) ? (cx.row % ep.S) : 0);
      const int half = ep.head_dim >> 1;
      const int i0 = (col0 % ep.head_dim) >> 1;
      const long off = static_cast<long>(pos) * half + i0;
      const float* cp = ep.cos_tab + off;
      const float* sp = ep.sin_tab + off;
      const bool in = CODA_IN(cx, off + 15, static_cast<long>(ep.S) * half);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        pr.c[q] = in ? ldg_nc_v4(cp + 4 * q) : make_uint4(0, 0, 0, 0);
        pr.s[q] = in ? ldg_nc_v4(sp + 4 * q) : make_uint4(0, 0, 0, 0);
      }
    }
  }
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 1;
  __device__ static int slots(const Params&) { return 1; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    if constexpr (kScale) st.rv = (cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) ? ep.r[cx.row] : 0.f;
  }
  __device__ static void chunk(State& st, const Params& ep, const EpiCtx& cx, int c, float (&acc)[32], const Pre& pr,
                               uint32_t, uint32_t box0, uint32_t) {
    const int col0 = cx.n0 + 32 * c;
    if constexpr (kScale) {
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] *= st.rv;
    }
    if (col0 < ep.rope_cols) {
      float cs[16], sn[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        cs[4 * q + 0] = __uint_as_float(pr.c[q].x);
        cs[4 * q + 1] = __uint_as_float(pr.c[q].y);
        cs[4 * q + 2] = __uint_as_float(pr.c[q].z);
        cs[4 * q + 3] = __uint_as_float(pr.c[q].w);
        sn[4 * q + 0] = __uint_as_float(pr.s[q].x);
        sn[4 * q + 1] = __uint_as_float(pr.s[q].y);
        sn[4 * q + 2] = __uint_as_float(pr.s[q].z);
        sn[4 * q + 3] = __uint_as_float(pr.s[q].w);
      }
      if (ep.lane_tables) {
        // (cs, sn) hold row p0's values: add the angle of this lane's offset
        const int j0 = ((col0 % ep.head_dim) >> 1) >> 2;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 lc = ld_shared_v4(lane_addr(cx.shared, 0, cx.lane, j0 + q));
          const uint4 ls = ld_shared_v4(lane_addr(cx.shared, 1, cx.lane, j0 + q));
          const float cl[4] = {__uint_as_float(lc.x), __uint_as_float(lc.y), __uint_as_float(lc.z),
                               __uint_as_float(lc.w)};
          const float sl[4] = {__uint_as_float(ls.x), __uint_as_float(ls.y), __uint_as_float(ls.z),
                               __uint_as_float(ls.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float cb = cs[4 * q + e], sb = sn[4 * q + e];
            cs[4 * q + e] = cb * cl[e] - sb * sl[e];
            sn[4 * q + e] = sb * cl[e] + cb * sl[e];
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float e = acc[2 * k], o = acc[2 * k + 1];
        const float s = kSign > 0 ? sn[k] : -sn[k];
        acc[2 * k] = e * cs[k] - o * s;
        acc[2 * k + 1] = e * s + o * cs[k];
      }
    }
    stage_row32(box0, cx.lane, acc);
  }
  CODA_STORE_SAME_COLS(0)
  __device__ static void end(State&, const Params&, const EpiCtx&) {}
};

// ---------------------------------------------------- cross-entropy forward
// Stateful online softmax over the tile's columns (CODA note, Key design 4):
// running max m and sum s of exp(l - m) per row, the tile argmax, and the
// target logit when the label falls in this tile. No tile is stored.
struct EpiCeLse {
  struct Params {
    const int32_t* labels;
    float* pmax;
    float* psum;
    int32_t* parg;  // nullable
    float* tgt;
    int* status;
  };
  struct State {
    float m, s;
    int best;
    int label;
  };
  CODA_NO_PREFETCH
  CODA_NO_INPUT
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 2;
  __device__ static int slots(const Params&) { return 0; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    st.m = -INFINITY;
    st.s = 0.f;
    st.best = -1;
    st.label = -1;
    if (cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) {
      st.label = ep.labels[cx.row];
      if (cx.n_blk == 0 && (st.label < 0 || st.label >= cx.N)) {
        atomicOr(ep.status, CODA_DEVST_BAD_LABEL);
        ep.tgt[cx.row] = __uint_as_float(0x7fc00000u);
      }
    }
  }
  __device__ static void chunk(State& st, const Params& ep, const EpiCtx& cx, int c, float (&acc)[32], const Pre&,
                               uint32_t, uint32_t, uint32_t) {
    const int col0 = cx.n0 + 32 * c;
    float cm = -INFINITY;
    int ci = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (col0 + j >= cx.N) acc[j] = -INFINITY;
      if (acc[j] > cm) {
        cm = acc[j];
        ci = j;
      }
    }
    if (cm > st.m) st.best = col0 + ci;
    const float nm = fmaxf(st.m, cm);
    if (nm != -INFINITY) {
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) sum += exp_f(acc[j] - nm);
      st.s = st.s * exp_f(st.m - nm) + sum;
      st.m = nm;
    }
    const int rel = st.label - col0;
    if (rel >= 0 && rel < 32 && cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) {
      float t = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j == rel) t = acc[j];
      ep.tgt[cx.row] = t;
    }
  }
  __device__ static void store_coord(const Params&, const EpiCtx&, int, int, int& map, int& x, int& y) {
    map = 0;
    x = 0;
    y = 0;
  }
  __device__ static void end(State& st, const Params& ep, const EpiCtx& cx) {
    const long i = static_cast<long>(cx.row) * cx.n_blocks + cx.n_blk;
    if (cx.row < cx.M && CODA_IN(cx, i, static_cast<long>(cx.M) * cx.n_blocks)) {
      ep.pmax[i] = st.m;
      ep.psum[i] = st.s;
      if (ep.parg) ep.parg[i] = st.best;
    }
  }
};

// --------------------------------------------------- cross-entropy backward
// dl = grad_scale * (exp(l - lse_row) - [j == label]) on the recomputed logits.
struct EpiCeBwd {
  struct Params {
    const int32_t* labels;
    const float* lse;
    float grad_scale;
  };
  struct State {
    int label;
    float lse;
  };
  CODA_NO_PREFETCH
  CODA_NO_INPUT
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 2;
  __device__ static int slots(const Params&) { return 1; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    const bool in = cx.row < cx.M && CODA_IN(cx, cx.row, cx.M);
    st.label = in ? ep.labels[cx.row] : -1;
    st.lse = in ? ep.lse[cx.row] : 0.f;
  }
  __device__ static void chunk(State& st, const Params& ep, const EpiCtx& cx, int c, float (&acc)[32], const Pre&,
                               uint32_t, uint32_t box0, uint32_t) {
    const int col0 = cx.n0 + 32 * c;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float pj = exp_f(acc[j] - st.lse);
      if (col0 + j == st.label) pj -= 1.0f;
      acc[j] = ep.grad_scale * pj;
    }
    stage_row32(box0, cx.lane, acc);
  }
  CODA_STORE_SAME_COLS(0)
  __device__ static void end(State&, const Params&, const EpiCtx&) {}
};

// ------------------------------------------ row statistic for RMSNorm backward
// In the GEMM that produces dY (CODA note, Key design 3): store dY, optionally
// dYr = r * dY, and the tile partial of sum_j dY[i,j] * Y[i,j].
struct EpiRowdot {
  struct Params {
    const __nv_bfloat16* Y;
    const float* r;  // nullable when dyr is not stored
    float* pdot;
    int store_dyr;
  };
  struct State {
    float dot, rv;
  };
  CODA_NO_PREFETCH
  CODA_INPUT_SAME_TILE  // Y
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 2;
  static constexpr int kStageBufs = 1;
  static constexpr int kInRingBytes = 4096;
  __device__ static int slots(const Params& ep) { return ep.store_dyr ? 2 : 1; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    st.dot = 0.f;
    st.rv = (ep.store_dyr && cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) ? ep.r[cx.row] : 0.f;
  }
  __device__ static void chunk(State& st, const Params& ep, const EpiCtx& cx, int, float (&acc)[32], const Pre&,
                               uint32_t in, uint32_t box0, uint32_t box1) {
    float y[32];
    uint4 u[4];
    box_row(in, cx.lane, u);
    unpack32(u, y);
#pragma unroll
    for (int i = 0; i < 32; ++i) st.dot = fmaf(acc[i], y[i], st.dot);
    stage_row32(box0, cx.lane, acc);
    if (ep.store_dyr) {
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] *= st.rv;
      stage_row32(box1, cx.lane, acc);
    }
  }
  CODA_STORE_SAME_COLS(1)
  __device__ static void end(State& st, const Params& ep, const EpiCtx& cx) {
    const long i = static_cast<long>(cx.row) * cx.n_blocks + cx.n_blk;
    if (cx.row < cx.M && CODA_IN(cx, i, static_cast<long>(cx.M) * cx.n_blocks)) ep.pdot[i] = st.dot;
  }
};

// ------------------------------------------------------ RMSNorm backward
// acc = G = dY W1^T. dh1 = r gamma G - r^2 s h1; column partial of r G h1 over
// the warp's 32 rows (the dgamma reduction's first level).
struct EpiRmsNormBwd {
  struct Params {
    const __nv_bfloat16* h1;
    const __nv_bfloat16* gamma;
    const float* r;
    const float* s;
    float* pdg;  // [ceil(M/32), d]
  };
  struct State {
    float rv, r2s;
  };
  struct Pre {
    uint4 g[4];
  };
  __device__ static void prefetch(const Params& ep, const EpiCtx& cx, int c, Pre& pr) {
    load_raw32(ep.gamma, 0, 1, cx.N, 0, cx.n0 + 32 * c, pr.g);
  }
  CODA_INPUT_SAME_TILE  // h1
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 1;
  static constexpr int kInRingBytes = 4096;
  __device__ static int slots(const Params&) { return 1; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    if (cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) {
      st.rv = ep.r[cx.row];
      st.r2s = st.rv * st.rv * ep.s[cx.row];
    } else {
      st.rv = 0.f;
      st.r2s = 0.f;
    }
  }
  __device__ static void chunk(State& st, const Params& ep, const EpiCtx& cx, int c, float (&acc)[32], const Pre& pr,
                               uint32_t in, uint32_t box0, uint32_t) {
    const int col0 = cx.n0 + 32 * c;
    float part[32];
    uint4 u[4];
    box_row(in, cx.lane, u);
    uint32_t hw[16], gw[16], w[16];
    words16(u, hw);
    words16(pr.g, gw);
    const float2 rv = splat2(st.rv), nr2s = splat2(-st.r2s);
    // columns 2j, 2j+1 as two-lane vectors: rG = r G; partial r G h; dh1 = gamma rG - r^2 s h1
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 h = make_float2(bf16_lo(hw[j]), bf16_hi(hw[j]));
      const float2 g = make_float2(bf16_lo(gw[j]), bf16_hi(gw[j]));
      const float2 rG = mul2(make_float2(acc[2 * j], acc[2 * j + 1]), rv);
      const float2 pt = mul2(rG, h);
      part[2 * j] = pt.x;
      part[2 * j + 1] = pt.y;
      const float2 o = fma2(g, rG, mul2(nr2s, h));
      w[j] = pack_bf16(o.x, o.y);
    }
    stage_words16(box0, cx.lane, w);
    const float tot = warp_colsum32(part, cx.lane);
    // rows past M contribute zeros; a warp slice that starts past M has no partial row
    const long ig = static_cast<long>(cx.wrow0 >> 5) * cx.N + col0 + cx.lane;
    if (cx.wrow0 < cx.M && col0 + cx.lane < cx.N && CODA_IN(cx, ig, static_cast<long>((cx.M + 31) >> 5) * cx.N))
      ep.pdg[ig] = tot;
  }
  CODA_STORE_SAME_COLS(0)
  __device__ static void end(State&, const Params&, const EpiCtx&) {}
};

// ------------------------------- SwiGLU backward with the row statistic
// Block chain, SwiGLU path: acc = dA[:, f0..f0+31] from dA = gh Wdn^T. As
// EpiSwiGLUBwd, plus the RMSNorm-backward row statistic of the rowscale GEMM
// that produced GU (CODA note, Key design 3: s = (1/d) rowsum(dGU (.) GU)
// formed in the GEMM that produces dGU; partial over the segment, fp32 dGU
// times the loaded bf16 GU), and the output stored already row-scaled,
// dGUr = r (.)row dGU, the form both consumers take (the weight gradient
// h2g^T dGUr and the RMSNorm-backward GEMM on dGUr Wgu^T = r (.)row G).
template <int kRing = 4096>
struct EpiSwiGLUBwdRowdot {
  struct Params {
    const __nv_bfloat16* gu;  // [M, 2F]
    const float* r;           // [M]
    float* pdot;              // [M, ceil(F/128)]
  };
  struct State {
    float2 dot;  // even and odd features' shares of the row dot
    float rv;
  };
  CODA_NO_PREFETCH
  static constexpr int kInBoxes = 2;  // ring bytes per chunk, filled by one 128-byte box (as EpiSwiGLUBwd)
  static constexpr int kInLoads = 1;
  __device__ static bool has_input(const Params&, const EpiCtx&, int) { return true; }
  __device__ static void in_coord(const Params&, const EpiCtx& cx, int c, int, int& map, int& x, int& y) {
    map = 0;
    x = 2 * (cx.n0 + 32 * c);
    y = cx.wrow0;
  }
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 2;
  static constexpr int kStageBufs = 1;
  static constexpr int kInRingBytes = kRing;  // 4096: one chunk of inputs in flight; 8192: two
  __device__ static int slots(const Params&) { return 1; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    st.dot = splat2(0.f);
    st.rv = (cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) ? ep.r[cx.row] : 0.f;
  }
  __device__ static void chunk(State& st, const Params&, const EpiCtx& cx, int, float (&acc)[32], const Pre&,
                               uint32_t in, uint32_t box0, uint32_t) {
    const float2 rv = splat2(st.rv);
    uint4 u[8];
    box128_row(in, cx.lane, u);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        w[4 * q] = u[4 * half + q].x;
        w[4 * q + 1] = u[4 * half + q].y;
        w[4 * q + 2] = u[4 * half + q].z;
        w[4 * q + 3] = u[4 * half + q].w;
      }
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        // r (dG, dU) from r dA; the row dot accumulates on the scaled values
        // and end() divides r out once
        float2 G, U, rdG, rdU;
        gu_unpack2(w[j], w[j + 1], G, U);
        swiglu_bwd2(mul2(make_float2(acc[16 * half + j], acc[16 * half + j + 1]), rv), G, U, rdG, rdU);
        st.dot = fma2(rdG, G, st.dot);
        st.dot = fma2(rdU, U, st.dot);
        w[j] = pack_bf16(rdG.x, rdU.x);
        w[j + 1] = pack_bf16(rdG.y, rdU.y);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        stage128_put(box0, cx.lane, 4 * half + q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
  }
  __device__ static void store_coord(const Params&, const EpiCtx& cx, int c, int, int& map, int& x, int& y) {
    map = 0;
    x = 2 * (cx.n0 + 32 * c);
    y = cx.wrow0;
  }
  __device__ static void end(State& st, const Params& ep, const EpiCtx& cx) {
    // r > 0 for every row inside M (r = 1 / sqrt(mean + eps))
    const long i = static_cast<long>(cx.row) * cx.n_blocks + cx.n_blk;
    if (cx.row < cx.M && CODA_IN(cx, i, static_cast<long>(cx.M) * cx.n_blocks))
      ep.pdot[i] = (st.dot.x + st.dot.y) / st.rv;
  }
};

// -------------------- RMSNorm backward with the residual-stream gradient
// Block chain: acc = Gr = dYr W^T = r (.)row G (the mainloop consumes the
// row-scaled gradient). dh = gamma (.) Gr - r^2 s h + dres, where dres is the
// gradient reaching h through the residual connection (a second input tile);
// column partial of Gr h (= r G h) over the warp's 32 rows.
template <int kRing = 4096>
struct EpiRmsNormBwdRes {
  struct Params {
    const __nv_bfloat16* h;
    const __nv_bfloat16* gamma;
    const float* r;
    const float* s;
    float* pdg;  // [ceil(M/32), d]
  };
  struct State {
    float r2s;
  };
  struct Pre {
    uint4 g[4];
  };
  __device__ static void prefetch(const Params& ep, const EpiCtx& cx, int c, Pre& pr) {
    load_raw32(ep.gamma, 0, 1, cx.N, 0, cx.n0 + 32 * c, pr.g);
  }
  // box 0: h (map 0), box 1: dres (map 1), both the chunk's 32 x 32 tile
  static constexpr int kInBoxes = 2;
  __device__ static bool has_input(const Params&, const EpiCtx&, int) { return true; }
  __device__ static void in_coord(const Params&, const EpiCtx& cx, int c, int b, int& map, int& x, int& y) {
    map = b;
    x = cx.n0 + 32 * c;
    y = cx.wrow0;
  }
  static constexpr int kChunksPerStore = 1;
  static constexpr int kMaxSlots = 1;
  static constexpr int kInRingBytes = kRing;  // 4096: one chunk of inputs in flight; 8192: two
  __device__ static int slots(const Params&) { return 1; }
  __device__ static void begin(State& st, const Params& ep, const EpiCtx& cx) {
    if (cx.row < cx.M && CODA_IN(cx, cx.row, cx.M)) {
      const float rv = ep.r[cx.row];
      st.r2s = rv * rv * ep.s[cx.row];
    } else {
      st.r2s = 0.f;
    }
  }
  __device__ static void chunk(State& st, const Params& ep, const EpiCtx& cx, int c, float (&acc)[32], const Pre& pr,
                               uint32_t in, uint32_t box0, uint32_t) {
    const int col0 = cx.n0 + 32 * c;
    float part[32];
    uint4 u[4], v[4];
    box_row(in, cx.lane, u);
    box_row(in + kInBoxBytes, cx.lane, v);
    uint32_t hw[16], dw[16], gw[16], w[16];
    words16(u, hw);
    words16(v, dw);
    words16(pr.g, gw);
    const float2 nr2s = splat2(-st.r2s);
    // columns 2j, 2j+1 as two-lane vectors: partial Gr h; dh = gamma Gr - r^2 s h + dres
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 h = make_float2(bf16_lo(hw[j]), bf16_hi(hw[j]));
      const float2 g = make_float2(bf16_lo(gw[j]), bf16_hi(gw[j]));
      const float2 dres = make_float2(bf16_lo(dw[j]), bf16_hi(dw[j]));
      const float2 Gr = make_float2(acc[2 * j], acc[2 * j + 1]);
      const float2 pt = mul2(Gr, h);
      part[2 * j] = pt.x;
      part[2 * j + 1] = pt.y;
      const float2 o = add2(fma2(g, Gr, mul2(nr2s, h)), dres);
      w[j] = pack_bf16(o.x, o.y);
    }
    stage_words16(box0, cx.lane, w);
    const float tot = warp_colsum32(part, cx.lane);
    const long ig = static_cast<long>(cx.wrow0 >> 5) * cx.N + col0 + cx.lane;
    if (cx.wrow0 < cx.M && col0 + cx.lane < cx.N && CODA_IN(cx, ig, static_cast<long>((cx.M + 31) >> 5) * cx.N))
      ep.pdg[ig] = tot;
  }
  CODA_STORE_SAME_COLS(0)
  __device__ static void end(State&, const Params&, const EpiCtx&) {}
};

}  // namespace coda
