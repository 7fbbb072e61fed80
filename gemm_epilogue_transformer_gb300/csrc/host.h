// Host-side internals shared by the translation units of libcoda:
// error reporting, per-device cache, tensor-map encoding, argument checks and
// the launch template for the fused GEMM kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/coda.h"

namespace coda {

// ---------------------------------------------------------------- errors
int fail(int code, const char* fmt, ...);
int fail_cuda(cudaError_t e, const char* what);

struct DeviceInfo {
  int ok;
  int sm_count;
  long long l2_bytes;  // L2 cache size
  int* status;  // device address of the status word
};
// Info for the current device (validated as sm_103); nullptr after fail().
const DeviceInfo* current_device();
unsigned long long wait_timeout_ns();
// 0 = choose per launch, 1 = single-SM tiles, 2 = SM-pair tiles (coda_set_cta_group).
int cta_group_setting();
// Consume the one-shot test fault set by coda_test_inject_missing_load().
int take_injected_fault();
// 0 = no stream-K split, 1 = where it is expected to pay (default), 2 = for
// every shape it applies to (coda_set_stream_k).
int stream_k_setting();

// Stream-K workspace of one stream: fp32 partial accumulators of split tiles
// and their arrival words, and this launch's epoch tag for those words.
struct SkWorkspace {
  void* part;
  unsigned* ctr;
  unsigned epoch;
};
// Bytes of partials a launch may use: one 256 KiB slot pair per SM
// ((clusters - 1) boundaries x 2 pieces x 128 x 256 fp32 per CTA of a cluster).
inline size_t sk_part_bytes(int sm_count) { return static_cast<size_t>(sm_count) * (size_t(256) << 10); }
// Arrival words: (clusters - 1) boundaries x 4 epilogue warps per CTA of a cluster.
inline int sk_ctr_words(int sm_count) { return sm_count * 4; }
// The calling stream's workspace on the current device, created by its first
// stream-K launch (cudaMalloc, arrival words zeroed on the stream); false when
// the stream is being captured, the thread is inside a NoAllocScope, or the
// workspace cannot be had, and the launch then runs without the stream-K split.
bool sk_workspace(const DeviceInfo* di, int dev, cudaStream_t stream, SkWorkspace* out);
// While one exists on a thread, launches from that thread allocate nothing
// (no stream-K workspace is created or used).
struct NoAllocScope {
  NoAllocScope();
  ~NoAllocScope();
};

// The C ABI's opaque stream handle as a CUDA stream.
inline cudaStream_t as_stream(coda_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// ---------------------------------------------------------------- checks
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

#define CODA_REQUIRE(cond, code, ...)        \
  do {                                       \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

#define CODA_REQ_PTR16(p) CODA_REQUIRE((p) != nullptr && aligned16(p), CODA_ERR_INVALID, "%s: " #p " must be a non-null 16-byte aligned device pointer", fn)
#define CODA_REQ_PTR4(p) CODA_REQUIRE((p) != nullptr && aligned4(p), CODA_ERR_INVALID, "%s: " #p " must be a non-null 4-byte aligned device pointer", fn)
#define CODA_REQ_OPT16(p) CODA_REQUIRE((p) == nullptr || aligned16(p), CODA_ERR_INVALID, "%s: " #p " must be 16-byte aligned", fn)
#define CODA_REQ_OPT4(p) CODA_REQUIRE((p) == nullptr || aligned4(p), CODA_ERR_INVALID, "%s: " #p " must be 4-byte aligned", fn)

// ---------------------------------------------------------------- tensor maps
// 2-D bf16 map over a row-major [outer, inner] array with row stride
// `row_bytes`, box {box_inner, box_outer}, the given swizzle.
int make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
// A row-major [k, mn] bf16 array read MN-major as boxes of `chunks` 64 x 64
// atoms (3-D map {64, k, mn/64}); mn a multiple of 64.
int make_map_bf16_mn3d(CUtensorMap* m, const void* base, uint64_t mn, uint64_t k, uint64_t row_bytes,
                       uint32_t chunks);
// The same for a byte array (FP8 operands).
int make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

}  // namespace coda
