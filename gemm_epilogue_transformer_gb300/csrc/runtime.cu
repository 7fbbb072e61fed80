// libcoda runtime: error text, per-device initialisation and the device
// status word, wait-timeout setting, tensor-map encoding via the driver entry
// point (no link-time dependency on libcuda).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "host.h"

namespace coda {

static thread_local char g_err[1024] = "";
// settings written by coda_set_* and read at every launch, possibly from other host threads
static std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
static std::atomic<int> g_cta_group{0};
static std::atomic<int> g_inject{0};
static std::atomic<int> g_stream_k{1};

// The device status word (CODA_DEVST_* bits). Kernels receive its device
// address, obtained per device with cudaGetSymbolAddress.
__device__ int g_device_status = 0;

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(CODA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

static std::mutex g_mu;
static DeviceInfo g_dev[64];

static const DeviceInfo* init_device(int dev) {
  if (dev < 0 || dev >= 64) {
    fail(CODA_ERR_INVALID, "device index %d out of range", dev);
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.ok) return &d;
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) {
    fail_cuda(e, "cudaGetDeviceProperties");
    return nullptr;
  }
  if (!(prop.major == 10 && prop.minor == 3)) {
    fail(CODA_ERR_UNSUPPORTED, "device %d is sm_%d%d (%s); libcoda is built for sm_103a (GB300)", dev, prop.major,
         prop.minor, prop.name);
    return nullptr;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_device_status);
  if (e != cudaSuccess) {
    fail_cuda(e, "cudaGetSymbolAddress(status word)");
    return nullptr;
  }
  d.sm_count = prop.multiProcessorCount;
  d.l2_bytes = prop.l2CacheSize;
  d.status = static_cast<int*>(p);
  d.ok = 1;
  return &d;
}

const DeviceInfo* current_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    fail_cuda(e, "cudaGetDevice");
    return nullptr;
  }
  return init_device(dev);
}

unsigned long long wait_timeout_ns() { return g_timeout_ns; }
int cta_group_setting() { return g_cta_group; }
int take_injected_fault() { return g_inject.exchange(0); }
int stream_k_setting() { return g_stream_k; }

// ------------------------------------------------- stream-K workspaces
// One per (device, stream handle), created by the stream's first stream-K
// launch and kept for the life of the process (one CUDA context per device,
// as for every per-device cache here). Launches on one stream run in order,
// so they can share its workspace; different streams never share one.
namespace {
struct SkEntry {
  int dev;
  cudaStream_t stream;
  unsigned long long sid;  // cudaStreamGetId of the stream the handle named when last used
  char* mem;               // partials, then the arrival words
  unsigned epoch;
};
constexpr int kMaxSkStreams = 64;
std::mutex g_sk_mu;
SkEntry g_sk[kMaxSkStreams];
int g_sk_n = 0;
thread_local int tl_no_alloc = 0;

size_t sk_ctr_bytes(int sm_count) { return static_cast<size_t>(sk_ctr_words(sm_count)) * sizeof(unsigned); }
}  // namespace

NoAllocScope::NoAllocScope() { ++tl_no_alloc; }
NoAllocScope::~NoAllocScope() { --tl_no_alloc; }

bool sk_workspace(const DeviceInfo* di, int dev, cudaStream_t stream, SkWorkspace* out) {
  if (tl_no_alloc) return false;
  // a captured launch would bake this launch's epoch into every replay
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (cs != cudaStreamCaptureStatusNone) return false;
  unsigned long long sid = 0;
  if (cudaStreamGetId(stream, &sid) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const size_t part = sk_part_bytes(di->sm_count), ctr = sk_ctr_bytes(di->sm_count);
  std::lock_guard<std::mutex> lk(g_sk_mu);
  SkEntry* e = nullptr;
  for (int i = 0; i < g_sk_n; ++i)
    if (g_sk[i].dev == dev && g_sk[i].stream == stream) e = &g_sk[i];
  if (e && e->sid != sid) {
    // The handle now names a new stream (the old one was destroyed): launches
    // of the old stream may still be running on this workspace.
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    const cudaError_t r = cudaDeviceSynchronize();
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (r != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    e->sid = sid;
  }
  if (!e) {
    if (g_sk_n == kMaxSkStreams) return false;
    void* mem = nullptr;
    // relaxed: the allocation must not disturb another thread's capture
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    cudaError_t r = cudaMalloc(&mem, part + ctr);
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (r != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    r = cudaMemsetAsync(static_cast<char*>(mem) + part, 0, ctr, stream);
    if (r != cudaSuccess) {
      cudaGetLastError();
      cudaFree(mem);
      return false;
    }
    e = &g_sk[g_sk_n++];
    e->dev = dev;
    e->stream = stream;
    e->sid = sid;
    e->mem = static_cast<char*>(mem);
    e->epoch = 0;
  }
  // Epoch tags are 30 bits; before they wrap, the words are zeroed on the
  // stream so no word left from 2^30 launches ago can match a new tag.
  if (++e->epoch >= (1u << 30)) {
    if (cudaMemsetAsync(e->mem + part, 0, ctr, stream) != cudaSuccess) {
      cudaGetLastError();
      --e->epoch;
      return false;
    }
    e->epoch = 1;
  }
  out->part = e->mem;
  out->ctr = reinterpret_cast<unsigned*>(e->mem + part);
  out->epoch = e->epoch;
  return true;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static int make_map(CUtensorMapDataType dt, CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CODA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(CODA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): inner %llu outer %llu stride %llu box %u x %u",
                static_cast<int>(r), (unsigned long long)inner, (unsigned long long)outer,
                (unsigned long long)row_bytes, box_inner, box_outer);
  return CODA_OK;
}

// A row-major [k, mn] bf16 operand used MN-major, viewed as 3-D {64, k, mn/64}
// (element in a 64-wide chunk, row, chunk) with strides {row_bytes, 128 B}, so
// that one box of {64, 64, chunks} lands in shared memory as `chunks`
// consecutive 128B-swizzled 64 x 64 atoms (8 KiB each): the layout of
// `chunks` separate 2-D boxes, in one copy. mn must be a multiple of 64 (a
// partial last chunk would read the next row instead of zeros).
int make_map_bf16_mn3d(CUtensorMap* m, const void* base, uint64_t mn, uint64_t k, uint64_t row_bytes,
                       uint32_t chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CODA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  if (mn % 64 != 0) return fail(CODA_ERR_INVALID, "3-D operand map needs a multiple of 64 columns (got %llu)",
                                (unsigned long long)mn);
  cuuint64_t dims[3] = {64, k, mn / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, 64, chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(CODA_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d): mn %llu k %llu stride %llu chunks %u",
                static_cast<int>(r), (unsigned long long)mn, (unsigned long long)k, (unsigned long long)row_bytes,
                chunks);
  return CODA_OK;
}

int make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  return make_map(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m, base, inner, outer, row_bytes, box_inner, box_outer, sw);
}

int make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  return make_map(CU_TENSOR_MAP_DATA_TYPE_UINT8, m, base, inner, outer, row_bytes, box_inner, box_outer, sw);
}

}  // namespace coda

using namespace coda;

extern "C" {

const char* coda_last_error(void) { return g_err; }

int coda_init(int device) {
  cudaError_t e = cudaSetDevice(device);
  if (e != cudaSuccess) return fail_cuda(e, "cudaSetDevice");
  return init_device(device) ? CODA_OK : CODA_ERR_UNSUPPORTED;
}

int coda_device_status(int clear) {
  const DeviceInfo* d = current_device();
  if (!d) return CODA_ERR_UNSUPPORTED;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e, "read status word");
  if (clear) {
    int z = 0;
    e = cudaMemcpy(d->status, &z, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e, "clear status word");
  }
  return v;
}

int coda_set_wait_timeout_ns(unsigned long long ns) {
  if (ns < 100000ull) return fail(CODA_ERR_INVALID, "coda_set_wait_timeout_ns: %llu ns is below 1e5", ns);
  g_timeout_ns = ns;
  return CODA_OK;
}

int coda_set_cta_group(int g) {
  if (g < 0 || g > 2) return fail(CODA_ERR_INVALID, "coda_set_cta_group: %d is not 0, 1 or 2", g);
  g_cta_group = g;
  return CODA_OK;
}

int coda_set_stream_k(int mode) {
  if (mode < 0 || mode > 2) return fail(CODA_ERR_INVALID, "coda_set_stream_k: %d is not 0, 1 or 2", mode);
  g_stream_k = mode;
  return CODA_OK;
}

int coda_test_inject_missing_load(void) {
  g_inject.store(1);
  return CODA_OK;
}

int coda_num_col_tiles(int N) { return N <= 0 ? 0 : (N + 127) / 128; }
int coda_num_row_tiles(int M) { return M <= 0 ? 0 : (M + 31) / 32; }

}  // extern "C"
