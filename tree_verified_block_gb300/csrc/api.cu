// Host-side plumbing of the C ABI: error text, device status, tensor maps.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "glance_internal.cuh"

namespace glance {

static thread_local char t_last_error[512] = "";

glance_status fail(glance_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

glance_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GLANCE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 1;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

cudaError_t ensure_smem(const void* func, int bytes) {
  struct Entry {
    const void* func;
    int dev;
    int bytes;
  };
  static Entry table[64];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (table[i].func == func && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n < 64) table[n++] = Entry{func, dev, bytes};
  return e;
}

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

glance_status make_map_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides_bytes, const uint32_t* box,
                            CUtensorMapSwizzle swz, const char* what) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(GLANCE_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", what);
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, s, b,
                   e, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GLANCE_ERR_INVALID_ARG, "%s: tensor map encode failed (%d)", what, (int)r);
  return GLANCE_OK;
}

}  // namespace glance

extern "C" {

const char* glance_last_error(void) { return glance::t_last_error; }

const char* glance_status_string(glance_status s) {
  switch (s) {
    case GLANCE_OK: return "GLANCE_OK";
    case GLANCE_ERR_INVALID_ARG: return "GLANCE_ERR_INVALID_ARG";
    case GLANCE_ERR_UNSUPPORTED: return "GLANCE_ERR_UNSUPPORTED";
    case GLANCE_ERR_CAPACITY: return "GLANCE_ERR_CAPACITY";
    case GLANCE_ERR_CUDA: return "GLANCE_ERR_CUDA";
    case GLANCE_ERR_DEVICE: return "GLANCE_ERR_DEVICE";
  }
  return "GLANCE_UNKNOWN_STATUS";
}

static glance_status read_all_status(int32_t* code_out, bool reset) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return glance::cuda_fail(e, "glance_device_status");
  int first = 0;
  cudaError_t (*fns[5])(int*, bool) = {glance::status_build_tree, glance::status_attention,
                                       glance::status_lmhead, glance::status_commit, glance::status_dense};
  for (auto fn : fns) {
    int v = 0;
    e = fn(&v, reset);
    if (e != cudaSuccess) return glance::cuda_fail(e, "glance_device_status");
    if (!first && v) first = v;
  }
  if (code_out) *code_out = first;
  if (first && !reset)
    return glance::fail(GLANCE_ERR_DEVICE, "device status word = %d", first);
  return GLANCE_OK;
}

glance_status glance_device_status(int32_t* code_out) { return read_all_status(code_out, false); }

namespace {

// out[0] = the first non-zero of out[1..n] (0 if none)
__global__ void first_status_kernel(int32_t* out, int n) {
  int first = 0;
  for (int i = 1; i <= n; ++i) {
    const int v = out[i];
    if (!first && v) first = v;
  }
  out[0] = first;
}

constexpr int kStatusUnits = 5;

}  // namespace

glance_status glance_get_status(int32_t* status_out, void* stream) {
  if (!status_out) return glance::fail(GLANCE_ERR_INVALID_ARG, "glance_get_status: null status_out");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t (*fns[kStatusUnits])(int*, cudaStream_t) = {
      glance::status_build_tree_async, glance::status_attention_async, glance::status_lmhead_async,
      glance::status_commit_async, glance::status_dense_async};
  for (int i = 0; i < kStatusUnits; ++i) {
    cudaError_t e = fns[i](status_out + 1 + i, s);
    if (e != cudaSuccess) return glance::cuda_fail(e, "glance_get_status");
  }
  first_status_kernel<<<1, 1, 0, s>>>(status_out, kStatusUnits);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return glance::cuda_fail(e, "glance_get_status");
  return GLANCE_OK;
}

glance_status glance_clear_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t (*fns[kStatusUnits])(void**) = {glance::status_build_tree_addr, glance::status_attention_addr,
                                              glance::status_lmhead_addr, glance::status_commit_addr,
                                              glance::status_dense_addr};
  for (int i = 0; i < kStatusUnits; ++i) {
    void* a = nullptr;
    cudaError_t e = fns[i](&a);
    if (e == cudaSuccess) e = cudaMemsetAsync(a, 0, sizeof(int), s);
    if (e != cudaSuccess) return glance::cuda_fail(e, "glance_clear_status");
  }
  return GLANCE_OK;
}

glance_status glance_reset_device_status(void) {
  int32_t dummy = 0;
  return read_all_status(&dummy, true);
}

int glance_version(void) { return 300; }

}  // extern "C"
