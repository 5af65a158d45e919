// Allocation-free variant of the dense decode: the split-K partials live in a fixed file-scope
// device array instead of a caller-provided workspace.
//
// Who needs it: code that may only hand over the tensors it already owns and must not allocate
// device memory while it runs -- for example a plugin boundary that passes just input and output
// pointers, or a host that has handed all device memory to its own pool. Such a caller cannot
// call cudaMalloc to build a workspace.
//
// Cost: every GPU that loads the library keeps kNoAllocScratchBytes of device memory for this
// array until the process exits.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "../../include/rkv.h"
#include "rkv_internal.h"

namespace rkv {

constexpr size_t kNoAllocScratchBytes = 8ull << 20;  // 8 MiB: status word + split partials

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch for the current device. In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device with that device
// current and cached.
static cudaError_t noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[128] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace rkv

using namespace rkv;

extern "C" rkv_status rkv_dense_decode_noalloc(const void* q, const void* k, const void* v,
                                               const int32_t* len, int n, int n_kv, int gqa,
                                               int head_dim, int max_len, float scale,
                                               void* out, void* stream) {
  RKV_TRACE();
  // sizes first: a problem beyond the fixed array is rejected before any pointer is looked at
  int bad = dense_check_sizes(n, n_kv, gqa, head_dim, max_len, scale);
  if (bad) return static_cast<rkv_status>(bad);
  const size_t need = kStatusBytes + dense_partials_bytes(n, n_kv, gqa, max_len);
  if (need > kNoAllocScratchBytes) return RKV_ERR_TOO_LARGE;
  bad = dense_check_pointers(q, k, v, len, out);
  if (bad) return static_cast<rkv_status>(bad);

  void* base = nullptr;
  if (noalloc_scratch(&base) != cudaSuccess) return RKV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero; the partials are fully rewritten by every call
  if (cudaMemsetAsync(base, 0, kStatusBytes, s) != cudaSuccess) return RKV_ERR_CUDA;
  const DenseArgs a = dense_args(q, k, v, len, n, n_kv, gqa, max_len, scale, out, base);
  return launch_dense(a, s) == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}
