// Allocation-free variant of the dense decode: the split-K partials live in a fixed file-scope
// device array instead of a caller-provided workspace.
//
// Who needs it: code that may only hand over the tensors it already owns and must not allocate
// device memory while it runs -- for example a plugin boundary that passes just input and output
// pointers, a host that has handed all device memory to its own pool, or a region that is being
// recorded into a CUDA graph. Such a caller cannot call cudaMalloc to build a workspace.
//
// Cost: every GPU that loads the library keeps kNoAllocScratchBytes of device memory for this
// array until the process exits.
#include <cuda_runtime.h>
#include <cmath>
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
  if (head_dim != kHeadDim) return RKV_ERR_UNSUPPORTED;
  if (!(gqa == 1 || gqa == 2 || gqa == 4 || gqa == 8)) return RKV_ERR_UNSUPPORTED;
  if (!q || !k || !v || !len || !out) return RKV_ERR_INVALID_ARG;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15u;
  if (mis) return RKV_ERR_INVALID_ARG;
  if (n <= 0 || n_kv <= 0 || max_len <= 0 || !(scale > 0.f) || !std::isfinite(scale))
    return RKV_ERR_INVALID_ARG;
  const size_t need = kStatusBytes + dense_partials_bytes(n, n_kv, gqa, max_len);
  if (need > kNoAllocScratchBytes) return RKV_ERR_TOO_LARGE;

  void* base = nullptr;
  if (noalloc_scratch(&base) != cudaSuccess) return RKV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero; the partials are fully rewritten by every call
  if (cudaMemsetAsync(base, 0, kStatusBytes, s) != cudaSuccess) return RKV_ERR_CUDA;

  DenseArgs a{};
  a.q = static_cast<const bf16*>(q);
  a.k = static_cast<const bf16*>(k);
  a.v = static_cast<const bf16*>(v);
  a.len = len;
  a.n = n;
  a.n_kv = n_kv;
  a.gqa = gqa;
  a.max_len = max_len;
  dense_plan(n, n_kv, max_len, &a.nsplit, &a.tokens_per_split);
  a.scale_log2 = scale * 1.4426950408889634f;
  const size_t rows = (size_t)n * n_kv * gqa * a.nsplit;
  unsigned char* p = static_cast<unsigned char*>(base) + kStatusBytes;
  a.part_m = reinterpret_cast<float*>(p);
  p += align_up(rows * 4, 256);
  a.part_l = reinterpret_cast<float*>(p);
  p += align_up(rows * 4, 256);
  a.part_o = reinterpret_cast<float*>(p);
  a.out = static_cast<bf16*>(out);
  a.status = static_cast<uint32_t*>(base);
  return launch_dense(a, s) == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}
