// C ABI of the RocketKV library: argument validation, workspace carving, kernel launches.
// Declarations and the contract of every entry point are in include/rkv.h.
#include <cuda_runtime.h>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/rkv.h"
#include "../../include/rkv_testing.h"
#include "rkv_internal.h"

using namespace rkv;

namespace rkv {

cudaError_t ensure_dyn_smem(const void* func, size_t bytes) {
  struct Entry {
    const void* func;
    int dev;
    size_t bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& x : done)
    if (x.func == func && x.dev == dev && x.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  for (Entry& x : done)
    if (x.func == func && x.dev == dev) {
      x.bytes = bytes;
      return cudaSuccess;
    }
  done.push_back({func, dev, bytes});
  return cudaSuccess;
}

int device_sm_count() {
  static std::mutex mu;
  static int cached[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    cudaGetLastError();
    return kFallbackSMs;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
      cudaGetLastError();
      return kFallbackSMs;
    }
    cached[dev] = sms;
  }
  return cached[dev];
}

}  // namespace rkv

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline uint32_t* status_ptr(void* ws) { return reinterpret_cast<uint32_t*>(ws); }
inline rkv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA; }
inline bool gqa_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxAvgKernel = (1 << 20) - 1;  // keeps a fixed-point window sum below 2^60

}  // namespace

extern "C" {

const char* rkv_status_string(rkv_status s) {
  switch (s) {
    case RKV_OK: return "ok";
    case RKV_ERR_INVALID_ARG: return "invalid argument";
    case RKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case RKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case RKV_ERR_CUDA: return "CUDA launch or runtime error";
    case RKV_ERR_DEVICE_STATUS: return "kernel reported inconsistent device data";
    case RKV_ERR_TOO_LARGE: return "problem too large for the fixed scratch of the allocation-free call";
  }
  return "unknown status";
}

rkv_status rkv_check_status(void* ws, void* stream, uint32_t* bits) {
  if (!ws) return RKV_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  uint32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return RKV_ERR_CUDA;
  if (bits) *bits = h;
  if (h == 0) return RKV_OK;
  e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? RKV_ERR_DEVICE_STATUS : RKV_ERR_CUDA;
}

rkv_status rkv_plan(int ctx, int budget, int head_dim, int page, int channels, int* keep,
                    int* page_out, int* channels_out, int* kernel_size) {
  if (ctx <= 0 || budget <= 0 || head_dim <= 0 || page < 0 || channels < 0)
    return RKV_ERR_INVALID_ARG;
  if (page == 0) page = 4;
  if (channels == 0) channels = head_dim / 4;
  if (channels < 1 || channels > head_dim || budget % 2 != 0 || budget / 2 < page)
    return RKV_ERR_INVALID_ARG;
  const long long want = (long long)budget * page * head_dim / channels;
  if (keep) *keep = (int)(want < ctx ? want : ctx);
  if (page_out) *page_out = page;
  if (channels_out) *channels_out = channels;
  if (kernel_size) *kernel_size = ctx <= 8192 ? 7 : (ctx <= 32768 ? 15 : 31);
  return RKV_OK;
}

// The overall ratio R = ctx / budget split evenly: sqrt(R) to each stage, and stage 2's share
// evenly between page size and channel reduction, the page rounded to the nearest power of two
// (in log2) within [1, min(64, budget / 2)] and the channels to the nearest integer in [1, d].
rkv_status rkv_plan_even_split(int ctx, int budget, int head_dim, int* keep, int* page_out,
                               int* channels_out, int* kernel_size) {
  if (ctx <= 0 || budget <= 1 || budget % 2 != 0 || head_dim <= 0) return RKV_ERR_INVALID_ARG;
  const double stage2 = std::sqrt((double)ctx / (double)budget);
  const double lp = std::floor(std::log2(stage2) / 2.0 + 0.5);
  int page = 1;
  for (int i = 0; i < (int)lp && page < 64 && page * 2 <= budget / 2; ++i) page *= 2;
  long long ch = std::llround((double)head_dim * page / stage2);
  if (ch < 1) ch = 1;
  if (ch > head_dim) ch = head_dim;
  const long long want = (long long)budget * page * head_dim / ch;
  if (keep) *keep = (int)(want < ctx ? want : ctx);
  if (page_out) *page_out = page;
  if (channels_out) *channels_out = (int)ch;
  if (kernel_size) *kernel_size = ctx <= 8192 ? 7 : (ctx <= 32768 ? 15 : 31);
  return RKV_OK;
}

// ------------------------------------------------------------------------------- stage 1
size_t rkv_snapkv_workspace_bytes(int n, int n_kv, int gqa, int max_len, int window) {
  if (n <= 0 || n_kv <= 0 || gqa <= 0 || max_len <= window || window <= 0) return 0;
  return kStatusBytes + snapkv_scratch_bytes(n, n_kv, gqa, max_len, window);
}

// per_head: every query head is its own unit (gqa units per K/V head, window rows of one head,
// own kept set); else the units are the K/V heads and their groups' rows are summed.
static rkv_status snapkv_impl(const void* k, const void* v, const int32_t* seq_lens,
                              const void* q_win, int n, int n_kv, int gqa, int head_dim,
                              int max_len, int window, int kernel_size, int keep, float scale,
                              void* k_out, void* v_out, int cap, int32_t* kept_idx,
                              int32_t* out_len, float* scores_out, void* ws, size_t ws_bytes,
                              void* stream, bool per_head, const PagedMap& out_pm,
                              int page = 0, int page_cap = 0, void* kmin = nullptr,
                              void* kmax = nullptr, bool pool_avg = false,
                              int kept_stride = 0, bool scores_only = false,
                              uint64_t wait_limit_ns = 0, int test_skip_tile = 0) {
  if (head_dim != kHeadDim) return RKV_ERR_UNSUPPORTED;
  if (scores_only) {  // scores only: no V, no selection or gather outputs
    if (!scores_out || v || k_out || v_out || kept_idx || out_len || kmin || kmax)
      return RKV_ERR_INVALID_ARG;
    kept_stride = 0;
    keep = window + 1;
    cap = keep;
  }
  // kept_stride > 0: index-only selection (no v, no compact cache, no gather)
  const bool index_only = kept_stride > 0;
  if (index_only) {
    if (k_out || v_out || kmin || kmax || kept_stride < keep) return RKV_ERR_INVALID_ARG;
    cap = keep;
  }
  if (!k || (!v && !index_only && !scores_only) || !seq_lens || !q_win ||
      (!index_only && !scores_only && (!k_out || !v_out)) ||
      (!scores_only && (!kept_idx || !out_len)))
    return RKV_ERR_INVALID_ARG;
  if (!aligned16(k) || (v && !aligned16(v)) || !aligned16(q_win) ||
      (k_out && !aligned16(k_out)) || (v_out && !aligned16(v_out)) ||
      (scores_out && !aligned16(scores_out)))
    return RKV_ERR_INVALID_ARG;
  if (n <= 0 || n_kv <= 0 || gqa <= 0 || window <= 0 || max_len <= window || keep <= window ||
      keep > cap || cap <= 0 || !(scale > 0.f) || !std::isfinite(scale))
    return RKV_ERR_INVALID_ARG;
  if (kernel_size < 0 || (kernel_size > 0 && kernel_size % 2 == 0)) return RKV_ERR_INVALID_ARG;
  if (pool_avg && kernel_size > kMaxAvgKernel) return RKV_ERR_INVALID_ARG;
  if (kmin || kmax) {  // page summaries built by the gather
    if (!kmin || !kmax || !aligned16(kmin) || !aligned16(kmax) || !pow2(page) || page > 64 ||
        page_cap <= 0 || page_cap % 8 != 0 || (keep + page - 1) / page > page_cap)
      return RKV_ERR_INVALID_ARG;
  }
  const int kv_div = per_head ? gqa : 1;
  if (per_head) {  // the kernels see n_kv * gqa units of one query head each
    n_kv *= gqa;
    gqa = 1;
  }
  if (gqa * window > 256) return RKV_ERR_UNSUPPORTED;
  const size_t need = rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window);
  if (!ws || !aligned16(ws) || ws_bytes < need) return RKV_ERR_WORKSPACE;

  SnapArgs a{};
  a.k = static_cast<const bf16*>(k);
  a.v = static_cast<const bf16*>(v);
  a.seq_lens = seq_lens;
  a.q_win = static_cast<const bf16*>(q_win);
  a.n = n;
  a.n_kv = n_kv;
  a.gqa = gqa;
  a.kv_div = kv_div;
  a.out_pm = out_pm;
  a.kmin = static_cast<bf16*>(kmin);
  a.kmax = static_cast<bf16*>(kmax);
  a.page = page;
  a.page_cap = page_cap;
  a.max_len = max_len;
  a.window = window;
  a.kernel_size = kernel_size;
  a.pool_avg = pool_avg ? 1 : 0;
  a.kept_stride = index_only ? kept_stride : keep;
  a.keep = keep;
  a.cap = cap;
  a.scale_log2 = scale * kLog2e;
  a.k_out = static_cast<bf16*>(k_out);
  a.v_out = static_cast<bf16*>(v_out);
  a.kept_idx = kept_idx;
  a.out_len = out_len;
  a.scores_only = scores_only ? 1 : 0;
  a.wait_limit_ns = wait_limit_ns;
  a.test_skip_tile = test_skip_tile;
  snapkv_plan(n, n_kv, gqa, max_len, window, &a.nsplit, &a.tokens_per_split, &a.rows_pad);
  // workspace carve: [status][pooled][scores (if not given)][split partials]
  unsigned char* p = static_cast<unsigned char*>(ws) + kStatusBytes;
  const size_t plen = align_up((size_t)n * n_kv * (max_len - window) * 4, 256);
  a.pooled = reinterpret_cast<float*>(p);
  p += plen;
  if (scores_out) {
    a.scores = scores_out;
  } else {
    a.scores = reinterpret_cast<float*>(p);
  }
  p += plen;
  a.part_ml = reinterpret_cast<float*>(p);
  p += align_up((size_t)n * n_kv * a.nsplit * a.rows_pad * 2 * 4, 256);
  a.nlse = reinterpret_cast<float*>(p);
  a.status = status_ptr(ws);
  return from_cuda(launch_snapkv(a, as_stream(stream)));
}

rkv_status rkv_snapkv_compress(const void* k, const void* v, const int32_t* seq_lens,
                               const void* q_win, int n, int n_kv, int gqa, int head_dim,
                               int max_len, int window, int kernel_size, int keep, float scale,
                               void* k_out, void* v_out, int cap, int32_t* kept_idx,
                               int32_t* out_len, float* scores_out, void* ws, size_t ws_bytes,
                               void* stream) {
  RKV_TRACE();
  return snapkv_impl(k, v, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window,
                     kernel_size, keep, scale, k_out, v_out, cap, kept_idx, out_len, scores_out,
                     ws, ws_bytes, stream, false, PagedMap{});
}

rkv_status rkv_snapkv_compress_avg_pool(const void* k, const void* v, const int32_t* seq_lens,
                                        const void* q_win, int n, int n_kv, int gqa,
                                        int head_dim, int max_len, int window, int kernel_size,
                                        int keep, float scale, void* k_out, void* v_out, int cap,
                                        int32_t* kept_idx, int32_t* out_len, float* scores_out,
                                        void* ws, size_t ws_bytes, void* stream) {
  RKV_TRACE();
  return snapkv_impl(k, v, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window,
                     kernel_size, keep, scale, k_out, v_out, cap, kept_idx, out_len, scores_out,
                     ws, ws_bytes, stream, false, PagedMap{}, 0, 0, nullptr, nullptr, true);
}

rkv_status rkv_snapkv_select(const void* k, const int32_t* seq_lens, const void* q_win, int n,
                             int n_kv, int gqa, int head_dim, int max_len, int window,
                             int kernel_size, int keep, float scale, int32_t* kept_idx,
                             int kept_stride, int32_t* out_len, float* scores_out, void* ws,
                             size_t ws_bytes, void* stream) {
  RKV_TRACE();
  if (kept_stride <= 0) return RKV_ERR_INVALID_ARG;
  return snapkv_impl(k, nullptr, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window,
                     kernel_size, keep, scale, nullptr, nullptr, keep, kept_idx, out_len,
                     scores_out, ws, ws_bytes, stream, false, PagedMap{}, 0, 0, nullptr, nullptr,
                     false, kept_stride);
}

rkv_status rkv_snapkv_scores(const void* k, const int32_t* seq_lens, const void* q_win, int n,
                             int n_kv, int gqa, int head_dim, int max_len, int window,
                             float scale, float* scores_out, void* ws, size_t ws_bytes,
                             void* stream) {
  RKV_TRACE();
  return snapkv_impl(k, nullptr, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window, 0, 0,
                     scale, nullptr, nullptr, 0, nullptr, nullptr, scores_out, ws, ws_bytes,
                     stream, false, PagedMap{}, 0, 0, nullptr, nullptr, false, 0, true);
}

rkv_status rkv_testing_scores_wait_timeout(const void* k, const int32_t* seq_lens,
                                           const void* q_win, int n, int n_kv, int gqa,
                                           int head_dim, int max_len, int window, float scale,
                                           float* scores_out, uint64_t wait_limit_ns, void* ws,
                                           size_t ws_bytes, void* stream) {
  RKV_TRACE();
  if (wait_limit_ns < 1000ull || wait_limit_ns > 1000000000ull) return RKV_ERR_INVALID_ARG;
  return snapkv_impl(k, nullptr, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window, 0, 0,
                     scale, nullptr, nullptr, 0, nullptr, nullptr, scores_out, ws, ws_bytes,
                     stream, false, PagedMap{}, 0, 0, nullptr, nullptr, false, 0, true,
                     wait_limit_ns, 1);
}

rkv_status rkv_testing_decode_layout(int layout) {
  return rkv::set_decode_layout(layout) == 0 ? RKV_OK : RKV_ERR_INVALID_ARG;
}

rkv_status rkv_snapkv_compress_summarized(const void* k, const void* v,
                                          const int32_t* seq_lens, const void* q_win, int n,
                                          int n_kv, int gqa, int head_dim, int max_len,
                                          int window, int kernel_size, int keep, float scale,
                                          void* k_out, void* v_out, int cap, int32_t* kept_idx,
                                          int32_t* out_len, float* scores_out, int page,
                                          int page_cap, void* kmin, void* kmax, void* ws,
                                          size_t ws_bytes, void* stream) {
  RKV_TRACE();
  if (!kmin || !kmax) return RKV_ERR_INVALID_ARG;
  return snapkv_impl(k, v, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window,
                     kernel_size, keep, scale, k_out, v_out, cap, kept_idx, out_len, scores_out,
                     ws, ws_bytes, stream, false, PagedMap{}, page, page_cap, kmin, kmax);
}

size_t rkv_snapkv_per_head_workspace_bytes(int n, int n_kv, int gqa, int max_len, int window) {
  if (gqa <= 0) return 0;
  return rkv_snapkv_workspace_bytes(n, n_kv * gqa, 1, max_len, window);
}

rkv_status rkv_snapkv_compress_per_head(const void* k, const void* v, const int32_t* seq_lens,
                                        const void* q_win, int n, int n_kv, int gqa,
                                        int head_dim, int max_len, int window, int kernel_size,
                                        int keep, float scale, void* k_out, void* v_out, int cap,
                                        int32_t* kept_idx, int32_t* out_len, float* scores_out,
                                        void* ws, size_t ws_bytes, void* stream) {
  RKV_TRACE();
  if (gqa <= 0) return RKV_ERR_INVALID_ARG;
  return snapkv_impl(k, v, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window,
                     kernel_size, keep, scale, k_out, v_out, cap, kept_idx, out_len, scores_out,
                     ws, ws_bytes, stream, true, PagedMap{});
}

// ------------------------------------------------------------------------------- summaries
size_t rkv_summaries_workspace_bytes(void) { return kStatusBytes; }

// Summaries of the cache (kept == nullptr) or of the kept sequence of the full cache.
static rkv_status summaries_impl(const void* k_cache, const int32_t* len, const int32_t* kept,
                                 const PagedMap& pm, int n, int n_kv, int head_dim, int cap,
                                 int vcap, int page, int page_cap, int first_token, void* kmin,
                                 void* kmax, void* ws, size_t ws_bytes, void* stream) {
  if (head_dim != kHeadDim) return RKV_ERR_UNSUPPORTED;
  if (!k_cache || !len || !kmin || !kmax) return RKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(kmin) || !aligned16(kmax)) return RKV_ERR_INVALID_ARG;
  if (n <= 0 || n_kv <= 0 || cap <= 0 || vcap <= 0 || !pow2(page) || page > 64 ||
      page_cap <= 0 || page_cap % 8 != 0 || first_token < 0)
    return RKV_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < kStatusBytes) return RKV_ERR_WORKSPACE;
  SummaryArgs a{};
  a.k_cache = static_cast<const bf16*>(k_cache);
  a.len = len;
  a.kept = kept;
  a.pm = pm;
  a.kmin = static_cast<bf16*>(kmin);
  a.kmax = static_cast<bf16*>(kmax);
  a.n = n;
  a.n_kv = n_kv;
  a.cap = cap;
  a.vcap = vcap;
  a.page = page;
  a.page_cap = page_cap;
  a.first_token = first_token;
  a.status = status_ptr(ws);
  return from_cuda(launch_summaries(a, as_stream(stream)));
}

rkv_status rkv_build_page_summaries(const void* k_cache, const int32_t* len, int n, int n_kv,
                                    int head_dim, int cap, int page, int page_cap,
                                    int first_token, void* kmin, void* kmax, void* ws,
                                    size_t ws_bytes, void* stream) {
  RKV_TRACE();
  return summaries_impl(k_cache, len, nullptr, PagedMap{}, n, n_kv, head_dim, cap, cap, page,
                        page_cap, first_token, kmin, kmax, ws, ws_bytes, stream);
}

rkv_status rkv_build_page_summaries_mt(const void* k_full, const int32_t* kept_idx,
                                       const int32_t* kept_len, int n, int n_kv, int head_dim,
                                       int full_cap, int kcap, int page, int page_cap,
                                       int first_token, void* kmin, void* kmax, void* ws,
                                       size_t ws_bytes, void* stream) {
  RKV_TRACE();
  if (!kept_idx) return RKV_ERR_INVALID_ARG;
  return summaries_impl(k_full, kept_len, kept_idx, PagedMap{}, n, n_kv, head_dim, full_cap, kcap,
                        page, page_cap, first_token, kmin, kmax, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------------------- hybrid
size_t rkv_hybrid_decode_workspace_bytes(int n, int n_kv, int gqa, int page_cap, int budget,
                                         int page) {
  (void)n_kv;
  (void)gqa;
  (void)page_cap;
  (void)budget;
  (void)page;
  return kStatusBytes + hybrid_counter_bytes(n);
}

// One decode step over the cache (kept == nullptr) or over the kept sequence of the full cache.
static rkv_status hybrid_impl(const void* q, const void* new_k, const void* new_v,
                              void* k_cache, void* v_cache, int32_t* len, int32_t* kept,
                              int32_t* full_len, const PagedMap& pm, void* kmin, void* kmax, int n,
                              int n_kv,
                              int gqa, int head_dim, int cap, int vcap, int page_cap, int budget,
                              int page, int channels, float scale, void* out,
                              int32_t* sel_channels, int32_t* sel_pages, float* approx_scores,
                              void* ws, size_t ws_bytes, void* stream) {
  if (head_dim != kHeadDim) return RKV_ERR_UNSUPPORTED;
  if (!gqa_ok(gqa)) return RKV_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !len || !kmin || !kmax || !out) return RKV_ERR_INVALID_ARG;
  if ((new_k == nullptr) != (new_v == nullptr)) return RKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(kmin) ||
      !aligned16(kmax) || !aligned16(out))
    return RKV_ERR_INVALID_ARG;
  if (n <= 0 || n_kv <= 0 || cap <= 0 || vcap <= 0 || page_cap <= 0 || page_cap % 8 != 0 ||
      !pow2(page) || page > 64 || budget <= 0 || budget % 2 != 0 || budget / 2 < page ||
      channels < 1 || channels > kHeadDim || !(scale > 0.f) || !std::isfinite(scale))
    return RKV_ERR_INVALID_ARG;
  const size_t smem = hybrid_smem_bytes(gqa, page_cap, budget, page);
  if (smem > kDecodeSmemMax) return RKV_ERR_UNSUPPORTED;
  if (!ws || !aligned16(ws) ||
      ws_bytes < rkv_hybrid_decode_workspace_bytes(n, n_kv, gqa, page_cap, budget, page))
    return RKV_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  HybridArgsAll a{};
  a.pm = pm;
  a.q = static_cast<const bf16*>(q);
  a.k_cache = static_cast<const bf16*>(k_cache);
  a.v_cache = static_cast<const bf16*>(v_cache);
  a.len = len;
  a.kmin = static_cast<const bf16*>(kmin);
  a.kmax = static_cast<const bf16*>(kmax);
  a.kept = kept;
  a.full_len = full_len;
  a.n = n;
  a.n_kv = n_kv;
  a.gqa = gqa;
  a.cap = cap;
  a.vcap = vcap;
  a.page_cap = page_cap;
  a.budget = budget;
  a.page = page;
  a.channels = channels;
  a.scale_log2 = scale * kLog2e;
  a.out = static_cast<bf16*>(out);
  a.sel_channels = sel_channels;
  a.sel_pages = sel_pages;
  a.approx = approx_scores;
  a.status = status_ptr(ws);
  a.ap.new_k = static_cast<const bf16*>(new_k);
  a.ap.new_v = static_cast<const bf16*>(new_v);
  a.ap.acount = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(ws) + kStatusBytes);
  return from_cuda(launch_hybrid(a, s));
}

rkv_status rkv_hybrid_decode(const void* q, const void* new_k, const void* new_v,
                             void* k_cache, void* v_cache, int32_t* len, void* kmin, void* kmax,
                             int n, int n_kv, int gqa, int head_dim, int cap, int page_cap,
                             int budget, int page, int channels, float scale, void* out,
                             int32_t* sel_channels, int32_t* sel_pages, float* approx_scores,
                             void* ws, size_t ws_bytes, void* stream) {
  RKV_TRACE();
  return hybrid_impl(q, new_k, new_v, k_cache, v_cache, len, nullptr, nullptr, PagedMap{}, kmin,
                     kmax, n, n_kv, gqa, head_dim, cap, cap, page_cap, budget, page, channels,
                     scale, out, sel_channels, sel_pages, approx_scores, ws, ws_bytes, stream);
}

rkv_status rkv_hybrid_decode_mt(const void* q, const void* new_k, const void* new_v,
                                void* k_full, void* v_full, int32_t* full_len, int32_t* kept_idx,
                                int32_t* kept_len, void* kmin, void* kmax, int n, int n_kv,
                                int gqa, int head_dim, int full_cap, int kcap, int page_cap,
                                int budget, int page, int channels, float scale, void* out,
                                int32_t* sel_channels, int32_t* sel_pages, float* approx_scores,
                                void* ws, size_t ws_bytes, void* stream) {
  RKV_TRACE();
  if (!kept_idx || !full_len) return RKV_ERR_INVALID_ARG;
  return hybrid_impl(q, new_k, new_v, k_full, v_full, kept_len, kept_idx, full_len, PagedMap{},
                     kmin, kmax, n, n_kv, gqa, head_dim, full_cap, kcap, page_cap, budget, page,
                     channels, scale, out, sel_channels, sel_pages, approx_scores, ws, ws_bytes,
                     stream);
}

// ------------------------------------------------------------------------------- paged
static bool paged_ok(const void* table, int num_blocks, int block, int max_blocks) {
  return table && num_blocks > 0 && max_blocks > 0 && pow2(block) && block <= 65536 &&
         (long long)max_blocks * block <= (1ll << 30);
}

rkv_status rkv_snapkv_compress_paged(const void* k, const void* v, const int32_t* seq_lens,
                                     const void* q_win, int n, int n_kv, int gqa, int head_dim,
                                     int max_len, int window, int kernel_size, int keep,
                                     float scale, void* k_pool, void* v_pool, int num_blocks,
                                     int block, const int32_t* block_table, int max_blocks,
                                     int32_t* kept_idx, int32_t* out_len, float* scores_out,
                                     void* ws, size_t ws_bytes, void* stream) {
  RKV_TRACE();
  if (!paged_ok(block_table, num_blocks, block, max_blocks)) return RKV_ERR_INVALID_ARG;
  const PagedMap pm{block_table, max_blocks, block, num_blocks};
  return snapkv_impl(k, v, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window,
                     kernel_size, keep, scale, k_pool, v_pool, max_blocks * block, kept_idx,
                     out_len, scores_out, ws, ws_bytes, stream, false, pm);
}

rkv_status rkv_build_page_summaries_paged(const void* k_pool, const int32_t* block_table,
                                          const int32_t* len, int n, int n_kv, int head_dim,
                                          int num_blocks, int block, int max_blocks, int page,
                                          int page_cap, int first_token, void* kmin, void* kmax,
                                          void* ws, size_t ws_bytes, void* stream) {
  RKV_TRACE();
  if (!paged_ok(block_table, num_blocks, block, max_blocks)) return RKV_ERR_INVALID_ARG;
  const PagedMap pm{block_table, max_blocks, block, num_blocks};
  const int capacity = max_blocks * block;
  return summaries_impl(k_pool, len, nullptr, pm, n, n_kv, head_dim, capacity, capacity, page,
                        page_cap, first_token, kmin, kmax, ws, ws_bytes, stream);
}

rkv_status rkv_hybrid_decode_paged(const void* q, const void* new_k, const void* new_v,
                                   void* k_pool, void* v_pool, const int32_t* block_table,
                                   int32_t* len, void* kmin, void* kmax, int n, int n_kv, int gqa,
                                   int head_dim, int num_blocks, int block, int max_blocks,
                                   int page_cap, int budget, int page, int channels, float scale,
                                   void* out, int32_t* sel_channels, int32_t* sel_pages,
                                   float* approx_scores, void* ws, size_t ws_bytes,
                                   void* stream) {
  RKV_TRACE();
  if (!paged_ok(block_table, num_blocks, block, max_blocks)) return RKV_ERR_INVALID_ARG;
  const PagedMap pm{block_table, max_blocks, block, num_blocks};
  const int capacity = max_blocks * block;
  return hybrid_impl(q, new_k, new_v, k_pool, v_pool, len, nullptr, nullptr, pm, kmin, kmax, n,
                     n_kv, gqa, head_dim, capacity, capacity, page_cap, budget, page, channels,
                     scale, out, sel_channels, sel_pages, approx_scores, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------------------- dense
size_t rkv_dense_decode_workspace_bytes(int n, int n_kv, int gqa, int max_len) {
  if (n <= 0 || n_kv <= 0 || gqa <= 0 || max_len <= 0) return 0;
  if ((long long)n * n_kv * gqa > INT_MAX) return 0;
  return kStatusBytes + dense_partials_bytes(n, n_kv, gqa, max_len);
}

rkv_status rkv_dense_decode(const void* q, const void* k, const void* v, const int32_t* len,
                            int n, int n_kv, int gqa, int head_dim, int max_len, float scale,
                            void* out, void* ws, size_t ws_bytes, void* stream) {
  RKV_TRACE();
  int bad = dense_check_sizes(n, n_kv, gqa, head_dim, max_len, scale);
  if (!bad) bad = dense_check_pointers(q, k, v, len, out);
  if (bad) return static_cast<rkv_status>(bad);
  const size_t need = rkv_dense_decode_workspace_bytes(n, n_kv, gqa, max_len);
  if (!ws || !aligned16(ws) || ws_bytes < need) return RKV_ERR_WORKSPACE;
  const DenseArgs a = dense_args(q, k, v, len, n, n_kv, gqa, max_len, scale, out, ws);
  return from_cuda(launch_dense(a, as_stream(stream)));
}

}  // extern "C"

namespace rkv {

int dense_check_sizes(int n, int n_kv, int gqa, int head_dim, int max_len, float scale) {
  if (head_dim != kHeadDim) return RKV_ERR_UNSUPPORTED;
  if (!gqa_ok(gqa)) return RKV_ERR_UNSUPPORTED;
  if (n <= 0 || n_kv <= 0 || max_len <= 0 || !(scale > 0.f) || !std::isfinite(scale))
    return RKV_ERR_INVALID_ARG;
  // one CTA per (unit, KV head) and split, one combine CTA per query head: grid limits
  if ((long long)n * n_kv * gqa > INT_MAX) return RKV_ERR_INVALID_ARG;
  return RKV_OK;
}

int dense_check_pointers(const void* q, const void* k, const void* v, const int32_t* len,
                         const void* out) {
  if (!q || !k || !v || !len || !out) return RKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return RKV_ERR_INVALID_ARG;
  return RKV_OK;
}

DenseArgs dense_args(const void* q, const void* k, const void* v, const int32_t* len, int n,
                     int n_kv, int gqa, int max_len, float scale, void* out, void* scratch) {
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
  a.scale_log2 = scale * kLog2e;
  const size_t rows = (size_t)n * n_kv * gqa * a.nsplit;
  unsigned char* p = static_cast<unsigned char*>(scratch) + kStatusBytes;
  a.part_m = reinterpret_cast<float*>(p);
  p += align_up(rows * 4, 256);
  a.part_l = reinterpret_cast<float*>(p);
  p += align_up(rows * 4, 256);
  a.part_o = reinterpret_cast<float*>(p);
  a.out = static_cast<bf16*>(out);
  a.status = static_cast<uint32_t*>(scratch);
  return a;
}

}  // namespace rkv
