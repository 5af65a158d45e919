// Internal launch interface between the C ABI (api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <nvtx3/nvToolsExt.h>

namespace rkv {

constexpr int kHeadDim = 128;
constexpr size_t kStatusBytes = 256;     // device status word + padding at the start of ws
constexpr int kDecodeThreads = 256;      // 8 warps per decode CTA
constexpr int kChunkTokens = 64;         // tokens per shared-memory stage in decode attention


typedef __nv_bfloat16 bf16;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------- decode side
// `len` counts the tokens of the sequence the decode sees; `cap` is the row capacity of k_cache.
// The plain decode's parameters stay within 128 bytes: a larger parameter block was measured to
// add 0.34 us to every launch, whatever the kernel reads.
struct HybridArgs {
  const bf16* q;
  const bf16* k_cache;
  const bf16* v_cache;
  const int32_t* len;
  const bf16* kmin;
  const bf16* kmax;
  int n, n_kv, gqa, cap, page_cap, budget, page, channels;
  float scale_log2;  // scale * log2(e)
  bf16* out;
  int32_t* sel_channels;
  int32_t* sel_pages;
  float* approx;
  uint32_t* status;
};
static_assert(sizeof(HybridArgs) <= 128, "plain-decode parameters must fit in 128 bytes");

// A decode step that first appends this step's token (new K / V rows [n][n_kv][128]) to every
// (unit, KV head): acount [n] counts the unit's KV-head CTAs that have read the unit's length;
// the last one advances it (zero at first use, back to zero after every launch).
struct AppendFields {
  const bf16* new_k;
  const bf16* new_v;
  int32_t* acount;
};

// Plain cache, with the append folded in.
struct HybridArgsApp : HybridArgs {
  AppendFields ap;
};

// RocketKV-MT: the sequence is kept[ukv][0 .. len-1], rows of the full cache (k_cache, cap rows,
// valid below full_len[u]); vcap (the kept list's capacity) bounds len. An appended token goes to
// row full_len[u] of the full cache and to the end of the kept list.
struct HybridArgsMT : HybridArgs {
  const int32_t* kept;
  const int32_t* full_len;
  int vcap;
  AppendFields ap;  // new_k == nullptr: no append
};

// Paged K/V cache: k_cache / v_cache are pools [num_blocks][n_kv][block][128]; token t of unit u
// (every K/V head g) lives in block table[u * max_blocks + t / block], row t % block. A table
// entry outside [0, num_blocks) is reported (RKV_DEV_BAD_INDEX) and block 0 used instead.
struct PagedMap {
  const int32_t* table;
  int max_blocks, block, num_blocks;
};

struct HybridArgsPaged : HybridArgs {
  PagedMap pm;
  AppendFields ap;  // new_k == nullptr: no append
};

// Launch-side view of every decode variant (only the fields of the chosen one are read).
struct HybridArgsAll : HybridArgsMT {
  PagedMap pm;
};

// Summaries of the sequence of `len` tokens: cache rows, or with `kept` set the rows
// kept[ukv][0 .. len-1] of the full cache (len <= vcap).
struct SummaryArgs {
  const bf16* k_cache;
  const int32_t* len;
  const int32_t* kept;
  PagedMap pm;  // table == nullptr: not paged
  bf16* kmin;
  bf16* kmax;
  int n, n_kv, cap, vcap, page, page_cap, first_token;
  uint32_t* status;
};

struct DenseArgs {
  const bf16* q;
  const bf16* k;
  const bf16* v;
  const int32_t* len;
  int n, n_kv, gqa, max_len, nsplit, tokens_per_split;
  float scale_log2;
  float* part_m;  // [n*Hq][nsplit]
  float* part_l;  // [n*Hq][nsplit]
  float* part_o;  // [n*Hq][nsplit][128]
  bf16* out;
  uint32_t* status;
};

// Raise a kernel's dynamic shared-memory limit once per (kernel, device); later calls are
// no-ops, so launches stay legal inside stream capture.
cudaError_t ensure_dyn_smem(const void* func, size_t bytes);

// Streaming multiprocessors of the current device, looked up once per device: persistent grids
// and split plans are sized in multiples of it. When no device answers (a host-only workspace
// query), the GB300's 152.
constexpr int kFallbackSMs = 152;
int device_sm_count();

// An NVTX range named after the entry point around each call that launches kernels, so that a
// profiler's timeline (or ncu --nvtx filters) shows the library's calls; without a tool attached
// NVTX returns at once.
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
};
#define RKV_TRACE() ::rkv::TraceRange rkv_trace_range_(__func__)

// split plan for dense decode, shared by the workspace query and the launch
void dense_plan(int n, int n_kv, int max_len, int* nsplit, int* tokens_per_split);
size_t dense_partials_bytes(int n, int n_kv, int gqa, int max_len);

// Argument checks of the dense decode, shared by the workspace and the allocation-free entry
// points: 0 when the call may proceed, else an rkv_status code. Sizes come first, so that a
// problem too large for a fixed scratch is reported before any pointer is looked at.
int dense_check_sizes(int n, int n_kv, int gqa, int head_dim, int max_len, float scale);
int dense_check_pointers(const void* q, const void* k, const void* v, const int32_t* len,
                         const void* out);
// The launch arguments over a scratch area whose first kStatusBytes hold the status word and the
// rest the split partials (dense_partials_bytes of them).
DenseArgs dense_args(const void* q, const void* k, const void* v, const int32_t* len, int n,
                     int n_kv, int gqa, int max_len, float scale, void* out, void* scratch);

// Dynamic shared memory of a decode CTA (ordinary layout), and its ceiling: the 227 KB a CTA
// may have less the kernel's static shared memory (about 29 KB), with a margin.
size_t hybrid_smem_bytes(int gqa, int page_cap, int budget, int page);
constexpr size_t kDecodeSmemMax = 190 * 1024;
// Shared-memory layout of later hybrid decode launches in this process
// (rkv_testing_decode_layout): 0 automatic, 1 always the ordinary layout, 2 the wide layout
// wherever it fits. Returns -1 for any other value.
int set_decode_layout(int layout);
size_t hybrid_counter_bytes(int n);  // the append counters after the status word
cudaError_t launch_hybrid(const HybridArgsAll& a, cudaStream_t s);
cudaError_t launch_summaries(const SummaryArgs& a, cudaStream_t s);
cudaError_t launch_dense(const DenseArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------- prefill side
struct SnapArgs {
  const bf16* k;
  const bf16* v;
  const int32_t* seq_lens;
  const bf16* q_win;
  int n, n_kv, gqa, max_len, window, kernel_size, keep, cap;
  float scale_log2;
  bf16* k_out;
  bf16* v_out;
  int32_t* kept_idx;
  int32_t* out_len;
  float* scores;       // [n][n_kv][max_len - window] (caller's buffer or workspace)
  float* pooled;       // workspace, same shape
  float* part_ml;      // workspace: [n*n_kv][nsplit][rows_pad][2] (max, sum) per split
  float* nlse;         // workspace: [n*n_kv][rows_pad] merged negated log2-sum-exp per row
  int nsplit, tokens_per_split, rows_pad;
  int kv_div;  // units per K/V head: 1, or gqa when every query head is its own unit
  PagedMap out_pm;  // table != nullptr: k_out / v_out are pools and rows go through the table
  bf16* kmin;       // != nullptr: page summaries of the compact cache, built by the gather
  bf16* kmax;
  int page, page_cap;
  int pool_avg;     // 1: average pooling over the clipped window instead of max pooling
  int kept_stride;  // entries between units' kept lists (>= keep)
  int scores_only;  // 1: stop after the score passes (no pooling, selection or gather)
  uint32_t* status;
  uint64_t wait_limit_ns;  // 0: the default bound of every mbarrier wait (1 s)
  int test_skip_tile;      // testing only (rkv_testing_scores_wait_timeout)
};

void snapkv_plan(int n, int n_kv, int gqa, int max_len, int window, int* nsplit,
                 int* tokens_per_split, int* rows_pad);
size_t snapkv_scratch_bytes(int n, int n_kv, int gqa, int max_len, int window);
cudaError_t launch_snapkv(const SnapArgs& a, cudaStream_t s);

}  // namespace rkv
