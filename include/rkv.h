/*
 * rkv.h -- C ABI of the RocketKV hot path on GB300 (sm_103a): SnapKV++ prefill eviction and
 * hybrid sparse decode attention, plus a dense decode used as the full-KV timing reference.
 *
 * The method is described in "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage KV
 * Cache Compression" (Behnam et al., arXiv 2502.14051). Sections cited below are those of the
 * authors' OpenReview responses on paperhub.cn (same title), which hold the method's details:
 *   [LAT]   "Lack of Direct Latency Comparison"           -- token budget split half / half
 *   [APPROX]"Explanation of Calculating Approximate Attention Scores" -- pages, Kmin/Kmax,
 *                                                             top-|q| channels, GQA group sums
 *   [PAGE]  "Is Page Always Divided Into 4?"              -- ratio decomposition, page size
 *   [EVICT] "Is Needle Among Evicted Tokens"              -- eviction per head and per layer
 *   [KSIZE] "Potential Sensitivity to Kernel Size in SnapKV++" -- adaptive pooling size
 *   [STEP]  "Are Different KV Tokens Retrieved at Each Decoding Step?" -- selection per step
 *   [SNAP++]"Novelty of SnapKV++"                          -- GQA-aware SnapKV scoring
 *   [MT]    "SCBench Results"                              -- RocketKV-MT: nothing evicted, the
 *                                                             decode selects among kept tokens
 * and [KEYPTS] = "Key points" of the summarizepaper.com summary (full-KV baseline, SnapKV++).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor pointer is DEVICE memory owned by the caller. The library allocates nothing
 *    and keeps no state between calls. bf16 tensors are passed as void* and must be 16-byte
 *    aligned. All integer tensors are int32.
 *  - n counts independent problems (batch x layers flattened; "unit" below = one of the n).
 *    Query heads of unit u: Hq = n_kv * gqa, query head h belongs to KV head h / gqa.
 *  - head_dim must be 128 (RKV_ERR_UNSUPPORTED otherwise).
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *    default stream). Arguments are validated on the host before any launch; an invalid
 *    argument returns RKV_ERR_INVALID_ARG / RKV_ERR_UNSUPPORTED / RKV_ERR_WORKSPACE and launches
 *    nothing. A failed launch returns RKV_ERR_CUDA.
 *  - ws / ws_bytes: scratch owned by the caller, at least the size the matching
 *    *_workspace_bytes() returns. Its first 256 bytes hold a device status word that kernels set
 *    when they detect an inconsistency in device-resident data (e.g. a length beyond capacity,
 *    a bounded wait that ran out). It must be zero before first use (allocate it zeroed).
 *    rkv_check_status() synchronises the stream, reads and clears it. Kernels never trap.
 *  - Two calls that share one workspace must not overlap on the GPU (same stream is fine).
 */
#ifndef RKV_H_
#define RKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RKV_OK = 0,
  RKV_ERR_INVALID_ARG = 1,
  RKV_ERR_UNSUPPORTED = 2,
  RKV_ERR_WORKSPACE = 3,
  RKV_ERR_CUDA = 4,
  RKV_ERR_DEVICE_STATUS = 5,
  RKV_ERR_TOO_LARGE = 6
} rkv_status;

/* Device status bits (reported by rkv_check_status through *bits). */
#define RKV_DEV_LEN_OVER_CAP   0x1u  /* a length exceeds cap / page_cap (work for it skipped) */
#define RKV_DEV_BAD_WINDOW     0x2u  /* a sequence shorter than the window (unit skipped)     */
#define RKV_DEV_WAIT_TIMEOUT   0x4u  /* a bounded mbarrier wait ran out (unit abandoned)      */
#define RKV_DEV_SELECT_FAILED  0x8u  /* a top-k selection produced the wrong count            */
#define RKV_DEV_BAD_INDEX      0x10u /* a kept index outside the valid rows (row 0 read)      */

/* Human-readable name of a status code (static string). */
const char* rkv_status_string(rkv_status s);

/* Synchronise `stream`, read the device status word in `ws`, clear it, and return RKV_OK if it
 * was zero or RKV_ERR_DEVICE_STATUS otherwise (bits in *bits when bits != NULL). */
rkv_status rkv_check_status(void* ws, void* stream, uint32_t* bits);

/* Pure host planner ([PAGE], [LAT], [KSIZE]). The overall ratio ctx / budget is split between
 * the two stages, and stage 2's share between the sequence dimension (page) and the head
 * dimension (head_dim / channels). page = 0 picks 4 and channels = 0 picks head_dim / 4; the
 * stage-1 keep is then min(ctx, budget * page * head_dim / channels), which makes the
 * approximation read exactly as many bytes as budget / 2 tokens of K and V. kernel_size: 7 for
 * ctx <= 8192, 15 for ctx <= 32768, else 31 (larger pooling for longer prompts). Any output
 * pointer may be NULL. Errors: RKV_ERR_INVALID_ARG for non-positive sizes, channels > head_dim,
 * budget odd or budget / 2 < page. */
rkv_status rkv_plan(int ctx, int budget, int head_dim, int page, int channels,
                    int* keep, int* page_out, int* channels_out, int* kernel_size);

/* The even split of [PAGE] for any ratio: with R = ctx / budget, each stage gets sqrt(R), and
 * stage 2's share is split evenly between the page size and the channel reduction, so that
 * page ~ R^(1/4) and head_dim / channels ~ R^(1/4) (128K tokens at budget 512: R = 256, page 4,
 * channels head_dim / 4, keep 8192). Where R^(1/4) is not a power of two the page is the power
 * of two nearest to it on a log2 scale (halves round up), within [1, min(64, budget / 2)];
 * channels = round(head_dim * page / sqrt(R)) within [1, head_dim]; keep and kernel_size as for
 * rkv_plan. Errors: RKV_ERR_INVALID_ARG for ctx <= 0, budget < 2 or odd, head_dim <= 0. */
rkv_status rkv_plan_even_split(int ctx, int budget, int head_dim, int* keep, int* page,
                               int* channels, int* kernel_size);

/* ------------------------------------------------------------------------------------------ */
/* Stage 1: SnapKV++ eviction ([SNAP++], [EVICT], [KSIZE], [KEYPTS])                            */
/* ------------------------------------------------------------------------------------------ */
size_t rkv_snapkv_workspace_bytes(int n, int n_kv, int gqa, int max_len, int window);

/* For each unit u and KV head g: score every prefix position i < L_u - window with the window
 * queries -- softmax(q . k / sqrt-scale) over all keys visible to each window query (the prefix
 * plus the causal part of the window), summed over the window and over the gqa query heads of
 * the group -- max-pool the scores with an odd kernel (stride 1, same length, clipped ends), keep
 * the keep - window highest (ties -> lower position) and append the window, then gather those
 * rows of K and V into the compact cache.
 *   k, v      [n][n_kv][max_len][128] bf16, rows >= L_u ignored
 *   seq_lens  [n] int32 on device, window <= L_u <= max_len
 *   q_win     [n][n_kv*gqa][window][128] bf16 -- the last `window` queries of every head
 *   window    1 <= window, gqa * window <= 256
 *   kernel_size odd >= 1, or 0 to pick it per sequence from L_u (7 / 15 / 31 as rkv_plan)
 *   keep      tokens kept per (unit, KV head) including the window; window < keep <= cap.
 *             A sequence with L_u <= keep keeps all L_u tokens.
 *   scale     logit scale (1/sqrt(128) for the usual attention)
 *   k_out, v_out [n][n_kv][cap][128] bf16: rows 0 .. out_len[u]-1 written (kept positions in
 *             ascending order, the window last)
 *   kept_idx  [n][n_kv][keep] int32: original positions of the kept rows; -1 past out_len[u]
 *   out_len   [n] int32: min(L_u, keep)
 *   scores_out NULL or [n][n_kv][max_len - window] fp32: the un-pooled prefix scores
 */
rkv_status rkv_snapkv_compress(const void* k, const void* v, const int32_t* seq_lens,
                               const void* q_win, int n, int n_kv, int gqa, int head_dim,
                               int max_len, int window, int kernel_size, int keep, float scale,
                               void* k_out, void* v_out, int cap, int32_t* kept_idx,
                               int32_t* out_len, float* scores_out, void* ws, size_t ws_bytes,
                               void* stream);

/* [SNAP++] The scoring half of rkv_snapkv_compress alone: for each unit u and KV head g, the
 * score of every prefix position i < L_u - window (softmax probabilities of the window queries
 * over the keys each may see, summed over the window and over the gqa query heads of the group),
 * with no pooling, selection or gather. For a caller that pools or selects by its own rule, and
 * for timing the two tensor-core score passes on their own.
 *   k, seq_lens, q_win, window, scale as rkv_snapkv_compress (no V needed)
 *   scores_out [n][n_kv][max_len - window] fp32 (required): entries i >= L_u - window of a
 *             unit are left untouched
 * Workspace rkv_snapkv_workspace_bytes; errors as rkv_snapkv_compress. */
rkv_status rkv_snapkv_scores(const void* k, const int32_t* seq_lens, const void* q_win, int n,
                             int n_kv, int gqa, int head_dim, int max_len, int window,
                             float scale, float* scores_out, void* ws, size_t ws_bytes,
                             void* stream);

/* [MT] The selection half of rkv_snapkv_compress (scores, pooling, top-k) without the gather:
 * RocketKV-MT evicts nothing, so each turn filters the full, unfiltered history again
 * ("SCBench Results": the next turn's prefill takes all earlier tokens as its prefix and SnapKV++
 * filters once more) and the decode reads the kept rows through the index list.
 *   k         [n][n_kv][max_len][128] bf16: the full cache, rows >= L_u ignored (no V needed)
 *   seq_lens  [n] int32: history length L_u this turn (earlier turns, generated tokens, the new
 *             input), window <= L_u <= max_len
 *   q_win     [n][n_kv*gqa][window][128] bf16: the last `window` queries of this turn's input
 *   kept_idx  [n][n_kv][kept_stride] int32, kept_stride >= keep: entries 0 .. keep-1 of each
 *             (unit, KV head) written as in rkv_snapkv_compress (-1 past out_len[u]); entries
 *             keep .. kept_stride-1 untouched, so the list can be handed to
 *             rkv_build_page_summaries_mt / rkv_hybrid_decode_mt with kcap = kept_stride
 *   out_len   [n] int32: min(L_u, keep), the kept_len of the MT calls
 * Other arguments, workspace (rkv_snapkv_workspace_bytes) and errors as rkv_snapkv_compress. */
rkv_status rkv_snapkv_select(const void* k, const int32_t* seq_lens, const void* q_win, int n,
                             int n_kv, int gqa, int head_dim, int max_len, int window,
                             int kernel_size, int keep, float scale, int32_t* kept_idx,
                             int kept_stride, int32_t* out_len, float* scores_out, void* ws,
                             size_t ws_bytes, void* stream);

/* rkv_snapkv_compress with average pooling in place of max pooling (a SnapKV pooling variant;
 * the pages describe max pooling only): each prefix score is replaced by the mean of the scores
 * over the in-range positions of its clipped window [max(0, i - r), min(n - 1, i + r)],
 * r = kernel_size / 2, before the top-k. The window sums are exact (fixed point), so the result
 * depends only on the fp32 scores. kernel_size odd in [1, 1048575], or 0 as above. Other
 * arguments, outputs, workspace and errors as rkv_snapkv_compress. */
rkv_status rkv_snapkv_compress_avg_pool(const void* k, const void* v, const int32_t* seq_lens,
                                        const void* q_win, int n, int n_kv, int gqa,
                                        int head_dim, int max_len, int window, int kernel_size,
                                        int keep, float scale, void* k_out, void* v_out, int cap,
                                        int32_t* kept_idx, int32_t* out_len, float* scores_out,
                                        void* ws, size_t ws_bytes, void* stream);

/* rkv_snapkv_compress followed by rkv_build_page_summaries(k_out, out_len, page, page_cap,
 * first_token = 0, kmin, kmax) in one pass: the gather builds the page summaries of the rows it
 * writes ([APPROX]), so the compact cache is not read back. Same outputs, bit for bit. page a
 * power of two <= 64; page_cap a multiple of 8 with page_cap * page >= keep; kmin, kmax
 * [n][n_kv][128][page_cap] bf16 (pages past ceil(out_len[u] / page) untouched). Workspace:
 * rkv_snapkv_workspace_bytes. */
rkv_status rkv_snapkv_compress_summarized(const void* k, const void* v,
                                          const int32_t* seq_lens, const void* q_win, int n,
                                          int n_kv, int gqa, int head_dim, int max_len,
                                          int window, int kernel_size, int keep, float scale,
                                          void* k_out, void* v_out, int cap, int32_t* kept_idx,
                                          int32_t* out_len, float* scores_out, int page,
                                          int page_cap, void* kmin, void* kmax, void* ws,
                                          size_t ws_bytes, void* stream);

/* The ablation without the GQA enhancement ([SNAP++], [KEYPTS]: plain SnapKV): every query
 * head is scored and filtered on its own -- its W window rows only, no sum over the group -- and
 * keeps its own copy of the selected rows of its K/V head h / gqa. Same arguments as
 * rkv_snapkv_compress, with the per-unit outputs per query head:
 *   k_out, v_out [n][n_kv*gqa][cap][128] bf16; kept_idx [n][n_kv*gqa][keep] int32;
 *   scores_out NULL or [n][n_kv*gqa][max_len - window] fp32; out_len [n] int32.
 * window <= 256. Workspace: rkv_snapkv_per_head_workspace_bytes. The result is a cache that the
 * decode calls use with n_kv*gqa K/V heads and gqa = 1. */
size_t rkv_snapkv_per_head_workspace_bytes(int n, int n_kv, int gqa, int max_len, int window);
rkv_status rkv_snapkv_compress_per_head(const void* k, const void* v, const int32_t* seq_lens,
                                        const void* q_win, int n, int n_kv, int gqa,
                                        int head_dim, int max_len, int window, int kernel_size,
                                        int keep, float scale, void* k_out, void* v_out, int cap,
                                        int32_t* kept_idx, int32_t* out_len, float* scores_out,
                                        void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Stage 2: page summaries ([APPROX])                                                          */
/* ------------------------------------------------------------------------------------------ */
size_t rkv_summaries_workspace_bytes(void);

/* Element-wise min and max of K over pages of `page` consecutive cache rows, stored
 * channel-major so that one channel of all pages is one contiguous row:
 *   k_cache [n][n_kv][cap][128] bf16, len [n] int32 (device)
 *   kmin, kmax [n][n_kv][128][page_cap] bf16; page p of unit u covers rows p*page ..
 *   min(len_u, (p+1)*page) - 1 (a partial last page uses its valid rows only).
 *   Pages from first_token / page up to the last page are (re)computed; first_token = 0
 *   rebuilds everything. page is a power of two <= 64; page_cap is a multiple of 8 and
 *   page_cap * page >= the largest len (checked on device: RKV_DEV_LEN_OVER_CAP).
 */
rkv_status rkv_build_page_summaries(const void* k_cache, const int32_t* len, int n, int n_kv,
                                    int head_dim, int cap, int page, int page_cap,
                                    int first_token, void* kmin, void* kmax, void* ws,
                                    size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Stage 2: hybrid sparse decode ([APPROX], [LAT], [STEP], [PAGE])                              */
/* ------------------------------------------------------------------------------------------ */
/* The decode's workspace: the status word and one append counter per unit (both zero at first
 * use; the counters are back at zero after every call). */
size_t rkv_hybrid_decode_workspace_bytes(int n, int n_kv, int gqa, int page_cap, int budget,
                                         int page);

/* One decode step. If new_k / new_v are given, token len_u is first appended to every KV head
 * of unit u (cache rows and the page summary it lands in) and len[u] is incremented, inside the
 * same launch; the new token can be selected in this step. Then, per (unit, KV head g):
 *   len_u <= budget: exact attention over every cached token;
 *   otherwise: the `channels` channels with the largest sum over the group of |q_h| (ties ->
 *   lower channel) are kept; with q_g = sum_h q_h, each page scores
 *   sum_{kept i} q_g[i] * (q_g[i] >= 0 ? Kmax[i][page] : Kmin[i][page]) (unscaled); the
 *   (budget/2)/page best pages (ties -> lower page) are selected and all gqa query heads attend
 *   exactly over their valid tokens.
 *   q        [n][n_kv*gqa][128] bf16
 *   new_k, new_v NULL (no append) or [n][n_kv][128] bf16
 *   k_cache, v_cache [n][n_kv][cap][128] bf16; len [n] int32 (device)
 *   kmin, kmax [n][n_kv][128][page_cap] bf16, as built by rkv_build_page_summaries
 *   budget    even, budget/2 >= page; page a power of two <= 64; 1 <= channels <= 128
 *   gqa       1, 2, 4 or 8
 *   out       [n][n_kv*gqa][128] bf16
 *   sel_channels NULL or [n][n_kv][channels] int32 (ascending; -1 on the dense path)
 *   sel_pages NULL or [n][n_kv][(budget/2)/page] int32 (ascending; -1 where unused)
 *   approx_scores NULL or [n][n_kv][page_cap] fp32 (pages >= ceil(len_u/page) untouched)
 * A decode CTA keeps one fp32 score per page of page_cap in shared memory: page_cap may be up to
 * 31,168 (fewer when budget/page is large: 27,136 at budget/page = 4096); beyond that the call
 * returns RKV_ERR_UNSUPPORTED. The same limit holds for the RocketKV-MT and paged variants.
 */
rkv_status rkv_hybrid_decode(const void* q, const void* new_k, const void* new_v,
                             void* k_cache, void* v_cache, int32_t* len, void* kmin, void* kmax,
                             int n, int n_kv, int gqa, int head_dim, int cap, int page_cap,
                             int budget, int page, int channels, float scale, void* out,
                             int32_t* sel_channels, int32_t* sel_pages, float* approx_scores,
                             void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------ */
/* RocketKV-MT: the full cache stays, the decode is restricted to the kept tokens ([MT])        */
/* ------------------------------------------------------------------------------------------ */
/* The multi-turn variant evicts nothing: every prompt token stays in the cache (the next turn
 * re-filters the whole history), and the decode selects only among the tokens SnapKV++ kept.
 * Here the kept tokens are named by an index list instead of being copied. For unit u and KV head
 * g the kept sequence is kept_idx[u][g][j], j = 0 .. kept_len[u]-1: rows of the full cache, in
 * the order the decode treats as token order (rkv_snapkv_compress writes such a list). Both calls
 * compute exactly what rkv_build_page_summaries / rkv_hybrid_decode compute on the compact cache
 * whose row j is k_full[u][g][kept_idx[u][g][j]] (same values, same order, same results); page
 * numbers (sel_pages, approx_scores, kmin / kmax columns) count pages of the kept sequence.
 *
 * Page summaries of the kept sequence:
 *   k_full [n][n_kv][full_cap][128] bf16; kept_idx [n][n_kv][kcap] int32; kept_len [n] int32
 *   kmin, kmax [n][n_kv][128][page_cap] bf16; page, page_cap, first_token as for
 *   rkv_build_page_summaries, with kept_len[u] <= kcap and <= page_cap * page (else
 *   RKV_DEV_LEN_OVER_CAP, unit skipped). A kept index outside [0, full_cap) sets
 *   RKV_DEV_BAD_INDEX and row 0 is read in its place. Workspace: rkv_summaries_workspace_bytes.
 */
rkv_status rkv_build_page_summaries_mt(const void* k_full, const int32_t* kept_idx,
                                       const int32_t* kept_len, int n, int n_kv, int head_dim,
                                       int full_cap, int kcap, int page, int page_cap,
                                       int first_token, void* kmin, void* kmax, void* ws,
                                       size_t ws_bytes, void* stream);

/* One decode step over the kept sequence. If new_k / new_v are given, each unit's new token is
 * first written to row full_len[u] of every KV head of the full cache, appended to the kept list
 * (kept_idx[u][g][kept_len[u]] = full_len[u]) and folded into the page summary it lands in; then
 * full_len[u] and kept_len[u] are incremented (RKV_DEV_LEN_OVER_CAP if full_len[u] = full_cap or
 * kept_len[u] = kcap: nothing appended). The rest is rkv_hybrid_decode on the kept sequence:
 * the dense path when kept_len[u] <= budget, else channel pick, page scores, page top-k and exact
 * attention over the selected pages' kept tokens. A kept index outside [0, full_len[u]) sets
 * RKV_DEV_BAD_INDEX and row 0 is read in its place.
 *   q, out [n][n_kv*gqa][128] bf16; new_k, new_v NULL or [n][n_kv][128] bf16
 *   k_full, v_full [n][n_kv][full_cap][128] bf16; full_len [n] int32
 *   kept_idx [n][n_kv][kcap] int32; kept_len [n] int32
 *   kmin, kmax, budget, page, page_cap, channels, gqa, sel_channels, sel_pages, approx_scores:
 *   as for rkv_hybrid_decode (pages of the kept sequence). Workspace:
 *   rkv_hybrid_decode_workspace_bytes.
 */
rkv_status rkv_hybrid_decode_mt(const void* q, const void* new_k, const void* new_v,
                                void* k_full, void* v_full, int32_t* full_len, int32_t* kept_idx,
                                int32_t* kept_len, void* kmin, void* kmax, int n, int n_kv,
                                int gqa, int head_dim, int full_cap, int kcap, int page_cap,
                                int budget, int page, int channels, float scale, void* out,
                                int32_t* sel_channels, int32_t* sel_pages, float* approx_scores,
                                void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Paged (block-table) compact cache, for serving engines that page their KV cache             */
/* ------------------------------------------------------------------------------------------ */
/* The same three steps -- stage 1 with its gather, page summaries, decode -- on a compact cache
 * held in fixed-size blocks of a shared pool instead of one contiguous region per unit (a
 * storage layout of the serving engine; the computation is that of the non-paged calls, with
 * identical results):
 *   k_pool, v_pool [num_blocks][n_kv][block][128] bf16; block a power of two <= 65536;
 *   block_table [n][max_blocks] int32: token t of unit u (every K/V head g) is row t % block of
 *   block block_table[u][t / block]; capacity = max_blocks * block tokens per unit.
 * Blocks are the caller's: every block a call may write (stage 1: tokens < keep; an append:
 * token len[u]) must be listed in the table beforehand. A table entry outside [0, num_blocks)
 * that a kernel meets sets RKV_DEV_BAD_INDEX and block 0 is used in its place.
 *
 * rkv_snapkv_compress_paged: rkv_snapkv_compress (workspace rkv_snapkv_workspace_bytes) whose
 *   kept rows go to the pools; keep <= capacity.
 * rkv_build_page_summaries_paged: rkv_build_page_summaries over the paged cache (len[u] <=
 *   capacity, else RKV_DEV_LEN_OVER_CAP); workspace rkv_summaries_workspace_bytes.
 * rkv_hybrid_decode_paged: rkv_hybrid_decode over the paged cache, appends included (len[u] <
 *   capacity to append); workspace rkv_hybrid_decode_workspace_bytes. */
rkv_status rkv_snapkv_compress_paged(const void* k, const void* v, const int32_t* seq_lens,
                                     const void* q_win, int n, int n_kv, int gqa, int head_dim,
                                     int max_len, int window, int kernel_size, int keep,
                                     float scale, void* k_pool, void* v_pool, int num_blocks,
                                     int block, const int32_t* block_table, int max_blocks,
                                     int32_t* kept_idx, int32_t* out_len, float* scores_out,
                                     void* ws, size_t ws_bytes, void* stream);
rkv_status rkv_build_page_summaries_paged(const void* k_pool, const int32_t* block_table,
                                          const int32_t* len, int n, int n_kv, int head_dim,
                                          int num_blocks, int block, int max_blocks, int page,
                                          int page_cap, int first_token, void* kmin, void* kmax,
                                          void* ws, size_t ws_bytes, void* stream);
rkv_status rkv_hybrid_decode_paged(const void* q, const void* new_k, const void* new_v,
                                   void* k_pool, void* v_pool, const int32_t* block_table,
                                   int32_t* len, void* kmin, void* kmax, int n, int n_kv, int gqa,
                                   int head_dim, int num_blocks, int block, int max_blocks,
                                   int page_cap, int budget, int page, int channels, float scale,
                                   void* out, int32_t* sel_channels, int32_t* sel_pages,
                                   float* approx_scores, void* ws, size_t ws_bytes,
                                   void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Full-KV decode attention, the baseline the method is compared against ([KEYPTS])            */
/* ------------------------------------------------------------------------------------------ */
size_t rkv_dense_decode_workspace_bytes(int n, int n_kv, int gqa, int max_len);

/* out[u][h] = softmax(scale * q[u][h] . K[u][g]^T) V[u][g] over the len_u cached tokens
 * (g = h / gqa), split over the sequence across thread blocks and merged.
 *   q [n][n_kv*gqa][128] bf16; k, v [n][n_kv][max_len][128] bf16; len [n] int32 (device,
 *   1 <= len_u <= max_len); out [n][n_kv*gqa][128] bf16; gqa 1, 2, 4 or 8.
 */
rkv_status rkv_dense_decode(const void* q, const void* k, const void* v, const int32_t* len,
                            int n, int n_kv, int gqa, int head_dim, int max_len, float scale,
                            void* out, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------ */
/* Allocation-free dense decode (a library convenience; the paper has no counterpart)          */
/* ------------------------------------------------------------------------------------------ */
/* Same computation, arguments and layouts as rkv_dense_decode, but without ws / ws_bytes: the
 * split-K partials go to an 8 MiB array of device memory that the library reserves statically
 * (every GPU that loads the library holds it until the process exits).
 *
 * It exists for callers that cannot call cudaMalloc to build a workspace: code that is only
 * handed its input and output tensors (a plugin boundary, say), or a host whose device memory
 * belongs entirely to its own pool. The caller still passes inputs and outputs; nothing is
 * allocated or freed by this call.
 *
 *  - Limit: 256 B + the partials of rkv_dense_decode_workspace_bytes(n, n_kv, gqa, max_len) must
 *    fit in 8 MiB; otherwise RKV_ERR_TOO_LARGE is returned and nothing is launched (the sizes
 *    are checked before the pointers).
 *  - Set-up: the first call on each device looks up the device address of the array (with that
 *    device current). Make that first call before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents. Each call clears the
 *    status word at its start; calls that overlap on the GPU (different streams, or different
 *    host threads) race on the array and must be serialised by the caller.
 *  - Device-detected inconsistencies (len > max_len is clamped) are not reported by this entry
 *    point. */
rkv_status rkv_dense_decode_noalloc(const void* q, const void* k, const void* v,
                                    const int32_t* len, int n, int n_kv, int gqa, int head_dim,
                                    int max_len, float scale, void* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RKV_H_ */
