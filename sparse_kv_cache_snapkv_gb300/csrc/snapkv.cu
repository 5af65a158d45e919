// Stage-1 kernels of RocketKV (SnapKV++ prefill eviction) on sm_103a.
//
// Method: "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage KV Cache
// Compression" -- summarizepaper.com "Key points" (SnapKV with the grouped-query enhancement),
// OpenReview author responses on paperhub.cn: "Novelty of SnapKV++" (scores summed over the
// query heads of a KV group, so each KV head selects once), "Potential Sensitivity to Kernel
// Size in SnapKV++" (1-D pooling whose size grows with the prompt length), "Is Needle Among
// Evicted Tokens" (eviction independent per head and per layer).
//
// Score computation, per (unit, KV head) with R = gqa * window window rows (padded to RP = 128
// or 256) and the prompt's K:
//   pass 1  D1 = Qwin . K^T on tcgen05 (M = 128 query rows per block, N = 128 tokens), TMEM
//           accumulators read back per row: online max / sum of 2^(scale*log2e*s) over the keys
//           each window row may see (prefix + causal window) -> per-split partial (m, l).
//   pass 2  D2 = K . Qwin^T (M = 128 tokens, N = RP rows): each TMEM lane is one token, so the
//           column sum over window rows and group heads, sum_r 2^(s*c - lse_r), is a per-thread
//           reduction. The partial (m, l) of all splits are merged into lse_r first.
// Both passes stream 128-token K tiles by TMA (SWIZZLE_128B, 2 x 64-column boxes) through a
// 4-stage mbarrier ring; one thread issues MMAs, eight warps run the epilogue; TMEM holds two
// accumulator buffers so the epilogue of tile i overlaps the MMA of tile i+1. Each pass is one
// persistent launch over every (unit, split) work item; pass 2 walks the units in reverse, so
// its first items find the K tiles pass 1 read last still in L2.
//   select  max-pool (odd kernel, clipped ends; or the average over the clipped window) + block
//           radix top-k, ascending kept positions
//   gather  kept K / V rows -> compact cache (16-byte vector copies)
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"
#include "rkv_internal.h"

namespace rkv {

constexpr int kTileTok = 128;
constexpr int kKStages = 4;
constexpr int kScoreThreads = 320;  // warp 0: TMA, warp 1: MMA, warps 2..9: epilogue
constexpr int kEpiThreads = 256;
constexpr int kTileBytes = kTileTok * kHeadDim * 2;  // 32 KB per K tile

// ------------------------------------------------------------------------------------------
// tcgen05 / TMA wrappers
// ------------------------------------------------------------------------------------------
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row core groups 1024 B
// apart (SBO), descriptor version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 accumulate, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__host__ __device__ inline int adaptive_kernel(int L) {
  return L <= 8192 ? 7 : (L <= 32768 ? 15 : 31);
}

// ------------------------------------------------------------------------------------------
// score kernel (both passes), persistent over work items
// ------------------------------------------------------------------------------------------
// A work item is one split (a contiguous range of 128-token tiles) of one (unit, KV head); the
// launch covers every item of every unit and each CTA streams its items (i = blockIdx.x,
// + gridDim.x, ...) through one continuous TMA -> MMA -> epilogue pipeline, so the pipeline fills
// once per launch. The Q tile of the next item is loaded into the other Q buffer while the
// current item's MMAs run (one buffer when G * W > 128, whose Q tile is twice the size).
struct ScoreParams {
  int n_kv, gqa, window, max_len, hq;
  int units, nsplit, tiles_per_split;
  int reverse;     // walk the units last-to-first (pass 2 starts where pass 1 ended: L2-warm)
  int kv_div;      // a unit reads the K rows of K/V head ukv / kv_div
  float scale_log2;
  const int32_t* seq_lens;
  float* part_ml;  // [units][nsplit][RP][2]: per-split (max, sum) of every window row (pass 1)
  const float* nlse;  // [units][RP]: merged, negated log2-sum-exp of every row (pass 2)
  float* scores;   // [units][max_len - window]
  uint32_t* status;
  uint64_t wait_limit_ns;  // bound of every mbarrier wait
  int test_skip_tile;      // testing only: CTA 0 never loads its first K tile of pass 1
};

template <int RB>
struct ScoreSmem {
  static constexpr int RP = RB * 128;
  static constexpr int kQBufs = RB == 1 ? 2 : 1;
  static constexpr size_t q_bytes = (size_t)RP * kHeadDim * 2;
  static constexpr size_t k_off = kQBufs * q_bytes;
  static constexpr size_t bar_off = k_off + (size_t)kKStages * kTileBytes;
  static constexpr size_t misc_off = bar_off + 256;
  static constexpr size_t total = misc_off + RP * 4 + 2 * 128 * 4 + 2 * 128 * 4 + 64 + 1024;
};

struct ItemInfo {
  int ukv, u, g, split, L, tile0, ntiles;
  bool bad;
};

template <int PASS>
__device__ __forceinline__ ItemInfo score_item(const ScoreParams& p, int i) {
  ItemInfo it;
  const int ui = i / p.nsplit;
  it.split = i - ui * p.nsplit;
  it.ukv = p.reverse ? (p.units - 1 - ui) : ui;
  it.u = it.ukv / p.n_kv;
  it.g = it.ukv - it.u * p.n_kv;
  int L = p.seq_lens[it.u];
  it.bad = L <= p.window || L > p.max_len;
  if (it.bad) L = 0;
  it.L = L;
  const int span = (PASS == 1) ? L : (L > p.window ? L - p.window : 0);
  const int tiles_all = (span + kTileTok - 1) / kTileTok;
  it.tile0 = it.split * p.tiles_per_split;
  it.ntiles = max(0, min(p.tiles_per_split, tiles_all - it.tile0));
  return it;
}

template <int PASS, int RB>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap qmap, ScoreParams p) {
  constexpr int RP = RB * 128;
  constexpr uint32_t kCols = (PASS == 1) ? (RB == 1 ? 256u : 512u) : (RP == 128 ? 256u : 512u);
  using SM = ScoreSmem<RB>;
  constexpr int QB = SM::kQBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem;
  uint8_t* ks = smem + SM::k_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::bar_off);
  uint64_t* empty = full + kKStages;
  uint64_t* tfull = empty + kKStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* qfull = tempty + 2;
  uint64_t* qempty = qfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qempty + 2);
  float* nlse_s = reinterpret_cast<float*>(smem + SM::misc_off);  // [RP] negated LSE (pass 2)
  float* xch_m = nlse_s + RP;                                      // [128] (pass 1 merge)
  float* xch_l = xch_m + 128;                                      // [128]
  float* spart = xch_l + 128;                                      // [2][128] (pass 2 merge)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int W = p.window;
  const int R = p.gqa * W;
  const int items = p.units * p.nsplit;
  const uint64_t lim = p.wait_limit_ns;

  if (tid == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiThreads / 32);
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(tmem_slot)), "r"(kCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();     // inputs (and the pass-1 results) come from earlier kernels in the stream
  pdl_trigger();
  bool aborted = false;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0, ic = 0;
      for (int i = blockIdx.x; i < items && !aborted; i += gridDim.x) {
        const ItemInfo itm = score_item<PASS>(p, i);
        if (itm.ntiles == 0) continue;
        const int qb = QB == 2 ? (ic & 1) : 0;
        if (ic >= QB && !mbar_wait(&qempty[qb], (uint32_t)(((ic / QB) - 1) & 1), lim)) {
          aborted = true;
          break;
        }
        uint8_t* qdst = qs + (size_t)qb * SM::q_bytes;
        const int qrow0 = (itm.u * p.hq + itm.g * p.gqa) * W;
        mbar_arrive_expect_tx(&qfull[qb], (uint32_t)(RP * kHeadDim * 2));
        for (int h = 0; h < 2; ++h)
          for (int rb = 0; rb < RB; ++rb)
            tma_load_2d(qdst + (size_t)h * RP * 128 + (size_t)rb * 128 * 128, &qmap, 64 * h,
                        qrow0 + rb * 128, &qfull[qb]);
        const int krow0 = (itm.ukv / p.kv_div) * p.max_len;
        for (int t = 0; t < itm.ntiles; ++t, ++it) {
          const int s = it % kKStages;
          if (it >= kKStages && !mbar_wait(&empty[s], (uint32_t)(((it / kKStages) - 1) & 1), lim)) {
            aborted = true;
            break;
          }
          // (testing: the first tile of CTA 0 is never loaded, so every wait on it runs out)
          if (PASS == 1 && p.test_skip_tile && blockIdx.x == 0 && it == 0) continue;
          uint8_t* dst = ks + (size_t)s * kTileBytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kTileBytes);
          const int y = krow0 + (itm.tile0 + t) * kTileTok;
          tma_load_2d(dst, &kmap, 0, y, &full[s]);
          tma_load_2d(dst + kTileBytes / 2, &kmap, 64, y, &full[s]);
        }
        ++ic;
      }
      if (aborted) {
        set_status(p.status, RKV_DEV_WAIT_TIMEOUT);
        for (int j = max(0, it - kKStages); j < it; ++j)  // let issued loads land
          mbar_wait(&full[j % kKStages], (uint32_t)((j / kKStages) & 1), lim);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, ic = 0;
      for (int i = blockIdx.x; i < items && !aborted; i += gridDim.x) {
        const ItemInfo itm = score_item<PASS>(p, i);
        if (itm.ntiles == 0) continue;
        const int qb = QB == 2 ? (ic & 1) : 0;
        if (!mbar_wait(&qfull[qb], (uint32_t)((ic / QB) & 1), lim)) {
          aborted = true;
          break;
        }
        const uint32_t qbase = smem_addr(qs + (size_t)qb * SM::q_bytes);
        for (int t = 0; t < itm.ntiles; ++t, ++it) {
          const int s = it % kKStages, b = it & 1;
          if (!mbar_wait(&full[s], (uint32_t)((it / kKStages) & 1), lim)) {
            aborted = true;
            break;
          }
          if (it >= 2 && !mbar_wait(&tempty[b], (uint32_t)(((it >> 1) - 1) & 1), lim)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t kbase = smem_addr(ks + (size_t)s * kTileBytes);
          if (PASS == 1) {
            constexpr uint32_t id = idesc_bf16(128, kTileTok);
#pragma unroll
            for (int rb = 0; rb < RB; ++rb) {
              const uint32_t d = tmem + (uint32_t)((b * RB + rb) * kTileTok);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off =
                    (uint32_t)((kk >> 2) * RP * 128 + rb * 128 * 128 + (kk & 3) * 32);
                const uint32_t koff = (uint32_t)((kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32);
                umma_bf16(d, desc_sw128(qbase + off), desc_sw128(kbase + koff), id, kk > 0);
              }
            }
          } else {
            constexpr uint32_t id = idesc_bf16(kTileTok, RP);
            const uint32_t d = tmem + (uint32_t)(b * RP);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t koff = (uint32_t)((kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32);
              const uint32_t qoff = (uint32_t)((kk >> 2) * RP * 128 + (kk & 3) * 32);
              umma_bf16(d, desc_sw128(kbase + koff), desc_sw128(qbase + qoff), id, kk > 0);
            }
          }
          umma_commit(&empty[s]);
          umma_commit(&tfull[b]);
        }
        if (aborted) break;
        umma_commit(&qempty[qb]);  // arrives once this item's MMAs are done with its Q tile
        ++ic;
      }
      if (aborted) set_status(p.status, RKV_DEV_WAIT_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int e = warp - 2;        // 0..7
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int hf = e >> 2;         // 0 / 1
    const int lrow = quarter * 32 + lane;
    const int etid = tid - 64;     // 0..255
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    int it = 0;
    for (int i = blockIdx.x; i < items; i += gridDim.x) {
      const ItemInfo itm = score_item<PASS>(p, i);
      if (PASS == 1 && itm.bad && itm.split == 0 && etid == 0)
        set_status(p.status, RKV_DEV_BAD_WINDOW);
      if (PASS == 1) {
        // row this thread owns and its visibility limit
        const int rb = (RB == 2) ? hf : 0;
        const int rg = rb * 128 + lrow;
        const bool row_ok = rg < R;
        const int lim = itm.L - W + (row_ok ? rg % W : 0);  // last visible key position
        const int c0 = (RB == 2) ? 0 : hf * 64;
        const int ncol = (RB == 2) ? 128 : 64;
        float m = -1e30f, l = 0.f;
        for (int t = 0; t < itm.ntiles; ++t, ++it) {
          const int b = it & 1;
          if (aborted) continue;
          if (!mbar_wait(&tfull[b], (uint32_t)((it >> 1) & 1), lim)) {
            aborted = true;
            continue;
          }
          tc_fence_after();
          const int t0 = (itm.tile0 + t) * kTileTok;
          for (int cc = 0; cc < ncol; cc += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_addr + (uint32_t)((b * RB + rb) * kTileTok + c0 + cc), r);
            const int tb = t0 + c0 + cc;
            // max on the raw logits (the scale is positive); only chunks that reach the causal
            // part of the window need the visibility mask
            float mt = -INFINITY;
            if (tb + 31 <= lim) {
#pragma unroll
              for (int j = 0; j < 32; ++j) mt = fmaxf(mt, __uint_as_float(r[j]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float x = (tb + j <= lim) ? __uint_as_float(r[j]) : -INFINITY;
                r[j] = __float_as_uint(x);
                mt = fmaxf(mt, x);
              }
            }
            const float mn = fmaxf(m, mt * p.scale_log2);
            const float nmn = -mn;
            float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 32; ++j)
              a4[j & 3] += fast_exp2(fmaf(__uint_as_float(r[j]), p.scale_log2, nmn));
            l = l * fast_exp2(m - mn) + ((a4[0] + a4[1]) + (a4[2] + a4[3]));
            m = mn;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[b]);
        }
        if (RB == 1) {
          if (hf == 1) {
            xch_m[lrow] = m;
            xch_l[lrow] = l;
          }
          named_bar_sync(1, kEpiThreads);
          if (hf == 0) {
            const float m2 = xch_m[lrow], l2 = xch_l[lrow];
            const float mn = fmaxf(m, m2);
            l = l * fast_exp2(m - mn) + l2 * fast_exp2(m2 - mn);
            m = mn;
          }
          named_bar_sync(1, kEpiThreads);  // xch is rewritten by the next item
        }
        if (RB == 2 || hf == 0) {
          float* dst =
              p.part_ml + (((size_t)itm.ukv * p.nsplit + itm.split) * RP + rb * 128 + lrow) * 2;
          dst[0] = m;  // an empty split publishes the neutral (-1e30, 0)
          dst[1] = l;
        }
      } else {
        // column sums: thread = token lrow of the tile, columns [c0, c0 + ncol) = window rows
        const int ncol = RP / 2;
        const int c0 = hf * ncol;
        const int prefix = itm.L - W;
        float* out = p.scores + (size_t)itm.ukv * (p.max_len - W);
        named_bar_sync(1, kEpiThreads);  // everyone is done with the previous item's rows
        if (etid < RP) nlse_s[etid] = p.nlse[(size_t)itm.ukv * RP + etid];
        named_bar_sync(1, kEpiThreads);
        // Every epilogue warp passes the named barrier once per tile, also after a failed wait,
        // so that a timeout in one warp can never leave the others waiting at the barrier.
        for (int t = 0; t < itm.ntiles; ++t, ++it) {
          const int b = it & 1;
          if (!aborted && !mbar_wait(&tfull[b], (uint32_t)((it >> 1) & 1), lim)) aborted = true;
          float acc = 0.f;
          if (!aborted) {
            tc_fence_after();
            float a4[4] = {0.f, 0.f, 0.f, 0.f};
            for (int cc = 0; cc < ncol; cc += 32) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_addr + (uint32_t)(b * RP + c0 + cc), r);
              const float4* nl = reinterpret_cast<const float4*>(nlse_s + c0 + cc);
#pragma unroll
              for (int i4 = 0; i4 < 8; ++i4) {
                const float4 v = nl[i4];  // negated log-sum-exp of four window rows
                a4[0] += fast_exp2(fmaf(__uint_as_float(r[4 * i4 + 0]), p.scale_log2, v.x));
                a4[1] += fast_exp2(fmaf(__uint_as_float(r[4 * i4 + 1]), p.scale_log2, v.y));
                a4[2] += fast_exp2(fmaf(__uint_as_float(r[4 * i4 + 2]), p.scale_log2, v.z));
                a4[3] += fast_exp2(fmaf(__uint_as_float(r[4 * i4 + 3]), p.scale_log2, v.w));
              }
            }
            acc = (a4[0] + a4[1]) + (a4[2] + a4[3]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
          }
          if (hf == 1) spart[b * 128 + lrow] = acc;
          named_bar_sync(1, kEpiThreads);
          if (hf == 0 && !aborted) {
            const int tt = (itm.tile0 + t) * kTileTok + lrow;
            if (tt < prefix) out[tt] = acc + spart[b * 128 + lrow];
          }
        }
      }
    }
    if (aborted) set_status(p.status, RKV_DEV_WAIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                 : "memory");
  }
}

// Merge the per-split (max, sum) of every window row into its negated log2-sum-exp (padded
// rows -> -1e30, so that they contribute nothing). Grid: units; block: RP threads.
__global__ void lse_merge_kernel(ScoreParams p, int rp) {
  const int ukv = blockIdx.x, r = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const int u = ukv / p.n_kv;
  const int L = p.seq_lens[u];
  const bool bad = L <= p.window || L > p.max_len;
  float m = -1e30f, l = 0.f;
  if (!bad && r < p.gqa * p.window) {
    const float2* pm = reinterpret_cast<const float2*>(p.part_ml) + (size_t)ukv * p.nsplit * rp + r;
    for (int s0 = 0; s0 < p.nsplit; s0 += 8) {
      float2 x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        x[j] = (s0 + j < p.nsplit) ? pm[(size_t)(s0 + j) * rp] : make_float2(-1e30f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float mn = fmaxf(m, x[j].x);
        l = l * fast_exp2(m - mn) + x[j].y * fast_exp2(x[j].x - mn);
        m = mn;
      }
    }
  }
  const_cast<float*>(p.nlse)[(size_t)ukv * rp + r] = (l > 0.f) ? -(m + log2f(l)) : -1e30f;
}

// ------------------------------------------------------------------------------------------
// average pooling: window sums in 32.32 fixed point. Scores lie in [0, G * W] with G * W <= 256
// and a window holds at most 2^20 - 1 of them, so a sum stays below 2^60: exact, independent of
// the order of its terms, and equal between the sliding sum of the shared-memory select and the
// direct sums of the general one.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ long long to_fixed(float v) { return __float2ll_rn(v * 4294967296.f); }

__device__ __forceinline__ float fixed_mean(long long s, int count) {
  return __fdiv_rn(__ll2float_rn(s) * 2.3283064365386963e-10f, (float)count);
}

// ------------------------------------------------------------------------------------------
// pooling + top-k selection: one CTA of 1024 threads per (unit, KV head)
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) select_kernel(SnapArgs a) {
  __shared__ SelectScratch sc;
  const int ukv = blockIdx.x;
  const int u = ukv / a.n_kv, g = ukv - u * a.n_kv;
  const int W = a.window;
  const int L = a.seq_lens[u];
  int32_t* kept = a.kept_idx + (size_t)ukv * a.kept_stride;
  if (L <= W || L > a.max_len) {
    for (int i = threadIdx.x; i < a.keep; i += blockDim.x) kept[i] = -1;
    if (g == 0 && threadIdx.x == 0) a.out_len[u] = 0;
    return;
  }
  if (L <= a.keep) {
    for (int i = threadIdx.x; i < a.keep; i += blockDim.x) kept[i] = i < L ? i : -1;
    if (g == 0 && threadIdx.x == 0) a.out_len[u] = L;
    return;
  }
  const int n = L - W;
  const int ks = a.kernel_size > 0 ? a.kernel_size : adaptive_kernel(L);
  const int r = ks / 2;
  const float* in = a.scores + (size_t)ukv * (a.max_len - W);
  float* pooled = a.pooled + (size_t)ukv * (a.max_len - W);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int lo = max(0, i - r), hi = min(n - 1, i + r);
    float m;
    if (a.pool_avg) {
      long long sum = 0;
      for (int j = lo; j <= hi; ++j) sum += to_fixed(in[j]);
      m = fixed_mean(sum, hi - lo + 1);
    } else {
      m = in[i];
      for (int j = lo; j <= hi; ++j) m = fmaxf(m, in[j]);
    }
    pooled[i] = m;
  }
  __syncthreads();
  const int want = a.keep - W;
  const int got = block_topk_ascending(pooled, n, want, kept, sc);
  if (got != want && threadIdx.x == 0) set_status(a.status, RKV_DEV_SELECT_FAILED);
  for (int j = threadIdx.x; j < W; j += blockDim.x) kept[want + j] = L - W + j;
  if (g == 0 && threadIdx.x == 0) a.out_len[u] = a.keep;
}

// ------------------------------------------------------------------------------------------
// pooling + top-k selection for long prompts: a cluster of kSelCluster CTAs per (unit, KV head)
// ------------------------------------------------------------------------------------------
// CTA c of the cluster owns the positions [c * span, (c + 1) * span) of the unit's n = L - W
// scores: it loads them with the pooling radius on each side, pools them (max, or the mean of
// the clipped window in 32.32 fixed point, as the other paths) into ordered keys in shared
// memory, and takes part in an MSB-first radix select over the whole unit (11, 11, 10 bits):
// every CTA builds a histogram of its keys, a cluster barrier publishes them, and every CTA
// reads all kSelCluster histograms through distributed shared memory and finds the same digit.
// The kept positions (ties -> lower position) are then written in ascending order from the
// CTAs' (above, equal) counts, exchanged the same way, and a block scan inside each CTA.
constexpr int kSelCluster = 8;
constexpr int kSelCThreads = 1024;
constexpr int kSelCBins = 2048;
constexpr int kSelCMaxSpan = 20480;   // positions per CTA (beyond: the one-CTA select)
constexpr int kSelCMaxRadius = 255;   // pooling radius (beyond: the one-CTA select)

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// 32-bit word at `local` (a shared address of this CTA) in the shared memory of CTA `rank`.
__device__ __forceinline__ uint32_t ld_peer_u32(const void* local, uint32_t rank) {
  uint32_t addr, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

struct SelCSmem {  // after the dynamic key / score arrays
  uint32_t hist[kSelCBins];
  unsigned long long tmp[33];
  uint32_t cnt[2];  // this CTA's (above, equal) counts of the final threshold
  int found[3];     // digit, keys above it, keys in its bin
};

size_t select_cluster_smem_bytes(int span, int r) {
  return align_up((size_t)(span + 2 * r) * 4, 16) + (size_t)span * 4 + sizeof(SelCSmem);
}

__global__ void __launch_bounds__(kSelCThreads, 1) select_cluster_kernel(SnapArgs a, int span) {
  extern __shared__ __align__(16) unsigned char smem_sel[];
  const int ukv = blockIdx.y;
  const uint32_t cr = cluster_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = ukv / a.n_kv, g = ukv - u * a.n_kv;
  const int W = a.window;
  const int L = a.seq_lens[u];
  int32_t* kept = a.kept_idx + (size_t)ukv * a.kept_stride;
  // every CTA of the cluster sees the same L: the early exits are taken by all or by none
  if (L <= W || L > a.max_len) {
    if (cr == 0) {
      for (int i = tid; i < a.keep; i += blockDim.x) kept[i] = -1;
      if (g == 0 && tid == 0) a.out_len[u] = 0;
    }
    return;
  }
  if (L <= a.keep) {
    if (cr == 0) {
      for (int i = tid; i < a.keep; i += blockDim.x) kept[i] = i < L ? i : -1;
      if (g == 0 && tid == 0) a.out_len[u] = L;
    }
    return;
  }
  const int n = L - W;
  const int ks = a.kernel_size > 0 ? a.kernel_size : adaptive_kernel(L);
  const int r = ks / 2;
  const int beg = min(n, (int)cr * span), end = min(n, beg + span);
  const int cnt_here = end - beg;
  const int rpad = (a.kernel_size > 0 ? a.kernel_size : 31) / 2;  // the launch's halo
  float* buf = reinterpret_cast<float*>(smem_sel);                  // positions beg-rpad ..
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_sel + align_up((size_t)(span + 2 * rpad) * 4, 16));
  SelCSmem& sm = *reinterpret_cast<SelCSmem*>(reinterpret_cast<unsigned char*>(keys) + (size_t)span * 4);
  const float* in = a.scores + (size_t)ukv * (a.max_len - W);

  // ---- load this CTA's scores with the pooling halo, then pool into ordered keys ----------
  for (int j = tid; j < cnt_here + 2 * r; j += blockDim.x) {
    const int i = beg - r + j;
    buf[j] = (i >= 0 && i < n) ? in[i] : -INFINITY;
  }
  __syncthreads();
  for (int q = tid; q < cnt_here; q += blockDim.x) {
    const int i = beg + q;
    float m;
    if (a.pool_avg) {
      const int lo = max(0, i - r), hi = min(n - 1, i + r);
      long long sum = 0;
      for (int j = lo; j <= hi; ++j) sum += to_fixed(buf[j - beg + r]);
      m = fixed_mean(sum, hi - lo + 1);
    } else {
      m = buf[q + r];
      for (int j = 0; j <= 2 * r; ++j) m = fmaxf(m, buf[q + j]);  // -inf outside [0, n)
    }
    keys[q] = ordered_key(m);
  }

  // ---- radix select over the cluster ---------------------------------------------------------
  const int want = a.keep - W;
  uint32_t prefix = 0u, mask = 0u;
  int remaining = want;
  bool inclusive = false;
  int start = 32;
  while (start > 0 && !inclusive) {
    const int nb = start >= 11 ? 11 : start;
    const int shift = start - nb;
    const uint32_t dmask = (1u << nb) - 1u;
    for (int b = tid; b < kSelCBins; b += blockDim.x) sm.hist[b] = 0u;
    __syncthreads();
    // pooled scores share few leading bits, so many keys of a warp fall in one bin: one atomic
    // per distinct bin and warp (its lanes' count)
    for (int q0 = 0; q0 < cnt_here; q0 += blockDim.x) {
      const int q = q0 + tid;
      const uint32_t k = q < cnt_here ? keys[q] : 0u;
      const bool in = q < cnt_here && (k & mask) == prefix;
      const uint32_t act = __ballot_sync(0xffffffffu, in);
      if (in) {
        const uint32_t bin = (k >> shift) & dmask;
        const uint32_t peers = __match_any_sync(act, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&sm.hist[bin], (uint32_t)__popc(peers));
      }
    }
    cluster_sync_all();  // every CTA's histogram is complete
    // thread t: bins 2047 - 2t and 2046 - 2t (descending), summed over the cluster
    uint32_t c0 = 0u, c1 = 0u;
    for (uint32_t c = 0; c < (uint32_t)kSelCluster; ++c) {
      c0 += ld_peer_u32(&sm.hist[kSelCBins - 1 - 2 * tid], c);
      c1 += ld_peer_u32(&sm.hist[kSelCBins - 2 - 2 * tid], c);
    }
    const unsigned long long tot = (unsigned long long)c0 + c1;
    const unsigned long long before = block_excl_scan64(tot, sm.tmp);
    if (before < (unsigned long long)remaining && before + tot >= (unsigned long long)remaining) {
      const bool first = before + c0 >= (unsigned long long)remaining;
      sm.found[0] = first ? kSelCBins - 1 - 2 * tid : kSelCBins - 2 - 2 * tid;
      sm.found[1] = (int)(first ? before : before + c0);
      sm.found[2] = (int)(first ? c0 : c1);
    }
    __syncthreads();
    const uint32_t digit = (uint32_t)sm.found[0];
    prefix |= (digit & dmask) << shift;
    mask |= dmask << shift;
    remaining -= sm.found[1];
    if (sm.found[2] == remaining) inclusive = true;
    start = shift;
    cluster_sync_all();  // no CTA clears its histogram while another still reads it
  }

  // ---- compaction in position order ----------------------------------------------------------
  // taken: (key & mask) > prefix, or == prefix: all of them when inclusive, else the first
  // `remaining` by position over the whole unit
  const int per = (cnt_here + (int)blockDim.x - 1) / (int)blockDim.x;
  const int q0 = min(cnt_here, tid * per), q1 = min(cnt_here, q0 + per);
  uint32_t gt = 0, eq = 0;
  for (int q = q0; q < q1; ++q) {
    const uint32_t k = keys[q] & mask;
    gt += k > prefix ? 1u : 0u;
    eq += k == prefix ? 1u : 0u;
  }
  const unsigned long long mine = ((unsigned long long)gt << 32) | eq;
  const unsigned long long bef = block_excl_scan64(mine, sm.tmp);
  if (tid == (int)blockDim.x - 1) {
    sm.cnt[0] = (uint32_t)((bef + mine) >> 32);
    sm.cnt[1] = (uint32_t)((bef + mine) & 0xffffffffull);
  }
  cluster_sync_all();
  uint32_t gt_cl = 0, eq_cl = 0;  // earlier CTAs of the cluster
  for (uint32_t c = 0; c < cr; ++c) {
    gt_cl += ld_peer_u32(&sm.cnt[0], c);
    eq_cl += ld_peer_u32(&sm.cnt[1], c);
  }
  const int need_eq = inclusive ? 0x7fffffff : remaining;
  int gt_before = (int)gt_cl + (int)(bef >> 32);
  int eq_before = (int)eq_cl + (int)(bef & 0xffffffffull);
  for (int q = q0; q < q1; ++q) {
    const uint32_t k = keys[q] & mask;
    bool take = k > prefix;
    if (k == prefix) {
      take = eq_before < need_eq;
      ++eq_before;
    }
    if (take) {
      const int pos = gt_before + min(eq_before - (k == prefix ? 1 : 0), need_eq);
      if (pos < want) kept[pos] = beg + q;
    }
    if (k > prefix) ++gt_before;
  }
  if (cr == 0) {
    for (int j = tid; j < W; j += blockDim.x) kept[want + j] = L - W + j;
    if (g == 0 && tid == 0) a.out_len[u] = a.keep;
  }
  cluster_sync_all();  // peers may still read this CTA's counts
}

// ------------------------------------------------------------------------------------------
// pooling + top-k selection with the whole unit in shared memory (n = L - W <= 32768 scores,
// pooling kernel 2^k - 1): one CTA of 1024 threads per (unit, KV head); thread t owns the 32
// consecutive positions [32t, 32t + 32).
// ------------------------------------------------------------------------------------------
constexpr int kSelThreads = 1024;
constexpr int kSelPerThread = 32;
constexpr int kSelMaxN = kSelThreads * kSelPerThread;  // 32768

// shared-memory slot of position i: one pad word per 32 keeps a thread's run conflict-free
__device__ __forceinline__ int sel_slot(int i) { return i + (i >> 5); }

size_t select_fast_smem_bytes() { return (size_t)(kSelMaxN + kSelMaxN / 32) * 4; }

// Max pooling in registers for r = 2^k - 1 <= 15 known at compile time. Thread t holds positions
// base .. base + 31 in x[] (-inf past n). A doubling step m_2w[q] = max(m_w[q], m_w[q + w]) takes
// the next thread's first w values by a shuffle, and lane 31 takes them from lane 0 of the next
// warp through xch (one buffer per step, so one barrier per step). Ascending q reads x[q + w]
// before it is updated.
template <int W>
__device__ __forceinline__ void reg_double_step(float (&x)[kSelPerThread], float* xch, int lane,
                                                int warp) {
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < W; ++j) xch[warp * 8 + j] = x[j];
  }
  float halo[W];
#pragma unroll
  for (int j = 0; j < W; ++j) halo[j] = __shfl_down_sync(0xffffffffu, x[j], 1);
  __syncthreads();
  if (lane == 31) {
#pragma unroll
    for (int j = 0; j < W; ++j)
      halo[j] = (warp + 1 < kSelThreads / 32) ? xch[(warp + 1) * 8 + j] : -INFINITY;
  }
#pragma unroll
  for (int q = 0; q < kSelPerThread; ++q)
    x[q] = fmaxf(x[q], (q + W < kSelPerThread) ? x[q + W] : halo[q + W - kSelPerThread]);
}

// After the doubling steps (w = R + 1): pooled[i] = max(m_w[max(0, i - R)], m_w[i]), with the
// previous thread's last R values by a shuffle (lane 0: from lane 31 of the previous warp through
// xch; thread 0 clips to position 0), written straight out as ordered keys with their range.
template <int R>
__device__ __forceinline__ void reg_pool_keys(const float (&x)[kSelPerThread], float* xch,
                                              uint32_t* key, int base, int n, int lane, int warp,
                                              uint32_t& hi, uint32_t& lo) {
  if constexpr (R > 0) {
    if (lane == 31) {
#pragma unroll
      for (int j = 0; j < R; ++j) xch[warp * 16 + j] = x[kSelPerThread - R + j];
    }
    __syncthreads();
  }
#pragma unroll
  for (int q = 0; q < kSelPerThread; ++q) {
    float m = x[q];
    if constexpr (R > 0) {
      float prev;
      if (q >= R) {
        prev = x[q - R];
      } else {
        prev = __shfl_up_sync(0xffffffffu, x[kSelPerThread - R + q], 1);
        if (lane == 0) prev = warp > 0 ? xch[(warp - 1) * 16 + q] : x[0];
      }
      m = fmaxf(m, prev);
    }
    const int i = base + q;
    if (i < n) {
      const uint32_t kk = ordered_key(m);
      key[sel_slot(i)] = kk;
      hi = max(hi, kk);
      lo = min(lo, kk);
    }
  }
}

template <int R>
__device__ __forceinline__ void reg_max_pool(float (&x)[kSelPerThread], float* xch, uint32_t* key,
                                             int base, int n, int lane, int warp, uint32_t& hi,
                                             uint32_t& lo) {
  if constexpr (R >= 1) reg_double_step<1>(x, xch + 0 * 256, lane, warp);
  if constexpr (R >= 3) reg_double_step<2>(x, xch + 1 * 256, lane, warp);
  if constexpr (R >= 7) reg_double_step<4>(x, xch + 2 * 256, lane, warp);
  if constexpr (R >= 15) reg_double_step<8>(x, xch + 3 * 256, lane, warp);
  reg_pool_keys<R>(x, xch + 4 * 256, key, base, n, lane, warp, hi, lo);
}

// Max pooling over [max(0, i - r), min(n - 1, i + r)] for 2r + 1 = 2^k - 1 by doubling: with
// m_w[i] = max over [i, min(i + w - 1, n - 1)], m_{2w}[i] = max(m_w[i], m_w[i + w]); once
// w = r + 1, the pooled value is max(m_w[max(0, i - r)], m_w[i]) (the two runs meet or overlap
// and end exactly at the window's clipped edges). Then a radix select over the ordered keys.
__global__ void __launch_bounds__(kSelThreads, 1) select_fast_kernel(SnapArgs a) {
  extern __shared__ __align__(16) float sh[];
  __shared__ uint32_t hist[2048];
  __shared__ int wsum[32], wsum2[32];
  __shared__ uint32_t wmax[32], wmin[32];
  __shared__ int found[4];
  __shared__ float xch[4 * 256 + 32 * 16];  // pooling exchange: 4 doubling steps, final step
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ukv = blockIdx.x;
  const int u = ukv / a.n_kv, g = ukv - u * a.n_kv;
  const int W = a.window;
  const int L = a.seq_lens[u];
  int32_t* kept = a.kept_idx + (size_t)ukv * a.kept_stride;
  if (L <= W || L > a.max_len) {
    for (int i = tid; i < a.keep; i += kSelThreads) kept[i] = -1;
    if (g == 0 && tid == 0) a.out_len[u] = 0;
    return;
  }
  if (L <= a.keep) {
    for (int i = tid; i < a.keep; i += kSelThreads) kept[i] = i < L ? i : -1;
    if (g == 0 && tid == 0) a.out_len[u] = L;
    return;
  }
  const int n = L - W;  // <= kSelMaxN (checked by the launcher)
  const int ks = a.kernel_size > 0 ? a.kernel_size : adaptive_kernel(L);
  const int r = ks / 2;
  const float* in = a.scores + (size_t)ukv * (a.max_len - W);
  // coalesced 4-byte asynchronous copies (position tid + 1024 q), all in flight at once
#pragma unroll
  for (int q = 0; q < kSelPerThread; ++q) {
    const int i = tid + q * kSelThreads;
    if (i < n) cp_async4(sh + sel_slot(i), in + i);
  }
  cp_async_commit();
  for (int i = tid; i < 2048; i += kSelThreads) hist[i] = 0u;
  cp_async_wait_all();
  __syncthreads();

  const int base = tid * kSelPerThread;
  float x[kSelPerThread];
  uint32_t hi = 0u, lo = 0xffffffffu;
  uint32_t* key = reinterpret_cast<uint32_t*>(sh);
  if (!a.pool_avg && (r == 0 || r == 1 || r == 3 || r == 7 || r == 15)) {
    // the thread's run, then pooling in registers; keys written by the last step
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q)
      x[q] = (base + q < n) ? sh[sel_slot(base + q)] : -INFINITY;
    switch (r) {
      case 0: reg_max_pool<0>(x, xch, key, base, n, lane, warp, hi, lo); break;
      case 1: reg_max_pool<1>(x, xch, key, base, n, lane, warp, hi, lo); break;
      case 3: reg_max_pool<3>(x, xch, key, base, n, lane, warp, hi, lo); break;
      case 7: reg_max_pool<7>(x, xch, key, base, n, lane, warp, hi, lo); break;
      default: reg_max_pool<15>(x, xch, key, base, n, lane, warp, hi, lo); break;
    }
  } else {
  if (a.pool_avg) {
    // mean over the clipped window: a fixed-point sum slid over the thread's 32 positions
    long long sum = 0;
    if (base < n) {
      const int hi0 = min(n - 1, base + r);
      for (int j = max(0, base - r); j <= hi0; ++j) sum += to_fixed(sh[sel_slot(j)]);
    }
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
      const int i = base + q;
      float v = 0.f;
      if (i < n) {
        if (q > 0) {
          if (i + r < n) sum += to_fixed(sh[sel_slot(i + r)]);
          if (i - r - 1 >= 0) sum -= to_fixed(sh[sel_slot(i - r - 1)]);
        }
        v = fixed_mean(sum, min(n - 1, i + r) - max(0, i - r) + 1);
      }
      x[q] = v;
    }
  } else {
    for (int w = 1; w <= r; w *= 2) {  // m_w -> m_2w until 2w = r + 1
#pragma unroll
      for (int q = 0; q < kSelPerThread; ++q) {
        const int i = base + q;
        float v = -INFINITY;
        if (i < n) {
          v = sh[sel_slot(i)];
          if (i + w < n) v = fmaxf(v, sh[sel_slot(i + w)]);
        }
        x[q] = v;
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < kSelPerThread; ++q)
        if (base + q < n) sh[sel_slot(base + q)] = x[q];
      __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
      const int i = base + q;
      float v = 0.f;
      if (i < n) v = fmaxf(sh[sel_slot(max(0, i - r))], sh[sel_slot(i)]);
      x[q] = v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kSelPerThread; ++q) {
    const int i = base + q;
    if (i < n) {
      const uint32_t kk = ordered_key(x[q]);
      key[sel_slot(i)] = kk;
      hi = max(hi, kk);
      lo = min(lo, kk);
    }
  }
  }
  hi = __reduce_max_sync(0xffffffffu, hi);
  lo = __reduce_min_sync(0xffffffffu, lo);
  if (lane == 0) {
    wmax[warp] = hi;
    wmin[warp] = lo;
  }
  __syncthreads();
  hi = 0u;
  lo = 0xffffffffu;
  for (int w = 0; w < 32; ++w) {
    hi = max(hi, wmax[w]);
    lo = min(lo, wmin[w]);
  }

  // ---- radix select of the `want` largest (ties -> lower position) -----------------------
  const int want = a.keep - W;
  const uint32_t diff = hi ^ lo;
  int start = diff ? 32 - __clz(diff) : 0;
  uint32_t mask = start >= 32 ? 0u : ~((1u << start) - 1u);
  uint32_t prefix = hi & mask;
  int remaining = want;
  bool inclusive = false;
  while (start > 0 && !inclusive) {
    const int nb = start < 11 ? start : 11;
    const int shift = start - nb;
    const uint32_t dmask = (1u << nb) - 1u;
    // counts, one atomic per run of equal digits (pooling repeats maxima)
    uint32_t run_d = 0u;
    uint32_t run_c = 0u;
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
      const int i = base + q;
      if (i < n) {
        const uint32_t kk = key[sel_slot(i)];
        if ((kk & mask) == prefix) {
          const uint32_t d = (kk >> shift) & dmask;
          if (run_c > 0u && d != run_d) {
            atomicAdd(&hist[run_d], run_c);
            run_c = 0u;
          }
          run_d = d;
          ++run_c;
        }
      }
    }
    if (run_c > 0u) atomicAdd(&hist[run_d], run_c);
    __syncthreads();
    // thread t holds bins 2047 - 2t and 2046 - 2t (descending), and clears them for the next pass
    const int c_hi = (int)hist[2047 - 2 * tid], c_lo = (int)hist[2046 - 2 * tid];
    hist[2047 - 2 * tid] = 0u;
    hist[2046 - 2 * tid] = 0u;
    const int own = c_hi + c_lo;
    const int incl_w = warp_incl_scan(own);
    if (lane == 31) wsum[warp] = incl_w;
    __syncthreads();
    int before;
    {  // the totals of the warps before this one, by a scan of all 32 in every warp
      const int xw = wsum[lane];
      before = __shfl_sync(0xffffffffu, warp_incl_scan(xw) - xw, warp);
    }
    const int incl = before + incl_w, excl = incl - own;
    if (excl < remaining && incl >= remaining) {
      if (excl + c_hi >= remaining) {
        found[0] = 2047 - 2 * tid;
        found[1] = excl;
        found[2] = c_hi;
      } else {
        found[0] = 2046 - 2 * tid;
        found[1] = excl + c_hi;
        found[2] = c_lo;
      }
    }
    __syncthreads();
    const int digit = found[0], above = found[1], in_bin = found[2];
    prefix |= (uint32_t)digit << shift;
    mask |= dmask << shift;
    remaining -= above;
    start = shift;
    if (in_bin == remaining) inclusive = true;
  }

  // ---- compaction in position order: block scan of (above, equal) counts -----------------
  const int need_eq = inclusive ? 0 : remaining;
  int cg = 0, ce = 0;
#pragma unroll
  for (int q = 0; q < kSelPerThread; ++q) {
    const int i = base + q;
    if (i < n) {
      const uint32_t kk = key[sel_slot(i)];
      cg += (inclusive ? kk >= prefix : kk > prefix) ? 1 : 0;
      ce += (!inclusive && kk == prefix) ? 1 : 0;
    }
  }
  const int ig = warp_incl_scan(cg), ie = warp_incl_scan(ce);
  if (lane == 31) {
    wsum[warp] = ig;
    wsum2[warp] = ie;
  }
  __syncthreads();
  // each warp scans the 32 per-warp totals itself (lane l holds warp l's) instead of a serial
  // loop over them in every thread
  int gb, eb, gtot, etot;
  {
    const int x1 = wsum[lane], x2 = wsum2[lane];
    const int s1 = warp_incl_scan(x1), s2 = warp_incl_scan(x2);
    gb = ig - cg + __shfl_sync(0xffffffffu, s1 - x1, warp);
    eb = ie - ce + __shfl_sync(0xffffffffu, s2 - x2, warp);
    gtot = __shfl_sync(0xffffffffu, s1, 31);
    etot = __shfl_sync(0xffffffffu, s2, 31);
  }
#pragma unroll
  for (int q = 0; q < kSelPerThread; ++q) {
    const int i = base + q;
    if (i < n) {
      const uint32_t kk = key[sel_slot(i)];
      const bool gsel = inclusive ? kk >= prefix : kk > prefix;
      const bool esel = !inclusive && kk == prefix;
      if (gsel) {
        const int pos = gb + min(eb, need_eq);
        if (pos < want) kept[pos] = i;
        ++gb;
      } else if (esel) {
        if (eb < need_eq && gb + eb < want) kept[gb + eb] = i;
        ++eb;
      }
    }
  }
  if (gtot + min(etot, need_eq) != want && tid == 0) set_status(a.status, RKV_DEV_SELECT_FAILED);
  for (int j = tid; j < W; j += kSelThreads) kept[want + j] = L - W + j;
  if (g == 0 && tid == 0) a.out_len[u] = a.keep;
}

// ------------------------------------------------------------------------------------------
// compaction gather: CTA = 64 kept rows of one (unit, KV head); each thread copies 16-byte
// chunks of K and V rows
// ------------------------------------------------------------------------------------------
// Page summaries of rows row0 .. min(cnt, row0 + 64) - 1 of a unit's compact cache, from the
// rows this CTA holds (kv[i] = row row0 + (tid >> 4) + 16 i, chunk tid & 15, valid where ok[i]).
__device__ __forceinline__ void gather_summaries(const SnapArgs& a, int ukv, int row0, int cnt,
                                                 const uint4 (&kv)[4], const bool (&ok)[4],
                                                 uint4* gsm) {
  const int tid = threadIdx.x, p = a.page;
  uint4* srow = gsm;                        // [64][16]
  uint4* smin = gsm + 64 * 16;              // [64 / p][16]
  uint4* smax = smin + (64 / p) * 16;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (ok[i]) srow[((tid >> 4) + 16 * i) * 16 + (tid & 15)] = kv[i];
  __syncthreads();
  const int nrows = min(64, cnt - row0);
  const int npg = (nrows + p - 1) / p;      // pages (the last may be partial)
  const __nv_bfloat162 pinf = __halves2bfloat162(__ushort_as_bfloat16(0x7F80),
                                                 __ushort_as_bfloat16(0x7F80));
  const __nv_bfloat162 ninf = __halves2bfloat162(__ushort_as_bfloat16(0xFF80),
                                                 __ushort_as_bfloat16(0xFF80));
  for (int it = tid; it < npg * 16; it += 256) {
    const int j = it >> 4, c = it & 15;
    const int r1 = min(nrows, (j + 1) * p);
    __nv_bfloat162 mn[4] = {pinf, pinf, pinf, pinf}, mx[4] = {ninf, ninf, ninf, ninf};
    for (int r = j * p; r < r1; ++r) {
      const uint4 x = srow[r * 16 + c];
      const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mn[e] = __hmin2(mn[e], y[e]);
        mx[e] = __hmax2(mx[e], y[e]);
      }
    }
    smin[j * 16 + c] = *reinterpret_cast<const uint4*>(mn);
    smax[j * 16 + c] = *reinterpret_cast<const uint4*>(mx);
  }
  __syncthreads();
  // channel-major rows: thread -> (channel, group of 8 pages)
  const int pg0 = row0 / p;
  const int ngrp = (npg + 7) / 8;
  const uint16_t* smin16 = reinterpret_cast<const uint16_t*>(smin);
  const uint16_t* smax16 = reinterpret_cast<const uint16_t*>(smax);
  uint16_t* kmin16 = reinterpret_cast<uint16_t*>(a.kmin);
  uint16_t* kmax16 = reinterpret_cast<uint16_t*>(a.kmax);
  for (int it = tid; it < kHeadDim * ngrp; it += 256) {
    const int ch = it / ngrp, j0 = (it - ch * ngrp) * 8;
    const size_t row = ((size_t)ukv * kHeadDim + ch) * a.page_cap + pg0 + j0;
    uint16_t vmin[8], vmax[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int j = min(j0 + t, npg - 1);
      vmin[t] = smin16[j * kHeadDim + ch];
      vmax[t] = smax16[j * kHeadDim + ch];
    }
    if (j0 + 8 <= npg && (pg0 & 7) == 0) {
      uint4 wmin, wmax;
      wmin.x = vmin[0] | ((uint32_t)vmin[1] << 16);
      wmin.y = vmin[2] | ((uint32_t)vmin[3] << 16);
      wmin.z = vmin[4] | ((uint32_t)vmin[5] << 16);
      wmin.w = vmin[6] | ((uint32_t)vmin[7] << 16);
      wmax.x = vmax[0] | ((uint32_t)vmax[1] << 16);
      wmax.y = vmax[2] | ((uint32_t)vmax[3] << 16);
      wmax.z = vmax[4] | ((uint32_t)vmax[5] << 16);
      wmax.w = vmax[6] | ((uint32_t)vmax[7] << 16);
      *reinterpret_cast<uint4*>(kmin16 + row) = wmin;
      *reinterpret_cast<uint4*>(kmax16 + row) = wmax;
    } else {
      for (int t = 0; t < 8 && j0 + t < npg; ++t) {
        kmin16[row + t] = vmin[t];
        kmax16[row + t] = vmax[t];
      }
    }
  }
}

// With a.kmin set the gather also builds the page summaries of the rows it writes: its 64 rows
// are whole pages (page | 64), staged in shared memory, reduced per (page, 16-byte chunk) and
// written channel-major like summaries_kernel. Dynamic shared memory: gather_smem_bytes(page).
size_t gather_smem_bytes(int page) {
  return (size_t)64 * 256 + 2 * (size_t)(64 / page) * 256;
}

__global__ void __launch_bounds__(256) gather_kernel(SnapArgs a) {
  extern __shared__ __align__(16) uint4 gsm[];
  const int ukv = blockIdx.y;
  const int u = ukv / a.n_kv;
  const int L = a.seq_lens[u];
  if (L <= a.window || L > a.max_len) return;
  const int cnt = min(L, a.keep);
  const int row0 = blockIdx.x * 64;
  if (row0 >= cnt) return;
  const int32_t* kept = a.kept_idx + (size_t)ukv * a.kept_stride;
  const size_t src_unit = (size_t)(ukv / a.kv_div);
  const uint4* ksrc = reinterpret_cast<const uint4*>(a.k + src_unit * a.max_len * kHeadDim);
  const uint4* vsrc = reinterpret_cast<const uint4*>(a.v + src_unit * a.max_len * kHeadDim);
  // destination: the unit's rows of k_out / v_out, or (paged) its pages in the pools
  const bool paged = a.out_pm.table != nullptr;
  const int g = ukv - u * a.n_kv;
  uint4* kdst = reinterpret_cast<uint4*>(paged ? a.k_out : a.k_out + (size_t)ukv * a.cap * kHeadDim);
  uint4* vdst = reinterpret_cast<uint4*>(paged ? a.v_out : a.v_out + (size_t)ukv * a.cap * kHeadDim);
  uint4 kv[4], vv[4];
  size_t dst[4];
  bool ok[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = threadIdx.x + 256 * i;  // 64 rows x 16 chunks
    const int row = row0 + (idx >> 4), ch = idx & 15;
    ok[i] = false;
    dst[i] = 0;
    if (row < cnt) {
      const int src = kept[row];
      if (src >= 0 && src < L) {
        kv[i] = ksrc[(size_t)src * 16 + ch];
        vv[i] = vsrc[(size_t)src * 16 + ch];
        const size_t r = paged ? paged_row(a.out_pm, paged_block(a.out_pm, u, row, a.status),
                                           a.n_kv, g, row)
                               : (size_t)row;
        dst[i] = r * 16 + ch;
        ok[i] = true;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (ok[i]) {
      kdst[dst[i]] = kv[i];
      vdst[dst[i]] = vv[i];
    }
  }
  if (a.kmin) gather_summaries(a, ukv, row0, cnt, kv, ok, gsm);
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
// Split plan: about 16 work items per SM for balance, at least 4 tiles per item.
void snapkv_plan(int n, int n_kv, int gqa, int max_len, int window, int* nsplit,
                 int* tokens_per_split, int* rows_pad) {
  (void)window;
  const int units = n * n_kv;
  const int tiles = (max_len + kTileTok - 1) / kTileTok;
  int ns = (16 * device_sm_count() + units - 1) / units;
  const int max_ns = tiles / 4 > 1 ? tiles / 4 : 1;
  ns = ns < 1 ? 1 : (ns > max_ns ? max_ns : ns);
  const int tps = (tiles + ns - 1) / ns;
  ns = (tiles + tps - 1) / tps;
  *nsplit = ns;
  *tokens_per_split = tps;  // in tiles
  *rows_pad = gqa * window <= 128 ? 128 : 256;
}

size_t snapkv_scratch_bytes(int n, int n_kv, int gqa, int max_len, int window) {
  int ns, tps, rp;
  snapkv_plan(n, n_kv, gqa, max_len, window, &ns, &tps, &rp);
  const size_t plen = align_up((size_t)n * n_kv * (max_len - window) * 4, 256);
  return 2 * plen + align_up((size_t)n * n_kv * ns * rp * 2 * 4, 256) +
         align_up((size_t)n * n_kv * rp * 4, 256);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// rows x 128 bf16, row-major, boxes of 128 rows x 64 columns, 128-byte swizzle
static bool make_rows_map(CUtensorMap* map, const void* base, uint64_t rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int PASS, int RB>
static cudaError_t launch_pass(const CUtensorMap& km, const CUtensorMap& qm,
                               const ScoreParams& sp, cudaStream_t s) {
  const size_t smem = ScoreSmem<RB>::total;
  cudaError_t e = ensure_dyn_smem((const void*)score_kernel<PASS, RB>, smem);
  if (e != cudaSuccess) return e;
  const int items = sp.units * sp.nsplit;
  const int sms = device_sm_count();
  const int grid = items < sms ? items : sms;
  e = launch_pdl_kernel(score_kernel<PASS, RB>, dim3(grid), dim3(kScoreThreads), smem, s, km, qm,
                        sp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_snapkv(const SnapArgs& a, cudaStream_t s) {
  CUtensorMap km, qm;
  const uint64_t krows = (uint64_t)a.n * (a.n_kv / a.kv_div) * a.max_len;
  const uint64_t qrows = (uint64_t)a.n * a.n_kv * a.gqa * a.window;
  if (!make_rows_map(&km, a.k, krows) || !make_rows_map(&qm, a.q_win, qrows))
    return cudaErrorInvalidValue;
  const int units = a.n * a.n_kv;
  ScoreParams sp{};
  sp.n_kv = a.n_kv;
  sp.gqa = a.gqa;
  sp.window = a.window;
  sp.max_len = a.max_len;
  sp.hq = a.n_kv * a.gqa;
  sp.units = units;
  sp.nsplit = a.nsplit;
  sp.kv_div = a.kv_div;
  sp.tiles_per_split = a.tokens_per_split;
  sp.scale_log2 = a.scale_log2;
  sp.seq_lens = a.seq_lens;
  sp.part_ml = a.part_ml;
  sp.nlse = a.nlse;
  sp.scores = a.scores;
  sp.status = a.status;
  sp.wait_limit_ns = a.wait_limit_ns ? a.wait_limit_ns : kWaitLimitNs;
  sp.test_skip_tile = a.test_skip_tile;
  cudaError_t e;
  sp.reverse = 0;
  e = a.rows_pad == 128 ? launch_pass<1, 1>(km, qm, sp, s) : launch_pass<1, 2>(km, qm, sp, s);
  if (e != cudaSuccess) return e;
  e = launch_pdl_kernel(lse_merge_kernel, dim3(units), dim3(a.rows_pad), 0, s, sp, a.rows_pad);
  if (e != cudaSuccess) return e;
  sp.reverse = 1;
  e = a.rows_pad == 128 ? launch_pass<2, 1>(km, qm, sp, s) : launch_pass<2, 2>(km, qm, sp, s);
  if (e != cudaSuccess) return e;
  if (a.scores_only) return cudaSuccess;
  // the whole-unit shared-memory select applies when every unit fits and the pooling kernel is
  // 2^k - 1 (the adaptive sizes 7 / 15 / 31 all are)
  const bool pow2_kernel =
      a.pool_avg || a.kernel_size <= 0 || ((a.kernel_size + 1) & a.kernel_size) == 0;
  const int nmax = a.max_len - a.window;
  const int span = ((nmax + kSelCluster - 1) / kSelCluster + 3) & ~3;
  const int rpad = (a.kernel_size > 0 ? a.kernel_size : 31) / 2;
  if (nmax <= kSelMaxN && pow2_kernel) {
    const size_t smem = select_fast_smem_bytes();
    e = ensure_dyn_smem((const void*)select_fast_kernel, smem);
    if (e != cudaSuccess) return e;
    select_fast_kernel<<<units, kSelThreads, smem, s>>>(a);
  } else if (span <= kSelCMaxSpan && rpad <= kSelCMaxRadius &&
             (long long)units * kSelCluster <= 4LL * device_sm_count()) {
    // long prompts and few units (one CTA per unit would leave most SMs idle): a cluster of
    // CTAs per (unit, KV head). Measured at 128K prompts: 8 units 55 against 307 us, 64 units
    // 272 against 311 us; with 128 units (ragged serving batch) the one-CTA select is faster
    // (164 against 340 us).
    const size_t smem = select_cluster_smem_bytes(span, rpad);
    e = ensure_dyn_smem((const void*)select_cluster_kernel, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kSelCluster, units);
    cfg.blockDim = dim3(kSelCThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSelCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, select_cluster_kernel, a, span);
    if (e != cudaSuccess) return e;
  } else {
    select_kernel<<<units, 1024, 0, s>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!a.k_out) return cudaSuccess;  // index-only selection (RocketKV-MT keeps every row)
  const size_t gsmem = a.kmin ? gather_smem_bytes(a.page) : 0;
  if (gsmem) {
    e = ensure_dyn_smem((const void*)gather_kernel, gsmem);
    if (e != cudaSuccess) return e;
  }
  gather_kernel<<<dim3((a.keep + 63) / 64, units), 256, gsmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace rkv
