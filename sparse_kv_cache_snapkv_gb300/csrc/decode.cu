// Stage-2 kernels of RocketKV on sm_103a: page summaries, decode-token append, the fused hybrid
// sparse decode (channel pick -> approximate page scores -> page top-k -> exact attention over
// the selected pages), and the dense split-K decode used as the full-KV reference.
//
// Method: "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage KV Cache
// Compression", OpenReview author responses (paperhub.cn): "Explanation of Calculating
// Approximate Attention Scores" (pages of consecutive tokens with element-wise Kmin / Kmax,
// only the top-|q| channels, the Kmin-or-Kmax pick by the sign of q, GQA group sums), "Lack of
// Direct Latency Comparison" (half of the budget to the approximation, half to exact sparse
// attention), "Are Different KV Tokens Retrieved at Each Decoding Step?" (selection per step).
//
// Memory movement: the approximate scores read the kept channels' summary rows straight from
// global memory into registers (a vector-matrix product: fp32 FMAs, no staging), after the
// channel pick has brought every channel that can still be picked into L2; the K/V rows of the
// selected pages are staged in shared memory by 16-byte cp.async copies, each warp the 16-token
// unit it attends over (the dense decode: each warp group a 64-token chunk), rows padded by
// 16 bytes so that ldmatrix reads them without bank conflicts.
//
// Attention arithmetic: warp-level mma.sync m16n8k16 (bf16 in, fp32 accumulate). The G query
// heads of a KV group are the rows of the A operand (padded to 16 with zeros); each warp takes 16
// tokens at a time: S = Q K^T (16 MMAs), an online softmax on the accumulator fragments, and
// O += P V (16 MMAs) with P re-packed from the accumulators as the next A operand.
#include <atomic>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "rkv_internal.h"

namespace rkv {

constexpr int kRowPad = 136;                                    // staged row stride (bf16)
constexpr int kStageElems = 2 * kChunkTokens * kRowPad;         // K rows then V rows
constexpr int kStageBytes = kStageElems * 2;                    // 34,816 B
constexpr int kDecStages = 2;                                   // one per warp group


// ------------------------------------------------------------------------------------------
// warp-level MMA helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A B + C for one m16n8k16 tile; only A rows 0..7 are ever non-zero here, so a1 = a3 = 0
// and the outputs of rows 8..15 are dropped.
__device__ __forceinline__ void mma_rows8(float& d0, float& d1, uint32_t a0, uint32_t a2,
                                          uint32_t b0, uint32_t b1) {
  float x2 = 0.f, x3 = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d0), "+f"(d1), "+f"(x2), "+f"(x3)
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------------------------------
// Warp attention state over 16-token groups of a stage.
// Lane roles (m16n8k16 fragments): r0 = lane / 4 is the query-head row (rows >= G are zero
// padding), t = lane % 4 picks the column pair 2t, 2t+1 of every 8-wide tile.
// ------------------------------------------------------------------------------------------
template <int G>
struct MmaAttn {
  const uint2* qf;  // Q A-fragments in shared memory: qf[ks * 32 + lane] = {a0, a2}
  float m, l;       // running max (log2 domain) and sum for row r0 (partial per lane)
  float o[16][2];   // row r0, channels 8nt + 2t, 8nt + 2t + 1
  int lane, r0, t;

  // Q fragments are shared by every warp of the CTA: built once in shared memory by one warp
  // from the fp32 copy of q (exact: the values are bf16); row r0 = lane / 4 < G holds query head
  // r0, rows >= G are zero.
  static __device__ __forceinline__ void build_fragments(const float* q_group, uint2* frag) {
    const int ln = threadIdx.x & 31, rr = ln >> 2, tt = ln & 3;
    const float* qr = q_group + rr * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint2 f = make_uint2(0u, 0u);
      if (rr < G) {
        const float2 x = *reinterpret_cast<const float2*>(qr + ks * 16 + 2 * tt);
        const float2 y = *reinterpret_cast<const float2*>(qr + ks * 16 + 8 + 2 * tt);
        f = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(y.x, y.y));
      }
      frag[ks * 32 + ln] = f;
    }
  }

  // The same fragments straight from the bf16 q rows in global memory.
  static __device__ __forceinline__ void build_fragments(const bf16* q_group, uint2* frag) {
    const int ln = threadIdx.x & 31, rr = ln >> 2, tt = ln & 3;
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(q_group + rr * kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      frag[ks * 32 + ln] = (rr < G) ? make_uint2(qw[ks * 8 + tt], qw[ks * 8 + 4 + tt])
                                    : make_uint2(0u, 0u);
  }

  __device__ __forceinline__ void init(const uint2* frag) {
    lane = threadIdx.x & 31;
    r0 = lane >> 2;
    t = lane & 3;
    qf = frag;
    m = -1e30f;
    l = 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = 0.f;
  }

  // Lane roles of the two ldmatrix operands: the K row (token n_k) and 16-byte half kh this lane
  // addresses for S = Q K^T, and the V row (token n_v) and column block cb for O += P V.
  static __device__ __forceinline__ int k_row(int ln) { return (ln & 7) + ((ln >> 4) << 3); }
  static __device__ __forceinline__ int k_col(int ln) { return ((ln >> 3) & 1) * 8; }
  static __device__ __forceinline__ int v_row(int ln) { return (ln & 7) + (((ln >> 3) & 1) << 3); }
  static __device__ __forceinline__ int v_col(int ln) { return (ln >> 4) << 3; }

  // tokens tok0 .. tok0 + 15 of a stage with `ntok` valid rows (rows >= ntok of V are zero)
  __device__ __forceinline__ void step16(const bf16* Ks, const bf16* Vs, int tok0, int ntok,
                                         float scale_log2) {
    step16_at(Ks + (tok0 + k_row(lane)) * kRowPad + k_col(lane),
              Vs + (tok0 + v_row(lane)) * kRowPad + v_col(lane), tok0, ntok, scale_log2);
  }

  // The same step with this lane's ldmatrix row addresses given (rows anywhere in shared memory,
  // each kRowPad-aligned as staged): kaddr = row k_row(lane) + k_col(lane), vaddr = row
  // v_row(lane) + v_col(lane) of the 16-token unit.
  __device__ __forceinline__ void step16_at(const bf16* kaddr, const bf16* vaddr, int tok0,
                                            int ntok, float scale_log2) {
    float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
    {
      const uint32_t base = smem_addr(kaddr);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(base + ks * 32, b0, b1, b2, b3);
        const uint2 qa = qf[ks * 32 + lane];
        mma_rows8(s00, s01, qa.x, qa.y, b0, b1);
        mma_rows8(s10, s11, qa.x, qa.y, b2, b3);
      }
    }
    const int j = tok0 + 2 * t;
    float s[4] = {s00 * scale_log2, s01 * scale_log2, s10 * scale_log2, s11 * scale_log2};
    s[0] = (j < ntok) ? s[0] : -INFINITY;
    s[1] = (j + 1 < ntok) ? s[1] : -INFINITY;
    s[2] = (j + 8 < ntok) ? s[2] : -INFINITY;
    s[3] = (j + 9 < ntok) ? s[3] : -INFINITY;
    float mt = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float mn = fmaxf(m, mt);
    const float alpha = fast_exp2(m - mn);
    m = mn;
    // P in bf16 (the A operand of P V); l sums the same rounded values
    const __nv_bfloat162 p01 = __floats2bfloat162_rn(fast_exp2(s[0] - mn), fast_exp2(s[1] - mn));
    const __nv_bfloat162 p23 = __floats2bfloat162_rn(fast_exp2(s[2] - mn), fast_exp2(s[3] - mn));
    const float2 f01 = __bfloat1622float2(p01), f23 = __bfloat1622float2(p23);
    l = l * alpha + ((f01.x + f01.y) + (f23.x + f23.y));
    const uint32_t pa0 = *reinterpret_cast<const uint32_t*>(&p01);
    const uint32_t pa2 = *reinterpret_cast<const uint32_t*>(&p23);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= alpha;
      o[nt][1] *= alpha;
    }
    {
      const uint32_t base = smem_addr(vaddr);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(base + np * 32, v0, v1, v2, v3);
        mma_rows8(o[2 * np][0], o[2 * np][1], pa0, pa2, v0, v1);
        mma_rows8(o[2 * np + 1][0], o[2 * np + 1][1], pa0, pa2, v2, v3);
      }
    }
  }

  __device__ __forceinline__ float row_l() const {
    float x = l;
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
  }
};

template <int G>
struct CombineSmem {
  float m[8][G];
  float l[8][G];
  float o[8][G][kHeadDim];
};

template <int G>
__device__ __forceinline__ void warp_deposit(const MmaAttn<G>& at, CombineSmem<G>* cs) {
  const int w = threadIdx.x >> 5;
  const float lt = at.row_l();
  if (at.r0 < G) {
    if (at.t == 0) {
      cs->m[w][at.r0] = at.m;
      cs->l[w][at.r0] = lt;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      cs->o[w][at.r0][nt * 8 + 2 * at.t] = at.o[nt][0];
      cs->o[w][at.r0][nt * 8 + 2 * at.t + 1] = at.o[nt][1];
    }
  }
}

// Merge the 8 warps for (h, c): unnormalised output relative to max M, with its sum L.
template <int G>
__device__ __forceinline__ void warp_merge(const CombineSmem<G>* cs, int h, int c, float* M,
                                           float* L, float* O) {
  float mm = -1e30f;
#pragma unroll
  for (int w = 0; w < 8; ++w) mm = fmaxf(mm, cs->m[w][h]);
  float ll = 0.f, oo = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float f = fast_exp2(cs->m[w][h] - mm);
    ll = fmaf(cs->l[w][h], f, ll);
    oo = fmaf(cs->o[w][h][c], f, oo);
  }
  *M = mm;
  *L = ll;
  *O = oo;
}

// Per-warp partial state in the warp's own staging rows (no other warp touches them, so no
// block barrier is needed before depositing): m[G], l[G], then o[G][kORow] (rows padded to 136
// floats so that the fragment stores of the G rows fall in distinct banks).
constexpr int kORow = 136;
template <int G>
__device__ __forceinline__ float* warp_state(bf16* stages, int w, size_t wstride) {
  return reinterpret_cast<float*>(stages + (size_t)w * wstride);
}
static_assert((2 * 8 + 8 * kORow) * 4 <= 2 * 16 * kRowPad * 2, "warp state fits its rows");

template <int G>
__device__ __forceinline__ void warp_deposit_own(const MmaAttn<G>& at, float* st) {
  const float lt = at.row_l();
  if (at.r0 < G) {
    if (at.t == 0) {
      st[at.r0] = at.m;
      st[G + at.r0] = lt;
    }
    float* o = st + 2 * G + at.r0 * kORow + 2 * at.t;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<float2*>(o + nt * 8) = make_float2(at.o[nt][0], at.o[nt][1]);
  }
}

// Zero V rows [ntok, round_up(ntok, 16)) of a partially filled stage so that P = 0 never meets
// stale bits there (0 * NaN would poison the accumulators). Called by the 128 threads of a group.
__device__ __forceinline__ void zero_tail_rows(bf16* Vs, int ntok, int gtid) {
  const int r1 = min(kChunkTokens, (ntok + 15) & ~15);
  const int n16 = (r1 - ntok) * 16;  // 16-byte words
  for (int i = gtid; i < n16; i += 128) {
    const int r = ntok + (i >> 4), c = i & 15;
    *reinterpret_cast<uint4*>(Vs + r * kRowPad + c * 8) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async();
}

__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + group) : "memory");
}

// ==========================================================================================
// Hybrid sparse decode: one CTA of 8 warps per (unit, KV head).
// ==========================================================================================
// The selected pages: the S = B / 2 / p of a sparse step, or every page of a dense one (a
// sequence of at most B tokens), never more than page_cap.
inline int sel_entries(int page_cap, int budget, int page) {
  const int dense_pages = (budget + page - 1) / page;
  return page_cap < dense_pages ? page_cap : dense_pages;
}

size_t hybrid_smem_bytes(int gqa, int page_cap, int budget, int page) {
  (void)gqa;
  size_t b = (size_t)kDecStages * kStageBytes;                       // K/V stages, warp states
  b += align_up((size_t)page_cap * 4, 16);                            // approximate scores
  b += align_up((size_t)sel_entries(page_cap, budget, page) * 4, 16);  // selected pages
  return b;
}

// Wide layout, for launches of at most one CTA per SM: the staging area holds either every kept
// channel's summary row at once (the page-score GEMV reads them from shared memory after one
// round of copies) or every selected token's K and V rows at once (each warp stages all of its
// 16-token units before it waits). Returns 0 when that does not fit beside the scores and the
// selection in kWideSmemMax bytes.
constexpr size_t kWideSmemMax = 190 * 1024;
constexpr size_t kUnitRowsBytes = (size_t)2 * 16 * kRowPad * 2;  // one 16-token unit, K + V

__host__ __device__ inline int wide_units_per_warp(int budget) {
  const int units = ((budget / 2) + 15) / 16;
  return (units + 7) / 8;
}

__host__ __device__ inline size_t wide_region_bytes(int channels, int page_cap, int budget) {
  const size_t gemv = (size_t)channels * page_cap * 2;
  const size_t att = (size_t)8 * wide_units_per_warp(budget) * kUnitRowsBytes;
  size_t r = gemv > att ? gemv : att;
  const size_t base = (size_t)kDecStages * kStageBytes;
  return align_up(r > base ? r : base, 16);
}

// After the region, the scores and the selection, the wide layout holds the kept rows'
// addresses (kHeadDim pointers); being larger, its size never equals the ordinary layout's, by
// which the kernel tells the two apart.
__host__ __device__ inline size_t wide_smem_bytes(int channels, int page_cap, int budget) {
  const size_t b = wide_region_bytes(channels, page_cap, budget) +
                   2 * align_up((size_t)page_cap * 4, 16) + kHeadDim * sizeof(void*);
  return b <= kWideSmemMax ? b : 0;
}

// MODE 0: the sequence is the cache itself (A = HybridArgs, whose smaller parameter block keeps
// the plain launch cheaper); 3: the same with this step's token appended first
// (A = HybridArgsApp); 1: the kept list of the full cache (RocketKV-MT, A = HybridArgsMT);
// 2: a paged cache (A = HybridArgsPaged). Modes 1 and 2 append when a.ap.new_k is set.
template <int G, int MODE, typename A>
__global__ void __launch_bounds__(kDecodeThreads, 2) hybrid_decode_kernel(A a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(16) uint32_t ukey[kHeadDim];  // ordered key of sum_h |q_h[c]|
  __shared__ float qg[kHeadDim];                     // sum_h q_h[c]
  __shared__ int chosen[kHeadDim];
  __shared__ int part_rank[kHeadDim];
  __shared__ int wcnt[4];
  __shared__ BinSelectSmem bsel;
  __shared__ union {
    SelectScratch generic;
    FastSelectSmem fast;
  } sel_smem;
  __shared__ uint2 qfrag[8 * 32];

  // The launch picks the layout through the dynamic shared-memory size: the wide one (see
  // wide_smem_bytes) when it allotted exactly that much.
  uint32_t dsmem;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dsmem));
  const size_t wbytes = wide_smem_bytes(a.channels, a.page_cap, a.budget);
  const bool wide = wbytes != 0 && dsmem == (uint32_t)wbytes;
  const size_t region = wide ? wide_region_bytes(a.channels, a.page_cap, a.budget)
                             : (size_t)kDecStages * kStageBytes;
  const int upw = wide ? wide_units_per_warp(a.budget) : 1;  // 16-token units staged per warp
  bf16* stages = reinterpret_cast<bf16*>(smem);
  float* scores = reinterpret_cast<float*>(smem + region);
  int* sel = reinterpret_cast<int*>(smem + region + align_up((size_t)a.page_cap * 4, 16));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ukv = blockIdx.x;
  const int u = ukv / a.n_kv;
  const int g = ukv - u * a.n_kv;
  const int hq = a.n_kv * G;
  pdl_wait();     // inputs may come from the kernel before this one in the stream
  pdl_trigger();  // the next decode step may be scheduled while this one runs
  // q and len are loaded together (q's address does not depend on len): thread c < 128 loads
  // channel c of every query head of the group
  const bf16* qgroup = a.q + ((size_t)u * hq + g * G) * kHeadDim;
  float qv[G];
  if (tid < kHeadDim) {
#pragma unroll
    for (int h = 0; h < G; ++h) qv[h] = __bfloat162float(qgroup[h * kHeadDim + tid]);
  }
  int len = a.len[u];
  int flen = a.cap;  // rows a kept index may name
  int vcap = a.cap;  // bound of len
  if constexpr (MODE == 1) {
    flen = a.full_len[u];
    vcap = a.vcap;
  }
  if constexpr (MODE == 2) vcap = a.pm.max_blocks * a.pm.block;
  bool appended = false;  // this launch appended the unit's token (length advanced at the end)
  const int len0 = len;
  int arow = 0;
  if constexpr (MODE != 0) {
    if (a.ap.new_k != nullptr) {
      // ---- append this step's token before attending (it is selectable in this step) ----
      // threads 0..127 write the K row and fold it into its page's Kmin / Kmax, threads
      // 128..255 the V row. The unit's length advances at the end of the launch: the last of
      // the unit's KV-head CTAs to finish (all of them read the length at their start) writes it.
      const int row = (MODE == 1) ? flen : len;  // cache row receiving the token
      arow = row;
      const int pg0 = len / a.page;
      const bool fits = len >= 0 && len < vcap && pg0 < a.page_cap && row >= 0 && row < a.cap;
      if (fits) {
        const int c = tid & (kHeadDim - 1);
        size_t dst;
        if constexpr (MODE == 2)
          dst = paged_row(a.pm, paged_block(a.pm, u, len, a.status), a.n_kv, g, len);
        else
          dst = (size_t)ukv * a.cap + row;
        const size_t src = (size_t)ukv * kHeadDim + c;
        if (tid < kHeadDim) {
          const size_t si = src * a.page_cap + pg0;
          const bf16 kval = a.ap.new_k[src];
          const bool fresh = len % a.page == 0;  // the token opens a new page
          bf16 omin = kval, omax = kval;
          if (!fresh) {
            omin = a.kmin[si];
            omax = a.kmax[si];
          }
          const float kf = __bfloat162float(kval);
          const_cast<bf16*>(a.k_cache)[dst * kHeadDim + c] = kval;
          const_cast<bf16*>(a.kmin)[si] = (fresh || kf < __bfloat162float(omin)) ? kval : omin;
          const_cast<bf16*>(a.kmax)[si] = (fresh || kf > __bfloat162float(omax)) ? kval : omax;
        } else {
          const_cast<bf16*>(a.v_cache)[dst * kHeadDim + c] = a.ap.new_v[src];
          if constexpr (MODE == 1) {
            if (c == 0) const_cast<int32_t*>(a.kept)[(size_t)ukv * vcap + len] = row;
          }
        }
        appended = true;
      } else if (tid == 0) {
        set_status(a.status, RKV_DEV_LEN_OVER_CAP);
      }
      __syncthreads();  // the new row and summary are visible to this CTA's reads below
      if (fits) {
        ++len;
        if constexpr (MODE == 1) flen = row + 1;
      }
    }
  }
  const int p = a.page;
  const int P = (len + p - 1) / p;
  const int S = (a.budget / 2) / p;
  const bool dense = len <= a.budget;
  const size_t cache_base = (size_t)ukv * a.cap;
  if (len <= 0 || len > vcap || P > a.page_cap) {
    if (tid == 0 && len != 0) set_status(a.status, RKV_DEV_LEN_OVER_CAP);
    if constexpr (MODE != 0) {
      if (appended && tid == 0 && atomicAdd(&a.ap.acount[u], 1) == a.n_kv - 1) {
        a.ap.acount[u] = 0;
        const_cast<int32_t*>(a.len)[u] = len0 + 1;
        if constexpr (MODE == 1) const_cast<int32_t*>(a.full_len)[u] = arow + 1;
      }
    }
    return;
  }

  // ---- group sums: |q| for the channel pick, signed q for the score --------------------
  if (tid < kHeadDim) {
    float s = 0.f, t = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      s += fabsf(qv[h]);
      t += qv[h];
    }
    ukey[tid] = ordered_key(s);
    qg[tid] = t;
  }
  __syncthreads();

  int nsel;
  if (!dense) {
    // ---- channel pick: top-c of sum_h |q_h| (ties -> lower channel), ascending -----------
    // Threads c and c + 128 rank channel c against channels 0..63 and 64..127 by the unique
    // order (key desc, channel asc); the ranks are a permutation, so exactly the channels of
    // rank < cn are taken, placed in channel order by the ballots of warps 0..3.
    const int cn = a.channels;
    {
      const int c = tid & (kHeadDim - 1), half = tid >> 7;
      const uint32_t mk = ukey[c];
      const uint4* k4 = reinterpret_cast<const uint4*>(ukey + 64 * half);
      int r = 0;
#pragma unroll 4
      for (int j4 = 0; j4 < 16; ++j4) {
        const uint4 x = k4[j4];
        const int j = 64 * half + 4 * j4;
        r += (x.x > mk || (x.x == mk && j < c)) ? 1 : 0;
        r += (x.y > mk || (x.y == mk && j + 1 < c)) ? 1 : 0;
        r += (x.z > mk || (x.z == mk && j + 2 < c)) ? 1 : 0;
        r += (x.w > mk || (x.w == mk && j + 3 < c)) ? 1 : 0;
      }
      if (half) part_rank[c] = r;
      __syncthreads();
      if (!half) {
        const bool take = r + part_rank[c] < cn;
        const uint32_t bt = __ballot_sync(0xffffffffu, take);
        if (lane == 0) wcnt[warp] = __popc(bt);
        group_sync(0);  // warps 0..3
        int before = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) before += (w < warp) ? wcnt[w] : 0;
        if (take) chosen[before + __popc(bt & ((1u << lane) - 1u))] = c;
      } else if (warp == 7) {
        MmaAttn<G>::build_fragments(qgroup, qfrag);
      }
    }
    __syncthreads();
    if (a.sel_channels && tid < cn) a.sel_channels[(size_t)ukv * cn + tid] = chosen[tid];

    // ---- approximate page scores -------------------------------------------------------
    // score[pg] = sum_i w_i R_i[pg] with w_i = q_g of kept channel i and R_i its summary row
    // (Kmax where q_g >= 0, else Kmin): a vector-matrix product over the kept rows, bound by
    // HBM, so plain fp32 FMAs on rows read straight from global memory (nothing staged).
    // Thread pair (2p, 2p + 1) takes the 8-page groups p, p + 128, ... (16 bytes of a row) over
    // the even / odd kept channels; one shuffle joins the pair's partial sums, and thread
    // 2p + h keeps pages 4h .. 4h + 3 of the group, so thread t holds pages 1024 r + 4 t + e.
    // The same pass records the range of the scores' ordered keys for the select.
    {
      const int h = tid & 1, pr = tid >> 1;
      const int ngroups = (P + 7) >> 3;
      const size_t rowbase = (size_t)ukv * kHeadDim;
      float* approx_row = a.approx ? a.approx + (size_t)ukv * a.page_cap : nullptr;
      uint32_t khi = 0u, klo = 0xffffffffu;
      if (wide) {
        // one round of 16-byte copies brings every kept row into shared memory (row i at
        // stages + i * page_cap); the GEMV below then reads 16 bytes per (row, 8-page group).
        // The rows' addresses are looked up once into shared memory, so that every thread
        // issues its copies back to back.
        const bf16** rowp = reinterpret_cast<const bf16**>(
            smem + region + 2 * align_up((size_t)a.page_cap * 4, 16));
        if (tid < cn) {
          const int c = chosen[tid] & (kHeadDim - 1);
          rowp[tid] = ((qg[c] >= 0.f) ? a.kmax : a.kmin) + (rowbase + c) * a.page_cap;
        }
        __syncthreads();
        for (int cc = tid; cc < ngroups; cc += kDecodeThreads) {
#pragma unroll 8
          for (int i = 0; i < cn; ++i)
            cp_async16(stages + (size_t)i * a.page_cap + cc * 8, rowp[i] + cc * 8);
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
      }
      for (int gb = 0; gb < ngroups; gb += kDecodeThreads / 2) {
        const int gi = gb + pr;
        const bool valid = gi < ngroups;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        if (valid && !wide) {
          const size_t col = (size_t)gi * 8;
#pragma unroll 16
          for (int i = h; i < cn; i += 2) {
            const int c = chosen[i] & (kHeadDim - 1);
            const float w = qg[c];
            const bf16* row = ((w >= 0.f) ? a.kmax : a.kmin) + (rowbase + c) * a.page_cap;
            // (the append variants may have written these rows in this launch: no
            // non-coherent loads there)
            const uint4 x = (MODE == 0) ? __ldg(reinterpret_cast<const uint4*>(row + col))
                                        : __ldcg(reinterpret_cast<const uint4*>(row + col));
            float f[8];
            unpack8(x, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(w, f[e], acc[e]);
          }
        } else if (valid) {
          const bf16* srow = stages + (size_t)gi * 8;
#pragma unroll 8
          for (int i = h; i < cn; i += 2) {
            const float w = qg[chosen[i] & (kHeadDim - 1)];
            const uint4 x = *reinterpret_cast<const uint4*>(srow + (size_t)i * a.page_cap);
            float f[8];
            unpack8(x, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(w, f[e], acc[e]);
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 1);
        if (valid) {
          // both threads of the pair hold the 8 sums; thread h publishes pages 4h .. 4h + 3
          const int p0 = gi * 8 + 4 * h;
          const float4 o = h ? make_float4(acc[4], acc[5], acc[6], acc[7])
                             : make_float4(acc[0], acc[1], acc[2], acc[3]);
          *reinterpret_cast<float4*>(scores + p0) = o;
          const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (p0 + e < P) {
              const uint32_t kk = ordered_key(ov[e]);
              khi = max(khi, kk);
              klo = min(klo, kk);
              if (approx_row) approx_row[p0 + e] = ov[e];
            }
          }
        }
      }
      bin_select_prepare(khi, klo, bsel);
      __syncthreads();
    }

    // ---- page top-k ----------------------------------------------------------------------
    if (S >= P) {
      for (int i = tid; i < P; i += kDecodeThreads) sel[i] = i;
      nsel = P;
    } else {
      bool done;
      if (P <= 1024)
        done = bin_topk<1>(scores, P, S, sel, bsel);
      else if (P <= 2048)
        done = bin_topk<2>(scores, P, S, sel, bsel);
      else if (P <= 3072)
        done = bin_topk<3>(scores, P, S, sel, bsel);
      else if (P <= 4096)
        done = bin_topk<4>(scores, P, S, sel, bsel);
      else
        done = false;
      if (!done) {
        // general select over the scores in shared memory (a range that is not a finite
        // positive number, a crowded k-th bin, or more than 4096 pages)
        if (tid < 8) {
          sel_smem.fast.wmax[tid] = bsel.wmax[tid];
          sel_smem.fast.wmin[tid] = bsel.wmin[tid];
        }
        fast_select_clear(sel_smem.fast);
        __syncthreads();
        int got;
        if (P <= 1024)
          got = block_topk_1024(scores, P, S, sel, sel_smem.fast);
        else if (P <= 2048)
          got = block_topk_fast<8>(scores, P, S, sel, sel_smem.fast);
        else if (P <= 4096)
          got = block_topk_fast<16>(scores, P, S, sel, sel_smem.fast);
        else
          got = block_topk_ascending(scores, P, S, sel, sel_smem.generic);
        if (got != S && tid == 0) set_status(a.status, RKV_DEV_SELECT_FAILED);
      }
      nsel = S;
    }
  } else {
    if (warp == 7) MmaAttn<G>::build_fragments(qgroup, qfrag);
    if (a.sel_channels && tid < a.channels) a.sel_channels[(size_t)ukv * a.channels + tid] = -1;
    for (int i = tid; i < P; i += kDecodeThreads) sel[i] = i;
    nsel = P;
  }
  __syncthreads();
  if (a.sel_pages) {
    for (int i = tid; i < S; i += kDecodeThreads)
      a.sel_pages[(size_t)ukv * S + i] = (!dense && i < nsel) ? sel[i] : -1;
  }

  // ---- exact attention over the selected pages -------------------------------------------
  // The selected pages' tokens, in page order, are cut into 16-token units; warp w takes units
  // w, w + 8, ...: it stages up to `upw` of them at a time (one in the ordinary layout, all of
  // its units in the wide one) with 16-byte cp.async into its own area (rows kRowPad apart),
  // waits for its own copies only, and runs one MMA step per unit.
  const int lp = __ffs(p) - 1;  // log2(page)
  const int ntok_all = (nsel - 1) * p + min(p, len - sel[nsel - 1] * p);
  const int nunits = (ntok_all + 15) >> 4;
  const size_t wstride = (size_t)upw * (2 * 16 * kRowPad);  // one warp's area (bf16)
  bf16* warea = stages + (size_t)warp * wstride;
  MmaAttn<G> at;
  at.init(qfrag);
  for (int t0 = warp; t0 < nunits; t0 += 8 * upw) {
    for (int j = 0; j < upw && t0 + 8 * j < nunits; ++j) {
      const int t = t0 + 8 * j;
      bf16* Kw = warea + (size_t)j * (2 * 16 * kRowPad);
      bf16* Vw = Kw + 16 * kRowPad;
      const int v0 = t * 16;
      const int nt = min(16, ntok_all - v0);
      // lanes 0..15 copy a K row, lanes 16..31 the V row of the same token, 16 bytes each
      const int half = (lane >> 4) & 1, c16 = lane & 15;
      const bf16* cache = half ? a.v_cache : a.k_cache;
      bf16* dst = (half ? Vw : Kw) + c16 * 8;
      if constexpr (MODE == 2) {
        // lane r looks up (and checks) the block of the unit's token r in the page table
        int kblk = 0;
        if (lane < nt) {
          const int v = v0 + lane;
          kblk = paged_block(a.pm, u, (sel[v >> lp] << lp) + (v & (p - 1)), a.status);
        }
        for (int r = 0; r < nt; ++r) {
          const int v = v0 + r;
          const int blk = __shfl_sync(0xffffffffu, kblk, r);
          const size_t row =
              paged_row(a.pm, blk, a.n_kv, g, (sel[v >> lp] << lp) + (v & (p - 1)));
          cp_async16(dst + r * kRowPad, cache + row * kHeadDim + c16 * 8);
        }
      } else if constexpr (MODE == 1) {
        // lane r fetches the cache row of the unit's token r from the kept list, checked
        int krow = 0;
        if (lane < nt) {
          const int v = v0 + lane;
          const int tk = (sel[v >> lp] << lp) + (v & (p - 1));
          krow = a.kept[(size_t)ukv * vcap + tk];
          if (krow < 0 || krow >= flen) {
            set_status(a.status, RKV_DEV_BAD_INDEX);
            krow = 0;
          }
        }
        for (int r = 0; r < nt; ++r) {
          const size_t tok = (size_t)__shfl_sync(0xffffffffu, krow, r);
          cp_async16(dst + r * kRowPad, cache + (cache_base + tok) * kHeadDim + c16 * 8);
        }
      } else {
        for (int r = 0; r < nt; ++r) {
          const int v = v0 + r;
          const size_t tok = ((size_t)sel[v >> lp] << lp) + (v & (p - 1));
          cp_async16(dst + r * kRowPad, cache + (cache_base + tok) * kHeadDim + c16 * 8);
        }
      }
      // V rows past the unit's tokens meet P = 0: make them zero, not stale bits (0 * NaN)
      for (int i = lane; i < (16 - nt) * 16; i += 32)
        *reinterpret_cast<uint4*>(Vw + (nt + (i >> 4)) * kRowPad + (i & 15) * 8) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncwarp();
    for (int j = 0; j < upw && t0 + 8 * j < nunits; ++j) {
      const bf16* Kw = warea + (size_t)j * (2 * 16 * kRowPad);
      at.step16(Kw, Kw + 16 * kRowPad, 0, min(16, ntok_all - (t0 + 8 * j) * 16), a.scale_log2);
    }
    __syncwarp();  // the next batch refills this warp's rows
  }
  __syncwarp();
  warp_deposit_own<G>(at, warp_state<G>(stages, warp, wstride));
  __syncthreads();
  // output pair (h, c): merge the 8 warps' partial states, each thread forming head h's factors
  for (int i = tid; i < G * kHeadDim / 2; i += kDecodeThreads) {
    const int h = i >> 6, c = (i & 63) * 2;
    float mw[8];
    float mm = -1e30f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      mw[w] = warp_state<G>(stages, w, wstride)[h];
      mm = fmaxf(mm, mw[w]);
    }
    float ll = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float* st = warp_state<G>(stages, w, wstride);
      const float f = fast_exp2(mw[w] - mm);
      const float2 x = *reinterpret_cast<const float2*>(st + 2 * G + h * kORow + c);
      ll = fmaf(st[G + h], f, ll);
      o0 = fmaf(f, x.x, o0);
      o1 = fmaf(f, x.y, o1);
    }
    const float inv = ll > 0.f ? 1.f / ll : 0.f;
    *reinterpret_cast<uint32_t*>(a.out + ((size_t)u * hq + g * G + h) * kHeadDim + c) =
        pack_bf16x2(o0 * inv, o1 * inv);
  }
  if constexpr (MODE != 0) {
    if (appended && tid == 0 && atomicAdd(&a.ap.acount[u], 1) == a.n_kv - 1) {
      a.ap.acount[u] = 0;
      const_cast<int32_t*>(a.len)[u] = len0 + 1;
      if constexpr (MODE == 1) const_cast<int32_t*>(a.full_len)[u] = arow + 1;
    }
  }
}

// Launch with programmatic stream serialisation (the kernel calls pdl_wait() before its first
// global read, so it is correct after any kind of predecessor).
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
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

// Layout policy of the hybrid decode (rkv_testing_decode_layout); 0: automatic.
static std::atomic<int> g_decode_layout{0};
int set_decode_layout(int layout) {
  if (layout < 0 || layout > 2) return -1;
  g_decode_layout.store(layout);
  return 0;
}

size_t hybrid_counter_bytes(int n) { return align_up((size_t)(n > 0 ? n : 0) * 4, 256); }

cudaError_t launch_hybrid(const HybridArgsAll& a, cudaStream_t s) {
  const HybridArgs& plain = a;
  const HybridArgsMT& mt = a;
  HybridArgsPaged pg;
  static_cast<HybridArgs&>(pg) = plain;
  pg.pm = a.pm;
  pg.ap = a.ap;
  HybridArgsApp app;
  static_cast<HybridArgs&>(app) = plain;
  app.ap = a.ap;
  // one CTA per (unit, KV head); the wide layout when they all fit one per SM (or as the test
  // hook asks: 1 never, 2 wherever it fits)
  const int layout = g_decode_layout.load();
  const size_t wbytes = wide_smem_bytes(a.channels, a.page_cap, a.budget);
  const bool wide = wbytes != 0 && layout != 1 &&
                    (layout == 2 || (long long)a.n * a.n_kv <= device_sm_count());
  const size_t smem = wide ? wbytes : hybrid_smem_bytes(a.gqa, a.page_cap, a.budget, a.page);
  const dim3 grid(a.n * a.n_kv), block(kDecodeThreads);
  cudaError_t e = cudaSuccess;
  switch (a.gqa) {
#define RKV_CASE(GG)                                                                         \
  case GG:                                                                                   \
    if (a.pm.table) {                                                                        \
      auto* k = hybrid_decode_kernel<GG, 2, HybridArgsPaged>;                                \
      e = ensure_dyn_smem((const void*)k, smem);                                             \
      if (e != cudaSuccess) return e;                                                        \
      e = launch_pdl(k, grid, block, smem, s, pg);                                           \
    } else if (a.kept) {                                                                     \
      auto* k = hybrid_decode_kernel<GG, 1, HybridArgsMT>;                                   \
      e = ensure_dyn_smem((const void*)k, smem);                                             \
      if (e != cudaSuccess) return e;                                                        \
      e = launch_pdl(k, grid, block, smem, s, mt);                                           \
    } else if (a.ap.new_k) {                                                                 \
      auto* k = hybrid_decode_kernel<GG, 3, HybridArgsApp>;                                  \
      e = ensure_dyn_smem((const void*)k, smem);                                             \
      if (e != cudaSuccess) return e;                                                        \
      e = launch_pdl(k, grid, block, smem, s, app);                                          \
    } else {                                                                                 \
      auto* k = hybrid_decode_kernel<GG, 0, HybridArgs>;                                     \
      e = ensure_dyn_smem((const void*)k, smem);                                             \
      if (e != cudaSuccess) return e;                                                        \
      e = launch_pdl(k, grid, block, smem, s, plain);                                        \
    }                                                                                        \
    if (e != cudaSuccess) return e;                                                          \
    break;
    RKV_CASE(1)
    RKV_CASE(2)
    RKV_CASE(4)
    RKV_CASE(8)
#undef RKV_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}


// ==========================================================================================
// Page summaries: CTA = (unit, KV head) x 32 pages. Reads rows coalesced (16 threads per
// 256-byte row, 16 bytes each), reduces with exact bf16 min / max, transposes through shared
// memory and writes channel rows 8 pages (16 bytes) at a time. Rows come from the cache, a kept
// list (RocketKV-MT) or a paged pool.
// ==========================================================================================
constexpr int kSumPages = 32;

// CTA = (unit, 32 pages). Thread t takes the 16-byte channel chunk t % 16 of pages t / 16 and
// t / 16 + 16: its 2 PG row loads are all issued before any is used. Per-page (min, max) go
// through shared memory so that each channel row of Kmin / Kmax is written 8 pages (16 bytes)
// at a time.
template <int PG>
__global__ void __launch_bounds__(256) summaries_kernel(SummaryArgs a) {
  __shared__ __align__(16) uint4 smin[kSumPages][kHeadDim / 8];
  __shared__ __align__(16) uint4 smax[kSumPages][kHeadDim / 8];
  const int ukv = blockIdx.x;
  const int u = ukv / a.n_kv;
  const int len = a.len[u];
  const int P = (len + PG - 1) / PG;
  if (len < 0 || len > a.vcap || P > a.page_cap) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_status(a.status, RKV_DEV_LEN_OVER_CAP);
    return;
  }
  const int pg0 = blockIdx.y * kSumPages;
  const int first_page = a.first_token / PG;
  if (pg0 >= P || pg0 + kSumPages <= first_page) return;
  const int c = threadIdx.x & 15, pl = threadIdx.x >> 4;
  const bool paged = a.pm.table != nullptr;
  const int g = ukv - u * a.n_kv;
  const uint4* kc = reinterpret_cast<const uint4*>(
      paged ? a.k_cache : a.k_cache + (size_t)ukv * a.cap * kHeadDim);
  const int32_t* kept = a.kept ? a.kept + (size_t)ukv * a.vcap : nullptr;
  // row (from kc) of sequence token t: itself, its kept index or its page's row (checked; row 0
  // of the unit, or block 0, if out of range)
  auto row_of = [&](int t) -> size_t {
    if (paged) return paged_row(a.pm, paged_block(a.pm, u, t, a.status), a.n_kv, g, t);
    if (!kept) return (size_t)t;
    const int r = kept[t];
    if (r < 0 || r >= a.cap) {
      set_status(a.status, RKV_DEV_BAD_INDEX);
      return 0;
    }
    return (size_t)r;
  };
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = pl + 16 * h;
    const int t0 = (pg0 + j) * PG;
    const int nt = min(PG, len - t0);  // rows of this page (<= 0: past the end)
    if (nt > 0) {
      const __nv_bfloat162 pinf = __halves2bfloat162(__ushort_as_bfloat16(0x7F80),
                                                     __ushort_as_bfloat16(0x7F80));
      const __nv_bfloat162 ninf = __halves2bfloat162(__ushort_as_bfloat16(0xFF80),
                                                     __ushort_as_bfloat16(0xFF80));
      __nv_bfloat162 mn[4] = {pinf, pinf, pinf, pinf}, mx[4] = {ninf, ninf, ninf, ninf};
      constexpr int kB = PG < 8 ? PG : 8;  // rows in flight per batch
#pragma unroll
      for (int r0 = 0; r0 < PG; r0 += kB) {
        uint4 x[kB];
        size_t rw[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) rw[b] = (r0 + b < nt) ? row_of(t0 + r0 + b) : 0;
#pragma unroll
        for (int b = 0; b < kB; ++b)
          if (r0 + b < nt) x[b] = kc[rw[b] * (kHeadDim / 8) + c];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          if (r0 + b < nt) {
            const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&x[b]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              mn[e] = __hmin2(mn[e], y[e]);
              mx[e] = __hmax2(mx[e], y[e]);
            }
          }
        }
      }
      smin[j][c] = *reinterpret_cast<const uint4*>(mn);
      smax[j][c] = *reinterpret_cast<const uint4*>(mx);
    }
  }
  __syncthreads();
  // write: thread -> (channel ch, 8-page group), pages [pg0, pg0 + 32) of channel row ch
  const int npg = min(kSumPages, P - pg0);
  const int first_j = max(0, first_page - pg0);
  const uint16_t* smin16 = reinterpret_cast<const uint16_t*>(&smin[0][0]);
  const uint16_t* smax16 = reinterpret_cast<const uint16_t*>(&smax[0][0]);
  uint16_t* kmin16 = reinterpret_cast<uint16_t*>(a.kmin);
  uint16_t* kmax16 = reinterpret_cast<uint16_t*>(a.kmax);
  for (int i = threadIdx.x; i < kHeadDim * (kSumPages / 8); i += blockDim.x) {
    const int ch = i >> 2, j0 = (i & 3) * 8;
    if (j0 >= npg) continue;
    const size_t row = ((size_t)ukv * kHeadDim + ch) * a.page_cap + pg0 + j0;
    uint16_t vmin[8], vmax[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int j = min(j0 + t, npg - 1);
      vmin[t] = smin16[j * kHeadDim + ch];
      vmax[t] = smax16[j * kHeadDim + ch];
    }
    if (j0 + 8 <= npg && j0 >= first_j) {
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
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int j = j0 + t;
        if (j < npg && j >= first_j) {
          kmin16[row + t] = vmin[t];
          kmax16[row + t] = vmax[t];
        }
      }
    }
  }
}

cudaError_t launch_summaries(const SummaryArgs& a, cudaStream_t s) {
  const dim3 grid(a.n * a.n_kv, (a.page_cap + kSumPages - 1) / kSumPages);
  switch (a.page) {
#define RKV_SUM(PGV)                                    \
  case PGV:                                             \
    summaries_kernel<PGV><<<grid, 256, 0, s>>>(a);      \
    break;
    RKV_SUM(1)
    RKV_SUM(2)
    RKV_SUM(4)
    RKV_SUM(8)
    RKV_SUM(16)
    RKV_SUM(32)
    RKV_SUM(64)
#undef RKV_SUM
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ==========================================================================================
// Dense decode (flash-decoding split-K): CTA = (unit, KV head, split). Each split's tokens are
// staged 64 rows at a time (16-byte cp.async copies, two warp groups with one stage each) and
// consumed by the same MMA warp code;
// per-split partials are merged by a second kernel.
// ==========================================================================================
void dense_plan(int n, int n_kv, int max_len, int* nsplit, int* tokens_per_split) {
  const long long units = (long long)n * n_kv;
  const long long target_ctas = 4LL * device_sm_count();  // two waves of two CTAs per SM
  int ns = (int)((target_ctas + units - 1) / units);
  const int max_ns = (max_len + 255) / 256;  // at least 256 tokens per split
  ns = ns < 1 ? 1 : (ns > max_ns ? max_ns : ns);
  int tps = (max_len + ns - 1) / ns;
  tps = (tps + kChunkTokens - 1) / kChunkTokens * kChunkTokens;
  ns = (max_len + tps - 1) / tps;
  *nsplit = ns;
  *tokens_per_split = tps;
}

size_t dense_partials_bytes(int n, int n_kv, int gqa, int max_len) {
  int ns, tps;
  dense_plan(n, n_kv, max_len, &ns, &tps);
  const size_t rows = (size_t)n * n_kv * gqa * ns;
  return align_up(rows * 4, 256) * 2 + align_up(rows * kHeadDim * 4, 256);
}

template <int G>
__global__ void __launch_bounds__(kDecodeThreads, 2) dense_split_kernel(DenseArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint2 qfrag[8 * 32];
  bf16* stages = reinterpret_cast<bf16*>(smem);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int ukv = blockIdx.x, split = blockIdx.y;
  const int u = ukv / a.n_kv, g = ukv - u * a.n_kv;
  const int hq = a.n_kv * G;
  int len = a.len[u];
  if (len > a.max_len) {
    if (tid == 0 && split == 0) set_status(a.status, RKV_DEV_LEN_OVER_CAP);
    len = a.max_len;
  }
  const int tb = split * a.tokens_per_split;
  const int te = min(len, tb + a.tokens_per_split);
  const int ntok_all = max(0, te - tb);
  const int nchunks = (ntok_all + kChunkTokens - 1) / kChunkTokens;
  const size_t base = ((size_t)ukv * a.max_len + tb) * kHeadDim;
  const bf16* qgroup = a.q + ((size_t)u * hq + g * G) * kHeadDim;
  const int wg = warp >> 2, wig = warp & 3, gtid = tid & 127;

  if (warp == 7) MmaAttn<G>::build_fragments(qgroup, qfrag);

  auto chunk_tokens = [&](int c) { return min(kChunkTokens, ntok_all - c * kChunkTokens); };
  // the 128 threads of a group stage one chunk of contiguous rows with 16-byte cp.async copies
  auto load = [&](int c) {
    bf16* Ks = stages + (size_t)wg * kStageElems;
    const int nt = chunk_tokens(c);
    const size_t row0 = base + (size_t)c * kChunkTokens * kHeadDim;
    for (int idx = gtid; idx < nt * 32; idx += 128) {
      const int r = idx >> 5, tv = (idx >> 4) & 1, c16 = idx & 15;
      const bf16* src = (tv ? a.v : a.k) + row0 + (size_t)r * kHeadDim + c16 * 8;
      cp_async16(Ks + tv * (kChunkTokens * kRowPad) + r * kRowPad + c16 * 8, src);
    }
    cp_async_commit();
  };
  if (wg < nchunks) load(wg);
  __syncthreads();  // Q fragments ready

  MmaAttn<G> at;
  at.init(qfrag);
  for (int c = wg; c < nchunks; c += 2) {
    cp_async_wait_all();
    group_sync(wg);
    const bf16* Ks = stages + (size_t)wg * kStageElems;
    bf16* Vs = stages + (size_t)wg * kStageElems + kChunkTokens * kRowPad;
    const int nt = chunk_tokens(c);
    if (nt < kChunkTokens) {
      zero_tail_rows(Vs, nt, gtid);
      group_sync(wg);
    }
    if (wig * 16 < nt) at.step16(Ks, Vs, wig * 16, nt, a.scale_log2);
    group_sync(wg);
    if (c + 2 < nchunks) load(c + 2);
  }
  __syncthreads();

  CombineSmem<G>* cs = reinterpret_cast<CombineSmem<G>*>(smem);
  warp_deposit<G>(at, cs);
  __syncthreads();
  for (int i = tid; i < G * kHeadDim; i += kDecodeThreads) {
    const int h = i >> 7, c = i & 127;
    float M, L, O;
    warp_merge<G>(cs, h, c, &M, &L, &O);
    const size_t row = ((size_t)u * hq + g * G + h) * a.nsplit + split;
    a.part_o[row * kHeadDim + c] = O;
    if (c == 0) {
      a.part_m[row] = M;
      a.part_l[row] = L;
    }
  }
}

__global__ void dense_combine_kernel(DenseArgs a) {
  const int row = blockIdx.x;  // (u, h)
  const int c = threadIdx.x;   // 128 channels
  const float* pm = a.part_m + (size_t)row * a.nsplit;
  const float* pl = a.part_l + (size_t)row * a.nsplit;
  const float* po = a.part_o + (size_t)row * a.nsplit * kHeadDim;
  float M = -1e30f;
  for (int s = 0; s < a.nsplit; ++s) M = fmaxf(M, pm[s]);
  float L = 0.f, O = 0.f;
  for (int s = 0; s < a.nsplit; ++s) {
    const float f = fast_exp2(pm[s] - M);
    L = fmaf(pl[s], f, L);
    O = fmaf(po[(size_t)s * kHeadDim + c], f, O);
  }
  a.out[(size_t)row * kHeadDim + c] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
}

cudaError_t launch_dense(const DenseArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)kDecStages * kStageBytes;
  const dim3 grid(a.n * a.n_kv, a.nsplit), block(kDecodeThreads);
  cudaError_t e = cudaSuccess;
  switch (a.gqa) {
#define RKV_CASE(GG)                                                                         \
  case GG:                                                                                   \
    e = ensure_dyn_smem((const void*)dense_split_kernel<GG>, smem);                          \
    if (e != cudaSuccess) return e;                                                          \
    dense_split_kernel<GG><<<grid, block, smem, s>>>(a);                                     \
    break;
    RKV_CASE(1)
    RKV_CASE(2)
    RKV_CASE(4)
    RKV_CASE(8)
#undef RKV_CASE
    default:
      return cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dense_combine_kernel<<<a.n * a.n_kv * a.gqa, kHeadDim, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace rkv
