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
// Memory movement: K/V rows of the selected pages are staged in shared memory by
// cp.async.bulk (one copy per page and tensor, completion on an mbarrier, kStages stages in
// flight); summary rows are read with 16-byte vector loads, 8 pages per load.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "rkv_internal.h"

namespace rkv {

// ==========================================================================================
// Warp-level online-softmax attention over rows staged in shared memory.
//
// Lane layout for q.k: lane = 8 * ts + e; ts (0..3) picks one of 4 tokens, e (0..7) owns 16
// channels [16e, 16e + 16) as two 16-byte chunks. Lanes e >= 4 read their two chunks in swapped
// order so that every quarter-warp touches 8 distinct 16-byte bank groups (conflict-free).
// Lane layout for p.v: lane owns output channels [4 * lane, 4 * lane + 4).
// Scores live in the log2 domain (q is pre-scaled by scale * log2(e)).
// ==========================================================================================
template <int G>
struct WarpAttn {
  float m[G];
  float l[G];
  float acc[G][4];
  float qr[G][16];
  int lane, ts, e, sw;

  __device__ __forceinline__ void init(const float* qs /* [G][128], scaled */) {
    lane = threadIdx.x & 31;
    ts = lane >> 3;
    e = lane & 7;
    sw = (e >> 2) & 1;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -1e30f;
      l[h] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[h][j] = 0.f;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int i = 0; i < 8; ++i) qr[h][jj * 8 + i] = qs[h * 128 + 16 * e + 8 * (jj ^ sw) + i];
    }
  }

  // Tokens t0 .. t0+3 of a stage holding `ntok` valid rows.
  __device__ __forceinline__ void step4(const bf16* Ks, const bf16* Vs, int t0, int ntok) {
    const int tk = t0 + ts;
    const bool valid = tk < ntok;
    float dot[G];
#pragma unroll
    for (int h = 0; h < G; ++h) dot[h] = 0.f;
    if (valid) {
      const uint4* row = reinterpret_cast<const uint4*>(Ks + tk * kHeadDim);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint4 c = row[2 * e + (jj ^ sw)];
        float f[8];
        unpack8(c, f);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int i = 0; i < 8; ++i) dot[h] = fmaf(qr[h][jj * 8 + i], f[i], dot[h]);
      }
    }
    float p[G], alpha[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float d = dot[h];
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      d += __shfl_xor_sync(0xffffffffu, d, 4);
      const float s = valid ? d : -INFINITY;
      float mt = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 8));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
      const float mn = fmaxf(m[h], mt);
      alpha[h] = exp2f(m[h] - mn);
      p[h] = exp2f(s - mn);
      m[h] = mn;
      l[h] = l[h] * alpha[h] + p[h];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[h][j] *= alpha[h];
    }
#pragma unroll
    for (int uu = 0; uu < 4; ++uu) {
      if (t0 + uu < ntok) {
        const uint2 vv =
            *reinterpret_cast<const uint2*>(Vs + (t0 + uu) * kHeadDim + 4 * lane);
        const float vf[4] = {bf16_lo(vv.x), bf16_hi(vv.x), bf16_lo(vv.y), bf16_hi(vv.y)};
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pu = __shfl_sync(0xffffffffu, p[h], uu * 8);
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[h][j] = fmaf(pu, vf[j], acc[h][j]);
        }
      }
    }
  }

  // Sum of l over the 4 token slots (every e-class ends up with the full sum).
  __device__ __forceinline__ float total_l(int h) const {
    float t = l[h];
    t += __shfl_xor_sync(0xffffffffu, t, 8);
    t += __shfl_xor_sync(0xffffffffu, t, 16);
    return t;
  }
};

// Shared-memory layout of the warp-combine step (re-uses the stage buffers).
template <int G>
struct CombineSmem {
  float m[8][G];
  float l[8][G];
  float o[8][G][kHeadDim];
};

// Each warp deposits its state; afterwards thread i < G*128 owns (h, c) = (i / 128, i % 128).
template <int G>
__device__ __forceinline__ void warp_deposit(const WarpAttn<G>& wa, CombineSmem<G>* cs) {
  const int w = threadIdx.x >> 5;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float lt = wa.total_l(h);
    if (wa.lane == 0) {
      cs->m[w][h] = wa.m[h];
      cs->l[w][h] = lt;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) cs->o[w][h][4 * wa.lane + j] = wa.acc[h][j];
  }
}

// Merge the 8 warps for (h, c): returns unnormalised output relative to max M, with L.
template <int G>
__device__ __forceinline__ void warp_merge(const CombineSmem<G>* cs, int h, int c, float* M,
                                           float* L, float* O) {
  float mm = -1e30f;
#pragma unroll
  for (int w = 0; w < 8; ++w) mm = fmaxf(mm, cs->m[w][h]);
  float ll = 0.f, oo = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float f = exp2f(cs->m[w][h] - mm);
    ll = fmaf(cs->l[w][h], f, ll);
    oo = fmaf(cs->o[w][h][c], f, oo);
  }
  *M = mm;
  *L = ll;
  *O = oo;
}

// ==========================================================================================
// Hybrid sparse decode: one CTA per (unit, KV head).
// ==========================================================================================
constexpr int kStageBytes = 2 * kChunkTokens * kHeadDim * 2;  // K + V rows of one stage

size_t hybrid_smem_bytes(int gqa, int page_cap, int budget, int page) {
  const int nsel_max = page_cap;  // selected-page list (dense path may select every page)
  size_t b = (size_t)kStages * kStageBytes;   // stages (re-used by the warp combine)
  b += align_up((size_t)page_cap * 4, 16);    // approximate scores
  b += align_up((size_t)nsel_max * 4, 16);    // selected pages
  (void)gqa;
  (void)budget;
  (void)page;
  return b;
}

template <int G>
__global__ void __launch_bounds__(kDecodeThreads, 2) hybrid_decode_kernel(HybridArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ float qs[G * kHeadDim];
  __shared__ float mag[kHeadDim];
  __shared__ float qg[kHeadDim];
  __shared__ int chosen[kHeadDim];
  __shared__ uint32_t ballots[4];
  __shared__ __align__(8) uint64_t bars[kStages];
  __shared__ SelectScratch sc;

  bf16* stages = reinterpret_cast<bf16*>(smem);
  float* scores = reinterpret_cast<float*>(smem + (size_t)kStages * kStageBytes);
  int* sel = reinterpret_cast<int*>(smem + (size_t)kStages * kStageBytes +
                                    align_up((size_t)a.page_cap * 4, 16));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ukv = blockIdx.x;
  const int u = ukv / a.n_kv;
  const int g = ukv - u * a.n_kv;
  const int hq = a.n_kv * G;
  const int len = a.len[u];
  const int p = a.page;
  const int P = (len + p - 1) / p;
  const int S = (a.budget / 2) / p;
  const bool dense = len <= a.budget;

  if (len <= 0 || len > a.cap || P > a.page_cap) {
    if (tid == 0 && len != 0) set_status(a.status, RKV_DEV_LEN_OVER_CAP);
    return;
  }

  // ---- q: raw values to shared memory -------------------------------------------------
  if (tid < G * 16) {
    const int h = tid >> 4, c8 = (tid & 15) * 8;
    const uint4 c = *reinterpret_cast<const uint4*>(
        a.q + ((size_t)u * hq + g * G + h) * kHeadDim + c8);
    float f[8];
    unpack8(c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) qs[h * kHeadDim + c8 + i] = f[i];
  }
  if (tid < kStages) mbar_init(&bars[tid], 1);
  fence_barrier_init();
  __syncthreads();

  // ---- group sums: |q| for the channel pick, signed q for the score --------------------
  if (tid < kHeadDim) {
    float s = 0.f, t = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float x = qs[h * kHeadDim + tid];
      s += fabsf(x);
      t += x;
    }
    mag[tid] = s;
    qg[tid] = t;
  }
  __syncthreads();

  int nsel;
  if (!dense) {
    // ---- channel pick: rank every channel (ties -> lower channel) ----------------------
    bool pick = false;
    if (tid < kHeadDim) {
      const float mine = mag[tid];
      int rank = 0;
      for (int j = 0; j < kHeadDim; ++j) {
        const float o = mag[j];
        rank += (o > mine) || (o == mine && j < tid);
      }
      pick = rank < a.channels;
    }
    const uint32_t picked = __ballot_sync(0xffffffffu, pick);
    if (lane == 0 && warp < 4) ballots[warp] = picked;
    __syncthreads();  // every warp's ballot is visible before any position is computed
    if (pick) {
      int pos = __popc(picked & ((1u << lane) - 1u));
      for (int w = 0; w < warp; ++w) pos += __popc(ballots[w]);
      chosen[pos] = tid;
    }
    if (tid == 0) {
      const int total = __popc(ballots[0]) + __popc(ballots[1]) + __popc(ballots[2]) +
                        __popc(ballots[3]);
      if (total != a.channels) set_status(a.status, RKV_DEV_SELECT_FAILED);
    }
    __syncthreads();
    if (a.sel_channels && tid < a.channels)
      a.sel_channels[(size_t)ukv * a.channels + tid] = chosen[tid];

    // ---- approximate page scores: 8 pages per 16-byte load, one load per kept channel ----
    const int nchunk = (P + 7) >> 3;
    const size_t rowbase = (size_t)ukv * kHeadDim;
    for (int ch = tid; ch < nchunk; ch += kDecodeThreads) {
      float s8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) s8[j] = 0.f;
      int i = 0;
      for (; i + 4 <= a.channels; i += 4) {
        uint4 raw[4];
        float w[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int c = chosen[i + r] & (kHeadDim - 1);
          w[r] = qg[c];
          const bf16* base = (w[r] >= 0.f) ? a.kmax : a.kmin;
          raw[r] = __ldg(reinterpret_cast<const uint4*>(
              base + (rowbase + c) * a.page_cap + (size_t)ch * 8));
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float f[8];
          unpack8(raw[r], f);
#pragma unroll
          for (int j = 0; j < 8; ++j) s8[j] = fmaf(w[r], f[j], s8[j]);
        }
      }
      for (; i < a.channels; ++i) {
        const int c = chosen[i] & (kHeadDim - 1);
        const float w = qg[c];
        const bf16* base = (w >= 0.f) ? a.kmax : a.kmin;
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
            base + (rowbase + c) * a.page_cap + (size_t)ch * 8));
        float f[8];
        unpack8(raw, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) s8[j] = fmaf(w, f[j], s8[j]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int pg = ch * 8 + j;
        if (pg < P) {
          scores[pg] = s8[j];
          if (a.approx) a.approx[(size_t)ukv * a.page_cap + pg] = s8[j];
        }
      }
    }
    __syncthreads();

    // ---- page top-k ----------------------------------------------------------------------
    if (S >= P) {
      for (int i = tid; i < P; i += kDecodeThreads) sel[i] = i;
      nsel = P;
    } else {
      const int got = block_topk_ascending(scores, P, S, sel, sc);
      if (got != S && tid == 0) set_status(a.status, RKV_DEV_SELECT_FAILED);
      nsel = S;
    }
  } else {
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
  const int ppc = kChunkTokens / p;  // pages per stage
  const int nchunks = (nsel + ppc - 1) / ppc;
  const size_t cache_base = (size_t)ukv * a.cap;

  auto issue = [&](int c) {  // warp 0 only
    const int s = c % kStages;
    bf16* Ks = stages + (size_t)s * (2 * kChunkTokens * kHeadDim);
    bf16* Vs = Ks + kChunkTokens * kHeadDim;
    const int j0 = c * ppc, j1 = min(nsel, j0 + ppc);
    if (lane == 0) {
      uint32_t bytes = 0;
      for (int j = j0; j < j1; ++j) {
        const int t0 = sel[j] * p;
        bytes += 2u * (uint32_t)min(p, len - t0) * (kHeadDim * 2);
      }
      mbar_arrive_expect_tx(&bars[s], bytes);
    }
    __syncwarp();
    for (int j = j0 + lane; j < j1; j += 32) {
      const int t0 = sel[j] * p;
      const uint32_t nb = (uint32_t)min(p, len - t0) * (kHeadDim * 2);
      const int r = (j - j0) * p;
      bulk_g2s(Ks + r * kHeadDim, a.k_cache + (cache_base + t0) * kHeadDim, nb, &bars[s]);
      bulk_g2s(Vs + r * kHeadDim, a.v_cache + (cache_base + t0) * kHeadDim, nb, &bars[s]);
    }
  };

  if (warp == 0)
    for (int c = 0; c < min(nchunks, kStages); ++c) issue(c);

  // q pre-scaled into registers
  __syncthreads();
  for (int i = tid; i < G * kHeadDim; i += kDecodeThreads) qs[i] *= a.scale_log2;
  __syncthreads();
  WarpAttn<G> wa;
  wa.init(qs);

  bool failed = false;
  for (int c = 0; c < nchunks; ++c) {
    const int s = c % kStages;
    const bool ok = mbar_wait(&bars[s], (uint32_t)((c / kStages) & 1));
    if (__syncthreads_or(!ok)) {
      failed = true;
      if (tid == 0) set_status(a.status, RKV_DEV_WAIT_TIMEOUT);
      // drain the copies still in flight (bounded) before leaving
      for (int c2 = c + 1; c2 < min(nchunks, c + kStages); ++c2)
        mbar_wait(&bars[c2 % kStages], (uint32_t)((c2 / kStages) & 1));
      break;
    }
    const bf16* Ks = stages + (size_t)s * (2 * kChunkTokens * kHeadDim);
    const bf16* Vs = Ks + kChunkTokens * kHeadDim;
    const int j0 = c * ppc, j1 = min(nsel, j0 + ppc);
    const int last_t0 = sel[j1 - 1] * p;
    const int ntok = (j1 - j0 - 1) * p + min(p, len - last_t0);
    wa.step4(Ks, Vs, warp * 8, ntok);
    wa.step4(Ks, Vs, warp * 8 + 4, ntok);
    __syncthreads();
    if (warp == 0 && c + kStages < nchunks) issue(c + kStages);
  }
  if (failed) return;

  CombineSmem<G>* cs = reinterpret_cast<CombineSmem<G>*>(smem);
  warp_deposit<G>(wa, cs);
  __syncthreads();
  for (int i = tid; i < G * kHeadDim; i += kDecodeThreads) {
    const int h = i >> 7, c = i & 127;
    float M, L, O;
    warp_merge<G>(cs, h, c, &M, &L, &O);
    a.out[((size_t)u * hq + g * G + h) * kHeadDim + c] = __float2bfloat16_rn(O / L);
  }
}

cudaError_t launch_hybrid(const HybridArgs& a, cudaStream_t s) {
  const size_t smem = hybrid_smem_bytes(a.gqa, a.page_cap, a.budget, a.page);
  const dim3 grid(a.n * a.n_kv), block(kDecodeThreads);
  cudaError_t e = cudaSuccess;
  switch (a.gqa) {
#define RKV_CASE(GG)                                                                         \
  case GG:                                                                                   \
    e = ensure_dyn_smem((const void*)hybrid_decode_kernel<GG>, smem);                        \
    if (e != cudaSuccess) return e;                                                          \
    hybrid_decode_kernel<GG><<<grid, block, smem, s>>>(a);                                   \
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
// Decode-token append: one CTA per unit writes the new row of every KV head and folds it into
// the page summary it lands in, then bumps len[u].
// ==========================================================================================
__global__ void append_kernel(AppendArgs a) {
  const int u = blockIdx.x, c = threadIdx.x;  // 128 threads: one channel each
  const int len = a.len[u];
  const int pg = len / a.page;
  const bool fits = len >= 0 && len < a.cap && pg < a.page_cap;
  if (fits) {
    for (int g = 0; g < a.n_kv; ++g) {
      const size_t ukv = (size_t)u * a.n_kv + g;
      const bf16 kval = a.new_k[ukv * kHeadDim + c];
      a.k_cache[(ukv * a.cap + len) * kHeadDim + c] = kval;
      a.v_cache[(ukv * a.cap + len) * kHeadDim + c] = a.new_v[ukv * kHeadDim + c];
      const size_t si = (ukv * kHeadDim + c) * a.page_cap + pg;
      if (len % a.page == 0) {
        a.kmin[si] = kval;
        a.kmax[si] = kval;
      } else {
        const float kf = __bfloat162float(kval);
        if (kf < __bfloat162float(a.kmin[si])) a.kmin[si] = kval;
        if (kf > __bfloat162float(a.kmax[si])) a.kmax[si] = kval;
      }
    }
  }
  __syncthreads();
  if (c == 0) {
    if (fits)
      a.len[u] = len + 1;
    else
      set_status(a.status, RKV_DEV_LEN_OVER_CAP);
  }
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  append_kernel<<<a.n, kHeadDim, 0, s>>>(a);
  return cudaGetLastError();
}

// ==========================================================================================
// Page summaries: CTA = (unit, KV head) x 32 pages. Reads rows coalesced (64 threads per
// 256-byte row, bf16x2 each), reduces with exact bf16 min / max, transposes through shared
// memory and writes 64-byte channel rows.
// ==========================================================================================
constexpr int kSumPages = 32;

__global__ void __launch_bounds__(256) summaries_kernel(SummaryArgs a) {
  __shared__ __align__(16) __nv_bfloat162 smin[kSumPages][kHeadDim / 2 + 1];
  __shared__ __align__(16) __nv_bfloat162 smax[kSumPages][kHeadDim / 2 + 1];
  const int ukv = blockIdx.x;
  const int u = ukv / a.n_kv;
  const int len = a.len[u];
  const int p = a.page;
  const int P = (len + p - 1) / p;
  if (len < 0 || len > a.cap || P > a.page_cap) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_status(a.status, RKV_DEV_LEN_OVER_CAP);
    return;
  }
  const int pg0 = blockIdx.y * kSumPages;
  const int first_page = a.first_token / p;
  if (pg0 >= P || pg0 + kSumPages <= first_page) return;
  const int cp = threadIdx.x & 63, sub = threadIdx.x >> 6;
  const __nv_bfloat162* kc =
      reinterpret_cast<const __nv_bfloat162*>(a.k_cache + (size_t)ukv * a.cap * kHeadDim);
  for (int j = sub; j < kSumPages; j += 4) {
    const int pg = pg0 + j;
    if (pg >= P) break;
    const int t0 = pg * p, t1 = min(len, t0 + p);
    __nv_bfloat162 mn = kc[(size_t)t0 * (kHeadDim / 2) + cp], mx = mn;
    for (int t = t0 + 1; t < t1; ++t) {
      const __nv_bfloat162 x = kc[(size_t)t * (kHeadDim / 2) + cp];
      mn = __hmin2(mn, x);
      mx = __hmax2(mx, x);
    }
    smin[j][cp] = mn;
    smax[j][cp] = mx;
  }
  __syncthreads();
  // write: thread -> (channel c, 8-page group), pages [pg0, pg0 + 32) of channel row c
  const int npg = min(kSumPages, P - pg0);
  for (int i = threadIdx.x; i < kHeadDim * (kSumPages / 8); i += blockDim.x) {
    const int c = i >> 2, grp = i & 3;
    const int j0 = grp * 8;
    if (j0 >= npg) continue;
    const size_t row = ((size_t)ukv * kHeadDim + c) * a.page_cap + pg0 + j0;
    const int half = c & 1, cpair = c >> 1;
    const int first_j = max(0, first_page - pg0);
    uint16_t vmin[8], vmax[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int j = min(j0 + t, npg - 1);
      const __nv_bfloat162 a2 = smin[j][cpair], b2 = smax[j][cpair];
      const bf16 x = half ? a2.y : a2.x, y = half ? b2.y : b2.x;
      vmin[t] = *reinterpret_cast<const uint16_t*>(&x);
      vmax[t] = *reinterpret_cast<const uint16_t*>(&y);
    }
    uint16_t* kmin16 = reinterpret_cast<uint16_t*>(a.kmin);
    uint16_t* kmax16 = reinterpret_cast<uint16_t*>(a.kmax);
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
  summaries_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ==========================================================================================
// Dense decode (flash-decoding split-K): CTA = (unit, KV head, split); contiguous token runs
// staged by two bulk copies (K rows, V rows) per 64-token stage; partials merged by a second
// kernel.
// ==========================================================================================
void dense_plan(int n, int n_kv, int max_len, int* nsplit, int* tokens_per_split) {
  const int units = n * n_kv;
  const int target_ctas = 152 * 4;  // two waves of two resident CTAs per SM
  int ns = (target_ctas + units - 1) / units;
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
  __shared__ float qs[G * kHeadDim];
  __shared__ __align__(8) uint64_t bars[kStages];
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

  if (tid < G * 16) {
    const int h = tid >> 4, c8 = (tid & 15) * 8;
    const uint4 c = *reinterpret_cast<const uint4*>(
        a.q + ((size_t)u * hq + g * G + h) * kHeadDim + c8);
    float f[8];
    unpack8(c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) qs[h * kHeadDim + c8 + i] = f[i] * a.scale_log2;
  }
  if (tid < kStages) mbar_init(&bars[tid], 1);
  fence_barrier_init();
  __syncthreads();

  auto issue = [&](int c) {  // one thread
    const int s = c % kStages;
    bf16* Ks = stages + (size_t)s * (2 * kChunkTokens * kHeadDim);
    bf16* Vs = Ks + kChunkTokens * kHeadDim;
    const int nt = min(kChunkTokens, ntok_all - c * kChunkTokens);
    const uint32_t nb = (uint32_t)nt * (kHeadDim * 2);
    mbar_arrive_expect_tx(&bars[s], 2 * nb);
    bulk_g2s(Ks, a.k + base + (size_t)c * kChunkTokens * kHeadDim, nb, &bars[s]);
    bulk_g2s(Vs, a.v + base + (size_t)c * kChunkTokens * kHeadDim, nb, &bars[s]);
  };
  if (tid == 0)
    for (int c = 0; c < min(nchunks, kStages); ++c) issue(c);

  WarpAttn<G> wa;
  wa.init(qs);
  for (int c = 0; c < nchunks; ++c) {
    const int s = c % kStages;
    const bool ok = mbar_wait(&bars[s], (uint32_t)((c / kStages) & 1));
    if (__syncthreads_or(!ok)) {
      if (tid == 0) set_status(a.status, RKV_DEV_WAIT_TIMEOUT);
      for (int c2 = c + 1; c2 < min(nchunks, c + kStages); ++c2)
        mbar_wait(&bars[c2 % kStages], (uint32_t)((c2 / kStages) & 1));
      return;
    }
    const bf16* Ks = stages + (size_t)s * (2 * kChunkTokens * kHeadDim);
    const bf16* Vs = Ks + kChunkTokens * kHeadDim;
    const int ntok = min(kChunkTokens, ntok_all - c * kChunkTokens);
    wa.step4(Ks, Vs, warp * 8, ntok);
    wa.step4(Ks, Vs, warp * 8 + 4, ntok);
    __syncthreads();
    if (tid == 0 && c + kStages < nchunks) issue(c + kStages);
  }

  CombineSmem<G>* cs = reinterpret_cast<CombineSmem<G>*>(smem);
  warp_deposit<G>(wa, cs);
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
    const float f = exp2f(pm[s] - M);
    L = fmaf(pl[s], f, L);
    O = fmaf(po[(size_t)s * kHeadDim + c], f, O);
  }
  a.out[(size_t)row * kHeadDim + c] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
}

cudaError_t launch_dense(const DenseArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)kStages * kStageBytes;
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
