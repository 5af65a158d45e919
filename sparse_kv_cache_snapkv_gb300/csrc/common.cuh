// Device-side building blocks shared by the RocketKV kernels (sm_103a).
//
//  * bf16 unpacking (exact widening to fp32)
//  * mbarrier + cp.async.bulk wrappers (non-tensor bulk copies global -> shared), with waits
//    bounded by the global timer so that no kernel can spin forever
//  * block-wide exclusive scan
//  * block-wide top-k radix select (largest keys first, ties -> lower index), emitting the
//    selected indices in ascending order
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "../../include/rkv.h"
#include "rkv_internal.h"

namespace rkv {

// ------------------------------------------------------------------------------------------
// status word
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------------------------------------------------
// bf16 helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4& c, float* f) {
  f[0] = bf16_lo(c.x); f[1] = bf16_hi(c.x);
  f[2] = bf16_lo(c.y); f[3] = bf16_hi(c.y);
  f[4] = bf16_lo(c.z); f[5] = bf16_hi(c.z);
  f[6] = bf16_lo(c.w); f[7] = bf16_hi(c.w);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------------------------------
// mbarrier / bulk copy
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies, tensor core).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete. Gives up after kWaitLimitNs of wall time and
// returns false (the caller records RKV_DEV_WAIT_TIMEOUT and abandons its unit).
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 1-D bulk copy global -> shared of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16-byte asynchronous global -> shared copies (LDGSTS). A thread waits for its own copies with
// cp_async_wait_all(); a barrier then publishes them to the other threads.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with programmatic stream serialisation may
// start while the previous kernel in the stream drains; pdl_wait() blocks until that kernel has
// completed and its writes are visible (a no-op for an ordinary launch). pdl_trigger() lets the
// next such kernel be scheduled early.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// warp / block reductions and scans
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// ------------------------------------------------------------------------------------------
// top-k radix select
// ------------------------------------------------------------------------------------------
// Order-preserving map float -> uint32 (larger float -> larger integer). -0 is folded to +0 so
// that the two zeros tie, as they do as real numbers.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  if (f == 0.0f) f = 0.0f;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct __align__(16) SelectScratch {
  uint32_t hist[8][256];  // one histogram per warp (warps w and w + 8 share one)
  unsigned long long tmp[33];
  uint32_t wmax[32], wmin[32];
  uint32_t digit;
  int above;
  int in_bin;
};

__device__ __forceinline__ unsigned long long warp_incl_scan64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive scan of 64-bit values over the block (contains __syncthreads()).
__device__ __forceinline__ unsigned long long block_excl_scan64(unsigned long long v,
                                                                unsigned long long* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned long long incl = warp_incl_scan64(v);
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = lane < nw ? tmp[lane] : 0ull;
    const unsigned long long wi = warp_incl_scan64(w);
    if (lane < nw) tmp[lane] = wi - w;
  }
  __syncthreads();
  const unsigned long long r = tmp[warp] + incl - v;
  __syncthreads();
  return r;
}

// Choose the k largest of keys[0..n) (ties -> lower index) and write their indices, ascending,
// to out[0..k). keys may live in shared or global memory. 1 <= k <= n. Every thread of the
// block (a multiple of 32 threads) must call it. Returns the number written.
//
// MSB-first radix select on order-preserving integer keys. The bits common to every key are
// found first (block max / min) and skipped, so the 8-bit histograms start where keys differ;
// the search stops as soon as the whole threshold bin is taken. The final pass writes the
// selected indices in index order using one block-wide scan of (above, equal) counts.
__device__ __noinline__ static int block_topk_ascending(const float* keys, int n, int k, int* out,
                                                        SelectScratch& sc) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int nw = nt >> 5;
  uint32_t hi = 0u, lo = 0xffffffffu;
  for (int i = tid; i < n; i += nt) {
    const uint32_t u = ordered_key(keys[i]);
    hi = max(hi, u);
    lo = min(lo, u);
  }
  hi = __reduce_max_sync(0xffffffffu, hi);
  lo = __reduce_min_sync(0xffffffffu, lo);
  if (lane == 0) {
    sc.wmax[warp] = hi;
    sc.wmin[warp] = lo;
  }
  __syncthreads();
  hi = sc.wmax[0];
  lo = sc.wmin[0];
  for (int w = 1; w < nw; ++w) {
    hi = max(hi, sc.wmax[w]);
    lo = min(lo, sc.wmin[w]);
  }
  const uint32_t diff = hi ^ lo;
  int start = diff ? 32 - __clz(diff) : 0;  // bits [start, 32) are equal in every key
  uint32_t mask = start >= 32 ? 0u : ~((1u << start) - 1u);
  uint32_t prefix = hi & mask;
  int remaining = k;
  bool inclusive = false;  // true: the selection is exactly {u >= prefix}
  while (start > 0) {
    const int nb = start < 8 ? start : 8;
    const int shift = start - nb;
    const uint32_t dmask = (1u << nb) - 1u;
    // Each warp counts into its own histogram: keys that share leading bits then contend only
    // within a warp, not across the block.
    for (int i = tid; i < 8 * 256; i += nt) (&sc.hist[0][0])[i] = 0;
    __syncthreads();
    uint32_t* myhist = sc.hist[warp & 7];
    for (int i = tid; i < n; i += nt) {
      const uint32_t u = ordered_key(keys[i]);
      if ((u & mask) == prefix) atomicAdd(&myhist[(u >> shift) & dmask], 1u);
    }
    __syncthreads();
    for (int b = tid; b < 256; b += nt) {
      uint32_t t = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) t += sc.hist[w][b];
      sc.hist[0][b] = t;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending); bins >= 2^nb are empty
      int cnt[8];
      int s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = (int)sc.hist[0][255 - 8 * lane - j];
        s += cnt[j];
      }
      const int incl = warp_incl_scan(s);
      const int excl = incl - s;
      if (excl < remaining && incl >= remaining) {
        int acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + cnt[j] >= remaining) {
            sc.digit = (uint32_t)(255 - 8 * lane - j);
            sc.above = acc;
            sc.in_bin = cnt[j];
            break;
          }
          acc += cnt[j];
        }
      }
    }
    __syncthreads();
    prefix |= sc.digit << shift;
    mask |= dmask << shift;
    remaining -= sc.above;
    start = shift;
    if (sc.in_bin == remaining) {
      inclusive = true;
      break;
    }
  }
  // keys above the threshold, and keys equal to it (the first `remaining` of them are taken)
  const int per = (n + nt - 1) / nt;
  const int beg = min(n, tid * per), end = min(n, beg + per);
  unsigned gt = 0, eq = 0;
  for (int i = beg; i < end; ++i) {
    const uint32_t u = ordered_key(keys[i]);
    if (inclusive) {
      gt += (u >= prefix);
    } else {
      gt += (u > prefix);
      eq += (u == prefix);
    }
  }
  const unsigned long long before =
      block_excl_scan64(((unsigned long long)gt << 32) | eq, sc.tmp);
  const int need_eq = inclusive ? 0 : remaining;
  const int eq_before = (int)(before & 0xffffffffull);
  const int gt_before = (int)(before >> 32);
  int pos = gt_before + min(eq_before, need_eq);
  int eq_seen = eq_before;
  for (int i = beg; i < end; ++i) {
    const uint32_t u = ordered_key(keys[i]);
    bool take;
    if (inclusive) {
      take = u >= prefix;
    } else {
      take = u > prefix;
      if (u == prefix) {
        take = eq_seen < need_eq;
        ++eq_seen;
      }
    }
    if (take) {
      if (pos < k) out[pos] = i;
      ++pos;
    }
  }
  // total selected: every thread's pos past its range adds up; report via the last thread
  if (tid == nt - 1) sc.above = pos;
  __syncthreads();
  const int total = sc.above;
  __syncthreads();
  return total;
}

// One warp chooses the k largest of keys[0..n) (n <= 128, keys in shared memory; ties -> lower
// index) and writes their indices ascending to out[0..k). Bit-plane radix select with ballots:
// no block barrier, no atomics. Every lane of the warp must call it. Returns the count written.
__device__ __forceinline__ int warp_topk_small(const float* keys, int n, int k, int* out) {
  const int lane = threadIdx.x & 31;
  uint32_t u[4];
  bool valid[4];
  uint32_t hi = 0u, lo = 0xffffffffu;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int idx = 4 * lane + j;
    valid[j] = idx < n;
    u[j] = valid[j] ? ordered_key(keys[idx]) : 0u;
    if (valid[j]) {
      hi = max(hi, u[j]);
      lo = min(lo, u[j]);
    }
  }
  hi = __reduce_max_sync(0xffffffffu, hi);
  lo = __reduce_min_sync(0xffffffffu, lo);
  const uint32_t diff = hi ^ lo;
  const int top = diff ? 31 - __clz(diff) : -1;  // highest bit where keys differ
  uint32_t prefix = top < 0 ? hi : (top >= 31 ? 0u : (hi & ~((2u << top) - 1u)));
  int remaining = k;
  for (int b = top; b >= 0; --b) {
    const uint32_t cand = prefix | (1u << b);
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      cnt += __popc(__ballot_sync(0xffffffffu, valid[j] && (u[j] >> b) == (cand >> b)));
    if (cnt >= remaining)
      prefix = cand;
    else
      remaining -= cnt;
  }
  // prefix is the k-th largest key; `remaining` keys equal to it are taken, lowest index first
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t eqb[4], selb[4];
  bool eq[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    eq[j] = valid[j] && u[j] == prefix;
    eqb[j] = __ballot_sync(0xffffffffu, eq[j]);
  }
  int eq_before = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) eq_before += __popc(eqb[j] & lt);
  bool take[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    take[j] = valid[j] && (u[j] > prefix || (eq[j] && eq_before < remaining));
    eq_before += eq[j] ? 1 : 0;
    selb[j] = __ballot_sync(0xffffffffu, take[j]);
  }
  int pos = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) pos += __popc(selb[j] & lt);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (take[j]) {
      if (pos < k) out[pos] = 4 * lane + j;
      ++pos;
    }
  }
  int total = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) total += __popc(selb[j]);
  return total;
}

// ------------------------------------------------------------------------------------------
// Low-latency top-k for one 256-thread block with at most NK * 256 keys.
// ------------------------------------------------------------------------------------------
struct __align__(16) FastSelectSmem {
  uint32_t hist[2][4][256];  // double-buffered; warps 2p (low 16 bits) and 2p+1 (high) share row p
  uint32_t wmax[8], wmin[8];
  int wsum[8];               // per-warp sums of the descending bin scan
  int found[4];              // digit, keys above, keys in the digit's bin
  uint32_t cnt[16][8];       // per key round and warp: (keys above << 16) | keys equal
};

// Same contract as block_topk_ascending (k largest, ties -> lower index, indices written
// ascending; returns the count), for blockDim.x == 256 and n <= NK * 256. Keys stay in
// registers (key i = 256 j + tid). MSB-first radix select with 8-bit digits after the bits all
// keys share; per pass: counts into per-warp-pair rows (atomics contend only within a warp
// pair), thread b totals bin 255 - b, warps scan 32 bins each, the thread whose bin holds the
// k-th key publishes it (three barriers). The search stops as soon as a whole bin is taken.
// The in-order compaction packs per-warp (above, equal) counts of every key round.
template <int NK>
__device__ __forceinline__ int block_topk_fast(const float* keys, int n, int k, int* out,
                                               FastSelectSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t u[NK];
  bool v[NK];
  uint32_t hi = 0u, lo = 0xffffffffu;
#pragma unroll
  for (int j = 0; j < NK; ++j) {
    const int idx = j * 256 + tid;
    v[j] = idx < n;
    u[j] = v[j] ? ordered_key(keys[idx]) : 0u;
    if (v[j]) {
      hi = max(hi, u[j]);
      lo = min(lo, u[j]);
    }
  }
  hi = __reduce_max_sync(0xffffffffu, hi);
  lo = __reduce_min_sync(0xffffffffu, lo);
  if (lane == 0) {
    sm.wmax[warp] = hi;
    sm.wmin[warp] = lo;
  }
  reinterpret_cast<uint4*>(&sm.hist[0][0][0])[tid] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  {
    const uint4 a0 = reinterpret_cast<const uint4*>(sm.wmax)[0];
    const uint4 a1 = reinterpret_cast<const uint4*>(sm.wmax)[1];
    const uint4 b0 = reinterpret_cast<const uint4*>(sm.wmin)[0];
    const uint4 b1 = reinterpret_cast<const uint4*>(sm.wmin)[1];
    hi = max(max(max(a0.x, a0.y), max(a0.z, a0.w)), max(max(a1.x, a1.y), max(a1.z, a1.w)));
    lo = min(min(min(b0.x, b0.y), min(b0.z, b0.w)), min(min(b1.x, b1.y), min(b1.z, b1.w)));
  }
  const uint32_t diff = hi ^ lo;
  int start = diff ? 32 - __clz(diff) : 0;
  uint32_t mask = start >= 32 ? 0u : ~((1u << start) - 1u);
  uint32_t prefix = hi & mask;
  int remaining = k;
  bool inclusive = false;
  const uint32_t inc = (warp & 1) ? 0x10000u : 1u;
  for (int pass = 0; start > 0; ++pass) {
    const int nb = start < 8 ? start : 8;
    const int shift = start - nb;
    const uint32_t dmask = (1u << nb) - 1u;
    uint32_t* H = &sm.hist[pass & 1][0][0];
    uint32_t* row = H + (warp >> 1) * 256;
#pragma unroll
    for (int j = 0; j < NK; ++j)
      if (v[j] && (u[j] & mask) == prefix) atomicAdd(&row[(u[j] >> shift) & dmask], inc);
    __syncthreads();
    // bin 255 - tid, summed over the four rows; warps scan their 32 bins in descending order
    const int bin = 255 - tid;
    int own = 0;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      const uint32_t w = H[pr * 256 + bin];
      own += (int)((w & 0xffffu) + (w >> 16));
    }
    const int incl_w = warp_incl_scan(own);
    if (lane == 31) sm.wsum[warp] = incl_w;
    // the other buffer is refilled next pass; its last readers finished before this pass began
    reinterpret_cast<uint4*>(&sm.hist[(pass + 1) & 1][0][0])[tid] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    int before = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) before += (w < warp) ? sm.wsum[w] : 0;
    const int incl = before + incl_w, excl = incl - own;
    if (own > 0 && excl < remaining && incl >= remaining) {
      sm.found[0] = bin;
      sm.found[1] = excl;
      sm.found[2] = own;
    }
    __syncthreads();
    const int digit = sm.found[0], above = sm.found[1], in_bin = sm.found[2];
    prefix |= (uint32_t)digit << shift;
    mask |= dmask << shift;
    remaining -= above;
    start = shift;
    if (in_bin == remaining) {
      inclusive = true;
      break;
    }
  }
  // compaction in index order (round j, then thread)
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t bg[NK], be[NK];
#pragma unroll
  for (int j = 0; j < NK; ++j) {
    const bool g = v[j] && (inclusive ? u[j] >= prefix : u[j] > prefix);
    const bool e = v[j] && !inclusive && u[j] == prefix;
    bg[j] = __ballot_sync(0xffffffffu, g);
    be[j] = __ballot_sync(0xffffffffu, e);
    if (lane == 0) sm.cnt[j][warp] = ((uint32_t)__popc(bg[j]) << 16) | (uint32_t)__popc(be[j]);
  }
  __syncthreads();
  const int need_eq = inclusive ? 0 : remaining;
  int gt_acc = 0, eq_acc = 0;
#pragma unroll
  for (int j = 0; j < NK; ++j) {
    const uint4 c0 = reinterpret_cast<const uint4*>(sm.cnt[j])[0];
    const uint4 c1 = reinterpret_cast<const uint4*>(sm.cnt[j])[1];
    const uint32_t c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint32_t below = 0u, all = 0u;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      below += (w < warp) ? c[w] : 0u;
      all += c[w];
    }
    const int eq_before = eq_acc + (int)(below & 0xffffu) + __popc(be[j] & lt);
    const int gt_before = gt_acc + (int)(below >> 16) + __popc(bg[j] & lt);
    const bool g = (bg[j] >> lane) & 1u, e = (be[j] >> lane) & 1u;
    const bool take = g || (e && eq_before < need_eq);
    const int pos = gt_before + min(eq_before, need_eq);
    if (take && pos < k) out[pos] = j * 256 + tid;
    gt_acc += (int)(all >> 16);
    eq_acc += (int)(all & 0xffffu);
  }
  __syncthreads();
  return gt_acc + min(eq_acc, need_eq);
}

}  // namespace rkv
