// Device-side building blocks shared by the RocketKV kernels (sm_103a).
//
//  * paged-cache addressing, bf16 unpacking (exact widening to fp32)
//  * mbarrier wrappers with waits bounded by the global timer, so that no kernel can spin
//    forever; 16-byte cp.async copies; programmatic-dependent-launch controls
//  * warp / block scans
//  * top-k selects (largest keys first, ties -> lower index, indices emitted in ascending order):
//    a general block radix select and low-latency block selects for <= NK * 256 keys (a
//    variant for <= 1024 keys with contiguous keys per thread)
#pragma once

#include <cstddef>
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
// paged cache addressing
// ------------------------------------------------------------------------------------------
// Block of token t of unit u, checked against the pool size (block 0 and RKV_DEV_BAD_INDEX if a
// table entry is out of range). t / block < max_blocks is the caller's bound (len <= capacity).
__device__ __forceinline__ int paged_block(const PagedMap& m, int u, int t, uint32_t* status) {
  int blk = m.table[(size_t)u * m.max_blocks + t / m.block];
  if (blk < 0 || blk >= m.num_blocks) {
    set_status(status, RKV_DEV_BAD_INDEX);
    blk = 0;
  }
  return blk;
}

// Row (128 elements) of a pool [num_blocks][n_kv][block][128] holding token t of head g in blk.
__device__ __forceinline__ size_t paged_row(const PagedMap& m, int blk, int n_kv, int g, int t) {
  return ((size_t)blk * n_kv + g) * m.block + (t % m.block);
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

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32, a few ulp of relative error).
// Results below the smallest normal float flush to zero; every caller sums or scales
// probabilities, where such a term is negligible. The score passes take one exponential per
// logit; with this instruction in place of exp2f they ran 14 % faster on GB300.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_addr(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// 16-byte asynchronous global -> shared copies (LDGSTS). A thread waits for its own copies with
// cp_async_wait_all(); a barrier then publishes them to the other threads.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}
// Hint: bring `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src_gmem, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes)
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

// ------------------------------------------------------------------------------------------
// Low-latency top-k for one 256-thread block with at most NK * 256 keys.
// ------------------------------------------------------------------------------------------
struct __align__(16) FastSelectSmem {
  uint32_t h11[2048];        // fine histogram of the first pass (up to 11 bits)
  uint32_t coarse[64];       // the same counts summed over 32 fine bins
  uint32_t hist[2][4][256];  // 8-bit fallback passes, double-buffered; warps 2p, 2p+1 share row p
  uint32_t wmax[8], wmin[8];
  int wsum[8];               // per-warp sums of a fallback pass's descending bin scan
  int found[4];              // fallback pass: digit, keys above, keys in the digit's bin
  uint32_t cnt[16][8];       // per key round and warp: (keys above << 16) | keys equal
  uint32_t cand_u[32];       // keys of a small final bin and their indices
  int cand_i[32];
  int ncand;
};
// every array read or cleared with 16-byte vector accesses starts on a 16-byte boundary
static_assert(offsetof(FastSelectSmem, h11) % 16 == 0, "h11 alignment");
static_assert(offsetof(FastSelectSmem, coarse) % 16 == 0, "coarse alignment");
static_assert(offsetof(FastSelectSmem, hist) % 16 == 0, "hist alignment");
static_assert(offsetof(FastSelectSmem, wmax) % 16 == 0, "wmax alignment");
static_assert(offsetof(FastSelectSmem, wmin) % 16 == 0, "wmin alignment");
static_assert(offsetof(FastSelectSmem, cnt) % 16 == 0, "cnt alignment");

// First phase of block_topk_fast, to be fused into whatever produces the keys: each thread
// passes the max / min of the ordered keys (ordered_key) it produced (0 / ~0 if none); this
// records the per-warp range and clears the histograms. A barrier must separate it from
// block_topk_fast (the one that publishes the keys serves).
// Clears the histograms and the candidate count (the part of fast_select_prepare that does not
// depend on the keys).
__device__ __forceinline__ void fast_select_clear(FastSelectSmem& sm) {
  const int tid = threadIdx.x;
  uint4* h = reinterpret_cast<uint4*>(sm.h11);
  h[2 * tid] = make_uint4(0u, 0u, 0u, 0u);
  h[2 * tid + 1] = make_uint4(0u, 0u, 0u, 0u);
  if (tid < 16) reinterpret_cast<uint4*>(sm.coarse)[tid] = make_uint4(0u, 0u, 0u, 0u);
  reinterpret_cast<uint4*>(&sm.hist[0][0][0])[tid] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) sm.ncand = 0;
}

__device__ __forceinline__ void fast_select_prepare(uint32_t hi, uint32_t lo, FastSelectSmem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  hi = __reduce_max_sync(0xffffffffu, hi);
  lo = __reduce_min_sync(0xffffffffu, lo);
  if (lane == 0) {
    sm.wmax[warp] = hi;
    sm.wmin[warp] = lo;
  }
  fast_select_clear(sm);
}

// Same contract as block_topk_ascending (k largest, ties -> lower index, indices written
// ascending; returns the count), for blockDim.x == 256, 1 <= k <= n <= NK * 256, after
// fast_select_prepare over the same keys. Keys stay in registers (key i = 256 j + tid).
// MSB-first radix select on the bits below those all keys share. First pass: up to 11 bits
// counted at once into a fine and a coarse histogram; every warp then finds the bin of the k-th
// key on its own (a scan of the 64 coarse bins, then of the 32 fine bins inside the chosen one),
// so no barrier is spent on publishing it. If that bin is taken whole the threshold is known;
// if it holds at most 32 keys they are gathered and every warp ranks them by (key desc, index
// asc), which yields the exact k-th key; otherwise 8-bit passes continue (three barriers each,
// warps scan 32 bins of per-warp-pair counts). The compaction packs per-warp (above, equal)
// counts of every key round. Ends without a barrier: the caller synchronises before reading
// out[] or reusing `sm`.
template <int NK>
__device__ __forceinline__ int block_topk_fast(const float* keys, int n, int k, int* out,
                                               FastSelectSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t u[NK];
  bool v[NK];
#pragma unroll
  for (int j = 0; j < NK; ++j) {
    const int idx = j * 256 + tid;
    v[j] = idx < n;
    u[j] = v[j] ? ordered_key(keys[idx]) : 0u;
  }
  uint32_t hi, lo;
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
  if (start > 0) {
    const int nb = start < 11 ? start : 11;
    const int shift = start - nb;
    const uint32_t dmask = (1u << nb) - 1u;
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      if (v[j]) {
        const uint32_t d = (u[j] >> shift) & dmask;
        atomicAdd(&sm.h11[d], 1u);
        atomicAdd(&sm.coarse[d >> 5], 1u);
      }
    }
    __syncthreads();
    // coarse bins in descending order: lane l holds bins 63 - 2l and 62 - 2l
    const uint2 cc = *reinterpret_cast<const uint2*>(&sm.coarse[62 - 2 * lane]);
    const int c_hi = (int)cc.y, c_lo = (int)cc.x;
    int incl = warp_incl_scan(c_hi + c_lo);
    int excl = incl - c_hi - c_lo;
    uint32_t b = __ballot_sync(0xffffffffu, excl < remaining && incl >= remaining);
    int src = __ffs(b) - 1;
    const int cbin_l = (excl + c_hi >= remaining) ? 63 - 2 * lane : 62 - 2 * lane;
    const int above_l = (excl + c_hi >= remaining) ? excl : excl + c_hi;
    const int cbin = __shfl_sync(0xffffffffu, cbin_l, src);
    const int above_c = __shfl_sync(0xffffffffu, above_l, src);
    // fine bins of that coarse bin, descending: lane l holds bin 32 cbin + 31 - l
    const int f = (int)sm.h11[cbin * 32 + 31 - lane];
    incl = warp_incl_scan(f) + above_c;
    excl = incl - f;
    b = __ballot_sync(0xffffffffu, excl < remaining && incl >= remaining);
    src = __ffs(b) - 1;
    const int digit = cbin * 32 + 31 - src;
    const int above = __shfl_sync(0xffffffffu, excl, src);
    const int in_bin = __shfl_sync(0xffffffffu, f, src);
    prefix |= (uint32_t)digit << shift;
    mask |= dmask << shift;
    remaining -= above;
    start = shift;
    if (in_bin == remaining) {
      inclusive = true;
      start = 0;
    } else if (start > 0 && in_bin <= 32) {
#pragma unroll
      for (int j = 0; j < NK; ++j) {
        if (v[j] && (u[j] & mask) == prefix) {
          const int slot = atomicAdd(&sm.ncand, 1);
          sm.cand_u[slot] = u[j];
          sm.cand_i[slot] = j * 256 + tid;
        }
      }
      __syncthreads();
      const bool mine = lane < in_bin;
      const uint32_t cu = mine ? sm.cand_u[lane] : 0u;
      const int ci = mine ? sm.cand_i[lane] : 0x7fffffff;
      int rank = 0, gt = 0;
      for (int m = 0; m < in_bin; ++m) {
        const uint32_t ou = __shfl_sync(0xffffffffu, cu, m);
        const int oi = __shfl_sync(0xffffffffu, ci, m);
        gt += ou > cu ? 1 : 0;
        rank += (ou > cu || (ou == cu && oi < ci)) ? 1 : 0;
      }
      b = __ballot_sync(0xffffffffu, mine && rank == remaining - 1);
      src = __ffs(b) - 1;
      prefix = __shfl_sync(0xffffffffu, cu, src);
      remaining -= __shfl_sync(0xffffffffu, gt, src);
      start = 0;
    }
  }
  const uint32_t inc = (warp & 1) ? 0x10000u : 1u;
  for (int pass = 0; start > 0 && !inclusive; ++pass) {
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
  return gt_acc + min(eq_acc, need_eq);
}

// block_topk_fast for n <= 1024 with thread t holding the contiguous keys 4t .. 4t + 3 (one
// 16-byte load; `keys` 16-byte aligned): the radix steps are the same, and the compaction needs
// one ballot per bit of a thread's 0..4 taken keys, because (warp, lane, j) is already index
// order. A ranked k-th key whose equal keys are all needed turns the rule into "take >= it",
// which skips the count of equal keys. Ends without a barrier.
__device__ __forceinline__ int block_topk_1024(const float* keys, int n, int k, int* out,
                                             FastSelectSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NK = 4;
  uint32_t u[NK];
  bool v[NK];
  {
    const int i0 = 4 * tid;
    if (i0 + 3 < n) {
      const float4 f = reinterpret_cast<const float4*>(keys)[tid];
      u[0] = ordered_key(f.x);
      u[1] = ordered_key(f.y);
      u[2] = ordered_key(f.z);
      u[3] = ordered_key(f.w);
      v[0] = v[1] = v[2] = v[3] = true;
    } else {
#pragma unroll
      for (int j = 0; j < NK; ++j) {
        v[j] = i0 + j < n;
        u[j] = v[j] ? ordered_key(keys[i0 + j]) : 0u;
      }
    }
  }
  uint32_t hi, lo;
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
  if (start > 0) {
    const int nb = start < 11 ? start : 11;
    const int shift = start - nb;
    const uint32_t dmask = (1u << nb) - 1u;
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      if (v[j]) {
        const uint32_t d = (u[j] >> shift) & dmask;
        atomicAdd(&sm.h11[d], 1u);
        atomicAdd(&sm.coarse[d >> 5], 1u);
      }
    }
    __syncthreads();
    const uint2 cc = *reinterpret_cast<const uint2*>(&sm.coarse[62 - 2 * lane]);
    const int c_hi = (int)cc.y, c_lo = (int)cc.x;
    int incl = warp_incl_scan(c_hi + c_lo);
    int excl = incl - c_hi - c_lo;
    uint32_t b = __ballot_sync(0xffffffffu, excl < remaining && incl >= remaining);
    int src = __ffs(b) - 1;
    const int cbin_l = (excl + c_hi >= remaining) ? 63 - 2 * lane : 62 - 2 * lane;
    const int above_l = (excl + c_hi >= remaining) ? excl : excl + c_hi;
    const int cbin = __shfl_sync(0xffffffffu, cbin_l, src);
    const int above_c = __shfl_sync(0xffffffffu, above_l, src);
    const int f = (int)sm.h11[cbin * 32 + 31 - lane];
    incl = warp_incl_scan(f) + above_c;
    excl = incl - f;
    b = __ballot_sync(0xffffffffu, excl < remaining && incl >= remaining);
    src = __ffs(b) - 1;
    const int digit = cbin * 32 + 31 - src;
    const int above = __shfl_sync(0xffffffffu, excl, src);
    const int in_bin = __shfl_sync(0xffffffffu, f, src);
    prefix |= (uint32_t)digit << shift;
    mask |= dmask << shift;
    remaining -= above;
    start = shift;
    if (in_bin == remaining) {
      inclusive = true;
      start = 0;
    } else if (start > 0 && in_bin <= 32) {
#pragma unroll
      for (int j = 0; j < NK; ++j) {
        if (v[j] && (u[j] & mask) == prefix) {
          const int slot = atomicAdd(&sm.ncand, 1);
          sm.cand_u[slot] = u[j];
          sm.cand_i[slot] = 4 * tid + j;
        }
      }
      __syncthreads();
      const bool mine = lane < in_bin;
      const uint32_t cu = mine ? sm.cand_u[lane] : 0u;
      const int ci = mine ? sm.cand_i[lane] : 0x7fffffff;
      int rank = 0, gt = 0, eq = 0;
      for (int m = 0; m < in_bin; ++m) {
        const uint32_t ou = __shfl_sync(0xffffffffu, cu, m);
        const int oi = __shfl_sync(0xffffffffu, ci, m);
        gt += ou > cu ? 1 : 0;
        eq += ou == cu ? 1 : 0;
        rank += (ou > cu || (ou == cu && oi < ci)) ? 1 : 0;
      }
      b = __ballot_sync(0xffffffffu, mine && rank == remaining - 1);
      src = __ffs(b) - 1;
      prefix = __shfl_sync(0xffffffffu, cu, src);
      const int gt_k = __shfl_sync(0xffffffffu, gt, src);
      const int eq_k = __shfl_sync(0xffffffffu, eq, src);
      // when every key equal to the k-th one is needed, the rule is simply "take >= prefix"
      if (eq_k == remaining - gt_k) {
        inclusive = true;
      } else {
        remaining -= gt_k;
      }
      start = 0;
    }
  }
  const uint32_t inc = (warp & 1) ? 0x10000u : 1u;
  for (int pass = 0; start > 0 && !inclusive; ++pass) {
    const int nb = start < 8 ? start : 8;
    const int shift = start - nb;
    const uint32_t dmask = (1u << nb) - 1u;
    uint32_t* H = &sm.hist[pass & 1][0][0];
    uint32_t* row = H + (warp >> 1) * 256;
#pragma unroll
    for (int j = 0; j < NK; ++j)
      if (v[j] && (u[j] & mask) == prefix) atomicAdd(&row[(u[j] >> shift) & dmask], inc);
    __syncthreads();
    const int bin = 255 - tid;
    int own = 0;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      const uint32_t w = H[pr * 256 + bin];
      own += (int)((w & 0xffffu) + (w >> 16));
    }
    const int incl_w = warp_incl_scan(own);
    if (lane == 31) sm.wsum[warp] = incl_w;
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
  // compaction in index order: thread t's keys are contiguous, so (warp, lane, j) is ascending
  const uint32_t lt = (1u << lane) - 1u;
  const int need_eq = inclusive ? 0 : remaining;
  int cg = 0, ce = 0;
  bool g[NK], e[NK];
#pragma unroll
  for (int j = 0; j < NK; ++j) {
    g[j] = v[j] && (inclusive ? u[j] >= prefix : u[j] > prefix);
    e[j] = v[j] && !inclusive && u[j] == prefix;
    cg += g[j] ? 1 : 0;
    ce += e[j] ? 1 : 0;
  }
  // warp-exclusive prefix of cg and ce (each 0..4) from the ballots of their bits
  const uint32_t g0 = __ballot_sync(0xffffffffu, cg & 1);
  const uint32_t g1 = __ballot_sync(0xffffffffu, cg & 2);
  const uint32_t g2 = __ballot_sync(0xffffffffu, cg & 4);
  int gb = __popc(g0 & lt) + 2 * __popc(g1 & lt) + 4 * __popc(g2 & lt);
  const int gw = __popc(g0) + 2 * __popc(g1) + 4 * __popc(g2);
  int eb = 0, ew = 0;
  if (!inclusive) {
    const uint32_t e0 = __ballot_sync(0xffffffffu, ce & 1);
    const uint32_t e1 = __ballot_sync(0xffffffffu, ce & 2);
    const uint32_t e2 = __ballot_sync(0xffffffffu, ce & 4);
    eb = __popc(e0 & lt) + 2 * __popc(e1 & lt) + 4 * __popc(e2 & lt);
    ew = __popc(e0) + 2 * __popc(e1) + 4 * __popc(e2);
  }
  if (lane == 0) sm.cnt[0][warp] = ((uint32_t)gw << 16) | (uint32_t)ew;
  __syncthreads();
  const uint4 c0 = reinterpret_cast<const uint4*>(sm.cnt[0])[0];
  const uint4 c1 = reinterpret_cast<const uint4*>(sm.cnt[0])[1];
  const uint32_t c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  uint32_t below = 0u, all = 0u;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    below += (w < warp) ? c[w] : 0u;
    all += c[w];
  }
  gb += (int)(below >> 16);
  eb += (int)(below & 0xffffu);
#pragma unroll
  for (int j = 0; j < NK; ++j) {
    const bool take = g[j] || (e[j] && eb < need_eq);
    const int pos = gb + min(eb, need_eq);
    if (take && pos < k) out[pos] = 4 * tid + j;
    gb += g[j] ? 1 : 0;
    eb += e[j] ? 1 : 0;
  }
  return (int)(all >> 16) + min((int)(all & 0xffffu), need_eq);
}

// ------------------------------------------------------------------------------------------
// Top-k of page scores by value bins, for one 256-thread block (the decode's page select)
// ------------------------------------------------------------------------------------------
// The scores are binned linearly in value between their minimum and maximum (kBinFine bins,
// bin 0 at the top, grouped into 32 coarse bins of 32). The map is monotone and deterministic,
// so every key of a higher bin is larger than every key of a lower bin, and equal keys share a
// bin. Every warp finds the fine bin F of the k-th largest key from the histograms on its own
// (a scan of the coarse bins, then of the 32 fine bins of the chosen one). When all of F's keys
// are needed -- with about one key per fine bin, nearly always -- the rule "bin <= F" selects the
// k largest. Otherwise F's keys are ranked exactly by (key desc, index asc) and the k-th one
// (key, index) decides: a page is taken iff its key is larger, or equal with an index not above.
// The result equals block_topk_ascending's (k largest, ties -> lower index, ascending).
constexpr int kBinFine = 1024;
constexpr int kMaxCand = 256;

struct __align__(16) BinSelectSmem {
  uint32_t fine[kBinFine];     // fine histogram (shared by the warps)
  uint32_t wh[8][32];          // per-warp coarse histograms (one word per thread)
  uint2 cand[kMaxCand];        // (ordered key, page) of the k-th key's fine bin
  uint32_t cnt[4][8];          // per key round and warp: pages taken
  uint32_t wmax[8], wmin[8];   // per-warp range of the ordered keys
  uint2 kth;
  int ncand;
};
static_assert(offsetof(BinSelectSmem, fine) % 16 == 0, "fine alignment");
static_assert(offsetof(BinSelectSmem, cnt) % 16 == 0, "cnt alignment");
static_assert(offsetof(BinSelectSmem, wmax) % 16 == 0, "wmax alignment");
static_assert(offsetof(BinSelectSmem, wmin) % 16 == 0, "wmin alignment");

// Inverse of ordered_key.
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// First phase, fused into whatever produces the keys: each thread passes the max / min of the
// ordered keys it produced (0 / ~0 if none). Records the per-warp range and clears the
// histograms. A barrier must separate it from bin_topk.
__device__ __forceinline__ void bin_select_prepare(uint32_t hi, uint32_t lo, BinSelectSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  hi = __reduce_max_sync(0xffffffffu, hi);
  lo = __reduce_min_sync(0xffffffffu, lo);
  if (lane == 0) {
    sm.wmax[warp] = hi;
    sm.wmin[warp] = lo;
  }
  reinterpret_cast<uint4*>(sm.fine)[tid] = make_uint4(0u, 0u, 0u, 0u);
  (&sm.wh[0][0])[tid] = 0u;
  if (tid == 0) sm.ncand = 0;
}

// k largest of scores[0..n) (1 <= k < n <= 1024 NR), page indices written ascending to
// out[0..k). Thread t reads the pages 1024 r + 4 t + e (r < NR, e < 4) as one float4 per round
// (`scores` 16-byte aligned, padded to a multiple of 4). Returns false, with nothing written
// and every thread agreeing, when the scores' range is not a normal finite
// positive number (NaN, infinities, all equal) or the k-th key's fine bin holds more than
// kMaxCand keys: the caller then runs a general select. Ends without a barrier on success.
template <int NR>
__device__ __forceinline__ bool bin_topk(const float* scores, int n, int k, int* out,
                                         BinSelectSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t hi, lo;
  {
    const uint4 a0 = reinterpret_cast<const uint4*>(sm.wmax)[0];
    const uint4 a1 = reinterpret_cast<const uint4*>(sm.wmax)[1];
    const uint4 b0 = reinterpret_cast<const uint4*>(sm.wmin)[0];
    const uint4 b1 = reinterpret_cast<const uint4*>(sm.wmin)[1];
    hi = max(max(max(a0.x, a0.y), max(a0.z, a0.w)), max(max(a1.x, a1.y), max(a1.z, a1.w)));
    lo = min(min(min(b0.x, b0.y), min(b0.z, b0.w)), min(min(b1.x, b1.y), min(b1.z, b1.w)));
  }
  const float smax = key_value(hi), smin = key_value(lo);
  const float range = smax - smin;
  if (!(range >= 1e-30f) || !(range <= 3.0e38f)) return false;
  const float inv = (float)kBinFine / range;
  float f[NR][4];
  bool v[NR][4];
  int fb[NR][4];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int p0 = 1024 * r + 4 * tid;
    const float4 x = p0 < n ? reinterpret_cast<const float4*>(scores)[256 * r + tid]
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    f[r][0] = x.x;
    f[r][1] = x.y;
    f[r][2] = x.z;
    f[r][3] = x.w;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[r][e] = p0 + e < n;
      fb[r][e] = min(kBinFine - 1, (int)((smax - f[r][e]) * inv));
      if (v[r][e]) {
        atomicAdd(&sm.fine[fb[r][e]], 1u);
        atomicAdd(&sm.wh[warp][fb[r][e] >> 5], 1u);
      }
    }
  }
  __syncthreads();
  // every warp: the coarse bin C of the k-th key (lane l = coarse bin l, from the top), then
  // the fine bin F inside it (lane l = fine bin 32 C + l)
  int c = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) c += (int)sm.wh[w][lane];
  int incl = warp_incl_scan(c);
  uint32_t b = __ballot_sync(0xffffffffu, incl >= k);
  const int C = __ffs(b) - 1;
  const int above_c = __shfl_sync(0xffffffffu, incl - c, C);
  const int cf = (int)sm.fine[32 * C + lane];
  incl = warp_incl_scan(cf) + above_c;
  b = __ballot_sync(0xffffffffu, incl >= k);
  const int fl = __ffs(b) - 1;
  const int F = 32 * C + fl;
  const int above = __shfl_sync(0xffffffffu, incl - cf, fl);
  const int nF = __shfl_sync(0xffffffffu, cf, fl);
  const int remaining = k - above;  // 1 .. nF keys of bin F are taken
  uint2 kth = make_uint2(0u, 0u);
  const bool whole = nF == remaining;
  if (!whole && nF > kMaxCand) return false;
  if (!whole) {
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (v[r][e] && fb[r][e] == F) {
          const int slot = atomicAdd(&sm.ncand, 1);
          sm.cand[slot] = make_uint2(ordered_key(f[r][e]), (uint32_t)(1024 * r + 4 * tid + e));
        }
    __syncthreads();
    if (tid < nF) {
      const uint2 me = sm.cand[tid];
      int rank = 0;
#pragma unroll 4
      for (int j = 0; j < nF; ++j) {
        const uint2 o = sm.cand[j];
        rank += (o.x > me.x || (o.x == me.x && o.y < me.y)) ? 1 : 0;
      }
      if (rank == remaining - 1) sm.kth = me;  // ranks are a permutation: exactly one writer
    }
    __syncthreads();
    kth = sm.kth;
  }
  // compaction in page order: (round, thread, e) is ascending
  const uint32_t lt = (1u << lane) - 1u;
  bool t[NR][4];
  int pre[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    int cr = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t pg = (uint32_t)(1024 * r + 4 * tid + e);
      bool take;
      if (whole) {
        take = fb[r][e] <= F;
      } else {
        const uint32_t key = ordered_key(f[r][e]);
        take = fb[r][e] < F ||
               (fb[r][e] == F && (key > kth.x || (key == kth.x && pg <= kth.y)));
      }
      t[r][e] = v[r][e] && take;
      cr += t[r][e] ? 1 : 0;
    }
    const uint32_t g0 = __ballot_sync(0xffffffffu, cr & 1);
    const uint32_t g1 = __ballot_sync(0xffffffffu, cr & 2);
    const uint32_t g2 = __ballot_sync(0xffffffffu, cr & 4);
    pre[r] = __popc(g0 & lt) + 2 * __popc(g1 & lt) + 4 * __popc(g2 & lt);
    if (lane == 0) sm.cnt[r][warp] = __popc(g0) + 2 * __popc(g1) + 4 * __popc(g2);
  }
  __syncthreads();
  int base = 0;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const uint4 c0 = reinterpret_cast<const uint4*>(sm.cnt[r])[0];
    const uint4 c1 = reinterpret_cast<const uint4*>(sm.cnt[r])[1];
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint32_t before = 0u, all = 0u;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      before += (w < warp) ? cw[w] : 0u;
      all += cw[w];
    }
    int pos = base + (int)before + pre[r];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (t[r][e]) out[pos++] = 1024 * r + 4 * tid + e;
    base += (int)all;
  }
  return true;
}

}  // namespace rkv
