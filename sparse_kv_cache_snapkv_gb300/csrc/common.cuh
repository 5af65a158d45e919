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

// Exclusive scan over the block (blockDim.x threads, multiple of 32). `tmp` holds >= 33 ints.
// Returns the exclusive prefix; *total receives the block sum. Contains __syncthreads().
__device__ __forceinline__ int block_excl_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = warp_incl_scan(v);
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? tmp[lane] : 0;
    int wi = warp_incl_scan(w);
    if (lane < nw) tmp[lane] = wi - w;
    if (lane == 31) tmp[32] = wi;
  }
  __syncthreads();
  int r = tmp[warp] + incl - v;
  *total = tmp[32];
  __syncthreads();
  return r;
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

struct SelectScratch {
  uint32_t hist[256];
  int tmp[33];
  uint32_t digit;
  int above;
};

// Choose the k largest of keys[0..n) (ties -> lower index) and write their indices, ascending,
// to out[0..k). keys may live in shared or global memory. 1 <= k <= n. Every thread of the
// block must call it. Returns the number written (== k unless something is badly wrong).
__device__ __noinline__ static int block_topk_ascending(const float* keys, int n, int k, int* out,
                                    SelectScratch& sc) {
  const int tid = threadIdx.x, nt = blockDim.x;
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nt) sc.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += nt) {
      const uint32_t u = ordered_key(keys[i]);
      if ((u & mask) == prefix) atomicAdd(&sc.hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      int cnt[8];
      int s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = (int)sc.hist[255 - 8 * tid - j];
        s += cnt[j];
      }
      const int incl = warp_incl_scan(s);
      const int excl = incl - s;
      // the bin holding the `remaining`-th largest lies in the lane whose range crosses it
      if (excl < remaining && incl >= remaining) {
        int acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + cnt[j] >= remaining) {
            sc.digit = (uint32_t)(255 - 8 * tid - j);
            sc.above = acc;
            break;
          }
          acc += cnt[j];
        }
      }
    }
    __syncthreads();
    prefix |= sc.digit << shift;
    mask |= 255u << shift;
    remaining -= sc.above;
    __syncthreads();
  }
  const uint32_t T = prefix;       // ordered key of the k-th largest
  const int need_eq = remaining;   // how many keys equal to T are taken (lowest indices)

  const int per = (n + nt - 1) / nt;
  const int beg = min(n, tid * per), end = min(n, beg + per);
  int gt = 0, eq = 0;
  for (int i = beg; i < end; ++i) {
    const uint32_t u = ordered_key(keys[i]);
    gt += (u > T);
    eq += (u == T);
  }
  int total;
  const int eq_before = block_excl_scan(eq, sc.tmp, &total);
  const int take_eq = max(0, min(eq, need_eq - eq_before));
  const int pos0 = block_excl_scan(gt + take_eq, sc.tmp, &total);
  int pos = pos0, eq_seen = 0;
  for (int i = beg; i < end; ++i) {
    const uint32_t u = ordered_key(keys[i]);
    bool sel = u > T;
    if (u == T) {
      sel = eq_seen < take_eq;
      ++eq_seen;
    }
    if (sel) {
      if (pos < k) out[pos] = i;
      ++pos;
    }
  }
  return total;
}

}  // namespace rkv
