// common.cuh -- device helpers shared by the kernels of the packed verify + OPD pass.
//
// Hand-written for sm_103a (GB300): bfloat16 unpacking, the MUFU base-2 exponential,
// mbarrier / bulk-copy (TMA engine) wrappers with bounded waits, cluster barriers,
// and the per-entry term of the clipped reverse KL that the forward screen and the
// backward both evaluate with the same instruction sequence.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/adaflash.h"

namespace adaflash {

// log2(e) as a float; exponentials are computed as 2^(x * log2 e).
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------------------
// status bits
// ---------------------------------------------------------------------------
__device__ __forceinline__ void flag_status(uint32_t* status, int code) {
  if (status) atomicOr(status, 1u << code);
}

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
struct F32 {
  using T = float;
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static float load(const void* base, int64_t i) {
    return __ldg(reinterpret_cast<const float*>(base) + i);
  }
};
struct BF16 {
  using T = uint16_t;
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static float load(const void* base, int64_t i) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(base) + i);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x on the MUFU unit (flush-to-zero; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// the per-entry term of the clipped reverse KL
// ---------------------------------------------------------------------------
// p_v = exp(z_v - lse_z), r_v = (z_v - t_v) - (lse_z - lse_t), term_v = p_v r_v.
// Written with explicit round-to-nearest intrinsics so that the forward's clip
// screen and the backward reach the same clip decision bit for bit.
struct TermConsts {
  float neg_lse_z_l2e;  // -lse_z * log2 e
  float dlse;           // lse_z - lse_t (float32 difference of the stored values)
};

__device__ __forceinline__ TermConsts make_term_consts(float lse_z, float lse_t) {
  TermConsts c;
  c.neg_lse_z_l2e = __fmul_rn(-lse_z, kLog2e);
  c.dlse = __fsub_rn(lse_z, lse_t);
  return c;
}

__device__ __forceinline__ void entry_term(float z, float t, const TermConsts& k, float& p, float& r,
                                           float& term) {
  p = ex2(__fmaf_rn(z, kLog2e, k.neg_lse_z_l2e));
  r = __fsub_rn(__fsub_rn(z, t), k.dlse);
  term = __fmul_rn(p, r);
}

// ---------------------------------------------------------------------------
// time, mbarriers, bulk copies, cluster barriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy and the cluster.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One test of phase `parity`; a thread whose phase is not complete is suspended
// for up to hint_ns (it wakes as soon as the phase completes), so waiting threads
// do not spin on the issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 1000000u) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after limit_ns.
// Returns false on timeout; the caller reports ADAFLASH_ERR_TIMEOUT.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t hint = limit_ns < 1000000ull ? static_cast<uint32_t>(limit_ns) : 1000000u;
  if (mbar_try_wait(bar, parity, hint)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity, hint)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// One-dimensional bulk copy global -> this CTA's shared memory on the TMA engine;
// completion is signalled as transaction bytes on `bar`.  dst, src and bytes must
// be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// L2 eviction priorities for bulk copies: keep (data read again soon) or stream.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_copy_g2s with an L2 eviction-priority policy.
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                   uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  cluster_arrive_release();
  cluster_wait_acquire();
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Generic address of the same shared-memory variable in CTA `rank` of the cluster.
template <typename T>
__device__ __forceinline__ T* map_to_rank(T* local, uint32_t rank) {
  uint64_t out;
  asm volatile("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(local)), "r"(rank));
  return reinterpret_cast<T*>(out);
}

// Request owning draft row d: the largest i in [0, R) with doff[i] <= d.
__device__ __forceinline__ int request_of_row(const int32_t* doff, int R, int d) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(doff + mid) <= d) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace adaflash

namespace adaflash {

// Exact 2^k for integer k <= 127 (0 below the normal range).
__device__ __forceinline__ float pow2i(int k) {
  return k < -126 ? 0.0f : __int_as_float((k + 127) << 23);
}

// Cluster-scope mbarrier helpers (arrive on a peer CTA's barrier; acquire-wait).
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* local_bar, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local_bar)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// Store v (a multiple of 16 bytes, 16-byte aligned) into `local_slot`'s copy in CTA
// `rank` of the cluster with asynchronous stores that report their bytes as
// transactions on that CTA's copy of `local_bar`: the receiver, which expects the
// bytes (mbarrier expect_tx) and waits on its barrier, sees the data with no fence
// on the sending side.
template <class T>
__device__ __forceinline__ void st_async_to_rank(const T& v, T* local_slot, uint64_t* local_bar, uint32_t rank) {
  static_assert(sizeof(T) % 16 == 0 && alignof(T) >= 16, "whole 16-byte words");
  uint32_t dst, bar;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(smem_addr(local_slot)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(bar) : "r"(smem_addr(local_bar)), "r"(rank));
  const uint4* w = reinterpret_cast<const uint4*>(&v);
#pragma unroll
  for (int i = 0; i < static_cast<int>(sizeof(T) / 16); ++i)
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     dst + 16 * i),
                 "r"(w[i].x), "r"(w[i].y), "r"(w[i].z), "r"(w[i].w), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 1000000u) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Warp-wide float max in one instruction (redux.sync, sm_100 family).
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Named barrier over the first `count` threads of the CTA (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync_id(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int count) {
  asm volatile("bar.sync 1, %0;" ::"r"(count) : "memory");
}

}  // namespace adaflash

namespace adaflash {

// Packed pairs of float32 in one 64-bit register (two lanes per instruction on the
// FMA pipe: fma/add/sub .f32x2).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

}  // namespace adaflash
