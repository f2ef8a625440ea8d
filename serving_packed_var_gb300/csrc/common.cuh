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

namespace adaflash {

// ---------------------------------------------------------------------------
// rows off the 16-byte grid
// ---------------------------------------------------------------------------
// A compile-time integer (a row's byte shift against the 16-byte grid, picked per
// row by a uniform switch, so each shift gets its own straight-line loads).
template <int N>
struct IntC {
  static constexpr int value = N;
};

// Words base[P .. P+N) of a 16-byte aligned array, each access the widest aligned
// one (128, 64 or 32 bits): a run that starts P words past a 16-byte boundary.
template <int P, int N>
__device__ __forceinline__ void lds_words(const uint32_t* base, uint32_t* w) {
  if constexpr (N > 0) {
    if constexpr (P % 4 == 0 && N >= 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(base + P);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      lds_words<P + 4, N - 4>(base, w + 4);
    } else if constexpr (P % 2 == 0 && N >= 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(base + P);
      w[0] = v.x; w[1] = v.y;
      lds_words<P + 2, N - 2>(base, w + 2);
    } else {
      w[0] = base[P];
      lds_words<P + 1, N - 1>(base, w + 1);
    }
  }
}

// The same from global memory through the read-only path.
template <int P, int N>
__device__ __forceinline__ void ldg_words(const uint32_t* base, uint32_t* w) {
  if constexpr (N > 0) {
    if constexpr (P % 4 == 0 && N >= 4) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + P));
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      ldg_words<P + 4, N - 4>(base, w + 4);
    } else if constexpr (P % 2 == 0 && N >= 2) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(base + P));
      w[0] = v.x; w[1] = v.y;
      ldg_words<P + 2, N - 2>(base, w + 2);
    } else {
      w[0] = __ldg(base + P);
      ldg_words<P + 1, N - 1>(base, w + 1);
    }
  }
}

// Streaming stores of x[0 .. N) to base[P .. P+N) (base 16-byte aligned), each the
// widest aligned store.
template <int P, int N>
__device__ __forceinline__ void stcs_words(float* base, const float* x) {
  if constexpr (N > 0) {
    if constexpr (P % 4 == 0 && N >= 4) {
      __stcs(reinterpret_cast<float4*>(base + P), make_float4(x[0], x[1], x[2], x[3]));
      stcs_words<P + 4, N - 4>(base, x + 4);
    } else if constexpr (P % 2 == 0 && N >= 2) {
      __stcs(reinterpret_cast<float2*>(base + P), make_float2(x[0], x[1]));
      stcs_words<P + 2, N - 2>(base, x + 2);
    } else {
      __stcs(base + P, x[0]);
      stcs_words<P + 1, N - 1>(base, x + 1);
    }
  }
}

// Eight float32 results to dst (4-byte aligned, q = (dst / 4) mod 4 words past a
// 16-byte boundary; q is uniform across a row, so the branch does not diverge).
// kShift = false: dst is 16-byte aligned (q = 0).
template <bool kShift = true>
__device__ __forceinline__ void store8_stream(float* dst, int q, const float x[8]) {
  if constexpr (!kShift) {
    stcs_words<0, 8>(dst, x);
    return;
  }
  float* base = dst - q;
  switch (q) {
    case 1: stcs_words<1, 8>(base, x); break;
    case 2: stcs_words<2, 8>(base, x); break;
    case 3: stcs_words<3, 8>(base, x); break;
    default: stcs_words<0, 8>(base, x); break;
  }
}

// Eight entries of a row whose group starts ZS two-byte units past a 16-byte
// boundary: words are read with aligned loads (lds_words / ldg_words, picked by
// kGlobal) from `base` (the 16-byte aligned address at or below the group), then
// widened.  ZS is even for float32 rows.  A bfloat16 group at an odd ZS straddles
// five words: its entries are the upper half of word i and the lower half of
// word i + 1.
template <class DT, int ZS, bool kGlobal>
__device__ __forceinline__ void load8_shifted(const uint32_t* base, float x[8]) {
  if constexpr (DT::kBytes == 4) {
    static_assert(ZS % 2 == 0, "float32 rows are 4-byte aligned");
    uint32_t w[8];
    if constexpr (kGlobal) ldg_words<ZS / 2, 8>(base, w); else lds_words<ZS / 2, 8>(base, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(w[i]);
  } else if constexpr (ZS % 2 == 0) {
    uint32_t w[4];
    if constexpr (kGlobal) ldg_words<ZS / 2, 4>(base, w); else lds_words<ZS / 2, 4>(base, w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_lo(w[i]);
      x[2 * i + 1] = bf16_hi(w[i]);
    }
  } else {
    uint32_t w[5];
    if constexpr (kGlobal) ldg_words<(ZS - 1) / 2, 5>(base, w); else lds_words<(ZS - 1) / 2, 5>(base, w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_hi(w[i]);
      x[2 * i + 1] = bf16_lo(w[i + 1]);
    }
  }
}

// Call f(IntC<zs2>{}) for a row's shift zs2 (in two-byte units, 0..7; only even
// shifts occur for float32 rows, so only those are instantiated).  kShift = false:
// every row is on the grid, only the shift-0 instance exists.
template <class DT, bool kShift = true, class F>
__device__ __forceinline__ void dispatch_shift(int zs2, F&& f) {
  if constexpr (!kShift) {
    f(IntC<0>{});
  } else if constexpr (DT::kBytes == 4) {
    switch (zs2) {
      case 2: f(IntC<2>{}); break;
      case 4: f(IntC<4>{}); break;
      case 6: f(IntC<6>{}); break;
      default: f(IntC<0>{}); break;
    }
  } else {
    switch (zs2) {
      case 1: f(IntC<1>{}); break;
      case 2: f(IntC<2>{}); break;
      case 3: f(IntC<3>{}); break;
      case 4: f(IntC<4>{}); break;
      case 5: f(IntC<5>{}); break;
      case 6: f(IntC<6>{}); break;
      case 7: f(IntC<7>{}); break;
      default: f(IntC<0>{}); break;
    }
  }
}

// Geometry of one row pair against the target row's 16-byte grid: the target row's
// first H entries (H < 16 / element bytes) lie before its first 16-byte boundary;
// the body [H, V) is copied in whole 16-byte words.  The draft row's body starts
// 2 * zs2 bytes past a 16-byte boundary (zs2 in 0..7).
struct RowGeom {
  int H;
  int zs2;
  const uint8_t* tb;  // target body (16-byte aligned)
  const uint8_t* zb;  // draft body (may be off the grid), nullptr for a target-only row
};

template <class DZ, class DT, bool kShift = true>
__device__ __forceinline__ RowGeom row_geom(const uint8_t* zrow, const uint8_t* trow, int V) {
  RowGeom g;
  if constexpr (!kShift) {  // every row on the grid
    g.H = 0;
    g.zs2 = 0;
    g.tb = trow;
    g.zb = zrow;
    return g;
  }
  const int off = static_cast<int>(reinterpret_cast<uintptr_t>(trow) & 15u);
  g.H = min(((16 - off) & 15) / DT::kBytes, V);
  g.tb = trow + static_cast<int64_t>(g.H) * DT::kBytes;
  g.zb = zrow ? zrow + static_cast<int64_t>(g.H) * DZ::kBytes : nullptr;
  g.zs2 = zrow ? static_cast<int>((reinterpret_cast<uintptr_t>(g.zb) & 15u) >> 1) : 0;
  return g;
}

}  // namespace adaflash
