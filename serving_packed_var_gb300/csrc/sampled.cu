// sampled.cu -- temperature-sampled verification of packed draft blocks.
//
// The target verifies the drafted tokens in parallel (AdaFlash article, "AdaFlash:
// Adaptive Speculative Decoding with Online Self-Improvement for High-Concurrency
// LLM Inference", opening section); the temperature is a tunable of the method
// (skill card "Adaflash Adaptive Speculative Decoding", "Implementation Steps").
// With p = softmax(z/T) and q = softmax(t/T) the rule is speculative sampling:
//
//   token j is accepted when u_j p(x_j) < q(x_j);
//   at the first rejection the emitted token is drawn from max(0, q - p) (q when
//   that is all zero); when all are accepted it is drawn from q at the bonus row;
//   a draw with uniform w is the smallest v whose prefix sum exceeds w * total.
//
// Two kernels:
//   S1 computes log-sum-exp(x / T) of every draft row and every target row, one
//      read of each logit.  A cluster of C CTAs shares a row (each a slice of its
//      8-entry groups); the partial (max, sum) pairs meet in CTA 0's shared memory.
//   S2 is one cluster of 8 CTAs per request, launched as a programmatic dependent
//      of S1: warp 0 applies the accept rule (k <= 16 lanes), then the cluster
//      draws the emitted token (fixed-order sums over one contiguous segment per
//      warp, CTA sums exchanged through distributed shared memory, and the warp
//      whose segment holds the threshold walks it).
#include <climits>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace adaflash {

namespace {

// S1: 256-thread CTAs with eight 16-byte loads in flight per thread, four resident
// CTAs per SM; a row is split over a cluster of up to 8 CTAs while there are fewer
// than 1.7 CTAs per SM (lse_cluster_size).  S2: 256-thread CTAs, eight resident per
// SM, so that 8 x 152 CTAs hold every request of a 128-request batch at once.
constexpr int kLseThreads = 256;
constexpr int kLseUnroll = 8;  // 16-byte loads in flight per thread
constexpr int kLseMinBlocks = 4;
constexpr int kLseCtasPerSmX10 = 17;  // 1.7 CTAs per SM
constexpr int kDrawMinBlocks = 8;
constexpr int kLseMaxCluster = 8;
constexpr int kDrawThreads = 256;  // per CTA
constexpr int kDrawCluster = 8;    // CTAs per request

// (max, sum of 2^{(x - max) * scale}); entries equal to -inf contribute nothing.
struct MaxSum {
  float m, s;
};

__device__ __forceinline__ void ms_add(MaxSum& a, float x, float scale) {
  if (x == kNegInf) return;
  if (x > a.m) {
    a.s = a.s * ex2((a.m - x) * scale);
    a.m = x;
  }
  a.s += ex2((x - a.m) * scale);
}

// E values at once: one rescale for the group's maximum, then E exponentials.
template <int E>
__device__ __forceinline__ void ms_add_group(MaxSum& a, const float (&x)[E], float scale) {
  float m = x[0];
#pragma unroll
  for (int e = 1; e < E; ++e) m = fmaxf(m, x[e]);
  if (m > a.m) {
    a.s = a.s * ex2((a.m - m) * scale);
    a.m = m;
  }
  if (a.m == kNegInf) return;
  float g = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) g += ex2((x[e] - a.m) * scale);
  a.s += g;
}

__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b, float scale) {
  const float m = fmaxf(a.m, b.m);
  if (m == kNegInf) return a;
  const float fa = (a.m == kNegInf) ? 0.f : ex2((a.m - m) * scale);
  const float fb = (b.m == kNegInf) ? 0.f : ex2((b.m - m) * scale);
  return MaxSum{m, a.s * fa + b.s * fb};
}

// Unpacks one 16-byte word into 4 (fp32) or 8 (bf16) values.
__device__ __forceinline__ void unpack16(const uint4& w, float (&x)[4]) {
  x[0] = __uint_as_float(w.x);
  x[1] = __uint_as_float(w.y);
  x[2] = __uint_as_float(w.z);
  x[3] = __uint_as_float(w.w);
}
__device__ __forceinline__ void unpack16(const uint4& w, float (&x)[8]) {
  x[0] = bf16_lo(w.x);
  x[1] = bf16_hi(w.x);
  x[2] = bf16_lo(w.y);
  x[3] = bf16_hi(w.y);
  x[4] = bf16_lo(w.z);
  x[5] = bf16_hi(w.z);
  x[6] = bf16_lo(w.w);
  x[7] = bf16_hi(w.w);
}

// Eight consecutive entries starting at v0 (a multiple of 8); 16-byte loads when
// the row starts on a 16-byte boundary, else eight element loads (the few groups
// left after the unrolled loops, and the draw's re-reads).
template <class DT>
__device__ __forceinline__ void load8(const uint8_t* row, bool aligned16, int v0, float (&x)[8]) {
  if (!aligned16) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = DT::load(row, v0 + e);
    return;
  }
  const uint4* p = reinterpret_cast<const uint4*>(row + static_cast<int64_t>(v0) * DT::kBytes);
  if constexpr (DT::kBytes == 2) {
    unpack16(__ldg(p), x);
  } else {
    float lo[4], hi[4];
    unpack16(__ldg(p), lo);
    unpack16(__ldg(p + 1), hi);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] = lo[e];
      x[4 + e] = hi[e];
    }
  }
}

// (max, sum) of slice `rank` of `C` of one row, reduced over the CTA (red holds
// 2 * 32 floats); the result is valid in every thread.  The row is cut into groups
// of 8 entries (C contiguous slices of groups) and a tail of V mod 8 entries (rank
// C - 1).  The order of operations depends only on V and C, not on the element
// type or the row's alignment, so rows holding equal values give equal results.
template <class DT>
__device__ MaxSum slice_maxsum(const uint8_t* row, int V, int rank, int C, float scale, float* red) {
  const int B = static_cast<int>(blockDim.x);
  const int tid = static_cast<int>(threadIdx.x);
  const bool a16 = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int ng = V >> 3;
  const int per = (ng + C - 1) / C;
  const int g0 = min(ng, rank * per), g1 = min(ng, g0 + per);
  MaxSum a{kNegInf, 0.f};
  int g = g0 + tid;
  if (a16) {
    // 16-byte words loaded first, unpacked as they are consumed
    constexpr int W = DT::kBytes / 2;                    // words per 8-entry group
    constexpr int U = kLseUnroll * 2 / DT::kBytes > 0 ? kLseUnroll * 2 / DT::kBytes : 1;  // same bytes in flight
    const uint4* rw = reinterpret_cast<const uint4*>(row);
    for (; g + (U - 1) * B < g1; g += U * B) {
      uint4 raw[U][W];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int q = 0; q < W; ++q) raw[u][q] = __ldcs(rw + static_cast<int64_t>(g + u * B) * W + q);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float x[8];
        if constexpr (W == 1) {
          unpack16(raw[u][0], x);
        } else {
          float lo[4], hi[4];
          unpack16(raw[u][0], lo);
          unpack16(raw[u][W - 1], hi);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[e] = lo[e];
            x[4 + e] = hi[e];
          }
        }
        ms_add_group<8>(a, x, scale);
      }
    }
  } else {
    // rows off the 16-byte grid: the same groups (so the same order of operations),
    // each read with the widest aligned loads at the row's byte shift, one loop
    // instance per shift, several groups in flight per thread
    const int zs2 = static_cast<int>((reinterpret_cast<uintptr_t>(row) & 15u) >> 1);
    dispatch_shift<DT>(zs2, [&](auto zs_c) {
      constexpr int ZS = decltype(zs_c)::value;
      constexpr int U = DT::kBytes == 2 ? 4 : 2;
      const uint32_t* base = reinterpret_cast<const uint32_t*>(row - 2 * ZS);  // the 16-byte boundary below
      for (; g + (U - 1) * B < g1; g += U * B) {
        float x[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u)
          load8_shifted<DT, ZS, true>(base + static_cast<int64_t>(g + u * B) * 2 * DT::kBytes, x[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) ms_add_group<8>(a, x[u], scale);
      }
    });
  }
  for (; g < g1; g += B) {
    float x[8];
    load8<DT>(row, a16, g << 3, x);
    ms_add_group<8>(a, x, scale);
  }
  if (rank == C - 1)
    for (int v = (ng << 3) + tid; v < V; v += B) ms_add(a, DT::load(row, v), scale);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    MaxSum b{__shfl_xor_sync(0xffffffffu, a.m, off), __shfl_xor_sync(0xffffffffu, a.s, off)};
    a = ms_merge(a, b, scale);
  }
  const int warp = tid >> 5, lane = tid & 31, nw = B >> 5;
  if (lane == 0) {
    red[warp] = a.m;
    red[32 + warp] = a.s;
  }
  __syncthreads();
  MaxSum t{kNegInf, 0.f};
  for (int w = 0; w < nw; ++w) t = ms_merge(t, MaxSum{red[w], red[32 + w]}, scale);
  return t;
}

// One 8-entry group from its 16-byte words (1 for bf16, 2 for fp32).
template <class DT>
__device__ __forceinline__ void unpack_group(const uint4* raw, float (&x)[8]) {
  if constexpr (DT::kBytes == 2) {
    unpack16(raw[0], x);
  } else {
    float lo[4], hi[4];
    unpack16(raw[0], lo);
    unpack16(raw[1], hi);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] = lo[e];
      x[4 + e] = hi[e];
    }
  }
}

// p = exp(x / T - lse) for one entry.
__device__ __forceinline__ float prob_at(float x, float inv_t, float lse) {
  return ex2(fmaf(x, inv_t, -lse) * kLog2e);
}

__device__ __forceinline__ bool is_aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

// ---- S1: log-sum-exp at temperature of every draft row and every target row ----
template <class DZ, class DT>
__global__ void __launch_bounds__(kLseThreads, kLseMinBlocks) lse_rows_kernel(const SampledParams P, int C) {
  __shared__ float red[64];
  __shared__ float part[2 * kLseMaxCluster];
  // S1 is a programmatic dependent of whatever the stream ran before it: nothing in
  // global memory is touched before that grid has completed.  Then S2 may be
  // scheduled; it waits for S1's results.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = static_cast<int>(blockIdx.x) / C;
  const int rank = static_cast<int>(blockIdx.x) % C;  // == %cluster_ctarank for a 1-D cluster of C
  const float scale = kLog2e * P.inv_t;
  MaxSum ms;
  if (b < P.N_d) {
    ms = slice_maxsum<DZ>(static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(b) * P.ld_z * DZ::kBytes, P.V,
                          rank, C, scale, red);
  } else {
    ms = slice_maxsum<DT>(static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(b - P.N_d) * P.ld_t * DT::kBytes,
                          P.V, rank, C, scale, red);
  }
  if (C == 1) {
    if (threadIdx.x == 0) P.row_lse[b] = ms.m * P.inv_t + logf(ms.s);  // lse = m / T + ln(s)
    return;
  }
  if (threadIdx.x == 0) {
    float* dst = map_to_rank(part, 0u);
    dst[2 * rank] = ms.m;
    dst[2 * rank + 1] = ms.s;
  }
  cluster_sync_all();
  if (rank == 0 && threadIdx.x == 0) {
    MaxSum t{kNegInf, 0.f};
    for (int r = 0; r < C; ++r) t = ms_merge(t, MaxSum{part[2 * r], part[2 * r + 1]}, scale);
    P.row_lse[b] = t.m * P.inv_t + logf(t.s);
  }
}

// ---- S2: the accept rule and the draw, one cluster of kDrawCluster CTAs per request ----
//
// The vocabulary is cut into one contiguous segment per warp of the cluster, each a
// whole number of tiles of 32 x 8 entries (lane l of a tile holds entries 8l..8l+7,
// so every load instruction of a warp reads consecutive 16-byte words).  The warp
// sums give, in vocabulary order, each warp's prefix; the owner warp stages its
// segment's weights in shared memory and walks it tile by tile.
template <class DZ, class DT>
__global__ void __launch_bounds__(kDrawThreads, kDrawMinBlocks) sampled_draw_kernel(const SampledParams P,
                                                                                              int seg_tiles) {
  extern __shared__ float wbuf[];  // seg_tiles * 256 weights of the owner warp's segment
  __shared__ float scan[kDrawThreads / 32];
  __shared__ float ctot[2][kDrawCluster];  // per pass: every CTA's sum, written into every CTA
  __shared__ int cown[kDrawCluster];       // every CTA's last candidate warp (or -1)
  __shared__ int s_L, s_owner;
  __shared__ float s_lse[2 * (ADAFLASH_MAX_K + 1)];  // lse of draft row d0+j and target row d0+i+j
  const int i = static_cast<int>(blockIdx.x) / kDrawCluster;
  const int rank = static_cast<int>(blockIdx.x) % kDrawCluster;  // == %cluster_ctarank
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d0 = __ldg(P.doff + i), d1 = __ldg(P.doff + i + 1);
  const int k = d1 - d0;
  const float inv_t = P.inv_t;
  bool ok = (k >= 1) && (k <= ADAFLASH_MAX_K) && (d0 >= 0) && (d1 <= P.N_d);
  if (i == 0 && d0 != 0) ok = false;
  if (i == P.R - 1 && d1 != P.N_d) ok = false;

  // The accept rule, evaluated by warp 0 of every CTA of the cluster (identical
  // inputs and instructions, so identical L); CTA 0 writes the outputs.  The
  // inputs it reads are fetched before waiting for S1, whose row_lse it then needs.
  const int d = d0 + lane, s = d0 + i + lane;
  const bool mine = (warp == 0) && ok && (lane < k);
  bool badtok = false;
  float zx = 0.f, tx = 0.f, ua = 0.f;
  if (mine) {
    const int x = __ldg(P.tokens + d);
    badtok = (x < 0) || (x >= P.V);
    if (!badtok) {
      zx = DZ::load(static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(d) * P.ld_z * DZ::kBytes, x);
      tx = DT::load(static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(s) * P.ld_t * DT::kBytes, x);
    }
    ua = __ldg(P.u_accept + d);
  }
  const float w = fminf(fmaxf(__ldg(P.u_sample + i), 0.f), 1.f);  // NaN -> 0
  asm volatile("griddepcontrol.wait;" ::: "memory");  // row_lse comes from S1
  // the next call's S1 may be scheduled now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0) {
    if (!ok) {
      if (lane == 0) {
        if (rank == 0) {
          P.accept_len[i] = -1;
          P.next_token[i] = -1;
          P.accept_rate[i] = -1.f;
          flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
        }
        s_L = -1;
      }
    } else {
      bool reject = badtok;
      // lanes j < k hold the lse of the pair at position j, lane k that of the bonus row
      const float lz = mine ? P.row_lse[d] : 0.f;
      const float lt = (lane <= k) ? P.row_lse[P.N_d + s] : 0.f;
      if (lane <= k) {
        s_lse[2 * lane] = lz;
        s_lse[2 * lane + 1] = lt;
      }
      if (mine && !badtok) reject = !(ua * prob_at(zx, inv_t, lz) < prob_at(tx, inv_t, lt));
      const unsigned rj = __ballot_sync(0xffffffffu, reject);
      const unsigned bt = __ballot_sync(0xffffffffu, badtok);
      if (lane == 0) {
        const int L = rj ? (__ffs(rj) - 1) : k;
        if (rank == 0) {
          P.accept_len[i] = L;
          P.accept_rate[i] = __fdiv_rn(static_cast<float>(L), static_cast<float>(k));
          if (bt) flag_status(P.status, ADAFLASH_ERR_BAD_TOKEN);
        }
        s_L = L;
      }
    }
  }
  __syncthreads();
  const int L = s_L;
  if (L < 0) return;  // malformed request: the whole cluster leaves before any cluster barrier

  const int V = P.V;
  // L < k: residual max(0, q - p) at the first rejected position; L = k: q at the bonus row
  int mode = (L < k) ? 0 : 1;
  const int dz = d0 + min(L, k - 1);  // draft row of the rejected position (unused when mode = 1)
  const int st = d0 + i + L;          // target row of the emitted position
  const uint8_t* zrow = static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(dz) * P.ld_z * DZ::kBytes;
  const uint8_t* trow = static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(st) * P.ld_t * DT::kBytes;
  const bool z16 = is_aligned16(zrow), t16 = is_aligned16(trow);
  const float lse_z = s_lse[2 * min(L, k - 1)];
  const float lse_t = s_lse[2 * L + 1];
  const int seg = seg_tiles * 256;                     // entries per warp segment
  const int gw = rank * (kDrawThreads / 32) + warp;    // warp index in vocabulary order
  const int s0 = min(V, gw * seg), s1 = min(V, s0 + seg);
  const int full_groups = V >> 3;                      // groups with all 8 entries in range

  auto weight_of = [&](float tv, float zv, int md) -> float {
    const float q = prob_at(tv, inv_t, lse_t);
    if (md == 1) return q;
    return fmaxf(q - prob_at(zv, inv_t, lse_z), 0.f);
  };
  // the 8 weights of group g (entries 8g .. 8g+7; those >= V weigh 0)
  auto group_weights = [&](int g, int md, float (&wv)[8]) {
    float tv[8], zv[8];
    if (g < full_groups) {
      load8<DT>(trow, t16, g << 3, tv);
      if (md == 0) {
        load8<DZ>(zrow, z16, g << 3, zv);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) zv[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) wv[e] = weight_of(tv[e], zv[e], md);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int v = (g << 3) + e;
        wv[e] = (v < V) ? weight_of(DT::load(trow, v), md == 0 ? DZ::load(zrow, v) : 0.f, md) : 0.f;
      }
    }
  };

  for (int pass = 0; pass < 2; ++pass) {
    // this lane's share of the warp segment: group lane of every tile, in order
    float own = 0.f;
    const int g0 = s0 >> 3, g1 = (s1 > s0) ? (s1 + 7) >> 3 : g0;  // an empty segment has no groups
    int g = g0 + lane;
    if (t16 && (mode == 1 || z16)) {
      // on the 16-byte grid: the words of several tiles issued before any is used
      constexpr int WT = DT::kBytes / 2, WZ = DZ::kBytes / 2;
      constexpr int U = 8 / (WT + WZ);  // tiles per round
      const uint4* tw = reinterpret_cast<const uint4*>(trow);
      const uint4* zw = reinterpret_cast<const uint4*>(zrow);
      for (; g + 32 * (U - 1) < min(g1, full_groups); g += 32 * U) {
        uint4 rt[U][WT], rz[U][WZ];
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
          for (int q = 0; q < WT; ++q) rt[u][q] = __ldg(tw + static_cast<int64_t>(g + 32 * u) * WT + q);
#pragma unroll
          for (int q = 0; q < WZ; ++q)
            rz[u][q] = (mode == 0) ? __ldg(zw + static_cast<int64_t>(g + 32 * u) * WZ + q) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float tv[8], zv[8];
          unpack_group<DT>(rt[u], tv);
          unpack_group<DZ>(rz[u], zv);
#pragma unroll
          for (int e = 0; e < 8; ++e) own += weight_of(tv[e], zv[e], mode);
        }
      }
    }
    for (; g < g1; g += 32) {
      float wv[8];
      group_weights(g, mode, wv);
#pragma unroll
      for (int e = 0; e < 8; ++e) own += wv[e];
    }
    // warp sum (fixed butterfly order), CTA prefix over warps, cluster prefix over CTAs
    float wsum = own;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    if (lane == 0) scan[warp] = wsum;
    __syncthreads();
    float before_w = 0.f, cta_total = 0.f;
    for (int ww = 0; ww < kDrawThreads / 32; ++ww) {
      if (ww < warp) before_w += scan[ww];
      cta_total += scan[ww];
    }
    if (tid < kDrawCluster) *map_to_rank(&ctot[pass][rank], static_cast<uint32_t>(tid)) = cta_total;
    cluster_sync_all();
    float before_c = 0.f, total = 0.f;
    for (int r = 0; r < kDrawCluster; ++r) {
      if (r < rank) before_c += ctot[pass][r];
      total += ctot[pass][r];
    }
    const float excl = before_c + before_w;  // this warp's prefix
    if (total > 0.f || mode == 1) {
      const float target = w * total;
      // The owner is the last warp (in vocabulary order) with positive mass whose
      // prefix does not pass the threshold.  The first such warp has prefix exactly
      // 0, so one exists whenever total > 0 whatever the rounding.
      if (tid == 0) s_owner = -1;
      __syncthreads();
      if (lane == 0 && wsum > 0.f && (excl <= target || !(target < total))) atomicMax(&s_owner, warp);
      __syncthreads();
      if (tid < kDrawCluster) *map_to_rank(&cown[rank], static_cast<uint32_t>(tid)) = s_owner;
      cluster_sync_all();  // the last cluster barrier: no remote writes after it
      int orank = -1;
      for (int r = 0; r < kDrawCluster; ++r)
        if (cown[r] >= 0) orank = r;
      if (orank < 0) {
        if (rank == 0 && tid == 0) P.next_token[i] = -1;  // no mass at all (non-finite logits)
      } else if (rank == orank) {
        // every warp of the owner CTA stages tiles of the owner warp's segment (coalesced);
        // the owner warp then walks it tile by tile: lane sums of 8 entries, a warp scan,
        // and the first lane whose running sum passes the threshold resolves within its
        // 8 entries
        const int ow = cown[orank];
        const int gwo = rank * (kDrawThreads / 32) + ow;
        const int s0o = min(V, gwo * seg), s1o = min(V, s0o + seg);
        const int ntiles = (s1o - s0o + 255) >> 8;
        for (int t = warp; t < ntiles; t += kDrawThreads / 32) {
          float wv[8];
          group_weights((s0o >> 3) + 32 * t + lane, mode, wv);
#pragma unroll
          for (int e = 0; e < 8; ++e) wbuf[(t << 8) + (lane << 3) + e] = wv[e];
        }
        __syncthreads();  // this CTA only: the owner CTA's warps all take this branch
        if (warp == ow) {
          float base = excl;
          int pick = -1, lastpos = -1;
          for (int t = 0; t < ntiles && pick < 0; ++t) {
            const float* tw8 = wbuf + (t << 8) + (lane << 3);
            float ls = 0.f;
            int lp = -1;
  #pragma unroll
            for (int e = 0; e < 8; ++e) {
              ls += tw8[e];
              if (tw8[e] > 0.f) lp = (t << 8) + (lane << 3) + e;
            }
            float inc = ls;
  #pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
              const float y = __shfl_up_sync(0xffffffffu, inc, off);
              if (lane >= off) inc += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, base + inc > target);
            if (hit) {
              const int hl = __ffs(hit) - 1;
              int pk = -1;
              if (lane == hl) {
                float acc = base + inc - ls;
                for (int e = 0; e < 8; ++e) {
                  acc += tw8[e];
                  if (acc > target) {
                    pk = (t << 8) + (lane << 3) + e;
                    break;
                  }
                }
                if (pk < 0) pk = lp;
              }
              pk = __shfl_sync(0xffffffffu, pk, hl);
              // a run with no positive entry: the last positive one before it
              const unsigned pos = __ballot_sync(0xffffffffu, lp >= 0) & (0xffffffffu >> (31 - hl));
              if (pk < 0 && pos) pk = __shfl_sync(0xffffffffu, lp, 31 - __clz(pos));
              if (pk < 0) pk = lastpos;
              pick = pk;
            } else {
              const unsigned pos = __ballot_sync(0xffffffffu, lp >= 0);
              if (pos) lastpos = __shfl_sync(0xffffffffu, lp, 31 - __clz(pos));
              base += __shfl_sync(0xffffffffu, inc, 31);
            }
          }
          if (pick < 0) pick = lastpos;  // the threshold lies past every partial sum
          if (lane == 0) P.next_token[i] = s0 + max(pick, 0);
        }
      }
      break;
    }
    // residual of identical distributions is all zero (the same verdict in every
    // CTA): draw from q instead
    mode = 1;
    __syncthreads();  // scan[] is rewritten by the next pass
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// S1 splits each row over the fewest CTAs that give 1.7 CTAs per SM (at most 8).
// Measured on GB300, k = 16 per request at V = 151936, bf16, us per sampled call (the
// earlier rule, doubling C up to 12 rows per SM, in brackets): one request C = 8 14.4
// graph-replayed (the same); 2 requests C = 4 16.4 (18.4); 4 requests C = 2 24.0
// (26.5); 8 requests C = 1 27.6 eager (33.6); 16 requests C = 1 45.6 (48.7); 32
// requests C = 1 67.9 (71.4).
static int lse_cluster_size(int rows, int num_sms) {
  const int64_t want = (static_cast<int64_t>(kLseCtasPerSmX10) * num_sms + 9) / 10;  // CTAs, rounded up
  const int64_t c = (want + rows - 1) / rows;
  return static_cast<int>(c < 1 ? 1 : (c > kLseMaxCluster ? kLseMaxCluster : c));
}

template <class DZ, class DT>
static cudaError_t launch_sampled_t(const SampledParams& p, int num_sms, cudaStream_t s) {
  if (p.R <= 0) return cudaSuccess;
  const int rows = p.N_d + p.N_t;
  const int C = lse_cluster_size(rows, num_sms);
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows * C));
    cfg.blockDim = dim3(kLseThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    count_launch();
    const cudaError_t e = cudaLaunchKernelEx(&cfg, lse_rows_kernel<DZ, DT>, p, C);
    if (e != cudaSuccess) return e;
  }
  const int warps = kDrawCluster * (kDrawThreads / 32);
  const int seg_tiles = ((p.V + 255) / 256 + warps - 1) / warps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.R * kDrawCluster));
  cfg.blockDim = dim3(kDrawThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(seg_tiles) * 256 * sizeof(float);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kDrawCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, sampled_draw_kernel<DZ, DT>, p, seg_tiles);
}

cudaError_t launch_sampled(const SampledParams& p, int z_dtype, int t_dtype, int num_sms, cudaStream_t s) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (zb && tb) return launch_sampled_t<BF16, BF16>(p, num_sms, s);
  if (!zb && tb) return launch_sampled_t<F32, BF16>(p, num_sms, s);
  if (zb && !tb) return launch_sampled_t<BF16, F32>(p, num_sms, s);
  return launch_sampled_t<F32, F32>(p, num_sms, s);
}

}  // namespace adaflash
