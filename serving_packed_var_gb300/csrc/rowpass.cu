// rowpass.cu -- K1: the fused streaming pass over packed logit rows.
//
// One work unit is either a PAIR (draft row d with its target row s) or a
// TARGET-ONLY row (a bonus row, or every row in verification-only mode).  A unit
// is handled by a cluster of C CTAs; CTA rank c owns the vocabulary slice
// [c*slice, (c+1)*slice).  Clusters are persistent: cluster k handles units
// k, k + #clusters, ...  Inside each CTA:
//
//   producer warp   : 1-D bulk copies (TMA engine) of chunks of z and t into a
//                     ring of shared-memory stages (mbarrier-signalled), running
//                     ahead across unit boundaries;
//   8 consumer warps: per 8-entry group, an online log-sum-exp of z and of t,
//                     sum_v e^{z_v}(z_v - t_v), max_v (z_v - t_v), the lowest-
//                     index argmax of t, and the group maximum of z kept in
//                     shared memory as a screening code.
//
// Slice results meet over distributed shared memory (remote stores + remote
// mbarrier arrivals, double-buffered by unit parity).  Every CTA combines them in
// the same fixed order and gets the row's log-sum-exps, the unclipped reverse KL
//     KL = sum_v p_v (z_v - t_v) - (lse_z - lse_t),
// and the bound term_v = p_v r_v <= p_v R, R = max_v(z_v - t_v) - (lse_z - lse_t).
// A term can exceed the clip c only where p_v > c / R, i.e. z_v > lse_z + log(c/R);
// each CTA compares its group codes with that threshold (no exponentials) and
// evaluates only the flagged groups exactly, re-reading those few entries.  The
// clipped KL is KL - sum_{term_v > c} (term_v - c): each logit byte is read from
// HBM once.
//
// Exponent offsets are integers in base 2 (n = -ceil(max * log2 e)), so every
// rescale and every combine of partial sums multiplies by an exact power of two;
// float64 is used for a handful of additions, two divisions and one series
// logarithm per row (GB300 has little float64 throughput).
//
// Operations: AdaFlash article ("AdaFlash: Adaptive Speculative Decoding with
// Online Self-Improvement for High-Concurrency LLM Inference"), sections
// "On-Policy Distillation (OPD) for Domain Adaptation" (reverse KL, top-1 hard
// label, per-vocabulary clipping) and the opening section (the target verifies the
// draft; its argmax is the greedy choice).
#include <cfloat>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace adaflash {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStages = 4;
constexpr int kChunk = 4096;  // entries of each tensor per stage
constexpr int kMaxCluster = 8;
constexpr int kNoOffset = 1 << 30;  // offset of an empty partial sum
constexpr double kLn2 = 0.69314718055994530942;

struct __align__(16) SlicePartial {
  double sz, szd, st;  // sums scaled by 2^{nz}, 2^{nz}, 2^{nt}
  int nz, nt;          // integer base-2 exponent offsets
  float mt, dmax;      // max of t (argmax value), max of z - t
  int bidx;
  int err;
};

struct __align__(16) SliceCorr {
  double corr, sclip;
  int nclip;
  int err;
};

struct RowConsts {
  double lse_z, lse_t;
  float theta;
  float lse_z_f, lse_t_f;
  int argmax;
  int err;
  int stop;  // every consumer thread leaves the unit loop together when set
};

// Per-thread running state: sz = sum_v 2^{z_v log2e + nz}, szd = sum_v 2^{z_v log2e + nz} (z_v - t_v),
// st = sum_v 2^{t_v log2e + nt}; nz, nt integers (nzf, ntf the same values as floats).
struct Acc {
  float mz, sz, szd, nzf;
  float mt, st, ntf;
  float dmax;
  int nz, nt;
  int bidx;
};

__device__ __forceinline__ void acc_init(Acc& a) {
  a.mz = kNegInf; a.sz = 0.f; a.szd = 0.f; a.nzf = 0.f; a.nz = kNoOffset;
  a.mt = kNegInf; a.st = 0.f; a.ntf = 0.f; a.nt = kNoOffset;
  a.dmax = kNegInf;
  a.bidx = INT_MAX;
}

// Integer offset for a new maximum m: -ceil(m log2 e) (clamped; logits are finite).
__device__ __forceinline__ int offset_for(float m) {
  const float x = fminf(fmaxf(m * kLog2e, -1048576.f), 1048576.f);
  return -static_cast<int>(ceilf(x));
}

// Lowest j < n with x[j] == v (some j holds it).
__device__ __forceinline__ int first_eq(const float x[8], float v, int n) {
  int j = n - 1;
#pragma unroll
  for (int jj = 6; jj >= 0; --jj)
    if (jj < n - 1 && x[jj] == v) j = jj;
  return j;
}

// Paired group: z[0..n), t[0..n) of vocabulary entries v0.., with group maxima vmz, vmt.
__device__ __forceinline__ void acc_pair(Acc& a, const float z[8], const float t[8], float vmz, float vmt,
                                         int n, int v0) {
  if (vmz > a.mz) {
    a.mz = vmz;
    const int nn = offset_for(vmz);
    if (nn < a.nz) {
      const float f = pow2i(nn - a.nz);
      a.sz *= f;
      a.szd *= f;
      a.nz = nn;
      a.nzf = static_cast<float>(nn);
    }
  }
  if (vmt > a.mt) {
    a.mt = vmt;
    a.bidx = v0 + first_eq(t, vmt, n);
    const int nn = offset_for(vmt);
    if (nn < a.nt) {
      a.st *= pow2i(nn - a.nt);
      a.nt = nn;
      a.ntf = static_cast<float>(nn);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < n) {
      const float ez = ex2(fmaf(z[j], kLog2e, a.nzf));
      const float et = ex2(fmaf(t[j], kLog2e, a.ntf));
      a.sz += ez;
      a.st += et;
      const float d = z[j] - t[j];
      a.szd = fmaf(ez, d, a.szd);
      a.dmax = fmaxf(a.dmax, d);
    }
  }
}

// Target-only group: argmax only.
__device__ __forceinline__ void acc_target(Acc& a, const float t[8], float vmt, int n, int v0) {
  if (vmt > a.mt) {
    a.mt = vmt;
    a.bidx = v0 + first_eq(t, vmt, n);
  }
}

template <class DT>
__device__ __forceinline__ void load8_smem(const uint8_t* base, int g, float x[8], float& vmax);

template <>
__device__ __forceinline__ void load8_smem<BF16>(const uint8_t* base, int g, float x[8], float& vmax) {
  const uint4 q = *reinterpret_cast<const uint4*>(base + 16 * g);
  const uint32_t m = bf16x2_max(bf16x2_max(q.x, q.y), bf16x2_max(q.z, q.w));
  vmax = fmaxf(bf16_lo(m), bf16_hi(m));
  x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x);
  x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
  x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z);
  x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
}

template <>
__device__ __forceinline__ void load8_smem<F32>(const uint8_t* base, int g, float x[8], float& vmax) {
  const float4 a = *reinterpret_cast<const float4*>(base + 32 * g);
  const float4 b = *reinterpret_cast<const float4*>(base + 32 * g + 16);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  vmax = fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
}

// Up to 8 entries straight from global memory (any alignment).
template <class DT>
__device__ __forceinline__ void load_global(const void* row, int64_t v0, int n, float x[8], float& vmax) {
  vmax = kNegInf;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    x[j] = (j < n) ? DT::load(row, v0 + j) : kNegInf;
    vmax = fmaxf(vmax, x[j]);
  }
}

// Warp-level combine of two thread states (exact power-of-two rescaling).
__device__ __forceinline__ void acc_merge(Acc& a, const Acc& b) {
  const int nz = min(a.nz, b.nz);
  const float fa = pow2i(nz - a.nz), fb = pow2i(nz - b.nz);
  a.sz = a.sz * fa + b.sz * fb;
  a.szd = a.szd * fa + b.szd * fb;
  a.nz = nz;
  a.mz = fmaxf(a.mz, b.mz);
  const int nt = min(a.nt, b.nt);
  a.st = a.st * pow2i(nt - a.nt) + b.st * pow2i(nt - b.nt);
  a.nt = nt;
  if (b.mt > a.mt || (b.mt == a.mt && b.bidx < a.bidx)) a.bidx = b.bidx;
  a.mt = fmaxf(a.mt, b.mt);
  a.dmax = fmaxf(a.dmax, b.dmax);
}

__device__ __forceinline__ Acc shfl_acc(const Acc& a, int off) {
  Acc b;
  b.mz = __shfl_xor_sync(0xffffffffu, a.mz, off);
  b.sz = __shfl_xor_sync(0xffffffffu, a.sz, off);
  b.szd = __shfl_xor_sync(0xffffffffu, a.szd, off);
  b.nz = __shfl_xor_sync(0xffffffffu, a.nz, off);
  b.mt = __shfl_xor_sync(0xffffffffu, a.mt, off);
  b.st = __shfl_xor_sync(0xffffffffu, a.st, off);
  b.nt = __shfl_xor_sync(0xffffffffu, a.nt, off);
  b.dmax = __shfl_xor_sync(0xffffffffu, a.dmax, off);
  b.bidx = __shfl_xor_sync(0xffffffffu, a.bidx, off);
  b.nzf = 0.f;
  b.ntf = 0.f;
  return b;
}

// Fixed-order float64 combine of partials (exact power-of-two scaling).
__device__ void combine_partials(const SlicePartial* parts, int n, SlicePartial& out) {
  int nz = kNoOffset, nt = kNoOffset, bidx = INT_MAX, err = 0;
  float mt = kNegInf, dmax = kNegInf;
  for (int i = 0; i < n; ++i) {
    nz = min(nz, parts[i].nz);
    nt = min(nt, parts[i].nt);
    dmax = fmaxf(dmax, parts[i].dmax);
    if (parts[i].mt > mt || (parts[i].mt == mt && parts[i].bidx < bidx)) bidx = parts[i].bidx;
    mt = fmaxf(mt, parts[i].mt);
    err |= parts[i].err;
  }
  double sz = 0.0, szd = 0.0, st = 0.0;
  for (int i = 0; i < n; ++i) {
    const double f = static_cast<double>(pow2i(nz - parts[i].nz));
    sz += parts[i].sz * f;
    szd += parts[i].szd * f;
    st += parts[i].st * static_cast<double>(pow2i(nt - parts[i].nt));
  }
  out.nz = nz; out.nt = nt; out.mt = mt; out.dmax = dmax; out.bidx = bidx; out.err = err;
  out.sz = sz; out.szd = szd; out.st = st;
}

// log sum e^x at float accuracy from a positive sum kept relative to offset n.
__device__ __forceinline__ double lse_approx(double sum, int n) {
  return -static_cast<double>(n) * kLn2 + static_cast<double>(logf(static_cast<float>(sum)));
}

struct Unit {
  bool pair, bad;
  int d, s;
};

__device__ __forceinline__ Unit map_unit(const RowPassParams& P, int u) {
  Unit U;
  U.pair = false;
  U.bad = false;
  U.d = -1;
  if (P.mode == kModeVerify) {
    U.s = u;
  } else if (u < P.N_d) {
    U.pair = true;
    U.d = u;
    const int i = request_of_row(P.doff, P.R, u);
    const int lo = __ldg(P.doff + i), hi = __ldg(P.doff + i + 1);
    U.bad = !(lo <= u && u < hi);
    U.s = u + i;
  } else {
    const int i = u - P.N_d;
    U.s = __ldg(P.doff + i + 1) + i;
  }
  if (U.s < 0 || U.s >= P.N_t) U.bad = true;
  return U;
}

}  // namespace

template <class DZ, class DT, bool kFast>
__global__ void __launch_bounds__(kThreads, 2) rowpass_kernel(const RowPassParams P) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages];
  __shared__ uint64_t empty_bar[kStages];
  __shared__ uint64_t part_bar[2];
  __shared__ uint64_t corr_bar[2];
  __shared__ SlicePartial slots[2][kMaxCluster];
  __shared__ SliceCorr cslots[2][kMaxCluster];
  __shared__ SlicePartial warp_part[kConsumerWarps];
  __shared__ double warp_corr[kConsumerWarps][2];
  __shared__ int warp_nclip[kConsumerWarps];
  __shared__ RowConsts rc;
  __shared__ int s_abort;
  __shared__ int s_unit_err;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int C = P.cluster;
  const int cid = static_cast<int>(blockIdx.x) / C;
  const int ncl = static_cast<int>(gridDim.x) / C;
  const int num_units = (P.mode == kModeVerify) ? P.N_t : (P.N_d + P.R);

  constexpr int kStageZ = kChunk * DZ::kBytes;
  constexpr int kStageT = kChunk * DT::kBytes;
  // 128-byte aligned base for the bulk-copy ring (the launch adds 128 bytes of slack).
  uint8_t* ring =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  float* codes = reinterpret_cast<float*>(ring + kStages * (kStageZ + kStageT));

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&part_bar[i], static_cast<uint32_t>(C));
      mbar_init(&corr_bar[i], static_cast<uint32_t>(C));
    }
    fence_barrier_init();
    s_abort = 0;
    s_unit_err = 0;
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrival

  volatile int* abort_flag = &s_abort;

  if (warp == kConsumerWarps) {
    // ---------------- producer warp: runs ahead across units ----------------
    if (kFast && lane == 0) {
      uint32_t cc = 0;
      for (int u = cid; u < num_units && !*abort_flag; u += ncl) {
        const Unit U = map_unit(P, u);
        const int v_begin = static_cast<int>(rank) * P.slice;
        const int v_end = U.bad ? v_begin : min(P.V, v_begin + P.slice);
        const int body = max(0, v_end - v_begin) & ~7;
        const uint8_t* zrow =
            U.pair ? static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(U.d) * P.ld_z * DZ::kBytes : nullptr;
        const uint8_t* trow =
            static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(max(U.s, 0)) * P.ld_t * DT::kBytes;
        for (int e0 = 0; e0 < body; e0 += kChunk, ++cc) {
          const int st = static_cast<int>(cc % kStages);
          if (cc >= static_cast<uint32_t>(kStages) &&
              !mbar_wait_bounded(&empty_bar[st], ((cc / kStages) & 1) ^ 1)) {
            *abort_flag = 1;
            break;
          }
          const int n = min(kChunk, body - e0);
          const uint32_t bz = U.pair ? static_cast<uint32_t>(n * DZ::kBytes) : 0u;
          const uint32_t bt = static_cast<uint32_t>(n * DT::kBytes);
          mbar_arrive_expect_tx(&full_bar[st], bz + bt);
          uint8_t* stage = ring + st * (kStageZ + kStageT);
          if (U.pair) bulk_copy_g2s(stage, zrow + static_cast<int64_t>(v_begin + e0) * DZ::kBytes, bz, &full_bar[st]);
          bulk_copy_g2s(stage + kStageZ, trow + static_cast<int64_t>(v_begin + e0) * DT::kBytes, bt, &full_bar[st]);
        }
      }
      // After an abort, let copies still in flight land before the CTA can exit.
      if (*abort_flag) {
        const uint32_t lo = cc > static_cast<uint32_t>(kStages) ? cc - kStages : 0u;
        for (uint32_t k = lo; k < cc; ++k)
          mbar_wait_bounded(&full_bar[k % kStages], (k / kStages) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    // ---------------- consumer warps ----------------
    uint32_t cc = 0;
    int it = 0, pit = 0;
    for (int u = cid; u < num_units; u += ncl, ++it) {
      const Unit U = map_unit(P, u);
      const int v_begin = static_cast<int>(rank) * P.slice;
      const int v_end = U.bad ? v_begin : min(P.V, v_begin + P.slice);
      const int len = max(0, v_end - v_begin);
      const int ngroups = (len + 7) >> 3;
      const int body = kFast ? (len & ~7) : 0;
      const uint8_t* zrow =
          U.pair ? static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(U.d) * P.ld_z * DZ::kBytes : nullptr;
      const uint8_t* trow =
          static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(max(U.s, 0)) * P.ld_t * DT::kBytes;

      Acc acc;
      acc_init(acc);
      if (kFast) {
        for (int e0 = 0; e0 < body; e0 += kChunk, ++cc) {
          const int st = static_cast<int>(cc % kStages);
          if (!mbar_wait_bounded(&full_bar[st], (cc / kStages) & 1)) {
            atomicOr(&s_unit_err, 1);
            *abort_flag = 1;
            break;
          }
          const int gcount = min(kChunk, body - e0) >> 3;
          const uint8_t* stage = ring + st * (kStageZ + kStageT);
          const int gbase = e0 >> 3;
          for (int g = tid; g < gcount; g += kConsumers) {
            float t[8], vmt;
            load8_smem<DT>(stage + kStageZ, g, t, vmt);
            const int v0 = v_begin + ((gbase + g) << 3);
            if (U.pair) {
              float z[8], vmz;
              load8_smem<DZ>(stage, g, z, vmz);
              codes[gbase + g] = vmz;
              acc_pair(acc, z, t, vmz, vmt, 8, v0);
            } else {
              acc_target(acc, t, vmt, 8, v0);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[st]);
        }
      }
      // Direct loads: the whole slice (unaligned rows) or the ragged tail group.
      for (int g = (body >> 3) + tid; g < ngroups; g += kConsumers) {
        const int64_t v0 = v_begin + (static_cast<int64_t>(g) << 3);
        const int n = min(8, v_end - static_cast<int>(v0));
        float t[8], vmt;
        load_global<DT>(trow, v0, n, t, vmt);
        if (U.pair) {
          float z[8], vmz;
          load_global<DZ>(zrow, v0, n, z, vmz);
          codes[g] = vmz;
          acc_pair(acc, z, t, vmz, vmt, n, static_cast<int>(v0));
        } else {
          acc_target(acc, t, vmt, n, static_cast<int>(v0));
        }
      }

      // ---- CTA reduction, then the exchange of slice partials ----
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc_merge(acc, shfl_acc(acc, off));
      if (lane == 0) {
        SlicePartial& w = warp_part[warp];
        w.nz = acc.nz; w.sz = acc.sz; w.szd = acc.szd;
        w.nt = acc.nt; w.st = acc.st; w.mt = acc.mt; w.dmax = acc.dmax; w.bidx = acc.bidx; w.err = 0;
      }
      named_bar_sync(kConsumers);

      const int buf = it & 1;
      if (tid == 0) {
        SlicePartial mine;
        combine_partials(warp_part, kConsumerWarps, mine);
        mine.err = s_unit_err;
        s_unit_err = 0;
        for (int r = 0; r < C; ++r) *map_to_rank(&slots[buf][rank], static_cast<uint32_t>(r)) = mine;
        for (int r = 0; r < C; ++r) mbar_arrive_remote(&part_bar[buf], static_cast<uint32_t>(r));
        int werr = 0;
        if (!mbar_wait_cluster_bounded(&part_bar[buf], (it >> 1) & 1)) {
          werr = 1;
          *abort_flag = 1;
        }
        SlicePartial all;
        combine_partials(slots[buf], C, all);
        rc.argmax = all.bidx;
        rc.err = all.err | werr;
        rc.stop = *abort_flag;
        if (U.pair && !U.bad) {
          const double lse_z = lse_approx(all.sz, all.nz);
          const double lse_t = lse_approx(all.st, all.nt);
          const float dlse = static_cast<float>(lse_z - lse_t);
          rc.lse_z = lse_z;
          rc.lse_t = lse_t;
          rc.lse_z_f = static_cast<float>(lse_z);
          rc.lse_t_f = static_cast<float>(lse_t);
          // Screen threshold on group maxima of z; the slack only adds candidates.
          const float R = all.dmax - dlse;
          const float Rp = R + 1e-4f * (1.f + fabsf(all.dmax) + fabsf(dlse));
          const float c = P.clip_c;
          if (!(c < INFINITY) || !(Rp > 0.f)) {
            rc.theta = INFINITY;
          } else {
            const double th = lse_z + static_cast<double>(logf(c / Rp)) - (1e-3 + 1e-6 * fabs(lse_z));
            rc.theta = __double2float_rd(th);
          }
        }
      }
      named_bar_sync(kConsumers);
      const bool stop = rc.stop != 0;  // read by every consumer thread from the same broadcast

      if (!U.pair) {
        if (rank == 0 && tid == 0) {
          if (U.bad) flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
          else {
            P.target_argmax[U.s] = rc.argmax;
            if (rc.err) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
          }
        }
        if (stop) break;
        continue;
      }

      // ---- exact evaluation of the screened groups ----
      double corr = 0.0, sclip = 0.0;
      int nclip = 0;
      {
        const float theta = U.bad ? INFINITY : rc.theta;
        const TermConsts tc = make_term_consts(rc.lse_z_f, rc.lse_t_f);
        const float c = P.clip_c;
        for (int g = tid; g < ngroups; g += kConsumers) {
          if (codes[g] > theta) {
            const int v0 = v_begin + (g << 3);
            const int n = min(8, v_end - v0);
            for (int j = 0; j < n; ++j) {
              const float zv = DZ::load(zrow, v0 + j);
              const float tv = DT::load(trow, v0 + j);
              float p, r, term;
              entry_term(zv, tv, tc, p, r, term);  // the backward's decision, bit for bit
              if (term > c) {
                // the clipped amount, from the log-sum-exps before float32 rounding
                const double zd = static_cast<double>(zv);
                const float arg = static_cast<float>((zd - rc.lse_z) * 1.4426950408889634);
                const double pd = static_cast<double>(ex2(arg));
                const double rd = (zd - static_cast<double>(tv)) - (rc.lse_z - rc.lse_t);
                corr += pd * rd - static_cast<double>(c);
                sclip += pd * (rd + 1.0);
                ++nclip;
              }
            }
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        corr += __shfl_xor_sync(0xffffffffu, corr, off);
        sclip += __shfl_xor_sync(0xffffffffu, sclip, off);
        nclip += __shfl_xor_sync(0xffffffffu, nclip, off);
      }
      if (lane == 0) {
        warp_corr[warp][0] = corr;
        warp_corr[warp][1] = sclip;
        warp_nclip[warp] = nclip;
      }
      named_bar_sync(kConsumers);
      const int cbuf = pit & 1;
      if (tid == 0) {
        SliceCorr mine;
        mine.corr = 0.0; mine.sclip = 0.0; mine.nclip = 0; mine.err = rc.err;
        for (int w = 0; w < kConsumerWarps; ++w) {
          mine.corr += warp_corr[w][0];
          mine.sclip += warp_corr[w][1];
          mine.nclip += warp_nclip[w];
        }
        *map_to_rank(&cslots[cbuf][rank], 0u) = mine;
        mbar_arrive_remote(&corr_bar[cbuf], 0u);
        if (rank == 0) {
          const bool ok = mbar_wait_cluster_bounded(&corr_bar[cbuf], (pit >> 1) & 1);
          if (!ok) *abort_flag = 1;
          if (U.bad) {
            flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
          } else {
            double corr_all = 0.0, sclip_all = 0.0;
            int nclip_all = 0, err_all = rc.err | (ok ? 0 : 1);
            for (int r = 0; r < C; ++r) {
              corr_all += cslots[cbuf][r].corr;
              sclip_all += cslots[cbuf][r].sclip;
              nclip_all += cslots[cbuf][r].nclip;
              err_all |= cslots[cbuf][r].err;
            }
            // Accurate difference of the log-sum-exps for the unclipped KL.
            SlicePartial all;
            combine_partials(slots[buf], C, all);
            const double dlse = static_cast<double>(all.nt - all.nz) * kLn2 + ln_series(all.sz / all.st);
            const double kl_unclip = all.szd / all.sz - dlse;
            const int a = rc.argmax;
            const double z_a = static_cast<double>(DZ::load(zrow, a));
            const int64_t d = U.d;
            P.kl_row[d] = static_cast<float>(kl_unclip - corr_all);
            P.ce_row[d] = static_cast<float>(rc.lse_z - z_a);
            P.row_stats[4 * d + 0] = rc.lse_z_f;
            P.row_stats[4 * d + 1] = rc.lse_t_f;
            P.row_stats[4 * d + 2] = static_cast<float>(kl_unclip + 1.0 - sclip_all);
            P.row_stats[4 * d + 3] = static_cast<float>(nclip_all);
            P.target_argmax[U.s] = a;
            if (err_all) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
          }
        }
      }
      ++pit;
      if (stop) break;
    }
    if (*abort_flag && tid == 0) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
  }

  __syncthreads();
  cluster_sync_all();  // no CTA leaves while a peer may still address its shared memory
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

int rowpass_cluster_size(int vocab) {
  // about 40K entries per CTA; at most 8 CTAs (the portable cluster size)
  int c = (vocab + 39999) / 40000;
  return c < 1 ? 1 : (c > kMaxCluster ? kMaxCluster : c);
}

int rowpass_slice(int vocab, int cluster) {
  const int per = (vocab + cluster - 1) / cluster;
  return (per + 7) & ~7;
}

namespace {
// Co-resident cluster counts, cached per (kernel, shared memory, cluster size, device).
struct OccEntry {
  const void* fn;
  size_t smem;
  int cluster;
  int device;
  int clusters;
};
OccEntry g_occ[64];
int g_occ_n = 0;
}  // namespace

template <class DZ, class DT, bool kFast>
static cudaError_t launch_one(const RowPassParams& p, cudaStream_t stream) {
  const size_t ring = static_cast<size_t>(kStages) * kChunk * (DZ::kBytes + DT::kBytes);
  const size_t smem = 128 + ring + static_cast<size_t>((p.slice + 7) / 8) * sizeof(float);
  auto kern = rowpass_kernel<DZ, DT, kFast>;
  const int units = (p.mode == kModeVerify) ? p.N_t : (p.N_d + p.R);
  if (units <= 0) return cudaSuccess;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;

  int clusters = -1;
  for (int i = 0; i < g_occ_n; ++i)
    if (g_occ[i].fn == reinterpret_cast<const void*>(kern) && g_occ[i].smem == smem &&
        g_occ[i].cluster == p.cluster && g_occ[i].device == device)
      clusters = g_occ[i].clusters;
  if (clusters < 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(p.cluster), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = 1;
    }
    clusters = n;
    if (g_occ_n < 64) g_occ[g_occ_n++] = OccEntry{reinterpret_cast<const void*>(kern), smem, p.cluster, device, n};
  }
  // One persistent cluster per co-resident slot (clusters never wait on one another).
  const int grid_clusters = units < clusters ? units : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(grid_clusters) * static_cast<unsigned>(p.cluster), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_rowpass(const RowPassParams& p, int z_dtype, int t_dtype, bool fast, cudaStream_t s) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (fast) {
    if (zb && tb) return launch_one<BF16, BF16, true>(p, s);
    if (!zb && tb) return launch_one<F32, BF16, true>(p, s);
    if (zb && !tb) return launch_one<BF16, F32, true>(p, s);
    return launch_one<F32, F32, true>(p, s);
  }
  if (zb && tb) return launch_one<BF16, BF16, false>(p, s);
  if (!zb && tb) return launch_one<F32, BF16, false>(p, s);
  if (zb && !tb) return launch_one<BF16, F32, false>(p, s);
  return launch_one<F32, F32, false>(p, s);
}

}  // namespace adaflash
