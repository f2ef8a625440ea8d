// rowpass.cu -- K1: the fused streaming pass over packed logit rows.
//
// One work unit is either a PAIR (draft row d with its target row s) or a
// TARGET-ONLY row (a bonus row, or every row in verification-only mode).  A unit
// is handled by a cluster of C CTAs; CTA rank c owns the vocabulary slice
// [c*slice, (c+1)*slice).  Each CTA streams its slice once from HBM:
//
//   producer warp : 1-D bulk copies (TMA engine) of chunks of z and t into a
//                   ring of shared-memory stages, signalled by mbarriers;
//   8 consumer warps: per 8-entry group, an online log-sum-exp of z and of t,
//                   sum_v e^{z_v - M}(z_v - t_v), max_v (z_v - t_v), the
//                   lowest-index argmax of t, and the group maximum of z kept in
//                   shared memory as a screening code.
//
// The slice results meet over distributed shared memory; every CTA combines them
// in the same fixed order (float64) and gets the row's log-sum-exps, the
// unclipped reverse KL
//     KL = sum_v p_v (z_v - t_v) - (lse_z - lse_t),
// and the bound term_v = p_v r_v <= p_v R with R = max_v(z_v - t_v) - (lse_z - lse_t).
// A term can exceed the clip c only where p_v > c / R, i.e. z_v > lse_z + log(c/R);
// the CTA scans its group codes against that threshold (no exponentials) and
// evaluates only the flagged groups exactly, re-reading those few entries.  The
// clipped KL is KL - sum_{term_v > c} (term_v - c), so each logit byte is read
// from HBM once.
//
// Operations: AdaFlash article ("AdaFlash: Adaptive Speculative Decoding with
// Online Self-Improvement for High-Concurrency LLM Inference"), sections
// "On-Policy Distillation (OPD) for Domain Adaptation" (reverse KL, top-1 hard
// label, per-vocabulary clipping) and the opening section (the target verifies the
// draft; its argmax is the greedy choice).
#include <cfloat>
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

struct __align__(16) SlicePartial {
  double sz, szd, st;  // sums scaled by 2^{nz}, 2^{nt} (see Acc)
  float nz, nt;        // exponent offsets actually used (float32 values, exact)
  float mt, dmax;      // max of t (for the argmax), max of z - t
  int bidx;
  int err;
};

struct __align__(16) SliceCorr {
  double corr, sclip;
  int nclip;
  int err;
};

struct RowConsts {
  double lse_z, lse_t, kl_unclip;
  float theta;
  float lse_z_f, lse_t_f;
  int argmax;
  int err;
};

// Per-thread running state.  Sums are kept relative to the exponent offset that
// is actually applied, nz = fl(-max(z) * log2 e):
//   sz = sum_v 2^{z_v log2e + nz},  szd = sum_v 2^{z_v log2e + nz} (z_v - t_v),
//   st = sum_v 2^{t_v log2e + nt}.
// Combining partials with their exact float offsets (rather than the maxima)
// keeps the rounding of -max*log2e out of the result.
struct Acc {
  float mz, nz, sz, szd;
  float mt, nt, st;
  float dmax;
  int bidx;
};

constexpr float kPosInf = __builtin_huge_valf();

__device__ __forceinline__ void acc_init(Acc& a) {
  a.mz = kNegInf; a.nz = kPosInf; a.sz = 0.f; a.szd = 0.f;
  a.mt = kNegInf; a.nt = kPosInf; a.st = 0.f;
  a.dmax = kNegInf;
  a.bidx = INT_MAX;
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
    const float nn = __fmul_rn(-vmz, kLog2e);
    const float f = ex2(nn - a.nz);
    a.sz *= f;
    a.szd *= f;
    a.mz = vmz;
    a.nz = nn;
  }
  if (vmt > a.mt) {
    const float nn = __fmul_rn(-vmt, kLog2e);
    const float f = ex2(nn - a.nt);
    a.st *= f;
    a.mt = vmt;
    a.nt = nn;
    a.bidx = v0 + first_eq(t, vmt, n);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < n) {
      const float ez = ex2(fmaf(z[j], kLog2e, a.nz));
      const float et = ex2(fmaf(t[j], kLog2e, a.nt));
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

// Group of 8 from a shared-memory stage (16-byte aligned).
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

// Warp-level combine of two thread states (float32, fixed xor pattern).
__device__ __forceinline__ void acc_merge(Acc& a, const Acc& b) {
  const float nz = fminf(a.nz, b.nz);
  const float fa = (a.nz == kPosInf) ? 0.f : ex2(nz - a.nz);
  const float fb = (b.nz == kPosInf) ? 0.f : ex2(nz - b.nz);
  a.sz = a.sz * fa + b.sz * fb;
  a.szd = a.szd * fa + b.szd * fb;
  a.nz = nz;
  a.mz = fmaxf(a.mz, b.mz);
  const float nt = fminf(a.nt, b.nt);
  const float ga = (a.nt == kPosInf) ? 0.f : ex2(nt - a.nt);
  const float gb = (b.nt == kPosInf) ? 0.f : ex2(nt - b.nt);
  a.st = a.st * ga + b.st * gb;
  a.nt = nt;
  if (b.mt > a.mt || (b.mt == a.mt && b.bidx < a.bidx)) a.bidx = b.bidx;
  a.mt = fmaxf(a.mt, b.mt);
  a.dmax = fmaxf(a.dmax, b.dmax);
}

__device__ __forceinline__ Acc shfl_acc(const Acc& a, int off) {
  Acc b;
  b.mz = __shfl_xor_sync(0xffffffffu, a.mz, off);
  b.nz = __shfl_xor_sync(0xffffffffu, a.nz, off);
  b.sz = __shfl_xor_sync(0xffffffffu, a.sz, off);
  b.szd = __shfl_xor_sync(0xffffffffu, a.szd, off);
  b.mt = __shfl_xor_sync(0xffffffffu, a.mt, off);
  b.nt = __shfl_xor_sync(0xffffffffu, a.nt, off);
  b.st = __shfl_xor_sync(0xffffffffu, a.st, off);
  b.dmax = __shfl_xor_sync(0xffffffffu, a.dmax, off);
  b.bidx = __shfl_xor_sync(0xffffffffu, a.bidx, off);
  return b;
}

// float64 combine of slice partials in a fixed order; offsets combine exactly.
__device__ void combine_partials(const SlicePartial* parts, int n, SlicePartial& out) {
  float nz = kPosInf, nt = kPosInf, mt = kNegInf, dmax = kNegInf;
  int bidx = INT_MAX, err = 0;
  for (int i = 0; i < n; ++i) {
    nz = fminf(nz, parts[i].nz);
    nt = fminf(nt, parts[i].nt);
    dmax = fmaxf(dmax, parts[i].dmax);
    if (parts[i].mt > mt || (parts[i].mt == mt && parts[i].bidx < bidx)) bidx = parts[i].bidx;
    mt = fmaxf(mt, parts[i].mt);
    err |= parts[i].err;
  }
  double sz = 0.0, szd = 0.0, st = 0.0;
  for (int i = 0; i < n; ++i) {
    if (parts[i].nz != kPosInf) {
      const double f = exp2(static_cast<double>(nz) - static_cast<double>(parts[i].nz));
      sz += parts[i].sz * f;
      szd += parts[i].szd * f;
    }
    if (parts[i].nt != kPosInf) {
      const double g = exp2(static_cast<double>(nt) - static_cast<double>(parts[i].nt));
      st += parts[i].st * g;
    }
  }
  out.nz = nz; out.nt = nt; out.mt = mt; out.dmax = dmax; out.bidx = bidx; out.err = err;
  out.sz = sz; out.szd = szd; out.st = st;
}

// log sum_v e^{x_v} from a sum kept relative to the exponent offset n (base 2).
__device__ __forceinline__ double lse_from(double sum, float n) {
  return -static_cast<double>(n) * 0.69314718055994530942 + log(sum);
}

}  // namespace

template <class DZ, class DT, bool kFast>
__global__ void __launch_bounds__(kThreads) rowpass_kernel(const RowPassParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[kStages];
  __shared__ uint64_t empty_bar[kStages];
  __shared__ SlicePartial slots[kMaxCluster];
  __shared__ SliceCorr cslots[kMaxCluster];
  __shared__ SlicePartial warp_part[kConsumerWarps];
  __shared__ double warp_corr[kConsumerWarps][2];
  __shared__ int warp_nclip[kConsumerWarps];
  __shared__ RowConsts rc;
  __shared__ int s_issued;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int C = P.cluster;
  const int unit = static_cast<int>(blockIdx.x) / C;

  // Pairs with the wait before the first store into a peer's shared memory.
  cluster_arrive_relaxed();

  // ---- unit -> rows (identical in every CTA of the cluster) ----
  bool pair = false, bad = false;
  int d = -1, s = -1;
  if (P.mode == kModeVerify) {
    s = unit;
  } else if (unit < P.N_d) {
    pair = true;
    d = unit;
    const int i = request_of_row(P.doff, P.R, d);
    const int lo = __ldg(P.doff + i), hi = __ldg(P.doff + i + 1);
    bad = !(lo <= d && d < hi);
    s = d + i;
  } else {
    const int i = unit - P.N_d;
    s = __ldg(P.doff + i + 1) + i;
  }
  if (s < 0 || s >= P.N_t) bad = true;

  const int v_begin = static_cast<int>(rank) * P.slice;
  const int v_end = bad ? v_begin : min(P.V, v_begin + P.slice);
  const int len = max(0, v_end - v_begin);
  const int ngroups = (len + 7) >> 3;
  const int body = kFast ? (len & ~7) : 0;
  const int nchunks = (body + kChunk - 1) / kChunk;

  const uint8_t* zrow = pair ? static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(d) * P.ld_z * DZ::kBytes
                             : nullptr;
  const uint8_t* trow = static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(max(s, 0)) * P.ld_t * DT::kBytes;

  constexpr int kStageZ = kChunk * DZ::kBytes;
  constexpr int kStageT = kChunk * DT::kBytes;
  // 128-byte aligned base for the bulk-copy ring (the launch adds 128 bytes of slack).
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem) + 127) & ~static_cast<uintptr_t>(127));
  float* codes = reinterpret_cast<float*>(ring + kStages * (kStageZ + kStageT));

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    fence_barrier_init();
    s_issued = 0;
  }
  __syncthreads();

  Acc acc;
  acc_init(acc);
  int err = 0;

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    if (kFast && lane == 0) {
      int k = 0;
      for (; k < nchunks; ++k) {
        const int st = k % kStages;
        if (k >= kStages && !mbar_wait_bounded(&empty_bar[st], ((k / kStages) - 1) & 1)) {
          err = 1;
          break;
        }
        const int e0 = k * kChunk;
        const int n = min(kChunk, body - e0);
        const uint32_t bz = pair ? static_cast<uint32_t>(n * DZ::kBytes) : 0u;
        const uint32_t bt = static_cast<uint32_t>(n * DT::kBytes);
        mbar_arrive_expect_tx(&full_bar[st], bz + bt);
        uint8_t* stage = ring + st * (kStageZ + kStageT);
        if (pair) bulk_copy_g2s(stage, zrow + static_cast<int64_t>(v_begin + e0) * DZ::kBytes, bz, &full_bar[st]);
        bulk_copy_g2s(stage + kStageZ, trow + static_cast<int64_t>(v_begin + e0) * DT::kBytes, bt, &full_bar[st]);
      }
      s_issued = k;
    }
  } else {
    // ---------------- consumer warps ----------------
    if (kFast) {
      for (int k = 0; k < nchunks; ++k) {
        const int st = k % kStages;
        if (!mbar_wait_bounded(&full_bar[st], (k / kStages) & 1)) {
          err = 1;
          break;
        }
        const int n = min(kChunk, body - k * kChunk);
        const int gcount = n >> 3;
        const uint8_t* stage = ring + st * (kStageZ + kStageT);
        const int gbase = (k * kChunk) >> 3;
        for (int g = tid; g < gcount; g += kConsumers) {
          float t[8], vmt;
          load8_smem<DT>(stage + kStageZ, g, t, vmt);
          const int v0 = v_begin + ((gbase + g) << 3);
          if (pair) {
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
      if (pair) {
        float z[8], vmz;
        load_global<DZ>(zrow, v0, n, z, vmz);
        codes[g] = vmz;
        acc_pair(acc, z, t, vmz, vmt, n, static_cast<int>(v0));
      } else {
        acc_target(acc, t, vmt, n, static_cast<int>(v0));
      }
    }
  }

  // ---- CTA reduction of the per-thread states ----
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc_merge(acc, shfl_acc(acc, off));
    if (lane == 0) {
      SlicePartial& w = warp_part[warp];
      w.nz = acc.nz; w.sz = acc.sz; w.szd = acc.szd;
      w.nt = acc.nt; w.st = acc.st; w.mt = acc.mt; w.dmax = acc.dmax; w.bidx = acc.bidx; w.err = 0;
    }
  }
  const int any_err = __syncthreads_or(err);

  // After a failed wait, let copies still in flight land before the CTA can exit.
  if (any_err && kFast && tid == kConsumers) {
    const int issued = s_issued;
    for (int k = max(0, issued - kStages); k < issued; ++k)
      mbar_wait_bounded(&full_bar[k % kStages], (k / kStages) & 1, 100000000ull);
  }

  // Peers have started (matching the relaxed arrive at entry) -> safe to push.
  cluster_wait_acquire();
  if (tid == 0) {
    SlicePartial mine;
    combine_partials(warp_part, kConsumerWarps, mine);
    mine.err = any_err;
    for (int r = 0; r < C; ++r) *map_to_rank(&slots[rank], static_cast<uint32_t>(r)) = mine;
  }
  cluster_sync_all();  // every CTA now holds all slice partials

  if (tid == 0) {
    SlicePartial all;
    combine_partials(slots, C, all);
    rc.argmax = all.bidx;
    rc.err = all.err;
    if (pair) {
      const double lse_z = lse_from(all.sz, all.nz);
      const double lse_t = lse_from(all.st, all.nt);
      const double dlse = lse_z - lse_t;
      rc.lse_z = lse_z;
      rc.lse_t = lse_t;
      rc.kl_unclip = all.szd / all.sz - dlse;
      rc.lse_z_f = static_cast<float>(lse_z);
      rc.lse_t_f = static_cast<float>(lse_t);
      // Screen threshold on group maxima of z (conservative: rounding only adds candidates).
      const double R = static_cast<double>(all.dmax) - dlse;
      const double Rp = R + 1e-4 * (1.0 + fabs(static_cast<double>(all.dmax)) + fabs(dlse));
      const double c = static_cast<double>(P.clip_c);
      if (!(c < INFINITY) || !(Rp > 0.0)) {
        rc.theta = INFINITY;
      } else {
        const double th = lse_z + log(c / Rp) - (1e-3 + 1e-6 * fabs(lse_z));
        rc.theta = __double2float_rd(th);
      }
    }
  }

  if (!pair) {
    if (rank == 0 && tid == 0) {
      if (bad) flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
      else {
        P.target_argmax[s] = rc.argmax;
        if (rc.err) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
      }
    }
    return;
  }
  __syncthreads();

  // ---- exact evaluation of the screened groups ----
  double corr = 0.0, sclip = 0.0;
  int nclip = 0;
  if (warp < kConsumerWarps) {
    const float theta = rc.theta;
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
            // the clipped amount itself in float64 from the float64 log-sum-exps
            const double pd = exp(static_cast<double>(zv) - rc.lse_z);
            const double rd = (static_cast<double>(zv) - static_cast<double>(tv)) - (rc.lse_z - rc.lse_t);
            corr += pd * rd - static_cast<double>(c);
            sclip += pd * (rd + 1.0);
            ++nclip;
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
  }
  __syncthreads();
  if (tid == 0) {
    SliceCorr mine;
    mine.corr = 0.0; mine.sclip = 0.0; mine.nclip = 0; mine.err = rc.err;
    for (int w = 0; w < kConsumerWarps; ++w) {
      mine.corr += warp_corr[w][0];
      mine.sclip += warp_corr[w][1];
      mine.nclip += warp_nclip[w];
    }
    *map_to_rank(&cslots[rank], 0u) = mine;
  }
  cluster_sync_all();  // rank 0 holds every slice's correction

  if (rank == 0 && tid == 0) {
    if (bad) {
      flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
      return;
    }
    double corr_all = 0.0, sclip_all = 0.0;
    int nclip_all = 0, err_all = rc.err;
    for (int r = 0; r < C; ++r) {
      corr_all += cslots[r].corr;
      sclip_all += cslots[r].sclip;
      nclip_all += cslots[r].nclip;
      err_all |= cslots[r].err;
    }
    const int a = rc.argmax;
    const double z_a = static_cast<double>(DZ::load(zrow, a));
    P.kl_row[d] = static_cast<float>(rc.kl_unclip - corr_all);
    P.ce_row[d] = static_cast<float>(rc.lse_z - z_a);
    float4 st;
    st.x = rc.lse_z_f;
    st.y = rc.lse_t_f;
    st.z = static_cast<float>(rc.kl_unclip + 1.0 - sclip_all);
    st.w = static_cast<float>(nclip_all);
    P.row_stats[4 * static_cast<int64_t>(d) + 0] = st.x;
    P.row_stats[4 * static_cast<int64_t>(d) + 1] = st.y;
    P.row_stats[4 * static_cast<int64_t>(d) + 2] = st.z;
    P.row_stats[4 * static_cast<int64_t>(d) + 3] = st.w;
    P.target_argmax[s] = a;
    if (err_all) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
  }
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

template <class DZ, class DT, bool kFast>
static cudaError_t launch_one(const RowPassParams& p, cudaStream_t stream) {
  const size_t ring = static_cast<size_t>(kStages) * kChunk * (DZ::kBytes + DT::kBytes);
  const size_t smem = 128 + ring + static_cast<size_t>((p.slice + 7) / 8) * sizeof(float);
  auto kern = rowpass_kernel<DZ, DT, kFast>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int units = (p.mode == kModeVerify) ? p.N_t : (p.N_d + p.R);
  if (units <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units) * static_cast<unsigned>(p.cluster), 1, 1);
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
