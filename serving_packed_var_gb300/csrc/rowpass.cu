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
//   consumer warps  : (8 in the forward, 4 with the gradient) per 8-entry group, an
//                     online log-sum-exp of z and of t, sum_v e^{z_v}(z_v - t_v)
//                     (packed f32x2 arithmetic), a bound on max_v (z_v - t_v), the
//                     lowest-index argmax of t, and the largest group maximum of z
//                     each thread sees.
//
// Slice results meet over distributed shared memory (asynchronous remote stores
// that complete on the receiver's mbarrier, double-buffered by unit parity).  Every
// CTA combines them in the same fixed order and gets the row's log-sum-exps, the
// unclipped reverse KL
//     KL = sum_v p_v (z_v - t_v) - (lse_z - lse_t),
// and the bound term_v = p_v r_v <= p_v R, R = max_v(z_v - t_v) - (lse_z - lse_t).
// A term can exceed the clip c only where p_v > c / R, i.e. z_v > lse_z + log(c/R);
// each thread compares the largest group maximum of z it saw with that threshold
// (no exponentials) and only when it is above, its groups are re-read and the ones
// above the threshold evaluated exactly.  The clipped KL is
// KL - sum_{term_v > c} (term_v - c): each logit byte is read from HBM once.
//
// Exponent offsets are integers in base 2 (n = -ceil(max * log2 e)), so every
// rescale and every combine of partial sums multiplies by an exact power of two.
// Everything is float32: on GB300 one float64 warp-instruction holds the small
// float64 pipe for a whole warp's worth of lanes, and the per-row tail of this
// kernel runs on a single thread.  The difference of log-sum-exps is taken as
// (n_t - n_z) ln 2 + ln(S_z / S_t), never as a difference of two large logs.
//
// The kGrad instantiation also writes dz: a second pass over each slice, served
// from the ring and from L2, once the row's constants and clip corrections are known
// (see the comments at second_pass_chunk and RowGrad below).
//
// Operations: AdaFlash article ("AdaFlash: Adaptive Speculative Decoding with
// Online Self-Improvement for High-Concurrency LLM Inference"), sections
// "On-Policy Distillation (OPD) for Domain Adaptation" (reverse KL, top-1 hard
// label, per-vocabulary clipping) and the opening section (the target verifies the
// draft; its argmax is the greedy choice).
#include <algorithm>
#include <atomic>
#include <cfloat>
#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "rowstats.cuh"

namespace adaflash {

namespace {

// CTA shape, ring depth, stage size and resident CTAs per SM, the measured best on
// GB300 for bf16 logits.  The forward: two CTAs per SM of 8 consumer warps, each with
// a 96 KB ring of three 8192-entry stages of z and t (one CTA of 16 warps, or 4096-
// entry stages, ran slower on the 128-request batch at V = 151936).  With the
// gradient: four CTAs per SM of 4 consumer warps with 48 KB rings of three 4096-entry
// stages (more CTAs per SM hide the per-row exchanges better: 237 -> 228 us on a
// 914-row batch at V = 151936; a fourth stage did not help either pass).
constexpr int kFwdConsumerWarps = 8;
constexpr int kFwdMinBlocks = 2;
constexpr int kFwdChunk = 8192;
constexpr int kGradConsumerWarps = 4;
constexpr int kGradMinBlocks = 4;
constexpr int kGradChunk = 4096;

template <bool kGrad>
struct RowCfg {
  static constexpr int kWarps = kGrad ? kGradConsumerWarps : kFwdConsumerWarps;
  static constexpr int kConsumers = kWarps * 32;
  static constexpr int kThreads = kConsumers + 32;  // + one producer warp
  static constexpr int kMinBlocks = kGrad ? kGradMinBlocks : kFwdMinBlocks;
  static constexpr int kChunk = kGrad ? kGradChunk : kFwdChunk;
  static_assert((kWarps & (kWarps - 1)) == 0, "a power-of-two number of consumer warps");
  static_assert((kChunk / 2) % (8 * kConsumers) == 0, "a chunk gives every consumer thread whole groups");
};

// Entries of each tensor per stage: the configuration's chunk for two 16-bit
// inputs, half of it when either input is float32 (the same ring bytes).
template <class DZ, class DT, bool kGrad>
__host__ __device__ constexpr int chunk_of() {
  return DZ::kBytes + DT::kBytes <= 4 ? RowCfg<kGrad>::kChunk : RowCfg<kGrad>::kChunk / 2;
}
// One ring stage: the target chunk, then the draft chunk with 16 bytes of room for a
// copy that starts at the 16-byte boundary below a draft body off the grid; the
// stage rounded to 128 bytes.
template <class DZ, class DT, bool kGrad>
struct StageLayout {
  static constexpr int kChunk = chunk_of<DZ, DT, kGrad>();
  static constexpr int kZOff = kChunk * DT::kBytes;
  static constexpr int kBytes = (kZOff + kChunk * DZ::kBytes + 16 + 127) / 128 * 128;
};

// Ring stages: three; four in the pass with the gradient when one input is float32 and
// the other bf16, whose 2048-entry stages are a quarter smaller than the bf16 pair's, so
// that the ring keeps about the same bytes (and the second pass takes four chunks from
// it instead of three).
template <class DZ, class DT, bool kGrad>
__host__ __device__ constexpr int stages_of() {
  return (kGrad && DZ::kBytes + DT::kBytes == 6) ? 4 : 3;
}


}  // namespace

// Per-row coefficients of the gradient (the backward's per-entry sequence).
struct RowGrad {
  TermConsts tc;
  float c;
  float k_m;     // 1 + beta - S   (inner factor where the term is kept: r + k_m)
  float k_clip;  // beta - S       (inner factor where the term is clipped)
  float g;       // upstream weight of the row
  float bg;      // beta * g, taken off at the target argmax
  float lse_z;
  float mt;      // the max of t
  int ga;        // slice-local body group holding the first max of t, -1 when not in this slice
  int head_arg;  // the first max of t lies in the row's head, which this CTA holds
  int stop;      // a wait gave up: every consumer thread leaves together
};

__device__ __forceinline__ float grad_of(float z, float t, const RowGrad& k) {
  float p, r, term;
  entry_term(z, t, k.tc, p, r, term);
  const float inner = (term <= k.c) ? __fadd_rn(r, k.k_m) : k.k_clip;
  return __fmul_rn(__fmul_rn(p, inner), k.g);
}

// grad_of on a group of 8 entries, two per instruction on the FMA pipe: the f32x2
// forms of the same round-to-nearest operations, so every lane equals grad_of bit
// for bit.
__device__ __forceinline__ void grad_of8(const float z[8], const float t[8], const RowGrad& k, float out[8]) {
  const uint64_t l2e = f2_pack(kLog2e, kLog2e);
  const uint64_t nl = f2_pack(k.tc.neg_lse_z_l2e, k.tc.neg_lse_z_l2e);
  const uint64_t dl = f2_pack(k.tc.dlse, k.tc.dlse);
  const uint64_t km = f2_pack(k.k_m, k.k_m);
  const uint64_t gg = f2_pack(k.g, k.g);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint64_t Z = f2_pack(z[2 * q], z[2 * q + 1]);
    const uint64_t T = f2_pack(t[2 * q], t[2 * q + 1]);
    float a0, a1;
    f2_unpack(f2_fma(Z, l2e, nl), a0, a1);
    const uint64_t P = f2_pack(ex2(a0), ex2(a1));
    const uint64_t R = f2_sub(f2_sub(Z, T), dl);  // r
    float m0, m1, r0, r1;
    f2_unpack(f2_mul(P, R), m0, m1);  // the terms p r
    f2_unpack(f2_add(R, km), r0, r1);
    const uint64_t I = f2_pack(m0 <= k.c ? r0 : k.k_clip, m1 <= k.c ? r1 : k.k_clip);
    f2_unpack(f2_mul(f2_mul(P, I), gg), out[2 * q], out[2 * q + 1]);
  }
}

// Reuse of the ring by the second pass (with the gradient): when a slice has at least
// kStages chunks, the last kStages chunks of the first pass are still in the ring, each
// in the stage that the second pass's first kStages positions land in (position ci of
// the second pass is ring position nch + ci after the first pass's 0 .. nch - 1).  They
// come first, in ascending order, with no copy; the rest follow from L2, last chunk
// first (the newest lines there).  With fewer chunks every chunk comes from L2.  The
// first pass asks L2 to drop those last chunks at once rather than keep them.  Measured
// on one box (us per call, 128 / 32 requests at V = 151936 bf16, ms on the 512-request
// stress batch; every chunk from L2 in brackets): 217.4 (218.6), 79.4 (79.1), 2.441
// (2.438); keeping the reused chunks in L2 as well: 219.6, 79.3, 2.465.
template <int kStages>
__device__ __forceinline__ bool second_pass_reuses(int ci, int nch) {
  return nch >= kStages && ci < kStages;
}
template <int kStages>
__device__ __forceinline__ int second_pass_chunk(int ci, int nch) {
  return second_pass_reuses<kStages>(ci, nch) ? nch - kStages + ci : nch - 1 - ci;
}

// kGrad: the single-pass forward + backward for batches of many rows.  After a
// pair unit's row constants and clip corrections are known, the producer's second
// pass over the same slice (queued right behind the first, so it is served from L2:
// the first pass asks L2 to keep the lines, the second to drop them) feeds the
// gradient, dz_v = g (p_v (m_v (r_v + 1) - S) + beta (p_v - [v == a])), written once
// with streaming stores.  Every CTA of the cluster gets the corrections (every CTA
// needs S).
//
// Rows need not start on the 16-byte grid.  A unit's vocabulary follows the target
// row's grid: its first H entries (the head, before the target row's first 16-byte
// boundary; H < 8) are group 0, read with element loads by rank 0, and the body
// [H, V) is cut into 8-entry groups 1, 2, ... and into slices of the cluster.  The
// target body is bulk-copied as it lies; the draft body, which may start 2 zs2
// bytes past a boundary, is bulk-copied from the boundary below it (16 bytes more)
// and read with aligned loads at that shift (one instance of the loop per shift).
// kShift = false is the instance for batches whose every row (and gradient row) starts
// on the 16-byte grid: no head, no shifted loads, plain 16-byte stores; its smaller
// code runs the aligned batch 6% faster than the general instance does.
template <class DZ, class DT, bool kGrad, bool kShift>
__global__ void __launch_bounds__(RowCfg<kGrad>::kThreads, RowCfg<kGrad>::kMinBlocks)
    rowpass_kernel(const RowPassParams P) {
  constexpr int kConsumerWarps = RowCfg<kGrad>::kWarps;
  constexpr int kConsumers = RowCfg<kGrad>::kConsumers;
  constexpr int kStages = stages_of<DZ, DT, kGrad>();
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages];
  __shared__ uint64_t empty_bar[kStages];
  __shared__ uint64_t part_bar[2];
  __shared__ uint64_t corr_bar[2];
  __shared__ SlicePartial slots[2][kMaxCluster];
  __shared__ SliceCorr cslots[2][kMaxCluster];
  __shared__ SlicePartial warp_part[kConsumerWarps];
  __shared__ float warp_corr[kConsumerWarps][2];
  __shared__ int warp_nclip[kConsumerWarps];
  __shared__ RowConsts rc;
  __shared__ RowGrad s_grad;
  __shared__ int s_abort;
  __shared__ int s_unit_err;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int C = P.cluster;
  const int cid = static_cast<int>(blockIdx.x) / C;
  const int ncl = static_cast<int>(gridDim.x) / C;
  const int num_units = P.unit_end;
  // Unit order.  Units are paired rows, then target-only rows; cluster cid takes every
  // ncl-th unit from cid on.  With the gradient, when one launch takes every unit, a
  // quarter of a wave of target-only rows (one cheap pass each) moves to the front, so
  // that a quarter of the clusters start their paired rows one short row later and the
  // clusters' first passes, exchanges and dz writes do not all fall in step; the other
  // target-only rows stay last, where they fill the final partial wave.
  const int early = (kGrad && P.unit_begin == 0 && P.unit_end == P.N_d + P.R) ? min(P.R, ncl / 4) : 0;
  auto unit_at = [&](int u) { return u < early ? P.N_d + u : (u < P.N_d + early ? u - early : u); };

  constexpr int kChunk = chunk_of<DZ, DT, kGrad>();
  constexpr int kGroupsPerThread = kChunk / 8 / kConsumers;  // 8-entry groups per consumer thread per chunk
  constexpr int kStageT = kChunk * DT::kBytes;
  constexpr int kZOff = StageLayout<DZ, DT, kGrad>::kZOff;
  constexpr int kStageBytes = StageLayout<DZ, DT, kGrad>::kBytes;
  // 128-byte aligned base for the bulk-copy ring (the launch adds 128 bytes of slack).
  uint8_t* ring =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  // One screening code per consumer thread and slot: slot c < #chunks covers the
  // thread's groups of ring chunk c, the slot after them one directly loaded group.
  uint16_t* codes = reinterpret_cast<uint16_t*>(ring + kStages * kStageBytes);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      // One local arrival per phase, made when the barrier is armed with the bytes it
      // expects (the peers' slices arrive as asynchronous-store transactions).  A
      // slot is armed for its next use right after its wait, before any peer can send
      // into it again; here for the first two uses.
      mbar_init(&part_bar[i], 1);
      mbar_init(&corr_bar[i], 1);
      mbar_arrive_expect_tx(&part_bar[i], static_cast<uint32_t>(C * sizeof(SlicePartial)));
      if (kGrad || rank == 0) mbar_arrive_expect_tx(&corr_bar[i], static_cast<uint32_t>(C * sizeof(SliceCorr)));
    }
    fence_barrier_init();
    s_abort = 0;
    s_unit_err = 0;
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrival

  // A bulk launch is a programmatic dependent of whatever the stream ran before it:
  // nothing in global memory is touched before that grid has completed.  Only then
  // may the kernels that follow (a tail launch, the acceptance scan / loss kernel)
  // be scheduled; they wait for this grid before reading what it writes.
  if (!P.wait_prior) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  volatile int* abort_flag = &s_abort;

  if (warp == kConsumerWarps) {
    // ---------------- producer warp: runs ahead across units ----------------
    if (lane == 0) {
      uint32_t cc = 0;
      uint64_t keep = 0, drop = 0;
      if (kGrad) {
        keep = l2_policy_evict_last();
        drop = l2_policy_evict_first();
      }
      for (int u = P.unit_begin + cid; u < num_units && !*abort_flag; u += ncl) {
        const Unit U = map_unit(P, unit_at(u));
        const uint8_t* zrow =
            U.pair ? static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(U.d) * P.ld_z * DZ::kBytes : nullptr;
        const uint8_t* trow =
            static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(max(U.s, 0)) * P.ld_t * DT::kBytes;
        const RowGeom G = row_geom<DZ, DT, kShift>(zrow, trow, P.V);
        const int v_begin = static_cast<int>(rank) * P.slice;  // in the body
        const int v_end = U.bad ? v_begin : min(P.V - G.H, v_begin + P.slice);
        const int body = max(0, v_end - v_begin) & ~7;
        const int zshift = 2 * G.zs2;  // bytes past the 16-byte boundary below the draft body
        const int passes = (kGrad && U.pair && !U.bad) ? 2 : 1;
        const int nch = (body + kChunk - 1) / kChunk;
        for (int pass = 0; pass < passes && !*abort_flag; ++pass) {
          for (int ci = 0; ci < nch; ++ci, ++cc) {
            const int e0 = (pass == 1 ? second_pass_chunk<kStages>(ci, nch) : ci) * kChunk;
            const int st = static_cast<int>(cc % kStages);
            if (cc >= static_cast<uint32_t>(kStages) &&
                !mbar_wait_bounded(&empty_bar[st], ((cc / kStages) & 1) ^ 1)) {
              *abort_flag = 1;
              break;
            }
            if (pass == 1 && second_pass_reuses<kStages>(ci, nch)) {
              mbar_arrive(&full_bar[st]);  // the chunk is still in this stage
              continue;
            }
            const int n = min(kChunk, body - e0);
            const uint32_t bz = U.pair ? static_cast<uint32_t>(n * DZ::kBytes + (zshift ? 16 : 0)) : 0u;
            const uint32_t bt = static_cast<uint32_t>(n * DT::kBytes);
            mbar_arrive_expect_tx(&full_bar[st], bz + bt);
            uint8_t* stage = ring + st * kStageBytes;
            const uint8_t* zsrc = U.pair ? G.zb + static_cast<int64_t>(v_begin + e0) * DZ::kBytes - zshift : nullptr;
            const uint8_t* tsrc = G.tb + static_cast<int64_t>(v_begin + e0) * DT::kBytes;
            if (kGrad && U.pair) {
              // L2 priority: keep the first pass's lines for the second, then drop them
              // (and drop at once the chunks the second pass takes from the ring)
              const bool reused = pass == 0 && nch >= kStages && ci >= nch - kStages;
              const uint64_t pol = (pass == 0 && !reused) ? keep : drop;
              bulk_copy_g2s_hint(stage + kZOff, zsrc, bz, &full_bar[st], pol);
              bulk_copy_g2s_hint(stage, tsrc, bt, &full_bar[st], pol);
            } else {
              if (U.pair) bulk_copy_g2s(stage + kZOff, zsrc, bz, &full_bar[st]);
              bulk_copy_g2s(stage, tsrc, bt, &full_bar[st]);
            }
          }
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
    for (int u = P.unit_begin + cid; u < num_units; u += ncl, ++it) {
      const Unit U = map_unit(P, unit_at(u));
      const uint8_t* zrow =
          U.pair ? static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(U.d) * P.ld_z * DZ::kBytes : nullptr;
      const uint8_t* trow =
          static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(max(U.s, 0)) * P.ld_t * DT::kBytes;
      const RowGeom G = row_geom<DZ, DT, kShift>(zrow, trow, P.V);
      const int Vb = P.V - G.H;
      const int v_begin = static_cast<int>(rank) * P.slice;  // in the body
      const int v_end = U.bad ? v_begin : min(Vb, v_begin + P.slice);
      const int len = max(0, v_end - v_begin);
      const int ngroups = (len + 7) >> 3;
      // Direct group index ngroups stands for the head (rank 0 only).
      const int has_head = (rank == 0 && !U.bad && G.H > 0) ? 1 : 0;
      const int ngx = ngroups + has_head;
      const int body = len & ~7;
      const int gfirst = 1 + (v_begin >> 3);  // row-global index of the slice's first group

      Acc acc;
      acc_init(acc);
      if (U.pair) {
        // The draft body's shift picks the loop instance (uniform per unit).
        dispatch_shift<DZ, kShift>(G.zs2, [&](auto zs_c) {
          constexpr int ZS = decltype(zs_c)::value;
          for (int e0 = 0; e0 < body; e0 += kChunk, ++cc) {
            const int st = static_cast<int>(cc % kStages);
            if (!mbar_wait_bounded(&full_bar[st], (cc / kStages) & 1)) {
              atomicOr(&s_unit_err, 1);
              *abort_flag = 1;
              break;
            }
            const int gcount = min(kChunk, body - e0) >> 3;
            const uint8_t* stage = ring + st * kStageBytes;
            const uint32_t* zw = reinterpret_cast<const uint32_t*>(stage + kZOff);
            const int gbase = gfirst + (e0 >> 3);
            float cm = kNegInf;
#pragma unroll
            for (int k = 0; k < kGroupsPerThread; ++k) {
              const int g = tid + k * kConsumers;
              if (g < gcount) {
                float z[8], t[8], vmt;
                load8_shifted<DZ, ZS, false>(zw + g * 2 * DZ::kBytes, z);
                const float vmz = max8(z);
                load8_smem<DT>(stage, g, t, vmt);
                acc_pair_nc(acc, z, t, vmz, vmt, gbase + g);
                cm = fmaxf(cm, vmz);
              }
            }
            acc.cmax = fmaxf(acc.cmax, cm);
            codes[(e0 / kChunk) * kConsumers + tid] = code_up(cm);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[st]);
          }
        });
      } else {
        for (int e0 = 0; e0 < body; e0 += kChunk, ++cc) {
          const int st = static_cast<int>(cc % kStages);
          if (!mbar_wait_bounded(&full_bar[st], (cc / kStages) & 1)) {
            atomicOr(&s_unit_err, 1);
            *abort_flag = 1;
            break;
          }
          const int gcount = min(kChunk, body - e0) >> 3;
          const uint8_t* stage = ring + st * kStageBytes;
          const int gbase = gfirst + (e0 >> 3);
#pragma unroll
          for (int k = 0; k < kGroupsPerThread; ++k) {
            const int g = tid + k * kConsumers;
            if (g < gcount) {
              float t[8], vmt;
              load8_smem<DT>(stage, g, t, vmt);
              acc_target(acc, vmt, gbase + g);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[st]);
        }
      }
      // Direct loads: the ragged end of the slice and (rank 0) the head.  Group g is
      // always handled by consumer thread g mod kConsumers, so a thread's group maximum
      // covers exactly the groups it re-reads.
      const int nchunks = (body + kChunk - 1) / kChunk;
      const int gd0 = (body >> 3) + ((tid - (body >> 3)) & (kConsumers - 1));  // this thread's first direct group
      for (int g = gd0, slot = nchunks; g < ngx; g += kConsumers, ++slot) {
        const bool head = g == ngroups;
        const int v0 = head ? 0 : G.H + v_begin + (g << 3);
        const int n = head ? G.H : min(8, v_end - (v_begin + (g << 3)));
        const int grp = head ? 0 : gfirst + g;
        float t[8], vmt;
        load_global<DT>(trow, v0, n, t, vmt);
        if (U.pair) {
          float z[8], vmz;
          load_global<DZ>(zrow, v0, n, z, vmz);
          acc_pair(acc, z, t, vmz, vmt, grp);
          codes[slot * kConsumers + tid] = code_up(vmz);
        } else {
          acc_target(acc, vmt, grp);
        }
      }

      // ---- CTA reduction, then the exchange of slice partials ----
      const AccS as = warp_reduce(acc_fold(acc));
      if (lane == 0) {
        SlicePartial& w = warp_part[warp];
        w.nz = as.nz; w.sz = as.sz; w.szd = as.szd;
        w.nt = as.nt; w.st = as.st; w.mt = as.mt; w.dmax = as.dmax; w.bgrp = as.bgrp; w.err = 0;
        w.cmax = as.cmax;
      }
      named_bar_sync(kConsumers);

      const int buf = it & 1;
      if (tid == 0) {
        SlicePartial mine;
        combine_partials(warp_part, kConsumerWarps, mine);
        mine.err = s_unit_err;
        s_unit_err = 0;
        const float own_cmax = mine.cmax;
        for (int r = 0; r < C; ++r) st_async_to_rank(mine, &slots[buf][rank], &part_bar[buf], static_cast<uint32_t>(r));
        int werr = 0;
        if (!mbar_wait_cluster_bounded(&part_bar[buf], (it >> 1) & 1)) {
          werr = 1;
          *abort_flag = 1;
        }
        SlicePartial all;
        combine_partials(slots[buf], C, all);
        mbar_arrive_expect_tx(&part_bar[buf], static_cast<uint32_t>(C * sizeof(SlicePartial)));  // armed for unit it + 2
        // The lowest index of the maximum lies in the first group holding it.  With the
        // gradient, a pair row's index is found in the second pass by the thread that
        // holds that group (no re-read here).
        rc.bgrp = all.bgrp;
        rc.mt = all.mt;
        rc.argmax = (rank == 0 && !U.bad && !(kGrad && U.pair))
                        ? resolve_argmax_grid<DZ, DT>(trow, zrow, all.bgrp, all.mt, P.V, G.H, &rc.za)
                        : -1;
        rc.err = all.err | werr;
        rc.stop = *abort_flag;
        if (U.pair && !U.bad) {
          row_consts(all, rc);
          // Screen threshold on group maxima of z; the slack only adds candidates.
          const float R = all.dmax - rc.dlse;
          const float Rp = R + 1e-4f * (1.f + fabsf(all.dmax) + fabsf(rc.dlse));
          const float c = P.clip_c;
          if (!(c < INFINITY) || !(Rp > 0.f)) {
            rc.theta = INFINITY;
          } else {
            const float th = rc.lse_z + logf(c / Rp);
            rc.theta = th - (1e-3f + 1e-5f * fabsf(th));
          }
          rc.scan = own_cmax > rc.theta;
          // The same decision in every CTA of the cluster: with no group maximum
          // above theta anywhere in the row, no term can clip and the exchange of
          // corrections is skipped.
          rc.any_scan = all.cmax > rc.theta;
        } else {
          rc.scan = 0;
          rc.any_scan = 0;
        }
      }
      named_bar_sync(kConsumers);
      const bool stop = rc.stop != 0;  // read by every consumer thread from the same broadcast

      if (!U.pair) {
        if (rank == 0 && tid == 0) {
          if (U.bad) flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
          else if (rc.argmax < 0 || rc.argmax >= P.V) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
          else {
            P.target_argmax[U.s] = rc.argmax;
            if (rc.err) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
          }
        }
        if (stop) break;
        continue;
      }

      // Rank 0 writes the row's outputs from the row constants and the summed corrections.
      auto finish_row = [&](float corr_all, float sclip_all, int nclip_all, int err_all) {
        if (U.bad) {
          flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
        } else if (kGrad) {
          // the argmax and the cross-entropy come from the second pass
          const int64_t d = U.d;
          P.kl_row[d] = rc.kl_unclip - corr_all;
          P.row_stats[4 * d + 0] = rc.lse_z;
          P.row_stats[4 * d + 1] = rc.lse_t;
          P.row_stats[4 * d + 2] = (rc.kl_unclip + 1.f) - sclip_all;
          P.row_stats[4 * d + 3] = static_cast<float>(nclip_all);
          if (err_all || rc.bgrp < (G.H > 0 ? 0 : 1) || rc.bgrp > (Vb + 7) / 8)
            flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
        } else if (rc.argmax < 0 || rc.argmax >= P.V) {
          // only after an aborted unit (no group was reduced): nothing valid to write
          flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
        } else {
          const int a = rc.argmax;
          const int64_t d = U.d;
          P.kl_row[d] = rc.kl_unclip - corr_all;
          P.ce_row[d] = rc.lse_z - rc.za;
          P.row_stats[4 * d + 0] = rc.lse_z;
          P.row_stats[4 * d + 1] = rc.lse_t;
          P.row_stats[4 * d + 2] = (rc.kl_unclip + 1.f) - sclip_all;
          P.row_stats[4 * d + 3] = static_cast<float>(nclip_all);
          P.target_argmax[U.s] = a;
          if (err_all) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
        }
      };
      // Gradient coefficients of the row from the summed corrections (tid 0), the
      // same float32 expressions as the stored row statistics the backward reads.
      auto set_grad = [&](float sclip_all) {
        const float S = (rc.kl_unclip + 1.f) - sclip_all;
        RowGrad k;
        k.tc = make_term_consts(rc.lse_z, rc.lse_t);
        k.c = P.clip_c;
        k.k_clip = __fsub_rn(P.ce_weight, S);
        k.k_m = __fadd_rn(1.0f, k.k_clip);
        k.g = P.grad_row ? __ldg(P.grad_row + U.d) : P.grad_scale;
        k.bg = __fmul_rn(P.ce_weight, k.g);
        k.lse_z = rc.lse_z;
        k.mt = rc.mt;
        const int ga = rc.bgrp - gfirst;  // slice-local group of the first max of t
        k.ga = (rc.bgrp >= 1 && ga >= 0 && ga < ngroups) ? ga : -1;
        k.head_arg = (has_head && rc.bgrp == 0) ? 1 : 0;
        k.stop = *abort_flag;
        s_grad = k;
      };
      if (!rc.any_scan) {
        if (rank == 0 && tid == 0) finish_row(0.f, 0.f, 0, rc.err);
        if constexpr (!kGrad) {
          if (stop) break;
          continue;
        } else {
          if (tid == 0) set_grad(0.f);
        }
      } else {

      // ---- exact evaluation of the screened groups ----
      float corr = 0.f, sclip = 0.f;
      int nclip = 0;
      {
        // A group can hold a clipped term only if its max z exceeds theta.  Each
        // thread compares the largest group maximum it saw with theta (rarely
        // above); only then does it walk its own codes and re-read, from global
        // memory, the groups of the slots whose code is above theta.
        const float theta = rc.theta;
        if (!U.bad && rc.scan && acc.cmax > theta) {
          const TermConsts tc = make_term_consts(rc.lse_z, rc.lse_t);
          const float c = P.clip_c;
          const int nslots = nchunks + (ngx > gd0 ? (ngx - gd0 + kConsumers - 1) / kConsumers : 0);
          for (int slot = 0; slot < nslots; ++slot) {
            if (!(code_value(codes[slot * kConsumers + tid]) > theta)) continue;
            for (int k = 0; k < (slot < nchunks ? kGroupsPerThread : 1); ++k) {
              int v0, n;
              if (slot < nchunks) {
                const int gl = tid + k * kConsumers;
                if (gl >= (min(kChunk, body - slot * kChunk) >> 3)) continue;
                const int g = slot * (kChunk / 8) + gl;
                v0 = G.H + v_begin + (g << 3);
                n = 8;
              } else {
                const int g = gd0 + (slot - nchunks) * kConsumers;
                if (g == ngroups) {
                  v0 = 0;
                  n = G.H;
                } else {
                  v0 = G.H + v_begin + (g << 3);
                  n = min(8, v_end - (v_begin + (g << 3)));
                }
              }
              float zs[8], ts[8];
              if (n == 8 && G.zs2 == 0 && v0 >= G.H) {
                load8_global_vec<DZ>(zrow, v0, zs);
                load8_global_vec<DT>(trow, v0, ts);
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  zs[j] = j < n ? DZ::load(zrow, v0 + j) : 0.f;
                  ts[j] = j < n ? DT::load(trow, v0 + j) : 0.f;
                }
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                if (j >= n) break;
                float p, r, term;
                entry_term(zs[j], ts[j], tc, p, r, term);  // the backward's evaluation, bit for bit
                if (term > c) {
                  corr += term - c;
                  sclip = fmaf(p, r + 1.f, sclip);
                  ++nclip;
                }
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
        mine.corr = 0.f; mine.sclip = 0.f; mine.nclip = 0; mine.err = rc.err;
        for (int w = 0; w < kConsumerWarps; ++w) {
          mine.corr += warp_corr[w][0];
          mine.sclip += warp_corr[w][1];
          mine.nclip += warp_nclip[w];
        }
        // To rank 0 only; with the gradient, to every CTA (each needs S).
        const int nto = kGrad ? C : 1;
        for (int r = 0; r < nto; ++r)
          st_async_to_rank(mine, &cslots[cbuf][rank], &corr_bar[cbuf], static_cast<uint32_t>(r));
        if (kGrad || rank == 0) {
          const bool ok = mbar_wait_cluster_bounded(&corr_bar[cbuf], (pit >> 1) & 1);
          if (!ok) *abort_flag = 1;
          float corr_all = 0.f, sclip_all = 0.f;
          int nclip_all = 0, err_all = rc.err | (ok ? 0 : 1);
          for (int r = 0; r < C; ++r) {
            corr_all += cslots[cbuf][r].corr;
            sclip_all += cslots[cbuf][r].sclip;
            nclip_all += cslots[cbuf][r].nclip;
            err_all |= cslots[cbuf][r].err;
          }
          mbar_arrive_expect_tx(&corr_bar[cbuf], static_cast<uint32_t>(C * sizeof(SliceCorr)));  // armed for pit + 2
          if (rank == 0) finish_row(corr_all, sclip_all, nclip_all, err_all);
          if (kGrad) set_grad(sclip_all);
        }
      }
      ++pit;
      }  // any_scan
      if constexpr (kGrad) {
        named_bar_sync(kConsumers);  // s_grad is set
        if (stop || s_grad.stop) break;
        if (!U.bad) {
          // ---- second pass over the slice (from L2): dz, written once ----
          const RowGrad k = s_grad;
          float* grow = P.grad + static_cast<int64_t>(U.d) * P.ld_g;  // the row
          float* gbody = grow + G.H + v_begin;                          // this slice of the body
          const int gq = static_cast<int>((reinterpret_cast<uintptr_t>(gbody) >> 2) & 3u);
          const int nch = (body + kChunk - 1) / kChunk;
          dispatch_shift<DZ, kShift>(G.zs2, [&](auto zs_c) {
            constexpr int ZS = decltype(zs_c)::value;
            for (int ci = 0; ci < nch; ++ci, ++cc) {
              const int e0 = second_pass_chunk<kStages>(ci, nch) * kChunk;  // the producer's second-pass order
              const int st = static_cast<int>(cc % kStages);
              if (!mbar_wait_bounded(&full_bar[st], (cc / kStages) & 1)) {
                atomicOr(&s_unit_err, 1);
                *abort_flag = 1;
                break;
              }
              const int gcount = min(kChunk, body - e0) >> 3;
              const uint8_t* stage = ring + st * kStageBytes;
              const uint32_t* zw = reinterpret_cast<const uint32_t*>(stage + kZOff);
#pragma unroll
              for (int kk = 0; kk < kGroupsPerThread; ++kk) {
                const int g = tid + kk * kConsumers;
                if (g < gcount) {
                  float z[8], t[8], out[8], vm;
                  load8_shifted<DZ, ZS, false>(zw + g * 2 * DZ::kBytes, z);
                  load8_smem<DT>(stage, g, t, vm);
                  // packed for float32 drafts (512 requests at V = 151937, float32 draft /
                  // bf16 target: 2.461 -> 2.436 ms); the scalar loop for bf16 drafts (128
                  // requests at V = 151936, bf16: 220.6 against 221.7 us packed)
                  if constexpr (DZ::kBytes == 4) {
                    grad_of8(z, t, k, out);
                  } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) out[e] = grad_of(z[e], t[e], k);
                  }
                  store8_stream<kShift>(gbody + e0 + (g << 3), gq, out);
                }
              }
              // The group holding the first max of t: the thread that just wrote it finds
              // the index, rewrites that entry with the hard-label term (program order makes
              // it the final value) and writes the argmax and the cross-entropy.
              const int lc = k.ga - (e0 >> 3);
              if (lc >= 0 && lc < gcount && tid == (lc & (kConsumers - 1))) {
                float zz[8], tt[8], vm;
                load8_shifted<DZ, ZS, false>(zw + lc * 2 * DZ::kBytes, zz);
                load8_smem<DT>(stage, lc, tt, vm);
                int j = -1;
                float zj = 0.f, tj = 0.f;
#pragma unroll
                for (int e = 7; e >= 0; --e)
                  if (tt[e] == k.mt) {
                    j = e;
                    zj = zz[e];
                    tj = tt[e];
                  }
                if (j >= 0) {
                  const int la = e0 + (lc << 3) + j;
                  gbody[la] = __fsub_rn(grad_of(zj, tj, k), k.bg);
                  P.target_argmax[U.s] = G.H + v_begin + la;
                  P.ce_row[U.d] = k.lse_z - zj;
                } else {
                  flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
                }
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(&empty_bar[st]);
            }
          });
          // The ragged end of the slice (fewer than 8 entries) and, in rank 0, the head,
          // straight from global memory; each entry is written by one thread, the argmax
          // by the thread holding it (the first entry of its group equal to the max).
          auto direct_entry = [&](int v, int g0, bool arg_group) {
            const float zv = DZ::load(zrow, v), tv = DT::load(trow, v);
            float o = grad_of(zv, tv, k);
            if (arg_group && tv == k.mt) {
              bool first = true;
              for (int u2 = g0; u2 < v; ++u2) first = first && !(DT::load(trow, u2) == k.mt);
              if (first) {
                o = __fsub_rn(o, k.bg);
                P.target_argmax[U.s] = v;
                P.ce_row[U.d] = k.lse_z - zv;
              }
            }
            grow[v] = o;
          };
          for (int v = body + tid; v < len; v += kConsumers)
            direct_entry(G.H + v_begin + v, G.H + v_begin + body, k.ga == (body >> 3));
          if (has_head)
            for (int v = tid; v < G.H; v += kConsumers) direct_entry(v, 0, k.head_arg != 0);
        }
      } else {
        if (stop) break;
      }
    }
    if (*abort_flag && tid == 0) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
  }

  __syncthreads();
  cluster_sync_all();  // no CTA leaves while a peer may still address its shared memory
  // A tail launch finishes only after the bulk launch before it, so whatever waits
  // on this launch also sees every unit of the bulk launch.
  if (P.wait_prior) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Entries of a row per CTA of the forward row pass, at most (V = 151936 gives one
// CTA per row when the batch fills the GPU).
constexpr int kSliceTarget = 160000;

int rowpass_cluster_size(int vocab, int units, int num_sms) {
  // At most kSliceTarget entries per CTA, and enough CTAs in
  // flight to fill the GPU (the resident CTAs per SM) when there are few rows; at most 8 (the
  // portable cluster size).
  int c = (vocab + kSliceTarget - 1) / kSliceTarget;
  if (c < 1) c = 1;
  while (c < kMaxCluster && static_cast<long long>(units) * c < static_cast<long long>(kFwdMinBlocks) * num_sms) ++c;
  return c > kMaxCluster ? kMaxCluster : c;
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
std::mutex g_occ_mu;
OccEntry g_occ[256];
int g_occ_n = 0;
}  // namespace

static int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  const int known = (dev >= 0 && dev < 64) ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (known) return known;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 152;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <class DZ, class DT, bool kGrad>
static size_t rowpass_smem(int slice) {
  constexpr int kChunk = chunk_of<DZ, DT, kGrad>();
  constexpr int kConsumers = RowCfg<kGrad>::kConsumers;
  const size_t ring = static_cast<size_t>(stages_of<DZ, DT, kGrad>()) * StageLayout<DZ, DT, kGrad>::kBytes;
  // screening codes: per consumer thread one slot per ring chunk, +1 for its one
  // directly loaded group (the ragged end of the slice or the head)
  const int slots = (slice + kChunk - 1) / kChunk + 1;
  return 128 + ring + static_cast<size_t>(slots) * kConsumers * sizeof(uint16_t);
}

// Co-resident clusters of this kernel at this cluster size (cached).
template <class DZ, class DT, bool kGrad, bool kShift>
static int active_clusters(int cluster, size_t smem) {
  auto kern = rowpass_kernel<DZ, DT, kGrad, kShift>;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return 1;
  {
    std::lock_guard<std::mutex> lock(g_occ_mu);
    for (int i = 0; i < g_occ_n; ++i)
      if (g_occ[i].fn == reinterpret_cast<const void*>(kern) && g_occ[i].smem == smem &&
          g_occ[i].cluster == cluster && g_occ[i].device == device)
        return g_occ[i].clusters;
  }
  // The query must see the shared-memory size the launch will use.
  if (raise_smem_limit(reinterpret_cast<const void*>(kern), smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(RowCfg<kGrad>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    n = sm_count() / cluster;  // one CTA per SM: always resident
    if (n < 1) n = 1;
  }
  std::lock_guard<std::mutex> lock(g_occ_mu);
  if (g_occ_n < 256) g_occ[g_occ_n++] = OccEntry{reinterpret_cast<const void*>(kern), smem, cluster, device, n};
  return n;
}

// One launch over units [p.unit_begin, p.unit_end), persistent clusters.
template <class DZ, class DT, bool kGrad, bool kShift>
static cudaError_t launch_range(const RowPassParams& p, bool programmatic, cudaStream_t stream) {
  const size_t smem = rowpass_smem<DZ, DT, kGrad>(p.slice);
  auto kern = rowpass_kernel<DZ, DT, kGrad, kShift>;
  const int units = p.unit_end - p.unit_begin;
  if (units <= 0) return cudaSuccess;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int clusters = active_clusters<DZ, DT, kGrad, kShift>(p.cluster, smem);
  cudaLaunchConfig_t cfg = {};
  const int grid_clusters = units < clusters ? units : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(grid_clusters) * static_cast<unsigned>(p.cluster), 1, 1);
  cfg.blockDim = dim3(RowCfg<kGrad>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Clusters placed for load balance rather than the default placement: measured on
  // GB300 (V = 151936, bf16), the step 220.3 -> 219.4 us on 128 requests and 80.7 ->
  // 78.6 us on 32, the forward 103.2 -> 102.1 us on 128 ("spread": no change).
  attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  attr[1].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
  attr[2].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[2].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 3 : 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Whole waves of units run at the requested cluster size; when the units do not
// fill the last wave, the remainder (the last rows, and the cheap target-only
// rows) runs as a second launch with larger clusters, so its rows are split
// over more CTAs instead of leaving a few CTAs to finish whole rows alone (with
// the gradient, a remainder of target-only rows only stays in the first launch).
// Every launch is programmatic: the first one waits for the stream's previous
// kernel before touching global memory; a second one starts as CTAs of the first
// retire and completes only after the first.
template <class DZ, class DT, bool kGrad, bool kShift>
static cudaError_t launch_one(const RowPassParams& p0, cudaStream_t stream) {
  const int units = (p0.mode == kModeVerify) ? p0.N_t : (p0.N_d + p0.R);
  if (units <= 0) return cudaSuccess;
  RowPassParams p = p0;
  p.unit_begin = 0;
  p.unit_end = units;
  p.wait_prior = 0;
  const int clusters = active_clusters<DZ, DT, kGrad, kShift>(p.cluster, rowpass_smem<DZ, DT, kGrad>(p.slice));
  const int split = (units / clusters) * clusters;
  // With the gradient, a last partial wave of target-only rows (cheap: no second pass)
  // stays in the one launch rather than costing a launch of its own.
  if (units <= clusters || split == units || p.cluster >= kMaxCluster ||
      (kGrad && p0.mode == kModeFwd && split >= p0.N_d))
    return launch_range<DZ, DT, kGrad, kShift>(p, true, stream);
  const RowPassParams base = p;
  p.unit_end = split;
  cudaError_t e = launch_range<DZ, DT, kGrad, kShift>(p, true, stream);
  if (e != cudaSuccess) return e;
  auto launch_tail = [&](int b, int end) {
    RowPassParams tail = base;
    tail.unit_begin = b;
    tail.unit_end = end;
    tail.wait_prior = 1;
    // the largest cluster that still fits all of the tail's rows in one wave (filling
    // the GPU instead took a second partial wave: 110.4 against 106.7 us for the
    // forward on a 128-request batch at V = 151936)
    const long long cap = static_cast<long long>(RowCfg<kGrad>::kMinBlocks) * sm_count();
    int c = 1;
    while (c < kMaxCluster && static_cast<long long>(end - b) * (c + 1) <= cap) ++c;
    tail.cluster = c;
    if (tail.cluster < p.cluster) tail.cluster = p.cluster;
    tail.slice = rowpass_slice(p.V, tail.cluster);
    return launch_range<DZ, DT, kGrad, kShift>(tail, true, stream);
  };
  // With the gradient, leftover paired rows and the cheap target-only rows get their
  // own launches, so the few expensive rows are split over the larger clusters their
  // count allows.
  if (kGrad && p0.mode == kModeFwd && split < p0.N_d && p0.N_d < units) {
    e = launch_tail(split, p0.N_d);
    if (e != cudaSuccess) return e;
    return launch_tail(p0.N_d, units);
  }
  return launch_tail(split, units);
}

// The largest cluster size (from 8 down to 1, or to 2 with the gradient) whose resident
// clusters take `units` row units in one round: more CTAs per row shorten each row, and
// no partly empty second round follows; 0 when no size does.
//
// The forward and verification use it for any batch (the units are its rows): measured
// on GB300, k = 16 per request at V = 151936, bf16, forward / verification us per call
// (the fill-the-GPU rule of rowpass_cluster_size in brackets): 3 requests C = 5 15.5 /
// 13.1 (18.1 / 15.0); 4 requests C = 4 16.0 / 14.1 (19.1 / 15.4); 8 requests C = 2 20.6
// / 12.8 (25.7 / 15.5); 16 requests C = 1 35.4 / 13.9 (41.4 / 17.9).
//
// The pass with the gradient uses it, counting paired rows only (the bonus rows, a
// quarter of a paired row's work each, may spill over), when every paired row fits the
// L2 budget at once: 3 requests C = 8 19.6 us (23.5 with the general rule's C = 6);
// 8 requests C = 4 40.5 (49.9); 4 and 6 requests unchanged (C = 8 and 6).
template <class DZ, class DT, bool kGrad, bool kShift>
static int one_round_cluster_t(int vocab, int units) {
  for (int c = kMaxCluster; c >= (kGrad ? 2 : 1); --c) {
    const size_t smem = rowpass_smem<DZ, DT, kGrad>(rowpass_slice(vocab, c));
    if (active_clusters<DZ, DT, kGrad, kShift>(c, smem) >= units) return c;
  }
  return 0;
}

template <bool kGrad, bool kShift>
static int one_round_cluster_dtypes(int z_dtype, int t_dtype, int vocab, int units) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (zb && tb) return one_round_cluster_t<BF16, BF16, kGrad, kShift>(vocab, units);
  if (!zb && tb) return one_round_cluster_t<F32, BF16, kGrad, kShift>(vocab, units);
  if (zb && !tb) return one_round_cluster_t<BF16, F32, kGrad, kShift>(vocab, units);
  return one_round_cluster_t<F32, F32, kGrad, kShift>(vocab, units);
}

int rowpass_one_round_cluster(int z_dtype, int t_dtype, bool aligned, int vocab, int units) {
  return aligned ? one_round_cluster_dtypes<false, false>(z_dtype, t_dtype, vocab, units)
                 : one_round_cluster_dtypes<false, true>(z_dtype, t_dtype, vocab, units);
}

int rowpass_grad_one_round_cluster(int z_dtype, int t_dtype, bool aligned, int vocab, int pairs) {
  return aligned ? one_round_cluster_dtypes<true, false>(z_dtype, t_dtype, vocab, pairs)
                 : one_round_cluster_dtypes<true, true>(z_dtype, t_dtype, vocab, pairs);
}

int rowpass_grad_cluster_size(int vocab, int units, int row_bytes, int chunk_entries, int num_sms, long long l2_bytes) {
  // The row pass's size, then at least 6 CTAs while each CTA's slice still holds four
  // ring chunks (C = 6 measured best on GB300 for bf16 rows and for fp32-draft /
  // bf16-target rows at V = 151936, against 4, 5, 7 and 8: more CTAs per row make the
  // per-row exchanges more frequent per byte, fewer put more rows in flight), then
  // raised until the rows in flight at once (resident CTAs / C rows of row_bytes) fit
  // three quarters of the L2, so that the second pass over each slice is served from L2.
  int c = rowpass_cluster_size(vocab, units, num_sms);
  const int floor_c = std::min(6, std::max(1, vocab / (4 * chunk_entries)));
  if (c < floor_c) c = floor_c;
  const long long budget = (l2_bytes > 0 ? l2_bytes : (126ll << 20)) * 3 / 4;
  while (c < kMaxCluster && static_cast<long long>(RowCfg<true>::kMinBlocks) * num_sms / c * row_bytes > budget) ++c;
  return c;
}

int rowpass_grad_chunk(int z_dtype, int t_dtype) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (zb && tb) return chunk_of<BF16, BF16, true>();
  if (!zb && tb) return chunk_of<F32, BF16, true>();
  if (zb && !tb) return chunk_of<BF16, F32, true>();
  return chunk_of<F32, F32, true>();
}

template <bool kGrad, bool kShift>
static cudaError_t launch_dtypes(const RowPassParams& p, int z_dtype, int t_dtype, cudaStream_t s) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (zb && tb) return launch_one<BF16, BF16, kGrad, kShift>(p, s);
  if (!zb && tb) return launch_one<F32, BF16, kGrad, kShift>(p, s);
  if (zb && !tb) return launch_one<BF16, F32, kGrad, kShift>(p, s);
  return launch_one<F32, F32, kGrad, kShift>(p, s);
}

cudaError_t launch_rowpass_grad(const RowPassParams& p, int z_dtype, int t_dtype, bool aligned, cudaStream_t s) {
  return aligned ? launch_dtypes<true, false>(p, z_dtype, t_dtype, s) : launch_dtypes<true, true>(p, z_dtype, t_dtype, s);
}

cudaError_t launch_rowpass(const RowPassParams& p, int z_dtype, int t_dtype, bool aligned, cudaStream_t s) {
  return aligned ? launch_dtypes<false, false>(p, z_dtype, t_dtype, s)
                 : launch_dtypes<false, true>(p, z_dtype, t_dtype, s);
}

}  // namespace adaflash
