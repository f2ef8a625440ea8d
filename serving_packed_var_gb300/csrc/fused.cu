// fused.cu -- K4: the forward and the backward of the OPD loss in one pass over each row.
//
// Training takes a step on the draft model right after each verification round
// (AdaFlash article, "AdaFlash: Adaptive Speculative Decoding with Online
// Self-Improvement for High-Concurrency LLM Inference", "On-Policy Distillation
// (OPD) for Domain Adaptation"); the target is fixed, so the gradient concerns the
// draft logits only.  The forward needs the final log-sum-exps of a row before any
// clipped term or gradient entry is known, so a purely streaming pass cannot write
// dz.  Here the row stays on chip instead: a cluster of C CTAs holds a (draft,
// target) row pair, each CTA its slice of z and t in shared memory (bulk copies on
// the TMA engine), and after the cluster has combined the slice statistics over
// distributed shared memory every CTA writes dz for its slice from shared memory.
// Each logit byte is read from HBM once for the whole training step, and dz is
// written once.
//
// The statistics, the clip screen and every output are those of the row pass (K1)
// and the backward (K3), with the same instruction sequences (rowstats.cuh,
// entry_term), so the outputs equal K1 + K3's bit for bit:
//   p = softmax(z), r_v = (z_v - t_v) - (lse_z - lse_t), term_v = p_v r_v,
//   KL = sum_v min(term_v, c),  S = sum_v [term_v <= c] p_v (r_v + 1),
//   dz_v = g ( p_v ([term_v <= c](r_v + 1) - S) + beta (p_v - [v == a]) ).
// Target-only units (the bonus rows) only find their argmax.
#include <algorithm>
#include <cfloat>
#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "rowstats.cuh"

namespace adaflash {

namespace {

constexpr int kFThreads = 256;  // a power of two
constexpr int kFWarps = kFThreads / 32;
constexpr uint32_t kPiece = 16384;  // bytes per bulk copy
// The shared-memory budget: two resident CTAs per SM (a slice of a bf16 pair at
// V = 151936 then needs clusters of 6).
constexpr int kFCtasPerSm = 2;
// The fused kernel takes batches whose clusters all run at once with one CTA per SM:
// with two CTAs on an SM its phases, one after another inside each CTA, leave the HBM
// stream idle, and the row pass with the gradient is faster (k = 16 per request at
// V = 151936, bf16, graph-replayed: one request 16.4 us fused against 18.4; two
// requests 22.5 fused against 20.5; a 128-request batch 384 us against 219.8).
constexpr size_t kSmemPerSm = 227 * 1024;
constexpr size_t kStaticReserve = 4096;  // static shared memory and the per-CTA reservation

struct GradCoef {
  TermConsts tc;
  float c;
  float k_m;     // 1 + beta - S   (inner factor where the term is kept: r + k_m)
  float k_clip;  // beta - S       (inner factor where the term is clipped)
  float g;
  float bg;      // beta * g, taken off at the argmax
};

__device__ __forceinline__ float grad_entry(float z, float t, const GradCoef& k) {
  float p, r, term;
  entry_term(z, t, k.tc, p, r, term);
  const float inner = (term <= k.c) ? __fadd_rn(r, k.k_m) : k.k_clip;
  return __fmul_rn(__fmul_rn(p, inner), k.g);
}

__host__ __device__ constexpr size_t round128(size_t x) { return (x + 127) & ~static_cast<size_t>(127); }

// Entry i of a slice held in shared memory.
template <class DT>
__device__ __forceinline__ float load_smem_entry(const uint8_t* buf, int i);
template <>
__device__ __forceinline__ float load_smem_entry<BF16>(const uint8_t* buf, int i) {
  return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(buf)[i]) << 16);
}
template <>
__device__ __forceinline__ float load_smem_entry<F32>(const uint8_t* buf, int i) {
  return reinterpret_cast<const float*>(buf)[i];
}

template <class DZ, class DT>
__host__ __device__ constexpr size_t fused_smem(int slice) {
  return 128 + round128(static_cast<size_t>(slice) * DZ::kBytes) + static_cast<size_t>(slice) * DT::kBytes;
}

}  // namespace

template <class DZ, class DT>
__global__ void __launch_bounds__(kFThreads, kFCtasPerSm) fused_kernel(const RowPassParams P) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar;
  __shared__ uint64_t part_bar[2];
  __shared__ uint64_t corr_bar[2];
  __shared__ SlicePartial slots[2][kMaxCluster];
  __shared__ SliceCorr cslots[2][kMaxCluster];
  __shared__ SlicePartial warp_part[kFWarps];
  __shared__ float warp_corr[kFWarps][2];
  __shared__ int warp_nclip[kFWarps];
  __shared__ RowConsts rc;
  __shared__ float s_mt;
  __shared__ int s_bgrp;
  __shared__ float s_corr_all, s_sclip_all;
  __shared__ int s_nclip_all, s_err_all;
  __shared__ int s_abort;

  // The acceptance scan / loss kernel that follows may be scheduled now; it waits
  // for this grid's completion before reading what this grid writes.
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int C = P.cluster;
  const int cid = static_cast<int>(blockIdx.x) / C;
  const int ncl = static_cast<int>(gridDim.x) / C;
  const int slice = P.slice;

  uint8_t* zbuf =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  uint8_t* tbuf = zbuf + round128(static_cast<size_t>(slice) * DZ::kBytes);

  if (tid == 0) {
    mbar_init(&full_bar, 1);
    for (int i = 0; i < 2; ++i) {
      // one local arrival per phase, made when armed with the expected bytes (the
      // peers' slices arrive as asynchronous-store transactions); re-armed after each wait
      mbar_init(&part_bar[i], 1);
      mbar_init(&corr_bar[i], 1);
      mbar_arrive_expect_tx(&part_bar[i], static_cast<uint32_t>(C * sizeof(SlicePartial)));
      mbar_arrive_expect_tx(&corr_bar[i], static_cast<uint32_t>(C * sizeof(SliceCorr)));
    }
    fence_barrier_init();
    s_abort = 0;
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrival

  uint32_t phase = 0;     // parity of full_bar's next phase
  bool in_flight = false;  // (thread 0) copies issued whose phase was not consumed
  int it = 0, pit = 0;
  for (int u = P.unit_begin + cid; u < P.unit_end; u += ncl, ++it) {
    const Unit U = map_unit(P, u);
    const int v_begin = static_cast<int>(rank) * slice;
    const int v_end = U.bad ? v_begin : min(P.V, v_begin + slice);
    const int len = max(0, v_end - v_begin);
    const int ngroups = (len + 7) >> 3;
    const int body = len & ~7;
    const int nbody = body >> 3;  // groups held in shared memory
    const uint8_t* zrow =
        U.pair ? static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(U.d) * P.ld_z * DZ::kBytes : nullptr;
    const uint8_t* trow = static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(max(U.s, 0)) * P.ld_t * DT::kBytes;

    // ---- the slice of z and t into shared memory (the previous unit's readers are done) ----
    if (body > 0) {
      if (tid == 0) {
        const uint32_t bz = U.pair ? static_cast<uint32_t>(body * DZ::kBytes) : 0u;
        const uint32_t bt = static_cast<uint32_t>(body * DT::kBytes);
        mbar_arrive_expect_tx(&full_bar, bz + bt);
        for (uint32_t off = 0; off < bz; off += kPiece)
          bulk_copy_g2s(zbuf + off, zrow + static_cast<int64_t>(v_begin) * DZ::kBytes + off,
                        bz - off < kPiece ? bz - off : kPiece, &full_bar);
        for (uint32_t off = 0; off < bt; off += kPiece)
          bulk_copy_g2s(tbuf + off, trow + static_cast<int64_t>(v_begin) * DT::kBytes + off,
                        bt - off < kPiece ? bt - off : kPiece, &full_bar);
        in_flight = true;
      }
      if (!mbar_wait_bounded(&full_bar, phase)) {
        s_abort = 1;
      } else if (tid == 0) {
        in_flight = false;
      }
      phase ^= 1u;
    }

    // ---- slice statistics: groups g = tid, tid + kFThreads, ... from shared memory ----
    Acc acc;
    acc_init(acc);
    const int gbase = v_begin >> 3;
    if (U.pair) {
      for (int g = tid; g < nbody; g += kFThreads) {
        float z[8], t[8], vmz, vmt;
        load8_smem<DZ>(zbuf, g, z, vmz);
        load8_smem<DT>(tbuf, g, t, vmt);
        acc_pair(acc, z, t, vmz, vmt, gbase + g);
      }
    } else {
      for (int g = tid; g < nbody; g += kFThreads) {
        float t[8], vmt;
        load8_smem<DT>(tbuf, g, t, vmt);
        acc_target(acc, vmt, gbase + g);
      }
    }
    // the ragged last group (fewer than 8 entries) straight from global memory
    const bool has_tail = ngroups > nbody;
    const int tail_tid = nbody & (kFThreads - 1);
    if (has_tail && tid == tail_tid) {
      const int n = len - body;
      float t[8], vmt;
      load_global<DT>(trow, v_begin + body, n, t, vmt);
      if (U.pair) {
        float z[8], vmz;
        load_global<DZ>(zrow, v_begin + body, n, z, vmz);
        acc_pair(acc, z, t, vmz, vmt, gbase + nbody);
      } else {
        acc_target(acc, vmt, gbase + nbody);
      }
    }

    // ---- CTA reduction, then the exchange of slice partials (every CTA gets all) ----
    const AccS as = warp_reduce(acc_fold(acc));
    if (lane == 0) {
      SlicePartial& w = warp_part[warp];
      w.nz = as.nz; w.sz = as.sz; w.szd = as.szd;
      w.nt = as.nt; w.st = as.st; w.mt = as.mt; w.dmax = as.dmax; w.bgrp = as.bgrp; w.err = 0;
      w.cmax = as.cmax;
    }
    __syncthreads();
    const int buf = it & 1;
    if (tid == 0) {
      SlicePartial mine;
      combine_partials(warp_part, kFWarps, mine);
      mine.err = s_abort;
      for (int r = 0; r < C; ++r) st_async_to_rank(mine, &slots[buf][rank], &part_bar[buf], static_cast<uint32_t>(r));
      int werr = 0;
      if (!mbar_wait_cluster_bounded(&part_bar[buf], (it >> 1) & 1)) {
        werr = 1;
        s_abort = 1;
      }
      SlicePartial all;
      combine_partials(slots[buf], C, all);
      mbar_arrive_expect_tx(&part_bar[buf], static_cast<uint32_t>(C * sizeof(SlicePartial)));  // armed for unit it + 2
      s_mt = all.mt;
      s_bgrp = all.bgrp;
      rc.err = all.err | werr;
      // The lowest index of the maximum lies in the first group holding it; the CTA
      // whose slice holds that group resolves it (from shared memory when it can).
      int a = -1;
      const int lg = all.bgrp - gbase;
      if (!U.bad && lg >= 0 && lg < ngroups) {
        if (lg < nbody) {
          float t[8], vmt;
          load8_smem<DT>(tbuf, lg, t, vmt);
          for (int j = 7; j >= 0; --j)
            if (t[j] == all.mt) a = (all.bgrp << 3) + j;
        } else {
          a = resolve_argmax<DT>(trow, all.bgrp, all.mt, P.V);
        }
      }
      rc.argmax = a;
      rc.stop = s_abort;
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
        // The same decision in every CTA of the cluster.
        rc.any_scan = all.cmax > rc.theta;
      } else {
        rc.any_scan = 0;
      }
    }
    __syncthreads();

    if (!U.pair) {
      if (tid == 0) {
        if (U.bad) {
          if (rank == 0) flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
        } else if (rc.argmax >= 0) {
          if (rc.argmax < P.V) P.target_argmax[U.s] = rc.argmax;
          if (rc.err) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
        }
      }
    } else {
      // ---- exact evaluation of the screened groups, summed over the cluster ----
      if (rc.any_scan) {
        float corr = 0.f, sclip = 0.f;
        int nclip = 0;
        const float theta = rc.theta;
        if (!U.bad && acc.cmax > theta) {
          const TermConsts tc = make_term_consts(rc.lse_z, rc.lse_t);
          const float c = P.clip_c;
          auto eval = [&](const float* z, const float* t, int n) {
            for (int j = 0; j < n; ++j) {
              float p, r, term;
              entry_term(z[j], t[j], tc, p, r, term);  // the backward's evaluation, bit for bit
              if (term > c) {
                corr += term - c;
                sclip = fmaf(p, r + 1.f, sclip);
                ++nclip;
              }
            }
          };
          for (int g = tid; g < nbody; g += kFThreads) {
            float z[8], t[8], vmz, vmt;
            load8_smem<DZ>(zbuf, g, z, vmz);
            if (!(vmz > theta)) continue;
            load8_smem<DT>(tbuf, g, t, vmt);
            eval(z, t, 8);
          }
          if (has_tail && tid == tail_tid) {
            const int n = len - body;
            float z[8], t[8], vmz, vmt;
            load_global<DZ>(zrow, v_begin + body, n, z, vmz);
            load_global<DT>(trow, v_begin + body, n, t, vmt);
            if (vmz > theta) eval(z, t, n);
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
        __syncthreads();
        const int cbuf = pit & 1;
        if (tid == 0) {
          SliceCorr mine;
          mine.corr = 0.f; mine.sclip = 0.f; mine.nclip = 0; mine.err = rc.err;
          for (int w = 0; w < kFWarps; ++w) {
            mine.corr += warp_corr[w][0];
            mine.sclip += warp_corr[w][1];
            mine.nclip += warp_nclip[w];
          }
          // every CTA needs S for its slice of dz: the corrections go to every rank
          for (int r = 0; r < C; ++r)
            st_async_to_rank(mine, &cslots[cbuf][rank], &corr_bar[cbuf], static_cast<uint32_t>(r));
          const bool ok = mbar_wait_cluster_bounded(&corr_bar[cbuf], (pit >> 1) & 1);
          if (!ok) s_abort = 1;
          float corr_all = 0.f, sclip_all = 0.f;
          int nclip_all = 0, err_all = rc.err | (ok ? 0 : 1);
          for (int r = 0; r < C; ++r) {
            corr_all += cslots[cbuf][r].corr;
            sclip_all += cslots[cbuf][r].sclip;
            nclip_all += cslots[cbuf][r].nclip;
            err_all |= cslots[cbuf][r].err;
          }
          mbar_arrive_expect_tx(&corr_bar[cbuf], static_cast<uint32_t>(C * sizeof(SliceCorr)));  // armed for pit + 2
          s_corr_all = corr_all;
          s_sclip_all = sclip_all;
          s_nclip_all = nclip_all;
          s_err_all = err_all;
        }
        ++pit;
        __syncthreads();
      } else if (tid == 0) {
        s_corr_all = 0.f;
        s_sclip_all = 0.f;
        s_nclip_all = 0;
        s_err_all = rc.err;
      }
      __syncthreads();

      const float S = (rc.kl_unclip + 1.f) - s_sclip_all;
      const int a = rc.argmax;  // valid only in the CTA whose slice holds it
      if (tid == 0 && !U.bad) {
        const int64_t d = U.d;
        if (rank == 0) {
          P.kl_row[d] = rc.kl_unclip - s_corr_all;
          P.row_stats[4 * d + 0] = rc.lse_z;
          P.row_stats[4 * d + 1] = rc.lse_t;
          P.row_stats[4 * d + 2] = S;
          P.row_stats[4 * d + 3] = static_cast<float>(s_nclip_all);
          if (s_err_all) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
        }
        if (a >= 0 && a < P.V) {
          const int la = a - v_begin;
          const float za = (la < body) ? load_smem_entry<DZ>(zbuf, la) : DZ::load(zrow, a);
          P.ce_row[d] = rc.lse_z - za;
          P.target_argmax[U.s] = a;
        }
      }
      if (U.bad) {
        if (rank == 0 && tid == 0) flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
      } else {
        // ---- dz for this slice, from shared memory ----
        GradCoef k;
        k.tc = make_term_consts(rc.lse_z, rc.lse_t);
        k.c = P.clip_c;
        k.k_clip = __fsub_rn(P.ce_weight, S);
        k.k_m = __fadd_rn(1.0f, k.k_clip);
        k.g = P.grad_row ? __ldg(P.grad_row + U.d) : P.grad_scale;
        k.bg = __fmul_rn(P.ce_weight, k.g);
        float* grow = P.grad + static_cast<int64_t>(U.d) * P.ld_g + v_begin;
        const int la = (a >= 0) ? a - v_begin : -1;
        for (int g = tid; g < nbody; g += kFThreads) {
          float z[8], t[8], vmz, vmt, out[8];
          load8_smem<DZ>(zbuf, g, z, vmz);
          load8_smem<DT>(tbuf, g, t, vmt);
#pragma unroll
          for (int e = 0; e < 8; ++e) out[e] = grad_entry(z[e], t[e], k);
          if ((la >> 3) == g) out[la & 7] = __fsub_rn(out[la & 7], k.bg);
          float4* dst = reinterpret_cast<float4*>(grow + (g << 3));
          __stcs(dst, make_float4(out[0], out[1], out[2], out[3]));
          __stcs(dst + 1, make_float4(out[4], out[5], out[6], out[7]));
        }
        if (has_tail && tid == tail_tid) {
          for (int v = body; v < len; ++v) {
            float o = grad_entry(DZ::load(zrow, v_begin + v), DT::load(trow, v_begin + v), k);
            if (v == la) o = __fsub_rn(o, k.bg);
            grow[v] = o;
          }
        }
      }
    }
    __syncthreads();  // shared memory is free for the next unit's copies
    if (s_abort) break;
  }
  if (s_abort && tid == 0) {
    flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
    // let copies still in flight land before the CTA can exit
    if (in_flight) mbar_wait_bounded(&full_bar, phase ^ 1u, 100000000ull);
  }
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while a peer may still address its shared memory
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

struct FOcc {
  const void* fn;
  int cluster;
  size_t smem;
  int device;
  int clusters;
};
std::mutex g_focc_mu;
FOcc g_focc[64];
int g_focc_n = 0;
}  // namespace

// Smallest cluster whose slices fit the shared-memory budget of kFCtasPerSm CTAs per
// SM (else of one CTA per SM); 0 when even 8 do not fit.
int fused_cluster_size(int vocab, int bytes_per_entry) {
  for (int pass = 0; pass < 2; ++pass) {
    const size_t budget = (pass == 0 ? kSmemPerSm / kFCtasPerSm : kSmemPerSm) - kStaticReserve;
    for (int c = 1; c <= kMaxCluster; ++c) {
      const int slice = rowpass_slice(vocab, c);
      // z and t share the slice; round128 of the z part adds at most 128 bytes
      if (static_cast<size_t>(slice) * bytes_per_entry + 256 <= budget) return c;
    }
  }
  return 0;
}

// Co-resident clusters of the fused kernel at cluster size C (cached per device).
template <class DZ, class DT>
static int fused_resident_clusters(int C, size_t smem, int num_sms) {
  auto kern = fused_kernel<DZ, DT>;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(g_focc_mu);
    for (int i = 0; i < g_focc_n; ++i)
      if (g_focc[i].fn == reinterpret_cast<const void*>(kern) && g_focc[i].cluster == C && g_focc[i].smem == smem &&
          g_focc[i].device == device)
        return g_focc[i].clusters;
  }
  if (raise_smem_limit(reinterpret_cast<const void*>(kern), smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C), 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
    (void)cudaGetLastError();
    clusters = num_sms / C;  // one CTA per SM: always resident
    if (clusters < 1) clusters = 1;
  }
  std::lock_guard<std::mutex> lock(g_focc_mu);
  if (g_focc_n < 64) g_focc[g_focc_n++] = FOcc{reinterpret_cast<const void*>(kern), C, smem, device, clusters};
  return clusters;
}

template <class DZ, class DT>
static int fused_max_units_t(int vocab, int num_sms) {
  const int C = fused_cluster_size(vocab, DZ::kBytes + DT::kBytes);
  if (C == 0) return 0;
  return std::min(fused_resident_clusters<DZ, DT>(C, fused_smem<DZ, DT>(rowpass_slice(vocab, C)), num_sms),
                  num_sms / C);
}

template <class DZ, class DT>
static cudaError_t launch_fused_t(const RowPassParams& p0, int num_sms, cudaStream_t stream) {
  RowPassParams p = p0;
  const int units = p.N_d + p.R;
  if (units <= 0) return cudaSuccess;
  const int C = fused_cluster_size(p.V, DZ::kBytes + DT::kBytes);
  if (C == 0) return cudaErrorNotSupported;
  p.cluster = C;
  p.slice = rowpass_slice(p.V, C);
  p.unit_begin = 0;
  p.unit_end = units;
  const size_t smem = fused_smem<DZ, DT>(p.slice);
  auto kern = fused_kernel<DZ, DT>;
  const int clusters = fused_resident_clusters<DZ, DT>(C, smem, num_sms);
  if (clusters < 1) return cudaErrorNotSupported;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int grid_clusters = units < clusters ? units : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(grid_clusters * C), 1, 1);
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, p);
}

int fused_max_units(int vocab, int z_dtype, int t_dtype, int num_sms) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (zb && tb) return fused_max_units_t<BF16, BF16>(vocab, num_sms);
  if (!zb && tb) return fused_max_units_t<F32, BF16>(vocab, num_sms);
  if (zb && !tb) return fused_max_units_t<BF16, F32>(vocab, num_sms);
  return fused_max_units_t<F32, F32>(vocab, num_sms);
}

cudaError_t launch_fused(const RowPassParams& p, int z_dtype, int t_dtype, int num_sms, cudaStream_t s) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (zb && tb) return launch_fused_t<BF16, BF16>(p, num_sms, s);
  if (!zb && tb) return launch_fused_t<F32, BF16>(p, num_sms, s);
  if (zb && !tb) return launch_fused_t<BF16, F32>(p, num_sms, s);
  return launch_fused_t<F32, F32>(p, num_sms, s);
}

}  // namespace adaflash
