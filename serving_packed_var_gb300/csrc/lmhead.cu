// lmhead.cu -- the verify + OPD-loss forward straight from final hidden states.
//
// The logits of a row are the LM head applied to its final hidden state, z = W_d h_d
// (draft) and t = W_t h_t (target); the verification and the loss are those of the
// row pass (AdaFlash article, "AdaFlash: Adaptive Speculative Decoding with Online
// Self-Improvement for High-Concurrency LLM Inference": the opening section and
// "On-Policy Distillation (OPD) for Domain Adaptation").  Here the logits are never
// written to memory:
//
//   L0 gathers the target hidden rows into pair order (the target row paired with
//      each draft row, then the bonus rows) in the caller's workspace;
//   L1 is a tcgen05 GEMM: one CTA per (128-row tile, 256-entry vocabulary tile)
//      computes the z and t tiles into TMEM (TMA loads of 128-byte-swizzled K-major
//      operands into a 2-stage shared-memory ring, one thread issuing the MMAs),
//      and its four epilogue warps reduce each row of the tile to a partial record:
//      max, sum of exponentials, sum of e^z (z - t), max (z - t), the two largest z
//      (with the index of the largest), the first index of the largest t and z there;
//   L2 combines a row's records in a fixed order into its log-sum-exps, the
//      unclipped reverse KL, the target argmax and the draft logit there (for the
//      CE), re-evaluates exactly (by dot products) only the entries whose term can
//      exceed the clip, and writes the outputs of the logits path (kl, ce, row
//      statistics, target argmax).
// A diagnostic entry point runs L1 with an epilogue that writes the logits instead.
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstring>

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace adaflash {

namespace {

constexpr int kBM = 128;  // rows per tile (TMEM lanes)
constexpr int kBN = 256;  // vocabulary entries per tile
constexpr int kBK = 64;   // hidden elements per k-block: one 128-byte swizzle row of bf16
constexpr int kLStages = 2;
constexpr int kLThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr uint32_t kTileA = kBM * kBK * 2;
constexpr uint32_t kTileB = kBN * kBK * 2;
constexpr uint32_t kStageBytes = 2 * kTileA + 2 * kTileB;
constexpr uint32_t kTmemCols = 512;  // z tile in columns 0..255, t tile in 256..511
constexpr int kCombThreads = 256;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

}  // namespace

// ---- L1: the head GEMM and the per-tile row reduction ----
__global__ void __launch_bounds__(kLThreads, 1)
    lmhead_gemm_kernel(const __grid_constant__ CUtensorMap map_hd, const __grid_constant__ CUtensorMap map_ht,
                       const __grid_constant__ CUtensorMap map_wd, const __grid_constant__ CUtensorMap map_wt,
                       const LmHeadParams P) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kLStages];
  __shared__ uint64_t empty_bar[kLStages];
  __shared__ uint64_t accum_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int s_err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = static_cast<int>(blockIdx.x), vt = static_cast<int>(blockIdx.y);
  const bool pair = mt < P.n_pair_tiles;
  // first row of the tile in the target operand (pair rows are also draft rows)
  const int row0 = pair ? mt * kBM : P.n_pair_rows + (mt - P.n_pair_tiles) * kBM;
  const int row_end = pair ? P.n_pair_rows : P.n_t_rows;
  const int v0 = vt * kBN;
  const int nkb = P.H / kBK;
  uint8_t* ring = align1024(smem_raw);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&accum_bar, 1);
    fence_barrier_init();
    s_err = 0;
    tma_prefetch_desc(&map_ht);
    tma_prefetch_desc(&map_wt);
    if (pair) {
      tma_prefetch_desc(&map_hd);
      tma_prefetch_desc(&map_wd);
    }
  }
  if (warp == 1) tmem_alloc(&tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      const uint32_t bytes = pair ? kStageBytes : (kTileA + kTileB);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kLStages;
        if (kb >= kLStages && !mbar_wait_bounded(&empty_bar[s], ((kb / kLStages) - 1) & 1)) {
          s_err = 1;
          break;
        }
        uint8_t* st = ring + s * kStageBytes;
        mbar_arrive_expect_tx(&full_bar[s], bytes);
        const int x = kb * kBK;
        if (pair) {
          tma_load_2d(st, &map_hd, x, row0, &full_bar[s]);
          tma_load_2d(st + 2 * kTileA, &map_wd, x, v0, &full_bar[s]);
        }
        tma_load_2d(st + kTileA, &map_ht, x, row0, &full_bar[s]);
        tma_load_2d(st + 2 * kTileA + kTileB, &map_wt, x, v0, &full_bar[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kLStages;
        if (!mbar_wait_bounded(&full_bar[s], (kb / kLStages) & 1)) {
          s_err = 1;
          break;
        }
        tc_fence_after();
        const uint32_t st = smem_addr(ring + s * kStageBytes);
        const uint64_t daz = sdesc_sw128(st), dat = sdesc_sw128(st + kTileA);
        const uint64_t dbz = sdesc_sw128(st + 2 * kTileA), dbt = sdesc_sw128(st + 2 * kTileA + kTileB);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
          const uint64_t step = static_cast<uint64_t>(kk * 2);  // 32 bytes per 16-element step, in 16-byte units
          if (pair) umma_bf16(tmem, daz + step, dbz + step, idesc, acc);
          umma_bf16(tmem + kBN, dat + step, dbt + step, idesc, acc);
        }
        umma_commit(&empty_bar[s]);
      }
      umma_commit(&accum_bar);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32 (w mod 4) .. +31 ----
    const int q = warp & 3;
    const int r = q * 32 + lane;  // row of the tile
    const int row = row0 + r;
    const bool valid_row = row < row_end;
    const bool ok = mbar_wait_bounded(&accum_bar, 0);
    tc_fence_after();
    if (!ok) s_err = 1;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    if (P.mode == 1) {
      // diagnostic: write the logits tiles
      for (int c = 0; c < kBN / 16; ++c) {
        uint32_t rt[16];
        tmem_ld16(tl + kBN + c * 16, rt);
        tmem_wait16(rt);
        if (ok && valid_row) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int v = v0 + c * 16 + j;
            if (v < P.V) P.out_t[static_cast<int64_t>(row) * P.ld_out + v] = __uint_as_float(rt[j]);
          }
        }
        if (pair) {
          uint32_t rz[16];
          tmem_ld16(tl + c * 16, rz);
          tmem_wait16(rz);
          if (ok && valid_row) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int v = v0 + c * 16 + j;
              if (v < P.V) P.out_z[static_cast<int64_t>(row) * P.ld_out + v] = __uint_as_float(rz[j]);
            }
          }
        }
      }
    } else {
      // statistics of this row over the tile's valid entries (natural exponentials
      // as 2^(x log2 e), every sum relative to the running maximum)
      float mz = kNegInf, sz = 0.f, szd = 0.f, dmax = kNegInf, z2 = kNegInf;
      float mt = kNegInf, st = 0.f, zat = 0.f;
      int az = -1, at = -1;
      for (int c = 0; c < kBN / 16; ++c) {
        uint32_t rt[16], rz[16];
        tmem_ld16(tl + kBN + c * 16, rt);
        tmem_wait16(rt);
        if (pair) {
          tmem_ld16(tl + c * 16, rz);
          tmem_wait16(rz);
        }
        const int vb = v0 + c * 16;
        const int nval = min(16, P.V - vb);  // entries of this chunk inside the vocabulary
        if (nval <= 0) continue;
        // t: maximum with its first index (and z there), then the rescaled sum
        float cmt = kNegInf, czat = 0.f;
        int cat = -1;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float t = __uint_as_float(rt[j]);
          if (j < nval && t > cmt) {
            cmt = t;
            cat = vb + j;
            if (pair) czat = __uint_as_float(rz[j]);
          }
        }
        if (cmt > mt) {
          st *= ex2((mt - cmt) * kLog2e);
          mt = cmt;
          at = cat;
          zat = czat;
        }
        float add_t = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < nval) add_t += ex2((__uint_as_float(rt[j]) - mt) * kLog2e);
        st += add_t;
        if (pair) {
          // z: the two largest values (first index of the largest), max (z - t)
          float c1 = kNegInf, c2 = kNegInf;
          int ci = -1;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float z = __uint_as_float(rz[j]);
            if (j < nval) {
              if (z > c1) {
                c2 = c1;
                c1 = z;
                ci = vb + j;
              } else if (z > c2) {
                c2 = z;
              }
              dmax = fmaxf(dmax, z - __uint_as_float(rt[j]));
            }
          }
          if (c1 > mz) {
            const float f = ex2((mz - c1) * kLog2e);
            sz *= f;
            szd *= f;
            z2 = fmaxf(mz, c2);
            mz = c1;
            az = ci;
          } else {
            z2 = fmaxf(z2, c1);
          }
          float add_z = 0.f, add_zd = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j < nval) {
              const float z = __uint_as_float(rz[j]);
              const float e = ex2((z - mz) * kLog2e);
              add_z += e;
              add_zd = fmaf(e, z - __uint_as_float(rt[j]), add_zd);
            }
          }
          sz += add_z;
          szd += add_zd;
        }
      }
      if (ok && valid_row) {
        LmPartial rec;
        rec.mz = mz;
        rec.sz = sz;
        rec.szd = szd;
        rec.dmax = dmax;
        rec.z2 = z2;
        rec.mt = mt;
        rec.st = st;
        rec.az = az;
        rec.at = at;
        rec.zat = zat;
        rec.pad1 = rec.pad2 = 0;
        P.partials[static_cast<int64_t>(row) * P.n_vtiles + vt] = rec;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && s_err) flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
}

}  // namespace adaflash

namespace adaflash {

// ---- L0: target hidden rows into pair order ----
// Target row s of request i (the largest i with doff[i] + i <= s) goes to row s - i
// when it is paired with a draft row, to row N_d + i when it is the bonus row.
__global__ void __launch_bounds__(128) lm_gather_kernel(const uint16_t* ht, int64_t ld_ht, const int32_t* doff, int R,
                                                         int N_d, int H, uint16_t* out, uint32_t* status) {
  const int s = static_cast<int>(blockIdx.x);
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(doff + mid) + mid <= s) lo = mid; else hi = mid - 1;
  }
  const int i = lo;
  const int a = __ldg(doff + i) + i, b = __ldg(doff + i + 1) + i;
  int dst;
  if (a <= s && s < b) dst = s - i;
  else if (s == b) dst = N_d + i;
  else dst = -1;
  if (dst < 0 || dst >= N_d + R || (s < b && dst >= N_d)) {
    if (threadIdx.x == 0) flag_status(status, ADAFLASH_ERR_BAD_OFFSETS);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(ht + static_cast<int64_t>(s) * ld_ht);
  uint4* d = reinterpret_cast<uint4*>(out + static_cast<int64_t>(dst) * H);
  for (int w = threadIdx.x; w < H / 8; w += blockDim.x) d[w] = __ldg(src + w);
}

namespace {

// Warp dot product of two bf16 rows of length H (H a multiple of 8, rows 16-byte aligned),
// fixed order: lane l takes 16-byte words l, l + 32, ..., then a butterfly.
__device__ __forceinline__ float warp_dot_bf16(const uint16_t* a, const uint16_t* b, int H) {
  const uint4* pa = reinterpret_cast<const uint4*>(a);
  const uint4* pb = reinterpret_cast<const uint4*>(b);
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int w = lane; w < H / 8; w += 32) {
    const uint4 x = __ldg(pa + w), y = __ldg(pb + w);
    acc = fmaf(bf16_lo(x.x), bf16_lo(y.x), acc);
    acc = fmaf(bf16_hi(x.x), bf16_hi(y.x), acc);
    acc = fmaf(bf16_lo(x.y), bf16_lo(y.y), acc);
    acc = fmaf(bf16_hi(x.y), bf16_hi(y.y), acc);
    acc = fmaf(bf16_lo(x.z), bf16_lo(y.z), acc);
    acc = fmaf(bf16_hi(x.z), bf16_hi(y.z), acc);
    acc = fmaf(bf16_lo(x.w), bf16_lo(y.w), acc);
    acc = fmaf(bf16_hi(x.w), bf16_hi(y.w), acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

struct RowAcc {
  float mz, sz, szd, dmax;
  float mt, st;
  int at;
  float zat;  // z at the first index of the largest t
};

__device__ __forceinline__ void racc_merge(RowAcc& a, const RowAcc& b) {
  const float m = fmaxf(a.mz, b.mz);
  if (m != kNegInf) {
    const float fa = (a.mz == kNegInf) ? 0.f : ex2((a.mz - m) * kLog2e);
    const float fb = (b.mz == kNegInf) ? 0.f : ex2((b.mz - m) * kLog2e);
    a.sz = a.sz * fa + b.sz * fb;
    a.szd = a.szd * fa + b.szd * fb;
    a.mz = m;
  }
  a.dmax = fmaxf(a.dmax, b.dmax);
  const float mt = fmaxf(a.mt, b.mt);
  if (mt != kNegInf) {
    const float fa = (a.mt == kNegInf) ? 0.f : ex2((a.mt - mt) * kLog2e);
    const float fb = (b.mt == kNegInf) ? 0.f : ex2((b.mt - mt) * kLog2e);
    a.st = a.st * fa + b.st * fb;
  }
  if (b.mt > a.mt || (b.mt == a.mt && b.at >= 0 && (a.at < 0 || b.at < a.at))) {
    a.at = b.at;
    a.zat = b.zat;
  }
  a.mt = mt;
}

}  // namespace

// ---- L2: per-row combine, exact re-evaluation of clip candidates, outputs ----
__global__ void __launch_bounds__(kCombThreads) lm_combine_kernel(const LmCombineParams P) {
  __shared__ RowAcc red[kCombThreads];
  __shared__ int s_cand[kCombThreads];  // entries of the current batch
  __shared__ float s_corr[kCombThreads], s_sclip[kCombThreads];
  __shared__ int s_nclip[kCombThreads];
  __shared__ float s_lse_z, s_lse_t, s_dlse, s_klu, s_theta, s_za;
  __shared__ int s_a, s_ok, s_d, s_s;
  const int r = static_cast<int>(blockIdx.x);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool pair = r < P.N_d;
  if (tid == 0) {
    int ok = 1, d = -1, s = -1;
    if (pair) {
      d = r;
      const int i = request_of_row(P.doff, P.R, d);
      const int lo = __ldg(P.doff + i), hi = __ldg(P.doff + i + 1);
      if (!(lo <= d && d < hi)) ok = 0;
      s = d + i;
    } else {
      const int i = r - P.N_d;
      s = __ldg(P.doff + i + 1) + i;
      if (s < 0 || s >= P.N_d + P.R) ok = 0;
    }
    s_ok = ok;
    s_d = d;
    s_s = s;
  }
  __syncthreads();
  if (!s_ok) {
    if (tid == 0) flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
    return;
  }
  // ---- fixed-order combine of the row's tile records ----
  const LmPartial* rec = P.partials + static_cast<int64_t>(r) * P.n_vtiles;
  RowAcc a{kNegInf, 0.f, 0.f, kNegInf, kNegInf, 0.f, -1, 0.f};
  for (int v = tid; v < P.n_vtiles; v += kCombThreads) {
    const LmPartial p = rec[v];
    RowAcc b{pair ? p.mz : kNegInf, pair ? p.sz : 0.f, pair ? p.szd : 0.f, pair ? p.dmax : kNegInf, p.mt, p.st, p.at,
             p.zat};
    racc_merge(a, b);
  }
  red[tid] = a;
  __syncthreads();
  for (int half = kCombThreads / 2; half > 0; half >>= 1) {
    if (tid < half) {
      RowAcc x = red[tid];
      racc_merge(x, red[tid + half]);
      red[tid] = x;
    }
    __syncthreads();
  }
  if (tid == 0) {
    const RowAcc& t = red[0];
    s_a = t.at;
    s_za = t.zat;  // the GEMM's own z at the target argmax: CE = lse_z - z_a from the same values
    s_lse_t = t.mt + logf(t.st);
    if (pair) {
      s_lse_z = t.mz + logf(t.sz);
      s_dlse = s_lse_z - s_lse_t;
      s_klu = t.szd / t.sz - s_dlse;
      const float R = t.dmax - s_dlse;
      const float Rp = R + 1e-4f * (1.f + fabsf(t.dmax) + fabsf(s_dlse));
      const float c = P.clip_c;
      if (!(c < INFINITY) || !(Rp > 0.f)) {
        s_theta = INFINITY;
      } else {
        const float th = s_lse_z + logf(c / Rp);
        s_theta = th - (1e-3f + 1e-5f * fabsf(th));
      }
    }
  }
  __syncthreads();
  const int a_idx = s_a;
  if (!pair) {
    if (tid == 0) {
      if (a_idx >= 0 && a_idx < P.V) P.target_argmax[s_s] = a_idx;
      else flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
    }
    return;
  }
  const int d = s_d;
  const uint16_t* hrow = P.hd + static_cast<int64_t>(d) * P.ld_hd;
  const uint16_t* trow = P.ht + static_cast<int64_t>(r) * P.H;
  // ---- exact terms of the entries that can exceed the clip ----
  // A tile is a candidate when its largest z clears theta; only its largest entry
  // can then clip unless its second largest z clears theta too, when every entry of
  // the tile is examined.  Entries are taken in vocabulary order, in batches.
  const float theta = s_theta;
  const float lse_z = s_lse_z, dlse = s_dlse, c = P.clip_c;
  const float nlz = -lse_z * kLog2e;
  float corr_all = 0.f, sclip_all = 0.f;
  int nclip_all = 0;
  int vt = 0, sub = 0;  // scan position (thread 0)
  while (true) {
    __syncthreads();
    if (tid == 0) {
      int n = 0;
      while (vt < P.n_vtiles && n < kCombThreads) {
        const LmPartial p = rec[vt];
        if (!(p.mz > theta)) {
          ++vt;
          continue;
        }
        if (!(p.z2 > theta)) {
          s_cand[n++] = p.az;
          ++vt;
          continue;
        }
        const int v0 = vt * 256;
        const int vend = min(P.V, v0 + 256);
        while (v0 + sub < vend && n < kCombThreads) s_cand[n++] = v0 + sub++;
        if (v0 + sub >= vend) {
          sub = 0;
          ++vt;
        }
      }
      s_nclip[0] = n;  // batch size
    }
    __syncthreads();
    const int n = s_nclip[0];
    if (n == 0) break;
    __syncthreads();
    for (int e = warp; e < n; e += kCombThreads / 32) {
      const int v = s_cand[e];
      float corr = 0.f, sc = 0.f;
      int nc = 0;
      if (v >= 0 && v < P.V) {
        const float z = warp_dot_bf16(hrow, P.wd + static_cast<int64_t>(v) * P.ld_wd, P.H);
        if (z > theta) {
          const float t = warp_dot_bf16(trow, P.wt + static_cast<int64_t>(v) * P.ld_wt, P.H);
          const float p = ex2(__fmaf_rn(z, kLog2e, nlz));
          const float rr = __fsub_rn(__fsub_rn(z, t), dlse);
          const float term = __fmul_rn(p, rr);
          if (term > c) {
            corr = term - c;
            sc = p * (rr + 1.f);
            nc = 1;
          }
        }
      }
      if (lane == 0) {
        s_corr[e] = corr;
        s_sclip[e] = sc;
        s_cand[e] = nc;  // reused: this entry's clip flag
      }
    }
    __syncthreads();
    if (tid == 0) {
      for (int e = 0; e < n; ++e) {
        corr_all += s_corr[e];
        sclip_all += s_sclip[e];
        nclip_all += s_cand[e];
      }
    }
  }
  if (tid == 0) {
    P.kl_row[d] = s_klu - corr_all;
    P.row_stats[4 * static_cast<int64_t>(d) + 0] = lse_z;
    P.row_stats[4 * static_cast<int64_t>(d) + 1] = s_lse_t;
    P.row_stats[4 * static_cast<int64_t>(d) + 2] = (s_klu + 1.f) - sclip_all;
    P.row_stats[4 * static_cast<int64_t>(d) + 3] = static_cast<float>(nclip_all);
    if (a_idx >= 0 && a_idx < P.V) {
      P.ce_row[d] = lse_z - s_za;
      P.target_argmax[s_s] = a_idx;
    } else {
      flag_status(P.status, ADAFLASH_ERR_TIMEOUT);
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      (void)cudaGetLastError();
  }
  return fn;
}

// bf16 matrix [rows, cols] with row stride ld elements, tiles of box_rows x 64 (128-byte swizzle).
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_lm_gather(const uint16_t* ht, int64_t ld_ht, const int32_t* doff, int R, int N_d, int H,
                             uint16_t* out, uint32_t* status, cudaStream_t s) {
  const int Nt = N_d + R;
  if (Nt <= 0) return cudaSuccess;
  count_launch();
  lm_gather_kernel<<<static_cast<unsigned>(Nt), 128, 0, s>>>(ht, ld_ht, doff, R, N_d, H, out, status);
  return cudaGetLastError();
}

cudaError_t launch_lm_gemm(const uint16_t* hd, int64_t ld_hd, const uint16_t* ht_pairs, int64_t ld_ht,
                           const uint16_t* wd, int64_t ld_wd, const uint16_t* wt, int64_t ld_wt,
                           const LmHeadParams& p, cudaStream_t s) {
  const int n_bonus_rows = p.n_t_rows - p.n_pair_rows;
  const int m_tiles = p.n_pair_tiles + (n_bonus_rows + kBM - 1) / kBM;
  if (m_tiles <= 0 || p.n_vtiles <= 0) return cudaSuccess;
  CUtensorMap mhd, mht, mwd, mwt;
  const bool have_pairs = p.n_pair_rows > 0;
  if (!make_map(&mht, ht_pairs, p.n_t_rows, p.H, ld_ht, kBM) || !make_map(&mwt, wt, p.V, p.H, ld_wt, kBN))
    return cudaErrorInvalidValue;
  if (have_pairs) {
    if (!make_map(&mhd, hd, p.n_pair_rows, p.H, ld_hd, kBM) || !make_map(&mwd, wd, p.V, p.H, ld_wd, kBN))
      return cudaErrorInvalidValue;
  } else {
    mhd = mht;
    mwd = mwt;
  }
  const size_t smem = static_cast<size_t>(kLStages) * kStageBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(lmhead_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  count_launch();
  lmhead_gemm_kernel<<<dim3(static_cast<unsigned>(m_tiles), static_cast<unsigned>(p.n_vtiles)), kLThreads, smem, s>>>(
      mhd, mht, mwd, mwt, p);
  return cudaGetLastError();
}

cudaError_t launch_lm_combine(const LmCombineParams& p, cudaStream_t s) {
  const int rows = p.N_d + p.R;
  if (rows <= 0) return cudaSuccess;
  count_launch();
  lm_combine_kernel<<<static_cast<unsigned>(rows), kCombThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace adaflash
