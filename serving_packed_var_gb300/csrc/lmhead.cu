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
//   L1 is a persistent tcgen05 GEMM: per (128-row tile, 256-entry vocabulary tile)
//      it computes the z and t tiles into TMEM (TMA loads of swizzled K-major
//      operands into a shared-memory ring, one thread issuing the MMAs), and its
//      epilogue warps reduce each row of the tile to a partial record:
//      max, sum of exponentials, sum of e^z (z - t), max (z - t), the two largest z
//      (with the index of the largest), the first index of the largest t and z there;
//   L2 combines a row's records in a fixed order into its log-sum-exps, the
//      unclipped reverse KL, the target argmax and the draft logit there (for the
//      CE), re-evaluates exactly (by dot products) only the entries whose term can
//      exceed the clip, and writes the outputs of the logits path (kl, ce, row
//      statistics, target argmax).
// A diagnostic entry point runs L1 with an epilogue that writes the logits instead.
#include <atomic>
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
// Hidden elements per k-block: 64, one 128-byte swizzle row of bf16.
constexpr int kBK = 64;
constexpr int kRowBytes = kBK * 2;  // one swizzle row
// Stage layout: A_z, A_t, then B_z and B_t, or a single B when the two heads are the
// same matrix (one weight tile feeds both products, and the ring has room for more stages).
template <bool kShared>
struct Ring {
  static constexpr uint32_t kB = kBN * kBK * 2;
  static constexpr uint32_t kA = kBM * kBK * 2;
  static constexpr uint32_t kStage = 2 * kA + (kShared ? 1 : 2) * kB;
  static constexpr int kStages = kShared ? 3 : 2;
  static constexpr uint32_t kOffBz = 2 * kA;
  static constexpr uint32_t kOffBt = kShared ? 2 * kA : 2 * kA + kB;
};
constexpr uint32_t kTileA = kBM * kBK * 2;
constexpr uint32_t kTileB = kBN * kBK * 2;
constexpr uint32_t kTmemCols = 512;  // z tile in columns 0..255, t tile in 256..511
constexpr int kCombThreads = 256;
constexpr int kMaxVTiles = (ADAFLASH_MAX_VOCAB + 255) / 256;  // vocabulary tiles of a row, at most
constexpr int kWin = 512;                                      // candidate entries per evaluation window

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

}  // namespace

// ---- L1: the head GEMM and the per-tile row reduction ----
//
// Persistent: CTA c takes tiles c, c + G, ... (row tiles fastest, so the CTAs at
// work at any time share weight tiles through L2).  The TMA warp runs ahead across
// tiles; the MMA warp starts a tile once the epilogue has read the accumulators of
// the previous one.  Sixteen epilogue warps split a tile: warp w reads TMEM lanes
// 32 (w mod 4) .. +31 (the hardware's lane quarters) and a quarter of the 256
// columns; the four quarter records of a row are merged in column order.

namespace {

constexpr int kEpiWarps = 16;
constexpr int kGemmThreads = 64 + kEpiWarps * 32;

struct EpiRec {
  float mz, sz, szd, dmax, z2, mt, st, zat;
  int az, at;
};

// Record b (columns after a's) merged into a: ties keep a's (lower) indices.
__device__ __forceinline__ void epi_merge(EpiRec& a, const EpiRec& b) {
  if (b.mz > a.mz) {
    const float f = (a.mz == kNegInf) ? 0.f : ex2((a.mz - b.mz) * kLog2e);
    a.sz = a.sz * f + b.sz;
    a.szd = a.szd * f + b.szd;
    a.z2 = fmaxf(a.mz, b.z2);
    a.mz = b.mz;
    a.az = b.az;
  } else if (b.mz != kNegInf) {
    const float f = ex2((b.mz - a.mz) * kLog2e);
    a.sz = a.sz + b.sz * f;
    a.szd = a.szd + b.szd * f;
    a.z2 = fmaxf(a.z2, b.mz);
  }
  a.dmax = fmaxf(a.dmax, b.dmax);
  if (b.mt > a.mt) {
    const float f = (a.mt == kNegInf) ? 0.f : ex2((a.mt - b.mt) * kLog2e);
    a.st = a.st * f + b.st;
    a.mt = b.mt;
    a.at = b.at;
    a.zat = b.zat;
  } else if (b.mt != kNegInf) {
    a.st = a.st + b.st * ex2((b.mt - a.mt) * kLog2e);
  }
}

}  // namespace

template <bool kShared>
__global__ void __launch_bounds__(kGemmThreads, 1)
    lmhead_gemm_kernel(const __grid_constant__ CUtensorMap map_hd, const __grid_constant__ CUtensorMap map_ht,
                       const __grid_constant__ CUtensorMap map_wd, const __grid_constant__ CUtensorMap map_wt,
                       const LmHeadParams P) {
  extern __shared__ uint8_t smem_raw[];
  using RG = Ring<kShared>;
  constexpr int kLStages = RG::kStages;
  constexpr uint32_t kStageBytes = RG::kStage;
  __shared__ uint64_t full_bar[kLStages];
  __shared__ uint64_t empty_bar[kLStages];
  __shared__ uint64_t accum_full, accum_empty;
  __shared__ uint32_t tmem_base;
  __shared__ int s_err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = P.n_pair_tiles + (P.n_t_rows - P.n_pair_rows + kBM - 1) / kBM;
  const int n_tiles = m_tiles * P.n_vtiles;
  const int nkb = P.H / kBK;
  uint8_t* ring = align1024(smem_raw);
  EpiRec* red = reinterpret_cast<EpiRec*>(ring + kLStages * kStageBytes);  // [4][kBM]

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&accum_full, 1);
    mbar_init(&accum_empty, kEpiWarps);
    fence_barrier_init();
    s_err = 0;
    tma_prefetch_desc(&map_ht);
    tma_prefetch_desc(&map_wt);
    tma_prefetch_desc(&map_hd);
    tma_prefetch_desc(&map_wd);
  }
  if (warp == 1) tmem_alloc(&tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* err = &s_err;  // after a failed wait, every role stops waiting

  if (warp == 0) {
    // ---- TMA producer: every k-block of every tile of this CTA ----
    if (lane == 0) {
      uint32_t g = 0;  // k-blocks issued so far
      for (int tile = blockIdx.x; tile < n_tiles && !*err; tile += gridDim.x) {
        const int mt = tile % m_tiles, vt = tile / m_tiles;
        const bool pair = mt < P.n_pair_tiles;
        const int row0 = pair ? mt * kBM : P.n_pair_rows + (mt - P.n_pair_tiles) * kBM;
        const uint32_t bytes = pair ? kStageBytes : (kTileA + kTileB);  // target-only tiles: A_t and B_t
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = static_cast<int>(g % kLStages);
          if (g >= static_cast<uint32_t>(kLStages) &&
              !mbar_wait_bounded(&empty_bar[s], ((g / kLStages) - 1) & 1)) {
            *err = 1;
            break;
          }
          uint8_t* st = ring + s * kStageBytes;
          mbar_arrive_expect_tx(&full_bar[s], bytes);
          const int x = kb * kBK;
          if (pair) {
            tma_load_2d(st, &map_hd, x, row0, &full_bar[s]);
            if (!kShared) tma_load_2d(st + RG::kOffBz, &map_wd, x, vt * kBN, &full_bar[s]);
          }
          tma_load_2d(st + kTileA, &map_ht, x, row0, &full_bar[s]);
          tma_load_2d(st + RG::kOffBt, &map_wt, x, vt * kBN, &full_bar[s]);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      uint32_t g = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < n_tiles && !*err; tile += gridDim.x, ++it) {
        const bool pair = (tile % m_tiles) < P.n_pair_tiles;
        // the epilogue has read the previous tile's accumulators
        if (it > 0 && !mbar_wait_bounded(&accum_empty, (it - 1) & 1)) {
          *err = 1;
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = static_cast<int>(g % kLStages);
          if (!mbar_wait_bounded(&full_bar[s], (g / kLStages) & 1)) {
            *err = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_addr(ring + s * kStageBytes);
          const uint64_t daz = sdesc_swizzled<kRowBytes>(st), dat = sdesc_swizzled<kRowBytes>(st + kTileA);
          const uint64_t dbz = sdesc_swizzled<kRowBytes>(st + RG::kOffBz);
          const uint64_t dbt = sdesc_swizzled<kRowBytes>(st + RG::kOffBt);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            const uint64_t step = static_cast<uint64_t>(kk * 2);  // 32 bytes per 16-element step, in 16-byte units
            if (pair) umma_bf16(tmem, daz + step, dbz + step, idesc, acc);
            umma_bf16(tmem + kBN, dat + step, dbt + step, idesc, acc);
          }
          umma_commit(&empty_bar[s]);
        }
        umma_commit(&accum_full);  // arrives once every MMA issued so far has completed
        if (!ok) break;
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue ----
    const int q = warp & 3;              // TMEM lane quarter
    const int j = (warp - 2) >> 2;       // column quarter: 64 j .. 64 j + 63
    const int r = q * 32 + lane;         // row of the tile
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      const int mt = tile % m_tiles, vt = tile / m_tiles;
      const bool pair = mt < P.n_pair_tiles;
      const int row0 = pair ? mt * kBM : P.n_pair_rows + (mt - P.n_pair_tiles) * kBM;
      const int row = row0 + r;
      const bool valid_row = row < (pair ? P.n_pair_rows : P.n_t_rows);
      // every epilogue warp runs every tile and every barrier below, whatever the
      // waits return, so the named barriers always see all sixteen warps
      const bool ok = !*err && mbar_wait_bounded(&accum_full, it & 1);
      tc_fence_after();
      if (!ok) *err = 1;
      EpiRec e{kNegInf, 0.f, 0.f, kNegInf, kNegInf, kNegInf, 0.f, 0.f, -1, -1};
      for (int c = 0; c < 4; ++c) {
        const int col = j * 64 + c * 16;
        uint32_t rt[16], rz[16];
        tmem_ld16(tl + kBN + col, rt);
        tmem_wait16(rt);
        if (pair) {
          tmem_ld16(tl + col, rz);
          tmem_wait16(rz);
        }
        const int vb = vt * kBN + col;
        const int nval = min(16, P.V - vb);  // entries of this chunk inside the vocabulary
        if (P.mode == 1) {
          if (ok && valid_row) {
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              if (x < nval) {
                P.out_t[static_cast<int64_t>(row) * P.ld_out + vb + x] = __uint_as_float(rt[x]);
                if (pair) P.out_z[static_cast<int64_t>(row) * P.ld_out + vb + x] = __uint_as_float(rz[x]);
              }
            }
          }
          continue;
        }
        if (nval <= 0) continue;
        // t: maximum with its first index (and z there), then the rescaled sum
        float cmt = kNegInf, czat = 0.f;
        int cat = -1;
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float t = __uint_as_float(rt[x]);
          if (x < nval && t > cmt) {
            cmt = t;
            cat = vb + x;
            if (pair) czat = __uint_as_float(rz[x]);
          }
        }
        if (cmt > e.mt) {
          e.st *= ex2((e.mt - cmt) * kLog2e);
          e.mt = cmt;
          e.at = cat;
          e.zat = czat;
        }
        float add_t = 0.f;
#pragma unroll
        for (int x = 0; x < 16; ++x)
          if (x < nval) add_t += ex2((__uint_as_float(rt[x]) - e.mt) * kLog2e);
        e.st += add_t;
        if (pair) {
          // z: the two largest values (first index of the largest), max (z - t)
          float c1 = kNegInf, c2 = kNegInf;
          int ci = -1;
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float z = __uint_as_float(rz[x]);
            if (x < nval) {
              if (z > c1) {
                c2 = c1;
                c1 = z;
                ci = vb + x;
              } else if (z > c2) {
                c2 = z;
              }
              e.dmax = fmaxf(e.dmax, z - __uint_as_float(rt[x]));
            }
          }
          if (c1 > e.mz) {
            const float f = ex2((e.mz - c1) * kLog2e);
            e.sz *= f;
            e.szd *= f;
            e.z2 = fmaxf(e.mz, c2);
            e.mz = c1;
            e.az = ci;
          } else {
            e.z2 = fmaxf(e.z2, c1);
          }
          float add_z = 0.f, add_zd = 0.f;
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            if (x < nval) {
              const float z = __uint_as_float(rz[x]);
              const float ez = ex2((z - e.mz) * kLog2e);
              add_z += ez;
              add_zd = fmaf(ez, z - __uint_as_float(rt[x]), add_zd);
            }
          }
          e.sz += add_z;
          e.szd += add_zd;
        }
      }
      // the accumulators are read: the next tile's MMAs may start
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accum_empty);
      if (P.mode == 1) continue;
      red[j * kBM + r] = e;
      named_bar_sync_id(1, kEpiWarps * 32);
      if (j == 0 && ok && valid_row) {
        EpiRec m = red[r];
        for (int jj = 1; jj < 4; ++jj) epi_merge(m, red[jj * kBM + r]);
        LmPartial rec;
        rec.mz = m.mz;
        rec.sz = m.sz;
        rec.szd = m.szd;
        rec.dmax = m.dmax;
        rec.z2 = m.z2;
        rec.mt = m.mt;
        rec.st = m.st;
        rec.az = m.az;
        rec.at = m.at;
        rec.zat = m.zat;
        rec.pad1 = rec.pad2 = 0;
        P.partials[static_cast<int64_t>(row) * P.n_vtiles + vt] = rec;
      }
      named_bar_sync_id(1, kEpiWarps * 32);  // red is rewritten by the next tile
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
  __shared__ int s_off[kMaxVTiles];  // candidate entries per tile, then their first list position
  __shared__ int s_wsum[kCombThreads / 32];
  __shared__ int s_total;
  __shared__ int s_list[kWin];  // vocabulary entries of the current window
  __shared__ float s_corr[kWin], s_sclip[kWin];
  __shared__ int s_flag[kWin];
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
  // the tile is examined.  The candidate count of every tile is found in parallel, a
  // block scan in tile order places the entries, and windows of kWin entries are
  // evaluated (one warp per entry) and summed in vocabulary order.
  const float theta = s_theta;
  const float lse_z = s_lse_z, dlse = s_dlse, c = P.clip_c;
  const float nlz = -lse_z * kLog2e;
  const int nt = P.n_vtiles;  // <= kMaxVTiles
  for (int v = tid; v < nt; v += kCombThreads) {
    const LmPartial p = rec[v];
    s_off[v] = !(p.mz > theta) ? 0 : (!(p.z2 > theta) ? 1 : min(256, P.V - v * 256));
  }
  __syncthreads();
  // exclusive scan of s_off over tiles: thread t owns tiles [t * per, (t + 1) * per)
  {
    const int per = (nt + kCombThreads - 1) / kCombThreads;
    const int t0 = min(nt, tid * per), t1 = min(nt, t0 + per);
    int mine = 0;
    for (int v = t0; v < t1; ++v) mine += s_off[v];
    int inc = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    if (lane == 31) s_wsum[warp] = inc;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kCombThreads / 32; ++w) {
      if (w < warp) before += s_wsum[w];
      total += s_wsum[w];
    }
    int run = before + inc - mine;
    for (int v = t0; v < t1; ++v) {
      const int cnt = s_off[v];
      s_off[v] = run;  // first list position of tile v
      run += cnt;
    }
    if (tid == 0) s_total = total;
  }
  __syncthreads();
  const int total = s_total;
  float corr_all = 0.f, sclip_all = 0.f;
  int nclip_all = 0;
  for (int lo = 0; lo < total; lo += kWin) {
    const int hi = min(total, lo + kWin);
    // place the entries of this window
    for (int v = tid; v < nt; v += kCombThreads) {
      const int o0 = s_off[v], o1 = (v + 1 < nt) ? s_off[v + 1] : total;
      if (o1 <= lo || o0 >= hi) continue;
      if (o1 - o0 == 1) {
        s_list[o0 - lo] = rec[v].az;
      } else {
        for (int x = max(o0, lo); x < min(o1, hi); ++x) s_list[x - lo] = v * 256 + (x - o0);
      }
    }
    __syncthreads();
    for (int e = warp; e < hi - lo; e += kCombThreads / 32) {
      const int v = s_list[e];
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
        s_flag[e] = nc;
      }
    }
    __syncthreads();
    if (tid == 0) {
      for (int e = 0; e < hi - lo; ++e) {
        corr_all += s_corr[e];
        sclip_all += s_sclip[e];
        nclip_all += s_flag[e];
      }
    }
    __syncthreads();
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

// bf16 matrix [rows, cols] with row stride ld elements, tiles of box_rows x kBK (swizzled at kBK * 2 bytes).
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The scratch of adaflash_lmhead_opd_fwd_static: one array per device, held while the
// library's LM-head code is loaded.  Host code cannot use the symbol as a device
// address; lm_static_scratch looks the address up once per device.
static __device__ __align__(256) uint8_t g_lm_static_scratch[ADAFLASH_LMHEAD_STATIC_SCRATCH_BYTES];

cudaError_t lm_static_scratch(void** ptr, int64_t* bytes) {
  static std::atomic<void*> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_lm_static_scratch);  // with this device current
    if (e != cudaSuccess) return e;
    cache[dev].store(p, std::memory_order_release);
  }
  *ptr = p;
  *bytes = ADAFLASH_LMHEAD_STATIC_SCRATCH_BYTES;
  return cudaSuccess;
}

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
  const bool shared = (wd == wt) && (ld_wd == ld_wt);
  const size_t smem = (shared ? static_cast<size_t>(Ring<true>::kStages) * Ring<true>::kStage
                              : static_cast<size_t>(Ring<false>::kStages) * Ring<false>::kStage) +
                      4 * kBM * sizeof(EpiRec) + 1024;
  auto kern = shared ? lmhead_gemm_kernel<true> : lmhead_gemm_kernel<false>;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  const long long tiles = static_cast<long long>(m_tiles) * p.n_vtiles;
  const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);  // one CTA per SM (shared memory)
  count_launch();
  kern<<<grid, kGemmThreads, smem, s>>>(mhd, mht, mwd, mwt, p);
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
