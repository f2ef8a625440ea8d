// rowstats.cuh -- per-row statistics shared by the row pass (K1) and the fused
// forward + backward pass (K4): the running sums of one thread, their warp and
// cluster combines, and the row constants derived from them.
//
// Sums are taken relative to integer base-2 exponent offsets, so every rescale and
// every combine multiplies by an exact power of two; everything is float32 (one
// float64 warp-instruction holds GB300's narrow float64 pipe for a whole warp).
// The difference of log-sum-exps is (n_t - n_z) ln 2 + ln(S_z / S_t), never a
// difference of two large logs.  Operations: AdaFlash article ("AdaFlash: Adaptive
// Speculative Decoding with Online Self-Improvement for High-Concurrency LLM
// Inference"), "On-Policy Distillation (OPD) for Domain Adaptation".
#pragma once

#include <cfloat>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace adaflash {

namespace {

constexpr int kMaxCluster = 8;
constexpr int kNoOffset = 1 << 30;  // offset of an empty partial sum
constexpr float kLn2 = 0.69314718055994530942f;

struct __align__(16) SlicePartial {
  float sz, szd, st;  // sums scaled by 2^{nz}, 2^{nz}, 2^{nt}
  int nz, nt;         // integer base-2 exponent offsets
  float mt, dmax;     // max of t, bound on max of z - t
  float cmax;         // largest group maximum of z in the slice
  int bgrp;           // first group holding the max of t
  int err;
};

struct __align__(16) SliceCorr {
  float corr, sclip;
  int nclip;
  int err;
};

struct RowConsts {
  float lse_z, lse_t, dlse, kl_unclip;
  float theta;
  int argmax;
  float za;  // the draft logit at argmax (pair rows of the forward)
  int bgrp;  // first (row-global) group holding the max of t
  float mt;  // the max of t
  int err;
  int stop;  // every consumer thread leaves the unit loop together when set
  int scan;      // some thread of this CTA saw a group maximum of z above the threshold
  int any_scan;  // some CTA of the cluster did (the corrections are exchanged)
};

// Per-thread running state.  Sums are kept relative to integer base-2 exponent
// offsets nz, nt and split over two accumulators (even / odd entries):
//   sz = sum_v 2^{z_v log2e + nz},  szd = sum_v 2^{z_v log2e + nz} (z_v - t_v),
//   st = sum_v 2^{t_v log2e + nt}.
// Offsets move lazily: only when a group maximum lands more than kHeadroom powers
// of two above the offset (a thread's first group, practically never after), so
// the rescale branch is uniform and rare.  The argmax of t is tracked without
// branches as (max value, first group holding it); the index inside that group
// is resolved once per row.  dmax bounds max_v (z_v - t_v) from above by
// max over groups of (max z - min t): it only sets the clip screen's threshold,
// where a larger bound can only add candidates.
constexpr float kHeadroom = 32.f;

struct Acc {
  float sz0, sz1, szd0, szd1, st0, st1;
  float nzf, ntf;    // offsets as floats (integer-valued)
  float zlim, tlim;  // a group maximum above these moves the offset
  float mt;          // max of t
  float dmax;        // bound on max (z - t)
  float cmax;        // largest group maximum of z among this thread's groups
  int nz, nt;
  int bgrp;          // first (row-global) group index holding mt
};

// Scalar form used once a thread's accumulators are folded (warp/CTA combine).
struct AccS {
  float sz, szd, st;
  float mt, dmax, cmax;
  int nz, nt;
  int bgrp;
};

__device__ __forceinline__ void acc_init(Acc& a) {
  a.sz0 = a.sz1 = a.szd0 = a.szd1 = a.st0 = a.st1 = 0.f;
  a.nzf = a.ntf = 0.f;
  a.zlim = a.tlim = kNegInf;
  a.mt = kNegInf;
  a.dmax = kNegInf;
  a.cmax = kNegInf;
  a.nz = a.nt = kNoOffset;
  a.bgrp = INT_MAX;
}

__device__ __forceinline__ AccS acc_fold(const Acc& a) {
  AccS s;
  s.sz = a.sz0 + a.sz1;
  s.szd = a.szd0 + a.szd1;
  s.st = a.st0 + a.st1;
  s.mt = a.mt; s.dmax = a.dmax; s.cmax = a.cmax; s.nz = a.nz; s.nt = a.nt; s.bgrp = a.bgrp;
  return s;
}

// Integer offset that maps a new maximum m to 2^{<= 0}: -ceil(m log2 e) (clamped; logits are finite).
__device__ __forceinline__ int offset_for(float m) {
  const float x = fminf(fmaxf(m * kLog2e, -1048576.f), 1048576.f);
  return -static_cast<int>(ceilf(x));
}

__device__ __forceinline__ void rescale_z(Acc& a, float vmz) {
  const int nn = offset_for(vmz);
  const float f = pow2i(nn - a.nz);
  a.sz0 *= f; a.sz1 *= f; a.szd0 *= f; a.szd1 *= f;
  a.nz = nn;
  a.nzf = static_cast<float>(nn);
  a.zlim = (kHeadroom - a.nzf) * 0.69314718f;  // z log2e + nz > kHeadroom  <=>  z > (kHeadroom - nz) ln 2
}

__device__ __forceinline__ void rescale_t(Acc& a, float vmt) {
  const int nn = offset_for(vmt);
  const float f = pow2i(nn - a.nt);
  a.st0 *= f; a.st1 *= f;
  a.nt = nn;
  a.ntf = static_cast<float>(nn);
  a.tlim = (kHeadroom - a.ntf) * 0.69314718f;
}

// Screening code: a group maximum of z rounded up to bfloat16 (exact for bf16
// logits), so a code at or below a threshold proves every entry below it.
__device__ __forceinline__ uint16_t code_up(float v) {
  const uint32_t b = __float_as_uint(v);
  return static_cast<uint16_t>((v > 0.f ? b + 0xffffu : b) >> 16);
}
__device__ __forceinline__ float code_value(uint16_t c) { return __uint_as_float(static_cast<uint32_t>(c) << 16); }

// Value given to the unused entries of a ragged group: finite, and so small that
// 2^{x log2e + n} is 0 and z - t is 0.
constexpr float kVoid = -1.0e30f;

// Sums of one paired group of 8 entries at the current offsets (no rescale check,
// no maxima of z): the caller has moved the offsets for this group's maxima.
__device__ __forceinline__ void acc_pair_sums(Acc& a, const float z[8], const float t[8], float vmt, int grp) {
  const bool nb = vmt > a.mt;
  a.mt = fmaxf(a.mt, vmt);
  a.bgrp = nb ? grp : a.bgrp;
  {
    // Two entries per instruction on the FMA pipe (f32x2): even/odd entries are the
    // two lanes of each packed register, matching the two accumulators.
    const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
    const uint64_t nz2 = f2_pack(a.nzf, a.nzf), nt2 = f2_pack(a.ntf, a.ntf);
    uint64_t SZ = f2_pack(a.sz0, a.sz1), ST = f2_pack(a.st0, a.st1), SD = f2_pack(a.szd0, a.szd1);
    float dm = a.dmax;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t Z = f2_pack(z[2 * q], z[2 * q + 1]);
      const uint64_t T = f2_pack(t[2 * q], t[2 * q + 1]);
      float az0, az1, at0, at1;
      f2_unpack(f2_fma(Z, l2e2, nz2), az0, az1);
      f2_unpack(f2_fma(T, l2e2, nt2), at0, at1);
      const uint64_t EZ = f2_pack(ex2(az0), ex2(az1));
      SZ = f2_add(SZ, EZ);
      ST = f2_add(ST, f2_pack(ex2(at0), ex2(at1)));
      const uint64_t D = f2_sub(Z, T);
      SD = f2_fma(EZ, D, SD);
      float d0, d1;
      f2_unpack(D, d0, d1);
      dm = fmax3f(dm, d0, d1);
    }
    f2_unpack(SZ, a.sz0, a.sz1);
    f2_unpack(ST, a.st0, a.st1);
    f2_unpack(SD, a.szd0, a.szd1);
    a.dmax = dm;
  }
}

// Paired group of 8 entries, row-global group index grp (unused entries of z and t
// hold kVoid).  vmz = max z, vmt = max t over the valid entries.  The caller keeps
// a.cmax (the largest group maximum of z) up to date.
__device__ __forceinline__ void acc_pair_nc(Acc& a, const float z[8], const float t[8], float vmz, float vmt,
                                            int grp) {
  if (vmz > a.zlim) rescale_z(a, vmz);
  if (vmt > a.tlim) rescale_t(a, vmt);
  acc_pair_sums(a, z, t, vmt, grp);
}

// The same, updating a.cmax.
__device__ __forceinline__ void acc_pair(Acc& a, const float z[8], const float t[8], float vmz, float vmt,
                                         int grp) {
  acc_pair_nc(a, z, t, vmz, vmt, grp);
  a.cmax = fmaxf(a.cmax, vmz);
}

// Target-only group: argmax only.
__device__ __forceinline__ void acc_target(Acc& a, float vmt, int grp) {
  const bool nb = vmt > a.mt;
  a.mt = fmaxf(a.mt, vmt);
  a.bgrp = nb ? grp : a.bgrp;
}

// Lowest index of the value mt inside group grp of a target row (-1 if absent).
template <class DT>
__device__ int resolve_argmax(const uint8_t* trow, int grp, float mt, int V) {
  if (grp < 0 || grp >= (V + 7) / 8) return -1;
  const int v0 = grp * 8;
  const int n = min(8, V - v0);
  for (int j = 0; j < n; ++j)
    if (DT::load(trow, v0 + j) == mt) return v0 + j;
  return -1;
}

// Group of 8 from a shared-memory stage (16-byte aligned): values, max and min.
template <class DT>
__device__ __forceinline__ void load8_smem(const uint8_t* base, int g, float x[8], float& vmax);

__device__ __forceinline__ float max8(const float x[8]) {
  return fmax3f(fmax3f(x[0], x[1], x[2]), fmax3f(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
}

template <>
__device__ __forceinline__ void load8_smem<BF16>(const uint8_t* base, int g, float x[8], float& vmax) {
  const uint4 q = *reinterpret_cast<const uint4*>(base + 16 * g);
  x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x);
  x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
  x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z);
  x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
  vmax = max8(x);
}

template <>
__device__ __forceinline__ void load8_smem<F32>(const uint8_t* base, int g, float x[8], float& vmax) {
  const float4 a = *reinterpret_cast<const float4*>(base + 32 * g);
  const float4 b = *reinterpret_cast<const float4*>(base + 32 * g + 16);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  vmax = max8(x);
}

// 8 entries from global memory with vector loads (v0 a multiple of 8, row on the
// 16-byte grid).
template <class DT>
__device__ __forceinline__ void load8_global_vec(const uint8_t* row, int64_t v0, float x[8]);
template <>
__device__ __forceinline__ void load8_global_vec<BF16>(const uint8_t* row, int64_t v0, float x[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(row + v0 * 2));
  x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x);
  x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
  x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z);
  x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
}
template <>
__device__ __forceinline__ void load8_global_vec<F32>(const uint8_t* row, int64_t v0, float x[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(row + v0 * 4));
  const float4 b = __ldg(reinterpret_cast<const float4*>(row + v0 * 4 + 16));
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Up to 8 entries straight from global memory (any alignment); unused entries get kVoid.
template <class DT>
__device__ __forceinline__ void load_global(const void* row, int64_t v0, int n, float x[8], float& vmax) {
  vmax = kNegInf;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < n) {
      x[j] = DT::load(row, v0 + j);
      vmax = fmaxf(vmax, x[j]);
    } else {
      x[j] = kVoid;
    }
  }
}

// Whole-warp combine: every lane first moves its sums to the warp's smallest
// offset (an exact power-of-two scale), so only the three sums need shuffles; the
// maxima and the argmax group use single-instruction warp reductions.  The xor
// butterfly gives every lane the same sums.
__device__ __forceinline__ AccS warp_reduce(const AccS& a) {
  AccS r;
  r.nz = __reduce_min_sync(0xffffffffu, a.nz);
  r.nt = __reduce_min_sync(0xffffffffu, a.nt);
  const float fz = pow2i(r.nz - a.nz), ft = pow2i(r.nt - a.nt);
  float sz = a.sz * fz, szd = a.szd * fz, st = a.st * ft;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sz += __shfl_xor_sync(0xffffffffu, sz, off);
    szd += __shfl_xor_sync(0xffffffffu, szd, off);
    st += __shfl_xor_sync(0xffffffffu, st, off);
  }
  r.sz = sz; r.szd = szd; r.st = st;
  r.mt = warp_max_f32(a.mt);
  r.bgrp = static_cast<int>(__reduce_min_sync(0xffffffffu, static_cast<unsigned>(a.mt == r.mt ? a.bgrp : INT_MAX)));
  r.dmax = warp_max_f32(a.dmax);
  r.cmax = warp_max_f32(a.cmax);
  return r;
}

// Fixed-order combine of partials; the power-of-two factors are exact.
__device__ void combine_partials(const SlicePartial* parts, int n, SlicePartial& out) {
  int nz = kNoOffset, nt = kNoOffset, bgrp = INT_MAX, err = 0;
  float mt = kNegInf, dmax = kNegInf, cmax = kNegInf;
  for (int i = 0; i < n; ++i) {
    cmax = fmaxf(cmax, parts[i].cmax);
    nz = min(nz, parts[i].nz);
    nt = min(nt, parts[i].nt);
    dmax = fmaxf(dmax, parts[i].dmax);
    if (parts[i].mt > mt || (parts[i].mt == mt && parts[i].bgrp < bgrp)) bgrp = parts[i].bgrp;
    mt = fmaxf(mt, parts[i].mt);
    err |= parts[i].err;
  }
  float sz = 0.f, szd = 0.f, st = 0.f;
  for (int i = 0; i < n; ++i) {
    const float f = pow2i(nz - parts[i].nz);
    sz = fmaf(parts[i].sz, f, sz);
    szd = fmaf(parts[i].szd, f, szd);
    st = fmaf(parts[i].st, pow2i(nt - parts[i].nt), st);
  }
  out.nz = nz; out.nt = nt; out.mt = mt; out.dmax = dmax; out.cmax = cmax; out.bgrp = bgrp; out.err = err;
  out.sz = sz; out.szd = szd; out.st = st;
}

// Row constants from the combined partials, all in float32:
//   lse   = -n ln2 + ln(S)                     (offsets are integers: n ln2 is near-exact),
//   dlse  = lse_z - lse_t = (nt - nz) ln2 + ln(Sz / St)   (no cancellation of two large logs),
//   KL    = Szd / Sz - dlse.
__device__ __forceinline__ void row_consts(const SlicePartial& all, RowConsts& rc) {
  constexpr float kLn2Lo = -1.9046542e-09f;  // ln 2 - kLn2
  const float nzf = static_cast<float>(all.nz), ntf = static_cast<float>(all.nt);
  rc.lse_z = fmaf(-nzf, kLn2, fmaf(-nzf, kLn2Lo, logf(all.sz)));
  rc.lse_t = fmaf(-ntf, kLn2, fmaf(-ntf, kLn2Lo, logf(all.st)));
  const float dn = static_cast<float>(all.nt - all.nz);
  rc.dlse = fmaf(dn, kLn2, fmaf(dn, kLn2Lo, logf(all.sz / all.st)));
  rc.kl_unclip = all.szd / all.sz - rc.dlse;
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

}  // namespace adaflash

namespace adaflash {
namespace {

// Lowest index of the value mt inside row-global group grp of a target row whose
// groups follow its 16-byte grid: group 0 is the head [0, H) and group G >= 1 holds
// entries [H + 8 (G - 1), H + 8 G) (-1 if absent or out of range).  With a draft row,
// *za receives the draft logit at that index.  Every entry of the group (and of the
// draft row's group) is loaded before the search, so the re-read costs one round trip
// to memory rather than one per entry.
template <class DZ, class DT>
__device__ int resolve_argmax_grid(const uint8_t* trow, const uint8_t* zrow, int grp, float mt, int V, int H,
                                   float* za) {
  if (grp < 0) return -1;
  int v0, n;
  if (grp == 0) {
    v0 = 0;
    n = H;
  } else {
    const long long s = static_cast<long long>(H) + 8ll * (grp - 1);
    if (s >= V) return -1;
    v0 = static_cast<int>(s);
    n = min(8, V - v0);
  }
  const float nan = __int_as_float(0x7fc00000);  // equal to nothing
  float t[8], z[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    t[j] = j < n ? DT::load(trow, v0 + j) : nan;
    z[j] = (zrow != nullptr && j < n) ? DZ::load(zrow, v0 + j) : 0.f;
  }
  int a = -1;
  float zv = 0.f;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (t[j] == mt) {
      a = v0 + j;
      zv = z[j];
    }
  }
  if (za != nullptr) *za = zv;
  return a;
}

}  // namespace
}  // namespace adaflash
