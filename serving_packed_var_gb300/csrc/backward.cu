// backward.cu -- K3: gradient of the OPD loss with respect to the draft logits.
//
// Training updates the serving draft model from verification results (AdaFlash
// article, "On-Policy Distillation (OPD) for Domain Adaptation"); the target
// model is fixed ("Decoupled training/inference": the target model never
// changes), so only the draft logits get a gradient.  For row r with upstream
// weight g, p = softmax(z), r_v = log p_v - log q_v, m_v = [p_v r_v <= c]:
//
//   dz_v = g * ( p_v (m_v (r_v + 1) - S) + beta (p_v - [v == a]) ),
//   S    = sum_u m_u p_u (r_u + 1)            (from the forward's row_stats),
//
// a streaming elementwise pass: z and t are read once, dz written once.  The clip
// decision m_v is evaluated with the same instruction sequence as the forward's
// screen, from the same stored float32 log-sum-exps.
#include "common.cuh"
#include "kernels.h"

#ifndef ADAFLASH_BWD_REVERSE
#define ADAFLASH_BWD_REVERSE 1
#endif

namespace adaflash {

namespace {
constexpr int kBwdThreads = 256;
constexpr int kPerThread = kBwdChunk / kBwdThreads;  // 32 entries = 4 groups of 8
static_assert(kPerThread % 8 == 0, "groups of 8");

struct RowCoef {
  TermConsts tc;
  float c;
  float k_m;     // 1 + beta - S   (inner factor where the term is kept: r + k_m)
  float k_clip;  // beta - S       (inner factor where the term is clipped)
  float g;
  int a;
};

__device__ __forceinline__ float grad_entry(float z, float t, const RowCoef& k) {
  float p, r, term;
  entry_term(z, t, k.tc, p, r, term);
  const float inner = (term <= k.c) ? __fadd_rn(r, k.k_m) : k.k_clip;
  return __fmul_rn(__fmul_rn(p, inner), k.g);
}

template <class DT>
__device__ __forceinline__ void load8_vec(const uint8_t* row, int64_t v0, float x[8]);

template <>
__device__ __forceinline__ void load8_vec<BF16>(const uint8_t* row, int64_t v0, float x[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(row + v0 * 2));
  x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x);
  x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
  x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z);
  x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
}

template <>
__device__ __forceinline__ void load8_vec<F32>(const uint8_t* row, int64_t v0, float x[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(row + v0 * 4));
  const float4 b = __ldg(reinterpret_cast<const float4*>(row + v0 * 4 + 16));
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
}  // namespace

template <class DZ, class DT, bool kFast>
__global__ void __launch_bounds__(kBwdThreads) bwd_kernel(const BwdParams P) {
  __shared__ RowCoef s_coef;
  __shared__ int s_ok;
  __shared__ int s_trow;
#if ADAFLASH_BWD_REVERSE
  // rows in reverse order: the forward's last rows, and the rows the next forward reads
  // first, are the ones still in L2
  const int d = P.N_d - 1 - static_cast<int>(blockIdx.x) / P.chunks_per_row;
#else
  const int d = static_cast<int>(blockIdx.x) / P.chunks_per_row;
#endif
  const int chunk = static_cast<int>(blockIdx.x) % P.chunks_per_row;

  if (threadIdx.x == 0) {
    const int i = request_of_row(P.doff, P.R, d);
    const int lo = __ldg(P.doff + i), hi = __ldg(P.doff + i + 1);
    const int s = d + i;
    bool ok = (lo <= d) && (d < hi) && (s < P.N_t);
    int a = ok ? __ldg(P.target_argmax + s) : -1;
    if (a < 0 || a >= P.V) ok = false;
    if (!ok) {
      if (chunk == 0) flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
    } else {
      const float lse_z = __ldg(P.row_stats + 4 * static_cast<int64_t>(d) + 0);
      const float lse_t = __ldg(P.row_stats + 4 * static_cast<int64_t>(d) + 1);
      const float S = __ldg(P.row_stats + 4 * static_cast<int64_t>(d) + 2);
      RowCoef k;
      k.tc = make_term_consts(lse_z, lse_t);
      k.c = P.clip_c;
      k.k_clip = __fsub_rn(P.ce_weight, S);
      k.k_m = __fadd_rn(1.0f, k.k_clip);
      k.g = P.grad_row ? __ldg(P.grad_row + d) : P.grad_scale;
      k.a = a;
      s_coef = k;
    }
    s_ok = ok;
    s_trow = s;
  }
  __syncthreads();
  if (!s_ok) return;
  const RowCoef k = s_coef;

  const uint8_t* zrow = static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(d) * P.ld_z * DZ::kBytes;
  const uint8_t* trow = static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(s_trow) * P.ld_t * DT::kBytes;
  float* grow = P.grad + static_cast<int64_t>(d) * P.ld_g;

  const int v_begin = chunk * kBwdChunk;
  const int v_end = min(P.V, v_begin + kBwdChunk);

  if (kFast) {
    const int body = (v_end - v_begin) & ~7;
#pragma unroll
    for (int j = 0; j < kPerThread / 8; ++j) {
      const int off = (j * kBwdThreads + static_cast<int>(threadIdx.x)) * 8;
      if (off < body) {
        const int64_t v0 = v_begin + off;
        float z[8], t[8], out[8];
        load8_vec<DZ>(zrow, v0, z);
        load8_vec<DT>(trow, v0, t);
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = grad_entry(z[e], t[e], k);
        float4* dst = reinterpret_cast<float4*>(grow + v0);
        __stcs(dst, make_float4(out[0], out[1], out[2], out[3]));
        __stcs(dst + 1, make_float4(out[4], out[5], out[6], out[7]));
      }
    }
    for (int v = v_begin + body + static_cast<int>(threadIdx.x); v < v_end; v += kBwdThreads)
      grow[v] = grad_entry(DZ::load(zrow, v), DT::load(trow, v), k);
  } else {
    for (int v = v_begin + static_cast<int>(threadIdx.x); v < v_end; v += kBwdThreads)
      __stcs(grow + v, grad_entry(DZ::load(zrow, v), DT::load(trow, v), k));
  }
  __syncthreads();
  // The hard-label term's -beta*g at the target argmax (written after the row's
  // stores above by the thread that owns that chunk).
  if (threadIdx.x == 0 && k.a >= v_begin && k.a < v_end) {
    const float base = grad_entry(DZ::load(zrow, k.a), DT::load(trow, k.a), k);
    grow[k.a] = __fsub_rn(base, __fmul_rn(P.ce_weight, k.g));
  }
}

template <class DZ, class DT, bool kFast>
static cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.N_d) * p.chunks_per_row;
  if (blocks <= 0) return cudaSuccess;
  count_launch();
  bwd_kernel<DZ, DT, kFast><<<static_cast<unsigned>(blocks), kBwdThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdParams& p, int z_dtype, int t_dtype, bool fast, cudaStream_t s) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (fast) {
    if (zb && tb) return launch_bwd_t<BF16, BF16, true>(p, s);
    if (!zb && tb) return launch_bwd_t<F32, BF16, true>(p, s);
    if (zb && !tb) return launch_bwd_t<BF16, F32, true>(p, s);
    return launch_bwd_t<F32, F32, true>(p, s);
  }
  if (zb && tb) return launch_bwd_t<BF16, BF16, false>(p, s);
  if (!zb && tb) return launch_bwd_t<F32, BF16, false>(p, s);
  if (zb && !tb) return launch_bwd_t<BF16, F32, false>(p, s);
  return launch_bwd_t<F32, F32, false>(p, s);
}

}  // namespace adaflash
