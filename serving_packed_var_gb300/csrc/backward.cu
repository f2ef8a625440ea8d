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

}  // namespace

// Rows need not start on the 16-byte grid: a row's vocabulary follows its target
// row's grid (the head, the first H < 8 entries before the target row's first
// 16-byte boundary, goes through element loads in the CTA of chunk 0; chunk c holds
// body entries [H + c * kBwdChunk, ...)).  Target groups are then 16-byte words; the
// draft row's groups sit 2 zs2 bytes past a boundary and are read with aligned loads
// at that shift (one loop instance per shift); dz is stored at the gradient row's
// own word offset.  kShift = false: every row of z, t and dz is on the grid (the
// shift-free instance, with less code).
template <class DZ, class DT, bool kShift>
__global__ void __launch_bounds__(kBwdThreads) bwd_kernel(const BwdParams P) {
  __shared__ RowCoef s_coef;
  __shared__ int s_ok;
  __shared__ int s_trow;
  // rows in reverse order: the forward's last rows, and the rows the next forward reads
  // first, are the ones still in L2 (287.7 -> 285.1 us for a 128-request forward and
  // backward at V = 151936)
  const int d = P.N_d - 1 - static_cast<int>(blockIdx.x) / P.chunks_per_row;
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
  const RowGeom G = row_geom<DZ, DT, kShift>(zrow, trow, P.V);

  const int b_begin = chunk * kBwdChunk;  // in the body
  const int b_end = min(P.V - G.H, b_begin + kBwdChunk);
  const int nb = max(0, b_end - b_begin);
  const int body = nb & ~7;
  float* gbody = grow + G.H + b_begin;
  const int gq = static_cast<int>((reinterpret_cast<uintptr_t>(gbody) >> 2) & 3u);
  const uint32_t* tw = reinterpret_cast<const uint32_t*>(G.tb + static_cast<int64_t>(b_begin) * DT::kBytes);
  const uint8_t* zb = G.zb + static_cast<int64_t>(b_begin) * DZ::kBytes;

  dispatch_shift<DZ, kShift>(G.zs2, [&](auto zs_c) {
    constexpr int ZS = decltype(zs_c)::value;
    const uint32_t* zw = reinterpret_cast<const uint32_t*>(zb - 2 * ZS);  // the 16-byte boundary below
#pragma unroll
    for (int j = 0; j < kPerThread / 8; ++j) {
      const int off = (j * kBwdThreads + static_cast<int>(threadIdx.x)) * 8;
      if (off < body) {
        float z[8], t[8], out[8];
        load8_shifted<DZ, ZS, true>(zw + off * DZ::kBytes / 4, z);
        load8_shifted<DT, 0, true>(tw + off * DT::kBytes / 4, t);
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = grad_entry(z[e], t[e], k);
        store8_stream<kShift>(gbody + off, gq, out);
      }
    }
  });
  // the ragged end of the chunk and, in chunk 0, the row's head: element loads
  for (int v = G.H + b_begin + body + static_cast<int>(threadIdx.x); v < G.H + b_end; v += kBwdThreads)
    grow[v] = grad_entry(DZ::load(zrow, v), DT::load(trow, v), k);
  if (chunk == 0)
    for (int v = static_cast<int>(threadIdx.x); v < G.H; v += kBwdThreads)
      grow[v] = grad_entry(DZ::load(zrow, v), DT::load(trow, v), k);
  __syncthreads();
  // The hard-label term's -beta*g at the target argmax (written after the row's
  // stores above by the CTA that holds that entry).
  const bool owns = (k.a >= G.H + b_begin && k.a < G.H + b_end) || (chunk == 0 && k.a < G.H);
  if (threadIdx.x == 0 && owns) {
    const float base = grad_entry(DZ::load(zrow, k.a), DT::load(trow, k.a), k);
    grow[k.a] = __fsub_rn(base, __fmul_rn(P.ce_weight, k.g));
  }
}

template <class DZ, class DT, bool kShift>
static cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t s) {
  const long long blocks = static_cast<long long>(p.N_d) * p.chunks_per_row;
  if (blocks <= 0) return cudaSuccess;
  count_launch();
  bwd_kernel<DZ, DT, kShift><<<static_cast<unsigned>(blocks), kBwdThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <bool kShift>
static cudaError_t launch_bwd_dtypes(const BwdParams& p, int z_dtype, int t_dtype, cudaStream_t s) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (zb && tb) return launch_bwd_t<BF16, BF16, kShift>(p, s);
  if (!zb && tb) return launch_bwd_t<F32, BF16, kShift>(p, s);
  if (zb && !tb) return launch_bwd_t<BF16, F32, kShift>(p, s);
  return launch_bwd_t<F32, F32, kShift>(p, s);
}

cudaError_t launch_bwd(const BwdParams& p, int z_dtype, int t_dtype, bool aligned, cudaStream_t s) {
  return aligned ? launch_bwd_dtypes<false>(p, z_dtype, t_dtype, s) : launch_bwd_dtypes<true>(p, z_dtype, t_dtype, s);
}

}  // namespace adaflash
