// sampled.cu -- temperature-sampled verification of packed draft blocks.
//
// The target verifies the drafted tokens in parallel (AdaFlash article, "AdaFlash:
// Adaptive Speculative Decoding with Online Self-Improvement for High-Concurrency
// LLM Inference", opening section); the temperature is a tunable of the method
// (skill card "AdaFlash Adaptive Speculative Decoding", "Implementation Steps").
// With p = softmax(z/T) and q = softmax(t/T) the rule is speculative sampling:
//
//   token j is accepted when u_j p(x_j) < q(x_j);
//   at the first rejection the emitted token is drawn from max(0, q - p) (q when
//   that is all zero); when all are accepted it is drawn from q at the bonus row;
//   a draw with uniform w is the smallest v whose prefix sum exceeds w * total.
//
// S1 computes log-sum-exp(x / T) of every draft row and every target row (one
// read of each logit, 128-bit loads where rows are 16-byte aligned), S2 applies the
// accept rule (one warp per request, k <= 16 lanes), S3 draws the emitted token
// (one CTA per request: fixed-order per-thread sums over contiguous chunks, a block
// scan, then one thread walks the chunk that holds the threshold).
#include <climits>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace adaflash {

namespace {

constexpr int kLseThreads = 256;
constexpr int kDrawThreads = 1024;

// (max, sum of 2^{(x - max) * scale}) per thread, combined by warps then CTA.
// Entries equal to -inf contribute nothing.
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

// ln sum_v exp(x_v / T) of one row, computed by the whole CTA (red holds 2 * 32
// floats).  Every thread gets the result.  The same sequence of operations for any
// row of one type and alignment, so equal rows give equal results bit for bit.
template <class DT>
__device__ float row_lse(const uint8_t* row, int V, bool vec, float inv_t, float* red) {
  const float scale = kLog2e * inv_t;
  MaxSum a{kNegInf, 0.f};
  int v0 = 0;
  if (vec) {
    constexpr int E = 16 / DT::kBytes;
    const int nvec = V / E;
    const uint4* rw = reinterpret_cast<const uint4*>(row);
    int j = threadIdx.x;
    for (; j + static_cast<int>(blockDim.x) < nvec; j += 2 * blockDim.x) {
      const uint4 w0 = __ldcs(rw + j), w1 = __ldcs(rw + j + blockDim.x);
      float x0[E], x1[E];
      unpack16(w0, x0);
      unpack16(w1, x1);
      ms_add_group<E>(a, x0, scale);
      ms_add_group<E>(a, x1, scale);
    }
    if (j < nvec) {
      float x0[E];
      unpack16(__ldcs(rw + j), x0);
      ms_add_group<E>(a, x0, scale);
    }
    v0 = nvec * E;
  }
  for (int v = v0 + threadIdx.x; v < V; v += blockDim.x) ms_add(a, DT::load(row, v), scale);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    MaxSum b{__shfl_xor_sync(0xffffffffu, a.m, off), __shfl_xor_sync(0xffffffffu, a.s, off)};
    a = ms_merge(a, b, scale);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) {
    red[warp] = a.m;
    red[32 + warp] = a.s;
  }
  __syncthreads();
  MaxSum t{kNegInf, 0.f};
  for (int w = 0; w < nw; ++w) t = ms_merge(t, MaxSum{red[w], red[32 + w]}, scale);
  // lse = m / T + ln(s)
  return t.m * inv_t + logf(t.s);
}

// p = exp(x / T - lse) for one entry.
__device__ __forceinline__ float prob_at(float x, float inv_t, float lse) {
  return ex2(fmaf(x, inv_t, -lse) * kLog2e);
}

}  // namespace

// ---- S1: log-sum-exp at temperature of every draft row and every target row ----
template <class DZ, class DT>
__global__ void __launch_bounds__(kLseThreads) lse_rows_kernel(const SampledParams P) {
  __shared__ float red[64];
  const int b = static_cast<int>(blockIdx.x);
  float lse;
  if (b < P.N_d) {
    lse = row_lse<DZ>(static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(b) * P.ld_z * DZ::kBytes, P.V,
                      P.z_vec != 0, P.inv_t, red);
  } else {
    lse = row_lse<DT>(static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(b - P.N_d) * P.ld_t * DT::kBytes,
                      P.V, P.t_vec != 0, P.inv_t, red);
  }
  if (threadIdx.x == 0) P.row_lse[b] = lse;
}

// ---- S2: the accept rule, one warp per request ----
template <class DZ, class DT>
__global__ void __launch_bounds__(256) sampled_accept_kernel(const SampledParams P) {
  const int lane = threadIdx.x & 31;
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (i >= P.R) return;
  const int d0 = __ldg(P.doff + i), d1 = __ldg(P.doff + i + 1);
  const int k = d1 - d0;
  bool ok = (k >= 1) && (k <= ADAFLASH_MAX_K) && (d0 >= 0) && (d1 <= P.N_d);
  if (i == 0 && d0 != 0) ok = false;
  if (i == P.R - 1 && d1 != P.N_d) ok = false;
  if (!ok) {
    if (lane == 0) {
      P.accept_len[i] = -1;
      P.next_token[i] = -1;
      P.accept_rate[i] = -1.f;
      flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
    }
    return;
  }
  bool reject = false, badtok = false;
  if (lane < k) {
    const int d = d0 + lane, s = d0 + i + lane;
    const int x = __ldg(P.tokens + d);
    badtok = (x < 0) || (x >= P.V);
    if (badtok) {
      reject = true;
    } else {
      const float zx = DZ::load(static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(d) * P.ld_z * DZ::kBytes, x);
      const float tx = DT::load(static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(s) * P.ld_t * DT::kBytes, x);
      const float p = prob_at(zx, P.inv_t, P.row_lse[d]);
      const float q = prob_at(tx, P.inv_t, P.row_lse[P.N_d + s]);
      reject = !(__ldg(P.u_accept + d) * p < q);
    }
  }
  const unsigned rj = __ballot_sync(0xffffffffu, reject);
  const unsigned bt = __ballot_sync(0xffffffffu, badtok);
  if (lane == 0) {
    const int L = rj ? (__ffs(rj) - 1) : k;
    P.accept_len[i] = L;
    P.accept_rate[i] = __fdiv_rn(static_cast<float>(L), static_cast<float>(k));
    if (bt) flag_status(P.status, ADAFLASH_ERR_BAD_TOKEN);
  }
}

// ---- S3: draw the emitted token, one CTA per request ----
template <class DZ, class DT>
__global__ void __launch_bounds__(kDrawThreads) sampled_draw_kernel(const SampledParams P) {
  __shared__ float scan[kDrawThreads / 32];
  __shared__ int s_mode, s_owner;
  const int i = blockIdx.x;
  const int L = P.accept_len[i];
  if (L < 0) return;  // malformed request (flagged by S2)
  const int d0 = __ldg(P.doff + i), d1 = __ldg(P.doff + i + 1);
  const int k = d1 - d0;
  const int V = P.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // L < k: residual max(0, q - p) at the first rejected position; L = k: q at the bonus row
  int mode = (L < k) ? 0 : 1;
  const int dz = d0 + min(L, k - 1);  // draft row of the rejected position (unused when mode = 1)
  const int st = d0 + i + L;          // target row of the emitted position
  const uint8_t* zrow = static_cast<const uint8_t*>(P.z) + static_cast<int64_t>(dz) * P.ld_z * DZ::kBytes;
  const uint8_t* trow = static_cast<const uint8_t*>(P.t) + static_cast<int64_t>(st) * P.ld_t * DT::kBytes;
  const float lse_z = P.row_lse[dz];
  const float lse_t = P.row_lse[P.N_d + st];
  const int per = (V + kDrawThreads - 1) / kDrawThreads;
  const int c0 = min(V, tid * per), c1 = min(V, c0 + per);
  const float w = fminf(fmaxf(__ldg(P.u_sample + i), 0.f), 1.f);  // NaN -> 0

  auto weight = [&](int v, int md) -> float {
    const float q = prob_at(DT::load(trow, v), P.inv_t, lse_t);
    if (md == 1) return q;
    return fmaxf(q - prob_at(DZ::load(zrow, v), P.inv_t, lse_z), 0.f);
  };

  for (int pass = 0; pass < 2; ++pass) {
    // fixed-order sum of this thread's contiguous chunk
    float own = 0.f;
    for (int v = c0; v < c1; ++v) own += weight(v, mode);
    // block inclusive scan of the chunk sums (warp shuffles, then warp totals)
    float incw = own;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incw, off);
      if (lane >= off) incw += y;
    }
    float exclw = __shfl_up_sync(0xffffffffu, incw, 1);
    if (lane == 0) exclw = 0.f;
    __syncthreads();
    if (lane == 31) scan[warp] = incw;
    __syncthreads();
    float before = 0.f, total = 0.f;
    for (int ww = 0; ww < kDrawThreads / 32; ++ww) {
      if (ww < warp) before += scan[ww];
      total += scan[ww];
    }
    const float excl = lane == 0 ? before : exclw + before;
    if (total > 0.f || mode == 1) {
      const float target = w * total;
      // The owner is the last thread with positive mass whose prefix does not pass
      // the threshold.  The first such thread has prefix exactly 0, so one exists
      // whenever total > 0, and rounding in the scan cannot leave it unassigned.
      if (tid == 0) s_owner = -1;
      __syncthreads();
      if (own > 0.f && (excl <= target || !(target < total))) atomicMax(&s_owner, tid);
      __syncthreads();
      if (tid == s_owner) {
        float acc = excl;
        int pick = -1, last = -1;
        for (int v = c0; v < c1; ++v) {
          const float wv = weight(v, mode);
          if (wv > 0.f) last = v;
          acc += wv;
          if (acc > target) {
            pick = v;
            break;
          }
        }
        P.next_token[i] = pick < 0 ? last : pick;
      } else if (tid == 0 && s_owner < 0) {
        P.next_token[i] = -1;  // no mass at all (non-finite logits)
      }
      break;
    }
    // residual of identical distributions is all zero: draw from q instead
    if (tid == 0) s_mode = 1;
    __syncthreads();
    mode = s_mode;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <class DZ, class DT>
static cudaError_t launch_sampled_t(const SampledParams& p, cudaStream_t s) {
  if (p.R <= 0) return cudaSuccess;
  count_launch();
  lse_rows_kernel<DZ, DT><<<static_cast<unsigned>(p.N_d + p.N_t), kLseThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch();
  sampled_accept_kernel<DZ, DT><<<static_cast<unsigned>((p.R * 32 + 255) / 256), 256, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch();
  sampled_draw_kernel<DZ, DT><<<static_cast<unsigned>(p.R), kDrawThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sampled(const SampledParams& p, int z_dtype, int t_dtype, cudaStream_t s) {
  const bool zb = (z_dtype == 1), tb = (t_dtype == 1);
  if (zb && tb) return launch_sampled_t<BF16, BF16>(p, s);
  if (!zb && tb) return launch_sampled_t<F32, BF16>(p, s);
  if (zb && !tb) return launch_sampled_t<BF16, F32>(p, s);
  return launch_sampled_t<F32, F32>(p, s);
}

}  // namespace adaflash
