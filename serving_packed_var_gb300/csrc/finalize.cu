// finalize.cu -- K2: per-request greedy acceptance over the packed offsets, and the
// batch loss as a fixed-order float64 sum.
//
// Greedy acceptance (AdaFlash article, opening section: the target verifies the
// drafted block in parallel): with a_j the target's choice at the position of
// draft token j, L_i is the first j whose token differs from a_j (k_i if none),
// the bonus token is the target's choice at the position right after the accepted
// prefix, and the acceptance rate L_i / k_i is the length head's free label
// (section "2. Adaptive Length Head for Token-Level Variance").  One warp handles
// one request: k_i <= 16 fits in one ballot.
//
// The loss is the mean over draft rows of kl + ce_weight * ce (the "mixture
// reverse-KL loss" of the AdaFlash README, "Released Checkpoint").
#include "common.cuh"
#include "kernels.h"

namespace adaflash {

namespace {
constexpr int kFinThreads = 1024;
}

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const FinalizeParams P) {
  // Launched as a programmatic dependent of the row pass: wait until its writes
  // (target_argmax, kl_row, ce_row) are complete and visible.  This grid releases
  // the next call's row pass only when it exits: released right after the wait, the
  // next persistent row pass was launched while these 1024-thread blocks still held
  // SMs, and on a 512-request batch the call took 3.63 ms instead of 2.51 ms.
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * kFinThreads + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * kFinThreads) >> 5;

  // The offsets and the tokens are inputs the row pass does not write: the first
  // request's are read before waiting for it.
  int d0 = 0, d1 = 0, tok = 0;
  auto load_inputs = [&](int r) {
    d0 = __ldg(P.doff + r);
    d1 = __ldg(P.doff + r + 1);
    const int k = d1 - d0;
    tok = (lane < k && k <= ADAFLASH_MAX_K && d0 >= 0 && d1 <= P.N_d) ? __ldg(P.tokens + d0 + lane) : 0;
  };
  if (gwarp < P.R) load_inputs(gwarp);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (int i = gwarp; i < P.R; i += nwarps) {
    if (i != gwarp) load_inputs(i);
    const int k = d1 - d0;
    bool ok = (k >= 1) && (k <= ADAFLASH_MAX_K) && (d0 >= 0) && (d1 <= P.N_d);
    if (i == 0 && d0 != 0) ok = false;
    if (i == P.R - 1 && d1 != P.N_d) ok = false;
    if (!ok) {
      if (lane == 0) {
        P.accept_len[i] = -1;
        P.bonus_token[i] = -1;
        P.accept_rate[i] = -1.0f;
        flag_status(P.status, ADAFLASH_ERR_BAD_OFFSETS);
      }
      continue;
    }
    // lanes 0..k read the target's choice at the request's k + 1 positions (the last one
    // is the bonus position), so the bonus token is a shuffle, not a second load
    const int a = lane <= k ? __ldg(P.target_argmax + d0 + i + lane) : -1;
    bool mismatch = false, badtok = false;
    if (lane < k) {
      badtok = (tok < 0) || (tok >= P.V);
      mismatch = badtok || (tok != a);
    }
    const unsigned mm = __ballot_sync(0xffffffffu, mismatch);
    const unsigned bt = __ballot_sync(0xffffffffu, badtok);
    const int L = mm ? (__ffs(mm) - 1) : k;
    const int bonus = __shfl_sync(0xffffffffu, a, L);
    if (lane == 0) {
      P.accept_len[i] = L;
      P.bonus_token[i] = bonus;
      P.accept_rate[i] = __fdiv_rn(static_cast<float>(L), static_cast<float>(k));
      if (bt) flag_status(P.status, ADAFLASH_ERR_BAD_TOKEN);
    }
  }

  if (P.kl_row == nullptr || blockIdx.x != 0) return;

  // Fixed-order float32 reduction (GB300's float64 pipe is narrow): each thread
  // sums a fixed strided subset with compensation (Kahan), then a fixed warp and
  // block tree.  The order never changes, so the loss is bitwise reproducible;
  // its relative error is about 1e-6, far below the loss tolerance.
  __shared__ float part[kFinThreads / 32];
  float acc = 0.f, comp = 0.f;
  for (int r = threadIdx.x; r < P.N_d; r += kFinThreads) {
    const float y = __fsub_rn(fmaf(P.ce_weight, P.ce_row[r], P.kl_row[r]), comp);
    const float t = __fadd_rn(acc, y);
    comp = __fsub_rn(__fsub_rn(t, acc), y);
    acc = t;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = part[threadIdx.x];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (threadIdx.x == 0) P.loss[0] = P.N_d > 0 ? v / static_cast<float>(P.N_d) : 0.0f;
  }
}

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s) {
  const int warps_per_block = kFinThreads / 32;
  int blocks = (p.R + warps_per_block - 1) / warps_per_block;
  if (blocks < 1) blocks = 1;
  if (blocks > 1024) blocks = 1024;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kFinThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, finalize_kernel, p);
}

// ---------------------------------------------------------------------------
// bounded-wait self-test: a barrier nothing completes, a wait that must give up
// ---------------------------------------------------------------------------
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Phase 0 never completes: nobody arrives.
  const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
  if (!ok && threadIdx.x == 0) flag_status(status, ADAFLASH_ERR_TIMEOUT);
}

cudaError_t launch_selftest_wait(uint32_t* status, int32_t limit_us, cudaStream_t s) {
  count_launch();
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError();
}

}  // namespace adaflash
