// kernels.h -- internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace adaflash {

enum RowPassMode : int32_t {
  kModeVerify = 0,  // every target row is a target-only unit (argmax only)
  kModeFwd = 1,     // draft rows are paired units, bonus target rows are target-only units
};

struct RowPassParams {
  const void* z;  // draft logits [N_d, ld_z]
  const void* t;  // target logits [N_t, ld_t]
  int64_t ld_z, ld_t;
  const int32_t* doff;
  int32_t R, N_d, N_t, V;
  int32_t mode;
  int32_t cluster;  // CTAs per row unit (1..8)
  int32_t slice;    // vocabulary entries per CTA (multiple of 8)
  int32_t unit_begin, unit_end;  // units handled by this launch (set by launch_rowpass)
  int32_t wait_prior;            // 1: complete only after the preceding launch has completed
  float clip_c;
  int32_t* target_argmax;
  float* kl_row;
  float* ce_row;
  float* row_stats;
  uint32_t* status;
  // fused forward + backward only (K4, and the row pass with the gradient)
  float ce_weight;
  const float* grad_row;  // NULL: grad_scale for every row
  float grad_scale;
  float* grad;            // [N_d, ld_g] float32
  int64_t ld_g;
};

struct FinalizeParams {
  const int32_t* tokens;
  const int32_t* doff;
  const int32_t* target_argmax;
  int32_t R, N_d, V;
  int32_t* accept_len;
  int32_t* bonus_token;
  float* accept_rate;
  const float* kl_row;  // NULL: no loss
  const float* ce_row;
  float ce_weight;
  float* loss;
  uint32_t* status;
};

struct BwdParams {
  const void* z;
  const void* t;
  int64_t ld_z, ld_t;
  const int32_t* doff;
  int32_t R, N_d, N_t, V;
  float clip_c, ce_weight;
  const int32_t* target_argmax;
  const float* row_stats;
  const float* grad_row;
  float grad_scale;
  float* grad;
  int64_t ld_g;
  int32_t chunks_per_row;
  uint32_t* status;
};

struct SampledParams {
  const void* z;  // draft logits [N_d, ld_z]
  const void* t;  // target logits [N_t, ld_t]
  int64_t ld_z, ld_t;
  const int32_t* doff;
  int32_t R, N_d, N_t, V;
  float inv_t;  // 1 / temperature
  const int32_t* tokens;
  const float* u_accept;  // [N_d]
  const float* u_sample;  // [R]
  float* row_lse;         // [N_d + N_t]: draft rows, then target rows
  int32_t* accept_len;
  int32_t* next_token;
  float* accept_rate;
  uint32_t* status;
};

// One row's statistics over one 256-entry vocabulary tile of the LM-head path.
struct __align__(16) LmPartial {
  float mz, sz, szd, dmax;  // max z, sum e^{z - mz}, sum e^{z - mz} (z - t), max (z - t)
  float z2, mt, st;         // second largest z, max t, sum e^{t - mt}
  int32_t az, at;           // first index of the largest z, of the largest t
  float zat;                // z at that index of t
  int32_t pad1, pad2;
};

struct LmHeadParams {
  int32_t n_pair_tiles;  // 128-row tiles of (draft row, paired target row)
  int32_t n_pair_rows;   // N_d
  int32_t n_t_rows;      // rows of the target operand: N_d paired rows, then the bonus rows
  int32_t V, H;
  int32_t n_vtiles;
  int32_t mode;          // 0: partial records, 1: write the logits (diagnostic)
  LmPartial* partials;   // [n_t_rows][n_vtiles]
  float* out_z;          // mode 1
  float* out_t;
  int64_t ld_out;
  uint32_t* status;
};

struct LmCombineParams {
  const uint16_t* hd;  // bf16 [N_d, ld_hd]
  const uint16_t* ht;  // bf16 gathered target rows [N_d + R, H] (pair order, then bonus rows)
  const uint16_t* wd;  // bf16 [V, ld_wd]
  const uint16_t* wt;
  int64_t ld_hd, ld_wd, ld_wt;
  const int32_t* doff;
  int32_t R, N_d, V, H, n_vtiles;
  float clip_c;
  const LmPartial* partials;
  int32_t* target_argmax;
  float* kl_row;
  float* ce_row;
  float* row_stats;
  uint32_t* status;
};

// Launch counter behind adaflash_kernel_launches (incremented once per launch).
void count_launch();
// Raises a kernel's dynamic shared-memory limit on the current device to at least
// `bytes`, never lowering it, so host threads launching one kernel with different
// sizes cannot undo each other's setting between setting it and launching.
cudaError_t raise_smem_limit(const void* fn, size_t bytes);

// dtype codes match adaflash_dtype (0 = fp32, 1 = bf16)
// The row pass (rows at any element-aligned address: each row follows its target
// row's 16-byte grid).  aligned: every row of z and t (and of the gradient) starts on
// the 16-byte grid, which selects the smaller shift-free instance.
cudaError_t launch_rowpass(const RowPassParams& p, int z_dtype, int t_dtype, bool aligned, cudaStream_t s);
// The row pass with the gradient (single-pass forward + backward, any element-aligned
// rows).  Cluster size: rowpass_grad_cluster_size (row_bytes = V (b_z + b_t)).
cudaError_t launch_rowpass_grad(const RowPassParams& p, int z_dtype, int t_dtype, bool aligned, cudaStream_t s);
int rowpass_grad_cluster_size(int vocab, int units, int row_bytes, int chunk_entries, int num_sms, long long l2_bytes);
// The largest cluster size that takes every row unit in one round of resident clusters
// (else 0): for the forward and verification (units: their rows), and for the pass with
// the gradient on batches whose paired rows all fit the L2 at once (pairs: paired rows).
int rowpass_one_round_cluster(int z_dtype, int t_dtype, bool aligned, int vocab, int units);
int rowpass_grad_one_round_cluster(int z_dtype, int t_dtype, bool aligned, int vocab, int pairs);
int rowpass_grad_chunk(int z_dtype, int t_dtype);  // vocabulary entries per ring stage
cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s);
// The backward (rows at any element-aligned address; aligned: every row of z, t and
// dz on the 16-byte grid, the shift-free instance).
cudaError_t launch_bwd(const BwdParams& p, int z_dtype, int t_dtype, bool aligned, cudaStream_t s);
// Fused forward + backward (K4).  fused_max_units is the largest batch (draft rows +
// requests) the fused kernel is used for (its clusters all resident with one CTA per
// SM): 0 when a row pair does not fit a cluster's shared memory; above it the caller
// runs the row pass with the gradient, which streams faster.
cudaError_t launch_fused(const RowPassParams& p, int z_dtype, int t_dtype, int num_sms, cudaStream_t s);
int fused_cluster_size(int vocab, int bytes_per_entry);
int fused_max_units(int vocab, int z_dtype, int t_dtype, int num_sms);
// LM-head path: gather of the target hidden rows into pair order (workspace), the
// tcgen05 GEMM with its per-tile reduction (or logits), and the per-row combine.
cudaError_t launch_lm_gather(const uint16_t* ht, int64_t ld_ht, const int32_t* doff, int R, int N_d, int H,
                             uint16_t* out, uint32_t* status, cudaStream_t s);
cudaError_t launch_lm_gemm(const uint16_t* hd, int64_t ld_hd, const uint16_t* ht_pairs, int64_t ld_ht,
                           const uint16_t* wd, int64_t ld_wd, const uint16_t* wt, int64_t ld_wt,
                           const LmHeadParams& p, cudaStream_t s);
cudaError_t launch_lm_combine(const LmCombineParams& p, cudaStream_t s);
// Device address (looked up once per device) and size of the static scratch array.
cudaError_t lm_static_scratch(void** ptr, int64_t* bytes);
cudaError_t launch_sampled(const SampledParams& p, int z_dtype, int t_dtype, int num_sms, cudaStream_t s);
cudaError_t launch_selftest_wait(uint32_t* status, int32_t limit_us, cudaStream_t s);

// Geometry chosen for a vocabulary size (shared by host validation and launches).
int rowpass_cluster_size(int vocab, int units, int num_sms);
int rowpass_slice(int vocab, int cluster);
constexpr int kBwdChunk = 8192;  // vocabulary entries per backward CTA

}  // namespace adaflash
