// api.cu -- the extern "C" entry points declared in include/adaflash.h.
//
// Host-side argument validation happens before any CUDA call, so malformed calls
// return at once and enqueue nothing.  Every accepted call enqueues its kernels on
// the caller's stream and returns without synchronising.
#include <atomic>
#include <mutex>
#include <vector>
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/adaflash.h"
#include "kernels.h"

using namespace adaflash;

namespace {

bool valid_dtype(adaflash_dtype t) { return t == ADAFLASH_FP32 || t == ADAFLASH_BF16; }
int dtype_bytes(adaflash_dtype t) { return t == ADAFLASH_FP32 ? 4 : 2; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Rows of a [N, ld] matrix start on 16-byte boundaries (bulk-copy / 128-bit path).
bool rows_16b(const void* base, int64_t ld, int bytes) {
  return aligned(base, 16) && ((ld * bytes) % 16 == 0);
}

// Shape checks shared by all entry points.
adaflash_status check_shape(int32_t R, int32_t N_d, int32_t V) {
  if (V < 1 || R < 0 || N_d < 0) return ADAFLASH_ERR_INVALID_ARG;
  if (V > ADAFLASH_MAX_VOCAB) return ADAFLASH_ERR_UNSUPPORTED;
  if (R == 0 && N_d != 0) return ADAFLASH_ERR_INVALID_ARG;
  if (static_cast<int64_t>(N_d) < R || static_cast<int64_t>(N_d) > static_cast<int64_t>(ADAFLASH_MAX_K) * R)
    return ADAFLASH_ERR_INVALID_ARG;
  if (static_cast<int64_t>(N_d) + R > INT32_MAX) return ADAFLASH_ERR_INVALID_ARG;
  return ADAFLASH_OK;
}

adaflash_status check_logits(const void* p, adaflash_dtype dt, int64_t ld, int32_t V) {
  if (!p || !valid_dtype(dt) || ld < V) return ADAFLASH_ERR_INVALID_ARG;
  if (!aligned(p, static_cast<uintptr_t>(dtype_bytes(dt)))) return ADAFLASH_ERR_INVALID_ARG;
  return ADAFLASH_OK;
}

bool int_ptr_ok(const void* p) { return p && aligned(p, 4); }

// The device must be compute capability 10.3 (checked once per device).
adaflash_status check_device() {
  static std::atomic<int> cache[64];  // 0 unknown, 1 ok, 2 unsupported (host threads may race: same value)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ADAFLASH_ERR_CUDA;
  const int known = (dev >= 0 && dev < 64) ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (known) return known == 1 ? ADAFLASH_OK : ADAFLASH_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ADAFLASH_ERR_CUDA;
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) cache[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? ADAFLASH_OK : ADAFLASH_ERR_UNSUPPORTED;
}

// Streaming multiprocessors of the current device (cached per device).
int num_sms() {
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

// L2 size of the current device in bytes (cached per device; 0 if unknown).
long long l2_bytes() {
  static std::atomic<long long> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const long long known = (dev >= 0 && dev < 64) ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (known) return known;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n < 1) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

#define ADAFLASH_TRY(expr)                          \
  do {                                              \
    const adaflash_status st_ = (expr);             \
    if (st_ != ADAFLASH_OK) return st_;             \
  } while (0)

#define ADAFLASH_CUDA(expr)                              \
  do {                                                   \
    if ((expr) != cudaSuccess) return ADAFLASH_ERR_CUDA; \
  } while (0)

// An empty batch (no requests, so no rows): nothing is read, whatever the row and
// token pointers hold (NULL included); the only write is loss = 0 where the entry
// point has a loss.
adaflash_status empty_batch(float* loss, bool has_loss, const uint32_t* d_status, cudaStream_t s) {
  if (has_loss && !int_ptr_ok(loss)) return ADAFLASH_ERR_INVALID_ARG;
  if (d_status && !aligned(d_status, 4)) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());
  if (has_loss) ADAFLASH_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), s));
  return ADAFLASH_OK;
}

// The acceptance scan and loss kernel (K2) after a row pass: the verification outputs,
// and the loss where kl_row is given.
cudaError_t finalize_after(const int32_t* tokens, const int32_t* doff, const int32_t* target_argmax, int32_t R,
                           int32_t N_d, int32_t V, int32_t* accept_len, int32_t* bonus_token, float* accept_rate,
                           const float* kl_row, const float* ce_row, float ce_weight, float* loss, uint32_t* status,
                           cudaStream_t s) {
  FinalizeParams f = {};
  f.tokens = tokens;
  f.doff = doff;
  f.target_argmax = target_argmax;
  f.R = R;
  f.N_d = N_d;
  f.V = V;
  f.accept_len = accept_len;
  f.bonus_token = bonus_token;
  f.accept_rate = accept_rate;
  f.kl_row = kl_row;
  f.ce_row = ce_row;
  f.ce_weight = ce_weight;
  f.loss = loss;
  f.status = status;
  return launch_finalize(f, s);
}

}  // namespace

namespace adaflash {
static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

cudaError_t raise_smem_limit(const void* fn, size_t bytes) {
  struct Limit {
    int device;
    const void* fn;
    size_t bytes;
  };
  static std::mutex mu;
  static std::vector<Limit> limits;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  Limit* found = nullptr;
  for (Limit& l : limits)
    if (l.device == device && l.fn == fn) found = &l;
  if (found != nullptr && found->bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (found != nullptr) found->bytes = bytes;
  else limits.push_back(Limit{device, fn, bytes});
  return cudaSuccess;
}
}  // namespace adaflash

extern "C" {

uint64_t adaflash_kernel_launches(void) { return adaflash::g_launches.load(std::memory_order_relaxed); }

const char* adaflash_status_string(adaflash_status s) {
  switch (s) {
    case ADAFLASH_OK: return "ADAFLASH_OK";
    case ADAFLASH_ERR_INVALID_ARG: return "ADAFLASH_ERR_INVALID_ARG";
    case ADAFLASH_ERR_UNSUPPORTED: return "ADAFLASH_ERR_UNSUPPORTED";
    case ADAFLASH_ERR_CUDA: return "ADAFLASH_ERR_CUDA";
    case ADAFLASH_ERR_TIMEOUT: return "ADAFLASH_ERR_TIMEOUT";
    case ADAFLASH_ERR_BAD_OFFSETS: return "ADAFLASH_ERR_BAD_OFFSETS";
    case ADAFLASH_ERR_BAD_TOKEN: return "ADAFLASH_ERR_BAD_TOKEN";
  }
  return "ADAFLASH_UNKNOWN_STATUS";
}

adaflash_status adaflash_verify_packed(const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
                                       const int32_t* draft_tokens, const int32_t* draft_offsets,
                                       int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
                                       int32_t* target_argmax, int32_t* accept_len, int32_t* bonus_token,
                                       float* accept_rate, uint32_t* d_status, void* stream) {
  ADAFLASH_TRY(check_shape(num_requests, num_draft_rows, vocab));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (num_requests == 0) return empty_batch(nullptr, false, d_status, s);
  ADAFLASH_TRY(check_logits(target_logits, t_dtype, ld_t, vocab));
  if (!int_ptr_ok(draft_tokens) || !int_ptr_ok(draft_offsets) || !int_ptr_ok(target_argmax) ||
      !int_ptr_ok(accept_len) || !int_ptr_ok(bonus_token) || !int_ptr_ok(accept_rate))
    return ADAFLASH_ERR_INVALID_ARG;
  if (d_status && !aligned(d_status, 4)) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());

  RowPassParams p = {};
  p.t = target_logits;
  p.ld_t = ld_t;
  p.doff = draft_offsets;
  p.R = num_requests;
  p.N_d = num_draft_rows;
  p.N_t = num_draft_rows + num_requests;
  p.V = vocab;
  p.mode = kModeVerify;
  // Target-only units read no draft row; the draft dtype only sizes the ring.
  const bool aligned = rows_16b(target_logits, ld_t, dtype_bytes(t_dtype));
  const int c = rowpass_one_round_cluster(1, t_dtype, aligned, vocab, p.N_t);
  p.cluster = c > 0 ? c : rowpass_cluster_size(vocab, p.N_t, num_sms());
  p.slice = rowpass_slice(vocab, p.cluster);
  p.clip_c = 1.0f;
  p.target_argmax = target_argmax;
  p.status = d_status;
  ADAFLASH_CUDA(launch_rowpass(p, 1, t_dtype, aligned, s));

  ADAFLASH_CUDA(finalize_after(draft_tokens, draft_offsets, target_argmax, num_requests, num_draft_rows, vocab,
                               accept_len, bonus_token, accept_rate, nullptr, nullptr, 0.0f, nullptr, d_status, s));
  return ADAFLASH_OK;
}

adaflash_status adaflash_opd_loss_fwd(const void* draft_logits, adaflash_dtype d_dtype, int64_t ld_d,
                                      const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
                                      const int32_t* draft_tokens, const int32_t* draft_offsets,
                                      int32_t num_requests, int32_t num_draft_rows, int32_t vocab, float clip_c,
                                      float ce_weight, int32_t* target_argmax, int32_t* accept_len,
                                      int32_t* bonus_token, float* accept_rate, float* kl_row, float* ce_row,
                                      float* row_stats, float* loss, uint32_t* d_status, void* stream) {
  ADAFLASH_TRY(check_shape(num_requests, num_draft_rows, vocab));
  if (!(clip_c > 0.0f) || !std::isfinite(ce_weight)) return ADAFLASH_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (num_requests == 0) return empty_batch(loss, true, d_status, s);
  ADAFLASH_TRY(check_logits(draft_logits, d_dtype, ld_d, vocab));
  ADAFLASH_TRY(check_logits(target_logits, t_dtype, ld_t, vocab));
  if (!int_ptr_ok(draft_tokens) || !int_ptr_ok(draft_offsets) || !int_ptr_ok(target_argmax) ||
      !int_ptr_ok(accept_len) || !int_ptr_ok(bonus_token) || !int_ptr_ok(accept_rate) || !int_ptr_ok(kl_row) ||
      !int_ptr_ok(ce_row) || !int_ptr_ok(row_stats) || !int_ptr_ok(loss))
    return ADAFLASH_ERR_INVALID_ARG;
  if (d_status && !aligned(d_status, 4)) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());

  RowPassParams p = {};
  p.z = draft_logits;
  p.t = target_logits;
  p.ld_z = ld_d;
  p.ld_t = ld_t;
  p.doff = draft_offsets;
  p.R = num_requests;
  p.N_d = num_draft_rows;
  p.N_t = num_draft_rows + num_requests;
  p.V = vocab;
  p.mode = kModeFwd;
  const bool aligned = rows_16b(draft_logits, ld_d, dtype_bytes(d_dtype)) &&
                       rows_16b(target_logits, ld_t, dtype_bytes(t_dtype));
  // all row units in one round of resident clusters where a cluster size allows it,
  // else enough CTAs to fill the GPU
  const int c = rowpass_one_round_cluster(d_dtype, t_dtype, aligned, vocab, p.N_d + p.R);
  p.cluster = c > 0 ? c : rowpass_cluster_size(vocab, p.N_d + p.R, num_sms());
  p.slice = rowpass_slice(vocab, p.cluster);
  p.clip_c = clip_c;
  p.target_argmax = target_argmax;
  p.kl_row = kl_row;
  p.ce_row = ce_row;
  p.row_stats = row_stats;
  p.status = d_status;
  ADAFLASH_CUDA(launch_rowpass(p, d_dtype, t_dtype, aligned, s));

  ADAFLASH_CUDA(finalize_after(draft_tokens, draft_offsets, target_argmax, num_requests, num_draft_rows, vocab,
                               accept_len, bonus_token, accept_rate, kl_row, ce_row, ce_weight, loss, d_status, s));
  return ADAFLASH_OK;
}

adaflash_status adaflash_opd_loss_bwd(const void* draft_logits, adaflash_dtype d_dtype, int64_t ld_d,
                                      const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
                                      const int32_t* draft_offsets, int32_t num_requests, int32_t num_draft_rows,
                                      int32_t vocab, float clip_c, float ce_weight, const int32_t* target_argmax,
                                      const float* row_stats, const float* grad_row, float grad_scale,
                                      float* grad_draft, int64_t ld_g, uint32_t* d_status, void* stream) {
  ADAFLASH_TRY(check_shape(num_requests, num_draft_rows, vocab));
  if (!(clip_c > 0.0f) || !std::isfinite(ce_weight) || !std::isfinite(grad_scale)) return ADAFLASH_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (num_requests == 0) return empty_batch(nullptr, false, d_status, s);
  ADAFLASH_TRY(check_logits(draft_logits, d_dtype, ld_d, vocab));
  ADAFLASH_TRY(check_logits(target_logits, t_dtype, ld_t, vocab));
  if (!int_ptr_ok(draft_offsets) || !int_ptr_ok(target_argmax) || !int_ptr_ok(row_stats) ||
      !int_ptr_ok(grad_draft) || ld_g < vocab)
    return ADAFLASH_ERR_INVALID_ARG;
  if (grad_row && !aligned(grad_row, 4)) return ADAFLASH_ERR_INVALID_ARG;
  if (d_status && !aligned(d_status, 4)) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());

  BwdParams p = {};
  p.z = draft_logits;
  p.t = target_logits;
  p.ld_z = ld_d;
  p.ld_t = ld_t;
  p.doff = draft_offsets;
  p.R = num_requests;
  p.N_d = num_draft_rows;
  p.N_t = num_draft_rows + num_requests;
  p.V = vocab;
  p.clip_c = clip_c;
  p.ce_weight = ce_weight;
  p.target_argmax = target_argmax;
  p.row_stats = row_stats;
  p.grad_row = grad_row;
  p.grad_scale = grad_scale;
  p.grad = grad_draft;
  p.ld_g = ld_g;
  p.chunks_per_row = (vocab + kBwdChunk - 1) / kBwdChunk;
  p.status = d_status;
  const bool aligned = rows_16b(draft_logits, ld_d, dtype_bytes(d_dtype)) &&
                       rows_16b(target_logits, ld_t, dtype_bytes(t_dtype)) && rows_16b(grad_draft, ld_g, 4);
  ADAFLASH_CUDA(launch_bwd(p, d_dtype, t_dtype, aligned, s));
  return ADAFLASH_OK;
}

adaflash_status adaflash_opd_loss_fwd_bwd(const void* draft_logits, adaflash_dtype d_dtype, int64_t ld_d,
                                          const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
                                          const int32_t* draft_tokens, const int32_t* draft_offsets,
                                          int32_t num_requests, int32_t num_draft_rows, int32_t vocab, float clip_c,
                                          float ce_weight, const float* grad_row, float grad_scale,
                                          int32_t* target_argmax, int32_t* accept_len, int32_t* bonus_token,
                                          float* accept_rate, float* kl_row, float* ce_row, float* row_stats,
                                          float* loss, float* grad_draft, int64_t ld_g, uint32_t* d_status,
                                          void* stream) {
  ADAFLASH_TRY(check_shape(num_requests, num_draft_rows, vocab));
  if (!(clip_c > 0.0f) || !std::isfinite(ce_weight) || !std::isfinite(grad_scale)) return ADAFLASH_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (num_requests == 0) return empty_batch(loss, true, d_status, s);
  ADAFLASH_TRY(check_logits(draft_logits, d_dtype, ld_d, vocab));
  ADAFLASH_TRY(check_logits(target_logits, t_dtype, ld_t, vocab));
  if (!int_ptr_ok(draft_tokens) || !int_ptr_ok(draft_offsets) || !int_ptr_ok(target_argmax) ||
      !int_ptr_ok(accept_len) || !int_ptr_ok(bonus_token) || !int_ptr_ok(accept_rate) || !int_ptr_ok(kl_row) ||
      !int_ptr_ok(ce_row) || !int_ptr_ok(row_stats) || !int_ptr_ok(loss) || !int_ptr_ok(grad_draft) || ld_g < vocab)
    return ADAFLASH_ERR_INVALID_ARG;
  if (grad_row && !aligned(grad_row, 4)) return ADAFLASH_ERR_INVALID_ARG;
  if (d_status && !aligned(d_status, 4)) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());

  RowPassParams p = {};
  p.z = draft_logits;
  p.t = target_logits;
  p.ld_z = ld_d;
  p.ld_t = ld_t;
  p.doff = draft_offsets;
  p.R = num_requests;
  p.N_d = num_draft_rows;
  p.N_t = num_draft_rows + num_requests;
  p.V = vocab;
  p.mode = kModeFwd;
  p.clip_c = clip_c;
  p.target_argmax = target_argmax;
  p.kl_row = kl_row;
  p.ce_row = ce_row;
  p.row_stats = row_stats;
  p.status = d_status;
  p.ce_weight = ce_weight;
  p.grad_row = grad_row;
  p.grad_scale = grad_scale;
  p.grad = grad_draft;
  p.ld_g = ld_g;
  // The on-chip fused kernel holds whole row pairs in shared memory (rows on the
  // 16-byte grid, a batch whose clusters all run at once with one CTA per SM);
  // otherwise the row pass with the gradient, which reads the logits from HBM once and
  // writes dz from a second pass over each slice served by L2 (any element-aligned
  // rows): 219.8 us on a 128-request batch at V = 151936, against 277.9 us for the
  // forward row pass and the backward kernel one after the other.
  const bool aligned16 = rows_16b(draft_logits, ld_d, dtype_bytes(d_dtype)) &&
                         rows_16b(target_logits, ld_t, dtype_bytes(t_dtype)) && rows_16b(grad_draft, ld_g, 4);
  const bool fused = aligned16 && num_draft_rows + num_requests <= fused_max_units(vocab, d_dtype, t_dtype, num_sms());
  if (fused) {
    ADAFLASH_CUDA(launch_fused(p, d_dtype, t_dtype, num_sms(), s));
  } else {
    const int row_bytes = vocab * (dtype_bytes(d_dtype) + dtype_bytes(t_dtype));
    int c = 0;
    if (static_cast<long long>(p.N_d) * row_bytes <= l2_bytes() * 3 / 4)
      c = rowpass_grad_one_round_cluster(d_dtype, t_dtype, aligned16, vocab, p.N_d);
    p.cluster = c > 0 ? c
                      : rowpass_grad_cluster_size(vocab, p.N_d + p.R, row_bytes, rowpass_grad_chunk(d_dtype, t_dtype),
                                                  num_sms(), l2_bytes());
    p.slice = rowpass_slice(vocab, p.cluster);
    ADAFLASH_CUDA(launch_rowpass_grad(p, d_dtype, t_dtype, aligned16, s));
  }

  ADAFLASH_CUDA(finalize_after(draft_tokens, draft_offsets, target_argmax, num_requests, num_draft_rows, vocab,
                               accept_len, bonus_token, accept_rate, kl_row, ce_row, ce_weight, loss, d_status, s));

  return ADAFLASH_OK;
}

// ---- LM-head path ----
namespace {
constexpr int kLmTileV = 256;  // vocabulary entries per tile of the head GEMM
constexpr int kLmTileM = 128;

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int64_t lm_ht_bytes(int64_t rows, int64_t H) { return round_up(rows * H * 2, 1024); }
int64_t lm_partial_bytes(int64_t rows, int64_t V) {
  return rows * ((V + kLmTileV - 1) / kLmTileV) * static_cast<int64_t>(sizeof(LmPartial));
}

adaflash_status check_bf16_rows(const void* p, int64_t ld, int32_t H) {
  if (!p || !aligned(p, 16) || ld < H || ld % 8 != 0) return ADAFLASH_ERR_INVALID_ARG;
  return ADAFLASH_OK;
}
}  // namespace

int64_t adaflash_lmhead_workspace_bytes(int32_t num_requests, int32_t num_draft_rows, int32_t vocab, int32_t hidden) {
  if (num_requests < 0 || num_draft_rows < 0 || vocab < 1 || hidden < 1) return -1;
  const int64_t rows = static_cast<int64_t>(num_requests) + num_draft_rows;
  return lm_ht_bytes(rows, hidden) + lm_partial_bytes(rows, vocab);
}

adaflash_status adaflash_lmhead_logits(const void* hidden_rows, int64_t ld_h, int32_t rows, const void* head,
                                       int64_t ld_w, int32_t vocab, int32_t hidden, float* logits, int64_t ld_out,
                                       uint32_t* d_status, void* stream) {
  if (rows < 0 || vocab < 1 || vocab > ADAFLASH_MAX_VOCAB || hidden < 64 || hidden % 64 != 0)
    return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_bf16_rows(hidden_rows, ld_h, hidden));
  ADAFLASH_TRY(check_bf16_rows(head, ld_w, hidden));
  if (!logits || !aligned(logits, 4) || ld_out < vocab) return ADAFLASH_ERR_INVALID_ARG;
  if (d_status && !aligned(d_status, 4)) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());
  if (rows == 0) return ADAFLASH_OK;
  LmHeadParams p = {};
  p.n_pair_tiles = 0;
  p.n_pair_rows = 0;
  p.n_t_rows = rows;
  p.V = vocab;
  p.H = hidden;
  p.n_vtiles = (vocab + kLmTileV - 1) / kLmTileV;
  p.mode = 1;
  p.out_t = logits;
  p.out_z = logits;
  p.ld_out = ld_out;
  p.status = d_status;
  const uint16_t* h = static_cast<const uint16_t*>(hidden_rows);
  const uint16_t* w = static_cast<const uint16_t*>(head);
  ADAFLASH_CUDA(launch_lm_gemm(h, ld_h, h, ld_h, w, ld_w, w, ld_w, p, static_cast<cudaStream_t>(stream)));
  return ADAFLASH_OK;
}

}  // extern "C"

namespace {
// Argument checks shared by the logit-free entry points (everything but the scratch).
adaflash_status check_lmhead_fwd_args(const void* draft_hidden, int64_t ld_hd, const void* target_hidden,
                                      int64_t ld_ht, const void* draft_head, int64_t ld_wd, const void* target_head,
                                      int64_t ld_wt, int32_t hidden, const int32_t* draft_tokens,
                                      const int32_t* draft_offsets, int32_t num_requests, int32_t num_draft_rows,
                                      int32_t vocab, float clip_c, float ce_weight, int32_t* target_argmax,
                                      int32_t* accept_len, int32_t* bonus_token, float* accept_rate, float* kl_row,
                                      float* ce_row, float* row_stats, float* loss, uint32_t* d_status) {
  ADAFLASH_TRY(check_shape(num_requests, num_draft_rows, vocab));
  if (hidden < 64 || hidden % 64 != 0) return ADAFLASH_ERR_INVALID_ARG;
  if (!(clip_c > 0.0f) || !std::isfinite(ce_weight)) return ADAFLASH_ERR_INVALID_ARG;
  if (num_requests == 0)  // an empty batch reads nothing: only the loss pointer matters
    return int_ptr_ok(loss) && (!d_status || aligned(d_status, 4)) ? ADAFLASH_OK : ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_bf16_rows(draft_hidden, ld_hd, hidden));
  ADAFLASH_TRY(check_bf16_rows(target_hidden, ld_ht, hidden));
  ADAFLASH_TRY(check_bf16_rows(draft_head, ld_wd, hidden));
  ADAFLASH_TRY(check_bf16_rows(target_head, ld_wt, hidden));
  if (!int_ptr_ok(draft_tokens) || !int_ptr_ok(draft_offsets) || !int_ptr_ok(target_argmax) ||
      !int_ptr_ok(accept_len) || !int_ptr_ok(bonus_token) || !int_ptr_ok(accept_rate) || !int_ptr_ok(kl_row) ||
      !int_ptr_ok(ce_row) || !int_ptr_ok(row_stats) || !int_ptr_ok(loss))
    return ADAFLASH_ERR_INVALID_ARG;
  if (d_status && !aligned(d_status, 4)) return ADAFLASH_ERR_INVALID_ARG;
  return ADAFLASH_OK;
}
}  // namespace

extern "C" {

adaflash_status adaflash_lmhead_opd_fwd(const void* draft_hidden, int64_t ld_hd, const void* target_hidden,
                                        int64_t ld_ht, const void* draft_head, int64_t ld_wd, const void* target_head,
                                        int64_t ld_wt, int32_t hidden, const int32_t* draft_tokens,
                                        const int32_t* draft_offsets, int32_t num_requests, int32_t num_draft_rows,
                                        int32_t vocab, float clip_c, float ce_weight, void* workspace,
                                        int64_t workspace_bytes, int32_t* target_argmax, int32_t* accept_len,
                                        int32_t* bonus_token, float* accept_rate, float* kl_row, float* ce_row,
                                        float* row_stats, float* loss, uint32_t* d_status, void* stream) {
  ADAFLASH_TRY(check_lmhead_fwd_args(draft_hidden, ld_hd, target_hidden, ld_ht, draft_head, ld_wd, target_head, ld_wt,
                                     hidden, draft_tokens, draft_offsets, num_requests, num_draft_rows, vocab, clip_c,
                                     ce_weight, target_argmax, accept_len, bonus_token, accept_rate, kl_row, ce_row,
                                     row_stats, loss, d_status));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (num_requests == 0) return empty_batch(loss, true, d_status, s);
  const int64_t need = adaflash_lmhead_workspace_bytes(num_requests, num_draft_rows, vocab, hidden);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());
  const int32_t Nt = num_draft_rows + num_requests;
  uint16_t* ht_pairs = static_cast<uint16_t*>(workspace);
  LmPartial* partials =
      reinterpret_cast<LmPartial*>(static_cast<uint8_t*>(workspace) + lm_ht_bytes(Nt, hidden));
  ADAFLASH_CUDA(launch_lm_gather(static_cast<const uint16_t*>(target_hidden), ld_ht, draft_offsets, num_requests,
                                 num_draft_rows, hidden, ht_pairs, d_status, s));
  LmHeadParams p = {};
  p.n_pair_tiles = (num_draft_rows + kLmTileM - 1) / kLmTileM;
  p.n_pair_rows = num_draft_rows;
  p.n_t_rows = Nt;
  p.V = vocab;
  p.H = hidden;
  p.n_vtiles = (vocab + kLmTileV - 1) / kLmTileV;
  p.mode = 0;
  p.partials = partials;
  p.status = d_status;
  ADAFLASH_CUDA(launch_lm_gemm(static_cast<const uint16_t*>(draft_hidden), ld_hd, ht_pairs, hidden,
                               static_cast<const uint16_t*>(draft_head), ld_wd,
                               static_cast<const uint16_t*>(target_head), ld_wt, p, s));
  LmCombineParams c = {};
  c.hd = static_cast<const uint16_t*>(draft_hidden);
  c.ht = ht_pairs;
  c.wd = static_cast<const uint16_t*>(draft_head);
  c.wt = static_cast<const uint16_t*>(target_head);
  c.ld_hd = ld_hd;
  c.ld_wd = ld_wd;
  c.ld_wt = ld_wt;
  c.doff = draft_offsets;
  c.R = num_requests;
  c.N_d = num_draft_rows;
  c.V = vocab;
  c.H = hidden;
  c.n_vtiles = p.n_vtiles;
  c.clip_c = clip_c;
  c.partials = partials;
  c.target_argmax = target_argmax;
  c.kl_row = kl_row;
  c.ce_row = ce_row;
  c.row_stats = row_stats;
  c.status = d_status;
  ADAFLASH_CUDA(launch_lm_combine(c, s));

  ADAFLASH_CUDA(finalize_after(draft_tokens, draft_offsets, target_argmax, num_requests, num_draft_rows, vocab,
                               accept_len, bonus_token, accept_rate, kl_row, ce_row, ce_weight, loss, d_status, s));
  return ADAFLASH_OK;
}

adaflash_status adaflash_lmhead_opd_fwd_static(const void* draft_hidden, int64_t ld_hd, const void* target_hidden,
                                               int64_t ld_ht, const void* draft_head, int64_t ld_wd,
                                               const void* target_head, int64_t ld_wt, int32_t hidden,
                                               const int32_t* draft_tokens, const int32_t* draft_offsets,
                                               int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
                                               float clip_c, float ce_weight, int32_t* target_argmax,
                                               int32_t* accept_len, int32_t* bonus_token, float* accept_rate,
                                               float* kl_row, float* ce_row, float* row_stats, float* loss,
                                               uint32_t* d_status, void* stream) {
  // the same argument checks as the workspace entry point, then the array's size
  ADAFLASH_TRY(check_lmhead_fwd_args(draft_hidden, ld_hd, target_hidden, ld_ht, draft_head, ld_wd, target_head, ld_wt,
                                     hidden, draft_tokens, draft_offsets, num_requests, num_draft_rows, vocab, clip_c,
                                     ce_weight, target_argmax, accept_len, bonus_token, accept_rate, kl_row, ce_row,
                                     row_stats, loss, d_status));
  if (num_requests == 0) return empty_batch(loss, true, d_status, static_cast<cudaStream_t>(stream));
  const int64_t need = adaflash_lmhead_workspace_bytes(num_requests, num_draft_rows, vocab, hidden);
  if (need < 0) return ADAFLASH_ERR_INVALID_ARG;
  if (need > ADAFLASH_LMHEAD_STATIC_SCRATCH_BYTES) return ADAFLASH_ERR_UNSUPPORTED;
  ADAFLASH_TRY(check_device());
  void* scratch = nullptr;
  int64_t bytes = 0;
  ADAFLASH_CUDA(lm_static_scratch(&scratch, &bytes));
  return adaflash_lmhead_opd_fwd(draft_hidden, ld_hd, target_hidden, ld_ht, draft_head, ld_wd, target_head, ld_wt,
                                 hidden, draft_tokens, draft_offsets, num_requests, num_draft_rows, vocab, clip_c,
                                 ce_weight, scratch, bytes, target_argmax, accept_len, bonus_token, accept_rate,
                                 kl_row, ce_row, row_stats, loss, d_status, stream);
}

adaflash_status adaflash_verify_sampled(const void* draft_logits, adaflash_dtype d_dtype, int64_t ld_d,
                                        const void* target_logits, adaflash_dtype t_dtype, int64_t ld_t,
                                        const int32_t* draft_tokens, const int32_t* draft_offsets,
                                        int32_t num_requests, int32_t num_draft_rows, int32_t vocab,
                                        float temperature, const float* u_accept, const float* u_sample,
                                        float* row_lse, int32_t* accept_len, int32_t* next_token,
                                        float* accept_rate, uint32_t* d_status, void* stream) {
  ADAFLASH_TRY(check_shape(num_requests, num_draft_rows, vocab));
  if (!(temperature > 0.0f) || !std::isfinite(temperature) || !std::isfinite(1.0f / temperature))
    return ADAFLASH_ERR_INVALID_ARG;
  if (num_requests == 0) return empty_batch(nullptr, false, d_status, static_cast<cudaStream_t>(stream));
  ADAFLASH_TRY(check_logits(draft_logits, d_dtype, ld_d, vocab));
  ADAFLASH_TRY(check_logits(target_logits, t_dtype, ld_t, vocab));
  if (!int_ptr_ok(draft_tokens) || !int_ptr_ok(draft_offsets) || !int_ptr_ok(u_accept) ||
      !int_ptr_ok(u_sample) || !int_ptr_ok(row_lse) || !int_ptr_ok(accept_len) || !int_ptr_ok(next_token) ||
      !int_ptr_ok(accept_rate))
    return ADAFLASH_ERR_INVALID_ARG;
  if (d_status && !aligned(d_status, 4)) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());

  SampledParams p = {};
  p.z = draft_logits;
  p.t = target_logits;
  p.ld_z = ld_d;
  p.ld_t = ld_t;
  p.doff = draft_offsets;
  p.R = num_requests;
  p.N_d = num_draft_rows;
  p.N_t = num_draft_rows + num_requests;
  p.V = vocab;
  p.inv_t = 1.0f / temperature;
  p.tokens = draft_tokens;
  p.u_accept = u_accept;
  p.u_sample = u_sample;
  p.row_lse = row_lse;
  p.accept_len = accept_len;
  p.next_token = next_token;
  p.accept_rate = accept_rate;
  p.status = d_status;
  ADAFLASH_CUDA(launch_sampled(p, d_dtype, t_dtype, num_sms(), static_cast<cudaStream_t>(stream)));
  return ADAFLASH_OK;
}

adaflash_status adaflash_selftest_bounded_wait(uint32_t* d_status, int32_t limit_us, void* stream) {
  if (!int_ptr_ok(d_status) || limit_us < 1 || limit_us > 1000000) return ADAFLASH_ERR_INVALID_ARG;
  ADAFLASH_TRY(check_device());
  ADAFLASH_CUDA(launch_selftest_wait(d_status, limit_us, static_cast<cudaStream_t>(stream)));
  return ADAFLASH_OK;
}

}  // extern "C"
