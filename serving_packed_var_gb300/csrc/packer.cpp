// packer.cpp -- host-side variable-length request packing with an EMA capacity estimate.
//
// The AdaFlash article ("AdaFlash: Adaptive Speculative Decoding with Online
// Self-Improvement for High-Concurrency LLM Inference", "Infrastructure: Async
// Training & Variable-Length Batching", "Variable-length request packing") packs
// requests of different predicted verification lengths into compact batches and
// sizes the next round from an exponential moving average, to use the GPU well
// without running out of memory.  Reading taken here:
//
//   a request of predicted draft length k occupies 2k + 1 logit rows in a round
//   (k draft rows and k + 1 target rows of the packed layout);
//   the estimate e of rows per request follows e <- alpha * x + (1 - alpha) * e,
//   x = a round's rows / its requests;
//   a round takes capacity = max(1, floor(row_budget / e)) requests from the front
//   of the queue, gives back the last ones while their rows exceed row_budget, and
//   packs the rest back to back (draft_offsets = exclusive prefix sum of their k).
//
// The EMA is float64 with the operations in that order (this file is compiled
// without floating-point contraction), so the decisions match a float64 restatement.
#include <cmath>
#include <cstdint>
#include <new>

#include "../../include/adaflash.h"

struct adaflash_packer {
  int32_t row_budget;
  double alpha;
  double e;  // rows per request
};

namespace {
constexpr int32_t kMaxK = ADAFLASH_MAX_K;
constexpr int32_t kMaxRows = 2 * kMaxK + 1;
inline int32_t rows_of(int32_t k) { return 2 * k + 1; }
}  // namespace

extern "C" {

adaflash_status adaflash_packer_create(int32_t row_budget, double alpha, double initial_rows_per_request,
                                       adaflash_packer** out) {
  if (!out) return ADAFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  if (row_budget < kMaxRows) return ADAFLASH_ERR_INVALID_ARG;
  if (!(alpha > 0.0) || !(alpha <= 1.0)) return ADAFLASH_ERR_INVALID_ARG;
  if (!(initial_rows_per_request > 0.0) || !std::isfinite(initial_rows_per_request)) return ADAFLASH_ERR_INVALID_ARG;
  adaflash_packer* p = new (std::nothrow) adaflash_packer;
  if (!p) return ADAFLASH_ERR_INVALID_ARG;
  p->row_budget = row_budget;
  p->alpha = alpha;
  p->e = initial_rows_per_request;
  *out = p;
  return ADAFLASH_OK;
}

adaflash_status adaflash_packer_destroy(adaflash_packer* p) {
  delete p;
  return ADAFLASH_OK;
}

adaflash_status adaflash_packer_plan(const adaflash_packer* p, const int32_t* queue_k, int32_t n_queue,
                                     int32_t* draft_offsets, int32_t* num_admitted, int32_t* capacity,
                                     int32_t* rows) {
  if (!p || n_queue < 0 || (n_queue > 0 && !queue_k) || !draft_offsets || !num_admitted || !capacity || !rows)
    return ADAFLASH_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_queue; ++i)
    if (queue_k[i] < 1 || queue_k[i] > kMaxK) return ADAFLASH_ERR_INVALID_ARG;
  int32_t cap = 0;
  if (n_queue > 0) {
    const double c = std::floor(static_cast<double>(p->row_budget) / p->e);
    cap = c < 1.0 ? 1 : (c >= static_cast<double>(n_queue) ? n_queue : static_cast<int32_t>(c));
  }
  int32_t admitted = cap;
  int64_t total = 0;
  for (int32_t i = 0; i < admitted; ++i) total += rows_of(queue_k[i]);
  while (admitted > 0 && total > p->row_budget) {
    --admitted;
    total -= rows_of(queue_k[admitted]);
  }
  draft_offsets[0] = 0;
  for (int32_t i = 0; i < admitted; ++i) draft_offsets[i + 1] = draft_offsets[i] + queue_k[i];
  *num_admitted = admitted;
  *capacity = cap;
  *rows = static_cast<int32_t>(total);
  return ADAFLASH_OK;
}

adaflash_status adaflash_packer_observe(adaflash_packer* p, int32_t rows, int32_t requests) {
  if (!p || rows < 0 || requests < 0) return ADAFLASH_ERR_INVALID_ARG;
  if (requests == 0) return ADAFLASH_OK;
  const double x = static_cast<double>(rows) / static_cast<double>(requests);
  const double a = p->alpha * x;
  const double b = (1.0 - p->alpha) * p->e;
  p->e = a + b;
  return ADAFLASH_OK;
}

adaflash_status adaflash_packer_estimate(const adaflash_packer* p, double* rows_per_request) {
  if (!p || !rows_per_request) return ADAFLASH_ERR_INVALID_ARG;
  *rows_per_request = p->e;
  return ADAFLASH_OK;
}

}  // extern "C"
