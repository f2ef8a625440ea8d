// opd_ref.cpp -- the CPU oracle of the packed verify + OPD-loss pass in plain C++.
//
// TEST INFRASTRUCTURE ONLY.  Loaded by tests/, __graft_entry__.smoke() and the
// CPU-baseline leg of bench.py through oracle/cpp.py; the CUDA library never links,
// includes or calls it, and it includes nothing of the CUDA sources.
//
// Everything is float64 and written as the plain definitions, one vocabulary entry
// at a time, left to right, with no blocking, online rescaling or fusion beyond what
// a definition states.  Inputs are the stored logits (float32, or bfloat16 bit
// patterns) widened exactly to double.
//
// Sources: "the AdaFlash article" is the page "AdaFlash: Adaptive Speculative
// Decoding with Online Self-Improvement for High-Concurrency LLM Inference"; "the
// AdaFlash README" is the page "AdaFlash: Adaptive Speculative Decoding via
// On-Policy Distilled Diffusion Drafters".  Readings where the pages leave a step
// open are the same as the Python oracle's (oracle/opd.py): greedy acceptance with
// the lowest index winning argmax ties, rate = L / k_i rounded once to float32, an
// upper clip min(p r, c) per vocabulary term, the hard-label weight beta and the
// mean over all draft rows, and a gradient that treats the target as a constant
// and passes through a term sitting exactly at the bound.
//
// Pinned by tests/test_oracle_cpp.py: element-by-element agreement with the Python
// oracle (itself pinned by brute force, closed forms and finite differences), and
// its own brute-force, closed-form and finite-difference checks.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// One stored logit widened to double: float32 as is, bfloat16 as the float32 whose
// upper half is the stored pattern (exact).
double widen(const void* row, int is_bf16, int64_t v) {
  if (is_bf16) {
    const uint16_t b = static_cast<const uint16_t*>(row)[v];
    const uint32_t w = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &w, sizeof f);
    return static_cast<double>(f);
  }
  return static_cast<double>(static_cast<const float*>(row)[v]);
}

void widen_row(const void* row, int is_bf16, int V, double* out) {
  for (int v = 0; v < V; ++v) out[v] = widen(row, is_bf16, v);
}

// log sum_v exp(x_v) in the max-shifted form m + log sum_v exp(x_v - m): the
// normaliser of the softmaxes p = softmax(z), q = softmax(t) of the AdaFlash
// article, "On-Policy Distillation (OPD) for Domain Adaptation".
double log_sum_exp(const double* x, int V) {
  double m = x[0];
  for (int v = 1; v < V; ++v) m = x[v] > m ? x[v] : m;
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += std::exp(x[v] - m);
  return m + std::log(s);
}

// The target's greedy choice: the smallest index holding the row maximum (AdaFlash
// article, opening section: the target verifies the drafted tokens).
int first_argmax(const double* x, int V) {
  int best = 0;
  for (int v = 1; v < V; ++v)
    if (x[v] > x[best]) best = v;
  return best;
}

struct RowResult {
  double kl, ce, loss_row, lse_z, lse_t, S, S_l1;
  int argmax, n_clipped;
};

// One (draft row z, target row t) pair, following the definitions in order:
//   log p = z - LSE(z), log q = t - LSE(t), p = exp(log p), r = log p - log q,
//   KL_clip = sum_v min(p_v r_v, c)              ("Reverse KL + Top-1 hard labels",
//                                                  "Per-vocabulary divergence clipping"),
//   CE = -log p_a, a = first argmax of t         ("Top-1 hard labels"),
//   loss_row = KL_clip + beta * CE               (README, "Released Checkpoint": a mixture),
//   S = sum_v [p_v r_v <= c] p_v (r_v + 1)       (the gradient's row constant),
//   S_l1 = sum_v [p_v r_v <= c] p_v |r_v + 1|    (the size of S's summands).
RowResult row_forward(const double* z, const double* t, int V, double c, double beta) {
  RowResult o{};
  o.lse_z = log_sum_exp(z, V);
  o.lse_t = log_sum_exp(t, V);
  double kl = 0.0, S = 0.0, S_l1 = 0.0;
  int nclip = 0;
  for (int v = 0; v < V; ++v) {
    const double log_p = z[v] - o.lse_z;
    const double log_q = t[v] - o.lse_t;
    const double p = std::exp(log_p);
    const double r = log_p - log_q;
    const double term = p * r;
    kl += term < c ? term : c;
    if (term <= c) {
      S += p * (r + 1.0);
      S_l1 += p * std::fabs(r + 1.0);
    } else {
      ++nclip;
    }
  }
  o.kl = kl;
  o.S = S;
  o.S_l1 = S_l1;
  o.n_clipped = nclip;
  o.argmax = first_argmax(t, V);
  o.ce = -(z[o.argmax] - o.lse_z);
  o.loss_row = o.kl + beta * o.ce;
  return o;
}

// d(g * loss_row)/dz_u = g [p_u (m_u (r_u + 1) - S) + beta (p_u - [u == a])], with
// m_u = [p_u r_u <= c]; the target and its argmax are constants (the target model
// never changes: AdaFlash article, "Decoupled training/inference").
void row_grad(const double* z, const double* t, int V, double c, double beta, double g, double* dz) {
  const double lse_z = log_sum_exp(z, V);
  const double lse_t = log_sum_exp(t, V);
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    const double log_p = z[v] - lse_z;
    const double p = std::exp(log_p);
    const double r = log_p - (t[v] - lse_t);
    if (p * r <= c) S += p * (r + 1.0);
  }
  const int a = first_argmax(t, V);
  for (int v = 0; v < V; ++v) {
    const double log_p = z[v] - lse_z;
    const double p = std::exp(log_p);
    const double r = log_p - (t[v] - lse_t);
    const double m = (p * r <= c) ? 1.0 : 0.0;
    const double onehot = (v == a) ? 1.0 : 0.0;
    dz[v] = g * (p * (m * (r + 1.0) - S) + beta * (p - onehot));
  }
}

// Run f(item) for item in [0, n) on `threads` std::threads (a shared counter).
template <class F>
void parallel_for(int64_t n, int threads, F f) {
  if (threads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  const int nt = static_cast<int>(std::min<int64_t>(threads, n));
  for (int k = 0; k < nt; ++k)
    pool.emplace_back([&] {
      for (int64_t i = next.fetch_add(1); i < n; i = next.fetch_add(1)) f(i);
    });
  for (auto& th : pool) th.join();
}

// Request owning draft row d: the largest i with doff[i] <= d.
int request_of(const int32_t* doff, int R, int d) {
  int i = 0;
  while (i + 1 < R && doff[i + 1] <= d) ++i;
  return i;
}

}  // namespace

extern "C" {

// One pair of float64 rows.  out: kl, ce, loss_row, lse_z, lse_t, S, S_l1;
// ints: argmax, n_clipped.
void oracle_row_forward(const double* z, const double* t, int V, double c, double beta, double* out, int* ints) {
  const RowResult r = row_forward(z, t, V, c, beta);
  out[0] = r.kl; out[1] = r.ce; out[2] = r.loss_row; out[3] = r.lse_z; out[4] = r.lse_t;
  out[5] = r.S; out[6] = r.S_l1;
  ints[0] = r.argmax;
  ints[1] = r.n_clipped;
}

void oracle_row_grad(const double* z, const double* t, int V, double c, double beta, double g, double* dz) {
  row_grad(z, t, V, c, beta, g, dz);
}

// Greedy verification of a packed batch (AdaFlash article, "Variable-length request
// packing": request i owns draft rows doff[i] .. doff[i+1]-1 and target rows
// doff[i]+i .. doff[i+1]+i; draft row doff[i]+j pairs with target row doff[i]+i+j,
// and target row doff[i+1]+i is the bonus position).  Every target row's first
// argmax, then per request the accepted prefix L_i (the first j whose token differs
// from the target's choice, k_i if none), the bonus token (the target's choice right
// after the prefix) and the rate L_i / k_i rounded once to float32 (the length
// head's free label: "2. Adaptive Length Head for Token-Level Variance").
void oracle_verify_packed(const void* target, int t_bf16, int64_t ld_t, const int32_t* tokens, const int32_t* doff,
                          int R, int V, int threads, int32_t* target_argmax, int32_t* accept_len,
                          int32_t* bonus_token, float* accept_rate) {
  const int64_t Nt = static_cast<int64_t>(doff[R]) + R;
  const int ew = t_bf16 ? 2 : 4;
  parallel_for(Nt, threads, [&](int64_t s) {
    std::vector<double> t(V);
    widen_row(static_cast<const uint8_t*>(target) + s * ld_t * ew, t_bf16, V, t.data());
    target_argmax[s] = first_argmax(t.data(), V);
  });
  for (int i = 0; i < R; ++i) {
    const int d0 = doff[i], k = doff[i + 1] - doff[i];
    int L = k;
    for (int j = 0; j < k; ++j)
      if (tokens[d0 + j] != target_argmax[d0 + i + j]) {
        L = j;
        break;
      }
    accept_len[i] = L;
    bonus_token[i] = target_argmax[d0 + i + L];
    accept_rate[i] = static_cast<float>(L) / static_cast<float>(k);
  }
}

// The forward (and, when grad is non-NULL, the gradient) of the listed draft rows of
// a packed batch.  rows[n] lists draft rows (NULL: every row 0 .. N_d-1, n = N_d).
// Per listed row (index n in the list): stats[8 n + 0..6] = kl, ce, loss_row, lse_z,
// lse_t, S, S_l1 and ints[2 n + 0..1] = argmax of the paired target row, n_clipped;
// grad[n V + v] = d(g_r loss_row)/dz_v with g_r = grad_row[r] (grad_row non-NULL) or
// grad_scale.  When every row is listed, *loss = (1 / N_d) sum_r loss_row_r, summed
// in row order.
void oracle_opd_rows(const void* draft, int d_bf16, int64_t ld_d, const void* target, int t_bf16, int64_t ld_t,
                     const int32_t* doff, int R, int V, double c, double beta, const int32_t* rows, int64_t n,
                     const double* grad_row, double grad_scale, int threads, double* stats, int32_t* ints,
                     double* grad, double* loss) {
  const int dw = d_bf16 ? 2 : 4, tw = t_bf16 ? 2 : 4;
  parallel_for(n, threads, [&](int64_t k) {
    const int d = rows ? rows[k] : static_cast<int>(k);
    const int i = request_of(doff, R, d);
    const int64_t s = static_cast<int64_t>(d) + i;
    std::vector<double> z(V), t(V);
    widen_row(static_cast<const uint8_t*>(draft) + static_cast<int64_t>(d) * ld_d * dw, d_bf16, V, z.data());
    widen_row(static_cast<const uint8_t*>(target) + s * ld_t * tw, t_bf16, V, t.data());
    const RowResult r = row_forward(z.data(), t.data(), V, c, beta);
    double* st = stats + 8 * k;
    st[0] = r.kl; st[1] = r.ce; st[2] = r.loss_row; st[3] = r.lse_z; st[4] = r.lse_t; st[5] = r.S; st[6] = r.S_l1;
    st[7] = 0.0;
    ints[2 * k] = r.argmax;
    ints[2 * k + 1] = r.n_clipped;
    if (grad) {
      const double g = grad_row ? grad_row[d] : grad_scale;
      row_grad(z.data(), t.data(), V, c, beta, g, grad + k * static_cast<int64_t>(V));
    }
  });
  if (loss && !rows) {
    double sum = 0.0;
    for (int64_t k = 0; k < n; ++k) sum += stats[8 * k + 2];
    *loss = n ? sum / static_cast<double>(n) : 0.0;
  }
}

}  // extern "C"
