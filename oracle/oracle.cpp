// Oracle for the top-p log-probability / entropy path and the GRPO/DAPO loss.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
// call this file; only the tests, the smoke check and the benchmark's CPU
// baseline leg use it.  It shares no code with the CUDA library.
//
// Plain fp64 on the host: full softmax, a full sort of the vocabulary, an
// explicit nucleus, compensated (Neumaier) sums.  No blocking, fusion or
// reordering beyond what the definitions below state.  Rows are spread over
// std::thread workers (static partition); every row is computed on its own,
// so the thread count never changes a result.
//
// Sources (the pages give semantics, not formulas):
//  * RL-Kernel, "Qwen3-8B VIME train-rollout consistency", section "ROCm
//    MI300X and gfx942": temperature finite and positive, top-p in (0,1], the
//    complete retained top-p set with no support cap, top-k and temperature 0
//    rejected; top-p < 1 scored by the sparse logp/monitoring-entropy fusion
//    over the retained support, top-p = 1 by the full-vocabulary scorer.
//  * RL-Kernel, "ROCm sparse performance" notes: temperature, softmax, sort and
//    top-p thresholding keep the sampler's native semantics; GRPO uses
//    standard-deviation normalisation; KL coefficient 0.01.
//  * LumenRL README, section "Rollout Correction": TIS clips large
//    importance ratios.
//  * prime-rl v0.10.0 release notes, section "1. Trainer Performance": the
//    loss is chunked so full logits need not exist at once (LM-head rows).
// Readings taken where the pages are silent: keep a token while the mass
// ranked strictly ahead of it is below top_p (so at least one is kept); equal
// logits are kept lower id first, -0 equal to +0; advantages use the n-1
// standard deviation plus 1e-6; the KL term is k3 = e^d - d - 1 with
// d = ref - new; clip bounds and the TIS cap are arguments; the loss is the
// token mean over the batch (or the mean of per-sequence token means).
//
// Parity pins: brute force on V = 8, closed forms (uniform, one-hot, two-level
// logits), top_p = 1 against a library log-softmax, invariants, hand-worked
// loss values and finite-difference gradients (tests/test_oracle_pins.py).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <thread>
#include <vector>

namespace {

const double kInf = std::numeric_limits<double>::infinity();
const double kNaN = std::numeric_limits<double>::quiet_NaN();

// Neumaier's compensated summation (an improved Kahan sum).
struct NeumaierSum {
  double s = 0.0, c = 0.0;
  void add(double x) {
    double t = s + x;
    if (std::fabs(s) >= std::fabs(x)) c += (s - t) + x;
    else c += (x - t) + s;
    s = t;
  }
  double value() const { return s + c; }
};

// bf16 is the upper half of an IEEE binary32; widening is exact.
double bf16_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

double load_logit(const void* logits, int dtype, int64_t row, int64_t ld, int64_t i) {
  if (dtype == 0) return bf16_to_double(static_cast<const uint16_t*>(logits)[row * ld + i]);
  return static_cast<double>(static_cast<const float*>(logits)[row * ld + i]);
}

template <class F>
void parallel_rows(int64_t n, int nthreads, F fn) {
  if (nthreads < 1) nthreads = 1;
  if (n < nthreads) nthreads = static_cast<int>(n > 0 ? n : 1);
  if (nthreads == 1) {
    for (int64_t r = 0; r < n; ++r) fn(r);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t) {
    int64_t lo = n * t / nthreads, hi = n * (t + 1) / nthreads;
    pool.emplace_back([lo, hi, &fn] { for (int64_t r = lo; r < hi; ++r) fn(r); });
  }
  for (auto& th : pool) th.join();
}

// Result of scoring one row.
struct RowResult {
  double logprob, entropy, gap;
  int64_t k;
};

// The logits path for one row of widened logits z[0..V).
//  1. x_i = z_i / T (T = the float temperature widened to double).
//  2. m = max x_i, w_i = exp(x_i - m), Z = sum w_i, p_i = w_i / Z.
//  3. pi = the vocabulary sorted by (z descending, id ascending); -0 == +0.
//  4. k* = V if top_p >= 1, else the least k with C_k = sum_{j<=k} p_pi(j) >= top_p
//     (V if rounding leaves no such k).
//  5. S = pi(1..k*), Z_S = sum_S w_i.
//  6. logprob(y) = (x_y - m) - ln Z_S if y in S, else -inf.
//  7. H = -sum_S q_i ln q_i with q_i = w_i / Z_S and 0 ln 0 = 0.
//  8. gap = min(|top_p - C_{k*-1}|, |C_{k*} - top_p|), +inf when top_p >= 1.
// force_k > 0 evaluates steps 5-7 at that k instead of k* (rows whose gap is
// too small for the nucleus to be unique).
// grad (optional, V entries): dL/dz for L = glp logprob + gh H with S held
// fixed (S moves only where a logit crosses the boundary, so almost everywhere
// it is locally constant):
//  9. grad_i = 0 for i outside S; for i in S, with q_i = w_i / Z_S,
//     grad_i = glp [y in S] ([i = y] - q_i) / T - gh q_i (ln q_i + H) / T.
// A row with no distribution gets NaN in every entry.
RowResult score_row(const std::vector<double>& z, int64_t y, double T, double p, int64_t force_k,
                    double glp = 0.0, double gh = 0.0, double* grad = nullptr) {
  const int64_t V = static_cast<int64_t>(z.size());
  RowResult r{kNaN, kNaN, kNaN, 0};
  bool bad = y < 0 || y >= V;         // selected id outside the vocabulary
  for (double v : z)
    if (!std::isfinite(v)) bad = true;  // non-finite logit: no distribution
  if (bad) {
    if (grad) std::fill(grad, grad + V, kNaN);
    return r;
  }

  std::vector<double> x(V), w(V);
  double m = -kInf;
  for (int64_t i = 0; i < V; ++i) {
    x[i] = z[i] / T;
    m = std::max(m, x[i]);
  }
  NeumaierSum zsum;
  for (int64_t i = 0; i < V; ++i) {
    w[i] = std::exp(x[i] - m);
    zsum.add(w[i]);
  }
  const double Z = zsum.value();

  std::vector<int64_t> order(V);
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
    if (z[a] != z[b]) return z[a] > z[b];  // -0.0 == +0.0 compares equal
    return a < b;
  });

  int64_t k = V;
  double c_prev = 0.0, c_at = 1.0;
  {
    NeumaierSum pre;
    double last = 0.0;
    bool found = false;
    for (int64_t j = 0; j < V; ++j) {
      pre.add(w[order[j]]);
      double c = pre.value() / Z;
      if (p < 1.0 && !found && c >= p) {
        k = j + 1;
        c_prev = last;
        c_at = c;
        found = true;
      }
      last = c;
    }
    if (p < 1.0 && !found) {  // rounding left the total below top_p
      k = V;
      c_at = last;
      NeumaierSum pre2;
      for (int64_t j = 0; j + 1 < V; ++j) pre2.add(w[order[j]]);
      c_prev = pre2.value() / Z;
    }
  }
  r.k = k;
  r.gap = (p >= 1.0) ? kInf : std::min(std::fabs(p - c_prev), std::fabs(c_at - p));

  const int64_t keff = force_k > 0 ? std::min(force_k, V) : k;
  std::vector<char> member(V, 0);
  NeumaierSum zs;
  for (int64_t j = 0; j < keff; ++j) {
    member[order[j]] = 1;
    zs.add(w[order[j]]);
  }
  const double ZS = zs.value();
  r.logprob = member[y] ? (x[y] - m) - std::log(ZS) : -kInf;

  NeumaierSum h;
  for (int64_t j = 0; j < keff; ++j) {
    double q = w[order[j]] / ZS;
    if (q > 0.0) h.add(-q * std::log(q));
  }
  r.entropy = h.value();
  if (grad) {
    const double H = r.entropy;
    for (int64_t i = 0; i < V; ++i) {
      if (!member[i]) {
        grad[i] = 0.0;
        continue;
      }
      const double q = w[i] / ZS;
      const double dlp = member[y] ? ((i == y ? 1.0 : 0.0) - q) / T : 0.0;
      const double lq = q > 0.0 ? std::log(q) : 0.0;   // q ln q -> 0 as q -> 0
      grad[i] = glp * dlp - gh * q * (lq + H) / T;
    }
  }
  return r;
}

std::vector<double> widen_row(const void* logits, int dtype, int64_t row, int64_t V, int64_t ld) {
  std::vector<double> z(V);
  for (int64_t i = 0; i < V; ++i) z[i] = load_logit(logits, dtype, row, ld, i);
  return z;
}

}  // namespace

extern "C" {

int oracle_version(void) { return 1; }

// Logits path over T rows.  logits: bf16 (dtype 0) or fp32 (dtype 1), row
// stride ld elements.  Outputs per row: logprob, entropy, k*, gap (any may be
// NULL).  force_k: NULL, or per-row k to evaluate at (<= 0 means k*).
int oracle_logprob_entropy(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld,
                           const int32_t* ids, float temperature, float top_p,
                           const int64_t* force_k, double* out_logprob, double* out_entropy,
                           int64_t* out_k, double* out_gap, int nthreads) {
  if (!logits || !ids || T < 0 || V < 1 || ld < V || (dtype != 0 && dtype != 1)) return 1;
  const double Td = static_cast<double>(temperature), pd = static_cast<double>(top_p);
  parallel_rows(T, nthreads, [&](int64_t row) {
    std::vector<double> z = widen_row(logits, dtype, row, V, ld);
    RowResult r = score_row(z, ids[row], Td, pd, force_k ? force_k[row] : 0);
    if (out_logprob) out_logprob[row] = r.logprob;
    if (out_entropy) out_entropy[row] = r.entropy;
    if (out_k) out_k[row] = r.k;
    if (out_gap) out_gap[row] = r.gap;
  });
  return 0;
}

// Gradient of the logits path (steps 1-9 of score_row): out_grad[T, V] (fp64,
// dense, row stride V) = dL/dz for L = sum_t g_lp[t] logprob_t + g_h[t] H_t,
// the retained sets held fixed.  g_lp / g_h may be NULL (zero); force_k as for
// oracle_logprob_entropy.
int oracle_logprob_entropy_backward(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld,
                                    const int32_t* ids, float temperature, float top_p,
                                    const int64_t* force_k, const float* g_lp, const float* g_h,
                                    double* out_grad, int nthreads) {
  if (!logits || !ids || !out_grad || T < 0 || V < 1 || ld < V || (dtype != 0 && dtype != 1))
    return 1;
  const double Td = static_cast<double>(temperature), pd = static_cast<double>(top_p);
  parallel_rows(T, nthreads, [&](int64_t row) {
    std::vector<double> z = widen_row(logits, dtype, row, V, ld);
    score_row(z, ids[row], Td, pd, force_k ? force_k[row] : 0,
              g_lp ? static_cast<double>(g_lp[row]) : 0.0,
              g_h ? static_cast<double>(g_h[row]) : 0.0, out_grad + row * V);
  });
  return 0;
}

// Log-probability and entropy over a retained set supplied by the sampler
// (the sparse path of RL-Kernel "Qwen3-8B VIME train-rollout consistency",
// section "ROCm MI300X and gfx942", which scores the complete retained
// support it is given).  Row r's retained set S is the list
// sup_ids[offsets[r] .. offsets[r+1]); every listed token is kept.
//  1. x_i = z_i / T for the listed i; m_S = max x_i over the list.
//  2. w_i = exp(x_i - m_S), Z_S = sum over the list (compensated).
//  3. logprob(y) = (x_y - m_S) - ln Z_S if y is listed, else -inf.
//  4. H = -sum over the list of q_i ln q_i, q_i = w_i / Z_S, 0 ln 0 = 0.
// A repeated id counts each time it is listed (the list is the caller's).
// Per-row status: 1 selected id outside [0, V); 8 an empty list, a listed id
// outside [0, V) or offsets that decrease; 2 a non-finite listed logit.  A
// row with a status gets NaN outputs.
int oracle_logprob_entropy_support(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld,
                                   const int32_t* ids, float temperature, const int64_t* offsets,
                                   const int32_t* sup_ids, double* out_logprob,
                                   double* out_entropy, int32_t* out_status, int nthreads) {
  if (!logits || !ids || !offsets || T < 0 || V < 1 || ld < V || (dtype != 0 && dtype != 1))
    return 1;
  const double Td = static_cast<double>(temperature);
  parallel_rows(T, nthreads, [&](int64_t row) {
    double lp = kNaN, ent = kNaN;
    int32_t st = 0;
    const int64_t a = offsets[row], b = offsets[row + 1];
    const int64_t y = ids[row];
    if (y < 0 || y >= V) st = 1;
    else if (b <= a) st = 8;
    else {
      for (int64_t j = a; j < b; ++j)
        if (sup_ids[j] < 0 || sup_ids[j] >= V) st = 8;
    }
    if (st == 0) {
      std::vector<double> x;
      x.reserve(static_cast<size_t>(b - a));
      bool y_in = false;
      double m = -kInf;
      for (int64_t j = a; j < b; ++j) {
        const double z = load_logit(logits, dtype, row, ld, sup_ids[j]);
        if (!std::isfinite(z)) st = 2;
        x.push_back(z / Td);
        m = std::max(m, x.back());
        if (sup_ids[j] == y) y_in = true;
      }
      if (st == 0) {
        NeumaierSum zs;
        for (double v : x) zs.add(std::exp(v - m));
        const double ZS = zs.value();
        lp = y_in ? (load_logit(logits, dtype, row, ld, y) / Td - m) - std::log(ZS) : -kInf;
        NeumaierSum h;
        for (double v : x) {
          const double q = std::exp(v - m) / ZS;
          if (q > 0.0) h.add(-q * std::log(q));
        }
        ent = h.value();
      }
    }
    if (st != 0) lp = ent = kNaN;
    if (out_logprob) out_logprob[row] = lp;
    if (out_entropy) out_entropy[row] = ent;
    if (out_status) out_status[row] = st;
  });
  return 0;
}

// Gradient of the supplied-support scorer with respect to the listed logits,
// the retained set held fixed (the sampler chose it):
//   d logprob / d z_i = ([i = y] - q_i) / T   for listed i, when y is listed
//                       (0 when y is not listed: its log-probability is -inf);
//   d H / d z_i       = -q_i (ln q_i + H) / T for listed i;
// with q_i = exp(x_i - m_S) / Z_S as in oracle_logprob_entropy_support.
// out_grad[j] = g_lp[row] d logprob/d z_{sup_ids[j]} + g_H[row] d H/d z_{sup_ids[j]}
// for every list position j (g_lp / g_H may be NULL, meaning 0).  Rows with
// a status (as in the forward) get NaN gradients.
int oracle_logprob_entropy_support_backward(const void* logits, int dtype, int64_t T, int64_t V,
                                            int64_t ld, const int32_t* ids, float temperature,
                                            const int64_t* offsets, const int32_t* sup_ids,
                                            const float* g_lp, const float* g_h, double* out_grad,
                                            int nthreads) {
  if (!logits || !ids || !offsets || !out_grad || T < 0 || V < 1 || ld < V ||
      (dtype != 0 && dtype != 1))
    return 1;
  const double Td = static_cast<double>(temperature);
  parallel_rows(T, nthreads, [&](int64_t row) {
    const int64_t a = offsets[row], b = offsets[row + 1];
    const int64_t y = ids[row];
    bool bad = y < 0 || y >= V || b <= a;
    for (int64_t j = a; j < b && !bad; ++j)
      if (sup_ids[j] < 0 || sup_ids[j] >= V) bad = true;
    std::vector<double> x;
    double m = -kInf;
    bool y_in = false;
    if (!bad) {
      for (int64_t j = a; j < b; ++j) {
        const double z = load_logit(logits, dtype, row, ld, sup_ids[j]);
        if (!std::isfinite(z)) bad = true;
        x.push_back(z / Td);
        m = std::max(m, x.back());
        if (sup_ids[j] == y) y_in = true;
      }
    }
    if (bad) {
      for (int64_t j = a; j < b; ++j) out_grad[j] = kNaN;
      return;
    }
    NeumaierSum zs;
    for (double v : x) zs.add(std::exp(v - m));
    const double ZS = zs.value();
    NeumaierSum h;
    std::vector<double> q(x.size());
    for (size_t i = 0; i < x.size(); ++i) {
      q[i] = std::exp(x[i] - m) / ZS;
      if (q[i] > 0.0) h.add(-q[i] * std::log(q[i]));
    }
    const double H = h.value();
    const double glp = g_lp ? static_cast<double>(g_lp[row]) : 0.0;
    const double gh = g_h ? static_cast<double>(g_h[row]) : 0.0;
    for (int64_t j = a; j < b; ++j) {
      const double qi = q[j - a];
      const double dlp = y_in ? ((sup_ids[j] == y ? 1.0 : 0.0) - qi) / Td : 0.0;
      const double lq = qi > 0.0 ? std::log(qi) : 0.0;   // q ln q -> 0 as q -> 0
      const double dh = -qi * (lq + H) / Td;
      out_grad[j] = glp * dlp + gh * dh;
    }
  });
  return 0;
}

// Draws one id per row from the renormalised truncated distribution by
// inverse CDF over S in the ranking order: the first j with
// sum_{i<=j} w_pi(i) >= u * Z_S.  u in [0,1) is supplied per row.
int oracle_sample_ids(const void* logits, int dtype, int64_t T, int64_t V, int64_t ld,
                      float temperature, float top_p, const double* u, int32_t* out_ids,
                      int nthreads) {
  if (!logits || !u || !out_ids || T < 0 || V < 1 || ld < V) return 1;
  const double Td = static_cast<double>(temperature), pd = static_cast<double>(top_p);
  parallel_rows(T, nthreads, [&](int64_t row) {
    std::vector<double> z = widen_row(logits, dtype, row, V, ld);
    RowResult r = score_row(z, 0, Td, pd, 0);
    if (!std::isfinite(r.entropy)) { out_ids[row] = 0; return; }
    std::vector<double> w(V);
    double m = -kInf;
    for (int64_t i = 0; i < V; ++i) m = std::max(m, z[i] / Td);
    for (int64_t i = 0; i < V; ++i) w[i] = std::exp(z[i] / Td - m);
    std::vector<int64_t> order(V);
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
      if (z[a] != z[b]) return z[a] > z[b];
      return a < b;
    });
    NeumaierSum zs;
    for (int64_t j = 0; j < r.k; ++j) zs.add(w[order[j]]);
    const double target = u[row] * zs.value();
    NeumaierSum c;
    int64_t pick = order[r.k - 1];
    for (int64_t j = 0; j < r.k; ++j) {
      c.add(w[order[j]]);
      if (c.value() >= target) { pick = order[j]; break; }
    }
    out_ids[row] = static_cast<int32_t>(pick);
  });
  return 0;
}

// Statistics slots written by oracle_grpo_loss (same meaning as the library's).
enum { ST_LOSS = 0, ST_TOKENS, ST_CLIP_LOW, ST_CLIP_HIGH, ST_TIS_MEAN, ST_TIS_CAPPED,
       ST_K3_MEAN, ST_PG_MEAN, ST_COUNT };

// GRPO/DAPO loss over packed sequences grouped contiguously (sequence s is in
// group s / group_size).
//  1. mu_g = mean R, sigma_g = sqrt(sum (R - mu_g)^2 / (G - 1)) (0 when G = 1),
//     A_s = (R_s - mu_g) / (sigma_g + 1e-6).
//  2. per token: r = exp(new - old); pg = -min(r A, clip(r, 1 - eps_low, 1 + eps_high) A);
//     w = min(exp(old - rollout), tis_cap); delta = ref - new,
//     k3 = exp(delta) - delta - 1; l = w pg + kl_coef k3.
//  3. agg 0 (token mean): L = sum m l / sum m, 0 when sum m = 0.
//     agg 1 (sequence mean of token means): L = mean over sequences with
//     sum m > 0 of (sum_s m l / sum_s m).
//  4. dL/dnew = (weight of the token in L) (w g_pg + kl_coef (1 - exp(delta))),
//     g_pg = -r A when the unclipped term is the active minimum (ties count as
//     unclipped), else 0.
// Inputs are the float values the library receives, widened to double.
int oracle_grpo_loss(const float* logp_new, const float* logp_old, const float* logp_rollout,
                     const float* logp_ref, const uint8_t* mask, const float* rewards,
                     const int32_t* seq_offsets, int32_t n_seq, int32_t group_size,
                     float eps_low, float eps_high, float tis_cap, float kl_coef, int agg,
                     double* out_loss, double* out_grad, double* out_adv, double* out_stats) {
  if (!logp_new || !logp_old || !logp_rollout || !logp_ref || !rewards || !seq_offsets) return 1;
  if (n_seq < 0 || group_size < 1 || n_seq % group_size != 0) return 1;
  const int64_t t0 = seq_offsets[0], t1 = seq_offsets[n_seq];
  const double el = eps_low, eh = eps_high, C = tis_cap, beta = kl_coef;

  std::vector<double> A(n_seq, 0.0);
  for (int32_t g = 0; g < n_seq / group_size; ++g) {
    const int32_t s0 = g * group_size;
    NeumaierSum sum;
    for (int32_t j = 0; j < group_size; ++j) sum.add(rewards[s0 + j]);
    const double mu = sum.value() / group_size;
    double sigma = 0.0;
    if (group_size > 1) {
      NeumaierSum ss;
      for (int32_t j = 0; j < group_size; ++j) {
        double d = rewards[s0 + j] - mu;
        ss.add(d * d);
      }
      sigma = std::sqrt(ss.value() / (group_size - 1));
    }
    for (int32_t j = 0; j < group_size; ++j) A[s0 + j] = (rewards[s0 + j] - mu) / (sigma + 1e-6);
  }
  if (out_adv)
    for (int32_t s = 0; s < n_seq; ++s) out_adv[s] = A[s];

  // Per-token terms.
  const int64_t n_tok = t1 - t0;
  std::vector<double> ell(n_tok > 0 ? n_tok : 0), dl(n_tok > 0 ? n_tok : 0);
  std::vector<double> msk(n_tok > 0 ? n_tok : 0);
  NeumaierSum msum, lsum, clo, chi, tis, tcap, k3s, pgs;
  for (int32_t s = 0; s < n_seq; ++s) {
    for (int64_t t = seq_offsets[s]; t < seq_offsets[s + 1]; ++t) {
      const double nw = logp_new[t], od = logp_old[t], ro = logp_rollout[t], rf = logp_ref[t];
      const double m = mask ? (mask[t] ? 1.0 : 0.0) : 1.0;
      const double r = std::exp(nw - od);
      const double a = A[s];
      const double rc = std::min(std::max(r, 1.0 - el), 1.0 + eh);
      const double unclipped = r * a, clipped = rc * a;
      const double pg = -std::min(unclipped, clipped);
      const double g_pg = (unclipped <= clipped) ? -r * a : 0.0;
      const double raw_w = std::exp(od - ro);
      const double w = std::min(raw_w, C);
      const double delta = rf - nw;
      const double k3 = std::exp(delta) - delta - 1.0;
      ell[t - t0] = w * pg + beta * k3;
      dl[t - t0] = w * g_pg + beta * (1.0 - std::exp(delta));
      msk[t - t0] = m;
      msum.add(m);
      lsum.add(m * ell[t - t0]);
      clo.add(m * ((a < 0.0 && r < 1.0 - el) ? 1.0 : 0.0));
      chi.add(m * ((a > 0.0 && r > 1.0 + eh) ? 1.0 : 0.0));
      tis.add(m * w);
      tcap.add(m * (raw_w > C ? 1.0 : 0.0));
      k3s.add(m * k3);
      pgs.add(m * pg);
    }
  }
  const double M = msum.value();
  double L = 0.0;
  std::vector<double> weight(n_tok > 0 ? n_tok : 0, 0.0);
  if (agg == 0) {
    L = M > 0.0 ? lsum.value() / M : 0.0;
    for (int64_t i = 0; i < n_tok; ++i) weight[i] = M > 0.0 ? msk[i] / M : 0.0;
  } else if (agg == 1) {
    int64_t n_live = 0;
    for (int32_t s = 0; s < n_seq; ++s) {
      NeumaierSum ms;
      for (int64_t t = seq_offsets[s]; t < seq_offsets[s + 1]; ++t) ms.add(msk[t - t0]);
      if (ms.value() > 0.0) ++n_live;
    }
    NeumaierSum total;
    for (int32_t s = 0; s < n_seq; ++s) {
      NeumaierSum ms, ls;
      for (int64_t t = seq_offsets[s]; t < seq_offsets[s + 1]; ++t) {
        ms.add(msk[t - t0]);
        ls.add(msk[t - t0] * ell[t - t0]);
      }
      const double mseq = ms.value();
      if (mseq > 0.0) {
        total.add(ls.value() / mseq);
        for (int64_t t = seq_offsets[s]; t < seq_offsets[s + 1]; ++t)
          weight[t - t0] = msk[t - t0] / mseq / static_cast<double>(n_live);
      }
    }
    L = n_live > 0 ? total.value() / static_cast<double>(n_live) : 0.0;
  } else {
    return 1;
  }
  if (out_loss) *out_loss = L;
  if (out_grad)
    for (int64_t i = 0; i < n_tok; ++i) out_grad[i] = weight[i] * dl[i];
  if (out_stats) {
    const double d = M > 0.0 ? M : 1.0;
    out_stats[ST_LOSS] = L;
    out_stats[ST_TOKENS] = M;
    out_stats[ST_CLIP_LOW] = clo.value() / d;
    out_stats[ST_CLIP_HIGH] = chi.value() / d;
    out_stats[ST_TIS_MEAN] = tis.value() / d;
    out_stats[ST_TIS_CAPPED] = tcap.value() / d;
    out_stats[ST_K3_MEAN] = k3s.value() / d;
    out_stats[ST_PG_MEAN] = pgs.value() / d;
  }
  return 0;
}

// Policy-loss variants.  Sources: prime-rl v0.10.0 release notes, section
// "2. RL Algorithms" (the IPO mask |pi_train(y) - pi_infer(y)| > eps with
// eps = 0.3 and no KL term; IcePop, which masks a token whose ratio
// pi_train / pi_infer leaves a fixed band; a length-weighted GRPO baseline and
// prompt-mean aggregation), LumenRL README, section "Rollout Correction" (TIS
// clips large ratios, MIS normalises them).  pi_train(y) = exp(new) and
// pi_infer(y) = exp(rollout).  Readings where the pages give no formula:
//  - IPO's surrogate is the importance-weighted policy gradient against the
//    inference policy, -rho A with rho = exp(new - rollout), on tokens the mask
//    keeps (no clipping);
//  - IcePop keeps the clipped (DAPO) term on tokens whose rho lies in
//    [band_low, band_high] and drops the others;
//  - MIS divides exp(old - rollout) by its mean over the batch's tokens with
//    mask 1 (no cap); TIS caps it at is_cap; none uses 1;
//  - the length-weighted baseline weights each reward by its sequence's packed
//    length, seq_offsets[s+1] - seq_offsets[s] (the plain mean when the group
//    has no tokens); the divisor stays the plain group standard deviation;
//  - prompt-mean aggregation averages, over groups with sum m > 0, each
//    group's token mean.
// Steps:
//  1. A_s = (R_s - b_g) / (sigma_g + 1e-6), b_g the plain or length-weighted
//     group mean, sigma_g as in oracle_grpo_loss.
//  2. per token: r = exp(new - old), rho = exp(new - rollout),
//     raw = exp(old - rollout);
//     type 0 (DAPO):   keep = 1; pg = -min(r A, clip(r) A); g = -r A if the
//                      unclipped term is the active minimum, else 0;
//     type 1 (IPO):    keep = [|exp(new) - exp(rollout)| <= ipo_eps];
//                      pg = -keep rho A; g = pg;
//     type 2 (IcePop): keep = [band_low <= rho <= band_high]; pg, g = keep x
//                      the DAPO ones;
//     w by is_method (0 none, 1 TIS, 2 MIS); delta = ref - new,
//     k3 = exp(delta) - delta - 1; l = w pg + kl_coef k3;
//     dl = w g + kl_coef (1 - exp(delta)).
//  3. agg 0 token mean, 1 sequence mean of token means, 2 prompt (group) mean
//     of token means.
//  4. dL/dnew = (weight of the token in L) dl.
// Stats: the eight of oracle_grpo_loss (clip fractions for types 0 and 2 only,
// the capped fraction for TIS only, slot 4 the mean of w) and slot 8, the
// fraction of mask-1 tokens the IPO / IcePop mask drops.
int oracle_policy_loss(const float* logp_new, const float* logp_old, const float* logp_rollout,
                       const float* logp_ref, const uint8_t* mask, const float* rewards,
                       const int32_t* seq_offsets, int32_t n_seq, int32_t group_size, int type,
                       float eps_low, float eps_high, float ipo_eps, float band_low,
                       float band_high, int is_method, float is_cap, float kl_coef, int baseline,
                       int agg, double* out_loss, double* out_grad, double* out_adv,
                       double* out_stats) {
  if (!logp_new || !logp_old || !logp_rollout || !logp_ref || !rewards || !seq_offsets) return 1;
  if (n_seq < 0 || group_size < 1 || n_seq % group_size != 0) return 1;
  if (type < 0 || type > 2 || is_method < 0 || is_method > 2 || baseline < 0 || baseline > 1 ||
      agg < 0 || agg > 2)
    return 1;
  const int64_t t0 = seq_offsets[0], t1 = seq_offsets[n_seq];
  const int64_t n_tok = t1 - t0;
  const double el = eps_low, eh = eps_high, beta = kl_coef;
  const int32_t n_grp = n_seq / group_size;

  // 1. advantages
  std::vector<double> A(n_seq, 0.0);
  for (int32_t g = 0; g < n_grp; ++g) {
    const int32_t s0 = g * group_size;
    NeumaierSum sum;
    for (int32_t j = 0; j < group_size; ++j) sum.add(rewards[s0 + j]);
    const double mu = sum.value() / group_size;
    double sigma = 0.0;
    if (group_size > 1) {
      NeumaierSum ss;
      for (int32_t j = 0; j < group_size; ++j) {
        const double d = rewards[s0 + j] - mu;
        ss.add(d * d);
      }
      sigma = std::sqrt(ss.value() / (group_size - 1));
    }
    double b = mu;
    if (baseline == 1) {
      NeumaierSum lw, ln;
      for (int32_t j = 0; j < group_size; ++j) {
        const double len = static_cast<double>(seq_offsets[s0 + j + 1] - seq_offsets[s0 + j]);
        lw.add(len * rewards[s0 + j]);
        ln.add(len);
      }
      if (ln.value() > 0.0) b = lw.value() / ln.value();
    }
    for (int32_t j = 0; j < group_size; ++j) A[s0 + j] = (rewards[s0 + j] - b) / (sigma + 1e-6);
  }
  if (out_adv)
    for (int32_t s = 0; s < n_seq; ++s) out_adv[s] = A[s];

  // the MIS normaliser: mean of exp(old - rollout) over tokens with mask 1
  double raw_mean = 1.0;
  if (is_method == 2) {
    NeumaierSum rs, ms;
    for (int64_t t = t0; t < t1; ++t) {
      const double m = mask ? (mask[t] ? 1.0 : 0.0) : 1.0;
      rs.add(m * std::exp(static_cast<double>(logp_old[t]) - logp_rollout[t]));
      ms.add(m);
    }
    if (ms.value() > 0.0) raw_mean = rs.value() / ms.value();
  }

  // 2. per-token terms
  std::vector<double> ell(n_tok > 0 ? n_tok : 0), dl(n_tok > 0 ? n_tok : 0);
  std::vector<double> msk(n_tok > 0 ? n_tok : 0);
  NeumaierSum msum, clo, chi, wsum, tcap, k3s, pgs, dropped;
  for (int32_t s = 0; s < n_seq; ++s) {
    const double a = A[s];
    for (int64_t t = seq_offsets[s]; t < seq_offsets[s + 1]; ++t) {
      const double nw = logp_new[t], od = logp_old[t], ro = logp_rollout[t], rf = logp_ref[t];
      const double m = mask ? (mask[t] ? 1.0 : 0.0) : 1.0;
      const double r = std::exp(nw - od), rho = std::exp(nw - ro), raw = std::exp(od - ro);
      double keep = 1.0, pg = 0.0, gpg = 0.0;
      if (type == 0 || type == 2) {
        const double rc = std::min(std::max(r, 1.0 - el), 1.0 + eh);
        pg = -std::min(r * a, rc * a);
        gpg = (r * a <= rc * a) ? -r * a : 0.0;
        if (type == 2) keep = (rho >= band_low && rho <= band_high) ? 1.0 : 0.0;
        pg *= keep;
        gpg *= keep;
        clo.add(m * ((a < 0.0 && r < 1.0 - el) ? 1.0 : 0.0));
        chi.add(m * ((a > 0.0 && r > 1.0 + eh) ? 1.0 : 0.0));
      } else {
        keep = std::fabs(std::exp(nw) - std::exp(ro)) <= ipo_eps ? 1.0 : 0.0;
        pg = -keep * rho * a;
        gpg = pg;
      }
      double w = 1.0;
      if (is_method == 1) {
        w = std::min(raw, static_cast<double>(is_cap));
        tcap.add(m * (raw > is_cap ? 1.0 : 0.0));
      } else if (is_method == 2) {
        w = raw / raw_mean;
      }
      const double delta = rf - nw;
      const double k3 = std::exp(delta) - delta - 1.0;
      ell[t - t0] = w * pg + beta * k3;
      dl[t - t0] = w * gpg + beta * (1.0 - std::exp(delta));
      msk[t - t0] = m;
      msum.add(m);
      wsum.add(m * w);
      k3s.add(m * k3);
      pgs.add(m * pg);
      dropped.add(m * (1.0 - keep));
    }
  }

  // 3. aggregation over units: the batch (0), sequences (1) or groups (2)
  const int32_t per_unit = agg == 1 ? 1 : group_size;
  const int32_t n_unit = agg == 0 ? 1 : (agg == 1 ? n_seq : n_grp);
  std::vector<double> weight(n_tok > 0 ? n_tok : 0, 0.0);
  std::vector<double> unit_mean(n_unit, 0.0), unit_m(n_unit, 0.0);
  int64_t n_live = 0;
  for (int32_t u = 0; u < n_unit; ++u) {
    const int64_t a0 = agg == 0 ? t0 : seq_offsets[u * per_unit];
    const int64_t a1 = agg == 0 ? t1 : seq_offsets[(u + 1) * per_unit];
    NeumaierSum ms, ls;
    for (int64_t t = a0; t < a1; ++t) {
      ms.add(msk[t - t0]);
      ls.add(msk[t - t0] * ell[t - t0]);
    }
    unit_m[u] = ms.value();
    if (unit_m[u] > 0.0) {
      unit_mean[u] = ls.value() / unit_m[u];
      ++n_live;
    }
  }
  NeumaierSum total;
  for (int32_t u = 0; u < n_unit; ++u) {
    if (unit_m[u] <= 0.0) continue;
    total.add(unit_mean[u]);
    const int64_t a0 = agg == 0 ? t0 : seq_offsets[u * per_unit];
    const int64_t a1 = agg == 0 ? t1 : seq_offsets[(u + 1) * per_unit];
    for (int64_t t = a0; t < a1; ++t)
      weight[t - t0] = msk[t - t0] / unit_m[u] / static_cast<double>(n_live);
  }
  const double L = n_live > 0 ? total.value() / static_cast<double>(n_live) : 0.0;
  if (out_loss) *out_loss = L;
  if (out_grad)
    for (int64_t i = 0; i < n_tok; ++i) out_grad[i] = weight[i] * dl[i];
  if (out_stats) {
    const double M = msum.value(), d = M > 0.0 ? M : 1.0;
    out_stats[ST_LOSS] = L;
    out_stats[ST_TOKENS] = M;
    out_stats[ST_CLIP_LOW] = clo.value() / d;
    out_stats[ST_CLIP_HIGH] = chi.value() / d;
    out_stats[ST_TIS_MEAN] = wsum.value() / d;
    out_stats[ST_TIS_CAPPED] = tcap.value() / d;
    out_stats[ST_K3_MEAN] = k3s.value() / d;
    out_stats[ST_PG_MEAN] = pgs.value() / d;
    out_stats[8] = dropped.value() / d;   // dropped by the IPO / IcePop mask
  }
  return 0;
}

// LM-head rows: z_i = sum_k h_k W_ik in fp64 from the exact bf16 values (never
// rounded to bf16), then the logits path above on that row.  hidden: bf16
// [T, H]; w_vocab: bf16 [V, H] row-major.  rows[0..n_rows) selects the rows.
int oracle_lmhead_rows(const uint16_t* hidden, const uint16_t* w_vocab, int64_t T, int64_t H,
                       int64_t V, const int64_t* rows, int64_t n_rows, const int32_t* ids,
                       float temperature, float top_p, double* out_logprob,
                       double* out_entropy, int64_t* out_k, int nthreads) {
  if (!hidden || !w_vocab || !rows || !ids || H < 1 || V < 1) return 1;
  const double Td = static_cast<double>(temperature), pd = static_cast<double>(top_p);
  parallel_rows(n_rows, nthreads, [&](int64_t j) {
    const int64_t row = rows[j];
    if (row < 0 || row >= T) {
      if (out_logprob) out_logprob[j] = kNaN;
      if (out_entropy) out_entropy[j] = kNaN;
      return;
    }
    std::vector<double> h(H), z(V);
    for (int64_t k = 0; k < H; ++k) h[k] = bf16_to_double(hidden[row * H + k]);
    for (int64_t i = 0; i < V; ++i) {
      const uint16_t* wr = w_vocab + i * H;
      double acc = 0.0;  // products of bf16 values are exact in fp64
      for (int64_t k = 0; k < H; ++k) acc += h[k] * bf16_to_double(wr[k]);
      z[i] = acc;
    }
    RowResult r = score_row(z, ids[row], Td, pd, 0);
    if (out_logprob) out_logprob[j] = r.logprob;
    if (out_entropy) out_entropy[j] = r.entropy;
    if (out_k) out_k[j] = r.k;
  });
  return 0;
}

// Gradient of the LM-head path (oracle_lmhead_rows, every row) for
// L = sum_t g_lp[t] logprob_t + g_h[t] H_t, the retained sets held fixed:
//  1. z = hidden W^T in fp64 from the exact bf16 values;
//  2. dz[t, :] = the logits-path gradient of row t (score_row, step 9);
//  3. out_dh = dz W ([T, H]); out_dw = dz^T hidden ([V, H]), each entry a
//     plain sum over the contracted index in increasing order.
// Rows with no distribution give NaN in their dz, so in dh and in every dw.
int oracle_lmhead_backward(const uint16_t* hidden, const uint16_t* w_vocab, int64_t T, int64_t H,
                           int64_t V, const int32_t* ids, float temperature, float top_p,
                           const float* g_lp, const float* g_h, double* out_dh, double* out_dw,
                           int nthreads) {
  if (!hidden || !w_vocab || !ids || T < 0 || H < 1 || V < 1 || !out_dh || !out_dw) return 1;
  const double Td = static_cast<double>(temperature), pd = static_cast<double>(top_p);
  std::vector<double> dz(static_cast<size_t>(T) * V);
  parallel_rows(T, nthreads, [&](int64_t row) {
    std::vector<double> h(H), z(V);
    for (int64_t k = 0; k < H; ++k) h[k] = bf16_to_double(hidden[row * H + k]);
    for (int64_t i = 0; i < V; ++i) {
      const uint16_t* wr = w_vocab + i * H;
      double acc = 0.0;  // products of bf16 values are exact in fp64
      for (int64_t k = 0; k < H; ++k) acc += h[k] * bf16_to_double(wr[k]);
      z[i] = acc;
    }
    score_row(z, ids[row], Td, pd, 0, g_lp ? static_cast<double>(g_lp[row]) : 0.0,
              g_h ? static_cast<double>(g_h[row]) : 0.0, dz.data() + row * V);
    // every out_dh[row, k] accumulates over i = 0, 1, ..., V-1 from 0; the
    // vocabulary loop is outermost so that W is read row by row
    double* dh = out_dh + row * H;
    for (int64_t k = 0; k < H; ++k) dh[k] = 0.0;
    for (int64_t i = 0; i < V; ++i) {
      const double d = dz[row * V + i];
      const uint16_t* wr = w_vocab + i * H;
      for (int64_t k = 0; k < H; ++k) dh[k] += d * bf16_to_double(wr[k]);
    }
  });
  parallel_rows(V, nthreads, [&](int64_t i) {
    for (int64_t k = 0; k < H; ++k) {
      double acc = 0.0;
      for (int64_t row = 0; row < T; ++row)
        acc += dz[row * V + i] * bf16_to_double(hidden[row * H + k]);
      out_dw[i * H + k] = acc;
    }
  });
  return 0;
}

}  // extern "C"
