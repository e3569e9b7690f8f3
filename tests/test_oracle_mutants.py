"""The oracle's pins have teeth: each plausible mistake below (a dropped term,
a wrong sign, index or operand, a strict comparison where the pages' rule is
inclusive, the wrong normaliser) is planted, one at a time, in a copy of
``oracle/oracle.cpp`` compiled on the CPU, and ``test_oracle_pins.py`` run
against that copy must fail.  Nothing here touches a GPU or the product.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

# (name, text in oracle.cpp, replacement); each text occurs exactly once.
MUTANTS = [
    # the logits path
    ("nucleus_strict", "if (p < 1.0 && !found && c >= p) {", "if (p < 1.0 && !found && c > p) {"),
    ("temperature_multiplies", "    x[i] = z[i] / T;\n    m = std::max(m, x[i]);",
     "    x[i] = z[i] * T;\n    m = std::max(m, x[i]);"),
    ("ties_high_id_first",
     "    if (z[a] != z[b]) return z[a] > z[b];  // -0.0 == +0.0 compares equal\n    return a < b;",
     "    if (z[a] != z[b]) return z[a] > z[b];  // -0.0 == +0.0 compares equal\n    return a > b;"),
    ("logprob_full_normaliser", "r.logprob = member[y] ? (x[y] - m) - std::log(ZS) : -kInf;",
     "r.logprob = member[y] ? (x[y] - m) - std::log(Z) : -kInf;"),
    ("entropy_sign", "    if (q > 0.0) h.add(-q * std::log(q));\n  }\n  r.entropy",
     "    if (q > 0.0) h.add(q * std::log(q));\n  }\n  r.entropy"),
    ("entropy_full_normaliser", "    double q = w[order[j]] / ZS;", "    double q = w[order[j]] / Z;"),
    ("gap_max", "r.gap = (p >= 1.0) ? kInf : std::min(", "r.gap = (p >= 1.0) ? kInf : std::max("),
    # the dense gradient
    ("grad_without_inverse_T",
     "const double dlp = member[y] ? ((i == y ? 1.0 : 0.0) - q) / T : 0.0;",
     "const double dlp = member[y] ? ((i == y ? 1.0 : 0.0) - q) : 0.0;"),
    ("grad_entropy_sign", "grad[i] = glp * dlp - gh * q * (lq + H) / T;",
     "grad[i] = glp * dlp + gh * q * (lq + H) / T;"),
    ("grad_ignores_y_outside_S",
     "const double dlp = member[y] ? ((i == y ? 1.0 : 0.0) - q) / T : 0.0;",
     "const double dlp = ((i == y ? 1.0 : 0.0) - q) / T;"),
    ("grad_drops_H", "grad[i] = glp * dlp - gh * q * (lq + H) / T;",
     "grad[i] = glp * dlp - gh * q * lq / T;"),
    # the GRPO/DAPO loss
    ("std_biased",
     "      sigma = std::sqrt(ss.value() / (group_size - 1));\n    }\n    for (int32_t j = 0; "
     "j < group_size; ++j) A[s0 + j] = (rewards[s0 + j] - mu) / (sigma + 1e-6);",
     "      sigma = std::sqrt(ss.value() / group_size);\n    }\n    for (int32_t j = 0; "
     "j < group_size; ++j) A[s0 + j] = (rewards[s0 + j] - mu) / (sigma + 1e-6);"),
    ("clip_bounds_swapped",
     "      const double rc = std::min(std::max(r, 1.0 - el), 1.0 + eh);\n      const double unclipped",
     "      const double rc = std::min(std::max(r, 1.0 - eh), 1.0 + el);\n      const double unclipped"),
    ("pg_max_not_min", "const double pg = -std::min(unclipped, clipped);",
     "const double pg = -std::max(unclipped, clipped);"),
    ("tis_ratio_inverted", "const double raw_w = std::exp(od - ro);",
     "const double raw_w = std::exp(ro - od);"),
    ("k3_delta_sign",
     "      const double delta = rf - nw;\n      const double k3 = std::exp(delta) - delta - 1.0;\n"
     "      ell[t - t0] = w * pg + beta * k3;\n      dl[t - t0] = w * g_pg",
     "      const double delta = nw - rf;\n      const double k3 = std::exp(delta) - delta - 1.0;\n"
     "      ell[t - t0] = w * pg + beta * k3;\n      dl[t - t0] = w * g_pg"),
    ("k3_grad_sign", "dl[t - t0] = w * g_pg + beta * (1.0 - std::exp(delta));",
     "dl[t - t0] = w * g_pg + beta * (std::exp(delta) - 1.0);"),
    ("clip_tie_rule", "const double g_pg = (unclipped <= clipped) ? -r * a : 0.0;",
     "const double g_pg = (unclipped < clipped) ? -r * a : 0.0;"),
    ("eps_inside_sqrt",
     "    for (int32_t j = 0; j < group_size; ++j) A[s0 + j] = (rewards[s0 + j] - mu) / "
     "(sigma + 1e-6);\n  }\n  if (out_adv)\n    for (int32_t s = 0; s < n_seq; ++s) out_adv[s] = "
     "A[s];\n\n  // Per-token terms.",
     "    for (int32_t j = 0; j < group_size; ++j) A[s0 + j] = (rewards[s0 + j] - mu) / "
     "std::sqrt(sigma * sigma + 1e-6);\n  }\n  if (out_adv)\n    for (int32_t s = 0; s < n_seq; "
     "++s) out_adv[s] = A[s];\n\n  // Per-token terms."),
    ("seq_mean_without_live_count",
     "weight[t - t0] = msk[t - t0] / mseq / static_cast<double>(n_live);",
     "weight[t - t0] = msk[t - t0] / mseq;"),
    # the loss variants
    ("ipo_on_log_ratio", "keep = std::fabs(std::exp(nw) - std::exp(ro)) <= ipo_eps ? 1.0 : 0.0;",
     "keep = std::fabs(nw - ro) <= ipo_eps ? 1.0 : 0.0;"),
    ("ipo_ratio_against_old", "pg = -keep * rho * a;", "pg = -keep * r * a;"),
    ("icepop_band_on_old_ratio",
     "if (type == 2) keep = (rho >= band_low && rho <= band_high) ? 1.0 : 0.0;",
     "if (type == 2) keep = (r >= band_low && r <= band_high) ? 1.0 : 0.0;"),
    ("mis_mean_over_all_tokens",
     "      rs.add(m * std::exp(static_cast<double>(logp_old[t]) - logp_rollout[t]));\n"
     "      ms.add(m);",
     "      rs.add(std::exp(static_cast<double>(logp_old[t]) - logp_rollout[t]));\n"
     "      ms.add(1.0);"),
    ("length_baseline_unweighted", "lw.add(len * rewards[s0 + j]);", "lw.add(rewards[s0 + j]);"),
    # the supplied support
    ("support_logprob_ignores_listing",
     "lp = y_in ? (load_logit(logits, dtype, row, ld, y) / Td - m) - std::log(ZS) : -kInf;",
     "lp = (load_logit(logits, dtype, row, ld, y) / Td - m) - std::log(ZS);"),
    ("support_grad_entropy_sign", "      const double dh = -qi * (lq + H) / Td;",
     "      const double dh = qi * (lq + H) / Td;"),
    ("support_grad_ignores_listing",
     "const double dlp = y_in ? ((sup_ids[j] == y ? 1.0 : 0.0) - qi) / Td : 0.0;",
     "const double dlp = ((sup_ids[j] == y ? 1.0 : 0.0) - qi) / Td;"),
    # the sampler
    ("sampler_full_normaliser", "for (int64_t j = 0; j < r.k; ++j) zs.add(w[order[j]]);",
     "for (int64_t j = 0; j < V; ++j) zs.add(w[order[j]]);"),
    ("sampler_strict_comparison", "if (c.value() >= target)", "if (c.value() > target + 1e-9)"),
    ("sampler_off_by_one", "{ pick = order[j]; break; }",
     "{ pick = order[j + 1 < r.k ? j + 1 : j]; break; }"),
    # the LM-head
    ("lmhead_rows_without_temperature",
     "    RowResult r = score_row(z, ids[row], Td, pd, 0);\n    if (out_logprob) out_logprob[j] = r.logprob;",
     "    RowResult r = score_row(z, ids[row], 1.0, pd, 0);\n    if (out_logprob) out_logprob[j] = r.logprob;"),
    ("lmhead_dh_shifted_column", "for (int64_t k = 0; k < H; ++k) dh[k] += d * bf16_to_double(wr[k]);",
     "for (int64_t k = 0; k < H; ++k) dh[k] += d * bf16_to_double(wr[(k + 1) % H]);"),
    ("lmhead_dw_first_row_only",
     "        acc += dz[row * V + i] * bf16_to_double(hidden[row * H + k]);",
     "        acc += dz[i] * bf16_to_double(hidden[row * H + k]);"),
]

_RUNNER = """
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle
oracle._LIB_PATH = {lib!r}
oracle._lib = None
oracle.build = lambda force=False: oracle._LIB_PATH
import pytest
sys.exit(pytest.main(['-q', '-x', '-p', 'no:cacheprovider', {pins!r}]))
"""


def _survives(mutant, work):
    """True when every pin passes with the mistake planted."""
    name, old, new = mutant
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: the text to mutate must occur once"
    d = os.path.join(work, name)
    os.makedirs(d)
    cpp = os.path.join(d, "oracle.cpp")
    with open(cpp, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(d, "liboracle.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-fno-fast-math",
                    "-ffp-contract=off", cpp, "-o", lib], check=True)
    code = _RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib,
                          pins=os.path.join(ROOT, "tests", "test_oracle_pins.py"))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900,
                       env=env)
    return r.returncode == 0


def test_pins_catch_every_planted_mistake(tmp_path):
    """All mutants, built and checked a few at a time (each is its own
    process); none may pass every pin."""
    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with ThreadPoolExecutor(workers) as pool:
        alive = list(pool.map(lambda m: _survives(m, str(tmp_path)), MUTANTS))
    survivors = [m[0] for m, a in zip(MUTANTS, alive) if a]
    assert not survivors, f"pins pass with these mistakes planted: {survivors}"
