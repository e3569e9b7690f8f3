"""Pins for the fp64 oracle: each test checks it against something other than
itself -- brute force, a closed form, a library routine, an invariant, or a
hand-worked value -- chosen so that a dropped term, a wrong sign, a wrong index
or a transposed operand in the oracle fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import workloads

TEMPS = (0.2, 0.7, 1.0, 1.8)   # the temperatures the RL-Kernel GPU suite exercises


def f32(x):
    return float(np.float32(x))


def score_all_ids(oracle, row, temperature, top_p):
    """Score one row once per vocabulary id (row repeated V times)."""
    row = np.asarray(row)
    V = row.shape[0]
    rep = np.ascontiguousarray(np.repeat(row[None, :], V, axis=0))
    return oracle.logprob_entropy(rep, np.arange(V, dtype=np.int32), temperature, top_p)


# --------------------------------------------------------------------------
# Brute force over every subset (V = 8).
# --------------------------------------------------------------------------

def brute_nucleus(z, temperature, top_p):
    """Smallest-cardinality id set with mass >= top_p; among those the largest
    mass; among equal masses the lexicographically smallest sorted id tuple."""
    T = f32(temperature)
    p = f32(top_p)
    x = [float(v) / T for v in z]
    mx = max(x)
    w = [math.exp(v - mx) for v in x]
    Z = math.fsum(w)
    V = len(z)
    best = None
    for size in range(1, V + 1):
        for ids in itertools.combinations(range(V), size):
            mass = math.fsum(w[i] for i in ids) / Z
            if mass >= p:
                key = (-mass, ids)
                if best is None or key < best[0]:
                    best = (key, ids)
        if best is not None:
            break
    S = best[1]
    ZS = math.fsum(w[i] for i in S)
    lp = {i: (x[i] - mx) - math.log(ZS) for i in S}
    H = -math.fsum((w[i] / ZS) * math.log(w[i] / ZS) for i in S)
    return set(S), lp, H


@pytest.mark.parametrize("temperature", [0.7, 1.0])
def test_bruteforce_v8(oracle, temperature):
    z, _ = workloads.brute_v8(seed=0)
    z = z.numpy()
    checked = 0
    for r in range(z.shape[0]):
        lp, ent, k, gap = score_all_ids(oracle, z[r], temperature, 0.9)
        if gap[0] < 1e-9:
            continue
        S, blp, bH = brute_nucleus(z[r], temperature, 0.9)
        members = {i for i in range(8) if np.isfinite(lp[i])}
        assert members == S
        assert k[0] == len(S)
        for i in range(8):
            if i in S:
                assert abs(lp[i] - blp[i]) < 1e-12
            else:
                assert lp[i] == -np.inf
        assert abs(ent[0] - bH) < 1e-12
        checked += 1
    assert checked >= 12


def test_bruteforce_ties_lower_id_first(oracle):
    # Equal logits: the brute force prefers the lexicographically smallest id set,
    # i.e. ties are kept lower id first.
    z = np.array([1.0, 2.0, 2.0, 0.5, 2.0, 1.0, -1.0, 2.0], np.float32)
    for p in (0.3, 0.5, 0.6, 0.75, 0.9, 0.97):
        lp, ent, k, gap = score_all_ids(oracle, z, 1.0, p)
        S, blp, bH = brute_nucleus(z, 1.0, p)
        assert {i for i in range(8) if np.isfinite(lp[i])} == S
        assert abs(ent[0] - bH) < 1e-12
    # bf16 bit patterns, including -0 and +0 which rank as equal values.
    bits = np.array([0x8000, 0x0000, 0x3F80, 0x3F80, 0x0000, 0xBF80, 0x8000, 0x3F80], np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    for p in (0.2, 0.45, 0.7, 0.8, 0.95):
        lp, ent, k, gap = score_all_ids(oracle, bits, 1.0, p)
        S, blp, bH = brute_nucleus(vals, 1.0, p)
        assert {i for i in range(8) if np.isfinite(lp[i])} == S
        assert abs(ent[0] - bH) < 1e-12


# --------------------------------------------------------------------------
# Closed forms.
# --------------------------------------------------------------------------

def test_uniform_logits_entropy_is_log_k(oracle):
    V = 1000
    row = np.full(V, 0.375, np.float32)
    # p = 0.9005: pV is not near an integer, so k* = ceil(pV) = 901 exactly.
    lp, ent, k, gap = score_all_ids(oracle, row, 0.7, 0.9005)
    assert k[0] == 901
    assert abs(ent[0] - math.log(901)) < 1e-12
    assert np.all(np.abs(lp[:901] + math.log(901)) < 1e-12)   # lower ids kept first
    assert np.all(lp[901:] == -np.inf)
    # top_p = 1 keeps the whole vocabulary.
    lp, ent, k, gap = score_all_ids(oracle, row, 0.7, 1.0)
    assert k[0] == V and gap[0] == np.inf
    assert abs(ent[0] - math.log(V)) < 1e-12


def test_uniform_gap_value(oracle):
    # float32(0.9) = 0.89999997615814...: C_899 = 0.899 < p <= C_900 = 0.9.
    row = np.zeros(1000, np.float32)
    lp, ent, k, gap = oracle.logprob_entropy(row[None, :], np.zeros(1, np.int32), 1.0, 0.9)
    p = f32(0.9)
    assert k[0] == 900
    assert abs(gap[0] - min(p - 0.899, 0.9 - p)) < 1e-15


@pytest.mark.parametrize("temperature", TEMPS)
def test_top_p_one_is_log_softmax(oracle, temperature):
    z, ids = workloads.tiny(seed=0)
    lp, ent, k, gap = oracle.logprob_entropy(z.numpy(), ids.numpy(), temperature, 1.0)
    zz = z.double() / f32(temperature)
    ref_lp = torch.log_softmax(zz, dim=1)
    ref_ent = torch.special.entr(torch.softmax(zz, dim=1)).sum(dim=1)
    sel = ref_lp[torch.arange(z.shape[0]), ids.long()].numpy()
    assert np.max(np.abs(lp - sel)) < 1e-12
    assert np.max(np.abs(ent - ref_ent.numpy())) < 1e-12
    assert np.all(k == z.shape[1])


def test_one_hot_peak(oracle):
    V = 500
    T = 0.7
    row = np.zeros(V, np.float32)
    row[123] = f32(60 * T + 1)
    lp, ent, k, gap = score_all_ids(oracle, row, T, 0.95)
    assert k[0] == 1
    assert lp[123] == 0.0
    assert ent[0] == 0.0
    assert np.all(np.delete(lp, 123) == -np.inf)


@pytest.mark.parametrize("a,b,alpha,beta,T,p", [
    (5, 300, 2.0, 0.0, 0.7, 0.6),
    (5, 300, 2.0, 0.0, 0.7, 0.95),
    (40, 10, 1.0, 0.5, 1.0, 0.5),
    (3, 997, 4.0, -1.0, 1.8, 0.93),
    (7, 50, 0.25, -0.25, 0.2, 0.999),
])
def test_two_level_logits(oracle, a, b, alpha, beta, T, p):
    V = a + b
    rng = np.random.default_rng(a * 1000 + b)
    pos = rng.permutation(V)
    hi_ids = np.sort(pos[:a])
    lo_ids = np.sort(pos[a:])
    row = np.empty(V, np.float32)
    row[hi_ids] = alpha
    row[lo_ids] = beta
    Tf, pf = f32(T), f32(p)
    wb = math.exp((beta - alpha) / Tf)       # w of a low token, w of a high token is 1
    Z = a + b * wb
    if pf * Z <= a:
        n_hi, n_lo = math.ceil(pf * Z), 0
    else:
        n_hi, n_lo = a, math.ceil((pf * Z - a) / wb)
    ZS = n_hi + n_lo * wb
    qa, qb = 1.0 / ZS, wb / ZS
    H = -(n_hi * qa * math.log(qa) + (n_lo * qb * math.log(qb) if n_lo else 0.0))
    lp, ent, k, gap = score_all_ids(oracle, row, T, p)
    assert gap[0] > 1e-9
    assert k[0] == n_hi + n_lo
    assert abs(ent[0] - H) < 1e-11
    members = set(hi_ids[:n_hi].tolist()) | set(lo_ids[:n_lo].tolist())
    assert {i for i in range(V) if np.isfinite(lp[i])} == members
    for i in hi_ids[:n_hi]:
        assert abs(lp[i] - math.log(qa)) < 1e-11
    for i in lo_ids[:n_lo]:
        assert abs(lp[i] - math.log(qb)) < 1e-11


# --------------------------------------------------------------------------
# Invariants.
# --------------------------------------------------------------------------

def _small_peaked(T=6, V=2000, seed=11):
    z, peaks = workloads.peaked_bf16(T, V, seed=seed)
    return workloads.bf16_bits(z)


@pytest.mark.parametrize("p", [0.5, 0.95, 1.0])
def test_members_sum_to_one_and_entropy_bounds(oracle, p):
    bits = _small_peaked()
    for r in range(bits.shape[0]):
        lp, ent, k, gap = score_all_ids(oracle, bits[r], 0.7, p)
        fin = np.isfinite(lp)
        assert fin.sum() == k[0]
        assert abs(math.fsum(np.exp(lp[fin])) - 1.0) < 1e-12
        assert -1e-12 <= ent[0] <= math.log(k[0]) + 1e-12


def test_k_monotone_in_top_p(oracle):
    bits = _small_peaked(T=8)
    ids = np.zeros(bits.shape[0], np.int32)
    prev = np.zeros(bits.shape[0], np.int64)
    for p in np.linspace(0.05, 1.0, 40):
        _, _, k, _ = oracle.logprob_entropy(bits, ids, 0.7, float(p))
        assert np.all(k >= prev)
        prev = k
    assert np.all(prev == bits.shape[1])


def test_shift_and_temperature_invariance(oracle):
    rng = np.random.default_rng(5)
    z = (rng.integers(-512, 512, size=(8, 700)) / 64.0).astype(np.float32)  # exact grid
    ids = rng.integers(0, 700, size=8).astype(np.int32)
    base = oracle.logprob_entropy(z, ids, 0.7, 0.9)
    shifted = oracle.logprob_entropy(z + np.float32(3.0), ids, 0.7, 0.9)
    assert np.array_equal(base[2], shifted[2])
    fin = np.isfinite(base[0])
    assert np.array_equal(fin, np.isfinite(shifted[0]))
    assert np.max(np.abs(base[0][fin] - shifted[0][fin])) < 1e-12
    assert np.max(np.abs(base[1] - shifted[1])) < 1e-12
    # z / 0.5 at temperature 1 is exactly z at temperature 0.5.
    a = oracle.logprob_entropy(z, ids, 0.5, 0.9)
    b = oracle.logprob_entropy(z * np.float32(2.0), ids, 1.0, 0.9)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bad_inputs_give_nan(oracle):
    z = np.zeros((3, 10), np.float32)
    z[1, 4] = np.inf
    ids = np.array([2, 3, 10], np.int32)   # row 2: id out of range
    lp, ent, k, gap = oracle.logprob_entropy(z, ids, 1.0, 0.9)
    assert np.isfinite(lp[0]) and np.isnan(lp[1]) and np.isnan(lp[2])
    assert np.isnan(ent[1]) and np.isnan(ent[2])


def test_sampler_draws_from_the_nucleus(oracle):
    bits = _small_peaked(T=64, V=1500, seed=3)
    u = workloads.uniforms(64, seed=1)
    ids = oracle.sample_ids(bits, 0.7, 0.95, u)
    lp, ent, k, gap = oracle.logprob_entropy(bits, ids, 0.7, 0.95)
    assert np.all(np.isfinite(lp))
    # u -> 0 picks the top-ranked token (the largest logit, lowest id on ties).
    first = oracle.sample_ids(bits, 0.7, 0.95, np.zeros(64))
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(first, np.argmax(vals, axis=1).astype(np.int32))


@pytest.mark.parametrize("T_,p", [(1.3, 0.95), (0.7, 0.6)])
def test_sampler_frequencies_are_the_nucleus_masses(oracle, T_, p):
    """One bf16 row (ties included) drawn at N evenly spaced u: each id's share
    of the draws is its renormalised mass exp(logprob) from the scorer to within
    1/N (each id owns an interval of u of that length), 0 off the nucleus; and
    as u grows the drawn ids follow the ranking order (logit descending, lower
    id first on ties) of a library sort."""
    V, N = 300, 4000
    bits = workloads.bf16_bits(workloads.normal_logits_fp32(1, V, 2.0, seed=9).to(torch.bfloat16))[0]
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    assert len(np.unique(vals)) < V                         # the row has ties
    u = (np.arange(N) + 0.5) / N
    ids = oracle.sample_ids(np.ascontiguousarray(np.repeat(bits[None, :], N, axis=0)), T_, p, u)
    lp, _, k, _ = score_all_ids(oracle, bits, T_, p)
    q = np.where(np.isfinite(lp), np.exp(lp), 0.0)
    assert 1 < k[0] < V
    freq = np.bincount(ids, minlength=V) / N
    assert np.all(np.abs(freq - q) <= 1.0 / N + 1e-12)
    order = np.lexsort((np.arange(V), -vals.astype(np.float64)))
    rank = np.empty(V, np.int64)
    rank[order] = np.arange(V)
    assert np.all(np.diff(rank[ids]) >= 0)


def test_sampler_uniform_row_closed_form(oracle):
    """V = 32 equal logits, top_p = 1/4: the nucleus is ids 0..7 (every mass
    1/32, exact), and u in the j-th eighth draws id j."""
    rows = np.zeros((8, 32), np.float32)
    ids = oracle.sample_ids(rows, 1.0, 0.25, (np.arange(8) + 0.5) / 8)
    assert list(ids) == list(range(8))
    ids = oracle.sample_ids(rows[:2], 1.0, 0.25, np.array([0.0, 0.999999]))
    assert list(ids) == [0, 7]
    # u on a boundary: the cumulative mass of ids 0..2 is exactly 3/8, so
    # u = 3/8 is reached at id 2 (the first token whose cumulative reaches u)
    ids = oracle.sample_ids(rows[:3], 1.0, 0.25, np.array([1 / 8, 3 / 8, 7 / 8]))
    assert list(ids) == [0, 2, 6]


# --------------------------------------------------------------------------
# GRPO / DAPO loss: hand-worked values.
# --------------------------------------------------------------------------

def test_advantages_hand_and_library(oracle):
    R = np.array([1, 0, 0, 1, 1, 1, 1, 1, 0.5, 0.0, 2.0, 1.5], np.float32)
    off = np.arange(13, dtype=np.int32)   # one token per sequence
    z = np.zeros(12, np.float32)
    _, _, adv, _ = oracle.grpo_loss(z, z, z, z, None, R, off, 4)
    sigma = math.sqrt(1.0 / 3.0)          # [1,0,0,1]: mean 0.5, sum sq 1, /(G-1)=1/3
    assert abs(adv[0] - 0.5 / (sigma + 1e-6)) < 1e-12
    assert abs(adv[1] + 0.5 / (sigma + 1e-6)) < 1e-12
    assert abs(adv[0] - 0.866024) < 1e-6
    assert np.all(adv[4:8] == 0.0)        # degenerate group: A = 0
    for g in range(3):
        r = R[4 * g:4 * g + 4].astype(np.float64)
        ref = (r - r.mean()) / (np.std(r, ddof=1) + 1e-6)
        assert np.max(np.abs(adv[4 * g:4 * g + 4] - ref)) < 1e-12


def test_clipped_ratio_tis_k3_hand_values(oracle):
    # Group [1,0,0,1]; four one-token sequences.  A = +a, -a, -a, +a.
    a = 0.5 / (math.sqrt(1.0 / 3.0) + 1e-6)
    ln15 = f32(math.log(1.5))
    r15 = math.exp(ln15)                          # the ratio the float inputs give
    ln07 = f32(math.log(0.7))
    new = np.array([ln15, ln15, ln07, 0.0], np.float32)
    old = np.zeros(4, np.float32)
    ro = np.array([0.0, 0.0, 0.0, f32(-math.log(3.0))], np.float32)   # old - rollout = ln 3
    ref = np.array([ln15, ln15 + f32(0.1), ln07, 0.0], np.float32)
    R = np.array([1, 0, 0, 1], np.float32)
    off = np.arange(5, dtype=np.int32)
    loss, grad, adv, st = oracle.grpo_loss(new, old, ro, ref, None, R, off, 4,
                                           0.2, 0.28, 2.0, 0.01)
    # token 0: r = 1.5 > 1.28, A > 0 -> clipped term active: pg = -1.28 a, grad_pg = 0.
    pg0 = -(1.0 + f32(0.28)) * a
    # token 1: r = 1.5, A < 0 -> unclipped -r A is larger: pg = r a.
    pg1 = r15 * a
    # token 2: r = 0.7 < 0.8, A < 0 -> clipped at 1 - 0.2: pg = 0.8 a.
    pg2 = (1.0 - f32(0.2)) * a
    # token 3: r = 1, A > 0 -> pg = -a; TIS weight exp(ln 3) = 3 capped to 2.
    pg3 = -a
    d1 = float(ref[1]) - float(new[1])                     # delta = ref - new (in double)
    k3_1 = math.exp(d1) - d1 - 1.0
    assert abs(k3_1 - 0.0051709) < 1e-6
    beta = f32(0.01)                                       # kl_coef as the float received
    ell = [pg0, pg1 + beta * k3_1, pg2, 2.0 * pg3]
    assert abs(pg0 + 1.108511) < 1e-5 and abs(pg1 - 1.299036) < 1e-5
    assert abs(pg2 - 0.692819) < 1e-5
    assert abs(loss - math.fsum(ell) / 4.0) < 1e-12
    # dL/dnew: token0 clipped -> 0; token1 -r A = r a; token2 clipped -> 0;
    # token3 unclipped: w (-r A) = 2 (-a).
    g = [0.0, r15 * a + beta * (1.0 - math.exp(d1)), 0.0, 2.0 * (-a)]
    assert np.max(np.abs(grad - np.array(g) / 4.0)) < 1e-12
    assert st["clip_high_frac"] == 0.25 and st["clip_low_frac"] == 0.25
    assert st["tis_capped_frac"] == 0.25 and abs(st["tis_mean"] - 1.25) < 1e-12
    assert st["tokens"] == 4.0


def test_k3_and_degenerate_group(oracle):
    new = np.array([0.0, -0.5, -1.0], np.float32)
    ref = new.copy()
    R = np.ones(3, np.float32)
    off = np.array([0, 1, 2, 3], np.int32)
    loss, grad, adv, st = oracle.grpo_loss(new, new, new, ref, None, R, off, 3)
    assert loss == 0.0 and np.all(adv == 0.0) and np.all(grad == 0.0)


def test_mask_and_empty(oracle):
    new = np.array([0.1, 0.2, 0.3, 0.4], np.float32)
    R = np.array([1, 0], np.float32)
    off = np.array([0, 2, 4], np.int32)
    m0 = np.zeros(4, np.uint8)
    loss, grad, _, st = oracle.grpo_loss(new, new, new, new, m0, R, off, 2)
    assert loss == 0.0 and np.all(grad == 0.0) and st["tokens"] == 0.0
    m = np.array([1, 0, 0, 1], np.uint8)
    full, _, _, _ = oracle.grpo_loss(new, new, new, new, None, R, off, 2)
    part, g, _, _ = oracle.grpo_loss(new, new, new, new, m, R, off, 2)
    # r = 1, w = 1, k3 = 0 everywhere: l = -A; A = +a for seq 0, -a for seq 1.
    a = 0.5 / (math.sqrt(0.5) + 1e-6)
    assert abs(part - (-a + a) / 2) < 1e-12
    assert g[1] == 0.0 and g[2] == 0.0


def test_seq_mean_aggregation_hand(oracle):
    # Two groups of one sequence each (G = 1 -> A = 0), lengths 1 and 3; only KL.
    new = np.zeros(4, np.float32)
    ref = np.array([0.1, 0.0, 0.2, -0.3], np.float32)
    off = np.array([0, 1, 4], np.int32)
    R = np.zeros(2, np.float32)
    k3 = [math.exp(float(d)) - float(d) - 1.0 for d in ref.astype(np.float64)]
    loss, _, _, _ = oracle.grpo_loss(new, new, new, ref, None, R, off, 1, kl_coef=0.5, agg=1)
    expect = 0.5 * (k3[0] + (k3[1] + k3[2] + k3[3]) / 3.0) / 2.0
    assert abs(loss - expect) < 1e-12
    loss0, _, _, _ = oracle.grpo_loss(new, new, new, ref, None, R, off, 1, kl_coef=0.5, agg=0)
    assert abs(loss0 - 0.5 * math.fsum(k3) / 4.0) < 1e-12


@pytest.mark.parametrize("agg", [0, 1])
def test_grad_matches_finite_differences(oracle, agg):
    rng = np.random.default_rng(7)
    off = np.array([0, 5, 9, 16, 20], np.int32)
    n = 20
    grid = 1.0 / 256.0
    new = (rng.integers(-200, 0, n) * grid).astype(np.float32)
    old = new + (rng.integers(-30, 30, n) * grid).astype(np.float32)
    ro = old + (rng.integers(-60, 60, n) * grid).astype(np.float32)
    ref = new + (rng.integers(-20, 20, n) * grid).astype(np.float32)
    R = np.array([1.0, 0.0, 0.3, 0.9], np.float32)
    mask = (rng.random(n) < 0.8).astype(np.uint8)
    kw = dict(eps_low=0.2, eps_high=0.28, tis_cap=2.0, kl_coef=0.05, agg=agg)
    _, grad, _, _ = oracle.grpo_loss(new, old, ro, ref, mask, R, off, 2, **kw)
    h = np.float32(2.0 ** -12)
    for t in range(n):
        up, dn = new.copy(), new.copy()
        up[t] += h
        dn[t] -= h
        lu = oracle.grpo_loss(up, old, ro, ref, mask, R, off, 2, **kw)[0]
        ld = oracle.grpo_loss(dn, old, ro, ref, mask, R, off, 2, **kw)[0]
        fd = (lu - ld) / (2 * float(h))
        assert abs(fd - grad[t]) < 2e-5, (t, fd, grad[t])


# --------------------------------------------------------------------------
# LM-head rows.
# --------------------------------------------------------------------------

def test_lmhead_rows_against_library_matmul(oracle):
    hidden, w, ids = workloads.lmhead_inputs(T=6, H=64, V=300, seed=4)
    hb, wb = workloads.bf16_bits(hidden), workloads.bf16_bits(w)
    rows = np.array([0, 2, 5], np.int64)
    lp, ent, k = oracle.lmhead_rows(hb, wb, rows, ids.numpy(), 0.7, 1.0)
    logits = (hidden.double() @ w.double().T) / f32(0.7)
    ref_lp = torch.log_softmax(logits, 1)
    ref_ent = torch.special.entr(torch.softmax(logits, 1)).sum(1)
    for j, r in enumerate(rows):
        assert abs(lp[j] - ref_lp[r, ids[r].long()].item()) < 1e-10
        assert abs(ent[j] - ref_ent[r].item()) < 1e-10
    assert np.all(k == 300)


# --------------------------------------------------------------------------
# The supplied-support scorer (retained set given by the sampler as a list).

def _nucleus_lists(hz, k):
    """The oracle's ranking (z descending, id ascending; -0 == +0) cut at k*."""
    vals = (hz.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return [np.lexsort((np.arange(vals.shape[1]), -vals[r]))[:k[r]] for r in range(vals.shape[0])]


@pytest.mark.parametrize("T,p", [(0.7, 0.5), (0.7, 0.95), (1.8, 0.95), (0.2, 0.9)])
def test_support_equals_topp_nucleus(oracle, T, p):
    """Given the top-p nucleus as its retained set -- in rank order or shuffled --
    the supplied-support scorer reproduces the top-p scorer."""
    z, _ = workloads.peaked_bf16(8, V=3000, seed=12)
    hz = workloads.bf16_bits(z)
    ids = oracle.sample_ids(hz, T, p, workloads.uniforms(8, 3))
    lp, ent, k, _ = oracle.logprob_entropy(hz, ids, T, p)
    lists = _nucleus_lists(hz, k)
    rng = np.random.default_rng(5)
    for shuffle in (False, True):
        ls = [rng.permutation(l) if shuffle else l for l in lists]
        off = np.concatenate([[0], np.cumsum([len(l) for l in ls])]).astype(np.int64)
        sup = np.concatenate(ls).astype(np.int32)
        slp, sent, st = oracle.logprob_entropy_support(hz, ids, T, off, sup)
        assert np.all(st == 0)
        assert np.allclose(slp, lp, rtol=0, atol=1e-11)
        assert np.allclose(sent, ent, rtol=0, atol=1e-11)
    # an id outside the nucleus scores -inf on both
    far = ((ids.astype(np.int64) + 1500) % 3000).astype(np.int32)
    lp2, _, _, _ = oracle.logprob_entropy(hz, far, T, p)
    off = np.concatenate([[0], np.cumsum([len(l) for l in lists])]).astype(np.int64)
    slp2, _, _ = oracle.logprob_entropy_support(hz, far, T, off, np.concatenate(lists).astype(np.int32))
    assert np.array_equal(np.isneginf(slp2), np.isneginf(lp2))


def test_support_closed_forms(oracle):
    V, T = 64, 0.7
    z = np.zeros((3, V), np.float32)
    z[1, :10] = 2.0          # two levels: 10 tokens at 2.0, the rest at 0.0
    z[2] = np.linspace(-3, 3, V, dtype=np.float32)
    # row 0: uniform logits, a support of k = 7 ids -> logprob -ln 7, H = ln 7
    s0 = np.array([3, 9, 11, 20, 33, 40, 63], np.int32)
    # row 1: 4 ids at 2.0 and 6 ids at 0.0
    s1 = np.array([0, 1, 2, 3, 30, 31, 32, 33, 34, 35], np.int32)
    # row 2: a single listed id -> logprob 0, H 0
    s2 = np.array([17], np.int32)
    off = np.array([0, 7, 17, 18], np.int64)
    ids = np.array([11, 31, 17], np.int32)
    lp, ent, st = oracle.logprob_entropy_support(z, ids, T, off, np.concatenate([s0, s1, s2]))
    assert np.all(st == 0)
    assert lp[0] == pytest.approx(-math.log(7), abs=1e-14)
    assert ent[0] == pytest.approx(math.log(7), abs=1e-14)
    a = math.exp(2.0 / float(np.float32(T)))   # the float32 temperature, widened
    Zs = 4 * a + 6
    q_hi, q_lo = a / Zs, 1 / Zs
    assert lp[1] == pytest.approx(math.log(q_lo), abs=1e-13)
    assert ent[1] == pytest.approx(-(4 * q_hi * math.log(q_hi) + 6 * q_lo * math.log(q_lo)), abs=1e-13)
    assert lp[2] == 0.0 and ent[2] == 0.0
    # shift invariance
    lp_s, ent_s, _ = oracle.logprob_entropy_support(z + np.float32(5.0), ids, T, off,
                                                    np.concatenate([s0, s1, s2]))
    assert np.allclose(lp_s, lp, atol=1e-12) and np.allclose(ent_s, ent, atol=1e-12)


def test_support_errors(oracle):
    V = 16
    z = np.zeros((5, V), np.float32)
    z[3, 2] = np.nan          # listed non-finite logit
    z[4, 9] = np.inf          # unlisted non-finite logit: not examined
    off = np.array([0, 0, 2, 4, 6, 8], np.int64)          # row 0: empty list
    sup = np.array([1, 16,  1, 2,  1, 2,  1, 2], np.int32)  # row 1: id 16 out of range
    ids = np.array([0, 1, 99, 1, 1], np.int32)             # row 2: selected id out of range
    lp, ent, st = oracle.logprob_entropy_support(z, ids, 1.0, off, sup)
    assert list(st) == [8, 8, 1, 2, 0]
    assert np.all(np.isnan(lp[:4])) and np.all(np.isnan(ent[:4]))
    assert lp[4] == pytest.approx(-math.log(2)) and ent[4] == pytest.approx(math.log(2))
    # offsets that decrease
    lp, ent, st = oracle.logprob_entropy_support(z[:2], ids[:2], 1.0,
                                                 np.array([0, 3, 1], np.int64), sup[:3])
    assert st[1] == 8 and np.isnan(lp[1])


def test_support_backward_matches_finite_differences(oracle):
    """The supplied-support gradient against central differences of the
    (pinned) supplied-support forward, sets held fixed; plus the shift
    invariance sum_j grad_j = 0 and the uniform closed form."""
    rng = np.random.default_rng(9)
    V, R, T = 12, 4, 0.7
    z = rng.normal(0, 1.5, (R, V)).astype(np.float32)
    lists = [np.array([0, 3, 5, 7, 11]), np.array([2, 4]), np.array([1, 6, 8, 9, 10, 3]),
             np.array([0, 1, 2])]
    ids = np.array([5, 4, 9, 7], np.int32)          # row 3: y not listed
    off = np.concatenate([[0], np.cumsum([len(l) for l in lists])]).astype(np.int64)
    sup = np.concatenate(lists).astype(np.int32)
    gl = rng.normal(0, 1, R).astype(np.float32)
    gh = rng.normal(0, 1, R).astype(np.float32)
    g = oracle.logprob_entropy_support_backward(z, ids, T, off, sup, gl, gh)

    def loss(zz):
        lp, ent, _ = oracle.logprob_entropy_support(zz, ids, T, off, sup)
        lp = np.where(np.isneginf(lp), 0.0, lp)       # y not listed: no log-prob term
        return gl.astype(np.float64) * lp + gh.astype(np.float64) * ent

    for r in range(R):
        for jj, i in enumerate(lists[r]):
            zp, zm = z.copy(), z.copy()
            zp[r, i] = np.float32(z[r, i] + 1e-3)
            zm[r, i] = np.float32(z[r, i] - 1e-3)
            h = float(zp[r, i]) - float(zm[r, i])
            fd = (loss(zp)[r] - loss(zm)[r]) / h
            assert g[off[r] + jj] == pytest.approx(fd, abs=2e-6)
        assert abs(g[off[r]:off[r + 1]].sum()) < 1e-12
    # uniform logits over k listed ids: the entropy part vanishes
    zu = np.zeros((1, V), np.float32)
    lst = np.array([2, 5, 9], np.int32)
    gu = oracle.logprob_entropy_support_backward(zu, np.array([5], np.int32), T,
                                                 np.array([0, 3], np.int64), lst,
                                                 np.array([1.5], np.float32), np.array([2.0], np.float32))
    T32 = float(np.float32(T))
    assert np.allclose(gu, [1.5 / T32 * (0 - 1 / 3), 1.5 / T32 * (1 - 1 / 3), 1.5 / T32 * (0 - 1 / 3)],
                       atol=1e-14)


def _dense_loss(oracle, z, ids, T, p, gl, gh):
    lp, ent, k, _ = oracle.logprob_entropy(z, ids, T, p)
    lp = np.where(np.isneginf(lp), 0.0, lp)           # y outside S: no log-prob term
    return gl.astype(np.float64) * lp + gh.astype(np.float64) * ent, k


@pytest.mark.parametrize("p", [0.5, 0.8, 1.0])
def test_dense_backward_matches_finite_differences(oracle, p):
    """The dense top-p gradient against central differences of the (pinned)
    forward wherever a step of +-1e-3 leaves k* alone: members and non-members
    alike (non-members must come out exactly 0)."""
    rng = np.random.default_rng(21)
    V, R, T = 16, 6, 0.8
    # distinct values 0.07 apart, so a 1e-3 step never reorders the ranking
    z = np.stack([rng.permutation(np.arange(V) * 0.07 * 3) for _ in range(R)]).astype(np.float32)
    ids = rng.integers(0, V, R).astype(np.int32)
    gl = rng.normal(0, 1, R).astype(np.float32)
    gh = rng.normal(0, 1, R).astype(np.float32)
    g = oracle.logprob_entropy_backward(z, ids, T, p, gl, gh)
    base, k0 = _dense_loss(oracle, z, ids, T, p, gl, gh)
    checked = 0
    for r in range(R):
        for i in range(V):
            zp, zm = z.copy(), z.copy()
            zp[r, i] = np.float32(z[r, i] + 1e-3)
            zm[r, i] = np.float32(z[r, i] - 1e-3)
            lp_, kp = _dense_loss(oracle, zp, ids, T, p, gl, gh)
            lm_, km = _dense_loss(oracle, zm, ids, T, p, gl, gh)
            if kp[r] != k0[r] or km[r] != k0[r]:
                continue                                # the step moved the boundary
            fd = (lp_[r] - lm_[r]) / (float(zp[r, i]) - float(zm[r, i]))
            assert g[r, i] == pytest.approx(fd, abs=2e-6)
            checked += 1
        assert abs(g[r].sum()) < 1e-12                  # shift invariance
    assert checked >= R * V * 3 // 4


def test_dense_backward_top_p_one_is_softmax_gradient(oracle):
    """top_p = 1, entropy weight 0: grad = g (onehot(y) - softmax(z / T)) / T,
    the softmax from the library."""
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    T = 0.7
    z = rng.normal(0, 2, (5, 300)).astype(np.float32)
    ids = rng.integers(0, 300, 5).astype(np.int32)
    gl = rng.normal(0, 1, 5).astype(np.float32)
    g = oracle.logprob_entropy_backward(z, ids, T, 1.0, gl, None)
    T32 = float(np.float32(T))
    q = softmax(z.astype(np.float64) / T32, axis=1)
    onehot = np.zeros_like(q)
    onehot[np.arange(5), ids] = 1.0
    assert np.allclose(g, gl[:, None].astype(np.float64) * (onehot - q) / T32, atol=1e-14)


def test_dense_backward_equals_support_backward_on_the_nucleus(oracle):
    """Restricted to its nucleus (found here by an independent sort), the
    dense gradient is the supplied-support gradient of that set; elsewhere 0.
    bf16 logits with many ties, so the id order inside the boundary value
    matters."""
    rng = np.random.default_rng(8)
    R, V, T, p = 6, 3000, 0.7, 0.9
    # a 0.25 grid: every value is shared by dozens of ids
    z = torch.from_numpy(np.round(rng.normal(0, 1, (R, V)) * 4).astype(np.float32) / 4).to(
        torch.bfloat16)
    hz = z.view(torch.int16).numpy().view(np.uint16)
    vals = (hz.astype(np.uint32) << 16).view(np.float32)
    ids = rng.integers(0, V, R).astype(np.int32)
    gl = rng.normal(0, 1, R).astype(np.float32)
    gh = rng.normal(0, 1, R).astype(np.float32)
    _, _, k, gap = oracle.logprob_entropy(hz, ids, T, p)
    g = oracle.logprob_entropy_backward(hz, ids, T, p, gl, gh)
    lists = [np.lexsort((np.arange(V), -vals[r]))[:k[r]] for r in range(R)]
    off = np.concatenate([[0], np.cumsum([len(l) for l in lists])]).astype(np.int64)
    sup = np.concatenate(lists).astype(np.int32)
    gs = oracle.logprob_entropy_support_backward(hz, ids, T, off, sup, gl, gh)
    for r in range(R):
        want = np.zeros(V)
        want[lists[r]] = gs[off[r]:off[r + 1]]
        assert np.allclose(g[r], want, rtol=1e-12, atol=1e-15)
        t = vals[r][lists[r][-1]]
        kept = (vals[r][lists[r]] == t).sum()
        assert 0 < kept < (vals[r] == t).sum()          # the boundary value's ties are split


def test_dense_backward_bad_rows_are_nan(oracle):
    z = np.zeros((3, 10), np.float32)
    z[1, 4] = np.inf
    g = oracle.logprob_entropy_backward(z, np.array([0, 1, 10], np.int32), 1.0, 0.9,
                                        np.ones(3, np.float32), np.ones(3, np.float32))
    assert np.all(np.isfinite(g[0])) and np.all(np.isnan(g[1])) and np.all(np.isnan(g[2]))


# ---------------------------------------------------------------- loss variants
GOLDEN = __import__("pathlib").Path(__file__).parent / "golden"


def _loss_batch(seed=3, n_prompts=4, group=4, lo=5, hi=40):
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi, n_prompts * group)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(off[-1])
    new = np.log(rng.uniform(0.05, 0.95, T)).astype(np.float32)
    old = (new + rng.normal(0, 0.2, T)).astype(np.float32)
    ro = (old + rng.normal(0, 0.3, T)).astype(np.float32)
    rf = (new + rng.normal(0, 0.1, T)).astype(np.float32)
    mask = (rng.uniform(size=T) > 0.15).astype(np.uint8)
    rew = rng.integers(0, 2, n_prompts * group).astype(np.float32)
    return new, old, ro, rf, mask, rew, off, group


def test_policy_loss_default_config_equals_grpo_loss(oracle):
    """Two independently written oracles: the variant loss at DAPO + TIS + mean
    baseline equals the GRPO/DAPO loss, for both of its aggregations."""
    new, old, ro, rf, mask, rew, off, G = _loss_batch()
    for agg in (0, 1):
        a = oracle.grpo_loss(new, old, ro, rf, mask, rew, off, G, agg=agg)
        b = oracle.policy_loss(new, old, ro, rf, mask, rew, off, G, agg=agg)
        assert b[0] == pytest.approx(a[0], rel=1e-12, abs=1e-15)
        assert np.allclose(b[1], a[1], rtol=1e-12, atol=1e-16)
        assert np.allclose(b[2], a[2], rtol=1e-12)
        for k, v in a[3].items():
            assert b[3][k] == pytest.approx(v, rel=1e-12, abs=1e-15)
        assert b[3]["mask_dropped"] == 0.0


def test_ipo_mask_on_the_pages_example(oracle):
    """The IPO mask keeps the rare token that moved 6x and masks the likely
    token that moved to 0.22x (tests/golden/ipo_mask_example.txt)."""
    rows = [l.split() for l in (GOLDEN / "ipo_mask_example.txt").read_text().splitlines()
            if l.strip() and not l.startswith("#")]
    for pi_inf, pi_tr, masked, ratio in rows:
        lp_tr = np.log(np.float32(pi_tr))
        lp_inf = np.log(np.float32(pi_inf))
        z = np.array([lp_tr], np.float32)
        _, g, _, st = oracle.policy_loss(z, z, np.array([lp_inf], np.float32), z, None,
                                         np.array([1.0], np.float32), [0, 1], 1,
                                         loss_type=oracle.LOSS_IPO, kl_coef=0.0,
                                         is_method=oracle.IS_NONE)
        assert st["mask_dropped"] == float(masked)
        assert float(np.exp(np.float64(lp_tr) - np.float64(lp_inf))) == pytest.approx(
            float(ratio), rel=1e-6)


def test_ipo_and_icepop_hand_values(oracle):
    """Two one-token sequences in one group, rewards 1 and 0: A = +-0.5 /
    (0.7071068 + 1e-6).  IPO (eps 0.3, no KL, no weight): the first token
    (0.5 vs 0.1) is masked, the second (0.5 vs 0.4) gives -1.25 A.  IcePop
    (band [0.5, 2]): rho = 5 is dropped, rho = 1.25 keeps the clipped term."""
    A = 0.5 / (np.sqrt(0.5) + 1e-6)
    new = np.log(np.array([0.5, 0.5], np.float32))
    ro = np.log(np.array([0.1, 0.4], np.float32))
    rho2 = float(np.exp(np.float64(new[1]) - np.float64(ro[1])))
    L, g, adv, st = oracle.policy_loss(new, new, ro, new, None, np.array([1, 0], np.float32),
                                       [0, 1, 2], 2, loss_type=oracle.LOSS_IPO, kl_coef=0.0,
                                       is_method=oracle.IS_NONE)
    assert adv == pytest.approx([A, -A], rel=1e-12)
    assert L == pytest.approx(0.5 * rho2 * A, rel=1e-12)
    assert g == pytest.approx([0.0, 0.5 * rho2 * A], rel=1e-12)
    assert st["mask_dropped"] == 0.5
    # IcePop: old = new, so r = 1 and the clipped term is -A; rho1 = 5 leaves the band
    L2, g2, _, st2 = oracle.policy_loss(new, new, ro, new, None, np.array([1, 0], np.float32),
                                        [0, 1, 2], 2, loss_type=oracle.LOSS_ICEPOP,
                                        band_low=0.5, band_high=2.0, kl_coef=0.0,
                                        is_method=oracle.IS_NONE)
    assert L2 == pytest.approx(0.5 * A, rel=1e-12)          # only the second: -(1)(-A)
    assert g2 == pytest.approx([0.0, 0.5 * A], rel=1e-12)
    assert st2["mask_dropped"] == 0.5


def test_mis_normalises_and_is_scale_invariant(oracle):
    """MIS: w = ratio / mean ratio.  Equal ratios give the unweighted loss;
    multiplying every ratio by one constant changes nothing."""
    new, old, ro, rf, mask, rew, off, G = _loss_batch(seed=5)
    flat = (old - np.float32(0.25)).astype(np.float32)       # every ratio exp(0.25)
    a = oracle.policy_loss(new, old, flat, rf, mask, rew, off, G, is_method=oracle.IS_MIS)
    b = oracle.policy_loss(new, old, flat, rf, mask, rew, off, G, is_method=oracle.IS_NONE)
    assert a[0] == pytest.approx(b[0], rel=1e-6)
    c = oracle.policy_loss(new, old, ro, rf, mask, rew, off, G, is_method=oracle.IS_MIS)
    d = oracle.policy_loss(new, old, (ro - np.float32(0.5)).astype(np.float32), rf, mask, rew,
                           off, G, is_method=oracle.IS_MIS)
    assert c[0] == pytest.approx(d[0], rel=1e-5)
    assert c[3]["tis_mean"] == pytest.approx(1.0, rel=1e-12)   # the weights average to 1


def test_length_weighted_baseline_and_prompt_mean(oracle):
    """Lengths 1 and 3, rewards 1 and 0: b = 0.25, sigma = 0.7071068, so
    A = 0.75 / (sigma + 1e-6) and -0.25 / (sigma + 1e-6); rewards 0 and 1:
    b = 0.75.  Prompt mean with one
    group is the token mean; with groups of one it is the sequence mean."""
    z = np.log(np.full(4, 0.5, np.float32))
    _, _, adv, _ = oracle.policy_loss(z, z, z, z, None, np.array([1, 0], np.float32),
                                      [0, 1, 4], 2, baseline=oracle.BASELINE_LENGTH_WEIGHTED)
    s = np.sqrt(0.5) + 1e-6
    assert adv == pytest.approx([0.75 / s, -0.25 / s], rel=1e-12)
    # rewards 0 and 1 on lengths 1 and 3: b = (1 * 0 + 3 * 1) / 4 = 0.75 (the
    # unweighted sum of rewards over the total length would give 0.25)
    _, _, adv, _ = oracle.policy_loss(z, z, z, z, None, np.array([0, 1], np.float32),
                                      [0, 1, 4], 2, baseline=oracle.BASELINE_LENGTH_WEIGHTED)
    assert adv == pytest.approx([-0.75 / s, 0.25 / s], rel=1e-12)
    new, old, ro, rf, mask, rew, off, G = _loss_batch(seed=7)
    n = len(rew)
    tok = oracle.policy_loss(new, old, ro, rf, mask, rew, off, n, agg=0)
    one = oracle.policy_loss(new, old, ro, rf, mask, rew, off, n, agg=2)
    assert one[0] == pytest.approx(tok[0], rel=1e-12) and np.allclose(one[1], tok[1], rtol=1e-12)
    seq = oracle.policy_loss(new, old, ro, rf, mask, rew, off, 1, agg=1)
    per = oracle.policy_loss(new, old, ro, rf, mask, rew, off, 1, agg=2)
    assert per[0] == pytest.approx(seq[0], rel=1e-12) and np.allclose(per[1], seq[1], rtol=1e-12)


@pytest.mark.parametrize("cfg", [
    dict(loss_type=0, is_method=2, agg=2),
    dict(loss_type=1, is_method=0, kl_coef=0.0, agg=0),
    dict(loss_type=1, is_method=1, kl_coef=0.02, agg=1),
    dict(loss_type=2, is_method=1, band_low=0.6, band_high=1.8, agg=2, baseline=1),
])
def test_policy_loss_gradient_matches_finite_differences(oracle, cfg):
    """dL/dnew against central differences of the loss, skipping tokens whose
    step crosses a clip bound or a mask edge (where L is not differentiable)."""
    new, old, ro, rf, mask, rew, off, G = _loss_batch(seed=11, n_prompts=2, group=3, lo=3, hi=9)
    L0, g, _, _ = oracle.policy_loss(new, old, ro, rf, mask, rew, off, G, **cfg)
    h, checked = 1e-3, 0
    for t in range(len(new)):
        up, dn = new.copy(), new.copy()
        up[t] = np.float32(new[t] + h)
        dn[t] = np.float32(new[t] - h)
        Lp, _, _, sp = oracle.policy_loss(up, old, ro, rf, mask, rew, off, G, **cfg)
        Lm, _, _, sm = oracle.policy_loss(dn, old, ro, rf, mask, rew, off, G, **cfg)
        _, _, _, s0 = oracle.policy_loss(new, old, ro, rf, mask, rew, off, G, **cfg)
        if any(sp[k] != s0[k] or sm[k] != s0[k]
               for k in ("clip_low_frac", "clip_high_frac", "mask_dropped")):
            continue
        r = np.exp(np.float64(new[t]) - old[t])
        if abs(r - 0.8) < 2e-3 or abs(r - 1.28) < 2e-3:   # at a clip bound
            continue
        fd = (Lp - Lm) / (float(up[t]) - float(dn[t]))
        assert g[t] == pytest.approx(fd, rel=2e-4, abs=2e-7), t
        checked += 1
    assert checked >= len(new) // 2


@pytest.mark.parametrize("p", [1.0, 0.9])
def test_lmhead_backward_is_the_chain_rule(oracle, p):
    """With small dyadic bf16 inputs every logit is exact in fp32, so the
    (pinned) dense logits gradient of z = h W^T applies as is: dL/dh = dz W
    and dL/dW = dz^T h, here by library matmuls in fp64."""
    rng = np.random.default_rng(6)
    T, H, V = 5, 16, 40
    h = (rng.integers(-4, 5, (T, H)) / 4.0).astype(np.float32)     # multiples of 1/4
    w = (rng.integers(-8, 9, (V, H)) / 8.0).astype(np.float32)     # multiples of 1/8
    hb = torch.from_numpy(h).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    wb = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    z = (h.astype(np.float64) @ w.T.astype(np.float64))
    assert np.array_equal(z.astype(np.float32).astype(np.float64), z)   # exact in fp32
    ids = rng.integers(0, V, T).astype(np.int32)
    gl = rng.normal(0, 1, T).astype(np.float32)
    gh = rng.normal(0, 1, T).astype(np.float32)
    dh, dw = oracle.lmhead_backward(hb, wb, ids, 0.7, p, gl, gh)
    dz = oracle.logprob_entropy_backward(z.astype(np.float32), ids, 0.7, p, gl, gh)
    assert np.allclose(dh, dz @ w.astype(np.float64), rtol=1e-12, atol=1e-14)
    assert np.allclose(dw, dz.T @ h.astype(np.float64), rtol=1e-12, atol=1e-14)
