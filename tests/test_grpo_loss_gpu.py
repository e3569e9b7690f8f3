"""GPU parity of rlk_grpo_loss (through the C ABI) against the fp64 oracle.

The loss gets the same fp32 inputs on both sides; the bar is relative error
<= 1e-4 on the loss and the statistics, and per-token gradients within
1e-4 of the largest gradient magnitude.  Results must repeat bitwise.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

REL = 1e-4


def make_batch(n_prompts, G, lo, hi, seed, cap_frac=0.05):
    off, R = workloads.grpo_batch(n_prompts, G, lo, hi, seed)
    n = int(off[-1])
    rng = np.random.default_rng(seed)
    new = np.log(rng.uniform(1e-4, 1.0, n)).astype(np.float32)
    old, ro, ref = workloads.perturbed_logps(new, seed)
    # a few tokens whose old/rollout ratio exceeds the TIS cap, and large ratios
    idx = rng.choice(n, max(1, int(cap_frac * n)), replace=False)
    ro[idx] -= np.float32(1.5)
    idx2 = rng.choice(n, max(1, int(0.05 * n)), replace=False)
    old[idx2] += rng.normal(0, 0.4, idx2.size).astype(np.float32)
    return off, R, new, old, ro, ref


def gpu_loss(rlk, off, R, new, old, ro, ref, G, mask=None, **kw):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    loss, grad, stats = rlk.grpo_loss(t(new), t(old), t(ro), t(ref), t(R), t(off), G,
                                      loss_mask=None if mask is None else t(mask), **kw)
    torch.cuda.synchronize()
    return float(loss.item()), grad.cpu().numpy(), stats.cpu().numpy()


def check(oracle, rlk, off, R, new, old, ro, ref, G, mask=None, agg=0, **kw):
    L, g, st = gpu_loss(rlk, off, R, new, old, ro, ref, G, mask, agg=agg, **kw)
    oL, og, _, ost = oracle.grpo_loss(new, old, ro, ref, mask, R, off, G, agg=agg,
                                      **{k: v for k, v in kw.items()})
    assert abs(L - oL) <= REL * max(abs(oL), 1e-6), (L, oL)
    scale = max(np.abs(og).max(), 1e-12)
    assert np.abs(g - og).max() <= REL * scale
    for i, name in enumerate(rlk.STAT_NAMES):
        assert abs(st[i] - ost[name]) <= REL * max(abs(ost[name]), 1e-3), (name, st[i], ost[name])
    return L, oL


@pytest.mark.parametrize("agg", [0, 1])
def test_dapo_config_loss(cuda_lib, oracle, agg):
    """64 prompts x group 8, lengths U{256..2048}, Bernoulli rewards, eps 0.2/0.28,
    TIS cap 2.0, k3 coefficient 0.01."""
    off, R, new, old, ro, ref = make_batch(64, 8, 256, 2048, seed=3)
    L, oL = check(oracle, cuda_lib, off, R, new, old, ro, ref, 8, agg=agg, eps_low=0.2,
                  eps_high=0.28, tis_cap=2.0, kl_coef=0.01)
    print("loss", L, "oracle", oL)


def test_mask_groups_and_degenerate_cases(cuda_lib, oracle):
    off, R, new, old, ro, ref = make_batch(6, 4, 1, 40, seed=8)
    rng = np.random.default_rng(1)
    mask = (rng.random(int(off[-1])) < 0.7).astype(np.uint8)
    R[:4] = 1.0                                   # a zero-variance group
    for agg in (0, 1):
        check(oracle, cuda_lib, off, R, new, old, ro, ref, 4, mask=mask, agg=agg)
        check(oracle, cuda_lib, off, R, new, old, ro, ref, 1, mask=mask, agg=agg)   # G = 1
    zero = np.zeros_like(mask)
    L, g, st = gpu_loss(cuda_lib, off, R, new, old, ro, ref, 4, zero)
    assert L == 0.0 and not g.any() and st[1] == 0.0


def test_empty_batch(cuda_lib):
    off = np.zeros(1, np.int32)
    e = np.zeros(0, np.float32)
    L, g, st = gpu_loss(cuda_lib, off, e, e, e, e, e, 1)
    assert L == 0.0 and g.size == 0


def test_loss_bitwise_repeat(cuda_lib):
    off, R, new, old, ro, ref = make_batch(16, 8, 100, 900, seed=4)
    a = gpu_loss(cuda_lib, off, R, new, old, ro, ref, 8)
    for _ in range(2):
        b = gpu_loss(cuda_lib, off, R, new, old, ro, ref, 8)
        assert np.float32(a[0]).tobytes() == np.float32(b[0]).tobytes()
        assert a[1].tobytes() == b[1].tobytes() and a[2].tobytes() == b[2].tobytes()


def test_chained_logits_to_loss(cuda_lib, oracle):
    """Qwen3-shaped logits -> GPU log-probs -> GPU loss, against the oracle's
    log-probs -> oracle loss.  The two loss inputs differ by the log-prob
    error d_t (<= 2e-4), so the losses may differ by at most
    sum_t s_t |d_t|, s_t bounding |dL/dlogp_t| over that interval:
    (w r e^|d| |A| + beta (e^(|ref - new| + |d|) + 1)) / N (the clipped
    term's slope is r |A| or 0; k3's is 1 - e^(ref - new)); plus the loss's
    own 1e-4 relative bar."""
    off, R = workloads.grpo_batch(4, 8, 16, 96, seed=3)
    n = int(off[-1])
    z, _ = workloads.peaked_bf16(n, seed=3, device="cuda")
    hz = workloads.bf16_bits(z)
    ids_h = oracle.sample_ids(hz, 0.7, 0.95, workloads.uniforms(n, 4))
    ids = torch.from_numpy(ids_h).cuda()
    lp, _ = cuda_lib.logprob_entropy(z, ids, 0.7, 0.95)
    olp, _, _, _ = oracle.logprob_entropy(hz, ids_h, 0.7, 0.95)
    new_gpu = lp.cpu().numpy()
    new_or = olp.astype(np.float32)
    assert np.all(np.isfinite(new_or))
    old, ro, ref = workloads.perturbed_logps(new_or, 5)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    loss, _, _ = cuda_lib.grpo_loss(t(new_gpu), t(old), t(ro), t(ref), t(R), t(off), 8)
    oL, _, adv, _ = oracle.grpo_loss(new_or, old, ro, ref, None, R, off, 8)
    d = np.abs(new_gpu.astype(np.float64) - new_or)
    assert np.all(d <= 2e-4 + 2.0 ** -22 * np.abs(new_or))            # the log-prob bar
    a_tok = np.repeat(np.abs(adv), np.diff(off))
    r = np.exp(new_or.astype(np.float64) - old)
    w = np.minimum(np.exp(old.astype(np.float64) - ro), 2.0)
    s = (w * r * np.exp(d) * a_tok + 0.01 * (np.exp(np.abs(ref - new_or) + d) + 1.0)) / n
    tol = (s * d).sum() + 1e-4 * max(abs(oL), 1e-6)
    err = abs(loss.item() - oL)
    print(f"chained loss {loss.item():.6f} oracle {oL:.6f} |diff| {err:.2e} bound {tol:.2e}")
    assert err <= tol


@pytest.mark.parametrize("case", ["decreasing", "past_end", "before_base"])
def test_bad_offsets_give_nan_and_stay_in_range(cuda_lib, case):
    """seq_offsets that decrease or leave the n_tok packed tokens: the loss,
    the statistics and the gradient come out NaN, and no gradient is written
    outside the n_tok tokens (canaries on both sides of the buffer)."""
    import ctypes
    lib = cuda_lib.load()
    off, R, new, old, ro, ref = make_batch(4, 4, 8, 40, seed=23)
    n = int(off[-1])
    bad = off.copy()
    if case == "decreasing":
        bad[5] = bad[3] - 1
    elif case == "past_end":
        bad[-1] = n + 50
    else:
        bad[2] = -7
    pad = 64
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tn, to, tr, tf, tR, toff = t(new), t(old), t(ro), t(ref), t(R), t(bad)
    gbuf = torch.full((n + 2 * pad,), 12345.0, device="cuda")
    grad = gbuf[pad:pad + n]
    loss = torch.zeros(1, device="cuda")
    stats = torch.zeros(cuda_lib.NSTATS, device="cuda")
    n_seq = off.size - 1
    wsb = cuda_lib.workspace_size(1, n, n_seq)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    p = lambda x: ctypes.c_void_p(x.data_ptr())
    code = lib.rlk_grpo_loss(p(tn), p(to), p(tr), p(tf), None, p(tR), p(toff), n_seq, 4, n, 0.2,
                             0.28, 2.0, 0.01, 0, p(loss), p(grad), p(stats), p(ws), wsb,
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    assert np.isnan(loss.item())
    assert np.all(np.isnan(stats.cpu().numpy()))
    g = gbuf.cpu().numpy()
    assert np.all(g[:pad] == 12345.0) and np.all(g[pad + n:] == 12345.0)
    written = g[pad:pad + n]
    assert np.all(np.isnan(written) | (written == 12345.0))
    # the same call with valid offsets is finite again
    loss2, _, _ = cuda_lib.grpo_loss(tn, to, tr, tf, tR, t(off), 4)
    torch.cuda.synchronize()
    assert np.isfinite(loss2.item())
