"""GPU parity of rlk_policy_loss (the loss variants, through the C ABI)
against the fp64 oracle, on the same fp32 inputs: relative error <= 1e-4 on
the loss and the statistics, per-token gradients within 1e-4 of the largest
gradient magnitude (the bar of rlk_grpo_loss).  The default configuration
must reproduce rlk_grpo_loss bit for bit.
"""
import numpy as np
import pytest
import torch

from test_grpo_loss_gpu import make_batch

pytestmark = pytest.mark.gpu

REL = 1e-4


def run(rlk, off, R, new, old, ro, ref, G, mask=None, **kw):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    loss, grad, stats = rlk.policy_loss(t(new), t(old), t(ro), t(ref), t(R), t(off), G,
                                        loss_mask=None if mask is None else t(mask), **kw)
    torch.cuda.synchronize()
    return float(loss.item()), grad.cpu().numpy(), stats.cpu().numpy()


def check(oracle, rlk, off, R, new, old, ro, ref, G, mask=None, **kw):
    L, g, st = run(rlk, off, R, new, old, ro, ref, G, mask, **kw)
    oL, og, _, ost = oracle.policy_loss(new, old, ro, ref, mask, R, off, G, **kw)
    assert abs(L - oL) <= REL * max(abs(oL), 1e-6), (L, oL)
    scale = max(np.abs(og).max(), 1e-12)
    assert np.abs(g - og).max() <= REL * scale
    for i, name in enumerate(oracle.POLICY_STAT_NAMES):
        assert abs(st[i] - ost[name]) <= REL * max(abs(ost[name]), 1e-3), (name, st[i], ost[name])
    return L, oL, st


CONFIGS = [
    dict(loss_type=0, is_method=1, agg=2),                                  # DAPO, prompt mean
    dict(loss_type=0, is_method=2, agg=0),                                  # MIS
    dict(loss_type=0, is_method=0, baseline=1, agg=1),                      # length-weighted
    dict(loss_type=1, is_method=0, kl_coef=0.0, ipo_eps=0.3, agg=0),       # the pages' IPO
    dict(loss_type=1, is_method=2, kl_coef=0.01, ipo_eps=0.05, agg=2),
    dict(loss_type=2, is_method=1, band_low=0.5, band_high=2.0, agg=0),    # IcePop
    dict(loss_type=2, is_method=2, band_low=0.8, band_high=1.25, baseline=1, agg=1),
]


@pytest.mark.parametrize("cfg", CONFIGS)
def test_policy_loss_variants(cuda_lib, oracle, cfg):
    """64 prompts x group 8, lengths U{256..2048}, Bernoulli rewards; a mask
    that drops ~10 % of the tokens; ratios spread wide enough that the IPO and
    IcePop masks drop some tokens."""
    off, R, new, old, ro, ref = make_batch(64, 8, 256, 2048, seed=13)
    rng = np.random.default_rng(1)
    mask = (rng.uniform(size=new.size) > 0.1).astype(np.uint8)
    _, _, st = check(oracle, cuda_lib, off, R, new, old, ro, ref, 8, mask=mask, **cfg)
    if cfg["loss_type"] != 0:
        assert st[cuda_lib.STAT_MASK_DROPPED] > 0.0          # the mask dropped something


def test_default_config_is_grpo_loss_bitwise(cuda_lib):
    off, R, new, old, ro, ref = make_batch(16, 4, 10, 300, seed=2)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    for agg in (0, 1, 2):
        a = cuda_lib.grpo_loss(t(new), t(old), t(ro), t(ref), t(R), t(off), 4, agg=agg)
        b = cuda_lib.policy_loss(t(new), t(old), t(ro), t(ref), t(R), t(off), 4, agg=agg)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        assert torch.equal(a[2], b[2][:cuda_lib.NSTATS])


def test_prompt_mean_edge_cases(cuda_lib, oracle):
    """Groups whose tokens are all masked (they drop out of the mean), empty
    sequences, G = 1, and a repeat that must give the same bits."""
    off, R, new, old, ro, ref = make_batch(6, 3, 0, 20, seed=4)
    mask = np.ones(new.size, np.uint8)
    mask[off[0]:off[3]] = 0                                # the first group: nothing counts
    for G in (3, 1):
        check(oracle, cuda_lib, off, R, new, old, ro, ref, G, mask=mask, agg=2, is_method=2)
        L, g, _ = run(cuda_lib, off, R, new, old, ro, ref, G, mask=mask, agg=2, is_method=2)
        L2, g2, _ = run(cuda_lib, off, R, new, old, ro, ref, G, mask=mask, agg=2, is_method=2)
        assert L == L2 and np.array_equal(g, g2)
    # nothing counts at all: loss 0, gradient 0
    L, g, _ = run(cuda_lib, off, R, new, old, ro, ref, 3, mask=np.zeros(new.size, np.uint8),
                  agg=2, is_method=2)
    assert L == 0.0 and not np.any(g)


def test_full_size_batch_variants(cuda_lib, oracle):
    """The 591,145-token GRPO batch, no mask, through the IPO and IcePop variants."""
    off, R, new, old, ro, ref = make_batch(64, 8, 256, 2048, seed=3)
    for cfg in (CONFIGS[3], CONFIGS[5]):
        check(oracle, cuda_lib, off, R, new, old, ro, ref, 8, **cfg)
