"""A seeded random sweep over the shapes and parameters the entry points
take: vocabulary sizes drawn log-uniformly from 2 to 200,000 and from a list
of step and tile boundaries (multiples of 8, 16, 256, 1024, the streaming
kernel's 14,336 and 174,080 limits and their neighbours), 1 to 40 rows,
padded strides, four temperatures, five top_p values, peaked, Gaussian,
0.25-grid and flat rows.  Each case checks

- the forward (with a row state) against the oracle, row by row;
- the sampler's three ways to a draw against each other, bit for bit, and
  their draws against the oracle's sorted inverse-CDF sampler;
- the dense backward: finite, and each row of dL/dlogits summing to zero
  (both the log-probability's and the entropy's gradient over the retained
  set do).
"""
import numpy as np
import pytest
import torch

import workloads
from _parity import compare_rows
from test_sampler_gpu import _check

pytestmark = pytest.mark.gpu

BOUNDARIES = [8, 9, 16, 17, 255, 256, 257, 1023, 1024, 1025, 2048, 2049, 8191, 8192, 8193,
              14335, 14336, 14337, 28672, 28673, 131072, 131073, 148256, 148255, 151936,
              174080, 174081]


def _case(rng):
    V = int(rng.choice(BOUNDARIES)) if rng.random() < 0.4 else \
        int(np.exp(rng.uniform(np.log(2), np.log(200000))))
    T = int(rng.choice([1, 2, 3, 5, 17, 40]))
    temp = float(rng.choice([0.5, 0.7, 1.0, 1.8]))
    p = float(rng.choice([0.5, 0.9, 0.95, 0.999, 1.0]))
    kind = str(rng.choice(["peaked", "normal", "grid", "flat"]))
    pad = int(rng.choice([0, 0, 3, 8]))
    return V, T, temp, p, kind, pad


def _rows(rng, V, T, kind, pad):
    if kind == "peaked":
        z, _ = workloads.peaked_bf16(T, V=V, seed=int(rng.integers(1 << 30)))
        z = z.float()
    else:
        scale = {"normal": 3.0, "grid": 2.0, "flat": 0.3}[kind]
        z = torch.from_numpy(rng.normal(0, scale, (T, V)).astype(np.float32))
        if kind == "grid":
            z = torch.round(z * 4) / 4
    base = torch.full((T, V + pad), -5.0)
    base[:, :V] = z
    return base.to(torch.bfloat16).cuda()[:, :V]


@pytest.mark.parametrize("seed", [11, 12, 13, 14])
def test_random_sweep(cuda_lib, oracle, seed):
    rng = np.random.default_rng(seed)
    for case in range(30):
        V, T, temp, p, kind, pad = _case(rng)
        label = f"seed {seed} case {case}: V={V} T={T} temp={temp} top_p={p} {kind} pad={pad}"
        z = _rows(rng, V, T, kind, pad)
        hz = workloads.bf16_bits(z)
        u = rng.random(T).astype(np.float32)
        ids_h = oracle.sample_ids(hz, temp, p, u.astype(np.float64)).astype(np.int32)
        ids = torch.from_numpy(ids_h).cuda()
        st = cuda_lib.new_row_state(T, z.device)
        lp, ent, k = cuda_lib.logprob_entropy(z, ids, temp, p, return_nucleus_size=True, row_state=st)
        torch.cuda.synchronize()
        lp_h = lp.cpu().numpy()
        compare_rows(oracle, hz, ids_h, temp, p, lp_h, ent.cpu().numpy(), k.cpu().numpy(), label=label)

        draws = []
        prev = cuda_lib.set_sampler_mode(1)
        try:
            for mode in (1, 0, 2):
                cuda_lib.set_sampler_mode(mode)
                draws.append(cuda_lib.sample_top_p(z, temp, p, torch.from_numpy(u).cuda(),
                                                   row_state=st).cpu().numpy())
        finally:
            cuda_lib.set_sampler_mode(prev)
        assert np.array_equal(draws[0], draws[1]) and np.array_equal(draws[0], draws[2]), label
        _check(hz, draws[0], u, temp, p, oracle)

        ones = torch.ones(T, device="cuda")
        g = cuda_lib.logprob_entropy_backward(z, ids, temp, st, ones, ones, grad_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.isfinite(g).all(), label
        fin = np.isfinite(lp_h)
        row_sum = g.double().sum(1).abs().cpu().numpy()[fin]
        row_abs = g.double().abs().sum(1).cpu().numpy()[fin]
        assert np.all(row_sum <= 1e-4 * row_abs + 2e-5), f"{label}: row sum {row_sum.max():.3e}"
