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


def test_random_lmhead_shapes(cuda_lib, oracle):
    """Random LM-head shapes (T from 1 to 513 rows across 128-row tiles, H
    from 64 to 1024, V from 1 to 20,000 across 256-column tiles): the fused
    forward at top_p = 1 against the oracle on sampled rows, dL/dhidden and
    dL/dW row by row (relative 4e-3 of the row's norm, the bf16 rounding of
    dz, with an absolute floor for the all-zero gradients of V = 1), and at
    top_p < 1 the same bits as the scorer on the GEMM's own logits rounded
    to bf16."""
    rng = np.random.default_rng(41)
    for case in range(24):
        T = int(rng.choice([1, 7, 127, 128, 129, 300, 513]))
        H = int(rng.choice([64, 128, 192, 512, 1024]))
        V = int(rng.choice([1, 3, 255, 256, 257, 4097, 20000]))
        temp = float(rng.choice([0.5, 0.7, 1.0]))
        p = float(rng.choice([1.0, 1.0, 0.9]))
        g = torch.Generator().manual_seed(int(rng.integers(1 << 30)))
        hidden = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
        w = (torch.randn(V, H, generator=g) * float(rng.choice([0.02, 0.1]))).to(torch.bfloat16).cuda()
        ids = torch.randint(0, V, (T,), generator=g, dtype=torch.int32).cuda()
        label = f"case {case}: T={T} H={H} V={V} temp={temp} top_p={p}"
        lse = torch.empty(T, device="cuda") if p == 1.0 else None
        lp, ent = cuda_lib.lmhead_logprob(hidden, w, ids, temp, p, out_lse=lse)
        torch.cuda.synchronize()
        if p < 1.0:
            logits, _, _ = cuda_lib.lmhead_logits_debug(hidden, w, ids, temp)
            slp, sent = cuda_lib.logprob_entropy(logits.to(torch.bfloat16).contiguous(), ids, temp, p)
            torch.cuda.synchronize()
            assert torch.equal(slp.view(torch.int32), lp.view(torch.int32)), label
            assert torch.equal(sent.view(torch.int32), ent.view(torch.int32)), label
            continue
        hb, wb = workloads.bf16_bits(hidden), workloads.bf16_bits(w)
        rows = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, 6)])).astype(np.int64)
        olp, oent, _ = oracle.lmhead_rows(hb, wb, rows, ids.cpu().numpy(), temp, 1.0)
        glp, gent = lp.cpu().numpy()[rows], ent.cpu().numpy()[rows]
        assert np.all(np.abs(glp - olp) <= 2e-4 + 2.0 ** -22 * np.abs(olp)), label
        assert np.all(np.abs(gent - oent) <= 2e-4), label
        if T * V * H > 4e8:
            continue   # the oracle's fp64 backward is O(T V H)
        ones = torch.ones(T, device="cuda")
        dh, dw = cuda_lib.lmhead_backward(hidden, w, ids, temp, lse, ent, ones, ones)
        torch.cuda.synchronize()
        odh, odw = oracle.lmhead_backward(hb, wb, ids.cpu().numpy(), temp, 1.0,
                                          np.ones(T, np.float32), np.ones(T, np.float32))
        for name, got, want in (("dL/dhidden", dh, odh), ("dL/dW", dw, odw)):
            got = got.double().cpu().numpy()
            floor = (1e-5 * np.sqrt(np.mean(want ** 2)) + 2e-5) * np.sqrt(want.shape[1])
            err = np.linalg.norm(got - want, axis=1)
            ref = np.linalg.norm(want, axis=1)
            assert np.all(err <= 4e-3 * ref + floor), f"{label}: {name}"
