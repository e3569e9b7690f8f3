"""Every benchmark leg at its own workload and launch configuration (the
inputs ``bench.py`` builds, the calls it times), checked on sampled rows
against the fp64 oracle, which computes a row on its own.

The rows sampled include the first and the last, and rows on both sides of
the grid-stride boundaries of the persistent kernels on a 152-SM part (760
CTAs for the sampler, 456 for the dense backward, 2432 for the supplied-support
kernels, 4096-row chunks for the LM-head), so the state a CTA carries from one
row to the next is exercised.  Where the oracle
cannot compute one output alone (a row of dL/dW sums over all 16,384 tokens),
a property that holds at any size stands in.  Tolerances are those of the
per-leg tests.
"""
import numpy as np
import pytest
import torch

import bench
import workloads
from _parity import ENT_TOL, LP_REL, LP_TOL, check_nucleus_sizes, compare_rows
from test_backward_gpu import _check as check_dense_grad
from test_sampler_gpu import _check as check_draws

pytestmark = pytest.mark.gpu

T, V, TEMP, P = bench.T_ROWS, bench.VOCAB, bench.TEMPERATURE, bench.TOP_P
SEED = bench.rank_seed(0)


def _rows(n_ctas, extra=()):
    r = {0, 1, T - 1, n_ctas - 1, n_ctas, n_ctas + 1, 2 * n_ctas, T // 2, *extra}
    return np.array(sorted(x for x in r if 0 <= x < T), np.int64)


def _close(lp, ent, olp, oent, label):
    assert np.array_equal(np.isneginf(lp), np.isneginf(olp)), f"{label}: -inf membership"
    fin = ~np.isneginf(olp)
    assert np.all(np.abs(lp[fin] - olp[fin]) <= LP_TOL + LP_REL * np.abs(olp[fin])), label
    assert np.all(np.abs(ent - oent) <= ENT_TOL), label


@pytest.fixture(scope="module")
def batch(cuda_lib):
    z, ids = bench.make_workload(torch.device("cuda"), seed=SEED)
    st = cuda_lib.new_row_state(T, z.device)
    lp, ent, k = cuda_lib.logprob_entropy(z, ids, TEMP, P, return_nucleus_size=True, row_state=st)
    torch.cuda.synchronize()
    return z, ids, st, k.cpu().numpy().astype(np.int64)


def test_dense_backward_bench_shape(cuda_lib, oracle, batch):
    """--op backward: bf16 gradients of all 4096 rows in one call."""
    z, ids, st, k = batch
    g = torch.Generator(device="cpu").manual_seed(SEED + 2)
    glp = torch.empty(T).uniform_(-1, 1, generator=g)
    gh = torch.empty(T).uniform_(-1, 1, generator=g)
    grad = torch.empty((T, V), device="cuda", dtype=torch.bfloat16)
    cuda_lib.logprob_entropy_backward(z, ids, TEMP, st, glp.cuda(), gh.cuda(), out=grad)
    torch.cuda.synchronize()
    rows = _rows(3 * 152, extra=(455, 911, 912, 3000))
    tr = torch.from_numpy(rows).cuda()
    hz = workloads.bf16_bits(z[tr])
    check_nucleus_sizes(oracle, hz, ids.cpu().numpy()[rows], TEMP, P, k[rows])
    og = oracle.logprob_entropy_backward(hz, ids.cpu().numpy()[rows], TEMP, P,
                                         glp.numpy()[rows], gh.numpy()[rows], force_k=k[rows])
    vals = (hz.astype(np.uint32) << 16).view(np.float32)
    check_dense_grad(grad[tr], og, vals, k[rows], rel=2.0 ** -8, label="bench backward")


def test_sampler_bench_shape(cuda_lib, oracle, batch):
    """--op sample: 4096 draws from the forward's row states."""
    z, _, st, _ = batch
    g = torch.Generator(device="cpu").manual_seed(SEED + 4)
    u = torch.rand(T, generator=g)
    out = cuda_lib.sample_top_p(z, TEMP, P, u.cuda(), row_state=st)
    torch.cuda.synchronize()
    rows = _rows(5 * 152, extra=range(0, T, 97))
    hz = workloads.bf16_bits(z[torch.from_numpy(rows).cuda()])
    check_draws(hz, out.cpu().numpy()[rows], u.numpy()[rows], TEMP, P, oracle)


def _sub_csr(off, sup, rows):
    lists = [sup[off[r]:off[r + 1]] for r in rows]
    o = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int64)
    return o, np.concatenate(lists).astype(np.int32)


def test_supplied_support_bench_shape(cuda_lib, oracle, batch):
    """--op support and --op support_backward: every row's top-p set as CSR."""
    z, ids, _, _ = batch
    off, sup = bench.make_supports(z, P, TEMP)
    lp, ent = cuda_lib.logprob_entropy_support(z, ids, TEMP, off, sup)
    g = torch.Generator(device="cpu").manual_seed(SEED + 1)
    glp = torch.empty(T).uniform_(-1, 1, generator=g)
    gh = torch.empty(T).uniform_(-1, 1, generator=g)
    grad = cuda_lib.logprob_entropy_support_backward(z, ids, TEMP, off, sup, glp.cuda(), gh.cuda())
    torch.cuda.synchronize()
    rows = _rows(16 * 152, extra=range(0, T, 331))
    off_h, sup_h = off.cpu().numpy(), sup.cpu().numpy()
    o, s = _sub_csr(off_h, sup_h, rows)
    hz = workloads.bf16_bits(z[torch.from_numpy(rows).cuda()])
    idr = ids.cpu().numpy()[rows]
    olp, oent, ost = oracle.logprob_entropy_support(hz, idr, TEMP, o, s)
    assert np.all(ost == 0)
    _close(lp.cpu().numpy()[rows].astype(np.float64), ent.cpu().numpy()[rows].astype(np.float64),
           olp, oent, "bench support")
    og = oracle.logprob_entropy_support_backward(hz, idr, TEMP, o, s, glp.numpy()[rows],
                                                 gh.numpy()[rows])
    gg = np.concatenate([grad.cpu().numpy()[off_h[r]:off_h[r + 1]] for r in rows]).astype(np.float64)
    assert np.all(np.abs(gg - og) <= 2e-5 + 1e-4 * np.abs(og)), np.abs(gg - og).max()


def test_canonical_partition_bench_shape(cuda_lib, oracle, batch):
    """--op canonical: top_p = 1 over the eight virtual shards."""
    z, ids, _, _ = batch
    lp, ent = cuda_lib.logprob_entropy_canonical(z, ids, TEMP)
    torch.cuda.synchronize()
    rows = _rows(8 * 152, extra=range(0, T, 257))
    hz = workloads.bf16_bits(z[torch.from_numpy(rows).cuda()])
    olp, oent, _, _ = oracle.logprob_entropy(hz, ids.cpu().numpy()[rows], TEMP, 1.0)
    _close(lp.cpu().numpy()[rows].astype(np.float64), ent.cpu().numpy()[rows].astype(np.float64),
           olp, oent, "bench canonical")


def test_canonical_topp_bench_shape(cuda_lib, oracle, batch):
    """--op canonical_topp: top_p 0.95 over the eight virtual shards (partials,
    window counts, combine) on sampled rows, k* included; rows on both sides
    of the window kernel's grid-stride boundary (2432 CTAs, a (row, shard)
    pair each per round: 304 rows)."""
    z, ids, _, _ = batch
    lp, ent, k = cuda_lib.logprob_entropy_canonical_topp(z, ids, TEMP, P)
    torch.cuda.synchronize()
    rows = _rows(16 * 152 // 8, extra=range(0, T, 257))
    hz = workloads.bf16_bits(z[torch.from_numpy(rows).cuda()])
    compare_rows(oracle, hz, ids.cpu().numpy()[rows], TEMP, P, lp.cpu().numpy()[rows],
                 ent.cpu().numpy()[rows], k.cpu().numpy()[rows], label="bench canonical top-p")


@pytest.fixture(scope="module")
def lmhead(cuda_lib):
    hidden, w, ids = workloads.lmhead_inputs(bench.LM_T, bench.LM_H, V, seed=4, device="cuda")
    return hidden, w, ids.to(torch.int32)


def test_lmhead_forward_bench_shape(cuda_lib, oracle, lmhead):
    """--op lmhead: hidden [16384, 4096], W [151936, 4096], top_p 1; the
    forward that saves the log-normaliser gives the same bits."""
    hidden, w, ids = lmhead
    lp, ent = cuda_lib.lmhead_logprob(hidden, w, ids, TEMP)
    lse = torch.empty(bench.LM_T, device="cuda")
    lp2, ent2 = cuda_lib.lmhead_logprob(hidden, w, ids, TEMP, out_lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(lp, lp2) and torch.equal(ent, ent2)
    rows = np.array([0, 127, 128, 4095, 4096, 8191, 8192, 12287, 12288, 16383], np.int64)
    olp, oent, _ = oracle.lmhead_rows(workloads.bf16_bits(hidden), workloads.bf16_bits(w), rows,
                                      ids.cpu().numpy(), TEMP, 1.0)
    assert np.abs(lp.cpu().numpy()[rows] - olp).max() <= 2e-4
    assert np.abs(ent.cpu().numpy()[rows] - oent).max() <= 2e-4


def test_lmhead_backward_bench_shape(cuda_lib, oracle, lmhead):
    """--op lmhead_backward: dL/dhidden rows against the oracle (a row of it
    depends on its own token only); dL/dW through the identity
    <dL/dW, W> = sum_t <dL/dhidden_t, hidden_t> (both equal sum dz z over
    every token and id, whatever dz is), and the zero column sums of dL/dW
    (each token's dz sums to zero over the vocabulary), up to the bf16
    rounding of dz."""
    hidden, w, ids = lmhead
    n, H = hidden.shape
    lse = torch.empty(n, device="cuda")
    _, ent = cuda_lib.lmhead_logprob(hidden, w, ids, TEMP, out_lse=lse)
    g = torch.Generator(device="cpu").manual_seed(SEED + 3)
    glp = torch.empty(n).uniform_(-1, 1, generator=g)
    gh = torch.empty(n).uniform_(-1, 1, generator=g)
    dh, dw = cuda_lib.lmhead_backward(hidden, w, ids, TEMP, lse, ent, glp.cuda(), gh.cuda())
    torch.cuda.synchronize()
    rows = np.array([0, 4095, 4096, 16383], np.int64)
    odh, _ = oracle.lmhead_backward(workloads.bf16_bits(hidden[torch.from_numpy(rows).cuda()]),
                                    workloads.bf16_bits(w),
                                    ids.cpu().numpy()[rows], TEMP, 1.0, glp.numpy()[rows],
                                    gh.numpy()[rows])
    got = dh.double().cpu().numpy()[rows]
    err = np.linalg.norm(got - odh, axis=1)
    assert np.all(err <= 4e-3 * np.linalg.norm(odh, axis=1)), err
    # the identity ties every entry of dL/dW to the checked dL/dhidden
    lhs = (dw.double() * w.double()).sum().item()
    per_t = (dh.double() * hidden.double()).sum(1)
    rhs = per_t.sum().item()
    scale = (dh.double() * hidden.double()).abs().sum().item()
    assert abs(lhs - rhs) <= 1e-5 * scale, (lhs, rhs, scale)
    # column sums: |sum_i dW[i, k]| against sum_i |dW[i, k]|; the bf16
    # rounding of dz leaves a residual near 2^-9 |dz_t| per token, random in
    # sign, far below 2^-11 of the column's absolute sum
    csum = dw.double().sum(0).abs()
    cabs = dw.double().abs().sum(0)
    assert torch.all(csum <= 2.0 ** -11 * cabs).item(), (csum / cabs).max().item()
