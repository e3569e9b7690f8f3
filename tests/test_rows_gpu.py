"""Per-row sampling parameters (rlk_logprob_entropy_rows), against the fp64
oracle row group by row group, plus the paths that read a row's temperature
from its state: the backward and the sampler.  Tolerances as for the scalar
entry points."""
import numpy as np
import pytest
import torch

import workloads
from _parity import LP_REL, LP_TOL, ENT_TOL, GAP_EXEMPT, check_nucleus_sizes

pytestmark = pytest.mark.gpu

PAIRS = [(0.2, 0.95), (0.7, 0.95), (1.0, 0.5), (1.8, 0.9), (0.7, 1.0), (1.0, 1.0)]


def _batch(V, R, seed):
    z, _ = workloads.peaked_bf16(R, V=V, seed=seed, device="cuda")
    hz = workloads.bf16_bits(z)
    pairs = np.array([PAIRS[r % len(PAIRS)] for r in range(R)], np.float32)
    return z, hz, pairs


def test_mixed_parameters_match_the_oracle(cuda_lib, oracle):
    R, V = 60, workloads.VOCAB
    z, hz, pairs = _batch(V, R, 51)
    ids = np.zeros(R, np.int32)
    for i, (T_, p) in enumerate(PAIRS):       # ids drawn from each row's own nucleus
        rows = np.arange(i, R, len(PAIRS))
        ids[rows] = oracle.sample_ids(hz[rows], T_, p, workloads.uniforms(len(rows), 3 + i))
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    lp, ent, k = cuda_lib.logprob_entropy_rows(z, d(ids), d(pairs[:, 0]), d(pairs[:, 1]),
                                               return_nucleus_size=True)
    torch.cuda.synchronize()
    lp, ent, k = lp.cpu().numpy().astype(np.float64), ent.cpu().numpy().astype(np.float64), k.cpu().numpy()
    for i, (T_, p) in enumerate(PAIRS):
        rows = np.arange(i, R, len(PAIRS))
        olp, oent, ok, gap = oracle.logprob_entropy(hz[rows], ids[rows], T_, p)
        sure = gap >= GAP_EXEMPT
        assert np.array_equal(k[rows][sure], ok[sure]), (T_, p)
        fin = sure & ~np.isneginf(olp)
        assert np.all(np.abs(lp[rows][fin] - olp[fin]) <= LP_TOL + LP_REL * np.abs(olp[fin])), (T_, p)
        assert np.all(np.abs(ent[rows][sure] - oent[sure]) <= ENT_TOL), (T_, p)


@pytest.mark.parametrize("T_,p", [(0.7, 0.95), (1.8, 1.0)])
def test_uniform_rows_equal_the_scalar_call(cuda_lib, T_, p):
    """An odd vocabulary keeps the scalar call on the per-row kernel too, so the
    bits must agree at top_p < 1 (at top_p = 1 the entropy within rounding)."""
    R, V = 24, 30011
    z, _ = workloads.peaked_bf16(R, V=V, seed=53, device="cuda")
    ids = torch.randint(0, V, (R,), dtype=torch.int32, device="cuda")
    a = cuda_lib.logprob_entropy(z, ids, T_, p)
    b = cuda_lib.logprob_entropy_rows(z, ids, torch.full((R,), T_, device="cuda"),
                                      torch.full((R,), p, device="cuda"))
    torch.cuda.synchronize()
    if p < 1.0:
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    else:   # the all-tokens branch of the top-p kernel sums the entropy in another order
        assert torch.equal(a[0], b[0])
        assert (a[1] - b[1]).abs().max().item() <= ENT_TOL


def test_bad_parameters(cuda_lib):
    R, V = 6, 5000
    z, _ = workloads.peaked_bf16(R, V=V, seed=55, device="cuda")
    ids = torch.zeros(R, dtype=torch.int32, device="cuda")
    temps = torch.tensor([0.7, 0.0, float("nan"), 0.7, -1.0, 1.0], device="cuda")
    tops = torch.tensor([0.9, 0.9, 0.9, 1.5, 0.9, 0.0], device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent = cuda_lib.logprob_entropy_rows(z, ids, temps, tops, status_word=st)
    torch.cuda.synchronize()
    assert torch.isnan(lp).cpu().tolist() == [False, True, True, True, True, True]
    assert int(st.item()) == cuda_lib.STATUS_BAD_PARAM


def test_backward_and_sampler_follow_each_rows_temperature(cuda_lib, oracle):
    R, V = 30, workloads.VOCAB
    z, hz, pairs = _batch(V, R, 57)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ids = torch.randint(0, V, (R,), dtype=torch.int32, device="cuda")
    st = cuda_lib.new_row_state(R, "cuda")
    _, _, k = cuda_lib.logprob_entropy_rows(z, ids, d(pairs[:, 0]), d(pairs[:, 1]), row_state=st,
                                            return_nucleus_size=True)
    rng = np.random.default_rng(1)
    glp, gh = rng.uniform(-1, 1, R).astype(np.float32), rng.uniform(-1, 1, R).astype(np.float32)
    # the call's temperature is a placeholder: every state carries its own
    g = cuda_lib.logprob_entropy_backward(z, ids, 1.0, st, d(glp), d(gh),
                                          grad_dtype=torch.float32)
    u = rng.uniform(0, 1, R).astype(np.float32)
    draws = cuda_lib.sample_top_p(z, 1.0, 1.0, d(u), row_state=st)
    torch.cuda.synchronize()
    g, k, draws = g.cpu().numpy().astype(np.float64), k.cpu().numpy().astype(np.int64), draws.cpu().numpy()
    idn = ids.cpu().numpy()
    for i, (T_, p) in enumerate(PAIRS):
        rows = np.arange(i, R, len(PAIRS))
        check_nucleus_sizes(oracle, hz[rows], idn[rows], T_, p, k[rows])
        og = oracle.logprob_entropy_backward(hz[rows], idn[rows], T_, p, glp[rows], gh[rows],
                                             force_k=k[rows])
        err = np.abs(g[rows] - og)
        assert np.all(err <= 2e-5 + 1e-4 * np.abs(og)), (T_, p, err.max())
        od = oracle.sample_ids(hz[rows], T_, p, u[rows].astype(np.float64))
        assert np.mean(draws[rows] == od) >= 0.8, (T_, p)   # neighbours only at cumulative ties
