"""rlk_logprob_entropy_support (retained set supplied by the sampler, CSR)
and its backward through the C ABI against the fp64 oracle.  Tolerances as for the top-p path:
|d logprob| <= 2e-4 (+ ~2 ulp of large values), |d entropy| <= 2e-4, -inf
where the oracle has -inf.  Given the top-p nucleus as its set, the supplied-
support path must also agree with rlk_logprob_entropy.
"""
import numpy as np
import pytest
import torch

import workloads
from _parity import LP_REL, LP_TOL, ENT_TOL

pytestmark = pytest.mark.gpu


def _csr(lists):
    off = np.concatenate([[0], np.cumsum([len(l) for l in lists])]).astype(np.int64)
    sup = (np.concatenate(lists) if off[-1] else np.zeros(0)).astype(np.int32)
    return off, sup


def _run(rlk, z, ids, T, off, sup, status=None):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sids = d(sup) if sup.size else torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent = rlk.logprob_entropy_support(z, d(ids), T, d(off), sids, status_word=status)
    torch.cuda.synchronize()
    return lp.cpu().numpy().astype(np.float64), ent.cpu().numpy().astype(np.float64)


def _check(lp, ent, olp, oent, label):
    inf_o, inf_g = np.isneginf(olp), np.isneginf(lp)
    assert np.array_equal(inf_o, inf_g), f"{label}: -inf membership differs"
    fin = ~inf_o
    tol = LP_TOL + LP_REL * np.abs(olp[fin])
    assert np.all(np.abs(lp[fin] - olp[fin]) <= tol), f"{label}: logprob"
    assert np.all(np.abs(ent - oent) <= ENT_TOL), f"{label}: entropy"


def _nucleus(hz, k):
    vals = (hz.astype(np.uint32) << 16).view(np.float32)
    return [np.lexsort((np.arange(vals.shape[1]), -vals[r]))[:k[r]] for r in range(vals.shape[0])]


@pytest.mark.parametrize("V", [151936, 20000])
@pytest.mark.parametrize("T,p", [(0.7, 0.95), (0.7, 0.5), (1.8, 0.95)])
def test_support_equals_topp_on_its_nucleus(cuda_lib, oracle, V, T, p):
    z, _ = workloads.peaked_bf16(48, V=V, seed=19, device="cuda")
    hz = workloads.bf16_bits(z)
    ids = oracle.sample_ids(hz, T, p, workloads.uniforms(48, 8))
    _, _, k, _ = oracle.logprob_entropy(hz, ids, T, p)
    rng = np.random.default_rng(2)
    lists = [rng.permutation(l) for l in _nucleus(hz, k)]
    off, sup = _csr(lists)
    lp, ent = _run(cuda_lib, z, ids, T, off, sup)
    olp, oent, st = oracle.logprob_entropy_support(hz, ids, T, off, sup)
    assert np.all(st == 0)
    _check(lp, ent, olp, oent, f"support V{V} T{T} p{p}")
    # the same rows through the top-p entry point
    tlp, tent = cuda_lib.logprob_entropy(z, torch.from_numpy(ids).cuda(), T, p)
    torch.cuda.synchronize()
    _check(lp, ent, tlp.cpu().numpy().astype(np.float64), tent.cpu().numpy().astype(np.float64),
           "support vs top-p")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_support_random_sets(cuda_lib, oracle, dtype):
    V, R = 30000, 40
    rng = np.random.default_rng(4)
    if dtype == "bf16":
        z, _ = workloads.peaked_bf16(R, V=V, seed=23, device="cuda")
        hz = workloads.bf16_bits(z)
    else:
        z = workloads.normal_logits_fp32(R, V, 2.0, seed=23, device="cuda")
        hz = z.cpu().numpy()
    sizes = np.concatenate([[1, 2, V], rng.integers(1, 6000, R - 3)])
    lists = [rng.choice(V, int(n), replace=False) for n in sizes]
    ids = np.array([rng.choice(l) if r % 3 else rng.integers(0, V) for r, l in enumerate(lists)],
                   np.int32)
    off, sup = _csr(lists)
    for T in (0.7, 1.0):
        lp, ent = _run(cuda_lib, z, ids, T, off, sup)
        olp, oent, st = oracle.logprob_entropy_support(hz, ids, T, off, sup)
        assert np.all(st == 0)
        _check(lp, ent, olp, oent, f"random {dtype} T{T}")


def test_support_bad_rows(cuda_lib, oracle):
    V = 5000
    z, _ = workloads.peaked_bf16(6, V=V, seed=3, device="cuda")
    z[3, 7] = float("nan")      # listed below
    z[5, 9] = float("inf")      # not listed: not read
    lists = [np.array([], np.int64), np.array([1, V]), np.array([1, 2]), np.array([7, 8]),
             np.array([4, 5]), np.array([10, 11])]
    off, sup = _csr(lists)
    ids = np.array([0, 1, 99999, 8, 4, 10], np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent = _run(cuda_lib, z, ids, 0.7, off, sup, st)
    assert np.all(np.isnan(lp[:4])) and np.all(np.isnan(ent[:4]))
    assert np.all(np.isfinite(lp[4:])) and np.all(np.isfinite(ent[4:]))
    assert int(st.item()) == (cuda_lib.STATUS_BAD_TOKEN_ID | cuda_lib.STATUS_NONFINITE |
                              cuda_lib.STATUS_BAD_SUPPORT)
    olp, oent, ost = oracle.logprob_entropy_support(workloads.bf16_bits(z), ids, 0.7, off, sup)
    assert list(ost) == [8, 8, 1, 2, 0, 0]
    _check(lp[4:], ent[4:], olp[4:], oent[4:], "good rows beside bad ones")
    # offsets that decrease
    off2 = np.array([0, 2, 1, 3], np.int64)
    st.zero_()
    lp, _ = _run(cuda_lib, z[:3].contiguous(), ids[[1, 4, 5]].copy(), 0.7, off2,
                 np.array([1, 2, 3], np.int32), st)
    assert np.isnan(lp[1]) and int(st.item()) & cuda_lib.STATUS_BAD_SUPPORT


def test_support_bitwise_batch_invariance_and_empty(cuda_lib, oracle):
    V = 151936
    z, _ = workloads.peaked_bf16(20, V=V, seed=31, device="cuda")
    hz = workloads.bf16_bits(z)
    ids = oracle.sample_ids(hz, 0.7, 0.95, workloads.uniforms(20, 6))
    _, _, k, _ = oracle.logprob_entropy(hz, ids, 0.7, 0.95)
    lists = _nucleus(hz, k)
    off, sup = _csr(lists)
    ref = _run(cuda_lib, z, ids, 0.7, off, sup)
    assert all(a.tobytes() == b.tobytes() for a, b in zip(ref, _run(cuda_lib, z, ids, 0.7, off, sup)))
    for r in (0, 7, 19):
        o1, s1 = _csr([lists[r]])
        one = _run(cuda_lib, z[r:r + 1].contiguous(), ids[r:r + 1].copy(), 0.7, o1, s1)
        assert one[0].tobytes() == ref[0][r:r + 1].tobytes()
        assert one[1].tobytes() == ref[1][r:r + 1].tobytes()
    e = torch.empty(0, V, dtype=torch.bfloat16, device="cuda")
    lp, ent = cuda_lib.logprob_entropy_support(e, torch.empty(0, dtype=torch.int32, device="cuda"),
                                               0.7, torch.zeros(1, dtype=torch.int64, device="cuda"),
                                               torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert lp.numel() == 0 and ent.numel() == 0


def _bwd(rlk, z, ids, T, off, sup, glp, gh, status=None):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g = rlk.logprob_entropy_support_backward(
        z, d(ids), T, d(off), d(sup), None if glp is None else d(glp.astype(np.float32)),
        None if gh is None else d(gh.astype(np.float32)), status_word=status)
    torch.cuda.synchronize()
    return g.cpu().numpy().astype(np.float64)


# Gradient tolerance: each component is (g_lp dlp + g_H dh) / T from float
# q_i (relative error a few ulp) and ln q_i (absolute error ~1e-6 from the
# row sums); |g| <= 3 and 1/T <= 2 keep the absolute error near 1e-5.
GRAD_ABS, GRAD_REL = 2e-5, 1e-4


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("T", [0.7, 1.0, 1.6])
def test_support_backward_matches_oracle(cuda_lib, oracle, dtype, T):
    V, R = 30000, 36
    rng = np.random.default_rng(11)
    if dtype == "bf16":
        z, _ = workloads.peaked_bf16(R, V=V, seed=41, device="cuda")
        hz = workloads.bf16_bits(z)
    else:
        z = workloads.normal_logits_fp32(R, V, 2.0, seed=41, device="cuda")
        hz = z.cpu().numpy()
    sizes = np.concatenate([[1, 2, 3000], rng.integers(1, 2500, R - 3)])
    lists = [rng.choice(V, int(n), replace=False) for n in sizes]
    ids = np.array([rng.choice(l) if r % 4 else rng.integers(0, V) for r, l in enumerate(lists)],
                   np.int32)
    off, sup = _csr(lists)
    glp = rng.uniform(-3, 3, R)
    gh = rng.uniform(-3, 3, R)
    for a, b in ((glp, gh), (glp, None), (None, gh)):
        g = _bwd(cuda_lib, z, ids, T, off, sup, a, b)
        og = oracle.logprob_entropy_support_backward(
            hz, ids, T, off, sup, np.zeros(R) if a is None else a.astype(np.float32),
            np.zeros(R) if b is None else b.astype(np.float32))
        assert np.all(np.isfinite(g))
        err = np.abs(g - og)
        assert np.all(err <= GRAD_ABS + GRAD_REL * np.abs(og)), f"max err {err.max():.3g}"


def test_support_backward_nucleus_full_vocab_and_determinism(cuda_lib, oracle):
    V, R, T, p = 151936, 24, 0.7, 0.95
    z, _ = workloads.peaked_bf16(R, V=V, seed=53, device="cuda")
    hz = workloads.bf16_bits(z)
    ids = oracle.sample_ids(hz, T, p, workloads.uniforms(R, 12))
    _, _, k, _ = oracle.logprob_entropy(hz, ids, T, p)
    lists = _nucleus(hz, k)
    lists[3] = np.arange(V)                              # a whole-vocabulary row
    off, sup = _csr(lists)
    rng = np.random.default_rng(5)
    glp, gh = rng.uniform(-1, 1, R), rng.uniform(-1, 1, R)
    g = _bwd(cuda_lib, z, ids, T, off, sup, glp, gh)
    og = oracle.logprob_entropy_support_backward(hz, ids, T, off, sup, glp.astype(np.float32),
                                                 gh.astype(np.float32))
    assert np.all(np.abs(g - og) <= GRAD_ABS + GRAD_REL * np.abs(og))
    # each row's gradient sums to zero (softmax over a fixed set)
    sums = np.add.reduceat(g, off[:-1])
    assert np.all(np.abs(sums) <= 1e-4)
    # bitwise: a repeat and each row alone give the same bits
    assert g.tobytes() == _bwd(cuda_lib, z, ids, T, off, sup, glp, gh).tobytes()
    for r in (0, 3, 23):
        o1, s1 = _csr([lists[r]])
        one = _bwd(cuda_lib, z[r:r + 1].contiguous(), ids[r:r + 1].copy(), T, o1, s1,
                   glp[r:r + 1], gh[r:r + 1])
        assert one.tobytes() == g[off[r]:off[r + 1]].tobytes()


def test_support_backward_bad_rows(cuda_lib, oracle):
    V = 5000
    z, _ = workloads.peaked_bf16(5, V=V, seed=3, device="cuda")
    z[2, 7] = float("nan")
    lists = [np.array([1, V]), np.array([1, 2]), np.array([7, 8]), np.array([4, 5]),
             np.array([10, 11, 12])]
    off, sup = _csr(lists)
    ids = np.array([1, 99999, 8, 4, 10], np.int32)
    ones = np.ones(5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = _bwd(cuda_lib, z, ids, 0.7, off, sup, ones, ones, st)
    og = oracle.logprob_entropy_support_backward(workloads.bf16_bits(z), ids, 0.7, off, sup,
                                                 ones, ones)
    assert np.all(np.isnan(g[:6])) and np.all(np.isnan(og[:6]))
    assert np.all(np.abs(g[6:] - og[6:]) <= GRAD_ABS + GRAD_REL * np.abs(og[6:]))
    assert int(st.item()) == (cuda_lib.STATUS_BAD_TOKEN_ID | cuda_lib.STATUS_NONFINITE |
                              cuda_lib.STATUS_BAD_SUPPORT)
