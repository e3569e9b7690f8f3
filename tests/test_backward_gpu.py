"""rlk_logprob_entropy_fwd / rlk_logprob_entropy_bwd (the dense gradient of
the top-p log-probability and entropy, retained sets held fixed) through the
C ABI against the fp64 oracle.

The forward's k* is checked against the oracle's (equal, or on rows whose
boundary gap is below rounding, one the oracle selects at a top_p within
1e-6); the oracle then evaluates each row at that k* (force_k), so both
sides hold the same set;
the set itself is checked exactly: every id outside it (found here by an
independent sort) must get a gradient of exactly 0.

Tolerance (fp32 gradients): each member's (g_lp dlp + g_H dh) / T is built
from fp32 q_i (a few ulp) and ln q_i (absolute ~1e-6 from ln Z_S), with
|g| <= 3 and 1/T <= 1.5: |d| <= 2e-5 + 1e-4 |oracle|.  bf16 gradients add
their own rounding, 2^-9 relative.
"""
import numpy as np
import pytest
import torch

import workloads
from _parity import check_nucleus_sizes

pytestmark = pytest.mark.gpu

GRAD_ABS, GRAD_REL = 2e-5, 1e-4


def _keys_sorted(vals):
    """Per row, ids in the ranking order (value descending, id ascending)."""
    V = vals.shape[1]
    return [np.lexsort((np.arange(V), -vals[r])) for r in range(vals.shape[0])]


def _run(rlk, z, ids_np, T, p, glp, gh, grad_dtype=torch.float32, out=None, status=None):
    ids = torch.from_numpy(ids_np).cuda()
    st = rlk.new_row_state(z.shape[0], z.device)
    lp, ent, k = rlk.logprob_entropy(z, ids, T, p, return_nucleus_size=True, row_state=st,
                                     status_word=status)
    d = lambda a: None if a is None else torch.from_numpy(a.astype(np.float32)).cuda()
    g = rlk.logprob_entropy_backward(z, ids, T, st, d(glp), d(gh), grad_dtype=grad_dtype, out=out,
                                     status_word=status)
    torch.cuda.synchronize()
    return g, k.cpu().numpy().astype(np.int64), st


def _check(g, og, vals, k, rows=None, rel=GRAD_REL, label=""):
    g = g.float().cpu().numpy().astype(np.float64) if torch.is_tensor(g) else g
    order = _keys_sorted(vals)
    for r in (range(g.shape[0]) if rows is None else rows):
        member = np.zeros(g.shape[1], bool)
        member[order[r][:k[r]]] = True
        assert np.all(g[r][~member] == 0.0), f"{label} row {r}: nonzero outside S"
        err = np.abs(g[r][member] - og[r][member])
        tol = GRAD_ABS + rel * np.abs(og[r][member])
        assert np.all(err <= tol), f"{label} row {r}: max err {err.max():.3g}"


def _vals(hz):
    return (hz.astype(np.uint32) << 16).view(np.float32) if hz.dtype == np.uint16 else hz


@pytest.mark.parametrize("T,p", [(0.7, 0.95), (1.0, 0.5), (1.4, 1.0)])
@pytest.mark.parametrize("V,pad", [(30011, 0), (30011, 5), (4099, 13)])
def test_backward_matches_oracle_bf16(cuda_lib, oracle, T, p, V, pad):
    """Per-row kernel shapes: odd V (ragged tail, unaligned rows) and padded
    strides on both the logits and the gradient."""
    R = 20
    rng = np.random.default_rng(7)
    z0, _ = workloads.peaked_bf16(R, V=V + pad, seed=61, device="cuda")
    z = z0[:, :V]
    hz = workloads.bf16_bits(z.contiguous())
    ids = oracle.sample_ids(hz, T, p, workloads.uniforms(R, 3))
    ids[::5] = rng.integers(0, V, len(ids[::5]))        # some ids outside the nucleus
    glp, gh = rng.uniform(-3, 3, R), rng.uniform(-3, 3, R)
    out = torch.full((R, V + 7), 123.0, device="cuda")[:, :V] if pad else None
    g, k, _ = _run(cuda_lib, z, ids, T, p, glp, gh, out=out)
    check_nucleus_sizes(oracle, hz, ids, T, p, k)
    og = oracle.logprob_entropy_backward(hz, ids, T, p, glp.astype(np.float32),
                                         gh.astype(np.float32), force_k=k)
    _check(g, og, _vals(hz), k, label=f"V{V} pad{pad}")
    if pad:
        assert torch.all(out.as_strided((R, 7), (V + 7, 1), V) == 123.0)   # padding untouched


@pytest.mark.parametrize("p", [0.95, 0.6, 1.0])
def test_backward_full_vocab_stream_rows(cuda_lib, oracle, p):
    """V = 151936 bf16: the streaming kernel's states (and the per-row
    recompute pass's), tie rows included; bf16 and fp32 gradients."""
    V, R, T = 151936, 24, 0.7
    rng = np.random.default_rng(17)
    z, _ = workloads.peaked_bf16(R, V=V, seed=71, device="cuda")
    z[3] = 0.0                                           # all equal: every tie kept or split
    z[5, :4000] = z[5, 4000:8000]                        # many duplicates near the top
    hz = workloads.bf16_bits(z)
    ids = oracle.sample_ids(hz, T, p, workloads.uniforms(R, 5))
    glp, gh = rng.uniform(-2, 2, R), rng.uniform(-2, 2, R)
    g, k, _ = _run(cuda_lib, z, ids, T, p, glp, gh)
    check_nucleus_sizes(oracle, hz, ids, T, p, k)
    og = oracle.logprob_entropy_backward(hz, ids, T, p, glp.astype(np.float32),
                                         gh.astype(np.float32), force_k=k)
    _check(g, og, _vals(hz), k, label="stream fp32 grads")
    gb, _, _ = _run(cuda_lib, z, ids, T, p, glp, gh, grad_dtype=torch.bfloat16)
    assert gb.dtype == torch.bfloat16
    # bf16 gradients are the fp32 ones rounded to nearest
    assert torch.equal(gb, g.to(torch.bfloat16))
    _check(gb, og, _vals(hz), k, rel=2.0 ** -8, label="stream bf16 grads")


@pytest.mark.parametrize("p", [0.9, 1.0])
def test_backward_fp32_logits(cuda_lib, oracle, p):
    V, R, T = 20000, 12, 0.8
    rng = np.random.default_rng(5)
    z = workloads.normal_logits_fp32(R, V, 2.0, seed=13, device="cuda")
    z[2, 100:200] = z[2, 0]                              # fp32 ties
    hz = z.cpu().numpy()
    ids = oracle.sample_ids(hz, T, p, workloads.uniforms(R, 9))
    glp, gh = rng.uniform(-3, 3, R), rng.uniform(-3, 3, R)
    g, k, _ = _run(cuda_lib, z, ids, T, p, glp, gh)
    check_nucleus_sizes(oracle, hz, ids, T, p, k)
    og = oracle.logprob_entropy_backward(hz, ids, T, p, glp.astype(np.float32),
                                         gh.astype(np.float32), force_k=k)
    _check(g, og, hz, k, label="fp32 logits")


def test_backward_split_ties_at_the_boundary(cuda_lib, oracle):
    """Logits on a coarse grid: the boundary value is shared by hundreds of
    ids and the set keeps only the lowest of them (the running tie count)."""
    V, R, T, p = 151936, 8, 1.0, 0.9
    rng = np.random.default_rng(2)
    z = torch.from_numpy((np.round(rng.normal(0, 1, (R, V)) * 4) / 4).astype(np.float32))
    z = z.to(torch.bfloat16).cuda()
    hz = workloads.bf16_bits(z)
    vals = _vals(hz)
    ids = rng.integers(0, V, R).astype(np.int32)
    glp, gh = rng.uniform(-1, 1, R), rng.uniform(-1, 1, R)
    g, k, st = _run(cuda_lib, z, ids, T, p, glp, gh)
    check_nucleus_sizes(oracle, hz, ids, T, p, k)
    og = oracle.logprob_entropy_backward(hz, ids, T, p, glp.astype(np.float32),
                                         gh.astype(np.float32), force_k=k)
    _check(g, og, vals, k, label="split ties")
    order = _keys_sorted(vals)
    for r in range(R):
        t = vals[r][order[r][k[r] - 1]]
        kept = (vals[r][order[r][:k[r]]] == t).sum()
        assert 0 < kept < (vals[r] == t).sum()          # the ties really are split


def test_backward_bad_rows_and_missing_state(cuda_lib, oracle):
    V, R = 5000, 5
    z, _ = workloads.peaked_bf16(R, V=V, seed=3, device="cuda")
    z[2, 17] = float("nan")
    ids = np.array([1, 99999, 8, 4, 10], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g, _, st = _run(cuda_lib, z, ids, 0.7, 0.9, np.ones(R), np.ones(R), status=status)
    gn = g.cpu().numpy()
    assert np.all(np.isnan(gn[1])) and np.all(np.isnan(gn[2]))
    assert np.all(np.isfinite(gn[[0, 3, 4]]))
    assert int(status.item()) == cuda_lib.STATUS_BAD_TOKEN_ID | cuda_lib.STATUS_NONFINITE
    # a state no forward wrote
    status.zero_()
    blank = torch.zeros_like(st)
    g2 = cuda_lib.logprob_entropy_backward(z, torch.from_numpy(ids).cuda(), 0.7, blank,
                                           status_word=status)
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(g2))
    assert int(status.item()) & cuda_lib.STATUS_NO_STATE


def test_backward_bitwise_repeat_and_batch_invariance(cuda_lib, oracle):
    V, R, T, p = 151936, 16, 0.7, 0.95
    rng = np.random.default_rng(12)
    z, _ = workloads.peaked_bf16(R, V=V, seed=81, device="cuda")
    hz = workloads.bf16_bits(z)
    ids = oracle.sample_ids(hz, T, p, workloads.uniforms(R, 4))
    glp, gh = rng.uniform(-1, 1, R), rng.uniform(-1, 1, R)
    g, _, _ = _run(cuda_lib, z, ids, T, p, glp, gh)
    g2, _, _ = _run(cuda_lib, z, ids, T, p, glp, gh)
    assert torch.equal(g, g2)
    for r in (0, 9, 15):
        one, _, _ = _run(cuda_lib, z[r:r + 1].contiguous(), ids[r:r + 1].copy(), T, p,
                         glp[r:r + 1], gh[r:r + 1])
        assert torch.equal(one[0], g[r])


def test_autograd_function(cuda_lib, oracle):
    V, R, T, p = 151936, 6, 0.7, 0.95
    rng = np.random.default_rng(4)
    z, _ = workloads.peaked_bf16(R, V=V, seed=91, device="cuda")
    hz = workloads.bf16_bits(z)
    ids_np = oracle.sample_ids(hz, T, p, workloads.uniforms(R, 2))
    w1 = torch.from_numpy(rng.uniform(-1, 1, R).astype(np.float32)).cuda()
    w2 = torch.from_numpy(rng.uniform(-1, 1, R).astype(np.float32)).cuda()
    x = z.float().requires_grad_(True)
    lp, ent = cuda_lib.logprob_entropy_autograd(x, torch.from_numpy(ids_np).cuda(), T, p)
    lp_fin = torch.where(torch.isinf(lp), torch.zeros_like(lp), lp)
    (lp_fin * w1 + ent * w2).sum().backward()
    _, _, k, _ = oracle.logprob_entropy(hz, ids_np, T, p)
    og = oracle.logprob_entropy_backward(hz, ids_np, T, p, w1.cpu().numpy(), w2.cpu().numpy(),
                                         force_k=k)
    _check(x.grad, og, _vals(hz), k, label="autograd")


def test_backward_empty_batch(cuda_lib):
    e = torch.empty(0, 1000, dtype=torch.bfloat16, device="cuda")
    st = cuda_lib.new_row_state(0, "cuda")
    g = cuda_lib.logprob_entropy_backward(e, torch.empty(0, dtype=torch.int32, device="cuda"),
                                          0.7, st)
    assert g.shape == (0, 1000)
