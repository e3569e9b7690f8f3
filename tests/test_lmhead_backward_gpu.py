"""GPU parity of rlk_lmhead_logprob_fwd / rlk_lmhead_logprob_bwd (the
gradients of the fused LM-head path) against the fp64 oracle.

Tolerance: the gradient logits dz are rounded to bf16 (relative error <= 2^-9
each, random in sign) before the two weight-side GEMMs, so a row of
dL/dhidden = dz W or of dL/dW = dz^T hidden carries a relative error near
2^-9 / sqrt(3) ~ 1e-3 in norm; each row must agree with the oracle to 4e-3 of
its norm (plus a floor of 1e-5 of the whole matrix's rms, for rows that are
nearly zero).  The row log-normaliser from the forward must agree with the
oracle's to 2e-4.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

REL = 4e-3


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _rows_close(got, want, label):
    got = got.double().cpu().numpy() if torch.is_tensor(got) else got
    floor = 1e-5 * np.sqrt(np.mean(want ** 2))
    err = np.linalg.norm(got - want, axis=1)
    ref = np.linalg.norm(want, axis=1)
    bad = err > REL * ref + floor * np.sqrt(want.shape[1])
    assert not bad.any(), f"{label}: {bad.sum()} rows, worst {np.max(err / (ref + 1e-30)):.3g}"


def _run(rlk, hidden, w, ids, T_, glp, gh, **kw):
    n = hidden.shape[0]
    lse = torch.empty(n, device="cuda")
    lp, ent = rlk.lmhead_logprob(hidden, w, ids, T_, out_lse=lse)
    dh, dw = rlk.lmhead_backward(hidden, w, ids, T_, lse, ent, glp, gh, **kw)
    torch.cuda.synchronize()
    return lp, ent, lse, dh, dw


@pytest.mark.parametrize("T,H,V", [(300, 256, 5000), (4500, 128, 2048)])
def test_lmhead_backward_matches_oracle(cuda_lib, oracle, T, H, V):
    """Ragged M and N tiles; the second shape spans two 4096-row chunks, so
    dL/dW sums two chunks."""
    hidden, w, ids = workloads.lmhead_inputs(T, H, V, seed=8, device="cuda")
    w = (w.float() * 2.5).to(torch.bfloat16)        # logits spread over a few units
    rng = np.random.default_rng(3)
    gl = rng.uniform(-2, 2, T).astype(np.float32)
    ge = rng.uniform(-2, 2, T).astype(np.float32)
    lp, ent, lse, dh, dw = _run(cuda_lib, hidden, w, ids, 0.7, torch.from_numpy(gl).cuda(),
                                torch.from_numpy(ge).cuda())
    hb, wb = _bits(hidden), _bits(w)
    odh, odw = oracle.lmhead_backward(hb, wb, ids.cpu().numpy(), 0.7, 1.0, gl, ge)
    _rows_close(dh, odh, "dL/dhidden")
    _rows_close(dw, odw, "dL/dW")
    # the log-normaliser, from the oracle's log-probability of the same rows
    olp, _, _ = oracle.lmhead_rows(hb, wb, np.arange(T), ids.cpu().numpy(), 0.7)
    z = hidden.double().cpu() @ w.double().cpu().T
    zy = z[torch.arange(T), ids.cpu().long()].numpy()
    assert np.abs(lse.cpu().numpy() - (zy / np.float32(0.7) - olp)).max() <= 2e-4


def test_lmhead_backward_entropy_only_and_accumulate(cuda_lib, oracle):
    T, H, V = 200, 128, 3000
    hidden, w, ids = workloads.lmhead_inputs(T, H, V, seed=9, device="cuda")
    w = (w.float() * 2.5).to(torch.bfloat16)
    ge = torch.ones(T, device="cuda")
    _, _, _, dh, dw = _run(cuda_lib, hidden, w, ids, 1.0, None, ge)
    odh, odw = oracle.lmhead_backward(_bits(hidden), _bits(w), ids.cpu().numpy(), 1.0, 1.0, None,
                                      np.ones(T, np.float32))
    _rows_close(dh, odh, "entropy-only dL/dhidden")
    _rows_close(dw, odw, "entropy-only dL/dW")
    base = torch.randn(V, H, device="cuda")
    lse = torch.empty(T, device="cuda")
    _, ent = cuda_lib.lmhead_logprob(hidden, w, ids, 1.0, out_lse=lse)
    _, dw2 = cuda_lib.lmhead_backward(hidden, w, ids, 1.0, lse, ent, None, ge,
                                      grad_w=base.clone(), accumulate_grad_w=True)
    torch.cuda.synchronize()
    assert torch.allclose(dw2, base + dw, rtol=1e-6, atol=1e-6)


def test_lmhead_backward_bitwise_repeat(cuda_lib):
    T, H, V = 300, 256, 5000
    hidden, w, ids = workloads.lmhead_inputs(T, H, V, seed=10, device="cuda")
    g = torch.rand(T, device="cuda")
    a = _run(cuda_lib, hidden, w, ids, 0.7, g, g)
    b = _run(cuda_lib, hidden, w, ids, 0.7, g, g)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_lmhead_backward_empty(cuda_lib):
    h = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(100, 128, dtype=torch.bfloat16, device="cuda")
    e = torch.empty(0, device="cuda")
    dh, dw = cuda_lib.lmhead_backward(h, w, torch.empty(0, dtype=torch.int32, device="cuda"), 0.7,
                                      e, e, grad_w=torch.zeros(100, 128, device="cuda"),
                                      accumulate_grad_w=True)
    assert dh.shape == (0, 128) and not dw.any()
