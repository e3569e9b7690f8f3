"""rlk_sample_top_p (deterministic inverse-CDF top-p sampling) against the
oracle's sampler, which sorts the vocabulary and takes the first id in ranking
order whose cumulative mass reaches u Z_S in fp64.

The kernel's masses are fixed-point (w 2^40, truncated) in fp32 exponent
arithmetic, so a draw whose u Z_S lies within ~1e-5 (relative) of a
cumulative boundary may land on the neighbouring token; such rows are
recognised from the oracle's own cumulative sums and only require the GPU's
id to be one of the two neighbours.  Rows whose nucleus the oracle finds
ambiguous (gap < 1e-6) are skipped.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _vals(hz):
    return (hz.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check(hz, ids_gpu, u, T_, p, oracle):
    oids = oracle.sample_ids(hz, T_, p, u.astype(np.float64))
    _, _, k, gap = oracle.logprob_entropy(hz, oids, T_, p)
    vals = _vals(hz)
    bad = []
    for r in range(hz.shape[0]):
        if gap[r] < 1e-6 or ids_gpu[r] == oids[r]:
            continue
        order = np.lexsort((np.arange(vals.shape[1]), -vals[r]))[:k[r]]
        x = vals[r][order] / np.float64(np.float32(T_))
        w = np.exp(x - x.max())
        cum = np.cumsum(w) / w.sum()
        j = int(np.nonzero(order == oids[r])[0][0])
        near = [order[j - 1]] if j > 0 else []
        near += [order[j + 1]] if j + 1 < len(order) else []
        edge = min(abs(cum[j] - u[r]), abs((cum[j - 1] if j else 0.0) - u[r]))
        if not (ids_gpu[r] in near and edge <= 1e-5):
            bad.append((r, int(ids_gpu[r]), int(oids[r]), edge))
    assert not bad, bad[:5]
    return oids


@pytest.mark.parametrize("T_,p", [(0.7, 0.95), (1.0, 0.5), (1.8, 0.9), (0.7, 1.0)])
def test_sampler_matches_oracle(cuda_lib, oracle, T_, p):
    R, V = 64, workloads.VOCAB
    z, _ = workloads.peaked_bf16(R, V=V, seed=43, device="cuda")
    hz = workloads.bf16_bits(z)
    u = workloads.uniforms(R, 11).astype(np.float32)
    ids = cuda_lib.sample_top_p(z, T_, p, torch.from_numpy(u).cuda())
    torch.cuda.synchronize()
    _check(hz, ids.cpu().numpy(), u, T_, p, oracle)


def test_sampler_edges_and_ties(cuda_lib, oracle):
    """u = 0 takes the top token (lowest id among equal maxima); u near 1 the
    last kept token; a 0.25-grid row whose boundary ties are split; a flat
    row; odd V and a padded stride."""
    R, V = 8, 30011
    rng = np.random.default_rng(4)
    base = torch.from_numpy((np.round(rng.normal(0, 1, (R, V + 5)) * 4) / 4).astype(np.float32))
    z = base.to(torch.bfloat16).cuda()[:, :V]
    z[1] = 0.0
    hz = workloads.bf16_bits(z.contiguous())
    u = np.array([0.0, 0.3, 0.999999, 0.5, 0.25, 0.75, 0.1, 0.9], np.float32)
    ids = cuda_lib.sample_top_p(z, 1.0, 0.9, torch.from_numpy(u).cuda())
    torch.cuda.synchronize()
    got = ids.cpu().numpy()
    vals = _vals(hz)
    top = np.lexsort((np.arange(V), -vals[0]))[0]
    assert got[0] == top
    k_flat = np.ceil(np.float64(np.float32(0.9)) * V)               # uniform row: k* = ceil(p V)
    assert got[1] == int(np.floor(np.float64(u[1]) * k_flat))       # and the draw's rank floor(u k*)
    _check(hz, got, u, 1.0, 0.9, oracle)


def test_sampler_bitwise_and_bad_rows(cuda_lib):
    R, V = 32, workloads.VOCAB
    z, _ = workloads.peaked_bf16(R, V=V, seed=47, device="cuda")
    u = torch.rand(R, device="cuda")
    a = cuda_lib.sample_top_p(z, 0.7, 0.95, u)
    b = cuda_lib.sample_top_p(z, 0.7, 0.95, u)
    one = cuda_lib.sample_top_p(z[5:6].contiguous(), 0.7, 0.95, u[5:6].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(a, b) and int(one.item()) == int(a[5].item())
    z[3, 10] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = cuda_lib.sample_top_p(z, 0.7, 0.95, u, status_word=st)
    torch.cuda.synchronize()
    assert int(ids[3].item()) == -1 and int(st.item()) & cuda_lib.STATUS_NONFINITE
    assert (ids.cpu().numpy()[[0, 1, 2, 4]] >= 0).all()
