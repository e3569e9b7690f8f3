"""The top-p sampler's two ways of reaching a draw against each other and
the oracle.

The direct mode reads a row once: members binned by key - boundary key with
fixed-point masses, and their positions listed, so the draw's tie group is
ranked from the list (a scan of the row in id order only when the list ran
out of room or the group is too large to rank; a debug mode turns the list
off so that scan serves every row).  The radix descent bins the
16-bit keys in two levels and finds the id by a scan in id order.  Both use
the same integer arithmetic (masses w 2^40 truncated, the target ceil(u Z),
the need-th lowest id of the draw's key), so their ids must be equal row by
row: peaked rows, rows with wide tie groups at the draw, rows whose members
overflow the list, coarse grids, a boundary that keeps every token, rows
without a valid state.  The draws are also checked against the oracle's
sorted inverse-CDF sampler.
"""
import numpy as np
import pytest
import torch

import workloads
from test_sampler_gpu import _check

pytestmark = pytest.mark.gpu


def _states(rlk, z, T_, p):
    st = rlk.new_row_state(z.shape[0], z.device)
    zeros = torch.zeros(z.shape[0], dtype=torch.int32, device=z.device)
    if torch.is_tensor(T_) or torch.is_tensor(p):
        full = lambda v: v if torch.is_tensor(v) else torch.full(
            (z.shape[0],), float(v), device=z.device, dtype=torch.float32)
        rlk.logprob_entropy_rows(z, zeros, full(T_), full(p), row_state=st)
    else:
        rlk.logprob_entropy(z, zeros, T_, p, row_state=st)
    return st


def _both(rlk, z, T_, p, u, state=None):
    """(direct-mode ids, radix-descent ids, their two status words); the
    direct mode without its member list must give the direct mode's ids and
    status."""
    if state is None:
        state = _states(rlk, z, T_, p)
    temp = 1.0 if torch.is_tensor(T_) else T_
    out = []
    prev = rlk.set_sampler_mode(1)
    try:
        for mode in (1, 0, 2):
            rlk.set_sampler_mode(mode)
            st = torch.zeros(1, dtype=torch.int32, device=z.device)
            ids = rlk.sample_top_p(z, temp, p, u, row_state=state, status_word=st)
            torch.cuda.synchronize()
            out.append((ids.cpu().numpy(), int(st.item())))
    finally:
        rlk.set_sampler_mode(prev)
    (a, sa), (b, sb), (c, sc) = out
    assert np.array_equal(a, c) and sa == sc, np.nonzero(a != c)[0]
    return a, b, sa, sb


def special_rows(V, seed):
    """Peaked Qwen-shaped rows mixed with rows of unusual shape."""
    z, _ = workloads.peaked_bf16(20, V=V, seed=seed)
    z = z.float()
    g = torch.Generator().manual_seed(seed)
    z[1] = torch.randn(V, generator=g) * 0.5                  # flat: tens of thousands of members
    z[2] = 1.5                                                 # all equal
    z[3] = 0.0; z[3, V // 3] = 60.0                            # one-hot
    z[4] = torch.randn(V, generator=g) * 3e4                   # huge logits
    z[5] = torch.randn(V, generator=g) * 3 - 20.0              # all negative
    z[6, :64] = z[6].max() + 0.5                               # 64-way tie at the top
    z[7] = torch.randn(V, generator=g) * 3; z[7, V - 1] = 40.0  # peak in the last column
    z[8] = torch.randn(V, generator=g) * 3; z[8, 0] = 40.0      # peak in the first column
    z[9, 100:4000:130] = z[9].max() + 0.25                     # 30-way tie at the top
    z[10] = torch.round(torch.randn(V, generator=g) * 8) / 8 + 4.0   # a coarse grid: wide ties
    z[11, 7] = z[11].max() + 20.0                              # one token takes all the mass
    z[12, 5000:7000] = z[12].max() + 1.0                       # a 2000-way tie: too large to rank
    return z.to(torch.bfloat16)


@pytest.mark.parametrize("T_,p", [(0.7, 0.95), (1.0, 0.5), (1.8, 0.9), (0.7, 0.999), (0.7, 1.0)])
def test_direct_matches_radix(cuda_lib, oracle, T_, p):
    z = special_rows(workloads.VOCAB, seed=61).cuda()
    u = workloads.uniforms(z.shape[0], 62).astype(np.float32)
    u[0], u[3] = 0.0, 0.99999994
    a, b, sa, sb = _both(cuda_lib, z, T_, p, torch.from_numpy(u).cuda())
    assert sa == 0 and sb == 0
    assert np.array_equal(a, b), np.nonzero(a != b)[0]
    _check(workloads.bf16_bits(z), a, u, T_, p, oracle)


def test_tie_groups_every_rank(cuda_lib):
    """Tie groups of 20, 300 (ranked from the list) and 1500 (too large: the
    scan in id order) at the top, drawn across their ranks: u sweeps the
    groups.  At top_p = 0.99 the boundary falls inside the two larger groups,
    so only their lowest ids are kept."""
    V = workloads.VOCAB
    sizes = (20, 300, 1500)
    base, _ = workloads.peaked_bf16(len(sizes), V=V, seed=71)
    base = base.float()
    for r, n in enumerate(sizes):
        cols = torch.arange(n) * 97 + 11
        base[r, cols] = base[r].max() + 8.0   # the group holds nearly all the mass
    reps = 96
    z = base.repeat_interleave(reps, dim=0).to(torch.bfloat16).cuda()
    u = np.tile(np.linspace(0.0, 0.999, reps, dtype=np.float32), len(sizes))
    a, b, sa, sb = _both(cuda_lib, z, 0.7, 0.99, torch.from_numpy(u).cuda())
    assert sa == 0 and sb == 0
    assert np.array_equal(a, b), np.nonzero(a != b)[0]
    # the draws walk each group in id order, at a rank close to u n
    for r, n in enumerate(sizes):
        cols = np.arange(n) * 97 + 11
        got = a[reps * r:reps * (r + 1)]
        assert np.isin(got, cols).all(), n
        rank = (got - 11) // 97
        assert np.all(np.diff(rank) >= 0), n
        assert np.all(np.abs(rank - u[:reps].astype(np.float64) * n) <= 0.02 * n + 1), n
        if n <= reps // 2:
            assert len(set(rank)) == n


@pytest.mark.parametrize("V,ld,off", [(14335, 14336, 0), (151931, 151936, 0), (151936, 151939, 0),
                                      (151936, 151944, 1), (174081, 174088, 0), (20000, 20480, 0),
                                      (148256, 148256, 0), (148255, 148256, 0), (2097153, 2097160, 0)])
@pytest.mark.parametrize("p", [0.9, 1.0])
def test_vocab_sizes_and_strides(cuda_lib, oracle, V, ld, off, p):
    """Partial last groups, padded strides that are not a multiple of 8
    logits, a base that is not 16-byte aligned (2-byte loads), row lengths
    whose groups do not fill the CTA's last step evenly (148,256 logits:
    18,532 groups, 100 past a whole number of 1,024-group steps, so some lanes
    of a warp hold groups in that step and others do not), and a vocabulary
    past 2^21 (no member list: the tie group from the scan in id order)."""
    rows = 12 if V < 1_000_000 else 3
    base, _ = workloads.peaked_bf16(rows, V=ld + off, seed=17, device="cuda")
    z = base[:, off:off + V]
    z[:, V - 3:] = 12.5   # kept tokens in the partial last group
    u = workloads.uniforms(rows, 18).astype(np.float32)
    a, b, sa, sb = _both(cuda_lib, z, 0.7, p, torch.from_numpy(u).cuda())
    assert sa == 0 and sb == 0
    assert np.array_equal(a, b), np.nonzero(a != b)[0]
    if V < 1_000_000:
        _check(workloads.bf16_bits(z), a, u, 0.7, p, oracle)


def test_batches_and_per_row_parameters(cuda_lib):
    """Batches of 1 .. 700 rows (fewer and more rows than CTAs), rows with
    their own temperature and top-p (the state's temperature sets the row's
    scale), and a row without a valid state (a NaN logit): -1 and the row's
    status in both modes; each row's id is the same in every batch."""
    z = special_rows(workloads.VOCAB, seed=81).cuda()
    n = 700
    idx = torch.arange(n) % z.shape[0]
    idx = idx[torch.randperm(n, generator=torch.Generator().manual_seed(2))]
    zz = z[idx.cuda()].contiguous()
    zz[13, 5] = float("nan")
    g = torch.Generator().manual_seed(83)
    temps = (0.5 + torch.rand(n, generator=g) * 1.5).cuda()
    tops = (0.5 + torch.rand(n, generator=g) * 0.5).cuda()
    tops[::7] = 1.0
    u = torch.rand(n, generator=g).cuda()
    state = _states(cuda_lib, zz, temps, tops)
    a, b, sa, sb = _both(cuda_lib, zz, temps, tops, u, state=state)
    assert np.array_equal(a, b), np.nonzero(a != b)[0]
    assert a[13] == -1 and sa == sb and sa & cuda_lib.STATUS_NONFINITE
    assert (np.delete(a, 13) >= 0).all()
    for rows in (1, 5, 152, 333):
        sub = slice(17, 17 + rows)
        c, d, _, _ = _both(cuda_lib, zz[sub].contiguous(), temps[sub].contiguous(),
                           tops[sub].contiguous(), u[sub].contiguous())
        assert np.array_equal(c, a[sub]) and np.array_equal(d, a[sub])


def test_subnormal_and_signed_zero_order(cuda_lib, oracle):
    """Rows made only of zeros of both signs, bf16 subnormals and the
    smallest normals of both signs.  Their weights are all equal, so the
    retained set, its boundary ties and the draw follow the exact order of
    these values (-0 == +0), which the packed bf16 compares must keep."""
    V = 20011   # p V = 10005.5: the boundary is not at a cumulative step
    pats = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x0002, 0x8002, 0x0040, 0x8040,
                     0x007F, 0x807F, 0x0080, 0x8080], np.uint16)
    rng = np.random.default_rng(5)
    hz = pats[rng.integers(0, len(pats), (8, V))]
    z = torch.from_numpy(hz.view(np.int16)).view(torch.bfloat16).cuda()
    u = workloads.uniforms(8, 6).astype(np.float32)
    a, b, sa, sb = _both(cuda_lib, z, 1.0, 0.5, torch.from_numpy(u).cuda())
    assert sa == 0 and sb == 0
    assert np.array_equal(a, b), np.nonzero(a != b)[0]
    _check(hz, a, u, 1.0, 0.5, oracle)


@pytest.mark.parametrize("V", [1, 5, 8, 9, 100, 1000])
@pytest.mark.parametrize("T_,p", [(0.7, 0.9), (1.0, 1.0)])
def test_small_vocabularies(cuda_lib, oracle, V, T_, p):
    """Rows shorter than one warp's groups (the loop bound, the queue and
    its last drain with a handful of lanes), with ties, against the oracle."""
    rng = np.random.default_rng(V)
    zf = np.round(rng.normal(0.0, 2.0, (16, V)) * 4) / 4   # a 0.25 grid: ties
    z = torch.from_numpy(zf.astype(np.float32)).to(torch.bfloat16).cuda()
    u = workloads.uniforms(16, V + 1).astype(np.float32)
    u[0] = 0.0
    a, b, sa, sb = _both(cuda_lib, z, T_, p, torch.from_numpy(u).cuda())
    assert sa == 0 and sb == 0
    assert np.array_equal(a, b), np.nonzero(a != b)[0]
    assert ((a >= 0) & (a < V)).all()
    _check(workloads.bf16_bits(z), a, u, T_, p, oracle)
