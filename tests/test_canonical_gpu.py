"""The canonical vocabulary partition (virtual tensor-parallel degree 8,
padded vocabulary 152576) through the C ABI.

- Against the fp64 oracle at top_p = 1: |d logprob|, |d entropy| <= 2e-4.
- Independence of the physical degree: splitting the eight shards over 1, 2,
  4 or 8 "ranks" (each computing its adjacent shards' partials from its own
  slice of the columns, then all partials combined in rank order) gives the
  canonical single-device result bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads
from _parity import LP_REL, LP_TOL, ENT_TOL, compare_rows

pytestmark = pytest.mark.gpu


def _check(lp, ent, olp, oent):
    lp, ent = lp.cpu().numpy().astype(np.float64), ent.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(lp), np.isneginf(olp))     # -inf: y outside the set
    fin = ~np.isneginf(olp)
    assert np.all(np.abs(lp[fin] - olp[fin]) <= LP_TOL + LP_REL * np.abs(olp[fin]))
    assert np.all(np.abs(ent - oent) <= ENT_TOL)


@pytest.mark.parametrize("T_", [0.7, 1.8])
def test_canonical_matches_oracle(cuda_lib, oracle, T_):
    R, V = 48, workloads.VOCAB
    z, _ = workloads.peaked_bf16(R, V=V, seed=33, device="cuda")
    hz = workloads.bf16_bits(z)
    ids = torch.from_numpy(oracle.sample_ids(hz, T_, 1.0, workloads.uniforms(R, 7))).cuda()
    lp, ent = cuda_lib.logprob_entropy_canonical(z, ids, T_)
    torch.cuda.synchronize()
    olp, oent, _, _ = oracle.logprob_entropy(hz, ids.cpu().numpy(), T_, 1.0)
    _check(lp, ent, olp, oent)
    # and within tolerance of the single-device scorer, whose boundaries differ
    dlp, dent = cuda_lib.logprob_entropy(z, ids, T_, 1.0)
    torch.cuda.synchronize()
    _check(lp, ent, dlp.cpu().numpy().astype(np.float64), dent.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_physical_degree_does_not_change_the_bits(cuda_lib, dtype):
    R, V = 40, workloads.VOCAB
    if dtype == "bf16":
        z, _ = workloads.peaked_bf16(R, V=V, seed=35, device="cuda")
    else:
        z = workloads.normal_logits_fp32(R, V, 3.0, seed=35, device="cuda")
    ids = torch.randint(0, V, (R,), dtype=torch.int32, device="cuda")
    ref = cuda_lib.logprob_entropy_canonical(z, ids, 0.7)
    for tp in (1, 2, 4, 8):
        parts = []
        for rank in range(tp):
            _, n, c0, w = cuda_lib.canonical_plan(tp, rank)
            local = z[:, c0:min(c0 + n * w, V)]            # this rank's columns only
            parts.append(cuda_lib.shard_partials(local, ids, 0.7, V, c0, w, n))
        lp, ent = cuda_lib.shard_combine(torch.cat(parts, 0), ids, 0.7, V, w)
        torch.cuda.synchronize()
        assert torch.equal(lp, ref[0]) and torch.equal(ent, ref[1]), tp


def test_padding_shards_and_small_vocabularies(cuda_lib, oracle):
    """A vocabulary of 1000 in a padded 2048 split eight ways: the last shards
    are padding only (empty partials); ragged shard ends; odd row stride."""
    R, V = 24, 1000
    base = workloads.normal_logits_fp32(R, V + 3, 2.0, seed=2, device="cuda")
    z = base[:, :V]                                    # fp32, row stride V + 3
    ids = torch.randint(0, V, (R,), dtype=torch.int32, device="cuda")
    lp, ent = cuda_lib.logprob_entropy_canonical(z, ids, 0.9, 8, 2048)
    torch.cuda.synchronize()
    olp, oent, _, _ = oracle.logprob_entropy(z.contiguous().cpu().numpy(), ids.cpu().numpy(),
                                             0.9, 1.0)
    _check(lp, ent, olp, oent)
    # rank 7 of 8 holds padding only: its partials are empty and change nothing
    parts = []
    for rank in range(8):
        _, n, c0, w = cuda_lib.canonical_plan(8, rank, 8, 2048)
        local = z[:, c0:min(c0 + n * w, V)] if c0 < V else z[:, :1]
        parts.append(cuda_lib.shard_partials(local, ids, 0.9, V, c0, w, n))
    lp2, ent2 = cuda_lib.shard_combine(torch.cat(parts, 0), ids, 0.9, V, w)
    torch.cuda.synchronize()
    assert torch.equal(lp2, lp) and torch.equal(ent2, ent)


def test_canonical_bad_rows(cuda_lib):
    R, V = 6, workloads.VOCAB
    z, _ = workloads.peaked_bf16(R, V=V, seed=3, device="cuda")
    z[2, 140000] = float("nan")        # in the last shard
    z[3, 5] = float("-inf")
    ids = torch.tensor([0, V, 1, 2, 3, -1], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent = cuda_lib.logprob_entropy_canonical(z, ids, 0.7, status_word=st)
    torch.cuda.synchronize()
    bad = torch.isnan(lp).cpu().tolist()
    assert bad == [False, True, True, True, False, True]
    assert int(st.item()) == cuda_lib.STATUS_BAD_TOKEN_ID | cuda_lib.STATUS_NONFINITE


def _csr(lists):
    off = np.concatenate([[0], np.cumsum([len(l) for l in lists])]).astype(np.int64)
    return off, np.concatenate(lists).astype(np.int32)


def test_supplied_support_under_the_partition(cuda_lib, oracle):
    """top_p < 1 rows as the sampler ships them (a retained set per row), under
    the canonical partition: against the supplied-support oracle, and the same
    bits for 1, 2, 4 and 8 emulated ranks.  Rows whose selected id is not
    listed get -inf; a bad list is flagged."""
    R, V = 32, workloads.VOCAB
    z, _ = workloads.peaked_bf16(R, V=V, seed=61, device="cuda")
    hz = workloads.bf16_bits(z)
    ids = oracle.sample_ids(hz, 0.7, 0.95, workloads.uniforms(R, 9))
    _, _, k, _ = oracle.logprob_entropy(hz, ids, 0.7, 0.95)
    vals = (hz.astype(np.uint32) << 16).view(np.float32)
    rng = np.random.default_rng(3)
    lists = [rng.permutation(np.lexsort((np.arange(V), -vals[r]))[:k[r]]) for r in range(R)]
    ids[5] = np.setdiff1d(np.arange(V), lists[5])[0]          # not listed
    off, sup = _csr(lists)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tid = d(ids)
    ref = None
    for tp in (1, 2, 4, 8):
        parts = []
        for rank in range(tp):
            _, n, c0, w = cuda_lib.canonical_plan(tp, rank)
            local = z[:, c0:min(c0 + n * w, V)]
            parts.append(cuda_lib.shard_partials_support(local, tid, 0.7, V, c0, w, n, d(off),
                                                         d(sup)))
        lp, ent = cuda_lib.shard_combine(torch.cat(parts, 0), tid, 0.7, V, w)
        torch.cuda.synchronize()
        if ref is None:
            ref = (lp, ent)
        else:
            assert torch.equal(lp, ref[0]) and torch.equal(ent, ref[1]), tp
    olp, oent, st = oracle.logprob_entropy_support(hz, ids, 0.7, off, sup)
    _check(ref[0], ref[1], olp, oent)
    assert np.isneginf(ref[0].cpu().numpy()[5]) and np.isneginf(olp[5])
    # a bad list: an empty row and an id out of range
    lists2 = [lists[0], np.array([], np.int64), np.array([3, V + 7])]
    off2, sup2 = _csr(lists2)
    stw = torch.zeros(1, dtype=torch.int32, device="cuda")
    p2 = cuda_lib.shard_partials_support(z[:3].contiguous(), tid[:3].contiguous(), 0.7, V, 0,
                                         19072, 8, d(off2), d(sup2))
    lp2, _ = cuda_lib.shard_combine(p2, tid[:3].contiguous(), 0.7, V, 19072, status_word=stw)
    torch.cuda.synchronize()
    assert torch.isnan(lp2).cpu().tolist() == [False, True, True]
    assert int(stw.item()) == cuda_lib.STATUS_BAD_SUPPORT


# ----------------------------------------------------------- top_p < 1
# Two exchanges: every shard's partial reaches every rank, which sets the
# row's window; each shard then counts its logits in the window per bf16 value
# and the counts are combined in shard order (RL-Kernel "Qwen3-8B VIME
# train-rollout consistency", section "Canonical topology strategy").

def _emulate_ranks(cuda_lib, z, ids, T_, p, tp):
    """tp ranks, each holding only its own columns: partials, the all-gather
    (a concatenation in rank order), window counts, the second all-gather, and
    the combine."""
    V = z.shape[1]
    plans = [cuda_lib.canonical_plan(tp, rank) for rank in range(tp)]
    local = [z[:, c0:min(c0 + n * w, V)] for _, n, c0, w in plans]
    parts = [cuda_lib.shard_partials(loc, ids, T_, V, c0, w, n)
             for loc, (_, n, c0, w) in zip(local, plans)]
    allp = torch.cat(parts, 0)
    cnts = [cuda_lib.shard_window_counts(loc, ids, T_, p, V, c0, w, n, allp)
            for loc, (_, n, c0, w) in zip(local, plans)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = cuda_lib.shard_combine_topp(allp, torch.cat(cnts, 0), ids, T_, p, V, plans[0][3],
                                      status_word=st)
    torch.cuda.synchronize()
    return out, int(st.item())


@pytest.mark.parametrize("T_,p", [(0.7, 0.95), (0.7, 0.5), (1.8, 0.9)])
def test_canonical_topp_matches_oracle(cuda_lib, oracle, T_, p):
    from _parity import compare_rows
    R, V = 48, workloads.VOCAB
    z, _ = workloads.peaked_bf16(R, V=V, seed=41, device="cuda")
    hz = workloads.bf16_bits(z)
    ids = torch.from_numpy(oracle.sample_ids(hz, T_, p, workloads.uniforms(R, 9))).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent, k = cuda_lib.logprob_entropy_canonical_topp(z, ids, T_, p, status_word=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    compare_rows(oracle, hz, ids.cpu().numpy(), T_, p, lp.cpu().numpy(), ent.cpu().numpy(),
                 k.cpu().numpy(), label=f"canonical top-p T{T_} p{p}")
    # ids mostly outside the nucleus: -inf log-probabilities, same sizes
    far = ((ids.long() + V // 2) % V).to(torch.int32)
    lp2, ent2, k2 = cuda_lib.logprob_entropy_canonical_topp(z, far, T_, p)
    torch.cuda.synchronize()
    compare_rows(oracle, hz, far.cpu().numpy(), T_, p, lp2.cpu().numpy(), ent2.cpu().numpy(),
                 k2.cpu().numpy(), label=f"canonical top-p far T{T_} p{p}")


def test_canonical_topp_bits_for_every_degree(cuda_lib, oracle):
    R, V = 40, workloads.VOCAB
    z, _ = workloads.peaked_bf16(R, V=V, seed=43, device="cuda")
    hz = workloads.bf16_bits(z)
    ids = torch.from_numpy(oracle.sample_ids(hz, 0.7, 0.95, workloads.uniforms(R, 11))).cuda()
    ref = cuda_lib.logprob_entropy_canonical_topp(z, ids, 0.7, 0.95)
    torch.cuda.synchronize()
    for tp in (1, 2, 4, 8):
        (lp, ent, k), st = _emulate_ranks(cuda_lib, z, ids, 0.7, 0.95, tp)
        assert st == 0
        assert torch.equal(lp, ref[0]) and torch.equal(ent, ref[1]) and torch.equal(k, ref[2]), tp


def test_canonical_topp_special_rows(cuda_lib, oracle):
    """Windows that cross zero (the near-zero bin inside the window), flat
    rows, wide tie groups, Zipf rows, and rows the path cannot resolve or must
    refuse."""
    from _parity import compare_rows
    V = workloads.VOCAB
    z, _ = workloads.peaked_bf16(12, V=V, seed=45)
    z = z.float()
    g = torch.Generator().manual_seed(45)
    z[1] = torch.randn(V, generator=g) * 0.5              # flat, around zero
    z[2] = torch.randn(V, generator=g) * 3 - 20.0         # all negative
    z[3, :64] = z[3].max() + 0.5                           # a wide tie group at the top
    zipf, _ = workloads.zipf_bf16(4, V=V, seed=46)
    z[4:8] = zipf.float()
    z[8] = 1.5                                             # all equal
    z = z.to(torch.bfloat16).cuda()
    hz = workloads.bf16_bits(z)
    for T_, p in ((0.7, 0.95), (1.0, 0.9)):
        ids_h = oracle.sample_ids(hz, T_, p, workloads.uniforms(12, 13))
        ids = torch.from_numpy(ids_h).cuda()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        lp, ent, k = cuda_lib.logprob_entropy_canonical_topp(z, ids, T_, p, status_word=st)
        torch.cuda.synchronize()
        lp, ent, k = lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy()
        unresolved = np.isnan(lp)
        # every row either matches the oracle or is reported unresolved
        assert (int(st.item()) & ~cuda_lib.STATUS_UNRESOLVED) == 0
        assert unresolved.sum() <= 2, f"rows left unresolved: {np.nonzero(unresolved)[0]}"
        ok = ~unresolved
        compare_rows(oracle, hz[ok], ids_h[ok], T_, p, lp[ok], ent[ok], k[ok],
                     label=f"canonical special T{T_} p{p}")
        for tp in (2, 8):
            (lp2, ent2, k2), _ = _emulate_ranks(cuda_lib, z, ids, T_, p, tp)
            assert np.array_equal(lp2.cpu().numpy().view(np.uint32), lp.view(np.uint32))
            assert np.array_equal(ent2.cpu().numpy().view(np.uint32), ent.view(np.uint32))


def test_canonical_topp_bad_rows(cuda_lib):
    V = workloads.VOCAB
    z, peaks = workloads.peaked_bf16(6, V=V, seed=47, device="cuda")
    z[1, 5] = float("nan")
    z[2, V - 1] = float("inf")
    z[3, 400] = float("-inf")
    ids = torch.tensor([int(peaks[0]), 1, 2, 3, V, -1], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent, k = cuda_lib.logprob_entropy_canonical_topp(z, ids, 0.7, 0.9, status_word=st)
    torch.cuda.synchronize()
    lp, ent, k = lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy()
    assert np.isfinite(lp[0]) and np.isfinite(ent[0]) and k[0] >= 1
    assert np.all(np.isnan(lp[1:])) and np.all(np.isnan(ent[1:])) and np.all(k[1:] == 0)
    assert int(st.item()) == (cuda_lib.STATUS_BAD_TOKEN_ID | cuda_lib.STATUS_NONFINITE)


def test_canonical_topp_boundaries_near_the_gap_threshold(cuda_lib, oracle):
    """Three peaked rows (V = 58,644, temperature 0.5, top_p 0.999) whose
    boundaries lie 0.7e-6, 1.18e-6 and 1.67e-6 from a cumulative step.  The
    combine's bin weights and the shards' sums must use one reference: a
    common factor between them as small as 2^-19 (a reference exponent
    rounded to fp32 on one side and not on the other) moves the second row's
    boundary by one token, outside the gap exemption."""
    z, _ = workloads.peaked_bf16(3, V=58644, seed=268817604, device="cuda")
    hz = workloads.bf16_bits(z)
    ids_h = oracle.sample_ids(hz, 0.5, 0.999, workloads.uniforms(3, 5))
    ids = torch.from_numpy(ids_h).cuda()
    lp, ent, k = cuda_lib.logprob_entropy_canonical_topp(z, ids, 0.5, 0.999)
    torch.cuda.synchronize()
    compare_rows(oracle, hz, ids_h, 0.5, 0.999, lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy(),
                 label="canonical near-threshold rows")
