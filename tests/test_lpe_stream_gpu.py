"""The streaming logprob/entropy path (bf16 rows of a large vocabulary)
against the fp64 oracle: rows it finishes itself, rows it hands to the
per-row kernel (windows that cross zero, flat rows), bad rows, vocabulary
sizes with a partial last unit, the smallest and largest vocabularies it
takes and one just past them, and batches smaller than the number of SMs.
Same tolerances as the other parity tests; outputs must be bitwise identical
whatever the batch around a row.
"""
import numpy as np
import pytest
import torch

import workloads
from _parity import compare_rows

pytestmark = pytest.mark.gpu

MARKS = (0x7FC0DEAD, 0x7FC0DEAE)   # the recompute marks: never a legal output


def run(rlk, logits, ids, T, p, status=None):
    lp, ent, k = rlk.logprob_entropy(logits, ids, T, p, return_nucleus_size=True,
                                     status_word=status)
    torch.cuda.synchronize()
    return lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy()


def special_rows(V, seed):
    """A batch mixing the peaked Qwen-shaped rows with rows of unusual shape."""
    z, peaks = workloads.peaked_bf16(16, V=V, seed=seed)
    z = z.float()
    g = torch.Generator().manual_seed(seed)
    z[1] = torch.randn(V, generator=g) * 0.5              # flat: window crosses zero
    z[2] = 1.5                                             # all equal
    z[3] = 0.0; z[3, V // 3] = 60.0                        # one-hot
    z[4] = torch.randn(V, generator=g) * 3e4               # huge logits
    z[5] = torch.randn(V, generator=g) * 3 - 20.0          # all negative, peak-free
    z[6, :64] = z[6].max() + 0.5                           # a wide tie group at the top
    z[7] = torch.randn(V, generator=g) * 3; z[7, V - 1] = 40.0   # peak in the last column
    z[8] = torch.randn(V, generator=g) * 3; z[8, 0] = 40.0       # peak in the first column
    return z.to(torch.bfloat16), peaks


def check(rlk, oracle, z, ids_h, T, p, label):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent, k = run(rlk, z, torch.from_numpy(ids_h).cuda(), T, p, st)
    assert not np.isin(lp.view(np.uint32), MARKS).any(), f"{label}: recompute marker leaked"
    assert int(st.item()) == 0, f"{label}: status {int(st.item())}"
    hz = workloads.bf16_bits(z)
    return compare_rows(oracle, hz, ids_h, T, p, lp, ent, k, label=label)


@pytest.mark.parametrize("T", [0.7, 1.8])
@pytest.mark.parametrize("p", [0.5, 0.95, 0.999, 1.0])
def test_stream_special_rows(cuda_lib, oracle, T, p):
    z, _ = special_rows(151936, seed=31)
    z = z.cuda()
    hz = workloads.bf16_bits(z)
    ids_h = oracle.sample_ids(hz, T, p, workloads.uniforms(z.shape[0], 41))
    check(cuda_lib, oracle, z, ids_h, T, p, f"special T{T} p{p}")
    # ids that are mostly outside the nucleus
    far = ((ids_h.astype(np.int64) + 151936 // 2) % 151936).astype(np.int32)
    check(cuda_lib, oracle, z, far, T, p, f"special-far T{T} p{p}")


@pytest.mark.parametrize("V,ld", [(14335, 14336), (14336, 14336), (151931, 151936),
                                  (174080, 174080), (174081, 174088), (20000, 20480)])
@pytest.mark.parametrize("p", [0.9, 1.0])
def test_stream_vocab_sizes(cuda_lib, oracle, V, ld, p):
    """Partial last units, the smallest and the largest vocabularies the
    streaming path takes (14,336 and 174,080) and one just outside each (the
    per-row kernel), padded row strides."""
    base, _ = workloads.peaked_bf16(12, V=ld, seed=17, device="cuda")
    z = base[:, :V]
    z[:, V - 3:] = 12.5   # tokens in the partial last group that are kept
    hz = workloads.bf16_bits(z)
    ids_h = oracle.sample_ids(hz, 0.7, p, workloads.uniforms(12, 43))
    ids_h[:4] = V - 1 - np.arange(4)
    check(cuda_lib, oracle, z, ids_h.astype(np.int32), 0.7, p, f"V{V} ld{ld} p{p}")


@pytest.mark.parametrize("p", [0.95, 1.0])
def test_stream_small_batches_bitwise(cuda_lib, oracle, p):
    """Batches of 1 .. 600 rows (fewer and more rows than SMs): each
    row's bits are the same in every batch, including rows that the per-row
    kernel recomputes."""
    z, _ = special_rows(151936, seed=5)
    z = z.cuda()
    hz = workloads.bf16_bits(z)
    ids_h = oracle.sample_ids(hz, 0.7, p, workloads.uniforms(16, 7))
    ids = torch.from_numpy(ids_h).cuda()
    ref = run(cuda_lib, z, ids, 0.7, p)
    compare_rows(oracle, hz, ids_h, 0.7, p, *ref, label=f"small p{p}")
    for r in (0, 1, 2, 9, 15):
        one = run(cuda_lib, z[r:r + 1].contiguous(), ids[r:r + 1].contiguous(), 0.7, p)
        for x, y in zip(ref, one):
            assert x[r:r + 1].tobytes() == y.tobytes()
    idx = torch.arange(600) % 16
    idx = idx[torch.randperm(600, generator=torch.Generator().manual_seed(3))].cuda()
    big = run(cuda_lib, z[idx].contiguous(), ids[idx].contiguous(), 0.7, p)
    ic = idx.cpu().numpy()
    for x, y in zip(ref, big):
        assert x[ic].tobytes() == y.tobytes()


def test_stream_bad_rows(cuda_lib):
    V = 151936
    z, peaks = workloads.peaked_bf16(8, V=V, seed=2, device="cuda")
    z[0, int(peaks[0])] = 30.0
    z[1, 5] = float("nan")
    z[2, V - 1] = float("inf")
    z[3, 40000] = float("-inf")
    z[4, 3] = float("nan"); z[4, 4] = float("-inf")
    ids = torch.tensor([int(peaks[0]), 1, 2, 3, 4, V, -1, int(peaks[7])],
                       dtype=torch.int32, device="cuda")
    for p in (1.0, 0.9):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        lp, ent, k = run(cuda_lib, z, ids, 0.7, p, st)
        assert np.isfinite(lp[0]) and np.isfinite(ent[0])
        assert np.isfinite(lp[7]) and np.isfinite(ent[7])
        assert np.all(np.isnan(lp[1:7])) and np.all(np.isnan(ent[1:7]))
        assert np.all(k[1:7] == 0)
        assert int(st.item()) == (cuda_lib.STATUS_BAD_TOKEN_ID | cuda_lib.STATUS_NONFINITE)


@pytest.mark.parametrize("p", [0.9, 0.95])
def test_stream_windows_across_zero(cuda_lib, oracle, p):
    """Rows whose window z >= m - L T crosses zero.  The long-response rows
    (Zipf-tilted means) are counted by the streaming kernel itself with
    compressed keys (the values within 2^-4 of zero share one bin summed in
    fixed point): at least four in five of them must not be handed on.  Rows
    whose boundary falls inside that shared bin (a tie group at 0.01, at -0.03)
    and rows with more near-zero tokens than its list holds must be handed on,
    and every row must match the oracle."""
    V = workloads.VOCAB
    z, _ = workloads.zipf_bf16(256, seed=9, kappa=workloads.ZIPF_KAPPA_CALIBRATED,
                               sigma=workloads.ZIPF_SIGMA)
    z = z.float()
    g = torch.Generator().manual_seed(10)
    for r, v in ((0, 0.01), (1, -0.03)):   # boundaries inside the shared bin
        z[r] = torch.randn(V, generator=g) - 12.0
        z[r, :3] = 2.0
        z[r, 1000:1400] = v
    z[2] = torch.randn(V, generator=g) * 0.02 - 30.0   # far below, and ...
    z[2, :500] = torch.randn(500, generator=g) * 0.03  # ... 500 tokens near zero
    z[2, 600] = 1.0
    z = z.to(torch.bfloat16).cuda()
    hz = workloads.bf16_bits(z)
    ids_h = oracle.sample_ids(hz, 0.7, p, workloads.uniforms(256, 12))
    ids = torch.from_numpy(ids_h).cuda()
    st = cuda_lib.new_row_state(256, z.device)
    lp, ent, k = cuda_lib.logprob_entropy(z, ids, 0.7, p, return_nucleus_size=True, row_state=st)
    torch.cuda.synchronize()
    compare_rows(oracle, hz, ids_h, 0.7, p, lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy(),
                 label=f"across zero p{p}")
    # the streaming kernel's reference exponent is an integer, the per-row kernel's is not
    E = st[:, 0].contiguous().view(torch.float32).cpu().numpy()
    streamed = E == np.floor(E)
    assert streamed[3:].mean() >= 0.8, streamed[3:].mean()
    assert not streamed[:2].any()


@pytest.mark.parametrize("p", [0.5, 0.95])
def test_stream_max_near_zero(cuda_lib, oracle, p):
    """Rows whose max lies within 2^-4 of zero.  A max just above zero makes
    the window cross zero from inside the shared near-zero bin: where the
    boundary lies below that bin the streaming kernel counts the row itself
    (the bin, max included, summed in fixed point); where the bin holds the
    boundary it hands the row on.  A max just below zero needs no shared bin
    (the window does not cross zero).  Every row against the oracle."""
    V = workloads.VOCAB
    g = torch.Generator().manual_seed(23)
    z = torch.randn(12, V, generator=g) - 6.0                 # the bulk, well below the max
    z[0, 100] = 0.03                                           # max just above zero
    z[1, 7] = 0.05; z[1, 9] = 0.01; z[1, 11] = -0.02          # a few near-zero tokens at the top
    z[2, V - 1] = -0.02                                        # max just below zero
    z[3, 0] = 0.0; z[3, 1] = -0.0; z[3, 2] = 0.001            # zeros of both signs at the top
    z[4] = torch.randn(V, generator=g) - 20.0                  # the bin holds nearly all the mass:
    z[4, 1000:1300] = 0.04                                     # the boundary lies in it
    z[4, 2000:2300] = -0.03
    z[5] = torch.randn(V, generator=g) * 1.5 - 8.0             # a wider bulk
    z[5, 50] = 0.06
    for r in range(6, 12):                                     # tilted like the long-response rows
        z[r] = -1.2 * torch.log(torch.randperm(V, generator=g).float() + 1.0) + \
               0.5 * torch.randn(V, generator=g) - 3.0
        z[r, r * 97] = 0.02 * (r - 8)
    z = z.to(torch.bfloat16).cuda()
    hz = workloads.bf16_bits(z)
    ids_h = oracle.sample_ids(hz, 0.7, p, workloads.uniforms(12, 24))
    ids_h[0], ids_h[2] = 100, V - 1                            # the max itself selected
    ids = torch.from_numpy(ids_h).cuda()
    st = cuda_lib.new_row_state(12, z.device)
    lp, ent, k = cuda_lib.logprob_entropy(z, ids, 0.7, p, return_nucleus_size=True, row_state=st)
    torch.cuda.synchronize()
    compare_rows(oracle, hz, ids_h, 0.7, p, lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy(),
                 label=f"max near zero p{p}")
    # the streaming kernel's reference exponent is an integer, the per-row
    # kernel's is not (row 8, whose max is 0, is left out: both are 0 there)
    E = st[:, 0].contiguous().view(torch.float32).cpu().numpy()
    streamed = E == np.floor(E)
    # streamed: boundaries far below the bin, and the rows whose max is below
    # zero; handed on: the bin holds the boundary (row 4's tie groups, and the
    # tilted rows with a positive max that alone is the nucleus)
    on = [0, 1, 2, 3, 6, 7] + ([5] if p < 0.9 else [])
    off = [4, 9, 10, 11]
    assert streamed[on].all() and not streamed[off].any(), streamed
