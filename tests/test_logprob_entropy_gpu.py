"""GPU parity of rlk_logprob_entropy (through the C ABI) against the fp64 oracle.

Tolerances: |dlogprob| <= 2e-4 and |dentropy| <= 2e-4 absolute; -inf matches
-inf; nucleus size identical on every row whose boundary mass gap is >= 1e-6
(rows below that are compared at the GPU's nucleus size and counted).
Outputs must also be bitwise identical across runs and batch compositions.
"""
import numpy as np
import pytest
import torch

import workloads
from _parity import compare_rows

pytestmark = pytest.mark.gpu

TEMPS = (0.2, 0.7, 1.0, 1.8)


def run(rlk, logits, ids, T, p):
    lp, ent, k = rlk.logprob_entropy(logits, ids, T, p, return_nucleus_size=True)
    torch.cuda.synchronize()
    return lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy()


def host(logits):
    if logits.dtype == torch.bfloat16:
        return workloads.bf16_bits(logits)
    return logits.detach().cpu().numpy()


def sample_ids(oracle, logits, T, p, seed):
    u = workloads.uniforms(logits.shape[0], seed)
    return torch.from_numpy(oracle.sample_ids(host(logits), T, p, u)).cuda()


def test_tiny_fp32_top_p_one(cuda_lib, oracle):
    z, ids = workloads.tiny(seed=0, device="cuda")
    lp, ent, k = run(cuda_lib, z, ids, 1.0, 1.0)
    rep = compare_rows(oracle, host(z), ids.cpu().numpy(), 1.0, 1.0, lp, ent, k, label="tiny")
    assert rep["members"] == 64 and np.all(k == 1000)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("T", [0.7, 1.0])
def test_bruteforce_v8(cuda_lib, oracle, dtype, T):
    z, _ = workloads.brute_v8(seed=0, device="cuda")
    if dtype == "bf16":
        z = z.to(torch.bfloat16)
    # every id of every row: repeat rows so each (row, id) pair is scored
    zz = z.repeat_interleave(8, dim=0).contiguous()
    ids = torch.arange(8, device="cuda", dtype=torch.int32).repeat(16)
    lp, ent, k = run(cuda_lib, zz, ids, T, 0.9)
    compare_rows(oracle, host(zz), ids.cpu().numpy(), T, 0.9, lp, ent, k, label="v8")


@pytest.mark.parametrize("T", TEMPS)
@pytest.mark.parametrize("p", [1.0, 0.999, 0.95, 0.5])
def test_qwen_rows_temperatures(cuda_lib, oracle, T, p):
    z, _ = workloads.peaked_bf16(40, seed=5, device="cuda")
    ids = sample_ids(oracle, z, T, p, seed=int(T * 100 + p * 1000))
    lp, ent, k = run(cuda_lib, z, ids, T, p)
    compare_rows(oracle, host(z), ids.cpu().numpy(), T, p, lp, ent, k, label=f"T{T} p{p}")


@pytest.mark.parametrize("V,ld", [(1001, 1001), (4099, 4104), (8, 8), (1, 1), (9, 24), (151936, 152064)])
@pytest.mark.parametrize("p", [1.0, 0.9])
def test_ragged_and_strided_rows(cuda_lib, oracle, V, ld, p):
    rows = 37
    base, _ = workloads.peaked_bf16(rows, V=ld, seed=7, device="cuda")
    z = base[:, :V]                           # row stride ld, possibly misaligned rows
    ids = sample_ids(oracle, z.contiguous(), 0.7, p, seed=V)
    lp, ent, k = run(cuda_lib, z, ids, 0.7, p)
    compare_rows(oracle, host(z.contiguous()), ids.cpu().numpy(), 0.7, p, lp, ent, k,
                 label=f"V{V} ld{ld}")


def test_qwen_config_full_size(cuda_lib, oracle):
    """T=4096, V=151936 bf16, temperature 0.7, top_p 0.95, ids drawn from the
    oracle's truncated distribution -- every row against the oracle."""
    z, _ = workloads.peaked_bf16(4096, seed=1, device="cuda")
    hz = host(z)
    u = workloads.uniforms(4096, 11)
    ids_h = oracle.sample_ids(hz, 0.7, 0.95, u)
    ids = torch.from_numpy(ids_h).cuda()
    lp, ent, k = run(cuda_lib, z, ids, 0.7, 0.95)
    rep = compare_rows(oracle, hz, ids_h, 0.7, 0.95, lp, ent, k, label="qwen-full")
    assert rep["members"] == 4096
    print("qwen full-size parity:", rep)


def test_bitwise_repeat_and_batch_invariance(cuda_lib, oracle):
    z, _ = workloads.peaked_bf16(96, seed=9, device="cuda")
    ids = sample_ids(oracle, z, 0.7, 0.95, seed=3)
    for p in (1.0, 0.95):
        ref = run(cuda_lib, z, ids, 0.7, p)
        for _ in range(2):
            again = run(cuda_lib, z, ids, 0.7, p)
            for x, y in zip(ref, again):
                assert np.array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                                      y.view(np.uint32) if y.dtype == np.float32 else y)
        # each row alone
        for r in (0, 17, 95):
            one = run(cuda_lib, z[r:r + 1].contiguous(), ids[r:r + 1].contiguous(), 0.7, p)
            for x, y in zip(ref, one):
                assert x[r:r + 1].tobytes() == y.tobytes()
        # permuted, duplicated and embedded at an odd offset in a bigger batch
        perm = torch.randperm(96, generator=torch.Generator().manual_seed(1)).cuda()
        zp = torch.cat([z[perm], z[:7], z[perm[:5]]]).contiguous()
        ip = torch.cat([ids[perm], ids[:7], ids[perm[:5]]]).contiguous()
        big = run(cuda_lib, zp, ip, 0.7, p)
        pc = perm.cpu().numpy()
        for x, y in zip(ref, big):
            assert x[pc].tobytes() == y[:96].tobytes()
            assert x[:7].tobytes() == y[96:103].tobytes()
        # the same rows under a padded row stride (152064 elements, still
        # 16-byte aligned rows): the layout does not change the bits
        wide = torch.zeros(96, 152064, dtype=torch.bfloat16, device="cuda")
        wide[:, :151936] = z
        pad = run(cuda_lib, wide[:, :151936], ids, 0.7, p)
        for x, y in zip(ref, pad):
            assert x.tobytes() == y.tobytes()
        # rows that are not 16-byte aligned (stride 151937) take the per-row
        # kernel: deterministic, within tolerance of the oracle
        odd = torch.zeros(96, 151937, dtype=torch.bfloat16, device="cuda")
        odd[:, :151936] = z
        mis = run(cuda_lib, odd[:, :151936], ids, 0.7, p)
        assert all(a.tobytes() == b.tobytes()
                   for a, b in zip(mis, run(cuda_lib, odd[:, :151936], ids, 0.7, p)))
        compare_rows(oracle, host(z), ids.cpu().numpy(), 0.7, p, *mis, label=f"odd-stride p{p}")


def _bits_row(vals):
    return torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)


def test_edge_rows(cuda_lib, oracle):
    V = 5000
    rows = []
    rows.append(torch.full((V,), 1.5))                                   # all equal
    one = torch.zeros(V); one[1234] = 60.0; rows.append(one)             # one-hot
    pm = torch.zeros(V); pm[::2] = -0.0; pm[7] = 0.5; rows.append(pm)     # +0 / -0 mix
    tiny = torch.randn(V, generator=torch.Generator().manual_seed(3)) * 1e-5
    tiny[10] = 1e-3; rows.append(tiny)                                    # near-zero bin
    two = torch.zeros(V); two[:40] = 2.0; two[40:] = 1.0; rows.append(two)  # wide tie groups
    big = torch.randn(V, generator=torch.Generator().manual_seed(4)) * 3e4  # huge logits
    rows.append(big)
    z = torch.stack(rows).to(torch.bfloat16).cuda()
    hz = host(z)
    for T in (0.2, 0.7, 1.8, 1e4):
        for p in (0.3, 0.9, 0.95, 0.999, 1.0):
            ids_h = oracle.sample_ids(hz, T, p, workloads.uniforms(z.shape[0], 5))
            ids = torch.from_numpy(ids_h).cuda()
            lp, ent, k = run(cuda_lib, z, ids, T, p)
            compare_rows(oracle, hz, ids_h, T, p, lp, ent, k, label=f"edge T{T} p{p}")
            # also a non-member id where one exists
            ids2_h = ((ids_h.astype(np.int64) + V // 2) % V).astype(np.int32)
            ids2 = torch.from_numpy(ids2_h).cuda()
            lp, ent, k = run(cuda_lib, z, ids2, T, p)
            compare_rows(oracle, hz, ids2_h, T, p, lp, ent, k, label=f"edge2 T{T} p{p}")


def test_ties_at_the_threshold(cuda_lib, oracle):
    """Rows where the boundary token's value is shared by tokens ranked just
    after it: the kept ones are the lowest ids of the tie group."""
    z, _ = workloads.peaked_bf16(32, V=20000, seed=13, device="cuda")
    hz = host(z).copy()
    vals = (hz.astype(np.uint32) << 16).view(np.float32)
    ids0 = np.zeros(32, np.int32)
    _, _, k0, _ = oracle.logprob_entropy(hz, ids0, 0.7, 0.95)
    tie_ids = []
    for r in range(32):
        order = np.lexsort((np.arange(vals.shape[1]), -vals[r]))
        b = order[k0[r] - 1]
        nxt = order[k0[r]:k0[r] + 3]
        hz[r, nxt] = hz[r, b]
        tie_ids.append(int(max(nxt.max(), b)))
    ids = np.array(tie_ids, np.int32)
    zt = torch.from_numpy(hz.view(np.int16)).view(torch.bfloat16).cuda()
    lp, ent, k = run(cuda_lib, zt, torch.from_numpy(ids).cuda(), 0.7, 0.95)
    compare_rows(oracle, hz, ids, 0.7, 0.95, lp, ent, k, label="ties")


def test_bad_rows_give_nan_and_status(cuda_lib):
    z, peaks = workloads.peaked_bf16(6, V=3000, seed=2, device="cuda")
    z[0, int(peaks[0])] = 30.0                 # row 0: a valid row whose id is surely kept
    z[1, 5] = float("nan")
    z[2, 7] = float("inf")
    z[3, 9] = float("-inf")
    ids = torch.tensor([int(peaks[0]), 1, 2, 3, 3000, -1], dtype=torch.int32, device="cuda")
    for p in (1.0, 0.9):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        lp, ent = cuda_lib.logprob_entropy(z, ids, 0.7, p, status_word=st)
        torch.cuda.synchronize()
        lp, ent = lp.cpu().numpy(), ent.cpu().numpy()
        assert np.isfinite(lp[0]) and np.isfinite(ent[0])
        assert np.all(np.isnan(lp[1:])) and np.all(np.isnan(ent[1:]))
        assert int(st.item()) == (cuda_lib.STATUS_BAD_TOKEN_ID | cuda_lib.STATUS_NONFINITE)


def test_empty_batch_and_graph_capture(cuda_lib, oracle):
    z = torch.empty(0, 100, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(0, dtype=torch.int32, device="cuda")
    lp, ent = cuda_lib.logprob_entropy(z, ids, 0.7, 0.9)
    assert lp.numel() == 0
    z, _ = workloads.peaked_bf16(64, V=30000, seed=21, device="cuda")
    ids = sample_ids(oracle, z, 0.7, 0.95, seed=2)
    out_lp = torch.empty(64, device="cuda")
    out_ent = torch.empty(64, device="cuda")
    eager = run(cuda_lib, z, ids, 0.7, 0.95)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cuda_lib.logprob_entropy(z, ids, 0.7, 0.95, out_logprob=out_lp, out_entropy=out_ent)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.logprob_entropy(z, ids, 0.7, 0.95, out_logprob=out_lp, out_entropy=out_ent)
    out_lp.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert out_lp.cpu().numpy().tobytes() == eager[0].tobytes()
    # replay after changing the inputs in place
    z2, _ = workloads.peaked_bf16(64, V=30000, seed=22, device="cuda")
    z.copy_(z2)
    g.replay()
    torch.cuda.synchronize()
    assert out_ent.cpu().numpy().tobytes() == run(cuda_lib, z, ids, 0.7, 0.95)[1].tobytes()
