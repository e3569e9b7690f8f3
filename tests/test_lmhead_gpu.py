"""GPU parity of rlk_lmhead_logprob (fused tcgen05 GEMM + online log-sum-exp).

1. The GEMM core on its own: the validation aid rlk_lmhead_logits_debug returns
   the fp32 logits the tensor cores produced; they must match a library fp32
   matrix product of the same bf16 values.
2. The fused outputs against the fp64 oracle (exact dot products, logits never
   rounded to bf16) on sampled rows: |dlogprob|, |dentropy| <= 2e-4.
3. Bitwise repeatability and batch-size invariance.
4. top_p < 1 (logits emitted as bf16 and scored by the top-p path): bit for
   bit the scorer's outputs on the GEMM's own logits, and against the oracle
   on inputs whose product is exact in fp32, where the oracle's bf16 logits
   are a CPU library product rounded to nearest even.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,H,V", [(128, 64, 256), (200, 128, 1000), (300, 4096, 5003),
                                   (37, 256, 777)])
def test_gemm_core_matches_library_matmul(cuda_lib, T, H, V):
    hidden, w, ids = workloads.lmhead_inputs(T, H, V, seed=4, device="cuda")
    logits, lp, ent = cuda_lib.lmhead_logits_debug(hidden, w, ids, 0.7)
    torch.cuda.synchronize()
    ref = hidden.double() @ w.double().T
    err = (logits.double() - ref).abs().max().item()
    scale = ref.abs().max().item()
    assert err <= 1e-4 * max(scale, 1.0), (err, scale)
    # the fused outputs at top_p = 1 agree with a library log-softmax of the same logits
    z = ref / np.float32(0.7)
    ref_lp = torch.log_softmax(z, 1)[torch.arange(T), ids.long()]
    ref_ent = torch.special.entr(torch.softmax(z, 1)).sum(1)
    assert (lp.double() - ref_lp).abs().max().item() <= 2e-4
    assert (ent.double() - ref_ent).abs().max().item() <= 2e-4


def test_fused_lmhead_against_oracle(cuda_lib, oracle):
    """hidden [T, 4096] ~ N(0,1), W [151936, 4096] ~ N(0, 0.02^2), temperature 0.7,
    top_p 1, uniform targets; rows sampled across several M tiles."""
    T, H, V = 640, 4096, workloads.VOCAB
    hidden, w, ids = workloads.lmhead_inputs(T, H, V, seed=4, device="cuda")
    lp, ent = cuda_lib.lmhead_logprob(hidden, w, ids, 0.7, 1.0)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 255, 300, 511, 512, 600, 639], np.int64)
    olp, oent, ok = oracle.lmhead_rows(workloads.bf16_bits(hidden), workloads.bf16_bits(w), rows,
                                       ids.cpu().numpy(), 0.7, 1.0)
    glp = lp.cpu().numpy()[rows]
    gent = ent.cpu().numpy()[rows]
    assert np.abs(glp - olp).max() <= 2e-4, np.abs(glp - olp).max()
    assert np.abs(gent - oent).max() <= 2e-4, np.abs(gent - oent).max()


def test_lmhead_bitwise_and_batch_invariant(cuda_lib):
    T, H, V = 300, 1024, 20000
    hidden, w, ids = workloads.lmhead_inputs(T, H, V, seed=9, device="cuda")
    a = cuda_lib.lmhead_logprob(hidden, w, ids, 0.7)
    b = cuda_lib.lmhead_logprob(hidden, w, ids, 0.7)
    torch.cuda.synchronize()
    assert a[0].cpu().numpy().tobytes() == b[0].cpu().numpy().tobytes()
    assert a[1].cpu().numpy().tobytes() == b[1].cpu().numpy().tobytes()
    # rows 130..199 computed inside a 70-row batch
    sub = cuda_lib.lmhead_logprob(hidden[130:200].contiguous(), w, ids[130:200].contiguous(), 0.7)
    torch.cuda.synchronize()
    assert a[0][130:200].cpu().numpy().tobytes() == sub[0].cpu().numpy().tobytes()
    assert a[1][130:200].cpu().numpy().tobytes() == sub[1].cpu().numpy().tobytes()


def test_lmhead_bad_ids(cuda_lib):
    hidden, w, ids = workloads.lmhead_inputs(8, 64, 300, seed=2, device="cuda")
    ids[3] = 300
    ids[5] = -2
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent = cuda_lib.lmhead_logprob(hidden, w, ids, 1.0, status_word=st)
    torch.cuda.synchronize()
    lp = lp.cpu().numpy()
    assert np.isnan(lp[3]) and np.isnan(lp[5]) and np.isfinite(lp[0])
    assert int(st.item()) & cuda_lib.STATUS_BAD_TOKEN_ID


@pytest.mark.parametrize("T,H,V,p", [(300, 256, 20000, 0.9), (4500, 128, 8192, 0.95),
                                     (130, 4096, 151936, 0.95)])
def test_lmhead_top_p_chunked_same_bits_as_the_scorer(cuda_lib, T, H, V, p):
    """top_p < 1: the GEMM emits bf16 logits chunk by chunk and the top-p path
    scores them; the outputs are bit for bit those of rlk_logprob_entropy on
    the GEMM's own logits rounded to bf16 (V % 8 == 0: same layout).  The
    second shape spans two 4096-row chunks."""
    hidden, w, ids = workloads.lmhead_inputs(T, H, V, seed=12, device="cuda")
    w = (w.float() * (8.0 if H <= 256 else 1.5)).to(torch.bfloat16)   # peaked enough for a nucleus
    lp, ent = cuda_lib.lmhead_logprob(hidden, w, ids, 0.7, p)
    logits, _, _ = cuda_lib.lmhead_logits_debug(hidden, w, ids, 0.7)
    dlp, dent = cuda_lib.logprob_entropy(logits.to(torch.bfloat16), ids, 0.7, p)
    torch.cuda.synchronize()
    assert torch.equal(lp, dlp) and torch.equal(ent, dent)


@pytest.mark.parametrize("T,H,V,p,s,L", [(300, 256, 20000, 0.9, 7, 7),
                                         (4500, 128, 8192, 0.95, 2, 1),
                                         (130, 4096, 151936, 0.95, 4, 1)])
def test_lmhead_top_p_against_oracle(cuda_lib, oracle, T, H, V, p, s, L):
    """top_p < 1 against the oracle on inputs whose product is exact in fp32
    in any summation order (hidden in {-L..L}, W in {-L..L} 2^-s): the
    oracle's logits are a CPU library product of the same bf16 values,
    rounded to bf16 to nearest even as the emit step rounds (a fifth of the
    logits of the first shape need rounding; the others fit bf16); then the
    fp64 logits path.  Nothing on the oracle side comes from the GPU.  The
    full-vocabulary shape has broad rows (median nucleus ~3000): rows whose
    boundary gap is below 1e-6 are not compared."""
    hidden, w, ids = workloads.lmhead_grid_inputs(T, H, V, seed=14, wshift=s, levels=L,
                                                  device="cuda")
    z = hidden.cpu().double() @ w.cpu().double().T                  # exact
    hz = workloads.bf16_bits(z.float().to(torch.bfloat16))          # z is exact in fp32
    ids_h = ids.cpu().numpy()
    drawn = oracle.sample_ids(hz, 0.7, p, workloads.uniforms(T, 21))
    ids_h[T // 4:] = drawn[T // 4:]                                 # a quarter keep uniform ids
    ids = torch.from_numpy(ids_h).cuda()
    lp, ent = cuda_lib.lmhead_logprob(hidden, w, ids, 0.7, p)
    torch.cuda.synchronize()
    olp, oent, ok, gap = oracle.logprob_entropy(hz, ids_h, 0.7, p)
    sure = gap > 1e-6
    assert sure.mean() > 0.75
    lp_, ent_ = lp.cpu().numpy().astype(np.float64), ent.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(lp_[sure]), np.isneginf(olp[sure]))
    fin = sure & ~np.isneginf(olp)
    assert np.all(np.abs(lp_[fin] - olp[fin]) <= 2e-4 + 2e-7 * np.abs(olp[fin]))
    assert np.all(np.abs(ent_[sure] - oent[sure]) <= 2e-4)
    assert np.median(ok) > 1                                        # real nuclei, not one token
    assert fin.sum() > T // 2                       # most ids drawn inside the nucleus
