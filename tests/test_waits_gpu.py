"""The expiry path of the bounded device waits, made to run out on purpose
without faulting anything: a debug setting makes the scorer's first CTA skip
one bulk copy (no copy is issued and no arrival made, so nothing is left in
flight) and shortens the wait limit to about a millisecond.  The call must
return, report RLK_STATUS_TIMEOUT, give NaN for every row of that CTA and
the normal bits for every other row; the next call, with the defaults back,
must be bitwise equal to a clean call.  The pages' validator seals a run on
any mismatch (RL-Kernel "ROCm sparse performance" notes): a timed-out row
must therefore never look like a result.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("p", [0.95, 1.0])
def test_withheld_copy_times_out_and_the_next_call_is_clean(cuda_lib, p):
    rlk = cuda_lib
    n, V = 600, 151936
    z, peaks = workloads.peaked_bf16(n, V=V, seed=11, device="cuda")
    ids = peaks.to(torch.int32).cuda()
    st0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp0, ent0 = rlk.logprob_entropy(z, ids, 0.7, p, status_word=st0)
    torch.cuda.synchronize()
    assert int(st0.item()) == 0
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    grid = min(n, nsm)
    old = rlk.set_wait_limit(2_000_000)   # about a millisecond
    try:
        rlk.withhold_copy(5)                # a stage of the first CTA's first row
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        lp, ent = rlk.logprob_entropy(z, ids, 0.7, p, status_word=st)
        torch.cuda.synchronize()
    finally:
        rlk.withhold_copy(-1)
        rlk.set_wait_limit(0)
    assert old > 2_000_000
    assert int(st.item()) & rlk.STATUS_TIMEOUT
    cta0 = np.zeros(n, bool)
    cta0[::grid] = True
    lp_h, ent_h = lp.cpu().numpy(), ent.cpu().numpy()
    assert np.all(np.isnan(lp_h[cta0])) and np.all(np.isnan(ent_h[cta0]))
    same = lambda a, b: a.cpu().contiguous().view(torch.int32).numpy()[~cta0] == \
        b.cpu().contiguous().view(torch.int32).numpy()[~cta0]
    assert np.all(same(lp, lp0)) and np.all(same(ent, ent0))
    # the context is usable and the next call is clean
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp2, ent2 = rlk.logprob_entropy(z, ids, 0.7, p, status_word=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.equal(lp2.view(torch.int32), lp0.view(torch.int32))
    assert torch.equal(ent2.view(torch.int32), ent0.view(torch.int32))


def test_lmhead_withheld_copy_times_out_and_the_next_call_is_clean(cuda_lib):
    """The same for the fused LM-head kernel: its first CTA never gets one
    operand copy, so that CTA's units (m-tile, vocabulary slice) stay
    unfinished; every row of those m-tiles must be NaN, the rest bitwise
    equal to a clean call."""
    rlk = cuda_lib
    T, H, V, BM, NSLICE = 4096, 512, 20000, 128, 19
    hidden, w, ids = workloads.lmhead_inputs(T, H, V, seed=21, device="cuda")
    st0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp0, ent0 = rlk.lmhead_logprob(hidden, w, ids, 0.7, status_word=st0)
    torch.cuda.synchronize()
    assert int(st0.item()) == 0
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    n_units = ((T + BM - 1) // BM) * NSLICE
    grid = min(n_units, nsm)
    old = rlk.set_wait_limit(2_000_000)
    try:
        rlk.withhold_copy(5)                # the second k-step of CTA 0's second tile
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        lp, ent = rlk.lmhead_logprob(hidden, w, ids, 0.7, status_word=st)
        torch.cuda.synchronize()
    finally:
        rlk.withhold_copy(-1)
        rlk.set_wait_limit(0)
    assert old > 2_000_000
    assert int(st.item()) & rlk.STATUS_TIMEOUT
    n_mt = (T + BM - 1) // BM

    def unit_tile(u, block=4):              # the kernel's unit order: slices in blocks of 4
        full, nfb = n_mt * block, NSLICE // block
        if u // full < nfb:
            return (u % full) // block
        return (u - nfb * full) // (NSLICE - nfb * block)

    bad = np.zeros(T, bool)
    for u in range(0, n_units, grid):       # the units of CTA 0, all unfinished
        mt = unit_tile(u)
        bad[mt * BM:(mt + 1) * BM] = True
    lp_h, ent_h = lp.cpu().numpy(), ent.cpu().numpy()
    assert np.all(np.isnan(lp_h[bad])) and np.all(np.isnan(ent_h[bad]))
    bits = lambda t: t.cpu().contiguous().view(torch.int32).numpy()[~bad]
    assert np.array_equal(bits(lp), bits(lp0)) and np.array_equal(bits(ent), bits(ent0))
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp2, ent2 = rlk.lmhead_logprob(hidden, w, ids, 0.7, status_word=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.equal(lp2.view(torch.int32), lp0.view(torch.int32))
    assert torch.equal(ent2.view(torch.int32), ent0.view(torch.int32))
