"""rlk_grpo_loss_noalloc through the C ABI.

This entry point serves callers that cannot allocate device memory -- a
framework that has reserved the whole device for its own pool, code running
inside an allocator callback, or a loop that bans cudaMalloc because it may
synchronise the device.  Its scratch lives in a static device array of the
library.  The test checks it against rlk_grpo_loss (caller-supplied
workspace) on the same inputs for every aggregation, on two calls in a row
(the second one reuses the array the first left behind).  Both run the same
three kernels in the same order on the same inputs, so the loss, the
gradient and the statistics must be bitwise equal.  Sizes beyond the array's
limit must be refused.  This file is collected last so a
run that stops at the first failure has run every other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point(cuda_lib):
    lib = cuda_lib.load()
    off, R = workloads.grpo_batch(16, 8, 64, 700, seed=11)
    n = int(off[-1])
    rng = np.random.default_rng(11)
    new = np.log(rng.uniform(1e-4, 1.0, n)).astype(np.float32)
    old, ro, ref = workloads.perturbed_logps(new, 11)
    ro[::37] -= np.float32(1.5)                      # some capped TIS weights
    mask = (rng.random(n) < 0.9).astype(np.uint8)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tn, to, tr, tf, tR, toff, tm = t(new), t(old), t(ro), t(ref), t(R), t(off), t(mask)
    n_seq = off.size - 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    bits = lambda t: t.cpu().contiguous().view(torch.int32).numpy()
    for agg in (0, 1, 2):
        ref_loss, ref_grad, ref_stats = cuda_lib.grpo_loss(tn, to, tr, tf, tR, toff, 8,
                                                           loss_mask=tm, agg=agg)
        torch.cuda.synchronize()
        for _ in range(2):
            loss = torch.full((1,), float("nan"), device="cuda")
            grad = torch.full((n,), float("nan"), device="cuda")
            stats = torch.full((cuda_lib.NSTATS,), float("nan"), device="cuda")
            code = lib.rlk_grpo_loss_noalloc(_ptr(tn), _ptr(to), _ptr(tr), _ptr(tf), _ptr(tm),
                                             _ptr(tR), _ptr(toff), n_seq, 8, n, 0.2, 0.28, 2.0,
                                             0.01, agg, _ptr(loss), _ptr(grad), _ptr(stats),
                                             stream)
            assert code == 0
            torch.cuda.synchronize()
            assert np.isfinite(loss.item())
            assert np.array_equal(bits(loss), bits(ref_loss)), f"agg {agg}: loss bits differ"
            assert np.array_equal(bits(grad), bits(ref_grad)), f"agg {agg}: gradient bits differ"
            assert np.array_equal(bits(stats), bits(ref_stats)), f"agg {agg}: statistics differ"


def test_noalloc_refuses_sizes_beyond_its_array(cuda_lib):
    lib = cuda_lib.load()
    fake = ctypes.c_void_p(0x10000)   # refused on the host before any device work
    too_many = cuda_lib.NOALLOC_MAX_SEQ + 8
    code = lib.rlk_grpo_loss_noalloc(fake, fake, fake, fake, None, fake, fake, too_many, 8, 10,
                                     0.2, 0.28, 2.0, 0.01, 0, fake, None, None, None)
    assert code == 1
