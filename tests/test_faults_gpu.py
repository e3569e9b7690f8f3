"""Failure handling on the GPU without a GPU fault.

- Host-side injected launch failures: an entry point whose arguments are good
  returns RLK_ERR_CUDA without launching, leaves its outputs untouched, and
  the next call works.
- Canaries: every output buffer sits inside a larger buffer filled with a
  sentinel; after the call the sentinel must be intact outside the output
  (no write lands outside what the ABI says is written).
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

PAD = 4096
SENT = 1.2345e-3


def guarded(n, dtype=torch.float32, fill=SENT):
    buf = torch.full((n + 2 * PAD,), fill, dtype=dtype, device="cuda")
    return buf, buf[PAD:PAD + n]


def intact(buf, n, fill=SENT):
    torch.cuda.synchronize()
    return bool((buf[:PAD] == fill).all()) and bool((buf[PAD + n:] == fill).all())


def test_injected_failure_leaves_outputs_and_recovers(cuda_lib):
    z, _ = workloads.peaked_bf16(16, V=151936, seed=3, device="cuda")
    ids = torch.zeros(16, dtype=torch.int32, device="cuda")
    lp = torch.full((16,), 7.0, device="cuda")
    ent = torch.full((16,), 7.0, device="cuda")
    assert cuda_lib.inject_launch_failures(1) == 0
    with pytest.raises(cuda_lib.RlkError):
        cuda_lib.logprob_entropy(z, ids, 0.7, 0.95, out_logprob=lp, out_entropy=ent)
    torch.cuda.synchronize()
    assert bool((lp == 7.0).all()) and bool((ent == 7.0).all())
    cuda_lib.logprob_entropy(z, ids, 0.7, 0.95, out_logprob=lp, out_entropy=ent)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(ent).all())
    # the loss and the LM-head take the same path
    off = torch.tensor([0, 3, 6], dtype=torch.int32, device="cuda")
    x = torch.full((6,), -1.0, device="cuda")
    r = torch.tensor([1.0, 0.0], device="cuda")
    assert cuda_lib.inject_launch_failures(2) == 0
    with pytest.raises(cuda_lib.RlkError):
        cuda_lib.grpo_loss(x, x, x, x, r, off, 2)
    h, w, hid = workloads.lmhead_inputs(128, 128, 1000, seed=1, device="cuda")
    with pytest.raises(cuda_lib.RlkError):
        cuda_lib.lmhead_logprob(h, w, hid, 0.7)
    assert cuda_lib.inject_launch_failures(0) == 0
    loss, _, _ = cuda_lib.grpo_loss(x, x, x, x, r, off, 2)
    torch.cuda.synchronize()
    assert torch.isfinite(loss).all()


def test_canaries_around_every_output(cuda_lib):
    T, V = 40, 151936
    z, _ = workloads.peaked_bf16(T, V=V, seed=5, device="cuda")
    ids = torch.randint(0, V, (T,), dtype=torch.int32, device="cuda")
    # forward outputs and the row state
    blp, lp = guarded(T)
    bent, ent = guarded(T)
    bst, st = guarded(T * 8, torch.int32, 0x5A5A5A5A)
    cuda_lib.logprob_entropy(z, ids, 0.7, 0.95, out_logprob=lp, out_entropy=ent,
                             row_state=st.view(T, 8))
    assert intact(blp, T) and intact(bent, T) and intact(bst, T * 8, 0x5A5A5A5A)
    # dense backward into a strided gradient: the row padding must stay too
    bg, gflat = guarded(T * (V + 16), torch.bfloat16, 3.0)
    g = gflat.view(T, V + 16)[:, :V]
    cuda_lib.logprob_entropy_backward(z, ids, 0.7, st.view(T, 8), torch.ones(T, device="cuda"),
                                      torch.ones(T, device="cuda"), out=g)
    assert intact(bg, T * (V + 16), 3.0)
    assert bool((gflat.view(T, V + 16)[:, V:] == 3.0).all())
    # supplied support and its backward
    k = 300
    off = torch.arange(0, (T + 1) * k, k, dtype=torch.int64, device="cuda")
    sup = torch.topk(z.float(), k, dim=1).indices.to(torch.int32).reshape(-1).contiguous()
    bsl, slp = guarded(T)
    bse, sent = guarded(T)
    cuda_lib.logprob_entropy_support(z, ids, 0.7, off, sup, out_logprob=slp, out_entropy=sent)
    assert intact(bsl, T) and intact(bse, T)
    bsg, sg = guarded(T * k)
    cuda_lib.logprob_entropy_support_backward(z, ids, 0.7, off, sup, torch.ones(T, device="cuda"),
                                              None, out=sg)
    assert intact(bsg, T * k)
    # canonical partials and the sampler
    lib = cuda_lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    bp, pflat = guarded(8 * T * 8)
    code = lib.rlk_shard_partials(z.data_ptr(), 0, T, V, V, 0, 19072, 8, ids.data_ptr(), 0.7,
                                  pflat.data_ptr(), stream)
    assert code == 0 and intact(bp, 8 * T * 8)
    bid, sid = guarded(T, torch.int32, 0x77777777)
    u = torch.rand(T, device="cuda")
    code = lib.rlk_sample_top_p(z.data_ptr(), 0, T, V, V, 0.7, st.data_ptr(), u.data_ptr(),
                                sid.data_ptr(), None, stream)
    assert code == 0 and intact(bid, T, 0x77777777)
    # the loss gradient
    n_tok = 6 * 50
    offs = torch.arange(0, n_tok + 1, 50, dtype=torch.int32, device="cuda")
    lpn = torch.log(torch.rand(n_tok, device="cuda") * 0.9 + 0.05)
    bl, lg = guarded(n_tok)
    wsz = cuda_lib.workspace_size(cuda_lib.OP_GRPO_LOSS, n_tok, 6, 0)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, device="cuda")
    rew = torch.rand(6, device="cuda")
    code = lib.rlk_grpo_loss(lpn.data_ptr(), lpn.data_ptr(), lpn.data_ptr(), lpn.data_ptr(), None,
                             rew.data_ptr(), offs.data_ptr(), 6, 3, n_tok,
                             0.2, 0.28, 2.0, 0.01, 0, loss.data_ptr(), lg.data_ptr(), None,
                             ws.data_ptr(), wsz, stream)
    assert code == 0 and intact(bl, n_tok)
