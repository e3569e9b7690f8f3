"""CUDA-graph capture of the training-side chain: forward with row state,
dense backward, sampler, the loss variants, and the LM-head forward and
backward (whose weight-side products are the library's tcgen05 GEMMs).  After one eager
warm-up (lazy attribute and handle set-up happens there), a captured graph
replays to the eager results bit for bit, and again after the inputs change
in place: nothing in these calls synchronises, allocates on its own or
depends on host state that a replay would not refresh.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _chain(rlk, z, ids, u, glp, gh, st, grad, lpo, ento, idso, loss_in, lossbufs, lm):
    rlk.logprob_entropy(z, ids, 0.7, 0.95, out_logprob=lpo, out_entropy=ento, row_state=st)
    rlk.logprob_entropy_backward(z, ids, 0.7, st, glp, gh, out=grad)
    idso.copy_(rlk.sample_top_p(z, 0.7, 0.95, u, row_state=st))
    new, old, ro, ref, rew, off = loss_in
    loss, lgrad, stats = rlk.policy_loss(new, old, ro, ref, rew, off, 4, loss_type=rlk.LOSS_IPO,
                                         is_method=rlk.IS_MIS, kl_coef=0.0,
                                         workspace=lossbufs[3])
    lossbufs[0].copy_(loss)
    lossbufs[1].copy_(lgrad)
    lossbufs[2].copy_(stats)
    h, w, hid, lse, lm_out, lm_ws, dh, dw, lm_g = lm
    lp, ent = rlk.lmhead_logprob(h, w, hid, 0.7, out_lse=lse, workspace=lm_ws[0])
    lm_out[0].copy_(lp)
    lm_out[1].copy_(ent)
    rlk.lmhead_backward(h, w, hid, 0.7, lse, ent, lm_g[0], lm_g[1],
                        grad_hidden=dh, grad_w=dw, workspace=lm_ws[1])


def test_training_chain_under_graph_capture(cuda_lib):
    rlk = cuda_lib
    R, V = 64, workloads.VOCAB
    z, _ = workloads.peaked_bf16(R, V=V, seed=71, device="cuda")
    ids = z.float().argmax(1).to(torch.int32)      # ranked first: always in the nucleus
    u = torch.rand(R, device="cuda")
    glp = torch.rand(R, device="cuda") - 0.5
    gh = torch.rand(R, device="cuda") - 0.5
    st = rlk.new_row_state(R, "cuda")
    grad = torch.empty((R, V), device="cuda", dtype=torch.bfloat16)
    lpo, ento = torch.empty(R, device="cuda"), torch.empty(R, device="cuda")
    idso = torch.empty(R, dtype=torch.int32, device="cuda")
    off = torch.arange(0, 8 * 40 + 1, 40, dtype=torch.int32, device="cuda")
    n_tok = 8 * 40
    g = torch.Generator(device="cuda").manual_seed(3)
    new = torch.log(torch.rand(n_tok, device="cuda", generator=g) * 0.9 + 0.05)
    loss_in = (new, new + 0.01, new - 0.02, new + 0.03, torch.tensor([1., 0., 1., 1., 0., 0., 1., 0.],
               device="cuda"), off)
    lossbufs = (torch.empty(1, device="cuda"), torch.empty(n_tok, device="cuda"),
                torch.empty(rlk.NSTATS_POLICY, device="cuda"),
                torch.empty(rlk.workspace_size(rlk.OP_GRPO_LOSS, n_tok, 8, 0), dtype=torch.uint8,
                            device="cuda"))
    T2, H, V2 = 256, 256, 5000
    h, w, hid = workloads.lmhead_inputs(T2, H, V2, seed=5, device="cuda")
    lm = (h, w, hid, torch.empty(T2, device="cuda"),
          (torch.empty(T2, device="cuda"), torch.empty(T2, device="cuda")),
          (torch.empty(rlk.workspace_size(rlk.OP_LMHEAD, T2, V2, H), dtype=torch.uint8,
                       device="cuda"),
           torch.empty(rlk.workspace_size(rlk.OP_LMHEAD_BWD, T2, V2, H), dtype=torch.uint8,
                       device="cuda")),
          torch.empty((T2, H), device="cuda"), torch.empty((V2, H), device="cuda"),
          (torch.rand(T2, device="cuda") - 0.5, torch.rand(T2, device="cuda") - 0.5))
    outs = lambda: [t.clone() for t in (lpo, ento, grad, idso, *lossbufs[:3], *lm[4], lm[6], lm[7])]
    args = (rlk, z, ids, u, glp, gh, st, grad, lpo, ento, idso, loss_in, lossbufs, lm)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # eager warm-up: lazy set-up happens here
        _chain(*args)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = outs()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _chain(*args)
    for t in (lpo, ento, idso, lossbufs[0]):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs()):
        assert torch.equal(a, b)
    # new inputs in place: the replay follows them
    z2, _ = workloads.peaked_bf16(R, V=V, seed=72, device="cuda")
    z.copy_(z2)
    u.copy_(torch.rand(R, device="cuda"))
    h.copy_(workloads.lmhead_inputs(T2, H, V2, seed=6, device="cuda")[0])
    graph.replay()
    torch.cuda.synchronize()
    replayed = outs()
    with torch.cuda.stream(s):
        _chain(*args)
    torch.cuda.synchronize()
    for a, b in zip(replayed, outs()):
        assert torch.equal(a, b)
    assert torch.isfinite(eager[0]).all()               # finite log-probabilities
    assert not torch.equal(replayed[1], eager[1])       # the forward saw the new logits
    assert not torch.equal(replayed[7], eager[7])       # the LM-head saw the new hidden
