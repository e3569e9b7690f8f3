"""Full-size workloads through the C ABI, in the launch configuration the
benchmark times (16-byte aligned bf16 rows of V = 151,936):

* the long-response batch: 8 responses x 6912 tokens (T = 55,296, 16.8 GB of
  logits resident at once), Zipf-tilted rows whose nucleus sizes span a few to
  tens of thousands of tokens, temperature 0.7, top_p 0.95, with some rows
  given exact ties at the threshold.  Sampled rows are checked against the
  oracle one by one; properties that hold at any size are checked on every
  row; and the sampled rows run alone give the same bits as in the batch.
* the GRPO/DAPO batch: 64 prompts x group 8, response lengths 256..2048
  (about 590k packed tokens), logits as above generated chunk by chunk, the
  kernel's log-probs of each chunk feeding the loss.  Sampled tokens'
  log-probs are checked against the oracle; the loss read straight from the
  forward's device buffer must give the same bits as over the same values
  passed through host memory.  (The loss at this size is held to the oracle
  in test_grpo_loss_gpu.py on inputs drawn for both sides; no oracle input
  here comes from the GPU.)
"""
import numpy as np
import pytest
import torch

import workloads
from _parity import compare_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

MARKS = (0x7FC0DEAD, 0x7FC0DEAE)   # the recompute marks
T_CFG2 = 8 * 6912
TEMP, TOP_P = 0.7, 0.95


def _run(rlk, z, ids):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp, ent, k = rlk.logprob_entropy(z, ids, TEMP, TOP_P, return_nucleus_size=True,
                                     status_word=st)
    torch.cuda.synchronize()
    return lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy(), int(st.item())


def _tie_row(oracle, bits_row):
    """Give the row's threshold value to the three tokens ranked right after
    the boundary token; returns the new row and the largest tied id."""
    vals = (bits_row.astype(np.uint32) << 16).view(np.float32)
    _, _, k0, _ = oracle.logprob_entropy(bits_row[None], np.zeros(1, np.int32), TEMP, TOP_P)
    order = np.lexsort((np.arange(vals.size), -vals))
    b = order[k0[0] - 1]
    nxt = order[k0[0]:k0[0] + 3]
    out = bits_row.copy()
    out[nxt] = out[b]
    return out, int(max(nxt.max(), b))


def test_long_response_batch_full_size(cuda_lib, oracle):
    z, _ = workloads.zipf_bf16(T_CFG2, seed=2, device="cuda")
    V = z.shape[1]
    sample = np.linspace(0, T_CFG2 - 1, 192).astype(np.int64)
    hz = workloads.bf16_bits(z[torch.from_numpy(sample).cuda()])
    # 1 % of the batch's rows (here: of the sampled ones) get exact ties at the threshold
    tie_rows = sample[::50]
    tie_ids = {}
    for r in tie_rows:
        j = int(np.nonzero(sample == r)[0][0])
        hz[j], tie_ids[int(r)] = _tie_row(oracle, hz[j])
        z[int(r)] = torch.from_numpy(hz[j].view(np.int16)).view(torch.bfloat16).cuda()
    ids_s = oracle.sample_ids(hz, TEMP, TOP_P, workloads.uniforms(sample.size, 21))
    for r, y in tie_ids.items():
        ids_s[int(np.nonzero(sample == r)[0][0])] = y
    ids = torch.argmax(z, dim=1).to(torch.int32)          # every other row: its top token
    ids[torch.from_numpy(sample).cuda()] = torch.from_numpy(ids_s).cuda()

    lp, ent, k, status = _run(cuda_lib, z, ids)
    assert status == 0
    # properties of every row
    assert not np.isin(lp.view(np.uint32), MARKS).any()
    assert np.all(np.isfinite(lp) | np.isneginf(lp)) and np.all(np.isfinite(ent))
    assert np.all((k >= 1) & (k <= V))
    assert np.all(ent >= -1e-5) and np.all(ent <= np.log(k) + 1e-4)
    # sampled rows against the oracle
    rep = compare_rows(oracle, hz, ids_s, TEMP, TOP_P, lp[sample], ent[sample], k[sample],
                       label="long-response")
    print("long-response full-size parity:", rep, "nucleus sizes", int(k.min()), int(np.median(k)),
          int(k.max()))
    # the sampled rows alone: the same bits
    zs = z[torch.from_numpy(sample).cuda()].contiguous()
    lp1, ent1, k1, _ = _run(cuda_lib, zs, ids[torch.from_numpy(sample).cuda()].contiguous())
    assert lp1.tobytes() == lp[sample].tobytes() and ent1.tobytes() == ent[sample].tobytes()
    assert np.array_equal(k1, k[sample])


def test_grpo_batch_chained_full_size(cuda_lib, oracle):
    off, R = workloads.grpo_batch(64, 8, 256, 2048, seed=3)
    n = int(off[-1])
    chunk = 8192
    new = torch.empty(n, device="cuda")
    rng = np.random.default_rng(7)
    picked_bits, picked_ids, picked_rows = [], [], []
    for c0 in range(0, n, chunk):
        rows = min(chunk, n - c0)
        z, _ = workloads.zipf_bf16(rows, seed=1000 + c0 // chunk, device="cuda")
        ids = torch.argmax(z, dim=1).to(torch.int32)
        sel = np.sort(rng.choice(rows, 2, replace=False))
        hb = workloads.bf16_bits(z[torch.from_numpy(sel).cuda()])
        y = oracle.sample_ids(hb, TEMP, TOP_P, workloads.uniforms(2, c0))
        ids[torch.from_numpy(sel).cuda()] = torch.from_numpy(y).cuda()
        cuda_lib.logprob_entropy(z, ids, TEMP, TOP_P, out_logprob=new[c0:c0 + rows])
        picked_bits.append(hb)
        picked_ids.append(y)
        picked_rows.append(sel + c0)
        del z
    torch.cuda.synchronize()
    new_h = new.cpu().numpy()
    assert np.all(np.isfinite(new_h))
    rows = np.concatenate(picked_rows)
    hb = np.concatenate(picked_bits)
    y = np.concatenate(picked_ids)
    olp, _, _, _ = oracle.logprob_entropy(hb, y, TEMP, TOP_P)
    fin = np.isfinite(olp)
    assert np.array_equal(fin, np.isfinite(new_h[rows]))
    assert np.all(np.abs(new_h[rows][fin] - olp[fin]) <= 2e-4 + 2.0 ** -22 * np.abs(olp[fin]))
    # the loss on these log-probs, straight from the device buffer the
    # forward wrote: the same bits as the loss over those values passed
    # through host memory (the loss itself is held to the oracle on this
    # batch size by test_grpo_loss_gpu.py, on inputs the oracle shares)
    old, ro, ref = workloads.perturbed_logps(new_h, 5)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    loss, grad, _ = cuda_lib.grpo_loss(new, t(old), t(ro), t(ref), t(R), t(off), 8)
    loss2, grad2, _ = cuda_lib.grpo_loss(t(new_h), t(old), t(ro), t(ref), t(R), t(off), 8)
    torch.cuda.synchronize()
    assert torch.equal(loss, loss2) and torch.equal(grad, grad2)
    assert np.isfinite(loss.item()) and bool(torch.isfinite(grad).all())
    print(f"GRPO full-size chained: {n} tokens, loss {loss.item():.6f}")
