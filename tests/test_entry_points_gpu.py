"""One row, one set of bits: the same bf16 rows scored through every entry
point that takes them -- rlk_logprob_entropy, the same call saving the row
state (rlk_logprob_entropy_fwd), rlk_logprob_entropy_rows with uniform and
with mixed per-row parameters, and a copy of the batch laid out with an odd
row stride (rows that are not 16-byte aligned, read with scalar loads) --
must give byte-identical log-probabilities, entropies and nucleus sizes.
The pages' consistency run fails on any compared value that is not bitwise
equal (RL-Kernel "Qwen3-8B VIME train-rollout consistency", launcher and
validation; RL-Kernel "ROCm sparse performance" notes, raw FP32 audit).
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.detach().cpu().contiguous().view(torch.int32).numpy()


def _rows(V, seed):
    z, _ = workloads.peaked_bf16(48, V=V, seed=seed)
    z = z.float()
    g = torch.Generator().manual_seed(seed)
    z[1] = 1.5                                         # all equal
    z[2] = 0.0; z[2, V // 3] = 60.0                    # one-hot
    z[3, :64] = z[3].max() + 0.5                       # a wide tie group at the top
    z[4] = torch.randn(V, generator=g) * 0.5           # flat: the window crosses zero
    z[5] = torch.randn(V, generator=g) * 3 - 20.0      # all negative
    return z.to(torch.bfloat16)


def _score_all(rlk, z, ids, T, p):
    n, V = z.shape
    dev = z.device
    out = {}
    lp, ent, k = rlk.logprob_entropy(z, ids, T, p, return_nucleus_size=True)
    out["scalar"] = (lp, ent, k)
    st = rlk.new_row_state(n, dev)
    out["fwd"] = rlk.logprob_entropy(z, ids, T, p, return_nucleus_size=True, row_state=st)
    temps = torch.full((n,), T, dtype=torch.float32, device=dev)
    tps = torch.full((n,), p, dtype=torch.float32, device=dev)
    out["rows"] = rlk.logprob_entropy_rows(z, ids, temps, tps, return_nucleus_size=True)
    # odd stride: each row starts 2 bytes past a 16-byte boundary
    buf = torch.zeros((n, V + 5), dtype=torch.bfloat16, device=dev)
    zs = buf[:, 1:V + 1]
    zs.copy_(z)
    out["strided"] = rlk.logprob_entropy(zs, ids, T, p, return_nucleus_size=True)
    # mixed per-row parameters: the rows with (T, p) must match the scalar call
    mix_t = temps.clone()
    mix_p = tps.clone()
    mix_t[1::3] = 1.8
    mix_p[2::3] = 0.5 if p != 0.5 else 0.9
    out["mixed"] = rlk.logprob_entropy_rows(z, ids, mix_t, mix_p, return_nucleus_size=True)
    same = ((mix_t == T) & (mix_p == p)).cpu().numpy()
    torch.cuda.synchronize()
    return out, same


@pytest.mark.parametrize("V", [151936, 151931, 50000])
@pytest.mark.parametrize("T,p", [(0.7, 0.95), (0.7, 1.0), (1.8, 0.5)])
def test_entry_points_give_the_same_bits(cuda_lib, oracle, V, T, p):
    z = _rows(V, seed=7).cuda()
    hz = workloads.bf16_bits(z)
    ids = oracle.sample_ids(hz, T, p, workloads.uniforms(z.shape[0], 9)).astype(np.int32)
    ids[:4] = [0, V - 1, V // 2, 1]
    ids_d = torch.from_numpy(ids).cuda()
    out, same = _score_all(cuda_lib, z, ids_d, T, p)
    ref = [_bits(x) for x in out["scalar"]]
    for name in ("fwd", "rows", "strided"):
        got = [_bits(x) for x in out[name]]
        for r, g_, what in zip(ref, got, ("logprob", "entropy", "nucleus size")):
            bad = np.nonzero(r != g_)[0]
            assert bad.size == 0, f"{name}: {what} bits differ at rows {bad[:10]}"
    got = [_bits(x) for x in out["mixed"]]
    for r, g_, what in zip(ref, got, ("logprob", "entropy", "nucleus size")):
        bad = np.nonzero((r != g_) & same)[0]
        assert bad.size == 0, f"mixed: {what} bits differ at rows {bad[:10]}"
