"""The per-row kernel's window pass on dense rows (a quarter of the groups
or more reach the window: near-flat rows, wide nuclei), where each thread
counts its own groups in place, against the oracle.  The selected id is put
on each side of the boundary's tie group -- its lowest id, the last id kept
and the first id dropped when top_p splits the group -- so the count of the
selected value's ties ahead of it decides membership.  Vocabularies: the
benchmark's (such rows cross zero with thousands of near-zero tokens and
the streaming kernel hands them on), one with a partial last group read
from rows that are not 16-byte aligned, a short one the per-row kernel
takes directly, and one too long for the group-max sketch (the queued
pass)."""
import numpy as np
import pytest
import torch

import workloads
from _parity import compare_rows

pytestmark = pytest.mark.gpu


def _values(hz):
    return (hz.astype(np.uint32) << 16).view(np.float32)


def _rows(V, seed):
    g = torch.Generator().manual_seed(seed)
    rows = [
        torch.round(torch.randn(V, generator=g) * 8) / 16,       # 0.5 N(0,1) on a 1/16 grid
        torch.randn(V, generator=g) * 1.3,                       # a random-init LM head's rows
        torch.round(torch.randn(V, generator=g) * 8) / 4,        # N(0, 4) on a 1/4 grid
        torch.round(torch.randn(V, generator=g) * 4) / 4 - 6.0,  # the same, all below zero
    ]
    return torch.stack(rows).to(torch.bfloat16)


def _boundary_ids(oracle, hz, temp, p):
    """Per row, three ids: the boundary tie group's lowest id, the last id
    kept, and the first id dropped (the group's last id if none is)."""
    n, V = hz.shape
    k = oracle.logprob_entropy(hz, np.zeros(n, np.int32), temp, p)[2]
    vals = _values(hz)
    ids = []
    for r in range(n):
        order = np.lexsort((np.arange(V), -vals[r]))   # value descending, id ascending
        b = vals[r, order[k[r] - 1]]
        group = np.nonzero(vals[r] == b)[0]
        kept = int(k[r] - np.count_nonzero(vals[r] > b))
        drop = group[kept] if kept < len(group) else group[-1]
        ids.append([group[0], group[kept - 1], drop])
    return np.asarray(ids, np.int32)


@pytest.mark.parametrize("V,off", [(151936, 0), (151931, 1), (5003, 0), (200003, 0)])
@pytest.mark.parametrize("temp,p", [(0.7, 0.9), (1.0, 0.5)])
def test_dense_rows_at_the_boundary(cuda_lib, oracle, V, off, temp, p):
    base = _rows(V, seed=V % 1000 + 7)
    hz0 = workloads.bf16_bits(base)
    ids = _boundary_ids(oracle, hz0, temp, p)
    z = base.repeat_interleave(3, dim=0)
    ids = ids.reshape(-1)
    n = z.shape[0]
    buf = torch.zeros((n, V + off + 3), dtype=torch.bfloat16, device="cuda")
    zd = buf[:, off:off + V]
    zd.copy_(z.cuda())
    hz = workloads.bf16_bits(zd)
    st = cuda_lib.new_row_state(n, zd.device)
    lp, ent, k = cuda_lib.logprob_entropy(zd, torch.from_numpy(ids).cuda(), temp, p,
                                          return_nucleus_size=True, row_state=st)
    torch.cuda.synchronize()
    compare_rows(oracle, hz, ids, temp, p, lp.cpu().numpy(), ent.cpu().numpy(), k.cpu().numpy(),
                 label=f"dense V={V} off={off} T={temp} p={p}")
    # the lowest id of the boundary group is always kept
    assert np.isfinite(lp.cpu().numpy()[0::3]).all()
    if V == 151936:
        # the streaming kernel hands these rows on (its reference exponent is
        # an integer, the per-row kernel's is not)
        E = st[:, 0].contiguous().view(torch.float32).cpu().numpy()
        assert (E[:3] != np.floor(E[:3])).all()
