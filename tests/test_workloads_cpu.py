"""The seeded input generators (CPU): draws are reproducible, any row subset
regenerates without the rest, and the exact-grid LM-head inputs really give
products exact in fp32 (a float32 library product, a float64 one and a sum in
reversed order agree bit for bit), which the LM-head top_p < 1 parity test
relies on."""
import numpy as np
import pytest
import torch

import workloads


def test_blocks_regenerate_independently():
    a, pa = workloads.peaked_bf16(2048 + 5, V=300, seed=3)
    b, pb = workloads.peaked_bf16(5, V=300, seed=3, row0=2048)
    assert torch.equal(a[2048:], b) and torch.equal(pa[2048:], pb)
    c, _ = workloads.peaked_bf16(2048 + 5, V=300, seed=3)
    assert torch.equal(a, c)


@pytest.mark.parametrize("H,V,s,L", [(256, 2000, 7, 7), (128, 1000, 2, 1), (4096, 600, 4, 1)])
def test_grid_lmhead_products_are_exact_in_fp32(H, V, s, L):
    h, w, ids = workloads.lmhead_grid_inputs(40, H, V, seed=14, wshift=s, levels=L)
    z64 = h.double() @ w.double().T
    z32 = h.float() @ w.float().T
    rev = (h.float().flip(1) @ w.float().flip(1).T)          # the other summation order
    assert torch.equal(z32.double(), z64) and torch.equal(rev.double(), z64)
    assert ids.dtype == torch.int32 and int(ids.min()) >= 0 and int(ids.max()) < V
    # values on the stated grid
    assert torch.equal((w.double() * 2.0 ** s).round(), w.double() * 2.0 ** s)
    assert float(h.abs().max()) <= L and float((w.double() * 2.0 ** s).abs().max()) <= L
