"""Seeded synthetic inputs for the logits path, the GRPO/DAPO loss and the LM-head.

This module holds random draws and data layout only -- none of the method's
arithmetic -- so that both the oracle and the CUDA path can be fed from it.
The real model and dataset the pages measure on (Qwen3-8B, DAPO-Math-17k) are
not available; these generators stand in for their shapes: vocabulary
151,936, temperature 0.7, top-p 0.95, group size 8, responses up to 6,912
tokens.

Large tensors are drawn in fixed blocks of ``BLOCK_ROWS`` rows, each block from
its own generator seeded by (seed, block index), so any subset of rows can be
regenerated without drawing the rest and the values never depend on how many
rows a caller asks for at once.
"""
from __future__ import annotations

import math

import numpy as np
import torch

BLOCK_ROWS = 1024
VOCAB = 151936          # Qwen3 vocabulary without padding
TEMPERATURE = 0.7
TOP_P = 0.95


def _gen(seed: int, block: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(block) * 7_919 + 12_345) % (2**63 - 1))
    return g


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns (for the oracle)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def uniforms(n: int, seed: int) -> np.ndarray:
    """Per-row uniforms in [0, 1) (float64), e.g. for inverse-CDF id draws."""
    return np.random.default_rng([int(seed), 0xC0FFEE]).random(int(n))


def uniform_ids(n: int, V: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, 10_000_019, device)
    return torch.randint(0, V, (int(n),), generator=g, device=device, dtype=torch.int64).to(torch.int32)


def normal_logits_fp32(T: int, V: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 logits, i.i.d. N(0, std^2)."""
    g = _gen(seed, 0, device)
    return torch.randn(T, V, generator=g, device=device, dtype=torch.float32) * float(std)


def tiny(seed: int = 0, device="cpu"):
    """Tiny case: T=64, V=1000, fp32 N(0, 2^2), ids uniform in [0, V)."""
    T, V = 64, 1000
    z = normal_logits_fp32(T, V, 2.0, seed, device)
    return z, uniform_ids(T, V, seed, device)


def brute_v8(seed: int = 0, device="cpu"):
    """Brute-force case: T=16, V=8, fp32 N(0, 2^2), ids uniform in [0, 8)."""
    T, V = 16, 8
    z = normal_logits_fp32(T, V, 2.0, seed + 101, device)
    return z, uniform_ids(T, V, seed + 101, device)


def peaked_bf16(T: int, V: int = VOCAB, seed: int = 1, device="cpu", row0: int = 0):
    """Qwen3-8B-shaped rows: bf16(3 N(0,1)), plus one peaked token per row whose
    logit gets + U(5, 15) before the (round-to-nearest-even) bf16 rounding.

    Returns (logits bf16 [T, V], peak ids int32 [T]).  ``row0`` selects the
    first global row, so chunks of a larger batch can be drawn on their own
    (row0 must be a multiple of BLOCK_ROWS).
    """
    assert row0 % BLOCK_ROWS == 0
    out = torch.empty(T, V, dtype=torch.bfloat16, device=device)
    peaks = torch.empty(T, dtype=torch.int32, device=device)
    for r in range(0, T, BLOCK_ROWS):
        n = min(BLOCK_ROWS, T - r)
        g = _gen(seed, (row0 + r) // BLOCK_ROWS, device)
        z = torch.randn(BLOCK_ROWS, V, generator=g, device=device, dtype=torch.float32)[:n]
        z.mul_(3.0)
        pid = torch.randint(0, V, (BLOCK_ROWS,), generator=g, device=device)[:n]
        bump = (torch.rand(BLOCK_ROWS, generator=g, device=device) * 10.0 + 5.0)[:n]
        rows = torch.arange(n, device=device)
        z[rows, pid] += bump
        out[r:r + n] = z.to(torch.bfloat16)
        peaks[r:r + n] = pid.to(torch.int32)
    return out, peaks


# The long-response configuration's rows, calibrated so that their nucleus
# sizes at temperature 0.7 / top_p 0.95 span 1 to ~5000 (tests/golden/
# zipf_calibration.py, whose output zipf_calibration.txt records the
# candidates and the histogram).  kappa = 1.0 gives a wider stress batch
# (nuclei up to ~34,000 tokens).
ZIPF_KAPPA_CALIBRATED = 1.15
ZIPF_SIGMA = 0.5


def zipf_bf16(T: int, V: int = VOCAB, seed: int = 2, kappa: float = 1.0, sigma: float = 0.5,
              device="cpu"):
    """Long-response rows with Zipf-tilted means.

    Per row: exponent s ~ U(0.8, 1.4); a row-specific permutation
    rank(i) = ((a i + b) mod V) + 1 with a coprime to V; logit
    z_i = bf16(-kappa s ln rank(i) + sigma N(0,1)).
    Returns (logits bf16 [T, V], s float32 [T]).
    """
    out = torch.empty(T, V, dtype=torch.bfloat16, device=device)
    svals = torch.empty(T, dtype=torch.float32, device=device)
    idx = torch.arange(V, device=device, dtype=torch.int64)
    for r in range(0, T, BLOCK_ROWS):
        n = min(BLOCK_ROWS, T - r)
        g = _gen(seed, r // BLOCK_ROWS, device)
        noise = torch.randn(BLOCK_ROWS, V, generator=g, device=device, dtype=torch.float32)[:n]
        s = (torch.rand(BLOCK_ROWS, generator=g, device=device) * 0.6 + 0.8)[:n]
        rng = np.random.default_rng([int(seed), r // BLOCK_ROWS, 77])
        a_list, b_list = [], []
        for _ in range(n):
            while True:
                a = int(rng.integers(1, V)) | 1
                if math.gcd(a, V) == 1:
                    break
            a_list.append(a)
            b_list.append(int(rng.integers(0, V)))
        a_t = torch.tensor(a_list, device=device, dtype=torch.int64)[:, None]
        b_t = torch.tensor(b_list, device=device, dtype=torch.int64)[:, None]
        rank = ((a_t * idx[None, :] + b_t) % V + 1).to(torch.float32)
        z = -float(kappa) * s[:, None] * torch.log(rank) + float(sigma) * noise
        out[r:r + n] = z.to(torch.bfloat16)
        svals[r:r + n] = s
    return out, svals


def grpo_batch(n_prompts: int = 64, group: int = 8, len_lo: int = 256, len_hi: int = 2048,
               seed: int = 3):
    """Packed ragged GRPO batch layout: response lengths ~ U{len_lo..len_hi},
    CSR offsets [n_seq + 1] (int32), rewards ~ Bernoulli(0.5) per sequence."""
    rng = np.random.default_rng([int(seed), 4242])
    n_seq = n_prompts * group
    lengths = rng.integers(len_lo, len_hi + 1, size=n_seq)
    offsets = np.zeros(n_seq + 1, np.int32)
    offsets[1:] = np.cumsum(lengths)
    rewards = (rng.random(n_seq) < 0.5).astype(np.float32)
    return offsets, rewards


def perturbed_logps(logp_new: np.ndarray, seed: int, std: float = 0.01):
    """old / rollout / ref log-probs = new + independent N(0, std^2), as float32."""
    rng = np.random.default_rng([int(seed), 999])
    new = np.asarray(logp_new, dtype=np.float32)
    outs = []
    for _ in range(3):
        outs.append((new.astype(np.float64) + rng.normal(0.0, std, new.shape)).astype(np.float32))
    return tuple(outs)


def lmhead_inputs(T: int, H: int, V: int, seed: int = 4, device="cpu"):
    """hidden bf16 [T, H] ~ N(0,1); W bf16 [V, H] ~ N(0, 0.02^2); ids uniform."""
    hidden = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    for r in range(0, T, BLOCK_ROWS):
        n = min(BLOCK_ROWS, T - r)
        g = _gen(seed, r // BLOCK_ROWS, device)
        hidden[r:r + n] = torch.randn(BLOCK_ROWS, H, generator=g, device=device)[:n].to(torch.bfloat16)
    w = torch.empty(V, H, dtype=torch.bfloat16, device=device)
    for r in range(0, V, 8192):
        n = min(8192, V - r)
        g = _gen(seed + 500, r // 8192, device)
        w[r:r + n] = (torch.randn(8192, H, generator=g, device=device)[:n] * 0.02).to(torch.bfloat16)
    return hidden, w, uniform_ids(T, V, seed, device)


def lmhead_grid_inputs(T: int, H: int, V: int, seed: int = 6, wshift: int = 4, levels: int = 1,
                       device="cpu"):
    """hidden and W on small integer grids: hidden uniform in {-L, ..., L},
    W uniform in {-L, ..., L} * 2^-wshift (L = levels), ids uniform.  Every
    partial sum of a dot product is a multiple of 2^-wshift of magnitude at
    most H L^2 2^-wshift (below 2^24 of those steps here), exact in fp32
    whatever the summation order, so a tensor-core product and a library
    product give the same logits bit for bit.  z has standard deviation
    sqrt(H) (L (L + 1) / 3) 2^-wshift; once |z| 2^wshift passes 256 the
    logits no longer fit bf16 and rounding them is exercised."""
    hidden = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    for r in range(0, T, BLOCK_ROWS):
        n = min(BLOCK_ROWS, T - r)
        g = _gen(seed, r // BLOCK_ROWS, device)
        hidden[r:r + n] = torch.randint(-levels, levels + 1, (BLOCK_ROWS, H), generator=g,
                                        device=device)[:n].to(torch.bfloat16)
    w = torch.empty(V, H, dtype=torch.bfloat16, device=device)
    for r in range(0, V, 8192):
        n = min(8192, V - r)
        g = _gen(seed + 700, r // 8192, device)
        w[r:r + n] = (torch.randint(-levels, levels + 1, (8192, H), generator=g,
                                    device=device)[:n].float() * 2.0 ** -wshift).to(torch.bfloat16)
    return hidden, w, uniform_ids(T, V, seed, device)
