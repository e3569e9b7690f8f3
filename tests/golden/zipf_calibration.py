"""Calibrates the long-response (Zipf-tilted) workload and writes
zipf_calibration.txt beside this file.

The long-response configuration asks for rows whose top-p nucleus sizes span
1 to about 5000 at temperature 0.7 and top_p 0.95.  The row recipe
(workloads.zipf_bf16: z_i = bf16(-kappa s ln rank(i) + sigma N(0,1)), s ~
U(0.8, 1.4) per row) does not fix kappa and sigma, so they are chosen here:
the fp64 oracle scores 1024 rows for each candidate kappa (sigma 0.5), and the
smallest kappa whose largest nucleus is at most ~5500 is kept.  The file
records the candidates' nucleus-size percentiles and the chosen pair's
histogram.  Only the oracle and the seeded input generator run here.

    python tests/golden/zipf_calibration.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads  # noqa: E402

ROWS, TEMPERATURE, TOP_P, SIGMA = 1024, 0.7, 0.95, 0.5
CANDIDATES = (1.0, 1.1, 1.15, 1.2, 1.3)
LIMIT = 5500


def main():
    oracle.build()
    lines = [f"# Zipf-tilted rows, V={workloads.VOCAB}, {ROWS} rows (seed 2), temperature "
             f"{TEMPERATURE}, top_p {TOP_P}, sigma {SIGMA}; nucleus sizes k* from the fp64 oracle",
             "# kappa  min  p10  median  p90  p99  max"]
    chosen = None
    for kappa in CANDIDATES:
        z, _ = workloads.zipf_bf16(ROWS, seed=2, kappa=kappa, sigma=SIGMA)
        hz = workloads.bf16_bits(z)
        _, _, k, _ = oracle.logprob_entropy(hz, np.zeros(ROWS, np.int32), TEMPERATURE, TOP_P)
        q = np.percentile(k, [10, 50, 90, 99])
        lines.append(f"{kappa:.2f} {k.min()} {q[0]:.0f} {q[1]:.0f} {q[2]:.0f} {q[3]:.0f} {k.max()}")
        if chosen is None and k.max() <= LIMIT:
            chosen = (kappa, k)
    kappa, k = chosen
    edges = [1, 2, 5, 10, 20, 50, 100, 200, 500, 1000, 2000, 5000, 10000, 200000]
    hist = np.histogram(k, bins=edges)[0]
    lines.append(f"chosen kappa {kappa:.2f} sigma {SIGMA}")
    lines.append("# k* histogram: [lo, hi) count")
    for lo, hi, n in zip(edges[:-1], edges[1:], hist):
        lines.append(f"[{lo}, {hi}) {n}")
    with open(os.path.join(HERE, "zipf_calibration.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")
    print("\n".join(lines))


if __name__ == "__main__":
    main()
