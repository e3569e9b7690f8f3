"""Comparison helpers shared by the GPU parity tests."""
import numpy as np

LP_TOL = 2e-4      # |delta logprob| (absolute) ...
LP_REL = 2.0 ** -22  # ... plus ~2 ulp of the fp32 output, which cannot hold 2e-4
                     # absolute once |logprob| exceeds ~1e3 (rows of huge logits)
ENT_TOL = 2e-4     # |delta entropy| (absolute)
GAP_EXEMPT = 1e-6  # rows whose boundary mass gap is below this may differ in k*


def check_nucleus_sizes(oracle, logits_host, ids_host, temperature, top_p, k, *, ref=None,
                        label=""):
    """The GPU's nucleus sizes k against the oracle's.  Where the oracle's
    boundary gap is at least GAP_EXEMPT they must be equal.  Elsewhere the
    prefix mass sits within GAP_EXEMPT of top_p and more than one size is
    correct to within rounding: k must lie between the sizes the oracle
    selects at top_p - GAP_EXEMPT and at top_p + GAP_EXEMPT.  Returns the
    oracle's (logprob, entropy, k, gap)."""
    k = np.asarray(k, np.int64)
    if ref is None:
        ref = oracle.logprob_entropy(logits_host, ids_host, temperature, top_p)
    _, _, ok, gap = ref
    exempt = gap < GAP_EXEMPT
    bad_k = (~exempt) & (k != ok)
    assert not bad_k.any(), f"{label}: nucleus size differs at rows {np.nonzero(bad_k)[0][:10]}"
    if exempt.any():
        rows = np.nonzero(exempt)[0]
        sub = np.ascontiguousarray(np.asarray(logits_host)[rows])
        sid = np.ascontiguousarray(np.asarray(ids_host)[rows])
        lo = oracle.logprob_entropy(sub, sid, temperature, top_p - GAP_EXEMPT)[2]
        hi = oracle.logprob_entropy(sub, sid, temperature, min(top_p + GAP_EXEMPT, 1.0))[2]
        out = (k[rows] < lo) | (k[rows] > hi)
        assert not out.any(), f"{label}: nucleus size outside the rounding range at rows {rows[out][:10]}"
    return ref


def compare_rows(oracle, logits_host, ids_host, temperature, top_p, lp, ent, k, *, ref=None,
                 label=""):
    """Compare GPU outputs with the oracle row by row.

    Rows with gap >= GAP_EXEMPT must have the same nucleus size and outputs
    within tolerance; rows below it must have a size the oracle selects at a
    top_p within GAP_EXEMPT (check_nucleus_sizes), and are compared against
    the oracle evaluated at that size (both memberships are correct there).
    Returns a small report dict.
    """
    lp = np.asarray(lp, np.float64)
    ent = np.asarray(ent, np.float64)
    k = np.asarray(k, np.int64)
    if ref is None:
        ref = oracle.logprob_entropy(logits_host, ids_host, temperature, top_p)
    ref = check_nucleus_sizes(oracle, logits_host, ids_host, temperature, top_p, k, ref=ref,
                              label=label)
    olp, oent, ok, gap = ref
    exempt = gap < GAP_EXEMPT
    if exempt.any():
        rows = np.nonzero(exempt)[0]
        force = np.zeros_like(k)
        force[rows] = k[rows]
        flp, fent, _, _ = oracle.logprob_entropy(logits_host, ids_host, temperature, top_p,
                                                 force_k=force)
        olp = olp.copy()
        oent = oent.copy()
        olp[rows] = flp[rows]
        oent[rows] = fent[rows]
    inf_o = np.isneginf(olp)
    inf_g = np.isneginf(lp)
    assert np.array_equal(inf_o, inf_g), f"{label}: -inf membership differs at {np.nonzero(inf_o != inf_g)[0][:10]}"
    fin = ~inf_o
    dlp = np.abs(lp[fin] - olp[fin])
    dent = np.abs(ent - oent)
    assert np.all(np.isfinite(lp[fin])) and np.all(np.isfinite(ent)), f"{label}: non-finite output"
    tol = LP_TOL + LP_REL * np.abs(olp[fin])
    assert dlp.size == 0 or np.all(dlp <= tol), f"{label}: max |dlogprob| {dlp.max():.3e}"
    assert dent.max() <= ENT_TOL, f"{label}: max |dentropy| {dent.max():.3e}"
    return {"rows": int(lp.size), "gap_exempt": int(exempt.sum()),
            "max_dlp": float(dlp.max()) if dlp.size else 0.0, "max_dent": float(dent.max()),
            "members": int(fin.sum())}
