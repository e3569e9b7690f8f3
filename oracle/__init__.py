"""fp64 CPU oracle for the top-p logprob/entropy path and the GRPO/DAPO loss.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports this package; only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` do.  It shares no code with the CUDA
path.  The arithmetic lives in ``oracle.cpp`` (plain C++17, fp64, full sort,
explicit nucleus); this module compiles it with g++ and marshals numpy arrays.

Every function here is pinned by ``tests/test_oracle_pins.py`` against brute
force, closed forms, library routines, invariants and hand-worked values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Statistic slots of grpo_loss (same order as the library's statistics).
STAT_NAMES = ("loss", "tokens", "clip_low_frac", "clip_high_frac", "tis_mean",
              "tis_capped_frac", "k3_mean", "pg_mean")


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so (host code only, portable flags)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, i32, f32, vp, i = (ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                   ctypes.c_void_p, ctypes.c_int)
            lib.oracle_logprob_entropy.argtypes = [vp, i, i64, i64, i64, vp, f32, f32, vp,
                                                   vp, vp, vp, vp, i]
            lib.oracle_sample_ids.argtypes = [vp, i, i64, i64, i64, f32, f32, vp, vp, i]
            lib.oracle_logprob_entropy_support.argtypes = [vp, i, i64, i64, i64, vp, f32, vp, vp,
                                                           vp, vp, vp, i]
            lib.oracle_logprob_entropy_support_backward.argtypes = [vp, i, i64, i64, i64, vp, f32,
                                                                    vp, vp, vp, vp, vp, i]
            lib.oracle_logprob_entropy_backward.argtypes = [vp, i, i64, i64, i64, vp, f32, f32,
                                                            vp, vp, vp, vp, i]
            lib.oracle_policy_loss.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i, f32, f32,
                                               f32, f32, f32, i, f32, f32, i, i, vp, vp, vp, vp]
            lib.oracle_lmhead_backward.argtypes = [vp, vp, i64, i64, i64, vp, f32, f32, vp, vp,
                                                   vp, vp, i]
            lib.oracle_grpo_loss.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, f32,
                                             f32, f32, i, vp, vp, vp, vp]
            lib.oracle_lmhead_rows.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp, f32, f32,
                                               vp, vp, vp, i]
            for fn in (lib.oracle_logprob_entropy, lib.oracle_sample_ids,
                       lib.oracle_logprob_entropy_support,
                       lib.oracle_logprob_entropy_support_backward,
                       lib.oracle_logprob_entropy_backward, lib.oracle_policy_loss,
                       lib.oracle_lmhead_backward, lib.oracle_grpo_loss, lib.oracle_lmhead_rows):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits_array(logits):
    """Accept a numpy float32 array, or uint16 bf16 bit patterns (dtype bf16)."""
    a = np.asarray(logits)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), 0
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), 1
    raise TypeError("oracle logits must be float32 or uint16 (bf16 bit patterns)")


def logprob_entropy(logits, ids, temperature, top_p, force_k=None, threads=None):
    """Score every row of ``logits`` [T, V]; returns (logprob, entropy, k, gap).

    ``temperature`` and ``top_p`` are rounded to float32 first, exactly like the
    values the library receives.  ``force_k`` evaluates rows at a given nucleus
    size instead of k* (entries <= 0 mean k*).
    """
    a, dt = _logits_array(logits)
    if a.ndim != 2:
        raise ValueError("logits must be 2-D")
    T, V = a.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    assert ids.shape == (T,)
    lp = np.empty(T, np.float64)
    ent = np.empty(T, np.float64)
    k = np.empty(T, np.int64)
    gap = np.empty(T, np.float64)
    fk = None if force_k is None else np.ascontiguousarray(force_k, dtype=np.int64)
    rc = _load().oracle_logprob_entropy(_ptr(a), dt, T, V, V, _ptr(ids),
                                        float(np.float32(temperature)),
                                        float(np.float32(top_p)), _ptr(fk), _ptr(lp),
                                        _ptr(ent), _ptr(k), _ptr(gap),
                                        threads or default_threads())
    if rc:
        raise ValueError("oracle_logprob_entropy rejected its arguments")
    return lp, ent, k, gap


def logprob_entropy_support(logits, ids, temperature, offsets, support_ids, threads=None):
    """Score every row of ``logits`` [T, V] over a supplied retained set: row r
    keeps the ids ``support_ids[offsets[r]:offsets[r+1]]``.  Returns (logprob,
    entropy, status) with status 0, 1 (bad selected id), 2 (non-finite listed
    logit) or 8 (empty list, listed id out of range, decreasing offsets)."""
    a, dt = _logits_array(logits)
    if a.ndim != 2:
        raise ValueError("logits must be 2-D")
    T, V = a.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    sup = np.ascontiguousarray(support_ids, dtype=np.int32)
    assert ids.shape == (T,) and off.shape == (T + 1,)
    lp = np.empty(T, np.float64)
    ent = np.empty(T, np.float64)
    st = np.empty(T, np.int32)
    rc = _load().oracle_logprob_entropy_support(_ptr(a), dt, T, V, V, _ptr(ids),
                                                float(np.float32(temperature)), _ptr(off),
                                                _ptr(sup), _ptr(lp), _ptr(ent), _ptr(st),
                                                threads or default_threads())
    if rc:
        raise ValueError("oracle_logprob_entropy_support rejected its arguments")
    return lp, ent, st


def logprob_entropy_backward(logits, ids, temperature, top_p, g_logprob=None, g_entropy=None,
                             force_k=None, threads=None):
    """Dense dL/dz [T, V] (fp64) of the logits path for
    L = sum_t g_logprob[t] logprob_t + g_entropy[t] H_t, each row's retained set
    held fixed; zero outside the set, NaN on rows with no distribution."""
    a, dt = _logits_array(logits)
    T, V = a.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gl = None if g_logprob is None else np.ascontiguousarray(g_logprob, dtype=np.float32)
    gh = None if g_entropy is None else np.ascontiguousarray(g_entropy, dtype=np.float32)
    fk = None if force_k is None else np.ascontiguousarray(force_k, dtype=np.int64)
    out = np.empty((T, V), np.float64)
    rc = _load().oracle_logprob_entropy_backward(
        _ptr(a), dt, T, V, V, _ptr(ids), float(np.float32(temperature)),
        float(np.float32(top_p)), _ptr(fk), _ptr(gl), _ptr(gh), _ptr(out),
        threads or default_threads())
    if rc:
        raise ValueError("oracle_logprob_entropy_backward rejected its arguments")
    return out


def logprob_entropy_support_backward(logits, ids, temperature, offsets, support_ids, g_logprob=None,
                                     g_entropy=None, threads=None):
    """dL/dz for every listed id (aligned with ``support_ids``), the retained
    sets held fixed, for L = sum_t g_logprob[t] logprob_t + g_entropy[t] H_t."""
    a, dt = _logits_array(logits)
    T, V = a.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    sup = np.ascontiguousarray(support_ids, dtype=np.int32)
    gl = None if g_logprob is None else np.ascontiguousarray(g_logprob, dtype=np.float32)
    gh = None if g_entropy is None else np.ascontiguousarray(g_entropy, dtype=np.float32)
    out = np.empty(int(off[-1]), np.float64)
    rc = _load().oracle_logprob_entropy_support_backward(
        _ptr(a), dt, T, V, V, _ptr(ids), float(np.float32(temperature)), _ptr(off), _ptr(sup),
        _ptr(gl), _ptr(gh), _ptr(out), threads or default_threads())
    if rc:
        raise ValueError("oracle_logprob_entropy_support_backward rejected its arguments")
    return out


def sample_ids(logits, temperature, top_p, u, threads=None):
    """Inverse-CDF draw from each row's renormalised nucleus; u in [0,1) per row."""
    a, dt = _logits_array(logits)
    T, V = a.shape
    u = np.ascontiguousarray(u, dtype=np.float64)
    out = np.empty(T, np.int32)
    rc = _load().oracle_sample_ids(_ptr(a), dt, T, V, V, float(np.float32(temperature)),
                                   float(np.float32(top_p)), _ptr(u), _ptr(out),
                                   threads or default_threads())
    if rc:
        raise ValueError("oracle_sample_ids rejected its arguments")
    return out


def grpo_loss(logp_new, logp_old, logp_rollout, logp_ref, mask, rewards, seq_offsets,
              group_size, eps_low=0.2, eps_high=0.28, tis_cap=2.0, kl_coef=0.01, agg=0):
    """GRPO/DAPO loss; returns (loss, grad[T], advantages[n_seq], stats dict)."""
    f = lambda x: np.ascontiguousarray(x, dtype=np.float32)
    new, old, ro, rf = f(logp_new), f(logp_old), f(logp_rollout), f(logp_ref)
    rw = f(rewards)
    off = np.ascontiguousarray(seq_offsets, dtype=np.int32)
    n_seq = off.shape[0] - 1
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    n_tok = int(off[-1] - off[0]) if n_seq >= 0 else 0
    loss = np.zeros(1, np.float64)
    grad = np.empty(max(n_tok, 0), np.float64)
    adv = np.empty(max(n_seq, 0), np.float64)
    stats = np.empty(len(STAT_NAMES), np.float64)
    rc = _load().oracle_grpo_loss(_ptr(new), _ptr(old), _ptr(ro), _ptr(rf), _ptr(m), _ptr(rw),
                                  _ptr(off), n_seq, int(group_size), float(eps_low),
                                  float(eps_high), float(tis_cap), float(kl_coef), int(agg),
                                  _ptr(loss), _ptr(grad), _ptr(adv), _ptr(stats))
    if rc:
        raise ValueError("oracle_grpo_loss rejected its arguments")
    return float(loss[0]), grad, adv, dict(zip(STAT_NAMES, stats.tolist()))


POLICY_STAT_NAMES = STAT_NAMES + ("mask_dropped",)
LOSS_DAPO, LOSS_IPO, LOSS_ICEPOP = 0, 1, 2
IS_NONE, IS_TIS, IS_MIS = 0, 1, 2
BASELINE_MEAN, BASELINE_LENGTH_WEIGHTED = 0, 1


def policy_loss(logp_new, logp_old, logp_rollout, logp_ref, mask, rewards, seq_offsets,
                group_size, loss_type=LOSS_DAPO, eps_low=0.2, eps_high=0.28, ipo_eps=0.3,
                band_low=0.5, band_high=2.0, is_method=IS_TIS, is_cap=2.0, kl_coef=0.01,
                baseline=BASELINE_MEAN, agg=0):
    """Policy-loss variants (DAPO / IPO / IcePop; none / TIS / MIS weights;
    mean or length-weighted baseline; token, sequence or prompt mean); returns
    (loss, grad[T], advantages[n_seq], stats dict)."""
    f = lambda x: np.ascontiguousarray(x, dtype=np.float32)
    new, old, ro, rf = f(logp_new), f(logp_old), f(logp_rollout), f(logp_ref)
    rw = f(rewards)
    off = np.ascontiguousarray(seq_offsets, dtype=np.int32)
    n_seq = off.shape[0] - 1
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    n_tok = int(off[-1] - off[0]) if n_seq >= 0 else 0
    loss = np.zeros(1, np.float64)
    grad = np.empty(max(n_tok, 0), np.float64)
    adv = np.empty(max(n_seq, 0), np.float64)
    stats = np.empty(len(POLICY_STAT_NAMES), np.float64)
    rc = _load().oracle_policy_loss(
        _ptr(new), _ptr(old), _ptr(ro), _ptr(rf), _ptr(m), _ptr(rw), _ptr(off), n_seq,
        int(group_size), int(loss_type), float(eps_low), float(eps_high), float(ipo_eps),
        float(band_low), float(band_high), int(is_method), float(is_cap), float(kl_coef),
        int(baseline), int(agg), _ptr(loss), _ptr(grad), _ptr(adv), _ptr(stats))
    if rc:
        raise ValueError("oracle_policy_loss rejected its arguments")
    return float(loss[0]), grad, adv, dict(zip(POLICY_STAT_NAMES, stats.tolist()))


def lmhead_rows(hidden_bits, w_bits, rows, ids, temperature, top_p=1.0, threads=None):
    """Logits = hidden @ W^T in fp64 for the selected rows, then the logits path."""
    h = np.ascontiguousarray(hidden_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    T, H = h.shape
    V, H2 = w.shape
    assert H == H2
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n = rows.shape[0]
    lp = np.empty(n, np.float64)
    ent = np.empty(n, np.float64)
    k = np.empty(n, np.int64)
    rc = _load().oracle_lmhead_rows(_ptr(h), _ptr(w), T, H, V, _ptr(rows), n, _ptr(ids),
                                    float(np.float32(temperature)), float(np.float32(top_p)),
                                    _ptr(lp), _ptr(ent), _ptr(k), threads or default_threads())
    if rc:
        raise ValueError("oracle_lmhead_rows rejected its arguments")
    return lp, ent, k


def lmhead_backward(hidden_bits, w_bits, ids, temperature, top_p=1.0, g_logprob=None,
                    g_entropy=None, threads=None):
    """Gradients of the LM-head path with the retained sets held fixed:
    (dL/dhidden [T, H], dL/dW [V, H]) in fp64."""
    h = np.ascontiguousarray(hidden_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    T, H = h.shape
    V, H2 = w.shape
    assert H == H2
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gl = None if g_logprob is None else np.ascontiguousarray(g_logprob, dtype=np.float32)
    gh = None if g_entropy is None else np.ascontiguousarray(g_entropy, dtype=np.float32)
    dh = np.empty((T, H), np.float64)
    dw = np.empty((V, H), np.float64)
    rc = _load().oracle_lmhead_backward(_ptr(h), _ptr(w), T, H, V, _ptr(ids),
                                        float(np.float32(temperature)), float(np.float32(top_p)),
                                        _ptr(gl), _ptr(gh), _ptr(dh), _ptr(dw),
                                        threads or default_threads())
    if rc:
        raise ValueError("oracle_lmhead_backward rejected its arguments")
    return dh, dw
