"""Python binding of librlk (argument marshalling only).

Every step of the computation runs in the CUDA kernels of ``librlk.so``; this
module only checks tensor placement, allocates outputs with PyTorch and passes
raw pointers plus the current CUDA stream through the C ABI declared in
``include/rlk.h``.  There is no CPU fallback: if the library is missing or the
tensors are not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "librlk.so")

RLK_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace",
                4: "CUDA error", 5: "timeout", 6: "bad input"}
STATUS_BAD_TOKEN_ID = 0x1
STATUS_NONFINITE = 0x2
OP_LOGPROB_ENTROPY, OP_GRPO_LOSS, OP_LMHEAD, OP_LMHEAD_BWD, OP_LMHEAD_TOPP = 0, 1, 2, 3, 4
OP_CANONICAL = 5
OP_CANONICAL_TOPP = 6
SHARD_COUNTS_BYTES = 8224   # rlk_shard_counts: one row's window counts of one shard
CANONICAL_TP, CANONICAL_VOCAB = 8, 152576
SHARD_PARTIAL_WORDS = 8   # rlk_shard_partial: 32 bytes per (shard, row)
AGG_TOKEN_MEAN, AGG_SEQ_MEAN_TOKEN_MEAN, AGG_PROMPT_MEAN = 0, 1, 2
LOSS_DAPO, LOSS_IPO, LOSS_ICEPOP = 0, 1, 2
IS_NONE, IS_TIS, IS_MIS = 0, 1, 2
BASELINE_MEAN, BASELINE_LENGTH_WEIGHTED = 0, 1
NSTATS_POLICY = 9
STAT_MASK_DROPPED = 8
NSTATS = 8
class LossConfig(ctypes.Structure):
    """rlk_loss_config."""
    _fields_ = [("type", ctypes.c_int), ("eps_low", ctypes.c_float), ("eps_high", ctypes.c_float),
                ("ipo_eps", ctypes.c_float), ("band_low", ctypes.c_float),
                ("band_high", ctypes.c_float), ("is_method", ctypes.c_int),
                ("is_cap", ctypes.c_float), ("kl_coef", ctypes.c_float),
                ("baseline", ctypes.c_int), ("agg", ctypes.c_int)]


STAT_NAMES = ("loss", "tokens", "clip_low_frac", "clip_high_frac", "tis_mean",
              "tis_capped_frac", "k3_mean", "pg_mean")
EXPORTS = ("rlk_version", "rlk_status_string", "rlk_workspace_size", "rlk_logprob_entropy",
           "rlk_logprob_entropy_fwd", "rlk_logprob_entropy_bwd", "rlk_logprob_entropy_rows",
           "rlk_logprob_entropy_support", "rlk_logprob_entropy_support_backward",
           "rlk_grpo_loss", "rlk_policy_loss", "rlk_lmhead_logprob", "rlk_lmhead_logprob_fwd",
           "rlk_lmhead_logprob_bwd", "rlk_shard_partials", "rlk_shard_combine",
           "rlk_shard_partials_support",
           "rlk_logprob_entropy_canonical", "rlk_sample_top_p",
           "rlk_shard_window_counts", "rlk_shard_combine_topp",
           "rlk_logprob_entropy_canonical_topp",
           "rlk_grpo_loss_noalloc")
NOALLOC_MAX_SEQ = 16384
DEBUG_EXPORTS = ("rlk_lmhead_logits_debug", "rlk_debug_inject_launch_failures",
                 "rlk_debug_set_wait_limit", "rlk_debug_withhold_copy",
                 "rlk_debug_set_sampler_mode")
STATUS_TIMEOUT = 0x4
STATUS_BAD_SUPPORT = 0x8
STATUS_NO_STATE = 0x10
STATUS_BAD_PARAM = 0x20
STATUS_UNRESOLVED = 0x40
ROW_STATE_WORDS = 8   # rlk_row_state: 32 bytes per row

_lock = threading.Lock()
_lib = None


class RlkError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)} ({code})")
        self.code = code


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def load(path: str | None = None):
    """Load librlk.so (built in-tree by ``build()``) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it first (entropy_logits_bf16_gb300.build())")
        lib = ctypes.CDLL(p)
        i64, i32, f32, vp, sz = (ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                 ctypes.c_void_p, ctypes.c_size_t)
        lib.rlk_version.restype = ctypes.c_int
        lib.rlk_status_string.argtypes = [ctypes.c_int]
        lib.rlk_status_string.restype = ctypes.c_char_p
        lib.rlk_workspace_size.argtypes = [ctypes.c_int, i64, i64, i64]
        lib.rlk_workspace_size.restype = sz
        lib.rlk_logprob_entropy.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, f32, f32, vp,
                                            vp, vp, vp, vp, sz, vp]
        lib.rlk_logprob_entropy.restype = ctypes.c_int
        lib.rlk_logprob_entropy_fwd.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, f32, f32, vp,
                                                vp, vp, vp, vp, vp]
        lib.rlk_logprob_entropy_fwd.restype = ctypes.c_int
        lib.rlk_logprob_entropy_rows.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, vp,
                                                 vp, vp, vp, vp, vp]
        lib.rlk_logprob_entropy_rows.restype = ctypes.c_int
        lib.rlk_logprob_entropy_bwd.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, f32, vp, vp,
                                                vp, vp, ctypes.c_int, i64, vp, vp]
        lib.rlk_logprob_entropy_bwd.restype = ctypes.c_int
        lib.rlk_logprob_entropy_support.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, f32, vp,
                                                    vp, vp, vp, vp, vp]
        lib.rlk_logprob_entropy_support.restype = ctypes.c_int
        lib.rlk_logprob_entropy_support_backward.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp,
                                                             f32, vp, vp, vp, vp, vp, vp, vp]
        lib.rlk_logprob_entropy_support_backward.restype = ctypes.c_int
        lib.rlk_policy_loss.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i64,
                                        ctypes.POINTER(LossConfig), vp, vp, vp, vp, sz, vp]
        lib.rlk_policy_loss.restype = ctypes.c_int
        lib.rlk_grpo_loss.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, f32, f32, f32,
                                      f32, ctypes.c_int, vp, vp, vp, vp, sz, vp]
        lib.rlk_grpo_loss.restype = ctypes.c_int
        lib.rlk_lmhead_logprob.argtypes = [vp, vp, i64, i64, i64, vp, f32, f32, vp, vp, vp, vp,
                                           sz, vp]
        lib.rlk_lmhead_logprob.restype = ctypes.c_int
        lib.rlk_sample_top_p.argtypes = [vp, ctypes.c_int, i64, i64, i64, f32, vp, vp, vp, vp, vp]
        lib.rlk_sample_top_p.restype = ctypes.c_int
        lib.rlk_debug_inject_launch_failures.argtypes = [ctypes.c_int]
        lib.rlk_debug_inject_launch_failures.restype = ctypes.c_int
        lib.rlk_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
        lib.rlk_debug_set_wait_limit.restype = ctypes.c_longlong
        lib.rlk_debug_withhold_copy.argtypes = [ctypes.c_longlong]
        lib.rlk_debug_withhold_copy.restype = ctypes.c_int
        lib.rlk_debug_set_sampler_mode.argtypes = [ctypes.c_int]
        lib.rlk_debug_set_sampler_mode.restype = ctypes.c_int
        lib.rlk_shard_partials.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, i64, i32, vp, f32,
                                           vp, vp]
        lib.rlk_shard_partials.restype = ctypes.c_int
        lib.rlk_shard_partials_support.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, i64, i32,
                                                   vp, f32, vp, vp, vp, vp]
        lib.rlk_shard_partials_support.restype = ctypes.c_int
        lib.rlk_shard_combine.argtypes = [vp, i32, i64, i64, i64, vp, f32, vp, vp, vp, vp]
        lib.rlk_shard_combine.restype = ctypes.c_int
        lib.rlk_logprob_entropy_canonical.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, f32, i32,
                                                      i64, vp, vp, vp, vp, sz, vp]
        lib.rlk_logprob_entropy_canonical.restype = ctypes.c_int
        lib.rlk_shard_window_counts.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, i64, i32, vp,
                                                f32, f32, vp, i32, vp, vp]
        lib.rlk_shard_window_counts.restype = ctypes.c_int
        lib.rlk_shard_combine_topp.argtypes = [vp, vp, i32, i64, i64, i64, vp, f32, f32, vp, vp,
                                               vp, vp, vp]
        lib.rlk_shard_combine_topp.restype = ctypes.c_int
        lib.rlk_logprob_entropy_canonical_topp.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, f32,
                                                           f32, i32, i64, vp, vp, vp, vp, vp, sz,
                                                           vp]
        lib.rlk_logprob_entropy_canonical_topp.restype = ctypes.c_int
        lib.rlk_lmhead_logprob_fwd.argtypes = [vp, vp, i64, i64, i64, vp, f32, f32, vp, vp, vp,
                                               vp, vp, sz, vp]
        lib.rlk_lmhead_logprob_fwd.restype = ctypes.c_int
        lib.rlk_lmhead_logprob_bwd.argtypes = [vp, vp, i64, i64, i64, vp, f32, vp, vp, vp, vp, vp,
                                               vp, ctypes.c_int, vp, sz, vp]
        lib.rlk_lmhead_logprob_bwd.restype = ctypes.c_int
        lib.rlk_lmhead_logits_debug.argtypes = [vp, vp, i64, i64, i64, vp, f32, vp, vp, vp, vp,
                                                vp, sz, vp]
        lib.rlk_lmhead_logits_debug.restype = ctypes.c_int
        lib.rlk_grpo_loss_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, f32, f32,
                                              f32, f32, ctypes.c_int, vp, vp, vp, vp]
        lib.rlk_grpo_loss_noalloc.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("librlk operates on CUDA tensors only")


def _check(fn, code):
    if code != RLK_OK:
        raise RlkError(fn, code)


def workspace_size(op: int, T: int, V: int, H: int = 0) -> int:
    return int(load().rlk_workspace_size(op, T, V, H))


def _logits_dtype(logits):
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit stride along the vocabulary")
    dt = {torch.bfloat16: 0, torch.float32: 1}.get(logits.dtype)
    if dt is None:
        raise ValueError("logits must be bf16 or fp32")
    return dt


def new_row_state(T: int, device) -> torch.Tensor:
    """Room for the per-row state the forward saves for the backward
    (rlk_row_state[T], 32 bytes a row)."""
    return torch.empty((T, ROW_STATE_WORDS), dtype=torch.int32, device=device)


def logprob_entropy(logits: torch.Tensor, token_ids: torch.Tensor, temperature: float,
                    top_p: float, *, out_logprob=None, out_entropy=None,
                    return_nucleus_size: bool = False, status_word: torch.Tensor | None = None,
                    row_state: torch.Tensor | None = None):
    """Top-p log-probability of the selected token and entropy of the retained set.

    logits: CUDA [T, V] bf16 or fp32 (rows may be strided, unit stride along V);
    token_ids: CUDA int32 [T].  Returns (logprob, entropy) fp32 [T], plus the
    nucleus sizes int32 [T] when ``return_nucleus_size``.  ``status_word`` (CUDA
    uint32/int32 [1]) receives the STATUS_* bits of bad rows.  ``row_state``
    (from ``new_row_state``) receives what ``logprob_entropy_backward`` needs.
    """
    lib = load()
    _need_cuda(logits, token_ids)
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit stride along the vocabulary")
    if logits.dtype == torch.bfloat16:
        dt = 0
    elif logits.dtype == torch.float32:
        dt = 1
    else:
        raise ValueError("logits must be bf16 or fp32")
    if token_ids.dtype != torch.int32 or not token_ids.is_contiguous():
        raise ValueError("token_ids must be contiguous int32")
    T, V = logits.shape
    ld = logits.stride(0) if T > 1 else V
    dev = logits.device
    lp = out_logprob if out_logprob is not None else torch.empty(T, device=dev, dtype=torch.float32)
    ent = out_entropy if out_entropy is not None else torch.empty(T, device=dev, dtype=torch.float32)
    ks = torch.empty(T, device=dev, dtype=torch.int32) if return_nucleus_size else None
    if row_state is not None:
        _need_cuda(row_state)
        if (row_state.dtype != torch.int32 or not row_state.is_contiguous()
                or row_state.numel() != T * ROW_STATE_WORDS):
            raise ValueError("row_state must come from new_row_state(T)")
        code = lib.rlk_logprob_entropy_fwd(_ptr(logits), dt, T, V, ld, _ptr(token_ids),
                                           float(temperature), float(top_p), _ptr(lp), _ptr(ent),
                                           _ptr(ks), _ptr(row_state), _ptr(status_word),
                                           _stream(dev))
        _check("rlk_logprob_entropy_fwd", code)
    else:
        code = lib.rlk_logprob_entropy(_ptr(logits), dt, T, V, ld, _ptr(token_ids),
                                       float(temperature), float(top_p), _ptr(lp), _ptr(ent),
                                       _ptr(ks), _ptr(status_word), None, 0, _stream(dev))
        _check("rlk_logprob_entropy", code)
    return (lp, ent, ks) if return_nucleus_size else (lp, ent)


def logprob_entropy_rows(logits: torch.Tensor, token_ids: torch.Tensor, temperatures: torch.Tensor,
                        top_ps: torch.Tensor, *, return_nucleus_size: bool = False,
                        status_word=None, row_state=None):
    """``logprob_entropy`` with per-row sampling parameters (CUDA fp32 [T]
    each).  ``row_state`` records each row's temperature for the backward and
    the sampler."""
    lib = load()
    _need_cuda(logits, token_ids, temperatures, top_ps, row_state)
    dt = _logits_dtype(logits)
    T, V = logits.shape
    for t in (temperatures, top_ps):
        if t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != T:
            raise ValueError("temperatures and top_ps must be contiguous fp32 [T]")
    if token_ids.dtype != torch.int32 or not token_ids.is_contiguous():
        raise ValueError("token_ids must be contiguous int32")
    if row_state is not None and (row_state.dtype != torch.int32 or not row_state.is_contiguous()
                                  or row_state.numel() != T * ROW_STATE_WORDS):
        raise ValueError("row_state must come from new_row_state(T)")
    ld = logits.stride(0) if T > 1 else V
    dev = logits.device
    lp = torch.empty(T, device=dev, dtype=torch.float32)
    ent = torch.empty(T, device=dev, dtype=torch.float32)
    ks = torch.empty(T, device=dev, dtype=torch.int32) if return_nucleus_size else None
    code = lib.rlk_logprob_entropy_rows(_ptr(logits), dt, T, V, ld, _ptr(token_ids),
                                        _ptr(temperatures), _ptr(top_ps), _ptr(lp), _ptr(ent),
                                        _ptr(ks), _ptr(row_state), _ptr(status_word), _stream(dev))
    _check("rlk_logprob_entropy_rows", code)
    return (lp, ent, ks) if return_nucleus_size else (lp, ent)


def logprob_entropy_backward(logits: torch.Tensor, token_ids: torch.Tensor, temperature: float,
                             row_state: torch.Tensor, grad_logprob=None, grad_entropy=None, *,
                             out=None, grad_dtype=None, status_word=None):
    """dL/dlogits [T, V] for L = sum grad_logprob * logprob + grad_entropy * H,
    each row's retained set (saved in ``row_state`` by the forward) held fixed;
    zero outside the set.  ``grad_dtype`` (bf16 or fp32) defaults to the
    logits' dtype; ``out`` may be a strided [T, V] tensor of that dtype."""
    lib = load()
    _need_cuda(logits, token_ids, row_state, grad_logprob, grad_entropy, out)
    dt = _logits_dtype(logits)
    if token_ids.dtype != torch.int32 or not token_ids.is_contiguous():
        raise ValueError("token_ids must be contiguous int32")
    T, V = logits.shape
    if (row_state.dtype != torch.int32 or not row_state.is_contiguous()
            or row_state.numel() != T * ROW_STATE_WORDS):
        raise ValueError("row_state must come from new_row_state(T)")
    for g in (grad_logprob, grad_entropy):
        if g is not None and (g.dtype != torch.float32 or not g.is_contiguous() or g.numel() != T):
            raise ValueError("gradients must be contiguous fp32 [T]")
    gdt = grad_dtype or (out.dtype if out is not None else logits.dtype)
    if out is None:
        out = torch.empty((T, V), device=logits.device, dtype=gdt)
    if out.dtype != gdt or out.shape != (T, V) or out.stride(1) != 1:
        raise ValueError("out must be [T, V] of grad_dtype with unit stride along V")
    gd = {torch.bfloat16: 0, torch.float32: 1}.get(gdt)
    if gd is None:
        raise ValueError("grad_dtype must be bf16 or fp32")
    ld = logits.stride(0) if T > 1 else V
    ldg = out.stride(0) if T > 1 else V
    code = lib.rlk_logprob_entropy_bwd(_ptr(logits), dt, T, V, ld, _ptr(token_ids),
                                       float(temperature), _ptr(row_state), _ptr(grad_logprob),
                                       _ptr(grad_entropy), _ptr(out), gd, ldg, _ptr(status_word),
                                       _stream(logits.device))
    _check("rlk_logprob_entropy_bwd", code)
    return out


class _LogprobEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, token_ids, temperature, top_p):
        state = new_row_state(logits.shape[0], logits.device)
        lp, ent = logprob_entropy(logits, token_ids, temperature, top_p, row_state=state)
        ctx.save_for_backward(logits, token_ids, state)
        ctx.temperature = temperature
        ctx.set_materialize_grads(False)
        return lp, ent

    @staticmethod
    def backward(ctx, g_lp, g_ent):
        logits, token_ids, state = ctx.saved_tensors
        if g_lp is None and g_ent is None:
            return None, None, None, None
        g = logprob_entropy_backward(
            logits, token_ids, ctx.temperature, state,
            None if g_lp is None else g_lp.float().contiguous(),
            None if g_ent is None else g_ent.float().contiguous())
        return g, None, None, None


def logprob_entropy_autograd(logits: torch.Tensor, token_ids: torch.Tensor, temperature: float,
                             top_p: float):
    """``logprob_entropy`` as a differentiable op: (logprob, entropy) whose
    backward is ``rlk_logprob_entropy_bwd`` (the retained sets held fixed)."""
    return _LogprobEntropy.apply(logits, token_ids, temperature, top_p)


def logprob_entropy_support(logits: torch.Tensor, token_ids: torch.Tensor, temperature: float,
                            support_offsets: torch.Tensor, support_ids: torch.Tensor, *,
                            out_logprob=None, out_entropy=None, status_word=None):
    """Log-probability of the selected token and entropy over a retained set
    supplied by the sampler: row t keeps the ids
    support_ids[support_offsets[t]:support_offsets[t+1]] (CUDA int64 offsets
    [T+1], int32 ids).  Returns (logprob, entropy) fp32 [T]."""
    lib = load()
    _need_cuda(logits, token_ids, support_offsets, support_ids)
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit stride along the vocabulary")
    if logits.dtype == torch.bfloat16:
        dt = 0
    elif logits.dtype == torch.float32:
        dt = 1
    else:
        raise ValueError("logits must be bf16 or fp32")
    if token_ids.dtype != torch.int32 or not token_ids.is_contiguous():
        raise ValueError("token_ids must be contiguous int32")
    if support_offsets.dtype != torch.int64 or not support_offsets.is_contiguous():
        raise ValueError("support_offsets must be contiguous int64")
    if support_ids.dtype != torch.int32 or not support_ids.is_contiguous():
        raise ValueError("support_ids must be contiguous int32")
    T, V = logits.shape
    if support_offsets.numel() != T + 1:
        raise ValueError("support_offsets must have T + 1 entries")
    ld = logits.stride(0) if T > 1 else V
    dev = logits.device
    lp = out_logprob if out_logprob is not None else torch.empty(T, device=dev, dtype=torch.float32)
    ent = out_entropy if out_entropy is not None else torch.empty(T, device=dev, dtype=torch.float32)
    code = lib.rlk_logprob_entropy_support(_ptr(logits), dt, T, V, ld, _ptr(token_ids),
                                           float(temperature), _ptr(support_offsets),
                                           _ptr(support_ids), _ptr(lp), _ptr(ent),
                                           _ptr(status_word), _stream(dev))
    _check("rlk_logprob_entropy_support", code)
    return lp, ent


def logprob_entropy_support_backward(logits: torch.Tensor, token_ids: torch.Tensor,
                                     temperature: float, support_offsets: torch.Tensor,
                                     support_ids: torch.Tensor, grad_logprob=None,
                                     grad_entropy=None, *, out=None, status_word=None):
    """dL/dz for every listed id (aligned with ``support_ids``; the retained
    sets held fixed) for L = sum grad_logprob * logprob + grad_entropy * H.
    Returns a CUDA fp32 tensor shaped like ``support_ids``."""
    lib = load()
    _need_cuda(logits, token_ids, support_offsets, support_ids, grad_logprob, grad_entropy)
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit stride along the vocabulary")
    dt = {torch.bfloat16: 0, torch.float32: 1}.get(logits.dtype)
    if dt is None:
        raise ValueError("logits must be bf16 or fp32")
    for t, want in ((token_ids, torch.int32), (support_offsets, torch.int64),
                    (support_ids, torch.int32)):
        if t.dtype != want or not t.is_contiguous():
            raise ValueError("token_ids int32, support_offsets int64 and support_ids int32, contiguous")
    for g in (grad_logprob, grad_entropy):
        if g is not None and (g.dtype != torch.float32 or not g.is_contiguous()):
            raise ValueError("gradients must be contiguous fp32")
    T, V = logits.shape
    ld = logits.stride(0) if T > 1 else V
    grad = out if out is not None else torch.empty(support_ids.shape, device=logits.device,
                                                   dtype=torch.float32)
    code = lib.rlk_logprob_entropy_support_backward(
        _ptr(logits), dt, T, V, ld, _ptr(token_ids), float(temperature), _ptr(support_offsets),
        _ptr(support_ids), _ptr(grad_logprob), _ptr(grad_entropy), _ptr(grad), _ptr(status_word),
        _stream(logits.device))
    _check("rlk_logprob_entropy_support_backward", code)
    return grad


def grpo_loss(logp_new, logp_old, logp_rollout, logp_ref, rewards, seq_offsets, group_size, *,
              loss_mask=None, eps_low=0.2, eps_high=0.28, tis_cap=2.0, kl_coef=0.01,
              agg=AGG_TOKEN_MEAN, want_grad=True, want_stats=True, workspace=None):
    """GRPO/DAPO loss with TIS and k3 KL.  Returns (loss[1], grad[T] or None,
    stats[NSTATS] or None), all CUDA fp32 tensors."""
    lib = load()
    _need_cuda(logp_new, logp_old, logp_rollout, logp_ref, rewards, seq_offsets, loss_mask)
    for t in (logp_new, logp_old, logp_rollout, logp_ref, rewards):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("log-probs and rewards must be contiguous fp32")
    if seq_offsets.dtype != torch.int32:
        raise ValueError("seq_offsets must be int32")
    if loss_mask is not None and loss_mask.dtype != torch.uint8:
        raise ValueError("loss_mask must be uint8")
    n_seq = seq_offsets.numel() - 1
    n_tok = logp_new.numel()
    dev = logp_new.device
    need = int(lib.rlk_workspace_size(OP_GRPO_LOSS, n_tok, n_seq, 0))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    loss = torch.empty(1, device=dev, dtype=torch.float32)
    grad = torch.empty(n_tok, device=dev, dtype=torch.float32) if want_grad else None
    stats = torch.empty(NSTATS, device=dev, dtype=torch.float32) if want_stats else None
    code = lib.rlk_grpo_loss(_ptr(logp_new), _ptr(logp_old), _ptr(logp_rollout), _ptr(logp_ref),
                             _ptr(loss_mask), _ptr(rewards), _ptr(seq_offsets), n_seq,
                             int(group_size), n_tok, float(eps_low), float(eps_high),
                             float(tis_cap), float(kl_coef), int(agg), _ptr(loss), _ptr(grad),
                             _ptr(stats), _ptr(workspace), workspace.numel(), _stream(dev))
    _check("rlk_grpo_loss", code)
    return loss, grad, stats


def policy_loss(logp_new, logp_old, logp_rollout, logp_ref, rewards, seq_offsets, group_size, *,
                loss_mask=None, loss_type=LOSS_DAPO, eps_low=0.2, eps_high=0.28, ipo_eps=0.3,
                band_low=0.5, band_high=2.0, is_method=IS_TIS, is_cap=2.0, kl_coef=0.01,
                baseline=BASELINE_MEAN, agg=AGG_TOKEN_MEAN, want_grad=True, want_stats=True,
                workspace=None):
    """rlk_policy_loss: the GRPO/DAPO loss with the IPO / IcePop policy terms,
    none / TIS / MIS weights, a mean or length-weighted baseline and token /
    sequence / prompt aggregation.  Returns (loss[1], grad[T] or None,
    stats[NSTATS_POLICY] or None), CUDA fp32 tensors."""
    lib = load()
    _need_cuda(logp_new, logp_old, logp_rollout, logp_ref, rewards, seq_offsets, loss_mask)
    for t in (logp_new, logp_old, logp_rollout, logp_ref, rewards):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("log-probs and rewards must be contiguous fp32")
    if seq_offsets.dtype != torch.int32:
        raise ValueError("seq_offsets must be int32")
    if loss_mask is not None and loss_mask.dtype != torch.uint8:
        raise ValueError("loss_mask must be uint8")
    n_seq = seq_offsets.numel() - 1
    n_tok = logp_new.numel()
    dev = logp_new.device
    need = int(lib.rlk_workspace_size(OP_GRPO_LOSS, n_tok, n_seq, 0))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    cfg = LossConfig(int(loss_type), float(eps_low), float(eps_high), float(ipo_eps),
                     float(band_low), float(band_high), int(is_method), float(is_cap),
                     float(kl_coef), int(baseline), int(agg))
    loss = torch.empty(1, device=dev, dtype=torch.float32)
    grad = torch.empty(n_tok, device=dev, dtype=torch.float32) if want_grad else None
    stats = torch.empty(NSTATS_POLICY, device=dev, dtype=torch.float32) if want_stats else None
    code = lib.rlk_policy_loss(_ptr(logp_new), _ptr(logp_old), _ptr(logp_rollout),
                               _ptr(logp_ref), _ptr(loss_mask), _ptr(rewards), _ptr(seq_offsets),
                               n_seq, int(group_size), n_tok, ctypes.byref(cfg), _ptr(loss),
                               _ptr(grad), _ptr(stats), _ptr(workspace), workspace.numel(),
                               _stream(dev))
    _check("rlk_policy_loss", code)
    return loss, grad, stats


def lmhead_logprob(hidden, w_vocab, token_ids, temperature, top_p=1.0, *, status_word=None,
                   workspace=None, out_lse=None):
    """Fused LM-head log-probability and entropy.  At top_p = 1 the logits never
    reach memory; at top_p < 1 they are emitted as bf16 4096 rows at a time
    and scored by the top-p path.  ``out_lse`` (CUDA fp32 [T], top_p = 1)
    receives each row's log-normaliser for ``lmhead_backward``."""
    lib = load()
    _need_cuda(hidden, w_vocab, token_ids)
    if hidden.dtype != torch.bfloat16 or w_vocab.dtype != torch.bfloat16:
        raise ValueError("hidden and w_vocab must be bf16")
    if not (hidden.is_contiguous() and w_vocab.is_contiguous()):
        raise ValueError("hidden and w_vocab must be contiguous")
    T, H = hidden.shape
    V, H2 = w_vocab.shape
    if H != H2:
        raise ValueError("hidden and w_vocab disagree on H")
    dev = hidden.device
    need = int(lib.rlk_workspace_size(OP_LMHEAD if top_p == 1.0 else OP_LMHEAD_TOPP, T, V, H))
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    lp = torch.empty(T, device=dev, dtype=torch.float32)
    ent = torch.empty(T, device=dev, dtype=torch.float32)
    wsb = 0 if workspace is None else workspace.numel()
    if out_lse is not None:
        _need_cuda(out_lse)
        if out_lse.dtype != torch.float32 or out_lse.numel() != T or not out_lse.is_contiguous():
            raise ValueError("out_lse must be contiguous fp32 [T]")
        code = lib.rlk_lmhead_logprob_fwd(_ptr(hidden), _ptr(w_vocab), T, H, V, _ptr(token_ids),
                                          float(temperature), float(top_p), _ptr(lp), _ptr(ent),
                                          _ptr(out_lse), _ptr(status_word), _ptr(workspace), wsb,
                                          _stream(dev))
        _check("rlk_lmhead_logprob_fwd", code)
    else:
        code = lib.rlk_lmhead_logprob(_ptr(hidden), _ptr(w_vocab), T, H, V, _ptr(token_ids),
                                      float(temperature), float(top_p), _ptr(lp), _ptr(ent),
                                      _ptr(status_word), _ptr(workspace), wsb, _stream(dev))
        _check("rlk_lmhead_logprob", code)
    return lp, ent


def lmhead_backward(hidden, w_vocab, token_ids, temperature, lse, entropy, grad_logprob=None,
                    grad_entropy=None, *, grad_hidden=None, grad_w=None, accumulate_grad_w=False,
                    workspace=None):
    """Gradients of the fused LM-head path: (dL/dhidden fp32 [T, H],
    dL/dW fp32 [V, H]); ``lse`` and ``entropy`` from the forward."""
    lib = load()
    _need_cuda(hidden, w_vocab, token_ids, lse, entropy, grad_logprob, grad_entropy, grad_hidden,
               grad_w)
    if hidden.dtype != torch.bfloat16 or w_vocab.dtype != torch.bfloat16:
        raise ValueError("hidden and w_vocab must be bf16")
    if not (hidden.is_contiguous() and w_vocab.is_contiguous()):
        raise ValueError("hidden and w_vocab must be contiguous")
    T, H = hidden.shape
    V, H2 = w_vocab.shape
    if H != H2:
        raise ValueError("hidden and w_vocab disagree on H")
    for t in (lse, entropy, grad_logprob, grad_entropy):
        if t is not None and (t.dtype != torch.float32 or t.numel() != T or not t.is_contiguous()):
            raise ValueError("lse, entropy and the gradients must be contiguous fp32 [T]")
    dev = hidden.device
    if grad_hidden is None:
        grad_hidden = torch.empty((T, H), device=dev, dtype=torch.float32)
    if grad_w is None:
        if accumulate_grad_w:
            raise ValueError("accumulate_grad_w needs grad_w")
        grad_w = torch.empty((V, H), device=dev, dtype=torch.float32)
    for t, shp in ((grad_hidden, (T, H)), (grad_w, (V, H))):
        if t.dtype != torch.float32 or tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError("grad_hidden / grad_w must be contiguous fp32 [T, H] / [V, H]")
    need = int(lib.rlk_workspace_size(OP_LMHEAD_BWD, T, V, H))
    if workspace is None:
        workspace = torch.empty(max(need, 256), device=dev, dtype=torch.uint8)
    code = lib.rlk_lmhead_logprob_bwd(_ptr(hidden), _ptr(w_vocab), T, H, V, _ptr(token_ids),
                                      float(temperature), _ptr(lse), _ptr(entropy),
                                      _ptr(grad_logprob), _ptr(grad_entropy), _ptr(grad_hidden),
                                      _ptr(grad_w), int(bool(accumulate_grad_w)), _ptr(workspace),
                                      workspace.numel(), _stream(dev))
    _check("rlk_lmhead_logprob_bwd", code)
    return grad_hidden, grad_w


def lmhead_logits_debug(hidden, w_vocab, token_ids, temperature):
    """Validation aid: the fused LM-head path that also returns the fp32 logits
    it computed ([T, V]); for small sizes only."""
    lib = load()
    _need_cuda(hidden, w_vocab, token_ids)
    T, H = hidden.shape
    V = w_vocab.shape[0]
    dev = hidden.device
    need = int(lib.rlk_workspace_size(OP_LMHEAD, T, V, H))
    ws = torch.empty(max(need, 16), device=dev, dtype=torch.uint8)
    logits = torch.empty(T, V, device=dev, dtype=torch.float32)
    lp = torch.empty(T, device=dev, dtype=torch.float32)
    ent = torch.empty(T, device=dev, dtype=torch.float32)
    code = lib.rlk_lmhead_logits_debug(_ptr(hidden), _ptr(w_vocab), T, H, V, _ptr(token_ids),
                                       float(temperature), _ptr(logits), _ptr(lp), _ptr(ent),
                                       None, _ptr(ws), ws.numel(), _stream(dev))
    _check("rlk_lmhead_logits_debug", code)
    return logits, lp, ent


# ------------------------------------------------------------ canonical partition
def canonical_plan(tp_size: int, tp_rank: int, n_virtual: int = CANONICAL_TP,
                   padded_vocab: int = CANONICAL_VOCAB):
    """The virtual shards a physical tensor-parallel rank holds: (first shard,
    number of shards, first global column, shard width).  Rank k of tp_size
    holds the adjacent shards [k n, (k + 1) n), n = n_virtual / tp_size."""
    if n_virtual % tp_size != 0 or not 0 <= tp_rank < tp_size:
        raise ValueError("tp_size must divide the virtual degree; 0 <= tp_rank < tp_size")
    if padded_vocab % n_virtual != 0:
        raise ValueError("the padded vocabulary must be a multiple of the virtual degree")
    n = n_virtual // tp_size
    width = padded_vocab // n_virtual
    return tp_rank * n, n, tp_rank * n * width, width


def shard_partials(logits, token_ids, temperature, V, first_col, shard_width, n_shards):
    """rlk_shard_partials: [n_shards, T, 8] fp32 partials of the shards whose
    columns ``logits`` ([T, cols], unit stride along the vocabulary) holds."""
    lib = load()
    _need_cuda(logits, token_ids)
    dt = _logits_dtype(logits)
    T = logits.shape[0]
    ld = logits.stride(0) if T > 1 else logits.shape[1]
    out = torch.empty((n_shards, T, SHARD_PARTIAL_WORDS), device=logits.device,
                      dtype=torch.float32)
    code = lib.rlk_shard_partials(_ptr(logits), dt, T, int(V), ld, int(first_col),
                                  int(shard_width), int(n_shards), _ptr(token_ids),
                                  float(temperature), _ptr(out), _stream(logits.device))
    _check("rlk_shard_partials", code)
    return out


def shard_partials_support(logits, token_ids, temperature, V, first_col, shard_width, n_shards,
                           support_offsets, support_ids):
    """rlk_shard_partials_support: [n_shards, T, 8] partials of a supplied
    retained set (CSR over global ids) restricted to this rank's shards."""
    lib = load()
    _need_cuda(logits, token_ids, support_offsets, support_ids)
    dt = _logits_dtype(logits)
    if support_offsets.dtype != torch.int64 or support_ids.dtype != torch.int32:
        raise ValueError("support_offsets int64, support_ids int32")
    T = logits.shape[0]
    ld = logits.stride(0) if T > 1 else logits.shape[1]
    out = torch.empty((n_shards, T, SHARD_PARTIAL_WORDS), device=logits.device,
                      dtype=torch.float32)
    code = lib.rlk_shard_partials_support(_ptr(logits), dt, T, int(V), ld, int(first_col),
                                          int(shard_width), int(n_shards), _ptr(token_ids),
                                          float(temperature), _ptr(support_offsets),
                                          _ptr(support_ids), _ptr(out), _stream(logits.device))
    _check("rlk_shard_partials_support", code)
    return out


def shard_combine(partials, token_ids, temperature, V, shard_width, *, status_word=None):
    """rlk_shard_combine: (logprob, entropy) from all shards' partials
    ([n_shards, T, 8], canonical order)."""
    lib = load()
    _need_cuda(partials, token_ids)
    if partials.dtype != torch.float32 or not partials.is_contiguous() or partials.dim() != 3:
        raise ValueError("partials must be contiguous fp32 [n_shards, T, 8]")
    n_shards, T = partials.shape[0], partials.shape[1]
    lp = torch.empty(T, device=partials.device, dtype=torch.float32)
    ent = torch.empty(T, device=partials.device, dtype=torch.float32)
    code = lib.rlk_shard_combine(_ptr(partials), n_shards, T, int(V), int(shard_width),
                                 _ptr(token_ids), float(temperature), _ptr(lp), _ptr(ent),
                                 _ptr(status_word), _stream(partials.device))
    _check("rlk_shard_combine", code)
    return lp, ent


def shard_window_counts(logits, token_ids, temperature, top_p, V, first_col, shard_width,
                        n_shards, all_partials):
    """rlk_shard_window_counts: [n_shards, T, 8224] uint8 window counts of this
    rank's shards (bf16 ``logits`` [T, cols]), given every shard's partial
    ([n_all, T, 8], canonical order)."""
    lib = load()
    _need_cuda(logits, token_ids, all_partials)
    dt = _logits_dtype(logits)
    T = logits.shape[0]
    ld = logits.stride(0) if T > 1 else logits.shape[1]
    if all_partials.dtype != torch.float32 or not all_partials.is_contiguous():
        raise ValueError("all_partials must be contiguous fp32 [n_all, T, 8]")
    out = torch.empty((n_shards, T, SHARD_COUNTS_BYTES), device=logits.device, dtype=torch.uint8)
    code = lib.rlk_shard_window_counts(_ptr(logits), dt, T, int(V), ld, int(first_col),
                                       int(shard_width), int(n_shards), _ptr(token_ids),
                                       float(temperature), float(top_p), _ptr(all_partials),
                                       int(all_partials.shape[0]), _ptr(out), _stream(logits.device))
    _check("rlk_shard_window_counts", code)
    return out


def shard_combine_topp(partials, counts, token_ids, temperature, top_p, V, shard_width, *,
                       status_word=None):
    """rlk_shard_combine_topp: (logprob, entropy, nucleus size) from all shards'
    partials and window counts (canonical order)."""
    lib = load()
    _need_cuda(partials, counts, token_ids)
    n_shards, T = partials.shape[0], partials.shape[1]
    if counts.shape[:2] != (n_shards, T) or not counts.is_contiguous():
        raise ValueError("counts must be contiguous [n_shards, T, 8224]")
    lp = torch.empty(T, device=partials.device, dtype=torch.float32)
    ent = torch.empty(T, device=partials.device, dtype=torch.float32)
    k = torch.empty(T, device=partials.device, dtype=torch.int32)
    code = lib.rlk_shard_combine_topp(_ptr(partials), _ptr(counts), n_shards, T, int(V),
                                      int(shard_width), _ptr(token_ids), float(temperature),
                                      float(top_p), _ptr(lp), _ptr(ent), _ptr(k), _ptr(status_word),
                                      _stream(partials.device))
    _check("rlk_shard_combine_topp", code)
    return lp, ent, k


def logprob_entropy_canonical_topp(logits, token_ids, temperature, top_p, n_virtual=CANONICAL_TP,
                                   padded_vocab=CANONICAL_VOCAB, *, status_word=None):
    """The canonical partition on one device at top_p < 1: (logprob, entropy,
    nucleus size)."""
    lib = load()
    _need_cuda(logits, token_ids)
    dt = _logits_dtype(logits)
    T, V = logits.shape
    ld = logits.stride(0) if T > 1 else V
    ws = torch.empty(max(int(lib.rlk_workspace_size(OP_CANONICAL_TOPP, T, n_virtual, 0)), 16),
                     device=logits.device, dtype=torch.uint8)
    lp = torch.empty(T, device=logits.device, dtype=torch.float32)
    ent = torch.empty(T, device=logits.device, dtype=torch.float32)
    k = torch.empty(T, device=logits.device, dtype=torch.int32)
    code = lib.rlk_logprob_entropy_canonical_topp(_ptr(logits), dt, T, V, ld, _ptr(token_ids),
                                                  float(temperature), float(top_p), int(n_virtual),
                                                  int(padded_vocab), _ptr(lp), _ptr(ent), _ptr(k),
                                                  _ptr(status_word), _ptr(ws), ws.numel(),
                                                  _stream(logits.device))
    _check("rlk_logprob_entropy_canonical_topp", code)
    return lp, ent, k


def logprob_entropy_canonical(logits, token_ids, temperature, n_virtual=CANONICAL_TP,
                              padded_vocab=CANONICAL_VOCAB, *, status_word=None):
    """The canonical partition on one device (top_p = 1)."""
    lib = load()
    _need_cuda(logits, token_ids)
    dt = _logits_dtype(logits)
    T, V = logits.shape
    ld = logits.stride(0) if T > 1 else V
    ws = torch.empty(max(int(lib.rlk_workspace_size(OP_CANONICAL, T, n_virtual, 0)), 16),
                     device=logits.device, dtype=torch.uint8)
    lp = torch.empty(T, device=logits.device, dtype=torch.float32)
    ent = torch.empty(T, device=logits.device, dtype=torch.float32)
    code = lib.rlk_logprob_entropy_canonical(_ptr(logits), dt, T, V, ld, _ptr(token_ids),
                                             float(temperature), int(n_virtual), int(padded_vocab),
                                             _ptr(lp), _ptr(ent), _ptr(status_word), _ptr(ws),
                                             ws.numel(), _stream(logits.device))
    _check("rlk_logprob_entropy_canonical", code)
    return lp, ent


def gather_shard_partials(local_partials, group=None):
    """All ranks' per-shard tensors ([n_local, T, ...] each: partials, or window
    counts) gathered in rank order, which is canonical shard order:
    [n_local * world, T, ...].  The exchange of the vocabulary-parallel path
    (once at top_p = 1, twice at top_p < 1)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(local_partials) for _ in range(world)]
    dist.all_gather(parts, local_partials.contiguous(), group=group)
    return torch.cat(parts, 0)


def vocab_parallel_logprob_entropy(local_logits, token_ids, temperature, V, group=None,
                                   n_virtual=CANONICAL_TP, padded_vocab=CANONICAL_VOCAB,
                                   top_p=1.0):
    """Tensor-parallel log-probability and entropy: this rank's canonical
    shards -> partials -> gather in rank order -> combine; at top_p < 1 the
    gathered partials set every shard's window, whose counts are gathered too
    and combined (returns (logprob, entropy, nucleus size) then).  The result is
    bitwise the same for every tensor-parallel degree."""
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    _, n, first_col, width = canonical_plan(world, rank, n_virtual, padded_vocab)
    part = shard_partials(local_logits, token_ids, temperature, V, first_col, width, n)
    allp = gather_shard_partials(part, group) if world > 1 else part
    if top_p >= 1.0:
        return shard_combine(allp, token_ids, temperature, V, width)
    cnt = shard_window_counts(local_logits, token_ids, temperature, top_p, V, first_col, width, n,
                              allp)
    allc = gather_shard_partials(cnt, group) if world > 1 else cnt
    return shard_combine_topp(allp, allc, token_ids, temperature, top_p, V, width)


def sample_top_p(logits, temperature, top_p, uniforms, *, row_state=None, status_word=None):
    """Deterministic top-p draw per row (rlk_sample_top_p): the id where the
    cumulative renormalised probability over the retained set, in ranking
    order, first reaches ``uniforms`` (CUDA fp32 [T]).  Without ``row_state``
    the forward runs first to select the sets; ``temperature`` and ``top_p``
    may then be CUDA fp32 [T] tensors (per-row parameters)."""
    lib = load()
    _need_cuda(logits, uniforms, row_state)
    if logits.dtype != torch.bfloat16:
        raise ValueError("the sampler takes bf16 logits")
    _logits_dtype(logits)
    if uniforms.dtype != torch.float32 or not uniforms.is_contiguous():
        raise ValueError("uniforms must be contiguous fp32")
    T, V = logits.shape
    if row_state is None:
        row_state = new_row_state(T, logits.device)
        zeros = torch.zeros(T, dtype=torch.int32, device=logits.device)
        if torch.is_tensor(temperature) or torch.is_tensor(top_p):   # per-row parameters
            full = lambda v: v if torch.is_tensor(v) else torch.full(
                (T,), float(v), device=logits.device, dtype=torch.float32)
            logprob_entropy_rows(logits, zeros, full(temperature), full(top_p),
                                 row_state=row_state)
            temperature = 1.0   # each state carries its row's
        else:
            logprob_entropy(logits, zeros, temperature, top_p, row_state=row_state)
    out = torch.empty(T, dtype=torch.int32, device=logits.device)
    ld = logits.stride(0) if T > 1 else V
    code = lib.rlk_sample_top_p(_ptr(logits), 0, T, V, ld, float(temperature), _ptr(row_state),
                                _ptr(uniforms), _ptr(out), _ptr(status_word),
                                _stream(logits.device))
    _check("rlk_sample_top_p", code)
    return out


def inject_launch_failures(n: int) -> int:
    """Host-side fault injection: the next ``n`` entry points that would launch
    return RLK_ERR_CUDA (raised as RlkError) without launching.  Returns the
    count that was pending."""
    return int(load().rlk_debug_inject_launch_failures(int(n)))


def set_wait_limit(cycles: int) -> int:
    """Debug: the clock cycles a bounded device wait may take before it gives
    up (<= 0 restores the default of about a second).  Returns the previous
    limit."""
    return int(load().rlk_debug_set_wait_limit(int(cycles)))


def withhold_copy(stage: int) -> None:
    """Debug: the next scorer (or LM-head forward) launch skips the bulk copy
    of the given stage in its first CTA, so the wait on it runs out; < 0
    clears it."""
    load().rlk_debug_withhold_copy(int(stage))


def set_sampler_mode(mode: int) -> int:
    """Debug: the ways rlk_sample_top_p may take to a draw: 1 the direct mode
    with its member list (default), 2 the direct mode without the list, 0 the
    radix descent only.  Returns the previous mode."""
    return int(load().rlk_debug_set_sampler_mode(int(mode)))
