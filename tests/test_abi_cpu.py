"""The C ABI without a GPU: the library builds and loads, exports every entry
point the header declares, and rejects bad arguments on the host before any
CUDA call (these calls never touch a device)."""
import ctypes
import math
import os
import re

import pytest

import entropy_logits_bf16_gb300 as rlk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: validation fails first


@pytest.fixture(scope="module")
def lib():
    rlk.build()
    return rlk.load()


def declared_functions(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rlk_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions("rlk.h")
    assert set(names) == set(rlk.EXPORTS)
    debug = declared_functions("rlk_debug.h")
    assert set(debug) == set(rlk.DEBUG_EXPORTS)
    for n in names + debug:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.rlk_version() >= 100
    for code in range(7):
        assert lib.rlk_status_string(code)
    assert lib.rlk_status_string(99) == b"unknown status"


def test_workspace_sizes(lib):
    assert lib.rlk_workspace_size(rlk.OP_LOGPROB_ENTROPY, 4096, 151936, 0) == 0
    n = lib.rlk_workspace_size(rlk.OP_GRPO_LOSS, 590000, 512, 0)
    assert n >= 512 * 8 * 4 and n % 256 == 0
    assert lib.rlk_workspace_size(rlk.OP_GRPO_LOSS, 1, -1, 0) == 0
    assert lib.rlk_workspace_size(99, 1, 1, 1) == 0


def lpe(lib, **kw):
    args = dict(logits=FAKE, dtype=0, T=4, V=100, ld=100, ids=FAKE, temperature=0.7, top_p=0.95,
                lp=FAKE, ent=FAKE, k=None, status=None)
    args.update(kw)
    return lib.rlk_logprob_entropy(args["logits"], args["dtype"], args["T"], args["V"], args["ld"],
                                   args["ids"], args["temperature"], args["top_p"], args["lp"],
                                   args["ent"], args["k"], args["status"], None, 0, None)


@pytest.mark.parametrize("kw", [
    dict(temperature=0.0), dict(temperature=-1.0), dict(temperature=math.inf),
    dict(temperature=math.nan), dict(top_p=0.0), dict(top_p=1.0000001), dict(top_p=-0.5),
    dict(top_p=math.nan), dict(T=-1), dict(V=0), dict(V=(1 << 24) + 1), dict(ld=99),
    dict(dtype=2), dict(logits=None), dict(ids=None), dict(lp=None), dict(ent=None),
    dict(logits=ctypes.c_void_p(0x10001)),
])
def test_logprob_entropy_rejects(lib, kw):
    assert lpe(lib, **kw) == 1


def test_top_k_and_zero_temperature_are_rejected_not_ignored(lib):
    # The sampling contract rejects temperature 0; there is no top-k argument at all.
    assert lpe(lib, temperature=0.0) == 1
    assert "top_k" not in open(os.path.join(ROOT, "include", "rlk.h")).read()


def test_empty_batch_is_a_no_op(lib):
    assert lpe(lib, T=0) == 0


def sup(lib, **kw):
    args = dict(logits=FAKE, dtype=0, T=4, V=100, ld=100, ids=FAKE, temperature=0.7, offs=FAKE,
                sids=FAKE, lp=FAKE, ent=FAKE)
    args.update(kw)
    return lib.rlk_logprob_entropy_support(args["logits"], args["dtype"], args["T"], args["V"],
                                           args["ld"], args["ids"], args["temperature"],
                                           args["offs"], args["sids"], args["lp"], args["ent"],
                                           None, None)


@pytest.mark.parametrize("kw", [
    dict(temperature=0.0), dict(temperature=math.nan), dict(temperature=-2.0), dict(T=-1),
    dict(V=0), dict(V=(1 << 24) + 1), dict(ld=99), dict(dtype=3), dict(logits=None),
    dict(ids=None), dict(offs=None), dict(lp=None), dict(ent=None),
    dict(logits=ctypes.c_void_p(0x10001)),
])
def test_support_rejects(lib, kw):
    assert sup(lib, **kw) == 1


def test_support_empty_batch_is_a_no_op(lib):
    assert sup(lib, T=0, logits=None, ids=None, offs=None, sids=None, lp=None, ent=None) == 0


def sup_bwd(lib, **kw):
    args = dict(logits=FAKE, dtype=0, T=4, V=100, ld=100, ids=FAKE, temperature=0.7, offs=FAKE,
                sids=FAKE, glp=None, gh=None, grad=FAKE)
    args.update(kw)
    return lib.rlk_logprob_entropy_support_backward(
        args["logits"], args["dtype"], args["T"], args["V"], args["ld"], args["ids"],
        args["temperature"], args["offs"], args["sids"], args["glp"], args["gh"], args["grad"],
        None, None)


@pytest.mark.parametrize("kw", [
    dict(temperature=0.0), dict(temperature=math.inf), dict(T=-1), dict(V=0),
    dict(V=(1 << 24) + 1), dict(ld=99), dict(dtype=2), dict(logits=None), dict(ids=None),
    dict(offs=None), dict(grad=None), dict(dtype=1, logits=ctypes.c_void_p(0x10002)),
])
def test_support_backward_rejects(lib, kw):
    assert sup_bwd(lib, **kw) == 1


def test_support_backward_empty_batch_is_a_no_op(lib):
    assert sup_bwd(lib, T=0, logits=None, ids=None, offs=None, sids=None, grad=None) == 0


def fwd(lib, **kw):
    args = dict(logits=FAKE, dtype=0, T=4, V=100, ld=100, ids=FAKE, temperature=0.7, top_p=0.9,
                lp=FAKE, ent=FAKE, state=FAKE)
    args.update(kw)
    return lib.rlk_logprob_entropy_fwd(args["logits"], args["dtype"], args["T"], args["V"],
                                       args["ld"], args["ids"], args["temperature"], args["top_p"],
                                       args["lp"], args["ent"], None, args["state"], None, None)


@pytest.mark.parametrize("kw", [
    dict(state=None), dict(state=ctypes.c_void_p(0x10008)), dict(top_p=0.0), dict(top_p=1.5),
    dict(temperature=0.0), dict(T=-1), dict(ld=99), dict(lp=None),
])
def test_forward_with_state_rejects(lib, kw):
    assert fwd(lib, **kw) == 1


def bwd(lib, **kw):
    args = dict(logits=FAKE, dtype=0, T=4, V=100, ld=100, ids=FAKE, temperature=0.7, state=FAKE,
                glp=None, gh=None, grad=FAKE, gdt=0, ldg=100)
    args.update(kw)
    return lib.rlk_logprob_entropy_bwd(args["logits"], args["dtype"], args["T"], args["V"],
                                       args["ld"], args["ids"], args["temperature"], args["state"],
                                       args["glp"], args["gh"], args["grad"], args["gdt"],
                                       args["ldg"], None, None)


@pytest.mark.parametrize("kw", [
    dict(temperature=0.0), dict(temperature=math.nan), dict(T=-1), dict(V=0),
    dict(V=(1 << 24) + 1), dict(ld=99), dict(ldg=99), dict(dtype=2), dict(gdt=5),
    dict(logits=None), dict(ids=None), dict(state=None), dict(grad=None),
    dict(state=ctypes.c_void_p(0x10004)), dict(gdt=1, grad=ctypes.c_void_p(0x10002)),
    dict(logits=ctypes.c_void_p(0x10001)),
])
def test_backward_rejects(lib, kw):
    assert bwd(lib, **kw) == 1


def test_backward_empty_batch_is_a_no_op(lib):
    assert bwd(lib, T=0, logits=None, ids=None, state=None, grad=None) == 0
    assert fwd(lib, T=0, logits=None, ids=None, lp=None, ent=None, state=None) == 0


def loss(lib, **kw):
    a = dict(n_seq=4, G=2, n_tok=10, el=0.2, eh=0.28, cap=2.0, kl=0.01, agg=0, ws=FAKE,
             ws_bytes=1 << 20, offs=FAKE, out=FAKE)
    a.update(kw)
    return lib.rlk_grpo_loss(FAKE, FAKE, FAKE, FAKE, None, FAKE, a["offs"], a["n_seq"], a["G"],
                             a["n_tok"], a["el"], a["eh"], a["cap"], a["kl"], a["agg"], a["out"],
                             None, None, a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw", [
    dict(n_seq=-1), dict(G=0), dict(n_seq=5, G=2), dict(n_tok=-1), dict(el=-0.1),
    dict(eh=math.inf), dict(cap=0.0), dict(cap=math.nan), dict(kl=-1.0), dict(agg=7),
    dict(offs=None), dict(out=None),
])
def test_grpo_loss_rejects(lib, kw):
    assert loss(lib, **kw) == 1


def test_grpo_loss_workspace_errors(lib):
    assert loss(lib, ws=None) == 3
    assert loss(lib, ws_bytes=16) == 3
    assert loss(lib, ws=ctypes.c_void_p(0x10004)) == 3


def pol(lib, **kw):
    import entropy_logits_bf16_gb300 as rlk
    cfg = dict(type=0, eps_low=0.2, eps_high=0.28, ipo_eps=0.3, band_low=0.5, band_high=2.0,
               is_method=1, is_cap=2.0, kl_coef=0.01, baseline=0, agg=0)
    args = dict(n_seq=4, group=2, n_tok=100, ws=FAKE, wsb=1 << 20, config=True)
    for k in list(kw):
        if k in cfg:
            cfg[k] = kw.pop(k)
    args.update(kw)
    c = rlk.LossConfig(**cfg)
    return lib.rlk_policy_loss(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, args["n_seq"],
                               args["group"], args["n_tok"],
                               ctypes.byref(c) if args["config"] else None, FAKE, None, None,
                               args["ws"], args["wsb"], None)


def test_loss_config_layout():
    import entropy_logits_bf16_gb300 as rlk
    assert ctypes.sizeof(rlk.LossConfig) == 44
    assert rlk.LossConfig.is_method.offset == 24 and rlk.LossConfig.agg.offset == 40


@pytest.mark.parametrize("kw", [
    dict(config=False), dict(type=3), dict(type=-1), dict(is_method=3), dict(baseline=2),
    dict(agg=3), dict(ipo_eps=-0.1), dict(ipo_eps=math.nan), dict(band_low=2.5),
    dict(band_low=-1.0), dict(band_high=math.inf), dict(is_cap=0.0), dict(kl_coef=-1.0),
    dict(eps_low=math.nan), dict(group=3), dict(n_seq=-2),
])
def test_policy_loss_rejects(lib, kw):
    assert pol(lib, **kw) == 1


def test_policy_loss_workspace_and_unused_cap(lib):
    assert pol(lib, ws=None) == 3
    assert pol(lib, wsb=16) == 3
    # the cap is checked only where TIS uses it: these reach the workspace check
    assert pol(lib, is_method=0, is_cap=0.0, ws=None) == 3
    assert pol(lib, is_method=2, is_cap=-1.0, ws=None) == 3


def test_lmhead_rejects(lib):
    f = lib.rlk_lmhead_logprob
    ok = dict(T=4, H=128, V=1000, temp=0.7, p=1.0)
    def call(**kw):
        a = dict(ok, **kw)
        return f(FAKE, FAKE, a["T"], a["H"], a["V"], FAKE, a["temp"], a["p"], FAKE, FAKE, None,
                 None, 0, None)
    assert call(H=100) == 1
    assert call(temp=0.0) == 1
    assert call(p=1.5) == 1
    assert call(V=0) == 1
    assert call(p=0.9) == 3          # top_p < 1 needs the chunk workspace
    assert lib.rlk_workspace_size(4, 100, 151936, 4096) >= 100 * 151936 * 2



def test_lmhead_fwd_bwd_reject(lib):
    ok = dict(T=4, H=128, V=1000, temp=0.7)
    def fwd(lse=FAKE, **kw):
        a = dict(ok, **kw)
        return lib.rlk_lmhead_logprob_fwd(FAKE, FAKE, a["T"], a["H"], a["V"], FAKE, a["temp"], 1.0,
                                          FAKE, FAKE, lse, None, FAKE, 1 << 30, None)
    assert fwd(lse=None) == 1
    assert fwd(H=96) == 1
    assert lib.rlk_lmhead_logprob_fwd(FAKE, FAKE, 4, 128, 1000, FAKE, 0.7, 0.9, FAKE, FAKE, FAKE,
                                      None, FAKE, 1 << 40, None) == 2   # the lse is top_p = 1 only
    def bwd(ws=FAKE, wsb=1 << 40, **kw):
        a = dict(dict(ok, lse=FAKE, ent=FAKE, gh=FAKE, gw=FAKE), **kw)
        return lib.rlk_lmhead_logprob_bwd(FAKE, FAKE, a["T"], a["H"], a["V"], FAKE, a["temp"],
                                          a["lse"], a["ent"], None, None, a["gh"], a["gw"], 0, ws,
                                          wsb, None)
    for kw in (dict(H=100), dict(H=0), dict(V=0), dict(T=-1), dict(temp=0.0), dict(lse=None),
               dict(ent=None), dict(gh=None), dict(gw=None), dict(gw=ctypes.c_void_p(0x10004))):
        assert bwd(**kw) == 1, kw
    assert bwd(ws=None) == 3
    assert bwd(wsb=1024) == 3
    assert bwd(ws=ctypes.c_void_p(0x10010)) == 3      # the workspace must be 256-byte aligned
    assert bwd(T=0, lse=None, ent=None, gh=None, gw=None, ws=None) == 0
    need = lib.rlk_workspace_size(3, 10000, 151936, 4096)
    assert need >= 4096 * 151936 * 2          # the gradient logits of one chunk of rows


def test_canonical_rejects(lib):
    def part(**kw):
        a = dict(dtype=0, T=4, V=1000, ld=1000, first=0, W=125, n=8, temp=0.7, out=FAKE)
        a.update(kw)
        return lib.rlk_shard_partials(FAKE, a["dtype"], a["T"], a["V"], a["ld"], a["first"], a["W"],
                                      a["n"], FAKE, a["temp"], a["out"], None)
    for kw in (dict(W=0), dict(n=0), dict(first=-125), dict(first=100), dict(ld=999), dict(dtype=7),
               dict(temp=0.0), dict(out=None), dict(out=ctypes.c_void_p(0x10008)), dict(V=0)):
        assert part(**kw) == 1, kw
    assert part(T=0, out=None) == 0
    def comb(**kw):
        a = dict(n=8, T=4, V=1000, W=125)
        a.update(kw)
        return lib.rlk_shard_combine(FAKE, a["n"], a["T"], a["V"], a["W"], FAKE, 0.7, FAKE, FAKE,
                                     None, None)
    assert comb(W=124) == 1                     # the shards must cover V
    assert comb(n=0) == 1
    def canon(**kw):
        a = dict(n=8, P=1000, ws=FAKE, wsb=1 << 20)
        a.update(kw)
        return lib.rlk_logprob_entropy_canonical(FAKE, 0, 4, 1000, 1000, FAKE, 0.7, a["n"], a["P"],
                                                 FAKE, FAKE, None, a["ws"], a["wsb"], None)
    assert canon(P=999) == 1 and canon(P=1001) == 1 and canon(n=0) == 1
    assert canon(ws=None) == 3 and canon(wsb=16) == 3
    assert lib.rlk_workspace_size(5, 100, 8, 0) == 100 * 8 * 32
    assert lib.rlk_workspace_size(6, 100, 8, 0) == 100 * 8 * (32 + 8224)
    def win(**kw):
        a = dict(dtype=0, T=4, V=1000, ld=1000, first=0, W=125, n=8, temp=0.7, p=0.9, nall=8,
                 allp=FAKE, out=FAKE)
        a.update(kw)
        return lib.rlk_shard_window_counts(FAKE, a["dtype"], a["T"], a["V"], a["ld"], a["first"],
                                           a["W"], a["n"], FAKE, a["temp"], a["p"], a["allp"],
                                           a["nall"], a["out"], None)
    for kw in (dict(p=1.0), dict(p=0.0), dict(nall=7), dict(W=0), dict(first=100), dict(ld=999),
               dict(allp=None), dict(out=ctypes.c_void_p(0x10008)), dict(temp=-1.0)):
        assert win(**kw) == 1, kw
    assert win(dtype=1) == 2                    # fp32 logits: no per-value counts
    assert win(T=0, out=None) == 0
    def ctp(**kw):
        a = dict(n=8, T=4, V=1000, W=125, p=0.9, cnt=FAKE)
        a.update(kw)
        return lib.rlk_shard_combine_topp(FAKE, a["cnt"], a["n"], a["T"], a["V"], a["W"], FAKE,
                                          0.7, a["p"], FAKE, FAKE, None, None, None)
    assert ctp(W=124) == 1 and ctp(p=1.0) == 1 and ctp(cnt=None) == 1
    def ctopp(**kw):
        a = dict(n=8, P=1000, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return lib.rlk_logprob_entropy_canonical_topp(FAKE, 0, 4, 1000, 1000, FAKE, 0.7, 0.9,
                                                      a["n"], a["P"], FAKE, FAKE, None, None,
                                                      a["ws"], a["wsb"], None)
    assert ctopp(P=999) == 1 and ctopp(n=0) == 1
    assert ctopp(ws=None) == 3 and ctopp(wsb=4 * 8 * (32 + 8224) - 1) == 3


def test_injected_launch_failures_come_before_any_launch(lib):
    """Host-side fault injection: calls whose arguments pass validation return
    RLK_ERR_CUDA without launching.  More failures are injected than calls are
    made, so no call here reaches a launch with the placeholder pointers."""
    assert lib.rlk_debug_inject_launch_failures(5) == 0
    assert lpe(lib) == 4
    assert sup(lib) == 4
    assert sup_bwd(lib) == 4
    assert lib.rlk_debug_inject_launch_failures(0) == 2      # two were left
    assert lib.rlk_debug_inject_launch_failures(-3) == 0     # a negative count clears


def test_binding_refuses_cpu_tensors(lib):
    import torch
    z = torch.zeros(2, 8, dtype=torch.bfloat16)
    ids = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):
        rlk.logprob_entropy(z, ids, 0.7, 0.95)


@pytest.fixture
def armed(lib):
    """Host-side fault injection armed for the test: a call whose arguments
    the host checks pass returns RLK_ERR_CUDA instead of launching, so the
    placeholder pointers below can never reach a device."""
    lib.rlk_debug_inject_launch_failures(1000)
    yield
    lib.rlk_debug_inject_launch_failures(0)


def test_rows_rejects(lib, armed):
    def rows(**kw):
        a = dict(logits=FAKE, dtype=0, T=4, V=100, ld=100, ids=FAKE, temps=FAKE, tops=FAKE,
                 lp=FAKE, ent=FAKE, state=None)
        a.update(kw)
        return lib.rlk_logprob_entropy_rows(a["logits"], a["dtype"], a["T"], a["V"], a["ld"],
                                            a["ids"], a["temps"], a["tops"], a["lp"], a["ent"],
                                            None, a["state"], None, None)
    for kw in (dict(dtype=3), dict(T=-1), dict(V=0), dict(V=(1 << 24) + 1), dict(ld=99),
               dict(logits=None), dict(ids=None), dict(temps=None), dict(tops=None),
               dict(lp=None), dict(ent=None), dict(logits=ctypes.c_void_p(0x10001)),
               dict(dtype=1, logits=ctypes.c_void_p(0x10002)),
               dict(state=ctypes.c_void_p(0x10008))):
        assert rows(**kw) == 1, kw
    assert rows(T=0, logits=None, ids=None, temps=None, tops=None, lp=None, ent=None) == 0
    assert rows() == 4 and rows(state=ctypes.c_void_p(0x10010)) == 4   # checks passed: injected


def test_sample_top_p_rejects(lib, armed):
    def smp(**kw):
        a = dict(logits=FAKE, dtype=0, T=4, V=100, ld=100, temp=0.7, state=FAKE, u=FAKE,
                 out=FAKE)
        a.update(kw)
        return lib.rlk_sample_top_p(a["logits"], a["dtype"], a["T"], a["V"], a["ld"], a["temp"],
                                    a["state"], a["u"], a["out"], None, None)
    for kw in (dict(dtype=3), dict(T=-1), dict(V=0), dict(ld=99), dict(temp=0.0),
               dict(temp=math.inf), dict(temp=math.nan), dict(logits=None), dict(state=None),
               dict(u=None), dict(out=None), dict(logits=ctypes.c_void_p(0x10001)),
               dict(state=ctypes.c_void_p(0x10008))):
        assert smp(**kw) == 1, kw
    assert smp(dtype=1) == 2                                  # fp32 logits: not supported
    assert smp(T=0, logits=None, state=None, u=None, out=None) == 0
    assert smp() == 4                                          # checks passed: injected


def test_shard_partials_support_rejects(lib, armed):
    def part(**kw):
        a = dict(dtype=0, T=4, V=1000, ld=1000, first=0, W=125, n=8, temp=0.7, off=FAKE,
                 out=FAKE)
        a.update(kw)
        return lib.rlk_shard_partials_support(FAKE, a["dtype"], a["T"], a["V"], a["ld"],
                                              a["first"], a["W"], a["n"], FAKE, a["temp"],
                                              a["off"], FAKE, a["out"], None)
    for kw in (dict(W=0), dict(n=0), dict(first=-125), dict(first=100), dict(ld=999),
               dict(dtype=7), dict(temp=0.0), dict(off=None), dict(out=None),
               dict(out=ctypes.c_void_p(0x10008)), dict(V=0)):
        assert part(**kw) == 1, kw
    assert part(T=0, off=None, out=None) == 0
    assert part() == 4                                         # checks passed: injected


def test_debug_settings_round_trip(lib):
    """The host-side debug settings return the previous value and restore
    their defaults (no device work)."""
    assert rlk.set_sampler_mode(0) == 1
    assert rlk.set_sampler_mode(2) == 0
    assert rlk.set_sampler_mode(7) == 2      # anything else: the default
    assert rlk.set_sampler_mode(1) == 1
    prev = rlk.set_wait_limit(1234)
    assert rlk.set_wait_limit(0) == 1234     # <= 0 restores the default
    assert rlk.set_wait_limit(prev) == prev
