"""Benchmark: tokens/s of top-p logprob + entropy at V=151936 bf16, and the
fraction of the HBM roofline the kernel reaches.

One step = one pass of the hot path over one batch of synthetic
Qwen3-8B-shaped logits (T=4096 rows, V=151936 bf16, temperature 0.7,
top_p 0.95; inputs 1.24 GB, larger than L2, so no flush is needed between
steps): rlk_logprob_entropy (max / log-sum-exp / entropy, nucleus select,
renormalisation) and then rlk_grpo_loss on the step's log-probs (64 responses
x 64 tokens in groups of 8).  The roofline figure is for the
rlk_logprob_entropy call, timed with its own events inside the step.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference] [--op logits|lmhead]

--op lmhead times the fused LM-head instead (its own metric and a tensor
roofline); the default line is the benchmark's.

Rows are independent, so N > 1 (one process per GPU via torchrun) runs N
replicas with no collective on the data path: weak scaling.  ``--impl
reference`` times the fp64 CPU oracle, as it stands, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

T_ROWS = 4096
VOCAB = 151936
TEMPERATURE = 0.7
TOP_P = 0.95
ROW_BYTES = VOCAB * 2
BYTES_PER_TOKEN = ROW_BYTES + 4 + 12     # logits row + id + (logprob, entropy, k*) outputs
METRIC = "tokens/s for top-p logprob+entropy at V=151936 bf16; % of HBM roofline"
KERNEL_SRC = os.path.join(ROOT, "entropy_logits_bf16_gb300", "csrc", "lpe_stream.cu")
PROFILE = os.path.join(ROOT, "profiles", "lpe_stream_kernel_qwen_T4096.txt")
WORKLOAD = (f"Qwen3-8B-shaped logits T={T_ROWS} V={VOCAB} bf16 = 3 N(0,1) + one peak U(5,15) "
            f"per row; temperature {TEMPERATURE}, top_p {TOP_P}; ids drawn from each row's "
            f"truncated distribution")
HBM_NOMINAL_GBS = 7900.0      # GB300 HBM3e nominal bandwidth
BF16_NOMINAL_TFLOPS = 2250.0  # GB300 dense bf16 nominal


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, dev) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: int, steps: int, ws: int, elapsed_ms: float) -> float:
    """Units all ranks processed per second over the (max-over-ranks) elapsed time."""
    return units_per_rank_step * steps * ws / (elapsed_ms / 1e3)


def rank_seed(rank: int) -> int:
    """Replicas draw different batches: rank r uses seed 1 + r."""
    return 1 + int(rank)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        # one earlier GB300 measurement: copy bandwidth, bf16 burst and sustained
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


BWD_SRC = os.path.join(ROOT, "entropy_logits_bf16_gb300", "csrc", "lpe_backward.cu")
BWD_PROFILE = os.path.join(ROOT, "profiles", "lpe_backward_pipe_kernel_qwen_T4096.txt")
CSRC = os.path.join(ROOT, "entropy_logits_bf16_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


def kernel_sha(src=KERNEL_SRC):
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(src=KERNEL_SRC, profile=PROFILE):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    try:
        kv = {}
        with open(profile) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_sha(src):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def sampled_ids(z, seed, temperature=TEMPERATURE, top_p=TOP_P):
    """Each row's selected id drawn from its temperature-scaled, top-p-truncated,
    renormalised distribution (the library's deterministic sampler, whose draws
    are tested against the oracle's inverse-CDF sampler), with seeded uniforms.
    Runs before any timed region."""
    import entropy_logits_bf16_gb300 as rlk
    import workloads
    u = torch.from_numpy(np.ascontiguousarray(workloads.uniforms(z.shape[0], seed),
                                              dtype=np.float32)).to(z.device)
    return rlk.sample_top_p(z, temperature, top_p, u)


def make_workload(device, seed):
    import workloads
    z, _ = workloads.peaked_bf16(T_ROWS, VOCAB, seed=seed, device=device)
    return z, sampled_ids(z, 1000 + seed)


def cpu_baseline(z, ids, min_seconds=10.0, max_reps=8):
    """The oracle, as it stands, on the whole batch of the same workload,
    repeated until at least min_seconds of CPU work have been timed."""
    import oracle
    import workloads
    hz = np.ascontiguousarray(workloads.bf16_bits(z))
    hid = ids.cpu().numpy()
    threads = oracle.default_threads()
    oracle.build()
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.logprob_entropy(hz, hid, TEMPERATURE, TOP_P, threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or reps >= max_reps:
            break
    return {"value": reps * T_ROWS / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"all {T_ROWS} rows of the workload x {reps}, fp64 oracle, {threads} threads, "
                      f"{dt:.2f} s"}


def run_reference(args):
    """--impl reference: the fp64 CPU oracle timed on the host cores."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    import workloads
    oracle.build()
    rows_per_step = 64
    z, peaks = workloads.peaked_bf16(rows_per_step * 4, VOCAB, seed=1, device="cpu")
    hz = workloads.bf16_bits(z)
    hid = oracle.sample_ids(hz, TEMPERATURE, TOP_P, workloads.uniforms(hz.shape[0], 1001))
    threads = oracle.default_threads()
    # the loss stage on each step's log-probs, as in the device step: the
    # sample's 64 tokens as 8 responses of 8 tokens in one group of 8;
    # old / rollout / reference log-probs from the first sample's plus N(0, 0.01^2)
    n_seq = rows_per_step // 8
    off_h = (np.arange(n_seq + 1) * 8).astype(np.int32)
    R_h = (np.random.default_rng(7).random(n_seq) < 0.5).astype(np.float32)
    lp0, _, _, _ = oracle.logprob_entropy(hz[:rows_per_step], hid[:rows_per_step], TEMPERATURE,
                                          TOP_P, threads=threads)
    old_h, ro_h, ref_h = workloads.perturbed_logps(lp0.astype(np.float32), 5)

    def step(i):
        s = (i % 4) * rows_per_step
        lp, _, _, _ = oracle.logprob_entropy(hz[s:s + rows_per_step], hid[s:s + rows_per_step],
                                             TEMPERATURE, TOP_P, threads=threads)
        new = np.where(np.isfinite(lp), lp, old_h).astype(np.float32)
        oracle.grpo_loss(new, old_h, ro_h, ref_h, None, R_h, off_h, 8)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = rows_per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": rows_per_step, "V": VOCAB,
                   "temperature": TEMPERATURE, "top_p": TOP_P, "global_batch": rows_per_step,
                   "loss": (f"GRPO/DAPO loss on the step's log-probs: {n_seq} sequences x 8 tokens, "
                            f"group 8, eps 0.2/0.28, TIS cap 2.0, k3 KL 0.01, token mean"),
                   "parallelism": "host cores, rank 0 only", "rows_per_step": rows_per_step,
                   "same_config": False,
                   "same_config_reason": (f"the fp64 oracle scores {rows_per_step} rows of the "
                                          f"{T_ROWS}-row device workload per step (a bounded "
                                          f"sample), then an {n_seq} x 8-token loss")},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} rows per step of the same workload, then "
                                   f"the loss on their log-probs ({n_seq} responses x 8 tokens, "
                                   f"groups of 8)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


GRPO_SEQ, GRPO_LEN, GRPO_G = 64, 64, 8          # 64 responses x 64 tokens, groups of 8
LOSS_CFG = (f"GRPO/DAPO loss on the step's log-probs: {GRPO_SEQ} sequences x {GRPO_LEN} tokens, "
            f"group {GRPO_G}, eps 0.2/0.28, TIS cap 2.0, k3 KL 0.01, token mean")
LM_T, LM_H = 16384, 4096
ZIPF_ROWS = 8 * 6912   # the long-response batch: 8 responses x 6912 tokens
LM_METRIC = "tokens/s for fused LM-head logprob+entropy (top_p 1) at V=151936, H=4096 bf16; % of bf16 peak"


def timed_steps(args, ws, dev, stream, parts, barrier):
    """W untimed steps, then K timed ones bracketed by barriers; returns
    (elapsed_ms over all steps, per-part mean ms, clock record).  `parts` are
    callables run in order each step, each bracketed by its own events."""
    for _ in range(max(args.warmup, 3)):
        for f in parts:
            f()
    barrier()
    clocks = ClockSampler(dist_env()[2] if ws > 1 else 0)
    clocks.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)]
           for _ in range(args.steps)]
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        evs[i][0].record(stream)
        for j, f in enumerate(parts):
            f()
            evs[i][j + 1].record(stream)
    t_stop.record(stream)
    barrier()
    elapsed_ms = t_start.elapsed_time(t_stop)
    part_ms = [sum(e[j].elapsed_time(e[j + 1]) for e in evs) / args.steps for j in range(len(parts))]
    clk = clocks.stop()
    return reduce_max(elapsed_ms, dev), part_ms, clk


def run_logits(args, ws, rank, dev, barrier):
    import entropy_logits_bf16_gb300 as rlk
    import workloads
    lib = rlk.load()
    stream = torch.cuda.current_stream(dev)
    z, ids = make_workload(dev, seed=rank_seed(rank))
    lp = torch.empty(T_ROWS, device=dev)
    ent = torch.empty(T_ROWS, device=dev)
    ks = torch.empty(T_ROWS, device=dev, dtype=torch.int32)

    def logprob():
        code = lib.rlk_logprob_entropy(
            rlk._ptr(z), 0, T_ROWS, VOCAB, VOCAB, rlk._ptr(ids), TEMPERATURE, TOP_P,
            rlk._ptr(lp), rlk._ptr(ent), rlk._ptr(ks), None, None, 0, rlk._stream(dev))
        if code != 0:
            raise RuntimeError(f"rlk_logprob_entropy returned {code}")

    # the loss stage: old / rollout / reference log-probs are the first step's
    # log-probs plus N(0, 0.01^2); rewards Bernoulli(0.5)
    logprob()
    torch.cuda.synchronize(dev)
    old_h, ro_h, ref_h = workloads.perturbed_logps(lp.cpu().numpy(), 5 + rank)
    rng = np.random.default_rng([7, rank])
    R_h = (rng.random(GRPO_SEQ) < 0.5).astype(np.float32)
    off_h = (np.arange(GRPO_SEQ + 1) * GRPO_LEN).astype(np.int32)
    assert off_h[-1] == T_ROWS
    tdev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    old, ro, ref, R, off = tdev(old_h), tdev(ro_h), tdev(ref_h), tdev(R_h), tdev(off_h)
    loss = torch.empty(1, device=dev)
    grad = torch.empty(T_ROWS, device=dev)
    stats = torch.empty(8, device=dev)
    wsb = rlk.workspace_size(1, T_ROWS, GRPO_SEQ)
    wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)

    def grpo(new=lp, o=old, r_=ro, f=ref, rw=R, of=off, out=loss):
        code = lib.rlk_grpo_loss(rlk._ptr(new), rlk._ptr(o), rlk._ptr(r_), rlk._ptr(f), None,
                                 rlk._ptr(rw), rlk._ptr(of), GRPO_SEQ, GRPO_G, T_ROWS, 0.2, 0.28,
                                 2.0, 0.01, 0, rlk._ptr(out), rlk._ptr(grad), rlk._ptr(stats),
                                 rlk._ptr(wsp), wsb, rlk._stream(dev))
        if code != 0:
            raise RuntimeError(f"rlk_grpo_loss returned {code}")

    elapsed_ms, part_ms, clk = timed_steps(args, ws, dev, stream, [logprob, grpo], barrier)

    # end to end through the public API: pinned host inputs -> device -> the
    # hot path -> the loss, log-probs and entropies back on the host.  The
    # host->device copy (~210 GB/s, whatever the number of streams) dominates,
    # so the rows go over in chunks and each chunk's kernels start as soon as
    # its copy has landed, on a second stream.
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
    host = [pin(t) for t in (z, ids, old, ro, ref, R, off)]
    dev_in = [torch.empty_like(t) for t in (z, ids, old, ro, ref, R, off)]
    out_h = torch.empty(2 * T_ROWS + 1, dtype=torch.float32, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 10))
    copy_s = torch.cuda.Stream(dev)
    n_chunk = 8
    rows_c = T_ROWS // n_chunk

    def e2e_step():
        hz, hids = host[0], host[1]
        dz, dids, dold, dro, dref, dR, doff = dev_in
        copy_s.wait_stream(stream)
        done = []
        with torch.cuda.stream(copy_s):
            for c in range(n_chunk):
                sl = slice(c * rows_c, (c + 1) * rows_c)
                dz[sl].copy_(hz[sl], non_blocking=True)
                dids[sl].copy_(hids[sl], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_s)
                done.append(ev)
            for d, h in zip(dev_in[2:], host[2:]):
                d.copy_(h, non_blocking=True)
        for c in range(n_chunk):
            sl = slice(c * rows_c, (c + 1) * rows_c)
            stream.wait_event(done[c])
            rlk.logprob_entropy(dz[sl], dids[sl], TEMPERATURE, TOP_P, out_logprob=lp[sl],
                                out_entropy=ent[sl])
        stream.wait_stream(copy_s)
        grpo(lp, dold, dro, dref, dR, doff, loss)
        out_h[:T_ROWS].copy_(lp, non_blocking=True)
        out_h[T_ROWS:2 * T_ROWS].copy_(ent, non_blocking=True)
        out_h[2 * T_ROWS:].copy_(loss, non_blocking=True)

    e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, dev)
    cpu_line = cpu_baseline(z, ids) if (ws == 1 and rank == 0 and not args.no_cpu_baseline) else None
    h2d_bytes = int(sum(t.numel() * t.element_size() for t in host))
    legs = None
    if not args.no_legs:   # every rank runs them (their timings cross ranks)
        del z, dev_in, host
        torch.cuda.empty_cache()
        legs = {}
        for name, fn in (("long_response_zipf_stress", lambda: leg_zipf(args, ws, rank, dev, barrier, 1.0)),
                         ("long_response_zipf_calibrated",
                          lambda: leg_zipf(args, ws, rank, dev, barrier, None)),
                         ("grpo_packed_591k", lambda: leg_grpo(args, ws, rank, dev, barrier)),
                         ("fused_lmhead", lambda: leg_lmhead(args, ws, rank, dev, barrier))):
            legs[name] = fn()
            torch.cuda.empty_cache()
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    launch_ms = part_ms[0]
    alg_bytes = BYTES_PER_TOKEN * T_ROWS
    achieved = alg_bytes / (launch_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": whole_job_rate(T_ROWS, args.steps, ws, elapsed_ms), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_ROWS, "V": VOCAB, "temperature": TEMPERATURE,
                   "top_p": TOP_P, "global_batch": T_ROWS * ws, "loss": LOSS_CFG,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "inputs (1.24 GB per GPU) larger than L2; no flush between steps",
                   "step_ms": {"logprob_entropy": part_ms[0], "grpo_loss": part_ms[1]}},
        "roofline": hbm_roofline(achieved, peaks, peak_kind, launch_ms, clk,
                                 kernel="lpe_stream_kernel<top_p<1> (+ the per-row recompute pass, "
                                        "timed together as one rlk_logprob_entropy call)",
                                 traffic=profiled_traffic(), bytes_per_token=BYTES_PER_TOKEN,
                                 tokens_per_launch=T_ROWS),
        "e2e": {"value": T_ROWS * ws / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": int(out_h.numel() * 4)},
        # streaming kernel + recompute pass + the loss's three kernels, per step
        "gpu_launches": 5 * args.steps,
        "clocks": clk,
    }
    if cpu_line is not None:
        line["cpu_baseline"] = cpu_line
    if legs is not None:
        line["legs"] = legs
    return line


def hbm_roofline(achieved, peaks, peak_kind, launch_ms, clk, **extra):
    """The HBM roofline entry: the fraction of the measured copy bandwidth
    (the task's denominator), with the nominal HBM3e bandwidth and the clock
    the launch ran at beside it."""
    r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": achieved / peaks["hbm_gbs"], "peak_source": peak_kind,
         "peak_nominal": HBM_NOMINAL_GBS, "frac_of_nominal": achieved / HBM_NOMINAL_GBS,
         "launch_ms": launch_ms}
    r.setdefault("traffic", None)
    r.update(extra)
    if clk:
        r["sm_mhz_median"] = clk["sm_mhz"]
        r["launch_ms_x_sm_ghz"] = launch_ms * clk["sm_mhz"] / 1e3
    return r


def leg_args(args, steps):
    class A:
        pass
    a = A()
    a.steps = min(args.steps, steps)
    a.warmup = max(args.warmup, 3)
    a.no_cpu_baseline = args.no_cpu_baseline
    return a


def leg_zipf(args, ws, rank, dev, barrier, kappa):
    """Long-response batch: 8 responses x 6912 tokens (T = 55,296 rows), V =
    151,936 bf16 rows with Zipf-tilted means, temperature 0.7, top_p 0.95, ids
    drawn from the truncated distributions.  kappa None: the calibrated rows
    (nucleus sizes 1 to ~5000); 1.0: the wider stress rows.  Rows the streaming
    kernel hands to the per-row kernel are counted from the row state (the
    per-row kernel's reference exponent is not an integer)."""
    import entropy_logits_bf16_gb300 as rlk
    import workloads
    rows = ZIPF_ROWS
    k = workloads.ZIPF_KAPPA_CALIBRATED if kappa is None else kappa
    z, _ = workloads.zipf_bf16(rows, seed=2 + 100 * rank, kappa=k, sigma=workloads.ZIPF_SIGMA,
                               device=dev)
    ids = sampled_ids(z, 2000 + rank)
    lp = torch.empty(rows, device=dev)
    ent = torch.empty(rows, device=dev)
    stream = torch.cuda.current_stream(dev)

    def f():
        rlk.logprob_entropy(z, ids, TEMPERATURE, TOP_P, out_logprob=lp, out_entropy=ent)

    la = leg_args(args, 5)
    elapsed_ms, part_ms, clk = timed_steps(la, ws, dev, stream, [f], barrier)
    st = rlk.new_row_state(rows, dev)
    _, _, ks = rlk.logprob_entropy(z, ids, TEMPERATURE, TOP_P, row_state=st, return_nucleus_size=True)
    E = st[:, 0].contiguous().view(torch.float32)
    recomputed = float((E != torch.floor(E)).float().mean().item())
    kq = torch.quantile(ks.float()[::7], torch.tensor([0.0, 0.5, 0.9, 0.99, 1.0], device=dev)).tolist()
    peaks, peak_kind = measured_peaks()
    achieved = rows * BYTES_PER_TOKEN / (part_ms[0] / 1e3) / 1e9
    out = {"metric": "tokens/s", "value": whole_job_rate(rows, la.steps, ws, elapsed_ms),
           "unit": "tokens/s", "steps": la.steps, "ms_per_step": elapsed_ms / la.steps,
           "config": {"workload": (f"long-response batch of {rows} rows (8 x 6912 = 55296 in full), V={VOCAB} bf16, "
                                   f"z = bf16(-kappa s ln rank + sigma N(0,1)), s ~ U(0.8,1.4), "
                                   f"kappa {k}, sigma {workloads.ZIPF_SIGMA}, temperature "
                                   f"{TEMPERATURE}, top_p {TOP_P}; ids from the truncated "
                                   f"distribution; boundary ties not injected"),
                      "T": rows, "V": VOCAB, "kappa": k, "sigma": workloads.ZIPF_SIGMA,
                      "nucleus_size_quantiles_0_50_90_99_100": [round(x) for x in kq],
                      "rows_recomputed_by_per_row_kernel": recomputed,
                      "l2": f"inputs ({rows * VOCAB * 2 / 1e9:.1f} GB) larger than L2"},
           "roofline": hbm_roofline(achieved, peaks, peak_kind, part_ms[0], clk,
                                    kernel="one rlk_logprob_entropy call (streaming kernel + "
                                           "per-row recompute pass)",
                                    bytes_per_token=BYTES_PER_TOKEN, tokens_per_launch=rows),
           "clocks": clk}
    if ws == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        sel = np.linspace(0, rows - 1, 96).astype(np.int64)
        sel_t = torch.from_numpy(sel).to(dev)
        hz = workloads.bf16_bits(z[sel_t])
        hid = ids[sel_t].cpu().numpy()
        threads = oracle.default_threads()
        oracle.build()
        t0 = time.perf_counter()
        oracle.logprob_entropy(hz, hid, TEMPERATURE, TOP_P, threads=threads)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": len(sel) / dt, "unit": "tokens/s", "cores": threads,
                               "kind": "oracle",
                               "sample": f"{len(sel)} evenly spaced rows, fp64 oracle, {threads} "
                                         f"threads, {dt:.2f} s"}
    del z
    return out


def run_zipf(args, ws, rank, dev, barrier):
    """--op zipf: the calibrated long-response leg on its own (--zipf-rows
    rows; 55,296 by default, fewer for a profile)."""
    out = leg_zipf(args, ws, rank, dev, barrier, None)
    if rank != 0:
        return None
    out.update({"metric": "tokens/s for top-p logprob+entropy on the calibrated long-response rows "
                          "at V=151936 bf16", "n_gpus": ws, "warmup": args.warmup,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic", "gpu_launches": 2 * out["steps"]})
    return out


def leg_grpo(args, ws, rank, dev, barrier):
    """GRPO/DAPO batch: 64 prompts x group 8, response lengths U{256..2048}
    packed (591,145 tokens at seed 3), logits as the Qwen3-shaped rows scored
    16,384 rows at a time (each chunk regenerated from the seeded generator
    before its scorer call, outside the timed events), then the loss over all
    tokens with old / rollout / reference log-probs = the first pass's
    log-probs + N(0, 0.01^2).  Timed: the scorer calls and the loss."""
    import entropy_logits_bf16_gb300 as rlk
    import workloads
    off_h, R_h = workloads.grpo_batch(64, 8, 256, 2048, seed=3)
    n = int(off_h[-1])
    CH = 16384
    chunks = [(c0, min(CH, n - c0)) for c0 in range(0, n, CH)]
    lp = torch.empty(n, device=dev)
    ent = torch.empty(n, device=dev)
    ids_all = torch.empty(n, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def chunk(c0, cn):
        z, _ = workloads.peaked_bf16(cn, VOCAB, seed=3 + 100 * rank, device=dev, row0=c0)
        return z

    for c0, cn in chunks:   # ids from each chunk's truncated distributions, and a first pass
        z = chunk(c0, cn)
        ids_all[c0:c0 + cn] = sampled_ids(z, 3000 + c0 + rank)
        rlk.logprob_entropy(z, ids_all[c0:c0 + cn], TEMPERATURE, TOP_P,
                            out_logprob=lp[c0:c0 + cn], out_entropy=ent[c0:c0 + cn])
        del z
    lp_h = lp.cpu().numpy()
    finite = np.isfinite(lp_h)
    old_h, ro_h, ref_h = workloads.perturbed_logps(np.where(finite, lp_h, -20.0), 9 + rank)
    tdev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    old, ro, ref, R, off = tdev(old_h), tdev(ro_h), tdev(ref_h), tdev(R_h), tdev(off_h)
    n_seq = len(R_h)
    wsb = rlk.workspace_size(1, n, n_seq)
    wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    loss = torch.empty(1, device=dev)
    grad = torch.empty(n, device=dev)
    new = torch.empty(n, device=dev)

    lib = rlk.load()
    stats = torch.empty(8, device=dev)

    def run_loss():
        torch.where(torch.isfinite(lp), lp, old, out=new)
        code = lib.rlk_grpo_loss(rlk._ptr(new), rlk._ptr(old), rlk._ptr(ro), rlk._ptr(ref), None,
                                 rlk._ptr(R), rlk._ptr(off), n_seq, 8, n, 0.2, 0.28, 2.0, 0.01, 0,
                                 rlk._ptr(loss), rlk._ptr(grad), rlk._ptr(stats), rlk._ptr(wsp),
                                 wsb, rlk._stream(dev))
        if code != 0:
            raise RuntimeError(f"rlk_grpo_loss returned {code}")

    steps = min(args.steps, 2)
    score_ms, loss_ms = [], []
    clocks = ClockSampler(dist_env()[2] if ws > 1 else 0)
    for it in range(steps + 1):
        if it == 1:
            clocks.start()
        t_sc = 0.0
        for c0, cn in chunks:
            z = chunk(c0, cn)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            e0.record(stream)
            rlk.logprob_entropy(z, ids_all[c0:c0 + cn], TEMPERATURE, TOP_P,
                                out_logprob=lp[c0:c0 + cn], out_entropy=ent[c0:c0 + cn])
            e1.record(stream)
            barrier()
            t_sc += e0.elapsed_time(e1)
            del z
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_loss()
        e1.record(stream)
        barrier()
        if it > 0:
            score_ms.append(t_sc)
            loss_ms.append(e0.elapsed_time(e1))
    clk = clocks.stop()
    sc = reduce_max(sum(score_ms) / steps, dev)
    ls = reduce_max(sum(loss_ms) / steps, dev)
    peaks, peak_kind = measured_peaks()
    achieved = n * BYTES_PER_TOKEN / (sc / 1e3) / 1e9
    out = {"metric": "tokens/s", "value": n * ws / ((sc + ls) / 1e3), "unit": "tokens/s",
           "steps": steps, "ms_per_step": sc + ls,
           "step_ms": {"logprob_entropy_all_chunks": sc, "grpo_loss": ls},
           "config": {"workload": (f"GRPO/DAPO: 64 prompts x group 8, lengths U{{256..2048}} packed "
                                   f"({n} tokens, seed 3); Qwen3-shaped logits V={VOCAB} bf16 "
                                   f"scored {CH} rows at a time ({len(chunks)} chunks, "
                                   f"regenerated outside the timed events); rewards "
                                   f"Bernoulli(0.5); old/rollout/ref = new + N(0, 0.01^2); "
                                   f"eps 0.2/0.28, TIS cap 2.0, k3 KL 0.01, token mean"),
                      "tokens": n, "sequences": n_seq, "chunk_rows": CH},
           "roofline": hbm_roofline(achieved, peaks, peak_kind, sc, clk,
                                    kernel="the rlk_logprob_entropy calls over all chunks",
                                    bytes_per_token=BYTES_PER_TOKEN, tokens_per_launch=n),
           "loss_roofline_note": "the loss reads ~21 B a token and is launch/latency-bound",
           "clocks": clk}
    if ws == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        threads = oracle.default_threads()
        oracle.build()
        z = chunk(0, CH)
        sel = np.arange(0, CH, 256)
        sel_t = torch.from_numpy(sel).to(dev)
        hz = workloads.bf16_bits(z[sel_t])
        hid = ids_all[sel_t].cpu().numpy()
        del z
        t0 = time.perf_counter()
        oracle.logprob_entropy(hz, hid, TEMPERATURE, TOP_P, threads=threads)
        t_rows = (time.perf_counter() - t0) / len(sel)
        new_h = np.where(finite, lp_h, old_h).astype(np.float32)
        t0 = time.perf_counter()
        oracle.grpo_loss(new_h, old_h, ro_h, ref_h, None, R_h, off_h, 8)
        t_loss = time.perf_counter() - t0
        est = n * t_rows + t_loss
        out["cpu_baseline"] = {"value": n / est, "unit": "tokens/s", "cores": threads,
                               "kind": "oracle",
                               "sample": (f"{len(sel)} rows (every 256th of the first chunk) "
                                          f"scored at {t_rows * 1e3:.1f} ms a row on {threads} "
                                          f"threads, extrapolated to all {n} rows, plus the "
                                          f"loss over all tokens ({t_loss:.2f} s)")}
    return out


def leg_lmhead(args, ws, rank, dev, barrier):
    """The fused LM-head (config 5) at top_p 1, as --op lmhead, without the
    end-to-end copy."""
    line = run_lmhead(leg_args(args, 5), ws, rank, dev, barrier, top_p=1.0, leg=True)
    return line


def run_lmhead(args, ws, rank, dev, barrier, top_p=1.0, leg=False):
    """--op lmhead: the fused LM-head (tcgen05 GEMM + online log-sum-exp
    epilogue) on hidden [16384, 4096] and W [151936, 4096] bf16, top_p 1.
    --op lmhead_topp: the same at top_p 0.95 (bf16 logits emitted 4096 rows at
    a time and scored by the top-p path)."""
    import entropy_logits_bf16_gb300 as rlk
    import workloads
    stream = torch.cuda.current_stream(dev)
    hidden, w, ids = workloads.lmhead_inputs(LM_T, LM_H, VOCAB, seed=4 + rank, device=dev)
    ids = ids.to(dev).to(torch.int32)
    wsb = rlk.workspace_size(rlk.OP_LMHEAD if top_p == 1.0 else rlk.OP_LMHEAD_TOPP, LM_T, VOCAB,
                             LM_H)
    wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    lp = torch.empty(LM_T, device=dev)

    def lm():
        rlk.lmhead_logprob(hidden, w, ids, TEMPERATURE, top_p, workspace=wsp)

    elapsed_ms, part_ms, clk = timed_steps(args, ws, dev, stream, [lm], barrier)
    if leg:
        peaks, peak_kind = measured_peaks()
        flops = 2.0 * LM_T * LM_H * VOCAB
        achieved = flops / (part_ms[0] / 1e3) / 1e12
        peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0))
        out = {"metric": "tokens/s", "value": whole_job_rate(LM_T, args.steps, ws, elapsed_ms),
               "unit": "tokens/s", "steps": args.steps, "ms_per_step": elapsed_ms / args.steps,
               "config": {"workload": f"fused LM-head: hidden [{LM_T}, {LM_H}] bf16 N(0,1), W_vocab "
                                      f"[{VOCAB}, {LM_H}] bf16 N(0, 0.02^2), temperature "
                                      f"{TEMPERATURE}, top_p 1, uniform ids; logits never stored"},
               "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                            "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_kind,
                            "peak_kind": "bf16 sustained (cuBLAS bf16 GEMM back to back)",
                            "peak_nominal": BF16_NOMINAL_TFLOPS,
                            "frac_of_nominal": achieved / BF16_NOMINAL_TFLOPS,
                            "kernel": "lmhead_kernel + lmhead_combine_kernel",
                            "flops_per_launch": flops, "launch_ms": part_ms[0]},
               "clocks": clk}
        if clk:
            out["roofline"]["sm_mhz_median"] = clk["sm_mhz"]
        if ws == 1 and rank == 0 and not args.no_cpu_baseline:
            import oracle
            rows = 64
            sel = np.linspace(0, LM_T - 1, rows).astype(np.int64)
            hb = workloads.bf16_bits(hidden[torch.from_numpy(sel).to(dev)])
            wb = workloads.bf16_bits(w)
            threads = oracle.default_threads()
            oracle.build()
            t0 = time.perf_counter()
            oracle.lmhead_rows(hb, wb, np.arange(rows), ids.cpu().numpy()[sel], TEMPERATURE, 1.0,
                               threads=threads)
            dt = time.perf_counter() - t0
            out["cpu_baseline"] = {"value": rows / dt, "unit": "tokens/s", "cores": threads,
                                   "kind": "oracle",
                                   "sample": f"{rows} evenly spaced rows, fp64 oracle, {threads} "
                                             f"threads, {dt:.2f} s"}
        del hidden, w
        return out
    host_h = torch.empty(hidden.shape, dtype=hidden.dtype, pin_memory=True).copy_(hidden)
    host_i = torch.empty(ids.shape, dtype=ids.dtype, pin_memory=True).copy_(ids)
    dh, di = torch.empty_like(hidden), torch.empty_like(ids)
    out_h = torch.empty(2 * LM_T, dtype=torch.float32, pin_memory=True)

    def e2e_step():
        dh.copy_(host_h, non_blocking=True)
        di.copy_(host_i, non_blocking=True)
        a, b = rlk.lmhead_logprob(dh, w, di, TEMPERATURE, top_p, workspace=wsp)
        out_h[:LM_T].copy_(a, non_blocking=True)
        out_h[LM_T:].copy_(b, non_blocking=True)

    e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(args.steps, 10))
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / n_e2e, dev)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    flops = 2.0 * LM_T * LM_H * VOCAB
    achieved = flops / (part_ms[0] / 1e3) / 1e12
    # the kernel runs back to back for seconds: the sustained (power-capped) peak
    peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0))
    line = {
        "metric": LM_METRIC if top_p == 1.0 else LM_METRIC.replace("(top_p 1)", f"(top_p {top_p})"),
        "value": whole_job_rate(LM_T, args.steps, ws, elapsed_ms), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"fused LM-head: hidden [{LM_T}, {LM_H}] bf16 N(0,1), W_vocab "
                               f"[{VOCAB}, {LM_H}] bf16 N(0, 0.02^2), temperature {TEMPERATURE}, "
                               f"top_p {top_p}, uniform ids; "
                               + ("logits never stored" if top_p == 1.0 else
                                  "bf16 logits of 4096 rows at a time in the workspace"),
                   "global_batch": LM_T * ws,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "W (1.24 GB) larger than L2; no flush between steps"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "peak_source": peak_kind,
                     "kernel": ("lmhead_kernel + lmhead_combine_kernel" if top_p == 1.0 else
                                "lmhead_kernel (emit) + the top-p logits path per chunk")
                               + " (one rlk_lmhead_logprob call)",
                     "flops_per_launch": flops, "launch_ms": part_ms[0]},
        "e2e": {"value": LM_T * ws / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(hidden.numel() * 2 + ids.numel() * 4),
                "d2h_bytes_per_step": int(out_h.numel() * 4),
                "note": "W_vocab (model state) stays resident; hidden states and ids are copied"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        rows = 256   # about 10 s of fp64 dot products on 16 cores
        sel = np.linspace(0, LM_T - 1, rows).astype(np.int64)
        hb = workloads.bf16_bits(hidden[torch.from_numpy(sel).to(dev)])
        wb = workloads.bf16_bits(w)
        threads = oracle.default_threads()
        oracle.build()
        t0 = time.perf_counter()
        oracle.lmhead_rows(hb, wb, np.arange(rows), ids.cpu().numpy()[sel], TEMPERATURE, top_p,
                           threads=threads)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": rows / dt, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{rows} evenly spaced rows, fp64 oracle, {threads} threads, "
                                          f"{dt:.2f} s"}
    return line


LMB_METRIC = ("tokens/s for the fused LM-head backward (dL/dhidden and dL/dW at top_p 1 by "
              "recompute) at V=151936, H=4096")


def run_lmhead_backward(args, ws, rank, dev, barrier):
    """--op lmhead_backward: rlk_lmhead_logprob_bwd on the LM-head benchmark
    shape (the forward, which saves each row's log-normaliser, runs once before
    the timed region).  Three GEMMs of 2 T V H flops each, all tcgen05: the
    recompute with the gradient epilogue and the two weight-side products."""
    import entropy_logits_bf16_gb300 as rlk
    import workloads
    stream = torch.cuda.current_stream(dev)
    hidden, w, ids = workloads.lmhead_inputs(LM_T, LM_H, VOCAB, seed=4 + rank, device=dev)
    ids = ids.to(dev).to(torch.int32)
    lse = torch.empty(LM_T, device=dev)
    _, ent = rlk.lmhead_logprob(hidden, w, ids, TEMPERATURE, out_lse=lse)
    g = torch.Generator(device="cpu").manual_seed(rank_seed(rank) + 3)
    glp = torch.empty(LM_T).uniform_(-1, 1, generator=g).to(dev)
    gh = torch.empty(LM_T).uniform_(-1, 1, generator=g).to(dev)
    dh = torch.empty((LM_T, LM_H), device=dev)
    dw = torch.empty((VOCAB, LM_H), device=dev)
    wsp = torch.empty(rlk.workspace_size(rlk.OP_LMHEAD_BWD, LM_T, VOCAB, LM_H), dtype=torch.uint8,
                      device=dev)

    def bwd():
        rlk.lmhead_backward(hidden, w, ids, TEMPERATURE, lse, ent, glp, gh, grad_hidden=dh,
                            grad_w=dw, workspace=wsp)

    elapsed_ms, part_ms, clk = timed_steps(args, ws, dev, stream, [bwd], barrier)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    flops = 3 * 2.0 * LM_T * LM_H * VOCAB
    achieved = flops / (part_ms[0] / 1e3) / 1e12
    peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0))
    n_chunks = (LM_T + 4095) // 4096
    return {
        "metric": LMB_METRIC, "value": whole_job_rate(LM_T, args.steps, ws, elapsed_ms),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"fused LM-head backward: hidden [{LM_T}, {LM_H}] bf16 N(0,1), "
                               f"W_vocab [{VOCAB}, {LM_H}] bf16 N(0, 0.02^2), temperature "
                               f"{TEMPERATURE}, top_p 1; dz recomputed 4096 rows at a time",
                   "global_batch": LM_T * ws,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "W (1.24 GB) and dW (2.49 GB) larger than L2; no flush between steps"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "peak_source": peak_kind,
                     "kernel": "lmhead_kernel (gradient epilogue) + two gemm_kernel products per chunk",
                     "flops_per_launch": flops, "launch_ms": part_ms[0]},
        "gpu_launches": 3 * n_chunks * args.steps,
        "clocks": clk,
    }


CAN_METRIC = ("tokens/s for top_p=1 logprob+entropy over the canonical vocabulary partition "
              "(virtual TP 8, padded vocabulary 152576) at V=151936 bf16")


def run_canonical(args, ws, rank, dev, barrier):
    """--op canonical: rlk_logprob_entropy_canonical on the benchmark rows
    (eight virtual shards' partials, then the fixed-order combine)."""
    import entropy_logits_bf16_gb300 as rlk
    stream = torch.cuda.current_stream(dev)
    z, ids = make_workload(dev, seed=rank_seed(rank))

    def call():
        rlk.logprob_entropy_canonical(z, ids, TEMPERATURE)

    elapsed_ms, part_ms, clk = timed_steps(args, ws, dev, stream, [call], barrier)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    alg = T_ROWS * (VOCAB * 2 + 4 + 8) + 2 * T_ROWS * rlk.CANONICAL_TP * 32   # logits, ids, outputs, partials
    achieved = alg / (part_ms[0] / 1e3) / 1e9
    return {
        "metric": CAN_METRIC, "value": whole_job_rate(T_ROWS, args.steps, ws, elapsed_ms),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD.replace("top_p 0.95", "top_p 1"), "T": T_ROWS, "V": VOCAB,
                   "virtual_tp": rlk.CANONICAL_TP, "padded_vocab": rlk.CANONICAL_VOCAB,
                   "global_batch": T_ROWS * ws,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": profiled_traffic(os.path.join(CSRC, "vocab_parallel.cu"),
                                                 os.path.join(PROFILES, "shard_partial_kernel_qwen_T4096.txt")),
                     "peak_source": peak_kind,
                     "kernel": "shard_partial_kernel + shard_combine_kernel (traffic: the partial kernel)",
                     "algorithmic_bytes_per_launch": alg, "launch_ms": part_ms[0]},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }


CAN_TOPP_METRIC = ("tokens/s for top-p logprob+entropy over the canonical vocabulary partition "
                   "(virtual TP 8, padded vocabulary 152576) at V=151936 bf16")


def run_canonical_topp(args, ws, rank, dev, barrier):
    """--op canonical_topp: rlk_logprob_entropy_canonical_topp on the benchmark
    rows at top_p 0.95 -- the eight virtual shards' partials, their window
    counts per bf16 value (a second read of each shard's logits, after the
    partials fix the row's max and Z), then the fixed-order combine."""
    import entropy_logits_bf16_gb300 as rlk
    stream = torch.cuda.current_stream(dev)
    z, ids = make_workload(dev, seed=rank_seed(rank))

    def call():
        rlk.logprob_entropy_canonical_topp(z, ids, TEMPERATURE, TOP_P)

    elapsed_ms, part_ms, clk = timed_steps(args, ws, dev, stream, [call], barrier)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    n = rlk.CANONICAL_TP
    # per row: the logits read twice (partials, then the window counts), the id,
    # the outputs (logprob, entropy, k*), the partials and the window counts
    # each written once and read once
    alg = T_ROWS * (2 * VOCAB * 2 + 4 + 12 + 2 * n * 32 + 2 * n * 8224)
    achieved = alg / (part_ms[0] / 1e3) / 1e9
    return {
        "metric": CAN_TOPP_METRIC, "value": whole_job_rate(T_ROWS, args.steps, ws, elapsed_ms),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_ROWS, "V": VOCAB, "virtual_tp": n,
                   "padded_vocab": rlk.CANONICAL_VOCAB, "global_batch": T_ROWS * ws,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": None, "peak_source": peak_kind,
                     "kernel": "shard_partial_kernel + shard_window_kernel + shard_combine_topp_kernel "
                               "(one rlk_logprob_entropy_canonical_topp call)",
                     "algorithmic_bytes_per_launch": alg, "launch_ms": part_ms[0]},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
    }


SMP_METRIC = ("tokens/s for deterministic top-p sampling (inverse CDF over the retained set "
              "in ranking order) at V=151936 bf16")


def run_sample(args, ws, rank, dev, barrier):
    """--op sample: rlk_sample_top_p on the benchmark rows (their retained sets
    from one forward before the timed region), one uniform per row."""
    import entropy_logits_bf16_gb300 as rlk
    stream = torch.cuda.current_stream(dev)
    z, ids = make_workload(dev, seed=rank_seed(rank))
    state = rlk.new_row_state(T_ROWS, dev)
    rlk.logprob_entropy(z, ids, TEMPERATURE, TOP_P, row_state=state)
    g = torch.Generator(device="cpu").manual_seed(rank_seed(rank) + 4)
    u = torch.rand(T_ROWS, generator=g).to(dev)

    def call():
        rlk.sample_top_p(z, TEMPERATURE, TOP_P, u, row_state=state)

    elapsed_ms, part_ms, clk = timed_steps(args, ws, dev, stream, [call], barrier)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    alg = T_ROWS * (VOCAB * 2 + 32 + 4 + 4)   # one read of the row, the state, u, the id
    achieved = alg / (part_ms[0] / 1e3) / 1e9
    return {
        "metric": SMP_METRIC, "value": whole_job_rate(T_ROWS, args.steps, ws, elapsed_ms),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD + "; one uniform per row", "T": T_ROWS, "V": VOCAB,
                   "global_batch": T_ROWS * ws,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": profiled_traffic(os.path.join(CSRC, "sampler.cu"),
                                                 os.path.join(PROFILES, "sample_kernel_qwen_T4096.txt")),
                     "peak_source": peak_kind,
                     "kernel": "sample_kernel (one rlk_sample_top_p call: each row read once, "
                               "tie groups ranked from the member list)",
                     "algorithmic_bytes_per_launch": alg, "launch_ms": part_ms[0]},
        "gpu_launches": args.steps,
        "clocks": clk,
    }


SUP_METRIC = ("tokens/s for supplied-support logprob+entropy (the top-p retained set given as "
              "CSR) at V=151936 bf16")


def make_supports(z, top_p, temperature, chunk=256):
    """Each row's top-p retained set (sorted by logit, lower id first on
    ties), as CSR int64 offsets [T+1] and int32 ids, built with library sorts on
    the device -- benchmark inputs, not the product path."""
    offs, lists = [0], []
    for r0 in range(0, z.shape[0], chunk):
        x = z[r0:r0 + chunk].float() / temperature
        order = torch.argsort(x, dim=1, descending=True, stable=True)   # ties: lower id first
        p = torch.softmax(x, dim=1).gather(1, order)
        c = torch.cumsum(p, dim=1)
        k = ((c < top_p).sum(dim=1) + 1).clamp(max=z.shape[1]).cpu()
        for i in range(x.shape[0]):
            lists.append(order[i, :int(k[i])].to(torch.int32))
            offs.append(offs[-1] + int(k[i]))
    return (torch.tensor(offs, dtype=torch.int64, device=z.device), torch.cat(lists))


SUP_BWD_METRIC = ("tokens/s for the supplied-support backward (gradient of logprob and entropy "
                  "over the top-p retained set given as CSR) at V=151936 bf16")


def run_support(args, ws, rank, dev, barrier, backward=False):
    """--op support / support_backward: rlk_logprob_entropy_support, or its
    backward, on the benchmark rows, each given its own top-p retained set."""
    import entropy_logits_bf16_gb300 as rlk
    stream = torch.cuda.current_stream(dev)
    z, ids = make_workload(dev, seed=rank_seed(rank))
    off, sup = make_supports(z, TOP_P, TEMPERATURE)
    lp = torch.empty(T_ROWS, device=dev)
    ent = torch.empty(T_ROWS, device=dev)
    g = torch.Generator(device="cpu").manual_seed(rank_seed(rank) + 1)
    glp = torch.empty(T_ROWS).uniform_(-1, 1, generator=g).to(dev)
    gh = torch.empty(T_ROWS).uniform_(-1, 1, generator=g).to(dev)
    grad = torch.empty(sup.shape, device=dev)

    def call():
        rlk.logprob_entropy_support(z, ids, TEMPERATURE, off, sup, out_logprob=lp, out_entropy=ent)

    def bcall():
        rlk.logprob_entropy_support_backward(z, ids, TEMPERATURE, off, sup, glp, gh, out=grad)

    elapsed_ms, part_ms, clk = timed_steps(args, ws, dev, stream, [bcall if backward else call],
                                           barrier)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    nnz = int(sup.numel())
    if backward:
        # ids + logits read once (the second pass hits L2), gradients written,
        # offsets, id and the two incoming gradients per row
        alg = nnz * (4 + 2 + 4) + T_ROWS * (8 + 4 + 8)
        sectors = nnz * 32 + nnz * 8 + T_ROWS * 20
        kernel = "support_backward_kernel (one rlk_logprob_entropy_support_backward call)"
    else:
        alg = nnz * (4 + 2) + T_ROWS * (8 + 4 + 8)   # listed ids + their logits, offsets, id, outputs
        sectors = nnz * 32 + nnz * 4 + T_ROWS * 20    # each listed logit costs one 32-byte sector
        kernel = "support_kernel (one rlk_logprob_entropy_support call)"
    achieved = alg / (part_ms[0] / 1e3) / 1e9
    return {
        "metric": SUP_BWD_METRIC if backward else SUP_METRIC,
        "value": whole_job_rate(T_ROWS, args.steps, ws, elapsed_ms),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD + "; each row's top-p retained set supplied as CSR",
                   "T": T_ROWS, "V": VOCAB, "listed_tokens": nnz,
                   "mean_listed_per_row": nnz / T_ROWS, "global_batch": T_ROWS * ws,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": profiled_traffic(
                         os.path.join(CSRC, "support.cu"),
                         os.path.join(PROFILES, ("support_backward_kernel_qwen_T4096.txt" if backward
                                                 else "support_kernel_qwen_T4096.txt"))),
                     "peak_source": peak_kind,
                     "kernel": kernel,
                     "algorithmic_bytes_per_launch": alg,
                     "sector_bytes_per_launch": sectors,
                     "sector_frac": sectors / (part_ms[0] / 1e3) / 1e9 / peaks["hbm_gbs"],
                     "launch_ms": part_ms[0]},
        "gpu_launches": args.steps,
        "clocks": clk,
    }


BWD_METRIC = ("tokens/s for the dense top-p backward (dL/dlogits over V=151936, bf16 logits and "
              "gradients, retained sets from the forward)")


def run_backward(args, ws, rank, dev, barrier):
    """--op backward: rlk_logprob_entropy_bwd on the benchmark rows (their row
    states saved by one forward before the timed region), bf16 gradients."""
    import entropy_logits_bf16_gb300 as rlk
    stream = torch.cuda.current_stream(dev)
    z, ids = make_workload(dev, seed=rank_seed(rank))
    state = rlk.new_row_state(T_ROWS, dev)
    rlk.logprob_entropy(z, ids, TEMPERATURE, TOP_P, row_state=state)
    g = torch.Generator(device="cpu").manual_seed(rank_seed(rank) + 2)
    glp = torch.empty(T_ROWS).uniform_(-1, 1, generator=g).to(dev)
    gh = torch.empty(T_ROWS).uniform_(-1, 1, generator=g).to(dev)
    grad = torch.empty((T_ROWS, VOCAB), device=dev, dtype=torch.bfloat16)

    def call():
        rlk.logprob_entropy_backward(z, ids, TEMPERATURE, state, glp, gh, out=grad)

    elapsed_ms, part_ms, clk = timed_steps(args, ws, dev, stream, [call], barrier)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    # logits read + gradients written, plus per row the state, id and two gradients
    alg = T_ROWS * VOCAB * (2 + 2) + T_ROWS * (32 + 4 + 8)
    achieved = alg / (part_ms[0] / 1e3) / 1e9
    return {
        "metric": BWD_METRIC, "value": whole_job_rate(T_ROWS, args.steps, ws, elapsed_ms),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD + "; gradients of logprob and entropy, bf16 out",
                   "T": T_ROWS, "V": VOCAB, "global_batch": T_ROWS * ws,
                   "l2": "inputs larger than L2 (1.24 GB read + 1.24 GB written per step)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": profiled_traffic(BWD_SRC, BWD_PROFILE), "peak_source": peak_kind,
                     "kernel": "lpe_backward_pipe_kernel (one rlk_logprob_entropy_bwd call)",
                     "algorithmic_bytes_per_launch": alg, "launch_ms": part_ms[0]},
        "gpu_launches": args.steps,
        "clocks": clk,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--op", default="logits", choices=["logits", "lmhead", "lmhead_backward", "support",
                                                       "support_backward", "backward",
                                                       "lmhead_topp", "canonical", "canonical_topp", "sample",
                                                       "zipf"],
                    help="logits: the benchmark (logprob/entropy + loss); lmhead: the fused "
                         "LM-head; support: the supplied-support scorer; support_backward: its "
                         "gradient; backward: the dense top-p gradient; lmhead_backward: the "
                         "LM-head gradients")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lm-rows", type=int, default=None,
                    help="rows of the LM-head workloads (default 16384; smaller for a profile)")
    ap.add_argument("--zipf-rows", type=int, default=None,
                    help="rows of the long-response workloads (default 55296; smaller for a profile)")
    ap.add_argument("--no-legs", action="store_true",
                    help="logits only: skip the long-response, packed GRPO and LM-head legs")
    args = ap.parse_args()
    global LM_T, ZIPF_ROWS
    if args.lm_rows:
        LM_T = int(args.lm_rows)
    if args.zipf_rows:
        ZIPF_ROWS = int(args.zipf_rows)
    if args.impl == "reference":
        run_reference(args)
        return
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import entropy_logits_bf16_gb300 as rlk
    rlk.build()
    rlk.load()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    run = {"logits": run_logits, "lmhead": run_lmhead, "support": run_support,
           "support_backward": lambda *a: run_support(*a, backward=True),
           "backward": run_backward, "lmhead_backward": run_lmhead_backward,
           "lmhead_topp": lambda *a: run_lmhead(*a, top_p=TOP_P),
           "canonical": run_canonical, "canonical_topp": run_canonical_topp,
           "sample": run_sample, "zipf": run_zipf}[args.op]
    line = run(args, ws, rank, dev, barrier)
    if line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
