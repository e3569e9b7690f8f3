"""The multi-process (N > 1) host logic of bench.py, on CPU with the gloo
backend and world size 2.  Rows are independent, so N GPUs run N replicas of
the hot path with no collective on the data path; what crosses ranks is the
timing: the job's time is the slowest rank's, and the whole-job throughput
counts every rank's rows over that time.  Each replica draws its own batch.

The vocabulary-parallel (canonical partition) path has one exchange: each
rank's shard partials are gathered in rank order; the plan of which virtual
shards a rank holds and that gather are tested here too.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        env = bench.dist_env()
        cpu = torch.device("cpu")
        t_max = bench.reduce_max(10.0 + 3.0 * rank, cpu)      # rank 1 is the slow one
        rate = bench.whole_job_rate(4096, 100, ws, t_max)
        seed = bench.rank_seed(rank)
        q.put((rank, env, t_max, rate, seed))
    finally:
        dist.destroy_process_group()


def test_replica_timing_and_seeds_over_two_gloo_ranks():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, t_max, rate, _ in res:
        assert env == (ws, rank, rank)
        assert t_max == pytest.approx(13.0)                    # max over ranks, on every rank
        assert rate == pytest.approx(4096 * 100 * ws / 13.0e-3)
    assert res[0][4] != res[1][4]                              # each replica its own batch


def test_single_process_helpers():
    import bench
    assert bench.reduce_max(7.5, torch.device("cpu")) == 7.5   # no process group: the value itself
    assert bench.whole_job_rate(4096, 10, 1, 5.0) == pytest.approx(4096 * 10 / 5.0e-3)


# ------------------------------------------------ canonical vocabulary partition
def test_canonical_plan_covers_every_shard_once():
    import entropy_logits_bf16_gb300 as rlk
    for tp in (1, 2, 4, 8):
        seen = []
        for r in range(tp):
            s0, n, c0, w = rlk.canonical_plan(tp, r)
            assert w == rlk.CANONICAL_VOCAB // rlk.CANONICAL_TP and c0 == s0 * w
            seen += list(range(s0, s0 + n))
        assert seen == list(range(rlk.CANONICAL_TP))          # adjacent, in rank order
    with pytest.raises(ValueError):
        rlk.canonical_plan(3, 0)


def _gather_worker(rank, ws, port, q):
    import torch.distributed as dist
    import entropy_logits_bf16_gb300 as rlk
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        s0, n, _, _ = rlk.canonical_plan(ws, rank)
        T = 5
        # each rank's partials carry their global shard index, so the gathered
        # order can be read back
        local = torch.arange(s0, s0 + n, dtype=torch.float32).view(n, 1, 1).expand(n, T, 8)
        full = rlk.gather_shard_partials(local.contiguous())
        # the second exchange at top_p < 1: each shard's window counts (bytes)
        cnt = torch.zeros((n, T, rlk.SHARD_COUNTS_BYTES), dtype=torch.uint8)
        cnt[:, :, 0] = torch.arange(s0, s0 + n, dtype=torch.uint8).view(n, 1)
        cnt[:, :, -1] = torch.arange(T, dtype=torch.uint8).view(1, T)
        fullc = rlk.gather_shard_partials(cnt)
        q.put((rank, full[:, 0, 0].tolist(), tuple(full.shape), fullc[:, 0, 0].tolist(),
               fullc[:, :, -1].tolist(), tuple(fullc.shape)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws", [2, 4])
def test_gather_shard_partials_in_canonical_order_over_gloo_ranks(ws):
    """The vocabulary-parallel exchanges: every rank ends with all eight shards'
    partials -- and, at top_p < 1, their window counts -- in shard order,
    whatever rank computed them (TP 2 and TP 4)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, order, shape, corder, crow, cshape in res:
        assert order == [float(s) for s in range(8)]
        assert shape == (8, 5, 8)
        assert corder == list(range(8)) and cshape == (8, 5, 8224)
        assert crow == [list(range(5))] * 8                    # rows stay in place


# ------------------------------------------------ the reference arm (the oracle on host cores)
def _bench(args, env=None):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    e = dict(os.environ)
    e.update(env or {})
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], cwd=root, env=e,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_prints_the_contract_line():
    import bench
    (line,) = _bench(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 1 and line["warmup"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    assert _bench(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"],
                  env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_peaks_file_and_fallback(tmp_path, monkeypatch):
    import json
    import bench
    peaks, kind = bench.measured_peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and peaks["hbm_gbs"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))          # no file there
    peaks, kind = bench.measured_peaks()
    assert kind == "fallback"
    assert peaks == {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1.0, "bf16_tflops": 2.0}))
    assert bench.measured_peaks() == ({"hbm_gbs": 1.0, "bf16_tflops": 2.0}, "measured")
