"""Host-side logic of bench.py: the replica aggregation across ranks (two gloo
ranks on CPU), and the step roofline arithmetic against the pages' shapes."""
import os
import socket

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
import la_inputs as I


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    tok, sec = bench.aggregate(100.0 * (rank + 1), 1.0 + rank)
    bench.barrier()
    q.put((rank, tok, sec))
    dist.destroy_process_group()


def test_replica_aggregation_gloo_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(60)
    res = sorted(q.get(timeout=10) for _ in range(2))
    # tokens sum over replicas, time is the slowest rank's
    assert res == [(0, 300.0, 2.0), (1, 300.0, 2.0)]


def test_single_process_aggregation_is_identity():
    assert bench.aggregate(7.0, 0.5) == (7.0, 0.5)


@pytest.mark.parametrize("name,T", [("7b", 121), ("13b", 81), ("34b", 57)])
def test_step_shapes_and_roofline_inputs(name, T):
    cfg = I.MODELS[name]
    W, N, G = I.LOOKAHEAD[name]
    assert 1 + (W + G) * (N - 1) == T
    by, fl = bench.step_model(cfg, T, 512)
    # weights dominate the bytes; FLOPs ~ 2 * params * T
    assert by > cfg.streamed_params() * 2
    assert fl > 2 * cfg.streamed_params() * T
    # arithmetic intensity is below the GB300 ridge (~290 FLOP/B): HBM bound
    assert fl / by < 290


def test_lookahead_overrides_and_sweep_shapes():
    """--wng / --preseed override the workload's settings; every sweep point
    fits the 128-row step and W = 0 points are the prompt-lookup mode (a
    prompt-seeded pool, no window)."""
    import argparse
    a = argparse.Namespace(workload="7b", wng="", preseed="auto")
    assert bench.lookahead_of(a) == (15, 5, 15, False)
    a = argparse.Namespace(workload="34b", wng="", preseed="auto")
    assert bench.lookahead_of(a) == (7, 5, 7, True)
    a = argparse.Namespace(workload="7b", wng="0,4,6", preseed="on")
    assert bench.lookahead_of(a) == (0, 4, 6, True)
    assert bench.SWEEP[0] == (0, 2, 0, False, False)
    assert any(d for *_, d in bench.SWEEP) and (15, 5, 15, False, True) in bench.SWEEP
    for W, N, G, pre, diag in bench.SWEEP:
        assert 1 + (W + G) * (N - 1) <= 128 and N >= 2
        if W == 0 and G > 0:
            assert pre


def test_batch_sweep_points_fit_one_pass():
    """Every point of bench.py --batch-sweep fits one 128-row forward pass,
    greedy runs from 1 to 128 sequences, and the workload's own lookahead
    setting is a batch-1 point."""
    import bench
    for W, N, G, b in bench.BATCH_SWEEP:
        assert b >= 1 and b * (1 + (W + G) * (N - 1)) <= 128, (W, N, G, b)
    greedy = sorted(b for W, N, G, b in bench.BATCH_SWEEP if W == 0 and G == 0)
    assert greedy[0] == 1 and greedy[-1] == 128
    assert (15, 5, 15, 1) in bench.BATCH_SWEEP
    assert bench.batch_points(128) == [(0, 2, 0, 128)] and bench.batch_points() == bench.BATCH_SWEEP
    assert bench.batch_points(2) == [(0, 2, 0, 2), (7, 5, 7, 2)] and bench.batch_points(7) == []


def test_attention_choice_of_the_benchmark():
    """--attn auto takes the tcgen05 attention where the library allows it
    (every step row within 31 positions of P, max_seq <= 4096): the 7B, 13B
    and 34B settings and greedy, not a 31-column window."""
    import bench
    for wl in ("7b", "13b", "34b"):
        W, N, G = bench.I.LOOKAHEAD[wl]
        assert bench.attn_tc_applies(W, N, 2600)
    assert bench.attn_tc_applies(0, 2, 800)
    assert not bench.attn_tc_applies(31, 3, 800)      # rows up to 32 positions past P
    assert not bench.attn_tc_applies(15, 5, 4097)


def test_reference_arm_line_on_the_tiny_workload():
    """bench.py --impl reference (the CPU oracle, no GPU) prints one JSON line
    with the benchmark contract's keys: the oracle's own tokens/s on the
    metric, a cpu_baseline describing the run and an e2e equal to the value
    with no host-device copies."""
    import json
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
