"""Host-side logic of bench.py (no GPU): the algorithmic work it divides by,
and the max-over-ranks reduction of the multi-process path on gloo ranks."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402


@pytest.mark.parametrize("lengths", [[8192], [300], [1, 64, 65, 66, 129, 5000], [0, 3]])
@pytest.mark.parametrize("kind", ["global", "local"])
def test_admitted_pairs_match_oracle_counts(lengths, kind):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    counts = oracle.key_counts(cu, oracle.KINDS[kind]["half_window"])
    assert bench.admitted_pairs(lengths, kind) == int(counts.astype(np.int64).sum())


def test_work_of_the_headline_workload():
    """The teardown's pair counts at n = 8192 times 256 flop per pair per
    head: 206.16 GFLOP (global) and 3.234 GFLOP (local); 50.33 MB."""
    g = bench.work([8192], "global")
    l = bench.work([8192], "local")
    assert g["flops"] == 67108864 * 256 * 12
    assert l["flops"] == 1052608 * 256 * 12
    assert g["bytes"] == l["bytes"] == 8192 * 6144


def test_work_of_the_22_layer_schedule():
    """32 sequences of 8192 tokens, layer i global iff i % 3 == 0: 8 global
    layers of 6.597 TFLOP and 14 local ones of 0.1035 TFLOP, 54.23 TFLOP in
    all; 1.611 GB per layer (qkv read once, out written once)."""
    from encoder_only_transformer_gb300 import workloads as W
    lengths = [8192] * 32
    kinds = [W.layer_kind(i) for i in range(22)]
    assert kinds.count("global") == 8 and kinds.count("local") == 14
    assert kinds[0] == "global" and kinds[1] == kinds[2] == "local"
    g, l = bench.work(lengths, "global"), bench.work(lengths, "local")
    assert g["flops"] == 32 * 8192 * 8192 * 256 * 12
    assert l["flops"] == 32 * (129 * 8192 - 64 * 65) * 256 * 12
    assert g["bytes"] == l["bytes"] == 32 * 8192 * 6144
    total = sum(bench.work(lengths, k)["flops"] for k in kinds)
    assert abs(total / 1e12 - 54.2252) < 1e-3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    worst = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    q.put((rank, worst, bench.whole_job_tokens_per_s(8192, world, worst)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    """Two gloo ranks: the timed region is the slowest rank's, and the value
    is the tokens of all ranks over that time (weak scaling)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert all(r[1] == 15.0 for r in res)
    assert all(abs(r[2] - 2 * 8192 / 0.015) < 1e-6 for r in res)


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the keys the benchmark contract asks of that arm."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--cpu-budget", "0.25"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["metric"] == bench.METRIC and rec["unit"] == bench.UNIT
    assert rec["higher_is_better"] is True and rec["steps"] == 1 and rec["warmup"] == 3
    assert rec["value"] > 0 and rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"] == {"value": rec["value"], "unit": rec["unit"],
                          "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
