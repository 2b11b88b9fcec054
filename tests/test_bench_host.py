"""Host-side logic of bench.py without a GPU: clock-log parsing, the
max-over-ranks reduction of step times across two gloo ranks on CPU, and
the reference arm's JSON line (it times the oracle on the host cores)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

CSV = """0, 1965, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
0, 1950, 2070, 1010.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active
0, 1980, 2070, 990.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
"""


def test_parse_clocks():
    c = bench.parse_clocks(CSV)
    assert c["sm_mhz"] == 1965.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clocks("")["sm_mhz"] is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        t = bench.max_over_ranks(1.5 + rank, ws)
        bench.barrier(ws)
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e")


def _bench(args, env_extra=None):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **(env_extra or {}))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], cwd=root, env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_line():
    """The reference arm times the oracle on the host cores (no GPU needed) and
    prints one line with the contract's keys on rank 0."""
    (line,) = _bench(["--impl", "reference", "--steps", "2", "--warmup", "0", "--ref-step-s", "0.2"])
    missing = [k for k in REQUIRED if k not in line]
    assert not missing, missing
    assert line["impl"] == "reference" and line["value"] > 0 and line["ms_per_step"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["single_core"]["value"] > 0
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "gauss_n70000_d64"


def test_reference_arm_other_ranks_print_nothing():
    lines = _bench(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                   {"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert lines == []
