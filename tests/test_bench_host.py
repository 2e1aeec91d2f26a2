"""Host logic of bench.py on CPU: byte accounting, the max-over-ranks timing
reduction with two gloo ranks, and the reference (oracle) arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from ternary_w2a8_linear_gb300 import inputs  # noqa: E402


def test_step_bytes():
    pk = 0
    act = 0
    for M in (1, 2, 4, 8):
        for _, K, N in inputs.BITNET2B_PROJ:
            pk += (N // 128) * (K // 128) * 4096
            act += M * K * 2
    assert bench.step_bytes() == pk + act
    # 17.37 MB of packed weights per layer set, four widths per step
    assert pk == 4 * 17_367_040


def test_ternarize_bytes():
    # fp32 weights of the seven projections once (69.47 M entries) plus their
    # packed form (17,367,040 bytes of tiles and seven 16-byte trailers)
    assert bench.ternarize_bytes() == 4 * 69_468_160 + 17_367_040 + 7 * 16 == 295_239_792


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), BITMTP_DIST_BACKEND="gloo")
    r, w = bench.dist_init()
    v = bench.dist_max(1.5 + rank, w)
    bench.dist_barrier(w)
    q.put((r, w, v))
    dist.destroy_process_group()


def test_dist_max_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 2.5), (1, 2, 2.5)]


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "1"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "config", "cpu_baseline", "e2e"):
        assert k in line
    assert line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
