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


def test_headline_step_bytes():
    # the 36-layer stack at widths 8, 12, 16: packed tiles of the layer set
    # (44,302,336 bytes) per layer and width, plus bf16 activation rows
    pk = sum((-(-N // 128)) * (-(-K // 128)) * 4096 for _, K, N in inputs.LARGE_PROJ)
    assert pk == 44_302_336
    act_k = sum(K for _, K, _ in inputs.LARGE_PROJ)
    want = sum(36 * (pk + M * act_k * 2) for M in (8, 12, 16))
    assert bench.headline_step_bytes() == want
    # 36 layer sets of packed weights = the 1.595 GB stack
    assert 36 * pk == 1_594_884_096


def test_layer_set_bytes():
    pk = sum((N // 128) * (K // 128) * 4096 for _, K, N in inputs.BITNET2B_PROJ)
    assert pk == 17_367_040
    for M in (1, 2, 4, 8, 16):
        assert bench.layer_set_bytes(inputs.BITNET2B_PROJ, M) == pk + M * 2 * (6 * 2560 + 6912)


def test_oracle_samples_cycle_the_workloads():
    seen = set()
    for i in range(21):
        T, w, x, is_bf16 = bench._oracle_sample("4", i)
        assert is_bf16 and x.shape[1] == T.shape[1] and x.shape[0] in (8, 12, 16)
        seen.add((x.shape[0], T.shape))
    assert len(seen) == 3 * 4  # widths x the layer set's four distinct (N, K) shapes
    T, w, x, is_bf16 = bench._oracle_sample("5", 3)  # sparsity 0, the draft group
    assert not is_bf16 and x.shape == (12, 2560) and T.shape == (2560, 2560)


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
