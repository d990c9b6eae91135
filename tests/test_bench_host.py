"""Host-side logic of bench.py: work counts, the reference arm, and the multi-rank
timing reduction over gloo (world size 2, CPU)."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from efficient_transformer_gb300 import inputs as gen


def test_path_counts_long_context_gqa():
    w = gen.WORKLOADS["gqa_causal_b1_hq32_hkv8_n65536_d128_bf16"]
    assert bench.path_bytes(w) == 3328 * 2**20
    assert abs(bench.path_flops(w) - 7.2155e11) / 7.2155e11 < 1e-3


def test_path_counts_bidirectional():
    w = gen.WORKLOADS["bidir_b2_h8_n2048_d64_bf16_elu1"]
    # fwd 2|q| + 2|kv| + bwd 3|q| + 4|kv|, |q| = |kv| = 4 MiB
    assert bench.path_bytes(w) == 11 * 4 * 2**20
    assert bench.path_flops(w) == 14 * 2 * 8 * 2048 * 64 * 64


def test_reference_arm_prints_one_line(capsys):
    rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3",
                     "--workload", "causal_b1_h2_n256_d32_f32"])
    assert rc == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "causal_b1_h2_n256_d32_f32"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + rank, world)     # rank 1 is the slow one
        bench.barrier(world)
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 11.0, 1: 11.0}


def test_config_names_workload_and_replicas():
    w = gen.WORKLOADS[gen.BENCH_WORKLOAD]
    c = bench.config_of(w, 2)
    assert c["workload"] == gen.BENCH_WORKLOAD and c["global_batch"] == 2 * w.B
    assert c["parallelism"] == "replicas2"
