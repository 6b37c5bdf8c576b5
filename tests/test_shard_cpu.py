"""Multi-process host logic of the bench (replicas, weak scaling) on CPU with
the gloo backend, world size 2, and the shard identities of the op on the
oracle: a column split of a packed layer gives the matching columns of y
exactly, and a row split (at group / segment boundaries) sums to y."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

import oracle as O
import synth
from helpers import exl2_case, gptq_case, oracle_W_exl2, oracle_W_gptq


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local = [10.0 + 5.0 * rank, 20.0 - rank]  # rank 1 is slower on the first, faster on the second
        out[rank] = bench.max_over_ranks(local, world)
    finally:
        dist.destroy_process_group()


def test_bench_times_are_the_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp

    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        got = dict(out)
    assert got[0] == got[1] == [15.0, 20.0]


def test_job_throughput_counts_every_replica():
    import bench
    # two replicas each streaming 1 GB per step, 10 steps in 100 ms -> 200 GB/s
    assert bench.job_throughput(10 ** 9, 10, 100.0, 2) == pytest.approx(200.0)
    assert bench.job_throughput(10 ** 9, 10, 100.0, 1) == pytest.approx(100.0)


def test_shard_reductions_gptq():
    # a column split at multiples of 8 keeps whole zero words; a row split at
    # group boundaries keeps whole groups
    g = gptq_case(512, 64, 128, act_order=False, seed=21)
    W = O.float64_from_fp16_bits(oracle_W_gptq(g))
    x = synth.activations(3, 512, seed=21).astype(np.float64)
    y = x @ W
    cols = [slice(0, 24), slice(24, 64)]
    assert np.array_equal(np.concatenate([x @ W[:, c] for c in cols], axis=1), y)
    rows = [slice(0, 256), slice(256, 512)]
    parts = sum(x[:, r] @ W[r, :] for r in rows)
    assert np.allclose(parts, y, rtol=1e-12, atol=1e-12)


def test_shard_reductions_exl2():
    # the row split is at a segment boundary (multiple of 32 stored rows)
    e = exl2_case(256, 40, bpw=4.0, permute=False, seed=22)
    W = O.float64_from_fp16_bits(oracle_W_exl2(e))
    x = synth.activations(2, 256, seed=22).astype(np.float64)
    y = x @ W
    assert np.array_equal(np.concatenate([x @ W[:, :16], x @ W[:, 16:]], axis=1), y)
    assert np.allclose(x[:, :96] @ W[:96] + x[:, 96:] @ W[96:], y, rtol=1e-12, atol=1e-12)


def test_reference_arm_prints_the_contract_line():
    # the --impl reference arm (the CPU oracle) runs on any host: one JSON line
    # with the fields the harness reads, its e2e moving no host-device bytes
    import json
    import subprocess
    import sys
    from pathlib import Path

    root = Path(__file__).resolve().parents[1]
    r = subprocess.run([sys.executable, str(root / "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=root,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 1 and line["warmup"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "decode_stream_70b_exl2_4p0bpw"
