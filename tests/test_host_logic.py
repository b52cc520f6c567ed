"""Host logic of the benchmark and the library, no GPU: the replica
aggregation bench.py uses for N > 1 (world-size-2 gloo process group on the
CPU), algorithmic byte counts, workspace sizes, the input generators, and the
reference arm's JSON line (the oracle timed on the host)."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from nf4_weight_quantized_gb300 import synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank: int, world: int, port: int, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        secs = 1.0 + 0.5 * rank  # rank 1 is the slow replica
        m = bench.reduce_max(dist, secs)
        q.put((rank, m, bench.replica_value(world, 12_719_616, 100, m)))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, value in got:
        assert m == 1.5  # both ranks see the max
        assert value == pytest.approx(2 * 12_719_616 * 100 / 1.5 / 1e9)


def test_reduce_max_without_a_process_group():
    assert bench.reduce_max(None, 3.25) == 3.25
    assert bench.replica_value(1, 10**9, 2, 2.0) == 1.0


def test_algorithmic_bytes():
    # codes K/2 + scales K/16 per row
    assert bench.bytes_of("residual", 2048, 11008)["total"] == 2048 * 11008 * 9 // 16 + 11008 * 2 + 2048 * 8
    assert bench.bytes_of("swiglu", 11008, 2048)["weight"] == 2 * 11008 * 2048 * 9 // 16
    assert bench.bytes_of("glu", 11008, 2048) == bench.bytes_of("swiglu", 11008, 2048)
    assert bench.bytes_of("argmax", 151936, 2048)["total"] == 151936 * 2048 * 9 // 16 + 4096 + 151936 * 4 + 8
    assert bench.bytes_of("chunk", 13824, 5120, 32)["total"] == 13824 * 5120 * 9 // 16 + 32 * 5120 * 2 + 32 * 13824 * 4
    qkv = bench.bytes_of("qkv", 2048, 2048, 1, 256)
    assert qkv["weight"] == 2560 * 2048 * 9 // 16 and qkv["total"] == qkv["weight"] + 4096 + 2560 * 8
    e = bench.bytes_of("embed", 151936, 2048, 4096)
    assert e["weight"] == 4096 * 1152 and e["total"] == 4096 * 1152 + 4096 * 8 + 4096 * 2048 * 2
    # RMSNorm: fp32 rows in, bf16 gain, bf16 rows out
    assert bench.bytes_of("rmsnorm", 32, 5120, 32)["total"] == 32 * 5120 * 6 + 5120 * 2


def test_every_reported_workload_is_defined():
    for name in bench.WORKLOADS:
        w = synth.WORKLOADS[name]
        d = synth.workload_inputs(w, M=min(w.M, 4)) if w.kind != "rmsnorm" else synth.workload_inputs(w)
        assert d
    r = synth.workload_inputs(synth.WORKLOADS["rmsnorm_chunk14b"])
    assert r["x"].shape == (32, 5120) and r["x"].dtype == np.float32 and r["w"].dtype == np.uint16


def test_all_core_oracle_worker_covers_its_rows():
    # one share of the all-core CPU baseline: the oracle on rows [r0, r1)
    import oracle

    codes, scales = oracle.quantize(synth.weights(90, 0, 64, 256))
    x = synth.normal_bf16(90, 1, 256)
    r = synth.normal_f32(90, 2, 64)
    n, secs = bench._oracle_rows_worker((codes, scales, x, r, 16, 48, 0.01))
    assert n >= 1 and secs > 0


def test_workload_inputs_are_seeded():
    w = synth.WORKLOADS["qkv3b"]
    a, b = synth.workload_inputs(w), synth.workload_inputs(w)
    assert set(a) == {"W", "Wk", "Wv", "x", "bq", "bk", "bv"}
    assert all(np.array_equal(a[k], b[k]) for k in a)
    # the interleaved gate/up workload holds the two-matrix SwiGLU weights
    g, sw = synth.workload_inputs(synth.WORKLOADS["glu3b"], M=6), synth.workload_inputs(synth.WORKLOADS["swiglu"], M=6)
    assert g["W"].shape == (12, 2048) and np.array_equal(g["x"], sw["x"])
    assert np.array_equal(g["W"][0::2], sw["W"]) and np.array_equal(g["W"][1::2], sw["Wu"])
    ids = synth.token_ids(6, 1, 4096, 151936)
    assert ids.dtype == np.int64 and ids.min() >= 0 and ids.max() < 151936
    assert np.array_equal(ids, synth.token_ids(6, 1, 4096, 151936))


def test_chunk_workspace_sizes(nf4_lib):
    nf4 = nf4_lib
    # 14B-shaped chunk: partials + one ticket per 128-row tile, within the no-alloc scratch
    n = nf4.nf4_workspace_bytes(13824, 5120, 32)
    assert 16 < n <= 8 << 20
    # many tiles per block: whole tiles, no partials (argmax-sized workspace)
    assert nf4.nf4_workspace_bytes(151936, 2048, 1) == 16
    # K % 256 != 0 (fallback kernel only) still has its split-K partials
    assert nf4.nf4_workspace_bytes(13824, 5056, 32) > 16


@pytest.fixture(scope="module")
def nf4_lib():
    from nf4_weight_quantized_gb300 import build

    if not os.path.exists(build.library_path()):
        build.build()
    from nf4_weight_quantized_gb300 import nf4 as mod

    return mod


def _bench_lines(*args, env=None):
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], capture_output=True, text=True,
                       cwd=root, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_reference_arm_line():
    # the reference arm (the oracle on the host) prints one JSON line on the
    # same metric, unit and workload as the GPU arm
    lines = _bench_lines("--impl", "reference", "--steps", "2", "--warmup", "3")
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"]["workload"] == bench.WORKLOAD_NAME and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] >= 3 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    assert _bench_lines("--impl", "reference", "--steps", "2", "--warmup", "3", env=env) == []


def _chunk_plan(M, K, B=152):
    """The stream-K plan of the TMA chunk kernel, restated: (tiles, units per
    tile, units, blocks, partial slots per tile, first unit of each block)."""
    tiles, NQ = (M + 127) // 128, K // 256
    U = tiles * NQ
    Bn = max(1, min(U, B))
    if tiles >= 4 * Bn:
        return tiles, NQ, U, Bn, 0, [(b * tiles // Bn) * NQ for b in range(Bn + 1)]
    mu = U // Bn
    return tiles, NQ, U, Bn, min((NQ + mu - 1) // mu + 1, Bn), [b * U // Bn for b in range(Bn + 1)]


@pytest.mark.parametrize("M,K,N", [(13824, 5120, 32), (2048, 2048, 7), (5120, 27648, 16), (1000, 512, 3),
                                   (300, 65536, 32), (27648, 5120, 32), (128, 256, 1)])
def test_chunk_processing_order_and_partial_slots(nf4_lib, M, K, N):
    # every unit is processed by exactly one block; a block's runs of units stay
    # inside one tile; a block takes the head of its last tile first only when
    # that tile continues in the next block; no tile spans more blocks than it
    # has partial slots, and the library's workspace holds them all
    tiles, NQ, U, B, maxseg, start = _chunk_plan(M, K)
    seen = []
    for b in range(B):
        u0, u1 = start[b], start[b + 1]
        nq = u1 - u0
        tB = (u1 - 1) // NQ
        uB = tB * NQ
        nh = u1 - uB if (maxseg and uB > u0 and u1 % NQ) else 0
        r0 = u0 % NQ
        unit = [uB + q if q < nh else u0 + q - nh for q in range(nq)]
        seen += unit
        q = 0
        while q < nq:  # seg_end as the kernel computes it
            e = nh if q < nh else min(q + NQ - (r0 + q - nh) % NQ, nq)
            assert e > q and len({unit[i] // NQ for i in range(q, e)}) == 1
            assert all(unit[i + 1] == unit[i] + 1 for i in range(q, e - 1))
            q = e
    assert sorted(seen) == list(range(U))
    if maxseg:
        owners = {}
        for b in range(B):
            for u in range(start[b], start[b + 1]):
                owners.setdefault(u // NQ, set()).add(b)
        assert max(len(v) for v in owners.values()) <= maxseg
        assert nf4_lib.nf4_workspace_bytes(M, K, N) >= tiles * maxseg * N * 128 * 4 + tiles * 4 + 16
