"""The N>1 bench path on CPU: replicas with gloo, world size 2.

Each rank runs its own batch (weak scaling, no data-path collective); the only
cross-rank step is the timing reduction (max over ranks) and the byte sum.
"""

import json
import os
import socket
import subprocess
import sys
import time

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_q):
    import bench
    from paged_kv_cache_296_gb300 import workloads as wl
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                                         rank=rank, world_size=world)
    dev = torch.device("cpu")
    mx = bench.max_over_ranks(1.5 + rank, world, dev)
    sm = bench.sum_over_ranks(10.0 * (rank + 1), world, dev)
    W = wl.make_workload(wl.SPECS[2], 2 + 1000 * rank)     # the seed rule bench.py uses
    out_q.put((rank, mx, sm, W.context_lens.tolist()))
    bench.barrier(world)
    torch.distributed.destroy_process_group()


def test_replica_reductions_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, mx0, sm0, lens0), (_, mx1, sm1, lens1) = res
    assert mx0 == mx1 == 2.5          # the slowest rank sets the time
    assert sm0 == sm1 == 30.0         # bytes add up over ranks
    assert lens0 != lens1             # each replica has its own batch


def _run_bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_prints_one_line():
    r = _run_bench(["--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3",
                    "--ref-seconds", "1"], {})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["steps"] == 2 and d["warmup"] == 3


def test_reference_arm_is_bounded_for_many_steps():
    # the whole run holds about --ref-seconds of oracle time whatever --steps is
    t0 = time.perf_counter()
    r = _run_bench(["--impl", "reference", "--config", "2", "--steps", "2000", "--warmup", "20",
                    "--ref-seconds", "2"], {})
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["steps"] == 2000 and d["value"] > 0
    assert wall < 120, f"2000 reference steps took {wall:.0f} s"


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_bench_rejects_short_warmup():
    r = _run_bench(["--impl", "reference", "--warmup", "2"], {})
    assert r.returncode != 0


def test_l2_plan_flushes_only_below_twice_l2(monkeypatch):
    # A step whose distinct bytes are under twice the L2 size gets a flush
    # buffer of twice the L2 size; at or above it, none.
    sys.path.insert(0, ROOT)
    import bench

    class Props:
        L2_cache_size = 1000

    monkeypatch.setattr(bench.torch.cuda, "get_device_properties", lambda device: Props())
    buf, text = bench.l2_plan("cpu", 1999)
    assert buf is not None and buf.numel() == 2000 and "flushed" in text
    buf, text = bench.l2_plan("cpu", 2000)
    assert buf is None and "no flush" in text


def test_reference_arm_config_is_the_workload_config():
    # The reference arm's config is exactly the dict the GPU arm prints for the
    # same workload and seed: the workload, the L2 rule and the parallelism.
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_296_gb300 import workloads as wl
    r = _run_bench(["--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3",
                    "--ref-seconds", "1"], {"CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    W = wl.make_workload(wl.SPECS[1], 1)
    want = bench.workload_config(wl.SPECS[1], W, bench.l2_text(bench.decode_distinct_bytes(W),
                                                             129 * 10 ** 6), 1, "seqs")
    assert d["config"] == json.loads(json.dumps(want))


def _shard_rank_main(rank, world, port, out_q):
    import numpy as np
    from oracle import paged_attention as ref
    from paged_kv_cache_296_gb300 import workloads as wl
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                                         rank=rank, world_size=world)
    spec = wl.Spec("gqa tiny", 3, 8, 4, 64, "bf16", "bf16", ("fixed", [5, 40, 17]))
    W = wl.make_workload(spec, 77)                  # every rank draws the same whole batch
    P = wl.shard_heads(W, rank, world)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    out = ref.paged_decode(bits(P.q), "bf16", bits(P.pool), P.block_tables.numpy(),
                           P.context_lens.numpy(), P.scale, "bf16")
    parts = [torch.zeros((3, 8 // world, 64), dtype=torch.float64) for _ in range(world)]
    torch.distributed.all_gather(parts, torch.from_numpy(np.ascontiguousarray(out)))
    if rank == 0:
        whole = ref.paged_decode(bits(W.q), "bf16", bits(W.pool), W.block_tables.numpy(),
                                 W.context_lens.numpy(), W.scale, "bf16")
        out_q.put((torch.cat(parts, dim=1).numpy(), whole, P.spec.num_kv_heads))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_kv_head_sharding_gloo_world2():
    # Each rank decodes its slice of KV heads (and the query heads that read
    # them) of one batch with no exchange; the slices, gathered along the head
    # axis, are the whole batch's output exactly.
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got, want, hkv_rank = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert hkv_rank == 2
    assert got.shape == want.shape == (3, 8, 64)
    assert (got == want).all()


def test_kv_head_ranges_partition_the_heads():
    from paged_kv_cache_296_gb300 import workloads as wl
    for hkv in (1, 2, 4, 8, 32):
        for world in (1, 2, 4, 8):
            if hkv % world:
                with pytest.raises(ValueError):
                    wl.kv_head_range(hkv, 0, world)
                continue
            covered = []
            for r in range(world):
                h0, h1 = wl.kv_head_range(hkv, r, world)
                assert h1 - h0 == hkv // world
                covered.extend(range(h0, h1))
            assert covered == list(range(hkv))
