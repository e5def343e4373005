"""Benchmark of the paged-KV-cache decode hot path on one GB300 (or N GPUs).

One step = the write of each sequence's new token into the paged pool plus
decode attention over every sequence, on a seeded synthetic batch whose KV
cache is already resident in HBM.  By default the step is pa_decode_append
(write, attention and split-KV merge in one launch); --path separate times
pa_reshape_and_cache followed by pa_decode.  The other path is timed after
the headline loop and reported under "other_path".

The headline workload is --config (default 3, the Llama-3-8B GQA batch); the
--also workloads (default 5, 4, 2: long-context E4M3, shared-prefix sampling,
Llama-2-7B MHA) are timed in the same process by the same rules and reported
under "also", each with its own roofline block and clock record.

Prints ONE JSON line (rank 0).  ``value`` is attended-KV GB/s of the whole job
(sum over ranks of sum_i L_i*Hkv*D*2*elt bytes per step / step time, max
over ranks).  ``roofline`` reports the decode call against the measured HBM
copy bandwidth.  ``e2e`` repeats the measurement through the public API with
every step's inputs copied in from pinned host memory and its output copied
back inside the timed region (on copy streams that overlap the neighbouring
steps' kernels, as a serving loop runs).  ``cpu_baseline`` times the float64
CPU oracle on a bounded sample of the same batch.  A workload whose distinct
bytes per step are under twice the L2 size is timed one step at a time, each
step after an untimed write of twice the L2 size (the line's config.l2 says
which); larger ones run back to back.  ``config`` names the workload only and
is the same on both arms; how the steps were launched is under ``run``.

N > 1 (torchrun, one rank per GPU): --shard seqs (default) gives every GPU its
own batch (replicas, weak scaling); --shard heads splits the KV heads of one
batch over the GPUs, each rank decoding its heads with no collective in
attention (strong scaling).

Other legs: --prefill N (causal prefill TFLOP/s against the bf16 tensor peak;
--prefill-kv e4m3 over an E4M3 cache), --prefix-cache (prefix-cached against
full prefill), --blocks (pa_copy_blocks against the HBM peak and the block
manager's host step).  --impl reference times the CPU oracle as the
reference arm, about --ref-seconds of oracle time whatever --steps is.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 3] [--also 5,4,2]
                    [--shard seqs|heads] [--impl reference]
"""

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

# The CPU oracle leg runs single-threaded; fix BLAS threads before NumPy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_296_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-decode attended-KV GB/s (fraction of GB300 HBM peak); µs per decode step"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_METRIC = "paged-prefill TFLOP/s (causal attention FLOPs); µs per prefill step"
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = ["pa_decode_kernel.cuh", "pa_decode_split.cuh", "pa_ptx.cuh", "pa_decode_launch.cuh",
                  "pa_cache.cu", "pa_decode_f16.cu", "pa_decode_bf16.cu", "pa_decode_e4m3.cu"]


# ---------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world, device):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor-core peak (TFLOP/s): the measured cuBLAS burst figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback bf16"


PREFILL_SOURCES = ["pa_prefill_tc.cuh", "pa_tcgen05.cuh", "pa_prefill_params.cuh", "pa_prefill_launch.cuh",
                   "pa_prefill.cu", "pa_prefill_fp8.cu", "pa_ptx.cuh", "pa_cache.cu"]


def kernel_source_hash(sources=None):
    h = hashlib.sha256()
    for name in (sources or KERNEL_SOURCES):
        with open(os.path.join(ROOT, "paged_kv_cache_296_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config_id, step_path):
    """DRAM bytes per decode call from the committed ncu summary of this step
    path, if it still describes the current kernel source (else None)."""
    name = "paged_decode_append" if step_path == "append" else "paged_decode_kernel"
    path = os.path.join(PROFILE_DIR, f"{name}_config{config_id}.md")
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_decode_call:\s*([0-9.eE+]+)", text)
    if not m_src or not m_tr or m_src.group(1) != kernel_source_hash():
        return None
    return float(m_tr.group(1))


def profiled_prefill_traffic(n, fp8=False):
    """DRAM bytes per pa_prefill call from the committed ncu summary of prefill
    workload ``n`` (over an E4M3 cache if ``fp8``), if it still describes the
    current kernel source (else None)."""
    path = os.path.join(PROFILE_DIR,
                        f"paged_prefill_tc_kernel_prefill{n}{'_e4m3' if fp8 else ''}.md")
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_prefill_call:\s*([0-9.eE+]+)", text)
    if not m_src or not m_tr or m_src.group(1) != kernel_source_hash(PREFILL_SOURCES):
        return None
    return float(m_tr.group(1))


def l2_plan(device, distinct):
    """How the timed steps keep L2 from serving one step's inputs to the next.

    ``distinct`` is the bytes one step reads or writes, each byte counted once.
    At twice the L2 size or more, a step has evicted most of what the step
    before it left in L2, so steps run back to back; below that, every timed
    step is preceded by an untimed write of twice the L2 size and timed by its
    own events.  Returns (flush buffer or None, the line's "l2" text)."""
    l2 = device_l2_bytes(device)
    if distinct >= 2 * l2:
        return None, l2_text(distinct, l2)
    return torch.empty(2 * l2, dtype=torch.uint8, device=device), l2_text(distinct, l2)


def time_each(run_one, n, flush_buf, stream):
    """Mean device ms of n steps, each run after a write of ``flush_buf``
    (larger than L2) and bracketed by its own events on ``stream``."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for i in range(n):
        flush_buf.fill_(i & 0x7F)
        ev[i][0].record(stream)
        run_one()
        ev[i][1].record(stream)
    stream.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def one_step_runner(fn, device, graphs, no_graph):
    """``fn`` as one replay of a CUDA graph of a single step (or a plain call)."""
    if no_graph:
        return fn
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize(device)
    with torch.cuda.graph(g):
        fn()
    g.replay()  # one untimed replay
    torch.cuda.synchronize(device)
    graphs.append(g)
    return g.replay


def pipelined_e2e(S, step_fn, device):
    """Steps through the public API with host buffers, as a serving loop runs
    them: every step copies its inputs in from pinned host memory (one packed
    buffer) and its output back.  Two device copies of the inputs and of the
    output let two copy streams (one per direction) move step i+1's inputs in
    and step i-1's output back while step i computes; each step still makes
    its own two copies.
    Returns (enqueue(k): k such steps on the current stream, verify(): the
    last enqueued step's output as copied back equals a plain step's bit for
    bit, h2d bytes per step, d2h bytes per step)."""
    names = list(getattr(S, "step_inputs", S.STEP_INPUTS))
    hosts, devs, sets = [], [], []
    for _ in range(2):
        h, d = S.stage_inputs()
        hosts.append(h)
        devs.append(d)
        sets.append({k: getattr(S, k) for k in names})
    outs = [S.out, torch.empty_like(S.out)]
    out_host = [torch.empty(S.out.shape, dtype=S.out.dtype).pin_memory() for _ in range(2)]
    xs = torch.cuda.Stream(device)   # host to device
    ys = torch.cuda.Stream(device)   # device to host
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    last = [0]

    def bind(b):
        for k, v in sets[b].items():
            setattr(S, k, v)
        S.out = outs[b]

    def verify():
        torch.cuda.synchronize(device)
        got = out_host[last[0]].clone()
        bind(0)
        step_fn()
        torch.cuda.synchronize(device)
        want = S.out.cpu()
        if not torch.equal(got.view(torch.uint8), want.view(torch.uint8)):
            raise RuntimeError("pipelined e2e output differs from a plain step's")

    def enqueue(k):
        cs = torch.cuda.current_stream(device)
        fork, join_x, join_y = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        fork.record(cs)
        xs.wait_event(fork)
        ys.wait_event(fork)
        for i in range(k):
            b = i % 2
            with torch.cuda.stream(xs):
                if i >= 2:
                    xs.wait_event(ev_done[b])        # step i-2 no longer reads buffer b
                devs[b].copy_(hosts[b], non_blocking=True)
                ev_in[b].record(xs)
            if i >= 1:
                with torch.cuda.stream(ys):
                    ys.wait_event(ev_done[1 - b])    # step i-1's output is final
                    out_host[1 - b].copy_(outs[1 - b], non_blocking=True)
                    ev_out[1 - b].record(ys)
            cs.wait_event(ev_in[b])
            if i >= 2:
                cs.wait_event(ev_out[b])             # step i-2's output has been read back
            bind(b)
            step_fn()
            ev_done[b].record(cs)
        b = (k - 1) % 2
        last[0] = b
        with torch.cuda.stream(ys):
            ys.wait_event(ev_done[b])
            out_host[b].copy_(outs[b], non_blocking=True)
            join_y.record(ys)
        join_x.record(xs)
        cs.wait_event(join_x)
        cs.wait_event(join_y)

    return (enqueue, verify, hosts[0].numel(),
            out_host[0].numel() * out_host[0].element_size())


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[4][1:5])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "power_w_max": max(r[3] for r in inside),
                "samples": len(inside), "reasons": reasons}


# ---------------------------------------------------------------- CPU oracle leg

class OracleSampler:
    """Times the float64 oracle on bounded samples of a decode workload.

    The unit of work is one sequence, all heads, over the first L' of its L
    tokens (a decode over a shorter context): the oracle's ``paged_decode`` on
    that problem.  L' is L when the time budget allows, else the share of it
    the oracle's measured rate fits into the budget (at least one block), so a
    sample never runs far past its budget.  Successive calls take the
    sequences in turn.
    """

    def __init__(self, W, pool_cpu_rows):
        self.W = W
        self.rows_fn = pool_cpu_rows
        spec = W.spec
        elt = 1 if spec.kv_dtype == "e4m3" else 2
        self.tok_bytes = spec.num_kv_heads * spec.head_size * 2 * elt
        self.q_bits = W.q.cpu().view(torch.int16).numpy().view(np.uint16)
        self.lens = W.context_lens.cpu().numpy()
        self.tables = W.block_tables.cpu().numpy()
        self.cursor = 0
        self.rate = None  # attended bytes per oracle second, once measured

    def sample(self, seconds):
        """Run samples until ``seconds`` of oracle time (at least one).
        Returns (attended bytes processed, elapsed s, samples)."""
        from oracle import paged_attention as ref  # test infrastructure: only these legs run it
        spec = self.W.spec
        done_bytes, elapsed, n = 0, 0.0, 0
        while n == 0 or elapsed < seconds:
            i = self.cursor % spec.num_seqs
            self.cursor += 1
            L = int(self.lens[i])
            budget = max(seconds - elapsed, 0.0)
            cap = L if self.rate is None else int(self.rate * budget / self.tok_bytes)
            Lp = min(L, max(16, cap, 0)) if L > 0 else 0
            nb = -(-Lp // 16)
            pool = self.rows_fn(self.tables[i, :nb].astype(np.int64))
            table = np.arange(max(nb, 1))[None, :]
            t = time.perf_counter()
            ref.paged_decode(self.q_bits[i:i + 1], spec.q_dtype, pool, table, np.array([Lp]),
                             self.W.scale, spec.kv_dtype, self.W.kv_scale)
            dt = time.perf_counter() - t
            elapsed += dt
            done_bytes += Lp * self.tok_bytes
            n += 1
            if Lp > 0 and dt > 0:
                r = Lp * self.tok_bytes / dt
                self.rate = r if self.rate is None else 0.5 * (self.rate + r)
        return done_bytes, elapsed, n


def oracle_rows_fn(W):
    """Pool rows of given physical blocks as the oracle sees them, built from the
    generator's own arrays (never from memory the CUDA path wrote): the 16-bit
    pool as drawn, or the oracle's quantisation of the fp32 source values."""
    if W.spec.kv_dtype == "e4m3":
        from oracle import paged_attention as ref

        def rows(blocks):
            src = W.pool_src[torch.from_numpy(blocks).to(W.pool_src.device)].cpu().contiguous()
            return ref.fp8_quantise(src.view(torch.int32).numpy().view(np.uint32), "f32",
                                    W.kv_scale)
        return rows

    def rows(blocks):
        t = W.pool[torch.from_numpy(blocks).to(W.pool.device)].cpu()
        return t.view(torch.int16).numpy().view(np.uint16)
    return rows


# The oracle on every host core: worker processes (spawn start, one BLAS
# thread each) attach to the pool rows in shared memory and decode whole
# sequences; the parent hands out sequences in turn and divides the attended
# bytes of the finished ones by the wall time.
_ORACLE_WORKER = {}


def _oracle_worker_init(shm_name, shape, dtype, q_bits, tables, q_dtype, kv_dtype, scale, kv_scale):
    from multiprocessing import shared_memory
    shm = shared_memory.SharedMemory(name=shm_name)
    _ORACLE_WORKER.update(shm=shm, pool=np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf),
                          q=q_bits, tables=tables, q_dtype=q_dtype, kv_dtype=kv_dtype,
                          scale=scale, kv_scale=kv_scale)


def _oracle_worker_decode(task):
    """One sequence (index, attended tokens): gather its rows, run the oracle."""
    from oracle import paged_attention as ref  # test infrastructure: the CPU baseline legs only
    i, L = task
    o = _ORACLE_WORKER
    nb = -(-L // 16)
    rows = o["pool"][o["tables"][i, :nb].astype(np.int64)]
    ref.paged_decode(o["q"][i:i + 1], o["q_dtype"], rows, np.arange(max(nb, 1))[None, :],
                     np.array([L]), o["scale"], o["kv_dtype"], o["kv_scale"])
    return L


class ParallelOracleSampler:
    """The float64 oracle over a decode workload on ``workers`` host processes.

    Over a 16-bit cache only (an E4M3 pool would have to be quantised by the
    oracle in every worker): the pool's rows as drawn go to shared memory once.
    ``sample(seconds)`` hands out whole sequences, in turn, until ``seconds`` of
    wall time have passed, waits for those in flight and returns (attended
    bytes, wall seconds, sequences).
    """

    def __init__(self, W, workers):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        spec = W.spec
        self.spec = spec
        self.workers = workers
        self.tok_bytes = spec.num_kv_heads * spec.head_size * 2 * 2
        pool = W.pool.cpu().view(torch.int16).numpy().view(np.uint16)
        self.shm = shared_memory.SharedMemory(create=True, size=max(pool.nbytes, 1))
        np.ndarray(pool.shape, dtype=pool.dtype, buffer=self.shm.buf)[...] = pool
        self.lens = W.context_lens.cpu().numpy()
        q_bits = W.q.cpu().view(torch.int16).numpy().view(np.uint16)
        tables = W.block_tables.cpu().numpy()
        self.pool = mp.get_context("spawn").Pool(
            processes=workers, initializer=_oracle_worker_init,
            initargs=(self.shm.name, pool.shape, pool.dtype.str, q_bits, tables, spec.q_dtype,
                      spec.kv_dtype, W.scale, W.kv_scale))
        self.cursor = 0
        # every worker started and warm (imports done) before any timing
        self.pool.map(_oracle_worker_decode, [(self._next(), 16)] * workers, chunksize=1)

    def _next(self):
        i = self.cursor % self.spec.num_seqs
        self.cursor += 1
        return i

    def sample(self, seconds):
        pending = []
        done_tok, n = 0, 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds or not (pending or n):
            while len(pending) < 2 * self.workers:
                i = self._next()
                pending.append(self.pool.apply_async(_oracle_worker_decode,
                                                     ((i, int(self.lens[i])),)))
            head = pending.pop(0)
            done_tok += head.get()
            n += 1
        for r in pending:
            done_tok += r.get()
            n += 1
        return done_tok * self.tok_bytes, time.perf_counter() - t0, n

    def close(self):
        self.pool.close()
        self.pool.join()
        self.shm.close()
        self.shm.unlink()


def shm_fits(nbytes):
    """Whether POSIX shared memory has room for ``nbytes`` (with a margin)."""
    try:
        st = os.statvfs("/dev/shm")
    except OSError:
        return False
    return st.f_bavail * st.f_frsize > 1.2 * nbytes


def parallel_oracle_ok(W, cores):
    """The parallel oracle runs over 16-bit caches, on several cores, when the
    pool fits in shared memory; else the one-core sampler runs."""
    return (W.spec.kv_dtype != "e4m3" and cores > 1
            and shm_fits(W.pool.numel() * W.pool.element_size()))


def oracle_baseline(W, seconds):
    """The cpu_baseline block: the oracle on every host core over ``seconds`` of
    wall time (16-bit caches), else on one core over ``seconds`` of its time."""
    cores = os.cpu_count() or 1
    if parallel_oracle_ok(W, cores):
        sampler = ParallelOracleSampler(W, cores)
        try:
            b, secs, nseq = sampler.sample(seconds)
        finally:
            sampler.close()
        where = f"{cores} worker processes (spawn), 1 BLAS thread each, wall time"
    else:
        b, secs, nseq = OracleSampler(W, oracle_rows_fn(W)).sample(seconds)
        cores = 1
        where = "1 BLAS thread, oracle time"
    return {"value": round(b / secs / 1e9, 4), "unit": "GB/s", "cores": cores,
            "host_cpus": os.cpu_count(), "kind": "oracle",
            "sample": f"float64 NumPy oracle, {nseq} sequences of this batch (all heads; a "
                      f"sequence cut to fewer tokens only on one core, if the time budget ends "
                      f"inside it), {secs:.1f} s, {where}"}


# ---------------------------------------------------------------- main legs

def parallelism(world, shard):
    """How the job is spread over GPUs, the same words on both arms."""
    if world <= 1:
        return "one device"
    if shard == "heads":
        return f"kv heads sharded over {world} GPUs (no collective in attention)"
    return f"replicas{world}"


def l2_text(distinct, l2_bytes):
    """The line's config.l2: which L2 rule the timed steps follow (see l2_plan)."""
    if distinct >= 2 * l2_bytes:
        return (f"inputs larger than L2: {distinct / 1e6:.0f} MB of distinct bytes per "
                f"step (L2 {l2_bytes / 1e6:.0f} MB), no flush")
    return (f"L2 flushed before every timed step by an untimed {2 * l2_bytes / 1e6:.0f} MB write "
            f"({distinct / 1e6:.1f} MB of distinct bytes per step, L2 {l2_bytes / 1e6:.0f} MB); "
            f"each step timed by its own CUDA events")


def device_l2_bytes(device=None):
    """L2 size of ``device`` (of GPU 0 if None; the nominal 129 MB where no GPU is visible)."""
    if device is None and not torch.cuda.is_available():
        return 129 * 10 ** 6
    props = torch.cuda.get_device_properties(device if device is not None else 0)
    return int(getattr(props, "L2_cache_size", 0) or 129 * 10 ** 6)


def decode_distinct_bytes(W):
    """Bytes one decode step reads or writes, each counted once (shared blocks once)."""
    from paged_kv_cache_296_gb300.runner import step_bytes, unique_kv_bytes
    total_bytes, kv_bytes, new_bytes = step_bytes(W)
    return unique_kv_bytes(W) + (total_bytes - kv_bytes) + new_bytes


def workload_config(spec, W, l2, world, shard):
    """The line's ``config``: the workload and the L2 rule only, identical on both
    arms for the same workload and seed (timing details go under ``run``)."""
    return {"workload": spec.name, "num_seqs": spec.num_seqs, "num_q_heads": spec.num_q_heads,
            "num_kv_heads": spec.num_kv_heads, "head_size": spec.head_size, "block_size": 16,
            "q_dtype": spec.q_dtype, "kv_dtype": spec.kv_dtype,
            "mean_context": float(W.context_lens.float().mean()),
            "num_blocks": W.num_blocks, "seed": W.seed, "l2": l2,
            "parallelism": parallelism(world, shard)}


def rank_workload(args, config_id, world, rank, device):
    """This rank's decode workload: its own batch (replicas, seed + 1000 * rank),
    or its slice of KV heads of the one shared batch (--shard heads).
    Returns (the whole workload this rank's slice comes from, the slice)."""
    spec = wl.SPECS[config_id]
    if args.shard == "heads" and world > 1:
        W = wl.make_workload(spec, config_id, device=str(device))
        return W, wl.shard_heads(W, rank, world)
    W = wl.make_workload(spec, config_id + 1000 * rank, device=str(device))
    return W, W


def decode_leg(args, config_id, world, rank, device, headline):
    """Build, warm up and time one decode workload.  The headline leg also times
    the other step path, the e2e path through host buffers and the CPU oracle;
    returns the JSON line (headline) or a compact record of the same figures."""
    from paged_kv_cache_296_gb300 import binding as pa
    from paged_kv_cache_296_gb300.runner import DecodeStep, step_bytes, unique_kv_bytes

    spec = wl.SPECS[config_id]
    W_all, W = rank_workload(args, config_id, world, rank, device)
    S = DecodeStep(W, device=device, partition_size=args.partition_size)
    total_bytes, kv_bytes, new_bytes = step_bytes(W)
    stream = torch.cuda.current_stream(device)
    path = args.path if headline else "append"
    step_fn = S.append if path == "append" else S.step

    for _ in range(args.warmup):
        step_fn()
    torch.cuda.synchronize(device)
    pa.pa_device_status(clear=True)
    flush_buf, _ = l2_plan(device, decode_distinct_bytes(W))
    l2 = l2_text(decode_distinct_bytes(W_all), device_l2_bytes(device))
    graphs = []  # kept alive until the leg ends

    def steps_per_graph(n):
        return max(d for d in range(1, min(n, 20) + 1) if n % d == 0)

    def make_runner(fn, n):
        """A callable that runs n steps of fn.  With graphs (the default) the
        steps are captured once, a few per CUDA graph (so the kernels of
        consecutive steps keep their programmatic-launch overlap), and the
        graph is replayed: every replay runs every kernel of those steps again,
        without the Python and launch overhead of issuing them one by one."""
        if args.no_graph:
            def run():
                for _ in range(n):
                    fn()
            return run
        spg = steps_per_graph(n)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(device)
        with torch.cuda.graph(g):
            for _ in range(spg):
                fn()
        g.replay()  # one untimed replay
        torch.cuda.synchronize(device)
        graphs.append(g)

        def run():
            for _ in range(n // spg):
                g.replay()
        return run

    def timed(which, n):
        """Time n steps of ``which``.  With inputs of twice the L2 size or more,
        CUDA events only at the ends of the region (an event between kernels
        would cost time and break their programmatic-launch overlap); with
        smaller ones, each step after an L2 flush, between its own events.
        Returns (ms per step, t0, t1)."""
        fn = S.append if which == "append" else S.step
        if flush_buf is not None:
            one = one_step_runner(fn, device, graphs, args.no_graph)
            barrier(world)
            torch.cuda.synchronize(device)
            t0 = time.time()
            ms = time_each(one, n, flush_buf, stream)
            barrier(world)
            return ms, t0, time.time()
        run = make_runner(fn, n)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(device)
        t0 = time.time()
        start.record(stream)
        run()
        end.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        t1 = time.time()
        return start.elapsed_time(end) / n, t0, t1

    def per_call(n):
        """Mean ms of the write call and of the decode call on the two-call path,
        each bracketed by its own events (outside the headline timing)."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        torch.cuda.synchronize(device)
        for i in range(n):
            if flush_buf is not None:
                flush_buf.fill_(i & 0x7F)
            ev[i][0].record(stream)
            S.write()
            ev[i][1].record(stream)
            S.decode()
            ev[i][2].record(stream)
        torch.cuda.synchronize(device)
        return (statistics.mean(e[0].elapsed_time(e[1]) for e in ev),
                statistics.mean(e[1].elapsed_time(e[2]) for e in ev))

    sampler = ClockSampler(device.index)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    n = args.steps
    ms_local, t_wall0, t_wall1 = timed(path, n)
    sampler.stop()
    ms_step = max_over_ranks(ms_local, world, device)
    status = pa.pa_device_status(clear=True)
    if status != 0:
        raise RuntimeError(f"device status {status:#x}: a kernel gave up waiting")
    # The step on the append path is one decode call (attention + merge), so
    # its mean duration over the timed region is the call's.
    if path == "append":
        dec_ms, write_ms = ms_local, 0.0
    else:
        write_ms, dec_ms = per_call(min(n, 500))

    all_kv = sum_over_ranks(kv_bytes, world, device)
    value = all_kv / (ms_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    if path == "append":
        call_bytes = total_bytes + new_bytes
        kernel = "pa_decode_append (token write + attention, then the split-KV merge)"
    else:
        call_bytes = total_bytes
        kernel = "pa_decode (attention + split-KV merge)"
    achieved = call_bytes / (dec_ms * 1e-3) / 1e9
    traffic = profiled_traffic(config_id, path) if args.shard != "heads" or world == 1 else None
    shared = spec.lens[0] == "shared_prefix"
    roofline = {"bound": "hbm", "kernel": kernel,
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                "algorithmic_bytes_per_launch": call_bytes, "traffic": traffic}
    if shared:
        # each shared block counted once: the bytes the step must move at least
        uniq = unique_kv_bytes(W) + (total_bytes - kv_bytes) + (new_bytes if path == "append" else 0)
        roofline["unique_bytes_per_launch"] = uniq
        roofline["frac_unique"] = round(uniq / (dec_ms * 1e-3) / 1e9 / peak, 4)
    run_info = {"step": path,
                "launch": "stream" if args.no_graph else
                          "CUDA graph replay, 1 step per graph" if flush_buf is not None else
                          f"CUDA graph replay, {steps_per_graph(n)} steps per graph",
                "partition_tokens": S.partition_tokens}
    clocks = sampler.summary(t_wall0, t_wall1)
    if not headline:
        rec = {"workload": spec.name, "config": workload_config(spec, W_all, l2, world, args.shard),
               "value": round(value, 2), "unit": "GB/s", "us_per_step": round(ms_step * 1e3, 2),
               "frac_of_hbm_peak": round(value / peak, 4),
               "seqs_per_s": round(spec.num_seqs * (1 if args.shard == "heads" else world)
                                   / (ms_step * 1e-3), 1),
               "roofline": roofline, "run": run_info,
               "gpu_launches": S.launches_per_step(path) * n, "clocks": clocks}
        if shared:
            rec["unique_kv_gbs"] = round(sum_over_ranks(unique_kv_bytes(W), world, device)
                                         / (ms_step * 1e-3) / 1e9, 2)
        return rec

    # The other way to run the same step, for comparison (not the headline).
    alt = None
    if not args.no_alt:
        other = "separate" if path == "append" else "append"
        fn = S.append if other == "append" else S.step
        for _ in range(args.warmup):
            fn()
        a_ms, _, _ = timed(other, n)
        alt = {"path": other, "us_per_step": round(max_over_ranks(a_ms, world, device) * 1e3, 2)}
        if other == "separate":
            w_ms, d_ms = per_call(min(n, 500))
            alt["us_write_call"] = round(w_ms * 1e3, 2)
            alt["us_decode_call"] = round(d_ms * 1e3, 2)

    # ---- e2e through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        # the step's inputs live packed in one pinned host buffer (q, new k/v,
        # slot mapping, block tables, lengths): one host-to-device copy per
        # step, overlapped with the previous step's kernels (double buffers)
        enqueue, verify, h2d, d2h = pipelined_e2e(S, step_fn, device)
        enqueue(max(2, args.warmup))
        torch.cuda.synchronize(device)
        if flush_buf is not None:
            # one step at a time after each flush: its copies in and out are
            # inside its events, with no overlap from a neighbouring step
            one = one_step_runner(lambda: enqueue(1), device, graphs, args.no_graph)
            run_e2e = None
        elif args.no_graph:
            def run_e2e():
                enqueue(n)
        else:
            spg = steps_per_graph(n)
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge):
                enqueue(spg)
            ge.replay()
            torch.cuda.synchronize(device)
            graphs.append(ge)

            def run_e2e():
                for _ in range(n // spg):
                    ge.replay()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        if run_e2e is None:
            e_local = time_each(one, n, flush_buf, stream)
        else:
            s2.record(stream)
            run_e2e()
            e2.record(stream)
            torch.cuda.synchronize(device)
            e_local = s2.elapsed_time(e2) / n
        barrier(world)
        verify()
        e2e_ms = max_over_ranks(e_local, world, device)
        e2e_gbs = all_kv / (e2e_ms * 1e-3) / 1e9
        e2e = {"value": round(e2e_gbs, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # ---- CPU oracle baseline (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(W, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "us_decode_call": round(dec_ms * 1e3, 2),
        "us_write_call": round(write_ms * 1e3, 2) if path != "append" else None,
        "frac_of_hbm_peak": round(value / peak, 4),
        "seqs_per_s": round(spec.num_seqs * (1 if args.shard == "heads" else world)
                            / (ms_step * 1e-3), 1),
        "higher_is_better": True,
        "scaling": "strong" if (args.shard == "heads" and world > 1) else "weak",
        "vs_baseline": None,
        "dtype": spec.kv_dtype if spec.kv_dtype == spec.q_dtype else f"{spec.q_dtype}+{spec.kv_dtype}",
        "data": "synthetic (seeded N(0,1) K/V/q; no model weights)",
        "config": workload_config(spec, W_all, l2, world, args.shard),
        "run": run_info,
        "roofline": roofline,
        "other_path": alt,
        "gpu_launches": S.launches_per_step(path) * n,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
    }
    if shared:
        line["unique_kv_gbs"] = round(sum_over_ranks(unique_kv_bytes(W), world, device)
                                      / (ms_step * 1e-3) / 1e9, 2)
    return line


def run_ours(args, world, rank, local):
    """The decode headline on --config, then every --also workload in the same
    process, each timed by the same rules; one JSON line with the others under
    ``also``."""
    from paged_kv_cache_296_gb300 import binding as pa

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    pa.load()
    if args.shard == "heads" and world > 1:
        for c in [args.config] + args.also:
            if wl.SPECS[c].num_kv_heads % world:
                raise SystemExit(f"--shard heads: workload {c} has {wl.SPECS[c].num_kv_heads} "
                                 f"KV heads, not a multiple of {world}")
    line = decode_leg(args, args.config, world, rank, device, headline=True)
    also = {}
    for c in args.also:
        if c != args.config:
            torch.cuda.empty_cache()
            also[f"config{c}"] = decode_leg(args, c, world, rank, device, headline=False)
    line["also"] = also or None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


class PrefillOracleSampler:
    """Times the float64 oracle on query rows of a prefill batch (all heads of
    each row), drawn over its sequences.  The oracle's pool after the step's
    write is built once."""

    def __init__(self, W):
        from oracle import paged_attention as ref  # test infrastructure: only these legs run it
        self.W = W
        dt = W.spec.dtype
        self.lens = W.context_lens.cpu().numpy()
        self.qsl = W.query_start_loc.cpu().numpy()
        self.tables = W.block_tables.cpu().numpy()
        self.q_bits = W.q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        pool = W.pool.cpu()
        self.pbits = ref.reshape_and_cache(pool.view(torch.int16).numpy().view(np.uint16),
                                           W.k_new.cpu().view(torch.int16).numpy().view(np.uint16),
                                           W.v_new.cpu().view(torch.int16).numpy().view(np.uint16),
                                           W.slot_mapping.cpu().numpy(), dt, dt)
        self.rng = np.random.default_rng(0)

    def sample(self, seconds):
        """Rows until ``seconds`` of oracle time (at least one row).
        Returns (flops, seconds, rows)."""
        from oracle import paged_attention as ref
        spec = self.W.spec
        dt = spec.dtype
        flops, elapsed, rows = 0, 0.0, 0
        while rows == 0 or elapsed < seconds:
            i = int(self.rng.integers(spec.num_seqs))
            n = int(self.qsl[i + 1] - self.qsl[i])
            if n == 0:
                continue
            t_ = int(self.rng.integers(n))
            pos = int(self.lens[i]) - n + t_
            nb = pos // 16 + 1
            sub = self.pbits[self.tables[i, :nb].astype(np.int64)]
            r = int(self.qsl[i]) + t_
            t0 = time.perf_counter()
            ref.paged_prefill(self.q_bits[r:r + 1], dt, sub, np.arange(nb)[None, :],
                              np.array([pos + 1]), np.array([0, 1]), self.W.scale, dt)
            elapsed += time.perf_counter() - t0
            flops += 4 * spec.head_size * spec.num_q_heads * (pos + 1)
            rows += 1
        return flops, elapsed, rows


def run_prefill(args, world, rank, local):
    """The prefill leg: one step = the write of the query tokens' K/V plus
    pa_prefill over a seeded prefill batch; value = causal attention TFLOP/s."""
    from paged_kv_cache_296_gb300 import binding as pa
    from paged_kv_cache_296_gb300.runner import PrefillStep, prefill_flops

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    pa.load()
    spec = wl.PREFILL_SPECS[args.prefill]
    W = wl.make_prefill_workload(spec, 10 + args.prefill + 1000 * rank, device=str(device))
    fp8 = args.prefill_kv == "e4m3"
    S = PrefillStep(W, device=device, kv_dtype=args.prefill_kv)
    flops = prefill_flops(W)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        S.step()
    torch.cuda.synchronize(device)
    pa.pa_device_status(clear=True)
    n = args.steps
    graphs = []
    # distinct bytes per step: the context K/V in the cache, q, out and the
    # query tokens' K/V sources
    kv_elt = S.pool.element_size()
    distinct = (int(W.context_lens.to(torch.int64).sum()) * spec.num_kv_heads * spec.head_size
                * 2 * kv_elt + 2 * S.q.numel() * S.q.element_size()
                + 2 * S.k_new.numel() * S.k_new.element_size())
    flush_buf, l2_text = l2_plan(device, distinct)

    def runner(fn):
        if args.no_graph:
            def run():
                for _ in range(n):
                    fn()
            return run, "stream"
        spg = max(d for d in range(1, min(n, 20) + 1) if n % d == 0)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(device)
        with torch.cuda.graph(g):
            for _ in range(spg):
                fn()
        g.replay()
        torch.cuda.synchronize(device)
        graphs.append(g)

        def run():
            for _ in range(n // spg):
                g.replay()
        return run, f"CUDA graph replay, {spg} steps per graph"

    def timed(run):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(device)
        t0 = time.time()
        a.record(stream)
        run()
        b.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        return a.elapsed_time(b) / n, t0, time.time()

    if flush_buf is not None:
        one = one_step_runner(S.step, device, graphs, args.no_graph)
        launch = "stream" if args.no_graph else "CUDA graph replay, 1 step per graph"
    else:
        run, launch = runner(S.step)
    sampler = ClockSampler(device.index)
    sampler.start()
    time.sleep(0.3)
    if flush_buf is not None:
        barrier(world)
        torch.cuda.synchronize(device)
        t0 = time.time()
        ms_local = time_each(one, n, flush_buf, stream)
        barrier(world)
        t1 = time.time()
    else:
        ms_local, t0, t1 = timed(run)
    sampler.stop()
    ms_step = max_over_ranks(ms_local, world, device)
    status = pa.pa_device_status(clear=True)
    if status != 0:
        raise RuntimeError(f"device status {status:#x}")
    # the attention kernel alone (the write is a small share of the step)
    def attention_call():
        pa.pa_prefill(S.out, S.q, S.k_cache, S.v_cache, S.block_tables, S.context_lens,
                      S.query_start_loc, S.max_query_len, S.scale, kv_scale=S.kv_scale)

    S.step()
    torch.cuda.synchronize(device)
    if flush_buf is not None:
        attn_ms = time_each(attention_call, min(n, 50), flush_buf, stream)
    else:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(stream)
        for _ in range(min(n, 50)):
            attention_call()
        ev[1].record(stream)
        torch.cuda.synchronize(device)
        attn_ms = ev[0].elapsed_time(ev[1]) / min(n, 50)

    e2e = None
    if not args.no_e2e:
        # inputs copied in and the output back every step, overlapped with the
        # neighbouring steps' kernels (double buffers)
        enqueue, verify, h2d, d2h = pipelined_e2e(S, S.step, device)
        enqueue(max(2, args.warmup))
        torch.cuda.synchronize(device)
        if flush_buf is not None:
            # one step at a time after each flush, its copies inside its events
            one_e2e = one_step_runner(lambda: enqueue(1), device, graphs, args.no_graph)
            barrier(world)
            e_ms = time_each(one_e2e, n, flush_buf, stream)
            barrier(world)
        else:
            if args.no_graph:
                def run_e2e():
                    enqueue(n)
            else:
                spg = max(d for d in range(1, min(n, 20) + 1) if n % d == 0)
                ge = torch.cuda.CUDAGraph()
                with torch.cuda.graph(ge):
                    enqueue(spg)
                ge.replay()
                torch.cuda.synchronize(device)
                graphs.append(ge)

                def run_e2e():
                    for _ in range(n // spg):
                        ge.replay()
            e_ms, _, _ = timed(run_e2e)
        verify()
        e_ms = max_over_ranks(e_ms, world, device)
        e2e = {"value": round(sum_over_ranks(flops, world, device) / (e_ms * 1e-3) / 1e12, 2),
               "unit": "TFLOP/s", "ms_per_step": round(e_ms, 5),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, secs, rows = PrefillOracleSampler(W).sample(args.cpu_seconds)
        cpu = {"value": round(f / secs / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
               "host_cpus": os.cpu_count(),
               "kind": "oracle",
               "sample": f"float64 NumPy oracle, {rows} query rows (all heads) of this batch, "
                         f"{secs:.1f} s, 1 BLAS thread"
                         + (" (on the 16-bit cache values: the same attention work)" if fp8 else "")}
    peak, peak_kind = tensor_peak()
    value = sum_over_ranks(flops, world, device) / (ms_step * 1e-3) / 1e12
    achieved = flops / (attn_ms * 1e-3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2), "us_prefill_call": round(attn_ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": spec.dtype, "data": "synthetic (seeded N(0,1) K/V/q; no model weights)",
        "config": {"workload": spec.name, "num_seqs": spec.num_seqs,
                   "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads,
                   "head_size": spec.head_size, "block_size": 16,
                   "query_tokens": int(W.q.shape[0]), "max_query_len": S.max_query_len,
                   "mean_context": float(W.context_lens.float().mean()),
                   "kv_dtype": "e4m3" if fp8 else spec.dtype,
                   "step": "pa_reshape_and_cache of the query tokens + pa_prefill",
                   "launch": launch,
                   "l2": l2_text + "; within a step, K/V re-read by a sequence's tiles comes from L2",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "paged_prefill_tc_kernel (tcgen05, S/P/O in TMEM)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "algorithmic_flops_per_launch": flops,
                     "traffic": profiled_prefill_traffic(args.prefill, fp8)},
        "gpu_launches": S.launches_per_step * n,
        "e2e": e2e, "cpu_baseline": cpu,
        "clocks": sampler.summary(t0, t1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


BLOCKS_METRIC = "block manager: pa_copy_blocks GB/s (copy-on-write block copies); host µs per decode step"


def run_blocks(args, world, rank, local):
    """The block manager leg.  GPU: pa_copy_blocks over 4096 (src, dst) pairs
    of 64 KB blocks (fp16 pool, 8 KV heads, d128), read + write bytes against
    the HBM peak.  Host: the native manager's decode step for 256 sequences
    (append one token each, export the block tables), microseconds per step."""
    from paged_kv_cache_296_gb300 import binding as pa

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    pa.load()
    nb, hkv, d, npairs = 16384, 8, 128, 4096
    pool = torch.empty((nb, 16, 2, hkv, d), dtype=torch.float16, device=device)
    pool.normal_()
    g = torch.Generator(device="cpu").manual_seed(7 + rank)
    perm = torch.randperm(nb, generator=g)
    pairs = torch.stack([perm[:npairs], perm[npairs:2 * npairs]], 1).to(torch.int64).to(device)
    block_bytes = pool[0].numel() * 2
    moved = 2 * npairs * block_bytes
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        pa.pa_copy_blocks(pool, pairs)
    torch.cuda.synchronize(device)
    n = args.steps
    sampler = ClockSampler(device.index)
    sampler.start()
    time.sleep(0.3)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    t0 = time.time()
    a.record(stream)
    for _ in range(n):
        pa.pa_copy_blocks(pool, pairs)
    b.record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    t1 = time.time()
    sampler.stop()
    ms = max_over_ranks(a.elapsed_time(b) / n, world, device)
    if pa.pa_device_status(clear=True) != 0:
        raise RuntimeError("pa_copy_blocks raised a device status bit")
    gbs = sum_over_ranks(moved, world, device) / (ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()

    # host: the manager's side of a decode step, 256 running sequences
    bm = pa.BlockManager(1 << 16)
    seqs = list(range(256))
    for s_ in seqs:
        bm.allocate(s_, 1000 + 7 * s_)
    for s_ in seqs[::4]:
        bm.fork(s_, 10000 + s_)                 # some shared blocks: copy-on-write happens
    ids = seqs + [10000 + s_ for s_ in seqs[::4]]
    host_steps = 200
    t_h = time.perf_counter()
    ids_np = np.array(ids, dtype=np.int64)
    ones = np.ones(len(ids), dtype=np.int64)
    for _ in range(host_steps):
        bm.append_batch(ids_np, ones, as_arrays=True)
        bm.block_tables(ids_np, 256)
    host_us = (time.perf_counter() - t_h) / host_steps * 1e6
    line = {
        "metric": BLOCKS_METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (N(0,1) pool, random block pairs)",
        "config": {"workload": f"{npairs} copies of 64 KB blocks (16 tokens x 2 x 8 heads x "
                               f"d128 fp16) in a {nb}-block pool",
                   "l2": f"{moved / 1e9:.2f} GB moved per step, larger than L2",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "copy_blocks_kernel", "achieved": round(gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                     "peak_kind": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": moved,
                     "traffic": None},
        "host": {"us_per_decode_step": round(host_us, 2), "sequences": len(ids),
                 "what": "pa_bm_append_batch (one token each) + pa_bm_block_tables (width 256), "
                         "through the Python binding"},
        "gpu_launches": n, "e2e": None, "cpu_baseline": None,
        "clocks": sampler.summary(t0, t1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


PREFIX_METRIC = ("prefix-cached prefill speed-up (x) for a 2000-token system prompt + "
                 "100-token user turn; µs per prefill step")


def run_prefix_cache(args, world, rank, local):
    """Prefix caching in the pages' system-prompt scenario (a 2K system prompt
    plus a 100-token user turn), 16 requests, Llama-3-8B-shaped heads, bf16.
    With the cache the block manager finds the system prompt's 125 blocks and
    the step writes and prefills only the 100 user tokens per request; without
    it, every request writes and prefills all 2100 tokens.  value = the ratio
    of the two step times."""
    from paged_kv_cache_296_gb300 import binding as pa

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    pa.load()
    B, sys_len, user_len, hq, hkv, d = 16, 2000, 100, 32, 8, 128
    L = sys_len + user_len
    nb = (B + 1) * (-(-L // 16)) + 16
    g = torch.Generator(device="cpu").manual_seed(21 + rank)
    system = torch.randint(0, 128000, (sys_len,), generator=g)
    users = torch.randint(0, 128000, (B, user_len), generator=g)
    pool = torch.empty((nb, 16, 2, hkv, d), dtype=torch.bfloat16, device=device)
    pool.normal_()
    kc, vc = pa.kv_views(pool)
    scale = 1.0 / math.sqrt(d)

    def build(cached_mode):
        bm = pa.BlockManager(nb)
        if cached_mode:
            bm.allocate_cached(10 ** 6, system.tolist() + [0])  # an earlier request warms the cache
        n_cached = []
        for i in range(B):
            toks = system.tolist() + users[i].tolist()
            n_cached.append(bm.allocate_cached(i, toks) if cached_mode else (bm.allocate(i, L) or 0))
        tables, lens = bm.block_tables(list(range(B)), -(-L // 16))
        nq = [L - c for c in n_cached]
        qsl = torch.tensor([0] + list(np.cumsum(nq)), dtype=torch.int32)
        slots = []
        for i in range(B):
            for p_ in range(n_cached[i], L):
                slots.append(int(tables[i, p_ // 16]) * 16 + p_ % 16)
        T = int(qsl[-1])
        st = {"bm": bm, "n_cached": n_cached, "tables": tables.to(device),
              "lens": lens.to(device), "qsl": qsl.to(device), "max_q": max(nq),
              "slots": torch.tensor(slots, dtype=torch.int64, device=device),
              "q": torch.randn((T, hq, d), generator=g).bfloat16().to(device),
              "k": torch.randn((T, hkv, d), generator=g).bfloat16().to(device),
              "v": torch.randn((T, hkv, d), generator=g).bfloat16().to(device)}
        st["out"] = torch.empty_like(st["q"])
        return st

    def step(st):
        pa.pa_reshape_and_cache(st["k"], st["v"], kc, vc, st["slots"])
        pa.pa_prefill(st["out"], st["q"], kc, vc, st["tables"], st["lens"], st["qsl"],
                      st["max_q"], scale)

    stream = torch.cuda.current_stream(device)
    n = args.steps
    spg = max(k for k in range(1, min(n, 20) + 1) if n % k == 0)
    results = {}
    graphs = []
    # one L2 plan for both modes, from the cached step's distinct bytes (the
    # smaller): the prompt's K/V once, the user tokens' K/V, q, out and the
    # user tokens' K/V sources, all bf16
    t_c = B * user_len
    flush_buf, l2_text = l2_plan(device, ((sys_len + t_c) * hkv * d * 2 + 2 * t_c * hq * d
                                          + 2 * t_c * hkv * d) * 2)
    sampler = ClockSampler(device.index)
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    for mode in ("cached", "full"):
        st = build(mode == "cached")
        for _ in range(args.warmup):
            step(st)
        torch.cuda.synchronize(device)
        if flush_buf is not None:
            one = one_step_runner(lambda st=st: step(st), device, graphs, args.no_graph)
            barrier(world)
            ms = time_each(one, n, flush_buf, stream)
            barrier(world)
            results[mode] = (max_over_ranks(ms, world, device), st)
            continue
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for _ in range(spg):
                step(st)
        gr.replay()
        torch.cuda.synchronize(device)
        graphs.append(gr)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        a.record(stream)
        for _ in range(n // spg):
            gr.replay()
        b.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        results[mode] = (max_over_ranks(a.elapsed_time(b) / n, world, device), st)
    t1 = time.time()
    sampler.stop()
    if pa.pa_device_status(clear=True) != 0:
        raise RuntimeError("a kernel raised a device status bit")
    ms_c, st_c = results["cached"]
    ms_f, st_f = results["full"]
    speedup = ms_f / ms_c
    line = {
        "metric": PREFIX_METRIC, "value": round(speedup, 2), "unit": "x", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(ms_c, 5),
        "us_per_step_cached": round(ms_c * 1e3, 2), "us_per_step_full": round(ms_f * 1e3, 2),
        "cached_tokens_per_request": st_c["n_cached"][0],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (random token ids, N(0,1) K/V/q; no model weights)",
        "config": {"workload": f"{B} requests: the same {sys_len}-token system prompt + "
                               f"{user_len} own tokens, 32/8 heads, d128, bf16",
                   "step": "pa_reshape_and_cache of the uncached tokens + pa_prefill of them",
                   "launch": f"CUDA graph replay, {spg} steps per graph" if flush_buf is None
                             else "stream" if args.no_graph else
                             "CUDA graph replay, 1 step per graph",
                   "l2": l2_text,
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"},
        "pages_context": "the pages quote 4x end-to-end for this scenario (180 ms -> 45 ms, "
                         "serving latency, hardware unstated); this is the attention step alone",
        "gpu_launches": 2 * n * 2, "e2e": None, "cpu_baseline": None, "roofline": None,
        "clocks": sampler.summary(t0, t1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference_prefill(args, world, rank, local):
    """The CPU oracle on a prefill workload: rank 0 alone, a bounded sample per step."""
    if rank != 0:
        return
    spec = wl.PREFILL_SPECS[args.prefill]
    W = wl.make_prefill_workload(spec, 10 + args.prefill, device="cpu")
    # the whole run holds about --ref-seconds of oracle time, whatever --steps
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    sampler = PrefillOracleSampler(W)
    for _ in range(args.warmup):
        sampler.sample(per_step)
    tot_f, tot_s, rows = 0, 0.0, 0
    for _ in range(args.steps):
        f, sec, r = sampler.sample(per_step)
        tot_f, tot_s, rows = tot_f + f, tot_s + sec, rows + r
    value = tot_f / tot_s / 1e12
    cpu = {"value": round(value, 6), "unit": "TFLOP/s", "cores": 1, "host_cpus": os.cpu_count(),
           "kind": "oracle",
           "sample": f"float64 NumPy oracle, {rows} query rows over {args.steps} steps "
                     f"({tot_s:.1f} s), 1 BLAS thread"}
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) K/V/q; no model weights)",
        "config": {"workload": spec.name, "parallelism": "host cores, one thread"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_reference(args, world, rank, local):
    """The CPU oracle as the reference arm: rank 0 alone, a bounded sample per step."""
    if rank != 0:
        return
    spec = wl.SPECS[args.config]
    W = wl.make_workload(spec, args.config, device="cpu")
    # the whole run holds about --ref-seconds of oracle time, whatever --steps
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    cores = os.cpu_count() or 1
    parallel = parallel_oracle_ok(W, cores)
    # every host core (16-bit caches: the pool in shared memory), else one
    sampler = ParallelOracleSampler(W, cores) if parallel else OracleSampler(W, oracle_rows_fn(W))
    try:
        tot_b, tot_s, nseq = 0, 0.0, 0
        if parallel:
            # the workers stay busy across steps: the warm-up and the timed steps
            # are two stretches of wall time (a per-step drain of the pool would
            # cost more than a step's budget)
            sampler.sample(per_step * args.warmup)
            tot_b, tot_s, nseq = sampler.sample(per_step * args.steps)
        else:
            for _ in range(args.warmup):
                sampler.sample(per_step)
            for _ in range(args.steps):
                b, s, k = sampler.sample(per_step)
                tot_b += b
                tot_s += s
                nseq += k
    finally:
        if parallel:
            sampler.close()
    value = tot_b / tot_s / 1e9
    cpu = {"value": round(value, 4), "unit": "GB/s", "cores": cores if parallel else 1,
           "host_cpus": os.cpu_count(), "kind": "oracle",
           "sample": (f"float64 NumPy oracle, {nseq} whole sequences over {args.steps} steps "
                      f"({tot_s:.1f} s of wall time), {cores} worker processes (spawn), "
                      f"1 BLAS thread each" if parallel else
                      f"float64 NumPy oracle, {nseq} sequence samples (all heads, contexts cut "
                      f"to the per-step time budget) over {args.steps} steps "
                      f"({tot_s:.1f} s), 1 BLAS thread")}
    # the same config as the GPU arm's line for this workload and seed
    l2 = l2_text(decode_distinct_bytes(W), device_l2_bytes())
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "strong" if (args.shard == "heads" and world > 1) else "weak",
            "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) K/V/q; no model weights)",
            "config": workload_config(spec, W, l2, world, args.shard),
            "run": {"where": (f"host cores, {cores} processes (rank 0 alone)" if parallel
                              else "host cores, one thread (rank 0 alone)")},
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--config", type=int, default=3, choices=sorted(wl.SPECS),
                   help="the headline decode workload (default: the Llama-3-8B GQA batch)")
    p.add_argument("--also", default="5,4,2",
                   help="other decode workloads timed in the same run, reported under 'also' "
                        "(comma list; '' for none)")
    p.add_argument("--shard", default="seqs", choices=["seqs", "heads"],
                   help="N>1: seqs = one batch per GPU (replicas, weak scaling); heads = the "
                        "KV heads of one batch split over the GPUs (strong scaling)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--partition-size", type=int, default=0)
    p.add_argument("--path", default="append", choices=["append", "separate"],
                   help="append: pa_decode_append (one launch per step); separate: "
                        "pa_reshape_and_cache then pa_decode")
    p.add_argument("--no-alt", action="store_true", help="skip timing the other path")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--ref-seconds", type=float, default=60.0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="issue every call from Python instead of replaying captured steps")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--prefill", type=int, default=0, choices=[0] + sorted(wl.PREFILL_SPECS),
                   help="time a prefill workload (pa_prefill) instead of the decode step")
    p.add_argument("--prefill-kv", default="same", choices=["same", "e4m3"],
                   help="with --prefill: a cache of q's dtype, or E4M3 codes of the same values")
    p.add_argument("--prefix-cache", action="store_true",
                   help="time prefix-cached against full prefill (system-prompt scenario)")
    p.add_argument("--blocks", action="store_true",
                   help="time the block manager (pa_copy_blocks; host step of pa_bm_*)")
    args = p.parse_args(argv)
    args.also = [int(x) for x in args.also.split(",") if x.strip()]
    for c in args.also:
        if c not in wl.SPECS:
            p.error(f"--also: no decode workload {c}")
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.blocks:
        run_blocks(args, world, rank, local)
    elif args.prefix_cache:
        run_prefix_cache(args, world, rank, local)
    elif args.prefill and args.impl == "ours":
        run_prefill(args, world, rank, local)
    elif args.prefill:
        run_reference_prefill(args, world, rank, local)
    elif args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
