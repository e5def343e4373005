"""Seeded synthetic inputs for paged decode: the one module both sides consume.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no attention, no quantisation, no slot decoding).  The
CUDA library and the CPU oracle each take what it returns and compute
independently.

Workloads follow the shapes of the pages' deployments ("vLLM 部署深度指南":
16-token blocks, section PagedAttention 方案; the pool layout
``[num_blocks, block_size, 2, num_kv_heads, head_size]``, section 代码层面理解;
Llama-class head shapes; shared prefixes, "vLLM GitHub 项目…" section 二 item 4).
No model weights, prompts or datasets are involved: every value is N(0, 1).

Draw order for a seed: context lengths -> physical block permutation ->
pool contents -> q -> the step's new k/v.  The generator is torch's seeded
CPU generator by default, so the same seed gives the same bytes on any
machine; ``device="cuda"`` draws on the GPU instead (faster, different
numbers) for timing runs that are not compared value by value.
"""

from dataclasses import dataclass, field, replace
import math

import numpy as np
import torch

BLOCK_SIZE = 16

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.uint8,
               "f32": torch.float32}

#: NaN bit patterns used to poison memory the path must never read.
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F}


@dataclass
class Spec:
    """Shape and distribution of one synthetic decode batch."""
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    q_dtype: str                      # "f16" | "bf16"
    kv_dtype: str                     # "f16" | "bf16" | "e4m3"
    lens: tuple                       # ("fixed", [..]) | ("uniform", lo, hi) |
                                      # ("loguniform", lo, hi) | ("shared_prefix", prompts, samples, prefix, suffix_hi)
    pool: tuple = ("factor", 1.25)    # ("fixed", num_blocks) | ("factor", f)
    partition_size: int = 512
    block_size: int = BLOCK_SIZE


#: The five benchmark workloads.  Seeds 1..5 belong to them.
SPECS = {
    1: Spec("tiny: 4 seqs, ctx {1,15,16,17}, 4/4 heads, d64, fp16",
            4, 4, 4, 64, "f16", "f16", ("fixed", [1, 15, 16, 17]), ("fixed", 64)),
    2: Spec("Llama-2-7B MHA decode: 64 seqs, ctx U[128,2048], 32/32 heads, d128, fp16",
            64, 32, 32, 128, "f16", "f16", ("uniform", 128, 2048)),
    3: Spec("Llama-3-8B GQA decode: 256 seqs, ctx logU[512,4096], 32/8 heads, d128, bf16",
            256, 32, 8, 128, "bf16", "bf16", ("loguniform", 512, 4096)),
    4: Spec("shared-prefix sampling: 16 prompts x 8 samples, 1024-token prefix, 32/8 heads, d128, fp16",
            128, 32, 8, 128, "f16", "f16", ("shared_prefix", 16, 8, 1024, 256)),
    5: Spec("long-context split-KV: 8 seqs, ctx U[16384,32768], 64/8 heads, d128, bf16 q, fp8-e4m3 KV",
            8, 64, 8, 128, "bf16", "e4m3", ("uniform", 16384, 32768)),
}


@dataclass
class Workload:
    """One decode step's inputs.  Tensors live on ``device``.

    ``pool`` is the cache state before the step (for e4m3, ``None`` until a
    side quantises ``pool_src``).  ``pool_src`` (e4m3 only) holds the fp32
    values the whole pool is filled from.  ``k_new``/``v_new``/``slot_mapping``
    are the step's write; ``context_lens`` already count the new token.
    """
    spec: Spec
    seed: int
    context_lens: torch.Tensor        # int32 [B]
    block_tables: torch.Tensor        # int32 [B, max_blocks]
    num_blocks: int
    pool: torch.Tensor                # [NB, BS, 2, Hkv, D] (f16/bf16) or None (e4m3)
    pool_src: torch.Tensor            # f32 [NB, BS, 2, Hkv, D] (e4m3 only) or None
    q: torch.Tensor                   # [B, Hq, D] q_dtype
    k_new: torch.Tensor               # [B, Hkv, D] q_dtype
    v_new: torch.Tensor               # [B, Hkv, D] q_dtype
    slot_mapping: torch.Tensor        # int64 [B]
    kv_scale: float
    scale: float
    shared_blocks: int = 0            # physical blocks referenced by more than one table
    extra: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self):
        return self.block_tables.shape[1]


def _draw_lens(spec, gen):
    kind = spec.lens[0]
    if kind == "fixed":
        return np.array(spec.lens[1], dtype=np.int64), None
    if kind == "uniform":
        lo, hi = spec.lens[1], spec.lens[2]
        lens = torch.randint(lo, hi + 1, (spec.num_seqs,), generator=gen)
        return lens.numpy().astype(np.int64), None
    if kind == "loguniform":
        lo, hi = spec.lens[1], spec.lens[2]
        u = torch.rand((spec.num_seqs,), generator=gen, dtype=torch.float64).numpy()
        lens = np.rint(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
        return np.clip(lens, lo, hi).astype(np.int64), None
    if kind == "shared_prefix":
        prompts, samples, prefix, suffix_hi = spec.lens[1:]
        # Tokens already cached after the prefix, per sample; the step's new
        # token extends that private suffix, so context = prefix + suffix + 1.
        suffix = torch.randint(0, suffix_hi + 1, (prompts * samples,), generator=gen).numpy()
        return (prefix + suffix + 1).astype(np.int64), (prompts, samples, prefix)
    raise ValueError(kind)


def _ceil_div(a, b):
    return -(-a // b)


def make_workload(spec, seed, device="cpu", poison=False, table_garbage=False):
    """Draw one decode step for ``spec``.

    ``poison``: fill every pool slot the step must not read (free blocks, the
    unused tail of each sequence's last block, the slots the step is about to
    write) with NaN, so that any stray read shows up as NaN in the output.
    Otherwise those slots hold N(0, 1) like the rest.
    ``table_garbage``: fill block-table entries past each sequence's last block
    with out-of-range ids instead of -1.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    bs = spec.block_size
    hkv, d = spec.num_kv_heads, spec.head_size

    lens, shared = _draw_lens(spec, gen)
    B = len(lens)
    assert B == spec.num_seqs
    nblk = [_ceil_div(int(L), bs) for L in lens]
    max_blocks = max(1, max(nblk))

    # Physical blocks each table needs (shared prefixes counted once).
    if shared is None:
        needed = sum(nblk)
    else:
        prompts, samples, prefix = shared
        pblk = prefix // bs
        needed = prompts * pblk + sum(n - pblk for n in nblk)
    if spec.pool[0] == "fixed":
        num_blocks = spec.pool[1]
    else:
        num_blocks = int(math.ceil(spec.pool[1] * needed))
    assert num_blocks >= needed
    perm = torch.randperm(num_blocks, generator=gen).numpy().astype(np.int64)

    tables = np.full((B, max_blocks), -1, dtype=np.int64)
    nxt = 0
    if shared is None:
        for i in range(B):
            tables[i, :nblk[i]] = perm[nxt:nxt + nblk[i]]
            nxt += nblk[i]
    else:
        prompts, samples, prefix = shared
        pblk = prefix // bs
        for p in range(prompts):
            pre = perm[nxt:nxt + pblk]
            nxt += pblk
            for s in range(samples):
                i = p * samples + s
                tables[i, :pblk] = pre
                priv = nblk[i] - pblk
                tables[i, pblk:nblk[i]] = perm[nxt:nxt + priv]
                nxt += priv
    if table_garbage:
        for i in range(B):
            junk = torch.randint(-(1 << 30), 1 << 30, (max_blocks - nblk[i],), generator=gen).numpy()
            junk = np.where((junk >= 0) & (junk < num_blocks), junk + num_blocks, junk)
            tables[i, nblk[i]:] = junk

    # The slot each sequence's new token (its last, index L-1) goes to; an
    # empty sequence writes nothing (slot -1, the padding convention).
    last = lens - 1
    slots = np.array([tables[i, last[i] // bs] * bs + last[i] % bs if lens[i] > 0 else -1
                      for i in range(B)], dtype=np.int64)

    # Which pool slots hold live (cached) tokens before the step.
    live = None
    if poison:
        live = np.zeros((num_blocks, bs), dtype=bool)
        for i in range(B):
            for j in range(int(lens[i]) - 1):
                live[tables[i, j // bs], j % bs] = True

    shape = (num_blocks, bs, 2, hkv, d)
    if spec.kv_dtype == "e4m3":
        pool_src = _randn(shape, torch.float32, gen, device)
        if poison:
            dead = torch.from_numpy(~live).to(device)
            pool_src[dead] = float("nan")
        pool = None
    else:
        pool = _randn(shape, TORCH_DTYPE[spec.kv_dtype], gen, device)
        if poison:
            dead = torch.from_numpy(~live).to(device)
            pool[dead] = float("nan")
        pool_src = None

    qd = TORCH_DTYPE[spec.q_dtype]
    q = _randn((B, spec.num_q_heads, d), qd, gen, device)
    k_new = _randn((B, hkv, d), qd, gen, device)
    v_new = _randn((B, hkv, d), qd, gen, device)

    kv_scale = 1.0
    if spec.kv_dtype == "e4m3":
        # Per-tensor calibration done by the caller before the path runs:
        # the largest finite magnitude the cache will hold, over the E4M3 maximum.
        amax = max(float(torch.nan_to_num(pool_src, nan=0.0).abs().max()),
                   float(k_new.float().abs().max()), float(v_new.float().abs().max()))
        kv_scale = amax / 448.0

    n_shared = 0
    if shared is not None:
        n_shared = shared[0] * (shared[2] // bs)

    return Workload(
        spec=spec, seed=seed,
        context_lens=torch.from_numpy(lens.astype(np.int32)).to(device),
        block_tables=torch.from_numpy(tables.astype(np.int32)).to(device),
        num_blocks=num_blocks, pool=pool, pool_src=pool_src,
        q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(slots).to(device),
        kv_scale=kv_scale, scale=1.0 / math.sqrt(d), shared_blocks=n_shared,
    )


def kv_head_range(num_kv_heads, rank, world):
    """KV heads ``[h0, h1)`` that rank ``rank`` of ``world`` holds when a batch's
    KV heads are split over GPUs in equal contiguous slices ("vLLM 部署深度指南",
    分布式推理: tensor parallelism over the GPUs of one node)."""
    if world < 1 or not 0 <= rank < world or num_kv_heads % world:
        raise ValueError(f"{num_kv_heads} KV heads do not split over {world} ranks")
    per = num_kv_heads // world
    return rank * per, (rank + 1) * per


def shard_heads(W, rank, world):
    """Rank ``rank``'s part of decode workload ``W`` when its KV heads are split
    over ``world`` GPUs: KV heads ``[h0, h1)`` of the pool and of the new
    tokens, and the query heads that read them, ``[h0*G, h1*G)`` (query head h
    reads KV head h // G).  Lengths, tables, slots and kv_scale are the whole
    batch's.  Every rank's slice is an independent decode; the outputs
    concatenated over ranks along the head axis are the whole batch's."""
    spec = W.spec
    h0, h1 = kv_head_range(spec.num_kv_heads, rank, world)
    g = spec.num_q_heads // spec.num_kv_heads
    sub = replace(spec, name=f"{spec.name} [kv heads {h0}..{h1 - 1}]",
                  num_q_heads=(h1 - h0) * g, num_kv_heads=h1 - h0)
    part = lambda t: None if t is None else t[:, :, :, h0:h1, :].contiguous()
    return replace(W, spec=sub,
                   pool=part(W.pool), pool_src=part(W.pool_src),
                   q=W.q[:, h0 * g:h1 * g, :].contiguous(),
                   k_new=W.k_new[:, h0:h1, :].contiguous(),
                   v_new=W.v_new[:, h0:h1, :].contiguous(),
                   extra=dict(W.extra, kv_heads=(h0, h1)))


def _randn(shape, dtype, gen, device):
    """N(0, 1) values of ``dtype``: drawn in float32 on the CPU generator, then cast."""
    if device == "cpu":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        return x.to(dtype)
    # GPU draw: seed a device generator from the CPU stream so runs stay reproducible.
    dgen = torch.Generator(device=device)
    dgen.manual_seed(int(torch.randint(0, 1 << 62, (1,), generator=gen)))
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(generator=dgen)
    return x.to(dtype)


def random_spec(seed, head_size=None, group=None, kv_dtype=None, max_len=70, max_seqs=5):
    """A small random shape for parity sweeps: few sequences, ragged lengths."""
    r = np.random.default_rng(seed)
    d = head_size or int(r.choice([64, 128]))
    g = group or int(r.choice([1, 2, 4, 8]))
    hkv = int(r.choice([1, 2, 3]))
    kvd = kv_dtype or str(r.choice(["f16", "bf16", "e4m3"]))
    qd = kvd if kvd != "e4m3" else str(r.choice(["f16", "bf16"]))
    B = int(r.integers(1, max_seqs + 1))
    lens = [int(x) for x in r.integers(0, max_len + 1, B)]
    lens[0] = max(lens[0], 1)
    return Spec(f"random seed {seed}", B, hkv * g, hkv, d, qd, kvd, ("fixed", lens),
                ("factor", 1.5), partition_size=int(r.choice([16, 32, 64, 512])))


# --------------------------------------------------------------------------
# Prefill (a prompt, or a chunk of one, per sequence)
# --------------------------------------------------------------------------

@dataclass
class PrefillSpec:
    """Shape of one synthetic prefill batch.

    ``context``: the sequences' lengths after the step, ``("fixed", [..])`` or
    ``("uniform", lo, hi)``.  ``query``: how many of each sequence's last tokens
    are this step's queries: ``("all",)`` (a whole prompt), ``("chunk", n)``
    (min(n, L) tokens: chunked prefill over an already cached prefix) or
    ``("fixed", [..])``.
    """
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    dtype: str                        # "f16" | "bf16" (q, cache, out)
    context: tuple
    query: tuple
    pool: tuple = ("factor", 1.25)
    block_size: int = BLOCK_SIZE


#: Prefill workloads (Llama-3-8B-shaped heads).  Seeds 11.. belong to them.
PREFILL_SPECS = {
    1: PrefillSpec("prefill: 4 prompts of 2048 tokens, 32/8 heads, d128, bf16",
                   4, 32, 8, 128, "bf16", ("fixed", [2048] * 4), ("all",)),
    2: PrefillSpec("chunked prefill: 16 seqs, context U[2048,8192], 512-token chunks, "
                   "32/8 heads, d128, bf16",
                   16, 32, 8, 128, "bf16", ("uniform", 2048, 8192), ("chunk", 512)),
}


@dataclass
class PrefillWorkload:
    """One prefill step's inputs.  ``pool`` is the cache before the step's write
    of the query tokens' K/V (``k_new``/``v_new`` at ``slot_mapping``)."""
    spec: PrefillSpec
    seed: int
    context_lens: torch.Tensor        # int32 [B]
    query_start_loc: torch.Tensor     # int32 [B + 1]
    block_tables: torch.Tensor        # int32 [B, max_blocks]
    num_blocks: int
    pool: torch.Tensor                # [NB, BS, 2, Hkv, D]
    q: torch.Tensor                   # [T, Hq, D]
    k_new: torch.Tensor               # [T, Hkv, D]
    v_new: torch.Tensor               # [T, Hkv, D]
    slot_mapping: torch.Tensor        # int64 [T]
    scale: float

    @property
    def max_blocks_per_seq(self):
        return self.block_tables.shape[1]

    @property
    def max_query_len(self):
        qsl = self.query_start_loc.cpu()
        return int((qsl[1:] - qsl[:-1]).max()) if len(qsl) > 1 else 0


def make_prefill_workload(spec, seed, device="cpu", poison=False):
    """Draw one prefill step for ``spec``.

    Draw order: context lengths -> query counts -> block permutation -> pool ->
    q -> the query tokens' k/v.  ``poison``: NaN in every slot the step must
    not read before writing it (free blocks, tails, the query tokens' own
    slots, which the step's write fills).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    bs = spec.block_size
    hkv, d = spec.num_kv_heads, spec.head_size
    B = spec.num_seqs
    if spec.context[0] == "fixed":
        lens = np.array(spec.context[1], dtype=np.int64)
    else:
        lens = torch.randint(spec.context[1], spec.context[2] + 1, (B,), generator=gen).numpy()
        lens = lens.astype(np.int64)
    assert len(lens) == B
    if spec.query[0] == "all":
        nq = lens.copy()
    elif spec.query[0] == "chunk":
        nq = np.minimum(lens, spec.query[1])
    else:
        nq = np.array(spec.query[1], dtype=np.int64)
    assert np.all((nq >= 0) & (nq <= lens))
    qsl = np.concatenate([[0], np.cumsum(nq)]).astype(np.int64)
    T = int(qsl[-1])

    nblk = [_ceil_div(int(L), bs) for L in lens]
    max_blocks = max(1, max(nblk))
    needed = sum(nblk)
    num_blocks = spec.pool[1] if spec.pool[0] == "fixed" else int(math.ceil(spec.pool[1] * needed))
    num_blocks = max(num_blocks, needed, 1)
    perm = torch.randperm(num_blocks, generator=gen).numpy().astype(np.int64)
    tables = np.full((B, max_blocks), -1, dtype=np.int64)
    nxt = 0
    for i in range(B):
        tables[i, :nblk[i]] = perm[nxt:nxt + nblk[i]]
        nxt += nblk[i]

    slots = np.empty(T, dtype=np.int64)
    for i in range(B):
        for t in range(int(nq[i])):
            pos = int(lens[i] - nq[i] + t)
            slots[qsl[i] + t] = tables[i, pos // bs] * bs + pos % bs

    shape = (num_blocks, bs, 2, hkv, d)
    dt = TORCH_DTYPE[spec.dtype]
    pool = _randn(shape, dt, gen, device)
    if poison:
        live = np.zeros((num_blocks, bs), dtype=bool)
        for i in range(B):
            for j in range(int(lens[i] - nq[i])):
                live[tables[i, j // bs], j % bs] = True
        pool[torch.from_numpy(~live).to(device)] = float("nan")
    q = _randn((T, spec.num_q_heads, d), dt, gen, device)
    k_new = _randn((T, hkv, d), dt, gen, device)
    v_new = _randn((T, hkv, d), dt, gen, device)
    return PrefillWorkload(
        spec=spec, seed=seed,
        context_lens=torch.from_numpy(lens.astype(np.int32)).to(device),
        query_start_loc=torch.from_numpy(qsl.astype(np.int32)).to(device),
        block_tables=torch.from_numpy(tables.astype(np.int32)).to(device),
        num_blocks=num_blocks, pool=pool, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(slots).to(device), scale=1.0 / math.sqrt(d))
