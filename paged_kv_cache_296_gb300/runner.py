"""One step of the hot path on the GPU, through the C ABI.

:class:`DecodeStep` holds a decode workload's device-resident state (pool,
tables, lengths, q, the step's new k/v, output, split-KV workspace);
:class:`PrefillStep` the same for a prefill (or chunked prefill) workload.
The pool is the cache: it stays in HBM between steps.
"""

import torch

from . import binding as pa
from .workloads import BLOCK_SIZE


def fill_fp8_pool(pool_src, kv_scale, device, rows_per_call=1 << 16):
    """An E4M3 pool quantised from fp32 values by pa_reshape_and_cache over every slot."""
    nb, bs, _, hkv, d = pool_src.shape
    pool = torch.zeros((nb, bs, 2, hkv, d), dtype=torch.uint8, device=device)
    kc, vc = pa.kv_views(pool)
    src = pool_src.reshape(nb * bs, 2, hkv, d)
    for r0 in range(0, nb * bs, rows_per_call):
        r1 = min(nb * bs, r0 + rows_per_call)
        part = src[r0:r1].to(device)
        slots = torch.arange(r0, r1, dtype=torch.int64, device=device)
        pa.pa_reshape_and_cache(part[:, 0].contiguous(), part[:, 1].contiguous(), kc, vc, slots,
                                kv_scale=kv_scale)
    return pool


class DecodeStep:
    """Device buffers for one workload plus the step that runs on them.

    ``shared``: decode with shared-prefix groups (pa_decode_shared /
    pa_decode_append_shared), each shared block read once for all the
    sequences whose tables hold it.  "auto" (the default) uses them when the
    tables have any (pa_find_shared_prefixes on the host copy of the tables).
    """

    def __init__(self, W, device="cuda", partition_size=0, shared="auto"):
        self.W = W
        self.device = torch.device(device)
        spec = W.spec
        if spec.kv_dtype == "e4m3":
            self.pool = fill_fp8_pool(W.pool_src, W.kv_scale, self.device)
        else:
            # a copy: the step writes into its pool, the workload keeps the drawn values
            self.pool = W.pool.to(self.device, copy=True)
        self.k_cache, self.v_cache = pa.kv_views(self.pool)
        self.q = W.q.to(self.device)
        self.k_new = W.k_new.to(self.device)
        self.v_new = W.v_new.to(self.device)
        self.slot_mapping = W.slot_mapping.to(self.device)
        self.block_tables = W.block_tables.to(self.device)
        self.context_lens = W.context_lens.to(self.device)
        self.out = torch.empty_like(self.q)
        self.partition_size = partition_size
        B, hq, d = self.q.shape
        groups = None
        if shared:
            groups = pa.pa_find_shared_prefixes(W.block_tables, W.context_lens, hq,
                                                spec.num_kv_heads)
            if groups.num_groups == 0:
                if shared != "auto":
                    raise ValueError("shared=True but the tables share no leading blocks")
                groups = None
        self.shared = groups is not None
        self.step_inputs = self.STEP_INPUTS
        if self.shared:
            self.grp_off = groups.offsets.to(self.device)
            self.grp_seq = groups.seqs.to(self.device)
            self.grp_blocks = groups.blocks.to(self.device)
            self.num_groups = groups.num_groups
            self.step_inputs = self.STEP_INPUTS + ("grp_off", "grp_seq", "grp_blocks")
            self.partition_tokens = 0
            nbytes = pa.pa_decode_shared_workspace_size(B, hq, spec.num_kv_heads, d,
                                                        W.max_blocks_per_seq, BLOCK_SIZE,
                                                        self.num_groups)
        else:
            self.partition_tokens = pa.pa_decode_partition_size(
                B, spec.num_kv_heads, W.max_blocks_per_seq, BLOCK_SIZE, partition_size)
            nbytes = pa.pa_decode_workspace_size(B, hq, spec.num_kv_heads, d,
                                                 W.max_blocks_per_seq, BLOCK_SIZE, partition_size)
        self.workspace = pa.alloc_workspace(nbytes, self.device)
        self.kv_scale = W.kv_scale
        self.scale = W.scale

    #: The step's per-call inputs, in the order they are packed by :meth:`stage_inputs`
    #: (a shared-prefix step adds its three group arrays).
    STEP_INPUTS = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")

    @property
    def groups(self):
        return pa.SharedGroups(self.grp_off, self.grp_seq, self.grp_blocks) if self.shared else None

    def stage_inputs(self):
        """Pack the per-step inputs into one device buffer and a pinned host twin.

        Each input becomes a view into a single device byte buffer (sections
        256-byte aligned), so a caller that keeps its step inputs in the
        pinned twin moves all of them with one host-to-device copy.  Returns
        ``(host, device)``, both uint8 of the same size; the host buffer
        already holds the current inputs.
        """
        align = lambda n: (n + 255) // 256 * 256
        names = getattr(self, "step_inputs", self.STEP_INPUTS)
        tensors = [getattr(self, k) for k in names]
        sizes = [t.numel() * t.element_size() for t in tensors]
        total = sum(align(n) for n in sizes)
        dev = torch.empty(total, dtype=torch.uint8, device=self.device)
        host = torch.empty(total, dtype=torch.uint8).pin_memory()
        off = 0
        for name, t, n in zip(names, tensors, sizes):
            view = dev[off:off + n].view(t.dtype).view(t.shape)
            view.copy_(t)
            host[off:off + n].copy_(view.view(torch.uint8).reshape(-1).cpu())
            setattr(self, name, view)
            off += align(n)
        return host, dev

    def launches_per_step(self, path="append"):
        """Kernels one step enqueues.

        "append": one (token write + attention), plus the merge kernel when a
        sequence can span more than one partition (always with the stream-K
        split).  "separate": the write kernel, then the same.
        """
        max_tokens = self.W.max_blocks_per_seq * BLOCK_SIZE
        split = self.partition_tokens == 0 or max_tokens > self.partition_tokens   # 0: stream-K
        n = 1 + (1 if split else 0)
        return n + (1 if path == "separate" else 0)

    def append(self):
        """The whole step in one call: pa_decode_append (or its shared-prefix form)."""
        if self.shared:
            pa.pa_decode_append_shared(self.out, self.q, self.k_new, self.v_new,
                                       self.slot_mapping, self.k_cache, self.v_cache,
                                       self.block_tables, self.context_lens, self.scale,
                                       self.groups, kv_scale=self.kv_scale,
                                       workspace=self.workspace)
            return self.out
        pa.pa_decode_append(self.out, self.q, self.k_new, self.v_new, self.slot_mapping,
                            self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                            self.scale, kv_scale=self.kv_scale,
                            partition_size=self.partition_size, workspace=self.workspace)
        return self.out

    def write(self):
        pa.pa_reshape_and_cache(self.k_new, self.v_new, self.k_cache, self.v_cache,
                                self.slot_mapping, kv_scale=self.kv_scale)

    def decode(self):
        if self.shared:
            pa.pa_decode_shared(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                self.context_lens, self.scale, self.groups,
                                kv_scale=self.kv_scale, workspace=self.workspace)
            return
        pa.pa_decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                     self.context_lens, self.scale, kv_scale=self.kv_scale,
                     partition_size=self.partition_size, workspace=self.workspace)

    def step(self):
        self.write()
        self.decode()
        return self.out


def step_bytes(W):
    """Algorithmic bytes of one step: (attended K/V + q + out, attended K/V, new-token bytes).

    Attended K/V counts every token of every sequence once per KV head:
    ``sum_i L_i * Hkv * D * 2 * elt``.  The new-token bytes are the write's:
    k_new/v_new read in the q dtype plus their cache rows written.
    """
    spec = W.spec
    elt = 1 if spec.kv_dtype == "e4m3" else 2
    kv = int(W.context_lens.to(torch.int64).sum()) * spec.num_kv_heads * spec.head_size * 2 * elt
    qo = 2 * W.q.numel() * W.q.element_size()
    n_new = int((W.slot_mapping >= 0).sum())
    new = n_new * spec.num_kv_heads * spec.head_size * 2 * (W.q.element_size() + elt)
    return kv + qo, kv, new


def unique_kv_bytes(W):
    """K/V bytes of distinct physical blocks' live tokens (shared prefixes counted once)."""
    spec = W.spec
    elt = 1 if spec.kv_dtype == "e4m3" else 2
    seen = set()
    total = 0
    bt = W.block_tables.cpu().numpy()
    for i, L in enumerate(W.context_lens.cpu().tolist()):
        for j in range(-(-L // BLOCK_SIZE)):
            b = int(bt[i, j])
            n = min(BLOCK_SIZE, L - j * BLOCK_SIZE)
            key = b
            if key in seen:
                continue
            seen.add(key)
            total += n
    return total * spec.num_kv_heads * spec.head_size * 2 * elt


class PrefillStep:
    """Device buffers for one prefill workload: the step writes the query
    tokens' K/V into the pool (pa_reshape_and_cache), then runs pa_prefill."""

    #: Per-step inputs, packed by :meth:`stage_inputs` for host-to-device copies.
    STEP_INPUTS = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens",
                   "query_start_loc")

    def __init__(self, W, device="cuda", kv_dtype=None):
        """``kv_dtype="e4m3"``: an E4M3 cache holding the workload's pool values
        (written through pa_reshape_and_cache with kv_scale = amax / 448 over
        them and the step's new K/V); else the workload's 16-bit pool."""
        self.W = W
        self.device = torch.device(device)
        for name in self.STEP_INPUTS:
            setattr(self, name, getattr(W, name).to(self.device))
        self.kv_scale = 1.0
        if kv_dtype == "e4m3":
            src = W.pool.to(self.device).float()
            amax = float(torch.nan_to_num(src, nan=0.0).abs().max())
            if self.k_new.numel():
                amax = max(amax, float(self.k_new.float().abs().max()),
                           float(self.v_new.float().abs().max()))
            self.kv_scale = amax / 448.0
            nb, bs, _, hkv, d = src.shape
            self.pool = torch.zeros((nb, bs, 2, hkv, d), dtype=torch.uint8, device=self.device)
            self.k_cache, self.v_cache = pa.kv_views(self.pool)
            flat = src.reshape(nb * bs, 2, hkv, d)
            slots = torch.arange(nb * bs, dtype=torch.int64, device=self.device)
            pa.pa_reshape_and_cache(flat[:, 0].contiguous(), flat[:, 1].contiguous(),
                                    self.k_cache, self.v_cache, slots, kv_scale=self.kv_scale)
            del src, flat
        else:
            self.pool = W.pool.to(self.device, copy=True)
            self.k_cache, self.v_cache = pa.kv_views(self.pool)
        self.out = torch.empty_like(self.q)
        self.max_query_len = W.max_query_len
        self.scale = W.scale

    stage_inputs = DecodeStep.stage_inputs

    def step(self):
        if self.q.shape[0]:
            pa.pa_reshape_and_cache(self.k_new, self.v_new, self.k_cache, self.v_cache,
                                    self.slot_mapping, kv_scale=self.kv_scale)
        pa.pa_prefill(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                      self.context_lens, self.query_start_loc, self.max_query_len, self.scale,
                      kv_scale=self.kv_scale)
        return self.out

    launches_per_step = 2


def prefill_flops(W):
    """Causal attention FLOPs of one prefill step: for every query (position p)
    and query head, 2*D multiply-adds for each of the p + 1 scores and 2*D for
    the weighted sum of as many V rows: 4 * D * Hq * sum (p + 1)."""
    lens = W.context_lens.cpu().long().tolist()
    qsl = W.query_start_loc.cpu().long().tolist()
    keys = 0
    for i, L in enumerate(lens):
        n = qsl[i + 1] - qsl[i]
        keys += (L - n) * n + n * (n + 1) // 2
    return 4 * W.spec.head_size * W.spec.num_q_heads * keys
