"""pa_decode_noalloc: decode with the library's fixed scratch instead of a caller workspace.

This entry point serves callers that cannot allocate device memory -- an
extension that its host runtime gives only input and output buffers, or a
serving loop that must not call cudaMalloc mid-flight because the call can
synchronise the device and eat into a memory budget fixed at start-up.  Its
output must match pa_decode's on the same inputs.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import pytest
import torch

from paged_kv_cache_296_gb300 import binding as pa
from paged_kv_cache_296_gb300 import workloads as wl
from paged_kv_cache_296_gb300.runner import DecodeStep



def test_rejects_sizes_beyond_the_fixed_scratch():
    """Host-side check, no GPU needed: too much scratch -> PA_ERR_WORKSPACE, nothing launched."""
    from paged_kv_cache_296_gb300 import build
    build()
    lib = pa.load()
    fake = ctypes.c_void_p(0x10000)
    # 4096 sequences x 64 heads x 64 partitions of 512 tokens: ~8.7 GB of partials.
    need = lib.pa_decode_workspace_size(4096, 64, 8, 128, 2048, 16, 512)
    assert need > pa.DECODE_NOALLOC_SCRATCH_BYTES
    st = lib.pa_decode_noalloc(fake, fake, fake, fake, fake, fake, 4096, 2048, 100000, 64, 8, 128,
                               16, 0.088, pa.PA_BF16, pa.PA_E4M3, 0.01, 512, ctypes.c_void_p(0))
    assert st == 3
    assert "scratch" in pa.pa_last_error()


def _compare_once(W, partition_size=0):
    """Run pa_decode (caller workspace) and pa_decode_noalloc on the same device
    state.  Both run the same kernels with the same partition plan on the same
    inputs, so their outputs must agree bit for bit."""
    S = DecodeStep(W, device="cuda", partition_size=partition_size)
    assert S.workspace is not None, "the batch must use split-KV scratch"
    S.write()
    S.decode()
    want = S.out.clone()
    got = torch.empty_like(S.out)
    pa.pa_decode_noalloc(got, S.q, S.k_cache, S.v_cache, S.block_tables, S.context_lens,
                         S.scale, kv_scale=S.kv_scale, partition_size=S.partition_size)
    torch.cuda.synchronize()
    assert torch.isfinite(got.float()).all()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
        (got.float() - want.float()).abs().max().item()


@pytest.mark.gpu
def test_noalloc_matches_pa_decode_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    pa.load()
    pa.pa_device_status(clear=True)
    # Call 1: fp8-E4M3 cache, long contexts, 8 query heads per KV head (16 partitions).
    long_fp8 = wl.Spec("long fp8", 4, 64, 8, 128, "bf16", "e4m3", ("uniform", 4096, 8192))
    _compare_once(wl.make_workload(long_fp8, 501, device="cuda"))
    # Call 2: fp16 MHA batch with a different partition count; it starts from
    # whatever call 1 left in the shared scratch.
    mha = wl.Spec("mha fp16", 16, 32, 32, 128, "f16", "f16", ("uniform", 128, 2048))
    _compare_once(wl.make_workload(mha, 502, device="cuda"), partition_size=256)
    assert pa.pa_device_status(clear=True) == 0
