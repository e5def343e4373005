"""The C ABI on the host (CPU only): the library loads, exports every symbol
include/pa.h declares, and rejects bad arguments before touching the GPU."""

import ctypes
import os
import re

import pytest

from paged_kv_cache_296_gb300 import binding as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_296_gb300 import build
    build()
    return pa.load()


def header_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = header_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_decode_workspace_size", "pa_gather_kv",
              "pa_check_tables", "pa_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    assert set(header_functions()) == set(pa.SIGNATURES), "binding and header disagree"


def test_version(lib):
    assert pa.pa_version() >= 100


FAKE = ctypes.c_void_p(0x10000)        # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x10008)
NULL = ctypes.c_void_p(0)


def decode_args(**over):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, B=4, mb=8, nb=64, hq=8, hkv=2,
             d=128, bs=16, scale=0.1, qd=pa.PA_F16, kvd=pa.PA_F16, kvs=1.0, part=0, ws=NULL,
             wsb=0, stream=NULL)
    a.update(over)
    return [a[k] for k in ("out", "q", "k", "v", "bt", "cl", "B", "mb", "nb", "hq", "hkv", "d",
                           "bs", "scale", "qd", "kvd", "kvs", "part", "ws", "wsb", "stream")]


@pytest.mark.parametrize("over,status", [
    (dict(out=NULL), 1),
    (dict(q=MISALIGNED), 1),
    (dict(d=96), 2),
    (dict(bs=32), 2),
    (dict(hq=6, hkv=4), 1),
    (dict(hq=32, hkv=2), 2),             # 16 query heads per KV head
    (dict(qd=pa.PA_E4M3), 2),
    (dict(kvd=pa.PA_BF16), 2),           # cache dtype differs from q and is not E4M3
    (dict(kvd=pa.PA_E4M3, kvs=0.0), 1),
    (dict(kvd=pa.PA_E4M3, kvs=float("inf")), 1),
    (dict(scale=float("nan")), 1),
    (dict(part=24), 1),                  # not a multiple of 16
    (dict(mb=100, part=512), 3),         # 1600 tokens > one 512-token partition: needs workspace
    (dict(nb=0), 1),
    (dict(B=-1), 1),
    (dict(B=70000), 2),
])
def test_decode_rejects_bad_arguments(lib, over, status):
    st = lib.pa_decode(*decode_args(**over))
    assert st == status
    assert pa.pa_last_error() != ""


def test_decode_workspace_must_be_aligned(lib):
    need = lib.pa_decode_workspace_size(4, 8, 2, 128, 100, 16, 0)
    st = lib.pa_decode(*decode_args(mb=100, ws=ctypes.c_void_p(0x10010), wsb=need))
    assert st == 1


def test_decode_zero_sequences_is_a_no_op(lib):
    assert lib.pa_decode(*decode_args(B=0, out=NULL, q=NULL)) == 0
    assert pa.pa_last_error() == ""


def test_workspace_size(lib):
    al = lambda x: (x + 255) // 256 * 256
    plan = 256                              # where a balanced split records its size
    # 64 x 32 (sequence, KV head) pairs: enough CTAs, no split below 8192 tokens, no workspace
    assert lib.pa_decode_workspace_size(64, 32, 32, 128, 128, 16, 0) == 0
    assert pa.pa_decode_partition_size(64, 32, 128) == 2048
    # 8 x 8 pairs: a balanced split (0), chosen on the device; the workspace
    # covers its smallest partition, 512 tokens: 32768 / 512 = 64 partitions
    assert pa.pa_decode_partition_size(8, 8, 2048) == 0
    rows = 8 * 64 * 64
    assert lib.pa_decode_workspace_size(8, 64, 8, 128, 2048, 16, 0) == \
        2 * al(rows * 4) + al(rows * 128 * 4) + plan
    # explicit sizes: 128 blocks = 2048 tokens = 4 partitions of 512
    rows = 64 * 32 * 4
    assert lib.pa_decode_workspace_size(64, 32, 32, 128, 128, 16, 512) == \
        2 * al(rows * 4) + al(rows * 128 * 4) + plan
    assert lib.pa_decode_workspace_size(64, 32, 32, 128, 128, 16, 256) == \
        2 * al(rows * 2 * 4) + al(rows * 2 * 128 * 4) + plan
    assert lib.pa_decode_workspace_size(64, 32, 32, 128, 128, 15, 0) == 0   # invalid block size
    # shared prefixes: cut partials of up to 1024 CTAs x 2 slots x (2 KV heads x
    # 32 columns), whole partials (prefix and suffix) per (sequence, query head),
    # the plan (8 ints + 8 per sequence)
    cut = 1024 * 2 * 64
    whole = 2 * 128 * 32
    assert lib.pa_decode_shared_workspace_size(128, 32, 8, 128, 81, 16, 16) == \
        2 * al(cut * 4) + al(cut * 128 * 4) + 2 * al(whole * 4) + al(whole * 128 * 4) \
        + al((8 + 8 * 128) * 4)
    # no groups: pa_decode's own choice and workspace
    assert lib.pa_decode_shared_workspace_size(8, 64, 8, 128, 2048, 16, 0) == \
        lib.pa_decode_workspace_size(8, 64, 8, 128, 2048, 16, 0)
    assert lib.pa_decode_shared_workspace_size(1025, 32, 8, 128, 81, 16, 1) == 0  # too many seqs
    assert lib.pa_decode_shared_workspace_size(8, 32, 8, 128, 81, 16, 1025) == 0  # too many groups
    # the library's choice
    assert pa.pa_decode_partition_size(4, 4, 2) == 32            # short: one partition
    assert pa.pa_decode_partition_size(1, 1, 100000) == 0        # few pairs: balanced split
    assert pa.pa_decode_partition_size(1024, 8, 4096) == 8192    # many pairs, 65536 tokens: capped
    assert pa.pa_decode_partition_size(64, 8, 128, partition_size=48) == 48
    assert pa.pa_decode_partition_size(64, 8, 128, partition_size=40) == -1


def cache_args(**over):
    a = dict(k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, sm=FAKE, n=4, stride=0, nb=64, hkv=2, d=128,
             bs=16, sd=pa.PA_F16, kd=pa.PA_F16, kvs=1.0, stream=NULL)
    a.update(over)
    return [a[k] for k in ("k", "v", "kc", "vc", "sm", "n", "stride", "nb", "hkv", "d", "bs",
                           "sd", "kd", "kvs", "stream")]


@pytest.mark.parametrize("over,status", [
    (dict(k=NULL), 1),
    (dict(kc=MISALIGNED), 1),
    (dict(sm=ctypes.c_void_p(0x10004)), 1),
    (dict(n=-1), 1),
    (dict(d=80), 2),
    (dict(bs=8), 2),
    (dict(sd=pa.PA_BF16), 2),                      # 16-bit cache from another dtype
    (dict(kd=pa.PA_F32, sd=pa.PA_F32), 2),
    (dict(kd=pa.PA_E4M3, sd=pa.PA_E4M3), 2),
    (dict(kd=pa.PA_E4M3, kvs=-1.0), 1),
    (dict(stride=100), 1),                         # smaller than Hkv*D
    (dict(stride=260), 1),                         # 520 bytes: not a multiple of 16
    (dict(nb=-5), 1),
])
def test_reshape_and_cache_rejects_bad_arguments(lib, over, status):
    assert lib.pa_reshape_and_cache(*cache_args(**over)) == status
    assert pa.pa_last_error() != ""


def test_reshape_and_cache_zero_tokens_is_a_no_op(lib):
    assert lib.pa_reshape_and_cache(*cache_args(n=0, k=NULL, v=NULL)) == 0


def test_gather_and_check_reject_bad_arguments(lib):
    st = lib.pa_gather_kv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 4, 8, 64, 2, 128, 16,
                          pa.PA_F16, NULL)
    assert st == 1
    st = lib.pa_gather_kv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, 64, 2, 128, 16,
                          pa.PA_F32, NULL)
    assert st == 2
    assert lib.pa_check_tables(FAKE, FAKE, FAKE, 4, 4, 8, 64, 16, NULL, NULL, NULL) == 1
    assert lib.pa_check_tables(FAKE, FAKE, FAKE, -1, 4, 8, 64, 16, FAKE, NULL, NULL) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("paged_kv_cache_296_gb300.binding")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError, match="missing"):
            mod.load(str(tmp_path / "nope.so"))
    finally:
        mod._lib = saved


def test_decode_append_requires_token_buffers(lib):
    args = decode_args()
    # pa_decode_append(out, q, k_new, v_new, slot_mapping, src_stride, k_cache, v_cache, ...)
    a = [args[0], args[1], NULL, FAKE, FAKE, 0] + args[2:]
    assert lib.pa_decode_append(*a) == 1
    a = [args[0], args[1], FAKE, FAKE, FAKE, 100] + args[2:]     # stride < Hkv*D
    assert lib.pa_decode_append(*a) == 1
    a = [args[0], args[1], MISALIGNED, FAKE, FAKE, 0] + args[2:]
    assert lib.pa_decode_append(*a) == 1
    a = [args[0], args[1], FAKE, FAKE, ctypes.c_void_p(0x10004), 0] + args[2:]
    assert lib.pa_decode_append(*a) == 1


def prefill_args(**over):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, qsl=FAKE, B=4, mq=64, mb=8, nb=64,
             hq=8, hkv=2, d=128, bs=16, scale=0.1, dt=pa.PA_F16, kvdt=pa.PA_F16, kvs=1.0,
             stream=NULL)
    a.update(over)
    return [a[k] for k in ("out", "q", "k", "v", "bt", "cl", "qsl", "B", "mq", "mb", "nb", "hq",
                           "hkv", "d", "bs", "scale", "dt", "kvdt", "kvs", "stream")]


@pytest.mark.parametrize("over,status", [
    (dict(out=NULL), 1),
    (dict(qsl=NULL), 1),
    (dict(q=MISALIGNED), 1),
    (dict(qsl=ctypes.c_void_p(0x10002)), 1),
    (dict(d=96), 2),
    (dict(bs=32), 2),
    (dict(hq=6, hkv=4), 1),
    (dict(dt=pa.PA_E4M3, kvdt=pa.PA_E4M3), 2),  # q is 16-bit
    (dict(dt=pa.PA_F32), 2),
    (dict(kvdt=pa.PA_BF16), 2),                 # a 16-bit cache is of q's dtype
    (dict(kvdt=pa.PA_E4M3, kvs=0.0), 1),        # an E4M3 cache needs a positive finite scale
    (dict(kvdt=pa.PA_E4M3, kvs=float("inf")), 1),
    (dict(kvdt=pa.PA_E4M3, kvs=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(mq=-1), 1),
    (dict(B=-1), 1),
    (dict(nb=0), 1),
])
def test_prefill_rejects_bad_arguments(lib, over, status):
    assert lib.pa_prefill(*prefill_args(**over)) == status
    assert pa.pa_last_error() != ""


def test_prefill_without_queries_is_a_no_op(lib):
    assert lib.pa_prefill(*prefill_args(mq=0, out=NULL, q=NULL)) == 0
    assert lib.pa_prefill(*prefill_args(B=0, out=NULL, q=NULL)) == 0


def test_a_plain_c_program_uses_the_library(lib, tmp_path):
    # The header is valid C99 and the shared library links into a C program
    # that runs the host-only calls (tests/c_consumer.c states its checks).
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(pa.LIB_PATH)
    exe = str(tmp_path / "c_consumer")
    subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_consumer.c"), "-o", exe,
                    "-L", libdir, "-lpagedattn", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
