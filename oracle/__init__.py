"""CPU oracle for paged-KV-cache decode: TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct definition of what the
GPU path computes, in NumPy float64.  It exists so that tests, the smoke
check and the benchmark's CPU baseline can test the CUDA library.  The
product path never imports, calls or links anything here, and nothing here
imports the product package: the two share no code.  Only the seeded input
generators (``paged_kv_cache_296_gb300.workloads``) feed both sides.

Sources (four web pages on vLLM's PagedAttention):
  * "vLLM 部署深度指南", section PagedAttention 方案 (16 tokens per block, the
    logical-view / block-table figure) and section 代码层面理解 (the pool
    ``[num_blocks, block_size, 2, num_heads, head_size]``, ``allocate`` with
    ceil rounding, ``append_kv`` writing into a physical block).
  * "vLLM GitHub 项目：探索高效 LLM 推理服务", section 二 (block table maps logical
    to physical blocks, blocks need not be contiguous, tables may share
    physical blocks).
  * FP8 KV cache: "vLLM 部署深度指南", 量化支持 table (FP8 row) and the
    ``--kv-cache-dtype fp8`` launch line; the byte format is OCP OFP8 E4M3.

Modules:
  e4m3             -- OCP E4M3 encode (round-to-nearest-even, saturating) / decode.
  paged_attention  -- reshape_and_cache, block-table gather, paged decode,
                      causal paged prefill, contiguous attention, split-KV
                      partials and their merge.
  block_manager    -- the block allocator: free list, ceil growth, sharing by
                      reference counts, copy-on-write of a shared last block.

Every function is pinned by ``tests/test_oracle_*.py`` (run with
``-m "not gpu"``) against library routines, closed forms, invariants and the
pages' worked figure.  No function is "parity unpinned".
"""

from . import e4m3, paged_attention  # noqa: F401
