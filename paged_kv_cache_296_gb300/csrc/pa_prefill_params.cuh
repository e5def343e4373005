// Paged prefill attention: causal multi-query attention over the paged pool.
//
// What it computes: sequence i has L_i cached tokens (its block table maps
// logical block j / 16 to a physical block of the pool [num_blocks, 16, 2, Hkv,
// D]); its n_i query tokens are its last n_i positions L_i - n_i .. L_i - 1,
// rows query_start_loc[i] .. query_start_loc[i+1]-1 of q [T, Hq, D].  The
// query at position p, head h, attends to the sequence's tokens 0..p of KV
// head h / G:  out = softmax(scale * q . K[0..p]^T) . V[0..p].  The pages
// schedule a prefill step beside decode steps ("vLLM 部署深度指南", section
// Continuous Batching, the scheduler sketch); causal attention over the
// prompt is the plainest reading of what that step attends to.
//
// This header holds the launch parameters shared by the host launcher and
// the kernel (pa_prefill_tc.cuh).
#pragma once

#include "pa_ptx.cuh"

namespace pa {

enum : unsigned { kErrBadQueryLayout = 2u };

struct PrefillParams {
  void* out;                      // [T, Hq, D], q dtype
  const void* q;                  // [T, Hq, D]
  const int32_t* block_tables;    // [B, max_blocks_per_seq]
  const int32_t* context_lens;    // [B]
  const int32_t* query_start_loc; // [B + 1]
  unsigned* status;
  int num_seqs;
  int max_query_len;
  int max_blocks_per_seq;
  int num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int group;                      // G = Hq / Hkv
  int tiles;                      // CTAs per (sequence, KV head): tiles of the longest query run
  int band;                       // tile indices per grid band (1: heaviest tiles first)
  float scale_log2;               // scale * log2(e) (times kv_scale for an E4M3 cache)
  float out_scale;                // kv_scale for an E4M3 cache (V holds its codes), else 1
};

// Two fp32 values rounded to a packed pair of the MMA type (QT: 0 = fp16, 1 = bf16).
template <int QT>
__device__ __forceinline__ uint32_t pf_pack(float lo, float hi) {
  if constexpr (QT == 0) {
    return pack_f16x2(lo, hi);
  } else {
    return pack_bf16x2(lo, hi);
  }
}

}  // namespace pa
