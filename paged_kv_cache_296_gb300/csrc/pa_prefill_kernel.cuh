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
// One CTA per (tile of 64 rows, KV head, sequence).  A row is one (query
// token, query head of the KV head's group) pair, token-major, so a tile holds
// 64 / G tokens' worth of the group's heads and every K/V byte it streams
// serves all of them.  Work inside a CTA (160 threads):
//   * warp 4 (producer): TMA loads of the sequence's K and V blocks 0 ..
//     ceil((last row's position + 1) / 16) - 1, one K tile and one V tile
//     (16 tokens x one head) per stage, into the same ring of full/empty
//     mbarriers as the decode kernel; every consumer warp reads every block,
//     so a stage's empty barrier counts 4 arrivals.
//   * warps 0-3 (consumers): 16 rows each.  Per block: S = Q K^T with
//     m16n8k16 tensor-core MMAs (rows as M, the block's 16 keys as N = 2 x 8,
//     head_size as K; Q held as A fragments for the whole CTA), the causal
//     mask (key > the row's position -> -inf), an online softmax on the
//     fragment (row statistics across the four lanes of a quad), then P
//     rounded to the MMA type is reused from registers as the A operand of
//     O += P V (V fragments by ldmatrix.trans; keys past L_i are zeroed, so
//     stale or poisoned slots never reach the sum).
//   * each warp normalises its rows and writes them; no cross-warp merge.
// fp32 accumulation throughout.  Tiles are visited heaviest first (the last
// rows of a sequence see the most keys).
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
  float scale_log2;               // scale * log2(e)
};

template <int D>
struct PrefillCfg {
  static constexpr int kRowBytes = D * 2;             // one token row of one head (16-bit)
  static constexpr int kTileBytes = 16 * kRowBytes;   // one block of K (or V), one head
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = (kStageBytes >= 8192) ? 8 : 16;  // a 64 KB ring
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kRows = 16 * kConsumerWarps;   // rows per CTA
  static constexpr int kSwizzle = (kRowBytes >= 128) ? 128 : 64;
  // Tiles land piece-major, [kRowBytes / 128][16 tokens][128 B] (one piece
  // for 64-byte rows); each piece is a 128B-swizzled 16-row tile.
  static constexpr int kPieceBytes = 16 * 128;
  static constexpr int kKSteps = D / 16;              // k-steps of Q K^T
  static constexpr int kDTiles = D / 8;               // n-tiles of O
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kRingBytes + 1024 + 2 * kStages * 8;
};

// Byte offset of (token row, byte column) inside a piece-major K or V tile.
template <int D>
__device__ __forceinline__ uint32_t pf_off(int tok, int col_bytes) {
  if constexpr (D * 2 >= 128) {
    const uint32_t off = (uint32_t)((col_bytes >> 7) * PrefillCfg<D>::kPieceBytes + tok * 128 +
                                    (col_bytes & 127));
    return off ^ (((off >> 7) & 7u) << 4);
  } else {
    const uint32_t off = (uint32_t)(tok * (D * 2) + col_bytes);
    return off ^ (((off >> 7) & 3u) << 4);
  }
}

template <int QT>
__device__ __forceinline__ uint32_t pf_pack(float lo, float hi) {
  if constexpr (QT == 0) {
    return pack_f16x2(lo, hi);
  } else {
    return pack_bf16x2(lo, hi);
  }
}

// Value of the low / high half of a packed pair of the MMA type.
template <int QT>
__device__ __forceinline__ float2 pf_unpack(uint32_t x) {
  if constexpr (QT == 0) {
    return __half22float2(*reinterpret_cast<const __half2*>(&x));
  } else {
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
  }
}

template <int QT>
__device__ __forceinline__ void pf_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  if constexpr (QT == 0) {
    mma_f16(d, a, b0, b1);
  } else {
    mma_bf16(d, a, b0, b1);
  }
}

// QT: 0 = fp16, 1 = bf16 (q, cache and out share it).
template <int D, int QT>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
  using C = PrefillCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kRingBytes);
  uint64_t* empty_bar = full_bar + C::kStages;

  if (threadIdx.x == C::kConsumerWarps * 32) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  // The kernel before this one on the stream (e.g. the write of the chunk's
  // K/V) may have written any input: wait for it before the first global read.
  griddep_wait();

  const int seq = blockIdx.z;
  const int kvh = blockIdx.y;
  const int tile = p.tiles - 1 - (int)blockIdx.x;  // heaviest tiles first
  const int r0q = p.query_start_loc[seq];
  const int nq = p.query_start_loc[seq + 1] - r0q;
  // A length past the table's capacity is cut to it: no entry past the row is read.
  const int L = min(p.context_lens[seq], p.max_blocks_per_seq * 16);
  if (nq <= 0) return;
  if (nq > L || nq > p.max_query_len) {
    if (threadIdx.x == 0 && tile == 0 && kvh == 0) atomicOr(p.status, kErrBadQueryLayout);
    return;
  }
  const int G = p.group;
  const int rows = nq * G;
  const int row0 = tile * C::kRows;
  if (row0 >= rows) return;
  const int last_row = min(rows, row0 + C::kRows) - 1;
  const int last_pos = L - nq + last_row / G;
  const int nkb = last_pos / 16 + 1;  // key blocks this tile attends to

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], C::kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int32_t* tbl = p.block_tables + (size_t)seq * p.max_blocks_per_seq;
    const int oob_row = p.num_blocks * 16;  // past the pool: TMA fills zeros
    const uint64_t pol = l2_evict_normal_policy();  // other tiles of the sequence reread it
    bool ok = true;
    int issued = 0;
    for (int base = 0; base < nkb; base += 32) {
      const int mine = (base + lane < nkb) ? __ldg(tbl + base + lane) : 0;
      const int cnt = min(32, nkb - base);
      for (int j = 0; j < cnt; ++j) {
        const int blk = __shfl_sync(0xffffffffu, mine, j);
        if (lane == 0 && ok) {
          const int it = base + j;
          const int s = it % C::kStages;
          const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
          if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, p.status)) {
            ok = false;
          } else {
            const int row = (blk >= 0 && blk < p.num_blocks) ? blk * 16 : oob_row;
            uint8_t* ks = smem + s * C::kStageBytes;
            mbar_arrive_expect_tx(&full_bar[s], C::kStageBytes);
            tma_load_4d(ks, &tmap_k, &full_bar[s], 0, row, 0, kvh, pol);
            tma_load_4d(ks + C::kTileBytes, &tmap_v, &full_bar[s], 0, row, 0, kvh, pol);
            ++issued;
          }
        }
      }
    }
    if (lane == 0) {
      const int first = max(0, issued - C::kStages);
      for (int it = first; it < issued; ++it) {
        mbar_wait_bounded(&full_bar[it % C::kStages], (uint32_t)(it / C::kStages) & 1u, p.status);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;  // fragment row within the warp's 16 (and row + 8)
  const int t = lane & 3;
  // This thread's two rows: warp rows wr and wr + 8.
  const int wr = row0 + warp * 16 + g;
  int pos[2];
  bool live[2];
  size_t qoff[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int r = wr + 8 * k;
    live[k] = r < rows;
    const int rr = live[k] ? r : rows - 1;
    const int tok = rr / G;
    pos[k] = L - nq + tok;
    qoff[k] = ((size_t)(r0q + tok) * p.num_q_heads + (size_t)kvh * G + (rr - tok * G)) * D;
  }
  // Q as A fragments: a0 = (row g, cols 2t..), a1 = (row g+8), a2/a3 = cols + 8.
  uint32_t qa[C::kKSteps][4];
  const uint16_t* q16 = reinterpret_cast<const uint16_t*>(p.q);
#pragma unroll
  for (int ks = 0; ks < C::kKSteps; ++ks) {
    const int c = 16 * ks + 2 * t;
    qa[ks][0] = live[0] ? *reinterpret_cast<const uint32_t*>(q16 + qoff[0] + c) : 0u;
    qa[ks][1] = live[1] ? *reinterpret_cast<const uint32_t*>(q16 + qoff[1] + c) : 0u;
    qa[ks][2] = live[0] ? *reinterpret_cast<const uint32_t*>(q16 + qoff[0] + c + 8) : 0u;
    qa[ks][3] = live[1] ? *reinterpret_cast<const uint32_t*>(q16 + qoff[1] + c + 8) : 0u;
  }

  float o[C::kDTiles][4];
#pragma unroll
  for (int i = 0; i < C::kDTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

  // ldmatrix lane addressing: K (non-transposed) and V (transposed), 16 rows.
  const int k_row = (lane & 7) + ((lane >> 4) & 1) * 8;
  const int k_col = ((lane >> 3) & 1) * 8;
  const int v_row = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int v_col = ((lane >> 4) & 1) * 8;

  for (int it = 0; it < nkb; ++it) {
    const int s = it % C::kStages;
    if (!mbar_wait_bounded(&full_bar[s], (uint32_t)(it / C::kStages) & 1u, p.status)) break;
    const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
    const uint32_t vbase = kbase + C::kTileBytes;

    // ---- S = Q K^T for the block's 16 keys (two n-tiles of 8)
    // Two accumulators per n-tile (even / odd k-steps): half-length MMA chains.
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < C::kKSteps; ++ks) {
      uint32_t b[4];
      ldsm_x4(b, kbase + pf_off<D>(k_row, (16 * ks + k_col) * 2));
      if (ks & 1) {
        pf_mma<QT>(sd[0], qa[ks], b[0], b[1]);
        pf_mma<QT>(sd[1], qa[ks], b[2], b[3]);
      } else {
        pf_mma<QT>(sc[0], qa[ks], b[0], b[1]);
        pf_mma<QT>(sc[1], qa[ks], b[2], b[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[j][e] = __fadd_rn(sc[j][e], sd[j][e]);
    }
    // ---- causal mask and online softmax (rows g: c0/c1, g+8: c2/c3)
    const int key0 = it * 16;
    float mx[2] = {m[0], m[1]};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + 8 * j + 2 * t + (e & 1);
        const int k = e >> 1;
        float v = __fmul_rn(sc[j][e], p.scale_log2);
        if (key > pos[k]) v = -INFINITY;
        sc[j][e] = v;
        mx[k] = fmaxf(mx[k], v);
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 1));
      mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 2));
    }
    // Every row sees key 0 in block 0, so mx is finite from the first block on.
    float alpha[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      alpha[k] = ex2_approx(__fsub_rn(m[k], mx[k]));
      m[k] = mx[k];
    }
    uint32_t pa[4];  // P as the A operand: (g, keys 2t..) (g+8) (g, keys 8+2t..) (g+8, 8+..)
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float p0 = ex2_approx(__fsub_rn(sc[j][2 * k], m[k]));
        const float p1 = ex2_approx(__fsub_rn(sc[j][2 * k + 1], m[k]));
        const uint32_t pk = pf_pack<QT>(p0, p1);
        const float2 r = pf_unpack<QT>(pk);  // the rounded values the MMA uses
        rs[k] = __fadd_rn(rs[k], __fadd_rn(r.x, r.y));
        pa[2 * j + k] = pk;
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) l[k] = __fmaf_rn(l[k], alpha[k], rs[k]);
    if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
      for (int i = 0; i < C::kDTiles; ++i) {
        o[i][0] = __fmul_rn(o[i][0], alpha[0]);
        o[i][1] = __fmul_rn(o[i][1], alpha[0]);
        o[i][2] = __fmul_rn(o[i][2], alpha[1]);
        o[i][3] = __fmul_rn(o[i][3], alpha[1]);
      }
    }
    // ---- O += P V; keys at or past L are zeroed in V (their slots may hold anything)
    const int valid = min(16, L - key0);
    const uint32_t mlo = (2 * t < valid ? 0x0000FFFFu : 0u) | (2 * t + 1 < valid ? 0xFFFF0000u : 0u);
    const uint32_t mhi =
        (2 * t + 8 < valid ? 0x0000FFFFu : 0u) | (2 * t + 9 < valid ? 0xFFFF0000u : 0u);
#pragma unroll
    for (int dt = 0; dt < C::kDTiles / 2; ++dt) {
      uint32_t b[4];
      ldsm_x4_trans(b, vbase + pf_off<D>(v_row, (16 * dt + v_col) * 2));
      if (valid < 16) {
        b[0] &= mlo; b[1] &= mhi; b[2] &= mlo; b[3] &= mhi;
      }
      pf_mma<QT>(o[2 * dt], pa, b[0], b[1]);
      pf_mma<QT>(o[2 * dt + 1], pa, b[2], b[3]);
    }
    // Release the stage (generic reads ordered before the async-proxy refill).
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
  }

  // ---- normalise and store: row g (c0, c1) and row g+8 (c2, c3)
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    l[k] = __fadd_rn(l[k], __shfl_xor_sync(0xffffffffu, l[k], 1));
    l[k] = __fadd_rn(l[k], __shfl_xor_sync(0xffffffffu, l[k], 2));
  }
  uint16_t* o16 = reinterpret_cast<uint16_t*>(p.out);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (!live[k]) continue;
    const float inv_ok = l[k] > 0.f ? 1.f : 0.f;
#pragma unroll
    for (int i = 0; i < C::kDTiles; ++i) {
      const float a = inv_ok > 0.f ? __fdiv_rn(o[i][2 * k], l[k]) : 0.f;
      const float b = inv_ok > 0.f ? __fdiv_rn(o[i][2 * k + 1], l[k]) : 0.f;
      *reinterpret_cast<uint32_t*>(o16 + qoff[k] + 8 * i + 2 * t) = pf_pack<QT>(a, b);
    }
  }
}

}  // namespace pa
