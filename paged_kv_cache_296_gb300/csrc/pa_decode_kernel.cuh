// Paged decode attention: one CTA per (KV head group, KV partition, sequence).
//
// What it computes ("vLLM GitHub 项目…" section 二; "vLLM 部署深度指南" sections
// PagedAttention 方案 and 代码层面理解): for every sequence i and query head h,
//   out[i, h] = softmax(scale * q[i, h] . K_i^T) . V_i
// where K_i / V_i are the sequence's first L_i tokens, found block by block
// through its block table (logical block j // 16 -> physical block, offset
// j % 16) in the pool [num_blocks, 16, 2, Hkv, D].  Query head h reads KV head
// h / G (G = Hq / Hkv), so each CTA serves the G query heads of its KV heads
// and reads every K/V byte of those heads once.  A CTA takes H adjacent KV
// heads (H = 1 for 16-bit caches, whose rows are 256 bytes; H = 2 for E4M3,
// so each token's K (and V) bytes of the group are one 256-byte run in the
// pool: measured on GB300, streaming that pattern in 128-byte runs tops out
// near 6.1 TB/s, in 256-byte runs near 6.7 TB/s).
//
// Layout of the work inside a CTA (4H consumer warps + 1 producer warp):
//   * the producer warp: one lane reads the partition's block-table entries
//     and issues one TMA load per 16-token block for K and one for V (all H
//     heads) into a ring of shared-memory stages, each guarded by a "full"
//     and an "empty" mbarrier.  Tiles land 128B-swizzled, so fragment loads
//     are bank-conflict free.
//   * consumers: warps 4j .. 4j+3 serve the group's head j; warp 4j + w takes
//     blocks w, w+4, ... and releases each stage once all H heads are done
//     with it (the empty barrier counts H arrivals).  For each block it
//     computes S^T = K . Q^T with m16n8k16 tensor-core MMAs (tokens as M = 16,
//     the G <= 8 query heads as N = 8, head_size as K), runs the online softmax
//     on the fragment, turns P^T into the B operand with movmatrix, and
//     accumulates O^T += V^T . P^T (head_size as M).  All accumulation is fp32.
//   * at the end each head's four warps' (m, l, O) states are merged through shared
//     memory; the CTA writes the normalised output (one partition) or an fp32
//     partial (m, l, O) that the merge kernel combines by log-sum-exp.
//
// fp8-E4M3 KV: bytes are widened exactly to f16 in registers (cvt.f16x2.e4m3x2);
// q is rounded to f16; the per-tensor kv_scale multiplies the logits and the
// output.  For the byte loads the head_size index of K is permuted (the same
// permutation is applied to q, so the dot product is unchanged) and the
// head_size index of V maps to output rows in a lane-contiguous order.
//
// This header holds the partition kernel (partitions of a given size, grid
// (KV head groups, partitions, sequences), or a balanced split of one wave
// planned in the kernel from the lengths) and the per-block step, query
// fragment load and fused token write that the shared-prefix kernel
// (pa_decode_split.cuh) shares with it, so both compute with the same bits.
#pragma once

#include "pa_ptx.cuh"

namespace pa {

enum KvKind { kKvF16 = 0, kKvBf16 = 1, kKvE4m3 = 2 };

struct DecodeParams {
  void* out;                    // [B, Hq, D], q dtype
  const void* q;                // [B, Hq, D]
  const int32_t* block_tables;  // [B, max_blocks_per_seq]
  const int32_t* context_lens;  // [B]
  float* part_m;                // [B, Hq, P]   (log2 domain)
  float* part_l;                // [B, Hq, P]
  float* part_o;                // [B, Hq, P, D]
  unsigned* status;             // device status word (error bits)
  int num_seqs;
  int max_blocks_per_seq;
  int num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int kv_groups;                // CTAs per (sequence, partition): ceil(num_kv_heads / H)
  int group;                    // G = Hq / Hkv, 1..8
  int partition_blocks;         // partition size in 16-token blocks; 0 = balanced (below)
  // Balanced split: the partition size is chosen in the kernel from the actual
  // context lengths, as the smallest one (>= min_partition_blocks) whose
  // partitions over all sequences and KV heads fit in `slots` resident CTAs.
  int min_partition_blocks;
  int slots;
  int num_partitions;           // P = partitions of the longest possible sequence
  float scale_log2;             // scale * log2(e) (* kv_scale for E4M3)
  float out_scale;              // kv_scale for E4M3, else 1
  float kv_scale;               // E4M3 write scale (fused write only)
  // Fused write of each sequence's new token (the last one, position L - 1).
  const uint8_t* k_new;         // [B, Hkv, D] of the q dtype, token stride src_stride_bytes
  const uint8_t* v_new;
  const int64_t* slot_mapping;  // [B]
  int64_t src_stride_bytes;
  uint8_t* k_cache;             // writable pool views
  uint8_t* v_cache;
  // ---- stream-K kernel only (pa_decode_split.cuh)
  int min_units;                // smallest range of blocks a CTA takes
  const int32_t* grp_off;       // [num_groups + 1] shared-prefix groups (CSR over grp_seq)
  const int32_t* grp_seq;       // sequence indices, group after group
  const int32_t* grp_blocks;    // [num_groups] leading table entries a group shares
  int num_groups;
  int cut_cols;                 // columns of one cut partial slot
  float* cut_m;                 // [CTAs][2][cut_cols]
  float* cut_l;
  float* cut_o;                 // [CTAs][2][cut_cols][D]
  float* whole_m;               // [2][B][Hq] (shared-prefix mode only)
  float* whole_l;
  float* whole_o;               // [2][B][Hq][D]
  int* plan;                    // the attention kernel's plan (balanced: its partition
                                // size; stream-K: the plan record), for the merge kernel
};


template <int D, int KV>
struct DecodeCfg {
  static constexpr int kElt = (KV == kKvE4m3) ? 1 : 2;
  static constexpr int kHeads = (KV == kKvE4m3) ? 2 : 1;  // KV heads per CTA (H)
  static constexpr int kRowBytes = D * kElt;          // one token row of one head
  static constexpr int kTileBytes = 16 * kHeads * kRowBytes;  // one block of K (or V), H heads
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
  static constexpr int kWarpsPerHead = 4;
  static constexpr int kConsumerWarps = kWarpsPerHead * kHeads;
  // Block `it` goes to stage it % kStages and to warp it % 4 of every head.
  // With kStages a multiple of 4, every stage has one consumer warp per head
  // that waits on its phases strictly in order, so a parity wait never runs
  // two phases ahead of its barrier (which would let it pass early).  Two or
  // more stages per warp let the producer run ahead while a warp computes.  A
  // CTA streams about (ring bytes) / (loaded memory latency, ~3.5 us on
  // GB300), so the ring is 64 KB whatever the stage size.
  static constexpr int kStages = (kStageBytes >= 8192) ? 8 : 16;
  static_assert(kStages % kWarpsPerHead == 0 && kStages >= 2 * kWarpsPerHead,
                "each stage must belong to exactly one consumer warp per head");
  static constexpr int kSwizzle = (kRowBytes >= 128) ? 128 : 64;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kMinCtasPerSm = (kHeads == 1) ? 4 : 2;  // register budget
  static constexpr int kMTiles = D / 16;              // m-tiles of O^T, k-steps of S^T
  static constexpr int kRedStride = D + 4;            // floats per head row in the merge buffer
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kRedBytes = kConsumerWarps * 8 * kRedStride * 4 + 2 * kConsumerWarps * 8 * 4;
  static constexpr int kSmemBytes = kRingBytes + 1024 /*align*/ + 2 * kStages * 8;
  static_assert(kRedBytes <= kRingBytes, "merge buffer must fit in the ring");
};

// Byte offset inside a swizzled tile of token rows (`row_bytes` per token).
template <int SW>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  if constexpr (SW == 128) {
    return off ^ (((off >> 7) & 7u) << 4);
  } else {
    return off ^ (((off >> 7) & 3u) << 4);
  }
}

template <int QT>
__device__ __forceinline__ float load_q_elem(const void* q, size_t idx) {
  if constexpr (QT == kKvF16) {
    return __half2float(reinterpret_cast<const __half*>(q)[idx]);
  } else {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(q)[idx]);
  }
}

template <int QT>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
  if constexpr (QT == kKvF16) {
    reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
  } else {
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  }
}

// Keep the halves of a packed pair whose token index is below `valid`.
__device__ __forceinline__ uint32_t token_mask(int tok, int valid) {
  return (tok < valid ? 0x0000FFFFu : 0u) | (tok + 1 < valid ? 0xFFFF0000u : 0u);
}

// One warp's online-softmax state for the 8 query-head columns of its MMA
// n-tile: lane (g, t) holds O^T rows (head_size) of columns 2t and 2t + 1 and
// the running maximum m and sum l of those two columns.
template <int D>
struct WarpState {
  float o[D / 16][4];
  float m0, m1, l0, l1;
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }
};

// B operand (Q^T) of the S^T MMAs: lane (g, t) holds query row `qrow`'s
// elements of k-steps 0 .. D/16-1 (zeros if !live).
template <int D, int KV, int QT>
__device__ __forceinline__ void load_q_frag(uint32_t (&qb)[D / 16][2], const void* q, size_t qrow,
                                            bool live) {
  const int t = threadIdx.x & 3;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    if (!live) {
      qb[s][0] = qb[s][1] = 0u;
    } else if constexpr (KV != kKvE4m3) {
      qb[s][0] = *reinterpret_cast<const uint32_t*>(
          reinterpret_cast<const uint16_t*>(q) + qrow + 16 * s + 2 * t);
      qb[s][1] = *reinterpret_cast<const uint32_t*>(
          reinterpret_cast<const uint16_t*>(q) + qrow + 16 * s + 2 * t + 8);
    } else {
      // head_size index permuted to match the K byte layout (see the header).
      const size_t d0 = qrow + (D / 4) * t + 4 * s;
      qb[s][0] = pack_f16x2(load_q_elem<QT>(q, d0), load_q_elem<QT>(q, d0 + 1));
      qb[s][1] = pack_f16x2(load_q_elem<QT>(q, d0 + 2), load_q_elem<QT>(q, d0 + 3));
    }
  }
}

// NB 16-token blocks of one head (NB = 1 or 2), for the calling warp's 8
// columns: S^T = K Q^T, online softmax, O^T += V^T P^T.  kbase[b] / vbase[b]:
// block b's K and V tiles in its stage (H heads, token-major); hsel: this
// warp's head within the tile; valid[b]: the block's tokens that exist (V rows
// past it are zeroed, their logits -inf).  kColMask: token r of block b counts
// for column 2t only if r < lim0[b] and for column 2t + 1 only if r < lim1[b]
// (columns of different sequences), and a column with no token so far keeps a
// zero state.  With NB = 2 the blocks' MMA chains interleave and they share
// one softmax step (one running-maximum update over their 32 tokens).
template <int D, int KV, bool kColMask, int NB>
__device__ __forceinline__ void decode_blocks(WarpState<D>& st, const uint32_t (&qb)[D / 16][2],
                                              const uint32_t (&kbase)[NB],
                                              const uint32_t (&vbase)[NB], int hsel,
                                              const int (&valid)[NB], float scale_log2,
                                              const int (&lim0)[NB], const int (&lim1)[NB]) {
  using C = DecodeCfg<D, KV>;
  constexpr bool kFp8 = (KV == kKvE4m3);
  // The P^T / V operands of the PV product are f16 unless the cache is bf16.
  constexpr bool kBf16Mma = (KV == kKvBf16);
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  // Byte offset of token `tok`'s row of this warp's head inside a tile.
  auto row_of = [&](int tok) { return (uint32_t)((tok * C::kHeads + hsel) * C::kRowBytes); };

  // ---- S^T = K . Q^T  (rows: tokens, columns: query heads)
  float sacc[NB][4];
#pragma unroll
  for (int b = 0; b < NB; ++b) sacc[b][0] = sacc[b][1] = sacc[b][2] = sacc[b][3] = 0.f;
  if constexpr (!kFp8) {
    const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < C::kMTiles; ++ks) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        uint32_t a[4];
        ldsm_x4(a, kbase[b] + swz<C::kSwizzle>(row_of(tok) + (ks * 2 + (lane >> 4)) * 16));
        if constexpr (kBf16Mma) {
          mma_bf16(sacc[b], a, qb[ks][0], qb[ks][1]);
        } else {
          mma_f16(sacc[b], a, qb[ks][0], qb[ks][1]);
        }
      }
    }
  } else {
    constexpr int kCpl = D / 64;  // 16-byte chunks per lane per row
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      uint32_t wa[C::kMTiles], wb[C::kMTiles];
#pragma unroll
      for (int i = 0; i < kCpl; ++i) {
        const uint4 xa = lds128(kbase[b] + swz<C::kSwizzle>(row_of(g) + (kCpl * t + i) * 16));
        const uint4 xb = lds128(kbase[b] + swz<C::kSwizzle>(row_of(g + 8) + (kCpl * t + i) * 16));
        wa[4 * i + 0] = xa.x; wa[4 * i + 1] = xa.y; wa[4 * i + 2] = xa.z; wa[4 * i + 3] = xa.w;
        wb[4 * i + 0] = xb.x; wb[4 * i + 1] = xb.y; wb[4 * i + 2] = xb.z; wb[4 * i + 3] = xb.w;
      }
#pragma unroll
      for (int ks = 0; ks < C::kMTiles; ++ks) {
        uint32_t a[4];
        a[0] = e4m3x2_to_f16x2((uint16_t)(wa[ks] & 0xFFFFu));
        a[1] = e4m3x2_to_f16x2((uint16_t)(wb[ks] & 0xFFFFu));
        a[2] = e4m3x2_to_f16x2((uint16_t)(wa[ks] >> 16));
        a[3] = e4m3x2_to_f16x2((uint16_t)(wb[ks] >> 16));
        mma_f16(sacc[b], a, qb[ks][0], qb[ks][1]);
      }
    }
  }

  // ---- online softmax on the fragments: c0/c1 token g, c2/c3 token g+8
  // Every rounding step below is spelled out (_rn intrinsics), so no
  // instantiation of this kernel contracts them into FMAs differently:
  // all variants produce the same bits.
  float sc[NB][4];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[b][i] = __fmul_rn(sacc[b][i], scale_log2);
    if (valid[b] < 16) {
      if (g >= valid[b]) sc[b][0] = sc[b][1] = -INFINITY;
      if (g + 8 >= valid[b]) sc[b][2] = sc[b][3] = -INFINITY;
    }
    if constexpr (kColMask) {
      if (g >= lim0[b]) sc[b][0] = -INFINITY;
      if (g >= lim1[b]) sc[b][1] = -INFINITY;
      if (g + 8 >= lim0[b]) sc[b][2] = -INFINITY;
      if (g + 8 >= lim1[b]) sc[b][3] = -INFINITY;
    }
  }
  float bm0 = fmaxf(sc[0][0], sc[0][2]), bm1 = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
  for (int b = 1; b < NB; ++b) {
    bm0 = fmaxf(bm0, fmaxf(sc[b][0], sc[b][2]));
    bm1 = fmaxf(bm1, fmaxf(sc[b][1], sc[b][3]));
  }
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
  }
  const float mn0 = fmaxf(st.m0, bm0), mn1 = fmaxf(st.m1, bm1);
  // A column none of whose tokens counted yet has mn = -inf: subtract 0
  // instead, so its weights come out 0 rather than NaN.
  const float mr0 = (kColMask && mn0 == -INFINITY) ? 0.f : mn0;
  const float mr1 = (kColMask && mn1 == -INFINITY) ? 0.f : mn1;
  const float al0 = ex2_approx(__fsub_rn(st.m0, mr0)), al1 = ex2_approx(__fsub_rn(st.m1, mr1));
  st.m0 = mn0;
  st.m1 = mn1;
  uint32_t P01[NB], P23[NB];
  float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const float p0 = ex2_approx(__fsub_rn(sc[b][0], mr0)), p1 = ex2_approx(__fsub_rn(sc[b][1], mr1));
    const float p2 = ex2_approx(__fsub_rn(sc[b][2], mr0)), p3 = ex2_approx(__fsub_rn(sc[b][3], mr1));
    float r0, r1, r2, r3;  // the rounded probabilities the MMA will use
    if constexpr (kBf16Mma) {
      P01[b] = pack_bf16x2(p0, p1);
      P23[b] = pack_bf16x2(p2, p3);
      r0 = __uint_as_float(P01[b] << 16); r1 = __uint_as_float(P01[b] & 0xFFFF0000u);
      r2 = __uint_as_float(P23[b] << 16); r3 = __uint_as_float(P23[b] & 0xFFFF0000u);
    } else {
      P01[b] = pack_f16x2(p0, p1);
      P23[b] = pack_f16x2(p2, p3);
      const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&P01[b]));
      const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&P23[b]));
      r0 = f01.x; r1 = f01.y; r2 = f23.x; r3 = f23.y;
    }
    if (b == 0) {
      sum0 = __fadd_rn(r0, r2);
      sum1 = __fadd_rn(r1, r3);
    } else {
      sum0 = __fadd_rn(sum0, __fadd_rn(r0, r2));
      sum1 = __fadd_rn(sum1, __fadd_rn(r1, r3));
    }
  }
  st.l0 = __fmaf_rn(st.l0, al0, sum0);
  st.l1 = __fmaf_rn(st.l1, al1, sum1);
  if (__any_sync(0xffffffffu, (al0 != 1.f) || (al1 != 1.f))) {
#pragma unroll
    for (int i = 0; i < C::kMTiles; ++i) {
      st.o[i][0] = __fmul_rn(st.o[i][0], al0); st.o[i][1] = __fmul_rn(st.o[i][1], al1);
      st.o[i][2] = __fmul_rn(st.o[i][2], al0); st.o[i][3] = __fmul_rn(st.o[i][3], al1);
    }
  }
  // P^T as the B operand: k = tokens (2t, 2t+1 | 2t+8, 2t+9), n = head g.
  uint32_t pb0[NB], pb1[NB], mlo[NB], mhi[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    pb0[b] = movmatrix_trans(P01[b]);
    pb1[b] = movmatrix_trans(P23[b]);
    mlo[b] = token_mask(2 * t, valid[b]);
    mhi[b] = token_mask(2 * t + 8, valid[b]);
  }

  // ---- O^T += V^T . P^T
  if constexpr (!kFp8) {
    const int mi = lane >> 3;
    const int tok = (lane & 7) + 8 * (mi >> 1);
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        uint32_t a[4];
        ldsm_x4_trans(a, vbase[b] + swz<C::kSwizzle>(row_of(tok) + (mt * 2 + (mi & 1)) * 16));
        if (valid[b] < 16) {
          a[0] &= mlo[b]; a[1] &= mlo[b]; a[2] &= mhi[b]; a[3] &= mhi[b];
        }
        if constexpr (kBf16Mma) {
          mma_bf16(st.o[mt], a, pb0[b], pb1[b]);
        } else {
          mma_f16(st.o[mt], a, pb0[b], pb1[b]);
        }
      }
    }
  } else {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      // Lane (g, t) owns head_size indices [D/8 * g, D/8 * (g+1)) of tokens
      // 2t, 2t+1, 2t+8, 2t+9; m-tile mt row g is index D/8*g + 2mt, row g+8
      // is the next one.
      uint32_t va[D / 32], vb[D / 32], vc[D / 32], vd[D / 32];
      if constexpr (D == 128) {
        const uint32_t col = g * 16;
        const uint4 x0 = lds128(vbase[b] + swz<C::kSwizzle>(row_of(2 * t) + col));
        const uint4 x1 = lds128(vbase[b] + swz<C::kSwizzle>(row_of(2 * t + 1) + col));
        const uint4 x2 = lds128(vbase[b] + swz<C::kSwizzle>(row_of(2 * t + 8) + col));
        const uint4 x3 = lds128(vbase[b] + swz<C::kSwizzle>(row_of(2 * t + 9) + col));
        va[0] = x0.x; va[1] = x0.y; va[2] = x0.z; va[3] = x0.w;
        vb[0] = x1.x; vb[1] = x1.y; vb[2] = x1.z; vb[3] = x1.w;
        vc[0] = x2.x; vc[1] = x2.y; vc[2] = x2.z; vc[3] = x2.w;
        vd[0] = x3.x; vd[1] = x3.y; vd[2] = x3.z; vd[3] = x3.w;
      } else {
        const uint32_t col = g * 8;
        const uint2 x0 = lds64(vbase[b] + swz<C::kSwizzle>(row_of(2 * t) + col));
        const uint2 x1 = lds64(vbase[b] + swz<C::kSwizzle>(row_of(2 * t + 1) + col));
        const uint2 x2 = lds64(vbase[b] + swz<C::kSwizzle>(row_of(2 * t + 8) + col));
        const uint2 x3 = lds64(vbase[b] + swz<C::kSwizzle>(row_of(2 * t + 9) + col));
        va[0] = x0.x; va[1] = x0.y; vb[0] = x1.x; vb[1] = x1.y;
        vc[0] = x2.x; vc[1] = x2.y; vd[0] = x3.x; vd[1] = x3.y;
      }
#pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) {
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
        const uint32_t lo = __byte_perm(va[mt >> 1], vb[mt >> 1], sel);  // tokens 2t, 2t+1
        const uint32_t hi = __byte_perm(vc[mt >> 1], vd[mt >> 1], sel);  // tokens 2t+8, 2t+9
        uint32_t a[4];
        a[0] = e4m3x2_to_f16x2((uint16_t)(lo & 0xFFFFu));
        a[1] = e4m3x2_to_f16x2((uint16_t)(lo >> 16));
        a[2] = e4m3x2_to_f16x2((uint16_t)(hi & 0xFFFFu));
        a[3] = e4m3x2_to_f16x2((uint16_t)(hi >> 16));
        if (valid[b] < 16) {
          a[0] &= mlo[b]; a[1] &= mlo[b]; a[2] &= mhi[b]; a[3] &= mhi[b];
        }
        mma_f16(st.o[mt], a, pb0[b], pb1[b]);
      }
    }
  }
}

// One block: decode_blocks with NB = 1.
template <int D, int KV, bool kColMask>
__device__ __forceinline__ void decode_block(WarpState<D>& st, const uint32_t (&qb)[D / 16][2],
                                             uint32_t kbase, uint32_t vbase, int hsel, int valid,
                                             float scale_log2, int lim0, int lim1) {
  const uint32_t kb[1] = {kbase}, vb[1] = {vbase};
  const int va[1] = {valid}, l0[1] = {lim0}, l1[1] = {lim1};
  decode_blocks<D, KV, kColMask, 1>(st, qb, kb, vb, hsel, va, scale_log2, l0, l1);
}

// Sum l over the 8 lanes that share t (tokens g and g+8 of every block).
template <int D>
__device__ __forceinline__ void finish_row_sums(WarpState<D>& st) {
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, x);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, x);
  }
}

// Store a warp's state to its slice of the merge buffer: O rows of columns
// 0..ncols-1 (ncols 4 or 8; stride kRedStride floats, head_size in natural
// order), m and l.
template <int D, int KV>
__device__ __forceinline__ void dump_state(const WarpState<D>& st, float* red_o, float* red_m,
                                           float* red_l, int ncols = 8) {
  using C = DecodeCfg<D, KV>;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  if (2 * t >= ncols) return;
#pragma unroll
  for (int mt = 0; mt < C::kMTiles; ++mt) {
    int d_lo, d_hi;
    if constexpr (KV == kKvE4m3) {
      d_lo = (D / 8) * g + 2 * mt;
      d_hi = d_lo + 1;
    } else {
      d_lo = 16 * mt + g;
      d_hi = d_lo + 8;
    }
    red_o[(2 * t) * C::kRedStride + d_lo] = st.o[mt][0];
    red_o[(2 * t + 1) * C::kRedStride + d_lo] = st.o[mt][1];
    red_o[(2 * t) * C::kRedStride + d_hi] = st.o[mt][2];
    red_o[(2 * t + 1) * C::kRedStride + d_hi] = st.o[mt][3];
  }
  if (g == 0) {
    red_m[2 * t] = st.m0;
    red_m[2 * t + 1] = st.m1;
    red_l[2 * t] = st.l0;
    red_l[2 * t + 1] = st.l1;
  }
}

// Eight source elements (16 bytes of q's dtype) to eight E4M3 codes:
// e4m3_rn_satfinite(x / kv_scale), x widened exactly to fp32, an IEEE division.
template <int QT>
__device__ __forceinline__ uint2 quantize8_e4m3(uint4 u, float kv_scale) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (QT == kKvF16) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    } else {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  uint32_t q8[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint16_t a = f32x2_to_e4m3x2(__fdiv_rn(x[4 * h], kv_scale), __fdiv_rn(x[4 * h + 1], kv_scale));
    const uint16_t b =
        f32x2_to_e4m3x2(__fdiv_rn(x[4 * h + 2], kv_scale), __fdiv_rn(x[4 * h + 3], kv_scale));
    q8[h] = (uint32_t)a | ((uint32_t)b << 16);
  }
  return make_uint2(q8[0], q8[1]);
}

// append_kv for one sequence's new token, KV heads kv0 .. kv0+H-1, by the
// calling warp: the same bytes pa_reshape_and_cache writes (a copy for a
// 16-bit cache, e4m3_rn_satfinite(x / kv_scale) for E4M3), then a proxy fence
// so this thread's later TMA loads of the block observe the write.
template <int D, int KV, int QT>
__device__ __forceinline__ void append_token(const DecodeParams& p, int seq, int kv0, int64_t slot) {
  using C = DecodeCfg<D, KV>;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int hh = 0; hh < C::kHeads; ++hh) {
    const int kvh = kv0 + hh;
    if (kvh < p.num_kv_heads && slot >= 0 && slot < (int64_t)p.num_blocks * 16) {
      constexpr int kSrcElt = 2;  // the new token comes in the q dtype
      const size_t src = (size_t)seq * p.src_stride_bytes + (size_t)kvh * D * kSrcElt;
      const size_t dst = (size_t)slot * (2ull * p.num_kv_heads * C::kRowBytes) +
                         (size_t)kvh * C::kRowBytes;
      if constexpr (KV != kKvE4m3) {
        constexpr int kVec = D * 2 / 16;  // 16-byte vectors per row
        if (lane < 2 * kVec) {
          const bool isv = lane >= kVec;
          const int j = isv ? lane - kVec : lane;
          const uint4 x = reinterpret_cast<const uint4*>((isv ? p.v_new : p.k_new) + src)[j];
          reinterpret_cast<uint4*>((isv ? p.v_cache : p.k_cache) + dst)[j] = x;
        }
      } else {
        constexpr int kGrp = D / 8;  // 8 elements -> 8 bytes per lane
        if (lane < 2 * kGrp) {
          const bool isv = lane >= kGrp;
          const int j = isv ? lane - kGrp : lane;
          const uint4 u = reinterpret_cast<const uint4*>((isv ? p.v_new : p.k_new) + src)[j];
          reinterpret_cast<uint2*>((isv ? p.v_cache : p.k_cache) + dst)[j] =
              quantize8_e4m3<QT>(u, p.kv_scale);
        }
      }
      fence_proxy_async_global();
    }
  }
  __syncwarp();
}

// append_kv for the new tokens of `nrows` sequences (rows[]), KV heads kv0 ..
// kv0+H-1, by `nthreads` threads (thread index `tid`): the same bytes as
// append_token, each thread taking 16-byte source pieces in turn, four at a
// time with all four loads issued before any store; then a proxy fence, so
// TMA loads issued after a barrier that follows observe the writes.
template <int D, int KV, int QT>
__device__ __forceinline__ void append_rows(const DecodeParams& p, const int* rows, int nrows,
                                            int kv0, int tid, int nthreads) {
  using C = DecodeCfg<D, KV>;
  constexpr int kUnits = D / 8;  // 16-byte source pieces per head row (8 elements)
  constexpr int kPerRow = C::kHeads * 2 * kUnits;
  constexpr int kBatch = 4;
  constexpr int kDstPiece = (KV == kKvE4m3) ? 8 : 16;
  const int total = nrows * kPerRow;
  const int64_t pool_rows = (int64_t)p.num_blocks * 16;
  for (int base = tid; base < total; base += kBatch * nthreads) {
    uint4 x[kBatch];
    uint8_t* dst[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int i = base + b * nthreads;
      dst[b] = nullptr;
      if (i < total) {
        const int r = i / kPerRow;
        const int rem = i - r * kPerRow;
        const int hh = rem / (2 * kUnits);
        const int isv = (rem - hh * 2 * kUnits) / kUnits;
        const int j = rem - hh * 2 * kUnits - isv * kUnits;
        const int seq = rows[r];
        const int kvh = kv0 + hh;
        const int L = min(max(p.context_lens[seq], 0), p.max_blocks_per_seq * 16);
        const int64_t slot = L > 0 ? p.slot_mapping[seq] : -1;
        if (kvh < p.num_kv_heads && slot >= 0 && slot < pool_rows) {
          const size_t src = (size_t)seq * p.src_stride_bytes + (size_t)kvh * D * 2 + (size_t)j * 16;
          x[b] = *reinterpret_cast<const uint4*>((isv ? p.v_new : p.k_new) + src);
          dst[b] = (isv ? p.v_cache : p.k_cache) +
                   (size_t)slot * (2ull * p.num_kv_heads * C::kRowBytes) +
                   (size_t)kvh * C::kRowBytes + (size_t)j * kDstPiece;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (dst[b] == nullptr) continue;
      if constexpr (KV != kKvE4m3) {
        *reinterpret_cast<uint4*>(dst[b]) = x[b];
      } else {
        *reinterpret_cast<uint2*>(dst[b]) = quantize8_e4m3<QT>(x[b], p.kv_scale);
      }
    }
  }
  fence_proxy_async_global();
}

// Issue the TMA loads of one 16-token block (K tile then V tile, H heads from
// kv0) into stage s, completing on full_bar[s].  An out-of-range block id
// reads the first row past the pool, which TMA fills with zeros.
template <int D, int KV>
__device__ __forceinline__ void load_block(uint8_t* stage, const CUtensorMap* tmap_k,
                                           const CUtensorMap* tmap_v, uint64_t* full, int blk,
                                           int num_blocks, int kv0, uint64_t policy) {
  using C = DecodeCfg<D, KV>;
  const int row = (blk >= 0 && blk < num_blocks) ? blk * 16 : num_blocks * 16;
  mbar_arrive_expect_tx(full, C::kStageBytes);
  if constexpr (C::kRowBytes > 128) {
    tma_load_4d(stage, tmap_k, full, 0, 0, kv0, row, policy);
    tma_load_4d(stage + C::kTileBytes, tmap_v, full, 0, 0, kv0, row, policy);
  } else {
    tma_load_3d(stage, tmap_k, full, 0, kv0, row, policy);
    tma_load_3d(stage + C::kTileBytes, tmap_v, full, 0, kv0, row, policy);
  }
}

// Balanced split (partition_blocks == 0).  The grid is one dimension of
// `slots` CTAs (one wave on this GPU, or the number of (sequence, KV head
// group) pairs if that is larger).  Every CTA computes the same plan from the
// actual context lengths:
//   pb = the smallest partition size in blocks, >= min_partition_blocks, with
//        kv_groups * sum_i max(1, ceil(ceil(L_i / 16) / pb)) <= slots;
// then takes work item blockIdx.x of the list ordered by (sequence, partition,
// KV head group) -- each sequence has at least one item, so empty sequences
// still get their zero output.  Items past the list's end exit at once.
//
// The plan is on every CTA's critical path, so it is a k-ary search: each
// round tests evenly spaced sizes at once (the count is monotone in pb) and
// keeps the interval where the test flips.  The interval starts narrow: with
// T blocks over V sequences, count(pb) <= T / pb + V, so every
// pb >= kv_groups * T / (slots - kv_groups * V) fits, while none below
// kv_groups * T / slots does; for a few long sequences that is a window of a
// few dozen sizes.  Up to 32 sequences, one warp does it all (a lane per
// sequence and a lane per tested size, 32 sizes a round, no barrier inside);
// beyond that the CTA's warps each test one size per round.
constexpr int kMaxBalancedSeqs = 512;  // the host only picks the mode below this

struct BalancedItem {
  int pb, seq, part, kvg;
  int len;  // the sequence's context length (-1: not known here)
  bool valid;
};

struct BalancedScratch {
  int nb[kMaxBalancedSeqs];  // blocks per sequence; -1: negative length (no item)
  int fits[2][32];           // per round parity, per warp
  int chunk[kMaxBalancedSeqs / 32];
  int pick[5];
};

__device__ __forceinline__ int parts_of(int n, int pbv) {
  return n < 0 ? 0 : max(1, (n + pbv - 1) / pbv);
}

// Up to 32 sequences: warp 0 computes the plan, every thread reads it.
__device__ __forceinline__ BalancedItem balanced_plan_small(const DecodeParams& p,
                                                           BalancedScratch& sc) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const int B = p.num_seqs;
    const int L = lane < B ? min(p.context_lens[lane], p.max_blocks_per_seq * 16) : -1;
    const int n = L > 0 ? (L + 15) >> 4 : (L == 0 ? 0 : -1);  // -1: no item
    int total = max(n, 0), maxnb = n, nvalid = n >= 0 ? 1 : 0;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) {
      total += __shfl_xor_sync(0xffffffffu, total, x);
      maxnb = max(maxnb, __shfl_xor_sync(0xffffffffu, maxnb, x));
      nvalid += __shfl_xor_sync(0xffffffffu, nvalid, x);
    }
    // The window's ends in float, widened so rounding cannot cut the answer
    // off: below lo nothing fits, from hi on everything does.
    const float tg = (float)total * (float)p.kv_groups;
    const float want = tg / (float)p.slots * 0.999f;
    int lo = max(p.min_partition_blocks, (int)fminf(want, 1.0e9f));
    int ub = maxnb;
    const int spare = p.slots - nvalid * p.kv_groups;
    if (spare > 0) ub = min(ub, (int)fminf(tg / (float)spare * 1.001f + 2.f, 1.0e9f));
    int hi = max(lo, ub);
    while (lo < hi) {
      const int span = hi - lo;
      const int c = lo + (int)((long long)span * (lane + 1) / 32);  // lane 31 tests hi
      int cnt = 0;
      for (int i = 0; i < B; ++i) cnt += parts_of(__shfl_sync(0xffffffffu, n, i), c);
      const unsigned fit =
          __ballot_sync(0xffffffffu, (long long)cnt * p.kv_groups <= p.slots);
      const int w = __ffs(fit) - 1;  // lane 31 (hi) always fits
      const int cw = __shfl_sync(0xffffffffu, c, w);
      const int cprev = __shfl_sync(0xffffffffu, c, w > 0 ? w - 1 : 0);
      hi = cw;
      lo = w > 0 ? cprev + 1 : lo;
    }
    const int pb = lo;
    const int mine = parts_of(n, pb);
    int incl = mine;
#pragma unroll
    for (int x = 1; x < 32; x <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, x);
      if (lane >= x) incl += o;
    }
    const int all = __shfl_sync(0xffffffffu, incl, 31);
    const int q = blockIdx.x / p.kv_groups;
    const int excl = incl - mine;
    const unsigned hit = __ballot_sync(0xffffffffu, q >= excl && q < excl + mine);
    if (lane == 0) {
      sc.pick[0] = hit ? __ffs(hit) - 1 : -1;
      sc.pick[2] = pb;
      sc.pick[3] = all;
    }
    if (hit && lane == __ffs(hit) - 1) {
      sc.pick[1] = q - excl;
      sc.pick[4] = L;
    }
  }
  __syncthreads();
  BalancedItem it;
  it.pb = sc.pick[2];
  const int q = blockIdx.x / p.kv_groups;
  it.valid = q < sc.pick[3] && sc.pick[0] >= 0;
  it.seq = it.valid ? sc.pick[0] : 0;
  it.part = it.valid ? sc.pick[1] : 0;
  it.kvg = blockIdx.x % p.kv_groups;
  it.len = it.valid ? sc.pick[4] : -1;
  return it;
}

template <int kThreads>
__device__ __forceinline__ BalancedItem balanced_plan(const DecodeParams& p, BalancedScratch& sc) {
  if (p.num_seqs <= 32) return balanced_plan_small(p, sc);
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = p.num_seqs;
  for (int i = threadIdx.x; i < B; i += kThreads) {
    const int L = min(p.context_lens[i], p.max_blocks_per_seq * 16);
    sc.nb[i] = L > 0 ? (L + 15) >> 4 : (L == 0 ? 0 : -1);
  }
  if (threadIdx.x == 0) sc.pick[0] = -1;
  __syncthreads();
  // Every warp reduces the totals itself: no barrier needed.
  int total = 0, maxnb = 0, nvalid = 0;
  for (int i = lane; i < B; i += 32) {
    const int n = sc.nb[i];
    total += max(n, 0);
    maxnb = max(maxnb, n);
    nvalid += n >= 0 ? 1 : 0;
  }
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) {
    total += __shfl_xor_sync(0xffffffffu, total, x);
    maxnb = max(maxnb, __shfl_xor_sync(0xffffffffu, maxnb, x));
    nvalid += __shfl_xor_sync(0xffffffffu, nvalid, x);
  }
  const long long tg = (long long)total * p.kv_groups;
  const long long want = (tg + p.slots - 1) / p.slots;
  int lo = max(p.min_partition_blocks, (int)(want < (1ll << 30) ? want : (1ll << 30)));
  // Every sequence in one partition (pb = maxnb) fits, as kv_groups * B <= slots.
  long long ub = maxnb;
  const long long spare = (long long)p.slots - (long long)nvalid * p.kv_groups;
  if (spare > 0) ub = min(ub, (tg + spare - 1) / spare);
  int hi = max(lo, (int)ub);
  for (int round = 0; lo < hi; ++round) {
    const long long span = hi - lo;
    const int c = lo + (int)(span * (warp + 1) / kWarps);  // the last warp tests hi
    int cnt = 0;
    for (int i = lane; i < B; i += 32) cnt += parts_of(sc.nb[i], c);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, x);
    int* fits = sc.fits[round & 1];  // alternate so the next round's writes race no reads
    if (lane == 0) fits[warp] = ((long long)cnt * p.kv_groups <= p.slots) ? 1 : 0;
    __syncthreads();
    int w = kWarps - 1;
#pragma unroll
    for (int k = kWarps - 2; k >= 0; --k) w = fits[k] ? k : w;
    hi = lo + (int)(span * (w + 1) / kWarps);
    lo = (w == 0) ? lo : lo + (int)(span * w / kWarps) + 1;
  }
  const int pb = lo;
  // The item's (sequence, partition): prefix sums of partitions over
  // sequences, by chunks of 32 sequences per warp.
  const int nchunks = (B + 31) / 32;
  for (int ch = warp; ch < nchunks; ch += kWarps) {
    const int i = ch * 32 + lane;
    int v = i < B ? parts_of(sc.nb[i], pb) : 0;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) v += __shfl_xor_sync(0xffffffffu, v, x);
    if (lane == 0) sc.chunk[ch] = v;
  }
  __syncthreads();
  const int q = blockIdx.x / p.kv_groups;  // the item's (sequence, partition) index
  int all = 0;
  for (int ch = 0; ch < nchunks; ++ch) all += sc.chunk[ch];
  for (int ch = warp; ch < nchunks; ch += kWarps) {
    int before = 0;
    for (int k = 0; k < ch; ++k) before += sc.chunk[k];
    const int i = ch * 32 + lane;
    const int mine = i < B ? parts_of(sc.nb[i], pb) : 0;
    int incl = mine;
#pragma unroll
    for (int x = 1; x < 32; x <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, x);
      if (lane >= x) incl += o;
    }
    const int excl = before + incl - mine;
    if (q >= excl && q < excl + mine) {
      sc.pick[0] = i;
      sc.pick[1] = q - excl;
    }
  }
  __syncthreads();
  BalancedItem it;
  it.pb = pb;
  it.valid = q < all && sc.pick[0] >= 0;
  it.seq = it.valid ? sc.pick[0] : 0;
  it.part = it.valid ? sc.pick[1] : 0;
  it.kvg = blockIdx.x % p.kv_groups;
  it.len = -1;
  return it;
}

template <int D, int KV, int QT, bool kAppend>
__global__ void __launch_bounds__(DecodeCfg<D, KV>::kThreads, DecodeCfg<D, KV>::kMinCtasPerSm)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using C = DecodeCfg<D, KV>;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kRingBytes);
  uint64_t* empty_bar = full_bar + C::kStages;

  // Launched with programmatic stream serialisation, this grid may start while
  // the kernel before it on the stream is still running; that kernel may have
  // written any input (q, tables, lengths, the pool), so every thread waits
  // for it before its first global read.  (The tensor maps are parameters.)
  if (threadIdx.x == C::kConsumerWarps * 32) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  griddep_wait();
  int kvg = blockIdx.x, part = blockIdx.y, seq = blockIdx.z;
  int pb = p.partition_blocks;
  int L = -1;
  if (pb == 0) {
    __shared__ BalancedScratch plan_scratch;
    const BalancedItem item = balanced_plan<C::kThreads>(p, plan_scratch);
    if (threadIdx.x == 0 && blockIdx.x == 0) *p.plan = item.pb;
    if (!item.valid) return;
    pb = item.pb;
    kvg = item.kvg;
    part = item.part;
    seq = item.seq;
    L = item.len;
  }
  // A length past the table's capacity is cut to it: no entry past the row is read.
  if (L < 0) L = min(p.context_lens[seq], p.max_blocks_per_seq * 16);
  const int part_tokens = pb * 16;
  const int tok0 = part * part_tokens;
  if (part > 0 && tok0 >= L) return;  // past the end of this sequence
  const int ntok = min(L - tok0, part_tokens);
  const int nblk = ntok > 0 ? (ntok + 15) >> 4 : 0;
  const int nparts_seq = (L + part_tokens - 1) / part_tokens;  // 0 when L == 0
  const int kv0 = kvg * C::kHeads;  // the group's first KV head

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], C::kHeads);
    }
    mbar_fence_init();
  }
  __syncthreads();

  WarpState<D> st;
  st.reset();

  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int32_t* tbl =
        p.block_tables + (size_t)seq * p.max_blocks_per_seq + (size_t)part * pb;
    int mine = (lane < nblk) ? __ldg(tbl + lane) : 0;
    if constexpr (kAppend) {
      // append_kv for this sequence's new token, the group's heads: the CTA
      // holding the partition with position L - 1 writes it, then makes the
      // write visible to its own TMA loads (generic -> async proxy) before
      // issuing them.
      const int64_t slot = (L > 0 && part == nparts_seq - 1) ? p.slot_mapping[seq] : -1;
      append_token<D, KV, QT>(p, seq, kv0, slot);
    }
    const uint64_t kv_policy = l2_evict_first_policy();  // the KV stream is read once
    bool ok = true;
    int issued = 0;
    for (int base = 0; base < nblk; base += 32) {
      if (base > 0) mine = (base + lane < nblk) ? __ldg(tbl + base + lane) : 0;
      const int cnt = min(32, nblk - base);
      for (int j = 0; j < cnt; ++j) {
        const int blk = __shfl_sync(0xffffffffu, mine, j);
        if (lane == 0 && ok) {
          const int it = base + j;
          const int s = it % C::kStages;
          const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
          if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, p.status)) {
            ok = false;
          } else {
            load_block<D, KV>(smem + s * C::kStageBytes, &tmap_k, &tmap_v, &full_bar[s], blk,
                              p.num_blocks, kv0, kv_policy);
            ++issued;
          }
        }
      }
    }
    // Never leave the CTA with copies in flight: wait (bounded) for the last
    // stages this producer filled.
    if (lane == 0) {
      const int first = max(0, issued - C::kStages);
      for (int it = first; it < issued; ++it) {
        mbar_wait_bounded(&full_bar[it % C::kStages], (uint32_t)(it / C::kStages) & 1u, p.status);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // Warp 4j + w serves head j of the group; a head past the last KV head
    // (odd count) sees zero-filled tiles and writes nothing.
    const int hsel = warp / C::kWarpsPerHead;
    const int kvh = kv0 + hsel;
    const int head0 = kvh * p.group;
    const int g = lane >> 2;
    const bool head_live = kvh < p.num_kv_heads && g < p.group;
    const size_t qrow = ((size_t)seq * p.num_q_heads + head0 + (head_live ? g : 0)) * D;
    uint32_t qb[C::kMTiles][2];
    load_q_frag<D, KV, QT>(qb, p.q, qrow, head_live);

    for (int it = warp % C::kWarpsPerHead; it < nblk; it += C::kWarpsPerHead) {
      const int s = it % C::kStages;
      const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
      if (!mbar_wait_bounded(&full_bar[s], ph, p.status)) break;
      const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
      const int valid = min(16, ntok - it * 16);
      decode_block<D, KV, false>(st, qb, kbase, kbase + C::kTileBytes, hsel, valid, p.scale_log2,
                                 16, 16);
      // Release the stage: this warp's reads of it (generic proxy) are ordered
      // before the TMA refill (async proxy) by the proxy fence, then the warp's
      // lanes by __syncwarp, then the producer by the mbarrier.
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    finish_row_sums(st);
  }

  // ---------------------------------------------------------------- merge warps
  __syncthreads();  // the ring is idle: reuse it for the per-warp states
  // All loads are done: the split-KV merge kernel may start launching; it
  // waits for this grid to finish before reading the partials.
  griddep_launch_dependents();
  float* red_o = reinterpret_cast<float*>(smem);                       // [warps][8][D+4]
  float* red_m = red_o + C::kConsumerWarps * 8 * C::kRedStride;          // [warps][8]
  float* red_l = red_m + C::kConsumerWarps * 8;                          // [warps][8]
  if (warp < C::kConsumerWarps) {
    dump_state<D, KV>(st, red_o + warp * 8 * C::kRedStride, red_m + warp * 8, red_l + warp * 8);
  }
  __syncthreads();

  // Combine each head's four warp states, four head_size elements per thread
  // and step (float4 reads of the buffer, 8- or 16-byte global stores).
  const bool direct = nparts_seq <= 1;
  constexpr int kQuads = D / 4;
  const int per_head = p.group * kQuads;
  for (int idx = threadIdx.x; idx < C::kHeads * per_head; idx += C::kThreads) {
    const int hs = idx / per_head;  // head of the group
    const int rem = idx - hs * per_head;
    const int h = rem / kQuads;
    const int d = (rem - h * kQuads) * 4;
    const int kvh = kv0 + hs;
    if (kvh >= p.num_kv_heads) break;  // later idx are past it too
    const int w0 = hs * C::kWarpsPerHead;
    float M = -INFINITY;
#pragma unroll
    for (int w = w0; w < w0 + C::kWarpsPerHead; ++w) M = fmaxf(M, red_m[w * 8 + h]);
    float num[4] = {0.f, 0.f, 0.f, 0.f}, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = w0; w < w0 + C::kWarpsPerHead; ++w) {
        const float wt = ex2_approx(__fsub_rn(red_m[w * 8 + h], M));
        const float4 ov = *reinterpret_cast<const float4*>(&red_o[(w * 8 + h) * C::kRedStride + d]);
        num[0] = __fmaf_rn(wt, ov.x, num[0]);
        num[1] = __fmaf_rn(wt, ov.y, num[1]);
        num[2] = __fmaf_rn(wt, ov.z, num[2]);
        num[3] = __fmaf_rn(wt, ov.w, num[3]);
        den = __fmaf_rn(wt, red_l[w * 8 + h], den);
      }
    }
    const int qh = kvh * p.group + h;
    if (direct) {
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[k] = (den > 0.f) ? __fmul_rn(__fdiv_rn(num[k], den), p.out_scale) : 0.f;
      uint2 pk;
      if constexpr (QT == kKvF16) {
        pk.x = pack_f16x2(v[0], v[1]);
        pk.y = pack_f16x2(v[2], v[3]);
      } else {
        pk.x = pack_bf16x2(v[0], v[1]);
        pk.y = pack_bf16x2(v[2], v[3]);
      }
      *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) +
                                ((size_t)seq * p.num_q_heads + qh) * D + d) = pk;
    } else {
      const size_t pi = ((size_t)seq * p.num_q_heads + qh) * p.num_partitions + part;
      *reinterpret_cast<float4*>(p.part_o + pi * D + d) = make_float4(num[0], num[1], num[2], num[3]);
      if (d == 0) {
        p.part_m[pi] = M;
        p.part_l[pi] = den;
      }
    }
  }
}

// Log-sum-exp merge of split-KV partials: one CTA of kMergeThreads per
// (sequence, query head).  The threads form kMergeThreads / D groups; group r
// takes partitions r, r + groups, ... and thread d of a group accumulates
// head_size element d with a running maximum (one pass: m, l and O of four
// partitions are loaded together, then folded in), so every partial's O row
// is read once, coalesced.  The groups' states are combined in a fixed order,
// so the result does not depend on timing.
constexpr int kMergeThreads = 256;

// Running log-sum-exp state of one head_size element: maximum M (log2
// domain), denominator and numerator, both scaled by 2^-M.
struct LseFold {
  float M = -INFINITY, acc = 0.f, den = 0.f;
  __device__ __forceinline__ void fold(float mx, int n, const float* mv, const float* lv,
                                       const float* ov) {
    const float Mn = fmaxf(M, mx);
    if (Mn == -INFINITY) return;  // nothing seen yet
    const float sc = ex2_approx(__fsub_rn(M, Mn));  // 0 when M is still -inf
    acc = __fmul_rn(acc, sc);
    den = __fmul_rn(den, sc);
    for (int u = 0; u < n; ++u) {
      const float w = ex2_approx(__fsub_rn(mv[u], Mn));
      den = __fmaf_rn(w, lv[u], den);
      acc = __fmaf_rn(w, ov[u], acc);
    }
    M = Mn;
  }
};

// Combine the kGroups fold states of element d (one per thread group, in
// group order) and store the normalised output; called by group 0's threads.
template <int D, int QT>
__device__ __forceinline__ void lse_combine_store(void* out, size_t row, int d, float out_scale,
                                                  const float (&red_acc)[kMergeThreads / D][D],
                                                  const float* red_den, const float* red_max) {
  constexpr int kGroups = kMergeThreads / D;
  float Mall = red_max[0];
#pragma unroll
  for (int g = 1; g < kGroups; ++g) Mall = fmaxf(Mall, red_max[g]);
  float a = 0.f, dn = 0.f;
  if (Mall != -INFINITY) {
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const float w = ex2_approx(__fsub_rn(red_max[g], Mall));
      a = __fmaf_rn(w, red_acc[g][d], a);
      dn = __fmaf_rn(w, red_den[g], dn);
    }
  }
  const float v = (dn > 0.f) ? __fmul_rn(__fdiv_rn(a, dn), out_scale) : 0.f;
  store_out<QT>(out, row * D + d, v);
}

template <int D, int QT>
__global__ void __launch_bounds__(kMergeThreads)
    paged_decode_merge_kernel(const DecodeParams p) {
  constexpr int kGroups = kMergeThreads / D;
  __shared__ float red_acc[kGroups][D];
  __shared__ float red_den[kGroups];
  __shared__ float red_max[kGroups];

  const int idx = blockIdx.x;  // sequence * num_q_heads + query head
  const int seq = idx / p.num_q_heads;
  // The kernel before this one is always the same call's attention kernel,
  // which writes no lengths: they may be read before the wait.
  const int L = min(p.context_lens[seq], p.max_blocks_per_seq * 16);
  // A balanced split never cuts a sequence shorter than its minimum partition.
  if (p.partition_blocks == 0 && L <= p.min_partition_blocks * 16) return;
  griddep_wait();  // the partials (and a balanced split's size) come from the attention kernel
  const int part_tokens = (p.partition_blocks ? p.partition_blocks : *p.plan) * 16;
  const int np = (L + part_tokens - 1) / part_tokens;
  if (np <= 1) return;  // written directly by the attention kernel
  const size_t base = (size_t)idx * p.num_partitions;
  const int tid = threadIdx.x;
  const int r = tid / D;
  const int d = tid - r * D;

  LseFold f;
  int i = r;
  for (; i + 3 * kGroups < np; i += 4 * kGroups) {
    float mv[4], lv[4], ov[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const size_t pi = base + i + u * kGroups;
      mv[u] = p.part_m[pi];
      lv[u] = p.part_l[pi];
      ov[u] = p.part_o[pi * D + d];
    }
    f.fold(fmaxf(fmaxf(mv[0], mv[1]), fmaxf(mv[2], mv[3])), 4, mv, lv, ov);
  }
  for (; i < np; i += kGroups) {
    const size_t pi = base + i;
    const float mv = p.part_m[pi], lv = p.part_l[pi], ov = p.part_o[pi * D + d];
    f.fold(mv, 1, &mv, &lv, &ov);
  }
  red_acc[r][d] = f.acc;
  if (d == 0) {
    red_den[r] = f.den;
    red_max[r] = f.M;
  }
  __syncthreads();
  if (r == 0) lse_combine_store<D, QT>(p.out, (size_t)idx, d, p.out_scale, red_acc, red_den, red_max);
}

}  // namespace pa
