// Paged decode attention: one CTA per (kv_head, KV partition, sequence).
//
// What it computes ("vLLM GitHub 项目…" section 二; "vLLM 部署深度指南" sections
// PagedAttention 方案 and 代码层面理解): for every sequence i and query head h,
//   out[i, h] = softmax(scale * q[i, h] . K_i^T) . V_i
// where K_i / V_i are the sequence's first L_i tokens, found block by block
// through its block table (logical block j // 16 -> physical block, offset
// j % 16) in the pool [num_blocks, 16, 2, Hkv, D].  Query head h reads KV head
// h / G (G = Hq / Hkv), so each CTA serves the G query heads of one KV head and
// reads every K/V byte of that head once.
//
// Layout of the work inside a CTA (160 threads):
//   * warp 4 (producer): one lane reads the partition's block-table entries
//     and issues one TMA load per 16-token block for K and one for V into a
//     ring of shared-memory stages, each guarded by a "full" and an "empty"
//     mbarrier.  Tiles land 128B-swizzled, so fragment loads are bank-conflict
//     free.
//   * warps 0-3 (consumers): warp w takes blocks w, w+4, ...  For each block it
//     computes S^T = K . Q^T with m16n8k16 tensor-core MMAs (tokens as M = 16,
//     the G <= 8 query heads as N = 8, head_size as K), runs the online softmax
//     on the fragment, turns P^T into the B operand with movmatrix, and
//     accumulates O^T += V^T . P^T (head_size as M).  All accumulation is fp32.
//   * at the end the four warps' (m, l, O) states are merged through shared
//     memory; the CTA writes the normalised output (one partition) or an fp32
//     partial (m, l, O) that the merge kernel combines by log-sum-exp.
//
// fp8-E4M3 KV: bytes are widened exactly to f16 in registers (cvt.f16x2.e4m3x2);
// q is rounded to f16; the per-tensor kv_scale multiplies the logits and the
// output.  For the byte loads the head_size index of K is permuted (the same
// permutation is applied to q, so the dot product is unchanged) and the
// head_size index of V maps to output rows in a lane-contiguous order.
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
  int group;                    // G = Hq / Hkv, 1..8
  int partition_blocks;         // partition size in 16-token blocks; 0 = balanced (below)
  // Balanced split: the partition size is chosen in the kernel from the actual
  // context lengths, as the smallest one (>= min_partition_blocks) whose
  // partitions over all sequences and KV heads fit in `slots` resident CTAs.
  int min_partition_blocks;
  int slots;
  int* plan;                    // balanced: the chosen size, for the merge kernel
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
};


template <int D, int KV>
struct DecodeCfg {
  static constexpr int kElt = (KV == kKvE4m3) ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;          // one token row of one head
  static constexpr int kTileBytes = 16 * kRowBytes;   // one block of K (or V) for one head
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
  static constexpr int kConsumerWarps = 4;
  // Block `it` goes to stage it % kStages and to consumer warp it % 4.  With
  // kStages a multiple of 4, every stage has one consumer warp that waits on
  // its phases strictly in order, so a parity wait never runs two phases ahead
  // of its barrier (which would let it pass early).  Two or more stages per
  // warp let the producer run ahead while a warp computes.  A CTA streams
  // about (ring bytes) / (loaded memory latency, ~3.5 us on GB300), so the
  // ring is 64 KB whatever the stage size.
  static constexpr int kStages = (kStageBytes >= 8192) ? 8 : 16;
  static_assert(kStages % kConsumerWarps == 0 && kStages >= 2 * kConsumerWarps,
                "each stage must belong to exactly one consumer warp");
  static constexpr int kSwizzle = (kRowBytes >= 128) ? 128 : 64;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kMTiles = D / 16;              // m-tiles of O^T, k-steps of S^T
  static constexpr int kRedStride = D + 4;            // floats per head row in the merge buffer
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kRingBytes + 1024 /*align*/ + 2 * kStages * 8;
  static_assert(kConsumerWarps * 8 * kRedStride * 4 + 2 * kConsumerWarps * 8 * 4 <= kRingBytes,
                "merge buffer must fit in the ring");
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

// Balanced split (partition_blocks == 0).  The grid is one dimension of
// `slots` CTAs (one wave on this GPU, or the number of (sequence, KV head)
// pairs if that is larger).  Every CTA computes the same plan from the actual
// context lengths:
//   pb = the smallest partition size in blocks, >= min_partition_blocks, with
//        num_kv_heads * sum_i max(1, ceil(ceil(L_i / 16) / pb)) <= slots;
// then takes work item blockIdx.x of the list ordered by (sequence, partition,
// KV head) -- each sequence has at least one item, so empty sequences still
// get their zero output.  Items past the list's end exit at once.
struct BalancedItem {
  int pb, seq, part, kvh;
  bool valid;
};

template <int kThreads>
__device__ __forceinline__ BalancedItem balanced_plan(const DecodeParams& p, int* red, int* pick) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kPer = 4;  // sequences per thread, contiguous (the mode has < 512 sequences)
  int nb[kPer];
  int total = 0, maxnb = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = threadIdx.x * kPer + k;
    const int L = i < p.num_seqs ? p.context_lens[i] : -1;
    nb[k] = L > 0 ? (L + 15) >> 4 : (L == 0 ? 0 : -1);  // -1: no such sequence
    total += max(nb[k], 0);
    maxnb = max(maxnb, nb[k]);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto block_reduce = [&](int v, bool is_max) {
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) {
      const int o = __shfl_xor_sync(0xffffffffu, v, x);
      v = is_max ? max(v, o) : v + o;
    }
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int r = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) r = is_max ? max(r, red[w]) : r + red[w];
    return r;
  };
  auto parts_of = [&](int pbv, int k) { return nb[k] < 0 ? 0 : max(1, (nb[k] + pbv - 1) / pbv); };
  total = block_reduce(total, false);
  maxnb = block_reduce(maxnb, true);
  const long long want = ((long long)total * p.num_kv_heads + p.slots - 1) / p.slots;
  int lo = max(p.min_partition_blocks, (int)(want < (1ll << 30) ? want : (1ll << 30)));
  int hi = max(lo, maxnb);  // count(maxnb) = pairs <= slots
  while (lo < hi) {
    const int mid = lo + (hi - lo) / 2;
    int c = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) c += parts_of(mid, k);
    if ((long long)block_reduce(c, false) * p.num_kv_heads <= p.slots) {
      hi = mid;
    } else {
      lo = mid + 1;
    }
  }
  const int pb = lo;
  // Exclusive prefix of partitions over sequences (threads hold consecutive
  // sequences), then find the item's sequence and partition.
  int mine = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) mine += parts_of(pb, k);
  int incl = mine;
#pragma unroll
  for (int x = 1; x < 32; x <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, x);
    if (lane >= x) incl += o;
  }
  __syncthreads();
  if (lane == 31) red[warp] = incl;
  if (threadIdx.x == 0) pick[0] = -1;
  __syncthreads();
  int before = incl - mine;
  for (int w = 0; w < warp; ++w) before += red[w];
  int all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) all += red[w];
  const int q = blockIdx.x / p.num_kv_heads;  // the item's (sequence, partition) index
  if (q >= before && q < before + mine) {
    int acc = before;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int n = parts_of(pb, k);
      if (q < acc + n) {
        pick[0] = threadIdx.x * kPer + k;
        pick[1] = q - acc;
        break;
      }
      acc += n;
    }
  }
  __syncthreads();
  BalancedItem it;
  it.pb = pb;
  it.valid = q < all && pick[0] >= 0;
  it.seq = it.valid ? pick[0] : 0;
  it.part = it.valid ? pick[1] : 0;
  it.kvh = blockIdx.x % p.num_kv_heads;
  return it;
}

template <int D, int KV, int QT, bool kAppend>
__global__ void __launch_bounds__(DecodeCfg<D, KV>::kThreads, 4)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using C = DecodeCfg<D, KV>;
  constexpr bool kFp8 = (KV == kKvE4m3);
  // The P^T / V operands of the PV product are f16 unless the cache is bf16.
  constexpr bool kBf16Mma = (KV == kKvBf16);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kRingBytes);
  uint64_t* empty_bar = full_bar + C::kStages;

  int kvh = blockIdx.x, part = blockIdx.y, seq = blockIdx.z;
  int pb = p.partition_blocks;
  if (pb == 0) {
    __shared__ int red[C::kThreads / 32];
    __shared__ int pick[2];
    const BalancedItem item = balanced_plan<C::kThreads>(p, red, pick);
    if (threadIdx.x == 0 && blockIdx.x == 0) *p.plan = item.pb;
    if (!item.valid) return;
    pb = item.pb;
    kvh = item.kvh;
    part = item.part;
    seq = item.seq;
  }
  const int L = p.context_lens[seq];
  const int part_tokens = pb * 16;
  const int tok0 = part * part_tokens;
  if (part > 0 && tok0 >= L) return;  // past the end of this sequence
  const int ntok = min(L - tok0, part_tokens);
  const int nblk = ntok > 0 ? (ntok + 15) >> 4 : 0;
  const int nparts_seq = (L + part_tokens - 1) / part_tokens;  // 0 when L == 0

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // Per-warp softmax state for heads 2t and 2t+1 (lane = 4g + t).
  const int g = lane >> 2;
  const int t = lane & 3;
  float o[C::kMTiles][4];
#pragma unroll
  for (int i = 0; i < C::kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
    }
    // The pool may have just been written by the preceding kernel (the step's
    // reshape_and_cache): wait for it before the first access to it.  Nothing
    // read before this point (q, tables, lengths) is written there.
    griddep_wait();
    if constexpr (kAppend) {
      // append_kv for this sequence's new token, head kvh: the CTA holding the
      // partition with position L - 1 writes it, then makes the write visible
      // to its own TMA loads (generic -> async proxy) before issuing them.
      if (L > 0 && part == nparts_seq - 1) {
        const int64_t slot = p.slot_mapping[seq];
        if (slot >= 0 && slot < (int64_t)p.num_blocks * 16) {
          constexpr int kSrcElt = 2;  // the new token comes in the q dtype
          const size_t src = (size_t)seq * p.src_stride_bytes + (size_t)kvh * D * kSrcElt;
          const size_t dst = (size_t)slot * (2ull * p.num_kv_heads * C::kRowBytes) +
                             (size_t)kvh * C::kRowBytes;
          if constexpr (!kFp8) {
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
                const uint16_t a = f32x2_to_e4m3x2(__fdiv_rn(x[4 * h], p.kv_scale),
                                                   __fdiv_rn(x[4 * h + 1], p.kv_scale));
                const uint16_t b = f32x2_to_e4m3x2(__fdiv_rn(x[4 * h + 2], p.kv_scale),
                                                   __fdiv_rn(x[4 * h + 3], p.kv_scale));
                q8[h] = (uint32_t)a | ((uint32_t)b << 16);
              }
              reinterpret_cast<uint2*>((isv ? p.v_cache : p.k_cache) + dst)[j] =
                  make_uint2(q8[0], q8[1]);
            }
          }
          fence_proxy_async_global();
        }
      }
      __syncwarp();
    }
    const int32_t* tbl =
        p.block_tables + (size_t)seq * p.max_blocks_per_seq + (size_t)part * pb;
    const int oob_row = p.num_blocks * 16;  // first token row past the pool: TMA fills zeros
    bool ok = true;
    int issued = 0;
    for (int base = 0; base < nblk; base += 32) {
      const int mine = (base + lane < nblk) ? __ldg(tbl + base + lane) : 0;
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
            const int row = (blk >= 0 && blk < p.num_blocks) ? blk * 16 : oob_row;
            uint8_t* ks = smem + s * C::kStageBytes;
            mbar_arrive_expect_tx(&full_bar[s], C::kStageBytes);
            if constexpr (C::kRowBytes > 128) {
              tma_load_4d(ks, &tmap_k, &full_bar[s], 0, 0, kvh, row);
              tma_load_4d(ks + C::kTileBytes, &tmap_v, &full_bar[s], 0, 0, kvh, row);
            } else {
              tma_load_3d(ks, &tmap_k, &full_bar[s], 0, kvh, row);
              tma_load_3d(ks + C::kTileBytes, &tmap_v, &full_bar[s], 0, kvh, row);
            }
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
    const int head0 = kvh * p.group;
    const bool head_live = g < p.group;
    const size_t qrow = ((size_t)seq * p.num_q_heads + head0 + (head_live ? g : 0)) * D;
    // B operand (Q^T): 2 registers per k-step.
    uint32_t qb[C::kMTiles][2];
#pragma unroll
    for (int s = 0; s < C::kMTiles; ++s) {
      if (!head_live) {
        qb[s][0] = qb[s][1] = 0u;
      } else if constexpr (!kFp8) {
        qb[s][0] = *reinterpret_cast<const uint32_t*>(
            reinterpret_cast<const uint16_t*>(p.q) + qrow + 16 * s + 2 * t);
        qb[s][1] = *reinterpret_cast<const uint32_t*>(
            reinterpret_cast<const uint16_t*>(p.q) + qrow + 16 * s + 2 * t + 8);
      } else {
        // head_size index permuted to match the K byte layout (see the header).
        const size_t d0 = qrow + (D / 4) * t + 4 * s;
        qb[s][0] = pack_f16x2(load_q_elem<QT>(p.q, d0), load_q_elem<QT>(p.q, d0 + 1));
        qb[s][1] = pack_f16x2(load_q_elem<QT>(p.q, d0 + 2), load_q_elem<QT>(p.q, d0 + 3));
      }
    }

    for (int it = warp; it < nblk; it += C::kConsumerWarps) {
      const int s = it % C::kStages;
      const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
      if (!mbar_wait_bounded(&full_bar[s], ph, p.status)) break;
      const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
      const uint32_t vbase = kbase + C::kTileBytes;
      const int valid = min(16, ntok - it * 16);

      // ---- S^T = K . Q^T  (rows: tokens, columns: query heads)
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (!kFp8) {
        const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int ks = 0; ks < C::kMTiles; ++ks) {
          uint32_t a[4];
          ldsm_x4(a, kbase + swz<C::kSwizzle>(tok * C::kRowBytes + (ks * 2 + (lane >> 4)) * 16));
          if constexpr (kBf16Mma) {
            mma_bf16(sacc, a, qb[ks][0], qb[ks][1]);
          } else {
            mma_f16(sacc, a, qb[ks][0], qb[ks][1]);
          }
        }
      } else {
        constexpr int kCpl = D / 64;  // 16-byte chunks per lane per row
        uint32_t wa[C::kMTiles], wb[C::kMTiles];
#pragma unroll
        for (int i = 0; i < kCpl; ++i) {
          const uint4 xa = lds128(kbase + swz<C::kSwizzle>(g * C::kRowBytes + (kCpl * t + i) * 16));
          const uint4 xb =
              lds128(kbase + swz<C::kSwizzle>((g + 8) * C::kRowBytes + (kCpl * t + i) * 16));
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
          mma_f16(sacc, a, qb[ks][0], qb[ks][1]);
        }
      }

      // ---- online softmax on the fragment: c0/c1 token g, c2/c3 token g+8
      // Every rounding step below is spelled out (_rn intrinsics), so no
      // instantiation of this kernel contracts them into FMAs differently:
      // all variants produce the same bits.
      float s0 = __fmul_rn(sacc[0], p.scale_log2), s1 = __fmul_rn(sacc[1], p.scale_log2);
      float s2 = __fmul_rn(sacc[2], p.scale_log2), s3 = __fmul_rn(sacc[3], p.scale_log2);
      if (valid < 16) {
        if (g >= valid) s0 = s1 = -INFINITY;
        if (g + 8 >= valid) s2 = s3 = -INFINITY;
      }
      float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
      }
      const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
      const float al0 = ex2_approx(__fsub_rn(m0, mn0)), al1 = ex2_approx(__fsub_rn(m1, mn1));
      m0 = mn0;
      m1 = mn1;
      const float p0 = ex2_approx(__fsub_rn(s0, mn0)), p1 = ex2_approx(__fsub_rn(s1, mn1));
      const float p2 = ex2_approx(__fsub_rn(s2, mn0)), p3 = ex2_approx(__fsub_rn(s3, mn1));
      uint32_t P01, P23;
      float r0, r1, r2, r3;  // the rounded probabilities the MMA will use
      if constexpr (kBf16Mma) {
        P01 = pack_bf16x2(p0, p1);
        P23 = pack_bf16x2(p2, p3);
        r0 = __uint_as_float(P01 << 16); r1 = __uint_as_float(P01 & 0xFFFF0000u);
        r2 = __uint_as_float(P23 << 16); r3 = __uint_as_float(P23 & 0xFFFF0000u);
      } else {
        P01 = pack_f16x2(p0, p1);
        P23 = pack_f16x2(p2, p3);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&P01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&P23));
        r0 = f01.x; r1 = f01.y; r2 = f23.x; r3 = f23.y;
      }
      l0 = __fmaf_rn(l0, al0, __fadd_rn(r0, r2));
      l1 = __fmaf_rn(l1, al1, __fadd_rn(r1, r3));
      if (__any_sync(0xffffffffu, (al0 != 1.f) || (al1 != 1.f))) {
#pragma unroll
        for (int i = 0; i < C::kMTiles; ++i) {
          o[i][0] = __fmul_rn(o[i][0], al0); o[i][1] = __fmul_rn(o[i][1], al1);
          o[i][2] = __fmul_rn(o[i][2], al0); o[i][3] = __fmul_rn(o[i][3], al1);
        }
      }
      // P^T as the B operand: k = tokens (2t, 2t+1 | 2t+8, 2t+9), n = head g.
      const uint32_t pb0 = movmatrix_trans(P01);
      const uint32_t pb1 = movmatrix_trans(P23);
      const uint32_t mlo = token_mask(2 * t, valid), mhi = token_mask(2 * t + 8, valid);

      // ---- O^T += V^T . P^T
      if constexpr (!kFp8) {
        const int mi = lane >> 3;
        const int tok = (lane & 7) + 8 * (mi >> 1);
#pragma unroll
        for (int mt = 0; mt < C::kMTiles; ++mt) {
          uint32_t a[4];
          ldsm_x4_trans(a, vbase + swz<C::kSwizzle>(tok * C::kRowBytes + (mt * 2 + (mi & 1)) * 16));
          if (valid < 16) {
            a[0] &= mlo; a[1] &= mlo; a[2] &= mhi; a[3] &= mhi;
          }
          if constexpr (kBf16Mma) {
            mma_bf16(o[mt], a, pb0, pb1);
          } else {
            mma_f16(o[mt], a, pb0, pb1);
          }
        }
      } else {
        // Lane (g, t) owns head_size indices [D/8 * g, D/8 * (g+1)) of tokens
        // 2t, 2t+1, 2t+8, 2t+9; m-tile mt row g is index D/8*g + 2mt, row g+8
        // is the next one.
        uint32_t va[D / 32], vb[D / 32], vc[D / 32], vd[D / 32];
        if constexpr (D == 128) {
          const uint32_t col = g * 16;
          const uint4 x0 = lds128(vbase + swz<C::kSwizzle>((2 * t) * C::kRowBytes + col));
          const uint4 x1 = lds128(vbase + swz<C::kSwizzle>((2 * t + 1) * C::kRowBytes + col));
          const uint4 x2 = lds128(vbase + swz<C::kSwizzle>((2 * t + 8) * C::kRowBytes + col));
          const uint4 x3 = lds128(vbase + swz<C::kSwizzle>((2 * t + 9) * C::kRowBytes + col));
          va[0] = x0.x; va[1] = x0.y; va[2] = x0.z; va[3] = x0.w;
          vb[0] = x1.x; vb[1] = x1.y; vb[2] = x1.z; vb[3] = x1.w;
          vc[0] = x2.x; vc[1] = x2.y; vc[2] = x2.z; vc[3] = x2.w;
          vd[0] = x3.x; vd[1] = x3.y; vd[2] = x3.z; vd[3] = x3.w;
        } else {
          const uint32_t col = g * 8;
          const uint2 x0 = lds64(vbase + swz<C::kSwizzle>((2 * t) * C::kRowBytes + col));
          const uint2 x1 = lds64(vbase + swz<C::kSwizzle>((2 * t + 1) * C::kRowBytes + col));
          const uint2 x2 = lds64(vbase + swz<C::kSwizzle>((2 * t + 8) * C::kRowBytes + col));
          const uint2 x3 = lds64(vbase + swz<C::kSwizzle>((2 * t + 9) * C::kRowBytes + col));
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
          if (valid < 16) {
            a[0] &= mlo; a[1] &= mlo; a[2] &= mhi; a[3] &= mhi;
          }
          mma_f16(o[mt], a, pb0, pb1);
        }
      }
      // Release the stage: this warp's reads of it (generic proxy) are ordered
      // before the TMA refill (async proxy) by the proxy fence, then the warp's
      // lanes by __syncwarp, then the producer by the mbarrier.
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    // Sum l over the 8 lanes that share t (tokens g and g+8 of every block).
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, x);
      l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    }
  }

  // ---------------------------------------------------------------- merge warps
  __syncthreads();  // the ring is idle: reuse it for the per-warp states
  // All loads are done: the split-KV merge kernel may start launching; it
  // waits for this grid to finish before reading the partials.
  griddep_launch_dependents();
  float* red_o = reinterpret_cast<float*>(smem);                       // [4][8][D+4]
  float* red_m = red_o + C::kConsumerWarps * 8 * C::kRedStride;          // [4][8]
  float* red_l = red_m + C::kConsumerWarps * 8;                          // [4][8]
  if (warp < C::kConsumerWarps) {
    float* mine = red_o + warp * 8 * C::kRedStride;
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt) {
      int d_lo, d_hi;
      if constexpr (kFp8) {
        d_lo = (D / 8) * g + 2 * mt;
        d_hi = d_lo + 1;
      } else {
        d_lo = 16 * mt + g;
        d_hi = d_lo + 8;
      }
      mine[(2 * t) * C::kRedStride + d_lo] = o[mt][0];
      mine[(2 * t + 1) * C::kRedStride + d_lo] = o[mt][1];
      mine[(2 * t) * C::kRedStride + d_hi] = o[mt][2];
      mine[(2 * t + 1) * C::kRedStride + d_hi] = o[mt][3];
    }
    if (g == 0) {
      red_m[warp * 8 + 2 * t] = m0;
      red_m[warp * 8 + 2 * t + 1] = m1;
      red_l[warp * 8 + 2 * t] = l0;
      red_l[warp * 8 + 2 * t + 1] = l1;
    }
  }
  __syncthreads();

  const bool direct = nparts_seq <= 1;
  for (int idx = threadIdx.x; idx < p.group * D; idx += C::kThreads) {
    const int h = idx / D;
    const int d = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) M = fmaxf(M, red_m[w * 8 + h]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < C::kConsumerWarps; ++w) {
        const float wt = ex2_approx(__fsub_rn(red_m[w * 8 + h], M));
        num = __fmaf_rn(wt, red_o[(w * 8 + h) * C::kRedStride + d], num);
        den = __fmaf_rn(wt, red_l[w * 8 + h], den);
      }
    }
    const int qh = kvh * p.group + h;
    if (direct) {
      const float v = (den > 0.f) ? __fmul_rn(__fdiv_rn(num, den), p.out_scale) : 0.f;
      store_out<QT>(p.out, ((size_t)seq * p.num_q_heads + qh) * D + d, v);
    } else {
      const size_t pi = ((size_t)seq * p.num_q_heads + qh) * p.num_partitions + part;
      p.part_o[pi * D + d] = num;
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
// head_size element d, so every partial's O row is read once, coalesced, with
// several independent loads in flight per thread.  The groups' sums are added
// in a fixed order, so the result does not depend on timing.
constexpr int kMergeThreads = 256;

template <int D, int QT>
__global__ void __launch_bounds__(kMergeThreads)
    paged_decode_merge_kernel(const DecodeParams p) {
  constexpr int kGroups = kMergeThreads / D;
  __shared__ float red_acc[kGroups][D];
  __shared__ float red_den[kGroups];
  __shared__ float red_max[kMergeThreads / 32];

  const int idx = blockIdx.x;  // sequence * num_q_heads + query head
  const int seq = idx / p.num_q_heads;
  const int L = p.context_lens[seq];
  // A balanced split never cuts a sequence shorter than its minimum partition.
  if (p.partition_blocks == 0 && L <= p.min_partition_blocks * 16) return;
  griddep_wait();  // the partials (and a balanced split's size) come from the attention kernel
  const int part_tokens = (p.partition_blocks ? p.partition_blocks : *p.plan) * 16;
  const int np = (L + part_tokens - 1) / part_tokens;
  if (np <= 1) return;  // written directly by the attention kernel
  const size_t base = (size_t)idx * p.num_partitions;
  const int tid = threadIdx.x;

  float M = -INFINITY;
  for (int i = tid; i < np; i += kMergeThreads) M = fmaxf(M, p.part_m[base + i]);
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
  if ((tid & 31) == 0) red_max[tid >> 5] = M;
  __syncthreads();
  M = red_max[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, red_max[w]);

  const int r = tid / D;
  const int d = tid - r * D;
  float acc = 0.f, den = 0.f;
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
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = ex2_approx(__fsub_rn(mv[u], M));
      den = __fmaf_rn(w, lv[u], den);
      acc = __fmaf_rn(w, ov[u], acc);
    }
  }
  for (; i < np; i += kGroups) {
    const size_t pi = base + i;
    const float w = ex2_approx(__fsub_rn(p.part_m[pi], M));
    den = __fmaf_rn(w, p.part_l[pi], den);
    acc = __fmaf_rn(w, p.part_o[pi * D + d], acc);
  }
  red_acc[r][d] = acc;
  if (d == 0) red_den[r] = den;
  __syncthreads();
  if (r == 0) {
    float a = red_acc[0][d], dn = red_den[0];
#pragma unroll
    for (int g = 1; g < kGroups; ++g) {
      a = __fadd_rn(a, red_acc[g][d]);
      dn = __fadd_rn(dn, red_den[g]);
    }
    const float v = (dn > 0.f) ? __fmul_rn(__fdiv_rn(a, dn), p.out_scale) : 0.f;
    store_out<QT>(p.out, (size_t)idx * D + d, v);
  }
}

}  // namespace pa
