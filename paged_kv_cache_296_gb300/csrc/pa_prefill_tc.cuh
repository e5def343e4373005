// Paged prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes is the causal paged prefill of pa_prefill_params.cuh: the
// query at position p of sequence i, head h, attends to that sequence's tokens
// 0..p of KV head h / G through its block table.
//
// One CTA per (two tiles of 128 rows, KV head, sequence), one CTA per SM; a
// row is one (query token, query head of the KV head's group) pair,
// token-major.  Keys go in chunks of 128 (8 blocks).  320 threads:
//   * warps 0-3 and 4-7 (softmax, one group per tile): thread r owns row r of
//     its tile, which is TMEM lane r of the tile's 256 columns.  They
//     stage Q into shared memory, run the online softmax on each S chunk read
//     from TMEM (in one load, or in two halves when an E4M3 cache leaves 128
//     registers a thread), write P (16-bit) back over it (keys 0..63 at columns
//     0..31, keys 64..127 at 64..95), rescale O in TMEM when a row's
//     running maximum grows by more than kRescale (log2 units; otherwise the
//     exponentials keep the older maximum, so P stays below 2^kRescale), and
//     finally normalise O and store the rows.
//   * warp 8 (producer): TMA loads of the chunks' K and V blocks into two
//     rings (K and V, each with full/empty mbarriers per chunk; K is released
//     as soon as S has read it, V after P V).  The rings are plane-major: each
//     128-byte piece of the rows has its own plane, 128B-swizzled, so the 8
//     blocks of a chunk are one 128-row operand.  It also zeroes the V rows
//     past the context's end in the last block (a P of 0 times a stale or
//     poisoned V must not reach the sum).
//   * warp 9 (MMA): owns the TMEM allocation; one thread issues, tile by tile,
//     O_t += P_t(c) V(c) (A = P from TMEM, B = each block's V rows, MN-major,
//     N = head size, K = 16) and then S_t(c + 1) = Q_t K(c + 1)^T (M = 128,
//     N = 128 keys, K = head size, A and B from shared memory) into the
//     columns P_t(c) occupied.  One thread's MMAs run in order, so P V(c) has
//     read P(c) before S(c + 1) overwrites it, and a completed S(c + 1) means
//     P V(c) is done too (the softmax may rescale O then).  The tensor core
//     works on one tile while the other tile's softmax runs.
// Accumulation in fp32 throughout; every wait is bounded.
#pragma once

#include "pa_ptx.cuh"
#include "pa_prefill_params.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

// Four E4M3 bytes (byte i -> element i) to four f16: elements 0, 1 in lo, 2, 3 in hi.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// KV8: the cache holds E4M3 codes.  The TMA then loads fp8 rows into rings of
// their own and eight converter warps (four for K, four for V) widen each chunk
// into 16-bit staging planes laid out like the 16-bit rings (one chunk of K; two
// of V, so that V(c + 1) is widened while the P V MMAs of chunk c read V(c)),
// which the MMAs read; the MMAs run in f16 (every E4M3 value is exact in
// f16).  The widening (cvt.f16x2.e4m3x2) is throughput-bound, so it is spread
// over many warps: 18 in all, 96 registers each (2 or 3 converter warps per
// operand measured slower).
template <int D, bool KV8>
struct PrefillTcCfg {
  static constexpr int kRows = 128;                        // rows of one tile (TMEM lanes)
  static constexpr int kTiles = 2;                         // tiles per CTA, one softmax group each
  static constexpr int kPieces = D * 2 / 128;              // 128-byte pieces of a 16-bit row
  static constexpr int kQTileBytes = kRows * D * 2;        // [pieces][128 rows][128 B]
  static constexpr int kQBytes = kTiles * kQTileBytes;
  static constexpr int kBlocksPerChunk = 8;                // 128 keys per S = Q K^T
  static constexpr int kBlockBytes = 16 * 128;             // one block, one piece: [16][128 B]
  static constexpr int kChunkBytes = kBlocksPerChunk * kBlockBytes;  // one chunk, one piece
  static constexpr int kChunkBytes8 = kBlocksPerChunk * 16 * D;      // one chunk of fp8 rows
  static constexpr int kRingBytes = KV8 ? 64 * 1024 : 128 * 1024;    // K and V rings
  static constexpr int kRing =                                        // chunks per ring
      KV8 ? kRingBytes / (2 * kChunkBytes8) : kRingBytes / (2 * kPieces * kChunkBytes);
  // one piece plane of K (or V): the whole ring, or (KV8) one staged chunk
  static constexpr int kPlaneBytes = KV8 ? kChunkBytes : kRing * kChunkBytes;
  static constexpr int kRingPart = KV8 ? kRing * kChunkBytes8 : kPieces * kPlaneBytes;
  static constexpr int kKOff = kQBytes;                    // K ring
  static constexpr int kVOff = kKOff + kRingPart;          // V ring
  static constexpr int kStBytes = kPieces * kPlaneBytes;  // KV8: one staged 16-bit chunk
  static constexpr int kVStages = 2;                       // KV8: staged V chunks
  static constexpr int kKStOff = kVOff + kRingPart;        // KV8: 16-bit K of one chunk
  static constexpr int kVStOff = kKStOff + (KV8 ? kStBytes : 0);  // KV8: 16-bit V, two chunks
  static constexpr int kBarOff = kVStOff + (KV8 ? kVStages * kStBytes : 0);
  // barriers: K full / empty, V full / empty per ring slot; s_full, p_full per
  // tile; q_ready, tail, o_done; KV8: staged K full / empty, staged V full and
  // empty per staged chunk
  static constexpr int kNumBars = 4 * kRing + 2 * kTiles + 3 + (KV8 ? 2 + 2 * kVStages : 0);
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static constexpr int kSoftmaxThreads = 128 * kTiles;
  static constexpr int kProducerWarp = kSoftmaxThreads / 32;
  static constexpr int kMmaWarp = kProducerWarp + 1;
  static constexpr int kConvWarp = kMmaWarp + 1;           // KV8: K converters, then V converters
  static constexpr int kConvWarps = 4;                     // KV8: warps per operand
  static constexpr int kThreads = kSoftmaxThreads + 64 + (KV8 ? 64 * kConvWarps : 0);
  // TMEM columns of tile t (base 256 t): O [0, D); S(c) in fp32 at [128, 256),
  // then P(c) (16-bit pairs) over it once the softmax has read it: keys 0..63
  // at [128, 160), keys 64..127 at [192, 224)
  static constexpr int kTileCols = 256;
  static constexpr int kS0 = 128;
  static constexpr int kTmemCols = kTileCols * kTiles;
  static constexpr float kRescale = 8.f;
  static_assert(D <= kS0 && kS0 + 128 <= kTileCols && kTmemCols <= 512, "TMEM layout");
  static_assert(kRing >= 2, "ring of at least two chunks");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// QT: 0 = fp16, 1 = bf16 (q and out); KV8: the cache holds E4M3 codes (else q's type).
template <int D, int QT, bool KV8>
__global__ void __launch_bounds__(PrefillTcCfg<D, KV8>::kThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
  using C = PrefillTcCfg<D, KV8>;
  constexpr int MT = KV8 ? 0 : QT;  // the MMAs' 16-bit type (P, and Q as staged)
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int kT = C::kTiles;
  constexpr int kR = C::kRing;
  constexpr int kBpc = C::kBlocksPerChunk;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full_k = bars;  // [kR] each
  uint64_t* empty_k = bars + kR;
  uint64_t* full_v = bars + 2 * kR;
  uint64_t* empty_v = bars + 3 * kR;
  uint64_t* s_full = bars + 4 * kR;  // [kT] each
  uint64_t* p_full = s_full + kT;
  uint64_t* q_ready = p_full + kT;
  uint64_t* tail_bar = q_ready + 1;
  uint64_t* o_done = q_ready + 2;
  uint64_t* kst_full = o_done + 1;  // KV8: the staged 16-bit K chunk
  uint64_t* kst_empty = o_done + 2;
  uint64_t* vst_full = o_done + 3;  // KV8: [kVStages] each, the staged 16-bit V chunks
  uint64_t* vst_empty = vst_full + C::kVStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == C::kProducerWarp * 32) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  griddep_wait();

  // One flat grid in bands of p.band tile indices, the heaviest (last) band
  // first; within a band the tiles of one (sequence, KV head) are adjacent so
  // that they run together and read its K/V through L2 once.  A band of 1
  // starts every CTA of a heavier tile index before any lighter one.
  int kvh, seq, group_tile;
  {
    const unsigned kBand = (unsigned)p.band;
    const unsigned groups = (unsigned)p.num_kv_heads * (unsigned)p.num_seqs;
    const unsigned full = ((unsigned)p.tiles / kBand) * kBand * groups;  // CTAs in full bands
    unsigned band, group, in_band;
    if (blockIdx.x < full) {
      band = blockIdx.x / (kBand * groups);
      const unsigned rem = blockIdx.x % (kBand * groups);
      group = rem / kBand;
      in_band = rem % kBand;
    } else {
      const unsigned tb = (unsigned)p.tiles % kBand;  // tiles of the last, partial band
      const unsigned rem = blockIdx.x - full;
      band = (unsigned)p.tiles / kBand;
      group = rem / tb;
      in_band = rem % tb;
    }
    kvh = (int)(group % (unsigned)p.num_kv_heads);
    seq = (int)(group / (unsigned)p.num_kv_heads);
    group_tile = p.tiles - 1 - (int)(band * kBand + in_band);
  }
  const int r0q = p.query_start_loc[seq];
  const int nq = p.query_start_loc[seq + 1] - r0q;
  const int L = min(p.context_lens[seq], p.max_blocks_per_seq * 16);
  if (nq <= 0) return;
  if (nq > L || nq > p.max_query_len) {
    if (threadIdx.x == 0 && group_tile == 0 && kvh == 0) atomicOr(p.status, kErrBadQueryLayout);
    return;
  }
  const int G = p.group;
  const int rows = nq * G;
  const int row0 = group_tile * kT * C::kRows;  // the CTA's first row (tile 0), tile t at + 128 t
  if (row0 >= rows) return;
  const int last_row = min(rows, row0 + kT * C::kRows) - 1;
  const int last_pos = L - nq + last_row / G;
  const int nkb = last_pos / 16 + 1;
  const int nchunks = (nkb + kBpc - 1) / kBpc;
  // The last block holds keys past the context's end when it is the block of
  // position L - 1 and L is not a multiple of 16.
  const bool has_tail = (nkb - 1 == (L - 1) / 16) && (L % 16 != 0);
  const bool bf16 = MT == 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kR; ++i) {
      // KV8: a ring slot is released by every lane of the operand's converter warps
      mbar_init(&full_k[i], 1);
      mbar_init(&empty_k[i], KV8 ? 32 * C::kConvWarps : 1);
      mbar_init(&full_v[i], 1);
      mbar_init(&empty_v[i], KV8 ? 32 * C::kConvWarps : 1);
    }
    if constexpr (KV8) {
      mbar_init(kst_full, 32 * C::kConvWarps);
      mbar_init(kst_empty, 1);
      for (int i = 0; i < C::kVStages; ++i) {
        mbar_init(&vst_full[i], 32 * C::kConvWarps);
        mbar_init(&vst_empty[i], 1);
      }
    }
    for (int t = 0; t < kT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
    }
    mbar_init(q_ready, C::kSoftmaxThreads);
    mbar_init(tail_bar, 1);
    mbar_init(o_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == C::kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() { atomicExch(abort_flag, 1); };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(abort_flag) != 0; };

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Chunk c goes to ring slot c % kR: block j of it lands at rows
    // 16 j .. 16 j + 15 of the slot in each piece's plane, K then V (KV8: at
    // rows 16 j .. of the slot's [128 rows][D bytes] tile, one load per block).
    const int32_t* tbl = p.block_tables + (size_t)seq * p.max_blocks_per_seq;
    const int oob_row = p.num_blocks * 16;
    const uint64_t pol = l2_evict_normal_policy();
    int issued = 0;  // chunks whose K and V are both in flight
    for (int c = 0; c < nchunks; ++c) {
      // lane j < nblk loads block j of the chunk, once lane 0 holds the slot
      const int b0 = kBpc * c;
      const int nblk = min(kBpc, nkb - b0);
      const int blk = lane < nblk ? __ldg(tbl + b0 + lane) : 0;
      const int brow = (blk >= 0 && blk < p.num_blocks) ? blk * 16 : oob_row;
      const int slot = c % kR;
      const uint32_t ph = ((uint32_t)(c / kR) & 1u) ^ 1u;
      const uint32_t bytes =
          (uint32_t)(KV8 ? nblk * 16 * D : nblk * C::kPieces * C::kBlockBytes);
      const uint32_t off = KV8 ? slot * C::kChunkBytes8 + lane * 16 * D
                               : slot * C::kChunkBytes + lane * C::kBlockBytes;
      int ok = 0;
      if (lane == 0 && !aborted() && mbar_wait_bounded(&empty_k[slot], ph, p.status)) {
        mbar_arrive_expect_tx(&full_k[slot], bytes);
        ok = 1;
      }
      if (!__shfl_sync(kAll, ok, 0)) break;
      if (lane < nblk) {
        if constexpr (KV8) {
          tma_load_3d(smem + C::kKOff + off, &tmap_k, &full_k[slot], 0, kvh, brow, pol);
        } else {
#pragma unroll
          for (int pc = 0; pc < C::kPieces; ++pc)
            tma_load_4d(smem + C::kKOff + pc * C::kPlaneBytes + off, &tmap_k, &full_k[slot], 0,
                        brow, pc, kvh, pol);
        }
      }
      ok = 0;
      if (lane == 0 && !aborted() && mbar_wait_bounded(&empty_v[slot], ph, p.status)) {
        mbar_arrive_expect_tx(&full_v[slot], bytes);
        ok = 1;
      }
      if (!__shfl_sync(kAll, ok, 0)) break;
      if (lane < nblk) {
        if constexpr (KV8) {
          tma_load_3d(smem + C::kVOff + off, &tmap_v, &full_v[slot], 0, kvh, brow, pol);
        } else {
#pragma unroll
          for (int pc = 0; pc < C::kPieces; ++pc)
            tma_load_4d(smem + C::kVOff + pc * C::kPlaneBytes + off, &tmap_v, &full_v[slot], 0,
                        brow, pc, kvh, pol);
        }
      }
      ++issued;
    }
    if (issued < nchunks && lane == 0) fail();
    if (!KV8 && lane == 0 && has_tail && !aborted() && issued == nchunks) {
      // zero the V rows of keys L .. 16 * nkb - 1 once the last chunk's V has landed
      // (KV8: the V converter writes zeros for them)
      const int c = nchunks - 1;
      const int slot = c % kR;
      const int j = nkb - 1 - kBpc * c;
      if (!mbar_wait_bounded(&full_v[slot], (uint32_t)(c / kR) & 1u, p.status)) {
        fail();
      } else {
        for (int key = L % 16; key < 16; ++key) {
          for (int pc = 0; pc < C::kPieces; ++pc) {
            uint4* row = reinterpret_cast<uint4*>(smem + C::kVOff + pc * C::kPlaneBytes +
                                                  slot * C::kChunkBytes + j * C::kBlockBytes +
                                                  key * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) row[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_shared();
        mbar_arrive(tail_bar);
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = umma_idesc(bf16, 128, 16 * kBpc, 0);
      const uint32_t id_pv = umma_idesc(bf16, 128, D, 1);
      // descriptors are formed once; an operand's step is a constant added to the low word
      const uint32_t q_lo = umma_desc_lo(sbase, 16);
      const uint32_t k_lo = umma_desc_lo(sbase + (KV8 ? C::kKStOff : C::kKOff), 16);
      const uint32_t v_lo = umma_desc_lo(sbase + (KV8 ? C::kVStOff : C::kVOff), C::kPlaneBytes);
      // KV8: one staged K chunk and two staged V chunks (each released once its MMAs
      // are done), else ring slots
      auto slot_lo = [&](int c) { return KV8 ? 0u : (uint32_t)((c % kR) * C::kChunkBytes >> 4); };
      auto vslot_lo = [&](int c) {
        return KV8 ? (uint32_t)((c % C::kVStages) * C::kStBytes >> 4) : slot_lo(c);
      };
      auto wait_k = [&](int c) {
        return KV8 ? mbar_wait_bounded(kst_full, (uint32_t)c & 1u, p.status)
                   : mbar_wait_bounded(&full_k[c % kR], (uint32_t)(c / kR) & 1u, p.status);
      };
      auto issue_s = [&](int t, int c) {  // S_t(c) = Q_t K(c)^T
        const uint32_t dcol = tmem + t * C::kTileCols + C::kS0;
        const uint32_t qa = q_lo + (uint32_t)(t * C::kQTileBytes >> 4);
        const uint32_t ka = k_lo + slot_lo(c);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          constexpr int kQStep = C::kRows * 128;
          const uint32_t qo = (uint32_t)(((k / 4) * kQStep + (k % 4) * 32) >> 4);
          const uint32_t ko = (uint32_t)(((k / 4) * C::kPlaneBytes + (k % 4) * 32) >> 4);
          umma_ss(dcol, umma_desc_join(qa + qo), umma_desc_join(ka + ko), id_s, k > 0 ? 1 : 0);
        }
        umma_commit(&s_full[t]);
      };
      bool ok = mbar_wait_bounded(q_ready, 0, p.status) && wait_k(0);
      tc_fence_after();
      if (ok) {
        for (int t = 0; t < kT; ++t) issue_s(t, 0);
        umma_commit(KV8 ? kst_empty : &empty_k[0]);
      }
      for (int c = 0; c < nchunks && ok; ++c) {
        const int slot = c % kR;
        const int nblk = min(kBpc, nkb - kBpc * c);
        const bool more = c + 1 < nchunks;
        if constexpr (KV8) {
          ok = mbar_wait_bounded(&vst_full[c % C::kVStages], (uint32_t)(c / C::kVStages) & 1u,
                                 p.status);
        } else {
          ok = mbar_wait_bounded(&full_v[slot], (uint32_t)(c / kR) & 1u, p.status);
          if (ok && has_tail && !more) ok = mbar_wait_bounded(tail_bar, 0, p.status);
        }
        for (int t = 0; t < kT && ok; ++t) {
          // O_t += P_t(c) V(c), then S_t(c + 1) into the same columns
          ok = mbar_wait_bounded(&p_full[t], (uint32_t)c & 1u, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t pcol = tmem + t * C::kTileCols + C::kS0;
          const uint32_t va = v_lo + vslot_lo(c);
          auto pv = [&](int j) {
            umma_ts(tmem + t * C::kTileCols, pcol + 64 * (j / 4) + 8 * (j % 4),
                    umma_desc_join(va + (uint32_t)(j * (C::kBlockBytes >> 4))), id_pv,
                    (c > 0 || j > 0) ? 1 : 0);
          };
          if (nblk == kBpc) {
#pragma unroll
            for (int j = 0; j < kBpc; ++j) pv(j);
          } else {
            for (int j = 0; j < nblk; ++j) pv(j);
          }
          if (t == kT - 1) umma_commit(KV8 ? &vst_empty[c % C::kVStages] : &empty_v[slot]);
          if (more) {
            if (t == 0) {
              ok = wait_k(c + 1);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(t, c + 1);
            if (t == kT - 1) umma_commit(KV8 ? kst_empty : &empty_k[(c + 1) % kR]);
          }
        }
      }
      if (ok) umma_commit(o_done);
      if (!ok) fail();
    }
    __syncwarp();
  } else if (KV8 && warp >= C::kConvWarp) {
    // ------------------------------------------------------------ converters (KV8)
    // Warps kConvWarp .. + kConvWarps - 1 widen K, the next kConvWarps V: each
    // 16-byte run of a landed fp8 row (16 codes) becomes 32 bytes of f16 in the
    // staging planes, at the positions the TMA would have put a 16-bit row; a
    // lane loads kBatch runs before converting them.  V rows of keys at or past
    // L become zeros (a P of 0 times a stale code must not reach the sum).
    const bool isv = warp >= C::kConvWarp + C::kConvWarps;
    const int cw = (warp - C::kConvWarp) % C::kConvWarps;  // this warp's share of the runs
    const int cl = cw * 32 + lane;
    uint64_t* full = isv ? full_v : full_k;
    uint64_t* empty = isv ? empty_v : empty_k;
    uint64_t* st_full = isv ? vst_full : kst_full;
    uint64_t* st_empty = isv ? vst_empty : kst_empty;
    const int nst = isv ? C::kVStages : 1;  // staged chunks of this operand
    const uint8_t* ring = smem + (isv ? C::kVOff : C::kKOff);
    uint8_t* st = smem + (isv ? C::kVStOff : C::kKStOff);
    constexpr int kRuns = D / 16;  // 16-byte runs of an fp8 row
    constexpr int kStride = 32 * C::kConvWarps;  // runs between one lane's consecutive runs
    static_assert(kStride % kRuns == 0, "a lane keeps one run index in every row");
    constexpr int kRStep = kStride / kRuns;  // rows between one lane's consecutive runs
    // run u = r * kRuns + j of a chunk: this lane takes j = cl % kRuns in rows
    // cl / kRuns, + kRStep, ...; its f16 elements 16 j .. 16 j + 15 go to piece
    // j / 4, 16-byte chunks 2 (j % 4) and + 1 of the staged row
    const int j = cl % kRuns;
    const int r_first = cl / kRuns;
    const int cc = 2 * (j % 4);
    uint8_t* const dst0 = st + (j / 4) * C::kPlaneBytes;
    for (int c = 0; c < nchunks; ++c) {
      const int slot = c % kR;
      const int si = c % nst;  // the staged chunk this chunk goes to
      uint8_t* const dst = dst0 + si * C::kStBytes;
      const bool w =
          mbar_wait_bounded(&full[slot], (uint32_t)(c / kR) & 1u, p.status) &&
          mbar_wait_bounded(&st_empty[si], ((uint32_t)(c / nst) & 1u) ^ 1u, p.status);
      if (!__all_sync(kAll, w)) {
        if (lane == 0) fail();
        break;
      }
      const int nrows = 16 * min(kBpc, nkb - kBpc * c);
      // V rows of keys at or past L are written as zeros
      const int live_rows = isv ? min(nrows, L - kBpc * 16 * c) : nrows;
      const uint8_t* src = ring + slot * C::kChunkBytes8;
      constexpr int kBatch = 4;  // runs loaded before any is converted
#pragma unroll 1
      for (int r0 = r_first; r0 < nrows; r0 += kBatch * kRStep) {
        uint4 x[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int r = r0 + b * kRStep;
          // the TMA's swizzle of the [16 rows][D bytes] tile: 16-byte chunk j of
          // row r sits at chunk j ^ (r & 7) (128-byte rows) or j ^ ((r >> 1) & 3)
          const int sw = D == 128 ? (r & 7) : ((r >> 1) & 3);
          if (r < nrows) x[b] = *reinterpret_cast<const uint4*>(src + r * D + ((j ^ sw) << 4));
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int r = r0 + b * kRStep;
          if (r >= nrows) break;
          uint4 y0 = make_uint4(0u, 0u, 0u, 0u), y1 = y0;
          if (r < live_rows) {
            e4m3x4_to_f16x4(x[b].x, y0.x, y0.y);
            e4m3x4_to_f16x4(x[b].y, y0.z, y0.w);
            e4m3x4_to_f16x4(x[b].z, y1.x, y1.y);
            e4m3x4_to_f16x4(x[b].w, y1.z, y1.w);
          }
          // the 16-bit row's 16-byte chunks cc and cc + 1, 128B-swizzled
          uint8_t* row = dst + r * 128;
          *reinterpret_cast<uint4*>(row + ((cc ^ (r & 7)) << 4)) = y0;
          *reinterpret_cast<uint4*>(row + (((cc + 1) ^ (r & 7)) << 4)) = y1;
        }
      }
      fence_proxy_async_shared();  // the MMAs read the staging through the async proxy
      mbar_arrive(&st_full[si]);
      mbar_arrive(&empty[slot]);
    }
  } else {
    // ------------------------------------------------------------ softmax groups
    // Group t (warps 4t .. 4t+3) owns tile t; thread r of the group owns row r
    // of the tile (TMEM lane r).  tcgen05.ld / st are warp-collective: every
    // decision that guards one is made uniform across the warp first.
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      const bool w = mbar_wait_bounded(bar, parity, p.status);
      return __all_sync(kAll, w) && !__any_sync(kAll, aborted());
    };
    const int t = threadIdx.x >> 7;
    const int r = threadIdx.x & 127;
    const uint32_t tcol = tmem + t * C::kTileCols;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t scol = tcol + lane_base + C::kS0;  // S(c), then P(c)
    const int R = row0 + t * C::kRows + r;
    const bool live = R < rows;
    const int RR = live ? R : rows - 1;
    const int tok = RR / G;
    const int pos = L - nq + tok;
    const size_t qoff = ((size_t)(r0q + tok) * p.num_q_heads + (size_t)kvh * G + (RR - tok * G)) * D;
    // stage Q: row r of tile t, piece-major, 128B-swizzled (zeros past the rows)
    {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) + qoff);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        uint4 v = live ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        if constexpr (KV8 && QT == 1) {
          // bf16 q to the MMAs' f16 (exact for magnitudes in f16's range, saturated above)
          auto cv = [](uint32_t x) {
            return pack_f16x2_satfinite(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
          };
          v = make_uint4(cv(v.x), cv(v.y), cv(v.z), cv(v.w));
        }
        const int piece = c / 8, cc = c % 8;
        *reinterpret_cast<uint4*>(smem + t * C::kQTileBytes + piece * (C::kRows * 128) + r * 128 +
                                  ((cc ^ (r & 7)) * 16)) = v;
      }
      fence_proxy_async_shared();
      mbar_arrive(q_ready);
    }
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    float m_run = -INFINITY, m_used = -INFINITY, l = 0.f;
    // scores of keys past the row's position (also keys past L and past the last block)
    auto mask_keys = [&](auto& v, int key_base) {
      constexpr int N = sizeof(v) / sizeof(float);
#pragma unroll
      for (int i = 0; i < N; ++i)
        if (key_base + i > pos) v[i] = -INFINITY;
    };
    // the maximum of raw scores (the scale is positive, so it commutes): eight
    // interleaved chains of 3-input max
    auto row_max = [&](const auto& v) {
      constexpr int N = sizeof(v) / sizeof(float);
      static_assert(N % 16 == 0, "whole 16-key groups");
      float mq[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mq[k] = v[k];
#pragma unroll
      for (int e = 8; e + 16 <= N; e += 16) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mq[k] = fmax3(mq[k], v[e + k], v[e + 8 + k]);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) mq[k] = fmaxf(mq[k], v[N - 8 + k]);
      return fmax3(fmax3(mq[0], mq[1], mq[2]), fmax3(mq[3], mq[4], mq[5]), fmaxf(mq[6], mq[7]));
    };
    // p = 2^(s * scale_log2 - m_used) for the keys of v (a multiple of 32 from key
    // 64 h), one rounding per exponent, stored as 16-bit pairs over the scores:
    // keys 0..63 at columns 0..31, keys 64..127 at 64..95 of the buffer; the
    // row sum in fp32 over two interleaved partial sums of pairs
    auto exp_store = [&](const auto& v, uint32_t col, uint64_t nm2, uint64_t& acc0,
                         uint64_t& acc1) {
      constexpr int N = sizeof(v) / sizeof(float);
#pragma unroll
      for (int q = 0; q < N / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const int e = 32 * q + 2 * i;
          const float2 x = f2_unpack(f2_fma(f2_pack(v[e], v[e + 1]), sc2, nm2));
          const float2 y = f2_unpack(f2_fma(f2_pack(v[e + 2], v[e + 3]), sc2, nm2));
          const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
          const float p2 = ex2_approx(y.x), p3 = ex2_approx(y.y);
          pk[i] = pf_pack<MT>(p0, p1);
          pk[i + 1] = pf_pack<MT>(p2, p3);
          acc0 = f2_add(acc0, f2_pack(p0, p1));
          acc1 = f2_add(acc1, f2_pack(p2, p3));
        }
        tmem_st16u(col + 64 * (q / 2) + 16 * (q % 2), pk);
      }
    };
    // the running maximum takes the chunk's; O (and l) of the rows whose maximum
    // grew by more than kRescale are rescaled: S(c) completed after P V(c - 1),
    // so O holds every earlier chunk (the warp's other rows take part with a
    // factor of 1); returns -m_used packed for exp_store
    auto update_max = [&](float mx, int c) {
      m_run = fmaxf(m_run, __fmul_rn(mx, p.scale_log2));
      const bool need = m_run > m_used + C::kRescale;
      if (c > 0 && __any_sync(kAll, need)) {
        const float alpha = need ? ex2_approx(__fsub_rn(m_used, m_run)) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
          float o[16];
          tmem_ld16(tcol + lane_base + c0, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __fmul_rn(o[i], alpha);
          tmem_st16(tcol + lane_base + c0, o);
        }
        l = __fmul_rn(l, alpha);
      }
      if (need) m_used = m_run;
      return f2_pack(-m_used, -m_used);
    };
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      if (!wait_all(&s_full[t], (uint32_t)c & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = 128 * c;
      const bool diag = __any_sync(kAll, key0 + 127 > pos);  // warp-uniform
      uint64_t acc0 = 0ull, acc1 = 0ull;
      if constexpr (!KV8) {
        // all of S(c) in registers: one load, one wait
        float sv[128];
        tmem_ld128(scol, sv);
        if (diag) mask_keys(sv, key0);
        const uint64_t nm2 = update_max(row_max(sv), c);
        exp_store(sv, scol, nm2, acc0, acc1);
      } else {
        // 96 registers a thread (18 warps): one 64-column half at a time, the
        // maxima of both, then half 1 and half 0 read again
        float mx;
        {
          float sh[64];
          tmem_ld64(scol, sh);
          if (diag) mask_keys(sh, key0);
          mx = row_max(sh);
        }
        float s1[64];
        tmem_ld64(scol + 64, s1);
        if (diag) mask_keys(s1, key0 + 64);
        const uint64_t nm2 = update_max(fmaxf(mx, row_max(s1)), c);
        exp_store(s1, scol + 64, nm2, acc0, acc1);
        {
          float sh[64];
          tmem_ld64(scol, sh);
          if (diag) mask_keys(sh, key0);
          exp_store(sh, scol, nm2, acc0, acc1);
        }
      }
      const float2 a0 = f2_unpack(acc0), a1 = f2_unpack(acc1);
      l = __fadd_rn(l, __fadd_rn(__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y)));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
    if (ok) ok = wait_all(o_done, 0);
    if (!ok) fail();
    tc_fence_after();
    if (ok) {  // every lane loads (warp-collective); only rows of the tile are stored
      const bool has = l > 0.f;
      // one reciprocal per row, then products: o * (s / l) within an ulp of o * s / l
      const float inv = has ? (KV8 ? __fdiv_rn(p.out_scale, l) : __frcp_rn(l)) : 0.f;
      uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + qoff;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float o[16];
        tmem_ld16(tcol + lane_base + c0, o);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // (KV8: V held codes, so the dequantised mean is out_scale = kv_scale times it)
          const float a = __fmul_rn(o[2 * i], inv);
          const float bv = __fmul_rn(o[2 * i + 1], inv);
          w[i] = pf_pack<QT>(a, bv);
        }
        if (live) {
          reinterpret_cast<uint4*>(dst + c0)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(dst + c0)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols));
  }
}

}  // namespace pa
