// Paged decode of a batch with shared-prefix groups, as a stream-K split.
//
// The work is laid out as lines of units, one unit = one 16-token block, two
// lines per KV head group (the same units for every group), and every CTA
// takes an equal range of one line:
//   * the suffix line: for each sequence i in order, the blocks of its own
//     part of the context, [P_i, ceil(L_i / 16)), where P_i is the length in
//     blocks of the shared prefix it belongs to (0 if none);
//   * the prefix line: for each shared-prefix group, the blocks [0, n_g) that
//     every member's table holds.  Parallel sampling forks several sequences
//     from one prompt, and their tables point at the same physical blocks
//     ("vLLM GitHub 项目…", section 二 item 4: block-level sharing, so shared
//     storage is not repeated); a prefix CTA streams each such block once and
//     computes the logits of all members' query heads against it, the
//     members x G heads forming up to 32 MMA columns (four n-tiles of 8; a
//     head's warps are 4 n-tiles x 2 block phases over a 16-bit cache, 4 x 1
//     over E4M3).
// CTA c serves KV head group c % kvgc, so the CTAs reading the adjacent head
// slices of the same blocks run side by side.  A CTA's range may end inside
// a row or span several rows; each stretch of a row it covers is a segment.
// A segment that covers a whole row of a sequence with no shared prefix
// writes the normalised output; every other segment writes an fp32 partial
// (m, l, O): "whole" partials per (sequence, query head), "cut" partials per
// (CTA, slot), slot 0 for the CTA's first segment and 1 for its last (a cut
// row is always one of the two).  The merge kernel finds, for every
// (sequence, query head), the partials that cover its context from the same
// plan and combines them by log-sum-exp.
//
// The plan is computed by every CTA from the context lengths (no host sync):
// prefix sums of row lengths, the number of CTAs each line gets (in
// proportion to its units, prefix units weighted by their cost) and the range width
// W = ceil(units / CTAs) of each line (at least min_units).  CTA 0 stores it
// for the merge kernel.
//
// Inside a CTA the ring, the producer and the per-block step are the fixed
// kernel's.  On the suffix line the consumer warps of a head take the blocks
// of the CTA's range in rotation (stage ownership never changes across
// segments); at a segment end each warp leaves its state in one of two slots
// of a merge buffer and goes on with the next segment, and a combiner warp
// merges the slot and writes the segment's result, so no consumer waits for
// another.  On the prefix line the n-tile warps of a block phase read each of
// its blocks, and at a segment end the phases' states are merged behind a
// barrier (a prefix CTA has one or two segments).  With the fused write
// (pa_decode_append_shared) the warp that takes a row's last block loads the
// row's new token when the segment starts, writes it into the stage once the
// block is in (the block as it is after the write) and into the pool, so no
// load waits for the write.
#pragma once

#include "pa_decode_kernel.cuh"
#include "pa_internal.h"

namespace pa {

// Plan record in the workspace (ints): [0] CTAs on each group's prefix line,
// [1] its range width, [2] the suffix line's width, [3] KV head groups; from
// kPlanHeader, per sequence i kPlanSeqInts ints: U_i (suffix blocks before i),
// n_i (its suffix blocks), g_i (its group or -1), j_i (its index among the
// group's members), and for a member its group's Up_g (prefix blocks before
// the group) and n_g (the group's prefix blocks).  CTA c of line position k
// serves KV head group c % kvgc with k = c / kvgc (prefix line first).
__host__ __device__ constexpr size_t split_plan_ints(int num_seqs) {
  return (size_t)kPlanHeader + kPlanSeqInts * (size_t)num_seqs;
}

// Shared-memory plan arrays (ints): sU[B+1], sP[B], sG[B], sJ[B], sUp[NG+1],
// and the inputs the CTAs read again: sL[B] (context lengths), sGo[2 NG]
// (each group's member range) and sMem[B] (member sequences, -1 if invalid).
__host__ __device__ constexpr size_t split_smem_plan_bytes(int num_seqs, int num_groups) {
  return (6 * (size_t)num_seqs + 3 * (size_t)num_groups + 2) * 4;
}

template <int D, int KV>
struct SplitCfg {
  using C = DecodeCfg<D, KV>;
  // Eight consumer warps whatever the cache: 8 per head for a 16-bit cache
  // (one KV head per CTA), 4 per head for E4M3 (two).  On the prefix line a
  // head's warps form 4 n-tiles x kPrefixPhases block phases.
  static constexpr int kConsumerWarps = 8;
  static constexpr int kWarpsPerHead = kConsumerWarps / C::kHeads;
  static constexpr int kPrefixPhases = kWarpsPerHead / 4;
  // consumers, then the producer warp, then the combiner warp
  static constexpr int kProducerWarp = kConsumerWarps;
  static constexpr int kCombinerWarp = kConsumerWarps + 1;
  static constexpr int kThreads = (kConsumerWarps + 2) * 32;
  static_assert(C::kStages % kWarpsPerHead == 0,
                "each stage must belong to exactly one consumer warp per head");
  static constexpr int kRedBytes =
      kConsumerWarps * 8 * C::kRedStride * 4 + 2 * kConsumerWarps * 8 * 4;
  static_assert(kRedBytes >= (3 * kMaxPlanGroups + 1) * 4,
                "the plan keeps the group arrays in the merge buffer");
  // Suffix segments' states: two slots of 4 columns per warp when G <= 4,
  // else one slot of 8 (the same bytes as the prefix phases' [warp][8] view).
  __host__ __device__ static constexpr int red_slot_cols(int group) { return group <= 4 ? 4 : 8; }
  __host__ __device__ static constexpr int red_slots(int group) { return group <= 4 ? 2 : 1; }
  __host__ __device__ static constexpr int red_slot_floats(int group) {
    return kConsumerWarps * red_slot_cols(group) * (C::kRedStride + 2);
  }
  static_assert(2 * kConsumerWarps * 4 * (C::kRedStride + 2) * 4 <= kRedBytes &&
                    kConsumerWarps * 8 * (C::kRedStride + 2) * 4 <= kRedBytes,
                "suffix merge slots must fit in the merge buffer");
  // Two CTAs per SM (shared memory allows no more).  The register cap this implies
  // is per SM sub-partition: 2 x 10 warps put 5 warps on each of the four
  // 16K-register files, so at most 96 registers a thread.
  static constexpr int kMinCtasPerSm = 2;
  // Suffix segments' query rows (H heads x up to 8 query heads x D, q's
  // dtype) and context length, prefetched by the producer: two slots.
  static constexpr int kQSlots = 2;
  static constexpr int kQSlotBytes = C::kHeads * 8 * D * 2;
  // ring (1024-aligned) | merge buffer | query slots | barriers (ring full and
  // empty, query slot full and empty, merge slot full and empty) | plan arrays
  static constexpr int kRedOffset = C::kRingBytes;
  static constexpr int kQOffset = kRedOffset + kRedBytes;
  static constexpr int kBarOffset = kQOffset + kQSlots * kQSlotBytes;
  static constexpr int kPlanOffset = kBarOffset + (2 * C::kStages + 2 * kQSlots + 4) * 8;
  __host__ __device__ static constexpr size_t smem_bytes(int num_seqs, int num_groups) {
    return 1024 + (size_t)kPlanOffset + split_smem_plan_bytes(num_seqs, num_groups);
  }
};

// Exclusive scan in place: on entry a[1..n] hold counts, on exit a[i] is the
// sum of the first i counts (a[0] = 0).  One warp.
__device__ __forceinline__ void warp_scan_counts(int* a, int n) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int base = 1; base <= n; base += 32) {
    const int i = base + lane;
    int v = i <= n ? a[i] : 0;
#pragma unroll
    for (int x = 1; x < 32; x <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, x);
      if (lane >= x) v += o;
    }
    if (i <= n) a[i] = v + carry;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) a[0] = 0;
}

// The segment of a line that starts at unit u (u inside the line, u < end).
struct Segment {
  int row;            // sequence (suffix line) or group (prefix line)
  int kvg;            // KV head group
  int b0;             // first block, counted from the row's first (shared) block
  int nblk;           // blocks in the segment
  bool whole;         // the segment is its row's whole range
  bool first;         // the segment starts the CTA's range (cut slot 0, else 1)
  bool row_end;       // the segment reaches its row's last block
};

// The segment of a KV head group's line that starts at unit u (u < u_end).
// Unit counts fit in 32 bits: the host admits a call only if (sequences +
// groups) x max_blocks_per_seq x num_kv_heads < 2^31.
__device__ __forceinline__ Segment segment_at(int u, int u_begin, int u_end, const int* base,
                                              int nrows, const int* first_blk) {
  // the row r with base[r] <= u < base[r + 1] (rows of no units skipped)
  int lo = 0, hi = nrows - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (base[mid + 1] > u) hi = mid; else lo = mid + 1;
  }
  Segment s;
  s.row = lo;
  s.kvg = 0;  // set by the caller: a CTA's line belongs to one KV head group
  const int row_start = base[lo];
  const int row_stop = base[lo + 1];
  const int seg_end = min(row_stop, u_end);
  s.b0 = (first_blk ? first_blk[lo] : 0) + (u - row_start);
  s.nblk = seg_end - u;
  s.whole = (u == row_start) && (seg_end == row_stop);
  s.first = (u == u_begin);
  s.row_end = (seg_end == row_stop);
  return s;
}

__device__ __forceinline__ void consumer_bar(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// A sequence's new token for KV head kvh (append_kv), held by one warp: lane
// i < 2 x D/8 has 16 source bytes (the K row's pieces, then the V row's), with
// the slot it goes to and the block the row's last table entry names.
struct NewToken {
  uint4 x;
  long long slot;  // < 0: nothing is written
  int blk;
};

// The loads are independent of one another, so they are in flight together.
template <int D>
__device__ __forceinline__ NewToken load_new_token(const DecodeParams& p, int seq, int kvh, int L,
                                                   int last_entry) {
  constexpr int kPieces = D / 8;
  const int lane = threadIdx.x & 31;
  NewToken tk;
  tk.x = make_uint4(0u, 0u, 0u, 0u);
  tk.slot = -1;
  tk.blk = -1;
  if (L <= 0 || kvh >= p.num_kv_heads) return tk;
  tk.slot = p.slot_mapping[seq];
  tk.blk = p.block_tables[(size_t)seq * p.max_blocks_per_seq + last_entry];
  if (lane < 2 * kPieces) {
    const int isv = lane / kPieces;
    const int j = lane - isv * kPieces;
    tk.x = *reinterpret_cast<const uint4*>((isv ? p.v_new : p.k_new) +
                                           (size_t)seq * p.src_stride_bytes +
                                           (size_t)kvh * D * 2 + (size_t)j * 16);
  }
  return tk;
}

// Write the token into the pool (the bytes append_rows writes) and, when its
// slot lies in the block just loaded into `stage` (the row's last), into the
// stage's row slot % 16 of head hsel: the block then reads as it does after
// the write.  A slot outside the pool writes nothing.
template <int D, int KV, int QT>
__device__ __forceinline__ void write_new_token(const DecodeParams& p, const NewToken& tk, int kvh,
                                                int hsel, uint8_t* stage) {
  using C = DecodeCfg<D, KV>;
  constexpr int kPieces = D / 8;
  constexpr int kDstPiece = (KV == kKvE4m3) ? 8 : 16;
  const int lane = threadIdx.x & 31;
  const long long pool_rows = (long long)p.num_blocks * 16;
  if (tk.slot >= 0 && tk.slot < pool_rows && lane < 2 * kPieces) {
    const int isv = lane / kPieces;
    const int j = lane - isv * kPieces;
    uint8_t* dst = (isv ? p.v_cache : p.k_cache) +
                   (size_t)tk.slot * (2ull * p.num_kv_heads * C::kRowBytes) +
                   (size_t)kvh * C::kRowBytes + (size_t)j * kDstPiece;
    uint8_t* sdst = nullptr;
    if (tk.slot / 16 == tk.blk) {
      const int row = (int)(tk.slot & 15);
      sdst = stage + (isv ? C::kTileBytes : 0) +
             swz<C::kSwizzle>((uint32_t)((row * C::kHeads + hsel) * C::kRowBytes + j * kDstPiece));
    }
    if constexpr (KV != kKvE4m3) {
      *reinterpret_cast<uint4*>(dst) = tk.x;
      if (sdst) *reinterpret_cast<uint4*>(sdst) = tk.x;
    } else {
      const uint2 c = quantize8_e4m3<QT>(tk.x, p.kv_scale);
      *reinterpret_cast<uint2*>(dst) = c;
      if (sdst) *reinterpret_cast<uint2*>(sdst) = c;
    }
  }
  __syncwarp();  // the stage row is written before any lane reads the block
}

template <int D, int KV, int QT, bool kAppend>
__global__ void __launch_bounds__(SplitCfg<D, KV>::kThreads, SplitCfg<D, KV>::kMinCtasPerSm)
    paged_decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                              const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using C = DecodeCfg<D, KV>;
  using SC = SplitCfg<D, KV>;
  constexpr int kT = SC::kThreads;
  constexpr int kConsumerWarps = SC::kConsumerWarps;
  constexpr int kWarpsPerHead = SC::kWarpsPerHead;
  constexpr int kConsumerThreads = kConsumerWarps * 32;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  float* red_o = reinterpret_cast<float*>(smem + SC::kRedOffset);    // [warps][8][D+4]
  float* red_m = red_o + kConsumerWarps * 8 * C::kRedStride;          // [warps][8]
  float* red_l = red_m + kConsumerWarps * 8;                          // [warps][8]
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + SC::kBarOffset);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* qfull_bar = empty_bar + C::kStages;
  uint64_t* qempty_bar = qfull_bar + SC::kQSlots;
  uint64_t* rfull_bar = qempty_bar + SC::kQSlots;   // [2] merge slot written by the consumers
  uint64_t* rempty_bar = rfull_bar + 2;             // [2] merge slot read by the combiner
  uint8_t* qslots = smem + SC::kQOffset;
  __shared__ int qslot_len[SC::kQSlots];
  __shared__ int abort_flag;

  const int B = p.num_seqs;
  const int NG = p.num_groups;
  const int kvgc = p.kv_groups;
  const int cap = p.max_blocks_per_seq * 16;
  int* sU = reinterpret_cast<int*>(smem + SC::kPlanOffset);  // [B+1]
  int* sP = sU + B + 1;                                      // [B]
  int* sG = sP + B;                                          // [B]
  int* sJ = sG + B;                                          // [B]
  int* sUp = sJ + B;                                         // [NG+1]
  int* sL = sUp + NG + 1;                                    // [B]
  int* sGo = sL + B;                                         // [2 NG]
  int* sMem = sGo + 2 * NG;                                  // [B]

  if (threadIdx.x == SC::kProducerWarp * 32) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  // Every input may come from the kernel before this one on the stream.
  griddep_wait();

  // ------------------------------------------------------------------ plan
  // Two rounds of global loads (every load of a round issued by its own
  // thread): lengths and group arrays, then the members' sequence ids.  The
  // merge buffer is free here and holds the group arrays meanwhile.
  const int tid = threadIdx.x;
  int* gOff = reinterpret_cast<int*>(red_o);  // [NG+1] group offsets as given
  int* gBlk = gOff + NG + 1;                  // [NG] shared blocks, clamped
  int* gMax = gBlk + NG;                      // [NG] longest member, in blocks
  for (int i = tid; i < B; i += kT) {
    const int L = min(max(p.context_lens[i], 0), cap);
    sL[i] = L;
    sU[i + 1] = (L + 15) >> 4;  // the sequence's blocks, for now
    sP[i] = 0;
    sG[i] = -1;
    sJ[i] = 0;
  }
  for (int g = tid; g <= NG; g += kT) {
    gOff[g] = p.grp_off[g];
    if (g < NG) {
      gBlk[g] = min(max(p.grp_blocks[g], 0), p.max_blocks_per_seq);
      gMax[g] = 0;
    }
  }
  if (tid == 0) abort_flag = 0;
  __syncthreads();
  // Groups: each member's suffix starts after the group's shared blocks.  A
  // group's prefix row has n_g = min(shared blocks, the longest member's
  // blocks) units.  Members past the columns a prefix CTA has (32 / G per KV
  // head) are left out of the group: their whole context is suffix.  One
  // (group, member slot) pair per item.
  // (A valid input lists each sequence at most once, so at most B members.)
  const int max_members = kPrefixCols / p.group;
  const int n_members = NG > 0 ? min(max(0, gOff[NG]), B) : 0;
  for (int g = tid; g < NG; g += kT) {
    const int o0 = min(max(gOff[g], 0), n_members);
    sGo[2 * g] = o0;
    sGo[2 * g + 1] = min(max(gOff[g + 1], o0), min(n_members, o0 + max_members));
  }
  for (int item = tid; item < NG * max_members; item += kT) {
    const int g = item / max_members;
    const int j = item - g * max_members;
    const int o0 = min(max(gOff[g], 0), n_members);
    const int o1 = min(max(gOff[g + 1], o0), min(n_members, o0 + max_members));
    if (o0 + j >= o1) continue;
    const int s = p.grp_seq[o0 + j];
    sMem[o0 + j] = (s >= 0 && s < B) ? s : -1;
    if (s < 0 || s >= B) continue;
    atomicMax(&gMax[g], sU[s + 1]);
    sP[s] = gBlk[g];
    sG[s] = g;
    sJ[s] = j;
  }
  __syncthreads();
  for (int g = tid; g < NG; g += kT) sUp[g + 1] = min(gBlk[g], gMax[g]);
  for (int i = tid; i < B; i += kT) sU[i + 1] = max(0, sU[i + 1] - sP[i]);
  __syncthreads();
  if (tid < 32) warp_scan_counts(sU, B);
  else if (tid < 64) warp_scan_counts(sUp, NG);
  __syncthreads();

  // Each KV head group has its own two lines (the units are the same for every
  // group); CTA c serves group c % kvgc, so the kvgc CTAs that read the same
  // blocks' adjacent head slices run side by side (DRAM pages are opened once
  // for all of them).  In the split of a group's CTAs between its lines a
  // prefix unit is weighted by its cost: a prefix CTA's n-tile warps each run
  // every block of their phase.
  const int Tp = sUp[NG];
  const int Ts = sU[B];
  const int Skv = (int)gridDim.x / kvgc;  // >= 2 (the launcher's rule)
  int n_pre;
  if (Tp == 0) {
    n_pre = 0;
  } else if (Ts == 0) {
    n_pre = Skv;
  } else {
    // A prefix unit costs its CTA more than a suffix unit: four n-tile warp
    // passes per block, shared by 4 x phases warps.  With one phase (E4M3) it
    // counts double; with two (16-bit) 5/4, the best of 1, 5/4 and 3/2 on the
    // shared-prefix sampling batch on GB300 (55.9, 52.1 and 54.0 us per step).
    const long long wp = SC::kPrefixPhases == 2 ? (5LL * Tp) / 4 : 2LL * Tp;
    n_pre = (int)(((long long)Skv * wp + (wp + Ts) / 2) / (wp + Ts));
    n_pre = min(max(n_pre, 1), Skv - 1);
  }
  const int Wp = n_pre ? max(p.min_units, (Tp + n_pre - 1) / n_pre) : 1;
  const int Ws = (Skv - n_pre) ? max(p.min_units, (Ts + (Skv - n_pre) - 1) / (Skv - n_pre)) : 1;
  if (blockIdx.x == 0) {
    if (tid == 0) {
      p.plan[0] = n_pre;
      p.plan[1] = Wp;
      p.plan[2] = Ws;
      p.plan[3] = kvgc;
    }
    for (int i = tid; i < B; i += kT) {
      int* r = p.plan + kPlanHeader + kPlanSeqInts * i;
      const int g = sG[i];
      *reinterpret_cast<int4*>(r) = make_int4(sU[i], sU[i + 1] - sU[i], g, sJ[i]);
      *reinterpret_cast<int4*>(r + 4) =
          g >= 0 ? make_int4(sUp[g], sUp[g + 1] - sUp[g], 0, 0) : make_int4(0, 0, 0, 0);
    }
  }
  const int my_kvg = (int)blockIdx.x % kvgc;
  const int ci = (int)blockIdx.x / kvgc;
  if (ci >= Skv) return;  // past the last whole set of kvgc CTAs
  const bool pre = ci < n_pre;
  const int cidx = pre ? ci : ci - n_pre;
  const int W = pre ? Wp : Ws;
  const int T = pre ? Tp : Ts;
  if ((long long)cidx * W >= T) return;  // no work for this CTA
  const int u_begin = cidx * W;
  const int u_end = (int)min((long long)T, (long long)u_begin + W);
  const int* line_base = pre ? sUp : sU;
  const int line_rows = pre ? NG : B;
  const int* line_first = pre ? nullptr : sP;

  const int warp = tid >> 5;
  const int lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      // suffix line: one consumer warp per head reads a stage; prefix line:
      // the four n-tile warps of its block phase, per head
      mbar_init(&empty_bar[s], pre ? 4 * C::kHeads : C::kHeads);
    }
    for (int q = 0; q < SC::kQSlots; ++q) {
      mbar_init(&qfull_bar[q], 1);
      mbar_init(&qempty_bar[q], kConsumerWarps);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&rfull_bar[r], kConsumerWarps);
      mbar_init(&rempty_bar[r], 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == SC::kProducerWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t kv_policy = l2_evict_first_policy();  // the KV stream is read once
    bool ok = true;
    int nseg = 0;  // suffix segments so far: segment k uses query slot k % kQSlots
    int issued = 0;
    int it = 0;
    for (int u = u_begin; u < u_end && ok;) {
      Segment sg = segment_at(u, u_begin, u_end, line_base, line_rows, line_first);
      sg.kvg = my_kvg;
      int seq = sg.row;
      if (pre) {
        // the table of the group's first listed sequence (all members share these blocks)
        const int o0 = sGo[2 * sg.row];
        const int o1 = sGo[2 * sg.row + 1];
        seq = -1;
        for (int k = o0; k < o1 && seq < 0; ++k) seq = sMem[k];
      }
      if (!pre) {
        // the segment's query rows and context length, into the next slot
        const int qs = nseg % SC::kQSlots;
        if (lane == 0 && ok) {
          if (!mbar_wait_bounded(&qempty_bar[qs], ((uint32_t)(nseg / SC::kQSlots) & 1u) ^ 1u,
                                 p.status)) {
            ok = false;
            abort_flag = 1;
          } else {
            const int kv0 = sg.kvg * C::kHeads;
            const uint32_t bytes =
                (uint32_t)(min(C::kHeads, p.num_kv_heads - kv0) * p.group * D * 2);
            qslot_len[qs] = sL[seq];
            mbar_arrive_expect_tx(&qfull_bar[qs], bytes);
            bulk_load(qslots + qs * SC::kQSlotBytes,
                      reinterpret_cast<const uint16_t*>(p.q) +
                          ((size_t)seq * p.num_q_heads + (size_t)kv0 * p.group) * D,
                      bytes, &qfull_bar[qs]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++nseg;
      }
      const int32_t* tbl = p.block_tables + (size_t)max(seq, 0) * p.max_blocks_per_seq + sg.b0;
      const int kv0 = sg.kvg * C::kHeads;
      for (int base = 0; base < sg.nblk; base += 32) {
        const int mine = (base + lane < sg.nblk) ? __ldg(tbl + base + lane) : 0;
        const int cnt = min(32, sg.nblk - base);
        for (int j = 0; j < cnt; ++j) {
          const int blk = __shfl_sync(0xffffffffu, mine, j);
          if (lane == 0 && ok) {
            const int s = it % C::kStages;
            const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
            if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, p.status)) {
              ok = false;
              abort_flag = 1;
            } else {
              load_block<D, KV>(smem + s * C::kStageBytes, &tmap_k, &tmap_v, &full_bar[s], blk,
                                p.num_blocks, kv0, kv_policy);
              ++issued;
            }
          }
          ++it;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      u += sg.nblk;
    }
    griddep_launch_dependents();
    // Never leave the CTA with copies in flight.
    if (lane == 0) {
      const int first = max(0, issued - C::kStages);
      for (int k = first; k < issued; ++k) {
        mbar_wait_bounded(&full_bar[k % C::kStages], (uint32_t)(k / C::kStages) & 1u, p.status);
      }
    }
    return;
  }

  // -------------------------------------------------------------- combiner
  if (warp == SC::kCombinerWarp) {
    if (!pre) {
      // Each suffix segment's result: the head's warp states from the merge
      // slot, combined by log-sum-exp, written as the output (a sequence with
      // no shared prefix whose whole suffix is the segment) or as a partial.
      const int cw = SC::red_slot_cols(p.group);
      const int R = SC::red_slots(p.group);
      constexpr int kQuads = D / 4;
      const int per_head = p.group * kQuads;
      int k = 0;
      for (int u = u_begin; u < u_end; ++k) {
        const Segment sg = segment_at(u, u_begin, u_end, line_base, line_rows, line_first);
        u += sg.nblk;
        const int r = k % R;
        if (*reinterpret_cast<volatile int*>(&abort_flag) != 0 ||
            !mbar_wait_bounded(&rfull_bar[r], (uint32_t)(k / R) & 1u, p.status)) {
          abort_flag = 1;
          break;
        }
        const float* so = red_o + r * SC::red_slot_floats(p.group);  // [warp][cw][stride]
        const float* sm = so + kConsumerWarps * cw * C::kRedStride;   // [warp][cw]
        const float* sl = sm + kConsumerWarps * cw;                   // [warp][cw]
        const int seq = sg.row;
        const bool direct = sg.whole && sG[seq] < 0;
        for (int idx = lane; idx < C::kHeads * per_head; idx += 32) {
          const int hs = idx / per_head;
          const int rem = idx - hs * per_head;
          const int h = rem / kQuads;
          const int d = (rem - h * kQuads) * 4;
          const int kvh2 = my_kvg * C::kHeads + hs;
          if (kvh2 >= p.num_kv_heads) break;
          const int w0 = hs * kWarpsPerHead;
          float M = -INFINITY;
#pragma unroll
          for (int w = w0; w < w0 + kWarpsPerHead; ++w) M = fmaxf(M, sm[w * cw + h]);
          float num[4] = {0.f, 0.f, 0.f, 0.f}, den = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int w = w0; w < w0 + kWarpsPerHead; ++w) {
              const float wt = ex2_approx(__fsub_rn(sm[w * cw + h], M));
              const float4 ov =
                  *reinterpret_cast<const float4*>(&so[(w * cw + h) * C::kRedStride + d]);
              num[0] = __fmaf_rn(wt, ov.x, num[0]);
              num[1] = __fmaf_rn(wt, ov.y, num[1]);
              num[2] = __fmaf_rn(wt, ov.z, num[2]);
              num[3] = __fmaf_rn(wt, ov.w, num[3]);
              den = __fmaf_rn(wt, sl[w * cw + h], den);
            }
          }
          const int qh = kvh2 * p.group + h;
          if (direct) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              v[e] = (den > 0.f) ? __fmul_rn(__fdiv_rn(num[e], den), p.out_scale) : 0.f;
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
            size_t pi;
            float *pm, *pl, *po;
            if (sg.whole) {  // a member's whole suffix
              pi = (size_t)B * p.num_q_heads + (size_t)seq * p.num_q_heads + qh;
              pm = p.whole_m; pl = p.whole_l; po = p.whole_o;
            } else {
              pi = ((size_t)blockIdx.x * 2 + (sg.first ? 0 : 1)) * p.cut_cols + hs * p.group + h;
              pm = p.cut_m; pl = p.cut_l; po = p.cut_o;
            }
            *reinterpret_cast<float4*>(po + pi * D + d) =
                make_float4(num[0], num[1], num[2], num[3]);
            if (d == 0) {
              pm[pi] = M;
              pl[pi] = den;
            }
          }
        }
        __syncwarp();  // every lane has read the slot
        if (lane == 0) mbar_arrive(&rempty_bar[r]);
      }
    }
    griddep_launch_dependents();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int hsel = warp / kWarpsPerHead;
  const int wq = warp % kWarpsPerHead;  // suffix: block rotation; prefix: n-tile + 4 x phase
  const int g = lane >> 2;
  const int t = lane & 3;
  float* my_o = red_o + warp * 8 * C::kRedStride;
  float* my_m = red_m + warp * 8;
  float* my_l = red_l + warp * 8;
  WarpState<D> st;
  uint32_t qb[C::kMTiles][2];
  int it0 = 0;
  int nseg = 0;  // suffix segments so far: query slot nseg % kQSlots, merge slot nseg % R

  for (int u = u_begin; u < u_end;) {
    Segment sg = segment_at(u, u_begin, u_end, line_base, line_rows, line_first);
    sg.kvg = my_kvg;
    const int kvh = sg.kvg * C::kHeads + hsel;
    st.reset();
    if (!pre) {
      // ------------------------------------------------ suffix line
      const int seq = sg.row;
      const int sidx = nseg++;
      const bool live = kvh < p.num_kv_heads && g < p.group;
      // the segment's query rows and length, prefetched by the producer
      const int qs = sidx % SC::kQSlots;
      bool aborted = *reinterpret_cast<volatile int*>(&abort_flag) != 0;
      if (!aborted &&
          !mbar_wait_bounded(&qfull_bar[qs], (uint32_t)(sidx / SC::kQSlots) & 1u, p.status)) {
        abort_flag = 1;
        aborted = true;
      }
      load_q_frag<D, KV, QT>(qb, qslots + qs * SC::kQSlotBytes,
                             (size_t)(hsel * p.group + (live ? g : 0)) * D, live && !aborted);
      const int L = qslot_len[qs];
      // tokens from the segment's first block to the context's end (the last
      // block of a row may be partial)
      const int seg_ntok = L - 16 * sg.b0;
      // block k of the segment sits at ring position it0 + k; this warp takes
      // the positions that are wq mod kWarpsPerHead, as in the fixed kernel
      const int k_first = (wq - it0) & (kWarpsPerHead - 1);
      const int k_last = sg.nblk - 1;
      // the fused write of the row's new token, by the warp of its last block
      const bool tok_mine = kAppend && sg.row_end && !aborted &&
                            ((k_last - k_first) & (kWarpsPerHead - 1)) == 0;
      NewToken tk;
      tk.slot = -1;
      if (tok_mine) tk = load_new_token<D>(p, seq, kvh, L, sg.b0 + k_last);
      // release the query slot (generic reads before the next bulk copy's writes)
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty_bar[qs]);
      for (int k = k_first; k < sg.nblk && !aborted; k += kWarpsPerHead) {
        const int it = it0 + k;
        const int s = it % C::kStages;
        if (!mbar_wait_bounded(&full_bar[s], (uint32_t)(it / C::kStages) & 1u, p.status)) {
          abort_flag = 1;
          aborted = true;
          break;
        }
        if (tok_mine && k == k_last)
          write_new_token<D, KV, QT>(p, tk, kvh, hsel, smem + s * C::kStageBytes);
        const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
        decode_block<D, KV, false>(st, qb, kbase, kbase + C::kTileBytes, hsel,
                                   min(16, seg_ntok - 16 * k), p.scale_log2, 16, 16);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      finish_row_sums(st);
      // Leave the state in the segment's merge slot for the combiner warp and
      // go on (the slot is free once the combiner has read its last use).
      const int R = SC::red_slots(p.group);
      const int cw = SC::red_slot_cols(p.group);
      const int r = sidx % R;
      if (!aborted &&
          !mbar_wait_bounded(&rempty_bar[r], ((uint32_t)(sidx / R) & 1u) ^ 1u, p.status)) {
        abort_flag = 1;
        aborted = true;
      }
      if (aborted) break;  // no barrier follows on this line
      float* so = red_o + r * SC::red_slot_floats(p.group);
      float* sm = so + kConsumerWarps * cw * C::kRedStride;
      dump_state<D, KV>(st, so + warp * cw * C::kRedStride, sm + warp * cw,
                        sm + kConsumerWarps * cw + warp * cw, cw);
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull_bar[r]);
    } else {
      // ------------------------------------------------ prefix line
      const int o0 = sGo[2 * sg.row];
      const int o1 = sGo[2 * sg.row + 1];
      const int mcnt = o1 - o0;
      const bool kv_live = kvh < p.num_kv_heads;
      const int nt = wq % 4;                     // this warp's n-tile of 8 columns
      const int phase = wq / 4;                  // and its block phase
      // B operand: this lane's column 8 nt + g -> member, query head of the group
      const int cb = 8 * nt + g;
      const int jb = cb / p.group;
      const int sb = (jb < mcnt) ? sMem[o0 + jb] : -1;
      const bool bl = kv_live && sb >= 0 && sb < B;
      load_q_frag<D, KV, QT>(
          qb, p.q, ((size_t)(bl ? sb : 0) * p.num_q_heads + kvh * p.group + cb % p.group) * D, bl);
      // C columns 2t, 2t+1 of the n-tile: their members' context lengths
      int lim[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = (8 * nt + 2 * t + c) / p.group;
        const int s = (j < mcnt) ? sMem[o0 + j] : -1;
        lim[c] = (s >= 0 && kv_live) ? sL[s] : -1;
      }
      // tokens past every live column's length are masked for the whole warp
      int vmax = max(lim[0], lim[1]);
#pragma unroll
      for (int x = 1; x < 32; x <<= 1) vmax = max(vmax, __shfl_xor_sync(0xffffffffu, vmax, x));
      const int seg_tok_end = 16 * (sg.b0 + sg.nblk);
      // a dead column (no member) keeps q = 0 and is never stored: no mask needed
      const int l0c = lim[0] < 0 ? (1 << 30) : lim[0];
      const int l1c = lim[1] < 0 ? (1 << 30) : lim[1];
      const bool need_mask = __any_sync(0xffffffffu, l0c < seg_tok_end || l1c < seg_tok_end);
      const bool aborted = *reinterpret_cast<volatile int*>(&abort_flag) != 0;
      // Blocks of this warp's phase two at a time over a 16-bit cache (their
      // MMA chains interleave and they share one softmax step), an odd last
      // one alone; one at a time over E4M3 (whose widening needs the registers).
      constexpr int kStep = SC::kPrefixPhases;
      constexpr bool kPairs = (KV != kKvE4m3);
      int k = (phase - it0) & (kStep - 1);
      while (k < sg.nblk && !aborted) {
        const bool two = kPairs && k + kStep < sg.nblk;
        const int itA = it0 + k;
        const int itB = itA + kStep;
        const int sA = itA % C::kStages;
        const int sB = itB % C::kStages;
        if (!mbar_wait_bounded(&full_bar[sA], (uint32_t)(itA / C::kStages) & 1u, p.status) ||
            (two &&
             !mbar_wait_bounded(&full_bar[sB], (uint32_t)(itB / C::kStages) & 1u, p.status))) {
          abort_flag = 1;
          break;
        }
        const uint32_t kA = smem_u32(smem + sA * C::kStageBytes);
        const uint32_t kB = smem_u32(smem + sB * C::kStageBytes);
        const int tokA = 16 * (sg.b0 + k);
        const int tokB = tokA + 16 * kStep;
        if (two) {
          const uint32_t kb[2] = {kA, kB};
          const uint32_t vb[2] = {kA + C::kTileBytes, kB + C::kTileBytes};
          const int va[2] = {min(16, vmax - tokA), min(16, vmax - tokB)};
          if (need_mask) {
            const int m0[2] = {l0c - tokA, l0c - tokB};
            const int m1[2] = {l1c - tokA, l1c - tokB};
            decode_blocks<D, KV, true, 2>(st, qb, kb, vb, hsel, va, p.scale_log2, m0, m1);
          } else {
            const int full[2] = {16, 16};
            decode_blocks<D, KV, false, 2>(st, qb, kb, vb, hsel, va, p.scale_log2, full, full);
          }
        } else {
          const int valid = min(16, vmax - tokA);
          if (need_mask) {
            decode_block<D, KV, true>(st, qb, kA, kA + C::kTileBytes, hsel, valid, p.scale_log2,
                                      l0c - tokA, l1c - tokA);
          } else {
            decode_block<D, KV, false>(st, qb, kA, kA + C::kTileBytes, hsel, valid,
                                       p.scale_log2, 16, 16);
          }
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty_bar[sA]);
          if (two) mbar_arrive(&empty_bar[sB]);
        }
        k += two ? 2 * kStep : kStep;
      }
      finish_row_sums(st);
      // The block phases' states of each n-tile merge into its 8 columns'
      // partials (one phase: a copy): every warp dumps its state, then the
      // consumers write (column, 4 head_size elements) items.
      dump_state<D, KV>(st, my_o, my_m, my_l);
      consumer_bar(kConsumerThreads);
      constexpr int kQuads = D / 4;
      for (int idx = tid; idx < C::kHeads * kPrefixCols * kQuads; idx += kConsumerThreads) {
        const int hs = idx / (kPrefixCols * kQuads);
        const int rem = idx - hs * (kPrefixCols * kQuads);
        const int col = rem / kQuads;             // 0..31: n-tile col / 8, column col % 8
        const int d = (rem - col * kQuads) * 4;
        const int j = col / p.group;
        const int kvh2 = sg.kvg * C::kHeads + hs;
        if (j >= mcnt || kvh2 >= p.num_kv_heads) continue;
        const int sq = sMem[o0 + j];
        if (sq < 0 || sq >= B) continue;
        const int c = col % 8;
        const int w0 = hs * kWarpsPerHead + col / 8;  // phase 0's warp of this n-tile
        float M = -INFINITY;
#pragma unroll
        for (int ph = 0; ph < SC::kPrefixPhases; ++ph) M = fmaxf(M, red_m[(w0 + 4 * ph) * 8 + c]);
        float num[4] = {0.f, 0.f, 0.f, 0.f}, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int ph = 0; ph < SC::kPrefixPhases; ++ph) {
            const int w = w0 + 4 * ph;
            const float wt = ex2_approx(__fsub_rn(red_m[w * 8 + c], M));
            const float4 ov = *reinterpret_cast<const float4*>(&red_o[(w * 8 + c) * C::kRedStride + d]);
            num[0] = __fmaf_rn(wt, ov.x, num[0]);
            num[1] = __fmaf_rn(wt, ov.y, num[1]);
            num[2] = __fmaf_rn(wt, ov.z, num[2]);
            num[3] = __fmaf_rn(wt, ov.w, num[3]);
            den = __fmaf_rn(wt, red_l[w * 8 + c], den);
          }
        }
        const int qh = kvh2 * p.group + col % p.group;
        size_t pi;
        float *pm, *pl, *po;
        if (sg.whole) {
          pi = (size_t)sq * p.num_q_heads + qh;
          pm = p.whole_m; pl = p.whole_l; po = p.whole_o;
        } else {
          pi = ((size_t)blockIdx.x * 2 + (sg.first ? 0 : 1)) * p.cut_cols + hs * kPrefixCols + col;
          pm = p.cut_m; pl = p.cut_l; po = p.cut_o;
        }
        *reinterpret_cast<float4*>(po + pi * D + d) = make_float4(num[0], num[1], num[2], num[3]);
        if (d == 0) {
          pm[pi] = M;
          pl[pi] = den;
        }
      }
      consumer_bar(kConsumerThreads);  // the buffer is free for the next segment
    }
    it0 += sg.nblk;
    u += sg.nblk;
  }
  griddep_launch_dependents();
}

// Log-sum-exp merge for the stream-K split: one warp per (sequence, query
// head), kSplitMergeWarps of them per CTA.  From the plan it lists the
// partials covering the sequence's context (its suffix: one whole partial, or
// the cut partials of the CTAs whose ranges meet its row; its shared prefix,
// if any, the same way on the prefix line).  Lanes resolve and load 32 of the
// partials' (m, l) at once; every lane then folds its D/32 head_size elements
// of each partial's O row (coalesced loads) into a running maximum, in list
// order, so the result does not depend on timing.  A sequence whose whole
// context one CTA wrote directly is skipped.
constexpr int kSplitMergeWarps = 8;

template <int D, int QT, int H>
__global__ void __launch_bounds__(kSplitMergeWarps * 32, 4)
    paged_decode_split_merge_kernel(const DecodeParams p) {
  constexpr int kPer = D / 32;  // head_size elements per lane
  const int lane = threadIdx.x & 31;
  const int idx = blockIdx.x * kSplitMergeWarps + (threadIdx.x >> 5);  // sequence * Hq + head
  if (idx >= p.num_seqs * p.num_q_heads) return;
  const int seq = idx / p.num_q_heads;
  const int h = idx - seq * p.num_q_heads;
  griddep_wait();  // the plan and the partials come from the attention kernel
  const int* plan = p.plan;
  const int n_pre = plan[0];
  const int Wp = plan[1], Ws = plan[2];
  const int kvgc = plan[3];
  const int4 r0 = *reinterpret_cast<const int4*>(plan + kPlanHeader + kPlanSeqInts * seq);
  const int4 r1 = *reinterpret_cast<const int4*>(plan + kPlanHeader + kPlanSeqInts * seq + 4);
  const int U = r0.x, nsuf = r0.y, grp = r0.z, mem = r0.w;
  const int pre_start = r1.x, pre_len = r1.y;
  const int G = p.group;
  const int kvh = h / G;
  const int kvg = kvh / H;
  const int hs = kvh - kvg * H;
  const int gh = h - kvh * G;

  // suffix partials
  const int s_start = U;
  int ns = 0, s_c0 = 0;
  bool s_whole = false;
  if (nsuf > 0) {
    s_c0 = s_start / Ws;
    const int c1 = (s_start + nsuf - 1) / Ws;
    if (s_c0 == c1) {
      if (grp < 0) return;  // written directly by the attention kernel
      s_whole = true;
      ns = 1;
    } else {
      ns = c1 - s_c0 + 1;
    }
  }
  // shared-prefix partials
  int np = 0, p_start = 0, p_c0 = 0;
  bool p_whole = false;
  if (grp >= 0) {
    const int npre = pre_len;
    if (npre > 0) {
      p_start = pre_start;
      p_c0 = p_start / Wp;
      const int c1 = (p_start + npre - 1) / Wp;
      if (p_c0 == c1) {
        p_whole = true;
        np = 1;
      } else {
        np = c1 - p_c0 + 1;
      }
    }
  }
  const size_t BH = (size_t)p.num_seqs * p.num_q_heads;
  const int K = ns + np;
  float M = -INFINITY, den = 0.f;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  for (int base = 0; base < K; base += 32) {
    // lane k of this chunk: partial base + k -> its (m, l) and O row
    const int k = base + lane;
    float mk = -INFINITY, lk = 0.f;
    const float* ok = p.cut_o;
    if (k < K) {
      const float *pm, *pl, *po;
      size_t pi;
      if (k < ns) {
        if (s_whole) {
          pi = BH + (size_t)seq * p.num_q_heads + h;
          pm = p.whole_m; pl = p.whole_l; po = p.whole_o;
        } else {
          const int c = s_c0 + k;
          const int slot = (c * Ws >= s_start) ? 0 : 1;
          pi = (((size_t)(n_pre + c) * kvgc + kvg) * 2 + slot) * p.cut_cols + hs * G + gh;
          pm = p.cut_m; pl = p.cut_l; po = p.cut_o;
        }
      } else if (p_whole) {
        pi = (size_t)seq * p.num_q_heads + h;
        pm = p.whole_m; pl = p.whole_l; po = p.whole_o;
      } else {
        const int c = p_c0 + (k - ns);
        const int slot = (c * Wp >= p_start) ? 0 : 1;
        pi = (((size_t)c * kvgc + kvg) * 2 + slot) * p.cut_cols + hs * kPrefixCols + mem * G + gh;
        pm = p.cut_m; pl = p.cut_l; po = p.cut_o;
      }
      mk = pm[pi];
      lk = pl[pi];
      ok = po + pi * D;
    }
    float cmax = mk;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, x));
    const float Mn = fmaxf(M, cmax);
    if (Mn == -INFINITY) continue;  // nothing but empty partials so far
    const float sc = ex2_approx(__fsub_rn(M, Mn));  // 0 while M is -inf
    den = __fmul_rn(den, sc);
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = __fmul_rn(acc[e], sc);
    const float wk = ex2_approx(__fsub_rn(mk, Mn));  // 0 for lanes past K
    float dl = __fmul_rn(wk, lk);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) dl = __fadd_rn(dl, __shfl_xor_sync(0xffffffffu, dl, x));
    den = __fadd_rn(den, dl);
    // O rows 4 at a time: all four loads are issued before any is used
    const int cnt = min(32, K - base);
    for (int j0 = 0; j0 < cnt; j0 += 4) {
      float w8[4];
      float row8[4][kPer];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jj = min(j0 + j, cnt - 1);
        w8[j] = (j0 + j < cnt) ? __shfl_sync(0xffffffffu, wk, jj) : 0.f;
        const float* row = reinterpret_cast<const float*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(ok), jj));
        if constexpr (kPer == 4) {
          const float4 v = reinterpret_cast<const float4*>(row)[lane];
          row8[j][0] = v.x; row8[j][1] = v.y; row8[j][2] = v.z; row8[j][3] = v.w;
        } else {
          const float2 v = reinterpret_cast<const float2*>(row)[lane];
          row8[j][0] = v.x; row8[j][1] = v.y;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j0 + j < cnt) {
#pragma unroll
          for (int e = 0; e < kPer; ++e) acc[e] = __fmaf_rn(w8[j], row8[j][e], acc[e]);
        }
      }
    }
    M = Mn;
  }
  float v[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e)
    v[e] = (den > 0.f) ? __fmul_rn(__fdiv_rn(acc[e], den), p.out_scale) : 0.f;
  uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + (size_t)idx * D + lane * kPer;
  if constexpr (kPer == 4) {
    uint2 pk;
    if constexpr (QT == kKvF16) {
      pk.x = pack_f16x2(v[0], v[1]);
      pk.y = pack_f16x2(v[2], v[3]);
    } else {
      pk.x = pack_bf16x2(v[0], v[1]);
      pk.y = pack_bf16x2(v[2], v[3]);
    }
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) =
        (QT == kKvF16) ? pack_f16x2(v[0], v[1]) : pack_bf16x2(v[0], v[1]);
  }
}

}  // namespace pa
