// The prefix line of the shared-prefix decode on the 5th-generation tensor
// cores (16-bit caches).
//
// A prefix CTA computes, for one KV head and each shared-prefix group its
// range meets, the logits of every member's query heads against the group's
// shared blocks and the weighted sum of their values ("vLLM GitHub 项目…",
// section 二 item 4: the samples' tables point at the same physical blocks, so
// the CTA reads each block once for all of them).  The members x G query rows
// (at most 32) are the rows of an M = 128 tile, the rest zero:
//   S(c) = Q K(c)^T   (tcgen05.mma kind::f16, A = Q and B = the chunk's K rows
//                      from shared memory, M = 128, N = 64 keys, into TMEM)
//   O  += P(c) V(c)   (A = P(c) from TMEM, B = the chunk's V rows, N = head size)
// over chunks of four 16-token blocks.  S is double-buffered in TMEM, so S(c+1)
// runs while the softmax of chunk c does.  TMEM per CTA (256 columns): O at
// [0, D), S of even chunks at [128, 192), of odd ones at [192, 256); P(c)
// (16-bit pairs) over S(c).  Roles: the producer warp loads each chunk's K and
// V blocks with TMA into a ring slot (piece-major, 128B-swizzled, each piece of
// the chunk one 64-row operand); the combiner warp's lane 0 allocates TMEM and
// issues the MMAs; the consumer warps stage Q per segment, and consumer warp 0
// (TMEM lanes 0-31: the live rows) runs the online softmax on each S chunk,
// writes P over it, and at the segment end writes the rows' partials
// (m, l, O) from TMEM.  Every wait is bounded.
#pragma once

#include "pa_decode_kernel.cuh"
#include "pa_decode_segment.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

template <int D>
struct PrefixTcCfg {
  static constexpr int kPieces = D * 2 / 128;          // 128-byte pieces of a 16-bit row
  static constexpr int kBlocks = 2;                     // blocks per chunk
  static constexpr int kKeys = 16 * kBlocks;            // N of S
  static constexpr int kBox = 16 * 128;                 // one block, one piece (a TMA box)
  static constexpr int kPlane = kKeys * 128;            // one piece of a chunk's K (or V)
  static constexpr int kOperand = kPieces * kPlane;     // K (or V) of a chunk
  static constexpr int kSlotBytes = 2 * kOperand;       // K then V
  static constexpr int kRows = 128;                     // M
  static constexpr int kQPlane = kRows * 128;
  static constexpr int kQBytes = kPieces * kQPlane;
  static constexpr int kTmemCols = 256;
  static constexpr int kS0 = 128;                       // S buffer 0; buffer 1 at kS0 + kKeys
  static constexpr float kRescale = 8.f;                // log2 units (see the prefill kernel)
  // barriers: full / empty per slot (up to 4), S full per buffer, P full, P V
  // done, O done, Q ready, TMEM free, MMAs drained
  static constexpr int kMaxSlots = 4;
  static constexpr int kNumBars = 2 * kMaxSlots + 2 + 6;
  static_assert(D <= kS0 && kS0 + 2 * kKeys <= kTmemCols, "TMEM layout");
};

// Barrier indices in the CTA's barrier array.
struct PrefixTcBars {
  uint64_t* b;
  int slots;
  __device__ uint64_t* full(int s) const { return b + s; }
  __device__ uint64_t* empty(int s) const { return b + 4 + s; }
  __device__ uint64_t* sfull(int buf) const { return b + 8 + buf; }
  __device__ uint64_t* pfull() const { return b + 10; }
  __device__ uint64_t* pvdone() const { return b + 11; }
  __device__ uint64_t* odone() const { return b + 12; }
  __device__ uint64_t* qready() const { return b + 13; }
  __device__ uint64_t* tfree() const { return b + 14; }
  __device__ uint64_t* drained() const { return b + 15; }
};

template <int D>
__device__ __forceinline__ void prefix_tc_init_bars(const PrefixTcBars& bars, int consumer_threads) {
  for (int s = 0; s < bars.slots; ++s) {
    mbar_init(bars.full(s), 1);
    mbar_init(bars.empty(s), 1);  // tcgen05.commit after the chunk's P V
  }
  mbar_init(bars.sfull(0), 1);
  mbar_init(bars.sfull(1), 1);
  mbar_init(bars.pfull(), 32);  // consumer warp 0
  mbar_init(bars.pvdone(), 1);
  mbar_init(bars.odone(), 1);
  mbar_init(bars.qready(), consumer_threads);
  mbar_init(bars.tfree(), 1);
  mbar_init(bars.drained(), 1);
}

// The group of prefix row `row`: its members' range in sMem and the first
// valid member (whose table the producer reads).
struct PrefixGroup {
  int o0, o1, lead;
};
__device__ __forceinline__ PrefixGroup prefix_group(const int* sGo, const int* sMem, int row) {
  PrefixGroup g;
  g.o0 = sGo[2 * row];
  g.o1 = sGo[2 * row + 1];
  g.lead = -1;
  for (int k = g.o0; k < g.o1 && g.lead < 0; ++k) g.lead = sMem[k];
  return g;
}

// Producer warp: chunk c of the CTA (counted over its segments) goes to slot
// c % slots; lane j loads block j of the chunk, every piece, K then V.
template <int D>
__device__ __forceinline__ bool prefix_tc_produce(const DecodeParams& p, const CUtensorMap* tmk,
                                                  const CUtensorMap* tmv, uint8_t* ring,
                                                  const PrefixTcBars& bars, const int* sUp, int NG,
                                                  const int* sGo, const int* sMem, int u_begin,
                                                  int u_end, int kvh, int* abort_flag,
                                                  int* chunks_out) {
  using TC = PrefixTcCfg<D>;
  const int lane = threadIdx.x & 31;
  const uint64_t pol = l2_evict_first_policy();
  const int oob_row = p.num_blocks * 16;
  bool ok = true;
  int gc = 0;
  for (int u = u_begin; u < u_end && ok;) {
    const Segment sg = segment_at(u, u_begin, u_end, sUp, NG, nullptr);
    u += sg.nblk;
    const PrefixGroup grp = prefix_group(sGo, sMem, sg.row);
    const int32_t* tbl =
        p.block_tables + (size_t)max(grp.lead, 0) * p.max_blocks_per_seq + sg.b0;
    const int nch = (sg.nblk + TC::kBlocks - 1) / TC::kBlocks;
    // the segment's table entries, 32 at a time (one load per lane), ahead of
    // the chunks that use them
    int ent = 0;
    for (int c = 0; c < nch && ok; ++c, ++gc) {
      const int slot = gc % bars.slots;
      const int nb = min(TC::kBlocks, sg.nblk - TC::kBlocks * c);
      const int b = TC::kBlocks * c;  // the chunk's first block in the segment
      if (b % 32 == 0) ent = (b + lane < sg.nblk) ? __ldg(tbl + b + lane) : 0;
      const int blk = __shfl_sync(0xffffffffu, ent, (b % 32) + min(lane, TC::kBlocks - 1));
      const int brow = (blk >= 0 && blk < p.num_blocks) ? blk * 16 : oob_row;
      int got = 0;
      if (lane == 0 && !*reinterpret_cast<volatile int*>(abort_flag) &&
          mbar_wait_bounded(bars.empty(slot), ((uint32_t)(gc / bars.slots) & 1u) ^ 1u, p.status)) {
        mbar_arrive_expect_tx(bars.full(slot), (uint32_t)(nb * TC::kPieces * 2 * TC::kBox));
        got = 1;
      }
      ok = __shfl_sync(0xffffffffu, got, 0) != 0;
      if (!ok) break;
      if (lane < nb) {
        uint8_t* dst = ring + slot * TC::kSlotBytes + lane * TC::kBox;
#pragma unroll
        for (int pc = 0; pc < TC::kPieces; ++pc) {
          tma_load_4d(dst + pc * TC::kPlane, tmk, bars.full(slot), 0, brow, pc, kvh, pol);
          tma_load_4d(dst + TC::kOperand + pc * TC::kPlane, tmv, bars.full(slot), 0, brow, pc,
                      kvh, pol);
        }
      }
    }
  }
  *chunks_out = gc;
  return ok;
}

// MMA issuer (one thread).  Per segment: wait for Q; S of the first two
// chunks; then per chunk c: wait for P(c), O += P(c) V(c) over its blocks,
// release the slot, and issue S(c + 2) into the buffer P(c) occupied (the
// thread's MMAs run in order, so P V(c) has read P(c) first).
template <int D, int KV>
__device__ __forceinline__ bool prefix_tc_mma(const DecodeParams& p, uint8_t* ring,
                                              const uint8_t* qtile, uint32_t tmem,
                                              const PrefixTcBars& bars, const int* sUp, int NG,
                                              int u_begin, int u_end, int* abort_flag) {
  using TC = PrefixTcCfg<D>;
  constexpr bool kBf16 = (KV == kKvBf16);
  const uint32_t id_s = umma_idesc(kBf16, 128, TC::kKeys, 0);
  const uint32_t id_pv = umma_idesc(kBf16, 128, D, 1);
  const uint32_t q_lo = umma_desc_lo(smem_u32(qtile), 16);
  const uint32_t k_lo = umma_desc_lo(smem_u32(ring), 16);
  const uint32_t v_lo = umma_desc_lo(smem_u32(ring) + TC::kOperand, TC::kPlane);
  auto alive = [&]() { return *reinterpret_cast<volatile int*>(abort_flag) == 0; };
  auto issue_s = [&](int g2) {
    const int slot = g2 % bars.slots;
    if (!alive() ||
        !mbar_wait_bounded(bars.full(slot), (uint32_t)(g2 / bars.slots) & 1u, p.status))
      return false;
    tc_fence_after();
    const uint32_t dcol = tmem + TC::kS0 + (uint32_t)(TC::kKeys * (g2 & 1));
    const uint32_t ka = k_lo + (uint32_t)(slot * TC::kSlotBytes >> 4);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t qo = (uint32_t)(((k / 4) * TC::kQPlane + (k % 4) * 32) >> 4);
      const uint32_t ko = (uint32_t)(((k / 4) * TC::kPlane + (k % 4) * 32) >> 4);
      umma_ss(dcol, umma_desc_join(q_lo + qo), umma_desc_join(ka + ko), id_s, k > 0 ? 1 : 0);
    }
    umma_commit(bars.sfull(g2 & 1));
    return true;
  };
  bool ok = true;
  int gc = 0, seg = 0;
  for (int u = u_begin; u < u_end && ok; ++seg) {
    const Segment sg = segment_at(u, u_begin, u_end, sUp, NG, nullptr);
    u += sg.nblk;
    const int nch = (sg.nblk + TC::kBlocks - 1) / TC::kBlocks;
    ok = alive() && mbar_wait_bounded(bars.qready(), (uint32_t)seg & 1u, p.status);
    if (!ok) break;
    tc_fence_after();
    ok = issue_s(gc) && (nch < 2 || issue_s(gc + 1));
    for (int c = 0; c < nch && ok; ++c) {
      const int g2 = gc + c;
      const int slot = g2 % bars.slots;
      const int nb = min(TC::kBlocks, sg.nblk - TC::kBlocks * c);
      ok = alive() && mbar_wait_bounded(bars.pfull(), (uint32_t)g2 & 1u, p.status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t pcol = tmem + TC::kS0 + (uint32_t)(TC::kKeys * (g2 & 1));
      const uint32_t va = v_lo + (uint32_t)(slot * TC::kSlotBytes >> 4);
      for (int j = 0; j < nb; ++j)
        umma_ts(tmem, pcol + 8 * j, umma_desc_join(va + (uint32_t)(j * (TC::kBox >> 4))), id_pv,
                (c > 0 || j > 0) ? 1 : 0);
      umma_commit(bars.empty(slot));
      umma_commit(bars.pvdone());
      if (c + 2 < nch) ok = issue_s(g2 + 2);
    }
    if (ok) umma_commit(bars.odone());
    gc += nch;
  }
  return ok;
}

}  // namespace pa

namespace pa {

// Consumer warps (nthreads threads, tid = threadIdx.x).  Per segment they stage
// Q (once the segment before has finished with it), and warp 0 runs the
// softmax over the segment's chunks and writes its rows' partials.
template <int D, int KV, int QT>
__device__ __forceinline__ bool prefix_tc_consume(const DecodeParams& p, uint8_t* ring,
                                                  uint8_t* qtile, uint32_t tmem,
                                                  const PrefixTcBars& bars, const int* sUp,
                                                  int NG, const int* sGo, const int* sMem,
                                                  const int* sL, int u_begin, int u_end, int kvh,
                                                  int nthreads, int* abort_flag) {
  using TC = PrefixTcCfg<D>;
  constexpr unsigned kAll = 0xffffffffu;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  const int B = p.num_seqs;
  auto alive = [&]() { return *reinterpret_cast<volatile int*>(abort_flag) == 0; };
  // warp-uniform bounded wait
  auto wait_all = [&](uint64_t* bar, uint32_t parity) {
    const bool w = alive() && mbar_wait_bounded(bar, parity, p.status);
    return __all_sync(kAll, w);
  };
  const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
  bool ok = true;
  int gc = 0, seg = 0;
  for (int u = u_begin; u < u_end && ok; ++seg) {
    const Segment sg = segment_at(u, u_begin, u_end, sUp, NG, nullptr);
    u += sg.nblk;
    const int o0 = sGo[2 * sg.row];
    const int mcnt = sGo[2 * sg.row + 1] - o0;
    const int nlive = min(mcnt * G, 32);
    const int nch = (sg.nblk + TC::kBlocks - 1) / TC::kBlocks;
    // ---- Q of the segment's rows: row r = member r / G, query head r % G of KV
    // head kvh; piece-major, 128B-swizzled; rows past the members are zero
    if (seg > 0) {
      const bool w = alive() && mbar_wait_bounded(bars.odone(), (uint32_t)(seg - 1) & 1u, p.status);
      if (!w) {
        atomicExch(abort_flag, 1);
        ok = false;
      }
    }
    {
      constexpr int kChunks = D / 8;  // 16-byte chunks of a row
      for (int item = tid; item < TC::kRows * kChunks; item += nthreads) {
        const int r = item / kChunks;
        const int cc = item - r * kChunks;
        const int s = (r < nlive) ? sMem[o0 + r / G] : -1;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (s >= 0 && s < B)
          v = *reinterpret_cast<const uint4*>(
              reinterpret_cast<const uint16_t*>(p.q) +
              ((size_t)s * p.num_q_heads + (size_t)kvh * G + (r % G)) * D + cc * 8);
        const int piece = cc / 8, c8 = cc % 8;
        *reinterpret_cast<uint4*>(qtile + piece * TC::kQPlane + r * 128 + ((c8 ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_shared();  // the MMAs read Q through the async proxy
      mbar_arrive(bars.qready());
    }
    if (warp == 0 && ok) {
      // ---- softmax: thread `lane` owns row `lane` (TMEM lane `lane`)
      const int r = lane;
      const int s_r = (r < nlive) ? sMem[o0 + r / G] : -1;
      const int lim = (s_r >= 0 && s_r < B) ? sL[s_r] : 0;  // tokens this row attends
      int vmax = lim;                                        // tokens any row attends
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) vmax = max(vmax, __shfl_xor_sync(kAll, vmax, x));
      float m_run = -INFINITY, m_used = -INFINITY, l = 0.f;
      for (int c = 0; c < nch && ok; ++c) {
        const int g2 = gc + c;
        const int buf = g2 & 1;
        const int slot = g2 % bars.slots;
        const int nb = min(TC::kBlocks, sg.nblk - TC::kBlocks * c);
        const int tok0 = 16 * (sg.b0 + TC::kBlocks * c);
        if (!wait_all(bars.sfull(buf), (uint32_t)(g2 >> 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t scol = tmem + TC::kS0 + (uint32_t)(TC::kKeys * buf);
        // keys past the loaded blocks or past the row's context count as -inf;
        // S is read in 16-column pieces (the register budget is 96 a thread)
        const int kend = min(16 * nb, lim - tok0);  // keys [0, kend) count
        auto load_masked = [&](int c0, float (&v)[16]) {
          tmem_ld16(scol + c0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c0 + i >= kend) v[i] = -INFINITY;
        };
        float mx = -INFINITY;
#pragma unroll
        for (int c0 = 0; c0 < TC::kKeys; c0 += 16) {
          float v[16];
          load_masked(c0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) mx = fmaxf(mx, v[i]);
        }
        m_run = fmaxf(m_run, __fmul_rn(mx, p.scale_log2));
        const bool need = m_run > m_used + TC::kRescale;
        if (c > 0 && __any_sync(kAll, need)) {
          // O may be rescaled only once P V(c - 1) has finished writing it.
          // P V(c) waits for this chunk's P, so P V(c - 1) is the last one that
          // can be in flight: the barrier is at most one phase short of it.
          if (!wait_all(bars.pvdone(), (uint32_t)(g2 - 1) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = need ? ex2_approx(__fsub_rn(m_used, m_run)) : 1.f;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 16) {
            float o[16];
            tmem_ld16(tmem + c0, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __fmul_rn(o[i], alpha);
            tmem_st16(tmem + c0, o);
          }
          l = __fmul_rn(l, alpha);
        }
        if (need) m_used = m_run;
        // P = 2^(s * scale - m_used), 16-bit pairs over S (keys 2i, 2i+1 in column i);
        // a row with no key so far keeps P = 0
        const bool any_key = m_used != -INFINITY;
        const uint64_t nm2 = f2_pack(any_key ? -m_used : 0.f, any_key ? -m_used : 0.f);
        uint64_t acc = 0ull;
        // keys 32 h .. 32 h + 31 -> columns 16 h .. 16 h + 15 (read before written)
#pragma unroll
        for (int h = 0; h < TC::kKeys / 32; ++h) {
          float v0[16], v1[16];
          load_masked(32 * h, v0);
          load_masked(32 * h + 16, v1);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float s0 = i < 8 ? v0[2 * i] : v1[2 * i - 16];
            const float s1 = i < 8 ? v0[2 * i + 1] : v1[2 * i - 15];
            float p0 = 0.f, p1 = 0.f;
            if (any_key) {
              const float2 x = f2_unpack(f2_fma(f2_pack(s0, s1), sc2, nm2));
              p0 = ex2_approx(x.x);
              p1 = ex2_approx(x.y);
            }
            pk[i] = (KV == kKvBf16) ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
            acc = f2_add(acc, f2_pack(p0, p1));
          }
          tmem_st16u(scol + 16 * h, pk);
        }
        const float2 a = f2_unpack(acc);
        l = __fadd_rn(l, __fadd_rn(a.x, a.y));
        // V rows of tokens no row attends (the last block of the group's
        // prefix may end inside it) hold stale or poisoned values: zero them
        // before P V reads them (a P of 0 times a NaN is NaN).
        if (tok0 + 16 * nb > vmax) {
          if (!wait_all(bars.full(slot), (uint32_t)(g2 / bars.slots) & 1u)) {
            ok = false;
            break;
          }
          const int k_first = max(vmax - tok0, 0);
          const int nrow = 16 * nb - k_first;
          uint8_t* vbase = ring + slot * TC::kSlotBytes + TC::kOperand;
          for (int it = lane; it < nrow * TC::kPieces * 8; it += 32) {
            const int rr = k_first + it / (TC::kPieces * 8);
            const int rem = it % (TC::kPieces * 8);
            const int pc = rem / 8;
            *reinterpret_cast<uint4*>(vbase + pc * TC::kPlane + rr * 128 + (rem % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_shared();
          __syncwarp();
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bars.pfull());
      }
      // ---- the rows' partials once every MMA of the segment is done
      if (ok && !wait_all(bars.odone(), (uint32_t)seg & 1u)) ok = false;
      if (ok) {
        tc_fence_after();
        const bool live = (r < nlive) && s_r >= 0 && s_r < B;
        const int col = r;  // row r <-> column r of the prefix partials
        const int qh = kvh * G + (r % G);
        size_t pi;
        float *pm, *pl, *po;
        if (sg.whole) {
          pi = (size_t)(live ? s_r : 0) * p.num_q_heads + qh;
          pm = p.whole_m; pl = p.whole_l; po = p.whole_o;
        } else {
          pi = ((size_t)blockIdx.x * 2 + (sg.first ? 0 : 1)) * p.cut_cols + col;
          pm = p.cut_m; pl = p.cut_l; po = p.cut_o;
        }
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
          float o[16];
          tmem_ld16(tmem + c0, o);  // warp-collective
          if (live) {
            float4* dst = reinterpret_cast<float4*>(po + pi * D + c0);
            dst[0] = make_float4(o[0], o[1], o[2], o[3]);
            dst[1] = make_float4(o[4], o[5], o[6], o[7]);
            dst[2] = make_float4(o[8], o[9], o[10], o[11]);
            dst[3] = make_float4(o[12], o[13], o[14], o[15]);
          }
        }
        if (live) {
          pm[pi] = m_used;
          pl[pi] = l;
        }
      }
    }
    if (!ok) atomicExch(abort_flag, 1);
    gc += nch;
  }
  if (warp == 0) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.tfree());
  }
  return ok;
}

}  // namespace pa
