// Paged prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes is the causal paged prefill of pa_prefill_kernel.cuh: the
// query at position p of sequence i, head h, attends to that sequence's tokens
// 0..p of KV head h / G through its block table.
//
// One CTA per (tile of 128 rows, KV head, sequence); a row is one (query token,
// query head of the KV head's group) pair, token-major.  192 threads:
//   * warps 0-3 (softmax): thread r owns row r, which is TMEM lane r.  They
//     stage Q into shared memory, run the online softmax on each S chunk read
//     from TMEM, write P (16-bit) back to TMEM, rescale O in TMEM when a row's
//     running maximum grows by more than kRescale (log2 units; otherwise the
//     exponentials keep the older maximum, so P stays below 2^kRescale), and
//     finally normalise O and store the rows.
//   * warp 4 (producer): TMA loads of the sequence's K/V blocks into a ring of
//     full/empty mbarriers (piece-major 128B-swizzled tiles), and zeroes the
//     V rows past the context's end in the last block (a P of 0 times a stale
//     or poisoned V must not reach the sum).
//   * warp 5 (MMA): owns the TMEM allocation; one thread issues, per chunk of
//     two blocks (32 keys), S = Q K^T (M = 128, N = 16 per block, K = head
//     size: kind::f16, A and B from shared memory) into one of two S buffers,
//     then O += P V for the previous chunk (A = P from TMEM, B = the V tile,
//     MN-major, N = head size, K = 16 per block), and releases ring stages,
//     S and P buffers with tcgen05.commit.
// Accumulation in fp32 throughout; every wait is bounded.
#pragma once

#include "pa_ptx.cuh"
#include "pa_prefill_kernel.cuh"

namespace pa {

template <int D>
struct PrefillTcCfg {
  static constexpr int kRows = 128;
  static constexpr int kPieces = D * 2 / 128;              // 128-byte pieces of a row
  static constexpr int kQBytes = kRows * D * 2;            // [pieces][128 rows][128 B]
  static constexpr int kTileBytes = 16 * D * 2;            // one block of K (or V), one head
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = (kStageBytes >= 8192) ? 8 : 16;  // 64 KB ring
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarOff = kQBytes + kRingBytes;
  // barriers: full, empty per stage; s_full, s_free, p_full, pv_done x2; q_ready, tail, o_done
  static constexpr int kNumBars = 2 * kStages + 8 + 3;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static constexpr int kThreads = 192;
  // TMEM columns: O [0, D), S buffers at kS0 + 32 b, P buffers at kP0 + 16 b
  static constexpr int kS0 = D;
  static constexpr int kP0 = D + 64;
  static constexpr int kTmemCols = 256;
  static constexpr float kRescale = 8.f;
  static_assert(kP0 + 32 <= kTmemCols, "TMEM layout");
};

__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16 instruction descriptor: f32 accumulator, A/B of type `bf16` (else
// f16), M, N, A K-major, B K-major (0) or MN-major (1).
__device__ __forceinline__ uint32_t umma_idesc(bool bf16, int m, int n, int b_mn) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                        int acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <int D, int QT>
__global__ void __launch_bounds__(PrefillTcCfg<D>::kThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
  using C = PrefillTcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + C::kStages;
  uint64_t* s_full = bars + 2 * C::kStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_full + 4;
  uint64_t* pv_done = s_full + 6;
  uint64_t* q_ready = s_full + 8;
  uint64_t* tail_bar = s_full + 9;
  uint64_t* o_done = s_full + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 4 * 32) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  griddep_wait();

  const int seq = blockIdx.z;
  const int kvh = blockIdx.y;
  const int tile = p.tiles - 1 - (int)blockIdx.x;  // heaviest tiles first
  const int r0q = p.query_start_loc[seq];
  const int nq = p.query_start_loc[seq + 1] - r0q;
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
  const int nkb = last_pos / 16 + 1;
  const int nchunks = (nkb + 1) / 2;
  // The last block holds keys past the context's end when it is the block of
  // position L - 1 and L is not a multiple of 16.
  const bool has_tail = (nkb - 1 == (L - 1) / 16) && (L % 16 != 0);
  const bool bf16 = QT == 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
      mbar_init(&p_full[b], 128);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(q_ready, 128);
    mbar_init(tail_bar, 1);
    mbar_init(o_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 5) {
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

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const int32_t* tbl = p.block_tables + (size_t)seq * p.max_blocks_per_seq;
    const int oob_row = p.num_blocks * 16;
    const uint64_t pol = l2_evict_normal_policy();
    int issued = 0;
    for (int base = 0; base < nkb; base += 32) {  // warp-uniform bounds (shuffles inside)
      const int mine = (base + lane < nkb) ? __ldg(tbl + base + lane) : 0;
      const int cnt = min(32, nkb - base);
      for (int j = 0; j < cnt; ++j) {
        const int blk = __shfl_sync(0xffffffffu, mine, j);
        if (lane == 0 && !aborted()) {
          const int it = base + j;
          const int s = it % C::kStages;
          if (!mbar_wait_bounded(&empty_bar[s], ((uint32_t)(it / C::kStages) & 1u) ^ 1u, p.status)) {
            fail();
          } else {
            const int row = (blk >= 0 && blk < p.num_blocks) ? blk * 16 : oob_row;
            uint8_t* ks = smem + C::kQBytes + s * C::kStageBytes;
            mbar_arrive_expect_tx(&full_bar[s], C::kStageBytes);
            tma_load_4d(ks, &tmap_k, &full_bar[s], 0, row, 0, kvh, pol);
            tma_load_4d(ks + C::kTileBytes, &tmap_v, &full_bar[s], 0, row, 0, kvh, pol);
            ++issued;
          }
        }
      }
    }
    if (lane == 0 && has_tail && !aborted() && issued == nkb) {
      // zero the V rows of keys L .. 16 * nkb - 1 once the last block has landed
      const int it = nkb - 1;
      const int s = it % C::kStages;
      if (!mbar_wait_bounded(&full_bar[s], (uint32_t)(it / C::kStages) & 1u, p.status)) {
        fail();
      } else {
        uint8_t* vs = smem + C::kQBytes + s * C::kStageBytes + C::kTileBytes;
        for (int key = L % 16; key < 16; ++key) {
          for (int piece = 0; piece < C::kPieces; ++piece) {
            uint4* row = reinterpret_cast<uint4*>(vs + piece * 16 * 128 + key * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_shared();
        mbar_arrive(tail_bar);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = umma_idesc(bf16, 128, 16, 0);
      const uint32_t id_pv = umma_idesc(bf16, 128, D, 1);
      bool ok = mbar_wait_bounded(q_ready, 0, p.status);
      tc_fence_after();
      auto issue_pv = [&](int c) {  // O += P(c) V(c); release its stages and P buffer
        const int b = c & 1;
        if (!mbar_wait_bounded(&p_full[b], (uint32_t)(c >> 1) & 1u, p.status)) return false;
        tc_fence_after();
        for (int j = 0; j < 2; ++j) {
          const int it = 2 * c + j;
          if (it >= nkb) break;
          if (has_tail && it == nkb - 1) {
            if (!mbar_wait_bounded(tail_bar, 0, p.status)) return false;
            tc_fence_after();
          }
          const int s = it % C::kStages;
          const uint32_t vaddr = sbase + C::kQBytes + s * C::kStageBytes + C::kTileBytes;
          umma_ts(tmem + 0, tmem + C::kP0 + 16 * b + 8 * j, umma_desc_sw128(vaddr, 2048, 1024),
                  id_pv, (c > 0 || j > 0) ? 1 : 0);
          umma_commit(&empty_bar[s]);
        }
        umma_commit(&pv_done[b]);
        return true;
      };
      for (int c = 0; c < nchunks && ok; ++c) {
        const int b = c & 1;
        if (c >= 2 && !mbar_wait_bounded(&s_free[b], (uint32_t)((c - 2) >> 1) & 1u, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int j = 0; j < 2 && ok; ++j) {
          const int it = 2 * c + j;
          if (it >= nkb) break;
          const int s = it % C::kStages;
          if (!mbar_wait_bounded(&full_bar[s], (uint32_t)(it / C::kStages) & 1u, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kaddr = sbase + C::kQBytes + s * C::kStageBytes;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t qoff = (k / 4) * (C::kRows * 128) + (k % 4) * 32;
            const uint32_t koff = (k / 4) * (16 * 128) + (k % 4) * 32;
            umma_ss(tmem + C::kS0 + 32 * b + 16 * j, umma_desc_sw128(sbase + qoff, 16, 1024),
                    umma_desc_sw128(kaddr + koff, 16, 1024), id_s, k > 0 ? 1 : 0);
          }
        }
        if (!ok) break;
        umma_commit(&s_full[b]);
        if (c >= 1 && !issue_pv(c - 1)) ok = false;
      }
      if (ok && !issue_pv(nchunks - 1)) ok = false;
      if (ok) umma_commit(o_done);
      if (!ok) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    const int r = threadIdx.x;  // row of the tile, TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const int R = row0 + r;
    const bool live = R < rows;
    const int RR = live ? R : rows - 1;
    const int tok = RR / G;
    const int pos = L - nq + tok;
    const size_t qoff = ((size_t)(r0q + tok) * p.num_q_heads + (size_t)kvh * G + (RR - tok * G)) * D;
    // stage Q: row r, piece-major, 128B-swizzled (zeros for rows past the tile's end)
    {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) + qoff);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = live ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        const int piece = c / 8, cc = c % 8;
        *reinterpret_cast<uint4*>(smem + piece * (C::kRows * 128) + r * 128 + ((cc ^ (r & 7)) * 16)) = v;
      }
      fence_proxy_async_shared();
      mbar_arrive(q_ready);
    }
    // tcgen05.ld / st are warp-collective: every decision that guards one is
    // made uniform across the warp (vote) before it is acted on.
    constexpr unsigned kAll = 0xffffffffu;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      const bool w = mbar_wait_bounded(bar, parity, p.status);
      return __all_sync(kAll, w) && !__any_sync(kAll, aborted());
    };
    float m_run = -INFINITY, m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      if (!wait_all(&s_full[b], (uint32_t)(c >> 1) & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[32];
      {
        float a[16], bb[16];
        tmem_ld16(tmem + lane_base + C::kS0 + 32 * b, a);
        tmem_ld16(tmem + lane_base + C::kS0 + 32 * b + 16, bb);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          s[i] = a[i];
          s[16 + i] = bb[i];
        }
      }
      tc_fence_before();
      mbar_arrive(&s_free[b]);
      const int key0 = 32 * c;
      float mx = m_run;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float v = __fmul_rn(s[i], p.scale_log2);
        if (key0 + i > pos) v = -INFINITY;  // causal (also covers keys past L and a missing block)
        s[i] = v;
        mx = fmaxf(mx, v);
      }
      m_run = mx;
      const bool need = m_run > m_used + C::kRescale;
      if (c > 0 && __any_sync(kAll, need)) {
        // rescale O (and l) of the rows that need it, once every earlier P V
        // has landed; the warp's other rows take part with a factor of 1
        if (!wait_all(&pv_done[(c - 1) & 1], (uint32_t)((c - 1) >> 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float alpha = need ? ex2_approx(__fsub_rn(m_used, m_run)) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
          float o[16];
          tmem_ld16(tmem + lane_base + c0, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __fmul_rn(o[i], alpha);
          tmem_st16(tmem + lane_base + c0, o);
        }
        tmem_wait_st();
        l = __fmul_rn(l, alpha);
      }
      if (need) m_used = m_run;
      // P buffer b was read by the P V of chunk c - 2: wait until it is done
      if (c >= 2) {
        if (!wait_all(&pv_done[b], (uint32_t)((c - 2) >> 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      uint32_t pk[16];
      float rs = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = ex2_approx(__fsub_rn(s[2 * i], m_used));
        const float p1 = ex2_approx(__fsub_rn(s[2 * i + 1], m_used));
        pk[i] = pf_pack<QT>(p0, p1);
        const float2 rr = pf_unpack<QT>(pk[i]);
        rs = __fadd_rn(rs, __fadd_rn(rr.x, rr.y));
      }
      l = __fadd_rn(l, rs);
      tmem_st16u(tmem + lane_base + C::kP0 + 16 * b, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    if (ok) ok = wait_all(o_done, 0);
    if (!ok) fail();
    tc_fence_after();
    if (ok) {  // every lane loads (warp-collective); only rows of the tile are stored
      const bool has = l > 0.f;
      uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + qoff;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float o[16];
        tmem_ld16(tmem + lane_base + c0, o);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float a = has ? __fdiv_rn(o[2 * i], l) : 0.f;
          const float bv = has ? __fdiv_rn(o[2 * i + 1], l) : 0.f;
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
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols));
  }
}

}  // namespace pa
