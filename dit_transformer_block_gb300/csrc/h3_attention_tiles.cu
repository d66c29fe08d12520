// Attention variants on one CTA per pair of 128-row query tiles (blog section
// 4.3, Fig. 6: SAGE quantisation and Skip-Softmax):
//   * Skip-Softmax over BF16 operands (attention_kernel<false, true>): the
//     softmax writes P over S in tensor memory; a key tile that every row of
//     a query tile finds negligible is left out (no exp2, no P, no P V);
//   * FP8 (SAGE) attention (attention_f8_kernel), with Skip-Softmax as an
//     option: Q, K, V and P in E4M3, S freed as soon as the softmax has read
//     it, P through shared memory.
#include <algorithm>

#include "h3_attn_common.cuh"

namespace h3 {
namespace {


// One KV tile of the online softmax for the calling thread's query row (TMEM
// lane). S_j is read from tS; P_j (bf16 pairs) is written over its first 64
// columns. valid = keys of this tile that are < L (>= BKV: none masked).
// o_live: O already holds earlier tiles (so raising the max rescales it).
// m, l: running max (times scale_log2) and row sum. Warp-collective.
// Skip-Softmax (SKIP): the four warps of a query tile vote (skip_vote, step
// vote_tag); when every valid row's tile maximum lies more than skip_log2
// below m_keep, the row's exact running maximum over the key tiles kept so
// far (rows >= L, row_valid false, vote to skip), the tile is skipped (no
// exp2, no P; the posts in flags tell the MMA warp to leave out its P V
// product) and the function returns true; otherwise m_keep takes in the
// tile's maximum. If the vote's wait runs out, ok is cleared and the function
// returns at once.
// F8: P is written as E4M3 codes (four per column, 32 columns) and the
// running max is kept an integer, so every P is an exact power-of-two multiple
// of the P against any other integer reference.
// Skip-Softmax vote of the four warps of a query tile on one KV tile (step
// vote_tag): each warp posts 2 * vote_tag + (every row of the warp votes to
// skip) in flags[quarter]. A warp that keeps the tile is done (one keeping
// warp keeps it); a warp that votes to skip reads the other three posts until
// all carry this step (bounded: on a timeout or another CTA's error, ok is
// cleared). Returns whether the tile is kept. The MMA warp reads the same
// posts (bit 0) after the tile's P barrier. A post is not overwritten before
// every warp has read it: flags alternate between two slots by step parity,
// and a warp reaches step j + 2 only after all four have taken S(j + 1).
__device__ __forceinline__ bool skip_vote(bool row_skip, volatile uint32_t* flags,
                                          uint32_t vote_tag, const DevErr& err, bool& ok) {
  const bool warp_skip = __all_sync(0xffffffffu, row_skip);
  const int quarter = (threadIdx.x >> 5) & 3;
  if ((threadIdx.x & 31) == 0) flags[quarter] = (vote_tag << 1) | (warp_skip ? 1u : 0u);
  __syncwarp();
  if (!warp_skip) return true;
  uint32_t f0, f1, f2, f3;
  uint32_t spins = 0;
  uint64_t t0 = 0;
  while (true) {
    f0 = flags[0], f1 = flags[1], f2 = flags[2], f3 = flags[3];
    if (((f0 | f1 | f2 | f3) >> 1) == vote_tag && ((f0 & f1 & f2 & f3) >> 1) == vote_tag) break;
    if ((++spins & 63u) == 0) {
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      if (*(volatile uint32_t*)err.word != 0u || now - t0 > err.timeout_ns) {
        atomicCAS(err.word, 0u, ERR_WAIT_ATTN_SOFTMAX);
        break;
      }
    }
  }
  if (!__all_sync(0xffffffffu, ((f0 & f1 & f2 & f3) >> 1) == vote_tag &&
                                   ((f0 | f1 | f2 | f3) >> 1) == vote_tag)) {
    ok = false;
    return false;
  }
  return !(f0 & f1 & f2 & f3 & 1u);
}

template <bool F8, bool SKIP>
__device__ __forceinline__ bool softmax_tile(uint32_t tS, uint32_t tO, int valid, bool o_live,
                                             float scale_log2, float& m, float& l,
                                             float skip_log2, float& m_keep, bool row_valid,
                                             volatile uint32_t* flags, uint32_t vote_tag,
                                             const DevErr& err, bool& ok) {
  uint32_t sr[128];
  {
    uint32_t (&c0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
    uint32_t (&c1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
    uint32_t (&c2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[64]);
    uint32_t (&c3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[96]);
    tmem_ld32(tS + 0, c0);
    tmem_ld32(tS + 32, c1);
    tmem_ld32(tS + 64, c2);
    tmem_ld32(tS + 96, c3);
    tmem_ld_wait();
    tmem_reg_fence(sr);
  }
  // Only the last tile holds keys >= L; mask them to -inf.
  if (valid < BKV) {
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (c >= valid) sr[c] = 0xff800000u;
  }
  if constexpr (!F8 && !SKIP) {
    if (o_live) {
      // Speculative pass (every tile after the first, whose running max is
      // finite for every row): the exponentials use the current running max
      // while the tile's max forms beside them, so the max is off the
      // critical path. When no row of the warp exceeds the running max by
      // more than the threshold — nearly always after the first tiles — this
      // is exactly the pass below with m unchanged (same operations, same
      // order); otherwise P is recomputed by the exact pass below.
      const float neg_m0 = -m;
      float sa = 0.f, sb = 0.f, sc = 0.f, sd = 0.f;
      float xa = -INFINITY, xb = -INFINITY, xc = -INFINITY, xd = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float s0 = __uint_as_float(sr[c * 32 + 2 * i]);
          const float s1 = __uint_as_float(sr[c * 32 + 2 * i + 1]);
          if ((i & 3) == 0)
            xa = max3f(xa, s0, s1);
          else if ((i & 3) == 1)
            xb = max3f(xb, s0, s1);
          else if ((i & 3) == 2)
            xc = max3f(xc, s0, s1);
          else
            xd = max3f(xd, s0, s1);
          float x0, x1;
          ffma2_bc(x0, x1, s0, s1, scale_log2, neg_m0);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          if (i & 1)
            fadd2(sc, sd, p0, p1);
          else
            fadd2(sa, sb, p0, p1);
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + c * 16, pk);
      }
      const float mxs = max3f(xa, xb, fmaxf(xc, xd)) * scale_log2;
      if (!__any_sync(0xffffffffu, mxs > m + RESCALE_THRESHOLD)) {
        l += (sa + sb) + (sc + sd);
        tmem_st_wait();
        return false;
      }
      tmem_st_wait();  // the exact pass overwrites P
    }
  }
  // Row max of the raw products (the scale is positive, so it commutes with
  // max), four independent 3-input max chains.
  float ma = -INFINITY, mb = -INFINITY, mc = -INFINITY, md = -INFINITY;
#pragma unroll
  for (int c = 0; c < 128; c += 8) {
    ma = max3f(ma, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
    mb = max3f(mb, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
    mc = max3f(mc, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
    md = max3f(md, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
  }
  const float mx = max3f(ma, mb, fmaxf(mc, md)) * scale_log2;
  if constexpr (SKIP) {
    // never on the first tile for a valid row (m_keep = -inf)
    if (!skip_vote(!row_valid || mx < m_keep - skip_log2, flags, vote_tag, err, ok)) return true;
    m_keep = fmaxf(m_keep, mx);
  }
  // Raise the running max only when it is exceeded by more than the
  // threshold; the decision is warp-uniform because the O rescale uses
  // warp-collective TMEM loads and stores.
  // FP8: the running max stays within 1 (log2) of the true one, so P <= 2
  // and 224 * P fits E4M3 (max 448) with small P still in its normal range.
  const bool need = mx > m + (F8 ? 1.0f : RESCALE_THRESHOLD);
  if (__any_sync(0xffffffffu, need)) {
    const float m_new = F8 ? ceilf(fmaxf(m, mx)) : fmaxf(m, mx);
    const float alpha = ex2_approx(m - m_new);  // 0 on the first tile
    l *= alpha;
    if (o_live) {
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {  // 16 columns at a time: the S row is live
        uint32_t ov[16];
        tmem_ld16(tO + c * 16, ov);
        tmem_ld_wait();
        tmem_reg_fence(ov);
#pragma unroll
        for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
        tmem_st16(tO + c * 16, ov);
      }
    }
    m = m_new;
  }
  // p = exp2(s * scale_log2 - m): one packed FMA per pair, two exp2, one
  // packed add into the row sum, one bf16x2 pack written over S.
  // FP8: P is carried as 224 * P (log2 224 added to the exponent); O and the
  // row sum carry the same factor, which cancels in O / l.
  const float neg_m = F8 ? (kLog2P8Scale - m) : -m;
  float la = 0.f, lb = 0.f, lc = 0.f, ld = 0.f;
  if constexpr (F8) {
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float x0, x1, x2, x3;
      ffma2_bc(x0, x1, __uint_as_float(sr[4 * i]), __uint_as_float(sr[4 * i + 1]), scale_log2,
               neg_m);
      ffma2_bc(x2, x3, __uint_as_float(sr[4 * i + 2]), __uint_as_float(sr[4 * i + 3]), scale_log2,
               neg_m);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
      fadd2(la, lb, p0, p1);
      fadd2(lc, ld, p2, p3);
      const uint32_t lo =
          __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi =
          __nv_cvt_float2_to_fp8x2(make_float2(p2, p3), __NV_SATFINITE, __NV_E4M3);
      pk[i] = lo | (hi << 16);
    }
    tmem_st32(tS, pk);
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float x0, x1;
        ffma2_bc(x0, x1, __uint_as_float(sr[c * 32 + 2 * i]),
                 __uint_as_float(sr[c * 32 + 2 * i + 1]), scale_log2, neg_m);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        if (i & 1)
          fadd2(lc, ld, p0, p1);
        else
          fadd2(la, lb, p0, p1);
        pk[i] = pack_bf16x2(p0, p1);
      }
      tmem_st16(tS + c * 16, pk);
    }
  }
  l += (la + lb) + (lc + ld);
  tmem_st_wait();
  return false;
}

// ---------------------------------------------------------------------------
// Two query tiles per CTA (256 rows of one head) sharing every K/V tile.
//   * warps 0-3 / 4-7: softmax of query tile 0 / 1 (thread = row = TMEM lane);
//   * warp 8: TMA producer (Q0, Q1 once; K_j and V_j through a 4-slot ring);
//   * warp 9: TMEM allocator (512 columns: S0, S1, O0, O1) and MMA issuer in
//     the order PV0(j), QK0(j+1), PV1(j), QK1(j+1), so each tile's softmax has
//     the other tile's two MMAs (1024 tensor clocks) to finish in; it commits
//     S0 and S1 once per KV step and O once at the end, and tile 1's softmax
//     frees the K/V slots (a commit covers every earlier product, so S1(j)
//     ready means K_j and V_{j-1} have been read);
//   * P_i is written over S_i; QK_i(j+1) is issued right behind PV_i(j) (MMAs
//     of one thread execute in issue order).
// Each K/V tile is read from shared memory by two Q tiles, which halves the
// shared-memory traffic per FLOP of the one-tile design.
constexpr int KV_SLOTS = 4;
constexpr size_t Q2_SMEM_BYTES = 1024 + (2 + KV_SLOTS) * TILE_BYTES + 256;

enum Bar2 {
  B2_Q = 0,
  B2_KV_FULL = 1,
  B2_KV_EMPTY = B2_KV_FULL + KV_SLOTS,
  B2_S = B2_KV_EMPTY + KV_SLOTS,
  B2_P = B2_S + 2,
  B2_O = B2_P + 2,
  B2_DRAIN = B2_O + 2,  // the MMA thread's last commit, waited on before exit
  B2_NUM = B2_DRAIN + 1
};
// barriers, the TMEM address word (padded to 16 bytes) and 16 vote flags
static_assert(B2_NUM * 8 + 16 + 16 * 4 <= 256, "barrier + flag region");

// F8: Q, K and V are E4M3 codes (one 128-byte TMA box per 128-row tile, 16
// KB), the MMAs are kind::f8f6f4 (K = 32 per instruction), P is written to
// TMEM as E4M3 and read back by the PV product, scores are scaled per (query
// tile, key tile) and the output per channel.
// SKIP: Skip-Softmax compiled in (a separate kernel, so the dense kernel
// carries none of its votes or branches).
template <bool F8, bool SKIP>
__global__ void __launch_bounds__(Q2_THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  constexpr int T_BYTES = F8 ? TILE_BYTES / 2 : TILE_BYTES;  // one Q/K/V tile in smem
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sKV = smem;                            // KV_SLOTS tiles
  uint8_t* sQ = smem + KV_SLOTS * T_BYTES;        // 2 tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sQ + 2 * T_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B2_NUM);
  // Skip-Softmax votes: [tile][parity of j][quarter]
  volatile uint32_t* skip_flags = tmem_slot + 4;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * 2 * BQ;
  const int col0 = blockIdx.y * DH;
  const int n = a.num_kv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < B2_NUM; ++i) mbar_init(bar(i), (i == B2_P || i == B2_P + 1) ? 128 : 1);
    fence_mbar_init();
    for (int i = 0; i < 16; ++i) skip_flags[i] = 0xffffffffu;  // no step's tag
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(B2_Q), 2 * T_BYTES);
      for (int i = 0; i < 2; ++i) {
        tma_load_2d(smem_u32(sQ + i * T_BYTES), &tmQ, bar(B2_Q), col0, q0 + i * BQ);
        if constexpr (!F8)
          tma_load_2d(smem_u32(sQ + i * T_BYTES + BOX_BYTES), &tmQ, bar(B2_Q), col0 + 64,
                      q0 + i * BQ);
      }
      int issued = 0;
      for (int t = 0; t < 2 * n; ++t) {  // even t: K_{t/2}, odd t: V_{t/2}
        const int slot = t % KV_SLOTS;
        const uint32_t use = static_cast<uint32_t>(t / KV_SLOTS);
        if (!mbar_wait(bar(B2_KV_EMPTY + slot), (use & 1u) ^ 1u, a.err, ERR_WAIT_ATTN_PRODUCER))
          break;
        const uint32_t full = bar(B2_KV_FULL + slot);
        mbar_arrive_expect_tx(full, T_BYTES);
        const CUtensorMap* m = (t & 1) ? &tmV : &tmK;
        uint8_t* dst = sKV + slot * T_BYTES;
        tma_load_2d(smem_u32(dst), m, full, col0, (t >> 1) * BKV);
        if constexpr (!F8)
          tma_load_2d(smem_u32(dst + BOX_BYTES), m, full, col0 + 64, (t >> 1) * BKV);
        issued = t + 1;
      }
      // No copy of this CTA may still be landing when it exits (after an
      // error the consumers may not have waited for them): wait, bounded, for
      // Q and for the last load of every slot. In a normal run these phases
      // completed long ago.
      const uint64_t t0 = globaltimer_ns();
      const uint64_t lim = drain_limit_ns(a.err);
      mbar_wait_drain(bar(B2_Q), 0u, t0, lim);
      for (int t = issued > KV_SLOTS ? issued - KV_SLOTS : 0; t < issued; ++t)
        mbar_wait_drain(bar(B2_KV_FULL + t % KV_SLOTS),
                        static_cast<uint32_t>(t / KV_SLOTS) & 1u, t0, lim);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = F8 ? idesc_e4m3_f32(BQ, BKV) : idesc_bf16_f32(BQ, BKV, false);
      constexpr uint32_t idesc_pv =
          F8 ? (idesc_e4m3_f32(BQ, DH) | (1u << 16)) : idesc_bf16_f32(BQ, DH, true);
      const uint32_t kv_addr = smem_u32(sKV), q_addr = smem_u32(sQ);
      auto slot_of = [](int t) { return t % KV_SLOTS; };
      auto wait_full = [&](int t) {
        return mbar_wait(bar(B2_KV_FULL + slot_of(t)),
                         static_cast<uint32_t>(t / KV_SLOTS) & 1u, a.err, ERR_WAIT_ATTN_MMA);
      };
      auto qk = [&](int i, int j) {  // S_i = Q_i K_j^T
        const uint32_t k_addr = kv_addr + slot_of(2 * j) * T_BYTES;
        const uint32_t qa = q_addr + i * T_BYTES;
        if constexpr (F8) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 32 codes = 32 bytes per step
            mma_ss_f8(tmem + i * 128, sdesc_sw128(qa + kk * 32, 16, 1024),
                      sdesc_sw128(k_addr + kk * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
            mma_ss(tmem + i * 128, sdesc_sw128(qa + off, 16, 1024),
                   sdesc_sw128(k_addr + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(B2_S + i));
      };
      int kept[2] = {0, 0};  // Skip-Softmax: key tiles kept per query tile
      auto pv = [&](int i, int j) {  // O_i += P_i V_j (left out when the tile was skipped)
        const uint32_t v_addr = kv_addr + slot_of(2 * j + 1) * T_BYTES;
        volatile uint32_t* f = skip_flags + (i * 2 + (j & 1)) * 4;
        const bool skipped = SKIP && (f[0] & f[1] & f[2] & f[3] & 1u);
        if (!skipped) {
          ++kept[i];
          if constexpr (F8) {
            // 32 keys per step: 32 rows of 128 bytes = 4 KB further; P codes
            // take 8 TMEM columns per step
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts_f8(tmem + 256 + i * 128, tmem + i * 128 + kk * 8,
                        sdesc_sw128(v_addr + kk * 4096, T_BYTES, 1024), idesc_pv,
                        (j > 0 || kk > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk)
              mma_ts(tmem + 256 + i * 128, tmem + i * 128 + kk * 8,
                     sdesc_sw128(v_addr + kk * 2048, BOX_BYTES, 1024), idesc_pv,
                     (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
      };
      bool ok = mbar_wait(bar(B2_Q), 0, a.err, ERR_WAIT_ATTN_MMA) && wait_full(0);
      if (ok) {
        tc_fence_after();
        qk(0, 0);
        qk(1, 0);
      }
      for (int j = 0; ok && j < n; ++j) {
        const uint32_t par = static_cast<uint32_t>(j) & 1u;
        if (!wait_full(2 * j + 1) || !mbar_wait(bar(B2_P), par, a.err, ERR_WAIT_ATTN_MMA)) break;
        tc_fence_after();
        pv(0, j);
        const bool more = j + 1 < n;
        if (more) {
          if (!wait_full(2 * j + 2)) break;
          tc_fence_after();
          qk(0, j + 1);
        }
        if (!mbar_wait(bar(B2_P + 1), par, a.err, ERR_WAIT_ATTN_MMA)) break;
        tc_fence_after();
        pv(1, j);
        if (more) qk(1, j + 1);
      }
      // O of both tiles is complete once every product issued so far is
      mma_commit(bar(B2_O));
      mma_commit(bar(B2_O + 1));
      if (SKIP && a.kept != nullptr && ok) {
        for (int i = 0; i < 2; ++i) {
          const int qt = blockIdx.x * 2 + i;
          if (qt * BQ < a.L) a.kept[qt * a.H + blockIdx.y] = kept[i];
        }
      }
      // Every MMA issued here must be done with shared and tensor memory
      // before the CTA frees them (after an error no consumer may have waited
      // for the last ones): commit and wait, bounded.
      mma_commit(bar(B2_DRAIN));
      mbar_wait_drain(bar(B2_DRAIN), 0u, globaltimer_ns(), drain_limit_ns(a.err));
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int tile = warp >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + tile * 128;
    const uint32_t tO = tmem + lane_base + 256 + tile * 128;
    float m = -INFINITY, l = 0.f;
    float m_keep = -INFINITY;  // Skip-Softmax: exact running max of the kept tiles
    bool ok = true;
    const bool row_valid = q0 + tile * BQ + quarter * 32 + lane < a.L;
    float sq_tile = 1.f;
    if constexpr (F8) {
      const int qt = blockIdx.x * 2 + tile;  // 128-row query tile index
      sq_tile = (qt * BQ < a.L) ? __ldg(a.sq + qt * a.H + blockIdx.y) : 0.f;
    }
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait_warp(bar(B2_S + tile), static_cast<uint32_t>(j) & 1u, a.err,
                     ERR_WAIT_ATTN_SOFTMAX)) {
        ok = false;
        break;
      }
      // S1(j) covers every product issued before it: K_j and V_{j-1} have
      // been read by both tiles, so one lane of tile 1 frees their slots
      if (tile == 1 && quarter == 0 && lane == 0) {
        mbar_arrive(bar(B2_KV_EMPTY + (2 * j) % KV_SLOTS));
        if (j > 0) mbar_arrive(bar(B2_KV_EMPTY + (2 * j - 1) % KV_SLOTS));
      }
      tc_fence_after();
      float mul = a.scale_log2;
      // a zero tile scale would turn masked (-inf) scores into NaN: keep the
      // multiplier positive
      if constexpr (F8) mul = fmaxf(mul * sq_tile * __ldg(a.sk + j * a.H + blockIdx.y), 1e-30f);
      softmax_tile<F8, SKIP>(tS, tO, a.L - j * BKV, j > 0, mul, m, l, a.skip_log2, m_keep,
                             row_valid, skip_flags + (tile * 2 + (j & 1)) * 4,
                             static_cast<uint32_t>(j), a.err, ok);
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(bar(B2_P + tile));
    }
    if (ok && mbar_wait_warp(bar(B2_O + tile), 0u, a.err, ERR_WAIT_ATTN_SOFTMAX)) {
      tc_fence_after();
      const int row = q0 + tile * BQ + quarter * 32 + lane;
      store_o_row(tO, l, a.o + static_cast<int64_t>(row) * a.ld_out + col0, row < a.L,
                  F8 ? a.sv + blockIdx.y * DH : nullptr);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// FP8 (SAGE) attention, one CTA per pair of 128-row query tiles of one head,
// with the same hand-off as the pair kernel: the softmax reads S_i into
// registers and frees it at once, so QK_i(j+1) overlaps the softmax of tile
// j; P_i (E4M3 codes) is formed in registers and stored to shared memory after
// PV_i(j-1) has finished with it; every product is an SS kind::f8f6f4 MMA.
//   warps 0-3 / 4-7: softmax of query tile 0 / 1 (thread = query row = TMEM
//     lane of S_i and O_i);
//   warp 8: TMA producer: Q0, Q1 once, then K_j and V_j (128 rows of 128
//     codes, 16 KB each) together into one 32 KB stage of a 4-stage ring;
//   warp 9: allocates TMEM (S0, S1, O0, O1); the whole warp runs the issue
//     loop, one elected lane issues: per KV step QK0(j+1), PV0(j), QK1(j+1),
//     PV1(j), then a commit frees stage j.
// Scores of (query tile t, key tile j, head h) are scaled by sq[t H + h] *
// sk[j H + h] (with the softmax scale); output channel d by sv[h 128 + d].
constexpr int F8_TILE = BQ * DH;          // 16 KB: one tile of E4M3 codes
constexpr int F8_STAGES = 4;
constexpr int F8_STAGE_BYTES = 2 * F8_TILE;  // K_j at 0, V_j at F8_TILE
constexpr size_t F8_SMEM_BYTES = 1024 + F8_STAGES * F8_STAGE_BYTES + 2 * F8_TILE + 2 * F8_TILE + 256;
static_assert(F8_SMEM_BYTES <= 227 * 1024, "fp8 attention shared memory");

enum BarF8 {
  BF_Q = 0,
  BF_FULL = 1,
  BF_EMPTY = BF_FULL + F8_STAGES,
  BF_S = BF_EMPTY + F8_STAGES,  // S_i written (MMA commit)
  BF_SFREE = BF_S + 2,          // S_i read by the softmax (4 warp arrivals)
  BF_P = BF_SFREE + 2,          // P_i written (4 warp arrivals)
  BF_PVD = BF_P + 2,            // P_i V_j done (MMA commit)
  BF_O = BF_PVD + 2,
  BF_DRAIN = BF_O + 1,
  BF_NUM = BF_DRAIN + 1
};
// barriers, the TMEM address word (padded to 16 bytes) and 16 vote flags
static_assert(BF_NUM * 8 + 16 + 16 * 4 <= 256, "barrier + flag region");

// softmax_tile<true, false>'s arithmetic for one KV tile (integer running max
// within 1 of the true one, P carried as 224 P, E4M3 codes), with the row's
// scores already in registers (sr) and the codes stored to shared memory at
// p_row = the P tile's address + 128 * row, 16-byte chunk c of the row at
// chunk c ^ r7 (r7 = row & 7: the 128-byte swizzle of a K-major tile). The
// codes, m and l are bitwise those of softmax_tile<true, false>. wait_pv() is
// called before the stores, or before an O rescale.
// SKIP: Skip-Softmax as in softmax_tile<false, true>: the tile's four warps
// vote through flags[quarter], each tagged with vote_tag (the KV step); when
// every valid row's tile maximum lies more than skip_log2 below m_keep (the
// row's exact running maximum over the kept tiles; rows >= L vote to skip),
// nothing is computed or stored and the MMA warp leaves out the tile's P V.
// Returns F8_KEPT, F8_SKIPPED, or F8_FAILED when a wait failed.
enum : int { F8_KEPT = 0, F8_SKIPPED = 1, F8_FAILED = -1 };
template <bool SKIP, class WaitPV>
__device__ __forceinline__ int softmax_tile_f8_smem(uint32_t (&sr)[128], uint32_t p_row,
                                                    uint32_t r7, uint32_t tO, int valid,
                                                    bool o_live, float scale_log2, float& m,
                                                    float& l, WaitPV&& wait_pv, float skip_log2,
                                                    float& m_keep, bool row_valid,
                                                    volatile uint32_t* flags, uint32_t vote_tag,
                                                    const DevErr& err) {
  if (valid < BKV) {
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (c >= valid) sr[c] = 0xff800000u;
  }
  float ma = -INFINITY, mb = -INFINITY, mc = -INFINITY, md = -INFINITY;
#pragma unroll
  for (int c = 0; c < 128; c += 8) {
    ma = max3f(ma, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
    mb = max3f(mb, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
    mc = max3f(mc, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
    md = max3f(md, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
  }
  const float mx = max3f(ma, mb, fmaxf(mc, md)) * scale_log2;
  if constexpr (SKIP) {
    // never on the first tile for a valid row (m_keep = -inf)
    bool ok = true;
    if (!skip_vote(!row_valid || mx < m_keep - skip_log2, flags, vote_tag, err, ok))
      return ok ? F8_SKIPPED : F8_FAILED;
    m_keep = fmaxf(m_keep, mx);
  }
  bool pv_done = !o_live;
  if (__any_sync(0xffffffffu, mx > m + 1.0f)) {
    const float m_new = ceilf(fmaxf(m, mx));
    const float alpha = ex2_approx(m - m_new);  // 0 on the first tile
    l *= alpha;
    if (o_live) {
      if (!wait_pv()) return F8_FAILED;
      pv_done = true;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t ov[16];
        tmem_ld16(tO + c * 16, ov);
        tmem_ld_wait();
        tmem_reg_fence(ov);
#pragma unroll
        for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
        tmem_st16(tO + c * 16, ov);
      }
      tmem_st_wait();
    }
    m = m_new;
  }
  const float neg_m = kLog2P8Scale - m;
  float la = 0.f, lb = 0.f, lc = 0.f, ld = 0.f;
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float x0, x1, x2, x3;
    ffma2_bc(x0, x1, __uint_as_float(sr[4 * i]), __uint_as_float(sr[4 * i + 1]), scale_log2,
             neg_m);
    ffma2_bc(x2, x3, __uint_as_float(sr[4 * i + 2]), __uint_as_float(sr[4 * i + 3]), scale_log2,
             neg_m);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
    fadd2(la, lb, p0, p1);
    fadd2(lc, ld, p2, p3);
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(p2, p3), __NV_SATFINITE, __NV_E4M3);
    pk[i] = lo | (hi << 16);
  }
  l += (la + lb) + (lc + ld);
  if (!pv_done && !wait_pv()) return F8_FAILED;
#pragma unroll
  for (uint32_t c = 0; c < 8; ++c)  // keys 16 c .. 16 c + 15
    st_shared_v4(p_row + ((c ^ r7) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
  return F8_KEPT;
}

// SKIP: Skip-Softmax compiled in (a separate instance, so the plain kernel
// carries none of its votes or branches).
template <bool SKIP>
__global__ void __launch_bounds__(Q2_THREADS, 1)
    attention_f8_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sKV = smem;                                // F8_STAGES stages
  uint8_t* sQ = smem + F8_STAGES * F8_STAGE_BYTES;    // 2 tiles
  uint8_t* sP = sQ + 2 * F8_TILE;                     // 2 tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * F8_TILE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + BF_NUM);
  // Skip-Softmax votes: [tile][parity of j][quarter]
  volatile uint32_t* skip_flags = tmem_slot + 4;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * 2 * BQ;
  const int col0 = blockIdx.y * DH;  // byte column of the head's codes
  const int n = a.num_kv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < BF_NUM; ++i) mbar_init(bar(i), (i >= BF_SFREE && i < BF_PVD) ? 4 : 1);
    fence_mbar_init();
    for (int i = 0; i < 16; ++i) skip_flags[i] = 0xffffffffu;  // no step's tag
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(BF_Q), 2 * F8_TILE);
      for (int i = 0; i < 2; ++i)
        tma_load_2d(smem_u32(sQ + i * F8_TILE), &tmQ, bar(BF_Q), col0, q0 + i * BQ);
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j % F8_STAGES;
        const uint32_t use = static_cast<uint32_t>(j / F8_STAGES);
        if (!mbar_wait(bar(BF_EMPTY + st), (use & 1u) ^ 1u, a.err, ERR_WAIT_ATTN_PRODUCER)) break;
        const uint32_t full = bar(BF_FULL + st);
        mbar_arrive_expect_tx(full, F8_STAGE_BYTES);
        const uint32_t dst = smem_u32(sKV + st * F8_STAGE_BYTES);
        tma_load_2d(dst, &tmK, full, col0, j * BKV);
        tma_load_2d(dst + F8_TILE, &tmV, full, col0, j * BKV);
        issued = j + 1;
      }
      // no copy of this CTA may still be landing when it exits
      const uint64_t t0 = globaltimer_ns();
      const uint64_t lim = drain_limit_ns(a.err);
      mbar_wait_drain(bar(BF_Q), 0u, t0, lim);
      for (int j = issued > F8_STAGES ? issued - F8_STAGES : 0; j < issued; ++j)
        mbar_wait_drain(bar(BF_FULL + j % F8_STAGES), static_cast<uint32_t>(j / F8_STAGES) & 1u,
                        t0, lim);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc_qk = idesc_e4m3_f32(BQ, BKV);
    constexpr uint32_t idesc_pv = idesc_e4m3_f32(BQ, DH) | (1u << 16);  // V MN-major
    const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dp = sdesc_sw128(smem_u32(sP), 16, 1024);
    const uint64_t dk = sdesc_sw128(smem_u32(sKV), 16, 1024);
    const uint64_t dv = sdesc_sw128(smem_u32(sKV) + F8_TILE, F8_TILE, 1024);
    auto wait = [&](int b, uint32_t parity) {
      return mbar_wait_warp(bar(b), parity, a.err, ERR_WAIT_ATTN_MMA);
    };
    auto wait_full = [&](int j) {
      return wait(BF_FULL + j % F8_STAGES, static_cast<uint32_t>(j / F8_STAGES) & 1u);
    };
    auto stage = [](int j) { return static_cast<uint32_t>((j % F8_STAGES) * (F8_STAGE_BYTES >> 4)); };
    auto qk = [&](int i, int j) {  // S_i = Q_i K_j^T; 32 codes (32 bytes) per instruction
      const uint64_t qd = dq + static_cast<uint32_t>(i * (F8_TILE >> 4));
      const uint64_t kd = dk + stage(j);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss_f8_el(tmem + i * 128, qd + kk * 2, kd + kk * 2, idesc_qk, kk > 0 ? 1u : 0u);
      mma_commit_el(bar(BF_S + i));
    };
    int kept[2] = {0, 0};  // Skip-Softmax: key tiles kept per query tile
    bool any_pv[2] = {false, false};
    auto pv = [&](int i, int j) {  // O_i += P_i V_j; 32 keys (32 rows of V, 4 KB) per instruction
      volatile uint32_t* f = skip_flags + (i * 2 + (j & 1)) * 4;
      const bool skipped = SKIP && (f[0] & f[1] & f[2] & f[3] & 1u);
      if (!skipped) {  // (the first tile is never skipped)
        ++kept[i];
        const uint64_t pd = dp + static_cast<uint32_t>(i * (F8_TILE >> 4));
        const uint64_t vd = dv + stage(j);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss_f8_el(tmem + 256 + i * 128, pd + kk * 2, vd + kk * (4096 >> 4), idesc_pv,
                       (any_pv[i] || kk > 0) ? 1u : 0u);
        any_pv[i] = true;
      }
      mma_commit_el(bar(BF_PVD + i));  // also for a skipped tile: the phase counts steps
    };
    bool ok = wait(BF_Q, 0u) && wait_full(0);
    if (ok) {
      tc_fence_after();
      qk(0, 0);
      qk(1, 0);
    }
    for (int j = 0; ok && j < n; ++j) {
      const uint32_t par = static_cast<uint32_t>(j) & 1u;
      const bool more = j + 1 < n;
      if (more) {
        if (!wait_full(j + 1) || !wait(BF_SFREE, par)) break;
        tc_fence_after();
        qk(0, j + 1);
      }
      if (!wait(BF_P, par)) break;
      tc_fence_after();
      pv(0, j);
      if (more) {
        if (!wait(BF_SFREE + 1, par)) break;
        tc_fence_after();
        qk(1, j + 1);
      }
      if (!wait(BF_P + 1, par)) break;
      tc_fence_after();
      pv(1, j);
      mma_commit_el(bar(BF_EMPTY + j % F8_STAGES));  // K_j, V_j read
    }
    mma_commit_el(bar(BF_O));
    if (SKIP && a.kept != nullptr && ok && lane == 0) {
      for (int i = 0; i < 2; ++i) {
        const int qt = blockIdx.x * 2 + i;
        if (qt * BQ < a.L) a.kept[qt * a.H + blockIdx.y] = kept[i];
      }
    }
    // every MMA must be done with shared and tensor memory before the CTA
    // frees them: commit and wait, bounded
    mma_commit_el(bar(BF_DRAIN));
    mbar_wait_drain(bar(BF_DRAIN), 0u, globaltimer_ns(), drain_limit_ns(a.err));
  } else {
    // ---------------------------------------------------------- softmax
    const int tile = warp >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + tile * 128;
    const uint32_t tO = tmem + lane_base + 256 + tile * 128;
    const uint32_t row = static_cast<uint32_t>(quarter * 32 + lane);
    const uint32_t p_row = smem_u32(sP + tile * F8_TILE) + row * 128;
    const int qt = blockIdx.x * 2 + tile;  // 128-row query tile index
    const float sq_tile = (qt * BQ < a.L) ? __ldg(a.sq + qt * a.H + blockIdx.y) : 0.f;
    float m = -INFINITY, l = 0.f;
    float m_keep = -INFINITY;  // Skip-Softmax: exact running max of the kept tiles
    const bool row_valid = q0 + tile * BQ + static_cast<int>(row) < a.L;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait_warp(bar(BF_S + tile), static_cast<uint32_t>(j) & 1u, a.err,
                          ERR_WAIT_ATTN_SOFTMAX)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
      {
        uint32_t (&c0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
        uint32_t (&c1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
        uint32_t (&c2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[64]);
        uint32_t (&c3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[96]);
        tmem_ld32(tS + 0, c0);
        tmem_ld32(tS + 32, c1);
        tmem_ld32(tS + 64, c2);
        tmem_ld32(tS + 96, c3);
        tmem_ld_wait();
        tmem_reg_fence(sr);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BF_SFREE + tile));  // S_i read
      // a zero tile scale would turn masked (-inf) scores into NaN: keep the
      // multiplier positive
      const float mul =
          fmaxf(a.scale_log2 * sq_tile * __ldg(a.sk + j * a.H + blockIdx.y), 1e-30f);
      auto wait_pv = [&]() {  // P_i V_{j-1} done with P_i and O_i
        const bool done = mbar_wait_warp(bar(BF_PVD + tile), static_cast<uint32_t>(j - 1) & 1u,
                                         a.err, ERR_WAIT_ATTN_SOFTMAX);
        tc_fence_after();
        return done;
      };
      if (softmax_tile_f8_smem<SKIP>(sr, p_row, row & 7u, tO, a.L - j * BKV, j > 0, mul, m, l,
                                     wait_pv, a.skip_log2, m_keep, row_valid,
                                     skip_flags + (tile * 2 + (j & 1)) * 4,
                                     static_cast<uint32_t>(j), a.err) == F8_FAILED) {
        ok = false;
        break;
      }
      fence_proxy_async_smem();  // the codes, for the tensor core's reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BF_P + tile));
    }
    if (ok && mbar_wait_warp(bar(BF_O), 0u, a.err, ERR_WAIT_ATTN_SOFTMAX)) {
      tc_fence_after();
      const int orow = q0 + tile * BQ + static_cast<int>(row);
      store_o_row(tO, l, a.o + static_cast<int64_t>(orow) * a.ld_out + col0, orow < a.L,
                  a.sv + blockIdx.y * DH);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <bool F8, bool SKIP>
static h3_status set_attention_smem() {
  static std::atomic<bool> done[64];
  const size_t bytes = F8 ? 1024 + (2 + KV_SLOTS) * (TILE_BYTES / 2) + 256 : Q2_SMEM_BYTES;
  return set_smem_limit(done, attention_kernel<F8, SKIP>, bytes,
                        "attention: set shared memory size");
}

h3_status launch_attention_skip(const void* q, const void* k, const void* v, int64_t ld_in,
                                void* o, int64_t ld_out, int L, int H, float scale,
                                cudaStream_t s, float skip_eps, int* kept) {
  h3_status st = set_attention_smem<false, true>();
  if (st != H3_OK) return st;
  AttnArgs a{};
  a.o = static_cast<__nv_bfloat16*>(o);
  a.ld_out = ld_out;
  a.L = L;
  a.H = H;
  a.num_kv = (L + BKV - 1) / BKV;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.skip_log2 = skip_eps > 0.f ? -log2f(skip_eps) : INFINITY;
  a.kept = skip_eps > 0.f ? kept : nullptr;  // the counts only when tiles may be skipped
  if ((st = dev_err(&a.err)) != H3_OK) return st;
  CUtensorMap tq, tk, tv;
  const uint64_t width = static_cast<uint64_t>(H) * DH;
  const uint64_t stride = static_cast<uint64_t>(ld_in) * 2;
  if ((st = make_tmap_bf16_2d(&tq, q, width, L, stride, 64, BQ)) != H3_OK) return st;
  if ((st = make_tmap_bf16_2d(&tk, k, width, L, stride, 64, BKV)) != H3_OK) return st;
  if ((st = make_tmap_bf16_2d(&tv, v, width, L, stride, 64, BKV)) != H3_OK) return st;
  dim3 grid((L + 2 * BQ - 1) / (2 * BQ), H);
  attention_kernel<false, true><<<grid, Q2_THREADS, Q2_SMEM_BYTES, s>>>(tq, tk, tv, a);
  return cuda_fail(cudaGetLastError(), "attention (skip) launch");
}

h3_status launch_attention_fp8(const void* qc, const void* kc, const void* vc, int64_t ld_codes,
                               const float* sq, const float* sk, const float* sv, void* o,
                               int64_t ld_out, int L, int H, float scale, cudaStream_t s,
                               float skip_eps, int* kept) {
  const bool skip = skip_eps >= 0.f;
  static std::atomic<bool> done[64], done_skip[64];
  h3_status st = skip ? set_smem_limit(done_skip, attention_f8_kernel<true>, F8_SMEM_BYTES,
                                       "attention (fp8, skip): set shared memory size")
                      : set_smem_limit(done, attention_f8_kernel<false>, F8_SMEM_BYTES,
                                       "attention (fp8): set shared memory size");
  if (st != H3_OK) return st;
  AttnArgs a{};
  a.o = static_cast<__nv_bfloat16*>(o);
  a.ld_out = ld_out;
  a.L = L;
  a.H = H;
  a.num_kv = (L + BKV - 1) / BKV;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.skip_log2 = skip_eps > 0.f ? -log2f(skip_eps) : INFINITY;
  a.kept = skip_eps > 0.f ? kept : nullptr;  // the counts only when tiles may be skipped
  if ((st = dev_err(&a.err)) != H3_OK) return st;
  CUtensorMap tq, tk, tv;
  const uint64_t width = static_cast<uint64_t>(H) * DH;  // bytes per row of codes
  if ((st = make_tmap_u8_2d(&tq, qc, width, L, ld_codes, 128, BQ)) != H3_OK) return st;
  if ((st = make_tmap_u8_2d(&tk, kc, width, L, ld_codes, 128, BKV)) != H3_OK) return st;
  if ((st = make_tmap_u8_2d(&tv, vc, width, L, ld_codes, 128, BKV)) != H3_OK) return st;
  dim3 grid((L + 2 * BQ - 1) / (2 * BQ), H);
  if (skip)
    attention_f8_kernel<true><<<grid, Q2_THREADS, F8_SMEM_BYTES, s>>>(tq, tk, tv, a);
  else
    attention_f8_kernel<false><<<grid, Q2_THREADS, F8_SMEM_BYTES, s>>>(tq, tk, tv, a);
  return cuda_fail(cudaGetLastError(), "attention (fp8) launch");
}

}  // namespace h3
