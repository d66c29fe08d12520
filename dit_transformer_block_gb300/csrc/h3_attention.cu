// Dense bidirectional attention over the valid length of a packed sequence,
// on tcgen05 tensor cores: CTA pairs (cta_group::2, M = 256 products), S, P
// and O in tensor memory.
//
// vLLM-Omni H3 blog, section 3.1: the attention backend receives the valid
// sequence length and the structural tail padding is dropped, so no key >= L
// takes part and no query row >= L is produced; section 3.3 / 4.3 name dense
// BF16 attention as the reference behaviour.
//
// The online softmax is base 2 with the scale folded in (packed FP32 FMA and
// add, 3-input max); the running max is raised only when a row's new max
// exceeds it by more than 8 (then O and the row sum are rescaled); only the
// last KV tile is masked. With Skip-Softmax (blog section 4.3, Fig. 6) a key
// tile that every row of a CTA's query tile finds negligible gives those rows
// nothing. The FP8 (SAGE) attention is in h3_attention_tiles.cu.
#include <algorithm>

#include "h3_attn_common.cuh"

namespace h3 {
namespace {

// ---------------------------------------------------------------------------
// CTA-pair form (tcgen05 cta_group::2). The two CTAs of a cluster run one head
// over 512 query rows as two M = 256 groups: group g covers rows
// p0 + 256 g .. p0 + 256 g + 255, and CTA r holds rows p0 + 256 g + 128 r ..
// + 127 of it (its query tile g). Every product is one M = 256 MMA issued by
// the MMA warp of the even CTA; each CTA supplies its own 128 rows of A (Q
// from its shared memory, or P from its tensor memory) and half of B: keys
// 64 r .. 64 r + 63 of K_j for S = Q K^T, head channels 64 r .. 64 r + 63 of
// V_j for O += P V. So each SM reads half of every K/V tile from its own
// shared memory and receives the other half from its peer.
//
// Tensor memory (512 columns): one S buffer that the two groups use in turn,
// O_0, O_1, and P_0, P_1 in columns of their own (bf16, two per column), so
// S is free as soon as a group's softmax has read it into registers: the
// other group's Q K^T then overwrites it while that softmax runs, and P V
// reads P from tensor memory. Shared memory carries only the Q tiles and the
// K/V stages (per KV step and CTA about 160 KB of operand reads and copies,
// against 2,048 cycles of MMA at 128 bytes per cycle); P stored with
// tcgen05.st takes about 190 cycles per tile, where the same stores to shared
// memory took about 460 while the P V products were reading it. The softmax
// of a group forms its whole P row in registers and waits for the group's
// previous P V only before storing it (or before an O rescale), so that
// product overlaps the exponentials.
// Roles per CTA (320 threads):
//   warps 0-3 / 4-7: softmax of the CTA's query tile 0 / 1: S from tensor
//     memory into registers, one lane per warp tells the even CTA's MMA warp
//     that S is free, then the tile's P is written to tensor memory and one
//     lane per warp tells the MMA warp that P is ready;
//   warp 8: TMA producer of the CTA's own halves: its Q tiles once, then, per
//     KV step, its K half and V half together into one 32 KB stage of a
//     3-stage ring, on its own barriers;
//   warp 9: allocates tensor memory (both CTAs together; S, O0, O1, P0, P1); in
//     the even CTA the whole warp runs the issue loop and one elected lane
//     issues each MMA and commit (both CTAs' barriers); in the odd CTA one
//     lane relays: each time one of its own stages has landed it arrives on
//     the even CTA's barrier of that stage, so the MMA issuer sees both halves.
// A stage is freed by a commit after the last product that reads it (PV1).
// Every wait is bounded; both CTAs meet at a cluster barrier before they free
// tensor memory, after the MMA issuer has waited for its last MMAs.
constexpr int P2_STAGES = 3;
constexpr int HALF_BYTES = TILE_BYTES / 2;   // 64 keys x 128 ch, or 128 keys x 64 ch (bf16)
constexpr int STAGE2_BYTES = 2 * HALF_BYTES; // K half at 0, V half at HALF_BYTES
// stages, Q tiles, barriers and flags (227 KB is the per-CTA limit)
constexpr size_t P2_SMEM_BYTES =
    1024 + P2_STAGES * STAGE2_BYTES + 2 * TILE_BYTES + 512;
static_assert(P2_SMEM_BYTES <= 227 * 1024, "pair kernel shared memory");

enum BarP {
  BP_Q = 0,
  BP_FULL = 1,                    // stage landed (both CTAs' halves, via the relay)
  BP_EMPTY = BP_FULL + P2_STAGES, // stage read by every product (MMA commit)
  BP_S = BP_EMPTY + P2_STAGES,    // S_g written (MMA commit)
  BP_SFREE = BP_S + 2,            // S_g read by the softmax (8 warp arrivals)
  BP_P = BP_SFREE + 2,            // P_g written (8 warp arrivals)
  BP_PVD = BP_P + 2,              // P_g V_j done (MMA commit)
  BP_O = BP_PVD + 2,
  BP_DRAIN = BP_O + 1,
  BP_NUM = BP_DRAIN + 1
};
// tensor-memory columns: S (one buffer, the two groups in turn), O_g, P_g
// (two bf16 per column)
constexpr uint32_t TM_S = 0, TM_O = 128, TM_P = 384;
// barriers, the TMEM address word (padded to 16 bytes), 16 vote flags, 16
// decisions of the peer CTA and 4 of its own
static_assert(BP_NUM * 8 + 16 + 16 * 4 + 16 * 4 + 4 * 4 <= 512, "barrier + flag region");

// One KV tile of the online softmax for the calling thread's query row (TMEM
// lane), in base 2 with the scale folded in (scale_log2 = softmax scale *
// log2(e)); the row's 128 scores are already in registers (sr); valid = keys
// of this tile below L (>= BKV: none masked); o_live: O already holds
// earlier tiles; m, l: running max (times scale_log2) and row sum. The
// running max is raised only when the tile's max exceeds it by more than
// RESCALE_THRESHOLD (then O and l are rescaled, warp-uniformly). P (bf16) is
// written to tensor memory at tP (the row's lane; keys 2c and 2c + 1 in
// column c, the even key in the low half), where the P V product reads it as
// its A operand. The whole P row
// is formed in registers first and stored last: wait_pv() (the previous P V
// of this tile has finished with P and O) is called only before the stores,
// or before an O rescale, so that wait overlaps the exponentials.
// SKIP: Skip-Softmax: the four warps of the CTA's query tile vote (skip_vote,
// step vote_tag); when every valid row's tile maximum lies more than
// skip_log2 below m_keep (the row's exact running maximum over the kept
// tiles; rows >= L vote to skip), the tile gives these rows nothing: the
// group's P V still runs for the peer CTA's rows, so P is set to zero
// (once: p_zero records that it already is).
// Returns TILE_KEPT, TILE_SKIPPED, or TILE_FAILED when a wait failed.
template <bool SKIP, class WaitPV>
__device__ __forceinline__ int softmax_tile_tm(uint32_t (&sr)[128], uint32_t tP,
                                                 uint32_t tO, int valid, bool o_live,
                                                 float scale_log2, float& m, float& l,
                                                 WaitPV&& wait_pv, float skip_log2, float& m_keep,
                                                 bool row_valid, volatile uint32_t* flags,
                                                 uint32_t vote_tag, bool& p_zero,
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
    if (!skip_vote(!row_valid || mx < m_keep - skip_log2, flags, vote_tag, err, ok)) {
      if (!ok) return TILE_FAILED;
      // also before the P arrive: the group's P barrier takes both CTAs'
      // warps, and its phase must not run ahead of the previous one
      if (o_live && !wait_pv()) return TILE_FAILED;
      if (!p_zero) {
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16(tP + c * 16, z);
        tmem_st_wait();
        p_zero = true;
      }
      return TILE_SKIPPED;
    }
    m_keep = fmaxf(m_keep, mx);
  }
  bool pv_done = !o_live;  // the first tile has no earlier product
  if (__any_sync(0xffffffffu, mx > m + RESCALE_THRESHOLD)) {
    const float m_new = fmaxf(m, mx);
    const float alpha = ex2_approx(m - m_new);  // 0 on the first tile
    l *= alpha;
    if (o_live) {
      if (!wait_pv()) return TILE_FAILED;
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
  const float neg_m = -m;
  float la = 0.f, lb = 0.f, lc = 0.f, ld = 0.f;
  uint32_t pk[64];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float x0, x1;
      ffma2_bc(x0, x1, __uint_as_float(sr[c * 32 + 2 * i]), __uint_as_float(sr[c * 32 + 2 * i + 1]),
               scale_log2, neg_m);
      const float p0 = ex2_approx(x0);
      const float p1 = ex2_approx(x1);
      if (i & 1)
        fadd2(lc, ld, p0, p1);
      else
        fadd2(la, lb, p0, p1);
      pk[c * 16 + i] = pack_bf16x2(p0, p1);
    }
  }
  l += (la + lb) + (lc + ld);
  if (!pv_done && !wait_pv()) return TILE_FAILED;
#pragma unroll
  for (int c = 0; c < 4; ++c)  // keys 32 c .. 32 c + 31
    tmem_st16(tP + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[c * 16]));
  tmem_st_wait();
  if constexpr (SKIP) p_zero = false;
  return TILE_KEPT;
}

// SKIP: Skip-Softmax compiled in (a separate instance, so the dense kernel
// carries none of its votes or branches).
template <bool SKIP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Q2_THREADS, 1)
    attention_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sKV = smem;                             // P2_STAGES stages
  uint8_t* sQ = smem + P2_STAGES * STAGE2_BYTES;   // 2 tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sQ + 2 * TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + BP_NUM);
  // Skip-Softmax votes of this CTA: [tile][parity of j][quarter]; in the even
  // CTA, the odd CTA's decisions (1: its query tile left the key tile out),
  // same layout
  volatile uint32_t* skip_flags = tmem_slot + 4;
  volatile uint32_t* peer_skip = skip_flags + 16;
  // in the even CTA, its own tiles' decisions [tile][parity of j] (each of
  // the tile's warps writes the same value)
  volatile uint32_t* own_skip = peer_skip + 16;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int p0 = (blockIdx.x >> 1) * 4 * BQ;
  const int col0 = blockIdx.y * DH;
  const int n = a.num_kv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < BP_NUM; ++i) {
      uint32_t count = 1;
      // the even CTA's Q and stage barriers also take the odd CTA's relay
      if (i == BP_Q || (i >= BP_FULL && i < BP_FULL + P2_STAGES)) count = leader ? 2 : 1;
      // one lane per softmax warp of the group, both CTAs
      if (i >= BP_SFREE && i < BP_PVD) count = 8;
      mbar_init(bar(i), count);
    }
    fence_mbar_init();
    if constexpr (SKIP)
      for (int i = 0; i < 16; ++i) skip_flags[i] = 0xffffffffu;  // no step's tag
  }
  if (warp == 9) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(BP_Q), 2 * TILE_BYTES);
      for (int g = 0; g < 2; ++g) {
        const int row = p0 + 2 * BQ * g + BQ * static_cast<int>(rank);
        tma_load_2d(smem_u32(sQ + g * TILE_BYTES), &tmQ, bar(BP_Q), col0, row);
        tma_load_2d(smem_u32(sQ + g * TILE_BYTES + BOX_BYTES), &tmQ, bar(BP_Q), col0 + 64, row);
      }
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j % P2_STAGES;
        const uint32_t use = static_cast<uint32_t>(j / P2_STAGES);
        if (!mbar_wait(bar(BP_EMPTY + st), (use & 1u) ^ 1u, a.err, ERR_WAIT_ATTN_PRODUCER))
          break;
        const uint32_t full = bar(BP_FULL + st);
        mbar_arrive_expect_tx(full, STAGE2_BYTES);
        const uint32_t dst = smem_u32(sKV + st * STAGE2_BYTES);
        const int key0 = j * BKV;
        const int k_row = key0 + 64 * static_cast<int>(rank);
        tma_load_2d(dst, &tmK, full, col0, k_row);
        tma_load_2d(dst + HALF_BYTES / 2, &tmK, full, col0 + 64, k_row);
        tma_load_2d(dst + HALF_BYTES, &tmV, full, col0 + 64 * static_cast<int>(rank), key0);
        issued = j + 1;
      }
      // No copy of this CTA may still be landing when it exits: wait, bounded,
      // for Q and for the last load of every stage (long done in a normal run).
      const uint64_t t0 = globaltimer_ns();
      const uint64_t lim = drain_limit_ns(a.err);
      mbar_wait_drain(bar(BP_Q), 0u, t0, lim);
      for (int j = issued > P2_STAGES ? issued - P2_STAGES : 0; j < issued; ++j)
        mbar_wait_drain(bar(BP_FULL + j % P2_STAGES), static_cast<uint32_t>(j / P2_STAGES) & 1u,
                        t0, lim);
    }
  } else if (warp == 9) {
    if (leader) {
      // -------------------------------------------------------- MMA issuer
      // The whole warp runs the loop; one elected lane issues. Descriptors
      // are a base plus a constant offset (start address field, in 16-byte
      // units; shared-memory addresses stay below 2^18, so no carry).
      constexpr uint32_t idesc_qk = idesc_bf16_f32(2 * BQ, BKV, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(2 * BQ, DH, true);
      const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk = sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t dv = sdesc_sw128(smem_u32(sKV) + HALF_BYTES, HALF_BYTES, 1024);
      constexpr uint16_t kBoth = 3;
      auto wait = [&](int b, uint32_t parity) {
        return mbar_wait_warp(bar(b), parity, a.err, ERR_WAIT_ATTN_MMA);
      };
      auto wait_full = [&](int j) {
        return wait(BP_FULL + j % P2_STAGES, static_cast<uint32_t>(j / P2_STAGES) & 1u);
      };
      // 16-byte offset of K step kk (16 elements) in a K-major 128-byte-swizzled tile
      auto kmaj = [](int kk, int box_bytes) {
        return static_cast<uint32_t>(((kk >> 2) * box_bytes + (kk & 3) * 32) >> 4);
      };
      auto qk = [&](int g, int j) {  // S = Q_g K_j^T over both CTAs' rows
        const uint64_t kd = dk + static_cast<uint32_t>((j % P2_STAGES) * (STAGE2_BYTES >> 4));
        const uint64_t qd = dq + static_cast<uint32_t>(g * (TILE_BYTES >> 4));
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk)
          mma_ss_pair_el(tmem + TM_S, qd + kmaj(kk, BOX_BYTES), kd + kmaj(kk, HALF_BYTES / 2),
                         idesc_qk, kk > 0 ? 1u : 0u);
        mma_commit_pair_mc_el(bar(BP_S + g), kBoth);
      };
      bool any_pv[2] = {false, false};
      auto pv = [&](int g, int j) {  // O_g += P_g V_j
        bool skipped = false;
        if constexpr (SKIP) {  // both CTAs' query tiles left key tile j out: no product
          const uint32_t own = own_skip[g * 2 + (j & 1)];
          const uint32_t peer = peer_skip[(g * 2 + (j & 1)) * 4];
          skipped = (own & peer) != 0u;
        }
        if (!skipped) {
          const uint64_t vd = dv + static_cast<uint32_t>((j % P2_STAGES) * (STAGE2_BYTES >> 4));
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)  // P_g from tensor memory, 16 keys = 8 columns
            mma_ts_pair_el(tmem + TM_O + g * 128, tmem + TM_P + g * 64 + kk * 8,
                           vd + kk * (2048 >> 4), idesc_pv, (any_pv[g] || kk > 0) ? 1u : 0u);
          any_pv[g] = true;
        }
        mma_commit_pair_mc_el(bar(BP_PVD + g), kBoth);  // also when left out: phases count steps
      };
      bool ok = wait(BP_Q, 0u) && wait_full(0);
      if (ok) {
        tc_fence_after();
        qk(0, 0);
        ok = wait(BP_SFREE, 0u);
        if (ok) {
          tc_fence_after();
          qk(1, 0);
        }
      }
      // Per KV step: QK0(j+1) once group 1 has read S1(j), PV0(j), QK1(j+1)
      // once group 0 has read S0(j+1), PV1(j); a stage is free once PV1 of it
      // is done. S is read while the other group's P V runs.
      for (int j = 0; ok && j < n; ++j) {
        const uint32_t par = static_cast<uint32_t>(j) & 1u;
        const bool more = j + 1 < n;
        if (more) {
          if (!wait_full(j + 1) || !wait(BP_SFREE + 1, par)) break;
          tc_fence_after();
          qk(0, j + 1);
        }
        if (!wait(BP_P, par)) break;
        tc_fence_after();
        pv(0, j);
        if (more) {
          if (!wait(BP_SFREE, par ^ 1u)) break;
          tc_fence_after();
          qk(1, j + 1);
        }
        if (!wait(BP_P + 1, par)) break;
        tc_fence_after();
        pv(1, j);
        mma_commit_pair_mc_el(bar(BP_EMPTY + j % P2_STAGES), kBoth);  // K_j, V_j read
      }
      // O of both groups is complete once every product issued so far is
      mma_commit_pair_mc_el(bar(BP_O), kBoth);
      // Every MMA issued here must be done with both CTAs' shared and tensor
      // memory before either frees them: commit and wait, bounded.
      mma_commit_pair_mc_el(bar(BP_DRAIN), 1);
      mbar_wait_drain(bar(BP_DRAIN), 0u, globaltimer_ns(), drain_limit_ns(a.err));
    } else if (lane == 0) {
      // ------------------------------------------------------------ relay
      if (mbar_wait(bar(BP_Q), 0, a.err, ERR_WAIT_ATTN_PRODUCER)) {
        mbar_arrive_remote(mapa_shared(bar(BP_Q), 0));
        for (int j = 0; j < n; ++j) {
          const int st = j % P2_STAGES;
          if (!mbar_wait(bar(BP_FULL + st), static_cast<uint32_t>(j / P2_STAGES) & 1u, a.err,
                         ERR_WAIT_ATTN_PRODUCER))
            break;
          mbar_arrive_remote(mapa_shared(bar(BP_FULL + st), 0));
        }
      }
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int tile = warp >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + TM_S;
    const uint32_t tO = tmem + lane_base + TM_O + tile * 128;
    const uint32_t tP = tmem + lane_base + TM_P + tile * 64;
    const uint32_t row = static_cast<uint32_t>(quarter * 32 + lane);
    // one lane per warp tells the even CTA's MMA warp
    auto tell = [&](int b) {
      if (lane == 0) {
        if (leader)
          mbar_arrive(bar(b));
        else
          mbar_arrive_remote(mapa_shared(bar(b), 0));
      }
    };
    float m = -INFINITY, l = 0.f;
    float m_keep = -INFINITY;  // Skip-Softmax: exact running max of the kept tiles
    // first row of the CTA's query tile
    auto qrow0 = [&]() { return p0 + 2 * BQ * tile + BQ * static_cast<int>(rank); };
    bool p_zero = false;
    int kept = 0;
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      if (!mbar_wait_warp(bar(BP_S + tile), static_cast<uint32_t>(j) & 1u, a.err,
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
      // S read: the next Q K^T of this group may overwrite it
      tc_fence_before();
      __syncwarp();
      tell(BP_SFREE + tile);
      // P_g V_{j-1} must be done before P_g is overwritten and O_g rescaled
      auto wait_pv = [&]() {
        const bool done = mbar_wait_warp(bar(BP_PVD + tile), static_cast<uint32_t>(j - 1) & 1u,
                                         a.err, ERR_WAIT_ATTN_SOFTMAX);
        tc_fence_after();
        return done;
      };
      const int got = softmax_tile_tm<SKIP>(sr, tP, tO, a.L - j * BKV, j > 0,
                                              a.scale_log2, m, l, wait_pv, a.skip_log2, m_keep,
                                              qrow0() + static_cast<int>(row) < a.L,
                                              skip_flags + (tile * 2 + (j & 1)) * 4,
                                              static_cast<uint32_t>(j), p_zero, a.err);
      if (got == TILE_FAILED) {
        ok = false;
        break;
      }
      if constexpr (SKIP) kept += got == TILE_KEPT ? 1 : 0;
      // P and any O rescale stored to tensor memory: tell the MMA warp
      tc_fence_before();
      __syncwarp();
      if constexpr (SKIP) {
        // with the tile's decision: the odd CTA stores it into the even CTA's
        // shared memory with st.async, whose 4 bytes complete on the P
        // barrier (each of the even CTA's warps adds 4 expected bytes)
        if (lane == 0) {
          if (leader) {
            own_skip[tile * 2 + (j & 1)] = got == TILE_SKIPPED ? 1u : 0u;
            mbar_arrive_expect_tx(bar(BP_P + tile), 4);
          } else {
            const uint32_t slot =
                smem_u32(const_cast<uint32_t*>(peer_skip) + (tile * 2 + (j & 1)) * 4 + quarter);
            const uint32_t pb = mapa_shared(bar(BP_P + tile), 0);
            st_async_u32(mapa_shared(slot, 0), got == TILE_SKIPPED ? 1u : 0u, pb);
            mbar_arrive_remote(pb);
          }
        }
      } else {
        tell(BP_P + tile);
      }
    }
    if (SKIP && ok && a.kept != nullptr && quarter == 0 && lane == 0 && qrow0() < a.L)
      a.kept[(qrow0() / BQ) * a.H + blockIdx.y] = kept;
    if (ok && mbar_wait_warp(bar(BP_O), 0u, a.err, ERR_WAIT_ATTN_SOFTMAX)) {
      tc_fence_after();
      const int orow = qrow0() + static_cast<int>(row);
      store_o_row(tO, l, a.o + static_cast<int64_t>(orow) * a.ld_out + col0, orow < a.L, nullptr);
    }
  }

  tc_fence_before();
  cluster_sync_all();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

// The pair kernel with or without Skip-Softmax (skip_eps < 0: dense).
static h3_status launch_pair(const void* q, const void* k, const void* v, int64_t ld_in, void* o,
                             int64_t ld_out, int L, int H, float scale, cudaStream_t s,
                             float skip_eps, int* kept) {
  const bool skip = skip_eps >= 0.f;
  static std::atomic<bool> done[64], done_skip[64];
  h3_status st = skip ? set_smem_limit(done_skip, attention_pair_kernel<true>, P2_SMEM_BYTES,
                                       "attention (skip): set shared memory size")
                      : set_smem_limit(done, attention_pair_kernel<false>, P2_SMEM_BYTES,
                                       "attention: set shared memory size");
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
  if ((st = make_tmap_bf16_2d(&tk, k, width, L, stride, 64, BKV / 2)) != H3_OK) return st;
  if ((st = make_tmap_bf16_2d(&tv, v, width, L, stride, 64, BKV)) != H3_OK) return st;
  // CTA pairs (a cluster of two along x), 512 query rows per pair
  dim3 grid(2 * ((L + 4 * BQ - 1) / (4 * BQ)), H);
  if (skip)
    attention_pair_kernel<true><<<grid, Q2_THREADS, P2_SMEM_BYTES, s>>>(tq, tk, tv, a);
  else
    attention_pair_kernel<false><<<grid, Q2_THREADS, P2_SMEM_BYTES, s>>>(tq, tk, tv, a);
  return cuda_fail(cudaGetLastError(), skip ? "attention (skip) launch" : "attention launch");
}

h3_status launch_attention(const void* q, const void* k, const void* v, int64_t ld_in,
                           void* o, int64_t ld_out, int L, int H, float scale, cudaStream_t s,
                           float skip_eps, int* kept) {
  return launch_pair(q, k, v, ld_in, o, ld_out, L, H, scale, s, skip_eps, kept);
}

}  // namespace h3
