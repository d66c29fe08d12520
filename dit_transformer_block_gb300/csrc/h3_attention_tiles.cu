// FP8 (SAGE) attention on one CTA per pair of 128-row query tiles (blog
// section 4.3, Fig. 6: Q, K, P and V in FP8 for the QK and PV products;
// Skip-Softmax as an option): one S buffer that the two query tiles use in
// turn, freed as soon as a softmax has read it, and P as E4M3 codes in tensor
// memory beside O. The BF16 attention (dense and Skip-Softmax) is in
// h3_attention.cu.
#include <algorithm>

#include "h3_attn_common.cuh"

namespace h3 {
namespace {


// ---------------------------------------------------------------------------
// FP8 (SAGE) attention, one CTA per pair of 128-row query tiles of one head,
// with the same hand-off and tensor-memory layout as the pair kernel: a
// softmax reads S into registers and frees it at once, so the other tile's
// Q K^T overlaps that softmax; P_i (E4M3 codes) is formed in registers and
// stored to tensor memory after PV_i(j-1) has finished with it; Q K^T is an
// SS kind::f8f6f4 MMA, P V the TS form (A = P_i from tensor memory).
//   warps 0-3 / 4-7: softmax of query tile 0 / 1 (thread = query row = TMEM
//     lane of S, O_i and P_i);
//   warp 8: TMA producer: Q0, Q1 once, then K_j and V_j (128 rows of 128
//     codes, 16 KB each) together into one 32 KB stage of a 4-stage ring;
//   warp 9: allocates TMEM (S, O0, O1, P0, P1); the whole warp runs the
//     issue loop, one elected lane issues: per KV step QK0(j+1) once tile 1
//     has read S1(j), PV0(j), QK1(j+1) once tile 0 has read S0(j+1), PV1(j),
//     then a commit frees stage j.
// Scores of (query tile t, key tile j, head h) are scaled by sq[t H + h] *
// sk[j H + h] (with the softmax scale); output channel d by sv[h 128 + d].
constexpr int F8_TILE = BQ * DH;          // 16 KB: one tile of E4M3 codes
constexpr int F8_STAGES = 4;
constexpr int F8_STAGE_BYTES = 2 * F8_TILE;  // K_j at 0, V_j at F8_TILE
constexpr size_t F8_SMEM_BYTES = 1024 + F8_STAGES * F8_STAGE_BYTES + 2 * F8_TILE + 256;
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
// tensor-memory columns: S (the two tiles in turn), O_i, P_i (four codes per
// column)
constexpr uint32_t TF_S = 0, TF_O = 128, TF_P = 384;
// barriers, the TMEM address word (padded to 16 bytes) and 16 vote flags
static_assert(BF_NUM * 8 + 16 + 16 * 4 <= 256, "barrier + flag region");

// One KV tile of the online softmax for the calling thread's query row, in
// base 2 with the scale folded in (scale_log2 = softmax scale * log2(e) *
// the tiles' FP8 scales): the row's scores are already in registers (sr);
// valid = keys of this tile below L (>= BKV: none masked); o_live: O already
// holds earlier tiles. The running max m is kept an integer within 1 of the
// true one (raised to the ceiling of the new max when the tile's max exceeds
// it by more than 1; then O and the row sum are rescaled), so every P is an
// exact power-of-two multiple of the P against any other integer reference;
// P is carried as 224 P (log2 224 added to the exponent), whose E4M3 codes
// are stored to tensor memory at tP (the row's lane; keys 4c .. 4c + 3 in
// column c, the lowest key in the low byte). The row sum l carries the same
// factor 224,
// which cancels in O / l. wait_pv() (the previous P V of this tile has
// finished with P and O) is called before the stores, or before an O
// rescale.
// SKIP: Skip-Softmax: the tile's four warps vote (skip_vote, step vote_tag);
// when every valid row's tile maximum lies more than skip_log2 below m_keep
// (the row's exact running maximum over the kept tiles; rows >= L vote to
// skip), nothing is computed or stored and the MMA warp leaves out the
// tile's P V.
// Returns TILE_KEPT, TILE_SKIPPED, or TILE_FAILED when a wait failed.
template <bool SKIP, class WaitPV>
__device__ __forceinline__ int softmax_tile_f8_tm(uint32_t (&sr)[128], uint32_t tP,
                                                    uint32_t tO, int valid,
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
    if (!skip_vote(!row_valid || mx < m_keep - skip_log2, flags, vote_tag, err, ok)) {
      if (!ok) return TILE_FAILED;
      // the tile's P barrier phase must not run ahead of the previous one
      return (o_live && !wait_pv()) ? TILE_FAILED : TILE_SKIPPED;
    }
    m_keep = fmaxf(m_keep, mx);
  }
  bool pv_done = !o_live;
  if (__any_sync(0xffffffffu, mx > m + 1.0f)) {
    const float m_new = ceilf(fmaxf(m, mx));
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
  if (!pv_done && !wait_pv()) return TILE_FAILED;
  tmem_st16(tP, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));  // keys 0 .. 63
  tmem_st16(tP + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
  tmem_st_wait();
  return TILE_KEPT;
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
  uint64_t* bars = reinterpret_cast<uint64_t*>(sQ + 2 * F8_TILE);
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
        mma_ss_f8_el(tmem + TF_S, qd + kk * 2, kd + kk * 2, idesc_qk, kk > 0 ? 1u : 0u);
      mma_commit_el(bar(BF_S + i));
    };
    int kept[2] = {0, 0};  // Skip-Softmax: key tiles kept per query tile
    bool any_pv[2] = {false, false};
    auto pv = [&](int i, int j) {  // O_i += P_i V_j; 32 keys (32 rows of V, 4 KB) per instruction
      volatile uint32_t* f = skip_flags + (i * 2 + (j & 1)) * 4;
      const bool skipped = SKIP && (f[0] & f[1] & f[2] & f[3] & 1u);
      if (!skipped) {  // (the first tile is never skipped)
        ++kept[i];
        const uint64_t vd = dv + stage(j);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_f8_el(tmem + TF_O + i * 128, tmem + TF_P + i * 32 + kk * 8,
                       vd + kk * (4096 >> 4), idesc_pv, (any_pv[i] || kk > 0) ? 1u : 0u);
        any_pv[i] = true;
      }
      mma_commit_el(bar(BF_PVD + i));  // also for a skipped tile: the phase counts steps
    };
    bool ok = wait(BF_Q, 0u) && wait_full(0);
    if (ok) {
      tc_fence_after();
      qk(0, 0);
      ok = wait(BF_SFREE, 0u);
      if (ok) {
        tc_fence_after();
        qk(1, 0);
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      const uint32_t par = static_cast<uint32_t>(j) & 1u;
      const bool more = j + 1 < n;
      if (more) {
        if (!wait_full(j + 1) || !wait(BF_SFREE + 1, par)) break;
        tc_fence_after();
        qk(0, j + 1);
      }
      if (!wait(BF_P, par)) break;
      tc_fence_after();
      pv(0, j);
      if (more) {
        if (!wait(BF_SFREE, par ^ 1u)) break;
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
    const uint32_t tS = tmem + lane_base + TF_S;
    const uint32_t tO = tmem + lane_base + TF_O + tile * 128;
    const uint32_t tP = tmem + lane_base + TF_P + tile * 32;
    const uint32_t row = static_cast<uint32_t>(quarter * 32 + lane);
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
      if (softmax_tile_f8_tm<SKIP>(sr, tP, tO, a.L - j * BKV, j > 0, mul, m, l,
                                     wait_pv, a.skip_log2, m_keep, row_valid,
                                     skip_flags + (tile * 2 + (j & 1)) * 4,
                                     static_cast<uint32_t>(j), a.err) == TILE_FAILED) {
        ok = false;
        break;
      }
      // the codes (and any O rescale) stored to tensor memory
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
