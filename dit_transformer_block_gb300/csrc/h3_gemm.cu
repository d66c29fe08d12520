// tcgen05 GEMM for the block projections: C[:L] = epilogue(A[:L] @ B^T),
// bf16 operands, FP32 accumulation in tensor memory, bf16 output.
//
// The matrix multiplies are the ones the fused small ops of the vLLM-Omni H3
// blog (section 3.2) sit around: QKV, attention output, FFN gate/up, FFN down.
//
// Design (one CTA per SM, persistent over output tiles):
//   * tile 128 x 256 (M x N), K step 64; A and B are K-major in global memory
//     and land in shared memory through TMA with 128-byte swizzle;
//   * a 4-stage ring of (A 16 KB + B 32 KB) stages, full/empty mbarriers;
//   * warp 0: TMA producer (one lane); warp 1: TMEM allocator and MMA issuer
//     (one lane, tcgen05.mma M=128 N=256 K=16); warps 2-5: epilogue, each owns
//     the 32 TMEM lanes (= tile rows) its warp index selects;
//   * two 256-column FP32 accumulators in TMEM so the epilogue of one tile
//     overlaps the main loop of the next;
//   * rows >= L are zero-filled by TMA on load and never stored.
// Epilogues (each rounds the product to bf16 first, like the unfused path):
//   * plain bf16 store;
//   * SwiGLU: the B tile's first 128 rows are gate rows and the last 128 the
//     matching up rows; the 128 output columns are SiLU(g) * u;
//   * residual: C is the FP32 residual stream and gets gate[col] * bf16(acc)
//     added with one fma, the arithmetic of the modulation kernel's residual
//     step, so the block's residual update needs no pass of its own;
//   * Q/K RMSNorm + RoPE: a 256-column tile is two 128-channel heads; a q or k
//     head of the thread's row is normalised by its RMS (a first pass over its
//     TMEM columns), scaled by the gain and rotated pair by pair with the row's
//     (cos, sin) table, then stored; v columns are stored as they are.
#include <cuda_bf16.h>

#include <algorithm>

#include "h3_internal.cuh"

namespace h3 {
namespace {

// BK counts bf16 elements; an FP8 stage holds 2 * BK codes in the same bytes.
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = BN * BK * 2;        // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;              // two accumulators of BN columns
constexpr int GROUP_M = 32;                 // raster: 32 M-blocks per N sweep
constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/;

struct GemmArgs {
  void* C;
  int64_t ldc;
  const float* sa;        // FP8: per-row scale of A [M]
  const float* sb;        // FP8: per-row scale of B [rows of B]
  int M, N, K;            // M = valid rows; N = output columns
  int num_m, num_n, num_k;
  int num_tiles;
  int ep;                 // GemmEpilogue
  int b_half_rows;        // SwiGLU: row offset of the up half inside B
  GemmExtra x;            // operands of the residual and Q/K-norm epilogues
  DevErr err;
};

__device__ __forceinline__ void tile_coords(int tile, const GemmArgs& a, int& mb, int& nb) {
  const int group_size = GROUP_M * a.num_n;
  const int group = tile / group_size;
  const int first_m = group * GROUP_M;
  const int gm = min(a.num_m - first_m, GROUP_M);
  const int r = tile - group * group_size;
  mb = first_m + r % gm;
  nb = r / gm;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// 8 accumulator columns [col, col + 8) of this thread's row (col a multiple
// of 8, relative to taddr's column), FP8-scaled when FP8, each rounded to
// bf16. Loads the 16-column block holding them.
template <bool FP8>
__device__ __forceinline__ void load8_bf16(uint32_t taddr, int col, float sa_row, const float* sb,
                                           float (&x)[8]) {
  uint32_t v[16];
  tmem_ld16(taddr + static_cast<uint32_t>(col & ~15), v);
  tmem_ld_wait();
  tmem_reg_fence(v);
  const bool hi = (col & 8) != 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float f = __uint_as_float(hi ? v[8 + j] : v[j]);
    if constexpr (FP8) f *= sa_row * __ldg(sb + col + j);
    x[j] = round_to_bf16(f);
  }
}

// 32 accumulator columns of this thread's row, FP8-scaled when FP8, each
// rounded to bf16 (returned as floats).
template <bool FP8>
__device__ __forceinline__ void load_chunk_bf16(uint32_t taddr, float sa_row, const float* sb,
                                                float (&x)[32]) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  tmem_ld_wait();
  tmem_reg_fence(v);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float f = __uint_as_float(v[j]);
    if constexpr (FP8) f *= sa_row * __ldg(sb + j);
    x[j] = round_to_bf16(f);
  }
}

// FP8 == true: A and B hold E4M3 codes (kind::f8f6f4, K = 32 per MMA, 128
// codes per 128-byte row of a stage) and the epilogue multiplies the FP32
// accumulator by sa[row] * sb[col] before rounding to bf16.
template <bool FP8>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs a) {
  constexpr int KB_ELEMS = FP8 ? 2 * BK : BK;  // elements per K block
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* full = bars;                 // [STAGES]
  uint64_t* empty = bars + STAGES;       // [STAGES]
  uint64_t* tfull = bars + 2 * STAGES;   // [2]
  uint64_t* tempty = tfull + 2;          // [2]
  uint64_t* drain = tempty + 2;          // the MMA thread's last commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int issued = 0;  // stage loads issued: load i went to stage i % STAGES, parity (i / STAGES) & 1
      for (int tile = blockIdx.x; tile < a.num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, a, mb, nb);
        int b_row0, b_row1;
        if (a.ep == GEMM_SWIGLU) {
          b_row0 = nb * (BN / 2);
          b_row1 = a.b_half_rows + nb * (BN / 2);
        } else {
          b_row0 = nb * BN;
          b_row1 = nb * BN + BN / 2;
        }
        for (int kb = 0; kb < a.num_k; ++kb) {
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, a.err, ERR_WAIT_GEMM_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const int kx = kb * KB_ELEMS;
          tma_load_2d(smem_u32(sA + stage * A_BYTES), &tmA, fb, kx, mb * BM);
          tma_load_2d(smem_u32(sB + stage * B_BYTES), &tmB, fb, kx, b_row0);
          tma_load_2d(smem_u32(sB + stage * B_BYTES + B_BYTES / 2), &tmB, fb, kx, b_row1);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // No copy of this CTA may still be landing when it exits (after an
      // error the consumer may not have waited for them): wait, bounded, for
      // the last load of every stage.
      const uint64_t t0 = globaltimer_ns();
      for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
        mbar_wait_drain(smem_u32(&full[i % STAGES]), static_cast<uint32_t>(i / STAGES) & 1u, t0,
                        drain_limit_ns(a.err));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = FP8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < a.num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, a.err, ERR_WAIT_GEMM_MMA)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < a.num_k; ++kb) {
          if (!mbar_wait(smem_u32(&full[stage]), phase, a.err, ERR_WAIT_GEMM_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = sdesc_sw128(a0 + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + k * 32, 16, 1024);
            if constexpr (FP8)
              mma_ss_f8(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            else
              mma_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&tfull[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued here must be done with shared and tensor memory
      // before the CTA frees them: commit and wait, bounded
      mma_commit(smem_u32(drain));
      mbar_wait_drain(smem_u32(drain), 0u, globaltimer_ns(), drain_limit_ns(a.err));
    }
  } else {
    // ------------------------------------------------------ epilogue warps
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < a.num_tiles; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, a, mb, nb);
      if (!mbar_wait_warp(smem_u32(&tfull[acc]), acc_phase, a.err, ERR_WAIT_GEMM_EPILOGUE)) break;
      tc_fence_after();
      const int row = mb * BM + quarter * 32 + lane;
      const bool row_ok = row < a.M;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      __nv_bfloat16* crow =
          static_cast<__nv_bfloat16*>(a.C) + static_cast<int64_t>(row) * a.ldc;
      const float sa_row = FP8 ? (row_ok ? __ldg(a.sa + row) : 0.f) : 1.f;
      if (a.ep == GEMM_SWIGLU) {
        const int col0 = nb * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2 / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(t_row + c * 32, g);
          tmem_ld32(t_row + BN / 2 + c * 32, u);
          tmem_ld_wait();
          tmem_reg_fence(g);
          tmem_reg_fence(u);
          if constexpr (FP8) {
            const float* sg = a.sb + col0 + c * 32;
            const float* su = a.sb + a.b_half_rows + col0 + c * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              g[j] = __float_as_uint(__uint_as_float(g[j]) * (sa_row * __ldg(sg + j)));
              u[j] = __float_as_uint(__uint_as_float(u[j]) * (sa_row * __ldg(su + j)));
            }
          }
          uint32_t o[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float g0 = round_to_bf16(__uint_as_float(g[2 * j]));
            const float g1 = round_to_bf16(__uint_as_float(g[2 * j + 1]));
            const float u0 = round_to_bf16(__uint_as_float(u[2 * j]));
            const float u1 = round_to_bf16(__uint_as_float(u[2 * j + 1]));
            o[j] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
          }
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(crow + col0 + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
        }
      } else if (a.ep == GEMM_RESIDUAL) {
        const int col0 = nb * BN;
        float* rrow = static_cast<float*>(a.C) + static_cast<int64_t>(row) * a.ldc + col0;
        const float* grow = a.x.gate + col0;
        if (a.x.seg != nullptr && row_ok)
          grow += static_cast<int64_t>(min(max(__ldg(a.x.seg + row), 0), a.x.num_seg - 1)) *
                  a.x.seg_stride;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float f[32];
          load_chunk_bf16<FP8>(t_row + c * 32, sa_row, a.sb + col0 + c * 32, f);
          if (row_ok) {
            float4* rp = reinterpret_cast<float4*>(rrow + c * 32);
            const float4* gp = reinterpret_cast<const float4*>(grow + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 r = __ldcs(rp + q);
              const float4 g = __ldg(gp + q);
              r.x = fmaf(g.x, f[4 * q + 0], r.x);
              r.y = fmaf(g.y, f[4 * q + 1], r.y);
              r.z = fmaf(g.z, f[4 * q + 2], r.z);
              r.w = fmaf(g.w, f[4 * q + 3], r.w);
              __stcs(rp + q, r);
            }
          }
        }
      } else if (a.ep == GEMM_QK_NORM_ROPE && nb * BN < 2 * a.x.d_model) {
        const float2* rope = a.x.rope + static_cast<int64_t>(row_ok ? row : 0) * 64;
#pragma unroll 1
        for (int hh = 0; hh < BN / 128; ++hh) {
          const int hcol = nb * BN + hh * 128;
          const float* gain = hcol < a.x.d_model ? a.x.q_gain : a.x.k_gain;
          const uint32_t t_head = t_row + hh * 128;
          // pass 1: sum of squares of the bf16-rounded head
          float ss = 0.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float f[32];
            load_chunk_bf16<FP8>(t_head + c * 32, sa_row, a.sb + hcol + c * 32, f);
#pragma unroll
            for (int j = 0; j < 32; ++j) ss = fmaf(f[j], f[j], ss);
          }
          const float inv = rsqrtf(ss * (1.0f / 128.0f) + a.x.eps);
          if (a.x.pairing == 1) {
            // pass 2, split-half pairs: eight pieces of eight pairs
#pragma unroll 1
            for (int pc = 0; pc < 8; ++pc) {
              const int f0 = a.x.piece_first[pc], s0 = a.x.piece_second[pc];
              const int p0 = a.x.piece_pair[pc];
              float xf[8], xs[8];
              load8_bf16<FP8>(t_head, f0, sa_row, a.sb + hcol, xf);
              load8_bf16<FP8>(t_head, s0, sa_row, a.sb + hcol, xs);
              float yf[8], ys[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float2 r = __ldg(rope + p0 + j);
                const float x0 = xf[j] * inv * __ldg(gain + f0 + j);
                const float x1 = xs[j] * inv * __ldg(gain + s0 + j);
                yf[j] = x0 * r.x - x1 * r.y;
                ys[j] = x0 * r.y + x1 * r.x;
              }
              if (row_ok) {
                *reinterpret_cast<uint4*>(crow + hcol + f0) =
                    make_uint4(pack_bf16x2(yf[0], yf[1]), pack_bf16x2(yf[2], yf[3]),
                               pack_bf16x2(yf[4], yf[5]), pack_bf16x2(yf[6], yf[7]));
                *reinterpret_cast<uint4*>(crow + hcol + s0) =
                    make_uint4(pack_bf16x2(ys[0], ys[1]), pack_bf16x2(ys[2], ys[3]),
                               pack_bf16x2(ys[4], ys[5]), pack_bf16x2(ys[6], ys[7]));
              }
            }
            continue;
          }
          // pass 2: scale, gain, rotate, store
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float f[32];
            load_chunk_bf16<FP8>(t_head + c * 32, sa_row, a.sb + hcol + c * 32, f);
            uint32_t o[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const float2 r = __ldg(rope + c * 16 + t);
              const float g0 = __ldg(gain + c * 32 + 2 * t);
              const float g1 = __ldg(gain + c * 32 + 2 * t + 1);
              const float x0 = f[2 * t] * inv * g0;
              const float x1 = f[2 * t + 1] * inv * g1;
              o[t] = pack_bf16x2(x0 * r.x - x1 * r.y, x0 * r.y + x1 * r.x);
            }
            if (row_ok) {
              uint4* dst = reinterpret_cast<uint4*>(crow + hcol + c * 32);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            }
          }
        }
      } else {
        const int col0 = nb * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(t_row + c * 32, v);
          tmem_ld_wait();
          tmem_reg_fence(v);
          if constexpr (FP8) {
            const float* sc = a.sb + col0 + c * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] = __float_as_uint(__uint_as_float(v[j]) * (sa_row * __ldg(sc + j)));
          }
          uint32_t o[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            o[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(crow + col0 + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

template <bool FP8>
static h3_status launch_gemm_impl(const void* A, int64_t lda_bytes, const float* sa, const void* B,
                                  int64_t ldb_bytes, const float* sb, void* C, int64_t ldc, int L,
                                  int N, int K, GemmEpilogue ep, cudaStream_t s,
                                  const GemmExtra* extra) {
  static std::atomic<bool> done[64];
  h3_status st = set_smem_limit(done, gemm_kernel<FP8>, SMEM_BYTES, "gemm: set shared memory size");
  if (st != H3_OK) return st;
  constexpr int kb_elems = FP8 ? 2 * BK : BK;
  GemmArgs a{};
  a.C = C;
  a.ldc = ldc;
  a.sa = sa;
  a.sb = sb;
  a.M = L;
  a.N = N;
  a.K = K;
  a.ep = ep;
  if (extra != nullptr) a.x = *extra;
  const int b_rows = (ep == GEMM_SWIGLU) ? 2 * N : N;
  const int tile_n = (ep == GEMM_SWIGLU) ? BN / 2 : BN;
  a.b_half_rows = (ep == GEMM_SWIGLU) ? N : 0;
  a.num_m = (L + BM - 1) / BM;
  a.num_n = N / tile_n;
  a.num_k = (K + kb_elems - 1) / kb_elems;
  a.num_tiles = a.num_m * a.num_n;
  st = dev_err(&a.err);
  if (st != H3_OK) return st;

  CUtensorMap tmA, tmB;
  auto tmap = FP8 ? make_tmap_u8_2d : make_tmap_bf16_2d;
  st = tmap(&tmA, A, static_cast<uint64_t>(K), static_cast<uint64_t>(L),
            static_cast<uint64_t>(lda_bytes), kb_elems, BM);
  if (st != H3_OK) return st;
  st = tmap(&tmB, B, static_cast<uint64_t>(K), static_cast<uint64_t>(b_rows),
            static_cast<uint64_t>(ldb_bytes), kb_elems, BN / 2);
  if (st != H3_OK) return st;
  const int grid = std::min(a.num_tiles, num_sms());
  gemm_kernel<FP8><<<grid, THREADS, SMEM_BYTES, s>>>(tmA, tmB, a);
  return cuda_fail(cudaGetLastError(), "gemm launch");
}

void rope_pieces(const int* axis_dims, GemmExtra* ex) {
  int n = 0, o = 0;
  for (int a = 0; a < 3; ++a) {
    const int d = axis_dims[a];
    for (int c = 0; c < d / 2 && n < 8; c += 8, ++n) {
      ex->piece_first[n] = o + c;
      ex->piece_second[n] = o + d / 2 + c;
      ex->piece_pair[n] = o / 2 + c;
    }
    o += d;
  }
  ex->pairing = 1;
}

h3_status launch_gemm(const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                      int64_t ldc, int L, int N, int K, GemmEpilogue ep, cudaStream_t s,
                      const GemmExtra* extra) {
  return launch_gemm_impl<false>(A, lda * 2, nullptr, B, ldb * 2, nullptr, C, ldc, L, N, K, ep, s,
                                 extra);
}

h3_status launch_gemm_fp8(const void* A, int64_t lda, const float* sa, const void* B, int64_t ldb,
                          const float* sb, void* C, int64_t ldc, int L, int N, int K,
                          GemmEpilogue ep, cudaStream_t s, const GemmExtra* extra) {
  return launch_gemm_impl<true>(A, lda, sa, B, ldb, sb, C, ldc, L, N, K, ep, s, extra);
}

}  // namespace h3
