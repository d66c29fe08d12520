// Pieces shared by the attention kernels (h3_attention.cu: dense attention
// by CTA pairs; h3_attention_tiles.cu: Skip-Softmax and FP8 attention):
// tile sizes, the kernel arguments, the O row store and a 16-byte shared
// store. Included by those two files only.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "h3_internal.cuh"

namespace h3 {
namespace {

constexpr int BQ = 128, BKV = 128, DH = 128;
constexpr int TILE_BYTES = BQ * DH * 2;        // 32 KB (two 64-column boxes)
constexpr int BOX_BYTES = TILE_BYTES / 2;      // 16 KB
constexpr float RESCALE_THRESHOLD = 8.0f;      // log2 units (factor 256)
constexpr float kLog2P8Scale = 7.807354922057604f;  // log2(224): FP8 P scale

struct AttnArgs {
  __nv_bfloat16* o;
  int64_t ld_out;
  int L;
  int num_kv;
  float scale_log2;  // softmax_scale * log2(e)
  float skip_log2;   // Skip-Softmax: skip a key tile when every valid row's tile max is below
                     // its exact running maximum over the kept tiles minus skip_log2
  int* kept;         // Skip-Softmax (optional): kept key tiles per (query tile, head)
  // FP8 operands: score multiplier of (query tile t, key tile j, head h) is
  // sq[t * H + h] * sk[j * H + h]; output column d of head h is scaled by
  // sv[h * 128 + d].
  const float* sq;
  const float* sk;
  const float* sv;
  int H;
  DevErr err;
};

constexpr int Q2_THREADS = 320;  // 10 warps: 8 softmax, TMA producer, MMA

// Normalises the thread's O row by 1/l and stores it (bf16) when row_ok.
// col_scale (FP8 operands): per-column factor of this head's output, or NULL.
__device__ __forceinline__ void store_o_row(uint32_t tO, float l, __nv_bfloat16* orow,
                                            bool row_ok, const float* col_scale) {
  const float inv_l = 1.0f / l;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t ov[32];
    tmem_ld32(tO + c * 32, ov);
    tmem_ld_wait();
    tmem_reg_fence(ov);
    if (col_scale != nullptr) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        ov[i] = __float_as_uint(__uint_as_float(ov[i]) * __ldg(col_scale + c * 32 + i));
    }
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
    if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
  }
}

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

// Outcome of one KV tile in a softmax warp.
enum : int { TILE_KEPT = 0, TILE_SKIPPED = 1, TILE_FAILED = -1 };

}  // namespace
}  // namespace h3
