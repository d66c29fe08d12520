// HBM-bound single-pass kernels of the DiT block: SwiGLU, per-head Q/K
// RMSNorm + RoPE, and FP32 modulation + LayerNorm + residual. Each reads its
// operands once with 16-byte (or 8-byte) vector loads, reduces with warp
// shuffles, and writes its result once; only rows < L are touched.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cmath>

#include "h3_internal.cuh"

namespace h3 {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }

// ------------------------------------------------------------------ SwiGLU
// vLLM-Omni H3 blog, section 3.2 (#6283): SiLU(g) * u in one launch.
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t swiglu_pair(uint32_t g, uint32_t u) {
  return pack_bf16x2(silu_f(bf16_lo(g)) * bf16_lo(u), silu_f(bf16_hi(g)) * bf16_hi(u));
}

constexpr int SWIGLU_THREADS = 256;
constexpr int SWIGLU_UNROLL = 4;

__global__ void __launch_bounds__(SWIGLU_THREADS)
    swiglu_kernel(const uint4* __restrict__ gu, uint4* __restrict__ out, int L, int F8) {
  for (int row = blockIdx.x; row < L; row += gridDim.x) {
    const uint4* g_row = gu + static_cast<int64_t>(row) * 2 * F8;
    const uint4* u_row = g_row + F8;
    uint4* o_row = out + static_cast<int64_t>(row) * F8;
    for (int c0 = threadIdx.x; c0 < F8; c0 += SWIGLU_THREADS * SWIGLU_UNROLL) {
      uint4 g[SWIGLU_UNROLL], u[SWIGLU_UNROLL];
#pragma unroll
      for (int i = 0; i < SWIGLU_UNROLL; ++i) {
        const int c = c0 + i * SWIGLU_THREADS;
        if (c < F8) {
          g[i] = ld_stream(g_row + c);
          u[i] = ld_stream(u_row + c);
        }
      }
#pragma unroll
      for (int i = 0; i < SWIGLU_UNROLL; ++i) {
        const int c = c0 + i * SWIGLU_THREADS;
        if (c < F8) {
          uint4 r;
          r.x = swiglu_pair(g[i].x, u[i].x);
          r.y = swiglu_pair(g[i].y, u[i].y);
          r.z = swiglu_pair(g[i].z, u[i].z);
          r.w = swiglu_pair(g[i].w, u[i].w);
          __stcs(o_row + c, r);
        }
      }
    }
  }
}

// ------------------------------------------------------ Q/K RMSNorm + RoPE
// vLLM-Omni H3 blog, section 3.2 (#5990) and section 3.1 (per-token RoPE rows).
// One warp owns one (row, tensor) pair: lanes 0-15 and 16-31 each cover one
// 128-wide head (8 channels = 4 rotation pairs per lane), so a head's RMS is a
// 16-lane shuffle reduction and every lane needs the angles of only its own
// four pairs, computed once per row.
constexpr int QK_HEAD_DIM = 128;
constexpr int QK_WARPS = 8;
// head pairs loaded per batch: interleaved pairs 11 (22 heads), split-half
// pairs, with more live values per head, 4 (measured: 0.367 / 0.446 ms at the
// 58,816-row size, against 0.372 / 0.455 with 8 for both)
template <bool HALF>
constexpr int QK_BATCH = HALF ? 4 : 11;

struct RopeTable {
  // turns per unit position of each pair, omega / (2 pi) in 0.64 fixed point
  // (omega / (2 pi) rounded to double, then scaled exactly by 2^64)
  uint64_t turn[QK_HEAD_DIM / 2];
  int axis[QK_HEAD_DIM / 2];      // which position (t, h, w) drives the pair
  // split-half layout, per 8-channel slice s of a head: the slice holding the
  // partners, whether s holds first elements, and the pair of its channel 0
  int half_src[QK_HEAD_DIM / 8];
  int half_first[QK_HEAD_DIM / 8];
  int half_pair0[QK_HEAD_DIM / 8];
};

// Angle of a pair at position p: its turns p * omega / (2 pi) modulo 1, exact
// in 64-bit fixed point (the integer product wraps modulo 2^64, i.e. whole
// turns), read as a signed fraction t of a half turn in [-1, 1) (one rounding
// to float32), then sin and cos of pi * t in FP32. No FP64 arithmetic, whose
// rate on this GPU is a small fraction of FP32's.
__device__ __forceinline__ void rope_angle(int32_t p, uint64_t turn, float& sn, float& cs) {
  const uint64_t f = static_cast<uint64_t>(static_cast<int64_t>(p)) * turn;
  const float t = __ll2float_rn(static_cast<int64_t>(f)) * 0x1p-63f;
  sincospif(t, &sn, &cs);
}

// One thread per (row, pair): out[row * 64 + pr] = (cos, sin).
__global__ void __launch_bounds__(256)
    rope_table_kernel(const int32_t* __restrict__ pos, int L, const RopeTable tab,
                      float2* __restrict__ out) {
  const int64_t i = blockIdx.x * 256LL + threadIdx.x;
  if (i >= static_cast<int64_t>(L) * (QK_HEAD_DIM / 2)) return;
  const int64_t row = i / (QK_HEAD_DIM / 2);
  const int pr = static_cast<int>(i - row * (QK_HEAD_DIM / 2));
  float sn, cs;
  rope_angle(__ldg(pos + 3 * row + tab.axis[pr]), tab.turn[pr], sn, cs);
  out[i] = make_float2(cs, sn);
}

// HALF: split-half pairs (o + j, o + d/2 + j) per section instead of
// interleaved ones. Each half of a section is a multiple of 8 channels, so a
// lane's slice holds only first or only second elements, of 8 consecutive
// pairs, and reads its partners from one other lane of its half-warp.
template <bool HALF>
__global__ void __launch_bounds__(QK_WARPS * 32)
    qk_norm_rope_kernel(__nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
                        int64_t row_stride, const float* __restrict__ q_gain,
                        const float* __restrict__ k_gain, const int32_t* __restrict__ pos,
                        int L, int H, float eps, const RopeTable tab) {
  const int warp = blockIdx.x * QK_WARPS + (threadIdx.x >> 5);
  const int row = warp >> 1;
  if (row >= L) return;
  const int which = warp & 1;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;   // 8-channel slice of the head
  const int half = lane >> 4;  // even / odd head of each pair

  __nv_bfloat16* base = (which ? k : q) + static_cast<int64_t>(row) * row_stride + sub * 8;
  const float* gp = (which ? k_gain : q_gain) + sub * 8;
  const float4 g0 = __ldg(reinterpret_cast<const float4*>(gp));
  const float4 g1 = __ldg(reinterpret_cast<const float4*>(gp + 4));
  const float gain[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};

  // the first batch of heads is requested before the angles are formed, so
  // the loads are in flight meanwhile
  uint4 v[QK_BATCH<HALF>];
  auto load_batch = [&](int h0) {
#pragma unroll
    for (int i = 0; i < QK_BATCH<HALF>; ++i) {
      const int head = h0 + 2 * i + half;
      v[i] = make_uint4(0, 0, 0, 0);
      if (head < H) v[i] = *reinterpret_cast<const uint4*>(base + head * QK_HEAD_DIM);
    }
  };
  load_batch(0);

  // Angles of this lane's pairs: 4 interleaved pairs; or, split-half, 8 pairs
  // shared with the partner lane, each lane evaluating 4 of them
  constexpr int NP = HALF ? 8 : 4;
  const int32_t p3[3] = {__ldg(pos + 3 * row), __ldg(pos + 3 * row + 1), __ldg(pos + 3 * row + 2)};
  float cs[NP], sn[NP];
  const int src_lane = (half << 4) + (HALF ? tab.half_src[sub] : 0);
  const bool first = HALF ? tab.half_first[sub] != 0 : true;
  const int pair0 = (HALF ? tab.half_pair0[sub] : sub * 4) + (first ? 0 : 4);
  float c4[4], s4[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int pr = pair0 + t;
    rope_angle(p3[tab.axis[pr]], tab.turn[pr], s4[t], c4[t]);
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    if constexpr (HALF) {
      const float oc = __shfl_sync(0xffffffffu, c4[t], src_lane);
      const float os = __shfl_sync(0xffffffffu, s4[t], src_lane);
      cs[t] = first ? c4[t] : oc;
      sn[t] = first ? s4[t] : os;
      cs[4 + t] = first ? oc : c4[t];
      sn[4 + t] = first ? os : s4[t];
    } else {
      cs[t] = c4[t];
      sn[t] = s4[t];
    }
  }

  for (int h0 = 0; h0 < H; h0 += 2 * QK_BATCH<HALF>) {
    if (h0 > 0) load_batch(h0);
#pragma unroll
    for (int i = 0; i < QK_BATCH<HALF>; ++i) {
      const int head = h0 + 2 * i + half;
      if (h0 + 2 * i >= H) break;  // uniform across the warp
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      float x[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[2 * j] = bf16_lo(w[j]);
        x[2 * j + 1] = bf16_hi(w[j]);
      }
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
#pragma unroll
      for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      const float inv = rsqrtf(ss * (1.0f / QK_HEAD_DIM) + eps);
      uint32_t o[4];
      if constexpr (HALF) {
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float a = x[j] * inv * gain[j];
          const float b = __shfl_sync(0xffffffffu, a, src_lane);  // the pair's other element
          // first elements: a c - b s; second elements: b s + a c
          y[j] = first ? a * cs[j] - b * sn[j] : b * sn[j] + a * cs[j];
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) o[t] = pack_bf16x2(y[2 * t], y[2 * t + 1]);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float a = x[2 * t] * inv * gain[2 * t];
          const float b = x[2 * t + 1] * inv * gain[2 * t + 1];
          o[t] = pack_bf16x2(a * cs[t] - b * sn[t], a * sn[t] + b * cs[t]);
        }
      }
      if (head < H)
        *reinterpret_cast<uint4*>(base + head * QK_HEAD_DIM) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// ----------------------------------------- modulation + LayerNorm + residual
// vLLM-Omni H3 blog, section 3.2 (#6281, #6878): FP32 modulation,
// normalisation and residual in one pass. One CTA per row; each thread keeps
// VPT float4 of the row in registers between the residual update and the
// two-pass mean/variance.
// 256 threads per row for the passes without a residual add, 512 for those
// with one: at the full width 256 threads beat 512 on the first kind
// (6.97 vs 6.28 TB/s) and 512 beat 256 on the second (6.65 vs 6.09 TB/s).
constexpr int MNR_THREADS = 256;
constexpr int MNR_THREADS_RESID = 512;

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// Block-wide max over T threads; red[] may still be read from a previous
// reduction, hence the leading barrier.
template <int T>
__device__ __forceinline__ float block_max_mnr(float v, float* red) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < T / 32) ? red[lane] : 0.f;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, m));
  return t;
}

template <int T>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] may still be read from a previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < T / 32) ? red[lane] : 0.f;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) t += __shfl_xor_sync(0xffffffffu, t, m);
  return t;
}

// seg (optional): token-group index of every row; group g reads its gate,
// shift and scale at an offset of g * seg_stride floats (a [G, 6, D] table).
// Indices outside [0, num_seg) are clamped so every read stays in the table.
// ROPE: the CTA also writes its row of the RoPE (cos, sin) table (threads
// 0-63, one pair each, while the row's loads are in flight).
// Q8: instead of the bf16 row, the row's E4M3 codes and scale, the per-row
// quantisation of quantize_fp8_rows applied to the bf16-rounded values (the
// same arithmetic, so the codes equal the unfused path's).
template <int VPT, bool ROPE, bool Q8, int T>
__global__ void __launch_bounds__(T)
    mod_norm_residual_kernel(float* __restrict__ resid, const __nv_bfloat16* __restrict__ delta,
                             const float* __restrict__ gate, const float* __restrict__ shift,
                             const float* __restrict__ scale, __nv_bfloat16* __restrict__ normed,
                             int D, float eps, const int32_t* __restrict__ seg, int num_seg,
                             int64_t seg_stride, const int32_t* __restrict__ pos,
                             float2* __restrict__ rope_out, const RopeTable tab,
                             uint8_t* __restrict__ codes, float* __restrict__ code_scale) {
  __shared__ float red[T / 32];
  const int row = blockIdx.x;
  if (seg != nullptr) {
    const int g = min(max(__ldg(seg + row), 0), num_seg - 1);
    const int64_t off = static_cast<int64_t>(g) * seg_stride;
    gate = gate ? gate + off : nullptr;
    shift = shift ? shift + off : nullptr;
    scale = scale ? scale + off : nullptr;
  }
  const int D4 = D >> 2;
  float4* rrow = reinterpret_cast<float4*>(resid + static_cast<int64_t>(row) * D);
  float4 x[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = threadIdx.x + v * T;
    x[v] = c < D4 ? rrow[c] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if constexpr (ROPE) {
    const int t = threadIdx.x;
    if (t < QK_HEAD_DIM / 2) {
      float sn, cs;
      rope_angle(__ldg(pos + 3LL * row + tab.axis[t]), tab.turn[t], sn, cs);
      rope_out[static_cast<int64_t>(row) * (QK_HEAD_DIM / 2) + t] = make_float2(cs, sn);
    }
  }
  if (delta != nullptr) {
    const uint2* drow = reinterpret_cast<const uint2*>(delta + static_cast<int64_t>(row) * D);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = threadIdx.x + v * T;
      if (c < D4) {
        const uint2 d = __ldcs(drow + c);
        const float4 g = __ldg(reinterpret_cast<const float4*>(gate) + c);
        x[v].x = fmaf(g.x, bf16_lo(d.x), x[v].x);
        x[v].y = fmaf(g.y, bf16_hi(d.x), x[v].y);
        x[v].z = fmaf(g.z, bf16_lo(d.y), x[v].z);
        x[v].w = fmaf(g.w, bf16_hi(d.y), x[v].w);
        rrow[c] = x[v];
      }
    }
  }
  if (!Q8 && normed == nullptr) return;
  float s = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) s += (x[v].x + x[v].y) + (x[v].z + x[v].w);
  const float mean = block_sum<T>(s, red) / static_cast<float>(D);
  float s2 = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = threadIdx.x + v * T;
    if (c < D4) {
      const float a = x[v].x - mean, b = x[v].y - mean, cc = x[v].z - mean, d = x[v].w - mean;
      s2 += (a * a + b * b) + (cc * cc + d * d);
    }
  }
  const float var = block_sum<T>(s2, red) / static_cast<float>(D);
  const float rstd = rsqrtf(var + eps);
  if constexpr (Q8) {
    float hv[VPT][4];
    float amax = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = threadIdx.x + v * T;
      hv[v][0] = hv[v][1] = hv[v][2] = hv[v][3] = 0.f;
      if (c < D4) {
        const float4 sc = __ldg(reinterpret_cast<const float4*>(scale) + c);
        const float4 sh = __ldg(reinterpret_cast<const float4*>(shift) + c);
        hv[v][0] = round_to_bf16(fmaf((x[v].x - mean) * rstd, 1.0f + sc.x, sh.x));
        hv[v][1] = round_to_bf16(fmaf((x[v].y - mean) * rstd, 1.0f + sc.y, sh.y));
        hv[v][2] = round_to_bf16(fmaf((x[v].z - mean) * rstd, 1.0f + sc.z, sh.z));
        hv[v][3] = round_to_bf16(fmaf((x[v].w - mean) * rstd, 1.0f + sc.w, sh.w));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(hv[v][0]), fabsf(hv[v][1])),
                                 fmaxf(fabsf(hv[v][2]), fabsf(hv[v][3]))));
      }
    }
    amax = block_max_mnr<T>(amax, red);
    const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 0.f;
    uint32_t* qrow = reinterpret_cast<uint32_t*>(codes + static_cast<int64_t>(row) * D);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = threadIdx.x + v * T;
      if (c < D4)
        qrow[c] = e4m3x4(__fmul_rn(hv[v][0], inv), __fmul_rn(hv[v][1], inv),
                         __fmul_rn(hv[v][2], inv), __fmul_rn(hv[v][3], inv));
    }
    if (threadIdx.x == 0) code_scale[row] = __fdiv_rn(amax, 448.0f);
    return;
  }
  uint2* hrow = reinterpret_cast<uint2*>(normed + static_cast<int64_t>(row) * D);
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = threadIdx.x + v * T;
    if (c < D4) {
      const float4 sc = __ldg(reinterpret_cast<const float4*>(scale) + c);
      const float4 sh = __ldg(reinterpret_cast<const float4*>(shift) + c);
      const float h0 = fmaf((x[v].x - mean) * rstd, 1.0f + sc.x, sh.x);
      const float h1 = fmaf((x[v].y - mean) * rstd, 1.0f + sc.y, sh.y);
      const float h2 = fmaf((x[v].z - mean) * rstd, 1.0f + sc.z, sh.z);
      const float h3v = fmaf((x[v].w - mean) * rstd, 1.0f + sc.w, sh.w);
      __stcs(hrow + c, make_uint2(pack_bf16x2(h0, h1), pack_bf16x2(h2, h3v)));
    }
  }
}

// --------------------------------------------------- GPU output preparation
// vLLM-Omni H3 blog, section 3.4: decoded FP32 BCTHW frames become contiguous
// uint8 BTHWC before they leave the GPU. Value map: round-half-even of
// clamp(x / 2 + 1/2, 0, 1) * 255, each step rounded in FP32 (no FMA).
// Each thread converts 4 consecutive pixels: one 16-byte load per channel
// plane, 4*C contiguous output bytes written as 32-bit words.
constexpr int U8_THREADS = 256;
constexpr int U8_MAX_C = 16;

__device__ __forceinline__ uint32_t frame_code(float x) {
  float t = __fadd_rn(__fmul_rn(x, 0.5f), 0.5f);
  t = fminf(fmaxf(t, 0.0f), 1.0f);
  return __float2uint_rn(__fmul_rn(t, 255.0f));
}

// CC > 0: channel count fixed at compile time (packing stays in registers);
// CC == 0: any C <= U8_MAX_C given at run time.
template <int CC>
__global__ void __launch_bounds__(U8_THREADS)
    frames_to_u8_kernel(const float* __restrict__ in, uint8_t* __restrict__ out, int C_rt,
                        int64_t N4 /* pixels per batch entry / 4 */, int64_t total4) {
  const int C = CC > 0 ? CC : C_rt;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(U8_THREADS) + threadIdx.x; i < total4;
       i += static_cast<int64_t>(gridDim.x) * U8_THREADS) {
    const int64_t b = i / N4;
    const int64_t p4 = i - b * N4;
    const float4* src = reinterpret_cast<const float4*>(in) + b * C * N4 + p4;
    uint32_t bytes[CC > 0 ? CC : U8_MAX_C];  // 4 pixels x C channels, little-endian
#pragma unroll
    for (int w = 0; w < (CC > 0 ? CC : U8_MAX_C); ++w) bytes[w] = 0;
#pragma unroll
    for (int c = 0; c < (CC > 0 ? CC : U8_MAX_C); ++c) {
      if (c >= C) break;
      const float4 v = __ldcs(src + static_cast<int64_t>(c) * N4);
      const float px[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int byte = k * C + c;  // pixel k, channel c
        bytes[byte >> 2] |= frame_code(px[k]) << (8 * (byte & 3));
      }
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + (b * N4 + p4) * 4 * C);
#pragma unroll
    for (int w = 0; w < (CC > 0 ? CC : U8_MAX_C); ++w)
      if (w < C) dst[w] = bytes[w];
  }
}

// ---------------------------------------------- FP8 per-row quantisation
// vLLM-Omni H3 blog, section 4.3 (online FP8: weights quantised at load
// time, activations online). One CTA per row: amax over the row, inv = 448 /
// amax, code = E4M3(x * inv) with saturation, scale = amax / 448; every step
// rounded in FP32 (IEEE division and multiply).
constexpr int Q8_THREADS = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < Q8_THREADS / 32) ? red[lane] : 0.f;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, m));
  return t;
}

template <int VPT>  // 8-element chunks per thread
__global__ void __launch_bounds__(Q8_THREADS)
    quantize_fp8_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx,
                             uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scale,
                             int K) {
  __shared__ float red[Q8_THREADS / 32];
  const int row = blockIdx.x;
  const int K8 = K >> 3;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(row) * ldx);
  uint4 v[VPT];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * Q8_THREADS;
    v[i] = c < K8 ? __ldcs(src + c) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
  amax = block_max(amax, red);
  const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(q + static_cast<int64_t>(row) * ldq);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * Q8_THREADS;
    if (c < K8) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      float f[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[2 * j] = __fmul_rn(bf16_lo(w[j]), inv);
        f[2 * j + 1] = __fmul_rn(bf16_hi(w[j]), inv);
      }
      dst[c] = make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
    }
  }
  if (threadIdx.x == 0) scale[row] = __fdiv_rn(amax, 448.0f);
}

}  // namespace

h3_status launch_quantize_fp8_rows(const void* x, int64_t ldx, void* q, int64_t ldq, float* scale,
                                   int R, int K, cudaStream_t s) {
  const int vpt = (K / 8 + Q8_THREADS - 1) / Q8_THREADS;
  const auto* xx = static_cast<const __nv_bfloat16*>(x);
  auto* qq = static_cast<uint8_t*>(q);
#define H3_Q8_CASE(V)                                                                   \
  case V:                                                                               \
    quantize_fp8_rows_kernel<V><<<R, Q8_THREADS, 0, s>>>(xx, ldx, qq, ldq, scale, K); \
    break;
  switch (vpt) {
    H3_Q8_CASE(1)
    H3_Q8_CASE(2)
    H3_Q8_CASE(3)
    H3_Q8_CASE(4)
    H3_Q8_CASE(5)
    H3_Q8_CASE(6)
    H3_Q8_CASE(7)
    H3_Q8_CASE(8)
    default:
      return fail(H3_ERR_UNSUPPORTED, "quantize_fp8_rows: K=%d exceeds 16384", K);
  }
#undef H3_Q8_CASE
  return cuda_fail(cudaGetLastError(), "quantize_fp8_rows launch");
}

h3_status launch_frames_to_u8(const float* in, uint8_t* out, int B, int C, int64_t N,
                              cudaStream_t s) {
  const int64_t N4 = N / 4;
  const int64_t total4 = static_cast<int64_t>(B) * N4;
  const int64_t want = (total4 + U8_THREADS - 1) / U8_THREADS;
  const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(num_sms()) * 8));
  if (C == 3)
    frames_to_u8_kernel<3><<<grid, U8_THREADS, 0, s>>>(in, out, C, N4, total4);
  else
    frames_to_u8_kernel<0><<<grid, U8_THREADS, 0, s>>>(in, out, C, N4, total4);
  return cuda_fail(cudaGetLastError(), "frames_to_u8 launch");
}

h3_status launch_swiglu(const void* gate_up, void* out, int L, int F, cudaStream_t s) {
  const int F8 = F / 8;
  const int grid = std::min(L, num_sms() * 8);
  swiglu_kernel<<<grid, SWIGLU_THREADS, 0, s>>>(static_cast<const uint4*>(gate_up),
                                                static_cast<uint4*>(out), L, F8);
  return cuda_fail(cudaGetLastError(), "swiglu launch");
}

constexpr double kTwoPi = 6.283185307179586476925286766559;

static RopeTable rope_table(const int* axis_dims, float theta) {
  RopeTable tab{};
  int pr = 0;
  int o = 0;  // first channel of section a
  for (int a = 0; a < 3; ++a) {
    const int d = axis_dims[a];
    for (int j = 0; j < d / 2; ++j, ++pr) {
      const double omega =
          std::pow(static_cast<double>(theta), -2.0 * j / static_cast<double>(d));
      // omega / (2 pi) < 1: scaled by 2^64 it is an integer below 2^63 with
      // at most 53 significant bits, which the conversion keeps exactly
      tab.turn[pr] = static_cast<uint64_t>(std::ldexp(omega / kTwoPi, 64));
      tab.axis[pr] = a;
    }
    // split-half slices (meaningful when d % 16 == 0): slice s of the first
    // half pairs with slice s + d/16 of the second half
    for (int c = 0; c + 8 <= d; c += 8) {
      const int s = (o + c) / 8;
      const bool fst = c < d / 2;
      tab.half_first[s] = fst ? 1 : 0;
      tab.half_src[s] = fst ? s + d / 16 : s - d / 16;
      tab.half_pair0[s] = o / 2 + (fst ? c : c - d / 2);
    }
    o += d;
  }
  return tab;
}

h3_status launch_rope_table(const int32_t* pos, const int* axis_dims, int L, float theta,
                            float2* out, cudaStream_t s) {
  const RopeTable tab = rope_table(axis_dims, theta);
  const int64_t n = static_cast<int64_t>(L) * (QK_HEAD_DIM / 2);
  const int grid = static_cast<int>((n + 255) / 256);
  rope_table_kernel<<<grid, 256, 0, s>>>(pos, L, tab, out);
  return cuda_fail(cudaGetLastError(), "rope_table launch");
}

h3_status launch_qk_norm_rope(void* q, void* k, int64_t row_stride, const float* q_gain,
                              const float* k_gain, const int32_t* pos, const int* axis_dims,
                              int L, int H, float theta, float eps, cudaStream_t s,
                              int pairing) {
  const RopeTable tab = rope_table(axis_dims, theta);
  const int64_t warps = 2LL * L;
  const int grid = static_cast<int>((warps + QK_WARPS - 1) / QK_WARPS);
  auto* qq = static_cast<__nv_bfloat16*>(q);
  auto* kk = static_cast<__nv_bfloat16*>(k);
  if (pairing == 1)
    qk_norm_rope_kernel<true><<<grid, QK_WARPS * 32, 0, s>>>(qq, kk, row_stride, q_gain, k_gain,
                                                             pos, L, H, eps, tab);
  else
    qk_norm_rope_kernel<false><<<grid, QK_WARPS * 32, 0, s>>>(qq, kk, row_stride, q_gain, k_gain,
                                                              pos, L, H, eps, tab);
  return cuda_fail(cudaGetLastError(), "qk_norm_rope launch");
}

template <int T, int V>
static void mnr_launch(bool rope, bool q8, int L, cudaStream_t s, float* resid,
                       const __nv_bfloat16* d, const float* gate, const float* shift,
                       const float* scale, __nv_bfloat16* n, int D, float eps, const int32_t* seg,
                       int num_seg, int64_t seg_stride, const int32_t* pos, float2* out,
                       const RopeTable& tab, uint8_t* codes, float* code_scale) {
#define H3_MNR_ARGS resid, d, gate, shift, scale, n, D, eps, seg, num_seg, seg_stride, pos, out, \
                    tab, codes, code_scale
  if (q8) {
    if (rope)
      mod_norm_residual_kernel<V, true, true, T><<<L, T, 0, s>>>(H3_MNR_ARGS);
    else
      mod_norm_residual_kernel<V, false, true, T><<<L, T, 0, s>>>(H3_MNR_ARGS);
  } else {
    if (rope)
      mod_norm_residual_kernel<V, true, false, T><<<L, T, 0, s>>>(H3_MNR_ARGS);
    else
      mod_norm_residual_kernel<V, false, false, T><<<L, T, 0, s>>>(H3_MNR_ARGS);
  }
#undef H3_MNR_ARGS
}

h3_status launch_mod_norm_residual(float* resid, const void* delta, const float* gate,
                                   const float* shift, const float* scale, void* normed, int L,
                                   int D, float eps, cudaStream_t s, const int32_t* seg,
                                   int num_seg, int64_t seg_stride, const RopeRequest* rope,
                                   uint8_t* codes, float* code_scale) {
  const auto* d = static_cast<const __nv_bfloat16*>(delta);
  auto* n = static_cast<__nv_bfloat16*>(normed);
  RopeTable tab{};
  if (rope != nullptr) tab = rope_table(rope->axis_dims, rope->theta);
  const int32_t* pos = rope ? rope->pos : nullptr;
  float2* out = rope ? rope->out : nullptr;
  const bool r = rope != nullptr, q = codes != nullptr;
  const bool wide = delta != nullptr && rope == nullptr;
  const int T = wide ? MNR_THREADS_RESID : MNR_THREADS;
  const int vpt = (D / 4 + T - 1) / T;
#define H3_MNR(TT, V)                                                                       \
  mnr_launch<TT, V>(r, q, L, s, resid, d, gate, shift, scale, n, D, eps, seg, num_seg,      \
                    seg_stride, pos, out, tab, codes, code_scale)
  if (wide) {
    switch (vpt) {
      case 1: H3_MNR(MNR_THREADS_RESID, 1); break;
      case 2: H3_MNR(MNR_THREADS_RESID, 2); break;
      case 3: H3_MNR(MNR_THREADS_RESID, 3); break;
      case 4: H3_MNR(MNR_THREADS_RESID, 4); break;
      default:
        return fail(H3_ERR_UNSUPPORTED, "mod_norm_residual: D=%d exceeds 8192", D);
    }
  } else {
    switch (vpt) {
      case 1: H3_MNR(MNR_THREADS, 1); break;
      case 2: H3_MNR(MNR_THREADS, 2); break;
      case 3: H3_MNR(MNR_THREADS, 3); break;
      case 4: H3_MNR(MNR_THREADS, 4); break;
      case 5: H3_MNR(MNR_THREADS, 5); break;
      case 6: H3_MNR(MNR_THREADS, 6); break;
      case 7: H3_MNR(MNR_THREADS, 7); break;
      case 8: H3_MNR(MNR_THREADS, 8); break;
      default:
        return fail(H3_ERR_UNSUPPORTED, "mod_norm_residual: D=%d exceeds 8192", D);
    }
  }
#undef H3_MNR
  return cuda_fail(cudaGetLastError(), "mod_norm_residual launch");
}

}  // namespace h3
