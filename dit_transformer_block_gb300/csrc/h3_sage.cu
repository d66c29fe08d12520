// FP8 operands for SAGE-style attention (vLLM-Omni H3 blog, section 4.3: Q, K,
// P and V quantised to FP8 for the QK and PV products).
//
//   1. kv_stats_partial / kv_stats_final: per (head, channel) mean of K and
//      absmax of V over the L valid rows. The K sum is exact: each 512-row
//      chunk is summed in 64-bit fixed point (units of 2^-40; exact for
//      nonzero |k| in [2^-33, 2^14), which bf16 keys of unit-RMS heads always
//      are), a chunk holding a value outside that range is summed in FP64
//      instead, and the chunks are combined in 128-bit integers. The exact sum
//      is rounded once to double, divided by L in FP64 and rounded once to
//      float32: the exact mean rounded once, whatever the order of the rows;
//   2. qk_tile_quant: Q, and K minus its mean, to E4M3 per (128-row tile,
//      head) block with absmax scaling;
//   3. v_quant: V to E4M3 per (head, channel) with the V absmax.
// Scaling: inv = 448 / amax (0 when amax == 0), code = E4M3_satfinite(x * inv),
// scale = amax / 448, every step rounded in FP32. Codes keep the [S, H, 128]
// row layout of the inputs (one byte per element); rows >= L are not written.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "h3_internal.cuh"

namespace h3 {
namespace {

constexpr int DH = 128;
constexpr int ST_ROWS = 512;  // rows per statistics chunk

// bf16 bits -> the value in units of 2^-40 when its exponent field lies in
// [94, 140] (magnitude in [2^-33, 2^14)), as a two's-complement integer of at
// most 55 bits; `in_range` tells whether it did (zero counts as in range).
__device__ __forceinline__ int64_t bf16_fixed40(uint32_t bits, bool& in_range) {
  const uint32_t e = (bits >> 7) & 0xFFu;
  const uint32_t mag_bits = bits & 0x7FFFu;
  in_range = mag_bits == 0u || (e >= 94u && e <= 140u);
  const uint32_t sh = e >= 94u ? min(e - 94u, 46u) : 0u;
  const int64_t mag = e >= 94u ? static_cast<int64_t>((128u | (bits & 0x7Fu))) << sh : 0;
  return (bits & 0x8000u) ? -mag : mag;
}

// grid (chunks, H), 128 threads. Thread t reads channels 8 (t % 16) ..
// 8 (t % 16) + 7 of head blockIdx.y with 16-byte loads, on every eighth row of
// the chunk starting at row t / 16; the eight row lanes of a channel are then
// added exactly in shared memory and thread d writes channel d.
// psum_i: the chunk's K sum in units of 2^-40 (at most 512 terms below 2^54,
// so no overflow); psum_d: 0, or the chunk's K sum in FP64 when one of its
// values lies outside the fixed-point range (psum_i is then 0).
__global__ void __launch_bounds__(DH)
    kv_stats_partial_kernel(const __nv_bfloat16* __restrict__ k,
                            const __nv_bfloat16* __restrict__ v, int64_t ld, int L,
                            int64_t* __restrict__ psum_i, double* __restrict__ psum_d,
                            float* __restrict__ pmax) {
  __shared__ long long s_acc[8][DH];
  __shared__ uint32_t s_vmax[8][DH];
  __shared__ uint32_t s_in[8][DH];
  const int chunk = blockIdx.x, h = blockIdx.y, H = gridDim.y;
  const int cg = threadIdx.x & 15, rl = threadIdx.x >> 4;
  const int r0 = chunk * ST_ROWS, r1 = min(L, r0 + ST_ROWS);
  const int64_t col = static_cast<int64_t>(h) * DH + cg * 8;
  int64_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  uint32_t vmax[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // |v| as bf16 bits (ordered as magnitudes)
  uint32_t in = 0xFFu;                          // bit c: channel c stayed in range
  int r = r0 + rl;
  auto take = [&](uint4 kr, uint4 vr) {
    const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
    const uint32_t vw[4] = {vr.x, vr.y, vr.z, vr.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t kb = (c & 1) ? (kw[c >> 1] >> 16) : (kw[c >> 1] & 0xFFFFu);
      const uint32_t vb = (c & 1) ? (vw[c >> 1] >> 16) : (vw[c >> 1] & 0xFFFFu);
      bool ok;
      acc[c] += bf16_fixed40(kb, ok);
      in &= ok ? 0xFFu : ~(1u << c);
      vmax[c] = max(vmax[c], vb & 0x7FFFu);
    }
  };
  // two rows per iteration, all four loads first
  for (; r + 8 < r1; r += 16) {
    const int64_t o0 = static_cast<int64_t>(r) * ld + col, o1 = o0 + 8 * ld;
    const uint4 k0 = __ldg(reinterpret_cast<const uint4*>(k + o0));
    const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(v + o0));
    const uint4 k1 = __ldg(reinterpret_cast<const uint4*>(k + o1));
    const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(v + o1));
    take(k0, v0);
    take(k1, v1);
  }
  if (r < r1) {
    const int64_t o0 = static_cast<int64_t>(r) * ld + col;
    take(__ldg(reinterpret_cast<const uint4*>(k + o0)), __ldg(reinterpret_cast<const uint4*>(v + o0)));
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    s_acc[rl][cg * 8 + c] = acc[c];
    s_vmax[rl][cg * 8 + c] = vmax[c];
    s_in[rl][cg * 8 + c] = (in >> c) & 1u;
  }
  __syncthreads();
  const int d = threadIdx.x;
  int64_t sum = 0;
  uint32_t vm = 0, all_in = 1;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    sum += s_acc[i][d];
    vm = max(vm, s_vmax[i][d]);
    all_in &= s_in[i][d];
  }
  double dsum = 0.0;
  if (!all_in) {  // rare: a value too small or too large for the fixed point
    sum = 0;
    for (int rr = r0; rr < r1; ++rr)
      dsum = __dadd_rn(dsum, static_cast<double>(__bfloat162float(
                                 k[static_cast<int64_t>(rr) * ld + static_cast<int64_t>(h) * DH + d])));
  }
  const int64_t o = (static_cast<int64_t>(chunk) * H + h) * DH + d;
  psum_i[o] = sum;
  psum_d[o] = dsum;
  pmax[o] = __uint_as_float(vm << 16);
}

// grid H, 128 threads: combine the chunks, mean = sum / L in FP64, rounded
// once to float32.
__global__ void __launch_bounds__(DH)
    kv_stats_final_kernel(const int64_t* __restrict__ psum_i, const double* __restrict__ psum_d,
                          const float* __restrict__ pmax, int chunks, int L,
                          float* __restrict__ k_mean, float* __restrict__ sv,
                          float* __restrict__ inv_v) {
  const int h = blockIdx.x, d = threadIdx.x, H = gridDim.x;
  __int128 si = 0;
  double sd = 0.0;
  float mx = 0.f;
  for (int ch = 0; ch < chunks; ++ch) {
    const int64_t o = (static_cast<int64_t>(ch) * H + h) * DH + d;
    si += psum_i[o];
    sd = __dadd_rn(sd, psum_d[o]);
    mx = fmaxf(mx, pmax[o]);
  }
  // the integer sum rounded once to double (exact below 2^53 units): split
  // into a high part that is a multiple of 2^32 and a low part, both exact in
  // double when |si| < 2^85, then one rounding in their sum
  const int64_t hi = static_cast<int64_t>(si >> 32);
  const double whole =
      __dadd_rn(static_cast<double>(hi) * 4294967296.0,
                static_cast<double>(static_cast<uint32_t>(si & 0xFFFFFFFFu)));
  const double sum = __dadd_rn(whole * 0x1p-40, sd);
  const int i = h * DH + d;
  k_mean[i] = __double2float_rn(__ddiv_rn(sum, static_cast<double>(L)));
  sv[i] = __fdiv_rn(mx, 448.0f);
  inv_v[i] = mx > 0.f ? __fdiv_rn(448.0f, mx) : 0.f;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

constexpr int QT_THREADS = 256;  // 16 rows x 16 chunks of 8 channels per pass, 8 passes

// grid (tiles, H, 2): z = 0 quantises Q, z = 1 quantises K - mean.
__global__ void __launch_bounds__(QT_THREADS)
    qk_tile_quant_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                         int64_t ld, const float* __restrict__ k_mean, int L,
                         uint8_t* __restrict__ qc, uint8_t* __restrict__ kc, int64_t ldc,
                         float* __restrict__ sq, float* __restrict__ sk) {
  __shared__ float red[QT_THREADS / 32];
  const int tile = blockIdx.x, h = blockIdx.y, which = blockIdx.z, H = gridDim.y;
  const __nv_bfloat16* src = which ? k : q;
  uint8_t* dst = which ? kc : qc;
  const int chunk = threadIdx.x & 15;   // channels 8*chunk .. 8*chunk+7
  const int rsub = threadIdx.x >> 4;    // row within a 16-row pass
  float mean[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mean[j] = which ? k_mean[h * DH + chunk * 8 + j] : 0.f;
  float x[8][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = tile * 128 + i * 16 + rsub;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (row < L)
      raw = *reinterpret_cast<const uint4*>(src + static_cast<int64_t>(row) * ld + h * DH +
                                            chunk * 8);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[i][2 * j] = row < L ? __fsub_rn(bf16_lo(w[j]), mean[2 * j]) : 0.f;
      x[i][2 * j + 1] = row < L ? __fsub_rn(bf16_hi(w[j]), mean[2 * j + 1]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[i][j]));
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < QT_THREADS / 32; ++w) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.f ? __fdiv_rn(448.0f, amax) : 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = tile * 128 + i * 16 + rsub;
    if (row < L) {
      float f[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(x[i][j], inv);
      *reinterpret_cast<uint2*>(dst + static_cast<int64_t>(row) * ldc + h * DH + chunk * 8) =
          make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
    }
  }
  if (threadIdx.x == 0) (which ? sk : sq)[tile * H + h] = __fdiv_rn(amax, 448.0f);
}

// One thread per 8 channels of one row.
__global__ void __launch_bounds__(256)
    v_quant_kernel(const __nv_bfloat16* __restrict__ v, int64_t ld, const float* __restrict__ inv_v,
                   int L, int H, uint8_t* __restrict__ vc, int64_t ldc) {
  const int64_t per_row = static_cast<int64_t>(H) * (DH / 8);
  const int64_t total = static_cast<int64_t>(L) * per_row;
  for (int64_t i = blockIdx.x * 256LL + threadIdx.x; i < total; i += gridDim.x * 256LL) {
    const int64_t row = i / per_row;
    const int64_t cc = i - row * per_row;  // chunk of 8 channels across heads
    const uint4 raw = *reinterpret_cast<const uint4*>(v + row * ld + cc * 8);
    const float4 i0 = *reinterpret_cast<const float4*>(inv_v + cc * 8);
    const float4 i1 = *reinterpret_cast<const float4*>(inv_v + cc * 8 + 4);
    const float inv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __fmul_rn(bf16_lo(w[j]), inv[2 * j]);
      f[2 * j + 1] = __fmul_rn(bf16_hi(w[j]), inv[2 * j + 1]);
    }
    *reinterpret_cast<uint2*>(vc + row * ldc + cc * 8) =
        make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
  }
}

}  // namespace

size_t sage_scratch_bytes(int L, int H) {
  const size_t chunks = (static_cast<size_t>(L) + ST_ROWS - 1) / ST_ROWS;
  return chunks * H * DH * (sizeof(int64_t) + sizeof(double) + sizeof(float)) +
         static_cast<size_t>(H) * DH * sizeof(float);
}

h3_status launch_sage_quantize(const void* q, const void* k, const void* v, int64_t ld, int L,
                               int H, uint8_t* qc, uint8_t* kc, uint8_t* vc, int64_t ldc,
                               float* sq, float* sk, float* sv, float* k_mean, void* scratch,
                               cudaStream_t s) {
  const int chunks = (L + ST_ROWS - 1) / ST_ROWS;
  const size_t n = static_cast<size_t>(chunks) * H * DH;
  int64_t* psum_i = static_cast<int64_t*>(scratch);
  double* psum_d = reinterpret_cast<double*>(psum_i + n);
  float* pmax = reinterpret_cast<float*>(psum_d + n);
  float* inv_v = pmax + n;
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  const auto* kk = static_cast<const __nv_bfloat16*>(k);
  const auto* vv = static_cast<const __nv_bfloat16*>(v);
  kv_stats_partial_kernel<<<dim3(chunks, H), DH, 0, s>>>(kk, vv, ld, L, psum_i, psum_d, pmax);
  kv_stats_final_kernel<<<H, DH, 0, s>>>(psum_i, psum_d, pmax, chunks, L, k_mean, sv, inv_v);
  const int tiles = (L + 127) / 128;
  qk_tile_quant_kernel<<<dim3(tiles, H, 2), QT_THREADS, 0, s>>>(qq, kk, ld, k_mean, L, qc, kc, ldc,
                                                               sq, sk);
  const int64_t work = static_cast<int64_t>(L) * H * (DH / 8);
  const int grid = static_cast<int>(std::min<int64_t>((work + 255) / 256, num_sms() * 8LL));
  v_quant_kernel<<<grid, 256, 0, s>>>(vv, ld, inv_v, L, H, vc, ldc);
  return cuda_fail(cudaGetLastError(), "sage quantize launch");
}

}  // namespace h3
