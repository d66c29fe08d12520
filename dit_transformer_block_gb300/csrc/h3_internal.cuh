// Host-side declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/h3block.h"
#include "h3_ptx.cuh"

namespace h3 {

// ---- error state (h3_abi.cu)
h3_status fail(h3_status s, const char* fmt, ...);
h3_status cuda_fail(cudaError_t e, const char* what);
void clear_error();
// Device error word and wait limit for kernels launched on the current device.
h3_status dev_err(DevErr* out);
int num_sms();

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device (done[] holds the devices already set; ordinals
// past its end are set on every call). Safe to call from several threads:
// the attribute call is idempotent and the flags are atomic.
template <typename Kernel>
h3_status set_smem_limit(std::atomic<bool> (&done)[64], Kernel kernel, size_t bytes,
                         const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, what);
  if (dev < 64 && done[dev].load(std::memory_order_acquire)) return H3_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e != cudaSuccess) return cuda_fail(e, what);
  if (dev < 64) done[dev].store(true, std::memory_order_release);
  return H3_OK;
}

// ---- TMA descriptors (h3_abi.cu). A 2D bf16 tensor of `outer` rows x `inner`
// elements with the given row stride, boxes of box_inner x box_outer, 128-byte
// swizzle, zero fill outside the tensor.
h3_status make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
// Same for a tensor of bytes (FP8 codes).
h3_status make_tmap_u8_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// ---- kernel launchers (arguments already validated)
h3_status launch_swiglu(const void* gate_up, void* out, int L, int F, cudaStream_t s);
// pairing: 0 interleaved pairs (2j, 2j + 1), 1 split-half pairs
// (o + j, o + d/2 + j) per section (every section a multiple of 16 wide).
h3_status launch_qk_norm_rope(void* q, void* k, int64_t row_stride, const float* q_gain,
                              const float* k_gain, const int32_t* pos, const int* axis_dims,
                              int L, int H, float theta, float eps, cudaStream_t s,
                              int pairing = 0);
// The RoPE (cos, sin) table of rows [0, L) (see launch_rope_table), written
// by the modulation kernel beside its own work when requested.
struct RopeRequest {
  const int32_t* pos;    // [L, 3] positions
  const int* axis_dims;  // host [3]
  float theta;
  float2* out;           // [L, 64]
};
// seg (optional): per-row token-group index into a table whose groups are
// seg_stride floats apart (gate/shift/scale point at group 0).
// codes (optional): write the normalised row as per-row E4M3 codes [L, D]
// and scales code_scale [L] (launch_quantize_fp8_rows of the bf16 row)
// instead of the bf16 row `normed`.
h3_status launch_mod_norm_residual(float* resid, const void* delta, const float* gate,
                                   const float* shift, const float* scale, void* normed, int L,
                                   int D, float eps, cudaStream_t s, const int32_t* seg = nullptr,
                                   int num_seg = 1, int64_t seg_stride = 0,
                                   const RopeRequest* rope = nullptr, uint8_t* codes = nullptr,
                                   float* code_scale = nullptr);

// (cos, sin) of every RoPE angle of rows [0, L): out[i * 64 + p] for channel
// pair p of a 128-channel head, the angle formed and reduced exactly as
// launch_qk_norm_rope does.
h3_status launch_rope_table(const int32_t* pos, const int* axis_dims, int L, float theta,
                            float2* out, cudaStream_t s);

// frames [B, C, N] float32 (N = T*H*W, N % 4 == 0) -> [B, N, C] uint8.
h3_status launch_frames_to_u8(const float* in, uint8_t* out, int B, int C, int64_t N,
                              cudaStream_t s);

enum GemmEpilogue : int {
  GEMM_STORE_BF16 = 0,     // C = bf16(acc)
  GEMM_SWIGLU = 1,         // B rows [gate | up] of F each; C[:, j] = SiLU(g) * u, width F
  GEMM_RESIDUAL = 2,       // C is the FP32 residual: C[:, j] += gate[j] * bf16(acc)
  GEMM_QK_NORM_ROPE = 3,   // C = bf16(acc), then RMSNorm + RoPE on the q and k heads
};
// Operands of the fused epilogues (unused fields may stay zero).
struct GemmExtra {
  // GEMM_RESIDUAL: per-column gate [N]; with seg, row i reads the gate at
  // gate + clamp(seg[i], 0, num_seg - 1) * seg_stride.
  const float* gate = nullptr;
  const int32_t* seg = nullptr;
  int num_seg = 1;
  int64_t seg_stride = 0;
  // GEMM_QK_NORM_ROPE: columns [0, d_model) are q heads, [d_model, 2 d_model)
  // k heads (128 channels each), the rest pass through; every head of a row is
  // rounded to bf16, scaled by 1/rms and its gain, rotated by the row's
  // (cos, sin) table [L, 64] (h3::launch_rope_table) and rounded again.
  const float* q_gain = nullptr;
  const float* k_gain = nullptr;
  const float2* rope = nullptr;
  int d_model = 0;
  float eps = 0.f;
  // split-half RoPE pairs (pairing 1): eight pieces of eight pairs, piece i
  // rotating columns piece_first[i] + j with piece_second[i] + j by table
  // entry piece_pair[i] + j (set by rope_pieces)
  int pairing = 0;
  int piece_first[8] = {};
  int piece_second[8] = {};
  int piece_pair[8] = {};
};
// Fills ex's split-half pieces for the RoPE sections axis_dims (each a
// multiple of 16, summing to 128) and sets ex->pairing = 1.
void rope_pieces(const int* axis_dims, GemmExtra* ex);
// C[:L, :] = epilogue(A[:L, :K] @ B^T). A row stride lda, B [N, K] row stride
// ldb, C row stride ldc (elements of C). For GEMM_SWIGLU, N is the width of C
// (= F) and B holds 2N rows.
h3_status launch_gemm(const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                      int64_t ldc, int L, int N, int K, GemmEpilogue ep, cudaStream_t s,
                      const GemmExtra* extra = nullptr);

// FP8 (E4M3) operands with per-row scales: C[:L] = epilogue(bf16-free
// (A @ B^T) * sa[row] * sb[col]). A [L, K] codes (row stride lda bytes), B
// [N or 2N, K] codes (row stride ldb bytes), sa [L], sb [N or 2N].
h3_status launch_gemm_fp8(const void* A, int64_t lda, const float* sa, const void* B, int64_t ldb,
                          const float* sb, void* C, int64_t ldc, int L, int N, int K,
                          GemmEpilogue ep, cudaStream_t s, const GemmExtra* extra = nullptr);
// Per-row absmax quantisation of bf16 x [R, K] (row stride ldx elements) to
// E4M3 codes q [R, K] (row stride ldq bytes) and float32 scales [R].
h3_status launch_quantize_fp8_rows(const void* x, int64_t ldx, void* q, int64_t ldq, float* scale,
                                   int R, int K, cudaStream_t s);

// o[:L] = attention(q, k, v); q/k/v rows of stride ld_in elements, o of ld_out.
// skip_eps < 0: dense attention (the CTA-pair kernel). skip_eps >= 0:
// Skip-Softmax (the pair kernel's instance with its vote), a key tile is left out for
// a query tile when every valid row's tile maximum is below eps times the
// row's exact running maximum over the kept tiles (eps = 0 never skips); kept
// (optional, [ceil(L/128), H]) receives the number of key tiles kept per
// (query tile, head).
h3_status launch_attention(const void* q, const void* k, const void* v, int64_t ld_in,
                           void* o, int64_t ld_out, int L, int H, float scale, cudaStream_t s,
                           float skip_eps = -1.f, int* kept = nullptr);

// SAGE-style FP8 attention: operands (h3_sage.cu) and the FP8 attention
// kernel (h3_attention.cu). Codes [L, H*128] bytes with row stride ldc; sq,
// sk [ceil(L/128), H]; sv, k_mean [H, 128]; scratch of sage_scratch_bytes.
size_t sage_scratch_bytes(int L, int H);
h3_status launch_sage_quantize(const void* q, const void* k, const void* v, int64_t ld, int L,
                               int H, uint8_t* qc, uint8_t* kc, uint8_t* vc, int64_t ldc,
                               float* sq, float* sk, float* sv, float* k_mean, void* scratch,
                               cudaStream_t s);
// skip_eps >= 0: Skip-Softmax on the FP8 logits (kept tile counts to `kept`
// [ceil(L/128), H] when not null), as in launch_attention.
h3_status launch_attention_fp8(const void* qc, const void* kc, const void* vc, int64_t ld_codes,
                               const float* sq, const float* sk, const float* sv, void* o,
                               int64_t ld_out, int L, int H, float scale, cudaStream_t s,
                               float skip_eps = -1.f, int* kept = nullptr);

}  // namespace h3
