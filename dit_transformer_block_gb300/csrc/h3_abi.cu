// C-ABI boundary of libh3block: argument validation, error reporting, TMA
// descriptor creation, and the block forward composed from the kernels.
// Every entry point validates on the host and launches nothing on error.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "h3_internal.cuh"

namespace h3 {

namespace {
thread_local char g_msg[512] = "";
uint64_t g_timeout_ns = 2000000000ull;
constexpr int kMaxDevices = 64;

// Device error word: first nonzero code recorded by a bounded wait.
__device__ uint32_t g_dev_error_word;

struct DeviceState {
  bool ready = false;
  uint32_t* err_word = nullptr;
  int sms = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

h3_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev >= kMaxDevices) return fail(H3_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dev_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    d.err_word = static_cast<uint32_t*>(p);
    d.sms = sms;
    d.ready = true;
  }
  *out = &d;
  return H3_OK;
}

__global__ void wait_timeout_kernel(DevErr err) {
  __shared__ uint64_t b;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&b), 1);
    fence_mbar_init();
    // nothing ever arrives: the wait must run out and record its code
    mbar_wait(smem_u32(&b), 0, err, ERR_WAIT_PROBE);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

const char* err_code_name(uint32_t c) {
  switch (c) {
    case ERR_WAIT_GEMM_PRODUCER: return "gemm TMA producer";
    case ERR_WAIT_GEMM_MMA: return "gemm MMA issuer";
    case ERR_WAIT_GEMM_EPILOGUE: return "gemm epilogue";
    case ERR_WAIT_ATTN_PRODUCER: return "attention TMA producer";
    case ERR_WAIT_ATTN_MMA: return "attention MMA issuer";
    case ERR_WAIT_ATTN_SOFTMAX: return "attention softmax";
    case ERR_WAIT_PROBE: return "wait-timeout probe";
    default: return "unknown";
  }
}
}  // namespace

h3_status fail(h3_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

h3_status cuda_fail(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return H3_OK;
  return fail(H3_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

void clear_error() { g_msg[0] = '\0'; }

h3_status dev_err(DevErr* out) {
  DeviceState* d = nullptr;
  h3_status st = device_state(&d);
  if (st != H3_OK) return st;
  out->word = d->err_word;
  out->timeout_ns = g_timeout_ns;
  return H3_OK;
}

int num_sms() {
  DeviceState* d = nullptr;
  if (device_state(&d) != H3_OK) return 1;
  return d->sms;
}

static h3_status make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base,
                              uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                              uint32_t box_inner, uint32_t box_outer);

h3_status make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_stride_bytes,
                      box_inner, box_outer);
}

h3_status make_tmap_u8_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, inner, outer, row_stride_bytes,
                      box_inner, box_outer);
}

static h3_status make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base,
                              uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                              uint32_t box_inner, uint32_t box_outer) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (g_encode == nullptr)
    return fail(H3_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(H3_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llux%llu stride %llu",
                static_cast<int>(r), static_cast<unsigned long long>(inner),
                static_cast<unsigned long long>(outer),
                static_cast<unsigned long long>(row_stride_bytes));
  return H3_OK;
}

}  // namespace h3

using namespace h3;

#define H3_REQUIRE(cond, code, ...) \
  do {                              \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

static h3_status check_rows(int S, int L) {
  H3_REQUIRE(S >= 0 && L >= 0, H3_ERR_INVALID_ARG, "negative size (S=%d, L=%d)", S, L);
  H3_REQUIRE(L <= S, H3_ERR_INVALID_ARG, "L=%d exceeds the buffer rows S=%d", L, S);
  return H3_OK;
}

extern "C" {

int h3_version(void) { return (1 << 16) | 0; }

const char* h3_last_error(void) { return g_msg; }

const char* h3_status_string(h3_status s) {
  switch (s) {
    case H3_OK: return "H3_OK";
    case H3_ERR_INVALID_ARG: return "H3_ERR_INVALID_ARG";
    case H3_ERR_UNSUPPORTED: return "H3_ERR_UNSUPPORTED";
    case H3_ERR_MISALIGNED: return "H3_ERR_MISALIGNED";
    case H3_ERR_WORKSPACE: return "H3_ERR_WORKSPACE";
    case H3_ERR_CUDA: return "H3_ERR_CUDA";
    case H3_ERR_TIMEOUT: return "H3_ERR_TIMEOUT";
  }
  return "H3_ERR_UNKNOWN";
}

void h3_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns = ns ? ns : 2000000000ull; }

h3_status h3_check_device_error(h3_stream_t stream) {
  clear_error();
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t code = 0;
  e = cudaMemcpyFromSymbol(&code, g_dev_error_word, sizeof(code));
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (code != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_dev_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    return fail(H3_ERR_TIMEOUT, "bounded wait ran out in %s (code 0x%x)", err_code_name(code),
                code);
  }
  return H3_OK;
}

h3_status h3_debug_wait_timeout(uint64_t timeout_ns, h3_stream_t stream) {
  clear_error();
  DevErr err;
  h3_status st = dev_err(&err);
  if (st != H3_OK) return st;
  err.timeout_ns = timeout_ns;
  wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
  return cuda_fail(cudaGetLastError(), "wait-timeout probe launch");
}

h3_status h3_mod_norm_residual(float* resid, const void* delta, const float* gate,
                               const float* shift, const float* scale, void* normed, int S,
                               int L, int D, float eps, h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(resid != nullptr, H3_ERR_INVALID_ARG, "resid is NULL");
  H3_REQUIRE(delta != nullptr || normed != nullptr, H3_ERR_INVALID_ARG,
             "neither delta nor normed given: nothing to do");
  H3_REQUIRE(delta == nullptr || gate != nullptr, H3_ERR_INVALID_ARG, "delta given without gate");
  H3_REQUIRE(normed == nullptr || (shift != nullptr && scale != nullptr), H3_ERR_INVALID_ARG,
             "normed given without shift and scale");
  H3_REQUIRE(D > 0 && D % 8 == 0, H3_ERR_UNSUPPORTED, "D=%d must be a positive multiple of 8", D);
  H3_REQUIRE(D <= 8192, H3_ERR_UNSUPPORTED, "D=%d exceeds 8192", D);
  H3_REQUIRE(eps >= 0.f, H3_ERR_INVALID_ARG, "eps < 0");
  H3_REQUIRE(aligned16(resid) && aligned16(delta) && aligned16(gate) && aligned16(shift) &&
                 aligned16(scale) && aligned16(normed),
             H3_ERR_MISALIGNED, "a pointer is not 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_mod_norm_residual(resid, delta, gate, shift, scale, normed, L, D, eps,
                                  reinterpret_cast<cudaStream_t>(stream));
}

// pairing 0: interleaved pairs; 1: split-half pairs, every section a
// multiple of 16 wide (so each half is whole 8-channel slices).
static h3_status check_pairing(const int* axis_dims, int pairing) {
  H3_REQUIRE(pairing == 0 || pairing == 1, H3_ERR_INVALID_ARG, "rope pairing %d (0 or 1)",
             pairing);
  if (pairing == 1)
    for (int a = 0; a < 3; ++a)
      H3_REQUIRE(axis_dims[a] % 16 == 0, H3_ERR_UNSUPPORTED,
                 "split-half RoPE needs sections that are multiples of 16 (axis_dims[%d]=%d)", a,
                 axis_dims[a]);
  return H3_OK;
}

static h3_status qk_norm_rope_impl(void* q, void* k, const float* q_gain, const float* k_gain,
                                   const int32_t* pos, const int* axis_dims, int S, int L, int H,
                                   int Dh, float theta, float eps, int pairing,
                                   h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(q && k && q_gain && k_gain && pos && axis_dims, H3_ERR_INVALID_ARG,
             "a required pointer is NULL");
  H3_REQUIRE(Dh == 128, H3_ERR_UNSUPPORTED, "head_dim %d unsupported (128 only)", Dh);
  H3_REQUIRE(H > 0, H3_ERR_INVALID_ARG, "H=%d", H);
  int sum = 0;
  for (int a = 0; a < 3; ++a) {
    H3_REQUIRE(axis_dims[a] >= 0 && axis_dims[a] % 2 == 0, H3_ERR_INVALID_ARG,
               "axis_dims[%d]=%d must be even and >= 0", a, axis_dims[a]);
    sum += axis_dims[a];
  }
  H3_REQUIRE(sum == Dh, H3_ERR_INVALID_ARG, "axis_dims sum %d != head_dim %d", sum, Dh);
  if ((st = check_pairing(axis_dims, pairing)) != H3_OK) return st;
  H3_REQUIRE(theta > 0.f && eps >= 0.f, H3_ERR_INVALID_ARG, "theta must be > 0 and eps >= 0");
  H3_REQUIRE(aligned16(q) && aligned16(k) && aligned16(q_gain) && aligned16(k_gain),
             H3_ERR_MISALIGNED, "q, k and the gains must be 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_qk_norm_rope(q, k, static_cast<int64_t>(H) * Dh, q_gain, k_gain, pos, axis_dims,
                             L, H, theta, eps, reinterpret_cast<cudaStream_t>(stream), pairing);
}

h3_status h3_qk_norm_rope(void* q, void* k, const float* q_gain, const float* k_gain,
                          const int32_t* pos, const int* axis_dims, int S, int L, int H, int Dh,
                          float theta, float eps, h3_stream_t stream) {
  return qk_norm_rope_impl(q, k, q_gain, k_gain, pos, axis_dims, S, L, H, Dh, theta, eps, 0,
                           stream);
}

h3_status h3_qk_norm_rope_layout(void* q, void* k, const float* q_gain, const float* k_gain,
                                 const int32_t* pos, const int* axis_dims, int S, int L, int H,
                                 int Dh, float theta, float eps, int pairing,
                                 h3_stream_t stream) {
  return qk_norm_rope_impl(q, k, q_gain, k_gain, pos, axis_dims, S, L, H, Dh, theta, eps,
                           pairing, stream);
}

h3_status h3_attention_varlen(const void* q, const void* k, const void* v, void* o, int S,
                              int L, int H, int Dh, float softmax_scale, h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(q && k && v && o, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  H3_REQUIRE(Dh == 128, H3_ERR_UNSUPPORTED, "head_dim %d unsupported (128 only)", Dh);
  H3_REQUIRE(H > 0 && H <= 65535, H3_ERR_INVALID_ARG, "H=%d", H);
  H3_REQUIRE(softmax_scale > 0.f, H3_ERR_INVALID_ARG, "softmax_scale must be > 0");
  H3_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(o), H3_ERR_MISALIGNED,
             "q, k, v, o must be 16-byte aligned");
  if (L == 0) return H3_OK;
  const int64_t ld = static_cast<int64_t>(H) * Dh;
  return launch_attention(q, k, v, ld, o, ld, L, H, softmax_scale,
                          reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_attention_varlen_skip(const void* q, const void* k, const void* v, void* o, int S,
                                   int L, int H, int Dh, float softmax_scale, float skip_eps,
                                   int32_t* kept_tiles, h3_stream_t stream) {
  clear_error();
  H3_REQUIRE(skip_eps >= 0.f && skip_eps < 1.f, H3_ERR_INVALID_ARG,
             "skip_eps=%g must be in [0, 1)", static_cast<double>(skip_eps));
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(q && k && v && o, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  H3_REQUIRE(Dh == 128, H3_ERR_UNSUPPORTED, "head_dim %d unsupported (128 only)", Dh);
  H3_REQUIRE(H > 0 && H <= 65535, H3_ERR_INVALID_ARG, "H=%d", H);
  H3_REQUIRE(softmax_scale > 0.f, H3_ERR_INVALID_ARG, "softmax_scale must be > 0");
  H3_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(o), H3_ERR_MISALIGNED,
             "q, k, v, o must be 16-byte aligned");
  if (L == 0) return H3_OK;
  const int64_t ld = static_cast<int64_t>(H) * Dh;
  return launch_attention(q, k, v, ld, o, ld, L, H, softmax_scale,
                          reinterpret_cast<cudaStream_t>(stream), skip_eps, kept_tiles);
}

size_t h3_sage_scratch_bytes(int L, int H) {
  clear_error();
  if (L < 0 || H <= 0) return 0;
  return sage_scratch_bytes(L, H);
}

h3_status h3_sage_quantize(const void* q, const void* k, const void* v, int S, int L, int H,
                           int Dh, void* qc, void* kc, void* vc, float* sq, float* sk, float* sv,
                           float* k_mean, void* scratch, size_t scratch_bytes,
                           h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(q && k && v && qc && kc && vc && sq && sk && sv && k_mean, H3_ERR_INVALID_ARG,
             "a required pointer is NULL");
  H3_REQUIRE(Dh == 128, H3_ERR_UNSUPPORTED, "head_dim %d unsupported (128 only)", Dh);
  H3_REQUIRE(H > 0 && H <= 65535, H3_ERR_INVALID_ARG, "H=%d", H);
  H3_REQUIRE(scratch != nullptr && scratch_bytes >= sage_scratch_bytes(L, H), H3_ERR_WORKSPACE,
             "scratch of %zu bytes given, %zu needed", scratch_bytes, sage_scratch_bytes(L, H));
  H3_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(qc) && aligned16(kc) &&
                 aligned16(vc) && aligned16(sv) && aligned16(scratch),
             H3_ERR_MISALIGNED, "operands, codes, sv and scratch must be 16-byte aligned");
  if (L == 0) return H3_OK;
  const int64_t ld = static_cast<int64_t>(H) * Dh;
  return launch_sage_quantize(q, k, v, ld, L, H, static_cast<uint8_t*>(qc),
                              static_cast<uint8_t*>(kc), static_cast<uint8_t*>(vc), ld, sq, sk, sv,
                              k_mean, scratch, reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_attention_fp8(const void* qc, const void* kc, const void* vc, const float* sq,
                           const float* sk, const float* sv, void* o, int S, int L, int H,
                           int Dh, float softmax_scale, h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(qc && kc && vc && sq && sk && sv && o, H3_ERR_INVALID_ARG,
             "a required pointer is NULL");
  H3_REQUIRE(Dh == 128, H3_ERR_UNSUPPORTED, "head_dim %d unsupported (128 only)", Dh);
  H3_REQUIRE(H > 0 && H <= 65535, H3_ERR_INVALID_ARG, "H=%d", H);
  H3_REQUIRE(softmax_scale > 0.f, H3_ERR_INVALID_ARG, "softmax_scale must be > 0");
  H3_REQUIRE(aligned16(qc) && aligned16(kc) && aligned16(vc) && aligned16(o), H3_ERR_MISALIGNED,
             "codes and o must be 16-byte aligned");
  if (L == 0) return H3_OK;
  const int64_t ld = static_cast<int64_t>(H) * Dh;
  return launch_attention_fp8(qc, kc, vc, ld, sq, sk, sv, o, ld, L, H, softmax_scale,
                              reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_attention_fp8_skip(const void* qc, const void* kc, const void* vc, const float* sq,
                                const float* sk, const float* sv, void* o, int S, int L, int H,
                                int Dh, float softmax_scale, float skip_eps, int32_t* kept_tiles,
                                h3_stream_t stream) {
  clear_error();
  H3_REQUIRE(skip_eps >= 0.f && skip_eps < 1.f, H3_ERR_INVALID_ARG,
             "skip_eps=%g must be in [0, 1)", static_cast<double>(skip_eps));
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(qc && kc && vc && sq && sk && sv && o, H3_ERR_INVALID_ARG,
             "a required pointer is NULL");
  H3_REQUIRE(Dh == 128, H3_ERR_UNSUPPORTED, "head_dim %d unsupported (128 only)", Dh);
  H3_REQUIRE(H > 0 && H <= 65535, H3_ERR_INVALID_ARG, "H=%d", H);
  H3_REQUIRE(softmax_scale > 0.f, H3_ERR_INVALID_ARG, "softmax_scale must be > 0");
  H3_REQUIRE(aligned16(qc) && aligned16(kc) && aligned16(vc) && aligned16(o), H3_ERR_MISALIGNED,
             "codes and o must be 16-byte aligned");
  H3_REQUIRE(reinterpret_cast<uintptr_t>(kept_tiles) % 4 == 0, H3_ERR_MISALIGNED,
             "kept_tiles must be 4-byte aligned");
  if (L == 0) return H3_OK;
  const int64_t ld = static_cast<int64_t>(H) * Dh;
  return launch_attention_fp8(qc, kc, vc, ld, sq, sk, sv, o, ld, L, H, softmax_scale,
                              reinterpret_cast<cudaStream_t>(stream), skip_eps, kept_tiles);
}

h3_status h3_swiglu(const void* gate_up, void* out, int S, int L, int F, h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(gate_up && out, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  H3_REQUIRE(F > 0 && F % 8 == 0, H3_ERR_UNSUPPORTED, "F=%d must be a positive multiple of 8", F);
  H3_REQUIRE(aligned16(gate_up) && aligned16(out), H3_ERR_MISALIGNED,
             "gate_up and out must be 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_swiglu(gate_up, out, L, F, reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_linear(const void* x, const void* w, void* y, int S, int L, int N, int K,
                    h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(x && w && y, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  H3_REQUIRE(N > 0 && N % 256 == 0, H3_ERR_UNSUPPORTED, "N=%d must be a multiple of 256", N);
  H3_REQUIRE(K > 0 && K % 64 == 0, H3_ERR_UNSUPPORTED, "K=%d must be a multiple of 64", K);
  H3_REQUIRE(aligned16(x) && aligned16(w) && aligned16(y), H3_ERR_MISALIGNED,
             "x, w, y must be 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_gemm(x, K, w, K, y, N, L, N, K, GEMM_STORE_BF16,
                     reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_linear_swiglu(const void* x, const void* w_gu, void* out, int S, int L, int F, int K,
                           h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(x && w_gu && out, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  H3_REQUIRE(F > 0 && F % 128 == 0, H3_ERR_UNSUPPORTED, "F=%d must be a multiple of 128", F);
  H3_REQUIRE(K > 0 && K % 64 == 0, H3_ERR_UNSUPPORTED, "K=%d must be a multiple of 64", K);
  H3_REQUIRE(aligned16(x) && aligned16(w_gu) && aligned16(out), H3_ERR_MISALIGNED,
             "x, w_gu, out must be 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_gemm(x, K, w_gu, K, out, F, L, F, K, GEMM_SWIGLU,
                     reinterpret_cast<cudaStream_t>(stream));
}

static h3_status check_axis_dims(const int* axis_dims) {
  H3_REQUIRE(axis_dims != nullptr, H3_ERR_INVALID_ARG, "axis_dims is NULL");
  int sum = 0;
  for (int a = 0; a < 3; ++a) {
    H3_REQUIRE(axis_dims[a] >= 0 && axis_dims[a] % 2 == 0, H3_ERR_INVALID_ARG,
               "axis_dims[%d]=%d must be even and >= 0", a, axis_dims[a]);
    sum += axis_dims[a];
  }
  H3_REQUIRE(sum == 128, H3_ERR_INVALID_ARG, "axis_dims sum %d != head_dim 128", sum);
  return H3_OK;
}

h3_status h3_rope_table(const int32_t* pos, const int* axis_dims, int S, int L, float theta,
                        float* table, h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(pos && table, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  if ((st = check_axis_dims(axis_dims)) != H3_OK) return st;
  H3_REQUIRE(theta > 0.f, H3_ERR_INVALID_ARG, "theta must be > 0");
  H3_REQUIRE(aligned16(table), H3_ERR_MISALIGNED, "table must be 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_rope_table(pos, axis_dims, L, theta, reinterpret_cast<float2*>(table),
                           reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_linear_qk_norm_rope(const void* x, const void* w_qkv, void* qkv,
                                 const float* q_gain, const float* k_gain,
                                 const float* rope_table, const int* axis_dims, int pairing,
                                 int S, int L, int H, int K, float eps, h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(x && w_qkv && qkv && q_gain && k_gain && rope_table, H3_ERR_INVALID_ARG,
             "a required pointer is NULL");
  H3_REQUIRE(H > 0 && H % 2 == 0, H3_ERR_UNSUPPORTED, "H=%d must be even", H);
  H3_REQUIRE(K > 0 && K % 64 == 0, H3_ERR_UNSUPPORTED, "K=%d must be a multiple of 64", K);
  H3_REQUIRE(eps >= 0.f, H3_ERR_INVALID_ARG, "eps must be >= 0");
  if ((st = check_axis_dims(axis_dims)) != H3_OK) return st;
  if ((st = check_pairing(axis_dims, pairing)) != H3_OK) return st;
  H3_REQUIRE(aligned16(x) && aligned16(w_qkv) && aligned16(qkv) && aligned16(q_gain) &&
                 aligned16(k_gain) && aligned16(rope_table),
             H3_ERR_MISALIGNED, "pointers must be 16-byte aligned");
  if (L == 0) return H3_OK;
  const int D = H * 128;
  GemmExtra ex;
  ex.q_gain = q_gain;
  ex.k_gain = k_gain;
  ex.rope = reinterpret_cast<const float2*>(rope_table);
  ex.d_model = D;
  ex.eps = eps;
  if (pairing == 1) rope_pieces(axis_dims, &ex);
  return launch_gemm(x, K, w_qkv, K, qkv, 3LL * D, L, 3 * D, K, GEMM_QK_NORM_ROPE,
                     reinterpret_cast<cudaStream_t>(stream), &ex);
}

h3_status h3_linear_residual(const void* x, const void* w, float* resid, const float* gate,
                             int S, int L, int N, int K, h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(x && w && resid && gate, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  H3_REQUIRE(N > 0 && N % 256 == 0, H3_ERR_UNSUPPORTED, "N=%d must be a multiple of 256", N);
  H3_REQUIRE(K > 0 && K % 64 == 0, H3_ERR_UNSUPPORTED, "K=%d must be a multiple of 64", K);
  H3_REQUIRE(aligned16(x) && aligned16(w) && aligned16(resid) && aligned16(gate),
             H3_ERR_MISALIGNED, "x, w, resid, gate must be 16-byte aligned");
  if (L == 0) return H3_OK;
  GemmExtra ex;
  ex.gate = gate;
  return launch_gemm(x, K, w, K, resid, N, L, N, K, GEMM_RESIDUAL,
                     reinterpret_cast<cudaStream_t>(stream), &ex);
}

static h3_status check_block_config(const h3_block_config* c) {
  H3_REQUIRE(c != nullptr, H3_ERR_INVALID_ARG, "config is NULL");
  h3_status st = check_rows(c->S, c->L);
  if (st != H3_OK) return st;
  H3_REQUIRE(c->Dh == 128, H3_ERR_UNSUPPORTED, "head_dim %d unsupported (128 only)", c->Dh);
  H3_REQUIRE(c->H > 0 && c->D == c->H * c->Dh, H3_ERR_INVALID_ARG, "D=%d != H*Dh=%d", c->D,
             c->H * c->Dh);
  H3_REQUIRE(c->D % 256 == 0 && c->D <= 8192, H3_ERR_UNSUPPORTED,
             "D=%d must be a multiple of 256 and at most 8192", c->D);
  H3_REQUIRE(c->F > 0 && c->F % 128 == 0, H3_ERR_UNSUPPORTED, "F=%d must be a multiple of 128",
             c->F);
  st = check_pairing(c->axis_dims, c->rope_pairing);
  if (st != H3_OK) return st;
  int sum = 0;
  for (int a = 0; a < 3; ++a) {
    H3_REQUIRE(c->axis_dims[a] >= 0 && c->axis_dims[a] % 2 == 0, H3_ERR_INVALID_ARG,
               "axis_dims[%d]=%d must be even and >= 0", a, c->axis_dims[a]);
    sum += c->axis_dims[a];
  }
  H3_REQUIRE(sum == c->Dh, H3_ERR_INVALID_ARG, "axis_dims sum %d != head_dim %d", sum, c->Dh);
  H3_REQUIRE(c->theta > 0.f && c->eps_ln >= 0.f && c->eps_qk >= 0.f, H3_ERR_INVALID_ARG,
             "theta must be > 0 and the epsilons >= 0");
  return H3_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace slices (bf16, S rows each): h [D] (h1, later h2), qkv [3D],
// attn [D], proj [D] (attention projection, later FFN down), ffn [F].
struct BlockWs {
  size_t h, qkv, attn, proj, ffn, rope, total;
};
static BlockWs block_ws(const h3_block_config* c) {
  BlockWs w;
  const size_t row = static_cast<size_t>(c->S) * 2;
  size_t off = 0;
  w.h = off;    off += align256(row * c->D);
  w.qkv = off;  off += align256(row * 3 * c->D);
  w.attn = off; off += align256(row * c->D);
  w.proj = off; off += align256(row * c->D);
  w.ffn = off;  off += align256(row * c->F);
  w.rope = off; off += align256(static_cast<size_t>(c->S) * 64 * sizeof(float2));
  w.total = off;
  return w;
}

size_t h3_block_workspace_bytes(const h3_block_config* cfg) {
  clear_error();
  if (check_block_config(cfg) != H3_OK) return 0;
  return block_ws(cfg).total;
}

static h3_status check_weights(const h3_block_weights* w) {
  H3_REQUIRE(w != nullptr, H3_ERR_INVALID_ARG, "weights struct is NULL");
  H3_REQUIRE(w->w_qkv && w->w_o && w->w_gu && w->w_down && w->q_gain && w->k_gain,
             H3_ERR_INVALID_ARG, "a weight pointer is NULL");
  H3_REQUIRE(aligned16(w->w_qkv) && aligned16(w->w_o) && aligned16(w->w_gu) &&
                 aligned16(w->w_down) && aligned16(w->q_gain) && aligned16(w->k_gain),
             H3_ERR_MISALIGNED, "weights and gains must be 16-byte aligned");
  return H3_OK;
}

// Runs num_blocks blocks in order over the residual stream. Block b uses
// w[b] and the modulation table mod + b * num_seg * 6 * D ([num_seg, 6, D]);
// with seg given, row i uses group seg[i] of that table. Fusions:
//   * the RoPE (cos, sin) table is built once, by the first modulated
//     LayerNorm pass (positions are shared by all blocks), and Q/K RMSNorm +
//     RoPE run in the QKV projection's epilogue;
//   * the residual update that ends block b and the modulated LayerNorm that
//     starts block b + 1 run as one pass over the residual;
//   * the last block's residual update runs in the down projection's
//     epilogue.
// events (one block only): recorded before every stage and after the last.
static h3_status stack_forward_impl(const h3_block_config* cfg, const h3_block_weights* w,
                                    int num_blocks, float* resid, const float* mod, int num_seg,
                                    const int32_t* seg, const int32_t* pos, void* workspace,
                                    size_t workspace_bytes, h3_stream_t stream,
                                    void* const* events, int num_events) {
  clear_error();
  h3_status st = check_block_config(cfg);
  if (st != H3_OK) return st;
  H3_REQUIRE(num_blocks >= 1, H3_ERR_INVALID_ARG, "num_blocks=%d", num_blocks);
  H3_REQUIRE(num_seg >= 1, H3_ERR_INVALID_ARG, "num_seg=%d", num_seg);
  H3_REQUIRE(seg != nullptr || num_seg == 1, H3_ERR_INVALID_ARG,
             "num_seg=%d needs a seg array", num_seg);
  H3_REQUIRE(w != nullptr, H3_ERR_INVALID_ARG, "weights array is NULL");
  for (int b = 0; b < num_blocks; ++b)
    if ((st = check_weights(&w[b])) != H3_OK) return st;
  H3_REQUIRE(resid && mod && pos, H3_ERR_INVALID_ARG, "resid, mod and pos must not be NULL");
  const BlockWs ws = block_ws(cfg);
  H3_REQUIRE(workspace != nullptr && workspace_bytes >= ws.total, H3_ERR_WORKSPACE,
             "workspace of %zu bytes given, %zu needed", workspace_bytes, ws.total);
  H3_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, H3_ERR_MISALIGNED,
             "workspace must be 256-byte aligned");
  H3_REQUIRE(aligned16(resid) && aligned16(mod), H3_ERR_MISALIGNED,
             "resid and mod must be 16-byte aligned");
  H3_REQUIRE(events == nullptr || (num_blocks == 1 && num_events == H3_BLOCK_STAGES + 1),
             H3_ERR_INVALID_ARG, "events: %d given, %d expected (one block)", num_events,
             H3_BLOCK_STAGES + 1);
  if (events != nullptr)
    for (int i = 0; i <= H3_BLOCK_STAGES; ++i)
      H3_REQUIRE(events[i] != nullptr, H3_ERR_INVALID_ARG, "events[%d] is NULL", i);
  if (cfg->L == 0) return H3_OK;

  const int L = cfg->L, D = cfg->D, H = cfg->H, F = cfg->F;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  void* h = base + ws.h;
  uint8_t* qkv = base + ws.qkv;
  void* attn = base + ws.attn;
  void* proj = base + ws.proj;
  void* ffn = base + ws.ffn;
  float2* rope = reinterpret_cast<float2*>(base + ws.rope);
  const int64_t ld_qkv = 3LL * D;
  const int64_t seg_stride = 6LL * D;  // floats between groups of one table
  const int64_t block_stride = static_cast<int64_t>(num_seg) * seg_stride;
  auto mark = [&](int i) -> h3_status {
    if (events == nullptr) return H3_OK;
    return cuda_fail(cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s), "event record");
  };
  auto mnr = [&](const void* delta, const float* gate, const float* shift, const float* scale,
                 void* normed, const RopeRequest* rope = nullptr) {
    return launch_mod_norm_residual(resid, delta, gate, shift, scale, normed, L, D, cfg->eps_ln,
                                    s, seg, num_seg, seg_stride, rope);
  };
#define H3_STAGE(i, call)                          \
  do {                                             \
    if ((st = mark(i)) != H3_OK) return st;        \
    if ((st = (call)) != H3_OK) return st;         \
  } while (0)

  for (int b = 0; b < num_blocks; ++b) {
    const h3_block_weights& wb = w[b];
    // (shift1, scale1, gate1, shift2, scale2, gate2) of group 0 of block b
    const float* m = mod + b * block_stride;
    const float* shift1 = m;
    const float* scale1 = m + D;
    const float* gate1 = m + 2 * D;
    const float* shift2 = m + 3 * D;
    const float* scale2 = m + 4 * D;
    const float* gate2 = m + 5 * D;
    // 0: h1 = LN(r) * (1 + scale1) + shift1 (fused into the previous block's
    //    last pass for b > 0); the same pass writes the RoPE table of every
    //    row, once per call
    if (b == 0) {
      const RopeRequest rq{pos, cfg->axis_dims, cfg->theta, rope};
      H3_STAGE(0, mnr(nullptr, nullptr, shift1, scale1, h, &rq));
    }
    // 1: [q | k | v] = h1 W_qkv^T; q, k <- RoPE(RMSNorm(q, k)) per head in the
    //    epilogue
    GemmExtra qk;
    qk.q_gain = wb.q_gain;
    qk.k_gain = wb.k_gain;
    qk.rope = rope;
    qk.d_model = D;
    qk.eps = cfg->eps_qk;
    if (cfg->rope_pairing == 1) rope_pieces(cfg->axis_dims, &qk);
    H3_STAGE(1, launch_gemm(h, D, wb.w_qkv, D, qkv, ld_qkv, L, 3 * D, D, GEMM_QK_NORM_ROPE, s,
                            &qk));
    // 2: a = softmax(q k^T / sqrt(Dh)) v over keys < L
    H3_STAGE(2, launch_attention(qkv, qkv + 2LL * D, qkv + 4LL * D, ld_qkv, attn, D, L, H,
                                 1.0f / sqrtf(static_cast<float>(cfg->Dh)), s));
    // 3: o = a W_o^T
    H3_STAGE(3, launch_gemm(attn, D, wb.w_o, D, proj, D, L, D, D, GEMM_STORE_BF16, s));
    // 4: r <- r + gate1 * o ; h2 = LN(r) * (1 + scale2) + shift2
    H3_STAGE(4, mnr(proj, gate1, shift2, scale2, h));
    // 5: s = SiLU(h2 W_g^T) * (h2 W_u^T), SwiGLU fused in the projection's epilogue
    H3_STAGE(5, launch_gemm(h, D, wb.w_gu, D, ffn, F, L, F, D, GEMM_SWIGLU, s));
    // 6: f = s W_down^T; r <- r + gate2 * f, in the epilogue for the last
    //    block, else in one pass with the next block's
    //    h1 = LN(r) * (1 + scale1') + shift1'
    if (b + 1 < num_blocks) {
      const float* mn = mod + (b + 1) * block_stride;
      H3_STAGE(6, launch_gemm(ffn, F, wb.w_down, F, proj, D, L, D, F, GEMM_STORE_BF16, s));
      if ((st = mnr(proj, gate2, mn, mn + D, h)) != H3_OK) return st;
    } else {
      GemmExtra res;
      res.gate = gate2;
      res.seg = seg;
      res.num_seg = num_seg;
      res.seg_stride = seg_stride;
      H3_STAGE(6, launch_gemm(ffn, F, wb.w_down, F, resid, D, L, D, F, GEMM_RESIDUAL, s, &res));
    }
  }
#undef H3_STAGE
  return mark(H3_BLOCK_STAGES);
}

static h3_status block_forward_impl(const h3_block_config* cfg, const h3_block_weights* w,
                                    float* resid, const float* mod, const int32_t* pos,
                                    void* workspace, size_t workspace_bytes, h3_stream_t stream,
                                    void* const* events, int num_events) {
  return stack_forward_impl(cfg, w, 1, resid, mod, 1, nullptr, pos, workspace, workspace_bytes,
                            stream, events, num_events);
}

h3_status h3_block_forward(const h3_block_config* cfg, const h3_block_weights* w, float* resid,
                           const float* mod, const int32_t* pos, void* workspace,
                           size_t workspace_bytes, h3_stream_t stream) {
  return block_forward_impl(cfg, w, resid, mod, pos, workspace, workspace_bytes, stream, nullptr,
                            0);
}

h3_status h3_block_forward_events(const h3_block_config* cfg, const h3_block_weights* w,
                                  float* resid, const float* mod, const int32_t* pos,
                                  void* workspace, size_t workspace_bytes, h3_stream_t stream,
                                  void* const* events, int num_events) {
  H3_REQUIRE(events != nullptr, H3_ERR_INVALID_ARG, "events is NULL");
  return block_forward_impl(cfg, w, resid, mod, pos, workspace, workspace_bytes, stream, events,
                            num_events);
}

h3_status h3_stack_forward(const h3_block_config* cfg, const h3_block_weights* w,
                           int num_blocks, float* resid, const float* mod, int num_seg,
                           const int32_t* seg, const int32_t* pos, void* workspace,
                           size_t workspace_bytes, h3_stream_t stream) {
  return stack_forward_impl(cfg, w, num_blocks, resid, mod, num_seg, seg, pos, workspace,
                            workspace_bytes, stream, nullptr, 0);
}

h3_status h3_mod_norm_residual_seg(float* resid, const void* delta, const float* gate,
                                   const float* shift, const float* scale, const int32_t* seg,
                                   int num_seg, int64_t seg_stride, void* normed, int S, int L,
                                   int D, float eps, h3_stream_t stream) {
  clear_error();
  H3_REQUIRE(seg != nullptr, H3_ERR_INVALID_ARG, "seg is NULL");
  H3_REQUIRE(num_seg >= 1, H3_ERR_INVALID_ARG, "num_seg=%d", num_seg);
  H3_REQUIRE(seg_stride >= D || num_seg == 1, H3_ERR_INVALID_ARG,
             "seg_stride=%lld is shorter than D=%d", static_cast<long long>(seg_stride), D);
  H3_REQUIRE(seg_stride % 4 == 0, H3_ERR_MISALIGNED,
             "seg_stride must be a multiple of 4 floats (16 bytes)");
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(resid != nullptr, H3_ERR_INVALID_ARG, "resid is NULL");
  H3_REQUIRE(delta != nullptr || normed != nullptr, H3_ERR_INVALID_ARG,
             "neither delta nor normed given: nothing to do");
  H3_REQUIRE(delta == nullptr || gate != nullptr, H3_ERR_INVALID_ARG, "delta given without gate");
  H3_REQUIRE(normed == nullptr || (shift != nullptr && scale != nullptr), H3_ERR_INVALID_ARG,
             "normed given without shift and scale");
  H3_REQUIRE(D > 0 && D % 8 == 0 && D <= 8192, H3_ERR_UNSUPPORTED,
             "D=%d must be a positive multiple of 8, at most 8192", D);
  H3_REQUIRE(eps >= 0.f, H3_ERR_INVALID_ARG, "eps < 0");
  H3_REQUIRE(aligned16(resid) && aligned16(delta) && aligned16(gate) && aligned16(shift) &&
                 aligned16(scale) && aligned16(normed),
             H3_ERR_MISALIGNED, "a pointer is not 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_mod_norm_residual(resid, delta, gate, shift, scale, normed, L, D, eps,
                                  reinterpret_cast<cudaStream_t>(stream), seg, num_seg,
                                  seg_stride);
}

h3_status h3_frames_to_u8(const float* frames, uint8_t* out, int B, int C, int T, int H, int W,
                          h3_stream_t stream) {
  clear_error();
  H3_REQUIRE(frames != nullptr && out != nullptr, H3_ERR_INVALID_ARG, "a pointer is NULL");
  H3_REQUIRE(B >= 0 && C >= 1 && T >= 0 && H >= 0 && W >= 0, H3_ERR_INVALID_ARG,
             "bad shape B=%d C=%d T=%d H=%d W=%d", B, C, T, H, W);
  H3_REQUIRE(C <= 16, H3_ERR_UNSUPPORTED, "C=%d exceeds 16 channels", C);
  const int64_t N = static_cast<int64_t>(T) * H * W;
  H3_REQUIRE(N % 4 == 0, H3_ERR_UNSUPPORTED, "T*H*W=%lld must be a multiple of 4",
             static_cast<long long>(N));
  H3_REQUIRE(aligned16(frames) && (reinterpret_cast<uintptr_t>(out) & 3u) == 0,
             H3_ERR_MISALIGNED, "frames must be 16-byte and out 4-byte aligned");
  if (B == 0 || N == 0) return H3_OK;
  return launch_frames_to_u8(frames, out, B, C, N, reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_quantize_fp8_rows(const void* x, void* q, float* scale, int R, int K,
                               h3_stream_t stream) {
  clear_error();
  H3_REQUIRE(x && q && scale, H3_ERR_INVALID_ARG, "a pointer is NULL");
  H3_REQUIRE(R >= 0, H3_ERR_INVALID_ARG, "R=%d", R);
  H3_REQUIRE(K > 0 && K % 8 == 0 && K <= 16384, H3_ERR_UNSUPPORTED,
             "K=%d must be a positive multiple of 8, at most 16384", K);
  H3_REQUIRE(aligned16(x) && aligned16(q), H3_ERR_MISALIGNED, "x and q must be 16-byte aligned");
  if (R == 0) return H3_OK;
  return launch_quantize_fp8_rows(x, K, q, K, scale, R, K,
                                  reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_linear_fp8(const void* qx, const float* sx, const void* qw, const float* sw, void* y,
                        int S, int L, int N, int K, h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(qx && sx && qw && sw && y, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  H3_REQUIRE(N > 0 && N % 256 == 0, H3_ERR_UNSUPPORTED, "N=%d must be a multiple of 256", N);
  H3_REQUIRE(K > 0 && K % 128 == 0, H3_ERR_UNSUPPORTED, "K=%d must be a multiple of 128", K);
  H3_REQUIRE(aligned16(qx) && aligned16(qw) && aligned16(y), H3_ERR_MISALIGNED,
             "qx, qw, y must be 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_gemm_fp8(qx, K, sx, qw, K, sw, y, N, L, N, K, GEMM_STORE_BF16,
                         reinterpret_cast<cudaStream_t>(stream));
}

h3_status h3_linear_swiglu_fp8(const void* qx, const float* sx, const void* qw_gu,
                               const float* sw_gu, void* out, int S, int L, int F, int K,
                               h3_stream_t stream) {
  clear_error();
  h3_status st = check_rows(S, L);
  if (st != H3_OK) return st;
  H3_REQUIRE(qx && sx && qw_gu && sw_gu && out, H3_ERR_INVALID_ARG, "a required pointer is NULL");
  H3_REQUIRE(F > 0 && F % 128 == 0, H3_ERR_UNSUPPORTED, "F=%d must be a multiple of 128", F);
  H3_REQUIRE(K > 0 && K % 128 == 0, H3_ERR_UNSUPPORTED, "K=%d must be a multiple of 128", K);
  H3_REQUIRE(aligned16(qx) && aligned16(qw_gu) && aligned16(out), H3_ERR_MISALIGNED,
             "qx, qw_gu, out must be 16-byte aligned");
  if (L == 0) return H3_OK;
  return launch_gemm_fp8(qx, K, sx, qw_gu, K, sw_gu, out, F, L, F, K, GEMM_SWIGLU,
                         reinterpret_cast<cudaStream_t>(stream));
}

// FP8 block workspace: the BF16 block's slices, one FP8 code buffer
// [S, max(D, F)] and one scale vector [S] for the projections, then the FP8
// attention operands (codes of q, k, v [S, D] each, tile scales sq, sk
// [ceil(L/128), H], channel scales sv and the K mean [H, 128], scratch).
struct BlockWsFp8 {
  BlockWs bf;
  size_t codes, scales, aq, ak, av, sq, sk, sv, kmean, scratch, total;
};
static BlockWsFp8 block_ws_fp8(const h3_block_config* c) {
  BlockWsFp8 w;
  w.bf = block_ws(c);
  const size_t S = static_cast<size_t>(c->S), D = static_cast<size_t>(c->D);
  const size_t tiles = (static_cast<size_t>(c->L) + 127) / 128 + 1;
  size_t off = w.bf.total;
  w.codes = off;   off += align256(S * std::max(c->D, c->F));
  w.scales = off;  off += align256(S * 4);
  w.aq = off;      off += align256(S * D);
  w.ak = off;      off += align256(S * D);
  w.av = off;      off += align256(S * D);
  w.sq = off;      off += align256(tiles * c->H * 4);
  w.sk = off;      off += align256(tiles * c->H * 4);
  w.sv = off;      off += align256(D * 4);
  w.kmean = off;   off += align256(D * 4);
  w.scratch = off; off += align256(sage_scratch_bytes(c->L, c->H));
  w.total = off;
  return w;
}

size_t h3_block_workspace_bytes_fp8(const h3_block_config* cfg) {
  clear_error();
  if (check_block_config(cfg) != H3_OK) return 0;
  if (cfg->D % 128 != 0) {
    fail(H3_ERR_UNSUPPORTED, "D=%d must be a multiple of 128 for FP8 projections", cfg->D);
    return 0;
  }
  return block_ws_fp8(cfg).total;
}

h3_status h3_block_forward_fp8(const h3_block_config* cfg, const h3_block_weights_fp8* w,
                               float* resid, const float* mod, const int32_t* pos,
                               int fp8_attention, void* workspace, size_t workspace_bytes,
                               h3_stream_t stream) {
  clear_error();
  h3_status st = check_block_config(cfg);
  if (st != H3_OK) return st;
  H3_REQUIRE(cfg->D % 128 == 0, H3_ERR_UNSUPPORTED, "D=%d must be a multiple of 128", cfg->D);
  H3_REQUIRE(w != nullptr, H3_ERR_INVALID_ARG, "weights struct is NULL");
  H3_REQUIRE(w->w_qkv && w->s_qkv && w->w_o && w->s_o && w->w_gu && w->s_gu && w->w_down &&
                 w->s_down && w->q_gain && w->k_gain,
             H3_ERR_INVALID_ARG, "a weight or scale pointer is NULL");
  H3_REQUIRE(aligned16(w->w_qkv) && aligned16(w->w_o) && aligned16(w->w_gu) &&
                 aligned16(w->w_down) && aligned16(w->q_gain) && aligned16(w->k_gain),
             H3_ERR_MISALIGNED, "weights and gains must be 16-byte aligned");
  H3_REQUIRE(resid && mod && pos, H3_ERR_INVALID_ARG, "resid, mod and pos must not be NULL");
  H3_REQUIRE(aligned16(resid) && aligned16(mod), H3_ERR_MISALIGNED,
             "resid and mod must be 16-byte aligned");
  const BlockWsFp8 ws = block_ws_fp8(cfg);
  H3_REQUIRE(workspace != nullptr && workspace_bytes >= ws.total, H3_ERR_WORKSPACE,
             "workspace of %zu bytes given, %zu needed", workspace_bytes, ws.total);
  H3_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, H3_ERR_MISALIGNED,
             "workspace must be 256-byte aligned");
  if (cfg->L == 0) return H3_OK;
  const int L = cfg->L, D = cfg->D, H = cfg->H, F = cfg->F;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* qkv = base + ws.bf.qkv;
  void* attn = base + ws.bf.attn;
  void* proj = base + ws.bf.proj;
  void* ffn = base + ws.bf.ffn;
  void* codes = base + ws.codes;
  float* sc = reinterpret_cast<float*>(base + ws.scales);
  float2* rope = reinterpret_cast<float2*>(base + ws.bf.rope);
  GemmExtra qk;
  qk.q_gain = w->q_gain;
  qk.k_gain = w->k_gain;
  qk.rope = rope;
  qk.d_model = D;
  qk.eps = cfg->eps_qk;
  if (cfg->rope_pairing == 1) rope_pieces(cfg->axis_dims, &qk);
  GemmExtra res;
  res.gate = mod + 5 * D;
  const int64_t ld_qkv = 3LL * D;
  const float* m = mod;
  auto quant = [&](const void* x, int K) {
    return launch_quantize_fp8_rows(x, K, codes, K, sc, L, K, s);
  };
  const float sm_scale = 1.0f / sqrtf(static_cast<float>(cfg->Dh));
  auto attention = [&](uint8_t* qkv_, void* out) -> h3_status {
    if (!fp8_attention)
      return launch_attention(qkv_, qkv_ + 2LL * D, qkv_ + 4LL * D, ld_qkv, out, D, L, H,
                              sm_scale, s);
    uint8_t* aq = base + ws.aq;
    uint8_t* ak = base + ws.ak;
    uint8_t* av = base + ws.av;
    float* sq = reinterpret_cast<float*>(base + ws.sq);
    float* sk = reinterpret_cast<float*>(base + ws.sk);
    float* sv = reinterpret_cast<float*>(base + ws.sv);
    float* km = reinterpret_cast<float*>(base + ws.kmean);
    h3_status r = launch_sage_quantize(qkv_, qkv_ + 2LL * D, qkv_ + 4LL * D, ld_qkv, L, H, aq, ak,
                                       av, D, sq, sk, sv, km, base + ws.scratch, s);
    if (r != H3_OK) return r;
    return launch_attention_fp8(aq, ak, av, D, sq, sk, sv, out, D, L, H, sm_scale, s);
  };
  const RopeRequest rq{pos, cfg->axis_dims, cfg->theta, rope};
  // the modulated LayerNorm passes write the FP8 codes of h1 / h2 directly
  uint8_t* c8 = static_cast<uint8_t*>(codes);
  if ((st = launch_mod_norm_residual(resid, nullptr, nullptr, m, m + D, nullptr, L, D,
                                     cfg->eps_ln, s, nullptr, 1, 0, &rq, c8, sc)) != H3_OK ||
      (st = launch_gemm_fp8(codes, D, sc, w->w_qkv, D, w->s_qkv, qkv, ld_qkv, L, 3 * D, D,
                            GEMM_QK_NORM_ROPE, s, &qk)) != H3_OK ||
      (st = attention(qkv, attn)) != H3_OK ||
      (st = quant(attn, D)) != H3_OK ||
      (st = launch_gemm_fp8(codes, D, sc, w->w_o, D, w->s_o, proj, D, L, D, D, GEMM_STORE_BF16,
                            s)) != H3_OK ||
      (st = launch_mod_norm_residual(resid, proj, m + 2 * D, m + 3 * D, m + 4 * D, nullptr, L,
                                     D, cfg->eps_ln, s, nullptr, 1, 0, nullptr, c8, sc)) !=
          H3_OK ||
      (st = launch_gemm_fp8(codes, D, sc, w->w_gu, D, w->s_gu, ffn, F, L, F, D, GEMM_SWIGLU,
                            s)) != H3_OK ||
      (st = quant(ffn, F)) != H3_OK ||
      (st = launch_gemm_fp8(codes, F, sc, w->w_down, F, w->s_down, resid, D, L, D, F,
                            GEMM_RESIDUAL, s, &res)) != H3_OK)
    return st;
  return H3_OK;
}

// Scratch of h3_block_forward_noalloc: a fixed array in the library's device
// data, so that entry point never allocates. Host code only sees a stand-in
// for this symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[H3_NOALLOC_SCRATCH_BYTES];
static void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
static h3_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev >= kMaxDevices) return fail(H3_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return H3_OK;
}

h3_status h3_block_forward_noalloc(const h3_block_config* cfg, const h3_block_weights* w,
                                   float* resid, const float* mod, const int32_t* pos,
                                   h3_stream_t stream) {
  clear_error();
  h3_status st = check_block_config(cfg);
  if (st != H3_OK) return st;
  const size_t need = block_ws(cfg).total;
  H3_REQUIRE(need <= H3_NOALLOC_SCRATCH_BYTES, H3_ERR_WORKSPACE,
             "this block needs %zu bytes of scratch; the no-alloc entry point has %u bytes "
             "(use h3_block_forward with a workspace)",
             need, static_cast<unsigned>(H3_NOALLOC_SCRATCH_BYTES));
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != H3_OK) return st;
  return block_forward_impl(cfg, w, resid, mod, pos, scratch, H3_NOALLOC_SCRATCH_BYTES, stream,
                            nullptr, 0);
}

}  // extern "C"
