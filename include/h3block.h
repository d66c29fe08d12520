/*
 * h3block — forward pass of one joint audio-video DiT block (MiniMax H3
 * style) on a single NVIDIA GB300 (sm_103a).
 *
 * The operations follow the vLLM-Omni MiniMax H3 serving blog ("vLLM-Omni 上的
 * MiniMax H3：从系统级优化到基于 FastVideo FastH3 的实时服务"):
 *   section 3.1  one packed sequence of text, audio and video tokens; the
 *                attention backend takes the valid length and does no work on
 *                the structural tail padding; RoPE rows come from each
 *                token's own positions; hidden width 5,376.
 *   section 3.2  fused Q/K RMSNorm + RoPE (#5990), merged FP32 modulation +
 *                normalisation + residual (#6281, #6878), fused SwiGLU in
 *                place of separate SiLU and multiply launches (#6283), all
 *                around the block's matrix multiplies.
 *
 * Conventions shared by every call
 *   - Pointers are device memory owned by the caller (unless a parameter says
 *     "host"). The library never allocates, frees or keeps a pointer after the
 *     call returns.
 *   - Tensors are row-major and contiguous. A "packed sequence" tensor has S
 *     buffer rows of which the first L are valid. Rows >= L of every output
 *     are left exactly as they were, and rows >= L of every input are never
 *     read (pad rows may hold anything).
 *   - bf16 tensors are passed as void* (IEEE bfloat16, 2 bytes per element).
 *   - Base pointers must be 16-byte aligned, else H3_ERR_MISALIGNED.
 *   - Work is queued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream). Calls return as soon as the work is queued and never
 *     synchronise. Argument errors are detected on the host before anything
 *     is launched; nothing is launched when a call returns an error.
 *   - L == 0 is an empty sequence: the call does nothing and returns H3_OK.
 *   - The device's current CUDA device must be the one that owns the memory.
 *   - Every device-side wait is bounded. A wait that runs out records a code
 *     in a device error word; h3_check_device_error() reports it.
 */
#ifndef H3BLOCK_H_
#define H3BLOCK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum h3_status {
  H3_OK = 0,
  H3_ERR_INVALID_ARG = 1,   /* null pointer, negative size, L > S, ...        */
  H3_ERR_UNSUPPORTED = 2,   /* a size this build has no kernel for            */
  H3_ERR_MISALIGNED = 3,    /* a pointer or row stride not 16-byte aligned    */
  H3_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required     */
  H3_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed              */
  H3_ERR_TIMEOUT = 6        /* a bounded device wait ran out (see below)      */
} h3_status;

/* ABI-identical to cudaStream_t. */
typedef struct CUstream_st* h3_stream_t;

/* Library version, (major << 16) | minor. */
int h3_version(void);

/* Message for the last error returned on the calling host thread (never NULL;
 * "" when the last call succeeded). Valid until the next call on that thread. */
const char* h3_last_error(void);

/* Name of a status code. */
const char* h3_status_string(h3_status s);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device. Returns H3_ERR_TIMEOUT (message names the waiting kernel
 * role) when a bounded wait in an earlier kernel ran out, H3_ERR_CUDA when the
 * stream reports an error, else H3_OK. */
h3_status h3_check_device_error(h3_stream_t stream);

/* Per-wait limit in nanoseconds used by kernels launched after this call
 * (default 2e9). Host-side setting, process-wide. 0 restores the default. */
void h3_set_wait_timeout_ns(uint64_t ns);

/*
 * a1 — FP32 modulation + normalisation + residual (blog section 3.2, #6281,
 * #6878), one pass per row:
 *   if delta != NULL:  resid[i,:] <- resid[i,:] + gate[:] * delta[i,:]   (FP32)
 *   if normed != NULL: normed[i,:] <- bf16( LN(resid[i,:]) * (1 + scale[:]) + shift[:] )
 * where LN is LayerNorm without affine over D with epsilon eps, computed in FP32
 * from the updated residual.
 *   resid  [S, D] float32, in/out          delta  [S, D] bf16 or NULL
 *   gate   [D] float32 (required iff delta) shift, scale [D] float32 (required iff normed)
 *   normed [S, D] bf16 or NULL
 * At least one of delta / normed must be given. D % 8 == 0, D <= 8192.
 */
h3_status h3_mod_norm_residual(float* resid, const void* delta, const float* gate,
                               const float* shift, const float* scale, void* normed,
                               int S, int L, int D, float eps, h3_stream_t stream);

/*
 * a2 — per-head Q/K RMSNorm followed by rotary position embedding, in place
 * (blog section 3.2, #5990; RoPE rows from per-token positions, section 3.1).
 * For every valid row i, head h and x in {q, k} (gain g_q / g_k):
 *   y = x[i,h,:] / sqrt(mean(x[i,h,:]^2) + eps) * g
 *   head_dim is split into sections of axis_dims[0..2] channels for the
 *   positions pos[i,0..2] = (t, h, w); inside section a the channel pair
 *   (o_a + 2j, o_a + 2j + 1) is rotated counter-clockwise by
 *   pos[i,a] * theta^(-2j / axis_dims[a]).
 *   q, k    [S, H, Dh] bf16 (row stride H*Dh), in/out
 *   q_gain, k_gain [Dh] float32
 *   pos     [S, 3] int32
 *   axis_dims  HOST array of 3 even non-negative ints summing to Dh
 * Dh == 128. FP32 arithmetic; the angle is reduced exactly in fixed point
 * (turns = pos * theta^(-2j/d) / (2 pi) modulo 1 in 64-bit integer arithmetic,
 * the per-pair factor rounded to double) and its sin/cos taken in FP32.
 */
h3_status h3_qk_norm_rope(void* q, void* k, const float* q_gain, const float* k_gain,
                          const int32_t* pos, const int* axis_dims, int S, int L, int H,
                          int Dh, float theta, float eps, h3_stream_t stream);

/*
 * a2 with a choice of channel pairing (the pages fix RoPE per token but not
 * its channel layout; interleaved pairs are the reading the block uses by
 * default). pairing 0: pairs (o_a + 2j, o_a + 2j + 1), exactly
 * h3_qk_norm_rope. pairing 1: split-half pairs (o_a + j, o_a + d_a/2 + j)
 * inside each section, the same angle for pair j; every axis_dims[a] must
 * then be a multiple of 16 (H3_ERR_UNSUPPORTED otherwise). Other arguments
 * as h3_qk_norm_rope.
 */
h3_status h3_qk_norm_rope_layout(void* q, void* k, const float* q_gain, const float* k_gain,
                                 const int32_t* pos, const int* axis_dims, int S, int L, int H,
                                 int Dh, float theta, float eps, int pairing,
                                 h3_stream_t stream);

/*
 * a3 — dense bidirectional attention over the valid length (blog section 3.1:
 * the backend takes the valid sequence length; no work on tail padding):
 *   o[i,h,:] = sum_{j<L} softmax_j(q[i,h,:] . k[j,h,:] * softmax_scale) v[j,h,:]
 * for i < L. Keys/values of rows >= L are never read; rows >= L of o are not
 * written.
 *   q, k, v, o [S, H, Dh] bf16 with row stride H*Dh
 * Dh == 128. bf16 tensor-core products, FP32 softmax and accumulation, bf16 out.
 */
h3_status h3_attention_varlen(const void* q, const void* k, const void* v, void* o, int S,
                              int L, int H, int Dh, float softmax_scale, h3_stream_t stream);

/*
 * a3 with Skip-Softmax (next step after dense attention; blog section 4.3,
 * Fig. 6: skip the softmax and P x V of tiles the QK scores show to be
 * negligible, decided per tile). Keys are taken in tiles of 128 from key 0 and
 * queries in tiles of 128 from row 0. A key tile is left out for a query tile
 * when, for every valid row of that query tile, the tile's largest base-2
 * logit (score * softmax_scale * log2(e)) lies more than log2(1/skip_eps)
 * below the row's exact running maximum over the key tiles kept so far (rows
 * >= L of a ragged last query tile take no part). The first key tile is never
 * skipped; skip_eps == 0 is exactly h3_attention_varlen.
 *   kept_tiles  [ceil(L/128), H] int32 device, or NULL: receives the number of
 *               key tiles kept for every (query tile, head), the first one
 *               included (only with skip_eps > 0; left untouched otherwise)
 * Other arguments as h3_attention_varlen; 0 <= skip_eps < 1; kept_tiles
 * 4-byte aligned.
 */
h3_status h3_attention_varlen_skip(const void* q, const void* k, const void* v, void* o, int S,
                                   int L, int H, int Dh, float softmax_scale, float skip_eps,
                                   int32_t* kept_tiles, h3_stream_t stream);

/*
 * a3 with FP8 ("SAGE") products (next step; blog section 4.3: Q, K, P and V
 * quantised to FP8 for the QK and PV products). Two steps:
 *
 * h3_sage_quantize: K is smoothed by subtracting its per-(head, channel)
 * mean over the L valid keys (their exact sum, taken in 64-bit fixed point
 * for keys whose nonzero magnitudes lie in [2^-33, 2^14) and in FP64 for a
 * 512-row chunk holding any other value, rounded once to double, divided by
 * L in double and rounded to float32), Q and the smoothed K are
 * quantised to E4M3 per (128-row tile, head) block and V per (head, channel),
 * all with absmax scaling (inv = 448 / amax, code = E4M3_satfinite(x * inv),
 * scale = amax / 448, float32 steps).
 *   q, k, v   [S, H, Dh] bf16 (row stride H*Dh)
 *   qc, kc, vc [S, H, Dh] E4M3 codes (bytes); rows >= L are not written
 *   sq, sk    [ceil(L/128), H] float32; sv, k_mean [H, Dh] float32
 *   scratch   device memory of h3_sage_scratch_bytes(L, H) bytes, 16-byte
 *             aligned
 *
 * h3_attention_fp8: o[i] = sum_j E4M3(P_ij) * vc[j] * sv / sum_j P_ij with
 * P_ij = 224 * 2^(z_ij - m_i), z_ij = (qc_i . kc_j) * sq * sk * softmax_scale
 * * log2(e), m_i an integer running maximum kept in [max_j z_ij - 1,
 * ceil(max_j z_ij)] (the kernel sees the keys once, so it cannot scale P by
 * the exact row maximum). P_ij is therefore 448 * p_ij (p_ij = 2^(z_ij -
 * max_j z_ij), P scaled by its row absmax) times a per-row factor in
 * (1/4, 1], and its E4M3 rounding differs from that of 448 * p_ij by at most
 * half an E4M3 step on each side. tcgen05 kind::f8f6f4 for QK and PV, FP32
 * softmax and accumulation, bf16 out. Dh == 128.
 */
size_t h3_sage_scratch_bytes(int L, int H);
h3_status h3_sage_quantize(const void* q, const void* k, const void* v, int S, int L, int H,
                           int Dh, void* qc, void* kc, void* vc, float* sq, float* sk, float* sv,
                           float* k_mean, void* scratch, size_t scratch_bytes,
                           h3_stream_t stream);
h3_status h3_attention_fp8(const void* qc, const void* kc, const void* vc, const float* sq,
                           const float* sk, const float* sv, void* o, int S, int L, int H,
                           int Dh, float softmax_scale, h3_stream_t stream);

/*
 * h3_attention_fp8 with Skip-Softmax (blog section 4.3, Fig. 6: SAGE
 * quantisation and Skip-Softmax together): the tile rule of
 * h3_attention_varlen_skip applied to the FP8 logits z_ij of h3_attention_fp8
 * (a key tile is left out for a 128-row query tile when every valid row's
 * largest z in it lies more than log2(1/skip_eps) below the row's exact
 * running maximum of z over the key tiles kept so far; the first key tile is
 * never left out); the kept tiles are then handled as in h3_attention_fp8,
 * whose result skip_eps == 0 reproduces bit for bit.
 *   kept_tiles  [ceil(L/128), H] int32 device, or NULL: the number of key
 *               tiles kept for every (query tile, head) (only with
 *               skip_eps > 0; left untouched otherwise); 4-byte aligned
 * Other arguments as h3_attention_fp8; 0 <= skip_eps < 1.
 */
h3_status h3_attention_fp8_skip(const void* qc, const void* kc, const void* vc, const float* sq,
                                const float* sk, const float* sv, void* o, int S, int L, int H,
                                int Dh, float softmax_scale, float skip_eps, int32_t* kept_tiles,
                                h3_stream_t stream);

/*
 * a5 — SwiGLU (blog section 3.2, #6283): out[i,j] = SiLU(g) * u with
 * g = gate_up[i,j], u = gate_up[i,F+j], SiLU(g) = g / (1 + exp(-g)), for i < L.
 *   gate_up [S, 2F] bf16, out [S, F] bf16. F % 8 == 0.
 */
h3_status h3_swiglu(const void* gate_up, void* out, int S, int L, int F, h3_stream_t stream);

/*
 * a4 — one block projection (the matrix multiplies the fused ops of blog
 * section 3.2 sit around): y[i,:] = bf16( x[i,:] @ w^T ) for i < L, no bias.
 *   x [S, K] bf16, w [N, K] bf16 (row n = output channel n), y [S, N] bf16.
 * K % 64 == 0, N % 256 == 0. bf16 tensor-core products, FP32 accumulation.
 */
h3_status h3_linear(const void* x, const void* w, void* y, int S, int L, int N, int K,
                    h3_stream_t stream);

/*
 * a4 + a5 fused — the FFN gate/up projection with SwiGLU in its epilogue
 * (blog section 3.2: SwiGLU without separate SiLU and multiply launches):
 *   out[i,j] = SiLU(bf16(x[i,:] . w_gu[j,:])) * bf16(x[i,:] . w_gu[F+j,:])   for i < L
 *   x [S, K] bf16, w_gu [2F, K] bf16 (rows [gate | up]), out [S, F] bf16.
 * F % 128 == 0, K % 64 == 0. The two products are rounded to bf16 before the
 * SiLU, so the result equals h3_linear followed by h3_swiglu.
 */
h3_status h3_linear_swiglu(const void* x, const void* w_gu, void* out, int S, int L, int F,
                           int K, h3_stream_t stream);

/*
 * a2 inputs, precomputed — the (cos, sin) of every RoPE angle of rows < L
 * (blog section 3.2: Q/K RMSNorm and RoPE fused, here into the QKV
 * projection's epilogue, which reads this table):
 *   table[i, p] = (cos phi, sin phi), phi = pos[i, a] * theta^(-2j / axis_dims[a])
 * for channel pair p of a 128-channel head (section a, pair j within it, as in
 * h3_qk_norm_rope), angle reduced to turns modulo 1 in 64-bit fixed point as
 * h3_qk_norm_rope does it, cos/sin in FP32.
 *   pos   [S, 3] int32; axis_dims HOST [3], even, sum 128
 *   table [S, 64, 2] float32 (rows >= L not written)
 */
h3_status h3_rope_table(const int32_t* pos, const int* axis_dims, int S, int L, float theta,
                        float* table, h3_stream_t stream);

/*
 * a4 + a2 fused — the QKV projection with Q/K RMSNorm + RoPE in its epilogue
 * (blog section 3.2: the small ops around the projections fused):
 *   qkv[i, :] = bf16(x[i, :] @ w_qkv^T) for i < L, then every q head (columns
 *   [0, 128H)) and k head (columns [128H, 256H)) of row i is normalised,
 *   scaled by q_gain / k_gain and rotated with table row i exactly as
 *   h3_qk_norm_rope would do it; v columns are the plain product.
 *   x [S, K] bf16, w_qkv [384H, K] bf16, qkv [S, 384H] bf16
 *   q_gain, k_gain [128] float32; rope_table from h3_rope_table
 *   axis_dims HOST [3] (sum 128), pairing as h3_qk_norm_rope_layout
 * H even, K % 64 == 0. Equals h3_linear followed by h3_qk_norm_rope_layout up
 * to the order of the FP32 sum of squares inside the RMS.
 */
h3_status h3_linear_qk_norm_rope(const void* x, const void* w_qkv, void* qkv,
                                 const float* q_gain, const float* k_gain,
                                 const float* rope_table, const int* axis_dims, int pairing,
                                 int S, int L, int H, int K, float eps, h3_stream_t stream);

/*
 * a4 + a1 fused — a projection whose product goes straight into the FP32
 * residual stream (blog section 3.2: FP32 residual merged into the
 * surrounding ops):
 *   resid[i, n] = fma(gate[n], bf16(x[i, :] . w[n, :]), resid[i, n])   for i < L
 * which is h3_linear followed by the residual step of h3_mod_norm_residual,
 * bit for bit.
 *   x [S, K] bf16, w [N, K] bf16, resid [S, N] float32 in/out, gate [N] float32
 * N % 256 == 0, K % 64 == 0.
 */
h3_status h3_linear_residual(const void* x, const void* w, float* resid, const float* gate,
                             int S, int L, int N, int K, h3_stream_t stream);

/* Shape and constants of one block. */
typedef struct h3_block_config {
  int S;             /* buffer rows                                   */
  int L;             /* valid rows, 0 <= L <= S                       */
  int D;             /* hidden width, D == H * Dh                     */
  int H;             /* heads                                         */
  int Dh;            /* head dim (128)                                */
  int F;             /* SwiGLU inner width                            */
  int axis_dims[3];  /* RoPE sections (t, h, w), sum == Dh            */
  float theta;       /* RoPE base                                     */
  float eps_ln;      /* LayerNorm epsilon of the modulation steps     */
  float eps_qk;      /* Q/K RMSNorm epsilon                           */
  int rope_pairing;  /* 0 interleaved, 1 split-half (h3_qk_norm_rope_layout) */
} h3_block_config;

/* Block weights (device pointers, caller-owned). */
typedef struct h3_block_weights {
  const void* w_qkv;    /* [3D, D] bf16, rows [q | k | v], each head-major */
  const void* w_o;      /* [D, D]  bf16                                    */
  const void* w_gu;     /* [2F, D] bf16, rows [gate | up]                  */
  const void* w_down;   /* [D, F]  bf16                                    */
  const float* q_gain;  /* [Dh] float32                                    */
  const float* k_gain;  /* [Dh] float32                                    */
} h3_block_weights;

/* Bytes of device workspace h3_block_forward needs for this config
 * (0 when the config is invalid; h3_last_error() says why). */
size_t h3_block_workspace_bytes(const h3_block_config* cfg);

/*
 * a6 — one whole block (blog sections 3.1-3.2), in this order, rows < L:
 *   (shift1, scale1, gate1, shift2, scale2, gate2) = mod[0..5, :]
 *   h1 = bf16(LN(r) * (1 + scale1) + shift1)
 *   [q | k | v] = h1 @ w_qkv^T ; q, k <- RoPE(RMSNorm(.))      (per head)
 *   a  = attention(q, k, v) over keys < L, scale Dh^-1/2
 *   r <- r + gate1 * (a @ w_o^T)
 *   h2 = bf16(LN(r) * (1 + scale2) + shift2)
 *   [g | u] = h2 @ w_gu^T ; s = SiLU(g) * u
 *   r <- r + gate2 * (s @ w_down^T)
 *   resid [S, D] float32 in/out (the residual stream r)
 *   mod   [6, D] float32
 *   pos   [S, 3] int32
 *   workspace: device memory of at least h3_block_workspace_bytes(cfg) bytes,
 *   256-byte aligned, owned by the caller, overwritten by the call.
 * Q/K RMSNorm + RoPE run in the QKV projection's epilogue
 * (h3_linear_qk_norm_rope), SwiGLU in the gate/up projection's
 * (h3_linear_swiglu) and the last residual update in the down projection's
 * (h3_linear_residual).
 */
h3_status h3_block_forward(const h3_block_config* cfg, const h3_block_weights* w, float* resid,
                           const float* mod, const int32_t* pos, void* workspace,
                           size_t workspace_bytes, h3_stream_t stream);

/*
 * a1 with token-group modulation (next step after the per-sample form):
 * the pages denoise conditioning and noisy tokens and video and audio tokens
 * (with their own sigma schedules) in one packed sequence (blog section 1,
 * Fig. 1; H3 blog PR, dual schedules). Row i takes its gate, shift and scale
 * from group seg[i] of a table: group g's vectors are at gate + g*seg_stride,
 * shift + g*seg_stride, scale + g*seg_stride (floats). Otherwise as
 * h3_mod_norm_residual.
 *   seg  [S] int32 device, values in [0, num_seg) (values outside are clamped
 *        to that range, so reads stay inside the table)
 *   seg_stride  floats between groups, >= D, multiple of 4
 */
h3_status h3_mod_norm_residual_seg(float* resid, const void* delta, const float* gate,
                                   const float* shift, const float* scale, const int32_t* seg,
                                   int num_seg, int64_t seg_stride, void* normed, int S, int L,
                                   int D, float eps, h3_stream_t stream);

/*
 * A stack of num_blocks blocks applied in order to the residual stream, the
 * way the denoiser runs its transformer blocks in every forward (blog
 * section 5). Block b uses w[b] and the modulation table
 *   mod + b * num_seg * 6 * D      ([num_seg, 6, D] float32, per block)
 * and, when seg is not NULL, row i uses group seg[i] of that table (see
 * h3_mod_norm_residual_seg; seg NULL requires num_seg == 1). The residual
 * update that ends block b and the modulated LayerNorm that starts block
 * b + 1 run as one pass over the residual. One workspace of
 * h3_block_workspace_bytes(cfg) serves the whole stack. With num_blocks == 1,
 * num_seg == 1 and seg == NULL this is h3_block_forward.
 *   w    host array of num_blocks weight structs
 */
h3_status h3_stack_forward(const h3_block_config* cfg, const h3_block_weights* w,
                           int num_blocks, float* resid, const float* mod, int num_seg,
                           const int32_t* seg, const int32_t* pos, void* workspace,
                           size_t workspace_bytes, h3_stream_t stream);

/*
 * GPU output preparation (blog section 3.4; a stage next to the block): decoded
 * video frames [B, C, T, H, W] float32 become contiguous [B, T, H, W, C]
 * uint8, a quarter of the bytes, before they leave the GPU. Each value maps to
 *   round_half_even( clamp(x * 0.5 + 0.5, 0, 1) * 255 )
 * with every step rounded in float32 (no fused multiply-add); NaN maps to 0.
 *   frames  16-byte aligned; out 4-byte aligned; T*H*W % 4 == 0; 1 <= C <= 16
 */
h3_status h3_frames_to_u8(const float* frames, uint8_t* out, int B, int C, int T, int H, int W,
                          h3_stream_t stream);

/*
 * Online FP8 projections (next step after the BF16 block; blog section 4.3,
 * "online FP8": eligible linear layers get FP8 weights and scales once at
 * load time, their activations are quantised online). Format: E4M3 codes,
 * one float32 scale per row (per output channel for weights, per token for
 * activations); value = code * scale.
 *
 * h3_quantize_fp8_rows: x [R, K] bf16 -> q [R, K] E4M3 codes (bytes), scale
 * [R] float32, per row: amax = max|x|, inv = 448 / amax (0 if amax == 0),
 * q = E4M3_satfinite(x * inv) (round to nearest even), scale = amax / 448,
 * each step rounded in float32. K % 8 == 0, K <= 16384. Serves both the
 * load-time weight quantisation and the online activation quantisation.
 */
h3_status h3_quantize_fp8_rows(const void* x, void* q, float* scale, int R, int K,
                               h3_stream_t stream);

/*
 * y[i, :] = bf16( (qx[i, :] . qw[j, :]) * sx[i] * sw[j] ) for i < L: an FP8
 * projection on tcgen05 (kind::f8f6f4), FP32 accumulation.
 *   qx [S, K] codes, sx [S]; qw [N, K] codes, sw [N]; y [S, N] bf16.
 *   K % 128 == 0, N % 256 == 0.
 */
h3_status h3_linear_fp8(const void* qx, const float* sx, const void* qw, const float* sw, void* y,
                        int S, int L, int N, int K, h3_stream_t stream);

/* FP8 gate/up projection with SwiGLU in the epilogue: as h3_linear_swiglu with
 * FP8 operands (qw_gu [2F, K] codes with scales sw_gu [2F]); the two products
 * are scaled and rounded to bf16 before the SiLU. F % 128 == 0, K % 128 == 0. */
h3_status h3_linear_swiglu_fp8(const void* qx, const float* sx, const void* qw_gu,
                               const float* sw_gu, void* out, int S, int L, int F, int K,
                               h3_stream_t stream);

/* Block weights with FP8 projections (codes from h3_quantize_fp8_rows). */
typedef struct h3_block_weights_fp8 {
  const void* w_qkv;  const float* s_qkv;   /* [3D, D] codes, [3D] scales */
  const void* w_o;    const float* s_o;     /* [D, D], [D]                */
  const void* w_gu;   const float* s_gu;    /* [2F, D], [2F]              */
  const void* w_down; const float* s_down;  /* [D, F], [D]                */
  const float* q_gain;                      /* [Dh]                       */
  const float* k_gain;                      /* [Dh]                       */
} h3_block_weights_fp8;

/* Workspace for h3_block_forward_fp8 (0 when the config is invalid). */
size_t h3_block_workspace_bytes_fp8(const h3_block_config* cfg);

/* h3_block_forward with the four projections in FP8: every projection input
 * (h1, the attention output, h2, the SwiGLU output) is quantised per token
 * as h3_quantize_fp8_rows does it before its FP8 GEMM (h1 and h2 by the
 * modulated LayerNorm passes themselves, from their bf16-rounded rows, so no
 * bf16 copy of them is written). fp8_attention != 0 also runs
 * the attention in FP8 (h3_sage_quantize + h3_attention_fp8); otherwise the
 * attention and everything else (modulation, Q/K RMSNorm + RoPE, SwiGLU) is
 * the BF16/FP32 path. D % 128 == 0, F % 128 == 0 in addition to
 * h3_block_forward's limits. */
h3_status h3_block_forward_fp8(const h3_block_config* cfg, const h3_block_weights_fp8* w,
                               float* resid, const float* mod, const int32_t* pos,
                               int fp8_attention, void* workspace, size_t workspace_bytes,
                               h3_stream_t stream);

/* Number of stages h3_block_forward runs, in the order listed above:
 * 0 modulation+LN (and the RoPE table), 1 QKV projection with Q/K
 * RMSNorm+RoPE in its epilogue, 2 attention, 3 output projection,
 * 4 residual+modulation+LN, 5 gate/up projection with SwiGLU in its epilogue,
 * 6 down projection with the residual update in its epilogue. */
#define H3_BLOCK_STAGES 7

/*
 * h3_block_forward, and records events[i] on `stream` just before stage i is
 * launched and events[H3_BLOCK_STAGES] after the last stage, so the caller
 * can time every stage on the launching stream. events: host array of
 * H3_BLOCK_STAGES + 1 cudaEvent_t handles created by the caller (num_events
 * must equal that count). The kernels launched are the same as those of
 * h3_block_forward.
 */
h3_status h3_block_forward_events(const h3_block_config* cfg, const h3_block_weights* w,
                                  float* resid, const float* mod, const int32_t* pos,
                                  void* workspace, size_t workspace_bytes, h3_stream_t stream,
                                  void* const* events, int num_events);

/* Bytes of the fixed device scratch array h3_block_forward_noalloc uses. */
#define H3_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * h3_block_forward for callers that cannot allocate device memory. The source
 * pages have no counterpart: this entry point exists for callers, not for the
 * method.
 *
 * Some callers cannot give the library a workspace: a host program or
 * plug-in whose device memory all belongs to a framework's pool and which may
 * not call cudaMalloc itself, or code that runs where an allocation is not
 * allowed. This variant takes its scratch from one array of
 * H3_NOALLOC_SCRATCH_BYTES (32 MiB) in the library's own device memory
 * instead; that array is reserved on every GPU that loads the library and
 * stays reserved until the process exits.
 *  - It allocates nothing: no cudaMalloc, cudaFree or allocating library
 *    routine is called.
 *  - A block whose h3_block_workspace_bytes(cfg) exceeds
 *    H3_NOALLOC_SCRATCH_BYTES is rejected with H3_ERR_WORKSPACE before
 *    anything is launched (the full 58,816-row block needs 5.5 GB; this entry
 *    point serves short sequences such as 256 rows of a 512-wide block).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current. Make that first call
 *    before any stream capture.
 *  - Every call on a device shares the one array, which keeps the last
 *    call's contents. The block writes every scratch element before it reads
 *    it, so nothing has to start at zero. Calls whose work overlaps on the
 *    GPU (different streams, or different host threads) race on the array:
 *    order them on one stream.
 * Arguments, results and errors are otherwise those of h3_block_forward.
 */
h3_status h3_block_forward_noalloc(const h3_block_config* cfg, const h3_block_weights* w,
                                   float* resid, const float* mod, const int32_t* pos,
                                   h3_stream_t stream);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier no one arrives at, with a wait limit of timeout_ns. The wait runs
 * out, the kernel records its code and returns; h3_check_device_error() then
 * reports H3_ERR_TIMEOUT. Nothing else is touched. */
h3_status h3_debug_wait_timeout(uint64_t timeout_ns, h3_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* H3BLOCK_H_ */
