/*
 * dit.h - C ABI of the GB300 (sm_103a) AdaLN diffusion-transformer block library (libdit.so).
 *
 * The library computes the forward of one AdaLN DiT block over a packed [text L | image N]
 * sequence, its int8lin-weight variant, the FlowMatch Euler step and a stacked-block denoise loop,
 * entirely in CUDA kernels on the caller's stream.
 *
 * Sources, cited by page title and section:
 *   [host contract]  "Host contract - RGBA-Image-2.1-Turbo (Core AI port of Qwen-Image-2.1-Turbo)",
 *                    sections 1 (DiT graph I/O, int8lin weights), 4 (sequence layout, RoPE tables),
 *                    5 (latent packing), 6 (FlowMatch Euler sampler).
 *   [gizai:dit]      the "gizai:dit" module reference: Block.forward, normedInto, linearInto,
 *                    gatedInto, prepOf, gluRows, weightAt, sinusoids, Modulation, Sequence.
 *   [klein]          "944 -> 346 ms: optimizing FLUX.2 klein-4B on one TPU v6e chip", sections 2
 *                    (cast points), 4.3 (flash attention, 1/sqrt(d) in fp32), 4.4 (fused qk prep).
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller owns every buffer. The
 *     library allocates nothing on these paths (a one-time 4-byte error word per device aside).
 *   - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16).
 *   - Matrices are row-major and densely packed unless a stride is given. Weights are [out, in].
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *     Validation happens before any launch: a call that returns an error launched nothing and left
 *     every output untouched.
 *   - Calls that share a workspace must not overlap on the device.
 *   - Device-side waits are bounded: a stuck pipeline sets the device error word, the kernel frees
 *     what it holds and returns. dit_check() reports it as DIT_ETIMEOUT.
 *   - Per-device state is created on the first call that needs it and kept until the process
 *     exits: the device addresses of the library's static device arrays (the error word, the
 *     no-allocation scratch), the int8lin side stream and its events, kernel attributes. It is keyed
 *     by device ordinal, so it does not survive cudaDeviceReset(): after a reset the cached
 *     addresses and handles are stale, and the library must not be called again in that process.
 */
#ifndef DIT_H_
#define DIT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DIT_API __attribute__((visibility("default")))
#else
#define DIT_API
#endif

typedef struct CUstream_st* dit_stream_t; /* same type as cudaStream_t */

/* Status codes. */
#define DIT_OK 0
#define DIT_EINVAL (-1)       /* null pointer, bad size, misaligned pointer (16 bytes for TMA operands) */
#define DIT_EUNSUPPORTED (-2) /* shape outside what the kernels implement (see each call) */
#define DIT_EWORKSPACE (-3)   /* workspace null or smaller than dit_workspace_bytes() */
#define DIT_ECUDA (-4)        /* a CUDA launch or runtime call failed */
#define DIT_ETIMEOUT (-5)     /* a bounded device wait gave up (reported by dit_check) */

/* Block dimensions. hidden H, heads nh, head_dim d = H / nh, ffn F.
 * Supported: d in {64, 128}; H % 256 == 0; F % 128 == 0. [gizai:dit, Arch]
 * rope_split selects the rotary layout of q and k:
 *   0: adjacent pairs (2i, 2i+1) over the whole head, tables [rows, d/2] [host contract, section 4]
 *   1: split halves over the first 3/4 of the head: values i and i + 3d/8 (i < 3d/8) turned by
 *      angle i, the last d/4 values unrotated, tables [rows, 3d/8] [gizai:dit, prepOf, HEAD] */
typedef struct {
  int hidden;
  int heads;
  int head_dim;
  int ffn;
  float eps;      /* modulated RMSNorm epsilon (1e-6 in every workload) */
  float qk_eps;   /* per-head query/key RMSNorm epsilon */
  int rope_split; /* 0 or 1, see above */
} dit_dims;

/* bf16 weights of one block. [gizai:dit, Block (indexes QKV, OUT, UP, DOWN, NORM1, NORM2, Q_NORM, K_NORM)]
 *   wqkv  [3H, H]: rows all queries, then all keys, then all values; head-major inside each
 *                  [gizai:dit, weightAt]
 *   wout  [H, H]
 *   wup   [2F, H]: gate row j at 2j, up row j at 2j + 1 [gizai:dit, gluRows]
 *   wdown [H, F]
 *   norm1, norm2 [H] fp32 affine weights of the two modulated norms, or NULL for ones
 *   q_norm, k_norm [d] fp32 head-norm weights, or NULL for ones
 * Weight pointers must be 16-byte aligned. */
typedef struct {
  const uint16_t* wqkv;
  const uint16_t* wout;
  const uint16_t* wup;
  const uint16_t* wdown;
  const float* norm1;
  const float* norm2;
  const float* q_norm;
  const float* k_norm;
} dit_block_w;

/* int8lin weights of one block [host contract, section 1]: each linear (0 qkv, 1 out, 2 up, 3 down)
 * as symmetric int8 values q [out, in] and one bf16 scale per 32 consecutive input elements
 * s [out, in / 32]; the weight is W[o, i] = bf16_rne(q[o, i] * s[o, i / 32]). Row orders as in
 * dit_block_w. Norm weights as in dit_block_w. */
typedef struct {
  const int8_t* q[4];
  const uint16_t* s[4];
  const float* norm1;
  const float* norm2;
  const float* q_norm;
  const float* k_norm;
} dit_block_w8;

/* W8A8 weights of one block [klein, section 5 (int8 detail) and its D4/D5 entries]: each linear
 * (0 qkv, 1 out, 2 up, 3 down) as symmetric int8 codes q [out, in] with one fp32 scale per output
 * channel, scale [out] (absmax / 127, as dit_w8a8_quantize_weight makes them), and an optional
 * SmoothQuant divisor smooth [in] (NULL: none) that was folded into the weight before its
 * quantisation and divides the activation before its per-token quantisation. Row orders and norm
 * weights as in dit_block_w. */
typedef struct {
  const int8_t* q[4];
  const float* scale[4];
  const float* smooth[4];
  const float* norm1;
  const float* norm2;
  const float* q_norm;
  const float* k_norm;
} dit_block_w8a8;

/* Modulation rows [gizai:dit, Modulation and Sequence.map]: rows [M, 6, H] fp32 holding, for each
 * modulation row, shift_a, scale_a, gate_a (attention) then shift_m, scale_m, gate_m (MLP).
 * map [L + N] int32 gives each packed row's modulation row (0 <= map[r] < M); NULL means row 0. */
typedef struct {
  const float* rows;
  const int32_t* map;
  int M;
} dit_mod;

/* LoRA adapters of a block's four linears [gizai:dit, Block (lora), loraOf, withLora, weightAt]:
 * for linear i (0 qkv, 1 out, 2 up, 3 down) with in_i inputs and out_i outputs, A[i] [rank, in_i]
 * and B[i] [out_i, rank] bf16 row-major; the linear becomes x W^T + (x A^T) B^T, the map of the
 * merged weight W + B A. A[i] = B[i] = NULL: no adapter on that linear. rank % 8 == 0,
 * 8 <= rank <= 1024. The caller owns the tensors. */
typedef struct {
  const uint16_t* A[4];
  const uint16_t* B[4];
  int rank;
} dit_lora;

/* ---------------------------------------------------------------------------------------------
 * Whole-block forward [gizai:dit, Block.forward]. For packed rows r = 0..L+N-1 (row r < L is
 * txt[r], else img[r - L]) and m = map[r]:
 *   h  = modnorm(x; norm1, shift_a, scale_a)      x * rsqrt(mean(x^2) + eps) * w * (1 + scale) + shift
 *   q,k,v = h Wqkv^T; per head q,k <- rmsnorm(.) * q_norm/k_norm, then rotated in adjacent pairs
 *           (2i, 2i+1) by the row's angle i (cos/sin tables) [host contract, section 4]
 *   o  = softmax(q k^T / sqrt(d)) v over all L+N rows, per head (no mask) [klein, section 4.3]
 *   x += gate_a * (o Wout^T)                      [gizai:dit, gatedInto]
 *   h2 = modnorm(x; norm2, shift_m, scale_m)
 *   x += gate_m * ((silu(h2 Wup_gate^T) * (h2 Wup_up^T)) Wdown^T)
 * txt [L, H] and img [N, H] fp32 are the residual stream, updated in place. L >= 0, N >= 1.
 * txt_cos/txt_sin [L, d/2] and img_cos/img_sin [N, d/2] fp32 are the per-row rotary tables
 * (dit_rope_tables builds them). GEMM operands are bf16 with fp32 accumulation; norms, softmax and
 * residual updates are fp32. ws: device workspace of at least dit_workspace_bytes(dims, L, N, 0)
 * bytes, 256-byte aligned. Errors: DIT_EINVAL, DIT_EUNSUPPORTED, DIT_EWORKSPACE, DIT_ECUDA.
 * ------------------------------------------------------------------------------------------- */
DIT_API int dit_block_forward(const dit_dims* dims, const dit_block_w* w, float* txt, int L, float* img, int N,
                      const float* txt_cos, const float* txt_sin, const float* img_cos, const float* img_sin,
                      const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream);

/* LoRA merge [gizai:dit, weightAt and loadBlock: a BF16 block's linear is loaded with its adapter's
 * update added, W + B A]: merged[o, i] = bf16_rne(W[o, i] + sum_r B[o, r] A[r, i]) for W [n_out, n_in],
 * A [rank, n_in], B [n_out, rank], all bf16 row-major (device). The sum over r is an fp32 FMA chain
 * in rank order (each product of two bf16 values is exact in fp32), W is added in fp32, then one
 * rounding to bf16, so a result differs from the rounding of the exact value only where that value
 * lies within the fp32 sum's rounding error of a bf16 rounding boundary. merged may be W itself (in
 * place) but must not otherwise overlap the inputs. The merged weights then serve any block form
 * (sequential, parallel, double-stream) with no adapter work per call. Errors: DIT_EINVAL for null
 * pointers or sizes < 1. */
DIT_API int dit_lora_merge(const uint16_t* W, int n_out, int n_in, const uint16_t* A, const uint16_t* B, int rank,
                           uint16_t* merged, dit_stream_t stream);

/* The bf16 block with LoRA adapters beside its linears (dit_lora): each adapted linear runs as
 * one GEMM for down = x A^T (bf16, [R, rank rounded up to 64], in the workspace) and the linear's
 * GEMM over [x | down] [W | B]^T with its usual epilogue (QK norm + rotary, gated residual, SwiGLU).
 * Workspace: dit_lora_workspace_bytes(dims, L, N, rank). Otherwise as dit_block_forward. */
DIT_API int dit_block_forward_lora(const dit_dims* dims, const dit_block_w* w, const dit_lora* lora, float* txt,
                                   int L, float* img, int N, const float* txt_cos, const float* txt_sin,
                                   const float* img_cos, const float* img_sin, const dit_mod* mod, void* ws,
                                   size_t ws_bytes, dit_stream_t stream);

/* The parallel and the double-stream blocks with LoRA adapters beside their linears [gizai:dit,
 * Block.parallel; withLora, loraOf, weightAt; klein article, sections 4.3-4.4 (double blocks)]:
 * each adapted linear runs as in dit_block_forward_lora (down = x A^T, then [x | down] [W | B]^T with
 * its usual epilogue). The parallel block then runs its four linears one by one (its fused GEMMs take
 * no per-part adapter factor), both output linears adding gate * (their product) to x; mod rows
 * [M, 3, H] as dit_parallel_block_forward. The double-stream block runs per stream, the text rows'
 * linears with lora_txt and the image rows' with lora_img (either may be NULL: no adapters on that
 * stream, but not both; lora_txt is ignored when L = 0). Workspace: dit_lora_workspace_bytes(dims,
 * L, N, rank) with the larger rank of the two sets. Otherwise as dit_parallel_block_forward and
 * dit_double_block_forward. */
DIT_API int dit_parallel_block_forward_lora(const dit_dims* dims, const dit_block_w* w, const dit_lora* lora,
                                            float* txt, int L, float* img, int N, const float* txt_cos,
                                            const float* txt_sin, const float* img_cos, const float* img_sin,
                                            const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream);
DIT_API int dit_double_block_forward_lora(const dit_dims* dims, const dit_block_w* w_txt, const dit_lora* lora_txt,
                                          const dit_block_w* w_img, const dit_lora* lora_img, float* txt, int L,
                                          float* img, int N, const float* txt_cos, const float* txt_sin,
                                          const float* img_cos, const float* img_sin, const dit_mod* mod, void* ws,
                                          size_t ws_bytes, dit_stream_t stream);
DIT_API size_t dit_lora_workspace_bytes(const dit_dims* dims, int L, int N, int rank);

/* The sandwich block [gizai:dit, POST_ATTN, POST_MLP]: dit_block_forward whose attention and MLP
 * outputs are normed before their gates: x += gate_a * rmsnorm(o Wout^T) * post_attn and
 * x += gate_m * rmsnorm(a Wdown^T) * post_mlp, rmsnorm(y) = y * rsqrt(mean(y^2) + eps) (dims.eps).
 * post_attn / post_mlp: [H] fp32, or NULL for a branch added as it is. Each normed branch runs as
 * its linear with an fp32 store and a row kernel for the norm and the residual (9 launches with
 * both). Workspace: dit_workspace_bytes(dims, L, N, 0). Otherwise as dit_block_forward. */
DIT_API int dit_block_forward_sandwich(const dit_dims* dims, const dit_block_w* w, const float* post_attn,
                                       const float* post_mlp, float* txt, int L, float* img, int N,
                                       const float* txt_cos, const float* txt_sin, const float* img_cos,
                                       const float* img_sin, const dit_mod* mod, void* ws, size_t ws_bytes,
                                       dit_stream_t stream);

/* The parallel and the double-stream sandwich blocks [gizai:dit, POST_ATTN, POST_MLP; Block.parallel;
 * klein article, sections 4.3-4.4]: branch outputs RMS-normed (the block's eps) times their post
 * weights ([H] fp32) before their gates. Parallel: x += gate * (rmsnorm(o Wout^T) post_attn +
 * rmsnorm(a Wdown^T) post_mlp), the one gate over both normed branches (a NULL weight leaves that
 * branch un-normed); the two output products are stored in fp32 and a row kernel applies the norms,
 * gate and residual. Double-stream: each stream's branches normed with that stream's weights
 * (post_*_txt for the text rows, post_*_img for the image rows; NULL: that stream's branch
 * un-normed). Workspace and other arguments as dit_parallel_block_forward / dit_double_block_forward
 * (variants 2 / 3). */
DIT_API int dit_parallel_block_forward_sandwich(const dit_dims* dims, const dit_block_w* w, const float* post_attn,
                                                const float* post_mlp, float* txt, int L, float* img, int N,
                                                const float* txt_cos, const float* txt_sin, const float* img_cos,
                                                const float* img_sin, const dit_mod* mod, void* ws, size_t ws_bytes,
                                                dit_stream_t stream);
DIT_API int dit_double_block_forward_sandwich(const dit_dims* dims, const dit_block_w* w_txt,
                                              const float* post_attn_txt, const float* post_mlp_txt,
                                              const dit_block_w* w_img, const float* post_attn_img,
                                              const float* post_mlp_img, float* txt, int L, float* img, int N,
                                              const float* txt_cos, const float* txt_sin, const float* img_cos,
                                              const float* img_sin, const dit_mod* mod, void* ws, size_t ws_bytes,
                                              dit_stream_t stream);

/* The same block with int8lin weights [host contract, section 1]: W = bf16_rne(q * s), then the
 * bf16 MMA. With at most 512 rows the GEMM's converter warps dequantize each weight k-block inside
 * the mainloop; with more rows (many M tiles per weight tile) each linear's weight is dequantized
 * once into the workspace by an HBM-bound kernel with the same arithmetic and the bf16 mainloop
 * runs on it (bitwise the same result). Those dequantizations run on a library-owned second stream
 * (created once per device), each one linear ahead into alternating workspace slots, forked from
 * and joined back to `stream` through events, so they overlap the previous linear's kernels; all
 * work stays ordered with respect to `stream`. Requires in % 256 == 0 for every linear.
 * Workspace: dit_workspace_bytes(dims, L, N, 1) (the bf16 block workspace plus two slots, each the
 * dequantized weight of the largest linear). */
DIT_API int dit_block_forward_int8(const dit_dims* dims, const dit_block_w8* w, float* txt, int L, float* img, int N,
                           const float* txt_cos, const float* txt_sin, const float* img_cos,
                           const float* img_sin, const dit_mod* mod, void* ws, size_t ws_bytes,
                           dit_stream_t stream);

/* The block with W8A8 linears (an opt-in lossy tier on the pages [klein, section 5]): before each
 * linear its activation (h, o, h2, a) is quantised per token, codes = clip(rint(v / s_r), -127, 127)
 * with s_r = max |v / smooth| / 127 over the row (float32, IEEE division, ties to even; a zero row has
 * scale 0), and the linear is the integer dot product of the codes times s_r times the weight's
 * per-channel scale, then the linear's usual epilogue. The codes are multiplied exactly on the bf16
 * tensor cores (integers up to 127 are bf16 values, their products fp32 values); the fp32
 * accumulation is exact while every partial sum stays below 2^24 in magnitude. The int8 weight codes
 * are widened to bf16 on a library-owned second stream one linear ahead (as in
 * dit_block_forward_int8). Workspace: dit_workspace_bytes(dims, L, N, 4). Errors as
 * dit_block_forward. */
DIT_API int dit_block_forward_w8a8(const dit_dims* dims, const dit_block_w8a8* w, float* txt, int L, float* img,
                                   int N, const float* txt_cos, const float* txt_sin, const float* img_cos,
                                   const float* img_sin, const dit_mod* mod, void* ws, size_t ws_bytes,
                                   dit_stream_t stream);

/* W8A8 weight quantisation [klein, D4 quantize_weight, D5 quantize_weight_smooth]: w bf16 [N, K]
 * (rows = output channels), smooth [K] fp32 or NULL: w' = fp32(w * smooth) (the fold), scale[n] =
 * max_k |w'[n, k]| / 127, q = clip(rint(w' / scale), -127, 127) int8 [N, K] (float32 decisions as in
 * dit_block_forward_w8a8). */
DIT_API int dit_w8a8_quantize_weight(const uint16_t* w, int N, int K, const float* smooth, int8_t* q, float* scale,
                                     dit_stream_t stream);

/* Per-token quantisation in place [klein, D4 quantize_rows]: x bf16 [R, K] (K % 8 == 0, 16-byte
 * aligned) is replaced by its codes (as bf16 integers), scale [R] fp32 receives the row scales. */
DIT_API int dit_w8a8_quantize_rows(uint16_t* x, int R, int K, const float* smooth, float* scale, dit_stream_t stream);

/* One W8A8 linear, fp32 out [M, N] = codes(a) codes(W)^T * s_a[row] * scale[col] (a bf16 [M, K] is not
 * modified; its codes go to the workspace). K and N multiples of 64.
 * Workspace: dit_linear_w8a8_workspace_bytes(M, N, K), 256-byte aligned. */
DIT_API int dit_linear_w8a8(const uint16_t* a, int M, int K, const int8_t* q, const float* scale, const float* smooth,
                            int N, float* out, void* ws, size_t ws_bytes, dit_stream_t stream);
DIT_API size_t dit_linear_w8a8_workspace_bytes(int M, int N, int K);

/* The parallel (single-stream) block [gizai:dit, Block.parallel]: x + gate * (attention + SwiGLU
 * MLP), both branches reading one modulated LayerNorm of x:
 *   h  = (x - mean(x)) * rsqrt(var(x) + eps) * norm1 * (1 + scale) + shift     (var biased, fp32)
 *   q,k,v = h Wqkv^T with the per-head QK norm and rotation of dit_block_forward
 *   o  = softmax(q k^T / sqrt(d)) v;   a = silu(h Wup_gate^T) * (h Wup_up^T) (interleaved rows)
 *   x += gate * (o Wout^T + a Wdown^T)
 * Weights as dit_block_forward (w->norm2 unused). mod->rows is [M, 3, H] fp32 here: shift, scale,
 * gate; map as dit_mod. The QKV and gate/up products run as one GEMM over [Wqkv ; Wup] and the
 * two output products as one GEMM over [o | a] [Wout | Wdown]^T (same arithmetic, fewer launches).
 * Workspace: dit_workspace_bytes(dims, L, N, 2), 256-byte aligned. Requires H % 256 == 0 and
 * ffn % 128 == 0 besides the dims rules. Errors as dit_block_forward. */
DIT_API int dit_parallel_block_forward(const dit_dims* dims, const dit_block_w* w, float* txt, int L, float* img,
                                       int N, const float* txt_cos, const float* txt_sin, const float* img_cos,
                                       const float* img_sin, const dit_mod* mod, void* ws, size_t ws_bytes,
                                       dit_stream_t stream);

/* The double-stream block [klein article, sections 4.3-4.4: the double blocks' per-stream
 * projections with the [txt | img] join on the prepared q, k, v]: dit_block_forward in which the
 * text rows [0, L) use w_txt and the image rows use w_img (all four linears and the four norm
 * weights), while the attention is one softmax over all L + N rows. mod as dit_block_forward
 * ([M, 6, H] and map): the map gives each stream its own modulation rows. w_txt may be NULL when
 * L = 0. With both streams present each norm and linear is one launch over all rows, the image
 * weights taken from row L on, each stream's rows padded to whole GEMM tiles when L is not on a tile
 * boundary, so no tile mixes the streams (7 launches); with one stream empty its norms and linears
 * run over the other's rows only. Any L works.
 * Workspace: dit_workspace_bytes(dims, L, N, 3).
 * Errors as dit_block_forward. */
DIT_API int dit_double_block_forward(const dit_dims* dims, const dit_block_w* w_txt, const dit_block_w* w_img,
                                     float* txt, int L, float* img, int N, const float* txt_cos,
                                     const float* txt_sin, const float* img_cos, const float* img_sin,
                                     const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream);

/* The int8lin forms of the parallel and the double-stream blocks [host contract, section 1 (the
 * int8 weight format); gizai:dit, Block.parallel; klein article, sections 4.3-4.4]: the blocks above
 * with every linear given as int8 values and bf16 block-32 scales (dit_block_w8), W = bf16_rne(q s).
 * Each weight is dequantised once per call, whatever the row count, on a library-owned second stream
 * that forks from and joins `stream` (as dit_block_forward_int8 does above 512 rows): for the
 * parallel block [Wqkv ; Wup] into one scratch slot while the norm runs, then Wout and Wdown into a
 * second while the first GEMM runs; for the double-stream block each linear's text and image
 * weights into one of two alternating slots, one linear ahead of its GEMM. The GEMMs are those of
 * the bf16 blocks on the dequantised weights, so each output equals the bf16 block's on
 * dit_dequant_int8 of the same weights bit for bit. Norm weights from the dit_block_w8 structs;
 * w_txt may be NULL when L = 0. Requires H % 256 == 0 and ffn % 256 == 0 besides the dims rules.
 * Workspace: dit_workspace_bytes(dims, L, N, 5) (parallel) and (dims, L, N, 6) (double-stream).
 * Errors as dit_block_forward. */
DIT_API int dit_parallel_block_forward_int8(const dit_dims* dims, const dit_block_w8* w, float* txt, int L,
                                            float* img, int N, const float* txt_cos, const float* txt_sin,
                                            const float* img_cos, const float* img_sin, const dit_mod* mod,
                                            void* ws, size_t ws_bytes, dit_stream_t stream);
DIT_API int dit_double_block_forward_int8(const dit_dims* dims, const dit_block_w8* w_txt,
                                          const dit_block_w8* w_img, float* txt, int L, float* img, int N,
                                          const float* txt_cos, const float* txt_sin, const float* img_cos,
                                          const float* img_sin, const dit_mod* mod, void* ws, size_t ws_bytes,
                                          dit_stream_t stream);

/* W8A8 weights of the parallel block [klein, section 5 (int8 detail: a single block's linear1 and
 * linear2) and its D4 / D5 entries]: linear1 = [Wqkv ; Wup] as one weight q1 [3H + 2F, H] (rows
 * all-Q, all-K, all-V, then the gate/up rows interleaved) and linear2 = [Wout | Wdown] as one weight
 * q2 [H, H + F] (inputs: the attention output's H, then the SwiGLU output's F), each quantised per
 * output channel over its whole row (dit_w8a8_quantize_weight of the joined matrix, after the fold
 * of its divisors), scale1 [3H + 2F] and scale2 [H] fp32; smooth1 [H] and smooth2 [H + F] fp32 the
 * SmoothQuant divisors used for them, or NULL. norm1, q_norm, k_norm as in dit_block_w. */
typedef struct {
  const int8_t* q1;
  const float* scale1;
  const float* smooth1;
  const int8_t* q2;
  const float* scale2;
  const float* smooth2;
  const float* norm1;
  const float* q_norm;
  const float* k_norm;
} dit_parallel_w8a8;

/* The W8A8 forms of the parallel and the double-stream blocks (an opt-in lossy tier, as for
 * dit_block_forward_w8a8) [klein, section 5 and its D4 / D5 entries]. Parallel: h (the modulated
 * LayerNorm's bf16 rows) is quantised per token (after the division by smooth1) and multiplied with
 * linear1's codes, the accumulator scaled by both scales before the QK-norm/rotary and SwiGLU
 * epilogues; the attention output o and the SwiGLU output a are quantised per token as one joined
 * row [o | a] (divisors smooth2) and multiplied with linear2's codes before the gated residual.
 * Double-stream: each stream's four linears are W8A8 linears with that stream's weights, scales
 * and divisors (w_txt for the text rows [0, L), w_img for the image rows; w_txt may be NULL when
 * L = 0), each activation quantised per token with its own stream's divisors. Weight codes are
 * widened to bf16 on the library's second stream one linear ahead; the integer dot products are
 * exact on the bf16 tensor cores while every partial sum stays below 2^24 in magnitude.
 * Workspace: dit_workspace_bytes(dims, L, N, 7) (parallel) and (dims, L, N, 8) (double-stream).
 * Requires H % 256 == 0 and ffn % 256 == 0 besides the dims rules. Errors as dit_block_forward. */
DIT_API int dit_parallel_block_forward_w8a8(const dit_dims* dims, const dit_parallel_w8a8* w, float* txt, int L,
                                            float* img, int N, const float* txt_cos, const float* txt_sin,
                                            const float* img_cos, const float* img_sin, const dit_mod* mod,
                                            void* ws, size_t ws_bytes, dit_stream_t stream);
DIT_API int dit_double_block_forward_w8a8(const dit_dims* dims, const dit_block_w8a8* w_txt,
                                          const dit_block_w8a8* w_img, float* txt, int L, float* img, int N,
                                          const float* txt_cos, const float* txt_sin, const float* img_cos,
                                          const float* img_sin, const dit_mod* mod, void* ws, size_t ws_bytes,
                                          dit_stream_t stream);

/* FlowMatch Euler step [host contract, section 6]: x[i] <- x[i] + (sigma_next - sigma) * vel[i],
 * each operation rounded separately in fp32 (no fused multiply-add). n >= 0. */
DIT_API int dit_euler_step(float* x, const float* vel, int64_t n, float sigma, float sigma_next, dit_stream_t stream);

/* Per-row rotary tables [host contract, section 4] for the packed sequence of L text tokens and an
 * h x w image grid: text token i at position (i, i, i), image token (y, x) at
 * (L, y - (h - h/2), x - (w - w/2)). Axis widths (16, 56, 56) for d = 128, (8, 28, 28) for d = 64;
 * column k of axis a holds the angle pos_a * theta^(-2k / width_a), evaluated in fp64 and rounded
 * once to fp32. cos, sin: device [L + h*w, d/2] fp32 (text rows first). */
DIT_API int dit_rope_tables(int L, int grid_h, int grid_w, int head_dim, float theta, float* cos, float* sin,
                    dit_stream_t stream);

/* Denoise model: the 32 (or `blocks`) stacked blocks plus the plain DiT around them.
 *   w_in   [H, C] bf16    patch-in of the packed latent tokens (C = latent_channels)
 *   w_t1   [H, 256] bf16  time MLP first linear;  w_t2 [H, H] bf16 second linear
 *   w_ada  [blocks, 6H, H] bf16  per-block modulation linear (shift_a, scale_a, gate_a, shift_m,
 *                                scale_m, gate_m); w_ada_f [2H, H] final norm (shift, scale)
 *   w_out  [C, H] bf16    patch-out to velocity
 *   block  [blocks]       the blocks' linears and norm weights (host array of device pointers)
 * No biases. Time embedding: temb = w_t2 silu(w_t1 [cos | sin](1000 t f_k)), f_k = 10000^(-k/128)
 * [gizai:dit, sinusoids]; every modulation is computed from silu(temb) with M = 1. */
typedef struct {
  dit_dims dims;
  int blocks;
  int latent_channels;
  const uint16_t* w_in;
  const uint16_t* w_t1;
  const uint16_t* w_t2;
  const uint16_t* w_ada;
  const uint16_t* w_ada_f;
  const uint16_t* w_out;
  const dit_block_w* block; /* HOST array of `blocks` descriptors */
} dit_model;

/* Full denoise loop [host contract, section 6] for `steps` Euler steps over sigmas[0..steps]
 * (HOST array, fp32): for each step i with t = sigmas[i], rows = [txt_feats ; x w_in^T] go through
 * every block, vel = modnorm(image rows; shift_f, scale_f) w_out^T, then
 * x <- x + (sigmas[i+1] - sigmas[i]) vel in fp32. x (img_tokens [N, C] fp32, device) holds the
 * packed noise on entry and the result on return. txt_feats [L, H] fp32. Rotary tables as in
 * dit_block_forward. The step-invariant work (time embeddings and every block's modulation for all
 * steps) is computed once up front. Any L >= 0 and N >= 1 (the host contract's graphs take
 * L = 8..512, N = 64..4096). Workspace: dit_denoise_workspace_bytes(). */
DIT_API int dit_denoise(const dit_model* model, float* img_tokens, int N, const float* txt_feats, int L,
                const float* sigmas, int steps, const float* txt_cos, const float* txt_sin,
                const float* img_cos, const float* img_sin, void* ws, size_t ws_bytes, dit_stream_t stream);

/* Workspace sizes. variant 0 = bf16 block, 1 = int8lin block, 2 = parallel block, 3 = double-stream
 * block, 4 = W8A8 block, 5 = int8lin parallel block, 6 = int8lin double-stream block, 7 = W8A8
 * parallel block, 8 = W8A8 double-stream block. Returns 0 for unsupported dims. */
DIT_API size_t dit_workspace_bytes(const dit_dims* dims, int L, int N, int variant);
DIT_API size_t dit_denoise_workspace_bytes(const dit_model* model, int L, int N, int steps);

/* Step-level entry points: each runs one step of the block forward on its own. The whole-block
 * calls above are sequences of these. ------------------------------------------------------ */

/* Modulated RMSNorm [gizai:dit, normedInto]: h[r] = bf16(x[r] * rsqrt(mean(x[r]^2) + eps) * w *
 * (1 + scale) + shift) with shift/scale the attention (which = 0) or MLP (which = 1) pair of
 * modulation row map[r]. h [L + N, H] bf16. w [H] or NULL. */
DIT_API int dit_modnorm(const dit_dims* dims, const float* txt, int L, const float* img, int N, const float* w,
                const dit_mod* mod, int which, uint16_t* h, dit_stream_t stream);

/* Stream-K scratch (no counterpart on the pages: a scheduling device of this library). The linears
 * below that take `ws` / `ws_bytes` run stream-K when their output tiles do not fill a whole number
 * of waves over the SMs and the scratch holds dit_stream_k_workspace_bytes(): the k-blocks of the
 * last tiles are divided evenly over all work units, each unit's share of a tile goes to the
 * scratch as an fp32 partial sum, and the unit that delivers a tile's last share adds the shares
 * in a fixed order and runs the epilogue (the result does not depend on timing; it differs from
 * the whole-tile result by the order of fp32 additions only). ws may be NULL (every tile whole);
 * when given it must be 256-byte aligned and not overlap the call's other buffers. The block calls
 * run their linears on whole tiles: on a GB300 at its power limit the partial sums cost energy and
 * bought no time (the GEMMs run at clocks the power limit sets, so an idle tail wave is not lost
 * time the way it is at a fixed clock). */
DIT_API size_t dit_stream_k_workspace_bytes(void);

/* QKV linear with its fused epilogue [gizai:dit, prepOf; klein, section 4.4]: qkv = h Wqkv^T;
 * q and k heads RMS-normed (times q_norm / k_norm, NULL = ones) then rotated by the tables;
 * stored bf16 as q, k [heads, R, d] (R = L + N) and v transposed as vt [heads, d, Rp] with
 * Rp = dit_vt_stride(R) (columns >= R unused). h [R, H] bf16. ws / ws_bytes: optional stream-K
 * scratch (see dit_stream_k_workspace_bytes). */
DIT_API int dit_qkv_rope(const dit_dims* dims, const uint16_t* h, int L, int N, const uint16_t* wqkv,
                 const float* q_norm, const float* k_norm, const float* txt_cos, const float* txt_sin,
                 const float* img_cos, const float* img_sin, uint16_t* q, uint16_t* k, uint16_t* vt,
                 void* ws, size_t ws_bytes, dit_stream_t stream);
DIT_API int dit_vt_stride(int R);

/* Joint attention [klein, section 4.3]: o[r, n*d + j] = sum_c softmax_c(q_n[r] . k_n[c] / sqrt(d))
 * vt_n[j, c] over all R rows, bf16 out [R, heads * d]. Layouts as dit_qkv_rope writes them.
 * ws / ws_bytes: optional scratch (16-byte aligned, not overlapping the other buffers) of at least
 * dit_attention_workspace_bytes(dims, R); NULL = one CTA per (pair of 128-row query tiles, head). */
DIT_API int dit_attention(const dit_dims* dims, int R, const uint16_t* q, const uint16_t* k, const uint16_t* vt,
                  uint16_t* o, void* ws, size_t ws_bytes, dit_stream_t stream);

/* Scratch for the persistent attention schedule (no counterpart on the pages: a scheduling device of
 * this library), 0 when it is not used for this shape. When the (query-tile pair, head) units leave
 * the last wave over the SMs part-empty, one CTA per SM takes an equal share of all the units' key
 * tiles; a unit cut between two CTAs is finished by the one holding its first key tiles, which
 * starts from the unnormalised output, row sum (and running maximum) the other left in the scratch
 * (133 KB per CTA at d = 128). The result does not depend on timing; it differs from the unscheduled
 * one in the cut units only: by the order of fp32 additions under the fixed maximum (within one bf16
 * step), by the bf16 rounding of each part's weights against its own maximum under a running one.
 * The block calls lend their h rows for it. Requires dims and R valid (else 0); reads the SM count
 * of the current device. */
DIT_API size_t dit_attention_workspace_bytes(const dit_dims* dims, int R);

/* The same attention for q and k rows as dit_qkv_rope writes them: RMS-normalised per head and
 * scaled by q_norm / k_norm ([d] fp32 each, NULL = ones; the caller vouches for this, the kernel
 * does not check it). Every scaled score then lies within a bound
 * B = (1 + 2^-6)^2 d max|q_norm| max|k_norm| log2(e) / sqrt(d) (log2 units; the margin covers the
 * bf16 rounding of q and k; 16.8 at d = 128 with unit weights); when B < 60 the softmax subtracts B
 * instead of a running row maximum, which lets it split each row over several warps (two, or four
 * at d = 128; the result differs from dit_attention by rounding only); otherwise it is
 * dit_attention. With weights other than ones (NULL counts as ones) B is computed on the device:
 * two kernels are launched and the one B does not choose returns at once. ws / ws_bytes as for
 * dit_attention. */
DIT_API int dit_attention_qknorm(const dit_dims* dims, int R, const uint16_t* q, const uint16_t* k, const uint16_t* vt,
                                 const float* q_norm, const float* k_norm, uint16_t* o, void* ws, size_t ws_bytes,
                                 dit_stream_t stream);

/* Linear with gated residual [gizai:dit, gatedInto]: x[r] += gate[map[r]] * (a[r] W^T) for the
 * attention (which = 0, W = wout [H, H], a [R, H]) or the MLP (which = 1, W = wdown [H, F],
 * a [R, F]) gate of the modulation rows. x rows < L in txt, others in img.
 * ws / ws_bytes: optional stream-K scratch (see dit_stream_k_workspace_bytes). */
DIT_API int dit_linear_gated(const dit_dims* dims, const uint16_t* a, int L, int N, const uint16_t* w,
                     const dit_mod* mod, int which, float* txt, float* img, void* ws, size_t ws_bytes,
                     dit_stream_t stream);

/* Up linear with SwiGLU epilogue [gizai:dit, gluRows]: u = h2 Wup^T [R, 2F];
 * a[r, j] = bf16(silu(u[r, 2j]) * u[r, 2j+1]) [R, F]. ws / ws_bytes: optional stream-K scratch
 * (see dit_stream_k_workspace_bytes). */
DIT_API int dit_linear_swiglu(const dit_dims* dims, const uint16_t* h2, int R, const uint16_t* wup, uint16_t* a,
                      void* ws, size_t ws_bytes, dit_stream_t stream);

/* Plain linear: out = a W^T with a [M, K] bf16, W [N, K] bf16; out fp32 (out_bf16 = 0) or bf16
 * (out_bf16 = 1), [M, N]. Supports K % 64 == 0 and N % 64 == 0. */
DIT_API int dit_linear(const uint16_t* a, int M, int K, const uint16_t* w, int N, void* out, int out_bf16,
               dit_stream_t stream);

/* int8lin dequantisation [host contract, section 1]: w[o, i] = bf16_rne(q[o, i] * s[o, i/32]),
 * the same arithmetic the int8 GEMM mainloop performs. cols % 32 == 0. */
DIT_API int dit_dequant_int8(const int8_t* q, const uint16_t* s, int64_t rows, int64_t cols, uint16_t* w,
                     dit_stream_t stream);

/* Plain linear with int8lin weights: out fp32 [M, N] = a W^T, W = bf16_rne(q * s) dequantized in
 * the mainloop (M <= 512) or once into the workspace (M > 512). K % 256 == 0, N % 128 == 0.
 * ws: dit_linear_int8_workspace_bytes(N, K) bytes, 256-byte aligned. */
DIT_API int dit_linear_int8(const uint16_t* a, int M, int K, const int8_t* wq, const uint16_t* w_scales, int N,
                            float* out, void* ws, size_t ws_bytes, dit_stream_t stream);
DIT_API size_t dit_linear_int8_workspace_bytes(int N, int K);

/* The whole-block forward for callers that cannot allocate device memory (no counterpart on the
 * pages: this entry point exists for callers, not for the method). A plugin running inside a host
 * application whose allocator owns the device memory, or a latency-bound loop where an allocation's
 * implicit device synchronisation is not allowed, cannot call cudaMalloc; such a caller passes only
 * inputs and outputs, exactly as for dit_block_forward, and the scratch lives in a static device
 * array of dit_block_noalloc_max_bytes() bytes (64 MiB) that every GPU loading the library holds
 * until the process exits. The call allocates nothing (no cudaMalloc/cudaFree, no allocating
 * library routine).
 *   - Limit: shapes whose dit_workspace_bytes(dims, L, N, 0) exceeds the array are rejected with
 *     DIT_EWORKSPACE before any launch (the 512x512 block, hidden 3072 / ffn 12288 / 1088 rows, fits;
 *     the 1024x1024 block does not).
 *   - Set-up: the first call on a device (with that device current) looks up the array's device
 *     address with cudaGetSymbolAddress; make that first call before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents; nothing in it needs to
 *     start at zero (each call writes every scratch byte before reading it). Calls that overlap on
 *     the GPU (other streams, other host threads) race on the array: serialise them.
 * Other arguments, results and errors as dit_block_forward. */
DIT_API int dit_block_forward_noalloc(const dit_dims* dims, const dit_block_w* w, float* txt, int L, float* img,
                                      int N, const float* txt_cos, const float* txt_sin, const float* img_cos,
                                      const float* img_sin, const dit_mod* mod, dit_stream_t stream);
DIT_API size_t dit_block_noalloc_max_bytes(void);

/* Synchronize `stream` and read (then clear) the device error word of the current device:
 * DIT_OK, DIT_ETIMEOUT, or DIT_ECUDA if the stream reported an error. */
DIT_API int dit_check(dit_stream_t stream);

/* Diagnostic of the failure-detection path (no counterpart on the pages): launches one warp that
 * waits, with the same bounded mbarrier wait every kernel here uses (1 s of the GPU's global
 * timer), on a barrier of its own that completes only when `complete` is nonzero. With
 * complete = 0 the wait gives up after about a second, records its site in the device error word
 * and the kernel returns, so the next dit_check(stream) returns DIT_ETIMEOUT and the context stays
 * usable; with complete != 0 dit_check returns DIT_OK. Returns DIT_OK once launched, DIT_ECUDA on a
 * launch error. */
DIT_API int dit_selftest_bounded_wait(int complete, dit_stream_t stream);

/* Static description of a status code. */
DIT_API const char* dit_status_string(int status);

/* Library version (major * 10000 + minor * 100 + patch). */
DIT_API int dit_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DIT_H_ */
