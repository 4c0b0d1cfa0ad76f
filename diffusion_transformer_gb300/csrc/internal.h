// Internal interface between the C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

#include "../../include/dit.h"

namespace dit {

// ------------------------------------------------------------------------------------------
// GEMM: C[M, N] = A[M, K] * B[N, K]^T, A and B bf16 K-major (row-major [rows, K]), fp32 accumulation
// in TMEM, one of several fused epilogues.
// ------------------------------------------------------------------------------------------
enum GemmEpilogue : int {
  kEpiStoreF32 = 0,     // out fp32 [M, N] (row stride ldo)
  kEpiStoreBF16 = 1,    // out bf16 [M, N]
  kEpiSiluBF16 = 2,     // out bf16 silu(acc)
  kEpiGated = 3,        // x[r, n] += gate[map[r]][n] * acc; x rows < L in txt, others in img (fp32, stride N)
  kEpiSwiGLU = 4,       // out bf16 [M, N/2]: a_j = silu(acc_{2j}) * acc_{2j+1}
  kEpiQKV = 5,          // QK-RMSNorm + RoPE on q/k columns -> q, k [heads, R, d]; v -> vt [heads, d, Rp]
  kEpiQKVSwiGLU = 6,    // columns < n_split as kEpiQKV, the rest as kEpiSwiGLU (parallel block)
};

struct GemmParams {
  int M, N, K;
  int* err;  // device error word
  // plain stores / swiglu
  void* out;
  long long ldo;
  // gated residual
  float* txt;
  float* img;
  int L;
  const float* gate;
  const int32_t* map;  // may be null: gate row 0 for every row
  long long gate_stride;
  // qkv epilogue
  uint16_t* q;
  uint16_t* k;
  uint16_t* vt;
  int H, heads, head_dim, Rp;
  const float *txt_cos, *txt_sin, *img_cos, *img_sin;  // [L, d/2], [R-L, d/2]
  const float *q_norm, *k_norm;                         // [d] or null
  float qk_eps;
  int rope_split;  // 0: adjacent pairs, tables [rows, d/2]; 1: split halves over 3d/4, tables [rows, 3d/8]
  // bf16 weights: caller scratch for stream-K (may be null: every tile whole). When the tiles are
  // not a whole number of waves, gemm_launch divides the k-blocks of the last sk_tiles tiles evenly
  // over the sk_units work units (CTAs or CTA pairs); a unit's share of a tile is a segment whose
  // fp32 partial accumulator goes to one of its two slots, and the unit that delivers a tile's
  // last segment sums the segments in order and runs the epilogue. Set by gemm_launch.
  void* split_ws;
  size_t split_ws_bytes;
  int sk_tiles, sk_units;
  float* sk_part;      // partial slots [2 * sk_units][slabs][128][BN] fp32 (slabs: 2 on CTA pairs)
  uint32_t* sk_cnt;    // arrivals per (stream-K tile, slab, 32-row quadrant); zero between launches
  // concatenated operands (0 = none): output columns >= n_split take B rows from the second B
  // (row n - n_split); inner indices >= k_split take A and B columns from the second A and B
  // (column k - k_split)
  int n_split, k_split;
  // rows of a sub-range of the sequence (one stream of a double-stream block): GEMM row r is sequence
  // row r + row_off for the QKV and gated epilogues; q, k and vt hold R_total rows (0: M)
  int row_off, R_total;
  // two row groups in one launch (double-stream block, m_split a multiple of 128): rows >= m_split
  // take B from the second B and, in the QKV epilogue, the head-norm weights q_norm2 / k_norm2
  int m_split;
  const float *q_norm2, *k_norm2;
  // TMA extents smaller than the GEMM's (0: the GEMM's): rows of B (columns past them read as zero)
  // and inner columns of the second B of a K-concatenation (LoRA factors of a rank below the tile)
  int b_rows, b2_inner;
  // set by the launcher for CTA-pair launches: a launch counter that picks the start-word set
  uint32_t pair_epoch;
  // W8A8 (both non-null): the accumulator is multiplied by a_scale[GEMM row] * w_scale[column]
  // before the epilogue (per-token and per-output-channel scales of integer codes); rows of the
  // second row group (m_split) take w_scale2 when it is given (the second stream's weight scales)
  const float *a_scale, *w_scale, *w_scale2;
};

// B operand in int8 with one bf16 scale per 32 consecutive K elements (int8lin weights). For row
// counts above kInt8MainloopMaxM the weight is first dequantised once into the caller's scratch
// (bf16 [N, K]) by the HBM-bound dequant kernel and the bf16 mainloop runs on it; below, the
// converter warps dequantise each k-block inside the mainloop (no scratch used).
struct GemmInt8B {
  const int8_t* q;     // [N, K]
  const uint16_t* s;   // [N, K/32] bf16 bits
  uint16_t* wbf;       // scratch [N, K] bf16 (may be null when M <= kInt8MainloopMaxM)
};
constexpr int kInt8MainloopMaxM = 512;
inline size_t gemm_int8_scratch_bytes(int N, int K) { return ((size_t(N) * K * 2) + 255) / 256 * 256; }

// Launch the GEMM. `a` is bf16 [M, K] (row stride lda elements), `b` bf16 [N, K] (stride K) unless
// `b8` is given. Returns a DIT_* status; checks shapes the kernels support.
// The same GEMM over concatenated bf16 operands: N-concatenation (p.n_split > 0: B = [b ; b2], b2
// the rows of output columns >= n_split), K-concatenation (p.k_split > 0: A = [a | a2],
// B = [b | b2], a2/b2 the columns from k_split on) or two row groups (p.m_split > 0: output rows
// >= m_split use the weights b2, [N, K] like b). Boundaries are multiples of the tile.
int gemm_launch_cat(const uint16_t* a, long long lda, const uint16_t* a2, long long lda2, const uint16_t* b,
                    long long ldb, const uint16_t* b2, long long ldb2, int epi, const GemmParams& p,
                    cudaStream_t stream);
int gemm_launch(const uint16_t* a, long long lda, const uint16_t* b, const GemmInt8B* b8, int epi,
                const GemmParams& p, cudaStream_t stream);
// Zero the stream-K arrival counters of the current device (after an aborted launch, which may
// leave some counted; dit_check does this when it finds the error word set). Synchronous.
int gemm_clear_stream_k_counters();

// ------------------------------------------------------------------------------------------
// attention
// ------------------------------------------------------------------------------------------
struct AttnParams {
  int R, heads, head_dim, Rp;
  const uint16_t *q, *k, *vt;  // [heads, R, d], [heads, R, d], [heads, d, Rp]
  uint16_t* o;                 // [R, heads * d]
  int* err;
  // qk_normed > 0: every q and k row was RMS-normalised per head and scaled by one of qk_normed (1 or
  // 2: the two streams of a double-stream block) sets of weights ([d] each, null = ones), as the QKV
  // epilogue does. The softmax may then subtract a fixed maximum (see attention.cu).
  int qk_normed;
  const float *qn0, *kn0, *qn1, *kn1;
  // optional scratch (16-byte aligned) for the persistent schedule: the unnormalised partials of
  // units split between two CTAs, 133 KB per CTA at d = 128; without it one CTA per unit
  void* part = nullptr;
  size_t part_bytes = 0;
  // set by attention_launch: key-tile steps per CTA, launch epoch of the ready words, and which of
  // a pair of launches this is (0: the only one; 1: fixed maximum, works when B < 60; 2: running
  // maximum, works when B >= 60)
  int work = 0;
  uint32_t epoch = 0;
  int select = 0;
};
int attention_launch(const AttnParams& p, cudaStream_t stream);
// Scratch the persistent schedule wants for R rows (0: it is not used for this shape).
size_t attention_part_bytes(int R, int heads, int head_dim);

// ------------------------------------------------------------------------------------------
// elementwise / row kernels
// ------------------------------------------------------------------------------------------
// h[r] = bf16( x[r] * rsqrt(mean(x[r]^2) + eps) * w * (1 + scale[m]) + shift[m] ), m = map[r] (or 0)
struct ModNormParams {
  const float* txt;
  const float* img;
  int L, R, H;
  long long ld_txt, ld_img;  // row strides (elements)
  const float* w;            // [H] or null
  const float* shift;        // row m at shift + m * mod_stride
  const float* scale;
  long long mod_stride;
  const int32_t* map;        // [R] or null (row 0)
  float eps;
  uint16_t* out;             // [R, H] bf16
  int layernorm;             // 0: RMS norm; 1: LayerNorm (mean subtracted first)
  int split_w;               // 1: rows >= L use w_img instead of w (per-stream norm weights)
  const float* w_img;        // [H] or null
};
int modnorm_launch(const ModNormParams& p, cudaStream_t stream);

// Sandwich residual: x[r] += gate[map[r]] * (f(y[r]) + f2(y2[r])), y [R, H] fp32 (a branch's linear
// output), f(y) = y * rsqrt(mean(y^2) + eps) * w for a normed row, y for an un-normed one; x rows < L
// in txt, others in img (row stride H). Text rows take (norm_txt, w), image rows (norm_img, w_img)
// (the double-stream block's per-stream post weights); the optional second branch y2 (the parallel
// block's MLP output under the same gate) is normed when norm2, with weight w2.
struct SandwichParams {
  float* txt;
  float* img;
  int L, R, H;
  const float* y;
  const float* gate;       // row m at gate + m * mod_stride
  long long mod_stride;
  const int32_t* map;      // [R] or null
  const float* w;          // [H] post-norm weight of the text rows or null (ones)
  float eps;
  int norm_txt, norm_img;  // text / image rows of y normed (1) or added as they are (0)
  const float* w_img;      // [H] post-norm weight of the image rows or null (ones)
  const float* y2;         // [R, H] second branch or null
  const float* w2;         // its post-norm weight or null (ones)
  int norm2;
};
int sandwich_launch(const SandwichParams& p, cudaStream_t stream);
// bounded-wait diagnostic (see dit_selftest_bounded_wait)
int wait_selftest_launch(int complete, int* err, cudaStream_t stream);

int euler_launch(float* x, const float* vel, long long n, float sigma, float sigma_next, cudaStream_t stream);
int rope_tables_launch(int L, int gh, int gw, int head_dim, float theta, float* cos, float* sin,
                       cudaStream_t stream);
int sinusoid_launch(const float* sigmas, int steps, int dim, uint16_t* out, cudaStream_t stream);
int f32_to_bf16_launch(const float* in, uint16_t* out, long long n, cudaStream_t stream);
int lora_merge_launch(const uint16_t* W, const uint16_t* A, const uint16_t* B, uint16_t* merged, int n_out, int n_in,
                      int rank, cudaStream_t stream);
int dequant_int8_launch(const int8_t* q, const uint16_t* s, uint16_t* w, long long rows, long long cols,
                        cudaStream_t stream);
// W8A8: per-token codes of x [rows, K] bf16 written over x (as bf16 integers) with scale[rows];
// per-output-channel codes of a bf16 weight [N, K] (int8) with scale[N]; int8 codes to bf16 (n % 16 == 0)
int quant_rows_launch(uint16_t* x, int rows, int K, const float* smooth, float* scale, cudaStream_t stream);
// The same over joined rows x[r, 0:K] ++ x2[r, 0:K2] (one code scale per joined row, divisors over the
// joined row), rows from row_split on taking the divisors smooth2 instead of smooth (NULL: none).
int quant_rows_joint_launch(uint16_t* x, int K, uint16_t* x2, int K2, int rows, const float* smooth,
                            const float* smooth2, int row_split, float* scale, cudaStream_t stream);
int quant_weight_launch(const uint16_t* w, int N, int K, const float* smooth, int8_t* q, float* scale,
                        cudaStream_t stream);
int codes_bf16_launch(const int8_t* q, uint16_t* w, long long n, cudaStream_t stream);

int num_sms();

// Launch `kern` on `stream` with programmatic dependent launch allowed (and a cluster of
// `cluster_x` CTAs when above 1). Only kernels that call pdl_wait() (ptx.cuh) before their first
// global memory access are launched this way.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  int n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = unsigned(cluster_x);
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = unsigned(n);
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Every check dit_block_forward makes before launching, except those on the workspace: DIT_OK, or the
// status it would return. Touches no CUDA state.
int check_block_call_without_workspace(const dit_dims* d, const dit_block_w* w, const float* txt, int L,
                                       const float* img, int N, const float* tc, const float* ts, const float* ic,
                                       const float* is, const dit_mod* mod);

// Raise a kernel's dynamic shared-memory limit on the current device (once per kernel and device).
bool smem_attr_once(const void* kernel, unsigned bytes);

}  // namespace dit
