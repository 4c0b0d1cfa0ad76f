// C ABI of libdit.so: argument validation, workspace carve-up and launch sequencing on the
// caller's stream. Every arithmetic step runs in the kernels of gemm.cu, attention.cu and
// elementwise.cu; this file only checks arguments and orders launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "tmap.h"

namespace dit {

// ------------------------------------------------------------------------------------------
// per-device state: error word address and SM count
// ------------------------------------------------------------------------------------------
static __device__ int g_error_word;

namespace {
constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];
std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int* err_word() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool dims_ok(const dit_dims* d) {
  if (!d) return false;
  if (d->head_dim != 64 && d->head_dim != 128) return false;
  if (d->heads <= 0 || d->hidden != d->heads * d->head_dim) return false;
  if (d->hidden % 256 != 0 || d->ffn <= 0 || d->ffn % 128 != 0) return false;
  if (!(d->eps >= 0.f) || !(d->qk_eps >= 0.f)) return false;
  if (d->rope_split != 0 && d->rope_split != 1) return false;
  return true;
}

struct BlockWs {
  uint16_t* h;   // [R, H]  norm outputs (h, then h2)
  uint16_t* q;   // [nh, R, d]
  uint16_t* k;   // [nh, R, d]
  uint16_t* vt;  // [nh, d, Rp]
  uint16_t* o;   // [R, H]  attention output
  uint16_t* a;   // [R, F]  SwiGLU output
  size_t bytes;
};

int vt_stride(int R) { return int(round_up(size_t(R), 8)); }

BlockWs carve_block_ws(const dit_dims* d, int R, void* base) {
  BlockWs w{};
  const size_t H = d->hidden, F = d->ffn, nh = d->heads, hd = d->head_dim;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* r = p ? p + off : nullptr;
    off += round_up(bytes, 256);
    return reinterpret_cast<uint16_t*>(r);
  };
  w.h = take(size_t(R) * H * 2);
  w.q = take(nh * size_t(R) * hd * 2);
  w.k = take(nh * size_t(R) * hd * 2);
  w.vt = take(nh * hd * size_t(vt_stride(R)) * 2);
  w.o = take(size_t(R) * H * 2);
  w.a = take(size_t(R) * F * 2);
  w.bytes = off;
  return w;
}

// Every block reads h (or its codes) only in the linears before attention and rewrites it only
// after: attention borrows the h rows as scratch for the partials of its persistent schedule.
void lend_h(AttnParams& ap, const BlockWs& b, int R, int H) {
  ap.part = b.h;
  ap.part_bytes = size_t(R) * H * 2;
}

// int8lin scratch of a block: two slots, each the dequantised weight of its largest linear (the
// weights are dequantised one linear ahead of their use, alternating slots)
size_t int8_slot_bytes(const dit_dims* d) {
  const int H = d->hidden, F = d->ffn;
  const int shapes[4][2] = {{3 * H, H}, {H, H}, {2 * F, H}, {H, F}};
  size_t tl = 0;
  for (auto& s : shapes) tl = std::max(tl, gemm_int8_scratch_bytes(s[0], s[1]));
  return tl;
}
size_t int8_scratch_bytes(const dit_dims* d) { return 2 * int8_slot_bytes(d); }
// int8lin parallel block: slot 0 = [Wqkv ; Wup] [3H + 2F, H], slot 1 = Wout [H, H] then Wdown [H, F]
size_t int8_parallel_slot0_bytes(const dit_dims* d) {
  return gemm_int8_scratch_bytes(3 * d->hidden + 2 * d->ffn, d->hidden);
}
size_t int8_parallel_scratch_bytes(const dit_dims* d) {
  return int8_parallel_slot0_bytes(d) + gemm_int8_scratch_bytes(d->hidden, d->hidden + d->ffn);
}
// int8lin double-stream block: two slots, each one linear's text weight followed by its image weight
size_t int8_double_scratch_bytes(const dit_dims* d) { return 4 * int8_slot_bytes(d); }

// Per device: a second stream and events for the int8lin block's weight dequantisation, which runs
// beside the block's kernels (fork from and join to the caller's stream through events). The mutex
// keeps one block's enqueue sequence whole when several host threads share the device.
struct SideStream {
  std::mutex mu;
  bool tried = false, ok = false;
  cudaStream_t s = nullptr;
  cudaEvent_t ev[8] = {};
};
SideStream g_side[kMaxDevices];
SideStream* side_stream() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  SideStream& ss = g_side[dev];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!ss.tried) {
    ss.tried = true;
    ss.ok = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) == cudaSuccess;
    for (auto& e : ss.ev) ss.ok = ss.ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
  }
  return ss.ok ? &ss : nullptr;
}

// The weights of a block's n <= 4 GEMMs prepared (dequantised, or widened from int8 codes) on the
// side stream one GEMM ahead of their use, into two alternating workspace slots: weight i goes to
// slot i % 2; weights 0 and 1 start at the fork, 2 once GEMM 0 has released slot 0, 3 once GEMM 1
// has released slot 1. Events: 0 fork, 1-4 weight i ready, 5-6 slot 0 / 1 free, 7 the join that
// every exit makes (the caller's stream then waits for all side work).
class WeightPrefetch {
 public:
  // prep(i, dst, stream) launches the preparation of linear i's weight into dst
  using Prep = int (*)(const void* ctx, int i, uint16_t* dst, cudaStream_t stream);
  WeightPrefetch(cudaStream_t st, uint16_t* slot0, size_t slot_bytes, Prep prep, const void* ctx, int n = 4)
      : st_(st), prep_(prep), ctx_(ctx), n_(n) {
    slot_[0] = slot0;
    slot_[1] = slot0 ? reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(slot0) + slot_bytes) : nullptr;
  }
  ~WeightPrefetch() {
    if (side_ && cudaEventRecord(side_->ev[7], side_->s) == cudaSuccess) cudaStreamWaitEvent(st_, side_->ev[7], 0);
  }
  // fork and start linears 0 and 1
  int start() {
    side_ = side_stream();
    if (!side_) return DIT_ECUDA;
    lock_ = std::unique_lock<std::mutex>(side_->mu);
    if (cudaEventRecord(side_->ev[0], st_) != cudaSuccess) return DIT_ECUDA;
    int r = ahead(0, 0);
    return r == DIT_OK && n_ > 1 ? ahead(1, -1) : r;
  }
  // the weight of linear i, ready for a launch on the caller's stream
  int use(int i, const uint16_t** w) {
    if (cudaStreamWaitEvent(st_, side_->ev[1 + i], 0) != cudaSuccess) return DIT_ECUDA;
    *w = slot_[i % 2];
    return DIT_OK;
  }
  // after GEMM i: its slot is free, and weight i + 2 (if any) may be prepared into it
  int done(int i) {
    if (i + 2 >= n_) return DIT_OK;
    if (cudaEventRecord(side_->ev[5 + i % 2], st_) != cudaSuccess) return DIT_ECUDA;
    return ahead(i + 2, 5 + i % 2);
  }

 private:
  int ahead(int i, int after) {
    if (after >= 0 && cudaStreamWaitEvent(side_->s, side_->ev[after], 0) != cudaSuccess) return DIT_ECUDA;
    int r = prep_(ctx_, i, slot_[i % 2], side_->s);
    if (r != DIT_OK) return r;
    return cudaEventRecord(side_->ev[1 + i], side_->s) == cudaSuccess ? DIT_OK : DIT_ECUDA;
  }
  cudaStream_t st_;
  Prep prep_;
  const void* ctx_;
  int n_;
  uint16_t* slot_[2];
  SideStream* side_ = nullptr;
  std::unique_lock<std::mutex> lock_;
};

// [out, in] of linear i (0 qkv, 1 out, 2 up, 3 down)
void linear_shape(const dit_dims* d, int i, int* n, int* k) {
  const int H = d->hidden, F = d->ffn;
  const int shp[4][2] = {{3 * H, H}, {H, H}, {2 * F, H}, {H, F}};
  *n = shp[i][0];
  *k = shp[i][1];
}

GemmParams base_params(int M, int N, int K, int* err) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.err = err;
  return p;
}

// QKV epilogue parameters: q, k, vt of the whole sequence (R rows, L text rows) in the block
// workspace, the rotary tables and the head-norm weights.
GemmParams qkv_params(const dit_dims* d, int M, int R, int L, const BlockWs& b, const float* tc, const float* ts,
                      const float* ic, const float* is, const float* qn, const float* kn, int* err) {
  GemmParams g = base_params(M, 3 * d->hidden, d->hidden, err);
  g.q = b.q;
  g.k = b.k;
  g.vt = b.vt;
  g.H = d->hidden;
  g.heads = d->heads;
  g.head_dim = d->head_dim;
  g.Rp = vt_stride(R);
  g.L = L;
  g.txt_cos = tc;
  g.txt_sin = ts;
  g.img_cos = ic;
  g.img_sin = is;
  g.q_norm = qn;
  g.k_norm = kn;
  g.qk_eps = d->qk_eps;
  g.rope_split = d->rope_split;
  return g;
}

struct ModRef {
  const float* rows;
  const int32_t* map;
  int M;
};

// One whole block on already-validated arguments. `w8` selects the int8lin path.
int lora_rank_pad(int rank) { return (rank + 63) / 64 * 64; }

// Linear i over the rows x [g.M, K] (bf16) with its LoRA adapter beside it when `lora` has factors
// for linear i [gizai:dit, loraOf, withLora]: down = x A_i^T into `down` ([g.M, rank padded to 64];
// the B operand's TMA map ends at the rank, so the padding columns come out as zeros), then one GEMM
// over [x | down] [W | B_i]^T through the linear's own epilogue. Without an adapter, the plain GEMM.
int gemm_with_lora(const dit_lora* lora, int i, const uint16_t* x, int K, const uint16_t* W, int epi, GemmParams g,
                   uint16_t* down, int* err, cudaStream_t st) {
  if (!lora || !lora->A[i]) return gemm_launch(x, K, W, nullptr, epi, g, st);
  const int rp = lora_rank_pad(lora->rank);
  GemmParams gd = base_params(g.M, rp, K, err);
  gd.out = down;
  gd.ldo = rp;
  gd.b_rows = lora->rank;
  int rc = gemm_launch(x, K, lora->A[i], nullptr, kEpiStoreBF16, gd, st);
  if (rc != DIT_OK) return rc;
  g.K = K + rp;
  g.k_split = K;
  g.b2_inner = lora->rank;
  return gemm_launch_cat(x, K, down, rp, W, K, lora->B[i], lora->rank, epi, g, st);
}

int run_block(const dit_dims* d, const dit_block_w* w, const dit_block_w8* w8, float* txt, int L, float* img, int N,
              const float* tc, const float* ts, const float* ic, const float* is, const ModRef& mod, void* ws,
              cudaStream_t st, const dit_lora* lora = nullptr, const float* post_attn = nullptr,
              const float* post_mlp = nullptr) {
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  const int R = L + N, H = d->hidden, F = d->ffn;
  const BlockWs b = carve_block_ws(d, R, ws);
  // linear i (0 qkv, 1 out, 2 up, 3 down) of input x [R, K]: with a LoRA adapter, down = x A^T into
  // the scratch after the block workspace ([R, rank padded to 64], the padding computed as zero from
  // A's missing rows), then [x | down] [W | B]^T through the linear's own epilogue
  uint16_t* lora_down = lora ? reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + b.bytes) : nullptr;
  auto linear = [&](int i, const uint16_t* x, int K, const uint16_t* W, const GemmInt8B* w8b, int epi,
                    GemmParams g) -> int {
    if (!lora || !lora->A[i]) return gemm_launch(x, K, W, w8b, epi, g, st);
    return gemm_with_lora(lora, i, x, K, W, epi, g, lora_down, err, st);
  };
  // a gated linear; with a post-norm weight (sandwich block) its output y goes to the h..vt span as
  // fp32 (consumed by then, and at least R * H * 4 bytes) and the sandwich kernel adds
  // gate * rmsnorm(y) * post to x
  auto gated_linear = [&](int i, const uint16_t* x, int K, const uint16_t* W, const GemmInt8B* w8b, GemmParams g,
                          const float* post, long long gate_row) -> int {
    if (!post) return linear(i, x, K, W, w8b, kEpiGated, g);
    float* y = reinterpret_cast<float*>(b.h);
    GemmParams gy = base_params(R, H, K, err);
    gy.out = y;
    gy.ldo = H;
    int rc = linear(i, x, K, W, w8b, kEpiStoreF32, gy);
    if (rc != DIT_OK) return rc;
    SandwichParams sp{txt, img, L, R, H, y, mod.rows + gate_row * H, 6LL * H, mod.map, post, d->eps, 1, 1, post};
    return sandwich_launch(sp, st);
  };
  // int8lin scratch after the block workspace: two slots of dequantised weights
  uint16_t* i8_tiles = w8 ? reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + b.bytes) : nullptr;
  // Rows above kInt8MainloopMaxM: each linear's weight is dequantised once (HBM-bound) on the side
  // stream one linear ahead, while the main stream runs the previous kernels; each GEMM then runs
  // the bf16 mainloop on its slot. (Fewer rows: the GEMMs dequantise inside their mainloop.)
  struct DequantCtx {
    const dit_dims* d;
    const dit_block_w8* w8;
  } dctx{d, w8};
  auto dequant = [](const void* c, int i, uint16_t* dst, cudaStream_t s2) -> int {
    const DequantCtx* x = static_cast<const DequantCtx*>(c);
    int n, k;
    linear_shape(x->d, i, &n, &k);
    return dequant_int8_launch(x->w8->q[i], x->w8->s[i], dst, n, k, s2);
  };
  const bool prefetch = w8 && R > kInt8MainloopMaxM;
  WeightPrefetch pf(st, i8_tiles, w8 ? int8_slot_bytes(d) : 0, dequant, &dctx);
  int rc;
  if (prefetch && (rc = pf.start()) != DIT_OK) return rc;
  // the int8lin GEMM of linear i: on the prefetched slot, or with the in-mainloop dequantisation
  auto gemm8 = [&](int i, const uint16_t* x, int K, int epi, const GemmParams& g) -> int {
    if (!prefetch) {
      GemmInt8B q8{w8->q[i], w8->s[i], i8_tiles};
      return gemm_launch(x, K, nullptr, &q8, epi, g, st);
    }
    const uint16_t* wb;
    int r = pf.use(i, &wb);
    if (r == DIT_OK) r = gemm_launch(x, K, wb, nullptr, epi, g, st);
    return r == DIT_OK ? pf.done(i) : r;
  };
  const float* norm1 = w8 ? w8->norm1 : w->norm1;
  const float* norm2 = w8 ? w8->norm2 : w->norm2;
  const float* qn = w8 ? w8->q_norm : w->q_norm;
  const float* kn = w8 ? w8->k_norm : w->k_norm;

  // 1. h = modnorm(x; norm1, shift_a, scale_a)
  ModNormParams mp{txt, img, L, R, H, H, H, norm1, mod.rows, mod.rows + H, 6LL * H, mod.map, d->eps, b.h};
  if ((rc = modnorm_launch(mp, st)) != DIT_OK) return rc;

  // 2. q, k, vt = qk-norm + rope epilogue of h Wqkv^T
  GemmParams g = qkv_params(d, R, R, L, b, tc, ts, ic, is, qn, kn, err);
  if ((rc = w8 ? gemm8(0, b.h, H, kEpiQKV, g) : linear(0, b.h, H, w->wqkv, nullptr, kEpiQKV, g)) != DIT_OK) return rc;

  // 3. o = attention(q, k, v); q and k rows QK-normed with qn, kn
  AttnParams ap{R, d->heads, d->head_dim, vt_stride(R), b.q, b.k, b.vt, b.o, err, 1, qn, kn, nullptr, nullptr};
  lend_h(ap, b, R, H);
  if ((rc = attention_launch(ap, st)) != DIT_OK) return rc;

  // 4. x += gate_a * (o Wout^T)
  g = base_params(R, H, H, err);
  g.txt = txt;
  g.img = img;
  g.L = L;
  g.gate = mod.rows + 2LL * H;
  g.map = mod.map;
  g.gate_stride = 6LL * H;
  if ((rc = w8 ? gemm8(1, b.o, H, kEpiGated, g) : gated_linear(1, b.o, H, w->wout, nullptr, g, post_attn, 2)) != DIT_OK)
    return rc;

  // 5. h2 = modnorm(x; norm2, shift_m, scale_m)
  mp.w = norm2;
  mp.shift = mod.rows + 3LL * H;
  mp.scale = mod.rows + 4LL * H;
  if ((rc = modnorm_launch(mp, st)) != DIT_OK) return rc;

  // 6. a = silu(h2 Wgate^T) * (h2 Wup^T), interleaved rows
  g = base_params(R, 2 * F, H, err);
  g.out = b.a;
  g.ldo = F;
  if ((rc = w8 ? gemm8(2, b.h, H, kEpiSwiGLU, g) : linear(2, b.h, H, w->wup, nullptr, kEpiSwiGLU, g)) != DIT_OK)
    return rc;

  // 7. x += gate_m * (a Wdown^T)
  g = base_params(R, H, F, err);
  g.txt = txt;
  g.img = img;
  g.L = L;
  g.gate = mod.rows + 5LL * H;
  g.map = mod.map;
  g.gate_stride = 6LL * H;
  // (int8lin: the down GEMM waits for its weight, the side stream's last work: the join)
  return w8 ? gemm8(3, b.a, F, kEpiGated, g) : gated_linear(3, b.a, F, w->wdown, nullptr, g, post_mlp, 5);
}

// W8A8 scratch after the block workspace: two slots of bf16-widened weight codes (as for int8lin),
// then the per-token scales [R] of the activation being quantised
size_t w8a8_extra_bytes(const dit_dims* d, int R) {
  return int8_scratch_bytes(d) + round_up(size_t(R) * sizeof(float), 256);
}

// The block with W8A8 linears [klein, section 5 and its D4/D5 entries]: each linear's activation
// (h, o, h2, a) is quantised per token in place (bf16 integer codes over the bf16 values; SmoothQuant
// divisor first when given) with its scales in the workspace; the weight's int8 codes are widened to
// bf16 on the side stream one linear ahead; the GEMM's integer-valued accumulator (exact while every
// partial sum stays below 2^24) is multiplied by the row's and the column's scales before the
// linear's usual epilogue.
int run_block_w8a8(const dit_dims* d, const dit_block_w8a8* w, float* txt, int L, float* img, int N,
                   const float* tc, const float* ts, const float* ic, const float* is, const ModRef& mod, void* ws,
                   cudaStream_t st) {
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  const int R = L + N, H = d->hidden, F = d->ffn;
  const BlockWs b = carve_block_ws(d, R, ws);
  uint16_t* slots = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + b.bytes);
  float* sa = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + b.bytes + int8_scratch_bytes(d));
  struct CodesCtx {
    const dit_dims* d;
    const dit_block_w8a8* w;
  } cctx{d, w};
  auto widen = [](const void* c, int i, uint16_t* dst, cudaStream_t s2) -> int {
    const CodesCtx* x = static_cast<const CodesCtx*>(c);
    int n, k;
    linear_shape(x->d, i, &n, &k);
    return codes_bf16_launch(x->w->q[i], dst, (long long)n * k, s2);
  };
  WeightPrefetch pf(st, slots, int8_slot_bytes(d), widen, &cctx);
  int rc;
  if ((rc = pf.start()) != DIT_OK) return rc;
  // linear i on activation codes x [R, K] (quantised in place first)
  auto linear = [&](int i, uint16_t* x, int K, int epi, GemmParams g) -> int {
    int r = quant_rows_launch(x, R, K, w->smooth[i], sa, st);
    if (r != DIT_OK) return r;
    const uint16_t* wc;
    if ((r = pf.use(i, &wc)) != DIT_OK) return r;
    g.a_scale = sa;
    g.w_scale = w->scale[i];
    if ((r = gemm_launch(x, K, wc, nullptr, epi, g, st)) != DIT_OK) return r;
    return pf.done(i);
  };
  auto gated = [&](int K, long long gate_row) {
    GemmParams g = base_params(R, H, K, err);
    g.txt = txt;
    g.img = img;
    g.L = L;
    g.gate = mod.rows + gate_row * H;
    g.map = mod.map;
    g.gate_stride = 6LL * H;
    return g;
  };

  // 1. h = modnorm(x; norm1, shift_a, scale_a)
  ModNormParams mp{txt, img, L, R, H, H, H, w->norm1, mod.rows, mod.rows + H, 6LL * H, mod.map, d->eps, b.h};
  if ((rc = modnorm_launch(mp, st)) != DIT_OK) return rc;
  // 2. q, k, vt from the W8A8 QKV linear with the QK-norm + rotary epilogue
  if ((rc = linear(0, b.h, H, kEpiQKV, qkv_params(d, R, R, L, b, tc, ts, ic, is, w->q_norm, w->k_norm, err))) !=
      DIT_OK)
    return rc;
  // 3. o = attention(q, k, v)
  AttnParams ap{R, d->heads, d->head_dim, vt_stride(R), b.q, b.k, b.vt, b.o, err, 1, w->q_norm, w->k_norm, nullptr,
                nullptr};
  lend_h(ap, b, R, H);
  if ((rc = attention_launch(ap, st)) != DIT_OK) return rc;
  // 4. x += gate_a * W8A8(o, Wout)
  if ((rc = linear(1, b.o, H, kEpiGated, gated(H, 2))) != DIT_OK) return rc;
  // 5. h2 = modnorm(x; norm2, shift_m, scale_m)
  mp.w = w->norm2;
  mp.shift = mod.rows + 3LL * H;
  mp.scale = mod.rows + 4LL * H;
  if ((rc = modnorm_launch(mp, st)) != DIT_OK) return rc;
  // 6. a = SwiGLU(W8A8(h2, Wup))
  GemmParams g = base_params(R, 2 * F, H, err);
  g.out = b.a;
  g.ldo = F;
  if ((rc = linear(2, b.h, H, kEpiSwiGLU, g)) != DIT_OK) return rc;
  // 7. x += gate_m * W8A8(a, Wdown)
  return linear(3, b.a, F, kEpiGated, gated(F, 5));
}

// The parallel (single-stream) block [gizai:dit, Block.parallel]: one modulated LayerNorm feeds
// both branches; mod rows [M, 3, H] = shift, scale, gate. Four launches: the norm, one GEMM over
// [Wqkv ; Wup] with the QKV epilogue on its first 3H columns and SwiGLU on the rest, the attention,
// and one GEMM over [o | a] [Wout | Wdown]^T with the gated residual. `w8` selects the int8lin
// weights: on the side stream, [Wqkv ; Wup] is dequantised into one scratch slot (overlapping the
// norm) and Wout, Wdown into a second (overlapping the first GEMM and the attention), whatever the
// row count; the GEMMs are then the bf16 ones on the slots.
int run_parallel_block(const dit_dims* d, const dit_block_w* w, const dit_block_w8* w8, const dit_parallel_w8a8* wq,
                       float* txt, int L, float* img, int N, const float* tc, const float* ts, const float* ic,
                       const float* is, const ModRef& mod, void* ws, cudaStream_t st, const dit_lora* lora = nullptr,
                       const float* post_attn = nullptr, const float* post_mlp = nullptr) {
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  const int R = L + N, H = d->hidden, F = d->ffn;
  const BlockWs b = carve_block_ws(d, R, ws);
  if (lora) {
    // Adapters beside the linears: the fused GEMMs cannot take a second K-concatenated factor per
    // fused part, so the four linears run one by one, each with its adapter (gemm_with_lora), the
    // two output linears both adding gate * (their product) to x.
    uint16_t* down = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + b.bytes);
    int rc;
    ModNormParams mp{txt, img, L, R, H, H, H, w->norm1, mod.rows, mod.rows + H, 3LL * H, mod.map, d->eps, b.h};
    mp.layernorm = 1;
    if ((rc = modnorm_launch(mp, st)) != DIT_OK) return rc;
    GemmParams g = qkv_params(d, R, R, L, b, tc, ts, ic, is, w->q_norm, w->k_norm, err);
    if ((rc = gemm_with_lora(lora, 0, b.h, H, w->wqkv, kEpiQKV, g, down, err, st)) != DIT_OK) return rc;
    g = base_params(R, 2 * F, H, err);
    g.out = b.a;
    g.ldo = F;
    if ((rc = gemm_with_lora(lora, 2, b.h, H, w->wup, kEpiSwiGLU, g, down, err, st)) != DIT_OK) return rc;
    AttnParams ap{R, d->heads, d->head_dim, vt_stride(R), b.q, b.k, b.vt, b.o, err, 1, w->q_norm, w->k_norm, nullptr,
                  nullptr};
    lend_h(ap, b, R, H);
    if ((rc = attention_launch(ap, st)) != DIT_OK) return rc;
    for (int i : {1, 3}) {
      g = base_params(R, H, i == 1 ? H : F, err);
      g.txt = txt;
      g.img = img;
      g.L = L;
      g.gate = mod.rows + 2LL * H;
      g.map = mod.map;
      g.gate_stride = 3LL * H;
      if ((rc = gemm_with_lora(lora, i, i == 1 ? b.o : b.a, i == 1 ? H : F, i == 1 ? w->wout : w->wdown, kEpiGated,
                               g, down, err, st)) != DIT_OK)
        return rc;
    }
    return DIT_OK;
  }
  struct DequantCtx {
    const dit_dims* d;
    const dit_block_w8* w8;
    const dit_parallel_w8a8* wq;
  } dctx{d, w8, wq};
  // weight 0: Wqkv then Wup (rows 3H on); weight 1: Wout then Wdown (at H * H). W8A8: the codes of
  // linear1 [3H + 2F, H] and of linear2 [H, H + F] widened to bf16
  auto dequant = [](const void* c, int i, uint16_t* dst, cudaStream_t s2) -> int {
    const DequantCtx* x = static_cast<const DequantCtx*>(c);
    const int H_ = x->d->hidden;
    if (x->wq) {
      const long long n = i == 0 ? (3LL * H_ + 2LL * x->d->ffn) * H_ : (long long)H_ * (H_ + x->d->ffn);
      return codes_bf16_launch(i == 0 ? x->wq->q1 : x->wq->q2, dst, n, s2);
    }
    const int first = i == 0 ? 0 : 1, second = i == 0 ? 2 : 3;
    int n, k;
    linear_shape(x->d, first, &n, &k);
    int r = dequant_int8_launch(x->w8->q[first], x->w8->s[first], dst, n, k, s2);
    if (r != DIT_OK) return r;
    uint16_t* dst2 = dst + (i == 0 ? size_t(3) * H_ * H_ : size_t(H_) * H_);
    linear_shape(x->d, second, &n, &k);
    return dequant_int8_launch(x->w8->q[second], x->w8->s[second], dst2, n, k, s2);
  };
  const bool slotted = w8 || wq;  // weights prepared into the slots after the block workspace
  uint16_t* slots = slotted ? reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + b.bytes) : nullptr;
  WeightPrefetch pf(st, slots, slotted ? int8_parallel_slot0_bytes(d) : 0, dequant, &dctx, 2);
  // W8A8: per-token scales of h and of [o | a], after the slots
  float* sa1 = wq ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + b.bytes + int8_parallel_scratch_bytes(d))
                  : nullptr;
  float* sa2 = wq ? sa1 + round_up(size_t(R), 64) : nullptr;
  int rc;
  if (slotted && (rc = pf.start()) != DIT_OK) return rc;
  const float* norm = wq ? wq->norm1 : w8 ? w8->norm1 : w->norm1;
  const float* qn = wq ? wq->q_norm : w8 ? w8->q_norm : w->q_norm;
  const float* kn = wq ? wq->k_norm : w8 ? w8->k_norm : w->k_norm;
  const uint16_t *wqkv = slotted ? nullptr : w->wqkv, *wup = slotted ? nullptr : w->wup;
  const uint16_t *wout = slotted ? nullptr : w->wout, *wdown = slotted ? nullptr : w->wdown;
  long long ld_out = H, ld_down = F;  // row strides of the two halves of the second GEMM's weight

  // 1. h = LayerNorm(x) * norm * (1 + scale) + shift (W8A8: then its per-token codes in place)
  ModNormParams mp{txt, img, L, R, H, H, H, norm, mod.rows, mod.rows + H, 3LL * H, mod.map, d->eps, b.h};
  mp.layernorm = 1;
  if ((rc = modnorm_launch(mp, st)) != DIT_OK) return rc;
  if (wq && (rc = quant_rows_launch(b.h, R, H, wq->smooth1, sa1, st)) != DIT_OK) return rc;

  // 2. q, k, vt (QK-norm + rope epilogue) and a (SwiGLU epilogue) from h [Wqkv ; Wup]^T
  GemmParams g = qkv_params(d, R, R, L, b, tc, ts, ic, is, qn, kn, err);
  g.N = 3 * H + 2 * F;
  g.out = b.a;
  g.ldo = F;
  g.n_split = 3 * H;
  if (slotted) {
    const uint16_t* s0;
    if ((rc = pf.use(0, &s0)) != DIT_OK) return rc;
    wqkv = s0;
    wup = s0 + size_t(3) * H * H;
  }
  if (wq) {
    g.a_scale = sa1;
    g.w_scale = wq->scale1;
  }
  if ((rc = gemm_launch_cat(b.h, H, nullptr, 0, wqkv, H, wup, H, kEpiQKVSwiGLU, g, st)) != DIT_OK) return rc;

  // 3. o = attention(q, k, v); q and k rows QK-normed
  AttnParams ap{R, d->heads, d->head_dim, vt_stride(R), b.q, b.k, b.vt, b.o, err, 1, qn, kn, nullptr, nullptr};
  lend_h(ap, b, R, H);
  if ((rc = attention_launch(ap, st)) != DIT_OK) return rc;
  // W8A8: codes of the joined rows [o | a] in place, one scale per row
  if (wq && (rc = quant_rows_joint_launch(b.o, H, b.a, F, R, wq->smooth2, nullptr, R, sa2, st)) != DIT_OK) return rc;

  // 4. x += gate * ([o | a] [Wout | Wdown]^T); with post-norm weights (a sandwich block) each output
  // product is stored in fp32 (o Wout^T over h and q, a Wdown^T over k and vt, consumed by now) and
  // the sandwich kernel adds gate * (rmsnorm(y1) post_attn + rmsnorm(y2) post_mlp) to x
  if (post_attn || post_mlp) {
    float* y1 = reinterpret_cast<float*>(b.h);
    float* y2 = reinterpret_cast<float*>(b.k);
    for (int i : {1, 3}) {
      g = base_params(R, H, i == 1 ? H : F, err);
      g.out = i == 1 ? y1 : y2;
      g.ldo = H;
      if ((rc = gemm_launch(i == 1 ? b.o : b.a, i == 1 ? H : F, i == 1 ? wout : wdown, nullptr, kEpiStoreF32, g, st)) !=
          DIT_OK)
        return rc;
    }
    SandwichParams sp{txt, img, L, R, H, y1, mod.rows + 2LL * H, 3LL * H, mod.map, post_attn, d->eps,
                      post_attn != nullptr, post_attn != nullptr, post_attn, y2, post_mlp, post_mlp != nullptr};
    return sandwich_launch(sp, st);
  }
  g = base_params(R, H, H + F, err);
  g.txt = txt;
  g.img = img;
  g.L = L;
  g.gate = mod.rows + 2LL * H;
  g.map = mod.map;
  g.gate_stride = 3LL * H;
  g.k_split = H;
  if (slotted) {
    const uint16_t* s1;
    if ((rc = pf.use(1, &s1)) != DIT_OK) return rc;
    if (wq) {
      // linear2's codes [H, H + F]: the first H columns multiply o, the rest a
      wout = s1;
      wdown = s1 + H;
      ld_out = ld_down = H + F;
      g.a_scale = sa2;
      g.w_scale = wq->scale2;
    } else {
      wout = s1;
      wdown = s1 + size_t(H) * H;
    }
  }
  return gemm_launch_cat(b.o, H, b.a, F, wout, ld_out, wdown, ld_down, kEpiGated, g, st);
}

// The double-stream block: the sequential block in which text rows [0, L) and image rows [L, R)
// each use their own linears and norm weights; the attention runs once over all R rows. Each
// stream's norms and GEMMs are launched over its own rows (row_off = its first sequence row), so any
// L works; the modulation map gives each stream its own modulation rows. `w8t`, `w8i` select the
// int8lin weights: linear i's text and image weights are dequantised on the side stream into one
// scratch slot (text first, none when L = 0), one linear ahead of their GEMM, whatever the row count.
int run_double_block(const dit_dims* d, const dit_block_w* wt, const dit_block_w* wi, const dit_block_w8* w8t,
                     const dit_block_w8* w8i, const dit_block_w8a8* wqt, const dit_block_w8a8* wqi, float* txt, int L,
                     float* img, int N, const float* tc, const float* ts, const float* ic, const float* is,
                     const ModRef& mod, void* ws, cudaStream_t st, const dit_lora* lora_t = nullptr,
                     const dit_lora* lora_i = nullptr, const float* const* post_t = nullptr,
                     const float* const* post_i = nullptr) {
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  const int R = L + N, H = d->hidden, F = d->ffn;
  const BlockWs b = carve_block_ws(d, R, ws);
  // int8lin / W8A8: the weights each GEMM reads live in the prefetch slots (dequantised, or codes
  // widened to bf16); tw8 / iw8 point at them, linear by linear, once the side stream has written them
  struct DequantCtx {
    const dit_dims* d;
    const dit_block_w8* t;
    const dit_block_w8* i;
    const dit_block_w8a8* qt;
    const dit_block_w8a8* qi;
    int L;
  } dctx{d, w8t, w8i, wqt, wqi, L};
  auto dequant = [](const void* c, int i, uint16_t* dst, cudaStream_t s2) -> int {
    const DequantCtx* x = static_cast<const DequantCtx*>(c);
    int n, k;
    linear_shape(x->d, i, &n, &k);
    if (x->L > 0) {
      int r = x->qi ? codes_bf16_launch(x->qt->q[i], dst, (long long)n * k, s2)
                    : dequant_int8_launch(x->t->q[i], x->t->s[i], dst, n, k, s2);
      if (r != DIT_OK) return r;
      dst += size_t(n) * k;
    }
    return x->qi ? codes_bf16_launch(x->qi->q[i], dst, (long long)n * k, s2)
                 : dequant_int8_launch(x->i->q[i], x->i->s[i], dst, n, k, s2);
  };
  const bool q8 = w8i != nullptr || wqi != nullptr;
  uint16_t* slots = q8 ? reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + b.bytes) : nullptr;
  WeightPrefetch pf(st, slots, q8 ? 2 * int8_slot_bytes(d) : 0, dequant, &dctx);
  // W8A8: per-token scales of the activation being quantised, after the slots
  float* sa = wqi ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + b.bytes + int8_double_scratch_bytes(d))
                  : nullptr;
  dit_block_w tw8{}, iw8{};
  if (q8) {
    if (wqi) {
      if (L > 0) tw8 = dit_block_w{nullptr, nullptr, nullptr, nullptr, wqt->norm1, wqt->norm2, wqt->q_norm, wqt->k_norm};
      iw8 = dit_block_w{nullptr, nullptr, nullptr, nullptr, wqi->norm1, wqi->norm2, wqi->q_norm, wqi->k_norm};
    } else {
      if (L > 0) tw8 = dit_block_w{nullptr, nullptr, nullptr, nullptr, w8t->norm1, w8t->norm2, w8t->q_norm, w8t->k_norm};
      iw8 = dit_block_w{nullptr, nullptr, nullptr, nullptr, w8i->norm1, w8i->norm2, w8i->q_norm, w8i->k_norm};
    }
    wt = &tw8;
    wi = &iw8;
    const int r = pf.start();
    if (r != DIT_OK) return r;
  }
  // W8A8: codes of activation x [R, K] in place before linear i, each stream's rows with its own
  // divisors, and the GEMM's scales (the image rows form the second row group when both streams run;
  // with L = 0 the image stream is the only one and takes every row)
  auto w8a8 = [&](int i, uint16_t* x, int K, GemmParams& g) -> int {
    if (!wqi) return DIT_OK;
    const int r = quant_rows_joint_launch(x, K, nullptr, 0, R, L > 0 ? wqt->smooth[i] : nullptr, wqi->smooth[i], L,
                                          sa, st);
    if (r != DIT_OK) return r;
    g.a_scale = sa;
    g.w_scale = L > 0 ? wqt->scale[i] : wqi->scale[i];
    g.w_scale2 = L > 0 ? wqi->scale[i] : nullptr;
    return DIT_OK;
  };
  // before linear i's GEMMs: its weights ready on the caller's stream; after them: the slot released
  auto before = [&](int i) -> int {
    if (!q8) return DIT_OK;
    const uint16_t* slot;
    const int r = pf.use(i, &slot);
    int n, k;
    linear_shape(d, i, &n, &k);
    const uint16_t* img_w = L > 0 ? slot + size_t(n) * k : slot;
    const uint16_t** ft[4] = {&tw8.wqkv, &tw8.wout, &tw8.wup, &tw8.wdown};
    const uint16_t** fi[4] = {&iw8.wqkv, &iw8.wout, &iw8.wup, &iw8.wdown};
    *ft[i] = L > 0 ? slot : nullptr;
    *fi[i] = img_w;
    return r;
  };
  auto after = [&](int i) -> int { return q8 ? pf.done(i) : DIT_OK; };
  struct Stream {
    const dit_block_w* w;
    int r0, n;
    bool text;
    const dit_lora* lora;  // adapters beside this stream's linears (per-stream launches), or null
  };
  const Stream S[2] = {{wt, 0, L, true, lora_t}, {wi, L, N, false, lora_i}};
  uint16_t* lora_down = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + b.bytes);
  // Sandwich post-norms per stream: post_t / post_i = {attention, MLP} weights of the text / image
  // stream (null entries: that stream's branch un-normed). A branch with a post weight on either
  // stream stores its linear's output in fp32 over h and q (consumed by then), then the sandwich
  // kernel adds gate * f(y) to x, f normalising the rows of the streams that have a weight.
  auto post_of = [&](const float* const* pw, int br) -> const float* { return pw ? pw[br] : nullptr; };
  auto has_post = [&](int br) { return (L > 0 && post_of(post_t, br)) || post_of(post_i, br); };
  float* ybuf = reinterpret_cast<float*>(b.h);
  auto sandwich = [&](int br, long long gate_row) {
    const float* wtx = L > 0 ? post_of(post_t, br) : nullptr;
    const float* wim = post_of(post_i, br);
    SandwichParams sp{txt, img, L, R, H, ybuf, mod.rows + gate_row * H, 6LL * H, mod.map, wtx, d->eps,
                      wtx != nullptr, wim != nullptr, wim};
    return sandwich_launch(sp, st);
  };
  int rc;
  // the text stream's rows are txt[0, L) (all below L); the image stream's img[0, N) (L = 0 here)
  auto norm = [&](const Stream& s, const float* w, long long shift_row) {
    ModNormParams mp{s.text ? txt : nullptr, s.text ? nullptr : img, s.text ? L : 0, s.n, H, H, H, w,
                     mod.rows + shift_row * H, mod.rows + (shift_row + 1) * H, 6LL * H,
                     mod.map ? mod.map + s.r0 : nullptr, d->eps, b.h + size_t(s.r0) * H};
    return modnorm_launch(mp, st);
  };
  auto gated = [&](const Stream& s, int K, long long gate_row) {
    GemmParams g = base_params(s.n, H, K, err);
    g.txt = txt;
    g.img = img;
    g.L = L;
    g.gate = mod.rows + gate_row * H;
    g.map = mod.map;
    g.gate_stride = 6LL * H;
    g.row_off = s.r0;
    return g;
  };

  if (L > 0 && N > 0 && !lora_t && !lora_i) {
    // Every norm and linear runs once over all rows, the GEMMs taking the image weights from row L on
    // (m_split; when L is not on a row-tile boundary each stream's rows are padded to whole tiles, so
    // no tile mixes the streams) and the norms the image norm weights.
    auto norm_all = [&](const float* w_t, const float* w_i, long long shift_row) {
      ModNormParams mp{txt, img, L, R, H, H, H, w_t, mod.rows + shift_row * H, mod.rows + (shift_row + 1) * H,
                       6LL * H, mod.map, d->eps, b.h};
      mp.split_w = 1;
      mp.w_img = w_i;
      return modnorm_launch(mp, st);
    };
    if ((rc = norm_all(wt->norm1, wi->norm1, 0)) != DIT_OK) return rc;
    GemmParams g = qkv_params(d, R, R, L, b, tc, ts, ic, is, wt->q_norm, wt->k_norm, err);
    g.q_norm2 = wi->q_norm;
    g.k_norm2 = wi->k_norm;
    g.m_split = L;
    if ((rc = w8a8(0, b.h, H, g)) != DIT_OK) return rc;
    if ((rc = before(0)) != DIT_OK) return rc;
    if ((rc = gemm_launch_cat(b.h, H, nullptr, 0, wt->wqkv, H, wi->wqkv, H, kEpiQKV, g, st)) != DIT_OK) return rc;
    if ((rc = after(0)) != DIT_OK) return rc;
    AttnParams ap{R, d->heads, d->head_dim, vt_stride(R), b.q, b.k, b.vt, b.o, err, 2, wt->q_norm, wt->k_norm,
                  wi->q_norm, wi->k_norm};
    lend_h(ap, b, R, H);
    if ((rc = attention_launch(ap, st)) != DIT_OK) return rc;
    g = gated(Stream{nullptr, 0, R, false}, H, 2);
    if (has_post(0)) {
      g = base_params(R, H, H, err);
      g.out = ybuf;
      g.ldo = H;
    }
    g.m_split = L;
    if ((rc = w8a8(1, b.o, H, g)) != DIT_OK) return rc;
    if ((rc = before(1)) != DIT_OK) return rc;
    if ((rc = gemm_launch_cat(b.o, H, nullptr, 0, wt->wout, H, wi->wout, H, has_post(0) ? kEpiStoreF32 : kEpiGated, g,
                              st)) != DIT_OK)
      return rc;
    if ((rc = after(1)) != DIT_OK) return rc;
    if (has_post(0) && (rc = sandwich(0, 2)) != DIT_OK) return rc;
    if ((rc = norm_all(wt->norm2, wi->norm2, 3)) != DIT_OK) return rc;
    g = base_params(R, 2 * F, H, err);
    g.out = b.a;
    g.ldo = F;
    g.m_split = L;
    if ((rc = w8a8(2, b.h, H, g)) != DIT_OK) return rc;
    if ((rc = before(2)) != DIT_OK) return rc;
    if ((rc = gemm_launch_cat(b.h, H, nullptr, 0, wt->wup, H, wi->wup, H, kEpiSwiGLU, g, st)) != DIT_OK) return rc;
    if ((rc = after(2)) != DIT_OK) return rc;
    g = gated(Stream{nullptr, 0, R, false}, F, 5);
    if (has_post(1)) {
      g = base_params(R, H, F, err);
      g.out = ybuf;
      g.ldo = H;
    }
    g.m_split = L;
    if ((rc = w8a8(3, b.a, F, g)) != DIT_OK) return rc;
    if ((rc = before(3)) != DIT_OK) return rc;
    if ((rc = gemm_launch_cat(b.a, F, nullptr, 0, wt->wdown, F, wi->wdown, F, has_post(1) ? kEpiStoreF32 : kEpiGated,
                              g, st)) != DIT_OK)
      return rc;
    return has_post(1) ? sandwich(1, 5) : DIT_OK;
  }

  // 1. h = modnorm(x; norm1, shift_a, scale_a), per stream
  for (const Stream& s : S)
    if (s.n > 0 && (rc = norm(s, s.w->norm1, 0)) != DIT_OK) return rc;
  // 2. q, k, vt per stream (its own Wqkv and q/k norm weights) into the joint layouts
  if ((rc = before(0)) != DIT_OK) return rc;
  for (const Stream& s : S) {
    if (s.n == 0) continue;
    GemmParams g = qkv_params(d, s.n, R, L, b, tc, ts, ic, is, s.w->q_norm, s.w->k_norm, err);
    g.row_off = s.r0;
    g.R_total = R;
    if ((rc = w8a8(0, b.h, H, g)) != DIT_OK) return rc;  // (one stream: it runs once)
    if ((rc = gemm_with_lora(s.lora, 0, b.h + size_t(s.r0) * H, H, s.w->wqkv, kEpiQKV, g, lora_down, err, st)) !=
        DIT_OK)
      return rc;
  }
  if ((rc = after(0)) != DIT_OK) return rc;
  // 3. o = attention over all rows (q and k QK-normed with the weights of the streams that have rows)
  const Stream* s0 = S[0].n > 0 ? &S[0] : &S[1];
  const Stream* s1 = (S[0].n > 0 && S[1].n > 0) ? &S[1] : nullptr;
  AttnParams ap{R, d->heads, d->head_dim, vt_stride(R), b.q, b.k, b.vt, b.o, err, s1 ? 2 : 1, s0->w->q_norm,
                s0->w->k_norm, s1 ? s1->w->q_norm : nullptr, s1 ? s1->w->k_norm : nullptr};
  lend_h(ap, b, R, H);
  if ((rc = attention_launch(ap, st)) != DIT_OK) return rc;
  // 4. x += gate_a * (o Wout^T), per stream
  if ((rc = before(1)) != DIT_OK) return rc;
  for (const Stream& s : S) {
    if (s.n == 0) continue;
    GemmParams g = gated(s, H, 2);
    if (has_post(0)) {
      g = base_params(s.n, H, H, err);
      g.out = ybuf + size_t(s.r0) * H;
      g.ldo = H;
    }
    if ((rc = w8a8(1, b.o, H, g)) != DIT_OK) return rc;
    if ((rc = gemm_with_lora(s.lora, 1, b.o + size_t(s.r0) * H, H, s.w->wout, has_post(0) ? kEpiStoreF32 : kEpiGated,
                             g, lora_down, err, st)) != DIT_OK)
      return rc;
  }
  if ((rc = after(1)) != DIT_OK) return rc;
  if (has_post(0) && (rc = sandwich(0, 2)) != DIT_OK) return rc;
  // 5. h2 = modnorm(x; norm2, shift_m, scale_m), per stream
  for (const Stream& s : S)
    if (s.n > 0 && (rc = norm(s, s.w->norm2, 3)) != DIT_OK) return rc;
  // 6. a = SwiGLU(h2 Wup^T), per stream
  if ((rc = before(2)) != DIT_OK) return rc;
  for (const Stream& s : S) {
    if (s.n == 0) continue;
    GemmParams g = base_params(s.n, 2 * F, H, err);
    g.out = b.a + size_t(s.r0) * F;
    g.ldo = F;
    if ((rc = w8a8(2, b.h, H, g)) != DIT_OK) return rc;
    if ((rc = gemm_with_lora(s.lora, 2, b.h + size_t(s.r0) * H, H, s.w->wup, kEpiSwiGLU, g, lora_down, err, st)) !=
        DIT_OK)
      return rc;
  }
  if ((rc = after(2)) != DIT_OK) return rc;
  // 7. x += gate_m * (a Wdown^T), per stream
  if ((rc = before(3)) != DIT_OK) return rc;
  for (const Stream& s : S) {
    if (s.n == 0) continue;
    GemmParams g = gated(s, F, 5);
    if (has_post(1)) {
      g = base_params(s.n, H, F, err);
      g.out = ybuf + size_t(s.r0) * H;
      g.ldo = H;
    }
    if ((rc = w8a8(3, b.a, F, g)) != DIT_OK) return rc;
    if ((rc = gemm_with_lora(s.lora, 3, b.a + size_t(s.r0) * F, F, s.w->wdown, has_post(1) ? kEpiStoreF32 : kEpiGated,
                             g, lora_down, err, st)) != DIT_OK)
      return rc;
  }
  return has_post(1) ? sandwich(1, 5) : DIT_OK;
}

int check_block_args(const dit_dims* d, const float* txt, int L, const float* img, int N, const float* tc,
                     const float* ts, const float* ic, const float* is, const dit_mod* mod, const void* ws,
                     size_t ws_bytes, int variant) {
  if (!d || !mod) return DIT_EINVAL;
  if (!dims_ok(d)) return DIT_EUNSUPPORTED;
  if (L < 0 || N < 1 || (L > 0 && (!txt || !tc || !ts)) || !img || !ic || !is) return DIT_EINVAL;
  if (!mod->rows || mod->M < 1) return DIT_EINVAL;
  if (!al16(txt) || !al16(img) || !al16(mod->rows)) return DIT_EINVAL;
  if (!ws) return DIT_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DIT_EINVAL;
  if (ws_bytes < dit_workspace_bytes(d, L, N, variant)) return DIT_EWORKSPACE;
  return DIT_OK;
}

}  // namespace

int check_block_call_without_workspace(const dit_dims* d, const dit_block_w* w, const float* txt, int L,
                                       const float* img, int N, const float* tc, const float* ts, const float* ic,
                                       const float* is, const dit_mod* mod) {
  if (!d || !mod) return DIT_EINVAL;
  if (!dims_ok(d)) return DIT_EUNSUPPORTED;
  if (L < 0 || N < 1 || (L > 0 && (!txt || !tc || !ts)) || !img || !ic || !is) return DIT_EINVAL;
  if (!mod->rows || mod->M < 1) return DIT_EINVAL;
  if (!al16(txt) || !al16(img) || !al16(mod->rows)) return DIT_EINVAL;
  if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
  if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  return DIT_OK;
}

EncodeTiledFn encode_tiled_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

bool smem_attr_once(const void* kernel, unsigned bytes) {
  const int dev = current_device();
  if (dev < 0) return false;
  constexpr int kKernels = 128;  // more than the library's kernel instantiations
  static const void* done[kMaxDevices][kKernels];
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < kKernels; ++i) {
    if (done[dev][i] == kernel) return true;
    if (!done[dev][i]) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) != cudaSuccess)
        return false;
      done[dev][i] = kernel;
      return true;
    }
  }
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) == cudaSuccess;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 1;
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

}  // namespace dit

using namespace dit;

extern "C" {

int dit_version(void) { return 100; }

const char* dit_status_string(int s) {
  switch (s) {
    case DIT_OK: return "ok";
    case DIT_EINVAL: return "invalid argument (null, size or alignment)";
    case DIT_EUNSUPPORTED: return "shape not supported by the kernels";
    case DIT_EWORKSPACE: return "workspace missing or too small";
    case DIT_ECUDA: return "CUDA error";
    case DIT_ETIMEOUT: return "a bounded device wait timed out";
    default: return "unknown status";
  }
}

size_t dit_workspace_bytes(const dit_dims* d, int L, int N, int variant) {
  if (!dims_ok(d) || L < 0 || N < 1 || variant < 0 || variant > 8) return 0;
  const size_t R = size_t(L) + N;
  size_t bytes = carve_block_ws(d, int(R), nullptr).bytes;
  if (variant == 1) bytes += int8_scratch_bytes(d);
  if (variant == 4) bytes += w8a8_extra_bytes(d, int(R));
  if (variant == 5) bytes += int8_parallel_scratch_bytes(d);
  if (variant == 6) bytes += int8_double_scratch_bytes(d);
  if (variant == 7) bytes += int8_parallel_scratch_bytes(d) + 2 * round_up(R, 64) * sizeof(float);
  if (variant == 8) bytes += int8_double_scratch_bytes(d) + round_up(R * sizeof(float), 256);
  return bytes;
}

int dit_vt_stride(int R) { return R < 0 ? 0 : vt_stride(R); }

int dit_selftest_bounded_wait(int complete, dit_stream_t stream) {
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  return wait_selftest_launch(complete, err, reinterpret_cast<cudaStream_t>(stream));
}

int dit_check(dit_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DIT_ECUDA;
  int* p = err_word();
  if (!p) return DIT_ECUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DIT_ECUDA;
  if (v != 0) {
    // an aborted launch may leave stream-K arrivals counted: clear them with the error word
    gemm_clear_stream_k_counters();
    const int z = 0;
    cudaMemcpy(p, &z, sizeof(int), cudaMemcpyHostToDevice);
    return DIT_ETIMEOUT;
  }
  return DIT_OK;
}

int dit_block_forward(const dit_dims* d, const dit_block_w* w, float* txt, int L, float* img, int N, const float* tc,
                      const float* ts, const float* ic, const float* is, const dit_mod* mod, void* ws,
                      size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 0);
  if (rc != DIT_OK) return rc;
  if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
  if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  return run_block(d, w, nullptr, txt, L, img, N, tc, ts, ic, is, ModRef{mod->rows, mod->map, mod->M}, ws,
                   reinterpret_cast<cudaStream_t>(stream));
}

int dit_parallel_block_forward(const dit_dims* d, const dit_block_w* w, float* txt, int L, float* img, int N,
                               const float* tc, const float* ts, const float* ic, const float* is, const dit_mod* mod,
                               void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 2);
  if (rc != DIT_OK) return rc;
  if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
  if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  if (d->hidden % 256 != 0 || d->ffn % 128 != 0) return DIT_EUNSUPPORTED;  // 256-wide tiles over 3H and 2F
  return run_parallel_block(d, w, nullptr, nullptr, txt, L, img, N, tc, ts, ic, is,
                            ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dit_double_block_forward(const dit_dims* d, const dit_block_w* w_txt, const dit_block_w* w_img, float* txt, int L,
                             float* img, int N, const float* tc, const float* ts, const float* ic, const float* is,
                             const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 3);
  if (rc != DIT_OK) return rc;
  for (const dit_block_w* w : {w_txt, w_img}) {
    if (w == w_txt && L == 0) continue;
    if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
    if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  }
  return run_double_block(d, w_txt, w_img, nullptr, nullptr, nullptr, nullptr, txt, L, img, N, tc, ts, ic, is,
                          ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dit_parallel_block_forward_int8(const dit_dims* d, const dit_block_w8* w, float* txt, int L, float* img, int N,
                                    const float* tc, const float* ts, const float* ic, const float* is,
                                    const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 5);
  if (rc != DIT_OK) return rc;
  if (!w) return DIT_EINVAL;
  if (d->hidden % 256 != 0 || d->ffn % 256 != 0) return DIT_EUNSUPPORTED;
  for (int i = 0; i < 4; ++i)
    if (!w->q[i] || !w->s[i] || !al16(w->q[i]) || !al16(w->s[i])) return DIT_EINVAL;
  return run_parallel_block(d, nullptr, w, nullptr, txt, L, img, N, tc, ts, ic, is,
                            ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dit_double_block_forward_int8(const dit_dims* d, const dit_block_w8* w_txt, const dit_block_w8* w_img, float* txt,
                                  int L, float* img, int N, const float* tc, const float* ts, const float* ic,
                                  const float* is, const dit_mod* mod, void* ws, size_t ws_bytes,
                                  dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 6);
  if (rc != DIT_OK) return rc;
  if (d->hidden % 256 != 0 || d->ffn % 256 != 0) return DIT_EUNSUPPORTED;
  for (const dit_block_w8* w : {w_txt, w_img}) {
    if (w == w_txt && L == 0) continue;
    if (!w) return DIT_EINVAL;
    for (int i = 0; i < 4; ++i)
      if (!w->q[i] || !w->s[i] || !al16(w->q[i]) || !al16(w->s[i])) return DIT_EINVAL;
  }
  return run_double_block(d, nullptr, nullptr, L > 0 ? w_txt : nullptr, w_img, nullptr, nullptr, txt, L, img, N, tc, ts,
                          ic, is, ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dit_parallel_block_forward_w8a8(const dit_dims* d, const dit_parallel_w8a8* w, float* txt, int L, float* img, int N,
                                    const float* tc, const float* ts, const float* ic, const float* is,
                                    const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 7);
  if (rc != DIT_OK) return rc;
  if (!w || !w->q1 || !w->scale1 || !w->q2 || !w->scale2) return DIT_EINVAL;
  if (!al16(w->q1) || !al16(w->q2)) return DIT_EINVAL;
  if (d->hidden % 256 != 0 || d->ffn % 256 != 0) return DIT_EUNSUPPORTED;
  return run_parallel_block(d, nullptr, nullptr, w, txt, L, img, N, tc, ts, ic, is,
                            ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dit_double_block_forward_w8a8(const dit_dims* d, const dit_block_w8a8* w_txt, const dit_block_w8a8* w_img,
                                  float* txt, int L, float* img, int N, const float* tc, const float* ts,
                                  const float* ic, const float* is, const dit_mod* mod, void* ws, size_t ws_bytes,
                                  dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 8);
  if (rc != DIT_OK) return rc;
  if (d->hidden % 256 != 0 || d->ffn % 256 != 0) return DIT_EUNSUPPORTED;
  for (const dit_block_w8a8* w : {w_txt, w_img}) {
    if (w == w_txt && L == 0) continue;
    if (!w) return DIT_EINVAL;
    for (int i = 0; i < 4; ++i)
      if (!w->q[i] || !w->scale[i] || !al16(w->q[i])) return DIT_EINVAL;
  }
  return run_double_block(d, nullptr, nullptr, nullptr, nullptr, L > 0 ? w_txt : nullptr, w_img, txt, L, img, N, tc,
                          ts, ic, is, ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dit_lora_merge(const uint16_t* W, int n_out, int n_in, const uint16_t* A, const uint16_t* B, int rank,
                   uint16_t* merged, dit_stream_t stream) {
  if (!W || !A || !B || !merged || n_out < 1 || n_in < 1 || rank < 1) return DIT_EINVAL;
  if ((n_out + 63) / 64 > 65535) return DIT_EUNSUPPORTED;
  return lora_merge_launch(W, A, B, merged, n_out, n_in, rank, reinterpret_cast<cudaStream_t>(stream));
}

size_t dit_lora_workspace_bytes(const dit_dims* d, int L, int N, int rank) {
  if (!dims_ok(d) || L < 0 || N < 1 || rank < 8 || rank > 1024 || rank % 8 != 0) return 0;
  return carve_block_ws(d, L + N, nullptr).bytes + (size_t(L + N) * lora_rank_pad(rank) * 2 + 255) / 256 * 256;
}

int dit_block_forward_lora(const dit_dims* d, const dit_block_w* w, const dit_lora* lora, float* txt, int L, float* img,
                           int N, const float* tc, const float* ts, const float* ic, const float* is, const dit_mod* mod,
                           void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (!lora) return DIT_EINVAL;
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 0);
  if (rc != DIT_OK) return rc;
  if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
  if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  if (lora->rank < 8 || lora->rank > 1024 || lora->rank % 8 != 0) return DIT_EUNSUPPORTED;
  for (int i = 0; i < 4; ++i) {
    if ((lora->A[i] == nullptr) != (lora->B[i] == nullptr)) return DIT_EINVAL;
    if (lora->A[i] && (!al16(lora->A[i]) || !al16(lora->B[i]))) return DIT_EINVAL;
  }
  if (ws_bytes < dit_lora_workspace_bytes(d, L, N, lora->rank)) return DIT_EWORKSPACE;
  return run_block(d, w, nullptr, txt, L, img, N, tc, ts, ic, is, ModRef{mod->rows, mod->map, mod->M}, ws,
                   reinterpret_cast<cudaStream_t>(stream), lora);
}

namespace {
// Pre-launch checks of a LoRA adapter set: rank within [8, 1024], a multiple of 8; each linear's two
// factors both given or both absent, 16-byte aligned.
int check_lora(const dit_lora* lora) {
  if (!lora) return DIT_EINVAL;
  if (lora->rank < 8 || lora->rank > 1024 || lora->rank % 8 != 0) return DIT_EUNSUPPORTED;
  for (int i = 0; i < 4; ++i) {
    if ((lora->A[i] == nullptr) != (lora->B[i] == nullptr)) return DIT_EINVAL;
    if (lora->A[i] && (!al16(lora->A[i]) || !al16(lora->B[i]))) return DIT_EINVAL;
  }
  return DIT_OK;
}
}  // namespace

int dit_parallel_block_forward_lora(const dit_dims* d, const dit_block_w* w, const dit_lora* lora, float* txt, int L,
                                    float* img, int N, const float* tc, const float* ts, const float* ic,
                                    const float* is, const dit_mod* mod, void* ws, size_t ws_bytes,
                                    dit_stream_t stream) {
  if (!lora) return DIT_EINVAL;
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 2);
  if (rc != DIT_OK) return rc;
  if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
  if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  if ((rc = check_lora(lora)) != DIT_OK) return rc;
  if (ws_bytes < dit_lora_workspace_bytes(d, L, N, lora->rank)) return DIT_EWORKSPACE;
  return run_parallel_block(d, w, nullptr, nullptr, txt, L, img, N, tc, ts, ic, is,
                            ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream), lora);
}

int dit_double_block_forward_lora(const dit_dims* d, const dit_block_w* w_txt, const dit_lora* lora_txt,
                                  const dit_block_w* w_img, const dit_lora* lora_img, float* txt, int L, float* img,
                                  int N, const float* tc, const float* ts, const float* ic, const float* is,
                                  const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 3);
  if (rc != DIT_OK) return rc;
  if (!lora_img && (L == 0 || !lora_txt)) return DIT_EINVAL;  // at least one adapter set
  int rank = 0;
  for (const dit_lora* lr : {L > 0 ? lora_txt : nullptr, lora_img}) {
    if (!lr) continue;
    if ((rc = check_lora(lr)) != DIT_OK) return rc;
    rank = std::max(rank, lr->rank);
  }
  for (const dit_block_w* w : {w_txt, w_img}) {
    if (w == w_txt && L == 0) continue;
    if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
    if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  }
  if (ws_bytes < dit_lora_workspace_bytes(d, L, N, rank)) return DIT_EWORKSPACE;
  return run_double_block(d, w_txt, w_img, nullptr, nullptr, nullptr, nullptr, txt, L, img, N, tc, ts, ic, is,
                          ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream),
                          L > 0 ? lora_txt : nullptr, lora_img);
}

int dit_parallel_block_forward_sandwich(const dit_dims* d, const dit_block_w* w, const float* post_attn,
                                        const float* post_mlp, float* txt, int L, float* img, int N, const float* tc,
                                        const float* ts, const float* ic, const float* is, const dit_mod* mod,
                                        void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 2);
  if (rc != DIT_OK) return rc;
  if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
  if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  if ((post_attn && !al16(post_attn)) || (post_mlp && !al16(post_mlp))) return DIT_EINVAL;
  return run_parallel_block(d, w, nullptr, nullptr, txt, L, img, N, tc, ts, ic, is,
                            ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream), nullptr,
                            post_attn, post_mlp);
}

int dit_double_block_forward_sandwich(const dit_dims* d, const dit_block_w* w_txt, const float* post_attn_txt,
                                      const float* post_mlp_txt, const dit_block_w* w_img, const float* post_attn_img,
                                      const float* post_mlp_img, float* txt, int L, float* img, int N,
                                      const float* tc, const float* ts, const float* ic, const float* is,
                                      const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 3);
  if (rc != DIT_OK) return rc;
  for (const dit_block_w* w : {w_txt, w_img}) {
    if (w == w_txt && L == 0) continue;
    if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
    if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  }
  for (const float* p : {post_attn_txt, post_mlp_txt, post_attn_img, post_mlp_img})
    if (p && !al16(p)) return DIT_EINVAL;
  const float* pt[2] = {post_attn_txt, post_mlp_txt};
  const float* pi[2] = {post_attn_img, post_mlp_img};
  return run_double_block(d, w_txt, w_img, nullptr, nullptr, nullptr, nullptr, txt, L, img, N, tc, ts, ic, is,
                          ModRef{mod->rows, mod->map, mod->M}, ws, reinterpret_cast<cudaStream_t>(stream), nullptr,
                          nullptr, pt, pi);
}

int dit_block_forward_sandwich(const dit_dims* d, const dit_block_w* w, const float* post_attn, const float* post_mlp,
                               float* txt, int L, float* img, int N, const float* tc, const float* ts, const float* ic,
                               const float* is, const dit_mod* mod, void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 0);
  if (rc != DIT_OK) return rc;
  if (!w || !w->wqkv || !w->wout || !w->wup || !w->wdown) return DIT_EINVAL;
  if (!al16(w->wqkv) || !al16(w->wout) || !al16(w->wup) || !al16(w->wdown)) return DIT_EINVAL;
  if ((post_attn && !al16(post_attn)) || (post_mlp && !al16(post_mlp))) return DIT_EINVAL;
  return run_block(d, w, nullptr, txt, L, img, N, tc, ts, ic, is, ModRef{mod->rows, mod->map, mod->M}, ws,
                   reinterpret_cast<cudaStream_t>(stream), nullptr, post_attn, post_mlp);
}

int dit_block_forward_w8a8(const dit_dims* d, const dit_block_w8a8* w, float* txt, int L, float* img, int N,
                           const float* tc, const float* ts, const float* ic, const float* is, const dit_mod* mod,
                           void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 4);
  if (rc != DIT_OK) return rc;
  if (!w) return DIT_EINVAL;
  for (int i = 0; i < 4; ++i)
    if (!w->q[i] || !w->scale[i] || !al16(w->q[i]) || !al16(w->scale[i])) return DIT_EINVAL;
  return run_block_w8a8(d, w, txt, L, img, N, tc, ts, ic, is, ModRef{mod->rows, mod->map, mod->M}, ws,
                        reinterpret_cast<cudaStream_t>(stream));
}

int dit_w8a8_quantize_weight(const uint16_t* w, int N, int K, const float* smooth, int8_t* q, float* scale,
                             dit_stream_t stream) {
  if (!w || !q || !scale || N < 1 || K < 1) return DIT_EINVAL;
  return quant_weight_launch(w, N, K, smooth, q, scale, reinterpret_cast<cudaStream_t>(stream));
}

int dit_w8a8_quantize_rows(uint16_t* x, int R, int K, const float* smooth, float* scale, dit_stream_t stream) {
  if (!x || !scale || R < 1 || K < 1) return DIT_EINVAL;
  if (K % 8 != 0) return DIT_EUNSUPPORTED;
  if (!al16(x)) return DIT_EINVAL;
  return quant_rows_launch(x, R, K, smooth, scale, reinterpret_cast<cudaStream_t>(stream));
}

size_t dit_linear_w8a8_workspace_bytes(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 1) return 0;
  return round_up(size_t(M) * K * 2, 256) + round_up(size_t(N) * K * 2, 256) + round_up(size_t(M) * 4, 256);
}

int dit_linear_w8a8(const uint16_t* a, int M, int K, const int8_t* q, const float* scale, const float* smooth, int N,
                    float* out, void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (!a || !q || !scale || !out || M < 1 || N < 1 || K < 1) return DIT_EINVAL;
  if (K % 64 != 0 || N % 64 != 0) return DIT_EUNSUPPORTED;
  if (!al16(a) || !al16(q) || !al16(out) || !ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DIT_EINVAL;
  if (ws_bytes < dit_linear_w8a8_workspace_bytes(M, N, K)) return DIT_EWORKSPACE;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* p = static_cast<uint8_t*>(ws);
  uint16_t* ac = reinterpret_cast<uint16_t*>(p);
  uint16_t* wc = reinterpret_cast<uint16_t*>(p + round_up(size_t(M) * K * 2, 256));
  float* sa = reinterpret_cast<float*>(p + round_up(size_t(M) * K * 2, 256) + round_up(size_t(N) * K * 2, 256));
  if (cudaMemcpyAsync(ac, a, size_t(M) * K * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return DIT_ECUDA;
  int rc = quant_rows_launch(ac, M, K, smooth, sa, st);
  if (rc == DIT_OK) rc = codes_bf16_launch(q, wc, (long long)N * K, st);
  if (rc != DIT_OK) return rc;
  GemmParams g = base_params(M, N, K, err);
  g.out = out;
  g.ldo = N;
  g.a_scale = sa;
  g.w_scale = scale;
  return gemm_launch(ac, K, wc, nullptr, kEpiStoreF32, g, st);
}

int dit_block_forward_int8(const dit_dims* d, const dit_block_w8* w, float* txt, int L, float* img, int N,
                           const float* tc, const float* ts, const float* ic, const float* is, const dit_mod* mod,
                           void* ws, size_t ws_bytes, dit_stream_t stream) {
  int rc = check_block_args(d, txt, L, img, N, tc, ts, ic, is, mod, ws, ws_bytes, 1);
  if (rc != DIT_OK) return rc;
  if (!w) return DIT_EINVAL;
  if (d->hidden % 256 != 0 || d->ffn % 256 != 0) return DIT_EUNSUPPORTED;  // int8lin: every K % 256 == 0
  for (int i = 0; i < 4; ++i)
    if (!w->q[i] || !w->s[i] || !al16(w->q[i]) || !al16(w->s[i])) return DIT_EINVAL;
  return run_block(d, nullptr, w, txt, L, img, N, tc, ts, ic, is, ModRef{mod->rows, mod->map, mod->M}, ws,
                   reinterpret_cast<cudaStream_t>(stream));
}

int dit_euler_step(float* x, const float* vel, int64_t n, float sigma, float sigma_next, dit_stream_t stream) {
  if (n < 0 || (n > 0 && (!x || !vel))) return DIT_EINVAL;
  return euler_launch(x, vel, n, sigma, sigma_next, reinterpret_cast<cudaStream_t>(stream));
}

int dit_rope_tables(int L, int gh, int gw, int head_dim, float theta, float* cos, float* sin, dit_stream_t stream) {
  if (L < 0 || gh < 1 || gw < 1 || !cos || !sin || !(theta > 0.f)) return DIT_EINVAL;
  if (head_dim != 64 && head_dim != 128) return DIT_EUNSUPPORTED;
  return rope_tables_launch(L, gh, gw, head_dim, theta, cos, sin, reinterpret_cast<cudaStream_t>(stream));
}

int dit_modnorm(const dit_dims* d, const float* txt, int L, const float* img, int N, const float* w,
                const dit_mod* mod, int which, uint16_t* h, dit_stream_t stream) {
  if (!d || !mod || !h || !img || L < 0 || N < 1 || (L > 0 && !txt) || (which != 0 && which != 1)) return DIT_EINVAL;
  if (d->hidden <= 0 || d->hidden % 4 != 0) return DIT_EUNSUPPORTED;
  if (!mod->rows || mod->M < 1 || !al16(img) || (txt && !al16(txt)) || !al16(mod->rows) || !al16(h) ||
      (w && !al16(w)))
    return DIT_EINVAL;
  const int H = d->hidden;
  ModNormParams mp{txt, img, L, L + N, H, H, H, w, mod->rows + 3LL * which * H, mod->rows + (3LL * which + 1) * H,
                   6LL * H, mod->map, d->eps, h};
  return modnorm_launch(mp, reinterpret_cast<cudaStream_t>(stream));
}

size_t dit_stream_k_workspace_bytes(void) {
  // two fp32 partial slots of a 128 x 256 tile slab per SM (CTA pairs: two slabs per pair unit)
  return size_t(num_sms()) * 2 * 128 * 256 * sizeof(float);
}

int dit_qkv_rope(const dit_dims* d, const uint16_t* h, int L, int N, const uint16_t* wqkv, const float* q_norm,
                 const float* k_norm, const float* tc, const float* ts, const float* ic, const float* is, uint16_t* q,
                 uint16_t* k, uint16_t* vt, void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (!d || !h || !wqkv || !q || !k || !vt || L < 0 || N < 1 || !ic || !is || (L > 0 && (!tc || !ts)))
    return DIT_EINVAL;
  if (!dims_ok(d)) return DIT_EUNSUPPORTED;
  if (!al16(h) || !al16(wqkv) || !al16(q) || !al16(k) || !al16(vt)) return DIT_EINVAL;
  if (ws && reinterpret_cast<uintptr_t>(ws) % 256 != 0) return DIT_EINVAL;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  const int R = L + N, H = d->hidden;
  GemmParams g = base_params(R, 3 * H, H, err);
  g.q = q;
  g.k = k;
  g.vt = vt;
  g.H = H;
  g.heads = d->heads;
  g.head_dim = d->head_dim;
  g.Rp = vt_stride(R);
  g.L = L;
  g.txt_cos = tc;
  g.txt_sin = ts;
  g.img_cos = ic;
  g.img_sin = is;
  g.q_norm = q_norm;
  g.k_norm = k_norm;
  g.qk_eps = d->qk_eps;
  g.rope_split = d->rope_split;
  g.split_ws = ws_bytes ? ws : nullptr;
  g.split_ws_bytes = ws ? ws_bytes : 0;
  return gemm_launch(h, H, wqkv, nullptr, kEpiQKV, g, reinterpret_cast<cudaStream_t>(stream));
}

size_t dit_attention_workspace_bytes(const dit_dims* d, int R) {
  if (!d || R < 1 || !dims_ok(d)) return 0;
  return attention_part_bytes(R, d->heads, d->head_dim);
}

int dit_attention(const dit_dims* d, int R, const uint16_t* q, const uint16_t* k, const uint16_t* vt, uint16_t* o,
                  void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (!d || R < 1 || !q || !k || !vt || !o) return DIT_EINVAL;
  if (!dims_ok(d)) return DIT_EUNSUPPORTED;
  if (!al16(q) || !al16(k) || !al16(vt) || !al16(o) || (ws && !al16(ws))) return DIT_EINVAL;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  AttnParams ap{R, d->heads, d->head_dim, vt_stride(R), q, k, vt, o, err};
  ap.part = ws_bytes ? ws : nullptr;
  ap.part_bytes = ws ? ws_bytes : 0;
  return attention_launch(ap, reinterpret_cast<cudaStream_t>(stream));
}

int dit_attention_qknorm(const dit_dims* d, int R, const uint16_t* q, const uint16_t* k, const uint16_t* vt,
                         const float* q_norm, const float* k_norm, uint16_t* o, void* ws, size_t ws_bytes,
                         dit_stream_t stream) {
  if (!d || R < 1 || !q || !k || !vt || !o) return DIT_EINVAL;
  if (!dims_ok(d)) return DIT_EUNSUPPORTED;
  if (!al16(q) || !al16(k) || !al16(vt) || !al16(o) || (ws && !al16(ws))) return DIT_EINVAL;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  AttnParams ap{R, d->heads, d->head_dim, vt_stride(R), q, k, vt, o, err, 1, q_norm, k_norm, nullptr, nullptr};
  ap.part = ws_bytes ? ws : nullptr;
  ap.part_bytes = ws ? ws_bytes : 0;
  return attention_launch(ap, reinterpret_cast<cudaStream_t>(stream));
}

int dit_linear_gated(const dit_dims* d, const uint16_t* a, int L, int N, const uint16_t* w, const dit_mod* mod,
                     int which, float* txt, float* img, void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (!d || !a || !w || !mod || !mod->rows || mod->M < 1 || !img || L < 0 || N < 1 || (L > 0 && !txt) ||
      (which != 0 && which != 1))
    return DIT_EINVAL;
  if (!dims_ok(d)) return DIT_EUNSUPPORTED;
  if (!al16(a) || !al16(w) || !al16(img) || (txt && !al16(txt)) || !al16(mod->rows)) return DIT_EINVAL;
  if (ws && reinterpret_cast<uintptr_t>(ws) % 256 != 0) return DIT_EINVAL;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  const int H = d->hidden, K = which == 0 ? H : d->ffn;
  GemmParams g = base_params(L + N, H, K, err);
  g.txt = txt;
  g.img = img;
  g.L = L;
  g.gate = mod->rows + (which == 0 ? 2LL : 5LL) * H;
  g.map = mod->map;
  g.gate_stride = 6LL * H;
  g.split_ws = ws_bytes ? ws : nullptr;
  g.split_ws_bytes = ws ? ws_bytes : 0;
  return gemm_launch(a, K, w, nullptr, kEpiGated, g, reinterpret_cast<cudaStream_t>(stream));
}

int dit_linear_swiglu(const dit_dims* d, const uint16_t* h2, int R, const uint16_t* wup, uint16_t* a, void* ws,
                      size_t ws_bytes, dit_stream_t stream) {
  if (!d || !h2 || !wup || !a || R < 1) return DIT_EINVAL;
  if (!dims_ok(d)) return DIT_EUNSUPPORTED;
  if (!al16(h2) || !al16(wup) || !al16(a)) return DIT_EINVAL;
  if (ws && reinterpret_cast<uintptr_t>(ws) % 256 != 0) return DIT_EINVAL;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  GemmParams g = base_params(R, 2 * d->ffn, d->hidden, err);
  g.out = a;
  g.ldo = d->ffn;
  g.split_ws = ws_bytes ? ws : nullptr;
  g.split_ws_bytes = ws ? ws_bytes : 0;
  return gemm_launch(h2, d->hidden, wup, nullptr, kEpiSwiGLU, g, reinterpret_cast<cudaStream_t>(stream));
}

int dit_linear(const uint16_t* a, int M, int K, const uint16_t* w, int N, void* out, int out_bf16,
               dit_stream_t stream) {
  if (!a || !w || !out || M < 1 || K < 1 || N < 1) return DIT_EINVAL;
  if (K % 64 != 0 || N % 64 != 0) return DIT_EUNSUPPORTED;
  if (!al16(a) || !al16(w) || !al16(out)) return DIT_EINVAL;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  GemmParams g = base_params(M, N, K, err);
  g.out = out;
  g.ldo = N;
  return gemm_launch(a, K, w, nullptr, out_bf16 ? kEpiStoreBF16 : kEpiStoreF32, g,
                     reinterpret_cast<cudaStream_t>(stream));
}

size_t dit_linear_int8_workspace_bytes(int N, int K) {
  if (N < 1 || K < 1) return 0;
  return gemm_int8_scratch_bytes(N, K);
}

int dit_linear_int8(const uint16_t* a, int M, int K, const int8_t* wq, const uint16_t* wsc, int N, float* out,
                    void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (!a || !wq || !wsc || !out || M < 1 || K < 1 || N < 1) return DIT_EINVAL;
  if (K % 256 != 0 || N % 128 != 0) return DIT_EUNSUPPORTED;
  if (!al16(a) || !al16(wq) || !al16(wsc) || !al16(out)) return DIT_EINVAL;
  if (!ws) return DIT_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DIT_EINVAL;
  if (ws_bytes < dit_linear_int8_workspace_bytes(N, K)) return DIT_EWORKSPACE;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  GemmParams g = base_params(M, N, K, err);
  g.out = out;
  g.ldo = N;
  GemmInt8B b8{wq, wsc, static_cast<uint16_t*>(ws)};
  return gemm_launch(a, K, nullptr, &b8, kEpiStoreF32, g, reinterpret_cast<cudaStream_t>(stream));
}

int dit_dequant_int8(const int8_t* q, const uint16_t* s, int64_t rows, int64_t cols, uint16_t* w,
                     dit_stream_t stream) {
  if (!q || !s || !w || rows < 0 || cols < 0) return DIT_EINVAL;
  if (cols % 32 != 0) return DIT_EUNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(w) % 16 || reinterpret_cast<uintptr_t>(q) % 16) return DIT_EINVAL;
  return dequant_int8_launch(q, s, w, rows, cols, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------------------------------
// denoise
// ------------------------------------------------------------------------------------------
namespace {
struct DenoiseWs {
  float* rows;      // [R, H] fp32: text rows then image rows
  uint8_t* block;   // block workspace
  uint16_t* xin;    // [N, C] bf16
  uint16_t* emb;    // [steps, 256] bf16
  uint16_t* t1;     // [steps, H] bf16
  uint16_t* st;     // [steps, H] bf16 = silu(temb)
  float* mods;      // [steps, blocks * 6H] fp32
  float* fin;       // [steps, 2H] fp32
  float* vel;       // [N, C] fp32
  size_t bytes;
};

DenoiseWs carve_denoise(const dit_model* m, int L, int N, int steps, void* base) {
  DenoiseWs w{};
  const size_t H = m->dims.hidden, C = m->latent_channels, R = size_t(L) + N;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* r = p ? p + off : nullptr;
    off += round_up(bytes, 256);
    return r;
  };
  w.rows = reinterpret_cast<float*>(take(R * H * 4));
  w.block = take(carve_block_ws(&m->dims, int(R), nullptr).bytes);
  w.xin = reinterpret_cast<uint16_t*>(take(size_t(N) * C * 2));
  w.emb = reinterpret_cast<uint16_t*>(take(size_t(steps) * 256 * 2));
  w.t1 = reinterpret_cast<uint16_t*>(take(size_t(steps) * H * 2));
  w.st = reinterpret_cast<uint16_t*>(take(size_t(steps) * H * 2));
  w.mods = reinterpret_cast<float*>(take(size_t(steps) * m->blocks * 6 * H * 4));
  w.fin = reinterpret_cast<float*>(take(size_t(steps) * 2 * H * 4));
  w.vel = reinterpret_cast<float*>(take(size_t(N) * C * 4));
  w.bytes = off;
  return w;
}

bool model_ok(const dit_model* m) {
  if (!m || !dims_ok(&m->dims) || m->blocks < 0 || m->latent_channels < 64 || m->latent_channels % 64 != 0)
    return false;
  return true;
}
}  // namespace

size_t dit_denoise_workspace_bytes(const dit_model* m, int L, int N, int steps) {
  if (!model_ok(m) || L < 0 || N < 1 || steps < 1 || steps > 64) return 0;
  return carve_denoise(m, L, N, steps, nullptr).bytes;
}

int dit_denoise(const dit_model* m, float* x, int N, const float* txt_feats, int L, const float* sigmas, int steps,
                const float* tc, const float* ts, const float* ic, const float* is, void* ws, size_t ws_bytes,
                dit_stream_t stream) {
  if (!m || !x || !sigmas || N < 1 || L < 0 || (L > 0 && (!txt_feats || !tc || !ts)) || !ic || !is) return DIT_EINVAL;
  if (!model_ok(m) || steps < 1 || steps > 64) return DIT_EUNSUPPORTED;
  if (!m->w_in || !m->w_t1 || !m->w_t2 || !m->w_ada_f || !m->w_out || (m->blocks > 0 && (!m->w_ada || !m->block)))
    return DIT_EINVAL;
  for (int b = 0; b < m->blocks; ++b) {
    const dit_block_w& bw = m->block[b];
    if (!bw.wqkv || !bw.wout || !bw.wup || !bw.wdown) return DIT_EINVAL;
    if (!al16(bw.wqkv) || !al16(bw.wout) || !al16(bw.wup) || !al16(bw.wdown)) return DIT_EINVAL;
  }
  if (!al16(x) || (txt_feats && !al16(txt_feats)) || !al16(m->w_in) || !al16(m->w_t1) || !al16(m->w_t2) ||
      (m->w_ada && !al16(m->w_ada)) || !al16(m->w_ada_f) || !al16(m->w_out))
    return DIT_EINVAL;
  if (!ws) return DIT_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DIT_EINVAL;
  if (ws_bytes < dit_denoise_workspace_bytes(m, L, N, steps)) return DIT_EWORKSPACE;
  int* err = err_word();
  if (!err) return DIT_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const dit_dims* d = &m->dims;
  const int H = d->hidden, C = m->latent_channels, R = L + N;
  const DenoiseWs w = carve_denoise(m, L, N, steps, ws);
  const long long SB = 6LL * H * m->blocks;
  int rc;

  // step-invariant work: time embeddings and every modulation row for all steps
  if ((rc = sinusoid_launch(sigmas, steps, 256, w.emb, st)) != DIT_OK) return rc;
  GemmParams g = base_params(steps, H, 256, err);
  g.out = w.t1;
  g.ldo = H;
  if ((rc = gemm_launch(w.emb, 256, m->w_t1, nullptr, kEpiSiluBF16, g, st)) != DIT_OK) return rc;
  g = base_params(steps, H, H, err);
  g.out = w.st;
  g.ldo = H;
  if ((rc = gemm_launch(w.t1, H, m->w_t2, nullptr, kEpiSiluBF16, g, st)) != DIT_OK) return rc;
  if (m->blocks > 0) {
    g = base_params(steps, int(SB), H, err);
    g.out = w.mods;
    g.ldo = SB;
    if ((rc = gemm_launch(w.st, H, m->w_ada, nullptr, kEpiStoreF32, g, st)) != DIT_OK) return rc;
  }
  g = base_params(steps, 2 * H, H, err);
  g.out = w.fin;
  g.ldo = 2 * H;
  if ((rc = gemm_launch(w.st, H, m->w_ada_f, nullptr, kEpiStoreF32, g, st)) != DIT_OK) return rc;

  float* txt_rows = w.rows;
  float* img_rows = w.rows + size_t(L) * H;
  for (int i = 0; i < steps; ++i) {
    if (L > 0 && cudaMemcpyAsync(txt_rows, txt_feats, size_t(L) * H * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return DIT_ECUDA;
    if ((rc = f32_to_bf16_launch(x, w.xin, (long long)N * C, st)) != DIT_OK) return rc;
    g = base_params(N, H, C, err);
    g.out = img_rows;
    g.ldo = H;
    if ((rc = gemm_launch(w.xin, C, m->w_in, nullptr, kEpiStoreF32, g, st)) != DIT_OK) return rc;
    for (int b = 0; b < m->blocks; ++b) {
      const ModRef mod{w.mods + i * SB + 6LL * H * b, nullptr, 1};
      if ((rc = run_block(d, &m->block[b], nullptr, txt_rows, L, img_rows, N, tc, ts, ic, is, mod, w.block, st)) !=
          DIT_OK)
        return rc;
    }
    const BlockWs bw = carve_block_ws(d, R, w.block);
    ModNormParams mp{nullptr, img_rows, 0, N, H, H, H, nullptr, w.fin + 2LL * H * i, w.fin + 2LL * H * i + H, 0,
                     nullptr, d->eps, bw.h};
    if ((rc = modnorm_launch(mp, st)) != DIT_OK) return rc;
    g = base_params(N, C, H, err);
    g.out = w.vel;
    g.ldo = C;
    if ((rc = gemm_launch(bw.h, H, m->w_out, nullptr, kEpiStoreF32, g, st)) != DIT_OK) return rc;
    if ((rc = euler_launch(x, w.vel, (long long)N * C, sigmas[i], sigmas[i + 1], st)) != DIT_OK) return rc;
  }
  return DIT_OK;
}

}  // extern "C"
