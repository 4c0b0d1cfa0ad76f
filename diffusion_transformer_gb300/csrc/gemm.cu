// Persistent warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
//   C[M, N] = A[M, K] * B[N, K]^T     A, B bf16 K-major, fp32 accumulators in TMEM
//
// One CTA per SM walks output tiles (128 x BN) in a static round-robin order. Warp 0 issues TMA
// loads of A and B k-blocks (64 wide, 128-byte swizzle) into a STAGES-deep shared-memory ring;
// warp 1 issues tcgen05.mma (M=128, N=BN, K=16) into one of two TMEM accumulators; warps 2-5 drain
// the other accumulator through the epilogue, so a tile's epilogue overlaps the next tile's
// mainloop. For int8lin weights (B8 = true) warps 6-9 convert each int8 k-block of B with its bf16
// block-32 scales (both brought in by TMA) into the bf16 swizzled tile the MMA reads:
// w = bf16_rne(q * s) (the host contract's int8lin scheme, section 1), inside the mainloop.
// PAIR = true: two CTAs of a cluster on two SMs share one 256 x BN tile (each brings its 128 rows
// of A and BN/2 rows of B; the first issues cta_group::2 MMAs over both), so a k-block costs each SM
// a third less shared-memory fill; every cross-CTA wait is a bounded mbarrier wait (see below).
// W8A8 (a_scale / w_scale set): the accumulator, an exact integer dot product of codes, is scaled
// in TMEM by the row's and the column's scales before the epilogue.
//
// Epilogues (the gizai:dit reference's linearInto / gatedInto / gluRows / prepOf):
//   kEpiStoreF32 / kEpiStoreBF16 / kEpiSiluBF16   plain stores
//   kEpiGated   x += gate[map[r]] * acc            (out and down linears)
//   kEpiSwiGLU  a_j = silu(acc_2j) * acc_2j+1      (up linear, interleaved rows)
//   kEpiQKV     per-head RMS norm * weight, rotary pairs (2i, 2i+1), head-major q/k stores and a
//               transposed v store for the attention kernel (klein article, section 4.4)
//   kEpiQKVSwiGLU  kEpiQKV on the columns below n_split, kEpiSwiGLU above (the parallel block)
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace dit {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kSkMaxParts = 3;  // stream-K segments per tile at most (the plan guarantees it)

template <int BN, bool B8, bool PAIR = false>
struct GemmCfg {
  // int8lin: 256-row CTA tiles (two M=128 MMAs share each converted B k-block), halving the
  // conversions per FLOP; bf16: 128-row tiles, or 256 x BN tiles shared by a CTA pair (PAIR: each CTA
  // brings its 128 rows of A and half of the B tile, the first CTA issues M=256 MMAs over both).
  static constexpr int kMH = (B8 && !PAIR) ? 2 : 1;  // 128-row halves per CTA tile
  static constexpr int kTileM = PAIR ? 2 * BM : BM * kMH;  // rows of one work tile
  static constexpr int kStages = B8 ? (PAIR ? 5 : (BN == 256 ? 3 : 4))
                                    : PAIR ? (BN == 256 ? 6 : 8) : (BN == 256 ? 4 : (BN == 128 ? 6 : 8));
  // TMEM accumulator sets: two (the epilogue drains one while the MMA fills the other) when they fit
  // in the 512 columns, else one.
  static constexpr int kAccBufs = (2 * kMH * BN <= 512) ? 2 : 1;
  static constexpr uint32_t kAHalf = BM * BK * 2;
  static constexpr uint32_t kABytes = kAHalf * kMH;
  static constexpr int kBRows = PAIR ? BN / 2 : BN;  // rows of B this CTA brings (PAIR: its half)
  static constexpr uint32_t kBLoad = kBRows * BK * 2;  // bf16 B bytes this CTA holds per stage (B8: converted)
  static constexpr uint32_t kB8Bytes = kBRows * BK;  // int8 tile TMA writes (B8 only)
  static constexpr uint32_t kSBytes = kBRows * 16;   // B8: scale tile [rows x 8 bf16] (4 k-blocks)
  static constexpr int kConvStages = PAIR ? 4 : 2;   // bf16 B tiles produced by the converters
  static constexpr int kConvThreads = 128;           // B8: converter warps 6..9, one per SM sub-partition
  static constexpr uint32_t kTmemCols = (kAccBufs * kMH * BN < 32) ? 32 : kAccBufs * kMH * BN;
  // epilogue warps: one per TMEM lane quadrant (two per quadrant, each taking half of the columns,
  // measured no faster)
  static constexpr int kEpiWarps = 4;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kEpiCols = BN / (kEpiWarps / 4);   // columns per epilogue warp
  static constexpr int kConvWarp0 = 2 + kEpiWarps;         // first converter warp (B8)
  static constexpr int kThreads = 64 + kEpiThreads + (B8 ? kConvThreads : 0);
  // smem: [A ring][B ring (bf16, or int8 + scales for B8)][B8: converted bf16 ring][barriers][tmem slot]
  static constexpr uint32_t kRingBytes = kStages * (kABytes + (B8 ? kB8Bytes + kSBytes : kBLoad));
  static constexpr uint32_t kConvBytes = B8 ? kConvStages * kBLoad : 0;
  static constexpr uint32_t kEpiBytes = kEpiWarps * 4096;   // epilogue staging, 4 KB per epilogue warp
  static constexpr uint32_t kBarBytes = 8 * (2 * kStages + 4 + 2 * kConvStages + 3) + 16;
  static constexpr uint32_t kSmemBytes = 1024 + kRingBytes + kConvBytes + kEpiBytes + kBarBytes;
};

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
    u.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
    u.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
    u.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
    d[c] = u;
  }
}

// ----------------------------------------------------------------------------------------------
// epilogues: thread `lane` of epilogue warp `quad` owns TMEM lane quad * 32 + lane, i.e. output row
// row0 + lane of the warp's 32-row slab; taddr points at (its lane, column n0). tcgen05.ld is
// warp-collective, so every lane loads even when its row is out of range. `stage` is this warp's
// 4 KB shared-memory scratch (the transposed v store, the gated residual's transpose). BN here is
// the warp's column count.
// ----------------------------------------------------------------------------------------------
template <int BN, int EPI, bool kRowPerThread>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t taddr, int row0, int row_end, int lane,
                                              int n0, uint8_t* stage) {
  const int row = row0 + lane;
  const bool row_ok = row < row_end;
  if constexpr (EPI == kEpiQKV) {
    const int d = p.head_dim;
    const int H = p.H;
    const int R = p.R_total > 0 ? p.R_total : p.M;  // rows of the q, k and vt layouts
    const int srow = row + p.row_off;                // sequence row of this thread's GEMM row
    const int tw = p.rope_split ? 3 * d / 8 : d / 2;  // rotary table columns per row
    for (int hh = 0; hh < BN / d; ++hh) {
      const int col0 = n0 + hh * d;
      const int which = col0 / H;              // 0 = q, 1 = k, 2 = v
      const int head = (col0 - which * H) / d;
      const uint32_t ta = taddr + hh * d;
      if (which == 2) {
        // v, transposed: vt[head*d + j][row]. Stage the warp's 32 rows x 32 values as bf16 (64 B
        // per row, 16-byte chunks XOR-swizzled by (row >> 1) & 3), then lane j writes value j of
        // all 32 rows as 64 contiguous bytes.
        uint32_t* st32 = reinterpret_cast<uint32_t*>(stage);
        for (int c = 0; c < d / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(ta + c * 32, v);
          tmem_ld_wait();
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int slot = q ^ ((lane >> 1) & 3);
            *reinterpret_cast<uint4*>(stage + lane * 64 + slot * 16) =
                make_uint4(pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
          }
          __syncwarp();
          const int j = lane;  // value index within the chunk
          uint32_t col[16];
#pragma unroll
          for (int r = 0; r < 32; r += 2) {
            const int o0 = r * 64 + (((j >> 3) ^ ((r >> 1) & 3)) << 4) + (j & 7) * 2;
            const int o1 = (r + 1) * 64 + (((j >> 3) ^ (((r + 1) >> 1) & 3)) << 4) + (j & 7) * 2;
            const uint32_t lo = *reinterpret_cast<const uint16_t*>(stage + o0);
            const uint32_t hi = *reinterpret_cast<const uint16_t*>(stage + o1);
            col[r >> 1] = lo | (hi << 16);
          }
          (void)st32;
          uint16_t* dst = p.vt + (size_t(head) * d + c * 32 + j) * p.Rp + row0 + p.row_off;
          if (row0 + 32 <= row_end && ((row0 + p.row_off) & 7) == 0) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);  // (row0 + row_off) % 8 == 0, Rp % 8 == 0: 16-byte aligned
#pragma unroll
            for (int q = 0; q < 4; ++q) d4[q] = make_uint4(col[4 * q], col[4 * q + 1], col[4 * q + 2], col[4 * q + 3]);
          } else {
#pragma unroll
            for (int r = 0; r < 32; ++r)
              if (row0 + r < row_end) dst[r] = uint16_t(r & 1 ? col[r >> 1] >> 16 : col[r >> 1] & 0xffffu);
          }
        }
        continue;
      }
      // pass 1: sum of squares of the head
      float ss = 0.f;
      for (int c = 0; c < d / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(ta + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float f = __uint_as_float(v[j]);
          ss = fmaf(f, f, ss);
        }
      }
      const float rstd = rsqrtf(ss / float(d) + p.qk_eps);
      const bool g2 = p.m_split > 0 && row >= p.m_split;  // second row group: its own head norms
      const float* wn = which == 0 ? (g2 ? p.q_norm2 : p.q_norm) : (g2 ? p.k_norm2 : p.k_norm);
      const float4* cs = reinterpret_cast<const float4*>(srow < p.L ? p.txt_cos + size_t(srow) * tw
                                                                      : p.img_cos + size_t(srow - p.L) * tw);
      const float4* sn = reinterpret_cast<const float4*>(srow < p.L ? p.txt_sin + size_t(srow) * tw
                                                                      : p.img_sin + size_t(srow - p.L) * tw);
      uint16_t* dst = (which == 0 ? p.q : p.k) + (size_t(head) * R + srow) * d;
      if (p.rope_split) {
        // pass 2, split halves: values i and i + hr (i < hr = 3d/8) turned by angle i, eight pairs
        // at a time; the last d/4 values are normalised and weighted only
        const int hr = 3 * d / 8;
        for (int i0 = 0; i0 < hr; i0 += 8) {
          uint32_t va[8], vb[8];
          tmem_ld8(ta + i0, va);
          tmem_ld8(ta + i0 + hr, vb);
          tmem_ld_wait();
          if (!row_ok) continue;
          const float4 c0 = __ldg(cs + i0 / 4), c1 = __ldg(cs + i0 / 4 + 1);
          const float4 s0 = __ldg(sn + i0 / 4), s1 = __ldg(sn + i0 / 4 + 1);
          const float cf[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          const float sf[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          uint32_t pa[4], pb[4];
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            float a[2], b[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              a[u] = __uint_as_float(va[j + u]) * rstd;
              b[u] = __uint_as_float(vb[j + u]) * rstd;
              if (wn) {
                a[u] *= __ldg(wn + i0 + j + u);
                b[u] *= __ldg(wn + i0 + hr + j + u);
              }
            }
            pa[j / 2] = pack_bf16x2(a[0] * cf[j] - b[0] * sf[j], a[1] * cf[j + 1] - b[1] * sf[j + 1]);
            pb[j / 2] = pack_bf16x2(a[0] * sf[j] + b[0] * cf[j], a[1] * sf[j + 1] + b[1] * cf[j + 1]);
          }
          *reinterpret_cast<uint4*>(dst + i0) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
          *reinterpret_cast<uint4*>(dst + i0 + hr) = make_uint4(pb[0], pb[1], pb[2], pb[3]);
        }
        for (int i0 = 2 * hr; i0 < d; i0 += 8) {
          uint32_t va[8];
          tmem_ld8(ta + i0, va);
          tmem_ld_wait();
          if (!row_ok) continue;
          uint32_t pa[4];
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            float a0 = __uint_as_float(va[j]) * rstd, a1 = __uint_as_float(va[j + 1]) * rstd;
            if (wn) {
              a0 *= __ldg(wn + i0 + j);
              a1 *= __ldg(wn + i0 + j + 1);
            }
            pa[j / 2] = pack_bf16x2(a0, a1);
          }
          *reinterpret_cast<uint4*>(dst + i0) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
        }
        continue;
      }
      // pass 2: normalise, weight, rotate adjacent pairs, store
      for (int c = 0; c < d / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(ta + c * 32, v);
        tmem_ld_wait();
        if (!row_ok) continue;
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float f = __uint_as_float(v[j]) * rstd;
          if (wn) f *= __ldg(wn + c * 32 + j);
          y[j] = f;
        }
        float cf[16], sf[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 c4 = __ldg(cs + c * 4 + q);
          const float4 s4 = __ldg(sn + c * 4 + q);
          cf[4 * q] = c4.x; cf[4 * q + 1] = c4.y; cf[4 * q + 2] = c4.z; cf[4 * q + 3] = c4.w;
          sf[4 * q] = s4.x; sf[4 * q + 1] = s4.y; sf[4 * q + 2] = s4.z; sf[4 * q + 3] = s4.w;
        }
        float o[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = y[2 * i], b = y[2 * i + 1];
          o[2 * i] = a * cf[i] - b * sf[i];
          o[2 * i + 1] = a * sf[i] + b * cf[i];
        }
        store_bf16x32(dst + c * 32, o);
      }
    }
  } else if constexpr (EPI == kEpiGated && kRowPerThread) {
    // x[r, n] += gate[map[r], n] * acc, one row per thread: the form for the int8 in-mainloop
    // kernel, whose 320 threads leave 168 registers each (the coalesced form below would spill).
    const int grow = (row_ok ? row : 0) + p.row_off;  // sequence row
    float* x = grow < p.L ? p.txt + size_t(grow) * p.N : p.img + size_t(grow - p.L) * p.N;
    const int m = (p.map && row_ok) ? __ldg(p.map + grow) : 0;
    const float* g = p.gate + size_t(m) * p.gate_stride;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(taddr + c * 32, v);
      const int n = n0 + c * 32;
      float4 xq[8], gq[8];
      const float4* xv = reinterpret_cast<const float4*>(x + n);
      const float4* gv = reinterpret_cast<const float4*>(g + n);
      if (row_ok) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          xq[q] = xv[q];
          gq[q] = __ldg(gv + q);
        }
      }
      tmem_ld_wait();
      if (row_ok) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          xq[q].x = fmaf(gq[q].x, __uint_as_float(v[4 * q + 0]), xq[q].x);
          xq[q].y = fmaf(gq[q].y, __uint_as_float(v[4 * q + 1]), xq[q].y);
          xq[q].z = fmaf(gq[q].z, __uint_as_float(v[4 * q + 2]), xq[q].z);
          xq[q].w = fmaf(gq[q].w, __uint_as_float(v[4 * q + 3]), xq[q].w);
        }
        float4* xo = reinterpret_cast<float4*>(x + n);
#pragma unroll
        for (int q = 0; q < 8; ++q) xo[q] = xq[q];
      }
    }
  } else if constexpr (EPI == kEpiGated) {
    // x[r, n] += gate[map[r], n] * acc. The accumulator chunk (32 rows x 32 columns, thread = row)
    // goes through the warp's 4 KB shared tile (16-byte chunks XOR-swizzled by row & 7), so the
    // global accesses are coalesced: lane handles rows (lane >> 3) + 4 i, i = 0..7, 16-byte column
    // chunk lane & 7, and every warp instruction moves four whole 128-byte lines of x or the gate.
    // The loads of chunk c + 1 are issued as soon as chunk c is stored. Every lane runs every
    // tcgen05.ld (warp-collective); only the global accesses are predicated.
    (void)row_ok;
    const int cq = lane & 7;
    float* xr[8];
    const float* gr[8];
    bool ok[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = row0 + (lane >> 3) + 4 * i;
      ok[i] = r < row_end;
      const int rr = (ok[i] ? r : 0) + p.row_off;  // sequence row
      xr[i] = (rr < p.L ? p.txt + size_t(rr) * p.N : p.img + size_t(rr - p.L) * p.N) + n0 + cq * 4;
      gr[i] = p.gate + size_t(p.map ? __ldg(p.map + rr) : 0) * p.gate_stride + n0 + cq * 4;
    }
    float4 xq[8], gq[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (ok[i]) {
        xq[i] = *reinterpret_cast<const float4*>(xr[i]);
        gq[i] = __ldg(reinterpret_cast<const float4*>(gr[i]));
      }
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(taddr + c * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(stage + lane * 128 + ((q ^ (lane & 7)) << 4)) =
            make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rl = (lane >> 3) + 4 * i;
        const float4 a = *reinterpret_cast<const float4*>(stage + rl * 128 + ((cq ^ (rl & 7)) << 4));
        if (ok[i]) {
          float4 o;
          o.x = fmaf(gq[i].x, a.x, xq[i].x);
          o.y = fmaf(gq[i].y, a.y, xq[i].y);
          o.z = fmaf(gq[i].z, a.z, xq[i].z);
          o.w = fmaf(gq[i].w, a.w, xq[i].w);
          *reinterpret_cast<float4*>(xr[i] + c * 32) = o;
        }
      }
      __syncwarp();
      if (c + 1 < BN / 32) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (ok[i]) {
            xq[i] = *reinterpret_cast<const float4*>(xr[i] + (c + 1) * 32);
            gq[i] = __ldg(reinterpret_cast<const float4*>(gr[i] + (c + 1) * 32));
          }
      }
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(taddr + c * 32, v);
      tmem_ld_wait();
      if (!row_ok) continue;
      const int n = n0 + c * 32;
      if constexpr (EPI == kEpiStoreF32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + size_t(row) * p.ldo + n);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                               __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
      } else if constexpr (EPI == kEpiStoreBF16 || EPI == kEpiSiluBF16) {
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          f[j] = __uint_as_float(v[j]);
          if constexpr (EPI == kEpiSiluBF16) f[j] = silu_f(f[j]);
        }
        store_bf16x32(static_cast<uint16_t*>(p.out) + size_t(row) * p.ldo + n, f);
      } else if constexpr (EPI == kEpiSwiGLU) {
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float a0 = silu_f(__uint_as_float(v[4 * j + 0])) * __uint_as_float(v[4 * j + 1]);
          const float a1 = silu_f(__uint_as_float(v[4 * j + 2])) * __uint_as_float(v[4 * j + 3]);
          w[j] = pack_bf16x2(a0, a1);
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + size_t(row) * p.ldo + n / 2);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  }
}

// ----------------------------------------------------------------------------------------------
// int8 -> bf16 conversion of one k-block of B: int8 tile [BN rows x 64] (row = 64 bytes, unswizzled)
// into the bf16 128-byte-swizzled tile [BN rows x 64]; each row's k-block has two bf16 scales (two
// groups of 32 inputs). The arithmetic is dequant16: bf16_rne(q * s) with one rounding.
// ----------------------------------------------------------------------------------------------
// Work item i of the converter threads = (row i / 4, 16-byte chunk i % 4 of that row's int8
// values): a warp reads 512 consecutive bytes of the int8 tile (no bank conflicts), takes the row's
// scale for that half k-block from the stage's scale tile, and writes the two swizzled 16-byte bf16
// chunks of its 16 values.
template <int BN, int NT>
__device__ __forceinline__ void convert_kblock(const uint8_t* src8, const uint16_t* sS, int s_col, uint8_t* dst16,
                                               int ct) {
  constexpr int kItems = BN * 4 / NT;  // work items per thread: rows r0, r0 + NT/4, ... at chunk q
  static_assert(BN * 4 % NT == 0, "converter work must divide evenly");
  const int q = ct & 3, r0 = ct >> 2;
  uint4 u[kItems];
  uint32_t sc[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {  // all loads first: independent shared-memory reads in flight
    const int r = r0 + k * (NT / 4);
    u[k] = *reinterpret_cast<const uint4*>(src8 + r * 64 + q * 16);
    sc[k] = sS[r * 8 + s_col + (q >> 1)];
  }
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int r = r0 + k * (NT / 4);
    uint32_t outw[8];
    dequant16(u[k], sc[k], outw);
    *reinterpret_cast<uint4*>(dst16 + sw128_offset(r, 2 * q)) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
    *reinterpret_cast<uint4*>(dst16 + sw128_offset(r, 2 * q + 1)) = make_uint4(outw[4], outw[5], outw[6], outw[7]);
  }
}

// ----------------------------------------------------------------------------------------------
// Work items of the persistent loop. Without stream-K (p.sk_tiles == 0) unit u takes tiles u,
// u + units, ... whole. With stream-K the last p.sk_tiles tiles (in tile order) form a region whose
// k-blocks, sk_tiles * KB of them in tile-major order, are cut into p.sk_units equal ranges; unit u
// first works through its range, tile segment by tile segment, then takes (tiles - sk_tiles) /
// sk_units whole tiles (an exact quotient by construction). Every unit thus does the same number of
// k-blocks to within one, whatever the tile count, and the partial tiles come first, so the work of
// finishing them overlaps whole tiles' mainloops. A range covers at most two partial segments (the
// one it starts in and the one it ends in), each with a slot of its own.
// ----------------------------------------------------------------------------------------------
struct WorkItem {
  int tile, k0, k1;
  int part;      // < 0: the whole tile; else this segment's index among the tile's segments
  int nparts;    // segments of the tile
  int u_first;   // unit of the tile's first segment (segment i is unit u_first + i's)
  int trel;      // tile index within the stream-K region
};

__host__ __device__ __forceinline__ int sk_begin(const GemmParams& p, int u, int KB) {
  return int((long long)u * p.sk_tiles * KB / p.sk_units);  // first k-block of unit u's range
}
// The unit whose range holds region k-block a: the largest u with sk_begin(u) <= a.
__host__ __device__ __forceinline__ int sk_unit_of(const GemmParams& p, int a, int KB) {
  const long long S = (long long)p.sk_tiles * KB;
  return int(((long long)(a + 1) * p.sk_units + S - 1) / S) - 1;
}
__host__ __device__ __forceinline__ int sk_segments(const GemmParams& p, int u, int KB) {
  const int a0 = sk_begin(p, u, KB), a1 = sk_begin(p, u + 1, KB);
  return a1 > a0 ? (a1 - 1) / KB - a0 / KB + 1 : 0;
}
__host__ __device__ __forceinline__ int unit_items(const GemmParams& p, int u, int units, int tiles, int KB) {
  if (p.sk_tiles <= 0) return u < tiles ? (tiles - u + units - 1) / units : 0;
  return sk_segments(p, u, KB) + (tiles - p.sk_tiles) / units;
}
__host__ __device__ __forceinline__ WorkItem unit_item(const GemmParams& p, int u, int i, int units, int tiles,
                                                       int KB) {
  if (p.sk_tiles <= 0) return WorkItem{u + i * units, 0, KB, -1, 1, 0, 0};
  const int nseg = sk_segments(p, u, KB);
  if (i >= nseg) return WorkItem{u + (i - nseg) * units, 0, KB, -1, 1, 0, 0};
  const int a0 = sk_begin(p, u, KB), a1 = sk_begin(p, u + 1, KB);
  const int trel = a0 / KB + i;
  const int k0 = i == 0 ? a0 - trel * KB : 0;
  const int k1 = i == nseg - 1 ? a1 - trel * KB : KB;
  const int tile = tiles - p.sk_tiles + trel;
  if (k0 == 0 && k1 == KB) return WorkItem{tile, 0, KB, -1, 1, 0, trel};
  const int uf = sk_unit_of(p, trel * KB, KB), ul = sk_unit_of(p, trel * KB + KB - 1, KB);
  return WorkItem{tile, k0, k1, u - uf, ul - uf + 1, uf, trel};
}
// Partial slot of unit v's segment on region tile trel: 2v for the tile its range starts in, 2v + 1
// for the tile it ends in.
__host__ __device__ __forceinline__ int sk_slot(const GemmParams& p, int v, int trel, int KB) {
  return 2 * v + (sk_begin(p, v, KB) < trel * KB ? 1 : 0);
}

// A warp's 32 rows x BN fp32 partial accumulator to its slot, in the thread-per-row layout
// [32-column chunk][float4 of the chunk][lane]: every store instruction writes 512 contiguous bytes.
template <int BN>
__device__ __forceinline__ void sk_store(uint32_t taddr, float* dst, int lane) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + c * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 8; ++q)
      __stcg(reinterpret_cast<float4*>(dst) + (c * 8 + q) * 32 + lane,
             make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                         __uint_as_float(v[4 * q + 3])));
  }
}

// The warp that delivered a tile quadrant's last segment: the sum of all segments' partials, in
// segment order (((p0 + p1) + p2) ..., the same whichever unit finishes), written over its own
// accumulator in TMEM; W8A8 accumulators (exact integer sums) are scaled by the row's and the
// column's scales after the sum, as a whole tile's are. The epilogue then runs on it unchanged.
// `part(i)` is segment i's slot (this warp's rows). The loads of parts 0 and 1 of a chunk are issued
// together (one L2 round trip for the usual two-part tile), a third part's after them.
template <int BN, typename PartFn>
__device__ __forceinline__ void sk_sum(const GemmParams& p, const float* w_scale, uint32_t taddr, PartFn part,
                                       int nparts, int lane, int row, int row_end, int n0) {
  static_assert(kSkMaxParts == 3, "parts 0 and 1 together, then part 2");
  const float sa = (p.a_scale && row < row_end) ? __ldg(p.a_scale + row) : 0.f;
  const float4* s0 = reinterpret_cast<const float4*>(part(0)) + lane;
  const float4* s1 = reinterpret_cast<const float4*>(part(1)) + lane;
  const float4* s2 = reinterpret_cast<const float4*>(part(nparts > 2 ? 2 : 1)) + lane;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float4 a[8], b[8];  // chunk c of a part: 8 float4 at part + c * 256 + q * 32
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      a[q] = __ldcg(s0 + c * 256 + q * 32);
      b[q] = __ldcg(s1 + c * 256 + q * 32);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      a[q].x += b[q].x;
      a[q].y += b[q].y;
      a[q].z += b[q].z;
      a[q].w += b[q].w;
    }
    if (nparts > 2) {
#pragma unroll
      for (int q = 0; q < 8; ++q) b[q] = __ldcg(s2 + c * 256 + q * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        a[q].x += b[q].x;
        a[q].y += b[q].y;
        a[q].z += b[q].z;
        a[q].w += b[q].w;
      }
    }
    uint32_t v[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[4 * q] = __float_as_uint(a[q].x);
      v[4 * q + 1] = __float_as_uint(a[q].y);
      v[4 * q + 2] = __float_as_uint(a[q].z);
      v[4 * q + 3] = __float_as_uint(a[q].w);
    }
    if (p.a_scale) {
      const float* sw = w_scale + n0 + c * 32;
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * sa * __ldg(sw + j));
    }
    tmem_st32(taddr + c * 32, v);
  }
  tmem_st_wait();
}

// Row tiles of a GEMM. With two row groups (m_split > 0) whose boundary is not on a tile boundary,
// each group is padded to whole tiles (group 0: rows [0, m_split), group 1: rows [m_split, M)), so
// no tile mixes the groups' weights; otherwise tiles are consecutive 'tile_m'-row blocks.
__host__ __device__ __forceinline__ bool row_groups_padded(const GemmParams& p, int tile_m) {
  return p.m_split > 0 && p.m_split % tile_m != 0;
}
__host__ __device__ __forceinline__ int row_tiles(const GemmParams& p, int tile_m) {
  if (row_groups_padded(p, tile_m))
    return (p.m_split + tile_m - 1) / tile_m + (p.M - p.m_split + tile_m - 1) / tile_m;
  return (p.M + tile_m - 1) / tile_m;
}
// First row, end of the valid rows and group of row tile mb.
struct TileRows {
  int base, end;
  bool g2;
};
__device__ __forceinline__ TileRows tile_rows(const GemmParams& p, int tile_m, int mb) {
  if (row_groups_padded(p, tile_m)) {
    const int nm0 = (p.m_split + tile_m - 1) / tile_m;
    if (mb < nm0) return TileRows{mb * tile_m, p.m_split, false};
    return TileRows{p.m_split + (mb - nm0) * tile_m, p.M, true};
  }
  return TileRows{mb * tile_m, p.M, p.m_split > 0 && mb * tile_m >= p.m_split};
}

// CTA pairs publish in global memory that their barriers are initialised, one word per CTA: it is
// set to 1 once the CTA's barriers are initialised and back to 0 when the CTA ends, and a CTA touches
// its peer's shared memory only after reading the peer's word as 1. Launches pick one of
// kPairSlots word sets in turn (host counter), so launches running at once on different streams
// use different words.
constexpr int kPairSlots = 64, kPairMaxCtas = 256;
__device__ uint32_t g_pair_started[kPairSlots * kPairMaxCtas];

// Stream-K arrival counters, one set per launch slot (launches take the kSkSlots sets in turn, so
// launches running at once on different streams count on different sets). The warp that brings a
// counter to its tile's segment count sets it back to zero, so every launch that finishes leaves
// its set at zero; an aborted launch may not, and dit_check() clears them all when it reports one.
constexpr int kSkSlots = 64, kSkMaxCounters = 2048;
__device__ uint32_t g_sk_cnt[kSkSlots * kSkMaxCounters];

template <int BN, int EPI, bool B8, bool PAIR>
__global__ void __launch_bounds__(GemmCfg<BN, B8, PAIR>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ CUtensorMap tmB2, const GemmParams p) {
  using Cfg = GemmCfg<BN, B8, PAIR>;
  constexpr int S = Cfg::kStages;
  constexpr int CS = Cfg::kConvStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * Cfg::kABytes;                              // bf16 ring, or int8 ring when B8
  uint8_t* sSc = sB + S * (B8 ? Cfg::kB8Bytes : Cfg::kBLoad);       // B8: scale-tile ring
  uint8_t* sC = sSc + (B8 ? S * Cfg::kSBytes : 0);                  // B8: converted bf16 ring
  uint8_t* sE = sC + Cfg::kConvBytes;                               // epilogue staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + Cfg::kEpiBytes);
  uint64_t* full = bars;                 // [S] TMA landed (PAIR: the first CTA's counts both CTAs' copies)
  uint64_t* empty = bars + S;            // [S] stage free (MMA done; B8: also converter done)
  uint64_t* tfull = bars + 2 * S;        // [2] accumulator ready
  uint64_t* tempty = bars + 2 * S + 2;   // [2] accumulator drained (PAIR: by both CTAs, first CTA's)
  uint64_t* cfull = bars + 2 * S + 4;    // [CS] converted B tile ready (B8)
  uint64_t* cempty = cfull + CS;         // [CS] converted B tile consumed (B8)
  uint64_t* drain = cempty + CS;         // [1] final MMA completion
  uint64_t* done = drain + 1;            // [1] PAIR: the peer CTA has finished with this CTA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  uint32_t* pair_ok = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = lane_id();
  // PAIR: CTAs 2u and 2u + 1 form cluster u; work unit = the pair, rank 0 issues the MMAs
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;
  const int unit = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);
  const int units = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);
  const int num_m = row_tiles(p, Cfg::kTileM);
  const int num_n = p.N / BN;
  // Tile order: consecutive tiles share the smaller operand's panel set, so the CTAs running at
  // once keep it in L2 and the larger operand streams from DRAM once. m fastest (A resident) when A
  // is the smaller operand, n fastest (B resident) otherwise.
  const bool n_fast = 2LL * p.M > (long long)p.N * (B8 ? 1 : 2);  // A bytes > B bytes (per k)
  auto tile_mn = [&](int tile, int& mb, int& nb) {
    if (n_fast) {
      mb = tile / num_n;
      nb = tile % num_n;
    } else {
      mb = tile % num_m;
      nb = tile / num_m;
    }
  };
  const int tiles = num_m * num_n;
  const int KB = p.K / BK;
  const int items = unit_items(p, unit, units, tiles, KB);  // this unit's work items

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), B8 ? 1 + Cfg::kConvThreads / 32 : 1);  // B8: MMA commit + converter warps
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), (PAIR ? 2 : 1) * Cfg::kEpiThreads);
    }
    for (int c = 0; c < CS; ++c) {
      mbar_init(smem_u32(&cfull[c]), (PAIR ? 2 : 1) * Cfg::kConvThreads / 32);  // converter warps (PAIR: both CTAs')
      mbar_init(smem_u32(&cempty[c]), 1);
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(done), 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (B8) tma_prefetch_desc(&tmS);
    if (p.k_split > 0) tma_prefetch_desc(&tmA2);
    if (p.k_split > 0 || p.n_split > 0 || p.m_split > 0) tma_prefetch_desc(&tmB2);
  }
  bool up = true;
  if constexpr (PAIR) {
    // barriers initialised here -> published; then a bounded wait for the peer's word
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t* words = g_pair_started + (p.pair_epoch % kPairSlots) * kPairMaxCtas;
      st_release_gpu(&words[blockIdx.x], 1u);
      const uint64_t t0 = globaltimer_ns();
      uint32_t ok = 1;
      while (ld_acquire_gpu(&words[blockIdx.x ^ 1u]) != 1u)
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicCAS(p.err, 0, kErrTimeoutPair);
          ok = 0;
          break;
        }
      asm volatile("fence.acq_rel.cluster;" ::: "memory");
      *pair_ok = ok;
    }
    __syncthreads();
    up = *pair_ok != 0;
    if (warp == 1) {
      tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
      tmem_relinquish_pair();
    }
  } else if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above (barriers, tensor memory, descriptor prefetch, the pair hand-shake on words of
  // this launch's own set) may overlap the previous kernel in the stream; its results only from here.
  pdl_wait();
  pdl_trigger();

  if (!up) {
    // the pair never formed: nothing to do
  } else if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_parity = 0;
      bool ok = true;
      // PAIR (bf16): both CTAs' copies complete on the first CTA's barrier, which expects both.
      // PAIR (int8): each CTA's copies complete on its own barrier, which its converters wait on.
      constexpr bool kLocalFull = !PAIR || B8;
      constexpr uint32_t kOwnBytes = Cfg::kABytes + (B8 ? Cfg::kB8Bytes + Cfg::kSBytes : Cfg::kBLoad);
      const uint32_t full0 = kLocalFull ? smem_u32(&full[0]) : mapa_shared(smem_u32(&full[0]), 0);
      for (int it = 0; it < items && ok; ++it) {
        const WorkItem w = unit_item(p, unit, it, units, tiles, KB);
        int mb, nb;
        tile_mn(w.tile, mb, nb);
        const TileRows tr = tile_rows(p, Cfg::kTileM, mb);
        for (int kb = w.k0; kb < w.k1; ++kb) {
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, p.err, kErrTimeoutProducer)) { ok = false; break; }
          const uint32_t fb = full0 + uint32_t(stage) * 8u;
          if (kLocalFull || rank == 0) mbar_arrive_expect_tx(smem_u32(&full[stage]), (kLocalFull ? 1 : 2) * kOwnBytes);
          // concatenated operands: the second A/B past the K boundary, the second B past the N boundary
          const bool k2 = p.k_split > 0 && kb * BK >= p.k_split;
          const bool n2 = p.n_split > 0 && nb * BN >= p.n_split;
          const bool m2 = tr.g2;
          const CUtensorMap* ma = k2 ? &tmA2 : &tmA;
          const CUtensorMap* mbm = (k2 || n2 || m2) ? &tmB2 : &tmB;
          const int kc = k2 ? kb * BK - p.k_split : kb * BK;
          const int nr = n2 ? nb * BN - p.n_split : nb * BN;
          if constexpr (B8) {
            // int8 B rows of this CTA (PAIR: its half of the tile) with their scales
            const int brow = nb * BN + int(rank) * Cfg::kBRows;
#pragma unroll
            for (int h = 0; h < Cfg::kMH; ++h)
              tma_load_2d(smem_u32(sA + stage * Cfg::kABytes + h * Cfg::kAHalf), ma, fb, kc,
                          tr.base + int(rank) * BM + h * BM);
            tma_load_2d(smem_u32(sB + stage * Cfg::kB8Bytes), &tmB, fb, kb * BK, brow);
            // scales of k-blocks (kb & ~3) .. (kb | 3): 8 bf16 per row, 16-byte aligned columns
            tma_load_2d(smem_u32(sSc + stage * Cfg::kSBytes), &tmS, fb, (kb * 2) & ~7, brow);
          } else if constexpr (PAIR) {
            tma_load_2d_pair(smem_u32(sA + stage * Cfg::kABytes), ma, fb, kc, tr.base + int(rank) * BM);
            tma_load_2d_pair(smem_u32(sB + stage * Cfg::kBLoad), mbm, fb, kc, nr + int(rank) * (BN / 2));
          } else {
            tma_load_2d(smem_u32(sA + stage * Cfg::kABytes), ma, fb, kc, tr.base);
            tma_load_2d(smem_u32(sB + stage * Cfg::kBLoad), mbm, fb, kc, nr);
          }
          issued_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      // every issued copy must have landed before the CTA exits (PAIR bf16: the first CTA's barriers
      // count the second's copies too, and the second waits for the first before it exits)
      if (kLocalFull || rank == 0)
        for (int s = 0; s < S; ++s)
          if (issued_mask & (1u << s))
            mbar_wait(smem_u32(&full[s]), (last_parity >> s) & 1u, p.err, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if ((!PAIR || rank == 0) && elect_one()) {
      constexpr uint32_t idesc = idesc_bf16(PAIR ? 2 * BM : BM, BN);
      int stage = 0, cstage = 0;
      uint32_t phase = 0, cphase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int it = 0; it < items && ok; ++it) {
        const WorkItem w = unit_item(p, unit, it, units, tiles, KB);
        if (!(PAIR ? mbar_wait_cluster(smem_u32(&tempty[acc]), acc_phase ^ 1, p.err, kErrTimeoutMma)
                   : mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1, p.err, kErrTimeoutMma)))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * Cfg::kMH * BN);
        for (int kb = w.k0; kb < w.k1; ++kb) {
          if (!mbar_wait(smem_u32(&full[stage]), phase, p.err, kErrTimeoutMma)) { ok = false; break; }
          uint32_t b_addr;
          if constexpr (B8) {
            // PAIR: the count covers both CTAs' converters, each of which waited for its own CTA's
            // copies of this stage (A included) before converting
            if (!(PAIR ? mbar_wait_cluster(smem_u32(&cfull[cstage]), cphase, p.err, kErrTimeoutMma)
                       : mbar_wait(smem_u32(&cfull[cstage]), cphase, p.err, kErrTimeoutMma))) {
              ok = false;
              break;
            }
            b_addr = smem_u32(sC + cstage * Cfg::kBLoad);
          } else {
            b_addr = smem_u32(sB + stage * Cfg::kBLoad);
          }
          tc_fence_after();
          const uint64_t bdesc = sw128_desc(b_addr);
#pragma unroll
          for (int h = 0; h < Cfg::kMH; ++h) {
            const uint64_t adesc = sw128_desc(smem_u32(sA + stage * Cfg::kABytes + h * Cfg::kAHalf));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {  // +32 bytes per K=16 step inside the swizzle atom
              if constexpr (PAIR)
                umma_bf16_pair(d, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), idesc, kb != w.k0 || kk != 0);
              else
                umma_bf16(d + uint32_t(h * BN), adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), idesc,
                          kb != w.k0 || kk != 0);
            }
          }
          if constexpr (PAIR) umma_commit_pair_both(smem_u32(&empty[stage]));
          else umma_commit(smem_u32(&empty[stage]));
          if constexpr (B8) {
            if constexpr (PAIR) umma_commit_pair_both(smem_u32(&cempty[cstage]));
            else umma_commit(smem_u32(&cempty[cstage]));
            if (++cstage == CS) { cstage = 0; cphase ^= 1; }
          }
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if constexpr (PAIR) umma_commit_pair_both(smem_u32(&tfull[acc]));
        else umma_commit(smem_u32(&tfull[acc]));
        if (++acc == Cfg::kAccBufs) { acc = 0; acc_phase ^= 1; }
      }
      // all MMAs issued by this thread complete before TMEM is released
      if constexpr (PAIR) umma_commit_pair(smem_u32(drain));
      else umma_commit(smem_u32(drain));
      mbar_wait(smem_u32(drain), 0, p.err, kErrTimeoutDrain);
    }
  } else if (warp < Cfg::kConvWarp0) {
    // ------------------------------------------------------------- epilogue warps
    const int quad = warp & 3;                       // TMEM lanes this warp may access
    const int col0 = ((warp - 2) >> 2) * Cfg::kEpiCols;  // its columns of the tile
    uint8_t* stage = sE + (warp - 2) * 4096;
    // PAIR: this CTA's 128 rows of the pair's tile; the accumulator is released on the first CTA
    const int rows_of = PAIR ? int(rank) * BM : 0;
    const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(&tempty[0]), 0) : smem_u32(&tempty[0]);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0; it < items; ++it) {
      const WorkItem w = unit_item(p, unit, it, units, tiles, KB);
      int mb, nb;
      tile_mn(w.tile, mb, nb);
      const TileRows tr = tile_rows(p, Cfg::kTileM, mb);
      if (!mbar_wait_warp(smem_u32(&tfull[acc]), acc_phase, p.err, kErrTimeoutEpilogue)) break;
      tc_fence_after();
      if constexpr (!B8) {
        static_assert(B8 || Cfg::kEpiCols == BN, "one epilogue warp per TMEM lane quadrant");
        const uint32_t taddr = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * BN);
        const int row = tr.base + rows_of + quad * 32 + lane;
        const float* w_scale = (tr.g2 && p.w_scale2) ? p.w_scale2 : p.w_scale;  // this row group's
        bool scaled = false;
        if (w.part >= 0) {
          // stream-K segment: publish this warp's partial, count it, and if it was the quadrant's
          // last segment sum them all into this accumulator and go on to the epilogue; otherwise
          // release the accumulator
          constexpr int kSlabs = PAIR ? 2 : 1;
          const size_t slab = size_t(BM) * BN, warp_off = size_t(quad) * 32 * BN;
          float* mine = p.sk_part + (size_t(sk_slot(p, unit, w.trel, KB)) * kSlabs + rank) * slab + warp_off;
          sk_store<BN>(taddr, mine, lane);
          __threadfence();
          __syncwarp();
          uint32_t* cnt = p.sk_cnt + (w.trel * kSlabs + int(rank)) * 4 + quad;
          int last = 0;
          if (lane == 0) last = atomicAdd(cnt, 1u) == uint32_t(w.nparts - 1);
          if (!__shfl_sync(0xffffffffu, last, 0)) {
            tc_fence_before();
            if constexpr (PAIR) mbar_arrive_cluster(tempty0 + uint32_t(acc) * 8u);
            else mbar_arrive(smem_u32(&tempty[acc]));
            if (++acc == Cfg::kAccBufs) { acc = 0; acc_phase ^= 1; }
            continue;
          }
          __threadfence();
          auto part = [&](int i) -> const float* {
            return p.sk_part + (size_t(sk_slot(p, w.u_first + i, w.trel, KB)) * kSlabs + rank) * slab + warp_off;
          };
          sk_sum<BN>(p, w_scale, taddr, part, w.nparts, lane, row, tr.end, nb * BN);
          if (lane == 0) atomicExch(cnt, 0u);  // zero again for the next launch
          scaled = true;
        }
        if (p.a_scale && !scaled) {
          // W8A8: the accumulator holds exact integer dot products of codes; scale it in place by
          // the row's and the column's scales, then run the epilogue on it as usual
          const float sa = row < tr.end ? __ldg(p.a_scale + row) : 0.f;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(taddr + c * 32, v);
            tmem_ld_wait();
            const float* sw = w_scale + nb * BN + c * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * sa * __ldg(sw + j));
            tmem_st32(taddr + c * 32, v);
          }
          tmem_st_wait();
        }
      }
#pragma unroll 1
      for (int h = 0; h < Cfg::kMH; ++h) {
        const uint32_t taddr =
            tmem_base + (uint32_t(quad * 32) << 16) + uint32_t((acc * Cfg::kMH + h) * BN + col0);
        const int row0 = tr.base + rows_of + h * BM + quad * 32, n0 = nb * BN + col0;
        if constexpr (EPI == kEpiQKVSwiGLU) {
          if (n0 < p.n_split)
            epilogue_tile<Cfg::kEpiCols, kEpiQKV, B8>(p, taddr, row0, tr.end, lane, n0, stage);
          else
            epilogue_tile<Cfg::kEpiCols, kEpiSwiGLU, B8>(p, taddr, row0, tr.end, lane, n0 - p.n_split, stage);
        } else {
          epilogue_tile<Cfg::kEpiCols, EPI, B8>(p, taddr, row0, tr.end, lane, n0, stage);
        }
      }
      tc_fence_before();
      if constexpr (PAIR) mbar_arrive_cluster(tempty0 + uint32_t(acc) * 8u);
      else mbar_arrive(smem_u32(&tempty[acc]));
      if (++acc == Cfg::kAccBufs) { acc = 0; acc_phase ^= 1; }
    }
  } else if constexpr (B8) {
    // ------------------------------------------------------------- int8 -> bf16 converters
    const int ct = threadIdx.x - 32 * Cfg::kConvWarp0;
    int stage = 0, cstage = 0;
    uint32_t phase = 0, cphase = 0;
    bool ok = true;
    // PAIR: the converted tile is read by the first CTA's MMAs, whose barrier counts both CTAs
    const uint32_t cfull0 = PAIR ? mapa_shared(smem_u32(&cfull[0]), 0) : smem_u32(&cfull[0]);
    for (int it = 0; it < items && ok; ++it) {
      const WorkItem w = unit_item(p, unit, it, units, tiles, KB);
      for (int kb = w.k0; kb < w.k1; ++kb) {
        // warp-uniform verdicts: the warp meets again at the __syncwarp below
        if (!mbar_wait_warp(smem_u32(&full[stage]), phase, p.err, kErrTimeoutConverter)) { ok = false; break; }
        if (!mbar_wait_warp(smem_u32(&cempty[cstage]), cphase ^ 1, p.err, kErrTimeoutConverter)) { ok = false; break; }
        convert_kblock<Cfg::kBRows, Cfg::kConvThreads>(sB + stage * Cfg::kB8Bytes,
                                                       reinterpret_cast<const uint16_t*>(sSc + stage * Cfg::kSBytes),
                                                       (kb * 2) & 7, sC + cstage * Cfg::kBLoad, ct);
        // every lane's writes to the async proxy, then one arrival per warp
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR) mbar_arrive_cluster(cfull0 + uint32_t(cstage) * 8u);
          else mbar_arrive(smem_u32(&cfull[cstage]));
          mbar_arrive(smem_u32(&empty[stage]));  // this warp is done reading the int8 stage
        }
        if (++cstage == CS) { cstage = 0; cphase ^= 1; }
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // Neither CTA leaves, nor frees its TMEM, while the other may still write its barriers, read its
    // shared memory or (first CTA's MMAs, drained above) write its TMEM. A peer still ending a
    // failed wait takes up to a second per role: allow a few.
    if (up) {
      if (threadIdx.x == 0) mbar_arrive_cluster(mapa_shared(smem_u32(done), rank ^ 1u));
      mbar_wait_cluster(smem_u32(done), 0, p.err, kErrTimeoutPair, 4 * kWaitLimitNs, false);
    }
    tc_fence_after();
    if (threadIdx.x == 0) g_pair_started[(p.pair_epoch % kPairSlots) * kPairMaxCtas + blockIdx.x] = 0u;
    if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  } else {
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

struct Maps {
  CUtensorMap a, b, s, a2, b2;  // s, a2, b2 unused unless int8 / concatenated operands (then copies)
};

// Work units (CTAs, or CTA pairs) that can be resident at once for a launch of `kern`.
int resident_units(const void* kern, bool pair, unsigned threads, unsigned smem) {
  if (!pair) return num_sms();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(num_sms() & ~1));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return num_sms() / 2;
  }
  return n < num_sms() / 2 ? n : num_sms() / 2;
}

std::atomic<uint32_t> g_pair_launches{0};
std::atomic<uint32_t> g_sk_launches{0};

// Device address of g_sk_cnt on the current device (looked up once per device).
uint32_t* sk_counters() {
  static uint32_t* addr[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sk_cnt) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint32_t*>(p);
  }
  return addr[dev];
}

// Stream-K plan of a bf16 launch over `units` work units of `slabs` 128-row slabs and tiles of BN
// columns: sets q.sk_* when it pays, else leaves q.sk_tiles = 0. With W whole waves and rem < units
// tiles over, the region is the last rem tiles (or rem + units when rem is below half the units, so
// that each unit's share stays at least half a tile and a tile meets at most three units); the
// critical path drops from W + 1 to W + rem / units tile-times, taken when that saves at least a
// tenth of a tile. Needs two partial slots per unit in the caller's scratch and at least eight
// k-blocks per tile.
void plan_stream_k(GemmParams& q, int tiles, int units, int slabs, int BN) {
  q.sk_tiles = 0;
  const int KB = q.K / BK;
  if (!q.split_ws || units < 2 || KB < 8) return;
  const int W = tiles / units, rem = tiles % units;
  if (rem == 0 || 10 * rem > 9 * units) return;
  int sk = rem;
  if (2 * sk < units) {
    if (W == 0) return;
    sk += units;
  }
  if (sk * slabs * 4 > kSkMaxCounters) return;
  if (size_t(2) * units * slabs * BM * BN * sizeof(float) > q.split_ws_bytes) return;
  GemmParams t = q;
  t.sk_tiles = sk;
  t.sk_units = units;
  for (int r = 0; r < sk; ++r)
    if (sk_unit_of(t, r * KB + KB - 1, KB) - sk_unit_of(t, r * KB, KB) + 1 > kSkMaxParts) return;
  uint32_t* cnt = sk_counters();
  if (!cnt) return;
  q.sk_tiles = sk;
  q.sk_units = units;
  q.sk_part = static_cast<float*>(q.split_ws);
  q.sk_cnt = cnt + size_t(g_sk_launches.fetch_add(1, std::memory_order_relaxed) % kSkSlots) * kSkMaxCounters;
}

template <int BN, int EPI, bool B8, bool PAIR>
int launch_one(const Maps& m, const GemmParams& p, cudaStream_t stream) {
  using Cfg = GemmCfg<BN, B8, PAIR>;
  static_assert(Cfg::kSmemBytes <= 227 * 1024, "shared memory budget");
  auto kern = gemm_kernel<BN, EPI, B8, PAIR>;
  if (!smem_attr_once(reinterpret_cast<const void*>(kern), Cfg::kSmemBytes)) return DIT_ECUDA;
  static int units_cached[64];  // resident units, queried once per kernel and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DIT_ECUDA;
  if (units_cached[dev] <= 0)
    units_cached[dev] = resident_units(reinterpret_cast<const void*>(kern), PAIR, Cfg::kThreads, Cfg::kSmemBytes);
  const int units_max = units_cached[dev];
  const int tiles = row_tiles(p, Cfg::kTileM) * (p.N / BN);
  GemmParams q = p;
  if constexpr (!B8) plan_stream_k(q, tiles, units_max, PAIR ? 2 : 1, BN);
  else q.sk_tiles = 0;
  const int units = q.sk_tiles > 0 ? units_max : (tiles < units_max ? tiles : units_max);
  if constexpr (PAIR) {
    if (2 * units > kPairMaxCtas) return DIT_EUNSUPPORTED;
    q.pair_epoch = g_pair_launches.fetch_add(1, std::memory_order_relaxed);
  }
  const int ctas = PAIR ? 2 * units : units;
  if (launch_pdl(kern, dim3(unsigned(ctas)), dim3(Cfg::kThreads), Cfg::kSmemBytes, stream, PAIR ? 2 : 1, m.a, m.b, m.s,
                 m.a2, m.b2, q) != cudaSuccess)
    return DIT_ECUDA;
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

template <int BN, bool B8, bool PAIR>
int dispatch_epi(int epi, const Maps& m, const GemmParams& p, cudaStream_t stream) {
  switch (epi) {
    case kEpiStoreF32: return launch_one<BN, kEpiStoreF32, B8, PAIR>(m, p, stream);
    case kEpiStoreBF16: return launch_one<BN, kEpiStoreBF16, B8, PAIR>(m, p, stream);
    case kEpiSiluBF16: return launch_one<BN, kEpiSiluBF16, B8, PAIR>(m, p, stream);
    case kEpiGated: return launch_one<BN, kEpiGated, B8, PAIR>(m, p, stream);
    case kEpiSwiGLU: return launch_one<BN, kEpiSwiGLU, B8, PAIR>(m, p, stream);
    case kEpiQKV: return launch_one<BN, kEpiQKV, B8, PAIR>(m, p, stream);
    case kEpiQKVSwiGLU:
      if constexpr (BN == 256 && !B8) return launch_one<BN, kEpiQKVSwiGLU, B8, PAIR>(m, p, stream);
      return DIT_EUNSUPPORTED;
    default: return DIT_EINVAL;
  }
}

}  // namespace

namespace {

int pick_bn(int N) { return (N % 256 == 0) ? 256 : (N % 128 == 0 ? 128 : 64); }

// bf16 mainloop on CTA pairs: 256-row tiles, each of the two SMs bringing its 128 rows of A and half
// of the B tile, so a k-block costs an SM 32 KB of shared-memory fill instead of 48 KB (BN = 256) and
// one MMA issue covers both. Needs tiles at least 128 wide and more than one 128-row block.
bool use_pair(int BN, const GemmParams& p) { return BN >= 128 && p.M > BM && num_sms() >= 2; }

// bf16 weights: the launch (stream-K is planned per kernel in launch_one, which knows its units)
int launch_bf16(const Maps& m, int BN, int epi, const GemmParams& q, bool pair, cudaStream_t stream) {
  switch (BN) {
    case 256: return pair ? dispatch_epi<256, false, true>(epi, m, q, stream) : dispatch_epi<256, false, false>(epi, m, q, stream);
    case 128: return pair ? dispatch_epi<128, false, true>(epi, m, q, stream) : dispatch_epi<128, false, false>(epi, m, q, stream);
    default: return dispatch_epi<64, false, false>(epi, m, q, stream);
  }
}

bool tmap_bf16(CUtensorMap* m, const uint16_t* ptr, int inner, int outer, long long ld, int box_outer) {
  return make_tmap_2d(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, ld * 2, BK, box_outer, true);
}

}  // namespace

int gemm_launch(const uint16_t* a, long long lda, const uint16_t* b, const GemmInt8B* b8, int epi,
                const GemmParams& p, cudaStream_t stream) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return DIT_EINVAL;
  if (p.K % BK != 0 || p.N % 64 != 0) return DIT_EUNSUPPORTED;
  if (p.n_split != 0 || p.k_split != 0 || epi == kEpiQKVSwiGLU) return DIT_EINVAL;  // gemm_launch_cat
  if (reinterpret_cast<uintptr_t>(a) % 16 || (lda * 2) % 16) return DIT_EINVAL;
  // tile width: 256 where it divides N (fewer A re-reads), else 128, else 64
  int BN = pick_bn(p.N);
  // QKV epilogue: a tile never straddles q/k/v and holds whole heads
  if (epi == kEpiQKV && (BN % p.head_dim != 0 || p.H % BN != 0)) return DIT_EUNSUPPORTED;
  Maps m;
  if (!tmap_bf16(&m.a, a, p.K, p.M, lda, BM)) return DIT_ECUDA;
  if (b8) {
    if (reinterpret_cast<uintptr_t>(b8->q) % 16 || reinterpret_cast<uintptr_t>(b8->s) % 16) return DIT_EINVAL;
    if (BN == 64 || p.K % 256 != 0) return DIT_EUNSUPPORTED;  // scale rows must be 16-byte multiples
    if (p.M > kInt8MainloopMaxM) {
      // Many M tiles: the in-mainloop converters would dequantise every weight tile once per M tile
      // (17 times at 4224 rows) and bound the GEMM at about 800 TFLOP/s, single CTAs or pairs alike;
      // dequantising the weight once, HBM-bound, and running the bf16 mainloop is faster (measured
      // 1.06-1.08 against 1.69 ms per 1024sq block).
      if (!b8->wbf || reinterpret_cast<uintptr_t>(b8->wbf) % 16) return DIT_EINVAL;
      const int rc = dequant_int8_launch(b8->q, b8->s, b8->wbf, p.N, p.K, stream);
      if (rc != DIT_OK) return rc;
      return gemm_launch(a, lda, b8->wbf, nullptr, epi, p, stream);
    }
    if (use_pair(BN, p)) {
      // CTA pairs: 256 x BN tiles, each CTA converting its half of every int8 k-block of B (BN/2
      // rows) into the bf16 tile the pair's MMAs read: the conversions per FLOP of the 256 x 128
      // single-CTA tile, with a third less shared-memory traffic per SM
      if (epi == kEpiQKV && (BN % p.head_dim != 0 || p.H % BN != 0)) return DIT_EUNSUPPORTED;
      if (!make_tmap_2d(&m.b, b8->q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.K, p.N, p.K, BK, BN / 2, false) ||
          !make_tmap_2d(&m.s, b8->s, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.K / 32, p.N, (long long)(p.K / 32) * 2, 8,
                        BN / 2, false))
        return DIT_ECUDA;
      m.a2 = m.a;
      m.b2 = m.b;
      return BN == 256 ? dispatch_epi<256, true, true>(epi, m, p, stream) : dispatch_epi<128, true, true>(epi, m, p, stream);
    }
    // int8lin tiles are 256 x 128: two M=128 MMAs share each converted B k-block and both accumulator
    // sets fit in TMEM. (256 x 256 tiles, with one accumulator set and no epilogue overlap, measured
    // 2.02 ms per 1024sq block against 1.87 ms.)
    BN = 128;
    if (epi == kEpiQKV && (BN % p.head_dim != 0 || p.H % BN != 0)) return DIT_EUNSUPPORTED;
    if (!make_tmap_2d(&m.b, b8->q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.K, p.N, p.K, BK, BN, false)) return DIT_ECUDA;
    if (!make_tmap_2d(&m.s, b8->s, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.K / 32, p.N, (long long)(p.K / 32) * 2, 8,
                      BN, false))
      return DIT_ECUDA;
    m.a2 = m.a;
    m.b2 = m.b;
    return dispatch_epi<128, true, false>(epi, m, p, stream);
  }
  if (reinterpret_cast<uintptr_t>(b) % 16) return DIT_EINVAL;
  const bool pair = use_pair(BN, p);
  if (!tmap_bf16(&m.b, b, p.K, p.b_rows > 0 ? p.b_rows : p.N, p.K, pair ? BN / 2 : BN)) return DIT_ECUDA;
  m.s = m.b;
  m.a2 = m.a;
  m.b2 = m.b;
  return launch_bf16(m, BN, epi, p, pair, stream);
}

int gemm_clear_stream_k_counters() {
  uint32_t* cnt = sk_counters();
  if (!cnt) return DIT_ECUDA;
  return cudaMemset(cnt, 0, sizeof(uint32_t) * kSkSlots * kSkMaxCounters) == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int gemm_launch_cat(const uint16_t* a, long long lda, const uint16_t* a2, long long lda2, const uint16_t* b,
                    long long ldb, const uint16_t* b2, long long ldb2, int epi, const GemmParams& p,
                    cudaStream_t stream) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return DIT_EINVAL;
  if (p.K % BK != 0 || p.N % 64 != 0) return DIT_EUNSUPPORTED;
  if ((p.n_split > 0) + (p.k_split > 0) + (p.m_split > 0) != 1) return DIT_EINVAL;  // exactly one kind
  const int BN = pick_bn(p.N);
  auto al = [](const void* q, long long ld) { return reinterpret_cast<uintptr_t>(q) % 16 == 0 && (ld * 2) % 16 == 0; };
  const bool pair = use_pair(BN, p);
  const int bbox = pair ? BN / 2 : BN;  // B rows one CTA loads per k-block
  Maps m;
  if (p.n_split > 0) {
    // B = [b ; b2]: rows [0, n_split) from b, the rest from b2, both [rows, K]
    if (p.n_split % BN != 0 || p.n_split >= p.N) return DIT_EUNSUPPORTED;
    if (epi == kEpiQKVSwiGLU && (BN != 256 || BN % p.head_dim != 0 || p.n_split != 3 * p.H)) return DIT_EUNSUPPORTED;
    if (!al(a, lda) || !al(b, ldb) || !al(b2, ldb2)) return DIT_EINVAL;
    if (!tmap_bf16(&m.a, a, p.K, p.M, lda, BM) || !tmap_bf16(&m.b, b, p.K, p.n_split, ldb, bbox) ||
        !tmap_bf16(&m.b2, b2, p.K, p.N - p.n_split, ldb2, bbox))
      return DIT_ECUDA;
    m.a2 = m.a;
  } else if (p.m_split > 0) {
    // rows [0, m_split) with the weights b, rows [m_split, M) with b2 (both [N, K]); a boundary inside
    // a row tile pads each group to whole tiles
    if (p.m_split >= p.M || epi == kEpiQKVSwiGLU) return DIT_EUNSUPPORTED;
    if (epi == kEpiQKV && (BN % p.head_dim != 0 || p.H % BN != 0)) return DIT_EUNSUPPORTED;
    if (!al(a, lda) || !al(b, ldb) || !al(b2, ldb2)) return DIT_EINVAL;
    if (!tmap_bf16(&m.a, a, p.K, p.M, lda, BM) || !tmap_bf16(&m.b, b, p.K, p.N, ldb, bbox) ||
        !tmap_bf16(&m.b2, b2, p.K, p.N, ldb2, bbox))
      return DIT_ECUDA;
    m.a2 = m.a;
  } else {
    // A = [a | a2], B = [b | b2]: inner columns [0, k_split) from a and b, the rest from a2 and b2
    if (p.k_split % BK != 0 || p.k_split >= p.K || epi == kEpiQKVSwiGLU) return DIT_EUNSUPPORTED;
    if (epi == kEpiQKV && (BN % p.head_dim != 0 || p.H % BN != 0)) return DIT_EUNSUPPORTED;
    if (!al(a, lda) || !al(a2, lda2) || !al(b, ldb) || !al(b2, ldb2)) return DIT_EINVAL;
    const int k2 = p.K - p.k_split, b2_inner = p.b2_inner > 0 ? p.b2_inner : k2;
    if (b2_inner > k2) return DIT_EINVAL;
    if (!tmap_bf16(&m.a, a, p.k_split, p.M, lda, BM) || !tmap_bf16(&m.a2, a2, k2, p.M, lda2, BM) ||
        !tmap_bf16(&m.b, b, p.k_split, p.N, ldb, bbox) || !tmap_bf16(&m.b2, b2, b2_inner, p.N, ldb2, bbox))
      return DIT_ECUDA;
  }
  m.s = m.b;
  return launch_bf16(m, BN, epi, p, pair, stream);
}

}  // namespace dit
