// Joint-sequence flash attention forward on tcgen05 for sm_103a.
//
//   o[r, n*d + j] = sum_c softmax_c( q_n[r] . k_n[c] / sqrt(d) ) v_n[c, j]      over all R rows, no mask
//
// The klein-4B article (section 4.3) gives the method: tile the queries, stream key/value tiles
// through on-chip memory and keep a running row max m and sum l, rescaling the accumulator by
// exp(m_old - m_new) ("online softmax", exact up to rounding order), applying 1/sqrt(d) in fp32.
//
// GB300 mapping: one CTA per (128-query tile, head). Warp 0 loads Q once and K/V tiles (128 keys)
// with TMA into a 2-deep ring; warp 1 issues S = Q K^T (M=128, N=128, K=d) into one of two TMEM
// S buffers and O += P V (M=128, N=d, K=128) into a TMEM O accumulator; warps 2-5 own one query
// row per thread: they read S from TMEM, do the online softmax in registers (exp2 in the log2
// domain), rescale O in TMEM when the max moves, and write P as bf16 into a swizzled shared tile
// the next MMA reads. S of tile j+1 is computed while the softmax of tile j runs.
// V arrives transposed ([d, keys]) from the QKV epilogue so both MMAs take K-major operands.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace dit {
namespace {

template <int D>
struct AttnCfg {
  static constexpr int kThreads = 192;
  static constexpr uint32_t kAtom = 128 * 128;          // one [128 rows x 64 bf16] swizzled atom
  static constexpr uint32_t kQBytes = 128 * D * 2;      // D/64 atoms
  static constexpr uint32_t kKBytes = 128 * D * 2;      // per stage, D/64 atoms
  static constexpr uint32_t kVAtom = D * 128;           // [D rows x 64 keys]
  static constexpr uint32_t kVBytes = 2 * kVAtom;       // per stage (128 keys)
  static constexpr uint32_t kPBytes = 2 * kAtom;        // [128 rows x 128 keys]
  static constexpr uint32_t kBarBytes = 8 * 16;
  static constexpr uint32_t kSmemNeed = 1024 + kQBytes + 2 * kKBytes + 2 * kVBytes + kPBytes + kBarBytes + 16;
  // at least 116 KB so that two CTAs never share an SM (each allocates all 512 TMEM columns)
  static constexpr uint32_t kSmemBytes = kSmemNeed > 116 * 1024 ? kSmemNeed : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;            // S0 [0,128), S1 [128,256), O [256, 256+D)
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnParams p, float scale_log2) {
  using Cfg = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + Cfg::kQBytes;
  uint8_t* sV = sK + 2 * Cfg::kKBytes;
  uint8_t* sP = sV + 2 * Cfg::kVBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + Cfg::kPBytes);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;     // [2]
  uint64_t* v_full = bars + 3;     // [2]
  uint64_t* kv_empty = bars + 5;   // [2]
  uint64_t* s_full = bars + 7;     // [2]
  uint64_t* p_full = bars + 9;
  uint64_t* o_done = bars + 10;
  uint64_t* drain = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);

  const int warp = threadIdx.x >> 5;
  const int lane = lane_id();
  const int qt = blockIdx.x;
  const int head = blockIdx.y;
  const int R = p.R;
  const int nkv = (R + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&kv_empty[s]), 1);
      mbar_init(smem_u32(&s_full[s]), 1);
    }
    mbar_init(smem_u32(p_full), 128);
    mbar_init(smem_u32(o_done), 1);
    mbar_init(smem_u32(drain), 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tmem_o = tmem_base + 256;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_one()) {
      const uint32_t qb = smem_u32(q_full);
      mbar_arrive_expect_tx(qb, Cfg::kQBytes);
      for (int a = 0; a < D / 64; ++a) tma_load_3d(smem_u32(sQ + a * Cfg::kAtom), &tmQ, qb, a * 64, qt * 128, head);
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int s = j & 1;
        if (!mbar_wait(smem_u32(&kv_empty[s]), ((j >> 1) & 1) ^ 1, p.err, kErrTimeoutProducer)) break;
        const uint32_t kb = smem_u32(&k_full[s]);
        mbar_arrive_expect_tx(kb, Cfg::kKBytes);
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(smem_u32(sK + s * Cfg::kKBytes + a * Cfg::kAtom), &tmK, kb, a * 64, j * 128, head);
        const uint32_t vb = smem_u32(&v_full[s]);
        mbar_arrive_expect_tx(vb, Cfg::kVBytes);
        for (int b = 0; b < 2; ++b)
          tma_load_3d(smem_u32(sV + s * Cfg::kVBytes + b * Cfg::kVAtom), &tmV, vb, j * 128 + b * 64, 0, head);
        issued = j + 1;
      }
      // every issued copy lands before the CTA exits
      mbar_wait(qb, 0, p.err, kErrTimeoutDrain);
      for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j) {
        mbar_wait(smem_u32(&k_full[j & 1]), (j >> 1) & 1, p.err, kErrTimeoutDrain);
        mbar_wait(smem_u32(&v_full[j & 1]), (j >> 1) & 1, p.err, kErrTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128);
      constexpr uint32_t idesc_o = idesc_bf16(128, D);
      bool ok = mbar_wait(smem_u32(q_full), 0, p.err, kErrTimeoutMma);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(smem_u32(&k_full[s]), (j >> 1) & 1, p.err, kErrTimeoutMma)) return false;
        tc_fence_after();
        const uint32_t dS = tmem_base + uint32_t(s * 128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a = kk >> 2, off = uint32_t(2 * (kk & 3));
          const uint64_t ad = sw128_desc(smem_u32(sQ + a * Cfg::kAtom)) + off;
          const uint64_t bd = sw128_desc(smem_u32(sK + s * Cfg::kKBytes + a * Cfg::kAtom)) + off;
          umma_bf16(dS, ad, bd, idesc_s, kk != 0);
        }
        umma_commit(smem_u32(&s_full[s]));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nkv && ok; ++j) {
        if (j + 1 < nkv && !issue_s(j + 1)) break;
        const int s = j & 1;
        if (!mbar_wait(smem_u32(p_full), j & 1, p.err, kErrTimeoutMma)) break;
        if (!mbar_wait(smem_u32(&v_full[s]), (j >> 1) & 1, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t b = kk >> 2, off = uint32_t(2 * (kk & 3));
          const uint64_t ad = sw128_desc(smem_u32(sP + b * Cfg::kAtom)) + off;
          const uint64_t bd = sw128_desc(smem_u32(sV + s * Cfg::kVBytes + b * Cfg::kVAtom)) + off;
          umma_bf16(tmem_o, ad, bd, idesc_o, (j | kk) != 0);
        }
        umma_commit(smem_u32(o_done));
        umma_commit(smem_u32(&kv_empty[s]));
      }
      umma_commit(smem_u32(drain));
      mbar_wait(smem_u32(drain), 0, p.err, kErrTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps 2..5
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_off = uint32_t(quad * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int s = j & 1;
      if (!mbar_wait_warp(smem_u32(&s_full[s]), (j >> 1) & 1, p.err, kErrTimeoutSoftmax)) { ok = false; break; }
      tc_fence_after();
      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem_base + lane_off + uint32_t(s * 128 + c * 32), r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(r[i]);
      }
      const int valid = R - j * 128;
      if (valid < 128) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= valid) sv[i] = -INFINITY;
      }
      float mx = sv[0];
#pragma unroll
      for (int i = 1; i < 128; ++i) mx = fmaxf(mx, sv[i]);
      const float m_new = fmaxf(m, mx * scale_log2);
      const float alpha = ex2_approx(m - m_new);
      float rowsum = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float p0 = ex2_approx(fmaf(sv[2 * i], scale_log2, -m_new));
        const float p1 = ex2_approx(fmaf(sv[2 * i + 1], scale_log2, -m_new));
        rowsum += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l = fmaf(l, alpha, rowsum);
      m = m_new;
      if (j > 0) {
        // PV of the previous tile must finish before O is rescaled and P is overwritten
        if (!mbar_wait_warp(smem_u32(o_done), (j - 1) & 1, p.err, kErrTimeoutSoftmax)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha < 1.0f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            const uint32_t ta = tmem_o + lane_off + uint32_t(c * 32);
            tmem_ld32(ta, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(ta, r);
          }
          tmem_st_wait();
        }
      }
#pragma unroll
      for (int k8 = 0; k8 < 16; ++k8) {
        uint8_t* atom = sP + (k8 >> 3) * Cfg::kAtom;
        *reinterpret_cast<uint4*>(atom + sw128_offset(uint32_t(row), uint32_t(k8 & 7))) =
            make_uint4(pk[4 * k8], pk[4 * k8 + 1], pk[4 * k8 + 2], pk[4 * k8 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(p_full));
    }
    if (ok && mbar_wait_warp(smem_u32(o_done), (nkv - 1) & 1, p.err, kErrTimeoutSoftmax)) {
      tc_fence_after();
      const int grow = qt * 128 + row;
      const float inv_l = 1.0f / l;
      const int H = p.heads * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem_o + lane_off + uint32_t(c * 32), r);
        tmem_ld_wait();
        if (grow < R) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + size_t(grow) * H + head * D + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * q + 0]) * inv_l, __uint_as_float(r[8 * q + 1]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv_l, __uint_as_float(r[8 * q + 3]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv_l, __uint_as_float(r[8 * q + 5]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv_l, __uint_as_float(r[8 * q + 7]) * inv_l));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

template <int D>
int launch_d(const AttnParams& p, cudaStream_t stream) {
  using Cfg = AttnCfg<D>;
  static_assert(Cfg::kSmemBytes <= 227 * 1024, "shared memory budget");
  CUtensorMap tq, tk, tv;
  const long long R = p.R, Rp = p.Rp, nh = p.heads;
  if (!make_tmap_3d_bf16(&tq, p.q, D, R, nh, D * 2, R * D * 2, 64, 128)) return DIT_ECUDA;
  if (!make_tmap_3d_bf16(&tk, p.k, D, R, nh, D * 2, R * D * 2, 64, 128)) return DIT_ECUDA;
  if (!make_tmap_3d_bf16(&tv, p.vt, R, D, nh, Rp * 2, D * Rp * 2, 64, D)) return DIT_ECUDA;
  auto kern = attn_kernel<D>;
  if (!smem_attr_once(reinterpret_cast<const void*>(kern), Cfg::kSmemBytes)) return DIT_ECUDA;
  const float scale_log2 = float(1.4426950408889634 / std::sqrt(double(D)));
  dim3 grid((p.R + 127) / 128, p.heads);
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, p, scale_log2);
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

}  // namespace

int attention_launch(const AttnParams& p, cudaStream_t stream) {
  if (p.R <= 0 || p.heads <= 0) return DIT_EINVAL;
  if (p.Rp % 8 != 0 || p.Rp < p.R) return DIT_EINVAL;
  switch (p.head_dim) {
    case 64: return launch_d<64>(p, stream);
    case 128: return launch_d<128>(p, stream);
    default: return DIT_EUNSUPPORTED;
  }
}

}  // namespace dit
