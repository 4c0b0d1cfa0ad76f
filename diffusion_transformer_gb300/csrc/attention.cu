// Joint-sequence flash attention forward on tcgen05 for sm_103a.
//
//   o[r, n*d + j] = sum_c softmax_c( q_n[r] . k_n[c] / sqrt(d) ) v_n[c, j]      over all R rows, no mask
//
// The klein-4B article (section 4.3) gives the method: tile the queries, stream key/value tiles
// through on-chip memory and keep a running row max m and sum l, rescaling the accumulator by
// exp(m_old - m_new) ("online softmax", exact up to rounding order), applying 1/sqrt(d) in fp32.
//
// GB300 mapping. A unit is (pair of 128-query tiles, head), its steps are its 128-key tiles. A CTA
// works through a range of steps: one whole unit, or (persistent schedule) an equal share of all
// units' steps per SM, a unit cut between two CTAs being finished by the one holding its first key
// tiles, which starts from the partial O, l (and m) the other left in the caller's scratch. Warp 0
// loads Q0, Q1 per unit and the K/V tiles with TMA into a 2-deep ring; warp 1 issues every MMA; the
// softmax warps turn S into P (running maximum: warps 2-5 tile 0, warps 6-9 tile 1, one query row
// per thread; fixed maximum: all of them on each tile in turn). While one tile's softmax runs, the
// tensor core runs the other tile's S = Q K^T and O += P V, so the exponentials and the MMAs of the
// two tiles overlap; under the fixed maximum the first half of each key part's P is announced
// early and half of the P V runs while the softmax finishes. Output tiles are normalised into a
// 128B-swizzled staging buffer and leave by TMA tensor stores. Tensor memory (512 columns):
//   [0, 128) S0, overwritten by P0   [128, 256) S1 / P1   [256, 256 + d) O0   [256 + d, 256 + 2d) O1
// The softmax reads S from TMEM, writes P (bf16, two keys per 32-bit column) back over the columns
// it has consumed, and the P V MMA reads A straight from TMEM. MMAs issued by one thread complete
// in order, so S(j+1) is issued right after P V(j) reads P(j) from the same columns, and the
// completion of S(j+1) also tells the softmax that P V(j) is done with O and P.
// The running max m only moves when a row's max exceeds it by more than 8 (log2 units), so the
// rescale of O in TMEM is rare; until then the weights exp2(s - m) stay below 2^8, and the final
// O / l is the same softmax.
// Fixed maximum: when q and k rows come RMS-normalised and weighted from the QKV epilogue,
// |q| <= sqrt(d) max|w_q| and |k| <= sqrt(d) max|w_k| (the rotation keeps the norm), so every scaled
// score lies in [-B, B], B = d max|w_q| max|w_k| scale (log2 units, with a margin for the bf16
// rounding). For B below 60 the softmax subtracts m = B throughout: the weights exp2(s - B) lie in
// [2^-120, 1], normal in fp32 and bf16, the same relative rounding as with a running max, and no row
// max is needed. Then no thread needs a whole row, and all the softmax warps work on each query
// tile in turn, warp (quadrant, part) taking 32 rows and 128 / parts of the keys (four parts and
// sixteen warps at d = 128, two parts and eight warps at d = 64): several warps per SM
// sub-partition share every softmax, so its latency drops and the next S no longer waits on it.
// P of key part p goes to the first half of that part's own S columns (inside what that warp has
// consumed), and the P V MMA reads it from there.
// V arrives transposed ([d, keys]) from the QKV epilogue so the P V MMA takes a K-major B operand.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace dit {

// Ready words of the persistent schedule: block (epoch % kAttnSlots) of a launch holds one word per
// CTA, set to the launch's epoch once that CTA's partial is complete. Launches on other streams take
// other epochs, hence other blocks or other values.
constexpr uint32_t kAttnSlots = 64;
constexpr int kAttnMaxCtas = 1024;
__device__ uint32_t g_attn_ready[kAttnSlots * kAttnMaxCtas];

namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct AttnCfg {
  static constexpr uint32_t kAtom = 128 * 128;          // one [128 rows x 64 bf16] swizzled atom
  static constexpr uint32_t kQBytes = 128 * D * 2;      // one query tile, D/64 atoms
  static constexpr uint32_t kKBytes = 128 * D * 2;      // per stage, D/64 atoms
  static constexpr uint32_t kVAtom = D * 128;           // [D rows x 64 keys]
  static constexpr uint32_t kVBytes = 2 * kVAtom;       // per stage (128 keys)
  static constexpr uint32_t kStageBytes = 128 * D * 2;  // one bf16 output tile
  static constexpr uint32_t kBarBytes = 8 * 24;
  static constexpr uint32_t kSmemNeed = 1024 + 2 * kQBytes + 2 * kKBytes + 2 * kVBytes + kStageBytes + kBarBytes + 16;
  // at least 116 KB so that two CTAs never share an SM (each allocates all 512 TMEM columns)
  static constexpr uint32_t kSmemBytes = kSmemNeed > 116 * 1024 ? kSmemNeed : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  // partial of a unit split between two CTAs: unnormalised O of both tiles ([tile][d / 4 groups of
  // four columns][128 rows] float4), then the row sums l and the running maxima m ([tile][128] each)
  static constexpr size_t kPartBytes = size_t(2) * 128 * D * 4 + 2 * 2 * 128 * 4;
};

// Softmax modes: running maximum, or fixed maximum (QK-normed rows whose bound B is below 60). With
// norm weights other than ones the bound is known only on the device: both kernels are launched
// one after the other (AttnParams::select), each computes B from the weights, and the one not
// chosen returns before its set-up (one kernel with both paths would take the running path's
// register allocation, and with it fewer softmax warps, for the common fixed case).
enum AttnMode : int { kAttnRunning = 0, kAttnFixed = 1 };
// Key parts per softmax row under the fixed maximum: four (sixteen softmax warps, four per SM
// sub-partition, 32 keys each) at d = 128, whose path needs about 100 registers; two at d = 64
// (d / 4 output columns would be narrower than one TMEM load). The running path keeps whole rows
// (168 registers) in two groups of four warps.
template <int D, int MODE>
struct AttnSplit {
  static constexpr int kParts = (MODE == kAttnFixed && D == 128) ? 4 : 2;
  static constexpr int kThreads = 64 + 128 * kParts;
};

// Output staging in the layout a TMA store with the 128-byte swizzle reads: the tile's columns in
// boxes of 64 (128 bytes a row), box b at b * 16 KB, the 16-byte chunk j of row r inside a box at
// r * 128 + ((j ^ (r & 7)) << 4), so that eight consecutive rows writing the same chunk hit
// distinct banks. One thread then stores the whole tile with D / 64 tensor stores (rows past R are
// not written), and the softmax warps go on while the copy engine moves it.
template <int D>
__device__ __forceinline__ void stage_chunk(uint8_t* stage, int r, int c, uint4 v) {
  *reinterpret_cast<uint4*>(stage + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
}
__device__ __forceinline__ uint4 pack8_scaled(const uint32_t* r, float s) {
  return make_uint4(pack_bf16x2(__uint_as_float(r[0]) * s, __uint_as_float(r[1]) * s),
                    pack_bf16x2(__uint_as_float(r[2]) * s, __uint_as_float(r[3]) * s),
                    pack_bf16x2(__uint_as_float(r[4]) * s, __uint_as_float(r[5]) * s),
                    pack_bf16x2(__uint_as_float(r[6]) * s, __uint_as_float(r[7]) * s));
}

// B = (1 + 2^-6)^2 d max|w_q| max|w_k| scale (log2 units) over the norm weights of every stream:
// every scaled score of QK-normed rows lies in [-B, B]. The margin per factor covers the bf16
// rounding of q and k and the fp32 normalisation. Computed by every warp (lane-strided max, then a
// butterfly), exactly the same in every warp and in both kernels of a pair of launches.
template <int D>
__device__ __noinline__ float qk_bound(const float* qn0, const float* kn0, const float* qn1, const float* kn1,
                                       int streams, float scale_log2) {
  const int lane = lane_id();
  float mq = 0.f, mk = 0.f;
  for (int i = lane; i < D; i += 32) {
    mq = fmaxf(mq, qn0 ? fabsf(qn0[i]) : 1.f);
    mk = fmaxf(mk, kn0 ? fabsf(kn0[i]) : 1.f);
    if (streams > 1) {
      mq = fmaxf(mq, qn1 ? fabsf(qn1[i]) : 1.f);
      mk = fmaxf(mk, kn1 ? fabsf(kn1[i]) : 1.f);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
    mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
  }
  return 1.015625f * mq * 1.015625f * mk * float(D) * scale_log2;
}

// Wait (bounded) until the ready word holds this launch's epoch; false after the limit or an error.
// The finisher is the word's only reader: it clears the word once seen, so that every launch starts
// from cleared words even when a captured graph replays the same epoch (the word's next writer is
// a later kernel in the stream).
__device__ __forceinline__ bool wait_ready(uint32_t* w, uint32_t epoch, int* err) {
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(w) != epoch)
    if (aborted(err) || globaltimer_ns() - t0 > 4 * kWaitLimitNs) {
      atomicCAS(err, 0, int(kErrTimeoutSoftmax));
      return false;
    }
  *w = 0u;
  return true;
}

template <int D, int MODE>
__global__ void __launch_bounds__(AttnSplit<D, MODE>::kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const AttnParams p,
                float scale_log2) {
  using Cfg = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                          // Q0, Q1
  uint8_t* sK = sQ + 2 * Cfg::kQBytes;         // 2 stages
  uint8_t* sV = sK + 2 * Cfg::kKBytes;         // 2 stages
  uint8_t* sStage = sV + 2 * Cfg::kVBytes;     // one output tile (and the parts' row sums)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + Cfg::kStageBytes);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;    // the segment's last S done: Q may be reloaded
  uint64_t* k_full = bars + 2;     // [2] per stage
  uint64_t* v_full = bars + 4;     // [2]
  uint64_t* k_empty = bars + 6;    // [2]
  uint64_t* v_empty = bars + 8;    // [2]
  uint64_t* s_full = bars + 10;    // [2] per query tile
  uint64_t* p_full = bars + 12;    // [2] per query tile
  uint64_t* o_done = bars + 14;    // [2] per query tile (a segment's last P V)
  uint64_t* o_ready = bars + 16;   // segment start: the last O read (and a finisher's partial put in)
  uint64_t* drain = bars + 17;
  uint64_t* p_half = bars + 18;    // [2] per query tile: the first half of each part's keys of P stored
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  uint32_t* ready_ok = tmem_slot + 1;  // finisher: the partial of the next CTA is there

  const int warp = threadIdx.x >> 5;
  const int lane = lane_id();
  const int R = p.R;
  const int nkv = (R + 127) / 128;   // key tiles (= query tiles)
  const int npairs = (nkv + 1) / 2;  // query-tile pairs per head
  // this CTA's steps [begin, end) of the unit-major sequence (unit u = head * npairs + pair, then
  // key tile); p.work = nkv gives one whole unit per CTA
  const int cta = int(blockIdx.y * gridDim.x + blockIdx.x);
  const long long total = (long long)p.heads * npairs * nkv;
  const long long begin = (long long)cta * p.work;
  const long long end = begin + p.work < total ? begin + p.work : total;
  auto seg_at = [&](long long s, int& u, int& j0, int& j1) {
    u = int(s / nkv);
    j0 = int(s - (long long)u * nkv);
    j1 = end - s < nkv - j0 ? j0 + int(end - s) : nkv;
  };
  auto slot_ptr = [&](int slot) { return reinterpret_cast<uint8_t*>(p.part) + size_t(slot) * Cfg::kPartBytes; };
  uint32_t* ready = g_attn_ready + (p.epoch % kAttnSlots) * kAttnMaxCtas;

  // the fixed maximum B from the norm weights (the same value in every warp and in either kernel of a
  // pair of launches)
  if (p.select != 0) {
    // one of a pair of launches over the same call (norm weights other than ones): the fixed kernel
    // works when B < 60, the running one otherwise; the other returns here, before any set-up
    // (the weights may come from the previous kernel in the stream, hence after its completion)
    pdl_wait();
    if ((p.select == 1) != (qk_bound<D>(p.qn0, p.kn0, p.qn1, p.kn1, p.qk_normed, scale_log2) < 60.f)) return;
  }
  float m_fixed = 0.f;
  constexpr bool fixed = MODE == kAttnFixed;
  constexpr int KS = AttnSplit<D, MODE>::kParts;
  const uint32_t softmax_warps = fixed ? 4 * KS : 8;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(q_empty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
      mbar_init(smem_u32(&s_full[s]), 1);
      // one arrival per softmax warp of the tile (each after its lanes' TMEM stores, fence and warp sync)
      mbar_init(smem_u32(&p_full[s]), fixed ? softmax_warps : 4);
      mbar_init(smem_u32(&p_half[s]), fixed ? softmax_warps : 4);
      mbar_init(smem_u32(&o_done[s]), 1);
    }
    mbar_init(smem_u32(o_ready), softmax_warps);
    mbar_init(smem_u32(drain), 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above may overlap the previous kernel in the stream; its results only from here
  pdl_wait();
  pdl_trigger();
  if constexpr (MODE == kAttnFixed) m_fixed = qk_bound<D>(p.qn0, p.kn0, p.qn1, p.kn1, p.qk_normed, scale_log2);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_one()) {
      int nq = 0, nk = 0, nv = 0;  // Q pairs, K tiles and V tiles issued
      bool ok = true;
      for (long long s = begin; s < end && ok;) {
        int u, j0, j1;
        seg_at(s, u, j0, j1);
        const int head = u / npairs, qp = u - head * npairs;
        // the previous segment's last S has read Q
        if (nq > 0 && !mbar_wait(smem_u32(q_empty), (nq - 1) & 1, p.err, kErrTimeoutProducer)) break;
        const uint32_t qb = smem_u32(q_full);
        mbar_arrive_expect_tx(qb, 2 * Cfg::kQBytes);
        for (int t = 0; t < 2; ++t)
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(smem_u32(sQ + t * Cfg::kQBytes + a * Cfg::kAtom), &tmQ, qb, a * 64, (2 * qp + t) * 128, head);
        ++nq;
        for (int j = j0; j < j1; ++j) {
          const int st = nk & 1;
          const uint32_t par = ((nk >> 1) & 1) ^ 1;
          if (!mbar_wait(smem_u32(&k_empty[st]), par, p.err, kErrTimeoutProducer)) { ok = false; break; }
          const uint32_t kb = smem_u32(&k_full[st]);
          mbar_arrive_expect_tx(kb, Cfg::kKBytes);
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(smem_u32(sK + st * Cfg::kKBytes + a * Cfg::kAtom), &tmK, kb, a * 64, j * 128, head);
          ++nk;
          if (!mbar_wait(smem_u32(&v_empty[st]), par, p.err, kErrTimeoutProducer)) { ok = false; break; }
          const uint32_t vb = smem_u32(&v_full[st]);
          mbar_arrive_expect_tx(vb, Cfg::kVBytes);
          for (int b = 0; b < 2; ++b)
            tma_load_3d(smem_u32(sV + st * Cfg::kVBytes + b * Cfg::kVAtom), &tmV, vb, j * 128 + b * 64, 0, head);
          ++nv;
        }
        s += j1 - j0;
      }
      // every issued copy lands before the CTA exits
      if (nq > 0) mbar_wait(smem_u32(q_full), (nq - 1) & 1, p.err, kErrTimeoutDrain);
      for (int i = nk - 2 < 0 ? 0 : nk - 2; i < nk; ++i)
        mbar_wait(smem_u32(&k_full[i & 1]), (i >> 1) & 1, p.err, kErrTimeoutDrain);
      for (int i = nv - 2 < 0 ? 0 : nv - 2; i < nv; ++i)
        mbar_wait(smem_u32(&v_full[i & 1]), (i >> 1) & 1, p.err, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128);
      constexpr uint32_t idesc_o = idesc_bf16(128, D);
      // descriptor low words of the three 1024-byte-aligned operand regions; tiles inside them add
      // their byte offset >> 4 (umma_bf16_lo), so each MMA costs two 32-bit adds besides itself
      const uint64_t dq = sw128_desc(smem_u32(sQ));
      const uint32_t q_lo = uint32_t(dq), d_hi = uint32_t(dq >> 32);
      const uint32_t k_lo = uint32_t(sw128_desc(smem_u32(sK))), v_lo = uint32_t(sw128_desc(smem_u32(sV)));
      auto issue_s = [&](int t, int g) {  // S_t = Q_t K^T (K tile g of the ring) into columns [128 t, 128 t + 128)
        const uint32_t dS = tmem_base + uint32_t(t * 128);
        const uint32_t qt = q_lo + uint32_t(t * (Cfg::kQBytes >> 4));
        const uint32_t ks = k_lo + uint32_t((g & 1) * (Cfg::kKBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t c = uint32_t((kk >> 2) * (Cfg::kAtom >> 4) + 2 * (kk & 3));
          umma_bf16_lo(dS, qt + c, ks + c, d_hi, idesc_s, kk != 0);
        }
        umma_commit(smem_u32(&s_full[t]));
      };
      // O_t += P_t V_g (O_t = on a segment's first tile unless it continues a partial); P_t in TMEM: keys 16 kk .. 16 kk + 15 at
      // column 128 t + 8 kk (running max), or inside their part's own S columns (fixed maximum: part
      // p of KP keys at 128 t + KP p)
      // In two halves: the key slices the softmax stores first (the first half of every part's keys,
      // or keys 0..63 under a running maximum), then the rest, so that half of P V runs while the
      // softmax finishes the tile.
      auto issue_pv = [&](int t, int g, bool first, int half) {
        const uint32_t dO = tmem_base + 256u + uint32_t(t * D);
        const uint32_t vs = v_lo + uint32_t((g & 1) * (Cfg::kVBytes >> 4));
        constexpr int KP = 128 / KS;  // keys per part (fixed maximum)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const bool in_first = fixed ? (kk * 16 % KP) < KP / 2 : kk < 4;
          if (in_first != (half == 0)) continue;
          const uint32_t c = uint32_t((kk >> 2) * (Cfg::kVAtom >> 4) + 2 * (kk & 3));
          const uint32_t pcol = fixed ? uint32_t(t * 128 + (kk * 16 / KP) * KP + (kk * 16 % KP) / 2) : uint32_t(t * 128 + kk * 8);
          umma_bf16_ts_lo(dO, tmem_base + pcol, vs + c, d_hi, idesc_o, !(first && kk == 0));
        }
      };
      int g = 0;     // key tiles consumed so far (ring position, s_full / p_full phase)
      int sidx = 0;  // segments started
      bool ok = true;
      for (long long s = begin; s < end && ok;) {
        int u, j0, j1;
        seg_at(s, u, j0, j1);
        const int n = j1 - j0;
        const bool finisher = j0 == 0 && j1 < nkv;  // O starts from the next CTA's partial
        if (!mbar_wait(smem_u32(q_full), sidx & 1, p.err, kErrTimeoutMma)) break;
        if (!mbar_wait(smem_u32(&k_full[g & 1]), (g >> 1) & 1, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
        issue_s(0, g);
        issue_s(1, g);
        umma_commit(smem_u32(&k_empty[g & 1]));
        if (n == 1) umma_commit(smem_u32(q_empty));
        for (int i = 0; i < n; ++i, ++g) {
          const int st = g & 1;
          const bool last = i + 1 == n;
          if (!mbar_wait(smem_u32(&v_full[st]), (g >> 1) & 1, p.err, kErrTimeoutMma)) { ok = false; break; }
          // K of the next tile is loaded long before the softmax of this one ends: wait for it
          // first, so that P V and the next S go out back to back once P is ready
          if (!last && !mbar_wait(smem_u32(&k_full[(g + 1) & 1]), ((g + 1) >> 1) & 1, p.err, kErrTimeoutMma)) { ok = false; break; }
          // tile 0: P V, then the next S over the same columns
          if (!mbar_wait(smem_u32(&p_half[0]), g & 1, p.err, kErrTimeoutMma)) { ok = false; break; }
          // a segment's first P V writes O: the softmax warps must have read the previous segment's
          // (and, for a finisher, put the partial in)
          if (i == 0 && !mbar_wait(smem_u32(o_ready), sidx & 1, p.err, kErrTimeoutMma)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, g, i == 0 && !finisher, 0);
          if (!mbar_wait(smem_u32(&p_full[0]), g & 1, p.err, kErrTimeoutMma)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, g, false, 1);
          if (last) umma_commit(smem_u32(&o_done[0]));
          else issue_s(0, g + 1);
          // tile 1
          if (!mbar_wait(smem_u32(&p_half[1]), g & 1, p.err, kErrTimeoutMma)) { ok = false; break; }
          tc_fence_after();
          issue_pv(1, g, i == 0 && !finisher, 0);
          if (!mbar_wait(smem_u32(&p_full[1]), g & 1, p.err, kErrTimeoutMma)) { ok = false; break; }
          tc_fence_after();
          issue_pv(1, g, false, 1);
          if (last) umma_commit(smem_u32(&o_done[1]));
          umma_commit(smem_u32(&v_empty[st]));
          if (!last) {
            issue_s(1, g + 1);
            umma_commit(smem_u32(&k_empty[(g + 1) & 1]));
            if (i + 2 == n) umma_commit(smem_u32(q_empty));  // the segment's last S
          }
        }
        ++sidx;
        s += n;
      }
      umma_commit(smem_u32(drain));
      mbar_wait(smem_u32(drain), 0, p.err, kErrTimeoutDrain);
    }
  } else if (fixed) {
    // ------------------------------------------------------------------ softmax warps, fixed max
    // warp (quad, part): rows quad * 32 + lane of each tile, keys [KP part, KP part + KP)
    constexpr int KP = 128 / KS, DC = D / KS;  // keys per part, output columns per warp
    const int part = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = uint32_t(quad * 32) << 16;
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    const uint64_t negm2 = f2_pack(-m_fixed, -m_fixed);
    float* lsum = reinterpret_cast<float*>(sStage);  // [tile][part][128 rows]
    const bool storer = threadIdx.x == 64;           // issues the tensor stores of the output
    bool ok = true;
    int g = 0, sidx = 0;
    for (long long s = begin; s < end;) {
      int u, j0, j1;
      seg_at(s, u, j0, j1);
      const int head = u / npairs, qp = u - head * npairs;
      const bool tail = j0 > 0;                   // the unit began on the previous CTA: leave a partial
      const bool finisher = j0 == 0 && j1 < nkv;  // the unit ends on the next CTA: start from its partial
      float l0 = 0.f, l1 = 0.f;  // row sums of the two tiles (scalars: an array indexed by t would sit in local memory)
      if (finisher) {
        // the next CTA left the partial at the start of its range, long before this point
        if (storer) *ready_ok = wait_ready(ready + cta + 1, p.epoch, p.err) ? 1u : 0u;
        asm volatile("bar.sync 1, %0;" ::"n"(128 * KS) : "memory");
        if (ok && *ready_ok) {
          const uint8_t* slot = slot_ptr(cta + 1);
          const float4* po = reinterpret_cast<const float4*>(slot) + size_t(part * (DC / 4)) * 128 + row;
#pragma unroll 1
          for (int t = 0; t < 2; ++t) {
#pragma unroll
            for (int c = 0; c < DC / 32; ++c) {
              uint32_t r[32];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float4 v = __ldcg(po + size_t(t * (D / 4) + c * 8 + k) * 128);
                r[4 * k] = __float_as_uint(v.x);
                r[4 * k + 1] = __float_as_uint(v.y);
                r[4 * k + 2] = __float_as_uint(v.z);
                r[4 * k + 3] = __float_as_uint(v.w);
              }
              tmem_st32(tmem_base + lane_off + 256u + uint32_t(t * D + part * DC + c * 32), r);
            }
          }
          if (part == 0) {  // the partial's row sums enter through part 0's
            const float* pl = reinterpret_cast<const float*>(slot + 2 * 128 * D * 4);
            l0 = __ldcg(pl + row);
            l1 = __ldcg(pl + 128 + row);
          }
          tmem_st_wait();
        }
      }
      // O is free for this segment's first P V (the previous segment's was read in its epilogue)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(o_ready));
      for (int j = j0; j < j1; ++j, ++g) {
        if (!ok) continue;
        const int valid = R - j * 128 - part * KP;  // keys of this part that exist (the same for the CTA)
        const bool full = valid >= KP;
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          if (!mbar_wait_warp(smem_u32(&s_full[t]), g & 1, p.err, kErrTimeoutSoftmax)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tS = tmem_base + lane_off + uint32_t(t * 128 + part * KP);
          uint32_t r[KP];
#pragma unroll
          for (int c = 0; c < KP / 32; ++c) tmem_ld32(tS + uint32_t(c * 32), *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
          tmem_ld_wait();
          uint64_t sum2[4] = {0, 0, 0, 0};  // eight fp32 partial sums (four packed pairs)
          // the first half of this part's keys, stored and announced (p_half), then the second
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[KP / 4];
#pragma unroll
            for (int i = 0; i < KP / 4; ++i) {
              const int k0 = h * (KP / 2) + 2 * i;
              const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(r[k0]), __uint_as_float(r[k0 + 1])), scale2, negm2);
              float p0 = ex2_approx(f2_lo(x2));
              float p1 = ex2_approx(f2_hi(x2));
              if (!full) {
                if (k0 >= valid) p0 = 0.f;
                if (k0 + 1 >= valid) p1 = 0.f;
              }
              sum2[i & 3] = f2_add(sum2[i & 3], f2_pack(p0, p1));
              pk[i] = pack_bf16x2(p0, p1);
            }
            tmem_st_cols(tS + uint32_t(h * (KP / 4)), pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(h == 0 ? &p_half[t] : &p_full[t]));
          }
          const uint64_t s01 = f2_add(sum2[0], sum2[1]), s23 = f2_add(sum2[2], sum2[3]);
          const uint64_t s4 = f2_add(s01, s23);
          const float ls = f2_lo(s4) + f2_hi(s4);
          if (t == 0) l0 += ls;
          else l1 += ls;
        }
      }
      // ---- segment end. Every softmax warp passes the same named barriers whatever happened.
      // MMAs complete in issue order, so once tile 0's last P V is done only tile 1's is left.
      bool done = ok && mbar_wait_warp(smem_u32(&o_done[0]), sidx & 1, p.err, kErrTimeoutSoftmax);
      if (storer) bulk_wait_read_all();  // the last tensor store has read the stage (row sums go there)
      asm volatile("bar.sync 1, %0;" ::"n"(128 * KS) : "memory");
      if (done) {
        lsum[(0 * KS + part) * 128 + row] = l0;
        lsum[(1 * KS + part) * 128 + row] = l1;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(128 * KS) : "memory");
      float lt0 = 0.f, lt1 = 0.f;
#pragma unroll
      for (int q = 0; q < KS; ++q) {
        lt0 += lsum[(0 * KS + q) * 128 + row];
        lt1 += lsum[(1 * KS + q) * 128 + row];
      }
      asm volatile("bar.sync 1, %0;" ::"n"(128 * KS) : "memory");  // row sums read: the stage is free
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        if (t == 1) done = done && mbar_wait_warp(smem_u32(&o_done[1]), sidx & 1, p.err, kErrTimeoutSoftmax);
        const uint32_t tO = tmem_base + lane_off + 256u + uint32_t(t * D + part * DC);
        if (tail) {
          // unnormalised O and the row sum of this unit's later key tiles, for the previous CTA
          float4* po = reinterpret_cast<float4*>(slot_ptr(cta)) + size_t(t * (D / 4) + part * (DC / 4)) * 128 + row;
          if (done) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < DC / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(tO + uint32_t(c * 32), r);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 8; ++k)
                __stcg(po + (c * 8 + k) * 128, make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                                          __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3])));
            }
            if (part == 0)
              __stcg(reinterpret_cast<float*>(slot_ptr(cta) + 2 * 128 * D * 4) + t * 128 + row, t == 0 ? lt0 : lt1);
          }
        } else {
          uint4 pk[DC / 8];  // this thread's normalised bf16 columns
          if (done) {
            tc_fence_after();
            const float inv_l = 1.0f / (t == 0 ? lt0 : lt1);
#pragma unroll
            for (int c = 0; c < DC / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(tO + uint32_t(c * 32), r);
              tmem_ld_wait();
#pragma unroll
              for (int q = 0; q < 4; ++q) pk[c * 4 + q] = pack8_scaled(&r[8 * q], inv_l);
            }
          }
          if (t == 1) {  // tile 0's store has read the stage
            if (storer) bulk_wait_read_all();
            asm volatile("bar.sync 1, %0;" ::"n"(128 * KS) : "memory");
          }
          if (done) {
#pragma unroll
            for (int q = 0; q < DC / 8; ++q) stage_chunk<D>(sStage, row, part * (DC / 8) + q, pk[q]);
          }
          fence_proxy_async_smem();
          asm volatile("bar.sync 1, %0;" ::"n"(128 * KS) : "memory");
          if (storer && done && (2 * qp + t) * 128 < R) {  // (a pair's second tile may lie past R)
            for (int b = 0; b < D / 64; ++b)
              tma_store_2d(&tmO, smem_u32(sStage + b * 16384), head * D + b * 64, (2 * qp + t) * 128);
            bulk_commit();
          }
        }
      }
      if (tail) {
        asm volatile("bar.sync 1, %0;" ::"n"(128 * KS) : "memory");  // every partial store issued
        if (storer && done) {
          __threadfence();
          st_release_gpu(ready + cta, p.epoch);
        }
      }
      ++sidx;
      s += j1 - j0;
    }
    if (storer) bulk_wait_all();
  } else {
    // ------------------------------------------------------------------ softmax warps 2..9, running max
    const int t = (warp - 2) >> 2;               // query tile of this warp group
    const int quad = warp & 3;                   // TMEM lanes this warp may access
    const int row = quad * 32 + lane;            // query row within the tile
    const uint32_t lane_off = uint32_t(quad * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + uint32_t(t * 128);
    const uint32_t tO = tmem_base + lane_off + 256u + uint32_t(t * D);
    const bool storer = threadIdx.x == 64 + 128 * t;  // first thread of each group: its tile's stores
    bool ok = true;
    int g = 0, sidx = 0;
    for (long long s = begin; s < end;) {
      int u, j0, j1;
      seg_at(s, u, j0, j1);
      const int head = u / npairs, qp = u - head * npairs;
      const bool tail = j0 > 0, finisher = j0 == 0 && j1 < nkv;
      float m = -INFINITY, l = 0.f;
      if (finisher) {
        // continue the online softmax from the state the next CTA left: its O, l and m
        if (threadIdx.x == 64) *ready_ok = wait_ready(ready + cta + 1, p.epoch, p.err) ? 1u : 0u;
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (ok && *ready_ok) {
          const uint8_t* slot = slot_ptr(cta + 1);
          const float4* po = reinterpret_cast<const float4*>(slot) + size_t(t * (D / 4)) * 128 + row;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float4 v = __ldcg(po + size_t(c * 8 + k) * 128);
              o[4 * k] = __float_as_uint(v.x);
              o[4 * k + 1] = __float_as_uint(v.y);
              o[4 * k + 2] = __float_as_uint(v.z);
              o[4 * k + 3] = __float_as_uint(v.w);
            }
            tmem_st32(tO + uint32_t(c * 32), o);
          }
          const float* pl = reinterpret_cast<const float*>(slot + 2 * 128 * D * 4);
          l = __ldcg(pl + t * 128 + row);
          m = __ldcg(pl + 2 * 128 + t * 128 + row);
          tmem_st_wait();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(o_ready));
      for (int j = j0; j < j1; ++j, ++g) {
        if (!ok) continue;
        if (!mbar_wait_warp(smem_u32(&s_full[t]), g & 1, p.err, kErrTimeoutSoftmax)) { ok = false; continue; }
        tc_fence_after();
        const int valid = R - j * 128;  // keys of this tile that exist (same for the whole CTA)
        const bool full = valid >= 128;
        // the whole S row in registers: four loads in flight, one wait
        uint32_t r[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + uint32_t(c * 32), *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
        tmem_ld_wait();
        // row max of the scaled scores (independent chains)
        float mx = -INFINITY;
        if (full) {
          float m8[8];
#pragma unroll
          for (int v = 0; v < 8; ++v) m8[v] = fmax3(__uint_as_float(r[v]), __uint_as_float(r[v + 8]), __uint_as_float(r[v + 16]));
#pragma unroll
          for (int k = 24; k < 128; k += 16) {
#pragma unroll
            for (int v = 0; v < 8; ++v) m8[v] = fmax3(m8[v], __uint_as_float(r[k + v]), __uint_as_float(r[k + 8 + v]));
          }
          // k = 24..119 covered in steps of 16 with two values each; the last 8 values (120..127)
#pragma unroll
          for (int v = 0; v < 8; ++v) m8[v] = fmaxf(m8[v], __uint_as_float(r[120 + v]));
          mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i < valid) mx = fmaxf(mx, __uint_as_float(r[i]));
        }
        mx *= scale_log2;
        float alpha = 1.f;
        if (mx > m + kRescaleThreshold) {  // also true on a fresh segment's first tile (m = -inf)
          alpha = ex2_approx(m - mx);
          m = mx;
        }
        // P = exp2(s * scale - m) as bf16 pairs into the consumed S columns; row sum in fp32
        const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
        const uint64_t negm2 = f2_pack(-m, -m);
        uint64_t sum2[4] = {0, 0, 0, 0};  // eight fp32 partial sums (four packed pairs)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int k0 = c * 32 + 2 * i;
            const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(r[k0]), __uint_as_float(r[k0 + 1])), scale2, negm2);
            float p0 = ex2_approx(f2_lo(x2));
            float p1 = ex2_approx(f2_hi(x2));
            if (!full) {
              if (k0 >= valid) p0 = 0.f;
              if (k0 + 1 >= valid) p1 = 0.f;
            }
            sum2[i & 3] = f2_add(sum2[i & 3], f2_pack(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + uint32_t(c * 16), pk);
        }
        const uint64_t s01 = f2_add(sum2[0], sum2[1]), s23 = f2_add(sum2[2], sum2[3]);
        const uint64_t s4 = f2_add(s01, s23);
        const float rowsum = f2_lo(s4) + f2_hi(s4);
        l = fmaf(l, alpha, rowsum);
        if ((j > j0 || finisher) && __any_sync(0xffffffffu, alpha < 1.0f)) {
          // O holds earlier tiles (or the partial): the wait on this S also covers the last P V
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + uint32_t(c * 32), o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + uint32_t(c * 32), o);
          }
        }
        // (a possible rescale of O precedes every P V of this tile: both halves announced together)
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&p_half[t]));
          mbar_arrive(smem_u32(&p_full[t]));
        }
      }
      // ---- segment end (both groups pass the same named barriers whatever happened)
      const bool done = ok && mbar_wait_warp(smem_u32(&o_done[t]), sidx & 1, p.err, kErrTimeoutSoftmax);
      if (tail) {
        uint8_t* slot = slot_ptr(cta);
        float4* po = reinterpret_cast<float4*>(slot) + size_t(t * (D / 4)) * 128 + row;  // [tile][D / 4][128 rows]
        float* pl = reinterpret_cast<float*>(slot + 2 * 128 * D * 4);                   // l, then m: [tile][128 rows]
        if (done) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + uint32_t(c * 32), o);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              __stcg(po + (c * 8 + k) * 128, make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                                        __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3])));
          }
          __stcg(pl + t * 128 + row, l);
          __stcg(pl + 2 * 128 + t * 128 + row, m);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");  // every partial store issued
        if (threadIdx.x == 64 && done) {
          __threadfence();
          st_release_gpu(ready + cta, p.epoch);
        }
      } else {
        // one staging buffer: tile 0's group stages first, tile 1's after tile 0's store has read it
        const float inv_l = 1.0f / l;
        if (t == 1) asm volatile("bar.sync 4, 256;" ::: "memory");
        else if (storer) bulk_wait_read_all();  // (the previous segment's tile 1 store: its group waited)
        if (t == 0) asm volatile("bar.sync 2, 128;" ::: "memory");
        if (done) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + uint32_t(c * 32), o);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q) stage_chunk<D>(sStage, row, c * 4 + q, pack8_scaled(&o[8 * q], inv_l));
          }
        }
        fence_proxy_async_smem();
        if (t == 0) asm volatile("bar.sync 2, 128;" ::: "memory");  // the tile's four warps
        else asm volatile("bar.sync 3, 128;" ::: "memory");
        if (storer && done && (2 * qp + t) * 128 < R) {  // (a pair's second tile may lie past R)
          for (int b = 0; b < D / 64; ++b)
            tma_store_2d(&tmO, smem_u32(sStage + b * 16384), head * D + b * 64, (2 * qp + t) * 128);
          bulk_commit();
        }
        if (t == 0) {
          if (storer) bulk_wait_read_all();
          asm volatile("bar.arrive 4, 256;" ::: "memory");
        } else if (storer) {
          bulk_wait_read_all();  // before the next segment's tile 0 stages
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
      }
      ++sidx;
      s += j1 - j0;
    }
    if (storer) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

// The persistent schedule: worth it when the units (query-tile pairs x heads, one per CTA, one CTA
// per SM) leave the last wave part-empty. Each CTA then takes ceil(steps / SMs) key-tile steps,
// at least one unit's worth, so a unit spans at most two CTAs. ctas = 0: one CTA per unit.
struct AttnPlan {
  long long ctas;
  int work;
};
AttnPlan attn_plan(long long R, long long heads) {
  const long long nkv = (R + 127) / 128, units = heads * ((nkv + 1) / 2), total = units * nkv;
  const long long sms = num_sms();
  if (sms <= 0 || units <= sms || units % sms == 0) return {0, 0};
  const long long work = (total + sms - 1) / sms;
  const long long ctas = (total + work - 1) / work;
  if (ctas > kAttnMaxCtas || work > (1LL << 30)) return {0, 0};
  return {ctas, int(work)};
}

uint32_t next_epoch() {
  static std::atomic<uint32_t> counter[64];
  int dev = 0;
  cudaGetDevice(&dev);
  uint32_t e = counter[dev & 63].fetch_add(1) + 1;
  if (e == 0) e = counter[dev & 63].fetch_add(1) + 1;  // 0 is the words' initial value
  return e;
}

template <int D>
int launch_d(const AttnParams& p0, cudaStream_t stream) {
  using Cfg = AttnCfg<D>;
  static_assert(Cfg::kSmemBytes <= 227 * 1024, "shared memory budget");
  AttnParams p = p0;
  CUtensorMap tq, tk, tv;
  const long long R = p.R, Rp = p.Rp, nh = p.heads;
  if (!make_tmap_3d_bf16(&tq, p.q, D, R, nh, D * 2, R * D * 2, 64, 128)) return DIT_ECUDA;
  if (!make_tmap_3d_bf16(&tk, p.k, D, R, nh, D * 2, R * D * 2, 64, 128)) return DIT_ECUDA;
  if (!make_tmap_3d_bf16(&tv, p.vt, R, D, nh, Rp * 2, D * Rp * 2, 64, D)) return DIT_ECUDA;
  CUtensorMap to;  // o [R, heads * d] bf16, stored in boxes of 64 columns x 128 rows
  if (!make_tmap_2d(&to, p.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, nh * D, R, nh * D * 2, 64, 128, true))
    return DIT_ECUDA;
  // unit norm weights give B = 1.0157^2 d scale = 16.8 (d = 128) or 11.9 (d = 64): always fixed
  const bool unit = !p.qn0 && !p.kn0 && (p.qk_normed < 2 || (!p.qn1 && !p.kn1));
  const float scale_log2 = float(1.4426950408889634 / std::sqrt(double(D)));
  // one CTA per (query-tile pair, head); or, when that leaves the last wave part-empty and the
  // caller lent scratch for the partials, one CTA per SM over an equal share of the key tiles
  const AttnPlan pl = attn_plan(p.R, p.heads);
  auto launch = [&](auto kern, int threads, int select) -> int {
    if (!smem_attr_once(reinterpret_cast<const void*>(kern), Cfg::kSmemBytes)) return DIT_ECUDA;
    AttnParams q = p;
    q.select = select;
    dim3 grid = dim3(unsigned((q.R + 255) / 256), unsigned(q.heads));
    q.work = (q.R + 127) / 128;
    q.epoch = 0;
    if (pl.ctas > 0 && q.part && size_t(pl.ctas) * Cfg::kPartBytes <= q.part_bytes &&
        (reinterpret_cast<uintptr_t>(q.part) & 15) == 0) {
      grid = dim3(unsigned(pl.ctas));
      q.work = pl.work;
      q.epoch = next_epoch();
    }
    if (launch_pdl(kern, grid, dim3(threads), Cfg::kSmemBytes, stream, 1, tq, tk, tv, to, q, scale_log2) != cudaSuccess)
      return DIT_ECUDA;
    return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
  };
  constexpr int kRunThreads = AttnSplit<D, kAttnRunning>::kThreads, kFixThreads = AttnSplit<D, kAttnFixed>::kThreads;
  if (p.qk_normed <= 0) return launch(attn_kernel<D, kAttnRunning>, kRunThreads, 0);
  if (unit) return launch(attn_kernel<D, kAttnFixed>, kFixThreads, 0);
  // the rare running case first, so that the common fixed kernel runs last and hands on directly
  const int rc = launch(attn_kernel<D, kAttnRunning>, kRunThreads, 2);
  return rc != DIT_OK ? rc : launch(attn_kernel<D, kAttnFixed>, kFixThreads, 1);
}

}  // namespace

size_t attention_part_bytes(int R, int heads, int head_dim) {
  if (R <= 0 || heads <= 0) return 0;
  const AttnPlan pl = attn_plan(R, heads);
  if (pl.ctas == 0) return 0;
  switch (head_dim) {
    case 64: return size_t(pl.ctas) * AttnCfg<64>::kPartBytes;
    case 128: return size_t(pl.ctas) * AttnCfg<128>::kPartBytes;
    default: return 0;
  }
}

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
