// HBM-bound row and elementwise kernels: modulated RMSNorm, FlowMatch Euler step, rotary tables,
// timestep sinusoids, fp32 -> bf16 conversion and the int8lin dequantisation used for checking.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kNormThreads = 256;

// Modulated RMSNorm (the gizai:dit reference's normedInto with its Modulation rows):
//   h[r] = bf16( x[r] * rsqrt(mean(x[r]^2) + eps) * w * (1 + scale[m]) + shift[m] )
// one CTA per row, fp32 statistics (klein article, section 2: fp32 RMSNorm -> bf16). Every load of
// the row (x, shift, scale, w) is issued before the reduction, so one pass over global memory
// serves both the statistics and the output. NC = float4 chunks per thread (H = NC * 4 * 256);
// NC = 0 is the generic two-pass form for other widths.
// Sum over the CTA (every thread gets the same total, added in the same order).
__device__ __forceinline__ float block_sum(float v, float* part) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();  // earlier readers of part are done
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += part[i];
  return tot;
}

// LN = false: RMS norm (the row's mean taken as 0, so (x - 0) is x exactly); LN = true: LayerNorm,
// the mean subtracted first and the variance taken over the deviations (two passes over values held
// in registers, no E[x^2] - mean^2 cancellation).
template <int NC, bool LN>
__global__ void __launch_bounds__(kNormThreads) modnorm_kernel(const ModNormParams p) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const float* x = r < p.L ? p.txt + size_t(r) * p.ld_txt : p.img + size_t(r - p.L) * p.ld_img;
  const int m = p.map ? __ldg(p.map + r) : 0;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const float4* sh4 = reinterpret_cast<const float4*>(p.shift + size_t(m) * p.mod_stride);
  const float4* sc4 = reinterpret_cast<const float4*>(p.scale + size_t(m) * p.mod_stride);
  const float4* w4 = reinterpret_cast<const float4*>((p.split_w && r >= p.L) ? p.w_img : p.w);
  const int n4 = p.H >> 2;
  __shared__ float part[kNormThreads / 32];

  if constexpr (NC > 0) {
    float4 xv[NC], sh[NC], sc[NC], wv[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      const int i = threadIdx.x + k * kNormThreads;
      xv[k] = x4[i];
      sh[k] = __ldg(sh4 + i);
      sc[k] = __ldg(sc4 + i);
      wv[k] = w4 ? __ldg(w4 + i) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
    float mean = 0.f;
    if constexpr (LN) {
      float s1 = 0.f;
#pragma unroll
      for (int k = 0; k < NC; ++k) s1 += (xv[k].x + xv[k].y) + (xv[k].z + xv[k].w);
      mean = block_sum(s1, part) / float(p.H);
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        xv[k].x -= mean;
        xv[k].y -= mean;
        xv[k].z -= mean;
        xv[k].w -= mean;
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      ss = fmaf(xv[k].x, xv[k].x, ss);
      ss = fmaf(xv[k].y, xv[k].y, ss);
      ss = fmaf(xv[k].z, xv[k].z, ss);
      ss = fmaf(xv[k].w, xv[k].w, ss);
    }
    const float rstd = rsqrtf(block_sum(ss, part) / float(p.H) + p.eps);
    uint2* out = reinterpret_cast<uint2*>(p.out + size_t(r) * p.H);
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      const float y0 = fmaf(xv[k].x * rstd * wv[k].x, 1.f + sc[k].x, sh[k].x);
      const float y1 = fmaf(xv[k].y * rstd * wv[k].y, 1.f + sc[k].y, sh[k].y);
      const float y2 = fmaf(xv[k].z * rstd * wv[k].z, 1.f + sc[k].z, sh[k].z);
      const float y3 = fmaf(xv[k].w * rstd * wv[k].w, 1.f + sc[k].w, sh[k].w);
      out[threadIdx.x + k * kNormThreads] = make_uint2(pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
    }
  } else {
    float mean = 0.f;
    if constexpr (LN) {
      float s1 = 0.f;
      for (int i = threadIdx.x; i < n4; i += kNormThreads) {
        const float4 v = x4[i];
        s1 += (v.x + v.y) + (v.z + v.w);
      }
      mean = block_sum(s1, part) / float(p.H);
    }
    float ss = 0.f;
    for (int i = threadIdx.x; i < n4; i += kNormThreads) {
      const float4 v = x4[i];
      const float a = v.x - mean, b = v.y - mean, c = v.z - mean, d = v.w - mean;
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
      ss = fmaf(c, c, ss);
      ss = fmaf(d, d, ss);
    }
    const float rstd = rsqrtf(block_sum(ss, part) / float(p.H) + p.eps);
    uint2* out = reinterpret_cast<uint2*>(p.out + size_t(r) * p.H);
    for (int i = threadIdx.x; i < n4; i += kNormThreads) {
      const float4 v = x4[i];
      const float4 shv = __ldg(sh4 + i);
      const float4 scv = __ldg(sc4 + i);
      float4 w = make_float4(1.f, 1.f, 1.f, 1.f);
      if (w4) w = __ldg(w4 + i);
      const float y0 = fmaf((v.x - mean) * rstd * w.x, 1.f + scv.x, shv.x);
      const float y1 = fmaf((v.y - mean) * rstd * w.y, 1.f + scv.y, shv.y);
      const float y2 = fmaf((v.z - mean) * rstd * w.z, 1.f + scv.z, shv.z);
      const float y3 = fmaf((v.w - mean) * rstd * w.w, 1.f + scv.w, shv.w);
      out[i] = make_uint2(pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
    }
  }
}

// FlowMatch Euler step (host contract, section 6): x + (sigma_next - sigma) * vel, each operation
// rounded separately in fp32.
__global__ void euler_kernel(float* __restrict__ x, const float* __restrict__ vel, long long n, float s0, float s1) {
  pdl_wait();
  pdl_trigger();
  const float dt = __fsub_rn(s1, s0);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    x[i] = __fadd_rn(x[i], __fmul_rn(dt, vel[i]));
}

__global__ void euler_kernel_v4(float4* __restrict__ x, const float4* __restrict__ vel, long long n4, float s0, float s1) {
  pdl_wait();
  pdl_trigger();
  const float dt = __fsub_rn(s1, s0);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 a = x[i];
    const float4 v = vel[i];
    a.x = __fadd_rn(a.x, __fmul_rn(dt, v.x));
    a.y = __fadd_rn(a.y, __fmul_rn(dt, v.y));
    a.z = __fadd_rn(a.z, __fmul_rn(dt, v.z));
    a.w = __fadd_rn(a.w, __fmul_rn(dt, v.w));
    x[i] = a;
  }
}

// Rotary tables (host contract, section 4): positions text i -> (i, i, i), image (y, x) ->
// (L, y - (h - h/2), x - (w - w/2)); axis widths (16, 56, 56) scaled by d / 128; column k of axis a
// holds pos_a * theta^(-2k / width_a), evaluated in fp64 and rounded once to fp32.
__global__ void rope_kernel(int L, int gh, int gw, int d, double theta, float* cos_out, float* sin_out, long long total) {
  pdl_wait();
  pdl_trigger();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int half = d / 2;
  const int r = int(idx / half);
  const int col = int(idx % half);
  const int w0 = 16 * d / 128, w1 = 56 * d / 128;
  int axis, k, width;
  if (col < w0 / 2) {
    axis = 0; k = col; width = w0;
  } else if (col < w0 / 2 + w1 / 2) {
    axis = 1; k = col - w0 / 2; width = w1;
  } else {
    axis = 2; k = col - w0 / 2 - w1 / 2; width = w1;
  }
  int pos;
  if (r < L) {
    pos = r;
  } else {
    const int t = r - L, y = t / gw, x = t % gw;
    pos = axis == 0 ? L : (axis == 1 ? y - (gh - gh / 2) : x - (gw - gw / 2));
  }
  const double f = 1.0 / pow(theta, double(2 * k) / double(width));
  const double ang = double(pos) * f;
  cos_out[idx] = float(cos(ang));
  sin_out[idx] = float(sin(ang));
}

struct SigmaList {
  float s[64];
};

// Timestep sinusoids (gizai:dit reference, sinusoids): row i = [cos | sin] of 1000 * t_i times
// 10000^(-k / (dim/2)), fp64 angles, stored bf16 as the time MLP's input.
__global__ void sinusoid_kernel(SigmaList sig, int steps, int dim, uint16_t* out) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int half = dim / 2;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const double f = pow(10000.0, -double(k) / double(half));
    const double ang = 1000.0 * double(sig.s[i]) * f;
    __nv_bfloat16 c = __double2bfloat16(cos(ang));
    __nv_bfloat16 s = __double2bfloat16(sin(ang));
    out[size_t(i) * dim + k] = *reinterpret_cast<uint16_t*>(&c);
    out[size_t(i) * dim + half + k] = *reinterpret_cast<uint16_t*>(&s);
  }
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ in, uint16_t* __restrict__ out, long long n) {
  pdl_wait();
  pdl_trigger();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    __nv_bfloat16 b = __float2bfloat16_rn(in[i]);
    out[i] = *reinterpret_cast<uint16_t*>(&b);
  }
}

// w[o, i] = bf16_rne(q[o, i] * s[o, i / 32]) with the same instructions as the GEMM converters:
// 16 consecutive values per chunk (cols % 32 == 0, so a chunk never straddles two scales); each
// thread keeps four chunks' loads in flight per iteration.
__global__ void dequant_kernel(const int8_t* __restrict__ q, const uint16_t* __restrict__ s, uint16_t* __restrict__ w,
                               long long rows, long long cols) {
  pdl_wait();
  pdl_trigger();
  constexpr int kU = 4;
  const long long chunks = rows * cols / 16;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long base = t; base < chunks; base += kU * nthreads) {
    uint4 q16[kU];
    uint32_t sc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long i = base + u * nthreads;
      if (i < chunks) {
        const long long e = 16 * i;
        q16[u] = *reinterpret_cast<const uint4*>(q + e);
        sc[u] = s[e >> 5];  // row * (cols / 32) + col / 32, since cols % 32 == 0
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long i = base + u * nthreads;
      if (i < chunks) {
        uint32_t out[8];
        dequant16(q16[u], sc[u], out);
        uint4* dst = reinterpret_cast<uint4*>(w + 16 * i);
        dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
        dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
      }
    }
  }
}

// Sandwich residual (branch outputs normed before their gate): one CTA per row, H/1024 float4
// chunks per thread of y (and y2) loaded before the reductions, then
// x += gate * (y * rstd * w + y2 * rstd2 * w2) with rstd = 1 and w = 1 for an un-normed branch.
template <int NC>
__global__ void __launch_bounds__(kNormThreads) sandwich_kernel(const SandwichParams p) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const bool text = r < p.L;
  float* x = text ? p.txt + size_t(r) * p.H : p.img + size_t(r - p.L) * p.H;
  const int m = p.map ? __ldg(p.map + r) : 0;
  const bool n1 = text ? p.norm_txt != 0 : p.norm_img != 0;  // the same for the whole CTA
  const bool two = p.y2 != nullptr;
  const bool n2 = two && p.norm2 != 0;
  const float4* y4 = reinterpret_cast<const float4*>(p.y + size_t(r) * p.H);
  const float4* z4 = two ? reinterpret_cast<const float4*>(p.y2 + size_t(r) * p.H) : nullptr;
  const float4* g4 = reinterpret_cast<const float4*>(p.gate + size_t(m) * p.mod_stride);
  const float4* w4 = n1 ? reinterpret_cast<const float4*>(text ? p.w : p.w_img) : nullptr;
  const float4* w24 = n2 ? reinterpret_cast<const float4*>(p.w2) : nullptr;
  float4* x4 = reinterpret_cast<float4*>(x);
  __shared__ float part[kNormThreads / 32];
  const int n4 = p.H >> 2;
  constexpr int K = NC > 0 ? NC : 1;
  float4 yv[K], zv[K];
  float ss = 0.f, ss2 = 0.f;
  auto acc = [](float s, float4 v) {
    s = fmaf(v.x, v.x, s);
    s = fmaf(v.y, v.y, s);
    s = fmaf(v.z, v.z, s);
    return fmaf(v.w, v.w, s);
  };
  if constexpr (NC > 0) {
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      yv[k] = y4[threadIdx.x + k * kNormThreads];
      if (two) zv[k] = z4[threadIdx.x + k * kNormThreads];
    }
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      ss = acc(ss, yv[k]);
      if (two) ss2 = acc(ss2, zv[k]);
    }
  } else {
    for (int i = threadIdx.x; i < n4; i += kNormThreads) {
      ss = acc(ss, y4[i]);
      if (two) ss2 = acc(ss2, z4[i]);
    }
  }
  const float rstd = n1 ? rsqrtf(block_sum(ss, part) / float(p.H) + p.eps) : 1.f;
  const float rstd2 = n2 ? rsqrtf(block_sum(ss2, part) / float(p.H) + p.eps) : 1.f;
  const float4 ones = make_float4(1.f, 1.f, 1.f, 1.f);
  auto apply = [&](int i, float4 v, float4 u) {
    const float4 g = __ldg(g4 + i);
    const float4 w = w4 ? __ldg(w4 + i) : ones;
    float4 b;  // the gated branches' sum before the gate
    b.x = v.x * rstd * w.x;
    b.y = v.y * rstd * w.y;
    b.z = v.z * rstd * w.z;
    b.w = v.w * rstd * w.w;
    if (two) {
      const float4 w2 = w24 ? __ldg(w24 + i) : ones;
      b.x += u.x * rstd2 * w2.x;
      b.y += u.y * rstd2 * w2.y;
      b.z += u.z * rstd2 * w2.z;
      b.w += u.w * rstd2 * w2.w;
    }
    float4 xv = x4[i];
    xv.x = fmaf(g.x, b.x, xv.x);
    xv.y = fmaf(g.y, b.y, xv.y);
    xv.z = fmaf(g.z, b.z, xv.z);
    xv.w = fmaf(g.w, b.w, xv.w);
    x4[i] = xv;
  };
  if constexpr (NC > 0) {
#pragma unroll
    for (int k = 0; k < NC; ++k) apply(threadIdx.x + k * kNormThreads, yv[k], two ? zv[k] : ones);
  } else {
    for (int i = threadIdx.x; i < n4; i += kNormThreads) apply(i, y4[i], two ? z4[i] : ones);
  }
}

// Diagnostic of the bounded-wait path every pipeline uses: one warp waits (mbar_wait_warp, the
// production wait with its 1 s limit) on an mbarrier of its own, which completes only when
// `complete` is set. Without it the wait gives up, the error word records the site and the kernel
// returns; nothing is trapped or left running.
constexpr int kErrTimeoutSelftest = 7;

__global__ void __launch_bounds__(32) wait_selftest_kernel(int complete, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (complete && threadIdx.x == 0) mbar_arrive(smem_u32(&bar));
  mbar_wait_warp(smem_u32(&bar), 0, err, kErrTimeoutSelftest);
}

int grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  const long long cap = 8LL * num_sms();
  if (g > cap) g = cap;
  return g < 1 ? 1 : int(g);
}

}  // namespace

int modnorm_launch(const ModNormParams& p, cudaStream_t stream) {
  if (p.R <= 0) return DIT_OK;
  const int chunks = p.H % (4 * kNormThreads) == 0 ? p.H / (4 * kNormThreads) : 0;
  cudaError_t rc;
  if (p.layernorm) {
    switch (chunks) {
      case 1: rc = launch_pdl(modnorm_kernel<1, true>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
      case 2: rc = launch_pdl(modnorm_kernel<2, true>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
      case 3: rc = launch_pdl(modnorm_kernel<3, true>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
      case 4: rc = launch_pdl(modnorm_kernel<4, true>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
      default: rc = launch_pdl(modnorm_kernel<0, true>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
    }
  } else {
    switch (chunks) {
      case 1: rc = launch_pdl(modnorm_kernel<1, false>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
      case 2: rc = launch_pdl(modnorm_kernel<2, false>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
      case 3: rc = launch_pdl(modnorm_kernel<3, false>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
      case 4: rc = launch_pdl(modnorm_kernel<4, false>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
      default: rc = launch_pdl(modnorm_kernel<0, false>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
    }
  }
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int euler_launch(float* x, const float* vel, long long n, float sigma, float sigma_next, cudaStream_t stream) {
  if (n <= 0) return DIT_OK;
  if (n % 4 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(vel) % 16 == 0) {
    if (launch_pdl(euler_kernel_v4, dim3(grid_for(n / 4, 256)), dim3(256), 0, stream, 1, reinterpret_cast<float4*>(x),
                   reinterpret_cast<const float4*>(vel), n / 4, sigma, sigma_next) != cudaSuccess)
      return DIT_ECUDA;
  } else {
    if (launch_pdl(euler_kernel, dim3(grid_for(n, 256)), dim3(256), 0, stream, 1, x, vel, n, sigma, sigma_next) !=
        cudaSuccess)
      return DIT_ECUDA;
  }
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int rope_tables_launch(int L, int gh, int gw, int head_dim, float theta, float* cos, float* sin, cudaStream_t stream) {
  const long long total = (long long)(L + gh * gw) * (head_dim / 2);
  if (total <= 0) return DIT_OK;
  rope_kernel<<<int((total + 255) / 256), 256, 0, stream>>>(L, gh, gw, head_dim, double(theta), cos, sin, total);
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int sinusoid_launch(const float* sigmas, int steps, int dim, uint16_t* out, cudaStream_t stream) {
  if (steps <= 0 || steps > 64) return DIT_EUNSUPPORTED;
  SigmaList sl{};
  for (int i = 0; i < steps; ++i) sl.s[i] = sigmas[i];
  if (launch_pdl(sinusoid_kernel, dim3(steps), dim3(128), 0, stream, 1, sl, steps, dim, out) != cudaSuccess)
    return DIT_ECUDA;
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int f32_to_bf16_launch(const float* in, uint16_t* out, long long n, cudaStream_t stream) {
  if (n <= 0) return DIT_OK;
  if (launch_pdl(f32_to_bf16_kernel, dim3(grid_for(n, 256)), dim3(256), 0, stream, 1, in, out, n) != cudaSuccess)
    return DIT_ECUDA;
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int sandwich_launch(const SandwichParams& p, cudaStream_t stream) {
  if (p.R <= 0) return DIT_OK;
  const int chunks = p.H % (4 * kNormThreads) == 0 ? p.H / (4 * kNormThreads) : 0;
  cudaError_t rc;
  switch (chunks) {
    case 1: rc = launch_pdl(sandwich_kernel<1>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
    case 2: rc = launch_pdl(sandwich_kernel<2>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
    case 3: rc = launch_pdl(sandwich_kernel<3>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
    case 4: rc = launch_pdl(sandwich_kernel<4>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
    default: rc = launch_pdl(sandwich_kernel<0>, dim3(p.R), dim3(kNormThreads), 0, stream, 1, p); break;
  }
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int wait_selftest_launch(int complete, int* err, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(complete, err);
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

// ----------------------------------------------------------------------------------------------
// W8A8 quantisers (klein article, section 5 and its D4/D5 entries): symmetric absmax / 127 codes,
// per token for activations (x / smooth first) and per output channel for weights (w * smooth,
// the SmoothQuant fold, first). Every decision in float32 with IEEE division (__fdiv_rn) and
// round-half-to-even (rintf), the codes clipped to [-127, 127]; a row of zeros has scale 0, codes 0.
// ----------------------------------------------------------------------------------------------
__device__ __forceinline__ float block_max(float v, float* part) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) m = fmaxf(m, part[i]);
  return m;
}

__device__ __forceinline__ float w8a8_code(float v, float scale) {
  if (scale == 0.f) return 0.f;
  return fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(v, scale))));
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// One CTA per row. The row is x[r, 0:K] followed by x2[r, 0:K2] (K2 = 0: x alone; both multiples of
// 8), quantised as one row: codes written over both as bf16 (exact small integers: the bf16 MMA then
// multiplies them exactly), the row's scale to scale[r]. The SmoothQuant divisors run over the
// joined row; rows from row_split on take smooth2 instead (the second stream's divisors; NULL: none).
// Two passes over the row (it is re-read from L2 after the maximum).
__global__ void __launch_bounds__(kNormThreads) quant_rows_kernel(uint16_t* x, int K, uint16_t* x2, int K2,
                                                                  const float* smooth, const float* smooth2,
                                                                  int row_split, float* scale) {
  pdl_wait();
  pdl_trigger();
  __shared__ float part[kNormThreads / 32];
  uint4* row = reinterpret_cast<uint4*>(x + size_t(blockIdx.x) * K);
  uint4* row2 = x2 ? reinterpret_cast<uint4*>(x2 + size_t(blockIdx.x) * K2) : nullptr;
  const int n8 = K / 8, n8_all = n8 + K2 / 8;
  const float* sm = int(blockIdx.x) >= row_split ? smooth2 : smooth;
  auto chunk = [&](int i) -> uint4* { return i < n8 ? row + i : row2 + (i - n8); };
  float m = 0.f;
  for (int i = threadIdx.x; i < n8_all; i += kNormThreads) {
    const uint4 u = *chunk(i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      if (sm) {
        a = __fdiv_rn(a, __ldg(sm + 8 * i + 2 * j));
        b = __fdiv_rn(b, __ldg(sm + 8 * i + 2 * j + 1));
      }
      m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
    }
  }
  const float sc = __fdiv_rn(block_max(m, part), 127.f);
  for (int i = threadIdx.x; i < n8_all; i += kNormThreads) {
    uint4* dst = chunk(i);
    const uint4 u = *dst;
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      if (sm) {
        a = __fdiv_rn(a, __ldg(sm + 8 * i + 2 * j));
        b = __fdiv_rn(b, __ldg(sm + 8 * i + 2 * j + 1));
      }
      o[j] = pack_bf16x2(w8a8_code(a, sc), w8a8_code(b, sc));  // integers up to 127: exact in bf16
    }
    *dst = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) scale[blockIdx.x] = sc;
}

__global__ void __launch_bounds__(kNormThreads) quant_weight_kernel(const uint16_t* w, int K, const float* smooth,
                                                                    int8_t* q, float* scale) {
  pdl_wait();
  pdl_trigger();
  __shared__ float part[kNormThreads / 32];
  const uint16_t* row = w + size_t(blockIdx.x) * K;
  auto val = [&](int k) {
    const float v = __uint_as_float(uint32_t(row[k]) << 16);
    return smooth ? __fmul_rn(v, __ldg(smooth + k)) : v;
  };
  float m = 0.f;
  for (int k = threadIdx.x; k < K; k += kNormThreads) m = fmaxf(m, fabsf(val(k)));
  const float sc = __fdiv_rn(block_max(m, part), 127.f);
  for (int k = threadIdx.x; k < K; k += kNormThreads) q[size_t(blockIdx.x) * K + k] = int8_t(w8a8_code(val(k), sc));
  if (threadIdx.x == 0) scale[blockIdx.x] = sc;
}

// int8 codes -> the same integers in bf16, 16 per thread step.
__global__ void codes_bf16_kernel(const int8_t* q, uint16_t* w, long long n16) {
  pdl_wait();
  pdl_trigger();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n16; i += (long long)gridDim.x * blockDim.x) {
    const uint4 u = reinterpret_cast<const uint4*>(q)[i];
    const uint32_t b[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int8_t* c = reinterpret_cast<const int8_t*>(&b[j]);
      o[2 * j] = pack_bf16x2(float(c[0]), float(c[1]));
      o[2 * j + 1] = pack_bf16x2(float(c[2]), float(c[3]));
    }
    uint4* dst = reinterpret_cast<uint4*>(w) + 2 * i;
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

int quant_rows_launch(uint16_t* x, int rows, int K, const float* smooth, float* scale, cudaStream_t stream) {
  return quant_rows_joint_launch(x, K, nullptr, 0, rows, smooth, nullptr, rows, scale, stream);
}

int quant_rows_joint_launch(uint16_t* x, int K, uint16_t* x2, int K2, int rows, const float* smooth,
                            const float* smooth2, int row_split, float* scale, cudaStream_t stream) {
  if (rows <= 0) return DIT_OK;
  if (K % 8 != 0 || K2 % 8 != 0 || (K2 > 0 && !x2)) return DIT_EUNSUPPORTED;
  if (launch_pdl(quant_rows_kernel, dim3(rows), dim3(kNormThreads), 0, stream, 1, x, K, x2, K2, smooth, smooth2,
                 row_split, scale) != cudaSuccess)
    return DIT_ECUDA;
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int quant_weight_launch(const uint16_t* w, int N, int K, const float* smooth, int8_t* q, float* scale,
                        cudaStream_t stream) {
  if (N <= 0 || K <= 0) return DIT_OK;
  quant_weight_kernel<<<N, kNormThreads, 0, stream>>>(w, K, smooth, q, scale);
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int codes_bf16_launch(const int8_t* q, uint16_t* w, long long n, cudaStream_t stream) {
  if (n <= 0) return DIT_OK;
  if (n % 16 != 0) return DIT_EUNSUPPORTED;
  codes_bf16_kernel<<<grid_for(n / 16, 256), 256, 0, stream>>>(q, w, n / 16);
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

// LoRA merge [gizai:dit, weightAt: a BF16 block's linear with its adapter's update B A added]:
// merged[o, i] = bf16_rne(W[o, i] + sum_r B[o, r] A[r, i]). One CTA per 64 x 64 output tile, 256
// threads with 4 x 4 outputs each; 32 ranks of B's rows and A's columns staged in shared memory (as
// fp32, zero past the edges) per step. Each product of two bf16 values is exact in fp32, so the sum
// over r is one fp32 FMA chain in rank order; W (exact in fp32) is added last, then one
// round-to-nearest-even to bf16. merged may be W itself (each element is read before it is written,
// by the thread that writes it).
constexpr int kMergeTile = 64, kMergeRanks = 32;
__global__ void __launch_bounds__(256) lora_merge_kernel(const uint16_t* W, const uint16_t* __restrict__ A,
                                                         const uint16_t* __restrict__ B, uint16_t* merged, int n_out,
                                                         int n_in, int rank) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sB[kMergeTile][kMergeRanks + 1];
  __shared__ float sA[kMergeRanks][kMergeTile];
  const int o0 = blockIdx.y * kMergeTile, i0 = blockIdx.x * kMergeTile;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int r0 = 0; r0 < rank; r0 += kMergeRanks) {
    for (int e = threadIdx.x; e < kMergeTile * kMergeRanks; e += 256) {
      const int rr = e % kMergeRanks, oo = e / kMergeRanks, o = o0 + oo, r = r0 + rr;
      sB[oo][rr] = (o < n_out && r < rank) ? __uint_as_float(uint32_t(B[size_t(o) * rank + r]) << 16) : 0.f;
    }
    for (int e = threadIdx.x; e < kMergeRanks * kMergeTile; e += 256) {
      const int ii = e % kMergeTile, rr = e / kMergeTile, i = i0 + ii, r = r0 + rr;
      sA[rr][ii] = (i < n_in && r < rank) ? __uint_as_float(uint32_t(A[size_t(r) * n_in + i]) << 16) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int rr = 0; rr < kMergeRanks; ++rr) {
      float b[4], a[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        b[k] = sB[ty + 16 * k][rr];
        a[k] = sA[rr][tx + 16 * k];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int l = 0; l < 4; ++l) acc[k][l] = __fmaf_rn(b[k], a[l], acc[k][l]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int o = o0 + ty + 16 * k;
    if (o >= n_out) continue;
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const int i = i0 + tx + 16 * l;
      if (i >= n_in) continue;
      const size_t at = size_t(o) * n_in + i;
      const float v = __fadd_rn(__uint_as_float(uint32_t(W[at]) << 16), acc[k][l]);
      __nv_bfloat16 h = __float2bfloat16_rn(v);
      merged[at] = *reinterpret_cast<uint16_t*>(&h);
    }
  }
}

int lora_merge_launch(const uint16_t* W, const uint16_t* A, const uint16_t* B, uint16_t* merged, int n_out, int n_in,
                      int rank, cudaStream_t stream) {
  if (n_out <= 0 || n_in <= 0) return DIT_OK;
  const dim3 grid((n_in + kMergeTile - 1) / kMergeTile, (n_out + kMergeTile - 1) / kMergeTile);
  if (grid.y > 65535u) return DIT_EUNSUPPORTED;
  lora_merge_kernel<<<grid, 256, 0, stream>>>(W, A, B, merged, n_out, n_in, rank);
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

int dequant_int8_launch(const int8_t* q, const uint16_t* s, uint16_t* w, long long rows, long long cols,
                        cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return DIT_OK;
  dequant_kernel<<<grid_for(rows * cols / 16, 256), 256, 0, stream>>>(q, s, w, rows, cols);
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ECUDA;
}

}  // namespace dit
