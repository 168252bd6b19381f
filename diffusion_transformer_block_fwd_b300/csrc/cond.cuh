// The conditioning around the block stacks and the sampler step
// ("FLUX.3 Image Klein support", comment "Structure (from dit.py)": timestep
// embedding into time_in / ref_time_in MLPEmbedders, per-stream modulation
// vectors, the image output layer; comment "Sampling": the Euler update).
//
//   timestep_embed_kernel  rows [cos(a), sin(a)], a_i = 1000 t 10000^(-i/128),
//                          in float64 (256 values per row)
//   rows_linear_kernel     y[m] (+)= W act(x[m]) for a few rows m (M <= 4):
//                          the MLPEmbedders, the modulation and adaLN linears.
//                          HBM-bound on W (bf16 [N, K], four independent
//                          16-byte loads in flight per lane, one warp per
//                          output, the activated rows in shared memory)
//   add_row_kernel         y[m] += r for the flow-map timestep term
//   euler_kernel           latent += (sigma_next - sigma) * velocity, and the
//                          new latent rounded to bf16 (the next call's input)
//   cfg_euler_kernel       the same with v = v_uncond + g (v_cond - v_uncond)
//   to_bf16_kernel         the first call's input from the initial latents

#pragma once

#include "flux3_internal.h"
#include "ptx.cuh"

namespace flux3 {

namespace cond_detail {

constexpr int kTimeDim = 256;
constexpr int kMaxRows = 4;
constexpr int kLoads = 4;     // 16-byte weight loads each lane has in flight

__global__ void timestep_embed_kernel(double t0, double t1, double t2, float *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 3 * kTimeDim) return;
  const int row = i / kTimeDim, j = i % kTimeDim, half = kTimeDim / 2;
  const double t = row == 0 ? t0 : row == 1 ? t1 : t2;
  const double f = exp(-log(10000.0) * (double)(j % half) / (double)half);
  const double a = 1000.0 * t * f;
  out[i] = (float)(j < half ? cos(a) : sin(a));
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }

// y[m * ldy + n] = (ACC ? y : 0) + sum_k W[n, k] * act(x[m * ldx + k]), m < M.
// K a multiple of 8; M * K floats fit the 48 KB of static-limit shared memory.
template <bool SILU_IN, bool ACC>
__global__ void __launch_bounds__(256) rows_linear_kernel(const __nv_bfloat16 *__restrict__ W, int N, int K,
                                                          const float *__restrict__ x, int ldx, int M,
                                                          float *__restrict__ y, int ldy) {
  extern __shared__ float xs[];   // [M][K], activated
  for (int i = threadIdx.x; i < M * K; i += blockDim.x) {
    const float v = x[(size_t)(i / K) * ldx + i % K];
    xs[i] = SILU_IN ? silu_f(v) : v;
  }
  __syncthreads();
  const int lane = threadIdx.x % 32;
  const int warps = gridDim.x * (blockDim.x / 32);
  for (int n = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; n < N; n += warps) {
    float acc[kMaxRows] = {0.f, 0.f, 0.f, 0.f};
    const uint4 *wr = reinterpret_cast<const uint4 *>(W + (size_t)n * K);
    for (int k0 = lane; k0 < K / 8; k0 += 32 * kLoads) {
      uint4 wv[kLoads];   // several independent 16-byte loads in flight per lane
#pragma unroll
      for (int l = 0; l < kLoads; ++l) {
        const int k8 = k0 + 32 * l;
        wv[l] = k8 < K / 8 ? __ldcs(wr + k8) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int l = 0; l < kLoads; ++l) {
        const int k8 = k0 + 32 * l;
        if (k8 >= K / 8) break;
        const uint32_t u[4] = {wv[l].x, wv[l].y, wv[l].z, wv[l].w};
        float w[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          w[2 * q] = __uint_as_float(u[q] << 16);
          w[2 * q + 1] = __uint_as_float(u[q] & 0xFFFF0000u);
        }
#pragma unroll
        for (int m = 0; m < kMaxRows; ++m) {
          if (m < M) {
            const float4 a = *reinterpret_cast<const float4 *>(xs + m * K + 8 * k8);
            const float4 b = *reinterpret_cast<const float4 *>(xs + m * K + 8 * k8 + 4);
            acc[m] = fmaf(w[0], a.x, fmaf(w[1], a.y, fmaf(w[2], a.z, fmaf(w[3], a.w,
                     fmaf(w[4], b.x, fmaf(w[5], b.y, fmaf(w[6], b.z, fmaf(w[7], b.w, acc[m]))))))));
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < kMaxRows; ++m) {
      float v = acc[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && m < M) {
        float *dst = y + (size_t)m * ldy + n;
        *dst = ACC ? *dst + v : v;
      }
    }
  }
}

__global__ void add_row_kernel(float *__restrict__ y, int ldy, int M, const float *__restrict__ r, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < M * n) y[(size_t)(i / n) * ldy + i % n] += r[i % n];
}

// The updates also write the new latent's bf16 rounding (the next call's
// image input) when `next_in` is given.
__global__ void euler_kernel(float *__restrict__ latent, const float *__restrict__ v, size_t n, float dt,
                             __nv_bfloat16 *__restrict__ next_in) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float y = fmaf(dt, v[i], latent[i]);
    latent[i] = y;
    if (next_in) next_in[i] = __float2bfloat16_rn(y);
  }
}

__global__ void cfg_euler_kernel(float *__restrict__ latent, const float *__restrict__ vu, const float *__restrict__ vc,
                                 size_t n, float g, float dt, __nv_bfloat16 *__restrict__ next_in) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float u = vu[i];
    const float y = fmaf(dt, fmaf(g, vc[i] - u, u), latent[i]);
    latent[i] = y;
    if (next_in) next_in[i] = __float2bfloat16_rn(y);
  }
}

__global__ void to_bf16_kernel(const float *__restrict__ src, size_t n, __nv_bfloat16 *__restrict__ dst) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

}  // namespace cond_detail

cudaError_t launch_timestep_embed(double t0, double t1, double t2, float *out, cudaStream_t s) {
  cond_detail::timestep_embed_kernel<<<3, 256, 0, s>>>(t0, t1, t2, out);
  return cudaGetLastError();
}

// y = W act(x) (+ y), M <= 4 rows, K % 8 == 0, M * K <= 12288.
cudaError_t launch_rows_linear(const __nv_bfloat16 *W, int N, int K, const float *x, int ldx, int M, float *y,
                               int ldy, bool silu_in, bool acc, cudaStream_t s) {
  using namespace cond_detail;
  if (M < 1 || M > kMaxRows || K % 8 != 0 || (size_t)M * K * 4 > 48 * 1024) return cudaErrorInvalidValue;
  const int grid = std::min((N + 7) / 8, num_sms() * 4);
  const size_t smem = (size_t)M * K * 4;
  if (silu_in && acc)
    rows_linear_kernel<true, true><<<grid, 256, smem, s>>>(W, N, K, x, ldx, M, y, ldy);
  else if (silu_in)
    rows_linear_kernel<true, false><<<grid, 256, smem, s>>>(W, N, K, x, ldx, M, y, ldy);
  else if (acc)
    rows_linear_kernel<false, true><<<grid, 256, smem, s>>>(W, N, K, x, ldx, M, y, ldy);
  else
    rows_linear_kernel<false, false><<<grid, 256, smem, s>>>(W, N, K, x, ldx, M, y, ldy);
  return cudaGetLastError();
}

cudaError_t launch_add_row(float *y, int ldy, int M, const float *r, int n, cudaStream_t s) {
  cond_detail::add_row_kernel<<<(M * n + 255) / 256, 256, 0, s>>>(y, ldy, M, r, n);
  return cudaGetLastError();
}

cudaError_t launch_euler(float *latent, const float *v, size_t n, float dt, __nv_bfloat16 *next_in, cudaStream_t s) {
  const int grid = (int)std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 8);
  cond_detail::euler_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(latent, v, n, dt, next_in);
  return cudaGetLastError();
}

cudaError_t launch_cfg_euler(float *latent, const float *vu, const float *vc, size_t n, float g, float dt,
                             __nv_bfloat16 *next_in, cudaStream_t s) {
  const int grid = (int)std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 8);
  cond_detail::cfg_euler_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(latent, vu, vc, n, g, dt, next_in);
  return cudaGetLastError();
}

cudaError_t launch_to_bf16(const float *src, size_t n, __nv_bfloat16 *dst, cudaStream_t s) {
  const int grid = (int)std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 8);
  cond_detail::to_bf16_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(src, n, dst);
  return cudaGetLastError();
}

}  // namespace flux3
