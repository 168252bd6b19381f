// Per-call preparation and the memory-bound LayerNorm + modulation kernel.
//
//   stream_ids   segment table -> uint8 stream id per token
//   rope_tables  pos ids [T, 4] -> cos / sin [T, 64] (pair p = 16 a + j of axis a)
//   prepare      both in one launch (the forward calls)
//   ln_modulate  x fp32 [T, 3072] -> h = (1 + scale[s]) * LN(x) + shift[s], bf16
//
// ln_modulate is HBM-bound: 12 KB read + 6 KB written per token.  One warp per
// token row, 16-byte loads, the row held in registers (96 floats per lane),
// two-pass mean / variance with warp-shuffle reductions.

#pragma once

#include "flux3_internal.h"
#include "ptx.cuh"

namespace flux3 {

namespace ew_detail {

struct SegTable {
  int start[FLUX3_MAX_SEGMENTS];
  int len[FLUX3_MAX_SEGMENTS];
  int stream[FLUX3_MAX_SEGMENTS];
  int n;
};


// Angles are carried in turns (angle / 2 pi) as an unevaluated float pair
// hi + lo: hi = pos * fh (rounded), lo = its exact rounding error (fma) plus
// pos * fl, where fh + fl is theta^(-2j/32) / (2 pi) split on the host from a
// double.  The pair holds the angle to ~2^-47 relative, so dropping the whole
// turns (hi - rint(hi) is exact) leaves the fraction of a turn accurate to
// ~3e-8 turns for |pos| < 2^20; sincospif of twice the fraction gives the
// table entries.  No float64 arithmetic runs on the device.
struct RopeFreqs {
  float hi[16], lo[16];
};

__device__ __forceinline__ void rope_entry(const float *pos, const RopeFreqs &fr, int i, float *cos_tab,
                                           float *sin_tab) {
  const int t = i / kRopePairs, p = i % kRopePairs;
  const int axis = p / 16, j = p % 16;
  const float x = __ldg(pos + (size_t)t * 4 + axis);
  const float th = x * fr.hi[j];
  const float tl = fmaf(x, fr.hi[j], -th) + x * fr.lo[j];
  const float frac = (th - rintf(th)) + tl;
  float sn, cs;
  sincospif(2.0f * frac, &sn, &cs);
  cos_tab[i] = cs;
  sin_tab[i] = sn;
}

__global__ void rope_tables_kernel(const float *pos, int T, RopeFreqs fr, float *cos_tab, float *sin_tab) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * kRopePairs) return;
  rope_entry(pos, fr, i, cos_tab, sin_tab);
}

__device__ __forceinline__ int stream_of(const SegTable &tab, int t) {
  int s = -1;
  for (int i = 0; i < tab.n; ++i)
    if (t >= tab.start[i] && t < tab.start[i] + tab.len[i]) s = tab.stream[i];
  if (s < 0) {  // the host validated coverage; keep the kernel honest anyway
    record_error(DEVERR_BOUNDS);
    s = 0;
  }
  return s;
}

__global__ void stream_ids_kernel(SegTable tab, int T, uint8_t *sid) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  sid[t] = (uint8_t)stream_of(tab, t);
}

// The per-call preparation in one launch: thread i writes RoPE pair i % 64 of
// token i / 64, and the token's first thread its stream id.
__global__ void prepare_kernel(SegTable tab, const float *pos, int T, RopeFreqs fr, uint8_t *sid, float *cos_tab,
                               float *sin_tab) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * kRopePairs) return;
  rope_entry(pos, fr, i, cos_tab, sin_tab);
  if (i % kRopePairs == 0) sid[i / kRopePairs] = (uint8_t)stream_of(tab, i / kRopePairs);
}

constexpr int kLnWarps = 8;

__global__ void __launch_bounds__(kLnWarps * 32, 2)
    ln_modulate_kernel(const float *__restrict__ x, int T, const uint8_t *__restrict__ sid,
                       const float *__restrict__ mod, float eps, __nv_bfloat16 *__restrict__ h, int early_release) {
  constexpr int kVec = kHidden / (32 * 4);  // 24 float4 per lane
  // early_release: the dependent (the in-projection) may start before this
  // kernel's own wait -- when nothing it reads before its wait (constant
  // weights) is written by a kernel still running
  if (early_release) griddep_launch_dependents();
  griddep_wait();
  if (!early_release) griddep_launch_dependents();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * kLnWarps + warp;
  if (t >= T) return;
  const int s = sid[t];   // issued with the row's loads: one round trip fewer before the modulation rows
  const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)t * kHidden);
  float4 v[kVec];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    v[i] = __ldcs(xr + i * 32 + lane);
    sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  }
  const float4 *shift = reinterpret_cast<const float4 *>(mod + (size_t)s * kModLen);
  const float4 *scale = reinterpret_cast<const float4 *>(mod + (size_t)s * kModLen + kHidden);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float mean = sum * (1.0f / kHidden);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, d = v[i].w - mean;
    sq += (a * a + b * b) + (c * c + d * d);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const float rstd = rsqrtf(sq * (1.0f / kHidden) + eps);
  uint2 *hr = reinterpret_cast<uint2 *>(h + (size_t)t * kHidden);
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const float4 sh = __ldg(shift + i * 32 + lane);
    const float4 sc = __ldg(scale + i * 32 + lane);
    const float a = fmaf((v[i].x - mean) * rstd, 1.0f + sc.x, sh.x);
    const float b = fmaf((v[i].y - mean) * rstd, 1.0f + sc.y, sh.y);
    const float c = fmaf((v[i].z - mean) * rstd, 1.0f + sc.z, sh.z);
    const float d = fmaf((v[i].w - mean) * rstd, 1.0f + sc.w, sh.w);
    hr[i * 32 + lane] = make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
  }
}

// Diagnostics: one CTA waits on an mbarrier that nothing arrives at; the
// bounded wait must give up after timeout_ns and record DEVERR_TIMEOUT.
__global__ void selftest_wait_kernel(unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort, timeout_ns);
  __syncthreads();
}

}  // namespace ew_detail

namespace ew_detail {

SegTable seg_table(const flux3_segment *segs, int n_segs) {
  SegTable tab{};
  tab.n = n_segs;
  for (int i = 0; i < n_segs; ++i) {
    tab.start[i] = segs[i].start;
    tab.len[i] = segs[i].len;
    tab.stream[i] = segs[i].stream;
  }
  return tab;
}

RopeFreqs rope_freqs(float theta) {
  RopeFreqs fr;
  const double inv_two_pi = 0.15915494309189535;
  for (int j = 0; j < 16; ++j) {
    const double turns = pow((double)theta, -2.0 * j / 32.0) * inv_two_pi;
    fr.hi[j] = (float)turns;
    fr.lo[j] = (float)(turns - (double)fr.hi[j]);
  }
  return fr;
}

}  // namespace ew_detail

cudaError_t launch_stream_ids(const flux3_segment *segs, int n_segs, int T, uint8_t *sid, cudaStream_t s) {
  using namespace ew_detail;
  stream_ids_kernel<<<(T + 255) / 256, 256, 0, s>>>(seg_table(segs, n_segs), T, sid);
  return cudaGetLastError();
}

cudaError_t launch_rope_tables(const float *pos, int T, float theta, float *cos_tab, float *sin_tab,
                               cudaStream_t s) {
  using namespace ew_detail;
  const int n = T * kRopePairs;
  rope_tables_kernel<<<(n + 255) / 256, 256, 0, s>>>(pos, T, rope_freqs(theta), cos_tab, sin_tab);
  return cudaGetLastError();
}

cudaError_t launch_prepare(const flux3_segment *segs, int n_segs, int T, uint8_t *sid, const float *pos, float theta,
                           float *cos_tab, float *sin_tab, cudaStream_t s) {
  using namespace ew_detail;
  const int n = T * kRopePairs;
  prepare_kernel<<<(n + 255) / 256, 256, 0, s>>>(seg_table(segs, n_segs), pos, T, rope_freqs(theta), sid, cos_tab,
                                                 sin_tab);
  return cudaGetLastError();
}

cudaError_t launch_ln_modulate(const float *x, int T, const uint8_t *sid, const float *mod, float eps,
                               __nv_bfloat16 *h, cudaStream_t s, bool pdl, bool early_release) {
  using namespace ew_detail;
  return launch_kernel(ln_modulate_kernel, dim3((T + kLnWarps - 1) / kLnWarps), dim3(kLnWarps * 32), 0, s, pdl, x,
                       T, sid, mod, eps, h, early_release ? 1 : 0);
}

cudaError_t launch_selftest_wait(unsigned long long timeout_ns, cudaStream_t s) {
  using namespace ew_detail;
  selftest_wait_kernel<<<1, 32, 0, s>>>(timeout_ns);
  return cudaGetLastError();
}

}  // namespace flux3
