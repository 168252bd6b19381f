// NVFP4 weights: e2m1 element codes (two per byte, element 2i in the low
// nibble), one e4m3 scale per 16 consecutive inputs of a row, and one float32
// scale per tensor.  The pages name the format only ("Welcome FLUX.3 Image
// Klein in Diffusers", section "Single-file format checkpoints": nvfp4
// checkpoints with fast kernels on Blackwell); the element and scale encodings
// are the published FP4 E2M1 / FP8 E4M3 definitions.
//
//   quantize    bf16 [rows, cols] -> codes, scales, global
//               global g = amax / (6 * 448) rounded to float32 (1 if amax = 0);
//               s_b = e4m3_RNE(amax_b / (6 g)), saturating at 448;
//               q = e2m1_RNE(w / (s_b g)), saturating at +-6, no negative zero.
//               Every rounding decision is taken in float64 on exactly the
//               quotients the definition names, so codes are reproducible.
//   dequantize  the packed block weights -> bf16: e2m1 * e4m3 (exact in
//               float32) times g, rounded to float32, then to bf16 (both
//               nearest even).
//
// The dequantised bf16 matrices feed the same tcgen05 GEMMs as bf16
// checkpoints (the activations stay bf16, so the FP4 tensor-core kinds, which
// need both operands in a narrow format, do not apply).  Dequantisation is
// HBM-bound: 9 bytes read and 32 written per 16 weights.

#pragma once

#include <algorithm>

#include "flux3_internal.h"
#include "ptx.cuh"

namespace flux3 {

namespace fp4_detail {

constexpr int kGroup = 16;            // inputs per e4m3 block scale
constexpr double kE2m1Max = 6.0;
constexpr double kE4m3Max = 448.0;

// e4m3 code of v >= 0, round to nearest even, saturating at 448 (code 0x7E).
__device__ __forceinline__ uint32_t e4m3_encode(double v) {
  v = fmin(v, kE4m3Max);
  if (v < 0.015625) {                      // below 2^-6: subnormal grid, step 2^-9
    return (uint32_t)rint(v * 512.0);      // 8 = 2^-6, the first normal code
  }
  int e;
  frexp(v, &e);                            // v in [2^(e-1), 2^e)
  int E = e - 1;
  uint32_t q = (uint32_t)rint(ldexp(v, 3 - E));   // 8 .. 16 (3 mantissa bits)
  if (q == 16) {
    q = 8;
    ++E;
  }
  const uint32_t code = ((uint32_t)(E + 7) << 3) | (q - 8);
  return code > 0x7Eu ? 0x7Eu : code;
}

__device__ __forceinline__ double e4m3_decode(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, (int)e - 10);
}

// e2m1 code of r, round to nearest even, saturating at +-6.  Ties: 0.25 -> 0,
// 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4 (even codes).
__device__ __forceinline__ uint32_t e2m1_encode(double r) {
  const double a = fabs(r);
  const uint32_t c = (uint32_t)(a > 0.25) + (uint32_t)(a >= 0.75) + (uint32_t)(a > 1.25) + (uint32_t)(a >= 1.75) +
                     (uint32_t)(a > 2.5) + (uint32_t)(a >= 3.5) + (uint32_t)(a > 5.0);
  return (c != 0 && r < 0.0) ? (c | 8u) : c;
}

// Magnitude of an e2m1 code as float: exponent field e (bits 2..1, bias 1),
// mantissa m (bit 0); e = 0 is subnormal (0.5 m).
__device__ __forceinline__ float e2m1_decode(uint32_t c) {
  const uint32_t mag = c & 7u;
  const float v = mag >= 2u ? __uint_as_float((mag << 22) + 0x3F000000u) : 0.5f * (float)mag;
  return (c & 8u) ? -v : v;
}

__device__ __forceinline__ float e4m3_decode_f(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// ---------------------------------------------------------------- quantiser
__global__ void amax_kernel(const __nv_bfloat16 *__restrict__ w, size_t n, unsigned int *amax_bits) {
  float m = 0.f;
  const size_t n8 = n / 8;
  const uint4 *w8 = reinterpret_cast<const uint4 *>(w);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(w8 + i);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m = fmaxf(m, fabsf(__uint_as_float(u[k] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(u[k] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));   // m >= 0: bit order = value order
}

__device__ __forceinline__ float global_scale_of(float amax) {
  return amax > 0.f ? __double2float_rn((double)amax / (kE2m1Max * kE4m3Max)) : 1.0f;
}

// One thread per 16-input group: block scale and 16 element codes.
__global__ void quantize_kernel(const __nv_bfloat16 *__restrict__ w, int rows, int cols,
                                const unsigned int *__restrict__ amax_bits, uint8_t *__restrict__ codes,
                                uint8_t *__restrict__ scales) {
  const int gpr = cols / kGroup;
  const size_t n_groups = (size_t)rows * gpr;
  const float g = global_scale_of(__uint_as_float(*amax_bits));
  const double g64 = (double)g;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_groups; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 *src = reinterpret_cast<const uint4 *>(w + i * kGroup);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float x[16];
    float amax_b = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[2 * k] = __uint_as_float(u[k] << 16);
      x[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
      amax_b = fmaxf(amax_b, fmaxf(fabsf(x[2 * k]), fabsf(x[2 * k + 1])));
    }
    const uint32_t sc = e4m3_encode((double)amax_b / (kE2m1Max * g64));
    const double denom = e4m3_decode(sc) * g64;   // exact: 4 x 24 significant bits
    uint32_t packed[2] = {0u, 0u};
    if (denom > 0.0) {
#pragma unroll
      for (int k = 0; k < 16; ++k) packed[k / 8] |= e2m1_encode((double)x[k] / denom) << (4 * (k % 8));
    }
    *reinterpret_cast<uint2 *>(codes + i * (kGroup / 2)) = make_uint2(packed[0], packed[1]);
    scales[i] = (uint8_t)sc;
  }
}

__global__ void finalize_global_kernel(unsigned int *amax_bits_then_global) {
  const float g = global_scale_of(__uint_as_float(*amax_bits_then_global));
  *reinterpret_cast<float *>(amax_bits_then_global) = g;
}

// ---------------------------------------------------------------- dequantiser
// One packed block in NVFP4 (see Fp4BlockView).  The in-projection rows are
// q | k | v | mlp_in (a/b interleaved in groups of 128), each tensor with its
// own global scale (indices 0..3); the out-projection rows hold attn_out's
// 3072 inputs then mlp_out's 9216 (global scales 4 and 5).
struct Fp4BlockView {
  const uint8_t *in_codes;    // [kInRows, kHidden / 2]
  const uint8_t *in_scales;   // [kInRows, kHidden / 16]
  const uint8_t *out_codes;   // [kHidden, kCatCols / 2]
  const uint8_t *out_scales;  // [kHidden, kCatCols / 16]
  const float *globals;       // [8]: q, k, v, mlp_in, attn_out, mlp_out
};

constexpr uint32_t kInGroups = (uint32_t)kInRows * (kHidden / kGroup);     // 5,308,416
constexpr uint32_t kOutGroups = (uint32_t)kHidden * (kCatCols / kGroup);   // 2,359,296


// One thread per 16-weight group: the 8 code bytes are decoded through a
// 256-entry shared table (byte -> the two e2m1 values), scaled by the group's
// e4m3 scale (exact) and the tensor's global scale with packed float-pair
// multiplies, and packed to bf16 pairs.
__global__ void __launch_bounds__(256)
    dequantize_block_kernel(Fp4BlockView v, __nv_bfloat16 *__restrict__ w_in, __nv_bfloat16 *__restrict__ w_out) {
  __shared__ float2 pair_of_byte[256];
  __shared__ float gs[6];
  pair_of_byte[threadIdx.x] = make_float2(e2m1_decode(threadIdx.x & 0xFu), e2m1_decode(threadIdx.x >> 4));
  // the expanded weights overwrite what the previous block's GEMMs read
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x < 6) gs[threadIdx.x] = v.globals[threadIdx.x];
  __syncthreads();
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < kInGroups + kOutGroups; i += gridDim.x * blockDim.x) {
    const bool in = i < kInGroups;
    const uint32_t gi = in ? i : i - kInGroups;
    float g;
    if (in) {
      const uint32_t row = gi / (kHidden / kGroup);
      g = gs[row < 3u * kHidden ? row / kHidden : 3];
    } else {
      const uint32_t col = (gi % (kCatCols / kGroup)) * kGroup;
      g = gs[col < (uint32_t)kHidden ? 4 : 5];
    }
    const uint2 c =
        __ldcs(reinterpret_cast<const uint2 *>((in ? v.in_codes : v.out_codes) + (size_t)gi * (kGroup / 2)));
    const float s = e4m3_decode_f(__ldcs((in ? v.in_scales : v.out_scales) + gi));
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t byte = ((k < 4 ? c.x : c.y) >> (8 * (k % 4))) & 0xFFu;
      float2 e = pair_of_byte[byte];
      mul2(e.x, e.y, s);   // exact: 2 x 4 significant bits
      mul2(e.x, e.y, g);
      o[k] = pack_bf16x2(e.x, e.y);
    }
    uint4 *dst = reinterpret_cast<uint4 *>((in ? w_in : w_out) + (size_t)gi * kGroup);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace fp4_detail

cudaError_t launch_quantize_nvfp4(const __nv_bfloat16 *w, int rows, int cols, uint8_t *codes, uint8_t *scales,
                                  float *global, cudaStream_t s) {
  using namespace fp4_detail;
  unsigned int *amax = reinterpret_cast<unsigned int *>(global);
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  const size_t n = (size_t)rows * cols;
  const int grid = (int)std::min<size_t>((n / 8 + 255) / 256, (size_t)num_sms() * 8);
  amax_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(w, n, amax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t groups = n / kGroup;
  const int qgrid = (int)std::min<size_t>((groups + 255) / 256, (size_t)num_sms() * 16);
  quantize_kernel<<<qgrid > 0 ? qgrid : 1, 256, 0, s>>>(w, rows, cols, amax, codes, scales);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  finalize_global_kernel<<<1, 1, 0, s>>>(amax);
  return cudaGetLastError();
}

cudaError_t launch_dequantize_block(const fp4_detail::Fp4BlockView &v, __nv_bfloat16 *w_in, __nv_bfloat16 *w_out,
                                    cudaStream_t s, bool pdl = false) {
  using namespace fp4_detail;
  return launch_kernel(fp4_detail::dequantize_block_kernel, dim3(num_sms() * 8), dim3(256), 0, s, pdl, v, w_in,
                       w_out);
}

}  // namespace flux3
