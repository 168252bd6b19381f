// Row-wise FP8 ("fp8r") weights: E4M3 element codes and one float32 scale per
// output row.  The pages name the variant only ("Welcome FLUX.3 Image Klein in
// Diffusers", section "Single-file format checkpoints": fp8r checkpoints with
// fast kernels on compute capability 8.9 and up); the element encoding is the
// published FP8 E4M3 definition and the recipe a reading:
//
//   quantize    bf16 [rows, cols] -> codes uint8 [rows, cols], scales float32 [rows]
//               s_r = amax_r / 448 rounded to float32 (1 for an all-zero row);
//               q = E4M3_RNE(w / s_r), saturating at +-448, no negative zero,
//               the decision taken in float64 on the quotient.
//   dequantize  e4m3(q) * s_r rounded to float32, then to bf16 (both nearest
//               even).
//
// As with NVFP4, the expanded bf16 matrices feed the bf16 tensor-core GEMMs:
// the activations stay bf16, and an FP8 tensor-core kind needs both operands in
// FP8.  Expansion is HBM-bound: 1 byte read and 2 written per weight.

#pragma once

#include "nvfp4.cuh"

namespace flux3 {

namespace fp8r_detail {

using fp4_detail::e4m3_decode_f;
using fp4_detail::e4m3_encode;

constexpr double kE4m3Max = 448.0;

// One warp per row: the row's amax, its scale, then 8 codes per lane step.
// cols is a multiple of 8 (16-byte loads of bf16, 8-byte stores of codes).
__global__ void quantize_fp8r_kernel(const __nv_bfloat16 *__restrict__ w, int rows, int cols,
                                     uint8_t *__restrict__ codes, float *__restrict__ scales) {
  const int lane = threadIdx.x % 32;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int n_warps = gridDim.x * blockDim.x / 32;
  for (int r = warp; r < rows; r += n_warps) {
    const uint4 *src = reinterpret_cast<const uint4 *>(w + (size_t)r * cols);
    float m = 0.f;
    for (int c = lane; c < cols / 8; c += 32) {
      const uint4 v = __ldg(src + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(u[k] << 16)), fabsf(__uint_as_float(u[k] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = m > 0.f ? __double2float_rn((double)m / kE4m3Max) : 1.0f;
    const double s64 = (double)s;
    uint2 *dst = reinterpret_cast<uint2 *>(codes + (size_t)r * cols);
    for (int c = lane; c < cols / 8; c += 32) {
      const uint4 v = __ldg(src + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      uint32_t packed[2] = {0u, 0u};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float x = __uint_as_float(k % 2 == 0 ? u[k / 2] << 16 : u[k / 2] & 0xFFFF0000u);
        uint32_t q = e4m3_encode(fabs((double)x) / s64);
        if (x < 0.f && q != 0u) q |= 0x80u;
        packed[k / 4] |= q << (8 * (k % 4));
      }
      dst[c] = make_uint2(packed[0], packed[1]);
    }
    if (lane == 0) scales[r] = s;
  }
}

// One packed block in fp8r.  The in-projection rows are q | k | v | mlp_in
// (a/b interleaved in groups of 128), one scale per row; the out-projection
// rows hold attn_out's 3072 inputs then mlp_out's 9216, with two scales per
// row (attn_out's, mlp_out's).
struct Fp8rBlockView {
  const uint8_t *in_codes;    // [kInRows, kHidden]
  const float *in_scales;     // [kInRows]
  const uint8_t *out_codes;   // [kHidden, kCatCols]
  const float *out_scales;    // [kHidden, 2]
};

constexpr uint32_t kChunk = 16;                                              // weights per thread step
constexpr uint32_t kInChunks = (uint32_t)kInRows * (kHidden / kChunk);      // 5,308,416
constexpr uint32_t kOutChunks = (uint32_t)kHidden * (kCatCols / kChunk);    // 2,359,296

// One thread per 16 weights: codes decoded through a 256-entry shared table
// (exact E4M3 values), scaled by the row's float32 scale (one rounding), packed
// to bf16 pairs.
__global__ void __launch_bounds__(256)
    dequantize_fp8r_block_kernel(Fp8rBlockView v, __nv_bfloat16 *__restrict__ w_in,
                                 __nv_bfloat16 *__restrict__ w_out) {
  __shared__ float value_of_code[256];
  {
    const uint32_t c = threadIdx.x;
    const float mag = e4m3_decode_f(c & 0x7Fu);
    value_of_code[c] = (c & 0x80u) ? -mag : mag;
  }
  // the expanded weights overwrite what the previous block's GEMMs read
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < kInChunks + kOutChunks; i += gridDim.x * blockDim.x) {
    const bool in = i < kInChunks;
    const uint32_t ci = in ? i : i - kInChunks;
    float s;
    if (in) {
      s = __ldg(v.in_scales + ci / (kHidden / kChunk));
    } else {
      const uint32_t row = ci / (kCatCols / kChunk), col = (ci % (kCatCols / kChunk)) * kChunk;
      s = __ldg(v.out_scales + 2 * row + (col < (uint32_t)kHidden ? 0 : 1));
    }
    const uint4 c = __ldcs(reinterpret_cast<const uint4 *>((in ? v.in_codes : v.out_codes) + (size_t)ci * kChunk));
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t word = words[k / 2];
      float a = value_of_code[(word >> (16 * (k % 2))) & 0xFFu];
      float b = value_of_code[(word >> (16 * (k % 2) + 8)) & 0xFFu];
      mul2(a, b, s);
      o[k] = pack_bf16x2(a, b);
    }
    uint4 *dst = reinterpret_cast<uint4 *>((in ? w_in : w_out) + (size_t)ci * kChunk);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace fp8r_detail

cudaError_t launch_quantize_fp8r(const __nv_bfloat16 *w, int rows, int cols, uint8_t *codes, float *scales,
                                 cudaStream_t s) {
  using namespace fp8r_detail;
  const int warps_per_cta = 8;
  const int grid = std::min((rows + warps_per_cta - 1) / warps_per_cta, num_sms() * 16);
  quantize_fp8r_kernel<<<grid > 0 ? grid : 1, warps_per_cta * 32, 0, s>>>(w, rows, cols, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_dequantize_fp8r_block(const fp8r_detail::Fp8rBlockView &v, __nv_bfloat16 *w_in,
                                         __nv_bfloat16 *w_out, cudaStream_t s, bool pdl = false) {
  return launch_kernel(fp8r_detail::dequantize_fp8r_block_kernel, dim3(num_sms() * 8), dim3(256), 0, s, pdl, v,
                       w_in, w_out);
}

}  // namespace flux3
