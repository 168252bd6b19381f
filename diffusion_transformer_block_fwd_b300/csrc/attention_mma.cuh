// Bidirectional attention over all tokens (24 heads x 128, no mask), online
// softmax, warp-level mma.sync (m16n8k16 bf16 -> fp32).
//
// CTA = (128 query rows, one head); 8 warps x 16 rows.  K/V tiles of 64 keys
// are double-buffered through cp.async into XOR-swizzled shared memory and
// read with ldmatrix; P stays in registers between the two MMAs.  Keys past T
// (zero-filled rows of the last tile) are masked to -inf before the softmax.

#pragma once

#include "flux3_internal.h"
#include "ptx.cuh"

namespace flux3 {
namespace attn_detail {

constexpr int kQRows = 128;
constexpr int kKRows = 64;
constexpr int kWarps = 8;
constexpr int kRowBytes = kHeadDim * 2;                 // 256 B per row
constexpr int kQBytes = kQRows * kRowBytes;             // 32 KB
constexpr int kKVBytes = kKRows * kRowBytes;            // 16 KB
constexpr int kSmem = kQBytes + 4 * kKVBytes;           // Q + 2 x (K, V) = 96 KB

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Copies `rows` rows of one head (128 bf16 = 16 chunks of 16 B) from the
// token-major [T, ld] matrix into swizzled shared memory; rows >= T read as 0.
template <int ROWS>
__device__ __forceinline__ void load_rows(uint32_t sbase, const __nv_bfloat16 *g, int ld, int row0, int T) {
  for (int i = threadIdx.x; i < ROWS * 16; i += kWarps * 32) {
    const int r = i / 16, c = i % 16;
    const int t = row0 + r;
    const bool valid = t < T;
    const __nv_bfloat16 *src = g + (size_t)(valid ? t : 0) * ld + c * 8;
    cp_async16(sbase + swz(r, c), src, valid);
  }
}

__global__ void __launch_bounds__(kWarps * 32, 1)
    attention_kernel(const __nv_bfloat16 *__restrict__ qkv, int T, __nv_bfloat16 *__restrict__ out) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_addr(smem);
  const uint32_t sK[2] = {sQ + kQBytes, sQ + kQBytes + 2 * kKVBytes};
  const uint32_t sV[2] = {sQ + kQBytes + kKVBytes, sQ + kQBytes + 3 * kKVBytes};

  const int head = blockIdx.y;
  const int q0 = blockIdx.x * kQRows;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, tq = lane & 3;

  const __nv_bfloat16 *Qg = qkv + head * kHeadDim;
  const __nv_bfloat16 *Kg = qkv + kHidden + head * kHeadDim;
  const __nv_bfloat16 *Vg = qkv + 2 * kHidden + head * kHeadDim;

  load_rows<kQRows>(sQ, Qg, kQkvCols, q0, T);
  cp_async_commit();
  load_rows<kKRows>(sK[0], Kg, kQkvCols, 0, T);
  load_rows<kKRows>(sV[0], Vg, kQkvCols, 0, T);
  cp_async_commit();

  cp_async_wait<1>();
  __syncthreads();

  // Q fragments of this warp's 16 rows for the 8 k-steps over head_dim.
  uint32_t qf[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int c = kk * 2 + (lane >> 4);
    ldsm_x4(sQ + swz(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kHeadDim);

  const int ntiles = (T + kKRows - 1) / kKRows;
  for (int j = 0; j < ntiles; ++j) {
    const int buf = j & 1;
    if (j + 1 < ntiles) {
      load_rows<kKRows>(sK[buf ^ 1], Kg, kQkvCols, (j + 1) * kKRows, T);
      load_rows<kKRows>(sV[buf ^ 1], Vg, kQkvCols, (j + 1) * kKRows, T);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    // S = Q K^T for 64 keys: 8 n-blocks of 8 keys.
    float s[8][4];
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
      for (int kk2 = 0; kk2 < 4; ++kk2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK[buf] + swz(nb * 8 + (lane & 7), kk2 * 4 + (lane >> 3)), b0, b1, b2, b3);
        mma16816(s[nb], qf[2 * kk2], b0, b1);
        mma16816(s[nb], qf[2 * kk2 + 1], b2, b3);
      }
    }
    // scale into the log2 domain; mask keys past T
    const int kbase = j * kKRows;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kbase + nb * 8 + 2 * tq + (e & 1);
        s[nb][e] = key < T ? s[nb][e] * scale_log2 : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nb][0], s[nb][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nb][2], s[nb][3]));
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = ex2_approx(m0 - mn0), al1 = ex2_approx(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t p[8][2];
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      const float p0 = ex2_approx(s[nb][0] - mn0), p1 = ex2_approx(s[nb][1] - mn0);
      const float p2 = ex2_approx(s[nb][2] - mn1), p3 = ex2_approx(s[nb][3] - mn1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      p[nb][0] = pack_bf16x2(p0, p1);
      p[nb][1] = pack_bf16x2(p2, p3);
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int db = 0; db < 16; ++db) {
      o[db][0] *= al0;
      o[db][1] *= al0;
      o[db][2] *= al1;
      o[db][3] *= al1;
    }
    // O += P V: 4 k-steps of 16 keys, 16 n-blocks of 8 dims.
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint32_t a[4] = {p[2 * ks][0], p[2 * ks][1], p[2 * ks + 1][0], p[2 * ks + 1][1]};
#pragma unroll
      for (int db = 0; db < 16; db += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sV[buf] + swz(ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, db + (lane >> 4)), b0, b1, b2, b3);
        mma16816(o[db], a, b0, b1);
        mma16816(o[db + 1], a, b2, b3);
      }
    }
    __syncthreads();  // buffer `buf` is refilled two iterations on
  }

#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int r0 = q0 + warp * 16 + g, r1 = r0 + 8;
  __nv_bfloat16 *ob = out + head * kHeadDim + 2 * tq;
#pragma unroll
  for (int db = 0; db < 16; ++db) {
    if (r0 < T)
      *reinterpret_cast<uint32_t *>(ob + (size_t)r0 * kCatCols + db * 8) = pack_bf16x2(o[db][0] * inv0, o[db][1] * inv0);
    if (r1 < T)
      *reinterpret_cast<uint32_t *>(ob + (size_t)r1 * kCatCols + db * 8) = pack_bf16x2(o[db][2] * inv1, o[db][3] * inv1);
  }
}

}  // namespace attn_detail

cudaError_t launch_attention(const __nv_bfloat16 *qkv, int T, __nv_bfloat16 *cat, cudaStream_t s) {
  using namespace attn_detail;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((T + kQRows - 1) / kQRows, kHeads);
  attention_kernel<<<grid, kWarps * 32, kSmem, s>>>(qkv, T, cat);
  return cudaGetLastError();
}

}  // namespace flux3
