// Bidirectional attention over all tokens of one sample (24 heads x 128, no
// mask), tcgen05 / TMEM flash attention.
//
// CTA = (128 query rows, one head), 192 threads:
//   warp 0      TMA producer: the Q tile once, then K and V tiles of 128 keys
//               into a 2-stage ring (128-byte swizzle, two 64-dim boxes each)
//   warp 1      owns the TMEM allocation (512 columns) and issues the MMAs
//               from one thread: S_j = Q K_j^T into one of two S buffers
//               (columns 0..127 / 128..255), then O += P_{j-1} V_{j-1}
//               (columns 256..383) with P read from tensor memory
//   warps 2..5  softmax, one query row per thread (TMEM lane = row): read the
//               S row, online max / exp2 / sum in fp32, write P as packed bf16
//               over the first 64 columns of the same S buffer; rescale the O
//               row in TMEM when the running max grows by more than 2^8
//               (otherwise the stale max is kept: P <= 2^8 is exact enough
//               for bf16 and the fp32 accumulator); finally O / l -> bf16.
// Keys past T (zero rows of the last tile) are masked to -inf.  Every wait is
// bounded; on a timeout the CTA drains, frees TMEM and returns.

#pragma once

#include "flux3_internal.h"
#include "ptx.cuh"

namespace flux3 {
namespace attn_tc {

constexpr int kRows = 128;                       // query rows per CTA and keys per tile
constexpr int kThreads = 192;
constexpr uint32_t kHalfBytes = kRows * 128;     // 128 rows x 64 bf16 (one 128-byte swizzle box)
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // 128 rows x 128 dims = 32 KB
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;

struct Ctl {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmem = 1024 + kTileBytes /*Q*/ + kStages * 2 * kTileBytes /*K, V*/ + sizeof(Ctl);

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      record_error(DEVERR_TIMEOUT);
      return;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_qkv, int T, __nv_bfloat16 *__restrict__ out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = smem + kTileBytes;                          // [stage][2 halves]
  uint8_t *sV = sK + kStages * kTileBytes;                  // [stage][2 halves]
  Ctl *ctl = reinterpret_cast<Ctl *>(sV + kStages * kTileBytes);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int head = blockIdx.y;
  const int q0 = blockIdx.x * kRows;
  const int nt = (T + kRows - 1) / kRows;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->kv_full[s], 1);
      mbar_init(&ctl->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->s_full[b], 1);
      mbar_init(&ctl->p_full[b], 128);
    }
    mbar_init(&ctl->o_done, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tm_qkv);
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int *abort = &ctl->abort;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const int xq = head * kHeadDim, xk = kHidden + head * kHeadDim, xv = 2 * kHidden + head * kHeadDim;
      mbar_arrive_expect_tx(&ctl->q_full, kTileBytes);
      tma_load_2d(sQ, &tm_qkv, &ctl->q_full, xq, q0);
      tma_load_2d(sQ + kHalfBytes, &tm_qkv, &ctl->q_full, xq + 64, q0);
      int last_phase[kStages] = {-1, -1};
      bool ok = true;
      for (int j = 0; j < nt; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!mbar_wait(&ctl->kv_empty[s], ph ^ 1, abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&ctl->kv_full[s], 2 * kTileBytes);
        uint8_t *k = sK + s * kTileBytes, *v = sV + s * kTileBytes;
        tma_load_2d(k, &tm_qkv, &ctl->kv_full[s], xk, j * kRows);
        tma_load_2d(k + kHalfBytes, &tm_qkv, &ctl->kv_full[s], xk + 64, j * kRows);
        tma_load_2d(v, &tm_qkv, &ctl->kv_full[s], xv, j * kRows);
        tma_load_2d(v + kHalfBytes, &tm_qkv, &ctl->kv_full[s], xv + 64, j * kRows);
        last_phase[s] = (int)ph;
      }
      drain_wait(&ctl->q_full, 0);
      if (!ok)
        for (int s = 0; s < kStages; ++s)
          if (last_phase[s] >= 0) drain_wait(&ctl->kv_full[s], (uint32_t)last_phase[s]);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc_s = idesc_bf16(kRows, kRows, false);   // B = K tile, K-major
      constexpr uint32_t idesc_o = idesc_bf16(kRows, kHeadDim, true); // B = V tile, MN-major
      const uint32_t q_addr = smem_addr(sQ);
      bool ok = mbar_wait(&ctl->q_full, 0, abort);
      for (int j = 0; ok && j <= nt; ++j) {
        if (j < nt) {
          const int s = j % kStages;
          if (!mbar_wait(&ctl->kv_full[s], (j / kStages) & 1, abort)) break;
          tc_fence_after();
          const uint32_t k_addr = smem_addr(sK + s * kTileBytes);
          const uint32_t d = tmem + (uint32_t)(j & 1) * kRows;
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t off = (uint32_t)(k / 4) * kHalfBytes + (uint32_t)(k % 4) * 32;
            mma_bf16_ss(d, smem_desc(q_addr + off, 16, 1024, kSwizzle128B),
                        smem_desc(k_addr + off, 16, 1024, kSwizzle128B), idesc_s, k > 0);
          }
          mma_commit(&ctl->s_full[j & 1]);
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int s = jj % kStages;
          if (!mbar_wait(&ctl->p_full[jj & 1], (jj >> 1) & 1, abort)) break;
          tc_fence_after();
          const uint32_t v_addr = smem_addr(sV + s * kTileBytes);
          const uint32_t p = tmem + (uint32_t)(jj & 1) * kRows;
          // 16 keys per MMA: P columns 8k .. 8k+7 (packed bf16 pairs), V rows 16k .. 16k+15;
          // V is MN-major: 64-dim halves 16 KB apart (leading offset), 8-row groups 1 KB apart.
#pragma unroll
          for (int k = 0; k < kRows / 16; ++k)
            mma_bf16_ts(tmem + kColO, p + k * 8, smem_desc(v_addr + k * 2048, kHalfBytes, 1024, kSwizzle128B),
                        idesc_o, (jj | k) != 0);
          mma_commit(&ctl->kv_empty[s]);
          mma_commit(&ctl->o_done);
        }
      }
      mma_commit(&ctl->drain);
      drain_wait(&ctl->drain, 0);
    }
  } else {
    // ---------------- softmax / correction / epilogue, one row per thread
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float scale_log2 = 1.4426950408889634f * rsqrtf((float)kHeadDim);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&ctl->s_full[sb], (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + sb * kRows + c * 32, sv[c]);
      const int valid = T - j * kRows;   // keys of this tile that exist
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float v = __uint_as_float(sv[c][i]) * scale_log2;
          if (c * 32 + i >= valid) v = -INFINITY;
          sv[c][i] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      const float m_new = fmaxf(m, mx);
      const bool need = (j > 0) && (m_new > m + 8.0f);
      bool waited = false;
      if (j == 0) {
        m = m_new;
      } else if (__any_sync(0xffffffffu, need)) {
        // O must hold every PV up to j-1 before it is rescaled
        if (!mbar_wait(&ctl->o_done, (j - 1) & 1, abort)) {
          ok = false;
          break;
        }
        waited = true;
        tc_fence_after();
        const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
        if (need) m = m_new;
        l *= alpha;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + kColO + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_off + kColO + c * 32, o);
        }
      }
      float sum = 0.f;
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(__uint_as_float(sv[c][2 * i]) - m);
          const float p1 = ex2_approx(__uint_as_float(sv[c][2 * i + 1]) - m);
          sum += p0 + p1;
          pk[c >> 1][(c & 1) * 16 + i] = pack_bf16x2(p0, p1);
        }
      l += sum;
      // keep o_done's phases in step: every PV completion is observed in order
      if (j > 0 && !waited) {
        if (!mbar_wait(&ctl->o_done, (j - 1) & 1, abort)) {
          ok = false;
          break;
        }
      }
      tmem_st32(tmem + lane_off + sb * kRows, pk[0]);
      tmem_st32(tmem + lane_off + sb * kRows + 32, pk[1]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctl->p_full[sb]);
    }
    if (ok && mbar_wait(&ctl->o_done, (nt - 1) & 1, abort)) {
      tc_fence_after();
      const float inv = 1.0f / l;
      const int t = q0 + row;
      uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)(t < T ? t : 0) * kCatCols + head * kHeadDim);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + kColO + c * 32, o);
        if (t < T) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[c * 4 + q] = make_uint4(
                pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace attn_tc

cudaError_t launch_attention(const __nv_bfloat16 *qkv, int T, __nv_bfloat16 *cat, cudaStream_t s) {
  using namespace attn_tc;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap tm;
  if (!make_tmap_bf16(&tm, qkv, (uint64_t)T, kQkvCols, kRows)) return cudaErrorInvalidValue;
  dim3 grid((T + kRows - 1) / kRows, kHeads);
  attention_kernel<<<grid, kThreads, kSmem, s>>>(tm, T, cat);
  return cudaGetLastError();
}

}  // namespace flux3
