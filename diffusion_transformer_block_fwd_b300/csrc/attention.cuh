// Bidirectional attention over all tokens of one sample (24 heads x 128, no
// mask), tcgen05 / TMEM flash attention with two query tiles per CTA.
//
// CTA = (256 query rows as two 128-row tiles A and B, one head), 384 threads
// in three warpgroups:
//   warps 0..3  softmax of tile A, one query row per thread (TMEM lane = row)
//   warps 4..7  softmax of tile B
//   warp 8      TMA producer: Q_A, Q_B once; K and V tiles of 128 keys in two
//               independent 2-stage rings (128-byte swizzle, two 64-dim boxes
//               per tile); K runs one tile ahead of V
//   warp 9      owns the TMEM allocation and issues every MMA from one thread
//   warps 10-11 complete the third warpgroup
// The softmax warpgroups take 216 registers per thread and the third
// warpgroup 72 (setmaxnreg), so a thread holds its row's 128 scores.
// TMEM (512 columns): S_A 0..127, S_B 128..255, O_A 256..383, O_B 384..511.
// P overwrites the first 64 columns of its S buffer as packed bf16 and is the
// A operand of O += P V.  MMA order per key tile j:
//   S_A(j), PV_B(j-1), S_B(j), PV_A(j)
// so while softmax A works on S_A(j) the tensor core runs PV_B(j-1) and
// S_B(j), and while softmax B works on S_B(j) it runs PV_A(j) and S_A(j+1).
// Softmax per key tile: the row's 128 scores in one TMEM round trip (two
// 64-column loads, one wait), the row max (3-input max, 4 chains), then
// p = exp2(s * log2(e)/sqrt(128) - m) with packed float-pair FMAs and adds and
// the MUFU exp2 (32 per clock per SM on this part), P rounded to bf16 and
// stored over S.  Online max in the log2 domain with lazy rescale (O is
// rescaled in TMEM only when a row's max grows by more than 2^8); row sums in
// fp32.  Keys past T are masked to -inf (last key tile only).
// Every wait is bounded; on a timeout the CTA drains, frees TMEM and returns.

#pragma once

#include "flux3_internal.h"
#include "ptx.cuh"

namespace flux3 {
namespace attn_tc {

constexpr int kRows = 128;                       // rows per query tile and keys per key tile
constexpr int kThreads = 384;                     // three warpgroups
constexpr int kWarpTma = 8, kWarpMma = 9;         // warps 10, 11 only complete the third warpgroup
// Register split (setmaxnreg): the launch gives every thread kLaunchRegs; the
// two softmax warpgroups take kSoftmaxRegs (a whole 128-column S row in
// registers), the producer / MMA warpgroup keeps kOtherRegs.  The shares add
// up to exactly the launch's allocation: 128 * (2 * 216 + 72) = 384 * 168.
constexpr int kLaunchRegs = 168, kSoftmaxRegs = 216, kOtherRegs = 72;
static_assert(128 * (2 * kSoftmaxRegs + kOtherRegs) == kThreads * kLaunchRegs, "register split");
constexpr uint32_t kHalfBytes = kRows * 128;     // 128 rows x 64 bf16 (one 128-byte swizzle box)
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // 128 rows x 128 dims = 32 KB
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int x) { return 128u * (uint32_t)x; }         // S_x / P_x
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u + 128u * (uint32_t)x; }  // O_x

struct Ctl {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmem = 1024 + 2 * kTileBytes /*Q_A, Q_B*/ + 2 * kStages * kTileBytes /*K, V*/ + sizeof(Ctl);

// Work items: item b < n_full is unit b (all keys); each later unit is split
// into `splits` key ranges, item n_full + v covering unit n_full + v / splits
// and its key tiles [ks * nt / splits, (ks + 1) * nt / splits), ks = v % splits.
// Units run head-major: unit u is query-tile pair u % n_qp of head u / n_qp.
// A split item writes its rows unnormalised to part[v] (kPartRowFloats floats
// per query row: 128 output values, the row max in the log2 domain, the row sum).
constexpr int kPartRowFloats = 132;
constexpr int kMaxSplits = 8;   // most key ranges a unit is split into
constexpr size_t kPartItemBytes = (size_t)2 * kRows * kPartRowFloats * 4;
struct Plan {
  int n_full, splits, n_qp;
  float *part;
};

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      record_error(DEVERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a, b) = (x0, x1) * s + (t, t) as one packed float-pair FMA.
__device__ __forceinline__ void fma2(float x0, float x1, float s, float t, float &a, float &b) {
  asm("{\n .reg .b64 x, m, c, d;\n mov.b64 x, {%2, %3};\n mov.b64 m, {%4, %4};\n mov.b64 c, {%5, %5};\n"
      " fma.rn.f32x2 d, x, m, c;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(a), "=f"(b)
      : "f"(x0), "f"(x1), "f"(s), "f"(t));
}

// (s0, s1) += (p0, p1) as one packed float-pair add.
__device__ __forceinline__ void add2(float &s0, float &s1, float p0, float p1) {
  asm("{\n .reg .b64 x, y, d;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n add.f32x2 d, x, y;\n"
      " mov.b64 {%0, %1}, d;\n}"
      : "+f"(s0), "+f"(s1)
      : "f"(p0), "f"(p1));
}

// The unit, key range and partial slot (-1: none) of work item b.
struct Item {
  int head, q0, j0, nt, slot;
};
__device__ __forceinline__ Item item_of(int b, int T, const Plan &plan) {
  const int nt_all = (T + kRows - 1) / kRows;
  Item it;
  int unit;
  if (b < plan.n_full) {
    unit = b;
    it.j0 = 0;
    it.nt = nt_all;
    it.slot = -1;
  } else {
    const int v = b - plan.n_full, ks = v % plan.splits;
    unit = plan.n_full + v / plan.splits;
    it.j0 = ks * nt_all / plan.splits;
    it.nt = (ks + 1) * nt_all / plan.splits - it.j0;
    it.slot = v;
  }
  it.head = unit / plan.n_qp;
  it.q0 = (unit % plan.n_qp) * 2 * kRows;
  return it;
}

// kSplit = false: grid (query-tile pairs, heads), every CTA a whole unit;
// kSplit = true: one CTA per work item of `plan` (whole units, then key ranges).
template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_qkv, int T, __nv_bfloat16 *__restrict__ out, Plan plan) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem;                                       // [tile A, B][2 halves]
  uint8_t *sK = smem + 2 * kTileBytes;                      // [stage][2 halves]
  uint8_t *sV = sK + kStages * kTileBytes;                  // [stage][2 halves]
  Ctl *ctl = reinterpret_cast<Ctl *>(sV + kStages * kTileBytes);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  Item item;
  if constexpr (kSplit) {
    item = item_of(blockIdx.x, T, plan);
  } else {
    item = Item{(int)blockIdx.y, (int)blockIdx.x * 2 * kRows, 0, (T + kRows - 1) / kRows, -1};
  }
  const int j0 = item.j0, nt = item.nt;   // this CTA's key tiles [j0, j0 + nt)

  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ctl->s_full[x], 1);
      mbar_init(&ctl->p_full[x], 128);
      mbar_init(&ctl->o_done[x], 1);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0) tma_prefetch_desc(&tm_qkv);
  if (warp == kWarpMma) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int *abort = &ctl->abort;
  // set-up above overlaps the previous kernel when launched as its programmatic
  // dependent.  The out-projection after attention is released before the
  // wait: before its own wait it only sets up and loads weights, which no
  // kernel of the block writes after the in-projection has started (and this
  // kernel starts only after that), so its CTAs can take SMs as the
  // in-projection's CTAs leave.
  griddep_launch_dependents();
  griddep_wait();

  if (warp >= kWarpTma) {
    // third warpgroup: one register share for all four of its warps (the
    // reallocation is a warpgroup-wide instruction), then the TMA and MMA roles
    regs_decrease<kOtherRegs>();
  }
  if (warp == kWarpTma) {
    if (lane == 0) {
      // ---------------- TMA producer: K_0, then per tile j: K_{j+1}, V_j
      const int head = item.head, q0 = item.q0;
      const int xq = head * kHeadDim, xk = kHidden + head * kHeadDim, xv = 2 * kHidden + head * kHeadDim;
      mbar_arrive_expect_tx(&ctl->q_full, 2 * kTileBytes);
      for (int x = 0; x < 2; ++x) {
        tma_load_2d(sQ + x * kTileBytes, &tm_qkv, &ctl->q_full, xq, q0 + x * kRows);
        tma_load_2d(sQ + x * kTileBytes + kHalfBytes, &tm_qkv, &ctl->q_full, xq + 64, q0 + x * kRows);
      }
      int k_last[kStages] = {-1, -1}, v_last[kStages] = {-1, -1};
      bool ok = true;
      auto load = [&](bool is_k, int j) -> bool {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        uint64_t *empty = is_k ? &ctl->k_empty[s] : &ctl->v_empty[s];
        uint64_t *full = is_k ? &ctl->k_full[s] : &ctl->v_full[s];
        if (!mbar_wait(empty, ph ^ 1, abort)) return false;
        mbar_arrive_expect_tx(full, kTileBytes);
        uint8_t *dst = (is_k ? sK : sV) + s * kTileBytes;
        const int x = is_k ? xk : xv;
        tma_load_2d(dst, &tm_qkv, full, x, (j0 + j) * kRows);
        tma_load_2d(dst + kHalfBytes, &tm_qkv, full, x + 64, (j0 + j) * kRows);
        (is_k ? k_last : v_last)[s] = (int)ph;
        return true;
      };
      ok = load(true, 0);
      for (int j = 0; ok && j < nt; ++j) {
        if (j + 1 < nt && !(ok = load(true, j + 1))) break;
        ok = load(false, j);
      }
      drain_wait(&ctl->q_full, 0);
      if (!ok)
        for (int s = 0; s < kStages; ++s) {
          if (k_last[s] >= 0) drain_wait(&ctl->k_full[s], (uint32_t)k_last[s]);
          if (v_last[s] >= 0) drain_wait(&ctl->v_full[s], (uint32_t)v_last[s]);
        }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc_s = idesc_bf16(kRows, kRows, false);   // B = K tile, K-major
      constexpr uint32_t idesc_o = idesc_bf16(kRows, kHeadDim, true); // B = V tile, MN-major
      // descriptors encoded once, moved by constant offsets per MMA (a few
      // instructions per MMA keep the issue ahead of the tensor core while the
      // softmax warps load the same sub-partitions)
      const SmemDesc dq = smem_desc_split(smem_addr(sQ), 16, 1024, kSwizzle128B);
      const SmemDesc dk = smem_desc_split(smem_addr(sK), 16, 1024, kSwizzle128B);
      const SmemDesc dv = smem_desc_split(smem_addr(sV), kHalfBytes, 1024, kSwizzle128B);
      auto issue_s = [&](int x, int s) {
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k) {
          const uint32_t off = (uint32_t)(k / 4) * kHalfBytes + (uint32_t)(k % 4) * 32;
          mma_bf16_ss_at(tmem + col_s(x), dq, x * kTileBytes + off, dk, s * kTileBytes + off, idesc_s, k > 0);
        }
        mma_commit(&ctl->s_full[x]);
      };
      // O_x += P_x V: 16 keys per MMA (P columns 8k.., V rows 16k..); V is
      // MN-major: 64-dim halves 16 KB apart, 8-row groups 1 KB apart.
      auto issue_pv = [&](int x, int s, bool first) {
#pragma unroll
        for (int k = 0; k < kRows / 16; ++k)
          mma_bf16_ts_at(tmem + col_o(x), tmem + col_s(x) + k * 8, dv, s * kTileBytes + k * 2048, idesc_o,
                         !(first && k == 0));
        mma_commit(&ctl->o_done[x]);
      };
      bool ok = mbar_wait(&ctl->q_full, 0, abort);
      for (int j = 0; ok && j < nt; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!(ok = mbar_wait(&ctl->k_full[s], ph, abort))) break;
        tc_fence_after();
        issue_s(0, s);
        if (j >= 1) {
          if (!(ok = mbar_wait(&ctl->p_full[1], (j - 1) & 1, abort))) break;
          tc_fence_after();
          issue_pv(1, (j - 1) % kStages, j - 1 == 0);
          mma_commit(&ctl->v_empty[(j - 1) % kStages]);
        }
        issue_s(1, s);
        mma_commit(&ctl->k_empty[s]);
        if (!(ok = mbar_wait(&ctl->v_full[s], ph, abort))) break;
        if (!(ok = mbar_wait(&ctl->p_full[0], j & 1, abort))) break;
        tc_fence_after();
        issue_pv(0, s, j == 0);
      }
      if (ok && mbar_wait(&ctl->p_full[1], (nt - 1) & 1, abort)) {
        tc_fence_after();
        issue_pv(1, (nt - 1) % kStages, nt - 1 == 0);
        mma_commit(&ctl->v_empty[(nt - 1) % kStages]);
      }
      mma_commit(&ctl->drain);
      drain_wait(&ctl->drain, 0);
    }
  } else if (warp < kWarpTma) {
    // ---------------- softmax / correction / epilogue of tile x, one row per thread
    regs_increase<kSoftmaxRegs>();
    const int x = warp / 4;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + col_s(x), t_o = tmem + lane_off + col_o(x);
    const float scale_log2 = 1.4426950408889634f * rsqrtf((float)kHeadDim);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      if (!(ok = mbar_wait(&ctl->s_full[x], j & 1, abort))) break;
      // S_x(j) complete implies PV_x(j-1) complete (MMAs finish in issue
      // order); observing o_done here keeps its phases in step.
      if (j > 0 && !(ok = mbar_wait(&ctl->o_done[x], (j - 1) & 1, abort))) break;
      tc_fence_after();
      const int valid = T - (j0 + j) * kRows;   // keys of this tile that exist (< 128 only in the last tile)
      // the row's 128 scores in registers, one TMEM round trip
      uint32_t sv[128];
      tmem_ld128(t_s, sv);
      if (valid < kRows) {               // the ragged last tile only (uniform branch)
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= valid) sv[i] = __float_as_uint(-INFINITY);
      }
      // row max of the raw scores, 4 chains of 3-input max (scale > 0 commutes with max)
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 64; ++i)
        m4[i & 3] = max3(m4[i & 3], __uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]));
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * scale_log2;
      const float m_new = fmaxf(m, mx);
      const bool need = (j > 0) && (m_new > m + 8.0f);
      if (j == 0) {
        m = m_new;
      } else if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
        if (need) m = m_new;
        l *= alpha;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(t_o + c * 32, o);
        }
      }
      // p = 2^(s * scale_log2 - m) in float pairs (packed FMA, MUFU exp2,
      // packed row sum in 4 pair accumulators), rounded to bf16 and packed in
      // place: pair k (columns 2k, 2k+1) -> sv[k]
      const float neg_m = -m;
      float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        float a, b;
        fma2(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]), scale_log2, neg_m, a, b);
        const float p0 = ex2_approx(a), p1 = ex2_approx(b);
        add2(sum[2 * (k & 3)], sum[2 * (k & 3) + 1], p0, p1);
        sv[k] = pack_bf16x2(p0, p1);
      }
      l += ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
      tmem_st32(t_s, *reinterpret_cast<uint32_t(*)[32]>(sv));
      tmem_st32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctl->p_full[x]);
    }
    // re-derived from the block index read afresh, so nothing of it is held
    // through the loop above
    Item it;
    if constexpr (kSplit) {
      uint32_t b;
      asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(b));
      it = item_of((int)b, T, plan);
    } else {
      it = Item{(int)blockIdx.y, (int)blockIdx.x * 2 * kRows, 0, nt, -1};
    }
    const int head = it.head, q0 = it.q0;
    if (kSplit && ok && it.slot >= 0 && mbar_wait(&ctl->o_done[x], (nt - 1) & 1, abort)) {
      // a key range of a split unit: unnormalised rows with their max and sum
      tc_fence_after();
      float4 *dst =
          reinterpret_cast<float4 *>(plan.part + ((size_t)it.slot * 2 * kRows + x * kRows + row) * kPartRowFloats);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(t_o + c * 32, o);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[c * 8 + q] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                       __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
      }
      dst[32] = make_float4(m, l, 0.f, 0.f);
    } else if (ok && mbar_wait(&ctl->o_done[x], (nt - 1) & 1, abort)) {
      tc_fence_after();
      const float inv = 1.0f / l;
      const int t = q0 + x * kRows + row;
      uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)(t < T ? t : 0) * kCatCols + head * kHeadDim);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(t_o + c * 32, o);
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
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// Combines the key ranges of each split unit, in range order (deterministic):
// with m* the largest range max, O = sum_r O_r 2^(m_r - m*) and
// l = sum_r l_r 2^(m_r - m*), the output row is O / l in bf16.  One warp per
// query row, four output values per lane.
__global__ void __launch_bounds__(256)
    attention_merge_kernel(const float *__restrict__ part, int T, Plan plan, __nv_bfloat16 *__restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int r = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x % 32;
  const int unit = plan.n_full + r / (2 * kRows), row_in_unit = r % (2 * kRows);
  const int t = (unit % plan.n_qp) * 2 * kRows + row_in_unit;
  if (t >= T) return;
  const int head = unit / plan.n_qp;
  const float *base = part + ((size_t)(unit - plan.n_full) * plan.splits * 2 * kRows + row_in_unit) * kPartRowFloats;
  const size_t item_stride = (size_t)2 * kRows * kPartRowFloats;
  // every range's (m, l, O slice) is loaded before any is used (one round
  // trip, not one per range); the sums run in range order
  float m[kMaxSplits], lk[kMaxSplits];
  float4 v[kMaxSplits];
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    if (k < plan.splits) {
      const float *p = base + k * item_stride;
      m[k] = __ldg(p + 128);
      lk[k] = __ldg(p + 129);
      v[k] = __ldg(reinterpret_cast<const float4 *>(p) + lane);
    }
  }
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k)
    if (k < plan.splits) mx = fmaxf(mx, m[k]);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxSplits; ++k) {
    if (k < plan.splits) {
      const float w = ex2_approx(m[k] - mx);
      o.x = fmaf(v[k].x, w, o.x);
      o.y = fmaf(v[k].y, w, o.y);
      o.z = fmaf(v[k].z, w, o.z);
      o.w = fmaf(v[k].w, w, o.w);
      l = fmaf(lk[k], w, l);
    }
  }
  const float inv = 1.0f / l;
  *reinterpret_cast<uint2 *>(out + (size_t)t * kCatCols + head * kHeadDim + lane * 4) =
      make_uint2(pack_bf16x2(o.x * inv, o.y * inv), pack_bf16x2(o.z * inv, o.w * inv));
}

// Split plan: the units that fill whole waves of one CTA per SM run whole;
// the units of the last, partial wave are split into the most key ranges (at
// most 8, each of at least 4 key tiles) that still fit in one wave and in the
// partial buffer.  No split without a buffer.
Plan attention_plan(int T, int sms, float *part, size_t part_bytes) {
  const int nt = (T + kRows - 1) / kRows;
  Plan p{};
  p.n_qp = (T + 2 * kRows - 1) / (2 * kRows);
  const int units = p.n_qp * kHeads;
  p.n_full = units;
  p.splits = 1;
  p.part = part;
  if (!part || sms < 1) return p;
  const int full = units / sms * sms, rem = units - full;
  if (rem == 0) return p;
  for (int S = kMaxSplits; S >= 2; --S) {
    if (rem * S > sms || nt / S < 4 || (size_t)rem * S * kPartItemBytes > part_bytes) continue;
    p.n_full = full;
    p.splits = S;
    return p;
  }
  return p;
}

}  // namespace attn_tc

cudaError_t launch_attention(const __nv_bfloat16 *qkv, int T, __nv_bfloat16 *cat, cudaStream_t s, bool pdl,
                             float *part, size_t part_bytes) {
  using namespace attn_tc;
  static std::atomic<bool> attr_set[kMaxDevices], attr_set_split[kMaxDevices];
  const int slot = device_slot();
  if (slot < 0 || !attr_set[slot].load(std::memory_order_acquire)) {
    // the warpgroup register split assumes exactly kLaunchRegs per thread at launch
    cudaFuncAttributes fa, fb;
    cudaError_t e = cudaFuncGetAttributes(&fa, attention_kernel<false>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fb, attention_kernel<true>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs || fb.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  }
  cudaError_t e = set_smem_once(attention_kernel<false>, (int)kSmem, attr_set);
  if (e == cudaSuccess) e = set_smem_once(attention_kernel<true>, (int)kSmem, attr_set_split);
  if (e != cudaSuccess) return e;
  CUtensorMap tm;
  if (!make_tmap_bf16(&tm, qkv, (uint64_t)T, kQkvCols, kRows)) return cudaErrorInvalidValue;
  const Plan plan = attention_plan(T, num_sms(), part, part_bytes);
  const int units = plan.n_qp * kHeads;
  if (plan.splits == 1)
    return launch_kernel(attention_kernel<false>, dim3(plan.n_qp, kHeads), dim3(kThreads), kSmem, s, pdl, tm, T, cat,
                         plan);
  const int items = plan.n_full + (units - plan.n_full) * plan.splits;
  const cudaError_t le =
      launch_kernel(attention_kernel<true>, dim3(items), dim3(kThreads), kSmem, s, pdl, tm, T, cat, plan);
  if (le != cudaSuccess) return le;
  return launch_kernel(attention_merge_kernel, dim3((units - plan.n_full) * 2 * kRows / 8), dim3(256), 0, s, pdl,
                       static_cast<const float *>(part), T, plan, cat);
}

}  // namespace flux3
