// Persistent, warp-specialised tcgen05 GEMM  C[M, N] = A[M, K] * B[N, K]^T
// (bf16 operands, fp32 accumulation in tensor memory) with the block's fused
// epilogues:
//   EPI_STORE         bf16 store of C
//   EPI_IN_PROJ       over the packed [Wq; Wk; Wv; Wmlp_in(a/b interleaved)]:
//                     per-head RMSNorm + 4-axis RoPE of q and k, plain v, and
//                     silu(a) * b of the MLP half
//   EPI_OUT_RESIDUAL  x += gate[stream] * C  (fp32 residual, in place)
//   EPI_STORE_F32     float32 store of C's first ldc columns (the embedders
//                     and the image output layer)
//
// CTA pairs (clusters of 2 on one TPC) share each 256 x 256 output tile:
// the even CTA of the pair (the leader) issues tcgen05.mma.cta_group::2 with
// M = 256, N = 256; each CTA holds its own 128 rows of the A tile and 128 of
// the 256 B rows in shared memory, and its own 128 accumulator rows in tensor
// memory.  Per SM that halves the B operand bytes the tensor core reads from
// shared memory and the bytes TMA writes, against a one-CTA 128 x 256 tile.
// For M <= 128 the one-CTA form runs instead (gemm1_kernel: 128 x 256 tiles,
// cta_group::1, all 256 B rows of a k-block in the CTA's shared memory, a
// 4-stage ring): a pair tile would be more than half padding there, and the
// 148 CTAs take twice as many tiles per round as 74 pairs.  Its weight loads
// carry an evict-first L2 policy (each weight line is read once).  Over NVFP4
// or fp8r weights (gemm1_fp4_kernel, gemm1_fp8_kernel) the codes arrive in a
// ring of their own and the epilogue warps expand each k-block into the bf16
// B stage in shared memory (see GemmCfg).
//
// Roles (320 threads per CTA): warp 0 issues the CTA's TMA loads (128 x 64
// of A, 128 x 64 of B, 128-byte swizzle) into a 6-stage ring, completing on
// the leader's stage barrier; warp 1 owns the 512-column TMEM allocation (two
// 256-column accumulators) and, in the leader, issues the MMAs from one
// thread and commits to both CTAs' barriers; warps 2-9 drain the other
// accumulator through tcgen05.ld (one output row and one 128-column half per
// thread) and run the epilogue, so the epilogue of tile i overlaps the MMAs
// of tile i+1.
// Units: the pairs (or CTAs) take units round robin.  Whole tiles fill complete
// rounds; when the last round would leave pairs idle, its tiles are split
// along K into ranges (out-projection only): each range stores its float32
// partial tile, and split_merge_residual_kernel sums a tile's ranges in a fixed
// order (deterministic) and applies the gated residual.
// Every wait is bounded (see mbar_wait); on a timeout the CTA drains its
// in-flight copies and MMAs, frees TMEM and returns.

#pragma once

#include <cuda_fp16.h>

#include "flux3_internal.h"
#include "ptx.cuh"

namespace flux3 {

namespace gemm_detail {

constexpr int kThreads = 320;
constexpr int kMaxSplitK = 12;   // most K ranges a split tile takes
constexpr int kEpiWarps = 8;
constexpr uint32_t kBoxBytes = 32 * 128;              // one epilogue output box: 32 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;                   // two 128-lane x 256-column fp32 accumulators

template <int kStages, int kCodeStages, int kBStages>
struct SharedCtl {
  uint64_t full[kStages];      // issuing CTA: the stage's TMA bytes (both CTAs' for a pair) landed
  uint64_t empty[kStages];     // every CTA: the stage's MMAs are done
  uint64_t tmem_full[2];       // every CTA: the accumulator holds a finished tile
  uint64_t tmem_empty[2];      // issuing CTA: every epilogue thread (of the pair) drained it
  uint64_t drain;
  uint64_t xbar[8];            // per epilogue warp: its residual box landed (out-projection)
  // NVFP4 weights (one-CTA form): the code ring and the converted B stages
  uint64_t cfull[kCodeStages];    // a k-block's e2m1 codes landed
  uint64_t cempty[kCodeStages];   // every converting thread has read them
  uint64_t bready[kBStages];      // every converting thread has written its B row of the stage
  uint64_t bempty[kBStages];      // the stage's MMAs are done (its B rows may be rewritten)
  uint32_t tmem_base;
  int abort;
};

// Weight formats of the B operand: bf16 through TMA, or codes expanded in
// shared memory by the epilogue warps (one-CTA form only).
enum : int { kWBf16 = 0, kWNvfp4 = 1, kWFp8r = 2 };

// The forms of the kernel.  Pair (kPair): a cluster of two CTAs on one TPC
// computes a 256 x 256 tile with cta_group::2 MMAs; each CTA stages 128 A
// rows and 128 B rows per k-block.  Single: one CTA computes a 128 x 256 tile
// with cta_group::1 MMAs and stages 128 A rows and all 256 B rows.  The
// single form serves M <= 128, where a pair tile would be at most half rows.
// Low-precision weights (single form only): B arrives as NVFP4 e2m1 codes (a
// quarter of the bf16 bytes) or fp8r e4m3 codes (half) in a ring of its own,
// and the epilogue warps, idle while the tile accumulates, expand each k-block
// into the bf16 B stage the MMA reads.  The A and B stages then form separate
// rings: A (from L2) four or five deep, the expanded B two deep (the expansion
// works out of shared memory, so one stage in hand while the MMAs read the
// other is enough).
template <bool kPair, int kWFmt = kWBf16>
struct GemmCfg {
  static constexpr bool kConv = kWFmt != kWBf16;
  static_assert(!(kPair && kConv), "low-precision weights are expanded in the one-CTA form only");
  static constexpr int kStages = kPair ? 6 : (kWFmt == kWNvfp4 ? 5 : 4);   // A stages (and B stages for bf16)
  static constexpr int kBStages = kConv ? 2 : kStages;
  static constexpr int kCodeStages = kWFmt == kWNvfp4 ? 5 : (kWFmt == kWFp8r ? 4 : 1);
  static constexpr int kCodeCols = kWFmt == kWNvfp4 ? kBK / 2 : kBK;        // code bytes per row of a k-block
  static constexpr int kTileM = kPair ? 256 : 128;                     // output rows per tile
  static constexpr uint32_t kABytes = 128 * kBK * 2;                   // 16 KB: 128 A rows per CTA
  static constexpr uint32_t kBBytes = (kPair ? 128 : 256) * kBK * 2;   // B rows per CTA
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kCodeBytes = kConv ? 256 * kCodeCols : 0;   // 8 KB (e2m1) or 16 KB (e4m3)
  // bytes completing on one stage barrier (with codes: A only)
  static constexpr uint32_t kTxBytes = kConv ? kABytes : (kPair ? 2 : 1) * kStageBytes;
  static constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kStages * kABytes + kBStages * kBBytes +
                                       (kConv ? kCodeStages * kCodeBytes : 0) + kEpiWarps * kBoxBytes +
                                       sizeof(SharedCtl<kStages, kCodeStages, kBStages>);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// One B row of a k-block from NVFP4: 64 e2m1 codes (32 bytes at `codes`, two
// per byte, the lower nibble first), their four e4m3 block scales (one per 16
// inputs, byte j of `scales4`) and the tensor's float32 scale g.  Each weight
// is e2m1 * e4m3 (exact in f16: at most 6 significant bits, within 2^-10 ..
// 2688), widened to float32, times g (rounded to float32), rounded to bf16 --
// the expansion kernel's arithmetic, so the MMA sees the same bf16 values.
// The row's eight 16-byte chunks go to the 128-byte-swizzled K-major layout
// of the B stage (row r of the stage at (r / 8) * 1024 + (r % 8) * 128).
__device__ __forceinline__ void expand_fp4_row(const uint8_t *codes, uint32_t scales4, float g, uint8_t *b_stage,
                                               int r) {
  const uint4 c0 = *reinterpret_cast<const uint4 *>(codes);
  const uint4 c1 = *reinterpret_cast<const uint4 *>(codes + 16);
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  uint32_t s01, s23;   // f16x2 pairs of the four block scales
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
      : "=r"(s01), "=r"(s23)
      : "r"(scales4));
  const __half2 sp[2] = {*reinterpret_cast<const __half2 *>(&s01), *reinterpret_cast<const __half2 *>(&s23)};
  uint8_t *row = b_stage + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q) {   // chunk q: inputs 8q .. 8q+7 of group q / 2
    uint32_t h[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        " cvt.rn.f16x2.e2m1x2 %1, b1;\n cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w[q]));
    const int grp = q >> 1;
    const __half2 s = (grp & 1) ? __high2half2(sp[grp >> 1]) : __low2half2(sp[grp >> 1]);
    uint32_t o[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&h[b]), s);   // exact
      float lo = __low2float(v), hi = __high2float(v);
      mul2(lo, hi, g);
      o[b] = pack_bf16x2(lo, hi);
    }
    *reinterpret_cast<uint4 *>(row + ((q ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// One B row of a k-block from fp8r: 64 e4m3 codes (64 bytes at `codes`) and
// the row's float32 scale s.  Each weight is e4m3 (exact in f16, and so in
// float32) times s, rounded to float32, then to bf16 -- the expansion kernel's
// arithmetic.  Same swizzled layout as expand_fp4_row.
__device__ __forceinline__ void expand_fp8_row(const uint8_t *codes, float s, uint8_t *b_stage, int r) {
  uint8_t *row = b_stage + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int h = 0; h < 4; ++h) {   // 16 codes: chunks 2h, 2h+1
    const uint4 c = *reinterpret_cast<const uint4 *>(codes + 16 * h);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t p01, p23;   // f16x2 of codes (0, 1) and (2, 3) of word k
      asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
          : "=r"(p01), "=r"(p23)
          : "r"(w[k]));
      const __half2 v01 = *reinterpret_cast<const __half2 *>(&p01), v23 = *reinterpret_cast<const __half2 *>(&p23);
      float a = __low2float(v01), b = __high2float(v01), c2 = __low2float(v23), d = __high2float(v23);
      mul2(a, b, s);
      mul2(c2, d, s);
      o[2 * k] = pack_bf16x2(a, b);
      o[2 * k + 1] = pack_bf16x2(c2, d);
    }
    *reinterpret_cast<uint4 *>(row + (((2 * h) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(row + (((2 * h + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// Waits for `bar` to pass `parity`, with a time limit only (used while
// draining after an abort, when the abort flag is already set).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      record_error(DEVERR_TIMEOUT);
      return;
    }
  }
}

// One 32-row x 64-column bf16 box of an epilogue warp's output: each lane
// writes its row's eight 16-byte chunks into the warp's 4 KB staging buffer
// in the 128-byte-swizzled layout of the tensor map, then one lane issues a
// TMA store, so global memory sees whole 128-byte lines instead of 16-byte
// pieces of 32 rows per instruction.
struct BoxWriter {
  uint8_t *buf;
  uint32_t lane;
  __device__ __forceinline__ void begin() const {   // the previous box has been read out of buf
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  }
  __device__ __forceinline__ void put(int q, uint32_t a, uint32_t b, uint32_t c, uint32_t d) const {
    *reinterpret_cast<uint4 *>(buf + lane * 128 + ((q ^ (lane & 7)) * 16)) = make_uint4(a, b, c, d);
  }
  __device__ __forceinline__ void store(const CUtensorMap *tm, int x, int y) const {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm, buf, x, y);
      bulk_commit();
    }
  }
};

// The out-projection's residual x goes through the same box (32 rows x 32
// fp32 columns): a TMA load fills it, each lane updates its row in place, and a
// TMA store writes it back.
__device__ __forceinline__ void load_x_box(const BoxWriter &bw, const CUtensorMap *tm, uint64_t *bar, int x, int y) {
  if (bw.lane == 0) {
    mbar_arrive_expect_tx(bar, kBoxBytes);
    tma_load_2d(bw.buf, tm, bar, x, y);
  }
}

__device__ __forceinline__ void put_chunk_bf16(const BoxWriter &bw, int q0, const uint32_t (&r)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    bw.put(q0 + q, pack_bf16x2(f32(r[8 * q + 0]), f32(r[8 * q + 1])), pack_bf16x2(f32(r[8 * q + 2]), f32(r[8 * q + 3])),
           pack_bf16x2(f32(r[8 * q + 4]), f32(r[8 * q + 5])), pack_bf16x2(f32(r[8 * q + 6]), f32(r[8 * q + 7])));
}

// Epilogue of one half (128 of the 256 columns) of the thread's accumulator
// row.  taddr: TMEM address of (this warp's lane quarter, column 0 of the
// tile).  Column half `half` is: for q / k tiles head `half` of the tile's two
// heads, for v and plain tiles columns 128*half .. +127, for MLP tiles the
// SwiGLU outputs 64*half .. +63 (a in columns 0..127, b in 128..255).
// bf16 outputs leave through the warp's staging box and TMA stores (tm0: C or
// qkv, tm1: cat); row0 is the first of the warp's 32 rows (stores clip rows
// past M).
// One 32-column chunk c of a q / k head: RMSNorm (inv, per-dim scales ns)
// then RoPE on the 16 adjacent pairs (cs, sn), packed to bf16 into the warp's
// box (chunk c fills the box's columns 32 * (c & 1) .. +31).
__device__ __forceinline__ void qk_rope_chunk(const BoxWriter &bw, const uint32_t (&r)[32], float inv,
                                              const float (&ns)[32], const float (&cs)[16], const float (&sn)[16],
                                              int c) {
  uint32_t o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float x0 = f32(r[2 * j]) * inv * ns[2 * j];
    const float x1 = f32(r[2 * j + 1]) * inv * ns[2 * j + 1];
    o[j] = pack_bf16x2(x0 * cs[j] - x1 * sn[j], x0 * sn[j] + x1 * cs[j]);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) bw.put(4 * (c & 1) + q, o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}

// kPipeTables: the q / k tiles' RoPE rows are loaded one chunk ahead with
// in-order loads (the forms whose epilogue warps hold no code-expansion state;
// in the others the extra registers would spill).
template <int EPI, bool kPipeTables = true>
__device__ __forceinline__ bool epilogue_half(uint32_t taddr, int row, int row0, int M, int n_blk, int half,
                                              const EpiParams &ep, const BoxWriter &bw, const CUtensorMap *tm0,
                                              const CUtensorMap *tm1, uint64_t *xbar, uint32_t &xphase,
                                              volatile int *abort) {
  const bool live = row < M;
  const int n0 = n_blk * kBN + half * 128;    // first output column of this half (not for MLP tiles)
  const uint32_t th = taddr + half * 128;
  uint32_t r[32];
  if constexpr (EPI == EPI_STORE) {
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      bw.begin();
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        tmem_ld32(th + (2 * b + c2) * 32, r);
        put_chunk_bf16(bw, 4 * c2, r);
      }
      bw.store(tm0, n0 + 64 * b, row0);
    }
  } else if constexpr (EPI == EPI_STORE_F32) {
    // four 32-row x 32-column float32 boxes; columns past ldc (rows of a
    // weight padded to the 256-column tile) are not stored
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      if (n0 + 32 * c >= ep.ldc) break;
      bw.begin();
      tmem_ld32(th + c * 32, r);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4 *>(bw.buf + bw.lane * 128 + ((q ^ (bw.lane & 7)) * 16)) =
            make_float4(f32(r[4 * q]), f32(r[4 * q + 1]), f32(r[4 * q + 2]), f32(r[4 * q + 3]));
      bw.store(tm0, n0 + 32 * c, row0);
    }
  } else if constexpr (EPI == EPI_OUT_RESIDUAL) {
    // x[row, n0 .. n0+127] += gate[stream(row)] * acc, as four 32-column boxes;
    // box 0's load was issued before the accumulator was waited for
    const int s = live ? ep.sid[row] : 0;
    const float4 *gate = reinterpret_cast<const float4 *>(ep.mod + (size_t)s * kModLen + 2 * kHidden + n0);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      if (!mbar_wait(xbar, xphase, abort)) return false;
      xphase ^= 1;
      tmem_ld32(th + c * 32, r);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 *p = reinterpret_cast<float4 *>(bw.buf + bw.lane * 128 + ((q ^ (bw.lane & 7)) * 16));
        const float4 g = __ldg(gate + c * 8 + q);
        float4 xv = *p;
        xv.x = fmaf(g.x, f32(r[4 * q + 0]), xv.x);
        xv.y = fmaf(g.y, f32(r[4 * q + 1]), xv.y);
        xv.z = fmaf(g.z, f32(r[4 * q + 2]), xv.z);
        xv.w = fmaf(g.w, f32(r[4 * q + 3]), xv.w);
        *p = xv;
      }
      bw.store(tm0, n0 + 32 * c, row0);
      if (c < 3) {
        bw.begin();
        load_x_box(bw, tm0, xbar, n0 + 32 * (c + 1), row0);
      }
    }
  } else {  // EPI_IN_PROJ
    constexpr int kQTiles = kHidden / kBN;          // 12
    constexpr int kVEnd = 3 * kHidden / kBN;        // 36
    if (n_blk < 2 * kQTiles) {
      // q or k, head `half` of the tile: RMSNorm over its 128 dims in fp32
      // straight from the accumulator, then RoPE on adjacent pairs; the 32
      // columns of chunk c are exactly RoPE axis c (t, h, w, l).
      const float4 *nscale4 = reinterpret_cast<const float4 *>(n_blk < kQTiles ? ep.qnorm : ep.knorm);
      const int rrow = live ? row : 0;
      const float4 *cs4 = reinterpret_cast<const float4 *>(ep.cos_tab + (size_t)rrow * kRopePairs);
      const float4 *sn4 = reinterpret_cast<const float4 *>(ep.sin_tab + (size_t)rrow * kRopePairs);
      float ss = 0.f;
      if constexpr (kPipeTables) {
        // The row's RoPE pairs stream one chunk ahead through in-order loads:
        // chunk 0's go out before the sum-of-squares pass, chunk c+1's before
        // chunk c's TMEM read, so no chunk waits a full memory round trip.
        float4 ca[4], sa[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) ca[q] = ldg_f4_in_order(cs4 + q), sa[q] = ldg_f4_in_order(sn4 + q);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(th + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) ss = fmaf(f32(r[i]), f32(r[i]), ss);
        }
        const float inv = rsqrtf(ss * (1.0f / kHeadDim) + ep.eps_rms);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          if ((c & 1) == 0) bw.begin();
          // this chunk's 16 RoPE pairs (loaded one chunk earlier) and 32 norm
          // scales (the same for every row: L1 hits after the first warp)
          float cs[16], sn[16], ns[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            cs[4 * q] = ca[q].x, cs[4 * q + 1] = ca[q].y, cs[4 * q + 2] = ca[q].z, cs[4 * q + 3] = ca[q].w;
            sn[4 * q] = sa[q].x, sn[4 * q + 1] = sa[q].y, sn[4 * q + 2] = sa[q].z, sn[4 * q + 3] = sa[q].w;
          }
          if (c < 3) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              ca[q] = ldg_f4_in_order(cs4 + (c + 1) * 4 + q), sa[q] = ldg_f4_in_order(sn4 + (c + 1) * 4 + q);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 a = ldg_f4_in_order(nscale4 + c * 8 + q);
            ns[4 * q] = a.x, ns[4 * q + 1] = a.y, ns[4 * q + 2] = a.z, ns[4 * q + 3] = a.w;
          }
          tmem_ld32(th + c * 32, r);
          qk_rope_chunk(bw, r, inv, ns, cs, sn, c);
          if (c & 1) bw.store(tm0, n0 + 64 * (c >> 1), row0);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(th + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) ss = fmaf(f32(r[i]), f32(r[i]), ss);
        }
        const float inv = rsqrtf(ss * (1.0f / kHeadDim) + ep.eps_rms);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          if ((c & 1) == 0) bw.begin();
          // this chunk's 16 RoPE pairs and 32 norm scales, 16-byte loads issued
          // ahead of the TMEM read
          float cs[16], sn[16], ns[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 a = __ldg(cs4 + c * 4 + q), b = __ldg(sn4 + c * 4 + q);
            cs[4 * q] = a.x, cs[4 * q + 1] = a.y, cs[4 * q + 2] = a.z, cs[4 * q + 3] = a.w;
            sn[4 * q] = b.x, sn[4 * q + 1] = b.y, sn[4 * q + 2] = b.z, sn[4 * q + 3] = b.w;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 a = __ldg(nscale4 + c * 8 + q);
            ns[4 * q] = a.x, ns[4 * q + 1] = a.y, ns[4 * q + 2] = a.z, ns[4 * q + 3] = a.w;
          }
          tmem_ld32(th + c * 32, r);
          qk_rope_chunk(bw, r, inv, ns, cs, sn, c);
          if (c & 1) bw.store(tm0, n0 + 64 * (c >> 1), row0);
        }
      }
    } else if (n_blk < kVEnd) {
#pragma unroll 1
      for (int b = 0; b < 2; ++b) {
        bw.begin();
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          tmem_ld32(th + (2 * b + c2) * 32, r);
          put_chunk_bf16(bw, 4 * c2, r);
        }
        bw.store(tm0, n0 + 64 * b, row0);
      }
    } else {
      // MLP tile m holds a[128m .. 128m+127] in columns 0..127 and the matching
      // b rows in columns 128..255 (interleaved when the weights were packed);
      // this half produces SwiGLU outputs 64*half .. 64*half+63 of the tile.
      const int m = n_blk - kVEnd;
      uint32_t b[32];
      bw.begin();
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const uint32_t ca = taddr + half * 64 + c * 32;
        tmem_ld32x2(ca, ca + 128, r, b);
        uint32_t o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float a0 = f32(r[2 * j]), a1 = f32(r[2 * j + 1]);
          // silu(a) = a / (1 + e^-a) with the fast division: 2 ulp in fp32, far
          // below the bf16 rounding of the output, and 0 for a below about -87
          // (where |silu(a)| < 1e-36).  The IEEE division measured 2.5x slower
          // in this epilogue, and 6x on the zero rows that pad a ragged tile.
          const float g0 = __fdividef(a0, 1.0f + __expf(-a0)) * f32(b[2 * j]);
          const float g1 = __fdividef(a1, 1.0f + __expf(-a1)) * f32(b[2 * j + 1]);
          o[j] = pack_bf16x2(g0, g1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) bw.put(4 * c + q, o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      }
      bw.store(tm1, kHidden + m * 128 + half * 64, row0);
    }
  }
  return true;
}

// Tile t of the pair schedule -> (row block, column block).
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, bool n_fast, int &m_blk, int &n_blk) {
  if (n_fast) {
    m_blk = t / num_n;
    n_blk = t % num_n;
  } else {
    m_blk = t % num_m;
    n_blk = t / num_m;
  }
}

// The pair schedule over units: units 0 .. n_full-1 are whole tiles (every
// k-block); each later tile is `splits` units, unit ks of it covering k-blocks
// [ks * num_kb / splits, (ks + 1) * num_kb / splits).  slot = -1 for a whole
// tile, else the unit's index among the split units (its partial buffer).
struct Unit {
  int m_blk, n_blk, kb0, kb1, slot;
};
__device__ __forceinline__ Unit unit_of(int u, int n_full, int splits, int num_m, int num_n, bool n_fast,
                                        int num_kb) {
  Unit r;
  int tile;
  if (u < n_full) {
    tile = u;
    r.kb0 = 0;
    r.kb1 = num_kb;
    r.slot = -1;
  } else {
    const int v = u - n_full, ks = v % splits;
    tile = n_full + v / splits;
    r.kb0 = ks * num_kb / splits;
    r.kb1 = (ks + 1) * num_kb / splits;
    r.slot = v;
  }
  tile_coords(tile, num_m, num_n, n_fast, r.m_blk, r.n_blk);
  return r;
}

// A split unit's fp32 accumulator rows go to its partial buffer (tile_m x 256
// float32 per unit, row = row in the tile) as four 32 x 32 boxes per half.
__device__ __forceinline__ void store_partial_half(uint32_t taddr, int slot, int row_box0, int rows_valid, int half,
                                                   int tile_m, const BoxWriter &bw, const CUtensorMap *tmP) {
  if (row_box0 >= rows_valid) return;   // the merge reads no row past M
  uint32_t r[32];
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    bw.begin();
    tmem_ld32(taddr + half * 128 + c * 32, r);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4 *>(bw.buf + bw.lane * 128 + ((q ^ (bw.lane & 7)) * 16)) =
          make_float4(f32(r[4 * q]), f32(r[4 * q + 1]), f32(r[4 * q + 2]), f32(r[4 * q + 3]));
    bw.store(tmP, half * 128 + c * 32, slot * tile_m + row_box0);
  }
}

// tmB: the bf16 weight, or the code bytes of a low-precision weight: NVFP4
// e2m1 codes [N, K / 2] (boxes of 32 bytes x 256 rows; ep.w_scales holds the
// e4m3 block scales [N, K / 16], ep.w_globals the tensors' float32 scales) or
// fp8r e4m3 codes [N, K] (boxes of 64 bytes x 256 rows; ep.w_scales holds the
// float32 row scales: [N] for the in-projection, [N][2] (attn_out, mlp_out)
// for the out-projection).
template <int EPI, bool kPair, int kWFmt>
__device__ __forceinline__ void gemm_body(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmO0,
                                          const CUtensorMap &tmO1, int M, int N, int K, int n_full, int splits,
                                          const EpiParams &ep) {
  using C = GemmCfg<kPair, kWFmt>;
  constexpr bool kConv = C::kConv;   // B from codes expanded by the epilogue warps
  constexpr int kStages = C::kStages;
  constexpr int kBStages = C::kBStages;
  constexpr int kCodeStages = C::kCodeStages;
  constexpr int kTileM = C::kTileM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *smA = smem;
  uint8_t *smB = smem + kStages * C::kABytes;
  uint8_t *smC = smB + kBStages * C::kBBytes;                        // NVFP4 code ring
  uint8_t *sOut = smC + (kConv ? kCodeStages * C::kCodeBytes : 0);   // [epilogue warp] 4 KB output box
  auto *ctl = reinterpret_cast<SharedCtl<kStages, kCodeStages, kBStages> *>(sOut + kEpiWarps * kBoxBytes);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = kPair ? cluster_ctarank() : 0;   // 0 = the CTA that issues the MMAs
  const bool leader = rank == 0;
  // a worker is a CTA pair or a single CTA
  const int worker = kPair ? blockIdx.x / 2 : blockIdx.x;
  const int num_workers = kPair ? gridDim.x / 2 : gridDim.x;
  const int num_m = (M + kTileM - 1) / kTileM;
  const int num_n = N / kBN;
  const int num_tiles = num_m * num_n;
  const int num_units = n_full + (num_tiles - n_full) * splits;
  const int num_kb = K / kBK;
  // Tile order: consecutive workers share the operand with more rows, so that
  // it is read from DRAM about once and the smaller one is re-read from L2.
  const bool n_fast = M > N;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tmem_full[a], 1);
      mbar_init(&ctl->tmem_empty[a], (kPair ? 2 : 1) * 256);
    }
    mbar_init(&ctl->drain, 1);
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(&ctl->xbar[w], 1);
    if constexpr (kConv) {
      for (int s = 0; s < kCodeStages; ++s) {
        mbar_init(&ctl->cfull[s], 1);
        mbar_init(&ctl->cempty[s], kEpiWarps * 32);
      }
      for (int s = 0; s < kBStages; ++s) {
        mbar_init(&ctl->bready[s], kEpiWarps * 32);
        mbar_init(&ctl->bempty[s], 1);
      }
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&ctl->tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (kPair)
    cluster_sync();        // both CTAs' barriers are initialised before any cross-CTA signal
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  volatile int *abort = &ctl->abort;
  // One-CTA form (small M, bound by streaming the weights B from DRAM): the
  // B halves of the first ring stages are loaded before griddep_wait, so the
  // DRAM latency of the first tiles passes while the previous kernel
  // finishes.  No kernel this one may overlap writes B: the weights (or their
  // codes) are constant, or expanded in HBM at the start of the block -- and
  // then LayerNorm releases the in-projection only after its own wait, so the
  // expansion has completed; the out-projection starts only after the
  // in-projection has.  The A halves, which the previous kernel may write,
  // follow after the wait.
  int n_pre = 0;
  if constexpr (kConv) {
    // the codes of the first k-blocks (lane 1 runs the code ring)
    if (warp == 0 && lane == 1 && worker < num_units) {
      const Unit un = unit_of(worker, n_full, splits, num_m, num_n, n_fast, num_kb);
      n_pre = un.kb1 - un.kb0 < kCodeStages ? un.kb1 - un.kb0 : kCodeStages;
      for (int i = 0; i < n_pre; ++i) {
        mbar_arrive_expect_tx(&ctl->cfull[i], C::kCodeBytes);
        tma_load_2d_hint(smC + i * C::kCodeBytes, &tmB, &ctl->cfull[i], (un.kb0 + i) * C::kCodeCols, un.n_blk * kBN,
                         l2_policy_evict_first());
      }
    }
  } else if constexpr (!kPair) {
    if (warp == 0 && lane == 0 && worker < num_units) {
      const Unit un = unit_of(worker, n_full, splits, num_m, num_n, n_fast, num_kb);
      n_pre = un.kb1 - un.kb0 < kStages ? un.kb1 - un.kb0 : kStages;
      for (int i = 0; i < n_pre; ++i) {
        uint8_t *b_dst = smB + i * C::kBBytes;
        mbar_arrive_expect_tx(&ctl->full[i], C::kTxBytes);
        const uint64_t pol = l2_policy_evict_first();
        tma_load_2d_hint(b_dst, &tmB, &ctl->full[i], (un.kb0 + i) * kBK, un.n_blk * kBN, pol);
        tma_load_2d_hint(b_dst + 128 * kBK * 2, &tmB, &ctl->full[i], (un.kb0 + i) * kBK, un.n_blk * kBN + 128, pol);
      }
    }
  }
  // set-up above overlaps the previous kernel when launched as its programmatic dependent
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: this CTA's 128 A rows and its B rows
      // (pair: 128, completing on the leader's full barrier; single: 256).
      // The one-CTA form reads each weight line once: its B loads are
      // evicted from L2 first, so they do not push out the small tensors the
      // epilogues and the next kernels read (RoPE tables, residual rows).
      uint64_t b_policy = 0;
      if constexpr (!kPair) b_policy = l2_policy_evict_first();
      int last_phase[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_phase[s] = -1;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int it = 0;   // k-blocks issued so far; the first n_pre have their B half in flight
      for (int u = worker; u < num_units && ok; u += num_workers) {
        const Unit un = unit_of(u, n_full, splits, num_m, num_n, n_fast, num_kb);
        const int a_row = un.m_blk * kTileM + (int)rank * 128;
        const int b_row = un.n_blk * kBN + (int)rank * 128;
        for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
          const bool pre = !kConv && it < n_pre;   // a fresh stage: no wait for it to drain
          if (!pre && !mbar_wait(&ctl->empty[stage], phase ^ 1, abort)) {
            ok = false;
            break;
          }
          uint8_t *a_dst = smA + stage * C::kABytes;
          uint8_t *b_dst = smB + stage * C::kBBytes;
          if constexpr (kPair) {
            const uint32_t full_leader = map_to_cta(smem_addr(&ctl->full[stage]), 0);
            if (leader) mbar_arrive_expect_tx(&ctl->full[stage], C::kTxBytes);
            tma_load_2d_pair(a_dst, &tmA, full_leader, kb * kBK, a_row);
            tma_load_2d_pair(b_dst, &tmB, full_leader, kb * kBK, b_row);
          } else if constexpr (kConv) {
            mbar_arrive_expect_tx(&ctl->full[stage], C::kTxBytes);   // B is written by the converting warps
            tma_load_2d(a_dst, &tmA, &ctl->full[stage], kb * kBK, a_row);
          } else {
            if (!pre) {
              mbar_arrive_expect_tx(&ctl->full[stage], C::kTxBytes);
              tma_load_2d_hint(b_dst, &tmB, &ctl->full[stage], kb * kBK, b_row, b_policy);
              tma_load_2d_hint(b_dst + 128 * kBK * 2, &tmB, &ctl->full[stage], kb * kBK, b_row + 128, b_policy);
            }
            tma_load_2d(a_dst, &tmA, &ctl->full[stage], kb * kBK, a_row);
          }
          last_phase[stage] = (int)phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok && leader) {  // every copy of a stage completes on the issuing CTA's barrier
        for (int s = 0; s < kStages; ++s)
          if (last_phase[s] >= 0) drain_wait(&ctl->full[s], (uint32_t)last_phase[s]);
      }
    } else if (kConv && lane == 1) {
      // ---------------- code ring: each k-block's 256 rows of code bytes
      const uint64_t b_policy = l2_policy_evict_first();
      int last_phase[kCodeStages];
#pragma unroll
      for (int s = 0; s < kCodeStages; ++s) last_phase[s] = -1;
      uint32_t cs = 0, cphase = 0;
      bool ok = true;
      int it = 0;   // the first n_pre k-blocks went out before griddep_wait
      for (int u = worker; u < num_units && ok; u += num_workers) {
        const Unit un = unit_of(u, n_full, splits, num_m, num_n, n_fast, num_kb);
        for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
          if (it >= n_pre) {
            if (!mbar_wait(&ctl->cempty[cs], cphase ^ 1, abort)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&ctl->cfull[cs], C::kCodeBytes);
            tma_load_2d_hint(smC + cs * C::kCodeBytes, &tmB, &ctl->cfull[cs], kb * C::kCodeCols, un.n_blk * kBN,
                             b_policy);
          }
          last_phase[cs] = (int)cphase;
          if (++cs == kCodeStages) {
            cs = 0;
            cphase ^= 1;
          }
        }
      }
      if (!ok)
        for (int s = 0; s < kCodeStages; ++s)
          if (last_phase[s] >= 0) drain_wait(&ctl->cfull[s], (uint32_t)last_phase[s]);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer: kTileM x 256 x 16 per instruction
      constexpr uint32_t idesc = idesc_bf16(kTileM, kBN, false);
      // descriptors encoded once and moved by constant offsets per MMA; a
      // 256-row B stage is one operand (row groups of 8 at 1024-byte strides)
      const SmemDesc da = smem_desc_split(smem_addr(smA), 16, 1024, kSwizzle128B);
      const SmemDesc db = smem_desc_split(smem_addr(smB), 16, 1024, kSwizzle128B);
      uint32_t stage = 0, phase = 0;
      uint32_t bstage = 0, bphase = 0;   // the B ring (its own with codes, else the same as the A ring)
      int local = 0;
      bool ok = true;
      for (int u = worker; u < num_units && ok; u += num_workers, ++local) {
        const Unit un = unit_of(u, n_full, splits, num_m, num_n, n_fast, num_kb);
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&ctl->tmem_empty[acc], acc_phase ^ 1, abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          if (!mbar_wait(&ctl->full[stage], phase, abort) ||
              (kConv && !mbar_wait(&ctl->bready[bstage], bphase, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t boff = (kConv ? bstage : stage) * C::kBBytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t accumulate = (kb != un.kb0 || k != 0) ? 1u : 0u;
            if constexpr (kPair)
              mma_bf16_ss_pair_at(d_tmem, da, stage * C::kABytes + k * 32, db, boff + k * 32, idesc, accumulate);
            else
              mma_bf16_ss_at(d_tmem, da, stage * C::kABytes + k * 32, db, boff + k * 32, idesc, accumulate);
          }
          if constexpr (kPair) {
            mma_commit_pair_mc(&ctl->empty[stage], 0x3);
          } else {
            mma_commit(&ctl->empty[stage]);
            if constexpr (kConv) mma_commit(&ctl->bempty[bstage]);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
          if (++bstage == kBStages) {
            bstage = 0;
            bphase ^= 1;
          }
        }
        if (ok) {
          if constexpr (kPair)
            mma_commit_pair_mc(&ctl->tmem_full[acc], 0x3);
          else
            mma_commit(&ctl->tmem_full[acc]);
        }
      }
      // all MMAs issued by this thread are complete once `drain` arrives
      if constexpr (kPair)
        mma_commit_pair(&ctl->drain);
      else
        mma_commit(&ctl->drain);
      drain_wait(&ctl->drain, 0);
    }
  } else {
    // ---------------- epilogue warps 2..9: this CTA's 128 rows; warp w reads
    // TMEM lane quarter w % 4, and takes column half (w - 2) / 4
    const int quarter = warp & 3;
    const int half = (warp - 2) / 4;
    const int row_in_tile = (int)rank * 128 + quarter * 32 + lane;
    const BoxWriter bw{sOut + (warp - 2) * kBoxBytes, (uint32_t)lane};
    if (lane == 0) {
      tma_prefetch_desc(&tmO0);
      tma_prefetch_desc(&tmO1);
    }
    uint64_t *xbar = &ctl->xbar[warp - 2];
    uint32_t xphase = 0;
    bool x_in_flight = false;   // broke out with a residual box load outstanding
    const uint32_t empty_leader0 = map_to_cta(smem_addr(&ctl->tmem_empty[0]), 0);
    const uint32_t empty_leader1 = map_to_cta(smem_addr(&ctl->tmem_empty[1]), 0);
    // NVFP4: this thread expands B row conv_r of every k-block, following the
    // code ring (cs) and the A / B stage ring (stage) in the producer's order
    const int conv_r = (warp - 2) * 32 + lane;
    uint32_t cs = 0, cphase = 0, bstage = 0, bphase = 0;
    int local = 0;
    for (int u = worker; u < num_units; u += num_workers, ++local) {
      const Unit un = unit_of(u, n_full, splits, num_m, num_n, n_fast, num_kb);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if constexpr (EPI == EPI_OUT_RESIDUAL) {
        // the residual does not depend on the accumulator: its first box is
        // loaded while the MMAs of this tile still run
        if (un.slot < 0) {
          bw.begin();
          load_x_box(bw, &tmO0, xbar, un.n_blk * kBN + half * 128, un.m_blk * kTileM + row_in_tile - lane);
        }
      }
      if constexpr (kConv) {
        static_assert(EPI == EPI_IN_PROJ || EPI == EPI_OUT_RESIDUAL, "low-precision weights of the block GEMMs only");
        const int brow = un.n_blk * kBN + conv_r;   // the weight row this thread expands
        // NVFP4: the tensor's float32 scale, by row block (q, k, v, mlp_in) for
        // the in-projection, by input column (attn_out, mlp_out) for the
        // out-projection; fp8r: the row's scale, for the out-projection one per
        // input half (attn_out, mlp_out)
        float g_lo, g_hi;
        const uint32_t *srow = nullptr;
        uint32_t s_cur = 0u, s_nxt = 0u;
        if constexpr (kWFmt == kWNvfp4) {
          srow = reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(ep.w_scales) + (size_t)brow * (K / 16));
          const int gi_q = un.n_blk / (kHidden / kBN);
          g_lo = __ldg(ep.w_globals + (EPI == EPI_IN_PROJ ? (gi_q < 3 ? gi_q : 3) : 4));
          g_hi = EPI == EPI_IN_PROJ ? g_lo : __ldg(ep.w_globals + 5);
          // the row's four block scales of a k-block are one 32-bit word; the
          // words go out two k-blocks ahead of their use
          s_cur = un.kb0 < un.kb1 ? __ldg(srow + un.kb0) : 0u;
          s_nxt = un.kb0 + 1 < un.kb1 ? __ldg(srow + un.kb0 + 1) : 0u;
        } else {
          const float *rs = static_cast<const float *>(ep.w_scales);
          g_lo = __ldg(rs + (EPI == EPI_IN_PROJ ? (size_t)brow : 2 * (size_t)brow));
          g_hi = EPI == EPI_IN_PROJ ? g_lo : __ldg(rs + 2 * (size_t)brow + 1);
        }
        bool conv_ok = true;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          const float g = (EPI == EPI_OUT_RESIDUAL && kb * kBK >= kHidden) ? g_hi : g_lo;
          const uint32_t s4 = s_cur;
          if constexpr (kWFmt == kWNvfp4) {
            s_cur = s_nxt;
            s_nxt = kb + 2 < un.kb1 ? __ldg(srow + kb + 2) : 0u;
          }
          if (!mbar_wait(&ctl->cfull[cs], cphase, abort) || !mbar_wait(&ctl->bempty[bstage], bphase ^ 1, abort)) {
            conv_ok = false;
            break;
          }
          if constexpr (kWFmt == kWNvfp4)
            expand_fp4_row(smC + cs * C::kCodeBytes + conv_r * C::kCodeCols, s4, g, smB + bstage * C::kBBytes, conv_r);
          else
            expand_fp8_row(smC + cs * C::kCodeBytes + conv_r * C::kCodeCols, g, smB + bstage * C::kBBytes, conv_r);
          fence_proxy_async_smem();       // the MMA reads the row through the async proxy
          mbar_arrive(&ctl->bready[bstage]);
          mbar_arrive(&ctl->cempty[cs]);
          if (++cs == kCodeStages) {
            cs = 0;
            cphase ^= 1;
          }
          if (++bstage == kBStages) {
            bstage = 0;
            bphase ^= 1;
          }
        }
        if (!conv_ok) {
          x_in_flight = EPI == EPI_OUT_RESIDUAL && un.slot < 0;
          break;
        }
      }
      if (!mbar_wait(&ctl->tmem_full[acc], acc_phase, abort)) {
        x_in_flight = EPI == EPI_OUT_RESIDUAL && un.slot < 0;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * kBN;
      if (un.slot >= 0) {
        store_partial_half(taddr, un.slot, row_in_tile - lane, M - un.m_blk * kTileM, half, kTileM, bw, &tmO1);
      } else if (!epilogue_half<EPI, !kConv>(taddr, un.m_blk * kTileM + row_in_tile, un.m_blk * kTileM + row_in_tile - lane,
                                     M, un.n_blk, half, ep, bw, &tmO0, &tmO1, xbar, xphase, abort)) {
        x_in_flight = true;   // only the residual box wait can fail
        break;
      }
      tc_fence_before();
      if constexpr (kPair)
        mbar_arrive_cluster_relaxed(acc ? empty_leader1 : empty_leader0);
      else
        mbar_arrive(&ctl->tmem_empty[acc]);
    }
    if (lane == 0) bulk_wait_all();   // this warp's output stores are complete before the CTA exits
    if (x_in_flight && lane == 0) drain_wait(xbar, xphase);   // the box must land before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();   // neither CTA leaves while its pair may still touch its memory
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1, int M, int N,
                int K, int n_full, int splits, EpiParams ep) {
  gemm_body<EPI, true, kWBf16>(tmA, tmB, tmO0, tmO1, M, N, K, n_full, splits, ep);
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm1_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1, int M, int N,
                 int K, int n_full, int splits, EpiParams ep) {
  gemm_body<EPI, false, kWBf16>(tmA, tmB, tmO0, tmO1, M, N, K, n_full, splits, ep);
}

// The one-CTA form over NVFP4 / fp8r weights (tmB: the code bytes).
template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm1_fp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1, int M, int N,
                     int K, int n_full, int splits, EpiParams ep) {
  gemm_body<EPI, false, kWNvfp4>(tmA, tmB, tmO0, tmO1, M, N, K, n_full, splits, ep);
}
template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm1_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1, int M, int N,
                     int K, int n_full, int splits, EpiParams ep) {
  gemm_body<EPI, false, kWFp8r>(tmA, tmB, tmO0, tmO1, M, N, K, n_full, splits, ep);
}

// Sums the split units of each trailing tile in a fixed order (unit 0 first)
// and applies the out-projection's epilogue: x[row, col] += gate[stream(row)]
// [col] * sum.  One thread per 4 columns of a row; tile i of the trailing
// tiles is tile n_full + i of the schedule.
__global__ void split_merge_residual_kernel(const float *__restrict__ part, int tile_m, int n_full, int splits,
                                            int num_m, int num_n, int n_fast, int M, float *__restrict__ x,
                                            const uint8_t *__restrict__ sid, const float *__restrict__ mod) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.y;                                 // trailing tile
  const int r = blockIdx.x * 4 + threadIdx.x / 64;          // row in the tile
  const int c = (threadIdx.x % 64) * 4;                     // column in the tile
  int m_blk, n_blk;
  tile_coords(n_full + i, num_m, num_n, n_fast != 0, m_blk, n_blk);
  const int row = m_blk * tile_m + r;
  if (r >= tile_m || row >= M) return;
  // every partial, x and the gate are loaded before any is used (one round
  // trip, not one per range); the sum runs in range order
  const int col = n_blk * kBN + c;
  float4 *xp = reinterpret_cast<float4 *>(x + (size_t)row * kHidden + col);
  float4 xv = *xp;
  const float4 g = __ldg(reinterpret_cast<const float4 *>(mod + (size_t)sid[row] * kModLen + 2 * kHidden + col));
  float4 p[kMaxSplitK];
#pragma unroll
  for (int ks = 0; ks < kMaxSplitK; ++ks)
    if (ks < splits)
      p[ks] = __ldcs(reinterpret_cast<const float4 *>(part + ((size_t)(i * splits + ks) * tile_m + r) * kBN + c));
  float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int ks = 0; ks < kMaxSplitK; ++ks) {
    if (ks < splits) {
      y.x += p[ks].x;
      y.y += p[ks].y;
      y.z += p[ks].z;
      y.w += p[ks].w;
    }
  }
  xv.x = fmaf(g.x, y.x, xv.x);
  xv.y = fmaf(g.y, y.y, xv.y);
  xv.z = fmaf(g.z, y.z, xv.z);
  xv.w = fmaf(g.w, y.w, xv.w);
  *xp = xv;
}

// ---------------------------------------------------------------- host launchers
// Split plan of a launch over `workers` (CTA pairs or single CTAs) with
// tile_m-row tiles: whole tiles fill complete rounds of the workers; the
// tiles of the last, partial round are split along K into `splits` ranges (a
// divisor of the k-block count leaving at least 16 k-blocks per range) so
// that their units fill that round.  Only the out-projection splits (its
// epilogue is linear in the product, so partial sums merge exactly as a sum);
// no split when the partial buffer is absent or too small, the round is
// full, or no divisor fits.
void split_plan(int EPI, int M, int N, int K, int tile_m, int workers, size_t part_bytes, int &n_full,
                int &splits) {
  const int tiles = ((M + tile_m - 1) / tile_m) * (N / kBN);
  const int num_kb = K / kBK;
  n_full = tiles;
  splits = 1;
  if (EPI != EPI_OUT_RESIDUAL || workers < 2) return;
  const int full = tiles / workers * workers, rem = tiles - full;
  if (rem == 0) return;
  const int cand[6] = {kMaxSplitK, 8, 6, 4, 3, 2};
  for (int S : cand) {
    const int units = rem * S;
    if (num_kb % S != 0 || num_kb / S < 16 || units > workers) continue;
    if ((size_t)units * tile_m * kBN * sizeof(float) > part_bytes) continue;
    n_full = full;
    splits = S;
    return;
  }
}

template <int EPI, bool kPair, int kWFmt = kWBf16>
cudaError_t launch_form(const CUtensorMap &tmA, const CUtensorMap &tmB, int M, int N, int K, const EpiParams &ep,
                        cudaStream_t s, bool pdl) {
  using C = GemmCfg<kPair, kWFmt>;
  auto kernel = [] {
    if constexpr (kWFmt == kWNvfp4)
      return gemm1_fp4_kernel<EPI>;
    else if constexpr (kWFmt == kWFp8r)
      return gemm1_fp8_kernel<EPI>;
    else
      return kPair ? gemm_kernel<EPI> : gemm1_kernel<EPI>;
  }();
  static std::atomic<bool> attr_set[kMaxDevices];
  const cudaError_t e = set_smem_once(kernel, (int)C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  const int tiles = ((M + C::kTileM - 1) / C::kTileM) * (N / kBN);
  const int workers = kPair ? num_sms() / 2 : num_sms();
  int n_full, splits;
  split_plan(EPI, M, N, K, C::kTileM, workers, ep.part ? ep.part_bytes : 0, n_full, splits);
  const int split_units = (tiles - n_full) * splits;
  // output boxes of 32 rows x 64 columns for the bf16 epilogues
  CUtensorMap tmO0 = tmA, tmO1 = tmA;
  if (EPI == EPI_STORE && !make_tmap_bf16(&tmO0, ep.C, (uint64_t)M, (uint64_t)ep.ldc, 32)) return cudaErrorInvalidValue;
  if (EPI == EPI_IN_PROJ && (!make_tmap_bf16(&tmO0, ep.qkv, (uint64_t)M, kQkvCols, 32) ||
                             !make_tmap_bf16(&tmO1, ep.cat, (uint64_t)M, kCatCols, 32)))
    return cudaErrorInvalidValue;
  if (EPI == EPI_OUT_RESIDUAL && !make_tmap_f32_box32(&tmO0, ep.x, (uint64_t)M, kHidden)) return cudaErrorInvalidValue;
  if (EPI == EPI_OUT_RESIDUAL && splits > 1 &&
      !make_tmap_f32_box32(&tmO1, ep.part, (uint64_t)split_units * C::kTileM, kBN))
    return cudaErrorInvalidValue;
  if (EPI == EPI_STORE_F32 && !make_tmap_f32_box32(&tmO0, ep.x, (uint64_t)M, (uint64_t)ep.ldc))
    return cudaErrorInvalidValue;
  const int units = n_full + split_units;
  const int grid = (kPair ? 2 : 1) * (units < workers ? units : workers);
  cudaError_t le = launch_kernel(kernel, dim3(grid), dim3(kThreads), C::kSmemBytes, s, pdl, tmA, tmB, tmO0, tmO1, M,
                                 N, K, n_full, splits, ep);
  if (le != cudaSuccess || splits == 1) return le;
  const int num_m = (M + C::kTileM - 1) / C::kTileM, num_n = N / kBN;
  return launch_kernel(split_merge_residual_kernel, dim3(C::kTileM / 4, tiles - n_full), dim3(256), 0, s, pdl,
                       static_cast<const float *>(ep.part), (int)C::kTileM, n_full, splits, num_m, num_n,
                       M > N ? 1 : 0, M, ep.x, ep.sid, ep.mod);
}

// M <= 128: single CTAs with 128-row tiles (a 256-row pair tile would be
// mostly padding, and twice the workers take the tiles); else CTA pairs.
template <int EPI>
cudaError_t launch_mode(const CUtensorMap &tmA, const CUtensorMap &tmB, int M, int N, int K, const EpiParams &ep,
                        cudaStream_t s, bool pdl) {
  if (M <= GemmCfg<false>::kTileM) return launch_form<EPI, false>(tmA, tmB, M, N, K, ep, s, pdl);
  return launch_form<EPI, true>(tmA, tmB, M, N, K, ep, s, pdl);
}

// Wraps the EPI_IN_PROJ / EPI_OUT_RESIDUAL low-precision forms (the only
// EPIs the expansion in the epilogue warps serves) for the switch below.
template <int EPI>
cudaError_t launch_lowp_mode(int fmt, const CUtensorMap &tmA, const CUtensorMap &tmCodes, int M, int N, int K,
                             const EpiParams &ep, cudaStream_t s, bool pdl) {
  if constexpr (EPI == EPI_IN_PROJ || EPI == EPI_OUT_RESIDUAL) {
    if (fmt == FLUX3_W_NVFP4) return launch_form<EPI, false, kWNvfp4>(tmA, tmCodes, M, N, K, ep, s, pdl);
    if (fmt == FLUX3_W_FP8R) return launch_form<EPI, false, kWFp8r>(tmA, tmCodes, M, N, K, ep, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gemm_detail

cudaError_t launch_gemm(int mode, const CUtensorMap &tmA, const CUtensorMap &tmB, int M, int N, int K,
                        const EpiParams &ep, cudaStream_t s, bool pdl) {
  using namespace gemm_detail;
  switch (mode) {
    case EPI_STORE: return launch_mode<EPI_STORE>(tmA, tmB, M, N, K, ep, s, pdl);
    case EPI_IN_PROJ: return launch_mode<EPI_IN_PROJ>(tmA, tmB, M, N, K, ep, s, pdl);
    case EPI_OUT_RESIDUAL: return launch_mode<EPI_OUT_RESIDUAL>(tmA, tmB, M, N, K, ep, s, pdl);
    case EPI_STORE_F32: return launch_mode<EPI_STORE_F32>(tmA, tmB, M, N, K, ep, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_lowp(int mode, int fmt, const CUtensorMap &tmA, const CUtensorMap &tmCodes, int M, int N,
                             int K, const EpiParams &ep, cudaStream_t s, bool pdl) {
  using namespace gemm_detail;
  if (M < 1 || M > kLowpGemmMaxRows || !ep.w_scales || (fmt == FLUX3_W_NVFP4 && !ep.w_globals))
    return cudaErrorInvalidValue;
  switch (mode) {
    case EPI_IN_PROJ: return launch_lowp_mode<EPI_IN_PROJ>(fmt, tmA, tmCodes, M, N, K, ep, s, pdl);
    case EPI_OUT_RESIDUAL: return launch_lowp_mode<EPI_OUT_RESIDUAL>(fmt, tmA, tmCodes, M, N, K, ep, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace flux3
