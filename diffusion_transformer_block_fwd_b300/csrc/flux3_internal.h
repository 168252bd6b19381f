// Internal launchers shared by the C-ABI layer and the kernel files.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "flux3.h"

namespace flux3 {

// Model constants the kernels are built for (issue #2142 tensor list).
constexpr int kHidden = 3072;
constexpr int kHeads = 24;
constexpr int kHeadDim = 128;
constexpr int kMlp = 9216;
constexpr int kModLen = 3 * kHidden;           // shift | scale | gate
constexpr int kQkvCols = 3 * kHidden;          // q^ | k^ | v
constexpr int kCatCols = kHidden + kMlp;       // attention | SwiGLU  (K of the out-projection)
constexpr int kInRows = 3 * kHidden + 2 * kMlp; // rows of the packed in-projection weight
constexpr int kRopePairs = kHeadDim / 2;       // 64 = 4 axes x 16 pairs

// GEMM tile shape (tcgen05, a CTA pair per 256 x 256 output tile; each CTA
// loads boxes of 128 rows x 64 columns of A and of B).
constexpr int kBM = 128;      // rows of one A box (one CTA's share of the 256-row tile)
constexpr int kBN = 256;      // output columns of a tile
constexpr int kBoxB = 128;    // rows of one B box (one CTA's share of the tile's 256 B rows)
constexpr int kBK = 64;

enum EpiMode : int { EPI_STORE = 0, EPI_IN_PROJ = 1, EPI_OUT_RESIDUAL = 2, EPI_STORE_F32 = 3 };

struct EpiParams {
  // EPI_STORE (bf16 C) and EPI_STORE_F32 (float32 C in x, ldc columns; tile
  // columns at or past ldc are not stored)
  __nv_bfloat16 *C;
  int ldc;
  // EPI_IN_PROJ
  __nv_bfloat16 *qkv;  // [M, 9216]
  __nv_bfloat16 *cat;  // [M, 12288]
  const float *cos_tab, *sin_tab;  // [M, 64]
  const float *qnorm, *knorm;      // [128]
  float eps_rms;
  // EPI_OUT_RESIDUAL
  float *x;             // [M, 3072] (EPI_STORE_F32: the float32 output [M, ldc])
  const uint8_t *sid;   // [M]
  const float *mod;     // [3, 9216]
  // EPI_OUT_RESIDUAL with a K split of the trailing tiles: float32 partial
  // tiles (tile rows x 256 per split unit); null / too small: no split
  float *part;
  size_t part_bytes;
  // Low-precision weights expanded inside the GEMM (launch_gemm_lowp): NVFP4
  // e4m3 block scales [N, K / 16] (4-byte aligned) and the block's float32
  // tensor scales (q, k, v, mlp_in, attn_out, mlp_out); fp8r float32 row scales
  // ([N], or [N][2] (attn_out, mlp_out) for the out-projection), no w_globals
  const void *w_scales;
  const float *w_globals;
};

// Size of the split partial buffer: 96 partial tiles of the CTA-pair form
// (256 x 256 float32, 256 KB each), or 192 of the one-CTA form.
constexpr int kMaxSplitUnits = 96;
constexpr size_t kSplitUnitBytes = 256 * 256 * 4;
constexpr size_t kSplitBytes = kMaxSplitUnits * kSplitUnitBytes;
static_assert(kSplitBytes == FLUX3_SPLIT_BYTES, "split scratch size of the header");

// Encodes a 2-D bf16 tensor map over a row-major [rows, cols] matrix with a
// {64 cols, box_rows} box and 128-byte swizzle.  Returns false on failure.
bool make_tmap_bf16(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// Encodes a 2-D uint8 tensor map over a row-major [rows, cols] byte matrix
// with a {box_cols, box_rows} box and no swizzle.  Returns false on failure.
bool make_tmap_u8(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                  uint32_t box_rows);

// Encodes a 2-D float32 tensor map over a row-major [rows, cols] matrix with a
// {32 cols, 32 rows} box and 128-byte swizzle.  Returns false on failure.
bool make_tmap_f32_box32(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols);

// Multiprocessor count of the current device.
int num_sms();

// The current device as an index into per-device state, or -1 when it has
// none (no current device, or an ordinal past kMaxDevices: the state is then
// set up on every call).  Function attributes and device properties belong to
// a device's context, so a process that drives several GPUs sets them up on
// each.
constexpr int kMaxDevices = 64;
int device_slot();

// Sets a kernel's dynamic shared-memory limit once per device.
template <typename Kernel>
cudaError_t set_smem_once(Kernel kernel, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  const int slot = device_slot();
  if (slot >= 0 && done[slot].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && slot >= 0) done[slot].store(true, std::memory_order_release);
  return e;
}

// Launches `kernel` on stream s.  With pdl, as a programmatic dependent launch
// of the previous kernel on s: the kernel may be scheduled while that one
// finishes (its CTAs set up, then wait in griddep_wait), which hides the
// launch gap between the kernels of a block.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

cudaError_t launch_gemm(int mode, const CUtensorMap &tmA, const CUtensorMap &tmB, int M, int N, int K,
                        const EpiParams &ep, cudaStream_t s, bool pdl = false);

// The block GEMMs (EPI_IN_PROJ, EPI_OUT_RESIDUAL) over NVFP4 or fp8r weights
// (fmt: FLUX3_W_NVFP4 / FLUX3_W_FP8R) for M <= kLowpGemmMaxRows (one-CTA
// tiles): tmCodes maps the code bytes (make_tmap_u8 with 256-row boxes of 32
// bytes for the e2m1 codes [N, K / 2], 64 bytes for the e4m3 codes [N, K]);
// ep.w_scales / ep.w_globals hold the scales.  The weights are expanded to
// bf16 in shared memory, never in HBM.
constexpr int kLowpGemmMaxRows = 128;
cudaError_t launch_gemm_lowp(int mode, int fmt, const CUtensorMap &tmA, const CUtensorMap &tmCodes, int M, int N,
                             int K, const EpiParams &ep, cudaStream_t s, bool pdl = false);

cudaError_t launch_stream_ids(const flux3_segment *segs, int n_segs, int T, uint8_t *sid, cudaStream_t s);
cudaError_t launch_rope_tables(const float *pos, int T, float theta, float *cos_tab, float *sin_tab,
                               cudaStream_t s);
// Stream ids and RoPE tables in one launch (the per-call preparation).
cudaError_t launch_prepare(const flux3_segment *segs, int n_segs, int T, uint8_t *sid, const float *pos, float theta,
                           float *cos_tab, float *sin_tab, cudaStream_t s);
// early_release (with pdl): the next kernel may be scheduled before this one's
// programmatic-dependent wait; only where that kernel reads nothing before its
// own wait that a still-running kernel writes.
cudaError_t launch_ln_modulate(const float *x, int T, const uint8_t *sid, const float *mod, float eps,
                               __nv_bfloat16 *h, cudaStream_t s, bool pdl = false, bool early_release = false);
cudaError_t launch_selftest_wait(unsigned long long timeout_ns, cudaStream_t s);
// part / part_bytes: scratch for the key-range split of the last, partial
// wave of units (null: no split).
cudaError_t launch_attention(const __nv_bfloat16 *qkv, int T, __nv_bfloat16 *cat, cudaStream_t s, bool pdl = false,
                             float *part = nullptr, size_t part_bytes = 0);

}  // namespace flux3
