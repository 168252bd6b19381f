// C ABI of the library (include/flux3.h): argument validation, weight
// packing, workspace carving, tensor-map set-up and the per-block launch
// sequence.  The kernels are compiled in this one translation unit.

#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "flux3_internal.h"
#include "ptx.cuh"

#include "attention.cuh"
#include "elementwise.cuh"
#include "gemm.cuh"
#include "nvfp4.cuh"
#include "fp8r.cuh"
#include "cond.cuh"

struct flux3_handle {
  flux3_config cfg;
  int n_blocks;
  const __nv_bfloat16 *w_in;   // bf16: [n_blocks][kInRows, kHidden]
  const __nv_bfloat16 *w_out;  // bf16: [n_blocks][kHidden, kCatCols]
  const float *norms;          // [n_blocks][2][kHeadDim]
  std::vector<CUtensorMap> tm_in, tm_out;               // bf16 only
  std::vector<flux3::fp4_detail::Fp4BlockView> fp4;    // NVFP4 only
  std::vector<flux3::fp8r_detail::Fp8rBlockView> fp8;  // fp8r only
};

// The non-block weights, copied into the caller's packed buffer.
struct flux3_cond {
  bool flow;                                            // ref_time_in present
  const __nv_bfloat16 *time_in_in, *time_in_out, *ref_in, *ref_out;
  const __nv_bfloat16 *early[3], *single[3], *final_adaln;
  CUtensorMap tm_emb[3];     // B operands of the embedders, by stream: emb_in.image, emb_in.image_cond, txt_in
  CUtensorMap tm_final;      // final_linear zero-padded to 256 rows (one N tile)
};

namespace flux3 {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

constexpr size_t kWInElems = (size_t)kInRows * kHidden;
constexpr size_t kWOutElems = (size_t)kHidden * kCatCols;
constexpr int kMaxTokensLimit = 65536;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool config_ok(const flux3_config *c) {
  return c && c->hidden == kHidden && c->heads == kHeads && c->head_dim == kHeadDim && c->mlp_hidden == kMlp &&
         c->n_blocks >= 1 && c->max_tokens >= 1 && c->max_tokens <= kMaxTokensLimit &&
         (c->wfmt == FLUX3_W_BF16 || c->wfmt == FLUX3_W_NVFP4 || c->wfmt == FLUX3_W_FP8R) &&
         c->rope_theta > 0.f && c->eps_ln > 0.f && c->eps_rms > 0.f;
}

// Bytes of the workspace for T tokens (each sub-buffer rounded up to 256 B);
// the order and sizes match workspace_layout below.
constexpr size_t ws_round(size_t v) { return (v + 255) / 256 * 256; }
// The out-projection's split partials reuse h and qkv (both dead once
// attention has run) when those hold kSplitBytes; below that size of T they
// get a region of their own.
constexpr bool split_in_place(size_t T) {
  return ws_round(T * kHidden * 2) + ws_round(T * kQkvCols * 2) >= kSplitBytes;
}
constexpr size_t workspace_total(size_t T) {
  return ws_round(T) + 2 * ws_round(T * kRopePairs * 4) + ws_round(T * kHidden * 2) + ws_round(T * kQkvCols * 2) +
         ws_round(T * kCatCols * 2) + (split_in_place(T) ? 0 : kSplitBytes);
}

// NVFP4 packed block: in-projection codes and scales, out-projection codes and
// scales, the six global scales.
constexpr size_t kFp4InCodes = (size_t)kInRows * kHidden / 2;
constexpr size_t kFp4InScales = (size_t)kInRows * kHidden / 16;
constexpr size_t kFp4OutCodes = (size_t)kHidden * kCatCols / 2;
constexpr size_t kFp4OutScales = (size_t)kHidden * kCatCols / 16;
constexpr size_t kFp4BlockBytes =
    ws_round(kFp4InCodes) + ws_round(kFp4InScales) + ws_round(kFp4OutCodes) + ws_round(kFp4OutScales) + 256;

// fp8r packed block: in-projection codes and row scales, out-projection codes
// and its two scales per row (attn_out's, mlp_out's).
constexpr size_t kFp8InCodes = (size_t)kInRows * kHidden;
constexpr size_t kFp8InScales = (size_t)kInRows * 4;
constexpr size_t kFp8OutCodes = (size_t)kHidden * kCatCols;
constexpr size_t kFp8OutScales = (size_t)kHidden * 2 * 4;
constexpr size_t kFp8BlockBytes =
    ws_round(kFp8InCodes) + ws_round(kFp8InScales) + ws_round(kFp8OutCodes) + ws_round(kFp8OutScales);

// Weights stored below bf16 are expanded to bf16 in the workspace, one block at a time.
bool lowp(int wfmt) { return wfmt == FLUX3_W_NVFP4 || wfmt == FLUX3_W_FP8R; }

struct Workspace {
  uint8_t *sid;
  float *cos_tab, *sin_tab;
  __nv_bfloat16 *h, *qkv, *cat;
  float *part;                   // the out-projection's split partials (kSplitBytes)
  __nv_bfloat16 *w_in, *w_out;   // NVFP4 / fp8r handles: the running block's weights in bf16
};

size_t workspace_layout(int T, uint8_t *base, Workspace *ws, bool fp4_weights = false) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return base ? base + o : nullptr;
  };
  uint8_t *sid = take((size_t)T);
  uint8_t *cs = take((size_t)T * kRopePairs * 4);
  uint8_t *sn = take((size_t)T * kRopePairs * 4);
  uint8_t *h = take((size_t)T * kHidden * 2);
  uint8_t *qkv = take((size_t)T * kQkvCols * 2);
  uint8_t *cat = take((size_t)T * kCatCols * 2);
  uint8_t *part = split_in_place((size_t)T) ? h : take(kSplitBytes);
  uint8_t *w_in = fp4_weights ? take(kWInElems * 2) : nullptr;
  uint8_t *w_out = fp4_weights ? take(kWOutElems * 2) : nullptr;
  if (ws) {
    ws->sid = sid;
    ws->cos_tab = reinterpret_cast<float *>(cs);
    ws->sin_tab = reinterpret_cast<float *>(sn);
    ws->h = reinterpret_cast<__nv_bfloat16 *>(h);
    ws->qkv = reinterpret_cast<__nv_bfloat16 *>(qkv);
    ws->cat = reinterpret_cast<__nv_bfloat16 *>(cat);
    ws->part = reinterpret_cast<float *>(part);
    ws->w_in = reinterpret_cast<__nv_bfloat16 *>(w_in);
    ws->w_out = reinterpret_cast<__nv_bfloat16 *>(w_out);
  }
  return off;
}

flux3_status segments_ok(const flux3_segment *segs, int n_segs, int T) {
  if (!segs || n_segs < 1 || n_segs > FLUX3_MAX_SEGMENTS || T < 1) return FLUX3_ERR_INVALID_ARG;
  int expect = 0;
  for (int i = 0; i < n_segs; ++i) {
    if (segs[i].start != expect || segs[i].len < 1 || segs[i].stream < 0 || segs[i].stream > 2)
      return FLUX3_ERR_INVALID_ARG;
    expect += segs[i].len;
    if (expect > T) return FLUX3_ERR_INVALID_ARG;
  }
  return expect == T ? FLUX3_OK : FLUX3_ERR_INVALID_ARG;
}

flux3_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FLUX3_OK : FLUX3_ERR_CUDA; }

#define F3_TRY(expr)                         \
  do {                                       \
    flux3_status _st = (expr);               \
    if (_st != FLUX3_OK) return _st;         \
  } while (0)
#define F3_CUDA(expr) F3_TRY(cuda_status(expr))

const float *block_norms(const flux3_handle *h, int b) { return h->norms + (size_t)b * 2 * kHeadDim; }

flux3_status run_in_projection(const flux3_handle *h, int b, const __nv_bfloat16 *hmod, int T, const float *cos_tab,
                               const float *sin_tab, __nv_bfloat16 *qkv, __nv_bfloat16 *cat, cudaStream_t s) {
  CUtensorMap tmA;
  if (!make_tmap_bf16(&tmA, hmod, (uint64_t)T, kHidden, kBM)) return FLUX3_ERR_CUDA;
  EpiParams ep{};
  ep.qkv = qkv;
  ep.cat = cat;
  ep.cos_tab = cos_tab;
  ep.sin_tab = sin_tab;
  ep.qnorm = block_norms(h, b);
  ep.knorm = block_norms(h, b) + kHeadDim;
  ep.eps_rms = h->cfg.eps_rms;
  return cuda_status(launch_gemm(EPI_IN_PROJ, tmA, h->tm_in[b], T, kInRows, kHidden, ep, s));
}

flux3_status run_out_projection(const flux3_handle *h, int b, const __nv_bfloat16 *cat, int T, const uint8_t *sid,
                                const float *mod, float *x, float *part, size_t part_bytes, cudaStream_t s) {
  CUtensorMap tmA;
  if (!make_tmap_bf16(&tmA, cat, (uint64_t)T, kCatCols, kBM)) return FLUX3_ERR_CUDA;
  EpiParams ep{};
  ep.x = x;
  ep.sid = sid;
  ep.mod = mod;
  ep.part = part;
  ep.part_bytes = part_bytes;
  return cuda_status(launch_gemm(EPI_OUT_RESIDUAL, tmA, h->tm_out[b], T, kHidden, kCatCols, ep, s));
}

// Sample boundaries of a batched call: 0 = start[0] < ... < start[n] = T,
// n <= FLUX3_MAX_SAMPLES, every segment inside one sample.  sample_of[i] is
// segment i's sample.
flux3_status samples_ok(const int *start, int n, int T, const flux3_segment *segs, int n_segs, int *sample_of) {
  if (!start || n < 1 || n > FLUX3_MAX_SAMPLES || start[0] != 0 || start[n] != T) return FLUX3_ERR_INVALID_ARG;
  for (int b = 0; b < n; ++b)
    if (start[b + 1] <= start[b]) return FLUX3_ERR_INVALID_ARG;
  for (int i = 0; i < n_segs; ++i) {
    int b = 0;
    while (b < n && segs[i].start >= start[b + 1]) ++b;
    if (b == n || segs[i].start + segs[i].len > start[b + 1]) return FLUX3_ERR_INVALID_ARG;
    sample_of[i] = b;
  }
  return FLUX3_OK;
}

// The blocks over one sample, or over a batch of samples (sample_start /
// n_samples): LayerNorm and both GEMMs over all rows, attention per sample,
// the modulation row of a token = 3 * sample + stream.
flux3_status forward_common(const flux3_handle *h, int first, int count, float *x, int T, const flux3_segment *segs,
                            int n_segs, const float *pos, const float *mod, void *workspace, size_t ws_bytes,
                            cudaStream_t s, const int *sample_start = nullptr, int n_samples = 1) {
  if (!h || !x || !pos || !mod || !workspace) return FLUX3_ERR_INVALID_ARG;
  if (first < 0 || count < 1 || first + count > h->n_blocks) return FLUX3_ERR_INVALID_ARG;
  if (T < 1 || T > h->cfg.max_tokens) return FLUX3_ERR_INVALID_ARG;
  F3_TRY(segments_ok(segs, n_segs, T));
  const int one_sample[2] = {0, T};
  int sample_of[FLUX3_MAX_SEGMENTS] = {0};
  if (sample_start) {
    F3_TRY(samples_ok(sample_start, n_samples, T, segs, n_segs, sample_of));
  } else {
    sample_start = one_sample;
    n_samples = 1;
  }
  flux3_segment rows[FLUX3_MAX_SEGMENTS];      // segments with the modulation row as their stream
  for (int i = 0; i < n_segs; ++i) {
    rows[i] = segs[i];
    rows[i].stream = 3 * sample_of[i] + segs[i].stream;
  }
  if (!aligned16(x) || !aligned16(pos) || !aligned16(mod) || !aligned16(workspace)) return FLUX3_ERR_ALIGNMENT;
  const bool fp4 = lowp(h->cfg.wfmt);
  Workspace ws;
  if (ws_bytes < workspace_layout(T, nullptr, nullptr, fp4)) return FLUX3_ERR_WORKSPACE;
  workspace_layout(T, static_cast<uint8_t *>(workspace), &ws, fp4);

  // the first launch waits for everything before it on the stream; each later
  // one is a programmatic dependent of the kernel before it (its set-up runs
  // while that kernel finishes)
  F3_CUDA(launch_prepare(rows, n_segs, T, ws.sid, pos, h->cfg.rope_theta, ws.cos_tab, ws.sin_tab, s));
  CUtensorMap tmH, tmCat, tmWin, tmWout;
  if (!make_tmap_bf16(&tmH, ws.h, (uint64_t)T, kHidden, kBM)) return FLUX3_ERR_CUDA;
  if (!make_tmap_bf16(&tmCat, ws.cat, (uint64_t)T, kCatCols, kBM)) return FLUX3_ERR_CUDA;
  if (fp4 && (!make_tmap_bf16(&tmWin, ws.w_in, kInRows, kHidden, kBoxB) ||
              !make_tmap_bf16(&tmWout, ws.w_out, kHidden, kCatCols, kBoxB)))
    return FLUX3_ERR_CUDA;
  // attention's key-range partials may use only memory that is dead while it
  // runs: h when the split region lies over h and qkv (attention reads qkv)
  const size_t attn_part_bytes = split_in_place((size_t)T) ? ws_round((size_t)T * kHidden * 2) : kSplitBytes;
  // NVFP4 / fp8r at small T: the GEMMs read the codes and expand them in
  // shared memory (the weight stream bounds them there); otherwise the block's
  // weights are expanded to bf16 in the workspace first
  const bool lowp_in_gemm = fp4 && T <= kLowpGemmMaxRows;
  const bool nv = h->cfg.wfmt == FLUX3_W_NVFP4;
  for (int b = first; b < first + count; ++b) {
    CUtensorMap tmCin, tmCout;
    const void *in_scales = nullptr, *out_scales = nullptr;
    const float *globals = nullptr;
    if (lowp_in_gemm) {
      const uint8_t *in_codes = nv ? h->fp4[b].in_codes : h->fp8[b].in_codes;
      const uint8_t *out_codes = nv ? h->fp4[b].out_codes : h->fp8[b].out_codes;
      const uint32_t cols = nv ? kBK / 2 : kBK;   // code bytes per row of a k-block
      if (!make_tmap_u8(&tmCin, in_codes, kInRows, (uint64_t)kHidden * cols / kBK, cols, 256) ||
          !make_tmap_u8(&tmCout, out_codes, kHidden, (uint64_t)kCatCols * cols / kBK, cols, 256))
        return FLUX3_ERR_CUDA;
      in_scales = nv ? static_cast<const void *>(h->fp4[b].in_scales) : static_cast<const void *>(h->fp8[b].in_scales);
      out_scales = nv ? static_cast<const void *>(h->fp4[b].out_scales) : static_cast<const void *>(h->fp8[b].out_scales);
      globals = nv ? h->fp4[b].globals : nullptr;
    } else if (nv) {
      F3_CUDA(launch_dequantize_block(h->fp4[b], ws.w_in, ws.w_out, s, true));
    } else if (h->cfg.wfmt == FLUX3_W_FP8R) {
      F3_CUDA(launch_dequantize_fp8r_block(h->fp8[b], ws.w_in, ws.w_out, s, true));
    }
    // LayerNorm releases the in-projection before its own wait unless this
    // block's weights were just expanded in HBM (the in-projection loads its
    // first weight stages before its wait)
    F3_CUDA(launch_ln_modulate(x, T, ws.sid, mod, h->cfg.eps_ln, ws.h, s, true, !fp4 || lowp_in_gemm));
    EpiParams ep{};
    ep.qkv = ws.qkv;
    ep.cat = ws.cat;
    ep.cos_tab = ws.cos_tab;
    ep.sin_tab = ws.sin_tab;
    ep.qnorm = block_norms(h, b);
    ep.knorm = block_norms(h, b) + kHeadDim;
    ep.eps_rms = h->cfg.eps_rms;
    if (lowp_in_gemm) {
      ep.w_scales = in_scales;
      ep.w_globals = globals;
      F3_CUDA(launch_gemm_lowp(EPI_IN_PROJ, h->cfg.wfmt, tmH, tmCin, T, kInRows, kHidden, ep, s, true));
    } else {
      F3_CUDA(launch_gemm(EPI_IN_PROJ, tmH, fp4 ? tmWin : h->tm_in[b], T, kInRows, kHidden, ep, s, true));
    }
    for (int smp = 0; smp < n_samples; ++smp) {   // attention within each sample
      const int r0 = sample_start[smp];
      F3_CUDA(launch_attention(ws.qkv + (size_t)r0 * kQkvCols, sample_start[smp + 1] - r0,
                               ws.cat + (size_t)r0 * kCatCols, s, true, ws.part, attn_part_bytes));
    }
    EpiParams eo{};
    eo.x = x;
    eo.sid = ws.sid;
    eo.mod = mod;
    eo.part = ws.part;
    eo.part_bytes = kSplitBytes;
    if (lowp_in_gemm) {
      eo.w_scales = out_scales;
      eo.w_globals = globals;
      F3_CUDA(launch_gemm_lowp(EPI_OUT_RESIDUAL, h->cfg.wfmt, tmCat, tmCout, T, kHidden, kCatCols, eo, s, true));
    } else {
      F3_CUDA(launch_gemm(EPI_OUT_RESIDUAL, tmCat, fp4 ? tmWout : h->tm_out[b], T, kHidden, kCatCols, eo, s, true));
    }
  }
  return FLUX3_OK;
}

// ---------------------------------------------------------------------------
// Scratch for flux3_block_forward_noalloc: a file-scope device array sized for
// FLUX3_NOALLOC_MAX_TOKENS tokens.  Every device that loads the library holds
// it until the process exits.  Host code only ever sees a host-side stand-in
// for the symbol, so the device address is looked up with cudaGetSymbolAddress
// in the current context.  The lookup runs on every call rather than being
// cached: the address belongs to a CUDA context, and a context can be replaced
// on the same device ordinal (cudaDeviceReset, or a host that drives the call
// under a context of its own).  Once the module is loaded the lookup is a
// host-side query that allocates nothing.
constexpr size_t kNoAllocScratchBytes = workspace_total(FLUX3_NOALLOC_MAX_TOKENS);
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context, or nullptr.
void *noalloc_scratch() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
  return p;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !aligned16(base) || (cols * 2) % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_u8(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                  uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !aligned16(base) || cols % 16 != 0 || box_cols % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_f32_box32(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !aligned16(base) || (cols * 4) % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_slot() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int num_sms() {
  static std::atomic<int> n[kMaxDevices];
  const int slot = device_slot();
  int v = slot >= 0 ? n[slot].load(std::memory_order_relaxed) : 0;
  if (v == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (v <= 0) v = 1;
    if (slot >= 0) n[slot].store(v, std::memory_order_relaxed);
  }
  return v;
}

}  // namespace flux3

using namespace flux3;

extern "C" {

void flux3_default_config(flux3_config *cfg) {
  if (!cfg) return;
  cfg->hidden = kHidden;
  cfg->heads = kHeads;
  cfg->head_dim = kHeadDim;
  cfg->mlp_hidden = kMlp;
  cfg->n_blocks = 28;
  cfg->max_tokens = 16384;
  cfg->wfmt = FLUX3_W_BF16;
  cfg->rope_theta = 10000.0f;
  cfg->eps_ln = 1e-6f;
  cfg->eps_rms = 1e-6f;
}

size_t flux3_packed_weight_bytes(const flux3_config *cfg) {
  if (!config_ok(cfg)) return 0;
  const size_t per_block = cfg->wfmt == FLUX3_W_NVFP4  ? kFp4BlockBytes
                           : cfg->wfmt == FLUX3_W_FP8R ? kFp8BlockBytes
                                                        : align_up(kWInElems * 2) + align_up(kWOutElems * 2);
  return (size_t)cfg->n_blocks * (per_block + align_up(2 * kHeadDim * 4));
}

size_t flux3_workspace_bytes(const flux3_config *cfg, int T) {
  if (!config_ok(cfg) || T < 1 || T > cfg->max_tokens) return 0;
  return workspace_layout(T, nullptr, nullptr, lowp(cfg->wfmt));
}

flux3_status flux3_block_init(flux3_handle **out, const flux3_config *cfg, const flux3_block_weights *w, int n_blocks,
                              void *packed, size_t packed_bytes, void *stream) {
  if (!out) return FLUX3_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w || !packed) return FLUX3_ERR_INVALID_ARG;
  if (cfg->wfmt != FLUX3_W_BF16) return FLUX3_ERR_INVALID_ARG;   // NVFP4 / fp8r: their own init
  if (!config_ok(cfg)) return FLUX3_ERR_UNSUPPORTED;
  if (n_blocks != cfg->n_blocks) return FLUX3_ERR_INVALID_ARG;
  if (packed_bytes < flux3_packed_weight_bytes(cfg)) return FLUX3_ERR_WORKSPACE;
  if (!aligned16(packed)) return FLUX3_ERR_ALIGNMENT;
  for (int b = 0; b < n_blocks; ++b) {
    const flux3_block_weights &bw = w[b];
    const void *ps[8] = {bw.q_proj, bw.k_proj, bw.v_proj, bw.attn_out, bw.mlp_in, bw.mlp_out, bw.query_norm, bw.key_norm};
    for (const void *p : ps) {
      if (!p) return FLUX3_ERR_INVALID_ARG;
      if (!aligned16(p)) return FLUX3_ERR_ALIGNMENT;
    }
  }
  if (!encode_fn()) return FLUX3_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  flux3_handle *h = new (std::nothrow) flux3_handle();
  if (!h) return FLUX3_ERR_CUDA;
  h->cfg = *cfg;
  h->n_blocks = n_blocks;
  uint8_t *base = static_cast<uint8_t *>(packed);
  const size_t in_bytes = align_up(kWInElems * 2), out_bytes = align_up(kWOutElems * 2);
  auto *w_in = reinterpret_cast<__nv_bfloat16 *>(base);
  auto *w_out = reinterpret_cast<__nv_bfloat16 *>(base + n_blocks * in_bytes);
  auto *norms = reinterpret_cast<float *>(base + n_blocks * (in_bytes + out_bytes));
  h->w_in = w_in;
  h->w_out = w_out;
  h->norms = norms;
  h->tm_in.resize(n_blocks);
  h->tm_out.resize(n_blocks);

  const size_t row = (size_t)kHidden * 2;  // bytes of one [*, 3072] row
  cudaError_t e = cudaSuccess;
  for (int b = 0; b < n_blocks && e == cudaSuccess; ++b) {
    const flux3_block_weights &bw = w[b];
    uint8_t *win = reinterpret_cast<uint8_t *>(w_in) + b * in_bytes;
    uint8_t *wout = reinterpret_cast<uint8_t *>(w_out) + b * out_bytes;
    // in-projection rows: q | k | v | mlp_in with a and b interleaved in groups of 128
    e = cudaMemcpyAsync(win, bw.q_proj, kHidden * row, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(win + kHidden * row, bw.k_proj, kHidden * row, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(win + 2 * kHidden * row, bw.v_proj, kHidden * row, cudaMemcpyDeviceToDevice, s);
    const uint8_t *mi = static_cast<const uint8_t *>(bw.mlp_in);
    uint8_t *wm = win + 3 * kHidden * row;
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(wm, 256 * row, mi, 128 * row, 128 * row, kMlp / 128, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(wm + 128 * row, 256 * row, mi + kMlp * row, 128 * row, 128 * row, kMlp / 128,
                            cudaMemcpyDeviceToDevice, s);
    // out-projection: [attn_out | mlp_out] concatenated along the input dimension
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(wout, kCatCols * 2, bw.attn_out, kHidden * 2, kHidden * 2, kHidden,
                            cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(wout + kHidden * 2, kCatCols * 2, bw.mlp_out, kMlp * 2, kMlp * 2, kHidden,
                            cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(norms + (size_t)b * 2 * kHeadDim, bw.query_norm, kHeadDim * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(norms + (size_t)b * 2 * kHeadDim + kHeadDim, bw.key_norm, kHeadDim * 4,
                          cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && (!make_tmap_bf16(&h->tm_in[b], win, kInRows, kHidden, kBoxB) ||
                             !make_tmap_bf16(&h->tm_out[b], wout, kHidden, kCatCols, kBoxB)))
      e = cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) {
    delete h;
    return FLUX3_ERR_CUDA;
  }
  *out = h;
  return FLUX3_OK;
}

flux3_status flux3_block_init_nvfp4(flux3_handle **out, const flux3_config *cfg, const flux3_block_weights_nvfp4 *w,
                                    int n_blocks, void *packed, size_t packed_bytes, void *stream) {
  if (!out) return FLUX3_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w || !packed) return FLUX3_ERR_INVALID_ARG;
  if (cfg->wfmt != FLUX3_W_NVFP4) return FLUX3_ERR_INVALID_ARG;
  if (!config_ok(cfg)) return FLUX3_ERR_UNSUPPORTED;
  if (n_blocks != cfg->n_blocks) return FLUX3_ERR_INVALID_ARG;
  if (packed_bytes < flux3_packed_weight_bytes(cfg)) return FLUX3_ERR_WORKSPACE;
  if (!aligned16(packed)) return FLUX3_ERR_ALIGNMENT;
  for (int b = 0; b < n_blocks; ++b) {
    const flux3_block_weights_nvfp4 &bw = w[b];
    const flux3_nvfp4_tensor *ts[6] = {&bw.q_proj, &bw.k_proj, &bw.v_proj, &bw.attn_out, &bw.mlp_in, &bw.mlp_out};
    for (const flux3_nvfp4_tensor *t : ts) {
      if (!t->codes || !t->scales || !t->global_scale) return FLUX3_ERR_INVALID_ARG;
      if (!aligned16(t->codes) || !aligned16(t->scales) || (reinterpret_cast<uintptr_t>(t->global_scale) & 3u))
        return FLUX3_ERR_ALIGNMENT;
    }
    if (!bw.query_norm || !bw.key_norm) return FLUX3_ERR_INVALID_ARG;
    if (!aligned16(bw.query_norm) || !aligned16(bw.key_norm)) return FLUX3_ERR_ALIGNMENT;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  flux3_handle *h = new (std::nothrow) flux3_handle();
  if (!h) return FLUX3_ERR_CUDA;
  h->cfg = *cfg;
  h->n_blocks = n_blocks;
  h->w_in = h->w_out = nullptr;
  uint8_t *base = static_cast<uint8_t *>(packed);
  auto *norms = reinterpret_cast<float *>(base + n_blocks * kFp4BlockBytes);
  h->norms = norms;
  h->fp4.resize(n_blocks);

  constexpr size_t in_row = kHidden / 2, in_srow = kHidden / 16;     // bytes per row: codes, scales
  constexpr size_t out_row = kCatCols / 2, out_srow = kCatCols / 16;
  constexpr size_t mlp_row = kMlp / 2, mlp_srow = kMlp / 16;          // mlp_out rows (9216 inputs)
  cudaError_t e = cudaSuccess;
  auto copy = [&](void *dst, const void *src, size_t bytes) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
  };
  auto copy2d = [&](void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, size_t height) {
    if (e == cudaSuccess) e = cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, cudaMemcpyDeviceToDevice, s);
  };
  for (int b = 0; b < n_blocks && e == cudaSuccess; ++b) {
    const flux3_block_weights_nvfp4 &bw = w[b];
    uint8_t *blk = base + b * kFp4BlockBytes;
    uint8_t *in_c = blk;
    uint8_t *in_s = in_c + ws_round(kFp4InCodes);
    uint8_t *out_c = in_s + ws_round(kFp4InScales);
    uint8_t *out_s = out_c + ws_round(kFp4OutCodes);
    float *globals = reinterpret_cast<float *>(out_s + ws_round(kFp4OutScales));
    // in-projection rows q | k | v | mlp_in (a and b interleaved in groups of 128), codes and scales alike
    const flux3_nvfp4_tensor *qkv[3] = {&bw.q_proj, &bw.k_proj, &bw.v_proj};
    for (int i = 0; i < 3; ++i) {
      copy(in_c + (size_t)i * kHidden * in_row, qkv[i]->codes, kHidden * in_row);
      copy(in_s + (size_t)i * kHidden * in_srow, qkv[i]->scales, kHidden * in_srow);
    }
    const uint8_t *mc = static_cast<const uint8_t *>(bw.mlp_in.codes);
    const uint8_t *ms = static_cast<const uint8_t *>(bw.mlp_in.scales);
    uint8_t *wc = in_c + 3 * kHidden * in_row, *wsc = in_s + 3 * kHidden * in_srow;
    copy2d(wc, 256 * in_row, mc, 128 * in_row, 128 * in_row, kMlp / 128);
    copy2d(wc + 128 * in_row, 256 * in_row, mc + kMlp * in_row, 128 * in_row, 128 * in_row, kMlp / 128);
    copy2d(wsc, 256 * in_srow, ms, 128 * in_srow, 128 * in_srow, kMlp / 128);
    copy2d(wsc + 128 * in_srow, 256 * in_srow, ms + kMlp * in_srow, 128 * in_srow, 128 * in_srow, kMlp / 128);
    // out-projection rows: attn_out's inputs then mlp_out's
    copy2d(out_c, out_row, bw.attn_out.codes, in_row, in_row, kHidden);
    copy2d(out_c + in_row, out_row, bw.mlp_out.codes, mlp_row, mlp_row, kHidden);
    copy2d(out_s, out_srow, bw.attn_out.scales, in_srow, in_srow, kHidden);
    copy2d(out_s + in_srow, out_srow, bw.mlp_out.scales, mlp_srow, mlp_srow, kHidden);
    const float *gsrc[6] = {bw.q_proj.global_scale, bw.k_proj.global_scale, bw.v_proj.global_scale,
                            bw.mlp_in.global_scale, bw.attn_out.global_scale, bw.mlp_out.global_scale};
    for (int i = 0; i < 6; ++i) copy(globals + i, gsrc[i], sizeof(float));
    copy(norms + (size_t)b * 2 * kHeadDim, bw.query_norm, kHeadDim * 4);
    copy(norms + (size_t)b * 2 * kHeadDim + kHeadDim, bw.key_norm, kHeadDim * 4);
    h->fp4[b] = fp4_detail::Fp4BlockView{in_c, in_s, out_c, out_s, globals};
  }
  if (e != cudaSuccess) {
    delete h;
    return FLUX3_ERR_CUDA;
  }
  *out = h;
  return FLUX3_OK;
}

flux3_status flux3_quantize_nvfp4(const void *w, int rows, int cols, void *codes, void *scales, float *global_scale,
                                  void *stream) {
  if (!w || !codes || !scales || !global_scale || rows < 1 || cols < 16 || cols % 16 != 0)
    return FLUX3_ERR_INVALID_ARG;
  if ((size_t)rows * (size_t)cols > (size_t)1 << 34) return FLUX3_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return FLUX3_ERR_ALIGNMENT;
  return cuda_status(launch_quantize_nvfp4(static_cast<const __nv_bfloat16 *>(w), rows, cols,
                                           static_cast<uint8_t *>(codes), static_cast<uint8_t *>(scales),
                                           global_scale, static_cast<cudaStream_t>(stream)));
}

flux3_status flux3_dequantize_block(const flux3_handle *h, int block_idx, void *w_in, void *w_out, void *stream) {
  if (!h || !w_in || !w_out || block_idx < 0 || block_idx >= h->n_blocks) return FLUX3_ERR_INVALID_ARG;
  if (!lowp(h->cfg.wfmt)) return FLUX3_ERR_UNSUPPORTED;
  if (!aligned16(w_in) || !aligned16(w_out)) return FLUX3_ERR_ALIGNMENT;
  auto *wi = static_cast<__nv_bfloat16 *>(w_in);
  auto *wo = static_cast<__nv_bfloat16 *>(w_out);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(h->cfg.wfmt == FLUX3_W_NVFP4 ? launch_dequantize_block(h->fp4[block_idx], wi, wo, s)
                                                   : launch_dequantize_fp8r_block(h->fp8[block_idx], wi, wo, s));
}

flux3_status flux3_quantize_fp8r(const void *w, int rows, int cols, void *codes, float *scales, void *stream) {
  if (!w || !codes || !scales || rows < 1 || cols < 16 || cols % 16 != 0) return FLUX3_ERR_INVALID_ARG;
  if ((size_t)rows * (size_t)cols > (size_t)1 << 34) return FLUX3_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u)) return FLUX3_ERR_ALIGNMENT;
  return cuda_status(launch_quantize_fp8r(static_cast<const __nv_bfloat16 *>(w), rows, cols,
                                          static_cast<uint8_t *>(codes), scales, static_cast<cudaStream_t>(stream)));
}

flux3_status flux3_block_init_fp8r(flux3_handle **out, const flux3_config *cfg, const flux3_block_weights_fp8r *w,
                                   int n_blocks, void *packed, size_t packed_bytes, void *stream) {
  if (!out) return FLUX3_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w || !packed) return FLUX3_ERR_INVALID_ARG;
  if (cfg->wfmt != FLUX3_W_FP8R) return FLUX3_ERR_INVALID_ARG;
  if (!config_ok(cfg)) return FLUX3_ERR_UNSUPPORTED;
  if (n_blocks != cfg->n_blocks) return FLUX3_ERR_INVALID_ARG;
  if (packed_bytes < flux3_packed_weight_bytes(cfg)) return FLUX3_ERR_WORKSPACE;
  if (!aligned16(packed)) return FLUX3_ERR_ALIGNMENT;
  for (int b = 0; b < n_blocks; ++b) {
    const flux3_block_weights_fp8r &bw = w[b];
    const flux3_fp8r_tensor *ts[6] = {&bw.q_proj, &bw.k_proj, &bw.v_proj, &bw.attn_out, &bw.mlp_in, &bw.mlp_out};
    for (const flux3_fp8r_tensor *t : ts) {
      if (!t->codes || !t->scales) return FLUX3_ERR_INVALID_ARG;
      if (!aligned16(t->codes) || (reinterpret_cast<uintptr_t>(t->scales) & 3u)) return FLUX3_ERR_ALIGNMENT;
    }
    if (!bw.query_norm || !bw.key_norm) return FLUX3_ERR_INVALID_ARG;
    if (!aligned16(bw.query_norm) || !aligned16(bw.key_norm)) return FLUX3_ERR_ALIGNMENT;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  flux3_handle *h = new (std::nothrow) flux3_handle();
  if (!h) return FLUX3_ERR_CUDA;
  h->cfg = *cfg;
  h->n_blocks = n_blocks;
  h->w_in = h->w_out = nullptr;
  uint8_t *base = static_cast<uint8_t *>(packed);
  auto *norms = reinterpret_cast<float *>(base + n_blocks * kFp8BlockBytes);
  h->norms = norms;
  h->fp8.resize(n_blocks);
  cudaError_t e = cudaSuccess;
  auto copy = [&](void *dst, const void *src, size_t bytes) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
  };
  auto copy2d = [&](void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, size_t height) {
    if (e == cudaSuccess) e = cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, cudaMemcpyDeviceToDevice, s);
  };
  for (int b = 0; b < n_blocks && e == cudaSuccess; ++b) {
    const flux3_block_weights_fp8r &bw = w[b];
    uint8_t *blk = base + b * kFp8BlockBytes;
    uint8_t *in_c = blk;
    float *in_s = reinterpret_cast<float *>(in_c + ws_round(kFp8InCodes));
    uint8_t *out_c = reinterpret_cast<uint8_t *>(in_s) + ws_round(kFp8InScales);
    float *out_s = reinterpret_cast<float *>(out_c + ws_round(kFp8OutCodes));
    // in-projection rows q | k | v | mlp_in (a and b interleaved in groups of 128), codes and row scales alike
    const flux3_fp8r_tensor *qkv[3] = {&bw.q_proj, &bw.k_proj, &bw.v_proj};
    for (int i = 0; i < 3; ++i) {
      copy(in_c + (size_t)i * kHidden * kHidden, qkv[i]->codes, (size_t)kHidden * kHidden);
      copy(in_s + (size_t)i * kHidden, qkv[i]->scales, kHidden * 4);
    }
    const uint8_t *mc = static_cast<const uint8_t *>(bw.mlp_in.codes);
    const float *ms = bw.mlp_in.scales;
    uint8_t *wc = in_c + (size_t)3 * kHidden * kHidden;
    float *wsc = in_s + 3 * kHidden;
    copy2d(wc, 256 * (size_t)kHidden, mc, 128 * (size_t)kHidden, 128 * (size_t)kHidden, kMlp / 128);
    copy2d(wc + 128 * (size_t)kHidden, 256 * (size_t)kHidden, mc + (size_t)kMlp * kHidden, 128 * (size_t)kHidden,
           128 * (size_t)kHidden, kMlp / 128);
    copy2d(wsc, 256 * 4, ms, 128 * 4, 128 * 4, kMlp / 128);
    copy2d(wsc + 128, 256 * 4, ms + kMlp, 128 * 4, 128 * 4, kMlp / 128);
    // out-projection rows: attn_out's inputs then mlp_out's; scales (attn_out's, mlp_out's) per row
    copy2d(out_c, kCatCols, bw.attn_out.codes, kHidden, kHidden, kHidden);
    copy2d(out_c + kHidden, kCatCols, bw.mlp_out.codes, kMlp, kMlp, kHidden);
    copy2d(out_s, 8, bw.attn_out.scales, 4, 4, kHidden);
    copy2d(out_s + 1, 8, bw.mlp_out.scales, 4, 4, kHidden);
    copy(norms + (size_t)b * 2 * kHeadDim, bw.query_norm, kHeadDim * 4);
    copy(norms + (size_t)b * 2 * kHeadDim + kHeadDim, bw.key_norm, kHeadDim * 4);
    h->fp8[b] = fp8r_detail::Fp8rBlockView{in_c, in_s, out_c, out_s};
  }
  if (e != cudaSuccess) {
    delete h;
    return FLUX3_ERR_CUDA;
  }
  *out = h;
  return FLUX3_OK;
}

flux3_status flux3_block_forward(const flux3_handle *h, int block_idx, float *x, int T, const flux3_segment *segs,
                                 int n_segs, const float *pos_ids, const float *mod, void *workspace, size_t ws_bytes,
                                 void *stream) {
  return forward_common(h, block_idx, 1, x, T, segs, n_segs, pos_ids, mod, workspace, ws_bytes,
                        static_cast<cudaStream_t>(stream));
}

flux3_status flux3_stack_forward(const flux3_handle *h, int first_block, int n_blocks, float *x, int T,
                                 const flux3_segment *segs, int n_segs, const float *pos_ids, const float *mod,
                                 void *workspace, size_t ws_bytes, void *stream) {
  return forward_common(h, first_block, n_blocks, x, T, segs, n_segs, pos_ids, mod, workspace, ws_bytes,
                        static_cast<cudaStream_t>(stream));
}

flux3_status flux3_mode_blocks_forward(const flux3_handle *const *mode_handles, int n_blocks, float *x, int T,
                                       const flux3_segment *segs, int n_segs, const float *pos_ids,
                                       const float *early_mod, void *workspace, size_t ws_bytes, void *stream) {
  if (!mode_handles || !x || !pos_ids || !early_mod || n_blocks < 1) return FLUX3_ERR_INVALID_ARG;
  F3_TRY(segments_ok(segs, n_segs, T));
  // each present mode must be one run of rows [row0, row0 + Tm)
  int first[3] = {-1, -1, -1}, last[3] = {-1, -1, -1};
  for (int i = 0; i < n_segs; ++i) {
    const int m = segs[i].stream;
    if (first[m] < 0) first[m] = i;
    last[m] = i;
  }
  for (int m = 0; m < 3; ++m) {
    if (first[m] < 0) continue;
    for (int i = first[m]; i <= last[m]; ++i)
      if (segs[i].stream != m) return FLUX3_ERR_INVALID_ARG;
    if (!mode_handles[m] || n_blocks > mode_handles[m]->n_blocks) return FLUX3_ERR_INVALID_ARG;
  }
  for (int m = 0; m < 3; ++m) {
    if (first[m] < 0) continue;
    const int row0 = segs[first[m]].start;
    const int tm = segs[last[m]].start + segs[last[m]].len - row0;
    const flux3_segment one{0, tm, m};
    F3_TRY(forward_common(mode_handles[m], 0, n_blocks, x + (size_t)row0 * kHidden, tm, &one, 1,
                          pos_ids + (size_t)row0 * 4, early_mod, workspace, ws_bytes,
                          static_cast<cudaStream_t>(stream)));
  }
  return FLUX3_OK;
}

flux3_status flux3_check_error(void *stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FLUX3_ERR_CUDA;
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
  if (e != cudaSuccess) return FLUX3_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return FLUX3_ERR_CUDA;
  }
  if (v == DEVERR_TIMEOUT) return FLUX3_ERR_TIMEOUT;
  if (v != 0) return FLUX3_ERR_DEVICE;
  return FLUX3_OK;
}

const char *flux3_status_string(flux3_status s) {
  switch (s) {
    case FLUX3_OK: return "ok";
    case FLUX3_ERR_INVALID_ARG: return "invalid argument";
    case FLUX3_ERR_UNSUPPORTED: return "unsupported configuration";
    case FLUX3_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FLUX3_ERR_WORKSPACE: return "buffer too small";
    case FLUX3_ERR_CUDA: return "CUDA runtime error";
    case FLUX3_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    case FLUX3_ERR_DEVICE: return "kernel bounds check failed";
  }
  return "unknown status";
}

void flux3_destroy(flux3_handle *h) { delete h; }

flux3_status flux3_stream_ids(const flux3_segment *segs, int n_segs, int T, uint8_t *stream_id, void *stream) {
  if (!stream_id) return FLUX3_ERR_INVALID_ARG;
  F3_TRY(segments_ok(segs, n_segs, T));
  return cuda_status(launch_stream_ids(segs, n_segs, T, stream_id, static_cast<cudaStream_t>(stream)));
}

flux3_status flux3_rope_tables(const float *pos_ids, int T, float theta, float *cos_tab, float *sin_tab,
                               void *stream) {
  if (!pos_ids || !cos_tab || !sin_tab || T < 1 || T > kMaxTokensLimit || !(theta > 0.f)) return FLUX3_ERR_INVALID_ARG;
  return cuda_status(launch_rope_tables(pos_ids, T, theta, cos_tab, sin_tab, static_cast<cudaStream_t>(stream)));
}

flux3_status flux3_prepare(const flux3_segment *segs, int n_segs, int T, const float *pos_ids, float theta,
                           uint8_t *stream_id, float *cos_tab, float *sin_tab, void *stream) {
  if (!stream_id || !pos_ids || !cos_tab || !sin_tab || !(theta > 0.f)) return FLUX3_ERR_INVALID_ARG;
  if (T > kMaxTokensLimit) return FLUX3_ERR_INVALID_ARG;
  F3_TRY(segments_ok(segs, n_segs, T));
  return cuda_status(launch_prepare(segs, n_segs, T, stream_id, pos_ids, theta, cos_tab, sin_tab,
                                    static_cast<cudaStream_t>(stream)));
}

flux3_status flux3_ln_modulate(const float *x, int T, const uint8_t *stream_id, const float *mod, float eps, void *hout,
                               void *stream) {
  if (!x || !stream_id || !mod || !hout || T < 1 || T > kMaxTokensLimit || !(eps > 0.f)) return FLUX3_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(mod) || !aligned16(hout)) return FLUX3_ERR_ALIGNMENT;
  return cuda_status(launch_ln_modulate(x, T, stream_id, mod, eps, static_cast<__nv_bfloat16 *>(hout),
                                        static_cast<cudaStream_t>(stream)));
}

flux3_status flux3_in_projection(const flux3_handle *h, int block_idx, const void *hmod, int T, const float *cos_tab,
                                 const float *sin_tab, void *qkv, void *cat, void *stream) {
  if (!h || !hmod || !cos_tab || !sin_tab || !qkv || !cat) return FLUX3_ERR_INVALID_ARG;
  if (block_idx < 0 || block_idx >= h->n_blocks || T < 1 || T > h->cfg.max_tokens) return FLUX3_ERR_INVALID_ARG;
  if (h->cfg.wfmt != FLUX3_W_BF16) return FLUX3_ERR_UNSUPPORTED;
  if (!aligned16(hmod) || !aligned16(qkv) || !aligned16(cat) || !aligned16(cos_tab) || !aligned16(sin_tab))
    return FLUX3_ERR_ALIGNMENT;
  return run_in_projection(h, block_idx, static_cast<const __nv_bfloat16 *>(hmod), T, cos_tab, sin_tab,
                           static_cast<__nv_bfloat16 *>(qkv), static_cast<__nv_bfloat16 *>(cat),
                           static_cast<cudaStream_t>(stream));
}

flux3_status flux3_attention(const void *qkv, int T, void *cat, void *split_buf, size_t split_bytes, void *stream) {
  if (!qkv || !cat || T < 1 || T > kMaxTokensLimit) return FLUX3_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(cat) || (split_buf && !aligned16(split_buf))) return FLUX3_ERR_ALIGNMENT;
  return cuda_status(launch_attention(static_cast<const __nv_bfloat16 *>(qkv), T, static_cast<__nv_bfloat16 *>(cat),
                                      static_cast<cudaStream_t>(stream), false, static_cast<float *>(split_buf),
                                      split_buf ? split_bytes : 0));
}

flux3_status flux3_out_projection(const flux3_handle *h, int block_idx, const void *cat, int T,
                                  const uint8_t *stream_id, const float *mod, float *x, void *split_buf,
                                  size_t split_bytes, void *stream) {
  if (!h || !cat || !stream_id || !mod || !x) return FLUX3_ERR_INVALID_ARG;
  if (block_idx < 0 || block_idx >= h->n_blocks || T < 1 || T > h->cfg.max_tokens) return FLUX3_ERR_INVALID_ARG;
  if (h->cfg.wfmt != FLUX3_W_BF16) return FLUX3_ERR_UNSUPPORTED;
  if (!aligned16(cat) || !aligned16(mod) || !aligned16(x)) return FLUX3_ERR_ALIGNMENT;
  if (split_buf && !aligned16(split_buf)) return FLUX3_ERR_ALIGNMENT;
  return run_out_projection(h, block_idx, static_cast<const __nv_bfloat16 *>(cat), T, stream_id, mod, x,
                            static_cast<float *>(split_buf), split_buf ? split_bytes : 0,
                            static_cast<cudaStream_t>(stream));
}

flux3_status flux3_gemm_bf16(const void *A, const void *B, void *C, int M, int N, int K, void *stream) {
  if (!A || !B || !C || M < 1 || N < kBN || K < kBK || N % kBN != 0 || K % kBK != 0) return FLUX3_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return FLUX3_ERR_ALIGNMENT;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, A, (uint64_t)M, (uint64_t)K, kBM) ||
      !make_tmap_bf16(&tb, B, (uint64_t)N, (uint64_t)K, kBoxB))
    return FLUX3_ERR_CUDA;
  EpiParams ep{};
  ep.C = static_cast<__nv_bfloat16 *>(C);
  ep.ldc = N;
  return cuda_status(launch_gemm(EPI_STORE, ta, tb, M, N, K, ep, static_cast<cudaStream_t>(stream)));
}

flux3_status flux3_block_forward_noalloc(const flux3_handle *h, int block_idx, float *x, int T,
                                         const flux3_segment *segs, int n_segs, const float *pos_ids,
                                         const float *mod, void *stream) {
  if (T > FLUX3_NOALLOC_MAX_TOKENS) return FLUX3_ERR_WORKSPACE;
  if (!h || T < 1) return FLUX3_ERR_INVALID_ARG;
  if (h->cfg.wfmt != FLUX3_W_BF16) return FLUX3_ERR_UNSUPPORTED;
  // the array is sized by workspace_total; the carving is workspace_layout's
  if (workspace_layout(FLUX3_NOALLOC_MAX_TOKENS, nullptr, nullptr, false) > kNoAllocScratchBytes)
    return FLUX3_ERR_WORKSPACE;
  void *scratch = noalloc_scratch();
  if (!scratch) return FLUX3_ERR_CUDA;
  return forward_common(h, block_idx, 1, x, T, segs, n_segs, pos_ids, mod, scratch, kNoAllocScratchBytes,
                        static_cast<cudaStream_t>(stream));
}

flux3_status flux3_selftest_wait_timeout(int timeout_us, void *stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return FLUX3_ERR_INVALID_ARG;
  return cuda_status(launch_selftest_wait(1000ull * (unsigned long long)timeout_us, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------- conditioning and the transformer call
namespace {

constexpr int kTimeDim = 256, kLatent = 128, kTxtFeat = 20480, kFinalPad = 256;

// packed cond weights: element counts, in this order
constexpr size_t kCondElems[] = {
    (size_t)kHidden * kTimeDim, (size_t)kHidden * kHidden,     // time_in
    (size_t)kHidden * kTimeDim, (size_t)kHidden * kHidden,     // ref_time_in
    (size_t)kModLen * kHidden, (size_t)kModLen * kHidden, (size_t)kModLen * kHidden,   // early
    (size_t)kModLen * kHidden, (size_t)kModLen * kHidden, (size_t)kModLen * kHidden,   // single
    (size_t)2 * kHidden * kHidden,                             // final adaLN [6144, 3072]
    (size_t)kHidden * kLatent, (size_t)kHidden * kLatent,      // emb_in image, image_cond
    (size_t)kHidden * kTxtFeat,                                // txt_in
    (size_t)kFinalPad * kHidden};                              // final linear, padded
constexpr int kCondParts = sizeof(kCondElems) / sizeof(kCondElems[0]);

size_t cond_offset(int part) {
  size_t off = 0;
  for (int i = 0; i < part; ++i) off += align_up(kCondElems[i] * 2);
  return off;
}

// conditioning scratch (floats): temb [3, 256], a [2, 3072], vec [2, 3072], ra [3072], r [3072]
constexpr size_t kCondScratchFloats = 3 * kTimeDim + 2 * kHidden + 2 * kHidden + kHidden + kHidden;

flux3_status run_conditioning(const flux3_cond *c, float t, float t_next, float *early, float *single, float *fin,
                              float *scratch, cudaStream_t s) {
  float *temb = scratch, *a = temb + 3 * kTimeDim, *vec = a + 2 * kHidden, *ra = vec + 2 * kHidden,
        *r = ra + kHidden;
  F3_CUDA(launch_timestep_embed((double)t, 0.0, (double)t_next, temb, s));
  F3_CUDA(launch_rows_linear(c->time_in_in, kHidden, kTimeDim, temb, kTimeDim, 2, a, kHidden, false, false, s));
  F3_CUDA(launch_rows_linear(c->time_in_out, kHidden, kHidden, a, kHidden, 2, vec, kHidden, true, false, s));
  if (c->flow) {
    F3_CUDA(launch_rows_linear(c->ref_in, kHidden, kTimeDim, temb + 2 * kTimeDim, kTimeDim, 1, ra, kHidden, false,
                               false, s));
    F3_CUDA(launch_rows_linear(c->ref_out, kHidden, kHidden, ra, kHidden, 1, r, kHidden, true, false, s));
    F3_CUDA(launch_add_row(vec, kHidden, 2, r, kHidden, s));
  }
  for (int st = 0; st < 3; ++st) {
    const float *v = vec + (st == FLUX3_STREAM_IMAGE ? 0 : kHidden);   // image at t, the others at 0
    F3_CUDA(launch_rows_linear(c->early[st], kModLen, kHidden, v, kHidden, 1, early + (size_t)st * kModLen, kModLen,
                               true, false, s));
    F3_CUDA(launch_rows_linear(c->single[st], kModLen, kHidden, v, kHidden, 1, single + (size_t)st * kModLen,
                               kModLen, true, false, s));
  }
  F3_CUDA(cudaMemsetAsync(fin + 2 * kHidden, 0, kHidden * 4, s));
  F3_CUDA(launch_rows_linear(c->final_adaln, 2 * kHidden, kHidden, vec, kHidden, 1, fin, 2 * kHidden, true, false,
                             s));
  return FLUX3_OK;
}

flux3_status inputs_ok(const void *const *inputs, const flux3_segment *segs, int n_segs) {
  if (!inputs) return FLUX3_ERR_INVALID_ARG;
  for (int i = 0; i < n_segs; ++i) {
    const void *p = inputs[segs[i].stream];
    if (!p) return FLUX3_ERR_INVALID_ARG;
    if (!aligned16(p)) return FLUX3_ERR_ALIGNMENT;
  }
  return FLUX3_OK;
}

flux3_status run_embed(const flux3_cond *c, const void *const *inputs, const flux3_segment *segs, int n_segs,
                       float *x, cudaStream_t s) {
  int row_of[3] = {0, 0, 0};   // next input row of each stream
  for (int i = 0; i < n_segs; ++i) {
    const int st = segs[i].stream, len = segs[i].len;
    const int K = st == FLUX3_STREAM_TXT ? kTxtFeat : kLatent;
    const __nv_bfloat16 *in = static_cast<const __nv_bfloat16 *>(inputs[st]) + (size_t)row_of[st] * K;
    row_of[st] += len;
    CUtensorMap tmA;
    if (!make_tmap_bf16(&tmA, in, (uint64_t)len, (uint64_t)K, kBM)) return FLUX3_ERR_CUDA;
    EpiParams ep{};
    ep.x = x + (size_t)segs[i].start * kHidden;
    ep.ldc = kHidden;
    F3_CUDA(launch_gemm(EPI_STORE_F32, tmA, c->tm_emb[st], len, kHidden, K, ep, s));
  }
  return FLUX3_OK;
}

size_t final_ws_bytes(int T) { return align_up((size_t)T) + align_up((size_t)T * kHidden * 2); }

flux3_status run_final(const flux3_cond *c, const float *x, const flux3_segment *segs, int n_segs, int T,
                       const float *fin, float *vel, uint8_t *ws, cudaStream_t s) {
  uint8_t *sid0 = ws;                                               // stream id 0 for every row: final_mod's row
  auto *h = reinterpret_cast<__nv_bfloat16 *>(ws + align_up((size_t)T));
  F3_CUDA(cudaMemsetAsync(sid0, 0, (size_t)T, s));
  int n_img = 0;
  for (int i = 0; i < n_segs; ++i) {
    if (segs[i].stream != FLUX3_STREAM_IMAGE) continue;
    F3_CUDA(launch_ln_modulate(x + (size_t)segs[i].start * kHidden, segs[i].len, sid0, fin, 1e-6f,
                               h + (size_t)n_img * kHidden, s));
    n_img += segs[i].len;
  }
  if (n_img == 0) return FLUX3_OK;
  CUtensorMap tmA;
  if (!make_tmap_bf16(&tmA, h, (uint64_t)n_img, kHidden, kBM)) return FLUX3_ERR_CUDA;
  EpiParams ep{};
  ep.x = vel;
  ep.ldc = kLatent;
  F3_CUDA(launch_gemm(EPI_STORE_F32, tmA, c->tm_final, n_img, kFinalPad, kHidden, ep, s));
  return FLUX3_OK;
}

// transformer workspace: x, early, single, final mods, cond scratch, final-layer scratch, block workspace
struct ModelWs {
  float *x, *early, *single, *fin, *scratch;
  uint8_t *final_ws, *block_ws;
  size_t block_bytes;
};
size_t model_ws_layout(const flux3_config *cfg, int T, uint8_t *base, ModelWs *w, int n_samples = 1) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return base ? base + o : nullptr;
  };
  uint8_t *x = take((size_t)T * kHidden * 4);
  uint8_t *e = take((size_t)3 * n_samples * kModLen * 4);
  uint8_t *sg = take((size_t)3 * n_samples * kModLen * 4);
  uint8_t *f = take((size_t)n_samples * kModLen * 4);
  uint8_t *sc = take(kCondScratchFloats * 4);
  uint8_t *fw = take(final_ws_bytes(T));
  const size_t bb = workspace_layout(T, nullptr, nullptr, lowp(cfg->wfmt));
  uint8_t *bw = take(bb);
  if (w) {
    w->x = reinterpret_cast<float *>(x);
    w->early = reinterpret_cast<float *>(e);
    w->single = reinterpret_cast<float *>(sg);
    w->fin = reinterpret_cast<float *>(f);
    w->scratch = reinterpret_cast<float *>(sc);
    w->final_ws = fw;
    w->block_ws = bw;
    w->block_bytes = bb;
  }
  return off;
}

}  // namespace

extern "C" {

size_t flux3_cond_packed_bytes(void) { return cond_offset(kCondParts); }

flux3_status flux3_cond_init(flux3_cond **out, const flux3_cond_weights *w, void *packed, size_t packed_bytes,
                             void *stream) {
  if (!out) return FLUX3_ERR_INVALID_ARG;
  *out = nullptr;
  if (!w || !packed) return FLUX3_ERR_INVALID_ARG;
  if (packed_bytes < flux3_cond_packed_bytes()) return FLUX3_ERR_WORKSPACE;
  if (!aligned16(packed)) return FLUX3_ERR_ALIGNMENT;
  const bool flow = w->ref_time_in_in != nullptr;
  if (flow != (w->ref_time_in_out != nullptr)) return FLUX3_ERR_INVALID_ARG;
  const void *src[kCondParts] = {w->time_in_in, w->time_in_out, w->ref_time_in_in, w->ref_time_in_out,
                                 w->early_mod[0], w->early_mod[1], w->early_mod[2], w->single_mod[0],
                                 w->single_mod[1], w->single_mod[2], w->final_adaln, w->emb_in_image,
                                 w->emb_in_image_cond, w->txt_in, w->final_linear};
  for (int i = 0; i < kCondParts; ++i) {
    if (!src[i] && !(i == 2 || i == 3)) return FLUX3_ERR_INVALID_ARG;
    if (src[i] && !aligned16(src[i])) return FLUX3_ERR_ALIGNMENT;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  flux3_cond *c = new (std::nothrow) flux3_cond();
  if (!c) return FLUX3_ERR_CUDA;
  uint8_t *base = static_cast<uint8_t *>(packed);
  auto part = [&](int i) { return reinterpret_cast<__nv_bfloat16 *>(base + cond_offset(i)); };
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < kCondParts && e == cudaSuccess; ++i) {
    if (!src[i]) continue;
    const size_t bytes = (i == kCondParts - 1 ? (size_t)kLatent * kHidden : kCondElems[i]) * 2;
    e = cudaMemcpyAsync(part(i), src[i], bytes, cudaMemcpyDeviceToDevice, s);
  }
  // rows 128..255 of the padded output linear are zero (their outputs are not stored either)
  if (e == cudaSuccess)
    e = cudaMemsetAsync(part(kCondParts - 1) + (size_t)kLatent * kHidden, 0, (size_t)kLatent * kHidden * 2, s);
  if (e != cudaSuccess) {
    delete c;
    return FLUX3_ERR_CUDA;
  }
  c->flow = flow;
  c->time_in_in = part(0);
  c->time_in_out = part(1);
  c->ref_in = part(2);
  c->ref_out = part(3);
  for (int st = 0; st < 3; ++st) {
    c->early[st] = part(4 + st);
    c->single[st] = part(7 + st);
  }
  c->final_adaln = part(10);
  if (!make_tmap_bf16(&c->tm_emb[FLUX3_STREAM_IMAGE], part(11), kHidden, kLatent, kBoxB) ||
      !make_tmap_bf16(&c->tm_emb[FLUX3_STREAM_IMAGE_COND], part(12), kHidden, kLatent, kBoxB) ||
      !make_tmap_bf16(&c->tm_emb[FLUX3_STREAM_TXT], part(13), kHidden, kTxtFeat, kBoxB) ||
      !make_tmap_bf16(&c->tm_final, part(14), kFinalPad, kHidden, kBoxB)) {
    delete c;
    return FLUX3_ERR_CUDA;
  }
  *out = c;
  return FLUX3_OK;
}

void flux3_cond_destroy(flux3_cond *c) { delete c; }

size_t flux3_cond_workspace_bytes(void) { return align_up(kCondScratchFloats * 4); }

flux3_status flux3_conditioning(const flux3_cond *c, float t, float t_next, float *early_mod, float *single_mod,
                                float *final_mod, void *workspace, size_t ws_bytes, void *stream) {
  if (!c || !early_mod || !single_mod || !final_mod || !workspace) return FLUX3_ERR_INVALID_ARG;
  if (!(t >= 0.f && t <= 1.f) || (c->flow && !(t_next >= 0.f && t_next <= 1.f))) return FLUX3_ERR_INVALID_ARG;
  if (ws_bytes < flux3_cond_workspace_bytes()) return FLUX3_ERR_WORKSPACE;
  if (!aligned16(early_mod) || !aligned16(single_mod) || !aligned16(final_mod) || !aligned16(workspace))
    return FLUX3_ERR_ALIGNMENT;
  return run_conditioning(c, t, c->flow ? t_next : 0.f, early_mod, single_mod, final_mod,
                          static_cast<float *>(workspace), static_cast<cudaStream_t>(stream));
}

flux3_status flux3_embed_tokens(const flux3_cond *c, const void *const *inputs, int T, const flux3_segment *segs,
                                int n_segs, float *x, void *stream) {
  if (!c || !x) return FLUX3_ERR_INVALID_ARG;
  F3_TRY(segments_ok(segs, n_segs, T));
  F3_TRY(inputs_ok(inputs, segs, n_segs));
  if (!aligned16(x)) return FLUX3_ERR_ALIGNMENT;
  return run_embed(c, inputs, segs, n_segs, x, static_cast<cudaStream_t>(stream));
}

size_t flux3_final_layer_workspace_bytes(int T) { return T < 1 ? 0 : final_ws_bytes(T); }

flux3_status flux3_final_layer(const flux3_cond *c, const float *x, int T, const flux3_segment *segs, int n_segs,
                               const float *final_mod, float *velocity, void *workspace, size_t ws_bytes,
                               void *stream) {
  if (!c || !x || !final_mod || !velocity || !workspace) return FLUX3_ERR_INVALID_ARG;
  F3_TRY(segments_ok(segs, n_segs, T));
  if (ws_bytes < final_ws_bytes(T)) return FLUX3_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(final_mod) || !aligned16(velocity) || !aligned16(workspace))
    return FLUX3_ERR_ALIGNMENT;
  return run_final(c, x, segs, n_segs, T, final_mod, velocity, static_cast<uint8_t *>(workspace),
                   static_cast<cudaStream_t>(stream));
}

size_t flux3_transformer_workspace_bytes(const flux3_config *joint_cfg, int T) {
  if (!config_ok(joint_cfg) || T < 1 || T > joint_cfg->max_tokens) return 0;
  return model_ws_layout(joint_cfg, T, nullptr, nullptr);
}

flux3_status flux3_transformer_forward(const flux3_cond *c, const flux3_handle *const *mode_handles,
                                       int n_mode_blocks, const flux3_handle *joint, const void *const *inputs,
                                       int T, const flux3_segment *segs, int n_segs, const float *pos_ids, float t,
                                       float t_next, float *velocity, void *workspace, size_t ws_bytes,
                                       void *stream) {
  if (!c || !joint || !pos_ids || !velocity || !workspace || n_mode_blocks < 0) return FLUX3_ERR_INVALID_ARG;
  if (n_mode_blocks > 0 && !mode_handles) return FLUX3_ERR_INVALID_ARG;
  if (T < 1 || T > joint->cfg.max_tokens) return FLUX3_ERR_INVALID_ARG;
  F3_TRY(segments_ok(segs, n_segs, T));
  F3_TRY(inputs_ok(inputs, segs, n_segs));
  if (!(t >= 0.f && t <= 1.f) || (c->flow && !(t_next >= 0.f && t_next <= 1.f))) return FLUX3_ERR_INVALID_ARG;
  if (!aligned16(workspace) || !aligned16(velocity) || !aligned16(pos_ids)) return FLUX3_ERR_ALIGNMENT;
  if (ws_bytes < model_ws_layout(&joint->cfg, T, nullptr, nullptr)) return FLUX3_ERR_WORKSPACE;
  ModelWs w;
  model_ws_layout(&joint->cfg, T, static_cast<uint8_t *>(workspace), &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  F3_TRY(run_conditioning(c, t, c->flow ? t_next : 0.f, w.early, w.single, w.fin, w.scratch, s));
  F3_TRY(run_embed(c, inputs, segs, n_segs, w.x, s));
  if (n_mode_blocks > 0)
    F3_TRY(flux3_mode_blocks_forward(mode_handles, n_mode_blocks, w.x, T, segs, n_segs, pos_ids, w.early,
                                     w.block_ws, w.block_bytes, stream));
  F3_TRY(forward_common(joint, 0, joint->n_blocks, w.x, T, segs, n_segs, pos_ids, w.single, w.block_ws,
                        w.block_bytes, s));
  return run_final(c, w.x, segs, n_segs, T, w.fin, velocity, w.final_ws, s);
}

flux3_status flux3_sigma_schedule(int steps, double alpha, float *sigmas) {
  if (steps < 1 || !(alpha > 0.0) || !sigmas) return FLUX3_ERR_INVALID_ARG;
  for (int k = 0; k <= steps; ++k) {
    const double t = 1.0 - (double)k / (double)steps;
    sigmas[k] = (float)(alpha * t / (1.0 + (alpha - 1.0) * t));
  }
  return FLUX3_OK;
}

flux3_status flux3_euler_step(float *latent, const float *velocity, size_t n, float sigma, float sigma_next,
                              void *next_input, void *stream) {
  if (!latent || !velocity || n == 0) return FLUX3_ERR_INVALID_ARG;
  const float dt = (float)((double)sigma_next - (double)sigma);
  return cuda_status(launch_euler(latent, velocity, n, dt, static_cast<__nv_bfloat16 *>(next_input),
                                  static_cast<cudaStream_t>(stream)));
}

flux3_status flux3_latents_to_bf16(const float *latent, size_t n, void *input, void *stream) {
  if (!latent || !input || n == 0) return FLUX3_ERR_INVALID_ARG;
  return cuda_status(launch_to_bf16(latent, n, static_cast<__nv_bfloat16 *>(input), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" {

flux3_status flux3_stack_forward_batch(const flux3_handle *h, int first_block, int n_blocks, float *x, int T,
                                       const flux3_segment *segs, int n_segs, const int *sample_start, int n_samples,
                                       const float *pos_ids, const float *mod, void *workspace, size_t ws_bytes,
                                       void *stream) {
  if (!sample_start) return FLUX3_ERR_INVALID_ARG;
  return forward_common(h, first_block, n_blocks, x, T, segs, n_segs, pos_ids, mod, workspace, ws_bytes,
                        static_cast<cudaStream_t>(stream), sample_start, n_samples);
}

size_t flux3_transformer_batch_workspace_bytes(const flux3_config *joint_cfg, int T, int n_samples) {
  if (!config_ok(joint_cfg) || T < 1 || T > joint_cfg->max_tokens || n_samples < 1 || n_samples > FLUX3_MAX_SAMPLES)
    return 0;
  return model_ws_layout(joint_cfg, T, nullptr, nullptr, n_samples);
}

flux3_status flux3_transformer_forward_batch(const flux3_cond *c, const flux3_handle *const *mode_handles,
                                             int n_mode_blocks, const flux3_handle *joint, const void *const *inputs,
                                             int T, const flux3_segment *segs, int n_segs, const int *sample_start,
                                             int n_samples, const float *pos_ids, const float *t, const float *t_next,
                                             float *velocity, void *workspace, size_t ws_bytes, void *stream) {
  if (!c || !joint || !pos_ids || !velocity || !workspace || !t || n_mode_blocks < 0 || !inputs)
    return FLUX3_ERR_INVALID_ARG;
  if (n_mode_blocks > 0 && !mode_handles) return FLUX3_ERR_INVALID_ARG;
  if (c->flow && !t_next) return FLUX3_ERR_INVALID_ARG;
  if (T < 1 || T > joint->cfg.max_tokens) return FLUX3_ERR_INVALID_ARG;
  F3_TRY(segments_ok(segs, n_segs, T));
  int sample_of[FLUX3_MAX_SEGMENTS] = {0};
  F3_TRY(samples_ok(sample_start, n_samples, T, segs, n_segs, sample_of));
  for (int b = 0; b < n_samples; ++b) {
    if (!(t[b] >= 0.f && t[b] <= 1.f) || (c->flow && !(t_next[b] >= 0.f && t_next[b] <= 1.f)))
      return FLUX3_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_segs; ++i) {
    const void *p = inputs[3 * sample_of[i] + segs[i].stream];
    if (!p) return FLUX3_ERR_INVALID_ARG;
    if (!aligned16(p)) return FLUX3_ERR_ALIGNMENT;
  }
  if (!aligned16(workspace) || !aligned16(velocity) || !aligned16(pos_ids)) return FLUX3_ERR_ALIGNMENT;
  if (ws_bytes < model_ws_layout(&joint->cfg, T, nullptr, nullptr, n_samples)) return FLUX3_ERR_WORKSPACE;
  ModelWs w;
  model_ws_layout(&joint->cfg, T, static_cast<uint8_t *>(workspace), &w, n_samples);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // per sample: conditioning rows 3b.., embedders, per-mode blocks on the sample's rows
  for (int b = 0; b < n_samples; ++b) {
    const int r0 = sample_start[b], tb = sample_start[b + 1] - r0;
    flux3_segment local[FLUX3_MAX_SEGMENTS], absolute[FLUX3_MAX_SEGMENTS];
    int n = 0;
    for (int i = 0; i < n_segs; ++i)
      if (sample_of[i] == b) {
        absolute[n] = segs[i];
        local[n] = segs[i];
        local[n].start -= r0;
        ++n;
      }
    F3_TRY(run_conditioning(c, t[b], c->flow ? t_next[b] : 0.f, w.early + (size_t)3 * b * kModLen,
                            w.single + (size_t)3 * b * kModLen, w.fin + (size_t)b * kModLen, w.scratch, s));
    F3_TRY(run_embed(c, inputs + 3 * b, absolute, n, w.x, s));
    if (n_mode_blocks > 0)
      F3_TRY(flux3_mode_blocks_forward(mode_handles, n_mode_blocks, w.x + (size_t)r0 * kHidden, tb, local, n,
                                       pos_ids + (size_t)r0 * 4, w.early + (size_t)3 * b * kModLen, w.block_ws,
                                       w.block_bytes, stream));
  }
  F3_TRY(forward_common(joint, 0, joint->n_blocks, w.x, T, segs, n_segs, pos_ids, w.single, w.block_ws,
                        w.block_bytes, s, sample_start, n_samples));
  int img_rows = 0;
  for (int b = 0; b < n_samples; ++b) {
    const int r0 = sample_start[b], tb = sample_start[b + 1] - r0;
    flux3_segment local[FLUX3_MAX_SEGMENTS];
    int n = 0, n_img = 0;
    for (int i = 0; i < n_segs; ++i)
      if (sample_of[i] == b) {
        local[n] = segs[i];
        local[n].start -= r0;
        if (segs[i].stream == FLUX3_STREAM_IMAGE) n_img += segs[i].len;
        ++n;
      }
    F3_TRY(run_final(c, w.x + (size_t)r0 * kHidden, local, n, tb, w.fin + (size_t)b * kModLen,
                     velocity + (size_t)img_rows * kLatent, w.final_ws, s));
    img_rows += n_img;
  }
  return FLUX3_OK;
}

flux3_status flux3_cfg_euler_step(float *latent, const float *v_uncond, const float *v_cond, size_t n,
                                  float guidance, float sigma, float sigma_next, void *next_input, void *stream) {
  if (!latent || !v_uncond || !v_cond || n == 0) return FLUX3_ERR_INVALID_ARG;
  const float dt = (float)((double)sigma_next - (double)sigma);
  return cuda_status(launch_cfg_euler(latent, v_uncond, v_cond, n, guidance, dt,
                                      static_cast<__nv_bfloat16 *>(next_input), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
