/*
 * flux3.h -- C ABI of the B300 (sm_103a) library for the FLUX.3 Image Klein
 * joint single_block forward pass.
 *
 * What the library computes (per block, for every token t of one sample):
 *   h    = (1 + scale[s]) * LayerNorm(x) + shift[s]        LayerNorm without affine, eps 1e-6
 *   q,k,v = h Wq^T, h Wk^T, h Wv^T                           24 heads x 128, no bias
 *   q^, k^ = RoPE4(RMSNorm(q) * query_norm), RoPE4(RMSNorm(k) * key_norm)   per head, eps 1e-6
 *   o    = softmax(q^ k^T / sqrt(128)) v                     all tokens attend to all tokens
 *   a|b  = h Wmlp_in^T,  g = silu(a) * b                     a = first 9216 outputs
 *   x'   = x + gate[s] * (o Wattn_out^T + g Wmlp_out^T)
 * s = the token's stream (image, image_cond, txt); each stream has its own
 * [shift | scale | gate] vector of 3 x 3072 floats.  Sources: "FLUX.3 Image
 * Klein support" (stable-diffusion.cpp issue #2142), comment "Structure (from
 * dit.py)" and its tensor list; "Welcome FLUX.3 Image Klein in Diffusers",
 * sections "Inside one block", "Two stages" and "Positions in four dimensions".
 *
 * Around the joint blocks the library also runs the 5 per-mode blocks (each
 * mode through its own weights, attention within the mode), weights stored
 * in NVFP4 or row-wise FP8, one whole transformer call (timestep
 * conditioning, embedders, both block stages, the image output layer), the
 * sampler updates, and batches of samples with attention per sample (the base
 * model's guided two-sample pack).  Each declaration below cites its passage.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers are ordinary process memory.  Each argument says which.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous on it; nothing synchronises except
 *     flux3_check_error().
 *   - All device memory (weights, packed weights, activations, workspace) is
 *     owned by the caller.  Weights are borrowed by the *_init calls only for
 *     the packing copies they enqueue; the packed buffer must outlive the
 *     handle.  Handles are freed by flux3_destroy / flux3_cond_destroy.
 *   - Layouts are row-major, token-major: a [T, C] tensor has element (t, c) at
 *     offset t*C + c.  bf16 is IEEE bfloat16 stored in 16 bits.
 *   - Errors are returned as flux3_status codes, never by aborting.  Argument
 *     errors are detected on the host before anything is enqueued.  Device-side
 *     failures (a pipeline wait that timed out, an index out of range) set a
 *     device error word that flux3_check_error() reads and clears.
 */
#ifndef FLUX3_H
#define FLUX3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FLUX3_API __attribute__((visibility("default")))

typedef enum flux3_status {
  FLUX3_OK = 0,
  FLUX3_ERR_INVALID_ARG = -1,   /* null pointer, bad size, bad segment table      */
  FLUX3_ERR_UNSUPPORTED = -2,   /* configuration the kernels are not built for    */
  FLUX3_ERR_ALIGNMENT = -3,     /* pointer not 16-byte aligned                    */
  FLUX3_ERR_WORKSPACE = -4,     /* workspace / packed buffer smaller than needed  */
  FLUX3_ERR_CUDA = -5,          /* a CUDA runtime call failed                     */
  FLUX3_ERR_TIMEOUT = -6,       /* a kernel pipeline wait ran out (device word)   */
  FLUX3_ERR_DEVICE = -7         /* a kernel's own bounds check fired (device word) */
} flux3_status;

/* Weight formats.  NVFP4 = e2m1 values with one e4m3 scale per 16 inputs and a
 * float32 per-tensor scale; FP8R = e4m3 values with one float32 scale per row
 * ("Welcome FLUX.3 Image Klein in Diffusers", section "Single-file format
 * checkpoints", names the nvfp4 and fp8r variants). */
typedef enum flux3_wfmt { FLUX3_W_BF16 = 0, FLUX3_W_NVFP4 = 1, FLUX3_W_FP8R = 2 } flux3_wfmt;

/* Token streams ("modes"): each selects its own modulation vector. */
typedef enum flux3_stream {
  FLUX3_STREAM_IMAGE = 0,
  FLUX3_STREAM_IMAGE_COND = 1,
  FLUX3_STREAM_TXT = 2
} flux3_stream;

/* Model configuration.  The kernels are built for hidden 3072, 24 heads of
 * 128, SwiGLU width 9216 (the shapes of the issue's tensor list); other values
 * return FLUX3_ERR_UNSUPPORTED.  max_tokens bounds T for workspace sizing. */
typedef struct flux3_config {
  int hidden;       /* 3072 */
  int heads;        /* 24   */
  int head_dim;     /* 128  */
  int mlp_hidden;   /* 9216 (mlp_in has 2 * mlp_hidden rows) */
  int n_blocks;     /* blocks held by a handle, 28 for the joint stack */
  int max_tokens;   /* largest T a forward call may use (<= 65536) */
  int wfmt;         /* flux3_wfmt */
  float rope_theta; /* 10000 */
  float eps_ln;     /* 1e-6 */
  float eps_rms;    /* 1e-6 */
} flux3_config;

/* One block's weights as the checkpoint stores them: device bf16 matrices of
 * shape [out, in] (row-major, no bias) and device float32 [128] norm scales.
 * Pointers must be 16-byte aligned. */
typedef struct flux3_block_weights {
  const void *q_proj;     /* [3072, 3072]  */
  const void *k_proj;     /* [3072, 3072]  */
  const void *v_proj;     /* [3072, 3072]  */
  const void *attn_out;   /* [3072, 3072]  */
  const void *mlp_in;     /* [18432, 3072] */
  const void *mlp_out;    /* [3072, 9216]  */
  const float *query_norm;/* [128] */
  const float *key_norm;  /* [128] */
} flux3_block_weights;

/* One weight matrix [rows, cols] in NVFP4 (cols a multiple of 16):
 *   codes         device uint8 [rows, cols / 2]: e2m1 codes (sign bit 3,
 *                 exponent bits 2..1 with bias 1, mantissa bit 0); element 2i
 *                 of a row is the low nibble of byte i, element 2i+1 the high
 *   scales        device uint8 [rows, cols / 16]: e4m3 bit patterns (sign 7,
 *                 exponent 6..3 with bias 7, mantissa 2..0); scale b of a row
 *                 covers its elements 16b .. 16b+15
 *   global_scale  device float32 [1]
 * weight[r, c] = e2m1(code[r, c]) * e4m3(scales[r, c / 16]) * global_scale.
 * The pages name the nvfp4 checkpoint variant ("Welcome FLUX.3 Image Klein in
 * Diffusers", section "Single-file format checkpoints") but not its layout;
 * this is the layout flux3_quantize_nvfp4 writes. */
typedef struct flux3_nvfp4_tensor {
  const void *codes;
  const void *scales;
  const float *global_scale;
} flux3_nvfp4_tensor;

/* One block's weights in NVFP4 (shapes as flux3_block_weights); the norm
 * scales stay float32.  Pointers must be 16-byte aligned (global_scale: 4). */
typedef struct flux3_block_weights_nvfp4 {
  flux3_nvfp4_tensor q_proj, k_proj, v_proj, attn_out, mlp_in, mlp_out;
  const float *query_norm;
  const float *key_norm;
} flux3_block_weights_nvfp4;

/* One weight matrix [rows, cols] in row-wise FP8 ("fp8r"):
 *   codes   device uint8 [rows, cols]: E4M3 bit patterns (sign 7, exponent
 *           6..3 with bias 7, mantissa 2..0); 0x7F / 0xFF (NaN) must not occur
 *   scales  device float32 [rows]: one scale per row (output feature)
 * weight[r, c] = e4m3(code[r, c]) * scales[r].  The pages name the fp8r
 * checkpoint variant ("Welcome FLUX.3 Image Klein in Diffusers", section
 * "Single-file format checkpoints") but not its layout; this is the layout
 * flux3_quantize_fp8r writes. */
typedef struct flux3_fp8r_tensor {
  const void *codes;
  const float *scales;
} flux3_fp8r_tensor;

/* One block's weights in fp8r (shapes as flux3_block_weights); the norm scales
 * stay float32.  codes and norm pointers 16-byte aligned, scales 4-byte. */
typedef struct flux3_block_weights_fp8r {
  flux3_fp8r_tensor q_proj, k_proj, v_proj, attn_out, mlp_in, mlp_out;
  const float *query_norm;
  const float *key_norm;
} flux3_block_weights_fp8r;

/* A contiguous run of tokens of one stream.  A forward call's segments must be
 * in increasing order, non-overlapping, non-empty, and cover [0, T) exactly;
 * at most FLUX3_MAX_SEGMENTS of them.  Any stream order is accepted. */
typedef struct flux3_segment {
  int start;
  int len;
  int stream;   /* flux3_stream */
} flux3_segment;

#define FLUX3_MAX_SEGMENTS 32

typedef struct flux3_handle flux3_handle;

/* Fills *cfg with the FLUX.3 Image Klein joint-block configuration
 * (3072 / 24 / 128 / 9216, 28 blocks, max_tokens 16384, bf16, theta 1e4,
 * eps 1e-6). */
FLUX3_API void flux3_default_config(flux3_config *cfg);

/* Bytes of the caller-owned buffer flux3_block_init (bf16),
 * flux3_block_init_nvfp4 (cfg->wfmt == FLUX3_W_NVFP4) or
 * flux3_block_init_fp8r (FLUX3_W_FP8R) packs the weights into (per block: the
 * q/k/v/mlp_in rows concatenated, the attn_out/mlp_out columns concatenated,
 * and the two norm scales; NVFP4 keeps codes, block scales and the six global
 * scales, 69.0 MB per block, fp8r codes and row scales, 122.9 MB, instead of
 * 245.4 MB).  0 if cfg is invalid. */
FLUX3_API size_t flux3_packed_weight_bytes(const flux3_config *cfg);

/* Bytes of workspace a forward call with T tokens needs (stream ids, RoPE
 * tables, modulated input, q/k/v, attention + SwiGLU output; with NVFP4 or
 * fp8r weights also one block's weights expanded to bf16, 245.4 MB, which
 * calls of up to 128 tokens leave unused).  0 if cfg is invalid or T is out of
 * range. */
FLUX3_API size_t flux3_workspace_bytes(const flux3_config *cfg, int T);

/* Creates a handle for n_blocks blocks (n_blocks == cfg->n_blocks).
 *   w        host array of n_blocks weight sets (device pointers inside)
 *   packed   device buffer of flux3_packed_weight_bytes(cfg) bytes (caller-owned)
 * Enqueues the packing copies on `stream`; the handle may be used for forward
 * calls on that stream right away (other streams: synchronise first).
 * Returns FLUX3_ERR_INVALID_ARG / _UNSUPPORTED / _ALIGNMENT / _WORKSPACE / _CUDA. */
FLUX3_API flux3_status flux3_block_init(flux3_handle **out, const flux3_config *cfg,
                                        const flux3_block_weights *w, int n_blocks,
                                        void *packed, size_t packed_bytes, void *stream);

/* flux3_block_init for NVFP4 weights (cfg->wfmt == FLUX3_W_NVFP4): packs the
 * codes, block scales, global scales and norm scales into `packed`
 * (flux3_packed_weight_bytes(cfg) bytes).  Every forward call then expands
 * each block's weights to bf16 (e2m1 * e4m3, exact in float32, times the
 * global scale rounded to float32, then to bf16; both nearest even) and the
 * projections run as bf16 tensor-core GEMMs with bf16 activations: above 128
 * tokens the expansion goes to the workspace just before the block runs, up to
 * 128 tokens the GEMMs expand the codes in shared memory (the same values).
 * Same errors as flux3_block_init. */
FLUX3_API flux3_status flux3_block_init_nvfp4(flux3_handle **out, const flux3_config *cfg,
                                              const flux3_block_weights_nvfp4 *w, int n_blocks,
                                              void *packed, size_t packed_bytes, void *stream);

/* Quantises a bf16 matrix to NVFP4 on the device:
 *   global_scale = float32(amax / (6 * 448))   (1 if the matrix is all zero)
 *   scale of block b = e4m3, nearest even, of amax_b / (6 * global_scale),
 *                      saturating at 448 (amax_b = largest |w| of the block)
 *   code = e2m1, nearest even, of w / (scale * global_scale), saturating at
 *          +-6; zero never carries a sign; a block whose scale is 0 is all 0
 * Every rounding decision is taken on the float64 quotient, so the result is
 * reproducible bit for bit.
 *   w             device bf16 [rows, cols], cols % 16 == 0, 16-byte aligned
 *   codes, scales device outputs in the flux3_nvfp4_tensor layout
 *   global_scale  device float32 [1] (output; it holds the amax bits while the
 *                 call's kernels run) */
FLUX3_API flux3_status flux3_quantize_nvfp4(const void *w, int rows, int cols, void *codes, void *scales,
                                            float *global_scale, void *stream);

/* The bf16 weights an NVFP4 or fp8r handle's block_idx runs with, as the forward pass
 * expands them: w_in device bf16 [27648, 3072] = rows of q | k | v | mlp_in
 * (mlp_in's a and b halves interleaved in groups of 128 rows: a[128m..],
 * b[128m..], ...), w_out device bf16 [3072, 12288] = [attn_out | mlp_out]
 * along the input dimension.  FLUX3_ERR_UNSUPPORTED for a bf16 handle. */
FLUX3_API flux3_status flux3_dequantize_block(const flux3_handle *h, int block_idx, void *w_in, void *w_out,
                                              void *stream);

/* A handle over fp8r weights (cfg->wfmt = FLUX3_W_FP8R), same conventions as
 * flux3_block_init_nvfp4: the codes and scales are copied into `packed`
 * (flux3_packed_weight_bytes(cfg) bytes: 122.9 MB per block), and every
 * forward call expands the running block's weights to bf16 (e4m3 * scale
 * rounded to float32, then to bf16, both nearest even) for the bf16 GEMMs: in
 * the workspace above 128 tokens, inside the GEMMs in shared memory up to 128. */
FLUX3_API flux3_status flux3_block_init_fp8r(flux3_handle **out, const flux3_config *cfg,
                                             const flux3_block_weights_fp8r *w, int n_blocks, void *packed,
                                             size_t packed_bytes, void *stream);

/* Row-wise FP8 quantisation of a device bf16 [rows, cols] matrix (cols a
 * multiple of 16, w and codes 16-byte aligned): per row s = amax / 448
 * rounded to float32 (1 for an all-zero row), codes = E4M3 of w / s, round to
 * nearest even, saturating at +-448, no negative zero (the decision taken in
 * float64).  codes: device uint8 [rows, cols]; scales: device float32 [rows]. */
FLUX3_API flux3_status flux3_quantize_fp8r(const void *w, int rows, int cols, void *codes, float *scales,
                                           void *stream);

/* One joint block (block_idx of the handle) applied in place.
 *   x        device float32 [T, 3072]: the residual stream, updated in place
 *   segs     host array of n_segs segments covering [0, T)
 *   pos_ids  device float32 [T, 4]: RoPE ids (t, h, w, l) per token
 *   mod      device float32 [3, 9216]: per stream (image, image_cond, txt) the
 *            shift | scale | gate vectors, each 3072 long
 *   workspace device buffer of at least flux3_workspace_bytes(cfg, T) bytes
 * 1 <= T <= cfg->max_tokens. */
FLUX3_API flux3_status flux3_block_forward(const flux3_handle *h, int block_idx, float *x, int T,
                                           const flux3_segment *segs, int n_segs,
                                           const float *pos_ids, const float *mod,
                                           void *workspace, size_t ws_bytes, void *stream);

/* Blocks first_block .. first_block + n_blocks - 1 applied in sequence to the
 * residual stream x (same arguments as flux3_block_forward).  All blocks use
 * the same `mod` (the joint blocks share one set of stream modulations: the
 * modulation tensors of the issue's list carry no block index).  The stream
 * ids and RoPE tables are built once per call. */
FLUX3_API flux3_status flux3_stack_forward(const flux3_handle *h, int first_block, int n_blocks,
                                           float *x, int T, const flux3_segment *segs, int n_segs,
                                           const float *pos_ids, const float *mod,
                                           void *workspace, size_t ws_bytes, void *stream);

/* The per-mode blocks that precede the joint stack ("FLUX.3 Image Klein
 * support", comment "Structure (from dit.py)"): five blocks per mode with
 * that mode's own weights; attention limited to the tokens of the same mode
 * in the same sample; modulation from the mode's early_stream_modulations
 * (tensor names content_mode_blocks.{image, image_cond}.{0..4} and
 * txt_mode_blocks.{0..4}).  Each mode's tokens run
 * through blocks 0 .. n_blocks-1 of that mode's handle as a sequence of their
 * own (attention block-diagonal by mode); x is updated in place.
 *   mode_handles  host array [3] indexed by flux3_stream: the handle holding
 *                 that mode's blocks; may be NULL for a mode with no tokens
 *   n_blocks      blocks per mode (5 in the checkpoint); 1 <= n_blocks <= each
 *                 used handle's block count
 *   x, T, segs, n_segs, pos_ids: as flux3_block_forward.  The segments of one
 *                 stream must be adjacent (one run of rows), as in the
 *                 pipeline's token order; otherwise FLUX3_ERR_INVALID_ARG.
 *   early_mod     device float32 [3, 9216]: per stream the shift | scale |
 *                 gate of early_stream_modulations
 *   workspace     device buffer of at least flux3_workspace_bytes(cfg, Tm)
 *                 bytes, Tm the largest mode's token count (T always
 *                 suffices); each used handle's max_tokens >= its mode's count
 * The modes run one after another on `stream`, each through the same kernels
 * as flux3_stack_forward on its rows. */
FLUX3_API flux3_status flux3_mode_blocks_forward(const flux3_handle *const *mode_handles, int n_blocks, float *x,
                                                 int T, const flux3_segment *segs, int n_segs,
                                                 const float *pos_ids, const float *early_mod, void *workspace,
                                                 size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * One transformer call around the block stacks ("FLUX.3 Image Klein support",
 * comment "Structure (from dit.py)"): timestep conditioning, per-stream
 * modulation vectors, input embedders, the image output layer; comment
 * "Sampling": the sigma schedule and the flow-map Euler update.
 * ------------------------------------------------------------------------ */

/* The non-block weights, device bf16 [out, in] (no biases), 16-byte aligned.
 * ref_time_in_* are NULL for a checkpoint without the flow-map timestep. */
typedef struct flux3_cond_weights {
  const void *time_in_in;       /* [3072, 256]   */
  const void *time_in_out;      /* [3072, 3072]  */
  const void *ref_time_in_in;   /* [3072, 256] or NULL */
  const void *ref_time_in_out;  /* [3072, 3072] or NULL */
  const void *early_mod[3];     /* [9216, 3072] per stream (image, image_cond, txt) */
  const void *single_mod[3];    /* [9216, 3072] per stream */
  const void *emb_in_image;     /* [3072, 128]   */
  const void *emb_in_image_cond;/* [3072, 128]   */
  const void *txt_in;           /* [3072, 20480] */
  const void *final_adaln;      /* [6144, 3072]  */
  const void *final_linear;     /* [128, 3072]   */
} flux3_cond_weights;

typedef struct flux3_cond flux3_cond;

/* Bytes of the caller-owned buffer flux3_cond_init copies the weights into. */
FLUX3_API size_t flux3_cond_packed_bytes(void);

/* Creates the conditioning handle; copies the weights into `packed`
 * (flux3_cond_packed_bytes() bytes, device, 16-byte aligned) on `stream`.  The
 * source weights may be freed once the stream has passed the copies. */
FLUX3_API flux3_status flux3_cond_init(flux3_cond **out, const flux3_cond_weights *w, void *packed,
                                       size_t packed_bytes, void *stream);

/* Frees the conditioning handle's host state (NULL is allowed); the packed
 * weight buffer stays the caller's. */
FLUX3_API void flux3_cond_destroy(flux3_cond *c);

/* Device workspace of flux3_conditioning (a few tens of KB). */
FLUX3_API size_t flux3_cond_workspace_bytes(void);

/* The modulation vectors of one call.  Per stream s the conditioning vector
 * vec_s = time_in(emb(t_s)) (+ ref_time_in(emb(t_next)) with the flow-map
 * weights), t_image = t and t_image_cond = t_txt = 0, emb(t) = [cos, sin] of
 * 1000 t 10000^(-i/128), i < 128, time_in = Linear, SiLU, Linear; then
 *   early_mod[s]  = early_stream_modulations[s](SiLU(vec_s))    device float32 [3, 9216]
 *   single_mod[s] = single_stream_modulations[s](SiLU(vec_s))   device float32 [3, 9216]
 *   final_mod     = adaLN(SiLU(vec_image)) = shift | scale, then 3072 zeros
 *                                                               device float32 [9216]
 * (SiLU before the modulation linears is a reading: the pages name only the
 * linear; the output layer's adaLN is stated as SiLU, Linear.)  t_next is
 * ignored without ref_time_in. */
FLUX3_API flux3_status flux3_conditioning(const flux3_cond *c, float t, float t_next, float *early_mod,
                                          float *single_mod, float *final_mod, void *workspace, size_t ws_bytes,
                                          void *stream);

/* The input embedders: x[row] = emb_s(input_s[k]) for the k-th token of
 * stream s in sequence order (emb_in.image / emb_in.image_cond on 128 latent
 * channels, txt_in on 20480 text features), float32, written for all T rows.
 *   inputs  host array [3] of device bf16 pointers indexed by flux3_stream:
 *           image [T_image, 128], image_cond [T_ref, 128], txt [T_txt, 20480]
 *           (16-byte aligned; NULL for a stream without tokens)
 *   x       device float32 [T, 3072]; segs as flux3_block_forward. */
FLUX3_API flux3_status flux3_embed_tokens(const flux3_cond *c, const void *const *inputs, int T,
                                          const flux3_segment *segs, int n_segs, float *x, void *stream);

/* Device workspace of flux3_final_layer for T tokens. */
FLUX3_API size_t flux3_final_layer_workspace_bytes(int T);

/* The output layer on the image tokens (in sequence order): h = (1 + scale) *
 * LayerNorm(x) + shift (eps 1e-6, shift | scale = final_mod's first 6144
 * values), velocity = h final_linear^T.
 *   x         device float32 [T, 3072]
 *   final_mod device float32 [9216] as flux3_conditioning writes it
 *   velocity  device float32 [T_image, 128] */
FLUX3_API flux3_status flux3_final_layer(const flux3_cond *c, const float *x, int T, const flux3_segment *segs,
                                         int n_segs, const float *final_mod, float *velocity, void *workspace,
                                         size_t ws_bytes, void *stream);

/* Device workspace of flux3_transformer_forward for T tokens with the joint
 * handle's configuration. */
FLUX3_API size_t flux3_transformer_workspace_bytes(const flux3_config *joint_cfg, int T);

/* One transformer call: conditioning, embedders, n_mode_blocks per-mode
 * blocks (flux3_mode_blocks_forward with the early modulations; 0 skips
 * them), the joint handle's blocks (single-stream modulations), the output
 * layer.  Arguments as the functions above; velocity device float32
 * [T_image, 128].  Each mode's token count must fit its mode handle's
 * max_tokens and T the joint handle's. */
FLUX3_API flux3_status flux3_transformer_forward(const flux3_cond *c, const flux3_handle *const *mode_handles,
                                                 int n_mode_blocks, const flux3_handle *joint,
                                                 const void *const *inputs, int T, const flux3_segment *segs,
                                                 int n_segs, const float *pos_ids, float t, float t_next,
                                                 float *velocity, void *workspace, size_t ws_bytes, void *stream);

/* Host: sigma_k = alpha t_k / (1 + (alpha - 1) t_k), t_k = 1 - k / steps,
 * k = 0..steps, into sigmas[steps + 1] (host float32; alpha 6.93 in the
 * pages). */
FLUX3_API flux3_status flux3_sigma_schedule(int steps, double alpha, float *sigmas);

/* latent[i] += (sigma_next - sigma) * velocity[i], i < n (device float32; the
 * difference is taken in double and rounded to float, the update is one fused
 * multiply-add).  next_input (device bf16 [n], or NULL): also receives the new
 * latent rounded to bf16, the image input of the next call. */
FLUX3_API flux3_status flux3_euler_step(float *latent, const float *velocity, size_t n, float sigma,
                                        float sigma_next, void *next_input, void *stream);

/* input[i] = bf16 rounding (nearest even) of latent[i], i < n: the first call's
 * image input from the initial latents. */
FLUX3_API flux3_status flux3_latents_to_bf16(const float *latent, size_t n, void *input, void *stream);

/* ------------------------------------------------------------------------
 * Several samples in one call: the base model guides its sampler with a
 * pack of two samples, the empty prompt's and the prompt's ("FLUX.3 Image
 * Klein support", comment "Sampling (sampling.py, pipeline.py)"), and a
 * token attends only within its own sample (comment "Structure (from
 * dit.py)").  The samples' tokens are concatenated: sample b owns rows
 * [sample_start[b], sample_start[b+1]).
 * ------------------------------------------------------------------------ */
#define FLUX3_MAX_SAMPLES 16

/* flux3_stack_forward over a batch of samples: LayerNorm and both projection
 * GEMMs run once over all T rows, attention runs per sample.
 *   sample_start host int [n_samples + 1], 0 = [0] < [1] < ... < [n] = T
 *   segs         as flux3_block_forward (stream = the token's mode), each
 *                segment inside one sample
 *   mod          device float32 [3 * n_samples, 9216]: row 3 b + stream
 * The rows of each sample come out as a flux3_stack_forward call on that
 * sample alone would leave them. */
FLUX3_API flux3_status flux3_stack_forward_batch(const flux3_handle *h, int first_block, int n_blocks, float *x,
                                                 int T, const flux3_segment *segs, int n_segs,
                                                 const int *sample_start, int n_samples, const float *pos_ids,
                                                 const float *mod, void *workspace, size_t ws_bytes, void *stream);

/* Device workspace of flux3_transformer_forward_batch. */
FLUX3_API size_t flux3_transformer_batch_workspace_bytes(const flux3_config *joint_cfg, int T, int n_samples);

/* flux3_transformer_forward over a batch of samples: conditioning per sample
 * (t[b], t_next[b]: host float arrays [n_samples]), embedders, per-mode blocks
 * per sample, the joint blocks batched (flux3_stack_forward_batch), the
 * output layer per sample.
 *   inputs    host array [n_samples * 3] of device bf16 pointers: sample b's
 *             image, image_cond, txt inputs at 3 b + stream
 *   velocity  device float32 [sum of the samples' image tokens, 128], the
 *             samples' image tokens one sample after the other */
FLUX3_API flux3_status flux3_transformer_forward_batch(const flux3_cond *c, const flux3_handle *const *mode_handles,
                                                       int n_mode_blocks, const flux3_handle *joint,
                                                       const void *const *inputs, int T, const flux3_segment *segs,
                                                       int n_segs, const int *sample_start, int n_samples,
                                                       const float *pos_ids, const float *t, const float *t_next,
                                                       float *velocity, void *workspace, size_t ws_bytes,
                                                       void *stream);

/* The guided update: latent[i] += (sigma_next - sigma) * (v_uncond[i] +
 * guidance (v_cond[i] - v_uncond[i])), i < n (device float32).  The pages
 * give the pack and the guidance scale (3.5), not the combination; this is
 * the classifier-free guidance form.  next_input as for flux3_euler_step. */
FLUX3_API flux3_status flux3_cfg_euler_step(float *latent, const float *v_uncond, const float *v_cond, size_t n,
                                            float guidance, float sigma, float sigma_next, void *next_input,
                                            void *stream);

/* Largest T flux3_block_forward_noalloc accepts (its scratch is ~51 MB). */
#define FLUX3_NOALLOC_MAX_TOKENS 512

/* flux3_block_forward for callers that must not allocate device memory.
 * The paper has no counterpart: this is a deployment variant.
 *
 * Some callers cannot call cudaMalloc (or any allocating routine) at the point
 * where they run a block: plug-in hosts whose device memory is owned by another
 * allocator, runtimes that reserve all memory up front and forbid allocation
 * afterwards, and real-time loops where an allocation's latency or failure is
 * not acceptable.  This entry point takes the same arguments as
 * flux3_block_forward minus the workspace: its scratch (stream ids, RoPE tables,
 * modulated input, q/k/v, attention + SwiGLU output) lives in a fixed device
 * array inside the library, sized for FLUX3_NOALLOC_MAX_TOKENS tokens, which
 * every GPU that loads the library holds until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   - T > FLUX3_NOALLOC_MAX_TOKENS returns FLUX3_ERR_WORKSPACE; a handle with
 *     NVFP4 or fp8r weights returns FLUX3_ERR_UNSUPPORTED (its expanded weights
 *     would not fit); other errors as flux3_block_forward.
 *   - Every call looks up the array's device address in the current CUDA
 *     context (cudaGetSymbolAddress; an address belongs to a context, which a
 *     device reset or a host's own context replaces).  The first call on a
 *     device may load the library's device code, so make it before any
 *     stream capture.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero: every call writes each scratch
 *     value before reading it.  Calls whose kernels overlap on the GPU (other
 *     streams, or other host threads) race on the array: serialise them. */
FLUX3_API flux3_status flux3_block_forward_noalloc(const flux3_handle *h, int block_idx, float *x, int T,
                                                   const flux3_segment *segs, int n_segs,
                                                   const float *pos_ids, const float *mod, void *stream);

/* Synchronises `stream`, then reads and clears the device error word.
 * Returns FLUX3_OK, FLUX3_ERR_TIMEOUT, FLUX3_ERR_DEVICE or FLUX3_ERR_CUDA. */
FLUX3_API flux3_status flux3_check_error(void *stream);

/* A static, NUL-terminated English name of a status code (never NULL; unknown
 * codes give a generic string).  The caller does not free it. */
FLUX3_API const char *flux3_status_string(flux3_status s);

/* Frees the handle's host state.  Does not touch caller-owned device memory. */
FLUX3_API void flux3_destroy(flux3_handle *h);

/* ------------------------------------------------------------------------
 * Step entry points: the stages of one block, exposed so each can be checked
 * on its own.  flux3_block_forward is flux3_prepare, flux3_ln_modulate,
 * flux3_in_projection, flux3_attention and flux3_out_projection in sequence
 * (its own launches after the first are programmatic dependents of the launch
 * before them, so each kernel's set-up overlaps the previous one's tail).
 * ------------------------------------------------------------------------ */

/* Per-token stream id from the segment table (validated as above).
 *   stream_id  device uint8 [T] (output) */
FLUX3_API flux3_status flux3_stream_ids(const flux3_segment *segs, int n_segs, int T,
                                        uint8_t *stream_id, void *stream);

/* RoPE tables: for token t, pair p = 16 a + j (axis a in t, h, w, l; j < 16):
 *   angle = pos_ids[t, a] * theta^(-2j/32);  cos_tab[t, p], sin_tab[t, p].
 * The 4 axes of 32 dims and theta are from the issue's "Structure" comment;
 * the frequency ladder within an axis is the standard RoPE one.
 *   pos_ids device float32 [T, 4]; cos_tab, sin_tab device float32 [T, 64] (outputs) */
FLUX3_API flux3_status flux3_rope_tables(const float *pos_ids, int T, float theta,
                                         float *cos_tab, float *sin_tab, void *stream);

/* flux3_stream_ids and flux3_rope_tables in one launch (what the forward
 * calls run once per call): stream_id [T], cos_tab, sin_tab [T, 64] as above. */
FLUX3_API flux3_status flux3_prepare(const flux3_segment *segs, int n_segs, int T, const float *pos_ids,
                                     float theta, uint8_t *stream_id, float *cos_tab, float *sin_tab,
                                     void *stream);

/* LayerNorm (no affine) + per-stream modulation:
 *   h[t] = (1 + scale[s(t)]) * (x[t] - mean) / sqrt(var + eps) + shift[s(t)]
 *   x device float32 [T, 3072]; stream_id device uint8 [T];
 *   mod device float32 [3, 9216]; h device bf16 [T, 3072] (output). */
FLUX3_API flux3_status flux3_ln_modulate(const float *x, int T, const uint8_t *stream_id,
                                         const float *mod, float eps, void *h, void *stream);

/* Step entry points flux3_in_projection and flux3_out_projection use the
 * handle's packed bf16 weights: with an NVFP4 or fp8r handle they return
 * FLUX3_ERR_UNSUPPORTED (the forward calls expand those weights themselves). */

/* The block's input projections with their fused epilogues (one tensor-core
 * GEMM over the concatenated [Wq; Wk; Wv; Wmlp_in] rows):
 *   qkv[t, 0:3072]      = RoPE4(RMSNorm(h Wq^T) * query_norm)   per head (bf16)
 *   qkv[t, 3072:6144]   = RoPE4(RMSNorm(h Wk^T) * key_norm)     per head (bf16)
 *   qkv[t, 6144:9216]   = h Wv^T                                 (bf16)
 *   cat[t, 3072:12288]  = silu(a) * b,  [a | b] = h Wmlp_in^T    (bf16)
 *   h device bf16 [T, 3072]; cos_tab/sin_tab from flux3_rope_tables;
 *   qkv device bf16 [T, 9216]; cat device bf16 [T, 12288] (columns 0..3071
 *   are left untouched: the attention writes them). */
FLUX3_API flux3_status flux3_in_projection(const flux3_handle *h, int block_idx, const void *hmod,
                                           int T, const float *cos_tab, const float *sin_tab,
                                           void *qkv, void *cat, void *stream);

/* Bidirectional attention over all T tokens, per head (24 x 128), scale
 * 1/sqrt(128), no mask:
 *   cat[t, 128 h : 128 h + 128] = softmax(q^_h k^_h^T / sqrt(128)) v_h
 *   qkv device bf16 [T, 9216] laid out as above; cat device bf16 [T, 12288]
 *   (only columns 0..3071 are written).
 * split_buf: optional device scratch (16-byte aligned, split_bytes long, at
 * most FLUX3_SPLIT_BYTES used; NULL for none).  With it, the (query-tile
 * pair, head) units of the last, partial wave of one CTA per SM are split
 * into key ranges that fill the wave; each range stores its unnormalised
 * rows with their running max and sum there, and a merge combines the ranges
 * in a fixed order.  The block forward calls do the same with their
 * workspace.  Without it no unit is split. */
FLUX3_API flux3_status flux3_attention(const void *qkv, int T, void *cat, void *split_buf, size_t split_bytes,
                                       void *stream);

/* Bytes of scratch the out-projection's K split can use (96 partial tiles of
 * 256 x 256 float32); the block workspace already holds it. */
#define FLUX3_SPLIT_BYTES ((size_t)96 * 256 * 256 * 4)

/* Output projection and gated residual (one GEMM with K = 3072 + 9216 over
 * cat = [attention | SwiGLU] against [Wattn_out | Wmlp_out]):
 *   x[t] += gate[s(t)] * (cat[t] [Wattn_out | Wmlp_out]^T)
 *   cat device bf16 [T, 12288]; stream_id device uint8 [T];
 *   mod device float32 [3, 9216]; x device float32 [T, 3072] (in place).
 * split_buf: optional device scratch (16-byte aligned, split_bytes long, at
 * most FLUX3_SPLIT_BYTES used; NULL for none).  With it, when the output
 * tiles leave SMs idle in the GEMM's last round of tiles, those tiles are
 * split along K, their float32 partial sums stored there and summed in a fixed
 * order (deterministic) before the gated residual; the block forward calls do
 * the same with their workspace.  Without it no tile is split. */
FLUX3_API flux3_status flux3_out_projection(const flux3_handle *h, int block_idx, const void *cat,
                                            int T, const uint8_t *stream_id, const float *mod,
                                            float *x, void *split_buf, size_t split_bytes,
                                            void *stream);

/* Plain tensor-core GEMM C = A B^T (fp32 accumulation, bf16 result), the core
 * the projections are built on.  A device bf16 [M, K], B device bf16 [N, K],
 * C device bf16 [M, N]; M >= 1, N % 256 == 0, K % 64 == 0, 16-byte aligned. */
FLUX3_API flux3_status flux3_gemm_bf16(const void *A, const void *B, void *C, int M, int N, int K,
                                       void *stream);

/* Diagnostics for the failure path: launches one CTA that waits on a pipeline
 * barrier nothing ever arrives at.  The wait gives up after timeout_us
 * (1 .. 1e6) and records a timeout in the device error word, exactly as a
 * stalled pipeline in a forward kernel would; flux3_check_error() then
 * returns FLUX3_ERR_TIMEOUT and the CUDA context stays usable. */
FLUX3_API flux3_status flux3_selftest_wait_timeout(int timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FLUX3_H */
