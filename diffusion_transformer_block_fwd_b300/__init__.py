"""Python binding of libflux3.so, the sm_103a library for the FLUX.3 Image
Klein joint single_block forward pass (C ABI: include/flux3.h).

The functions below carry the C entry points' names and only marshal
arguments (ctypes); every step of the block runs in the library's CUDA
kernels.  PyTorch is used for device memory and streams only.  There is no
fallback: if the library is missing or cannot be loaded, importing the
binding's functions raises.
"""

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libflux3.so")

FLUX3_OK = 0
FLUX3_ERR_INVALID_ARG = -1
FLUX3_ERR_UNSUPPORTED = -2
FLUX3_ERR_ALIGNMENT = -3
FLUX3_ERR_WORKSPACE = -4
FLUX3_ERR_CUDA = -5
FLUX3_ERR_TIMEOUT = -6
FLUX3_ERR_DEVICE = -7

FLUX3_W_BF16 = 0
FLUX3_W_NVFP4 = 1
FLUX3_W_FP8R = 2
FLUX3_STREAM_IMAGE = 0
FLUX3_STREAM_IMAGE_COND = 1
FLUX3_STREAM_TXT = 2
FLUX3_MAX_SEGMENTS = 32
FLUX3_NOALLOC_MAX_TOKENS = 512
FLUX3_MAX_SAMPLES = 16

EXPORTED = (
    "flux3_default_config", "flux3_packed_weight_bytes", "flux3_workspace_bytes", "flux3_block_init",
    "flux3_block_forward", "flux3_stack_forward", "flux3_check_error", "flux3_status_string", "flux3_destroy",
    "flux3_stream_ids", "flux3_rope_tables", "flux3_prepare", "flux3_ln_modulate", "flux3_in_projection", "flux3_attention",
    "flux3_out_projection", "flux3_gemm_bf16", "flux3_selftest_wait_timeout", "flux3_block_forward_noalloc",
    "flux3_block_init_nvfp4", "flux3_quantize_nvfp4", "flux3_dequantize_block", "flux3_mode_blocks_forward",
    "flux3_block_init_fp8r", "flux3_quantize_fp8r",
    "flux3_cond_packed_bytes", "flux3_cond_init", "flux3_cond_destroy", "flux3_cond_workspace_bytes",
    "flux3_conditioning", "flux3_embed_tokens", "flux3_final_layer_workspace_bytes", "flux3_final_layer",
    "flux3_transformer_workspace_bytes", "flux3_transformer_forward", "flux3_sigma_schedule", "flux3_euler_step",
    "flux3_stack_forward_batch", "flux3_transformer_batch_workspace_bytes", "flux3_transformer_forward_batch",
    "flux3_cfg_euler_step", "flux3_latents_to_bf16",
)


class Flux3Error(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class flux3_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("mlp_hidden", ctypes.c_int), ("n_blocks", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("wfmt", ctypes.c_int), ("rope_theta", ctypes.c_float), ("eps_ln", ctypes.c_float),
                ("eps_rms", ctypes.c_float)]


class flux3_block_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q_proj", "k_proj", "v_proj", "attn_out", "mlp_in", "mlp_out",
                                                "query_norm", "key_norm")]


class flux3_nvfp4_tensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


NVFP4_MATRICES = ("q_proj", "k_proj", "v_proj", "attn_out", "mlp_in", "mlp_out")


class flux3_block_weights_nvfp4(ctypes.Structure):
    _fields_ = [(n, flux3_nvfp4_tensor) for n in NVFP4_MATRICES] + [("query_norm", ctypes.c_void_p),
                                                                    ("key_norm", ctypes.c_void_p)]


class flux3_fp8r_tensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class flux3_block_weights_fp8r(ctypes.Structure):
    _fields_ = [(n, flux3_fp8r_tensor) for n in NVFP4_MATRICES] + [("query_norm", ctypes.c_void_p),
                                                                   ("key_norm", ctypes.c_void_p)]


COND_KEYS = ("time_in_in", "time_in_out", "ref_time_in_in", "ref_time_in_out", "early_mod", "single_mod",
             "emb_in_image", "emb_in_image_cond", "txt_in", "final_adaln", "final_linear")


class flux3_cond_weights(ctypes.Structure):
    _fields_ = [("time_in_in", ctypes.c_void_p), ("time_in_out", ctypes.c_void_p),
                ("ref_time_in_in", ctypes.c_void_p), ("ref_time_in_out", ctypes.c_void_p),
                ("early_mod", ctypes.c_void_p * 3), ("single_mod", ctypes.c_void_p * 3),
                ("emb_in_image", ctypes.c_void_p), ("emb_in_image_cond", ctypes.c_void_p),
                ("txt_in", ctypes.c_void_p), ("final_adaln", ctypes.c_void_p), ("final_linear", ctypes.c_void_p)]


class flux3_segment(ctypes.Structure):
    _fields_ = [("start", ctypes.c_int), ("len", ctypes.c_int), ("stream", ctypes.c_int)]


_lib = None


def lib():
    """The loaded library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libflux3.so not built ({LIB_PATH}); run "
                               "python -m diffusion_transformer_block_fwd_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        cfgp = ctypes.POINTER(flux3_config)
        segp = ctypes.POINTER(flux3_segment)
        sig = {
            "flux3_default_config": (None, [cfgp]),
            "flux3_packed_weight_bytes": (sz, [cfgp]),
            "flux3_workspace_bytes": (sz, [cfgp, i]),
            "flux3_block_init": (i, [ctypes.POINTER(vp), cfgp, ctypes.POINTER(flux3_block_weights), i, vp, sz, vp]),
            "flux3_block_forward": (i, [vp, i, vp, i, segp, i, vp, vp, vp, sz, vp]),
            "flux3_stack_forward": (i, [vp, i, i, vp, i, segp, i, vp, vp, vp, sz, vp]),
            "flux3_check_error": (i, [vp]),
            "flux3_status_string": (ctypes.c_char_p, [i]),
            "flux3_destroy": (None, [vp]),
            "flux3_stream_ids": (i, [segp, i, i, vp, vp]),
            "flux3_rope_tables": (i, [vp, i, f, vp, vp, vp]),
            "flux3_prepare": (i, [segp, i, i, vp, f, vp, vp, vp, vp]),
            "flux3_ln_modulate": (i, [vp, i, vp, vp, f, vp, vp]),
            "flux3_in_projection": (i, [vp, i, vp, i, vp, vp, vp, vp, vp]),
            "flux3_attention": (i, [vp, i, vp, vp, sz, vp]),
            "flux3_out_projection": (i, [vp, i, vp, i, vp, vp, vp, vp, sz, vp]),
            "flux3_gemm_bf16": (i, [vp, vp, vp, i, i, i, vp]),
            "flux3_selftest_wait_timeout": (i, [i, vp]),
            "flux3_block_forward_noalloc": (i, [vp, i, vp, i, segp, i, vp, vp, vp]),
            "flux3_block_init_nvfp4": (i, [ctypes.POINTER(vp), cfgp, ctypes.POINTER(flux3_block_weights_nvfp4), i,
                                           vp, sz, vp]),
            "flux3_quantize_nvfp4": (i, [vp, i, i, vp, vp, vp, vp]),
            "flux3_dequantize_block": (i, [vp, i, vp, vp, vp]),
            "flux3_mode_blocks_forward": (i, [ctypes.POINTER(vp), i, vp, i, segp, i, vp, vp, vp, sz, vp]),
            "flux3_block_init_fp8r": (i, [ctypes.POINTER(vp), cfgp, ctypes.POINTER(flux3_block_weights_fp8r), i,
                                          vp, sz, vp]),
            "flux3_quantize_fp8r": (i, [vp, i, i, vp, vp, vp]),
            "flux3_cond_packed_bytes": (sz, []),
            "flux3_cond_init": (i, [ctypes.POINTER(vp), ctypes.POINTER(flux3_cond_weights), vp, sz, vp]),
            "flux3_cond_destroy": (None, [vp]),
            "flux3_cond_workspace_bytes": (sz, []),
            "flux3_conditioning": (i, [vp, f, f, vp, vp, vp, vp, sz, vp]),
            "flux3_embed_tokens": (i, [vp, ctypes.POINTER(vp), i, segp, i, vp, vp]),
            "flux3_final_layer_workspace_bytes": (sz, [i]),
            "flux3_final_layer": (i, [vp, vp, i, segp, i, vp, vp, vp, sz, vp]),
            "flux3_transformer_workspace_bytes": (sz, [cfgp, i]),
            "flux3_transformer_forward": (i, [vp, ctypes.POINTER(vp), i, vp, ctypes.POINTER(vp), i, segp, i, vp, f, f,
                                              vp, vp, sz, vp]),
            "flux3_sigma_schedule": (i, [i, ctypes.c_double, ctypes.POINTER(ctypes.c_float)]),
            "flux3_euler_step": (i, [vp, vp, sz, f, f, vp, vp]),
            "flux3_latents_to_bf16": (i, [vp, sz, vp, vp]),
            "flux3_stack_forward_batch": (i, [vp, i, i, vp, i, segp, i, ctypes.POINTER(i), i, vp, vp, vp, sz, vp]),
            "flux3_transformer_batch_workspace_bytes": (sz, [cfgp, i, i]),
            "flux3_transformer_forward_batch": (i, [vp, ctypes.POINTER(vp), i, vp, ctypes.POINTER(vp), i, segp, i,
                                                    ctypes.POINTER(i), i, vp, ctypes.POINTER(f), ctypes.POINTER(f),
                                                    vp, vp, sz, vp]),
            "flux3_cfg_euler_step": (i, [vp, vp, vp, sz, f, f, f, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status):
    return lib().flux3_status_string(int(status)).decode()


def _check(status, what):
    if status != FLUX3_OK:
        raise Flux3Error(status, what)


def segments_array(segments):
    """[(start, len, stream), ...] -> ctypes array of flux3_segment."""
    arr = (flux3_segment * max(1, len(segments)))()
    for k, (s, n, st) in enumerate(segments):
        arr[k].start, arr[k].len, arr[k].stream = int(s), int(n), int(st)
    return arr


# ---------------------------------------------------------------- C entry points
def flux3_default_config():
    cfg = flux3_config()
    lib().flux3_default_config(ctypes.byref(cfg))
    return cfg


def flux3_packed_weight_bytes(cfg):
    return int(lib().flux3_packed_weight_bytes(ctypes.byref(cfg)))


def flux3_workspace_bytes(cfg, T):
    return int(lib().flux3_workspace_bytes(ctypes.byref(cfg), int(T)))


def flux3_block_init(cfg, weights, packed_ptr, packed_bytes, stream=0):
    """weights: list of dicts of device pointers (ints) keyed like
    flux3_block_weights.  Returns the handle (an int)."""
    n = len(weights)
    arr = (flux3_block_weights * n)()
    for b, w in enumerate(weights):
        for k, _ in flux3_block_weights._fields_:
            setattr(arr[b], k, int(w[k]))
    h = ctypes.c_void_p()
    _check(lib().flux3_block_init(ctypes.byref(h), ctypes.byref(cfg), arr, n, packed_ptr, packed_bytes, stream),
           "flux3_block_init")
    return h.value


def flux3_block_init_nvfp4(cfg, weights, packed_ptr, packed_bytes, stream=0):
    """weights: list of dicts: for each matrix name a (codes, scales, global)
    triple of device pointers, and query_norm / key_norm device pointers."""
    n = len(weights)
    arr = (flux3_block_weights_nvfp4 * n)()
    for b, w in enumerate(weights):
        for k in NVFP4_MATRICES:
            c, sc, g = w[k]
            t = getattr(arr[b], k)
            t.codes, t.scales, t.global_scale = int(c), int(sc), int(g)
        arr[b].query_norm, arr[b].key_norm = int(w["query_norm"]), int(w["key_norm"])
    h = ctypes.c_void_p()
    _check(lib().flux3_block_init_nvfp4(ctypes.byref(h), ctypes.byref(cfg), arr, n, packed_ptr, packed_bytes, stream),
           "flux3_block_init_nvfp4")
    return h.value


def flux3_quantize_nvfp4(w, rows, cols, codes, scales, global_scale, stream=0):
    _check(lib().flux3_quantize_nvfp4(w, rows, cols, codes, scales, global_scale, stream), "flux3_quantize_nvfp4")


def flux3_block_init_fp8r(cfg, weights, packed_ptr, packed_bytes, stream=0):
    """weights: list of dicts: for each matrix name a (codes, scales) pair of
    device pointers, and query_norm / key_norm device pointers."""
    n = len(weights)
    arr = (flux3_block_weights_fp8r * n)()
    for b, w in enumerate(weights):
        for k in NVFP4_MATRICES:
            c, sc = w[k]
            t = getattr(arr[b], k)
            t.codes, t.scales = int(c), int(sc)
        arr[b].query_norm, arr[b].key_norm = int(w["query_norm"]), int(w["key_norm"])
    h = ctypes.c_void_p()
    _check(lib().flux3_block_init_fp8r(ctypes.byref(h), ctypes.byref(cfg), arr, n, packed_ptr, packed_bytes, stream),
           "flux3_block_init_fp8r")
    return h.value


def flux3_quantize_fp8r(w, rows, cols, codes, scales, stream=0):
    _check(lib().flux3_quantize_fp8r(w, rows, cols, codes, scales, stream), "flux3_quantize_fp8r")


def _ptr3(ptrs):
    return (ctypes.c_void_p * 3)(*[(int(p) if p else None) for p in ptrs])


def flux3_cond_packed_bytes():
    return int(lib().flux3_cond_packed_bytes())


def flux3_cond_init(weights, packed_ptr, packed_bytes, stream=0):
    """weights: dict of device pointers keyed like flux3_cond_weights
    (early_mod / single_mod: three pointers each; ref_time_in_*: 0 or None
    without the flow-map timestep).  Returns the handle (an int)."""
    w = flux3_cond_weights()
    for k in COND_KEYS:
        v = weights.get(k)
        if k in ("early_mod", "single_mod"):
            for j in range(3):
                getattr(w, k)[j] = int(v[j])
        else:
            setattr(w, k, int(v) if v else None)
    h = ctypes.c_void_p()
    _check(lib().flux3_cond_init(ctypes.byref(h), ctypes.byref(w), packed_ptr, packed_bytes, stream),
           "flux3_cond_init")
    return h.value


def flux3_cond_destroy(c):
    lib().flux3_cond_destroy(c)


def flux3_cond_workspace_bytes():
    return int(lib().flux3_cond_workspace_bytes())


def flux3_conditioning(c, t, t_next, early_mod, single_mod, final_mod, workspace, ws_bytes, stream=0):
    _check(lib().flux3_conditioning(c, t, t_next, early_mod, single_mod, final_mod, workspace, ws_bytes, stream),
           "flux3_conditioning")


def flux3_embed_tokens(c, inputs, T, segments, x, stream=0):
    segs = segments_array(segments)
    _check(lib().flux3_embed_tokens(c, _ptr3(inputs), T, segs, len(segments), x, stream), "flux3_embed_tokens")


def flux3_final_layer_workspace_bytes(T):
    return int(lib().flux3_final_layer_workspace_bytes(int(T)))


def flux3_final_layer(c, x, T, segments, final_mod, velocity, workspace, ws_bytes, stream=0):
    segs = segments_array(segments)
    _check(lib().flux3_final_layer(c, x, T, segs, len(segments), final_mod, velocity, workspace, ws_bytes, stream),
           "flux3_final_layer")


def flux3_transformer_workspace_bytes(cfg, T):
    return int(lib().flux3_transformer_workspace_bytes(ctypes.byref(cfg), int(T)))


def flux3_transformer_forward(c, mode_handles, n_mode_blocks, joint, inputs, T, segments, pos_ids, t, t_next,
                              velocity, workspace, ws_bytes, stream=0):
    segs = segments_array(segments)
    _check(lib().flux3_transformer_forward(c, _ptr3(mode_handles), n_mode_blocks, joint, _ptr3(inputs), T, segs,
                                           len(segments), pos_ids, t, t_next, velocity, workspace, ws_bytes,
                                           stream), "flux3_transformer_forward")


def flux3_sigma_schedule(steps, alpha=6.93):
    out = (ctypes.c_float * (steps + 1))()
    _check(lib().flux3_sigma_schedule(steps, alpha, out), "flux3_sigma_schedule")
    return list(out)


def flux3_euler_step(latent, velocity, n, sigma, sigma_next, next_input=None, stream=0):
    _check(lib().flux3_euler_step(latent, velocity, n, sigma, sigma_next, next_input, stream), "flux3_euler_step")


def flux3_latents_to_bf16(latent, n, inp, stream=0):
    _check(lib().flux3_latents_to_bf16(latent, n, inp, stream), "flux3_latents_to_bf16")


def _ints(v):
    return (ctypes.c_int * len(v))(*[int(a) for a in v])


def _floats(v):
    return (ctypes.c_float * len(v))(*[float(a) for a in v])


def flux3_stack_forward_batch(h, first_block, n_blocks, x, T, segments, sample_start, pos_ids, mod, workspace,
                              ws_bytes, stream=0):
    segs = segments_array(segments)
    _check(lib().flux3_stack_forward_batch(h, first_block, n_blocks, x, T, segs, len(segments), _ints(sample_start),
                                           len(sample_start) - 1, pos_ids, mod, workspace, ws_bytes, stream),
           "flux3_stack_forward_batch")


def flux3_transformer_batch_workspace_bytes(cfg, T, n_samples):
    return int(lib().flux3_transformer_batch_workspace_bytes(ctypes.byref(cfg), int(T), int(n_samples)))


def flux3_transformer_forward_batch(c, mode_handles, n_mode_blocks, joint, inputs, T, segments, sample_start,
                                    pos_ids, t, t_next, velocity, workspace, ws_bytes, stream=0):
    """inputs: per sample three device pointers (image, image_cond, txt);
    t, t_next: per-sample timesteps."""
    flat = [p for per in inputs for p in per]
    ptrs = (ctypes.c_void_p * len(flat))(*[(int(p) if p else None) for p in flat])
    segs = segments_array(segments)
    _check(lib().flux3_transformer_forward_batch(c, _ptr3(mode_handles), n_mode_blocks, joint, ptrs, T, segs,
                                                 len(segments), _ints(sample_start), len(sample_start) - 1, pos_ids,
                                                 _floats(t), _floats(t_next), velocity, workspace, ws_bytes, stream),
           "flux3_transformer_forward_batch")


def flux3_cfg_euler_step(latent, v_uncond, v_cond, n, guidance, sigma, sigma_next, next_input=None, stream=0):
    _check(lib().flux3_cfg_euler_step(latent, v_uncond, v_cond, n, guidance, sigma, sigma_next, next_input, stream),
           "flux3_cfg_euler_step")


def flux3_dequantize_block(h, block_idx, w_in, w_out, stream=0):
    _check(lib().flux3_dequantize_block(h, block_idx, w_in, w_out, stream), "flux3_dequantize_block")


def flux3_block_forward(h, block_idx, x, T, segments, pos_ids, mod, workspace, ws_bytes, stream=0):
    segs = segments_array(segments)
    _check(lib().flux3_block_forward(h, block_idx, x, T, segs, len(segments), pos_ids, mod, workspace, ws_bytes,
                                     stream), "flux3_block_forward")


def flux3_mode_blocks_forward(mode_handles, n_blocks, x, T, segments, pos_ids, early_mod, workspace, ws_bytes,
                              stream=0):
    """mode_handles: three handles (ints, or None for a mode without tokens),
    indexed by stream id."""
    hs = (ctypes.c_void_p * 3)(*[(int(h) if h else None) for h in mode_handles])
    segs = segments_array(segments)
    _check(lib().flux3_mode_blocks_forward(hs, n_blocks, x, T, segs, len(segments), pos_ids, early_mod, workspace,
                                           ws_bytes, stream), "flux3_mode_blocks_forward")


def flux3_stack_forward(h, first_block, n_blocks, x, T, segments, pos_ids, mod, workspace, ws_bytes, stream=0):
    segs = segments_array(segments)
    _check(lib().flux3_stack_forward(h, first_block, n_blocks, x, T, segs, len(segments), pos_ids, mod, workspace,
                                     ws_bytes, stream), "flux3_stack_forward")


def flux3_check_error(stream=0):
    return int(lib().flux3_check_error(stream))


def flux3_destroy(h):
    lib().flux3_destroy(h)


def flux3_stream_ids(segments, T, stream_id, stream=0):
    segs = segments_array(segments)
    _check(lib().flux3_stream_ids(segs, len(segments), T, stream_id, stream), "flux3_stream_ids")


def flux3_rope_tables(pos_ids, T, theta, cos_tab, sin_tab, stream=0):
    _check(lib().flux3_rope_tables(pos_ids, T, theta, cos_tab, sin_tab, stream), "flux3_rope_tables")


def flux3_prepare(segments, T, pos_ids, theta, stream_id, cos_tab, sin_tab, stream=0):
    """flux3_stream_ids and flux3_rope_tables in one launch."""
    segs = segments_array(segments)
    _check(lib().flux3_prepare(segs, len(segments), T, pos_ids, theta, stream_id, cos_tab, sin_tab, stream),
           "flux3_prepare")


def flux3_ln_modulate(x, T, stream_id, mod, eps, h, stream=0):
    _check(lib().flux3_ln_modulate(x, T, stream_id, mod, eps, h, stream), "flux3_ln_modulate")


def flux3_in_projection(h, block_idx, hmod, T, cos_tab, sin_tab, qkv, cat, stream=0):
    _check(lib().flux3_in_projection(h, block_idx, hmod, T, cos_tab, sin_tab, qkv, cat, stream),
           "flux3_in_projection")


def flux3_attention(qkv, T, cat, stream=0, split_buf=None, split_bytes=0):
    _check(lib().flux3_attention(qkv, T, cat, split_buf, split_bytes, stream), "flux3_attention")


FLUX3_SPLIT_BYTES = 96 * 256 * 256 * 4


def flux3_out_projection(h, block_idx, cat, T, stream_id, mod, x, stream=0, split_buf=None, split_bytes=0):
    _check(lib().flux3_out_projection(h, block_idx, cat, T, stream_id, mod, x, split_buf, split_bytes, stream),
           "flux3_out_projection")


def flux3_gemm_bf16(A, B, C, M, N, K, stream=0):
    _check(lib().flux3_gemm_bf16(A, B, C, M, N, K, stream), "flux3_gemm_bf16")


def flux3_block_forward_noalloc(h, block_idx, x, T, segments, pos_ids, mod, stream=0):
    """flux3_block_forward with the library's built-in scratch (T <= 512)."""
    segs = segments_array(segments)
    _check(lib().flux3_block_forward_noalloc(h, block_idx, x, T, segs, len(segments), pos_ids, mod, stream),
           "flux3_block_forward_noalloc")


def flux3_selftest_wait_timeout(timeout_us, stream=0):
    _check(lib().flux3_selftest_wait_timeout(timeout_us, stream), "flux3_selftest_wait_timeout")


from .model import Flux3Blocks, Flux3Conditioning, Flux3Transformer, quantize_fp8r, quantize_nvfp4  # noqa: E402,F401  (torch-owned buffers around the handle)
