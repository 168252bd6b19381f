"""Host-side checks of the C ABI that need no GPU: the library loads, every
entry point the header declares is exported, configuration and sizing
helpers, and argument validation that returns before anything is enqueued."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import diffusion_transformer_block_fwd_b300 as F3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from diffusion_transformer_block_fwd_b300 import build
    build.build()


def header_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"FLUX3_API\s+[\w\s\*]+?\b(flux3_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = header_functions()
    for must in ("flux3_block_init", "flux3_block_forward", "flux3_stack_forward", "flux3_check_error",
                 "flux3_workspace_bytes", "flux3_packed_weight_bytes"):
        assert must in names
    assert sorted(F3.EXPORTED) == names


def test_library_exports_every_declared_symbol():
    L = F3.lib()
    for n in header_functions():
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", F3.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (flux3_\w+)", out))
    assert exported == set(header_functions())


def test_default_config_and_sizes():
    cfg = F3.flux3_default_config()
    assert (cfg.hidden, cfg.heads, cfg.head_dim, cfg.mlp_hidden, cfg.n_blocks) == (3072, 24, 128, 9216, 28)
    assert abs(cfg.rope_theta - 1e4) < 1e-3 and abs(cfg.eps_ln - 1e-6) < 1e-12 and abs(cfg.eps_rms - 1e-6) < 1e-12
    per_block = (27648 * 3072 + 3072 * 12288) * 2 + 256 * 4
    assert F3.flux3_packed_weight_bytes(cfg) >= 28 * per_block
    assert F3.flux3_packed_weight_bytes(cfg) < 28 * (per_block + 3 * 256)
    ws = F3.flux3_workspace_bytes(cfg, 4608)
    assert ws >= 4608 * (1 + 2 * 64 * 4 + (3072 + 9216 + 12288) * 2)
    assert F3.flux3_workspace_bytes(cfg, 0) == 0
    assert F3.flux3_workspace_bytes(cfg, cfg.max_tokens + 1) == 0
    bad = F3.flux3_default_config()
    bad.hidden = 2048
    assert F3.flux3_packed_weight_bytes(bad) == 0


def test_status_strings():
    for s in range(-7, 1):
        assert F3.status_string(s)
    assert F3.status_string(0) == "ok"


def _segs(lst):
    return F3.segments_array(lst), len(lst)


@pytest.mark.parametrize("segments,T", [
    ([], 10),                                   # no segments
    ([(0, 5, 0), (6, 4, 2)], 10),                # gap
    ([(0, 5, 0), (4, 6, 2)], 10),                # overlap
    ([(0, 5, 0), (5, 4, 2)], 10),                # short of T
    ([(0, 5, 0), (5, 6, 2)], 10),                # past T
    ([(0, 10, 3)], 10),                          # bad stream
    ([(0, 0, 0), (0, 10, 1)], 10),               # empty segment
    ([(i, 1, 0) for i in range(33)], 33),        # too many
])
def test_segment_validation_rejects_bad_tables(segments, T):
    arr, n = _segs(segments)
    st = F3.lib().flux3_stream_ids(arr, n, T, ctypes.c_void_p(16), None)
    assert st == F3.FLUX3_ERR_INVALID_ARG
    st = F3.lib().flux3_prepare(arr, n, T, 16, ctypes.c_float(1e4), 16, 16, 16, None)
    assert st == F3.FLUX3_ERR_INVALID_ARG


def test_forward_argument_validation_before_any_launch():
    L = F3.lib()
    arr, n = _segs([(0, 8, 0)])
    # null handle
    assert L.flux3_block_forward(None, 0, 16, 8, arr, n, 16, 16, 16, 1 << 20, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_stack_forward(None, 0, 28, 16, 8, arr, n, 16, 16, 16, 1 << 20, None) == F3.FLUX3_ERR_INVALID_ARG
    # init: null output, null weights, wrong block count, small packed buffer, misaligned pointers
    cfg = F3.flux3_default_config()
    cfg.n_blocks = 1
    h = ctypes.c_void_p()
    w = (F3.flux3_block_weights * 1)()
    assert L.flux3_block_init(None, ctypes.byref(cfg), w, 1, 256, 1 << 40, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_block_init(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1 << 40, None) == F3.FLUX3_ERR_INVALID_ARG
    for k, _ in F3.flux3_block_weights._fields_:
        setattr(w[0], k, 4096)
    assert L.flux3_block_init(ctypes.byref(h), ctypes.byref(cfg), w, 2, 256, 1 << 40, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_block_init(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1024, None) == F3.FLUX3_ERR_WORKSPACE
    assert L.flux3_block_init(ctypes.byref(h), ctypes.byref(cfg), w, 1, 264, 1 << 40, None) == F3.FLUX3_ERR_ALIGNMENT
    w[0].mlp_in = 4100
    assert L.flux3_block_init(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1 << 40, None) == F3.FLUX3_ERR_ALIGNMENT
    bad = F3.flux3_default_config()
    bad.heads = 16
    assert L.flux3_block_init(ctypes.byref(h), ctypes.byref(bad), w, 28, 256, 1 << 40, None) == F3.FLUX3_ERR_UNSUPPORTED
    assert h.value is None
    # step entry points
    assert L.flux3_gemm_bf16(16, 16, 16, 128, 200, 64, None) == F3.FLUX3_ERR_INVALID_ARG     # N % 256
    assert L.flux3_gemm_bf16(16, 16, 16, 128, 256, 96, None) == F3.FLUX3_ERR_INVALID_ARG     # K % 64
    assert L.flux3_gemm_bf16(18, 16, 16, 128, 256, 64, None) == F3.FLUX3_ERR_ALIGNMENT
    assert L.flux3_attention(16, 0, 16, None, 0, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_attention(16, 8, 16, 24, 1 << 20, None) == F3.FLUX3_ERR_ALIGNMENT
    assert L.flux3_ln_modulate(16, 4, 16, 16, ctypes.c_float(0.0), 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_rope_tables(16, 4, ctypes.c_float(-1.0), 16, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_prepare(arr, n, 8, 16, ctypes.c_float(-1.0), 16, 16, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_prepare(arr, n, 8, None, ctypes.c_float(1e4), 16, 16, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_selftest_wait_timeout(0, None) == F3.FLUX3_ERR_INVALID_ARG


def test_nvfp4_sizes_and_validation():
    L = F3.lib()
    cfg = F3.flux3_default_config()
    cfg.wfmt = F3.FLUX3_W_NVFP4
    per_block = 27648 * 3072 // 2 + 27648 * 3072 // 16 + 3072 * 12288 // 2 + 3072 * 12288 // 16
    assert per_block == 69_009_408                      # 4.5 bits per weight
    assert 28 * per_block <= F3.flux3_packed_weight_bytes(cfg) < 28 * (per_block + 8 * 256)
    bf = F3.flux3_default_config()
    # the NVFP4 workspace adds one block's weights in bf16
    assert F3.flux3_workspace_bytes(cfg, 4608) - F3.flux3_workspace_bytes(bf, 4608) >= (27648 + 12288) * 3072 * 2
    cfg.n_blocks = 1
    h = ctypes.c_void_p()
    w = (F3.flux3_block_weights_nvfp4 * 1)()
    # bf16 init refuses an NVFP4 config and vice versa
    wb = (F3.flux3_block_weights * 1)()
    for k, _ in F3.flux3_block_weights._fields_:
        setattr(wb[0], k, 4096)
    assert L.flux3_block_init(ctypes.byref(h), ctypes.byref(cfg), wb, 1, 256, 1 << 40, None) == F3.FLUX3_ERR_INVALID_ARG
    bf.n_blocks = 1
    assert L.flux3_block_init_nvfp4(ctypes.byref(h), ctypes.byref(bf), w, 1, 256, 1 << 40, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_block_init_nvfp4(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1 << 40, None) == \
        F3.FLUX3_ERR_INVALID_ARG                         # null tensors
    for k in F3.NVFP4_MATRICES:
        t = getattr(w[0], k)
        t.codes, t.scales, t.global_scale = 4096, 8192, 12288
    w[0].query_norm, w[0].key_norm = 256, 512
    assert L.flux3_block_init_nvfp4(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1024, None) == \
        F3.FLUX3_ERR_WORKSPACE
    w[0].mlp_out.global_scale = 12290
    assert L.flux3_block_init_nvfp4(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1 << 40, None) == \
        F3.FLUX3_ERR_ALIGNMENT
    assert h.value is None
    # quantiser: cols must be a multiple of 16, pointers aligned
    assert L.flux3_quantize_nvfp4(16, 4, 40, 16, 16, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_quantize_nvfp4(16, 0, 32, 16, 16, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_quantize_nvfp4(18, 4, 32, 16, 16, 16, None) == F3.FLUX3_ERR_ALIGNMENT
    assert L.flux3_dequantize_block(None, 0, 16, 16, None) == F3.FLUX3_ERR_INVALID_ARG


def test_mode_blocks_validation_before_any_launch():
    L = F3.lib()
    none3 = (ctypes.c_void_p * 3)(None, None, None)
    ok_segs, n_ok = _segs([(0, 4, 2), (4, 8, 0), (12, 4, 1)])
    # no handle array, zero blocks, null buffers
    assert L.flux3_mode_blocks_forward(None, 5, 16, 16, ok_segs, n_ok, 16, 16, 16, 1 << 20, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_mode_blocks_forward(none3, 0, 16, 16, ok_segs, n_ok, 16, 16, 16, 1 << 20, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_mode_blocks_forward(none3, 5, None, 16, ok_segs, n_ok, 16, 16, 16, 1 << 20, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    # a mode split into two runs of rows (txt | image | txt)
    split, n_split = _segs([(0, 4, 2), (4, 8, 0), (12, 4, 2)])
    assert L.flux3_mode_blocks_forward(none3, 5, 16, 16, split, n_split, 16, 16, 16, 1 << 20, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    # a mode with tokens but no handle
    assert L.flux3_mode_blocks_forward(none3, 5, 16, 16, ok_segs, n_ok, 16, 16, 16, 1 << 20, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    # a bad segment table
    bad, n_bad = _segs([(0, 4, 2), (5, 11, 0)])
    assert L.flux3_mode_blocks_forward(none3, 5, 16, 16, bad, n_bad, 16, 16, 16, 1 << 20, None) == \
        F3.FLUX3_ERR_INVALID_ARG


def test_fp8r_sizes_and_validation():
    L = F3.lib()
    cfg = F3.flux3_default_config()
    cfg.wfmt = F3.FLUX3_W_FP8R
    per_block = 27648 * 3072 + 27648 * 4 + 3072 * 12288 + 3072 * 2 * 4
    assert per_block == 122_818_560                     # 8 bits per weight + one float per row
    assert 28 * per_block <= F3.flux3_packed_weight_bytes(cfg) < 28 * (per_block + 8 * 256)
    bf = F3.flux3_default_config()
    assert F3.flux3_workspace_bytes(cfg, 4608) - F3.flux3_workspace_bytes(bf, 4608) >= (27648 + 12288) * 3072 * 2
    cfg.n_blocks = 1
    h = ctypes.c_void_p()
    w = (F3.flux3_block_weights_fp8r * 1)()
    # the other formats' inits refuse an fp8r config and the fp8r init refuses theirs
    wb = (F3.flux3_block_weights * 1)()
    for k, _ in F3.flux3_block_weights._fields_:
        setattr(wb[0], k, 4096)
    assert L.flux3_block_init(ctypes.byref(h), ctypes.byref(cfg), wb, 1, 256, 1 << 40, None) == F3.FLUX3_ERR_INVALID_ARG
    w4 = (F3.flux3_block_weights_nvfp4 * 1)()
    assert L.flux3_block_init_nvfp4(ctypes.byref(h), ctypes.byref(cfg), w4, 1, 256, 1 << 40, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    bf.n_blocks = 1
    assert L.flux3_block_init_fp8r(ctypes.byref(h), ctypes.byref(bf), w, 1, 256, 1 << 40, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_block_init_fp8r(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1 << 40, None) == \
        F3.FLUX3_ERR_INVALID_ARG                         # null tensors
    for k in F3.NVFP4_MATRICES:
        t = getattr(w[0], k)
        t.codes, t.scales = 4096, 8192
    w[0].query_norm, w[0].key_norm = 256, 512
    assert L.flux3_block_init_fp8r(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1024, None) == \
        F3.FLUX3_ERR_WORKSPACE
    w[0].mlp_in.scales = 8194
    assert L.flux3_block_init_fp8r(ctypes.byref(h), ctypes.byref(cfg), w, 1, 256, 1 << 40, None) == \
        F3.FLUX3_ERR_ALIGNMENT
    assert h.value is None
    assert L.flux3_quantize_fp8r(16, 4, 40, 16, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_quantize_fp8r(16, 0, 32, 16, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_quantize_fp8r(18, 4, 32, 16, 16, None) == F3.FLUX3_ERR_ALIGNMENT
    assert L.flux3_quantize_fp8r(16, 4, 32, 16, 18, None) == F3.FLUX3_ERR_ALIGNMENT


def test_sigma_schedule_host_entry_point_matches_oracle():
    from oracle import flux3_model as M
    for steps in (16, 50):
        got = np.array(F3.flux3_sigma_schedule(steps, 6.93), dtype=np.float32)
        assert np.array_equal(got, M.sigma_schedule(steps).astype(np.float32))
    assert F3.lib().flux3_sigma_schedule(0, ctypes.c_double(6.93), (ctypes.c_float * 1)()) == F3.FLUX3_ERR_INVALID_ARG


def test_model_entry_points_validation_before_any_launch():
    L = F3.lib()
    h = ctypes.c_void_p()
    w = F3.flux3_cond_weights()
    assert L.flux3_cond_init(None, ctypes.byref(w), 256, 1 << 40, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_cond_init(ctypes.byref(h), ctypes.byref(w), 256, 1 << 40, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_cond_init(ctypes.byref(h), ctypes.byref(w), 256, 1024, None) == F3.FLUX3_ERR_WORKSPACE
    w.time_in_in = 4096
    w.ref_time_in_in = 4096          # ref_time_in_out missing: both or neither
    assert L.flux3_cond_init(ctypes.byref(h), ctypes.byref(w), 256, 1 << 40, None) == F3.FLUX3_ERR_INVALID_ARG
    assert h.value is None
    assert F3.flux3_cond_packed_bytes() > (3072 * 20480 + 6 * 9216 * 3072) * 2
    assert L.flux3_conditioning(None, ctypes.c_float(0.5), ctypes.c_float(0.4), 16, 16, 16, 16, 1 << 20, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    segs, n = _segs([(0, 8, 0)])
    ins = (ctypes.c_void_p * 3)(16, 16, 16)
    assert L.flux3_embed_tokens(None, ins, 8, segs, n, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_final_layer(None, 16, 8, segs, n, 16, 16, 16, 1 << 20, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_transformer_forward(None, None, 0, None, ins, 8, segs, n, 16, ctypes.c_float(0.5),
                                       ctypes.c_float(0.4), 16, 16, 1 << 20, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_euler_step(None, 16, 8, ctypes.c_float(1.0), ctypes.c_float(0.9), None, None) == \
        F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_latents_to_bf16(None, 8, 16, None) == F3.FLUX3_ERR_INVALID_ARG
    assert L.flux3_cfg_euler_step(16, None, 16, 8, ctypes.c_float(3.5), ctypes.c_float(1.0), ctypes.c_float(0.9),
                                  None, None) == F3.FLUX3_ERR_INVALID_ARG
    cfg = F3.flux3_default_config()
    assert F3.flux3_transformer_workspace_bytes(cfg, 4608) > F3.flux3_workspace_bytes(cfg, 4608) + 4608 * 3072 * 4
    assert F3.flux3_transformer_workspace_bytes(cfg, 0) == 0


def test_every_entry_point_is_documented_in_the_header():
    """Each FLUX3_API declaration of include/flux3.h follows its own comment
    block (the operation, its arguments, layouts and errors)."""
    lines = open(os.path.join(ROOT, "include", "flux3.h")).read().split("\n")
    undocumented = []
    for i, line in enumerate(lines):
        if not line.startswith("FLUX3_API"):
            continue
        j = i - 1
        while j >= 0 and not lines[j].strip():
            j -= 1
        if not lines[j].rstrip().endswith("*/"):
            undocumented.append(line.split("(")[0].split()[-1])
    assert not undocumented, undocumented
