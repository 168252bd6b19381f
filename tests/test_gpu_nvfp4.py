"""NVFP4 weights on the GPU against the CPU oracle.

* flux3_quantize_nvfp4: codes, block scales and the global scale bit for bit
  against oracle.nvfp4.quantize (integer results decided by floating point:
  both sides decide on the float64 quotients the definition names).
* flux3_dequantize_block: each bf16 weight equals e2m1 * e4m3 (exact) times
  the global scale rounded to float32, then rounded to bf16 (both nearest
  even), from the oracle's codes and scales.
* Up to 128 tokens the GEMMs expand the codes in shared memory: the block
  equals a bf16 handle holding the expanded weights bit for bit (also at 129
  tokens, where the expansion goes through HBM).
* The block with NVFP4 weights: the oracle runs on the exactly dequantised
  weights (quantised by the oracle itself; no GPU value feeds the oracle);
  criterion max|err| <= 5e-2 RMS(x'), cosine >= 0.998 on x', plus the bf16
  path's update criterion (the GPU's only extra rounding is that of each
  weight to bf16).
* The 28-block stack at 1024x1024 + ten 512x512 references (14848 tokens):
  properties at full size.
"""

import numpy as np
import pytest
import torch

import diffusion_transformer_block_fwd_b300 as F3
import oracle as O
import synth
from _f3 import DEV, assert_block_output, assert_close, f64, layout_tensors, sample_rows
from oracle import nvfp4 as Q

pytestmark = pytest.mark.gpu

MATS = ("q_proj", "k_proj", "v_proj", "attn_out", "mlp_in", "mlp_out")
RAGGED = [("txt", 37), ("image", (9, 11)), ("image_cond", (5, 7))]


def _stream():
    return torch.cuda.current_stream().cuda_stream


def gpu_quantize(w_bf16_dev):
    codes, scales, g = F3.quantize_nvfp4(w_bf16_dev)
    assert F3.flux3_check_error(_stream()) == 0
    return codes, scales, g


def dequant_f32_then_bf16(codes, scales, g):
    """The expansion the forward pass uses, from the oracle's codes and scales:
    e2m1 * e4m3 is exact in float32; times g rounded to float32 (numpy float32
    multiply, nearest even); then to bf16 (torch's nearest-even cast)."""
    p = Q.dequantize(codes, scales, 1.0).astype(np.float32)          # exact
    w = p * np.float32(g)
    return torch.from_numpy(w).to(torch.bfloat16)


def bf16_bits(t):
    return t.view(torch.int16).cpu().numpy()


def check_quantizer(w):
    """GPU quantiser vs the oracle on the bf16 matrix w (CPU tensor)."""
    codes, scales, g = gpu_quantize(w.to(DEV))
    rc, rs, rg = Q.quantize(f64(w))
    assert np.float32(g.item()) == np.float32(rg)
    assert np.array_equal(scales.cpu().numpy(), rs), "block scales differ"
    c = codes.cpu().numpy()
    bad = c != rc
    assert not bad.any(), f"{int(bad.sum())} code bytes differ"


def test_quantize_crafted_ties_zeros_subnormal_scales():
    # global amax 2.625 = 2688 * 2^-10 -> g = 2^-10 exactly; block 1 has scale 1.0
    # so its elements land exactly on every e2m1 tie point (ties go to even codes)
    g = 2.0 ** -10
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    rows = np.zeros((6, 64))
    rows[0, :16] = 2.625
    rows[1, 16:32] = np.concatenate([ties, -ties]) * g
    rows[2, :16] = 0.0                                   # all-zero block -> scale 0, codes 0
    rows[2, 16:32] = -0.0                                # negative zeros carry no sign
    rows[3, :16] = np.linspace(-1, 1, 16) * 3e-5         # small block: subnormal e4m3 scale
    rows[4, :16] = np.linspace(-1, 1, 16) * 1e-9         # scale rounds to 0 -> codes 0
    rows[5, 48:64] = np.array([6.1, -5.9, 3.0, 0.3] * 4) * g * 7.0   # scale 7 (exact), saturation near 6
    w = torch.from_numpy(rows).to(torch.bfloat16)
    check_quantizer(w)
    codes, scales, gg = gpu_quantize(w.to(DEV))
    assert gg.item() == g
    assert list(Q.E2M1_TABLE[np.concatenate([[b & 15, b >> 4] for b in codes[1, 8:16].cpu().numpy()])]) == \
        [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -0.0, -1.0, -1.0, -2.0, -2.0, -4.0, -4.0, -6.0]


def test_quantize_all_zero_matrix():
    w = torch.zeros((5, 32), dtype=torch.bfloat16)
    codes, scales, g = gpu_quantize(w.to(DEV))
    assert g.item() == 1.0 and not codes.any() and not scales.any()
    check_quantizer(w)


@pytest.mark.parametrize("rows,cols,dist", [(1, 16, "normal"), (3, 48, "normal"), (77, 320, "heavy"),
                                            (256, 3072, "normal"), (129, 9216, "heavy")])
def test_quantize_random_shapes(rows, cols, dist):
    g = torch.Generator().manual_seed(rows * 7 + cols)
    w = torch.randn((rows, cols), generator=g) * 0.02
    if dist == "heavy":
        w = w * torch.exp(2.0 * torch.randn((rows, cols), generator=g))
    check_quantizer(w.to(torch.bfloat16))


def test_quantize_full_size_projection():
    w = synth.block_weights(31, 0)["q_proj"]            # [3072, 3072] N(0, 0.02) bf16
    check_quantizer(w)


# ---------------------------------------------------------------- one NVFP4 block
@pytest.fixture(scope="module")
def fp4_block():
    """Block weights quantised by the oracle; the GPU handle gets the oracle's
    codes, the oracle runs on their exact dequantisation."""
    w = synth.block_weights(2468, 0)
    dev, wdq, raw = {}, {}, {}
    for k in MATS:
        c, s, g = Q.quantize(f64(w[k]))
        dev[k] = (torch.from_numpy(c).to(DEV), torch.from_numpy(s).to(DEV),
                  torch.tensor([g], dtype=torch.float32, device=DEV))
        wdq[k] = Q.dequantize(c, s, g)
        raw[k] = (c, s, g)
    for k in ("query_norm", "key_norm"):
        dev[k] = w[k].to(DEV)
        wdq[k] = f64(w[k])
    blocks = F3.Flux3Blocks([dev], max_tokens=16384, wfmt="nvfp4")
    return blocks, wdq, raw


def test_dequantize_block_bit_exact(fp4_block):
    blocks, _, raw = fp4_block
    w_in = torch.empty((27648, 3072), dtype=torch.bfloat16, device=DEV)
    w_out = torch.empty((3072, 12288), dtype=torch.bfloat16, device=DEV)
    F3.flux3_dequantize_block(blocks.handle, 0, w_in.data_ptr(), w_out.data_ptr(), _stream())
    assert F3.flux3_check_error(_stream()) == 0
    gin = bf16_bits(w_in)
    for i, k in enumerate(("q_proj", "k_proj", "v_proj")):
        assert np.array_equal(gin[3072 * i:3072 * (i + 1)], bf16_bits(dequant_f32_then_bf16(*raw[k]))), k
    # mlp_in rows interleaved in groups of 128: a[128m..], b[128m..]
    mi = bf16_bits(dequant_f32_then_bf16(*raw["mlp_in"])).reshape(2, 72, 128, 3072).transpose(1, 0, 2, 3)
    assert np.array_equal(gin[9216:], mi.reshape(18432, 3072)), "mlp_in"
    cat = np.concatenate([bf16_bits(dequant_f32_then_bf16(*raw["attn_out"])),
                          bf16_bits(dequant_f32_then_bf16(*raw["mlp_out"]))], axis=1)
    assert np.array_equal(bf16_bits(w_out), cat), "attn_out | mlp_out"


def _run(blocks, lay, x, mods):
    pos, _ = layout_tensors(lay)
    y = x.clone()
    blocks.forward(y, lay.segments, pos, mods)
    assert F3.flux3_check_error(_stream()) == 0
    return y


@pytest.mark.parametrize("name,spec", [("block_t96", synth.WORKLOADS["block_t96"]["spec"]), ("ragged_t171", RAGGED),
                                       ("one_token", [("image_cond", (1, 1))])])
def test_nvfp4_block_matches_oracle(fp4_block, name, spec):
    blocks, wdq, _ = fp4_block
    lay = synth.build_layout(spec)
    x = synth.activations(41, lay.T, device=DEV)
    mods = synth.modulation(41, device=DEV)
    y = _run(blocks, lay, x, mods)
    m = f64(mods)
    parts = O.single_block_parts(f64(x), wdq, m, lay.stream_id, lay.pos.astype(np.float64))
    assert_close(f64(y), parts["out"], 5e-2, 0.998, name + " x' (NVFP4 criterion)")
    assert_block_output(f64(y), parts["out"], f64(x), m[lay.stream_id, 6144:], parts["y"], name)


@pytest.fixture(scope="module")
def bf16_twin(fp4_block):
    """A bf16 handle whose weights are the NVFP4 block's exact expansion."""
    _, _, raw = fp4_block
    w = synth.block_weights(2468, 0)
    dev = {k: dequant_f32_then_bf16(*raw[k]).to(DEV) for k in MATS}
    dev.update({k: w[k].to(DEV) for k in ("query_norm", "key_norm")})
    return F3.Flux3Blocks([dev], max_tokens=1024)


@pytest.mark.parametrize("name,spec", [("one_token", [("txt", 1)]), ("block_t96", synth.WORKLOADS["block_t96"]["spec"]),
                                       ("t128", [("txt", 64), ("image", (8, 8))]),
                                       ("t129_expanded", [("txt", 65), ("image", (8, 8))])])
def test_nvfp4_block_equals_bf16_block_on_expanded_weights(fp4_block, bf16_twin, name, spec):
    """Up to 128 tokens the NVFP4 GEMMs read the e2m1 codes and expand them in
    shared memory; from 129 on the block's weights are expanded in HBM first.
    Both feed the tensor cores the same bf16 values as a bf16 handle holding
    the expanded weights, so the block output equals that handle's bit for
    bit."""
    blocks, _, _ = fp4_block
    lay = synth.build_layout(spec)
    x = synth.activations(44, lay.T, device=DEV)
    mods = synth.modulation(44, device=DEV)
    a = _run(blocks, lay, x, mods)
    b = _run(bf16_twin, lay, x, mods)
    assert not torch.equal(a, x)
    assert torch.equal(a, b), f"{name}: max |diff| {float((a - b).abs().max())}"


def test_nvfp4_stack_small_t_equals_blocks_one_by_one(fp4_block):
    """Two NVFP4 blocks at 96 tokens (codes expanded inside the GEMMs, the
    kernels chained by programmatic dependent launches across the blocks):
    the stack call equals the blocks called one at a time bit for bit."""
    _, _, raw = fp4_block
    w = synth.block_weights(2468, 0)
    dev = {k: tuple(torch.from_numpy(v).to(DEV) if isinstance(v, np.ndarray)
                    else torch.tensor([v], dtype=torch.float32, device=DEV) for v in raw[k]) for k in MATS}
    dev.update({k: w[k].to(DEV) for k in ("query_norm", "key_norm")})
    blocks = F3.Flux3Blocks([dev, dev], max_tokens=256, wfmt="nvfp4")
    lay = synth.build_layout(synth.WORKLOADS["block_t96"]["spec"])
    pos, _ = layout_tensors(lay)
    x = synth.activations(45, lay.T, device=DEV)
    mods = synth.modulation(45, device=DEV)
    a = x.clone()
    blocks.forward(a, lay.segments, pos, mods)
    b = x.clone()
    for i in range(2):
        blocks.forward(b, lay.segments, pos, mods, first_block=i, n_blocks=1)
    assert F3.flux3_check_error(_stream()) == 0
    assert torch.isfinite(a).all() and torch.equal(a, b)
    blocks.close()


def test_nvfp4_block_full_size_sampled_rows(fp4_block):
    """One block at the 14848-token layout (1024x1024 + ten 512x512 references)."""
    blocks, wdq, _ = fp4_block
    lay = synth.build_layout(synth.WORKLOADS["stack28_nvfp4_1024sq_10ref512_t14848"]["spec"])
    x = synth.activations(42, lay.T, device=DEV)
    mods = synth.modulation(42, device=DEV)
    y = _run(blocks, lay, x, mods)
    rows = sample_rows(lay.T, lay.segments, n_random=16)
    m = f64(mods)
    parts = O.single_block_parts(f64(x), wdq, m, lay.stream_id, lay.pos.astype(np.float64), rows=rows)
    assert_close(f64(y)[rows], parts["out"], 5e-2, 0.998, "t14848 x' (NVFP4 criterion)")
    assert_block_output(f64(y)[rows], parts["out"], f64(x)[rows], m[lay.stream_id[rows], 6144:], parts["y"],
                        "t14848")


def test_nvfp4_stack28_full_size_properties():
    """28 NVFP4 blocks (quantised on the GPU) over 14848 tokens: finite, the
    stack call equals the 28 blocks called one by one bit for bit, and zero
    gates make every block the identity bit for bit."""
    ws = []
    for b in range(28):
        w = synth.block_weights(97, b, device=DEV)
        q = {k: gpu_quantize(w[k]) for k in MATS}
        q.update({k: w[k] for k in ("query_norm", "key_norm")})
        ws.append(q)
        del w
    blocks = F3.Flux3Blocks(ws, max_tokens=14848, wfmt="nvfp4")
    del ws
    lay = synth.build_layout(synth.WORKLOADS["stack28_nvfp4_1024sq_10ref512_t14848"]["spec"])
    pos, _ = layout_tensors(lay)
    x = synth.activations(43, lay.T, device=DEV)
    mods = synth.modulation(43, device=DEV)
    a = x.clone()
    blocks.forward(a, lay.segments, pos, mods)
    assert F3.flux3_check_error(_stream()) == 0
    assert torch.isfinite(a).all() and not torch.equal(a, x)
    b = x.clone()
    for i in range(28):
        blocks.forward(b, lay.segments, pos, mods, first_block=i, n_blocks=1)
    assert F3.flux3_check_error(_stream()) == 0
    assert torch.equal(a, b)
    m0 = mods.clone()
    m0[:, 6144:] = 0.0
    c = x.clone()
    blocks.forward(c, lay.segments, pos, m0)
    assert F3.flux3_check_error(_stream()) == 0
    assert torch.equal(c, x)
    blocks.close()


def test_nvfp4_handle_rejects_bf16_only_calls(fp4_block):
    blocks, _, _ = fp4_block
    sp = _stream()
    T = 8
    buf = torch.zeros(T * 12288, dtype=torch.bfloat16, device=DEV)
    st = F3.lib().flux3_in_projection(blocks.handle, 0, buf.data_ptr(), T, buf.data_ptr(), buf.data_ptr(),
                                      buf.data_ptr(), buf.data_ptr(), sp)
    assert st == F3.FLUX3_ERR_UNSUPPORTED
    x = torch.zeros((T, 3072), device=DEV)
    segs = F3.segments_array([(0, T, 0)])
    st = F3.lib().flux3_block_forward_noalloc(blocks.handle, 0, x.data_ptr(), T, segs, 1, buf.data_ptr(),
                                              buf.data_ptr(), sp)
    assert st == F3.FLUX3_ERR_UNSUPPORTED


@pytest.mark.slow
def test_nvfp4_stack28_t14848_every_block_sampled_rows():
    """Every block of a 28-block NVFP4 stack at the 14848-token layout
    (1024x1024 + ten 512x512 references).  The oracle quantises each block's
    seeded weights itself (worker processes) and the GPU handle is built from
    the oracle's codes; each block gets a seeded input of its own (made on the
    CPU), and its output rows (segment ends, the ragged tail, random rows)
    are checked against the oracle run on the exactly dequantised weights:
    5e-2 RMS / cosine 0.998 on x', plus the bf16 path's update criterion."""
    import multiprocessing as mp

    import _oracle_pool

    with mp.get_context("spawn").Pool(6) as pool:
        qs = pool.map(_oracle_pool.quantize_block, [(1357, b) for b in range(28)])
    dev = []
    for q in qs:
        d = {k: (torch.from_numpy(q[k][0]).to(DEV), torch.from_numpy(q[k][1]).to(DEV),
                 torch.tensor([q[k][2]], dtype=torch.float32, device=DEV)) for k in MATS}
        d.update({k: torch.from_numpy(q[k].astype(np.float32)).to(DEV) for k in ("query_norm", "key_norm")})
        dev.append(d)
    blocks = F3.Flux3Blocks(dev, max_tokens=14848, wfmt="nvfp4")
    del dev
    lay = synth.build_layout(synth.WORKLOADS["stack28_nvfp4_1024sq_10ref512_t14848"]["spec"])
    assert lay.T == 14848
    pos, _ = layout_tensors(lay)
    pos64 = lay.pos.astype(np.float64)
    rows = sample_rows(lay.T, lay.segments, n_random=8)
    mods = synth.modulation(1358, device=DEV)
    m64 = f64(mods)
    for b in range(28):
        wdq = {k: Q.dequantize(*qs[b][k]) for k in MATS}
        wdq.update({k: qs[b][k] for k in ("query_norm", "key_norm")})
        x_in = synth.activations(1400 + b, lay.T, device=DEV)
        xg = x_in.clone()
        blocks.forward(xg, lay.segments, pos, mods, first_block=b, n_blocks=1)
        x64 = f64(x_in)
        parts = O.single_block_parts(x64, wdq, m64, lay.stream_id, pos64, rows=rows)
        assert F3.flux3_check_error(_stream()) == 0
        got = f64(xg)[rows]
        assert_close(got, parts["out"], 5e-2, 0.998, f"t14848 block {b} x' (NVFP4 criterion)")
        assert_block_output(got, parts["out"], x64[rows], m64[lay.stream_id[rows], 6144:], parts["y"],
                            f"t14848 block {b}")
    blocks.close()
