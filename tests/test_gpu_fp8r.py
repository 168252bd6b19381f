"""Row-wise FP8 ("fp8r") weights on the GPU against the oracle (oracle/fp8r.py):

* The quantiser: codes and row scales bit-exact (every rounding decision is
  taken on the same float64 quotient on both sides) on crafted rows (ties,
  saturation, zero rows, subnormal codes), random matrices and a full-size
  projection.
* The expansion of a packed block to bf16: bit-exact against the oracle's
  codes and scales expanded the same way (e4m3 * s rounded to float32, then to
  bf16).
* Up to 128 tokens the GEMMs expand the codes in shared memory: the block
  equals a bf16 handle holding the expanded weights bit for bit (also at 129
  tokens, where the expansion goes through HBM).
* The block with fp8r weights: the oracle runs on the exactly dequantised
  weights (quantised by the oracle itself; no GPU value feeds the oracle);
  the block criterion of the bf16 path on x' and on the update (the GPU's only
  extra rounding is that of each weight to bf16), at 96 and 171 tokens and on
  sampled rows of the 8704-token layout."""

import numpy as np
import pytest
import torch

import diffusion_transformer_block_fwd_b300 as F3
import oracle as O
import synth
from _f3 import DEV, assert_block_output, f64, layout_tensors, sample_rows
from oracle import fp8r as R
from oracle import nvfp4 as Q

pytestmark = pytest.mark.gpu

MATS = ("q_proj", "k_proj", "v_proj", "attn_out", "mlp_in", "mlp_out")
RAGGED = [("txt", 37), ("image", (9, 11)), ("image_cond", (5, 7))]


def _stream():
    return torch.cuda.current_stream().cuda_stream


def gpu_quantize(w_bf16_dev):
    codes, scales = F3.quantize_fp8r(w_bf16_dev)
    assert F3.flux3_check_error(_stream()) == 0
    return codes, scales


def check_quantizer(w):
    """GPU quantiser vs the oracle on the bf16 matrix w (CPU tensor)."""
    codes, scales = gpu_quantize(w.to(DEV))
    rc, rs = R.quantize(f64(w))
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32)), "row scales differ"
    bad = codes.cpu().numpy() != rc
    assert not bad.any(), f"{int(bad.sum())} codes differ"


def expand_f32_then_bf16(codes, scales):
    """The expansion the forward pass uses, from the oracle's codes and scales:
    e4m3 value (exact in float32) times the row scale rounded to float32
    (numpy float32 multiply, nearest even), then to bf16 (torch's nearest-even
    cast)."""
    v = Q.E4M3_TABLE[codes].astype(np.float32)
    return torch.from_numpy(v * scales[:, None]).to(torch.bfloat16)


def bf16_bits(t):
    return t.view(torch.int16).cpu().numpy()


def test_quantize_crafted_rows():
    rows = np.zeros((6, 48))
    # row 0: amax 448 -> scale 1 exactly; the elements sit on E4M3 tie points
    ties = Q.E4M3_TABLE[8:24] * 0.5 + Q.E4M3_TABLE[9:25] * 0.5
    rows[0, :16] = ties
    rows[0, 16:32] = -ties
    rows[0, 47] = 448.0
    rows[1, :] = 0.0                                        # all-zero row: scale 1, codes 0
    rows[2, :] = np.linspace(-1, 1, 48) * 3e-3              # ordinary row
    rows[3, :8] = [1.0, -1.0, 2.0 ** -12, -(2.0 ** -12), 0.0, 1e-30, 0.5, -0.25]   # subnormal / zero codes
    rows[4, :] = 7.0                                        # constant row: every code 448
    rows[5, ::2] = -1e-4
    rows[5, 1::2] = 1e-4
    w = torch.from_numpy(rows).to(torch.bfloat16)
    check_quantizer(w)
    codes, scales = gpu_quantize(w.to(DEV))
    assert scales[0].item() == 1.0 and scales[1].item() == 1.0
    assert not codes[1].any()
    assert (codes[4] == 0x7E).all()


@pytest.mark.parametrize("rows,cols,dist", [(1, 16, "normal"), (3, 48, "normal"), (77, 320, "heavy"),
                                            (256, 3072, "normal"), (129, 9216, "heavy")])
def test_quantize_random_shapes(rows, cols, dist):
    g = torch.Generator().manual_seed(rows * 11 + cols)
    w = torch.randn((rows, cols), generator=g) * 0.02
    if dist == "heavy":
        w = w * torch.exp(2.0 * torch.randn((rows, cols), generator=g))
    check_quantizer(w.to(torch.bfloat16))


def test_quantize_full_size_projection():
    check_quantizer(synth.block_weights(33, 0)["mlp_in"])   # [18432, 3072]


@pytest.fixture(scope="module")
def fp8_block():
    """Block weights quantised by the oracle; the GPU handle gets the oracle's
    codes and scales, the oracle runs on their exact dequantisation."""
    w = synth.block_weights(1357, 0)
    dev, wdq, raw = {}, {}, {}
    for k in MATS:
        c, s = R.quantize(f64(w[k]))
        dev[k] = (torch.from_numpy(c).to(DEV), torch.from_numpy(s).to(DEV))
        wdq[k] = R.dequantize(c, s)
        raw[k] = (c, s)
    for k in ("query_norm", "key_norm"):
        dev[k] = w[k].to(DEV)
        wdq[k] = f64(w[k])
    blocks = F3.Flux3Blocks([dev], max_tokens=16384, wfmt="fp8r")
    return blocks, wdq, raw


def test_expand_block_bit_exact(fp8_block):
    blocks, _, raw = fp8_block
    w_in = torch.empty((27648, 3072), dtype=torch.bfloat16, device=DEV)
    w_out = torch.empty((3072, 12288), dtype=torch.bfloat16, device=DEV)
    F3.flux3_dequantize_block(blocks.handle, 0, w_in.data_ptr(), w_out.data_ptr(), _stream())
    assert F3.flux3_check_error(_stream()) == 0
    gin = bf16_bits(w_in)
    for i, k in enumerate(("q_proj", "k_proj", "v_proj")):
        assert np.array_equal(gin[3072 * i:3072 * (i + 1)], bf16_bits(expand_f32_then_bf16(*raw[k]))), k
    mi = bf16_bits(expand_f32_then_bf16(*raw["mlp_in"])).reshape(2, 72, 128, 3072).transpose(1, 0, 2, 3)
    assert np.array_equal(gin[9216:], mi.reshape(18432, 3072)), "mlp_in"
    cat = np.concatenate([bf16_bits(expand_f32_then_bf16(*raw["attn_out"])),
                          bf16_bits(expand_f32_then_bf16(*raw["mlp_out"]))], axis=1)
    assert np.array_equal(bf16_bits(w_out), cat), "attn_out | mlp_out"


def _run(blocks, lay, x, mods):
    pos, _ = layout_tensors(lay)
    y = x.clone()
    blocks.forward(y, lay.segments, pos, mods)
    assert F3.flux3_check_error(_stream()) == 0
    return y


@pytest.mark.parametrize("name,spec", [("block_t96", synth.WORKLOADS["block_t96"]["spec"]), ("ragged_t171", RAGGED)])
def test_fp8r_block_against_oracle(fp8_block, name, spec):
    blocks, wdq, _ = fp8_block
    lay = synth.build_layout(spec)
    x = synth.activations(61, lay.T, device=DEV)
    mods = synth.modulation(61, device=DEV)
    y = _run(blocks, lay, x, mods)
    m = f64(mods)
    parts = O.single_block_parts(f64(x), wdq, m, lay.stream_id, lay.pos.astype(np.float64))
    assert_block_output(f64(y), parts["out"], f64(x), m[lay.stream_id, 6144:], parts["y"], name)


@pytest.fixture(scope="module")
def bf16_twin(fp8_block):
    """A bf16 handle whose weights are the fp8r block's exact expansion."""
    _, _, raw = fp8_block
    w = synth.block_weights(1357, 0)
    dev = {k: expand_f32_then_bf16(*raw[k]).to(DEV) for k in MATS}
    dev.update({k: w[k].to(DEV) for k in ("query_norm", "key_norm")})
    return F3.Flux3Blocks([dev], max_tokens=1024)


@pytest.mark.parametrize("name,spec", [("one_token", [("txt", 1)]), ("block_t96", synth.WORKLOADS["block_t96"]["spec"]),
                                       ("t128", [("txt", 64), ("image", (8, 8))]),
                                       ("t129_expanded", [("txt", 65), ("image", (8, 8))])])
def test_fp8r_block_equals_bf16_block_on_expanded_weights(fp8_block, bf16_twin, name, spec):
    """Up to 128 tokens the fp8r GEMMs read the e4m3 codes and expand them in
    shared memory; from 129 on the block's weights are expanded in HBM first.
    Both feed the tensor cores the same bf16 values as a bf16 handle holding
    the expanded weights, so the block output equals that handle's bit for
    bit."""
    blocks, _, _ = fp8_block
    lay = synth.build_layout(spec)
    x = synth.activations(63, lay.T, device=DEV)
    mods = synth.modulation(63, device=DEV)
    a = _run(blocks, lay, x, mods)
    b = _run(bf16_twin, lay, x, mods)
    assert not torch.equal(a, x)
    assert torch.equal(a, b), f"{name}: max |diff| {float((a - b).abs().max())}"


def test_fp8r_stack_small_t_equals_blocks_one_by_one(fp8_block):
    """Two fp8r blocks at 96 tokens (codes expanded inside the GEMMs): the
    stack call equals the blocks called one at a time bit for bit."""
    _, _, raw = fp8_block
    w = synth.block_weights(1357, 0)
    dev = {k: (torch.from_numpy(raw[k][0]).to(DEV), torch.from_numpy(raw[k][1]).to(DEV)) for k in MATS}
    dev.update({k: w[k].to(DEV) for k in ("query_norm", "key_norm")})
    blocks = F3.Flux3Blocks([dev, dev], max_tokens=256, wfmt="fp8r")
    lay = synth.build_layout(synth.WORKLOADS["block_t96"]["spec"])
    pos, _ = layout_tensors(lay)
    x = synth.activations(64, lay.T, device=DEV)
    mods = synth.modulation(64, device=DEV)
    a = x.clone()
    blocks.forward(a, lay.segments, pos, mods)
    b = x.clone()
    for i in range(2):
        blocks.forward(b, lay.segments, pos, mods, first_block=i, n_blocks=1)
    assert F3.flux3_check_error(_stream()) == 0
    assert torch.isfinite(a).all() and torch.equal(a, b)
    blocks.close()


def test_fp8r_block_full_size_sampled_rows(fp8_block):
    blocks, wdq, _ = fp8_block
    lay = synth.build_layout(synth.WORKLOADS["block_1024sq_ref1_t8704"]["spec"])
    x = synth.activations(62, lay.T, device=DEV)
    mods = synth.modulation(62, device=DEV)
    y = _run(blocks, lay, x, mods)
    rows = sample_rows(lay.T, lay.segments, n_random=16)
    m = f64(mods)
    parts = O.single_block_parts(f64(x), wdq, m, lay.stream_id, lay.pos.astype(np.float64), rows=rows)
    assert_block_output(f64(y)[rows], parts["out"], f64(x)[rows], m[lay.stream_id[rows], 6144:], parts["y"], "t8704")


def test_fp8r_handle_rejects_bf16_only_calls(fp8_block):
    blocks, _, _ = fp8_block
    sp = _stream()
    T = 8
    buf = torch.zeros(T * 12288, dtype=torch.bfloat16, device=DEV)
    L = F3.lib()
    p = buf.data_ptr()
    assert L.flux3_in_projection(blocks.handle, 0, p, T, p, p, p, p, sp) == F3.FLUX3_ERR_UNSUPPORTED
    x = torch.zeros((T, 3072), device=DEV)
    assert L.flux3_out_projection(blocks.handle, 0, p, T, p, p, x.data_ptr(), None, 0, sp) == F3.FLUX3_ERR_UNSUPPORTED
    segs = F3.segments_array([(0, T, 0)])
    assert L.flux3_block_forward_noalloc(blocks.handle, 0, x.data_ptr(), T, segs, 1, p, p, sp) == \
        F3.FLUX3_ERR_UNSUPPORTED
