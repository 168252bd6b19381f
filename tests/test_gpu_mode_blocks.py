"""The per-mode blocks (flux3_mode_blocks_forward, "FLUX.3 Image Klein
support", comment "Structure (from dit.py)": the first 5 blocks are per mode,
own weights, attention only among the mode's own tokens, early_stream
modulations).

* 112 tokens (txt 32, image 8x8, one 4x4 reference), 5 blocks per mode:
  every block teacher-forced against the oracle (the GPU block runs on the
  oracle's own input of that block, fp32-rounded; values flow oracle -> GPU
  only) under the block criterion, and the entry point's free-running result
  against the oracle chain.
* The full 8704-token layout (txt 512, image 64x64, one 64x64 reference): the
  entry point equals per-mode stack calls on the modes' rows bit for bit, the
  modes are isolated, and each mode's first block meets the block criterion on
  sampled rows (both ends of the mode, random rows)."""

import numpy as np
import pytest
import torch

import diffusion_transformer_block_fwd_b300 as F3
from diffusion_transformer_block_fwd_b300.model import mode_blocks_forward
import oracle as O
import synth
from _f3 import DEV, assert_block_output, assert_close, f64, layout_tensors, weights_f64

pytestmark = pytest.mark.gpu
N_BLOCKS = 5


@pytest.fixture(scope="module")
def modes():
    ws = [[synth.block_weights(6000 + m, b, device=DEV) for b in range(N_BLOCKS)] for m in range(3)]
    mb = [F3.Flux3Blocks(ws[m], max_tokens=8704) for m in range(3)]
    return ws, mb


def _sync_ok():
    assert F3.flux3_check_error(torch.cuda.current_stream().cuda_stream) == 0


def _mode_rows(lay, m):
    return np.nonzero(lay.stream_id == m)[0]


def test_mode_blocks_small_against_oracle(modes):
    ws, mb = modes
    lay = synth.build_layout(synth.WORKLOADS["modes5_t112"]["spec"])
    pos, _ = layout_tensors(lay)
    pos64 = lay.pos.astype(np.float64)
    x = synth.activations(91, lay.T, device=DEV)
    mods = synth.modulation(91, device=DEV)
    m64 = f64(mods)
    # free-running entry point, 5 blocks per mode
    xg = x.clone()
    mode_blocks_forward(mb, xg, lay.segments, pos, mods)
    _sync_ok()
    # oracle chain, weights converted one block at a time
    ref = O.mode_blocks_forward(f64(x), [(weights_f64(w) for w in ws[m]) for m in range(3)], m64,
                                lay.stream_id, pos64)
    assert_close(f64(xg), ref, 2e-2, 0.9995, "5 per-mode blocks, free-running")
    # teacher-forced per block: the entry point with one block, on the oracle's own input
    xo = f64(x)
    for b in range(N_BLOCKS):
        one = [F3.Flux3Blocks([ws[m][b]], max_tokens=512) for m in range(3)]
        x_in = torch.from_numpy(xo.astype(np.float32)).to(DEV)
        xg1 = x_in.clone()
        mode_blocks_forward(one, xg1, lay.segments, pos, mods)
        _sync_ok()
        xin64 = f64(x_in)
        out = xin64.copy()
        for m in range(3):
            r = _mode_rows(lay, m)
            parts = O.single_block_parts(xin64[r], weights_f64(ws[m][b]), m64, lay.stream_id[r], pos64[r])
            out[r] = parts["out"]
            gate = m64[lay.stream_id[r], 6144:]
            assert_block_output(f64(xg1)[r], parts["out"], xin64[r], gate, parts["y"], f"block {b} mode {m}")
        for o in one:
            o.close()
        xo = out


def test_mode_order_does_not_matter(modes):
    """The same tokens with the modes in another order give the same rows, bit
    for bit (each mode's rows are the same sub-sequence either way)."""
    _, mb = modes
    lay = synth.build_layout(synth.WORKLOADS["modes5_t112"]["spec"])
    pos, _ = layout_tensors(lay)
    x = synth.activations(92, lay.T, device=DEV)
    mods = synth.modulation(92, device=DEV)
    a = x.clone()
    mode_blocks_forward(mb, a, lay.segments, pos, mods)
    order = np.concatenate([_mode_rows(lay, m) for m in (0, 1, 2)])    # image, image_cond, txt
    segs, start = [], 0
    for m in (0, 1, 2):
        n = int((lay.stream_id == m).sum())
        segs.append((start, n, m))
        start += n
    idx = torch.from_numpy(order).to(DEV)
    b = x[idx].contiguous()
    mode_blocks_forward(mb, b, segs, pos[idx].contiguous(), mods)
    _sync_ok()
    assert torch.equal(a[idx], b)


def test_mode_blocks_full_size(modes):
    ws, mb = modes
    lay = synth.build_layout(synth.WORKLOADS["modes5_1024sq_ref1_t8704"]["spec"])
    pos, _ = layout_tensors(lay)
    x = synth.activations(93, lay.T, device=DEV)
    mods = synth.modulation(93, device=DEV)
    a = x.clone()
    mode_blocks_forward(mb, a, lay.segments, pos, mods)
    _sync_ok()
    assert torch.isfinite(a).all()
    # the entry point is the per-mode stacks on the modes' rows, bit for bit
    b = x.clone()
    for m in range(3):
        r = _mode_rows(lay, m)
        r0, n = int(r[0]), len(r)
        sub = b[r0:r0 + n]
        mb[m].forward(sub, [(0, n, m)], pos[r0:r0 + n].contiguous(), mods)
    _sync_ok()
    assert torch.equal(a, b)
    # isolation: changing the txt tokens changes only the txt rows
    x2 = x.clone()
    t = torch.from_numpy(_mode_rows(lay, 2)).to(DEV)
    x2[t] += 0.5 * synth.activations(94, len(t), device=DEV)
    c = x2.clone()
    mode_blocks_forward(mb, c, lay.segments, pos, mods)
    _sync_ok()
    keep = torch.from_numpy(np.nonzero(lay.stream_id != 2)[0]).to(DEV)
    assert torch.equal(a[keep], c[keep])
    assert (a[t] != c[t]).any(dim=1).all()
    # each mode's first block on sampled rows
    d = x.clone()
    mode_blocks_forward(mb, d, lay.segments, pos, mods, n_blocks=1)
    _sync_ok()
    m64, x64, pos64, got = f64(mods), f64(x), lay.pos.astype(np.float64), f64(d)
    rng = np.random.default_rng(95)
    for m in range(3):
        r = _mode_rows(lay, m)
        n = len(r)
        local = np.unique(np.concatenate([[0, 1, n - 2, n - 1], rng.choice(n, 12, replace=False)]))
        parts = O.single_block_parts(x64[r], weights_f64(ws[m][0]), m64, lay.stream_id[r], pos64[r], rows=local)
        gate = m64[lay.stream_id[r][local], 6144:]
        assert_block_output(got[r][local], parts["out"], x64[r][local], gate, parts["y"], f"mode {m} sampled rows")
