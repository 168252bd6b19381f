"""Whole-block parity (flux3_block_forward through the C ABI) against the CPU
oracle, and the invariants that hold at any size."""

import numpy as np
import pytest
import torch

import diffusion_transformer_block_fwd_b300 as F3
import oracle as O
import synth
from _f3 import DEV, assert_block_output, assert_close, f64, layout_tensors, sample_rows, weights_f64

pytestmark = pytest.mark.gpu

RAGGED = [("txt", 37), ("image", (9, 11)), ("image_cond", (5, 7))]


@pytest.fixture(scope="module")
def blk():
    w = synth.block_weights(1234, 0, device=DEV)
    return w, weights_f64(w), F3.Flux3Blocks([w], max_tokens=16384)


def run_block(blocks, lay, x, mods):
    pos, _ = layout_tensors(lay)
    y = x.clone()
    blocks.forward(y, lay.segments, pos, mods)
    assert F3.flux3_check_error(torch.cuda.current_stream().cuda_stream) == 0
    return y


@pytest.mark.parametrize("name,spec", [("block_t96", synth.WORKLOADS["block_t96"]["spec"]),
                                       ("ragged_t171", RAGGED),
                                       ("ragged_t300", [("image", (10, 17)), ("txt", 80), ("image_cond", (5, 10))]),
                                       ("one_token", [("txt", 1)])])
def test_block_full_oracle(blk, name, spec):
    w, wf, blocks = blk
    lay = synth.build_layout(spec)
    x = synth.activations(5, lay.T, device=DEV)
    mods = synth.modulation(5, device=DEV)
    y = run_block(blocks, lay, x, mods)
    m = f64(mods)
    parts = O.single_block_parts(f64(x), wf, m, lay.stream_id, lay.pos.astype(np.float64))
    assert_block_output(f64(y), parts["out"], f64(x), m[lay.stream_id, 6144:], parts["y"], name)


# the default max_tokens (16384): 1024 text tokens + 64x64 image + eleven 32x32 references
MAX_TOKENS_SPEC = [("txt", 1024), ("image", (64, 64))] + [("image_cond", (32, 32))] * 11


# 1792 and 2048 tokens (512 text + a 40x32 or 48x32 image): on 148 SMs attention splits the units of its last
# wave into key ranges (3 and 2 ranges) whose partials must fit in h (6 KB per token: attention still reads qkv
# behind it), and the out-projection splits its trailing 10 tiles in 6 ranges (1792) and 22 in 3 (2048)
MID_SPECS = {"mid_t1792": [("txt", 512), ("image", (40, 32))], "mid_t2048": [("txt", 512), ("image", (48, 32))]}


@pytest.mark.parametrize("workload", ["mid_t1792", "mid_t2048", "block_1024sq_t4608", "block_1024sq_ref1_t8704",
                                      "max_tokens_t16384"])
def test_block_full_size_sampled_rows(blk, workload):
    w, wf, blocks = blk
    spec = (MAX_TOKENS_SPEC if workload == "max_tokens_t16384" else MID_SPECS[workload] if workload in MID_SPECS
            else synth.WORKLOADS[workload]["spec"])
    lay = synth.build_layout(spec)
    x = synth.activations(6, lay.T, device=DEV)
    mods = synth.modulation(6, device=DEV)
    y = run_block(blocks, lay, x, mods)
    rows = sample_rows(lay.T, lay.segments)
    m = f64(mods)
    parts = O.single_block_parts(f64(x), wf, m, lay.stream_id, lay.pos.astype(np.float64), rows=rows)
    assert_block_output(f64(y)[rows], parts["out"], f64(x)[rows], m[lay.stream_id[rows], 6144:], parts["y"],
                        workload)


def test_zero_gate_is_bit_exact_identity(blk):
    _, _, blocks = blk
    lay = synth.build_layout(synth.WORKLOADS["block_1024sq_ref1_t8704"]["spec"])
    x = synth.activations(7, lay.T, device=DEV)
    mods = synth.modulation(7, device=DEV)
    mods[:, 6144:] = 0.0
    y = run_block(blocks, lay, x, mods)
    assert torch.equal(y, x)
    # a zero gate for one stream leaves exactly that stream's rows unchanged
    mods = synth.modulation(8, device=DEV)
    mods[1, 6144:] = 0.0
    y = run_block(blocks, lay, x, mods)
    ic = torch.from_numpy(lay.stream_id == 1).to(DEV)
    assert torch.equal(y[ic], x[ic]) and not torch.equal(y[~ic], x[~ic])


def test_stream_isolation_bit_exact(blk):
    _, _, blocks = blk
    lay = synth.build_layout(synth.WORKLOADS["block_1024sq_t4608"]["spec"])   # no image_cond tokens
    x = synth.activations(9, lay.T, device=DEV)
    mods = synth.modulation(9, device=DEV)
    y1 = run_block(blocks, lay, x, mods)
    mods[1] = torch.randn(9216, device=DEV)
    y2 = run_block(blocks, lay, x, mods)
    assert torch.equal(y1, y2)


def test_deterministic_repeat(blk):
    _, _, blocks = blk
    lay = synth.build_layout(synth.WORKLOADS["block_1024sq_ref1_t8704"]["spec"])
    x = synth.activations(10, lay.T, device=DEV)
    mods = synth.modulation(10, device=DEV)
    assert torch.equal(run_block(blocks, lay, x, mods), run_block(blocks, lay, x, mods))


def test_permutation_equivariance(blk):
    """Permuting the tokens together with their ids and streams permutes the
    output (a permuted layout is given as one segment per token run)."""
    _, _, blocks = blk
    lay = synth.build_layout(RAGGED)
    T = lay.T
    x = synth.activations(11, T, device=DEV)
    mods = synth.modulation(11, device=DEV)
    y = run_block(blocks, lay, x, mods)
    perm = np.random.default_rng(0).permutation(T)
    sid_p = lay.stream_id[perm]
    segs = []
    for t in range(T):
        if segs and segs[-1][2] == sid_p[t]:
            segs[-1][1] += 1
        else:
            segs.append([t, 1, int(sid_p[t])])
    if len(segs) > F3.FLUX3_MAX_SEGMENTS:       # keep the table within the ABI limit: sort by stream
        order = np.argsort(sid_p, kind="stable")
        perm = perm[order]
        sid_p = lay.stream_id[perm]
        segs = []
        for t in range(T):
            if segs and segs[-1][2] == sid_p[t]:
                segs[-1][1] += 1
            else:
                segs.append([t, 1, int(sid_p[t])])
    lp = synth.Layout([tuple(s) for s in segs], lay.pos[perm], sid_p)
    yp = run_block(blocks, lp, x[torch.from_numpy(perm).to(DEV)].contiguous(), mods)
    from _f3 import assert_close
    assert_close(f64(yp), f64(y)[perm], 2e-2, 0.9995, "permuted x'")
    assert_close(f64(yp) - f64(x)[perm], f64(y)[perm] - f64(x)[perm], 1e-1, 0.9999, "permuted update")


def test_stack_forward_equals_block_sequence():
    ws = [synth.block_weights(99, b, device=DEV) for b in range(3)]
    blocks = F3.Flux3Blocks(ws, max_tokens=1024)
    lay = synth.build_layout(RAGGED)
    pos, _ = layout_tensors(lay)
    x = synth.activations(12, lay.T, device=DEV)
    mods = synth.modulation(12, device=DEV)
    a = x.clone()
    blocks.forward(a, lay.segments, pos, mods)                 # stack of 3
    b = x.clone()
    for i in range(3):
        blocks.forward(b, lay.segments, pos, mods, first_block=i, n_blocks=1)
    assert F3.flux3_check_error(torch.cuda.current_stream().cuda_stream) == 0
    assert torch.equal(a, b)
