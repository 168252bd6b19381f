"""One transformer call around the block stacks on the GPU against the oracle
(oracle/flux3_model.py): conditioning vectors, input embedders and the image
output layer at full size, the Euler step, and the composed call
(conditioning, embedders, per-mode blocks, joint blocks, output layer) at 112
tokens against the oracle's chain and at 4608 tokens against its own steps.
No GPU value ever feeds the oracle."""

import numpy as np
import pytest
import torch

import diffusion_transformer_block_fwd_b300 as F3
from diffusion_transformer_block_fwd_b300.model import mode_blocks_forward
import oracle as O
import synth
from _f3 import DEV, assert_close, f64, layout_tensors, weights_f64
from oracle import flux3_model as M

pytestmark = pytest.mark.gpu


def _sync_ok():
    assert F3.flux3_check_error(torch.cuda.current_stream().cuda_stream) == 0


def _cond64(w):
    out = {}
    for k, v in w.items():
        if v is None:
            out[k] = None
        elif isinstance(v, list):
            out[k] = [f64(t) for t in v]
        else:
            out[k] = f64(v)
    return out


@pytest.fixture(scope="module", params=[True, False], ids=["flow_map", "base"])
def cond(request):
    w = synth.cond_weights(700, device=DEV, flow=request.param)
    return w, F3.Flux3Conditioning(w), _cond64(w)


def test_conditioning_matches_oracle(cond):
    _, c, w64 = cond
    for t, tn in ((0.73, 0.61), (1.0, 0.97), (0.02, 0.0)):
        early, single, fin = c.modulations(t, tn)
        _sync_ok()
        vec = M.stream_vectors(t, tn, w64)
        for got, lins in ((early, w64["early_mod"]), (single, w64["single_mod"])):
            ref = M.modulation_vectors(vec, lins)
            assert_close(f64(got), ref, 1e-4, 0.99999999, f"modulation t={t}")
        ref_fin = np.asarray(O.silu(vec[0]) @ w64["final_adaln"].T)
        assert_close(f64(fin)[:6144], ref_fin, 1e-4, 0.99999999, f"final adaLN t={t}")
        assert not fin[6144:].any()


@pytest.mark.parametrize("workload", ["block_1024sq_t4608", "block_1024sq_ref1_t8704"])
def test_embed_tokens_full_size(cond, workload):
    """Exact bf16 inputs and weights, float32 accumulation in the tensor core
    against float64: over K = 20480 text features the largest deviation seen
    is ~1.3e-4 of RMS(x); bound 1e-3 (a quarter of one bf16 rounding) and
    cosine 0.9999999."""
    _, c, w64 = cond
    lay = synth.build_layout(synth.WORKLOADS[workload]["spec"])
    ins = synth.stream_inputs(71, lay, device=DEV)
    x = c.embed(ins, lay.segments, lay.T)
    _sync_ok()
    ref = M.embed_tokens([f64(t) if t is not None else None for t in ins], lay.stream_id, w64)
    for s in range(3):
        r = lay.stream_id == s
        if r.any():
            assert_close(f64(x)[r], ref[r], 1e-3, 0.9999999, f"stream {s}")


def test_final_layer_full_size(cond):
    _, c, w64 = cond
    lay = synth.build_layout(synth.WORKLOADS["block_1024sq_ref1_t8704"]["spec"])
    x = synth.activations(72, lay.T, device=DEV)
    _, _, fin = c.modulations(0.5, 0.4)
    v = c.final_layer(x, lay.segments, fin)
    _sync_ok()
    img = np.nonzero(lay.stream_id == 0)[0]
    vec = M.stream_vectors(0.5, 0.4, w64)
    ref = M.final_layer(f64(x)[img], vec[0], w64["final_adaln"], w64["final_linear"])
    assert v.shape == (len(img), 128)
    assert_close(f64(v), ref, 2e-2, 0.9995, "velocity")


def test_euler_step():
    lat = synth.activations(73, 64, device=DEV)[:, :128].contiguous()
    v = synth.activations(74, 64, device=DEV)[:, :128].contiguous()
    sig = F3.flux3_sigma_schedule(16)
    x = lat.clone()
    nxt = torch.empty(x.shape, dtype=torch.bfloat16, device=DEV)
    F3.flux3_euler_step(x.data_ptr(), v.data_ptr(), x.numel(), sig[3], sig[4], nxt.data_ptr())
    _sync_ok()
    dt = np.float32(np.float64(sig[4]) - np.float64(sig[3]))
    want = (f64(lat) + np.float64(dt) * f64(v)).astype(np.float32)     # one rounding: fused multiply-add
    assert np.array_equal(x.cpu().numpy(), want)
    assert torch.equal(nxt.cpu(), torch.from_numpy(want).to(torch.bfloat16))   # the next input: nearest-even bf16
    first = torch.empty(x.shape, dtype=torch.bfloat16, device=DEV)
    F3.flux3_latents_to_bf16(lat.data_ptr(), lat.numel(), first.data_ptr())
    _sync_ok()
    assert torch.equal(first.cpu(), lat.cpu().to(torch.bfloat16))


def test_transformer_small_against_oracle(cond):
    """112 tokens (txt 32, image 8x8, one 4x4 reference), 2 per-mode blocks
    per mode, 3 joint blocks; the oracle's chain from the same inputs."""
    w, c, w64 = cond
    lay = synth.build_layout(synth.WORKLOADS["modes5_t112"]["spec"])
    pos, _ = layout_tensors(lay)
    mw = [[synth.block_weights(7100 + m, b, device=DEV) for b in range(2)] for m in range(3)]
    jw = [synth.block_weights(7200, b, device=DEV) for b in range(3)]
    mb = [F3.Flux3Blocks(mw[m], max_tokens=512) for m in range(3)]
    joint = F3.Flux3Blocks(jw, max_tokens=512)
    model = F3.Flux3Transformer(c, mb, joint)
    ins = synth.stream_inputs(75, lay, device=DEV)
    v = model.forward(ins, lay.segments, pos, 0.81, 0.7)
    _sync_ok()
    ref = M.transformer_forward([f64(t) for t in ins], lay.stream_id, lay.pos.astype(np.float64), 0.81, 0.7, w64,
                                [(weights_f64(b) for b in mw[m]) for m in range(3)],
                                (weights_f64(b) for b in jw))
    assert_close(f64(v), ref, 2e-2, 0.9995, "velocity")


def test_transformer_full_size_is_its_steps():
    """4608 tokens (txt 512, image 64x64), 5 per-mode blocks, 28 joint blocks:
    the call equals conditioning, embedders, per-mode blocks, joint blocks and
    output layer run one by one, bit for bit; finite."""
    w = synth.cond_weights(701, device=DEV)
    c = F3.Flux3Conditioning(w)
    lay = synth.build_layout(synth.WORKLOADS["block_1024sq_t4608"]["spec"])
    pos, _ = layout_tensors(lay)
    counts = [int((lay.stream_id == m).sum()) for m in range(3)]
    mb = [F3.Flux3Blocks([synth.block_weights(7300 + m, b, device=DEV) for b in range(5)], max_tokens=4608)
          if counts[m] else None for m in range(3)]
    joint = F3.Flux3Blocks([synth.block_weights(7400, b, device=DEV) for b in range(28)], max_tokens=4608)
    model = F3.Flux3Transformer(c, mb, joint)
    ins = synth.stream_inputs(76, lay, device=DEV)
    v = model.forward(ins, lay.segments, pos, 0.9, 0.8)
    _sync_ok()
    assert torch.isfinite(v).all() and v.shape == (4096, 128)
    early, single, fin = c.modulations(0.9, 0.8)
    x = c.embed(ins, lay.segments, lay.T)
    mode_blocks_forward(mb, x, lay.segments, pos, early)
    joint.forward(x, lay.segments, pos, single)
    v2 = c.final_layer(x, lay.segments, fin)
    _sync_ok()
    assert torch.equal(v, v2)
