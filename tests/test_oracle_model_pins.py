"""Pins of the oracle's parts around the block stacks (oracle/flux3_model.py):
the sigma schedule against the figures the pages print, the timestep
embedding's closed forms, torch.nn.functional restatements of the embedder,
modulation and output layer, and the stream rules of the conditioning."""

import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle as O
from oracle import flux3_model as M


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# Schedule ("Welcome FLUX.3 Image Klein in Diffusers", section "The denoising
# loop": the shift 6.93, 44 of 50 steps above sigma 0.5, sigma near 0.97 at
# step 10; "FLUX.3 Image Klein support", comment "Sampling (sampling.py,
# pipeline.py)": the shifted map of evenly spaced t from 1 to 0)
# --------------------------------------------------------------------------
def test_schedule_matches_the_printed_figures():
    s = M.sigma_schedule(50)
    assert len(s) == 51 and s[0] == 1.0 and s[-1] == 0.0
    assert int((s[:50] > 0.5).sum()) == 44
    assert abs(s[10] - 0.97) < 0.005
    assert np.all(np.diff(s) < 0)


def test_schedule_inverse_map_and_sixteen_steps():
    # sigma(t) inverts to t = sigma / (alpha - (alpha - 1) sigma)
    s = M.sigma_schedule(16)
    t = s / (M.SHIFT - (M.SHIFT - 1.0) * s)
    np.testing.assert_allclose(t, np.linspace(1, 0, 17), rtol=0, atol=1e-15)
    # alpha = 1 is the identity schedule
    np.testing.assert_allclose(M.sigma_schedule(8, alpha=1.0), np.linspace(1, 0, 9), atol=1e-15)


def test_euler_steps_telescope():
    rng = _rng(1)
    x0, v = rng.standard_normal(10), rng.standard_normal(10)
    s = M.sigma_schedule(16)
    x = x0
    for k in range(16):
        x = M.euler_step(x, v, s[k], s[k + 1])
    np.testing.assert_allclose(x, x0 - v, rtol=1e-13, atol=1e-13)   # sum of steps = sigma_16 - sigma_0 = -1


# --------------------------------------------------------------------------
# Timestep embedding (comment "Structure (from dit.py)": a 256-wide embedding
# of cosines then sines of 1000 t times the frequencies)
# --------------------------------------------------------------------------
def test_timestep_embedding_closed_forms():
    e0 = M.timestep_embedding(0.0)
    assert e0.shape == (256,) and np.all(e0[:128] == 1.0) and np.all(e0[128:] == 0.0)
    for t in (0.03, 0.5, 0.97, 1.0):
        e = M.timestep_embedding(t)
        np.testing.assert_allclose(e[:128] ** 2 + e[128:] ** 2, 1.0, rtol=1e-14)     # one (cos, sin) pair per freq
        assert e[0] == math.cos(1000.0 * t) and e[128] == math.sin(1000.0 * t)      # the first frequency is 1
    # the ladder runs from 1 down towards 1/max_period
    a = np.arctan2(M.timestep_embedding(1e-3)[128:], M.timestep_embedding(1e-3)[:128]) / 1.0
    np.testing.assert_allclose(a, 10000.0 ** (-np.arange(128) / 128), rtol=1e-12)


# --------------------------------------------------------------------------
# Embedders, modulation, output layer: torch.nn.functional restatements
# --------------------------------------------------------------------------
def _t(a):
    return torch.from_numpy(np.asarray(a, np.float64))


def test_mlp_embedder_and_modulation_match_library():
    rng = _rng(2)
    x = rng.standard_normal(16)
    w_in, w_out = rng.standard_normal((24, 16)) * 0.3, rng.standard_normal((24, 24)) * 0.3
    ref = F.linear(F.silu(F.linear(_t(x), _t(w_in))), _t(w_out)).numpy()
    np.testing.assert_allclose(M.mlp_embedder(x, w_in, w_out), ref, rtol=1e-13, atol=1e-14)
    vec = rng.standard_normal((3, 24))
    lins = [rng.standard_normal((72, 24)) * 0.2 for _ in range(3)]
    ref = np.stack([F.linear(F.silu(_t(vec[s])), _t(lins[s])).numpy() for s in range(3)])
    np.testing.assert_allclose(M.modulation_vectors(vec, lins), ref, rtol=1e-13, atol=1e-14)


def test_final_layer_matches_library():
    rng = _rng(3)
    D = 32
    x = rng.standard_normal((7, D))
    vec = rng.standard_normal(D)
    w_ada, w_lin = rng.standard_normal((2 * D, D)) * 0.2, rng.standard_normal((8, D)) * 0.2
    mod = F.linear(F.silu(_t(vec)), _t(w_ada))
    shift, scale = mod.chunk(2)
    h = (1 + scale) * F.layer_norm(_t(x), (D,), eps=1e-6) + shift
    np.testing.assert_allclose(M.final_layer(x, vec, w_ada, w_lin), F.linear(h, _t(w_lin)).numpy(),
                               rtol=1e-12, atol=1e-13)


def _tiny_cond(rng, D=32, flow=True):
    c = {"time_in_in": rng.standard_normal((D, 256)) * 0.1, "time_in_out": rng.standard_normal((D, D)) * 0.2,
         "early_mod": [rng.standard_normal((3 * D, D)) * 0.2 for _ in range(3)],
         "single_mod": [rng.standard_normal((3 * D, D)) * 0.2 for _ in range(3)],
         "emb_in_image": rng.standard_normal((D, 8)) * 0.3, "emb_in_image_cond": rng.standard_normal((D, 8)) * 0.3,
         "txt_in": rng.standard_normal((D, 40)) * 0.1, "final_adaln": rng.standard_normal((2 * D, D)) * 0.2,
         "final_linear": rng.standard_normal((8, D)) * 0.2}
    if flow:
        c["ref_time_in_in"] = rng.standard_normal((D, 256)) * 0.1
        c["ref_time_in_out"] = rng.standard_normal((D, D)) * 0.2
    return c


def test_stream_vectors_follow_the_timestep_rules():
    rng = _rng(4)
    c = _tiny_cond(rng)
    v = M.stream_vectors(0.6, 0.4, c)
    assert np.array_equal(v[1], v[2])                      # image_cond and txt both at timestep 0
    assert not np.allclose(v[0], v[1])
    v0 = M.stream_vectors(0.0, 0.4, c)
    assert np.array_equal(v0[0], v0[1])                    # at t = 0 the image stream matches them
    # the flow-map term is the same for every stream
    d = M.stream_vectors(0.6, 0.4, c) - M.stream_vectors(0.6, 0.1, c)
    np.testing.assert_allclose(d[0], d[1], rtol=0, atol=1e-15)
    np.testing.assert_allclose(d[0], d[2], rtol=0, atol=1e-15)
    assert np.any(d != 0)
    c.pop("ref_time_in_in"), c.pop("ref_time_in_out")
    assert np.array_equal(M.stream_vectors(0.6, 0.4, c), M.stream_vectors(0.6, 0.1, c))


def test_embed_tokens_routes_each_stream_through_its_embedder():
    rng = _rng(5)
    c = _tiny_cond(rng)
    sid = np.array([2, 2, 0, 0, 0, 1, 1, 0])
    ins = [rng.standard_normal((4, 8)), rng.standard_normal((2, 8)), rng.standard_normal((2, 40))]
    x = M.embed_tokens(ins, sid, c)
    np.testing.assert_allclose(x[[2, 3, 4, 7]], F.linear(_t(ins[0]), _t(c["emb_in_image"])).numpy(), rtol=1e-13)
    np.testing.assert_allclose(x[[5, 6]], F.linear(_t(ins[1]), _t(c["emb_in_image_cond"])).numpy(), rtol=1e-13)
    np.testing.assert_allclose(x[[0, 1]], F.linear(_t(ins[2]), _t(c["txt_in"])).numpy(), rtol=1e-13)


def test_transformer_output_is_the_image_tokens_only():
    """Velocity rows = image tokens in sequence order; text and reference
    inputs reach them only through the joint blocks (zero joint blocks: the
    image velocity ignores the other streams entirely)."""
    from test_oracle_pins import _tiny_block
    rng = _rng(6)
    c = _tiny_cond(rng)
    mode_blocks = [[_tiny_block(rng)] for _ in range(3)]
    joint = [_tiny_block(rng)]
    sid = np.array([2, 2, 2, 0, 0, 0, 0, 1, 1])
    pos = np.zeros((9, 4))
    ins = [rng.standard_normal((4, 8)), rng.standard_normal((2, 8)), rng.standard_normal((3, 40))]
    v = M.transformer_forward(ins, sid, pos, 0.7, 0.5, c, mode_blocks, joint)
    assert v.shape == (4, 8)
    ins2 = [ins[0], ins[1], ins[2] + 1.0]
    assert not np.allclose(M.transformer_forward(ins2, sid, pos, 0.7, 0.5, c, mode_blocks, joint), v)
    assert np.array_equal(M.transformer_forward(ins2, sid, pos, 0.7, 0.5, c, mode_blocks, []),
                          M.transformer_forward(ins, sid, pos, 0.7, 0.5, c, mode_blocks, []))


# --------------------------------------------------------------------------
# Batches of samples (the base model's CFG pack)
# --------------------------------------------------------------------------
def _torch_batch_block(x, w, mods, sample_id, sid, pos):
    """One joint block over concatenated samples in one pass: attention with a
    block-diagonal boolean mask by sample (scaled_dot_product_attention), each
    token's modulation row 3 * sample + stream.  fp64 torch."""
    T, D = x.shape
    d = len(w["query_norm"])
    H = D // d
    tx = _t(x)
    rows = torch.from_numpy(3 * sample_id + sid).long()
    tm = _t(mods)[rows]
    shift, scale, gate = tm[:, :D], tm[:, D:2 * D], tm[:, 2 * D:]
    h = (1 + scale) * F.layer_norm(tx, (D,), eps=1e-6) + shift
    W = {k: _t(v) for k, v in w.items()}
    q, k, v = (F.linear(h, W[n]).view(T, H, d) for n in ("q_proj", "k_proj", "v_proj"))

    def rms(t_, s_):
        return t_ * torch.rsqrt(t_.pow(2).mean(-1, keepdim=True) + 1e-6) * s_

    n = d // 4
    freqs = torch.cat([1e4 ** (-torch.arange(0, n, 2, dtype=torch.float64) / n)] * 4)
    axis = torch.arange(d // 2) // (n // 2)
    rot = torch.polar(torch.ones(T, d // 2, dtype=torch.float64), _t(pos)[:, axis] * freqs)[:, None, :]

    def rope(t_):
        return torch.view_as_real(torch.view_as_complex(t_.reshape(T, H, d // 2, 2).contiguous()) * rot).reshape(T, H, d)

    q, k = rope(rms(q, W["query_norm"])), rope(rms(k, W["key_norm"]))
    smp = torch.from_numpy(sample_id)
    o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                       attn_mask=smp[:, None] == smp[None, :]).transpose(0, 1).reshape(T, D)
    a, b = F.linear(h, W["mlp_in"]).chunk(2, dim=-1)
    return (tx + gate * (F.linear(o, W["attn_out"]) + F.linear(F.silu(a) * b, W["mlp_out"]))).numpy()


def test_batch_matches_sample_masked_restatement():
    from test_oracle_pins import _tiny_block, _tiny_inputs
    rng = _rng(20)
    ws = [_tiny_block(rng) for _ in range(2)]
    x, _, sid, pos = _tiny_inputs(rng, T=15)
    sample_id = np.array([0] * 6 + [1] * 9)
    mods = 0.3 * rng.standard_normal((6, 96))
    y = x
    for w in ws:
        y = _torch_batch_block(y, w, mods, sample_id, sid, pos)
    np.testing.assert_allclose(M.stack_forward_batch(x, ws, mods, sample_id, sid, pos), y, rtol=1e-9, atol=1e-10)


def test_batch_samples_are_isolated():
    from test_oracle_pins import _tiny_block, _tiny_inputs
    rng = _rng(21)
    ws = [_tiny_block(rng)]
    x, _, sid, pos = _tiny_inputs(rng, T=12)
    sample_id = np.array([0] * 5 + [1] * 7)
    mods = 0.3 * rng.standard_normal((6, 96))
    out = M.stack_forward_batch(x, ws, mods, sample_id, sid, pos)
    x2, m2 = x.copy(), mods.copy()
    x2[:5] += 1.0
    m2[:3] += 0.5                                            # sample 0's inputs and modulation only
    out2 = M.stack_forward_batch(x2, ws, m2, sample_id, sid, pos)
    assert np.array_equal(out[5:], out2[5:])
    assert np.all(np.any(out[:5] != out2[:5], axis=1))


def test_cfg_closed_forms():
    rng = _rng(22)
    u, c, x = rng.standard_normal((3, 40))
    np.testing.assert_allclose(M.cfg_velocity(u, c, 1.0), c, rtol=0, atol=1e-15)
    assert np.array_equal(M.cfg_velocity(u, c, 0.0), u)
    np.testing.assert_allclose(M.cfg_velocity(u, c, 3.5), 3.5 * c - 2.5 * u, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(M.cfg_euler_step(x, u, c, 1.0, 0.8, 0.5), x - 0.3 * c, rtol=1e-14, atol=1e-14)


# --------------------------------------------------------------------------
# One whole transformer call against a torch.nn.functional restatement
# (comment "Structure (from dit.py)": embedders, time_in / ref_time_in, the
# per-mode blocks under the early modulations, the joint blocks under the
# single-stream modulations, the image output layer)
# --------------------------------------------------------------------------
def _torch_transformer_call(ins, sid, pos, t, t_next, c, mode_blocks, joint):
    """The call restated in fp64 torch, written apart from the oracle: the
    timestep embedding from its definition, each MLPEmbedder and modulation
    linear with F.linear / F.silu, the per-mode blocks as block-diagonal
    masked passes over the whole sequence, the joint blocks as full passes,
    the output layer with F.layer_norm."""
    from test_oracle_pins import _torch_block, _torch_mode_block

    def temb(tt):
        i = torch.arange(128, dtype=torch.float64)
        a = 1000.0 * tt * torch.exp(-math.log(10000.0) * i / 128.0)
        return torch.cat([torch.cos(a), torch.sin(a)])

    def embedder(e, w_in, w_out):
        return F.linear(F.silu(F.linear(e, _t(w_in))), _t(w_out))

    v_img = embedder(temb(t), c["time_in_in"], c["time_in_out"])
    v_rest = embedder(temb(0.0), c["time_in_in"], c["time_in_out"])
    vec = torch.stack([v_img, v_rest, v_rest])          # rows: image, image_cond, txt
    if "ref_time_in_in" in c:
        vec = vec + embedder(temb(t_next), c["ref_time_in_in"], c["ref_time_in_out"])[None, :]
    early = torch.stack([F.linear(F.silu(vec[s]), _t(c["early_mod"][s])) for s in range(3)]).numpy()
    single = torch.stack([F.linear(F.silu(vec[s]), _t(c["single_mod"][s])) for s in range(3)]).numpy()
    emb = [c["emb_in_image"], c["emb_in_image_cond"], c["txt_in"]]
    T, D = len(sid), vec.shape[1]
    x = torch.zeros((T, D), dtype=torch.float64)
    for s in range(3):
        x[torch.from_numpy(sid == s)] = F.linear(_t(ins[s]), _t(emb[s]))
    x = x.numpy()
    for b in range(len(mode_blocks[0])):
        x = _torch_mode_block(x, [mode_blocks[m][b] for m in range(3)], early, sid, pos)
    for w in joint:
        x = _torch_block(x, w, single, sid, pos)
    ada = F.linear(F.silu(vec[0]), _t(c["final_adaln"]))
    shift, scale = ada[:D], ada[D:]
    img = _t(x)[torch.from_numpy(sid == 0)]
    h = (1.0 + scale) * F.layer_norm(img, (D,), eps=1e-6) + shift
    return F.linear(h, _t(c["final_linear"])).numpy()


def _tiny_call(seed):
    from test_oracle_pins import _tiny_block
    rng = _rng(seed)
    c = _tiny_cond(rng)
    mode_blocks = [[_tiny_block(rng) for _ in range(2)] for _ in range(3)]
    joint = [_tiny_block(rng) for _ in range(2)]
    sid = np.array([2, 2, 2, 0, 0, 0, 0, 0, 0, 1, 1, 1, 1])
    pos = np.zeros((13, 4))
    pos[:3, 3] = np.arange(3)
    pos[3:9, 1], pos[3:9, 2] = np.repeat(np.arange(2), 3) * 0.5, np.tile(np.arange(3), 2) * 0.5
    pos[9:, 1], pos[9:, 2], pos[9:, 3] = np.repeat(np.arange(2), 2) * 0.5, np.tile(np.arange(2), 2) * 0.5, -1.0
    ins = [rng.standard_normal((6, 8)), rng.standard_normal((4, 8)), rng.standard_normal((3, 40))]
    return ins, sid, pos, c, mode_blocks, joint


def test_transformer_call_matches_library_restatement():
    ins, sid, pos, c, mode_blocks, joint = _tiny_call(40)
    for t, t_next in ((0.8, 0.6), (1.0, 0.75)):
        got = M.transformer_forward(ins, sid, pos, t, t_next, c, mode_blocks, joint)
        ref = _torch_transformer_call(ins, sid, pos, t, t_next, c, mode_blocks, joint)
        assert got.shape == (6, 8)
        np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-11)


def test_transformer_call_restatement_catches_planted_wiring_mistakes():
    """Mistakes planted in the oracle's wiring (on the CPU, in copies of its
    inputs) must break the agreement above: the early and single modulation
    sets swapped, the image stream conditioned on t_next instead of t, the
    per-mode and joint blocks run in the other order."""
    ins, sid, pos, c, mode_blocks, joint = _tiny_call(41)
    ref = _torch_transformer_call(ins, sid, pos, 0.8, 0.6, c, mode_blocks, joint)
    scale = float(np.sqrt(np.mean(ref ** 2)))
    swapped = dict(c, early_mod=c["single_mod"], single_mod=c["early_mod"])
    planted = [M.transformer_forward(ins, sid, pos, 0.8, 0.6, swapped, mode_blocks, joint),
               M.transformer_forward(ins, sid, pos, 0.6, 0.6, c, mode_blocks, joint)]
    # blocks in the other order: the joint blocks first, then the per-mode ones
    vec = M.stream_vectors(0.8, 0.6, c)
    x = M.embed_tokens(ins, sid, c)
    x = O.stack_forward(x, joint, M.modulation_vectors(vec, c["single_mod"]), sid, pos)
    x = O.mode_blocks_forward(x, mode_blocks, M.modulation_vectors(vec, c["early_mod"]), sid, pos)
    planted.append(M.final_layer(x[sid == 0], vec[0], c["final_adaln"], c["final_linear"]))
    for p in planted:
        assert np.abs(p - ref).max() > 1e-3 * scale
