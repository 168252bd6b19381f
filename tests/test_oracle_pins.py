"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each check is a value printed
by the pages (tests/golden/), a closed form, an invariant of the operation, a
brute-force definition on tiny inputs, or a library routine that computes the
same textbook operation.  Each is chosen so that a plausible slip (a dropped
term, a wrong sign or index, a swapped chunk) fails it.
"""

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle as O
import synth


def _rng(seed=0):
    return np.random.default_rng(seed)


def _tiny_block(rng, hidden=32, head_dim=8, mlp_hidden=48, std=0.3):
    shapes = O.block_weight_shapes(hidden, head_dim, mlp_hidden)
    w = {}
    for name, shape in shapes.items():
        if name.endswith("norm"):
            w[name] = 1.0 + 0.1 * rng.standard_normal(shape)
        else:
            w[name] = std * rng.standard_normal(shape)
    return w


def _tiny_inputs(rng, T=11, hidden=32, streams=(0, 1, 2)):
    x = rng.standard_normal((T, hidden))
    mods = 0.3 * rng.standard_normal((3, 3 * hidden))
    sid = np.array([streams[i % len(streams)] for i in range(T)])
    pos = np.stack([rng.integers(0, 3, T), rng.integers(0, 5, T) * 0.5,
                    rng.integers(0, 5, T) * 0.5, -rng.integers(0, 4, T)], axis=1).astype(np.float64)
    return x, mods, sid, pos


# --------------------------------------------------------------------------
# P1: shapes and parameter totals printed by the pages
# --------------------------------------------------------------------------
def test_checkpoint_totals_match_printed(golden_dir):
    vals = {}
    for line in open(os.path.join(golden_dir, "checkpoint_totals.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = v
    inv = O.checkpoint_inventory()
    assert len(inv) == int(vals["tensors"])
    total = sum(int(np.prod(s)) for _, s in inv)
    assert round(total / 1e9, 3) == float(vals["params_billions_3dp"])
    # the single-block share of it: 6 matrices + 2 norm scales
    per_block = sum(int(np.prod(s)) for s in O.block_weight_shapes().values())
    assert per_block == 4 * 3072 * 3072 + 18432 * 3072 + 3072 * 9216 + 2 * 128


def test_block_shapes_are_the_listed_ones():
    s = O.block_weight_shapes()
    assert s["mlp_in"] == (18432, 3072) and s["mlp_out"] == (3072, 9216)
    assert s["q_proj"] == s["k_proj"] == s["v_proj"] == s["attn_out"] == (3072, 3072)
    assert s["query_norm"] == s["key_norm"] == (128,)
    assert O.HEADS * O.HEAD_DIM == O.HIDDEN and sum(O.ROPE_AXES) == O.HEAD_DIM


# --------------------------------------------------------------------------
# RoPE ids: the page table and the token layout of the synthetic workloads
# --------------------------------------------------------------------------
def _golden_rope_rows(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "rope_ids.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        kind, idx, *vals = line.split()
        rows.append((kind, [float(v) for v in idx.split(",")], [float(v) for v in vals]))
    return rows


def test_rope_id_table(golden_dir):
    for kind, idx, want in _golden_rope_rows(golden_dir):
        if kind == "txt":
            got = O.rope_ids_from_table("txt", i=idx[0])
        elif kind == "image":
            got = O.rope_ids_from_table("image", row=idx[0], col=idx[1])
        else:
            got = O.rope_ids_from_table("image_cond", row=idx[0], col=idx[1], k=idx[2])
        assert list(got) == want, (kind, idx)


def test_synth_layout_follows_rope_table(golden_dir):
    refs = [("image_cond", (32, 32))] * 10
    lay = synth.build_layout([("txt", 160), ("image", (64, 64))] + refs)
    assert lay.T == 160 + 4096 + 10 * 1024
    for kind, idx, want in _golden_rope_rows(golden_dir):
        if kind == "txt":
            t = int(idx[0])
        elif kind == "image":
            t = 160 + int(idx[0]) * 64 + int(idx[1])
        else:
            t = 160 + 4096 + int(idx[2]) * 1024 + int(idx[0]) * 32 + int(idx[1])
        assert list(lay.pos[t].astype(np.float64)) == want, (kind, idx)
    assert [s[2] for s in lay.segments] == [synth.STREAM_TXT, synth.STREAM_IMAGE] + [synth.STREAM_IMAGE_COND] * 10


def test_token_counts_of_the_speed_figure(golden_dir):
    for line in open(os.path.join(golden_dir, "token_counts.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        name, total, img, refs = line.split()
        w, h = (int(v) for v in img.split("x"))
        n_img = (w // 16) * (h // 16)
        n_ref = 0 if refs == "-" else sum((int(a) // 16) * (int(b) // 16)
                                          for a, b in (r.split("x") for r in refs.split(",")))
        n_txt = int(total) - n_img - n_ref
        assert n_txt > 0 and n_txt % 80 == 0 and n_txt <= 4096, name
    # the workloads' own counts
    assert synth.build_layout(synth.WORKLOADS["block_1024sq_t4608"]["spec"]).T == 4608
    assert synth.build_layout(synth.WORKLOADS["block_1024sq_ref1_t8704"]["spec"]).T == 8704
    assert synth.build_layout(synth.WORKLOADS["stack28_1024sq_2ref512_t6656"]["spec"]).T == 6656
    assert synth.build_layout(synth.WORKLOADS["stack28_nvfp4_1024sq_10ref512_t14848"]["spec"]).T == 14848
    assert synth.build_layout(synth.WORKLOADS["block_t96"]["spec"]).T == 96


# --------------------------------------------------------------------------
# P2: RoPE
# --------------------------------------------------------------------------
def test_rope_identity_at_zero_and_norm_preserving():
    rng = _rng(1)
    x = rng.standard_normal((5, 3, 128))
    assert np.array_equal(O.apply_rope(x, np.zeros((5, 4))), x)
    pos = rng.standard_normal((5, 4)) * 50
    y = O.apply_rope(x, pos)
    # every rotated pair keeps its length
    np.testing.assert_allclose(y[..., 0::2] ** 2 + y[..., 1::2] ** 2,
                               x[..., 0::2] ** 2 + x[..., 1::2] ** 2, rtol=1e-12, atol=1e-12)


def test_rope_matches_complex_rotation_of_pairs():
    """A pair (x0, x1) read as the complex number x0 + i x1 is multiplied by
    exp(i * angle): the textbook statement of a rotation (catches a sign slip)."""
    rng = _rng(2)
    x = rng.standard_normal((7, 2, 128))
    pos = np.array([[0, 1.5, 3.0, -2.0]] * 7) + rng.integers(0, 4, (7, 4))
    y = O.apply_rope(x, pos)
    xt = torch.view_as_complex(torch.from_numpy(x.reshape(7, 2, 64, 2)).contiguous())
    ang = torch.from_numpy(O.rope_angles(pos))[:, None, :]
    yt = torch.view_as_real(xt * torch.polar(torch.ones_like(ang), ang)).reshape(7, 2, 128).numpy()
    np.testing.assert_allclose(y, yt, rtol=1e-12, atol=1e-12)


def test_rope_first_pair_of_each_axis_turns_by_the_position():
    """The highest frequency of each axis is 1 rad per unit of position: a unit
    vector in pair 0 of axis a at position pi/2 on that axis turns by 90 degrees."""
    for a in range(4):
        x = np.zeros((1, 1, 128))
        x[0, 0, 32 * a] = 1.0
        pos = np.zeros((1, 4))
        pos[0, a] = math.pi / 2
        y = O.apply_rope(x, pos)
        want = np.zeros(128)
        want[32 * a + 1] = 1.0
        np.testing.assert_allclose(y[0, 0], want, atol=1e-15)
    f = O.rope_frequencies()
    assert all(len(fa) == 16 and fa[0] == 1.0 and np.all(np.diff(fa) < 0) for fa in f)
    # theta sets the slowest pair: 16 pairs span a factor theta^(30/32)
    np.testing.assert_allclose(f[0][0] / f[0][-1], 1e4 ** (30 / 32), rtol=1e-12)


def test_rope_each_axis_owns_its_quarter():
    rng = _rng(3)
    x = rng.standard_normal((4, 2, 128))
    base = rng.standard_normal((4, 4))
    y0 = O.apply_rope(x, base)
    for a in range(4):
        p = base.copy()
        p[:, a] += 0.75
        y1 = O.apply_rope(x, p)
        changed = np.any(np.abs(y1 - y0) > 1e-12, axis=(0, 1))
        assert np.all(changed[32 * a:32 * a + 32]) and not np.any(np.delete(changed, np.s_[32 * a:32 * a + 32]))


def test_rope_relative_position_property():
    """<rope(q, p), rope(k, p')> depends only on p - p' (per axis), including
    half-integer and negative shifts."""
    rng = _rng(4)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    p = np.array([[0.0, 3.5, 7.0, -1.0]])
    pk = np.array([[0.0, 1.0, 0.5, 5.0]])
    ref = np.sum(O.apply_rope(q, p) * O.apply_rope(k, pk))
    for delta in ([0, 0.5, -3.5, -4.0], [2, 17.5, 100.0, 333.0], [-1, -0.5, 0.0, -7.0]):
        d = np.array([delta], np.float64)
        got = np.sum(O.apply_rope(q, p + d) * O.apply_rope(k, pk + d))
        assert abs(got - ref) < 1e-9 * (1 + abs(ref))
    # and it does depend on the difference
    other = np.sum(O.apply_rope(q, p + np.array([[0, 1.0, 0, 0]])) * O.apply_rope(k, pk))
    assert abs(other - ref) > 1e-6


# --------------------------------------------------------------------------
# LayerNorm, modulation, RMSNorm
# --------------------------------------------------------------------------
def test_layer_norm_matches_library_and_has_zero_mean_unit_variance():
    rng = _rng(5)
    x = rng.standard_normal((6, 3072)) * 3 + 1.5
    y = O.layer_norm(x)
    yt = F.layer_norm(torch.from_numpy(x), (3072,), eps=1e-6).numpy()
    np.testing.assert_allclose(y, yt, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(y.mean(1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(1), 1 - 1e-6 / x.var(1), rtol=1e-9)


def test_modulation_uses_the_tokens_stream_and_the_one_plus_scale_form():
    rng = _rng(6)
    D = 16
    x = rng.standard_normal((3, D))
    mods = rng.standard_normal((3, 3 * D))
    sid = np.array([2, 0, 1])
    # scale = -1 removes the normalised input entirely: h = shift
    m2 = mods.copy()
    m2[:, D:2 * D] = -1.0
    np.testing.assert_allclose(O.modulate(x, m2, sid), m2[sid, :D], atol=1e-15)
    # scale = 0, shift = 0 is plain LayerNorm
    m3 = np.zeros_like(mods)
    np.testing.assert_allclose(O.modulate(x, m3, sid), O.layer_norm(x), atol=1e-15)
    # each row uses its own stream's vector
    h = O.modulate(x, mods, sid)
    for t, s in enumerate(sid):
        ln = F.layer_norm(torch.from_numpy(x[t]), (D,), eps=1e-6).numpy()
        np.testing.assert_allclose(h[t], (1 + mods[s, D:2 * D]) * ln + mods[s, :D], rtol=1e-12, atol=1e-12)


def test_rms_norm_closed_form():
    c = np.array([[[-2.5] * 128, [0.125] * 128]])
    scale = np.linspace(0.5, 1.5, 128)
    y = O.rms_norm(c, scale)
    np.testing.assert_allclose(y[0, 0], -2.5 / math.sqrt(6.25 + 1e-6) * scale, rtol=1e-14)
    np.testing.assert_allclose(y[0, 1], 0.125 / math.sqrt(0.015625 + 1e-6) * scale, rtol=1e-14)
    # scale-invariance of the input (up to eps)
    rng = _rng(7)
    v = rng.standard_normal((3, 128))
    np.testing.assert_allclose(O.rms_norm(1000 * v, scale), O.rms_norm(v, scale), rtol=1e-6)


# --------------------------------------------------------------------------
# P3: attention
# --------------------------------------------------------------------------
def _attention_triple_loop(q, k, v):
    T, H, d = q.shape
    out = np.zeros((T, H, v.shape[2]))
    for h in range(H):
        for i in range(T):
            logits = [sum(q[i, h, c] * k[j, h, c] for c in range(d)) / math.sqrt(d) for j in range(k.shape[0])]
            m = max(logits)
            e = [math.exp(s - m) for s in logits]
            z = sum(e)
            for j in range(k.shape[0]):
                for c in range(v.shape[2]):
                    out[i, h, c] += e[j] / z * v[j, h, c]
    return out


def test_attention_equals_brute_force_on_tiny_inputs():
    rng = _rng(8)
    for T in (1, 3, 8):
        q, k, v = (rng.standard_normal((T, 2, 4)) * 2 for _ in range(3))
        np.testing.assert_allclose(O.attention(q, k, v, chunk=2), _attention_triple_loop(q, k, v),
                                   rtol=1e-12, atol=1e-12)


def test_attention_rows_sum_to_one_and_match_library():
    rng = _rng(9)
    q, k, v = (rng.standard_normal((300, 3, 128)) for _ in range(3))
    ones = np.ones_like(v)
    np.testing.assert_allclose(O.attention(q, k, ones), 1.0, atol=1e-12)
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(a).transpose(0, 1) for a in (q, k, v)))
    np.testing.assert_allclose(O.attention(q, k, v, chunk=64), ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)


def test_attention_scale_is_inverse_sqrt_head_dim():
    """Two keys whose logits differ by sqrt(d): weights are 1/(1+e) and e/(1+e)."""
    d = 128
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 1.0
    k = np.zeros((2, 1, d))
    k[1, 0, 0] = math.sqrt(d)
    v = np.zeros((2, 1, d))
    v[0, 0, 0] = 1.0
    v[1, 0, 1] = 1.0
    o = O.attention(q, k, v)
    np.testing.assert_allclose(o[0, 0, :2], [1 / (1 + math.e), math.e / (1 + math.e)], rtol=1e-14)


# --------------------------------------------------------------------------
# SwiGLU chunk order
# --------------------------------------------------------------------------
def test_swiglu_gates_the_second_half_by_silu_of_the_first():
    ab = np.concatenate([np.full((1, 4), 1.0), np.full((1, 4), 2.0)], axis=1)
    np.testing.assert_allclose(O.swiglu(ab), 2.0 / (1 + math.exp(-1.0)), rtol=1e-15)
    np.testing.assert_allclose(O.silu(np.array([-1.0, 0.0, 3.0])),
                               F.silu(torch.tensor([-1.0, 0.0, 3.0], dtype=torch.float64)).numpy(), rtol=1e-15)


# --------------------------------------------------------------------------
# Block: P3 (library restatement), P4 (zero gate), P5 (permutation), P6
# --------------------------------------------------------------------------
def _torch_block(x, w, mods, sid, pos):
    """Independent restatement with torch.nn.functional routines in fp64:
    layer_norm, scaled_dot_product_attention, silu; RoPE as complex
    multiplication; RMSNorm written out."""
    T, D = x.shape
    d = len(w["query_norm"])
    H = D // d
    tx = torch.from_numpy(x)
    tm = torch.from_numpy(mods)[torch.from_numpy(sid).long()]
    shift, scale, gate = tm[:, :D], tm[:, D:2 * D], tm[:, 2 * D:]
    h = (1 + scale) * F.layer_norm(tx, (D,), eps=1e-6) + shift
    W = {k: torch.from_numpy(np.asarray(v)) for k, v in w.items()}
    q, k, v = (F.linear(h, W[n]).view(T, H, d) for n in ("q_proj", "k_proj", "v_proj"))

    def rms(t, s):
        return t * torch.rsqrt(t.pow(2).mean(-1, keepdim=True) + 1e-6) * s

    n = d // 4
    freqs = torch.cat([1e4 ** (-torch.arange(0, n, 2, dtype=torch.float64) / n)] * 4)
    axis = torch.arange(d // 2) // (n // 2)
    ang = torch.from_numpy(pos)[:, axis] * freqs
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]

    def rope(t):
        return torch.view_as_real(torch.view_as_complex(t.reshape(T, H, d // 2, 2).contiguous()) * rot).reshape(T, H, d)

    q, k = rope(rms(q, W["query_norm"])), rope(rms(k, W["key_norm"]))
    o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1)).transpose(0, 1)
    a, b = F.linear(h, W["mlp_in"]).chunk(2, dim=-1)
    out = F.linear(o.reshape(T, D), W["attn_out"]) + F.linear(F.silu(a) * b, W["mlp_out"])
    return (tx + gate * out).numpy()


def test_block_matches_library_restatement():
    rng = _rng(10)
    w = _tiny_block(rng)
    x, mods, sid, pos = _tiny_inputs(rng)
    np.testing.assert_allclose(O.single_block(x, w, mods, sid, pos), _torch_block(x, w, mods, sid, pos),
                               rtol=1e-10, atol=1e-11)


def test_block_full_width_matches_library_restatement():
    """The real sizes (3072 wide, 24 x 128 heads, 9216 SwiGLU) on a few tokens."""
    rng = _rng(11)
    w = {k: (1.0 + 0.1 * rng.standard_normal(s)) if k.endswith("norm") else 0.02 * rng.standard_normal(s)
         for k, s in O.block_weight_shapes().items()}
    lay = synth.build_layout([("txt", 3), ("image", (2, 3)), ("image_cond", (1, 2))])
    x = rng.standard_normal((lay.T, 3072))
    mods = 0.1 * rng.standard_normal((3, 9216))
    got = O.single_block(x, w, mods, lay.stream_id, lay.pos)
    np.testing.assert_allclose(got, _torch_block(x, w, mods, lay.stream_id, lay.pos.astype(np.float64)),
                               rtol=1e-9, atol=1e-10)


def test_zero_gate_is_identity_and_per_stream():
    rng = _rng(12)
    w = _tiny_block(rng)
    x, mods, sid, pos = _tiny_inputs(rng)
    m0 = mods.copy()
    m0[:, 64:] = 0.0
    assert np.array_equal(O.single_block(x, w, m0, sid, pos), x)
    m1 = mods.copy()
    m1[1, 64:] = 0.0                      # only image_cond gated off
    out = O.single_block(x, w, m1, sid, pos)
    assert np.array_equal(out[sid == 1], x[sid == 1])
    assert np.all(np.any(out[sid != 1] != x[sid != 1], axis=1))


def test_permutation_equivariance():
    rng = _rng(13)
    w = _tiny_block(rng)
    x, mods, sid, pos = _tiny_inputs(rng, T=13)
    perm = rng.permutation(13)
    out = O.single_block(x, w, mods, sid, pos)
    outp = O.single_block(x[perm], w, mods, sid[perm], pos[perm])
    np.testing.assert_allclose(outp, out[perm], rtol=1e-10, atol=1e-12)


def test_stream_isolation_of_modulation():
    rng = _rng(14)
    w = _tiny_block(rng)
    x, mods, sid, pos = _tiny_inputs(rng, streams=(0, 2))
    m2 = mods.copy()
    m2[1] = rng.standard_normal(m2.shape[1])     # image_cond vector, no image_cond tokens
    assert np.array_equal(O.single_block(x, w, mods, sid, pos), O.single_block(x, w, m2, sid, pos))


def test_sampled_rows_equal_full_block():
    rng = _rng(15)
    w = _tiny_block(rng)
    x, mods, sid, pos = _tiny_inputs(rng, T=17)
    rows = np.array([0, 5, 16, 7])
    np.testing.assert_allclose(O.single_block(x, w, mods, sid, pos, rows=rows),
                               O.single_block(x, w, mods, sid, pos)[rows], rtol=1e-12, atol=1e-13)


def test_stack_is_blocks_in_sequence_sharing_modulation():
    rng = _rng(16)
    ws = [_tiny_block(rng) for _ in range(3)]
    x, mods, sid, pos = _tiny_inputs(rng)
    y = x
    for w in ws:
        y = _torch_block(y, w, mods, sid, pos)
    np.testing.assert_allclose(O.stack_forward(x, ws, mods, sid, pos), y, rtol=1e-9, atol=1e-10)


# --------------------------------------------------------------------------
# Per-mode blocks ("FLUX.3 Image Klein support", "Structure (from dit.py)":
# the first 5 blocks are per mode, own weights, attention only among the
# mode's own tokens, modulation from early_stream_modulations)
# --------------------------------------------------------------------------
def _torch_mode_block(x, w_by_mode, mods, sid, pos):
    """Independent restatement over the whole sequence at once: each token's
    projections, norm scales and output projections are those of its mode
    (computed with all three modes' weights, the token's row selected), and
    attention is scaled_dot_product_attention with a block-diagonal boolean
    mask (query and key of the same mode).  fp64 torch."""
    T, D = x.shape
    d = len(w_by_mode[0]["query_norm"])
    H = D // d
    tx = torch.from_numpy(x)
    ts = torch.from_numpy(sid).long()
    tm = torch.from_numpy(mods)[ts]
    shift, scale, gate = tm[:, :D], tm[:, D:2 * D], tm[:, 2 * D:]
    h = (1 + scale) * F.layer_norm(tx, (D,), eps=1e-6) + shift
    Ws = [{k: torch.from_numpy(np.asarray(v)) for k, v in w.items()} for w in w_by_mode]
    rows = torch.arange(T)

    def per_mode(fn):
        return torch.stack([fn(W) for W in Ws])[ts, rows]

    def rms(t, s):
        return t * torch.rsqrt(t.pow(2).mean(-1, keepdim=True) + 1e-6) * s

    n = d // 4
    freqs = torch.cat([1e4 ** (-torch.arange(0, n, 2, dtype=torch.float64) / n)] * 4)
    axis = torch.arange(d // 2) // (n // 2)
    ang = torch.from_numpy(pos)[:, axis] * freqs
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]

    def rope(t):
        return torch.view_as_real(torch.view_as_complex(t.reshape(T, H, d // 2, 2).contiguous()) * rot).reshape(T, H, d)

    q = per_mode(lambda W: rope(rms(F.linear(h, W["q_proj"]).view(T, H, d), W["query_norm"])))
    k = per_mode(lambda W: rope(rms(F.linear(h, W["k_proj"]).view(T, H, d), W["key_norm"])))
    v = per_mode(lambda W: F.linear(h, W["v_proj"]).view(T, H, d))
    mask = ts[:, None] == ts[None, :]
    o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                       attn_mask=mask).transpose(0, 1).reshape(T, D)

    def mlp(W):
        a, b = F.linear(h, W["mlp_in"]).chunk(2, dim=-1)
        return F.linear(F.silu(a) * b, W["mlp_out"])

    out = per_mode(lambda W: F.linear(o, W["attn_out"])) + per_mode(mlp)
    return (tx + gate * out).numpy()


def test_mode_blocks_match_masked_restatement():
    """Modes interleaved (each mode in several runs), two blocks per mode with
    different weights: the oracle's per-mode sub-sequences against one
    block-diagonal masked pass over the whole sequence per block."""
    rng = _rng(30)
    blocks = [[_tiny_block(rng) for _ in range(2)] for _ in range(3)]
    x, mods, sid, pos = _tiny_inputs(rng, T=14)
    y = x
    for b in range(2):
        y = _torch_mode_block(y, [blocks[m][b] for m in range(3)], mods, sid, pos)
    np.testing.assert_allclose(O.mode_blocks_forward(x, blocks, mods, sid, pos), y, rtol=1e-9, atol=1e-10)


def test_mode_blocks_attend_within_their_mode_only():
    rng = _rng(31)
    blocks = [[_tiny_block(rng)] for _ in range(3)]
    x, mods, sid, pos = _tiny_inputs(rng, T=12)
    out = O.mode_blocks_forward(x, blocks, mods, sid, pos)
    x2 = x.copy()
    x2[sid == 2] += rng.standard_normal(x2[sid == 2].shape)   # change only the txt tokens
    out2 = O.mode_blocks_forward(x2, blocks, mods, sid, pos)
    assert np.array_equal(out[sid != 2], out2[sid != 2])
    assert np.all(np.any(out[sid == 2] != out2[sid == 2], axis=1))
    # and the joint block mixes them
    j1 = O.single_block(x, blocks[0][0], mods, sid, pos)
    j2 = O.single_block(x2, blocks[0][0], mods, sid, pos)
    assert np.all(np.any(j1[sid == 0] != j2[sid == 0], axis=1))


def test_mode_blocks_one_mode_is_that_modes_stack():
    rng = _rng(32)
    blocks = [[_tiny_block(rng) for _ in range(2)] for _ in range(3)]
    x, mods, _, pos = _tiny_inputs(rng, T=9)
    sid = np.full(9, 1)
    np.testing.assert_allclose(O.mode_blocks_forward(x, blocks, mods, sid, pos),
                               O.stack_forward(x, blocks[1], mods, sid, pos), rtol=1e-12, atol=1e-13)
