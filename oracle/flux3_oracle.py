"""fp64 NumPy oracle of the FLUX.3 Image Klein joint ``single_block``.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Notation follows the pages: D = hidden 3072, H = 24 heads of d = 128,
F = 9216 SwiGLU width (mlp_in has 2F rows), three token streams ("modes")
image / image_cond / txt, per-stream modulation vector of 3D values in the
chunk order shift, scale, gate.  Linear layers are ``y = x @ W.T`` with the
checkpoint's ``[out, in]`` weight shapes and no bias.

Everything is float64.  Inputs that are bf16 on the device (weights,
activations) are read exactly into float64; the oracle rounds nothing.
"""

import numpy as np

HIDDEN = 3072
HEADS = 24
HEAD_DIM = 128
MLP_HIDDEN = 9216
ROPE_AXES = (32, 32, 32, 32)   # (t, h, w, l)
ROPE_THETA = 10000.0
EPS_LN = 1e-6
EPS_RMS = 1e-6

STREAM_IMAGE = 0
STREAM_IMAGE_COND = 1
STREAM_TXT = 2
N_STREAMS = 3

BLOCK_TENSORS = ("q_proj", "k_proj", "v_proj", "attn_out", "mlp_in", "mlp_out",
                 "query_norm", "key_norm")

__all__ = [
    "HIDDEN", "HEADS", "HEAD_DIM", "MLP_HIDDEN", "ROPE_AXES", "ROPE_THETA",
    "EPS_LN", "EPS_RMS", "STREAM_IMAGE", "STREAM_IMAGE_COND", "STREAM_TXT",
    "N_STREAMS", "BLOCK_TENSORS",
    "block_weight_shapes", "checkpoint_inventory", "rope_ids_from_table",
    "split_modulation", "layer_norm", "modulate", "rms_norm", "rope_frequencies",
    "rope_angles", "apply_rope", "attention", "silu", "swiglu", "qkv_heads",
    "single_block", "single_block_parts", "stack_forward", "mode_blocks_forward",
]


# --------------------------------------------------------------------------
# Shapes ("FLUX.3 Image Klein support", comment "Tensor names (distilled
# checkpoint)"): each block has q_proj, k_proj, v_proj [3072,3072],
# attn_out [3072,3072], mlp_in [18432,3072], mlp_out [3072,9216] and the two
# [128] norm scales.
# --------------------------------------------------------------------------
def block_weight_shapes(hidden=HIDDEN, head_dim=HEAD_DIM, mlp_hidden=MLP_HIDDEN):
    return {
        "q_proj": (hidden, hidden),
        "k_proj": (hidden, hidden),
        "v_proj": (hidden, hidden),
        "attn_out": (hidden, hidden),
        "mlp_in": (2 * mlp_hidden, hidden),
        "mlp_out": (hidden, mlp_hidden),
        "query_norm": (head_dim,),
        "key_norm": (head_dim,),
    }


def checkpoint_inventory():
    """Every tensor of the distilled checkpoint as (name, shape).

    Follows the tensor list in "FLUX.3 Image Klein support", comment "Tensor
    names (distilled checkpoint)": embedders, time_in / ref_time_in, the six
    stream modulation linears, 5 content-mode blocks for image and image_cond,
    5 txt-mode blocks, 28 single blocks and the image final layer.  The same
    comment states the totals (359 tensors, 5.549 B parameters) that pin it.
    """
    inv = [("emb_in.image.weight", (3072, 128)),
           ("emb_in.image_cond.weight", (3072, 128)),
           ("txt_in.weight", (3072, 20480))]
    for emb in ("time_in", "ref_time_in"):
        inv += [(f"{emb}.in_layer.weight", (3072, 256)),
                (f"{emb}.out_layer.weight", (3072, 3072))]
    for group in ("early_stream_modulations", "single_stream_modulations"):
        for mode in ("image", "image_cond", "txt"):
            inv.append((f"{group}.{mode}.lin.weight", (9216, 3072)))
    prefixes = ([f"content_mode_blocks.image.{i}" for i in range(5)]
                + [f"content_mode_blocks.image_cond.{i}" for i in range(5)]
                + [f"txt_mode_blocks.{i}" for i in range(5)]
                + [f"single_blocks.{i}" for i in range(28)])
    names = {"query_norm": "norm.query_norm.scale", "key_norm": "norm.key_norm.scale"}
    for p in prefixes:
        for t, shape in block_weight_shapes().items():
            inv.append((f"{p}.{names.get(t, t + '.weight')}", shape))
    inv += [("final_layer.image.adaLN_modulation.1.weight", (6144, 3072)),
            ("final_layer.image.linear.weight", (128, 3072))]
    return inv


# --------------------------------------------------------------------------
# RoPE ids ("Welcome FLUX.3 Image Klein in Diffusers", table in "Positions in
# four dimensions"; same ids in "FLUX.3 Image Klein support", "Structure"):
#   text token i            -> (0, 0, 0, i)
#   image token (row, col)  -> (0, row/2, col/2, 0)
#   reference k (row, col)  -> (0, row/2, col/2, -(k+1))
# --------------------------------------------------------------------------
def rope_ids_from_table(kind, i=None, row=None, col=None, k=None):
    if kind == "txt":
        return (0.0, 0.0, 0.0, float(i))
    if kind == "image":
        return (0.0, row / 2.0, col / 2.0, 0.0)
    if kind == "image_cond":
        return (0.0, row / 2.0, col / 2.0, -(k + 1.0))
    raise ValueError(kind)


# --------------------------------------------------------------------------
# Modulation ("FLUX.3 Image Klein support", tensor list: modulation linears
# are [9216, 3072] = 3 x 3072: shift, scale, gate).
# --------------------------------------------------------------------------
def split_modulation(mod_row, hidden=HIDDEN):
    mod_row = np.asarray(mod_row, dtype=np.float64)
    return mod_row[..., :hidden], mod_row[..., hidden:2 * hidden], mod_row[..., 2 * hidden:3 * hidden]


def layer_norm(x, eps=EPS_LN):
    """LayerNorm over the last axis with no learned scale or bias, epsilon
    1e-6 and the biased variance ("FLUX.3 Image Klein support", comment
    "Structure (from dit.py)", the block's x_mod line; the variance form is a
    reading)."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def modulate(x, mods, stream_id, eps=EPS_LN):
    """x_mod = (1 + scale) * LayerNorm(x) + shift, with each token's shift and
    scale taken from the modulation vector of the token's own mode ("FLUX.3
    Image Klein support", comment "Structure (from dit.py)", on the shared
    blocks; "Welcome FLUX.3 Image Klein in Diffusers", section "Inside one
    block")."""
    x = np.asarray(x, np.float64)
    shift, scale, _ = split_modulation(np.asarray(mods)[np.asarray(stream_id)], x.shape[-1])
    return (1.0 + scale) * layer_norm(x, eps) + shift


def rms_norm(x, scale, eps=EPS_RMS):
    """RMSNorm of each head's 128 values: x / sqrt(mean(x^2) + eps) * scale,
    with epsilon 1e-6 and a learned scale of length 128 shared by the heads
    ("FLUX.3 Image Klein support", comment "Structure (from dit.py)", applied
    to q and k before RoPE)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * np.asarray(scale, np.float64)


def rope_frequencies(axes=ROPE_AXES, theta=ROPE_THETA):
    """Per axis of width n the n/2 rotation frequencies theta^(-2j/n),
    j = 0..n/2-1 (4 axes of 32, theta 10000: "Structure").  The pages give only
    the axis widths and theta; the per-axis frequency ladder is the standard
    RoPE one.  Returns a list of arrays, one per axis."""
    return [theta ** (-2.0 * np.arange(n // 2, dtype=np.float64) / n) for n in axes]


def rope_angles(pos, axes=ROPE_AXES, theta=ROPE_THETA):
    """Angles [T, sum(axes)/2]: axis a contributes pos[:, a] * freq_a[j]."""
    pos = np.asarray(pos, dtype=np.float64)
    freqs = rope_frequencies(axes, theta)
    return np.concatenate([pos[:, a:a + 1] * f[None, :] for a, f in enumerate(freqs)], axis=1)


def apply_rope(x, pos, axes=None, theta=ROPE_THETA):
    """Rotate x [T, H, d] by 4-axis RoPE ("Positions in four dimensions": each
    axis owns a quarter of every head, in the order t, h, w, l).

    Within axis a (dims [32a, 32a+32)) pair j is the adjacent pair
    (32a+2j, 32a+2j+1), rotated by angle pos[t, a] * freq_a[j]:
    (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos).  The pair layout is a
    reading: the pages are silent on it (parity unpinned beyond the RoPE
    invariants; see the module's tests)."""
    x = np.asarray(x, dtype=np.float64)
    if axes is None:                                 # four equal axes: a quarter of the head each
        axes = (x.shape[-1] // 4,) * 4
    ang = rope_angles(pos, axes, theta)              # [T, d/2], pair index = global pair
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def attention(q, k, v, chunk=256):
    """Bidirectional full attention, no mask: for each head h,
    O_h = softmax(Q_h K_h^T / sqrt(d)) V_h  ("Two stages": in the joint blocks
    everything attends to everything; "From prompt to tokens": the padding is
    attended too).  q, k, v: [T, H, d].  Query rows are processed in chunks
    only to bound memory; each row's softmax is over all T keys."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    tq, nh, d = q.shape
    out = np.empty((tq, nh, v.shape[-1]), dtype=np.float64)
    inv_sqrt_d = 1.0 / np.sqrt(d)
    for h in range(nh):
        kh = k[:, h, :]
        vh = v[:, h, :]
        for r0 in range(0, tq, chunk):
            s = (q[r0:r0 + chunk, h, :] @ kh.T) * inv_sqrt_d
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            out[r0:r0 + chunk, h, :] = p @ vh
    return out


def silu(x):
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(-x))


def swiglu(ab, mlp_hidden=None):
    """SwiGLU of the mlp_in output: with a its first half and b its second,
    returns silu(a) * b ("FLUX.3 Image Klein support", comment "Structure
    (from dit.py)", the block line; which half gates is a reading)."""
    ab = np.asarray(ab, np.float64)
    if mlp_hidden is None:
        mlp_hidden = ab.shape[-1] // 2
    return silu(ab[..., :mlp_hidden]) * ab[..., mlp_hidden:2 * mlp_hidden]


def qkv_heads(h, w, pos, rows=None):
    """Projections of the modulated input and the q/k treatment of the block
    ("Structure": separate q, k, v projections; per-head RMSNorm on q and k,
    then RoPE).  Returns (q_hat, k_hat, v) as [T, H, d]; if ``rows`` is given,
    q_hat holds only those query rows."""
    T, hidden = h.shape
    d = len(w["query_norm"])
    nh = hidden // d
    hq = h if rows is None else h[rows]
    posq = pos if rows is None else np.asarray(pos)[rows]
    q = (hq @ np.asarray(w["q_proj"], np.float64).T).reshape(hq.shape[0], nh, d)
    k = (h @ np.asarray(w["k_proj"], np.float64).T).reshape(T, nh, d)
    v = (h @ np.asarray(w["v_proj"], np.float64).T).reshape(T, nh, d)
    q_hat = apply_rope(rms_norm(q, w["query_norm"]), posq)
    k_hat = apply_rope(rms_norm(k, w["key_norm"]), pos)
    return q_hat, k_hat, v


def single_block_parts(x, w, mods, stream_id, pos, rows=None):
    """The block step by step; returns a dict of intermediates and the output.

    Follows "FLUX.3 Image Klein support", comment "Structure (from dit.py)"
    (the block line), and "Welcome FLUX.3 Image Klein in Diffusers", section
    "Inside one block":
      h      = (1 + scale) * LayerNorm(x) + shift          (per token's stream)
      q, k, v = separate projections of h
      q, k   = RoPE(RMSNorm(q)), RoPE(RMSNorm(k))          (per head)
      attn   = attention(q, k, v)                          (all tokens)
      g      = silu(a) * b,  [a | b] = h mlp_in^T (halves of 9216)
      x'     = x + gate * (attn_out(attn) + mlp_out(g))    (per token's stream)
    ``rows`` restricts the outputs (and q, attention, MLP) to those tokens;
    keys and values always cover all T tokens.  Sizes are taken from the
    arguments (head_dim = len(query_norm)), so the same code runs the full
    3072-wide block and the tiny cases of the tests.
    """
    x = np.asarray(x, np.float64)
    stream_id = np.asarray(stream_id)
    mods = np.asarray(mods, np.float64)
    h = modulate(x, mods, stream_id)
    q_hat, k_hat, v = qkv_heads(h, w, pos, rows)
    o = attention(q_hat, k_hat, v).reshape(q_hat.shape[0], x.shape[1])
    hr = h if rows is None else h[rows]
    ab = hr @ np.asarray(w["mlp_in"], np.float64).T
    g = swiglu(ab)
    y = o @ np.asarray(w["attn_out"], np.float64).T + g @ np.asarray(w["mlp_out"], np.float64).T
    sr = stream_id if rows is None else stream_id[rows]
    _, _, gate = split_modulation(mods[sr], x.shape[1])
    xr = x if rows is None else x[rows]
    out = xr + gate * y
    return {"h": h, "q_hat": q_hat, "k_hat": k_hat, "v": v, "attn": o, "ab": ab,
            "g": g, "y": y, "out": out}


def single_block(x, w, mods, stream_id, pos, rows=None):
    """One joint single_block: returns x' (all tokens, or ``rows``)."""
    return single_block_parts(x, w, mods, stream_id, pos, rows)["out"]


def stack_forward(x, blocks, mods, stream_id, pos):
    """The joint blocks applied in sequence to the residual stream; all blocks
    share the one set of per-stream modulation vectors (the modulation linears'
    names carry no block index: "Tensor names (distilled checkpoint)")."""
    x = np.asarray(x, np.float64)
    for w in blocks:
        x = single_block(x, w, mods, stream_id, pos)
    return x


def mode_blocks_forward(x, mode_blocks, early_mods, stream_id, pos):
    """The per-mode blocks that come before the joint ones ("FLUX.3 Image
    Klein support", comment "Structure (from dit.py)"): five blocks for each
    mode, with weights of that mode alone; a token's attention is limited to
    tokens of its own mode within its sample; the modulation comes from the
    mode's early_stream_modulations linear (weight names
    content_mode_blocks.{image,image_cond}.* and txt_mode_blocks.* in the
    comment's tensor list).

    mode_blocks: for each stream id (image, image_cond, txt) the list of that
    mode's block weights, in order.  early_mods: [3, 3D].  The tokens of each
    mode are taken out of the sequence (keeping their order), run through that
    mode's blocks as a sequence of their own, and written back in place."""
    x = np.array(x, dtype=np.float64)
    stream_id = np.asarray(stream_id)
    pos = np.asarray(pos, np.float64)
    for m in range(N_STREAMS):
        idx = np.nonzero(stream_id == m)[0]
        if idx.size == 0:
            continue
        xm = x[idx]
        for w in mode_blocks[m]:
            xm = single_block(xm, w, early_mods, stream_id[idx], pos[idx])
        x[idx] = xm
    return x
