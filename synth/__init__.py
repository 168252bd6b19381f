"""Seeded synthetic inputs for the joint single_block: token layouts, RoPE
position ids, random-init weights, activations and modulation vectors.

This module serves both the CUDA path (tests, bench) and the CPU oracle.  It
holds none of the block's arithmetic: it only draws seeded random numbers and
lays tokens out the way the pipeline does before the blocks run.

Distributions (random-init stand-ins for the gated checkpoint):
  weights      N(0, 0.02) rounded to bf16, [out, in], no biases
  norm scales  1 + N(0, 0.1), float32 [128]
  activations  N(0, 1) rounded to bf16, held as float32 (the residual stream)
  modulation   N(0, 0.1) float32, one [3 * 3072] vector per stream

Token layouts follow the pipeline's packing: one token per 16x16-pixel patch
(a 1024x1024 image is a 64x64 grid), text first, then the noisy image, then
the references, and the 4-axis ids of the "Positions in four dimensions" table
of "Welcome FLUX.3 Image Klein in Diffusers": text i -> (0,0,0,i); image
(row, col) -> (0, row/2, col/2, 0); reference k -> (0, row/2, col/2, -(k+1)).
"""

from dataclasses import dataclass, field
import zlib

import numpy as np
import torch

STREAM_IMAGE = 0
STREAM_IMAGE_COND = 1
STREAM_TXT = 2
STREAM_OF = {"image": STREAM_IMAGE, "image_cond": STREAM_IMAGE_COND, "txt": STREAM_TXT}

HIDDEN = 3072
MLP_HIDDEN = 9216
HEAD_DIM = 128
HEADS = 24


@dataclass
class Layout:
    """segments: list of (start, length, stream); pos: float32 [T, 4]."""
    segments: list
    pos: np.ndarray
    stream_id: np.ndarray = field(repr=False)

    @property
    def T(self):
        return int(self.pos.shape[0])


def build_layout(spec, l_offset=0.0):
    """spec: list of ('txt', n) | ('image', (rows, cols)) | ('image_cond', (rows, cols)).
    References are numbered k = 0, 1, ... in the order they appear; ``l_offset``
    is added to every reference's l id (0 keeps the table's -(k+1))."""
    segments, pos = [], []
    start, k = 0, 0
    for kind, size in spec:
        if kind == "txt":
            n = int(size)
            p = np.zeros((n, 4), np.float32)
            p[:, 3] = np.arange(n, dtype=np.float32)
        else:
            rows, cols = size
            r, c = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
            n = rows * cols
            p = np.zeros((n, 4), np.float32)
            p[:, 1] = r.reshape(-1) * 0.5
            p[:, 2] = c.reshape(-1) * 0.5
            if kind == "image_cond":
                p[:, 3] = -(k + 1.0) + l_offset
                k += 1
        if n == 0:
            continue
        segments.append((start, n, STREAM_OF[kind]))
        pos.append(p)
        start += n
    pos = np.concatenate(pos, 0) if pos else np.zeros((0, 4), np.float32)
    sid = np.zeros(start, np.uint8)
    for s0, n, st in segments:
        sid[s0:s0 + n] = st
    return Layout(segments, pos, sid)


@dataclass
class Pack:
    """Several samples concatenated: layouts[b] is sample b's own layout;
    segments, pos, stream_id cover the whole pack; sample_start [n + 1];
    sample_id [T]."""
    layouts: list
    segments: list
    pos: np.ndarray
    stream_id: np.ndarray = field(repr=False)
    sample_id: np.ndarray = field(repr=False)
    sample_start: list = field(default_factory=list)

    @property
    def T(self):
        return int(self.pos.shape[0])


def build_pack(specs):
    """One layout per spec, concatenated sample after sample."""
    lays = [build_layout(sp) for sp in specs]
    segments, starts, off = [], [0], 0
    for lay in lays:
        segments += [(s0 + off, n, st) for s0, n, st in lay.segments]
        off += lay.T
        starts.append(off)
    return Pack(lays, segments, np.concatenate([l.pos for l in lays]), np.concatenate([l.stream_id for l in lays]),
                np.concatenate([np.full(l.T, b, np.int64) for b, l in enumerate(lays)]), starts)


# The benchmark and parity workloads (text padded to a multiple of 80 by the
# pipeline is only a sizing rule; these use the stated counts).
WORKLOADS = {
    # one block, 32 txt + 8x8 image (128x128 px)
    "block_t96": dict(spec=[("txt", 32), ("image", (8, 8))], blocks=1, calls=1, wfmt="bf16"),
    # one block at 1024x1024: 512 txt + 64x64 image
    "block_1024sq_t4608": dict(spec=[("txt", 512), ("image", (64, 64))], blocks=1, calls=1, wfmt="bf16"),
    # one block, 1024x1024 target + one 1024x1024 reference
    "block_1024sq_ref1_t8704": dict(spec=[("txt", 512), ("image", (64, 64)), ("image_cond", (64, 64))],
                                    blocks=1, calls=1, wfmt="bf16"),
    # 28-block stack, 1024x1024 + two 512x512 references, 16 calls
    "stack28_1024sq_2ref512_t6656": dict(spec=[("txt", 512), ("image", (64, 64))] + [("image_cond", (32, 32))] * 2,
                                         blocks=28, calls=16, wfmt="bf16"),
    # 28-block stack, 1024x1024 target + one 1024x1024 reference (the one-block layout above)
    "stack28_1024sq_ref1_t8704": dict(spec=[("txt", 512), ("image", (64, 64)), ("image_cond", (64, 64))],
                                      blocks=28, calls=1, wfmt="bf16"),
    # the per-mode blocks (5 per mode, each mode attending only to itself): a small case
    # and the 1024x1024 + one 1024x1024 reference layout
    "modes5_t112": dict(spec=[("txt", 32), ("image", (8, 8)), ("image_cond", (4, 4))],
                        blocks=5, calls=1, wfmt="bf16", stage="modes"),
    "modes5_1024sq_ref1_t8704": dict(spec=[("txt", 512), ("image", (64, 64)), ("image_cond", (64, 64))],
                                     blocks=5, calls=1, wfmt="bf16", stage="modes"),
    # the 16-step flow-map sampler at 1024x1024 text-to-image: each step one transformer call
    # (conditioning, embedders, 5 per-mode blocks, 28 joint blocks, output layer) and the Euler update
    "sample16_1024sq_t4608": dict(spec=[("txt", 512), ("image", (64, 64))], blocks=28, calls=16, wfmt="bf16",
                                  stage="model", mode_blocks=5),
    # the base model's 50-step sampler with guidance on the two-sample pack
    # [empty prompt (80 padded text tokens) | prompt (160)], both with the 1024x1024 image
    "cfg50_1024sq_pack2": dict(specs=[[("txt", 80), ("image", (64, 64))], [("txt", 160), ("image", (64, 64))]],
                               blocks=28, calls=50, wfmt="bf16", stage="cfg", mode_blocks=5),
    # 28-block stack, row-wise FP8 weights, 1024x1024 + one 1024x1024 reference
    "stack28_fp8r_1024sq_ref1_t8704": dict(spec=[("txt", 512), ("image", (64, 64)), ("image_cond", (64, 64))],
                                           blocks=28, calls=1, wfmt="fp8r"),
    # 28-block stack, NVFP4 weights, 1024x1024 + ten 512x512 references
    "stack28_nvfp4_1024sq_10ref512_t14848": dict(
        spec=[("txt", 512), ("image", (64, 64))] + [("image_cond", (32, 32))] * 10,
        blocks=28, calls=1, wfmt="nvfp4"),
    # the 28-block stack at the small block's 96 tokens, bf16 and NVFP4 weights:
    # the weight stream bounds it (245 MB of bf16 weights per block, 69 MB NVFP4)
    "stack28_t96": dict(spec=[("txt", 32), ("image", (8, 8))], blocks=28, calls=1, wfmt="bf16"),
    "stack28_nvfp4_t96": dict(spec=[("txt", 32), ("image", (8, 8))], blocks=28, calls=1, wfmt="nvfp4"),
    "stack28_fp8r_t96": dict(spec=[("txt", 32), ("image", (8, 8))], blocks=28, calls=1, wfmt="fp8r"),
    # two NVFP4 blocks at 96 tokens: a small case of the above for kernel captures
    "stack2_nvfp4_t96": dict(spec=[("txt", 32), ("image", (8, 8))], blocks=2, calls=1, wfmt="nvfp4"),
}


def _seed(*parts):
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def block_weights(seed, block, device="cpu", hidden=HIDDEN, mlp_hidden=MLP_HIDDEN, head_dim=HEAD_DIM,
                  std=0.02):
    """Random-init weights of one block: bf16 [out, in] matrices and float32
    [head_dim] norm scales.  Values depend on (seed, block, tensor) and on the
    device the generator runs on."""
    shapes = {"q_proj": (hidden, hidden), "k_proj": (hidden, hidden), "v_proj": (hidden, hidden),
              "attn_out": (hidden, hidden), "mlp_in": (2 * mlp_hidden, hidden),
              "mlp_out": (hidden, mlp_hidden)}
    w = {}
    for name, shape in shapes.items():
        g = _gen(device, _seed(seed, block, name))
        w[name] = (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    for name in ("query_norm", "key_norm"):
        g = _gen(device, _seed(seed, block, name))
        w[name] = 1.0 + 0.1 * torch.randn((head_dim,), generator=g, device=device, dtype=torch.float32)
    return w


def activations(seed, T, device="cpu", hidden=HIDDEN, std=1.0):
    """Residual-stream input: N(0, std) rounded to bf16, returned as float32."""
    g = _gen(device, _seed(seed, "x", T))
    return (torch.randn((T, hidden), generator=g, device=device) * std).to(torch.bfloat16).float()


def bf16_matrix(seed, rows, cols, device="cpu", std=1.0, tag="m"):
    """A bf16 [rows, cols] N(0, std) tensor (inputs of single-step tests)."""
    g = _gen(device, _seed(seed, tag, rows, cols))
    return (torch.randn((rows, cols), generator=g, device=device) * std).to(torch.bfloat16)


def modulation(seed, call=0, device="cpu", hidden=HIDDEN, std=0.1):
    """Per-stream modulation vectors [3, 3*hidden] float32 (rows: image,
    image_cond, txt; columns: shift | scale | gate)."""
    g = _gen(device, _seed(seed, "mod", call))
    return torch.randn((3, 3 * hidden), generator=g, device=device) * std


COND_SHAPES = {"time_in_in": (3072, 256), "time_in_out": (3072, 3072), "ref_time_in_in": (3072, 256),
               "ref_time_in_out": (3072, 3072), "emb_in_image": (3072, 128), "emb_in_image_cond": (3072, 128),
               "txt_in": (3072, 20480), "final_adaln": (6144, 3072), "final_linear": (128, 3072)}


def cond_weights(seed, device="cpu", std=0.02, flow=True):
    """The non-block weights (time_in, ref_time_in, the six stream modulation
    linears, the embedders, the image output layer): N(0, std) rounded to
    bf16, shapes of the checkpoint's tensor list.  Without ``flow`` the
    ref_time_in weights are None."""
    w = {}
    for k, shape in COND_SHAPES.items():
        if k.startswith("ref_time_in") and not flow:
            w[k] = None
            continue
        g = _gen(device, _seed(seed, "cond", k))
        w[k] = (torch.randn(shape, generator=g, device=device) * std).to(torch.bfloat16)
    for grp in ("early_mod", "single_mod"):
        w[grp] = []
        for s in range(3):
            g = _gen(device, _seed(seed, "cond", grp, s))
            w[grp].append((torch.randn((9216, 3072), generator=g, device=device) * std).to(torch.bfloat16))
    return w


def stream_inputs(seed, lay, device="cpu"):
    """Per stream the embedder inputs of its tokens in sequence order, bf16
    N(0, 1): image and image_cond 128 latent channels, txt 20480 features
    (None for a stream without tokens)."""
    out = []
    for s, ch in ((STREAM_IMAGE, 128), (STREAM_IMAGE_COND, 128), (STREAM_TXT, 20480)):
        n = int((lay.stream_id == s).sum())
        if n == 0:
            out.append(None)
            continue
        g = _gen(device, _seed(seed, "inputs", s))
        out.append(torch.randn((n, ch), generator=g, device=device).to(torch.bfloat16))
    return out


def to_f64(t):
    """Exact float64 NumPy copy of a (bf16 or float32) torch tensor."""
    return t.detach().to("cpu", torch.float64).numpy()
