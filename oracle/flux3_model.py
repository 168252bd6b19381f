"""fp64 NumPy oracle of the parts around the block stacks: timestep
conditioning, per-stream modulation vectors, input embedders, the image output
layer, the sigma schedule and the sampler step.  Together with
``flux3_oracle.mode_blocks_forward`` and ``flux3_oracle.stack_forward`` they
make one transformer call.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
* "FLUX.3 Image Klein support" (stable-diffusion.cpp issue #2142), comment
  "Structure (from dit.py)": the time conditioning is a 256-wide sinusoidal
  embedding (cosines and sines of 1000 t times a frequency ladder with period
  scale 10000) fed to an MLPEmbedder (Linear, SiLU, Linear); the image mode is
  conditioned on the current t and the other two modes on 0; the flow-map
  checkpoint adds the ref_time_in embedding of t_next to the vector of every
  mode; only image tokens reach the output, a LayerNorm modulated by a shift
  and scale from adaLN_modulation (SiLU, then a Linear to 2 x 3072) followed
  by a linear to 128 channels.  Comment "Sampling (sampling.py,
  pipeline.py)": the sigma schedule alpha t / (1 + (alpha - 1) t) over t
  evenly spaced from 1 to 0 in `steps` intervals, alpha 6.93; the flow map
  takes (sigma_k, sigma_{k+1}) and the latents move by
  (sigma_{k+1} - sigma_k) times the velocity.
  Tensor list: emb_in.{image,image_cond} [3072,128], txt_in [3072,20480],
  time_in / ref_time_in in_layer [3072,256] and out_layer [3072,3072], the
  modulation linears [9216,3072], final_layer adaLN [6144,3072] and linear
  [128,3072].
* "Welcome FLUX.3 Image Klein in Diffusers", "Every token gets its own
  timestep" (text and reference tokens at timestep 0; the flow map's second
  timestep embedding added to every token's modulation), "The denoising loop"
  (shift 6.93; 44 of the 50 steps above sigma = 0.5; sigma about 0.97 at step
  10), "Two stages" (only the image tokens reach the output layers).

Readings (the pages are silent): the frequency ladder freqs_i =
max_period^(-i/128), i = 0..127; the modulation vectors are Linear(SiLU(vec))
like the output layer's adaLN (the pages name only the linear); the output
LayerNorm is the blocks' one (no learned parameters, epsilon 1e-6); adaLN chunk order shift,
scale; the embedders, like every matrix of the checkpoint, have no bias.
"""

import numpy as np

from .flux3_oracle import (EPS_LN, N_STREAMS, STREAM_IMAGE, STREAM_IMAGE_COND, STREAM_TXT, layer_norm,
                           mode_blocks_forward, silu, stack_forward)

TIME_DIM = 256
MAX_PERIOD = 10000.0
TIME_FACTOR = 1000.0
LATENT_CH = 128
TXT_FEAT = 20480
SHIFT = 6.93

__all__ = ["TIME_DIM", "MAX_PERIOD", "TIME_FACTOR", "LATENT_CH", "TXT_FEAT", "SHIFT",
           "timestep_embedding", "mlp_embedder", "stream_vectors", "modulation_vectors", "embed_tokens",
           "final_layer", "transformer_forward", "sigma_schedule", "euler_step", "stack_forward_batch",
           "cfg_velocity", "cfg_euler_step", "transformer_forward_batch"]


def timestep_embedding(t, dim=TIME_DIM, max_period=MAX_PERIOD, time_factor=TIME_FACTOR):
    """[cos(a), sin(a)] with a_i = time_factor * t * max_period^(-i/half),
    i = 0..half-1 (the cosines first)."""
    half = dim // 2
    freqs = np.exp(-np.log(max_period) * np.arange(half, dtype=np.float64) / half)
    a = time_factor * float(t) * freqs
    return np.concatenate([np.cos(a), np.sin(a)])


def mlp_embedder(x, w_in, w_out):
    """MLPEmbedder: Linear, SiLU, Linear (no biases)."""
    x = np.asarray(x, np.float64)
    return silu(x @ np.asarray(w_in, np.float64).T) @ np.asarray(w_out, np.float64).T


def stream_vectors(t, t_next, cond):
    """The conditioning vector of each stream [3, D]: the image stream's from
    timestep t, image_cond's and txt's from timestep 0; with ref_time_in
    (flow map) every stream adds the embedding of t_next."""
    vec = np.empty((N_STREAMS, np.asarray(cond["time_in_out"]).shape[0]))
    v_t = mlp_embedder(timestep_embedding(t), cond["time_in_in"], cond["time_in_out"])
    v_0 = mlp_embedder(timestep_embedding(0.0), cond["time_in_in"], cond["time_in_out"])
    vec[STREAM_IMAGE] = v_t
    vec[STREAM_IMAGE_COND] = v_0
    vec[STREAM_TXT] = v_0
    if cond.get("ref_time_in_in") is not None:
        vec += mlp_embedder(timestep_embedding(t_next), cond["ref_time_in_in"], cond["ref_time_in_out"])
    return vec


def modulation_vectors(vec, lins):
    """Per stream s: lins[s](SiLU(vec[s])) -> [3, 3D] (shift | scale | gate)."""
    vec = np.asarray(vec, np.float64)
    return np.stack([silu(vec[s]) @ np.asarray(lins[s], np.float64).T for s in range(N_STREAMS)])


def embed_tokens(inputs, stream_id, cond):
    """x [T, D]: each token's input row through its stream's embedder
    (emb_in.image, emb_in.image_cond: 128 latent channels; txt_in: 20480 text
    features).  inputs[s] holds stream s's rows in sequence order."""
    stream_id = np.asarray(stream_id)
    W = {STREAM_IMAGE: cond["emb_in_image"], STREAM_IMAGE_COND: cond["emb_in_image_cond"],
         STREAM_TXT: cond["txt_in"]}
    D = np.asarray(W[STREAM_IMAGE]).shape[0]
    x = np.zeros((len(stream_id), D))
    for s in range(N_STREAMS):
        idx = np.nonzero(stream_id == s)[0]
        if idx.size:
            x[idx] = np.asarray(inputs[s], np.float64) @ np.asarray(W[s], np.float64).T
    return x


def final_layer(x_img, vec_img, w_adaln, w_linear, eps=EPS_LN):
    """Image tokens only: (shift, scale) = chunk(adaLN(SiLU(vec)), 2);
    h = (1 + scale) * LayerNorm(x) + shift; velocity = h @ linear^T."""
    mod = silu(np.asarray(vec_img, np.float64)) @ np.asarray(w_adaln, np.float64).T
    D = mod.shape[-1] // 2
    shift, scale = mod[:D], mod[D:]
    h = (1.0 + scale) * layer_norm(x_img, eps) + shift
    return h @ np.asarray(w_linear, np.float64).T


def transformer_forward(inputs, stream_id, pos, t, t_next, cond, mode_blocks, joint_blocks):
    """One call: embed, the per-mode blocks (early modulations), the joint
    blocks (single-stream modulations), the output layer on the image tokens
    (in sequence order).  Returns the velocity [T_image, 128]."""
    stream_id = np.asarray(stream_id)
    vec = stream_vectors(t, t_next, cond)
    early = modulation_vectors(vec, cond["early_mod"])
    single = modulation_vectors(vec, cond["single_mod"])
    x = embed_tokens(inputs, stream_id, cond)
    x = mode_blocks_forward(x, mode_blocks, early, stream_id, pos)
    x = stack_forward(x, joint_blocks, single, stream_id, pos)
    img = np.nonzero(stream_id == STREAM_IMAGE)[0]
    return final_layer(x[img], vec[STREAM_IMAGE], cond["final_adaln"], cond["final_linear"])


def sigma_schedule(steps, alpha=SHIFT):
    """sigma_k for t_k = 1 - k/steps, k = 0..steps."""
    t = np.linspace(1.0, 0.0, steps + 1)
    return alpha * t / (1.0 + (alpha - 1.0) * t)


def euler_step(x, v, sigma, sigma_next):
    return np.asarray(x, np.float64) + (sigma_next - sigma) * np.asarray(v, np.float64)


# --------------------------------------------------------------------------
# Several samples in one call: the base model guides its sampler with a pack
# of two samples, the empty prompt's and the prompt's (comment "Sampling
# (sampling.py, pipeline.py)"); a token attends only within its own sample
# (comment "Structure (from dit.py)").  The guidance combination is a reading: the pages
# give the pack and the scale (3.5), not the formula; this is the usual
# classifier-free guidance form.
# --------------------------------------------------------------------------
def stack_forward_batch(x, blocks, mods, sample_id, stream_id, pos):
    """Joint blocks over concatenated samples: each sample's rows run through
    the blocks as a sequence of their own, a token's modulation row being
    mods[3 * sample + stream]."""
    x = np.array(x, dtype=np.float64)
    sample_id = np.asarray(sample_id)
    stream_id = np.asarray(stream_id)
    pos = np.asarray(pos, np.float64)
    mods = np.asarray(mods, np.float64)
    blocks = list(blocks)
    for b in np.unique(sample_id):
        idx = np.nonzero(sample_id == b)[0]
        x[idx] = stack_forward(x[idx], blocks, mods[3 * b:3 * b + 3], stream_id[idx], pos[idx])
    return x


def cfg_velocity(v_uncond, v_cond, guidance):
    v_uncond = np.asarray(v_uncond, np.float64)
    return v_uncond + guidance * (np.asarray(v_cond, np.float64) - v_uncond)


def cfg_euler_step(x, v_uncond, v_cond, guidance, sigma, sigma_next):
    return euler_step(x, cfg_velocity(v_uncond, v_cond, guidance), sigma, sigma_next)


def transformer_forward_batch(samples, t, t_next, cond, mode_blocks, joint_blocks):
    """samples: per sample (inputs, stream_id, pos); t, t_next per sample.
    Each sample is one transformer call of its own; the velocities of the
    samples' image tokens are returned one sample after the other."""
    return np.concatenate([transformer_forward(ins, sid, pos, t[b], t_next[b], cond, mode_blocks, joint_blocks)
                           for b, (ins, sid, pos) in enumerate(samples)])
