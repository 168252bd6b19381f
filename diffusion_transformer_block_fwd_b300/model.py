"""Flux3Blocks: a handle plus the torch-allocated device buffers it needs
(packed weights, workspace).  Argument marshalling only; the forward pass is
flux3_stack_forward / flux3_block_forward / flux3_mode_blocks_forward of the C
library."""

import torch

from . import (FLUX3_W_BF16, FLUX3_W_FP8R, FLUX3_W_NVFP4, NVFP4_MATRICES, flux3_block_forward, flux3_block_init,
               flux3_block_init_fp8r, flux3_block_init_nvfp4, flux3_default_config, flux3_destroy,
               flux3_mode_blocks_forward, flux3_packed_weight_bytes, flux3_quantize_fp8r, flux3_quantize_nvfp4,
               flux3_stack_forward, flux3_workspace_bytes, flux3_cond_packed_bytes, flux3_cond_init,
               flux3_cond_destroy, flux3_cond_workspace_bytes, flux3_conditioning, flux3_embed_tokens,
               flux3_final_layer_workspace_bytes, flux3_final_layer, flux3_transformer_workspace_bytes,
               flux3_transformer_forward, flux3_sigma_schedule, flux3_euler_step, flux3_stack_forward_batch,
               flux3_transformer_batch_workspace_bytes, flux3_transformer_forward_batch, flux3_cfg_euler_step,
               flux3_latents_to_bf16)

WEIGHT_KEYS = ("q_proj", "k_proj", "v_proj", "attn_out", "mlp_in", "mlp_out", "query_norm", "key_norm")


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def quantize_nvfp4(w, stream=None):
    """NVFP4 of a bf16 [rows, cols] device matrix through flux3_quantize_nvfp4:
    returns (codes uint8 [rows, cols/2], scales uint8 [rows, cols/16],
    global float32 [1]) device tensors."""
    assert w.dtype == torch.bfloat16 and w.is_contiguous() and w.dim() == 2
    rows, cols = w.shape
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=w.device)
    g = torch.empty(1, dtype=torch.float32, device=w.device)
    flux3_quantize_nvfp4(w.data_ptr(), rows, cols, codes.data_ptr(), scales.data_ptr(), g.data_ptr(),
                         _stream_ptr(stream))
    return codes, scales, g


def quantize_fp8r(w, stream=None):
    """Row-wise FP8 of a bf16 [rows, cols] device matrix through
    flux3_quantize_fp8r: returns (codes uint8 [rows, cols], scales float32
    [rows]) device tensors."""
    assert w.dtype == torch.bfloat16 and w.is_contiguous() and w.dim() == 2
    rows, cols = w.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=w.device)
    scales = torch.empty(rows, dtype=torch.float32, device=w.device)
    flux3_quantize_fp8r(w.data_ptr(), rows, cols, codes.data_ptr(), scales.data_ptr(), _stream_ptr(stream))
    return codes, scales


class Flux3Blocks:
    """Joint single_blocks on one CUDA device.

    weights: list (one per block) of dicts of device tensors.  bf16 format:
    bf16 [out, in] matrices q_proj, k_proj, v_proj, attn_out, mlp_in, mlp_out.
    nvfp4 format: each of those is a (codes, scales, global) triple as
    quantize_nvfp4 returns; fp8r format: a (codes, scales) pair as
    quantize_fp8r returns.  All: float32 [128] query_norm, key_norm.  The
    weights are copied into the packed buffer at construction and not
    referenced afterwards."""

    def __init__(self, weights, max_tokens=16384, stream=None, wfmt="bf16"):
        fp4 = wfmt == "nvfp4"
        fp8 = wfmt == "fp8r"
        lowp = fp4 or fp8
        dev = (weights[0]["q_proj"][0] if lowp else weights[0]["q_proj"]).device
        self.device = dev
        self.wfmt = wfmt
        self.cfg = flux3_default_config()
        self.cfg.n_blocks = len(weights)
        self.cfg.max_tokens = int(max_tokens)
        self.cfg.wfmt = FLUX3_W_NVFP4 if fp4 else FLUX3_W_FP8R if fp8 else FLUX3_W_BF16
        nbytes = flux3_packed_weight_bytes(self.cfg)
        if nbytes == 0:
            raise ValueError("unsupported configuration")
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        ptrs = []
        for w in weights:
            for k in WEIGHT_KEYS[6:]:
                assert w[k].dtype == torch.float32 and w[k].is_contiguous(), k
            if fp4:
                for k in NVFP4_MATRICES:
                    c, sc, g = w[k]
                    assert c.dtype == torch.uint8 and sc.dtype == torch.uint8 and g.dtype == torch.float32, k
                    assert c.is_contiguous() and sc.is_contiguous() and c.device == dev, k
                d = {k: tuple(t.data_ptr() for t in w[k]) for k in NVFP4_MATRICES}
                d.update({k: w[k].data_ptr() for k in WEIGHT_KEYS[6:]})
                ptrs.append(d)
            elif fp8:
                for k in NVFP4_MATRICES:
                    c, sc = w[k]
                    assert c.dtype == torch.uint8 and sc.dtype == torch.float32, k
                    assert c.is_contiguous() and sc.is_contiguous() and c.device == dev, k
                d = {k: (w[k][0].data_ptr(), w[k][1].data_ptr()) for k in NVFP4_MATRICES}
                d.update({k: w[k].data_ptr() for k in WEIGHT_KEYS[6:]})
                ptrs.append(d)
            else:
                for k in WEIGHT_KEYS[:6]:
                    assert w[k].dtype == torch.bfloat16 and w[k].is_contiguous() and w[k].device == dev, k
                ptrs.append({k: w[k].data_ptr() for k in WEIGHT_KEYS})
        sp = _stream_ptr(stream)
        init = flux3_block_init_nvfp4 if fp4 else flux3_block_init_fp8r if fp8 else flux3_block_init
        self.handle = init(self.cfg, ptrs, self.packed.data_ptr(), nbytes, sp)
        (stream or torch.cuda.current_stream()).synchronize()   # source weights may be freed after this
        self._ws = torch.empty(0, dtype=torch.uint8, device=dev)

    @property
    def n_blocks(self):
        return self.cfg.n_blocks

    def workspace(self, T):
        need = flux3_workspace_bytes(self.cfg, T)
        if need == 0:
            raise ValueError(f"T={T} out of range (max_tokens={self.cfg.max_tokens})")
        if self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x, segments, pos_ids, mod, first_block=0, n_blocks=None, stream=None):
        """Applies blocks first_block .. first_block + n_blocks - 1 to x in place.
        x: float32 [T, 3072]; pos_ids: float32 [T, 4]; mod: float32 [3, 9216]."""
        T = x.shape[0]
        n = self.n_blocks - first_block if n_blocks is None else n_blocks
        for t, dt in ((x, torch.float32), (pos_ids, torch.float32), (mod, torch.float32)):
            assert t.dtype == dt and t.is_contiguous() and t.device == self.device
        ws = self.workspace(T)
        sp = _stream_ptr(stream)
        if n == 1:
            flux3_block_forward(self.handle, first_block, x.data_ptr(), T, segments, pos_ids.data_ptr(),
                                mod.data_ptr(), ws.data_ptr(), ws.numel(), sp)
        else:
            flux3_stack_forward(self.handle, first_block, n, x.data_ptr(), T, segments, pos_ids.data_ptr(),
                                mod.data_ptr(), ws.data_ptr(), ws.numel(), sp)
        return x

    def forward_batch(self, x, segments, sample_start, pos_ids, mod, first_block=0, n_blocks=None, stream=None):
        """The blocks over several samples concatenated in x (sample b owns
        rows sample_start[b] .. sample_start[b + 1] - 1): LayerNorm and the
        projections over all rows, attention within each sample, in place.
        mod: float32 [3 * n_samples, 9216], row 3 b + stream."""
        T = x.shape[0]
        n = self.n_blocks - first_block if n_blocks is None else n_blocks
        for t in (x, pos_ids, mod):
            assert t.dtype == torch.float32 and t.is_contiguous() and t.device == self.device
        assert sample_start[0] == 0 and sample_start[-1] == T
        ws = self.workspace(T)
        flux3_stack_forward_batch(self.handle, first_block, n, x.data_ptr(), T, segments, list(sample_start),
                                  pos_ids.data_ptr(), mod.data_ptr(), ws.data_ptr(), ws.numel(), _stream_ptr(stream))
        return x

    def close(self):
        if getattr(self, "handle", None):
            flux3_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mode_blocks_forward(mode_blocks, x, segments, pos_ids, early_mod, n_blocks=None, stream=None):
    """The per-mode blocks through flux3_mode_blocks_forward, in place on x.

    mode_blocks: three Flux3Blocks (or None for a mode without tokens), indexed
    by stream id (image, image_cond, txt), each holding that mode's blocks.
    x: float32 [T, 3072]; pos_ids: float32 [T, 4]; early_mod: float32 [3, 9216];
    the segments of one stream must be adjacent."""
    used = [b for b in mode_blocks if b is not None]
    assert used, "no mode blocks"
    dev = used[0].device
    for t in (x, pos_ids, early_mod):
        assert t.dtype == torch.float32 and t.is_contiguous() and t.device == dev
    n = min(b.n_blocks for b in used) if n_blocks is None else n_blocks
    counts = [0, 0, 0]
    for _, ln, st in segments:
        counts[st] += ln
    big = max(range(3), key=lambda m: counts[m])   # the workspace is sized for the largest mode
    ws = mode_blocks[big].workspace(counts[big])
    flux3_mode_blocks_forward([b.handle if b is not None else None for b in mode_blocks], n, x.data_ptr(),
                              x.shape[0], segments, pos_ids.data_ptr(), early_mod.data_ptr(), ws.data_ptr(),
                              ws.numel(), _stream_ptr(stream))
    return x


class Flux3Conditioning:
    """The non-block weights (time_in, ref_time_in, the stream modulation
    linears, the embedders, the output layer) on one device, through
    flux3_cond_init.  weights: dict of bf16 device tensors keyed like the C
    struct (early_mod / single_mod: lists of three; ref_time_in_* may be
    absent)."""

    def __init__(self, weights, stream=None):
        dev = weights["time_in_in"].device
        self.device = dev
        ptrs = {}
        for k, v in weights.items():
            if v is None:
                continue
            ts = v if isinstance(v, (list, tuple)) else [v]
            for t in ts:
                assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.device == dev, k
            ptrs[k] = [t.data_ptr() for t in ts] if isinstance(v, (list, tuple)) else v.data_ptr()
        nbytes = flux3_cond_packed_bytes()
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.handle = flux3_cond_init(ptrs, self.packed.data_ptr(), nbytes, _stream_ptr(stream))
        (stream or torch.cuda.current_stream()).synchronize()
        self._ws = torch.empty(flux3_cond_workspace_bytes(), dtype=torch.uint8, device=dev)

    def modulations(self, t, t_next=0.0, stream=None):
        """(early [3, 9216], single [3, 9216], final [9216]) float32."""
        early = torch.empty((3, 9216), dtype=torch.float32, device=self.device)
        single = torch.empty((3, 9216), dtype=torch.float32, device=self.device)
        fin = torch.empty(9216, dtype=torch.float32, device=self.device)
        flux3_conditioning(self.handle, float(t), float(t_next), early.data_ptr(), single.data_ptr(), fin.data_ptr(),
                           self._ws.data_ptr(), self._ws.numel(), _stream_ptr(stream))
        return early, single, fin

    def embed(self, inputs, segments, T, stream=None):
        """inputs: three bf16 tensors (or None) indexed by stream id; returns x
        float32 [T, 3072]."""
        x = torch.empty((T, 3072), dtype=torch.float32, device=self.device)
        flux3_embed_tokens(self.handle, [t.data_ptr() if t is not None else None for t in inputs], T, segments,
                           x.data_ptr(), _stream_ptr(stream))
        return x

    def final_layer(self, x, segments, final_mod, stream=None):
        T = x.shape[0]
        n_img = sum(n for _, n, st in segments if st == 0)
        v = torch.empty((n_img, 128), dtype=torch.float32, device=self.device)
        ws = torch.empty(flux3_final_layer_workspace_bytes(T), dtype=torch.uint8, device=self.device)
        flux3_final_layer(self.handle, x.data_ptr(), T, segments, final_mod.data_ptr(), v.data_ptr(), ws.data_ptr(),
                          ws.numel(), _stream_ptr(stream))
        return v

    def close(self):
        if getattr(self, "handle", None):
            flux3_cond_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Flux3Transformer:
    """One transformer call through flux3_transformer_forward: conditioning,
    embedders, the per-mode blocks, the joint blocks, the output layer."""

    def __init__(self, cond, mode_blocks, joint, n_mode_blocks=None):
        self.cond, self.mode_blocks, self.joint = cond, list(mode_blocks), joint
        used = [b for b in self.mode_blocks if b is not None]
        self.n_mode_blocks = (min(b.n_blocks for b in used) if used else 0) if n_mode_blocks is None else n_mode_blocks
        self._ws = torch.empty(0, dtype=torch.uint8, device=joint.device)

    def forward(self, inputs, segments, pos_ids, t, t_next=0.0, stream=None, velocity=None):
        T = pos_ids.shape[0]
        need = flux3_transformer_workspace_bytes(self.joint.cfg, T)
        if self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.joint.device)
        n_img = sum(n for _, n, st in segments if st == 0)
        if velocity is None:
            velocity = torch.empty((n_img, 128), dtype=torch.float32, device=self.joint.device)
        flux3_transformer_forward(self.cond.handle, [b.handle if b is not None else None for b in self.mode_blocks],
                                  self.n_mode_blocks, self.joint.handle,
                                  [t_.data_ptr() if t_ is not None else None for t_ in inputs], T, segments,
                                  pos_ids.data_ptr(), float(t), float(t_next), velocity.data_ptr(),
                                  self._ws.data_ptr(), self._ws.numel(), _stream_ptr(stream))
        return velocity

    def forward_batch(self, inputs, segments, sample_start, pos_ids, t, t_next=None, stream=None, velocity=None):
        """Several samples through flux3_transformer_forward_batch.  inputs: per
        sample three bf16 tensors (or None); t, t_next: per-sample timesteps;
        returns the samples' image-token velocities one after the other."""
        T = pos_ids.shape[0]
        n = len(sample_start) - 1
        need = flux3_transformer_batch_workspace_bytes(self.joint.cfg, T, n)
        if self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.joint.device)
        n_img = sum(k for _, k, st in segments if st == 0)
        if velocity is None:
            velocity = torch.empty((n_img, 128), dtype=torch.float32, device=self.joint.device)
        ptrs = [[t_.data_ptr() if t_ is not None else None for t_ in per] for per in inputs]
        tn = t_next if t_next is not None else [0.0] * n
        flux3_transformer_forward_batch(self.cond.handle, [b.handle if b is not None else None for b in self.mode_blocks],
                                        self.n_mode_blocks, self.joint.handle, ptrs, T, segments, sample_start,
                                        pos_ids.data_ptr(), t, tn, velocity.data_ptr(), self._ws.data_ptr(),
                                        self._ws.numel(), _stream_ptr(stream))
        return velocity

    def sample_cfg(self, latents, uncond_inputs, cond_inputs, segments, sample_start, pos_ids, steps=50, alpha=6.93,
                   guidance=3.5, stream=None):
        """The base model's sampler: per step one call on the two-sample pack
        [unconditional, conditional] (both samples carry the current latents as
        their image input) and the guided Euler update of the latents.
        segments / sample_start / pos_ids describe the pack."""
        sig = flux3_sigma_schedule(steps, alpha)
        n_img = latents.shape[0]
        sp = _stream_ptr(stream)
        v = torch.empty((2 * n_img, 128), dtype=torch.float32, device=latents.device)
        img = torch.empty(latents.shape, dtype=torch.bfloat16, device=latents.device)
        u = list(uncond_inputs)
        c = list(cond_inputs)
        u[0] = c[0] = img
        flux3_latents_to_bf16(latents.data_ptr(), latents.numel(), img.data_ptr(), sp)
        for k in range(steps):
            self.forward_batch([u, c], segments, sample_start, pos_ids, [sig[k], sig[k]], stream=stream, velocity=v)
            flux3_cfg_euler_step(latents.data_ptr(), v[:n_img].data_ptr(), v[n_img:].data_ptr(), latents.numel(),
                                 guidance, sig[k], sig[k + 1], img.data_ptr(), sp)
        return latents

    def sample(self, latents, inputs, segments, pos_ids, steps=16, alpha=6.93, flow_map=True, stream=None):
        """The flow-map sampler: for k < steps, v = forward(sigma_k, sigma_{k+1})
        on the current latents (their bf16 rounding, written by the library, is
        the image input), then latents += (sigma_{k+1} - sigma_k) v.  latents:
        float32 [T_image, 128], updated in place."""
        sig = flux3_sigma_schedule(steps, alpha)
        sp = _stream_ptr(stream)
        v = torch.empty_like(latents)
        img = torch.empty(latents.shape, dtype=torch.bfloat16, device=latents.device)
        ins = list(inputs)
        ins[0] = img
        flux3_latents_to_bf16(latents.data_ptr(), latents.numel(), img.data_ptr(), sp)
        for k in range(steps):
            self.forward(ins, segments, pos_ids, sig[k], sig[k + 1] if flow_map else 0.0, stream=stream, velocity=v)
            flux3_euler_step(latents.data_ptr(), v.data_ptr(), latents.numel(), sig[k], sig[k + 1], img.data_ptr(), sp)
        return latents
