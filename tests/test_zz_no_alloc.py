"""flux3_block_forward_noalloc: the block forward for callers that cannot
allocate device memory (plug-in hosts whose memory belongs to another
allocator, runtimes that reserve everything up front, real-time loops).  Its
scratch is a fixed array inside the library, so its output must match the
ordinary entry point (caller-provided workspace) on the same inputs, call
after call.  This file is collected last on purpose."""


import pytest
import torch

import diffusion_transformer_block_fwd_b300 as F3
import synth
from _f3 import DEV, layout_tensors

pytestmark = pytest.mark.gpu


def test_noalloc_matches_block_forward_on_two_calls_in_a_row():
    """The largest call first (T = 512 fills the array), then a smaller ragged
    one (T = 171, not a multiple of the 128-row tiles), so stale rows of the
    first call sit past the second call's T in every scratch buffer.  Both
    entry points run the same deterministic kernels on the same inputs, so the
    outputs must be equal bit for bit."""
    w = synth.block_weights(555, 0, device=DEV)
    blocks = F3.Flux3Blocks([w], max_tokens=F3.FLUX3_NOALLOC_MAX_TOKENS)
    sp = torch.cuda.current_stream().cuda_stream
    specs = [[("txt", 160), ("image", (16, 20)), ("image_cond", (4, 8))],        # T = 512, the maximum
             [("txt", 37), ("image", (9, 11)), ("image_cond", (5, 7))]]          # T = 171
    for call, spec in enumerate(specs):
        lay = synth.build_layout(spec)
        pos, _ = layout_tensors(lay)
        x = synth.activations(600 + call, lay.T, device=DEV)
        mods = synth.modulation(600 + call, device=DEV)
        ref = x.clone()
        blocks.forward(ref, lay.segments, pos, mods)                           # workspace entry point
        got = x.clone()
        F3.flux3_block_forward_noalloc(blocks.handle, 0, got.data_ptr(), lay.T, lay.segments, pos.data_ptr(),
                                       mods.data_ptr(), sp)                    # raises on a status other than ok
        assert F3.flux3_check_error(sp) == F3.FLUX3_OK
        assert not torch.equal(got, x), f"call {call}: the block changed nothing"
        assert torch.equal(got, ref), f"call {call}: differs from flux3_block_forward"


def test_noalloc_rejects_more_tokens_than_its_scratch_holds():
    w = synth.block_weights(556, 0, device=DEV)
    blocks = F3.Flux3Blocks([w], max_tokens=4096)
    T = F3.FLUX3_NOALLOC_MAX_TOKENS + 1
    x = torch.zeros((T, 3072), device=DEV)
    pos = torch.zeros((T, 4), device=DEV)
    mods = torch.zeros((3, 9216), device=DEV)
    segs = F3.segments_array([(0, T, 0)])
    st = F3.lib().flux3_block_forward_noalloc(blocks.handle, 0, x.data_ptr(), T, segs, 1, pos.data_ptr(),
                                              mods.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == F3.FLUX3_ERR_WORKSPACE
