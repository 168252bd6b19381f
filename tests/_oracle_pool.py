"""Oracle work run in worker processes (started with the spawn method) for
the full-size parity tests: seeded block weights quantised by the oracle.
Imports only NumPy, the seeded generators and the oracle."""

import synth
from oracle import nvfp4 as Q

MATS = ("q_proj", "k_proj", "v_proj", "attn_out", "mlp_in", "mlp_out")


def quantize_block(args):
    """(seed, block) -> {matrix: (codes, scales, g)} plus the two norm scales
    as float64, for the block's seeded bf16 weights."""
    seed, block = args
    w = synth.block_weights(seed, block)
    out = {k: Q.quantize(synth.to_f64(w[k])) for k in MATS}
    out.update({k: synth.to_f64(w[k]) for k in ("query_norm", "key_norm")})
    return out
