"""Parity of each step of the block (through the C ABI) against the CPU
oracle, on seeded inputs that span several tiles and a ragged tail."""

import numpy as np
import pytest
import torch

import diffusion_transformer_block_fwd_b300 as F3
import oracle as O
import synth
from _f3 import (DEV, assert_bf16_elementwise, assert_close, f64, layout_tensors, sample_rows, weights_f64)

pytestmark = pytest.mark.gpu

RAGGED = [("txt", 37), ("image", (9, 11)), ("image_cond", (5, 7))]          # T = 171, three streams


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.fixture(scope="module")
def block1():
    w = synth.block_weights(7, 0, device=DEV)
    blocks = F3.Flux3Blocks([w], max_tokens=16384)
    return w, blocks


def test_stream_ids_bit_exact():
    for spec in (RAGGED, synth.WORKLOADS["stack28_nvfp4_1024sq_10ref512_t14848"]["spec"], [("image", (1, 1))]):
        lay = synth.build_layout(spec)
        out = torch.full((lay.T,), 255, dtype=torch.uint8, device=DEV)
        F3.flux3_stream_ids(lay.segments, lay.T, out.data_ptr(), _stream())
        assert F3.flux3_check_error(_stream()) == 0
        assert np.array_equal(out.cpu().numpy(), lay.stream_id)


def test_rope_tables_match_oracle_angles():
    lay = synth.build_layout(synth.WORKLOADS["stack28_nvfp4_1024sq_10ref512_t14848"]["spec"])
    rng = np.random.default_rng(3)
    extra = np.stack([rng.integers(0, 5, 500), rng.integers(0, 128, 500) * 0.5, rng.integers(0, 128, 500) * 0.5,
                      rng.integers(-4096, 4096, 500)], 1).astype(np.float32)
    pos = np.concatenate([lay.pos, extra])
    T = pos.shape[0]
    pd = torch.from_numpy(pos).to(DEV)
    cs = torch.empty((T, 64), device=DEV)
    sn = torch.empty((T, 64), device=DEV)
    F3.flux3_rope_tables(pd.data_ptr(), T, 1e4, cs.data_ptr(), sn.data_ptr(), _stream())
    ang = O.rope_angles(pos.astype(np.float64))
    assert np.abs(cs.cpu().numpy() - np.cos(ang)).max() < 1e-6
    assert np.abs(sn.cpu().numpy() - np.sin(ang)).max() < 1e-6


def test_prepare_equals_stream_ids_and_rope_tables():
    """The forward calls' one-launch preparation writes exactly what the two
    separate step entry points write."""
    for spec in (RAGGED, synth.WORKLOADS["stack28_nvfp4_1024sq_10ref512_t14848"]["spec"], [("image", (1, 1))]):
        lay = synth.build_layout(spec)
        T = lay.T
        pd = torch.from_numpy(lay.pos).to(DEV)
        sid = torch.full((T,), 255, dtype=torch.uint8, device=DEV)
        cs, sn = torch.empty((T, 64), device=DEV), torch.empty((T, 64), device=DEV)
        F3.flux3_prepare(lay.segments, T, pd.data_ptr(), 1e4, sid.data_ptr(), cs.data_ptr(), sn.data_ptr(), _stream())
        sid2 = torch.full((T,), 255, dtype=torch.uint8, device=DEV)
        cs2, sn2 = torch.empty((T, 64), device=DEV), torch.empty((T, 64), device=DEV)
        F3.flux3_stream_ids(lay.segments, T, sid2.data_ptr(), _stream())
        F3.flux3_rope_tables(pd.data_ptr(), T, 1e4, cs2.data_ptr(), sn2.data_ptr(), _stream())
        assert F3.flux3_check_error(_stream()) == 0
        assert np.array_equal(sid.cpu().numpy(), lay.stream_id)
        assert torch.equal(sid, sid2) and torch.equal(cs, cs2) and torch.equal(sn, sn2)


@pytest.mark.parametrize("T", [1, 37, 171, 4608])
def test_ln_modulate(T):
    lay = synth.build_layout(RAGGED) if T == 171 else None
    x = synth.activations(11, T, device=DEV) * 1.7 + 0.3
    mods = synth.modulation(11, device=DEV)
    sid_np = lay.stream_id if lay else (np.arange(T) % 3).astype(np.uint8)
    sid = torch.from_numpy(sid_np).to(DEV)
    h = torch.empty((T, 3072), dtype=torch.bfloat16, device=DEV)
    F3.flux3_ln_modulate(x.data_ptr(), T, sid.data_ptr(), mods.data_ptr(), 1e-6, h.data_ptr(), _stream())
    assert F3.flux3_check_error(_stream()) == 0
    ref = O.modulate(f64(x), f64(mods), sid_np)
    assert_bf16_elementwise(f64(h), ref, 1e-4, "ln_modulate")


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (100, 512, 192), (128, 256, 3072), (129, 768, 3072),
                                   (300, 1024, 640), (1000, 256, 12288), (4608, 3072, 3072)])
def test_gemm_bf16(M, N, K):
    A = synth.bf16_matrix(1, M, K, device=DEV)
    B = synth.bf16_matrix(2, N, K, device=DEV, std=0.05)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    F3.flux3_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, _stream())
    assert F3.flux3_check_error(_stream()) == 0
    a, b = f64(A), f64(B)
    rows = np.arange(M) if M <= 1000 else sample_rows(M, [(0, M, 0)], 64)
    ref = a[rows] @ b.T
    absprod = np.abs(a[rows]) @ np.abs(b).T
    assert_bf16_elementwise(f64(C)[rows], ref, 2e-5 * absprod, f"gemm {M}x{N}x{K}")


# Layouts of the projection tests by token count: up to 128 tokens the GEMM
# runs one-CTA 128-row tiles, above it CTA-pair 256-row tiles.
STEP_SPECS = {1: [("txt", 1)], 96: synth.WORKLOADS["block_t96"]["spec"], 128: [("txt", 64), ("image", (8, 8))],
              129: [("txt", 65), ("image", (8, 8))], 171: RAGGED,
              512: [("txt", 160), ("image", (16, 20)), ("image_cond", (4, 8))],
              4608: synth.WORKLOADS["block_1024sq_t4608"]["spec"],
              6656: synth.WORKLOADS["stack28_1024sq_2ref512_t6656"]["spec"]}


@pytest.mark.parametrize("T", [1, 96, 128, 129, 171, 4608])
def test_in_projection(block1, T):
    w, blocks = block1
    lay = synth.build_layout(STEP_SPECS[T])
    assert lay.T == T
    pos, _ = layout_tensors(lay)
    hmod = synth.bf16_matrix(5, T, 3072, device=DEV)
    cs = torch.empty((T, 64), device=DEV)
    sn = torch.empty((T, 64), device=DEV)
    F3.flux3_rope_tables(pos.data_ptr(), T, 1e4, cs.data_ptr(), sn.data_ptr(), _stream())
    qkv = torch.full((T, 9216), float("nan"), dtype=torch.bfloat16, device=DEV)
    cat = torch.full((T, 12288), float("nan"), dtype=torch.bfloat16, device=DEV)
    F3.flux3_in_projection(blocks.handle, 0, hmod.data_ptr(), T, cs.data_ptr(), sn.data_ptr(), qkv.data_ptr(),
                           cat.data_ptr(), _stream())
    assert F3.flux3_check_error(_stream()) == 0
    wf = weights_f64(w)
    rows = np.arange(T) if T <= 200 else sample_rows(T, lay.segments)
    h64 = f64(hmod)
    hr = h64[rows]
    pr = lay.pos[rows].astype(np.float64)
    d = 128
    q = O.apply_rope(O.rms_norm((hr @ wf["q_proj"].T).reshape(-1, 24, d), wf["query_norm"]), pr).reshape(-1, 3072)
    k = O.apply_rope(O.rms_norm((hr @ wf["k_proj"].T).reshape(-1, 24, d), wf["key_norm"]), pr).reshape(-1, 3072)
    v = hr @ wf["v_proj"].T
    g = O.swiglu(hr @ wf["mlp_in"].T)
    got = f64(qkv)[rows]
    gcat = f64(cat)[rows]
    for name, gv, rv in (("q^", got[:, :3072], q), ("k^", got[:, 3072:6144], k), ("v", got[:, 6144:], v),
                         ("g", gcat[:, 3072:], g)):
        rms = float(np.sqrt(np.mean(rv * rv)))
        assert_bf16_elementwise(gv, rv, 2e-3 * rms, f"in_projection {name} T={T}")
        assert_close(gv, rv, 1.0, 0.99999, f"in_projection {name} T={T}")     # cosine; the bound above is the max
    assert torch.isnan(cat[:, :3072].float()).all(), "attention columns must be left untouched"


def check_attention(got, ref, ref_abs, what):
    """P and the output are rounded to bf16 (relative error <= 2^-8 each), so
    |err| <= 2^-8 * sum_j p_j |v_j| + 2^-8 |o| (+ a 1e-5 slack for the fp32
    logits and exp2); plus cosine >= 0.9999."""
    bound = 2.0 ** -8 * (ref_abs + np.abs(ref)) * 1.01 + 1e-5 * ref_abs + 1e-6
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside the bf16 bound"
    assert_close(got, ref, 1.0, 0.9999, what)


def _qkv_inputs(T, seed, q_scale=1.0):
    qkv = synth.bf16_matrix(seed, T, 9216, device=DEV)
    if q_scale != 1.0:
        qkv[:, :3072] = (qkv[:, :3072].float() * q_scale).to(torch.bfloat16)
    return qkv


@pytest.mark.parametrize("T,q_scale", [(1, 1.0), (5, 1.0), (64, 1.0), (65, 1.0), (127, 1.0), (128, 1.0),
                                       (129, 1.0), (300, 1.0), (1000, 1.0), (300, 6.0), (1000, 12.0)])
def test_attention(T, q_scale):
    qkv = _qkv_inputs(T, 21 + T, q_scale)
    cat = torch.full((T, 12288), float("nan"), dtype=torch.bfloat16, device=DEV)
    F3.flux3_attention(qkv.data_ptr(), T, cat.data_ptr(), _stream(), *_split_args(True))
    assert F3.flux3_check_error(_stream()) == 0
    a = f64(qkv).reshape(T, 3, 24, 128)
    ref = O.attention(a[:, 0], a[:, 1], a[:, 2]).reshape(T, 3072)
    ref_abs = O.attention(a[:, 0], a[:, 1], np.abs(a[:, 2])).reshape(T, 3072)
    got = f64(cat)[:, :3072]
    check_attention(got, ref, ref_abs, f"attention T={T} qscale={q_scale}")
    assert torch.isnan(cat[:, 3072:].float()).all(), "SwiGLU columns must be left untouched"


_SPLIT_BUF = {}


def _split_args(split):
    """(split_buf, split_bytes) for the attention / out-projection step entry points."""
    if not split:
        return (None, 0)
    if "buf" not in _SPLIT_BUF:
        _SPLIT_BUF["buf"] = torch.empty(F3.FLUX3_SPLIT_BYTES // 4, dtype=torch.float32, device=DEV)
    return (_SPLIT_BUF["buf"].data_ptr(), F3.FLUX3_SPLIT_BYTES)


# 4256 = 160 text + 64x64 image tokens, the pages' text-to-image count per call (a ragged last key tile).
# With the split buffer on 148 SMs: 2048 tokens split their last 44 units in 3 key ranges, 6656 their last 32
# in 4, 14848 and 16384 their last 60 and 56 in 2; 4256, 4608 and 8704 split nothing.  The sampled rows meet
# the trailing units (the last heads) in every query tile they fall in.
@pytest.mark.parametrize("T,split", [(2048, True), (4256, True), (4608, True), (6656, True), (6656, False),
                                     (8704, True), (14848, True), (16384, True), (16384, False)])
def test_attention_full_size_sampled_rows(T, split):
    qkv = _qkv_inputs(T, 31, 3.0)
    cat = torch.empty((T, 12288), dtype=torch.bfloat16, device=DEV)
    F3.flux3_attention(qkv.data_ptr(), T, cat.data_ptr(), _stream(), *_split_args(split))
    assert F3.flux3_check_error(_stream()) == 0
    rows = sample_rows(T, [(0, T, 0)], 40)
    a = f64(qkv).reshape(T, 3, 24, 128)
    ref = O.attention(a[rows, 0], a[:, 1], a[:, 2]).reshape(len(rows), 3072)
    ref_abs = O.attention(a[rows, 0], a[:, 1], np.abs(a[:, 2])).reshape(len(rows), 3072)
    check_attention(f64(cat)[rows, :3072], ref, ref_abs, f"attention T={T} split={split}")


def test_attention_split_against_unsplit():
    """Split and unsplit outputs differ only where units were split (the last
    heads' columns), and there only by rounding: each range rounds its P to
    bf16 relative to its own running max, and the merge rescales the ranges
    in float32.  Each output is within the bf16 bound of the exact value
    (2^-8 (sum_j p_j |v_j| + |o|), test above), so the two are within twice
    that of each other: checked on sampled rows of the split heads with the
    oracle's sum_j p_j |v_j|; and the difference's RMS over every row stays
    within 5e-3 of the output's."""
    T = 6656
    qkv = _qkv_inputs(T, 32, 3.0)
    a = torch.empty((T, 12288), dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    F3.flux3_attention(qkv.data_ptr(), T, a.data_ptr(), _stream())
    F3.flux3_attention(qkv.data_ptr(), T, b.data_ptr(), _stream(), *_split_args(True))
    assert F3.flux3_check_error(_stream()) == 0
    # units 592..623 (head 22 from query-tile pair 20, head 23) are the split ones
    assert torch.equal(a[:, :22 * 128], b[:, :22 * 128])
    assert torch.equal(a[:5120, 22 * 128:23 * 128], b[:5120, 22 * 128:23 * 128])
    fa, fb = f64(a[:, 22 * 128:3072]), f64(b[:, 22 * 128:3072])
    assert not np.array_equal(fa, fb)
    rms = np.sqrt(np.mean(fa * fa))
    assert np.sqrt(np.mean((fa - fb) ** 2)) <= 5e-3 * rms
    rows = sample_rows(T, [(0, T, 0)], 40)
    q = f64(qkv).reshape(T, 3, 24, 128)[:, :, 22:24]
    ref = O.attention(q[rows, 0], q[:, 1], q[:, 2]).reshape(len(rows), 256)
    ref_abs = O.attention(q[rows, 0], q[:, 1], np.abs(q[:, 2])).reshape(len(rows), 256)
    bound = 2 * 2.0 ** -8 * (ref_abs + np.abs(ref)) * 1.01 + 2e-5 * ref_abs + 2e-6
    assert (np.abs(fa[rows] - fb[rows]) <= bound).all()


@pytest.mark.parametrize("T,split", [(1, True), (96, False), (96, True), (128, True), (129, True), (171, False),
                                     (171, True), (512, True), (4608, True), (6656, False), (6656, True)])
def test_out_projection(block1, T, split):
    """With a split buffer, the tiles of the GEMM's last, partial round of
    tiles are split along K: up to 128 tokens the 12 one-CTA tiles in 12 ranges
    each, at 129 and 171 tokens the 12 pair tiles in 6, at 512 the 24 pair
    tiles in 3, at 6656 the 16 trailing pair tiles in 4; none at 4608, whose
    last round is nearly full.  Without the buffer no tile is split.  Both
    against the float64 product."""
    w, blocks = block1
    lay = synth.build_layout(STEP_SPECS[T])
    assert lay.T == T
    _, sid = layout_tensors(lay)
    cat = synth.bf16_matrix(9, T, 12288, device=DEV)
    x = synth.activations(9, T, device=DEV)
    x0 = x.clone()
    mods = synth.modulation(9, device=DEV)
    F3.flux3_out_projection(blocks.handle, 0, cat.data_ptr(), T, sid.data_ptr(), mods.data_ptr(), x.data_ptr(),
                            _stream(), *_split_args(split))
    assert F3.flux3_check_error(_stream()) == 0
    wf = weights_f64(w)
    rows = np.arange(T) if T <= 600 else sample_rows(T, lay.segments)
    if T == 6656:   # every row of the trailing tiles (row blocks 24 and 25)
        rows = np.union1d(rows, np.arange(6144, 6656, 7))
    c = f64(cat)[rows]
    y = c[:, :3072] @ wf["attn_out"].T + c[:, 3072:] @ wf["mlp_out"].T
    gate = f64(mods)[lay.stream_id[rows], 6144:]
    ref_delta = gate * y
    got_delta = f64(x)[rows] - f64(x0)[rows]
    assert_close(got_delta, ref_delta, 1e-3, 0.999999, f"out_projection T={T} split={split}")


@pytest.mark.parametrize("T,row0", [(6656, 6144), (96, 0)])
def test_out_projection_split_matches_unsplit_up_to_summation_order(block1, T, row0):
    """The split changes only the order of the float32 sums of the trailing
    tiles (rows row0 and on): the two results agree to float32 rounding, and
    rows outside the trailing tiles are equal bit for bit."""
    _, blocks = block1
    lay = synth.build_layout(STEP_SPECS[T])
    _, sid = layout_tensors(lay)
    cat = synth.bf16_matrix(10, T, 12288, device=DEV)
    x = synth.activations(10, T, device=DEV)
    mods = synth.modulation(10, device=DEV)
    a, b = x.clone(), x.clone()
    F3.flux3_out_projection(blocks.handle, 0, cat.data_ptr(), T, sid.data_ptr(), mods.data_ptr(), a.data_ptr(),
                            _stream(), *_split_args(False))
    F3.flux3_out_projection(blocks.handle, 0, cat.data_ptr(), T, sid.data_ptr(), mods.data_ptr(), b.data_ptr(),
                            _stream(), *_split_args(True))
    assert F3.flux3_check_error(_stream()) == 0
    assert torch.equal(a[:row0], b[:row0])
    da, db = f64(a[row0:]) - f64(x[row0:]), f64(b[row0:]) - f64(x[row0:])
    assert not np.array_equal(da, db)
    # float32 sums of 12288 products in another grouping: ~1e-5 of RMS per
    # element, its maximum over up to 1.5 M elements a few times that; both
    # bounds are far inside the 1e-3 the oracle comparison above allows
    rms = np.sqrt(np.mean(da * da))
    assert np.abs(da - db).max() <= 5e-4 * rms
    assert np.sqrt(np.mean((da - db) ** 2)) <= 5e-5 * rms
    # and twice the same split call: bit for bit (fixed merge order)
    c = x.clone()
    F3.flux3_out_projection(blocks.handle, 0, cat.data_ptr(), T, sid.data_ptr(), mods.data_ptr(), c.data_ptr(),
                            _stream(), *_split_args(True))
    assert F3.flux3_check_error(_stream()) == 0
    assert torch.equal(b, c)


def test_timeout_path_reports_and_context_survives():
    F3.flux3_selftest_wait_timeout(20000, _stream())
    assert F3.flux3_check_error(_stream()) == F3.FLUX3_ERR_TIMEOUT
    assert F3.flux3_check_error(_stream()) == F3.FLUX3_OK          # the word was cleared
    A = synth.bf16_matrix(1, 128, 64, device=DEV)
    C = torch.empty((128, 256), dtype=torch.bfloat16, device=DEV)
    B = synth.bf16_matrix(2, 256, 64, device=DEV)
    F3.flux3_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), 128, 256, 64, _stream())
    assert F3.flux3_check_error(_stream()) == F3.FLUX3_OK
    np.testing.assert_allclose(f64(C), f64(A) @ f64(B).T, rtol=2 ** -8, atol=1e-3)
