"""Host-side pieces of bench.py that need no GPU: the reference arm's JSON
line (the CPU oracle timed on whole blocks), the CPU baseline of our line, and
the rule that keys a captured DRAM traffic figure to a kernel's device code."""

import importlib.util
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _reference_line(workload, steps=2, warmup=3):
    env = dict(os.environ, RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          workload, "--steps", str(steps), "--warmup", str(warmup)],
                         capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["block_t96", "modes5_t112"])
def test_reference_line_keeps_the_contract_and_the_workloads_unit(workload):
    """The reference line states a measured time: each timed step is one whole
    block over the workload's layout.  A single-block workload's step is the
    call our line repeats, so the units agree; for a multi-block workload the
    line is per block and the call-scaled figure sits under its own key, in
    the unit of our line."""
    b = _bench()
    tokens, flops, unit = b.workload_call(workload)
    d = _reference_line(workload)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["config"]["workload"] == workload and d["config"]["T"] == tokens
    assert d["value"] > 0 and d["higher_is_better"] is True
    # value = tokens of one block / measured seconds of one block
    assert d["value"] == pytest.approx(tokens / (d["ms_per_step"] * 1e-3), rel=1e-9)
    # the timed region holds the steps it reports
    assert d["wall_s_timed_region"] >= d["steps"] * d["ms_per_step"] * 1e-3 * 0.999
    single = flops == b.block_flops(tokens)
    assert d["unit"] == (unit if single else b.UNIT_ONE_BLOCK)
    assert ("call_extrapolation" in d) != single
    if not single:
        ce = d["call_extrapolation"]
        assert ce["unit"] == unit
        assert ce["value"] == pytest.approx(tokens / (ce["ms_per_call"] * 1e-3), rel=1e-9)
        assert ce["ms_per_call"] == pytest.approx(d["ms_per_step"] * flops / b.block_flops(tokens), rel=1e-9)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_baseline_is_measured_whole_blocks():
    b = _bench()
    cb = b.oracle_baseline([("txt", 8), ("image", (4, 4))], 0.0)
    assert cb["kind"] == "oracle" and cb["unit"] == b.UNIT and cb["cores"] >= 1
    assert cb["value"] == pytest.approx(24 / (cb["ms_per_block"] * 1e-3), rel=1e-9)
    assert "whole block" in cb["sample"] and "1 measured rep" in cb["sample"]
    ex = cb["sampled_extrapolation"]
    assert ex["unit"] == b.UNIT and "scaled" in ex["sample"]


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "block_t96", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert out.returncode == 0 and not out.stdout.strip()


def test_workload_calls_scale_with_their_blocks():
    b = _bench()
    T, f1, u1 = b.workload_call("block_1024sq_ref1_t8704")
    T28, f28, u28 = b.workload_call("stack28_1024sq_ref1_t8704")
    assert T == T28 == 8704 and f28 == 28 * f1 and u1 == b.UNIT and u28 == b.UNIT_STACK
    # the block formula: 245,366,784 T + 12,288 T^2
    assert f1 == 245_366_784 * T + 12_288 * T * T
    # per-mode blocks: the formula at each mode's own count (512 txt, 4096 image, 4096 reference)
    _, fm, um = b.workload_call("modes5_1024sq_ref1_t8704")
    assert fm == 5 * (b.block_flops(512) + 2 * b.block_flops(4096)) and um == b.UNIT_MODES
    # the guided pack: joint attention within each sample, so less than one joint sequence of both
    Tp, fc, uc = b.workload_call("cfg50_1024sq_pack2")
    assert Tp == 80 + 4096 + 160 + 4096 and uc == b.UNIT_CFG
    assert fc < b.model_call_flops([8192, 0, 240], 5, 28)


def test_traffic_key_covers_device_code_only():
    b = _bench()
    dev = b"__global__ void k() {}\n"
    host = b"cudaError_t launch() { return cudaSuccess; }\n"
    assert b.device_part(dev + b.HOST_MARKER + host) == dev
    assert b.device_part(dev + b.HOST_MARKER + host + b"// edited\n") == dev
    assert b.device_part(dev + host) == dev + host          # no marker: the whole file
    # comments do not enter the key; code does; literals holding // or /* stay code
    code = b'__global__ void k(int *p) {  // store\n  /* one */ *p = 1;\n  const char *s = "// x";\n}\n'
    recommented = b'__global__ void k(int *p) {\n  // the store\n  *p = 1;  /* two */\n  const char *s = "// x";\n}\n'
    edited = code.replace(b"*p = 1", b"*p = 2")
    assert b.strip_comments(code) == b.strip_comments(recommented)
    assert b.strip_comments(code) != b.strip_comments(edited)
    assert b'"// x"' in b.strip_comments(code)
    # every kernel source a traffic figure is keyed to has the marker once
    for tr in b.TRAFFIC.values():
        with open(os.path.join(ROOT, tr["src"]), "rb") as f:
            assert f.read().count(b.HOST_MARKER) == 1, tr["src"]


def test_split_plan_mirrors():
    """bench.py counts each launch of the timed region, so it mirrors the
    library's split plans on 148 SMs: the out-projection's K ranges (one-CTA
    128-row tiles up to 128 tokens, CTA-pair 256-row tiles above) and
    attention's key ranges of a partial last wave; a split adds one merge
    launch.  The values are those the step tests name for each size."""
    b = _bench()
    out = {1: 12, 96: 12, 128: 12, 129: 6, 171: 6, 512: 3, 4608: 1, 6656: 4, 14848: 2}
    for T, S in out.items():
        assert b.out_proj_splits(T, 148) == S, (T, b.out_proj_splits(T, 148), S)
    attn = {2048: 3, 4256: 1, 4608: 1, 6656: 4, 8704: 1, 14848: 2, 16384: 2}
    for T, S in attn.items():
        assert b.attn_splits(T, 148) == S, (T, b.attn_splits(T, 148), S)
    assert b.merges(96, 148) == 1 and b.merges(4608, 148) == 0 and b.merges(6656, 148) == 2
