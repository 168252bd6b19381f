"""Benchmark of the joint single_block forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one joint single_block over one batch of synthetic tokens (default
the 1024x1024 workload: 512 text + 64x64 image tokens = 4608): stream ids,
RoPE tables, LayerNorm + modulation, the fused in-projection GEMM (q/k/v with
QK-RMSNorm + RoPE, SwiGLU), attention, and the out-projection GEMM with the
gated residual.  Inputs are resident in HBM when the timed region starts;
L2 is flushed (a 256 MiB write, then a 256 MiB read of another buffer, which
drains the write's dirty lines) between timed steps, outside the per-step
events.  For N > 1 (torchrun) every rank runs an independent replica (the
path needs no exchange): the value is the tokens of all ranks over the
slowest rank's time.

Each timed step is one replay of a CUDA graph of that launch sequence, so
the per-kernel events (event-record nodes in the graph) measure device time
without host launch gaps.  `--workload` selects another configuration: the
other single-block layouts, or a 28-block stack (bf16 or NVFP4 weights), where
a step is one call of the stack per sampler step of the workload (16 for the
two-reference stack, each with fresh modulation vectors).

One JSON line is printed by rank 0.  `--impl reference` times the CPU oracle
on the host cores instead (rank 0 only).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "single_block tokens/s and TFLOP/s at 1024² (4608 tok), % of B300 BF16 peak"
UNIT = "tokens/s"
# the unit of the other workloads' lines: tokens per second of the call a step repeats
UNIT_STACK = "tokens/s (per stack call)"
UNIT_MODES = "tokens/s (per-mode blocks)"
UNIT_MODEL = "tokens/s (transformer calls of the sampler)"
UNIT_CFG = "tokens/s (two-sample guided calls of the sampler)"
UNIT_ONE_BLOCK = "tokens/s (one joint block over the workload's token layout)"

# Algorithmic FLOPs of one block over T tokens: 2 x (MACs of the six
# projections) + QK^T + PV = 245,366,784 T + 12,288 T^2.
def block_flops(T):
    D, F = 3072, 9216
    proj = 2 * T * D * (3 * D + 2 * F) + 2 * T * (D + F) * D
    attn = 4 * T * T * D
    return proj + attn


def kernel_flops(T):
    return {"in_projection": 2 * T * 3072 * 27648, "attention": 4 * T * T * 3072,
            "out_projection": 2 * T * 12288 * 3072}


def out_proj_splits(T, sms):
    """K ranges of the out-projection's trailing tiles at T tokens on `sms`
    SMs (1: no split), the plan the library takes: tiles are 128 x 256 on
    single CTAs for T <= 128, else 256 x 256 on CTA pairs; the last, partial
    round of tiles is split by the largest of 12, 8, 6, 4, 3, 2 that divides
    the 192 k-blocks into ranges of >= 16 and keeps the units within the
    workers and their partial tiles within the 24 MiB split buffer.  A split
    adds one merge launch."""
    tile_m, workers = (128, sms) if T <= 128 else (256, sms // 2)
    tiles = -(-T // tile_m) * 12
    rem = tiles % workers
    if rem == 0 or workers < 2:
        return 1
    for S in (12, 8, 6, 4, 3, 2):
        if 192 % S == 0 and 192 // S >= 16 and rem * S <= workers and \
                rem * S * tile_m * 256 * 4 <= 96 * 256 * 256 * 4:
            return S
    return 1


def attn_splits(T, sms):
    """Key ranges the attention's trailing units take at T tokens on `sms`
    SMs (1: no split), the plan the library takes: the units of the last,
    partial wave of one CTA per SM are split into the most ranges (<= 8, each
    of >= 4 key tiles) that fit in that wave and in the 24 MiB split buffer.
    A split adds one merge launch."""
    units = -(-T // 256) * 24
    rem = units % sms if units >= sms else units
    nt = -(-T // 128)
    if rem == 0:
        return 1
    for S in range(8, 1, -1):
        if rem * S <= sms and nt // S >= 4 and rem * S * 2 * 128 * 132 * 4 <= 96 * 256 * 256 * 4:
            return S
    return 1


def merges(T, sms):
    """Merge launches of one block at T tokens (out-projection, attention)."""
    return (out_proj_splits(T, sms) > 1) + (attn_splits(T, sms) > 1)


def kernel_bytes(T):
    """Algorithmic HBM bytes per launch of the memory-bound kernels."""
    return {"ln_modulate": T * (3072 * 4 + 3072 * 2), "rope_tables": T * (16 + 2 * 64 * 4), "stream_ids": T}


# DRAM traffic per launch from an ncu capture, valid only for the kernel
# source it was taken on: the sha256 of the file's device code (the text
# before its host-launcher marker line, the whole file if it has none; comments
# stripped); null otherwise.
TRAFFIC = {
    # gemm_kernel<EPI_IN_PROJ>, T = 4608: dram__bytes_read.sum 207.53 MB + dram__bytes_write.sum 154.16 MB
    # (ncu --metrics ... --clock-control none, one launch; profiles/gemm_tcgen05_block_1024sq_t4608.md)
    "in_projection": {"src": "diffusion_transformer_block_fwd_b300/csrc/gemm.cuh", "src_sha": "118222b384e5fa29", "T": 4608,
                      "bytes_per_launch": 361_686_016},
}

HOST_MARKER = b"// ---------------------------------------------------------------- host launchers\n"


def device_part(text):
    """The device code of a kernel source: everything before its host-launcher marker."""
    i = text.find(HOST_MARKER)
    return text if i < 0 else text[:i]


def strip_comments(text):
    """C / C++ source bytes without their // and /* */ comments (string and
    character literals kept), runs of blanks collapsed, empty lines dropped: a
    comment or layout edit leaves a kernel's key unchanged, a code edit does
    not."""
    out, i, n = bytearray(), 0, len(text)
    while i < n:
        c = text[i:i + 1]
        if c in (b'"', b"'"):
            j = i + 1
            while j < n and text[j:j + 1] != c:
                j += 2 if text[j:j + 1] == b"\\" else 1
            out += text[i:j + 1]
            i = j + 1
        elif text.startswith(b"//", i):
            j = text.find(b"\n", i)
            i = n if j < 0 else j
        elif text.startswith(b"/*", i):
            j = text.find(b"*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out += c
            i += 1
    lines = [b" ".join(l.split()) for l in bytes(out).split(b"\n")]   # blanks collapsed
    return b"\n".join(l for l in lines if l)


def src_sha(path):
    with open(os.path.join(ROOT, path), "rb") as f:
        return hashlib.sha256(strip_comments(device_part(f.read()))).hexdigest()[:16]


class L2Flush:
    """Evicts the step's data from L2 between timed steps: a 256 MiB write
    (larger than the 126 MB L2), then a 256 MiB read of a second buffer, so
    that the write's dirty lines are written back before the next step starts
    instead of during its first kernels.  Runs outside the step's events."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
        self.r = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.r.sum()


L2_NOTE = "flushed between timed steps (256 MiB write, then a 256 MiB read of another buffer), outside the events"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), d.get("bf16_tflops_sustained"), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


def smi_target(dev_index):
    """The nvidia-smi id of CUDA device `dev_index`: its PCI bus id (nvidia-smi
    numbers GPUs in PCI order and ignores CUDA_VISIBLE_DEVICES), else the
    ordinal."""
    try:
        import torch
        p = torch.cuda.get_device_properties(dev_index)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return str(dev_index)


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs, on the
    GPU the CUDA device maps to."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.target = None
        self.proc = None
        self.path = None
        self.out = None

    def _close_out(self):
        if self.out is not None:
            self.out.close()
            self.out = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            for target in dict.fromkeys((smi_target(self.index), str(self.index))):
                self.out = open(self.path, "w")
                self.proc = subprocess.Popen(["nvidia-smi", "-i", target, f"--query-gpu={self.FIELDS}",
                                              "--format=csv,noheader,nounits", "-lms", "50"],
                                             stdout=self.out, stderr=subprocess.DEVNULL)
                # accepted once a sample line arrives; an id nvidia-smi rejects ends the process
                t_end = time.time() + 2.0
                while time.time() < t_end and self.proc.poll() is None and os.path.getsize(self.path) == 0:
                    time.sleep(0.05)
                if self.proc.poll() is None:
                    self.target = target
                    break
                self.proc = None
                self._close_out()
        except Exception:
            self.proc = None
            self._close_out()

    def stop(self):
        if self.proc is None:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._close_out()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons),
                "gpu": self.target}


# ---------------------------------------------------------------- CPU oracle timing
class OracleBlock:
    """The CPU oracle running one joint block over a workload's token layout
    (seeded inputs, float64).  `run()` times the whole block: every output
    row, keys and values over all T tokens.  `run_sampled()` times the block
    output for `rows_n` query tokens only (keys and values still over all
    tokens), for warm-up and for a labelled FLOP-scaled estimate."""

    def __init__(self, spec, rows_n=128):
        import oracle as O
        import synth
        self.O = O
        self.lay = synth.build_layout(spec)
        T = self.T = self.lay.T
        w = synth.block_weights(1, 0, device="cpu")
        self.wf = {k: synth.to_f64(v) for k, v in w.items()}
        self.x = synth.to_f64(synth.activations(1, T))
        self.mods = synth.to_f64(synth.modulation(1))
        self.pos = self.lay.pos.astype(np.float64)
        self.rows = np.linspace(0, T - 1, rows_n).astype(np.int64)
        D, F = 3072, 9216
        sample_flops = 4 * T * D * D + rows_n * (2 * D * D + 4 * D * F + 2 * (D + F) * D + 4 * T * D)
        self.sample_scale = block_flops(T) / sample_flops
        self.rows_n = rows_n

    def run(self):
        """Seconds of one whole block (measured)."""
        t0 = time.perf_counter()
        self.O.single_block(self.x, self.wf, self.mods, self.lay.stream_id, self.pos)
        return time.perf_counter() - t0

    def run_sampled(self):
        """Seconds of the sampled block (measured, not scaled)."""
        t0 = time.perf_counter()
        self.O.single_block(self.x, self.wf, self.mods, self.lay.stream_id, self.pos, rows=self.rows)
        return time.perf_counter() - t0

    def describe(self, reps):
        return (f"fp64 NumPy oracle: one whole block over the workload's {self.T} tokens (every output row), "
                f"{reps} measured rep(s)")

    def describe_sampled(self, reps):
        return (f"fp64 NumPy oracle: block output for {self.rows_n} of {self.T} query tokens (keys/values over all "
                f"tokens), {reps} rep(s), time scaled to a whole block by algorithmic FLOPs x{self.sample_scale:.2f}")


def pin_blas_threads():
    """Pins the BLAS thread pool to the cores this process may run on and
    returns that count (the core count the oracle's time is quoted for)."""
    cores = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(limits=cores, user_api="blas")
    except Exception:
        pass
    return cores


def host_cores():
    cores = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            cores = max(n)
    except Exception:
        pass
    return cores


def oracle_baseline(spec, seconds):
    """The oracle timed in full on this host: whole blocks until `seconds` have
    passed (at least one); the 128-row FLOP-scaled estimate is reported beside
    it under its own key."""
    pin_blas_threads()
    s = OracleBlock(spec)
    s.run_sampled()                                    # warm-up (BLAS threads, page faults)
    est = s.run_sampled() * s.sample_scale
    times = []
    t_end = time.perf_counter() + seconds
    while not times or time.perf_counter() < t_end:
        times.append(s.run())
    t_block = statistics.mean(times)
    return {"value": s.T / t_block, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "sample": s.describe(len(times)), "ms_per_block": 1e3 * t_block,
            "sampled_extrapolation": {"value": s.T / est, "unit": UNIT, "ms_per_block": 1e3 * est,
                                      "sample": s.describe_sampled(1)}}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores.  A
    timed step is one whole joint block over the workload's token layout,
    measured (no scaling).  For a single-block workload that is the call our
    arm's step repeats, so the line has our line's unit; for the multi-block
    workloads (stacks, samplers, per-mode blocks) the line's unit is one
    block, and the call-scaled figure is reported under its own key.
    Warm-up steps run the sampled block (the same code on 128 query rows) so
    that the whole run ends within a few minutes."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import synth
    cores = pin_blas_threads()
    wl = synth.WORKLOADS[args.workload]
    spec = wl["spec"] if "spec" in wl else wl["specs"][-1]   # a pack: the conditional sample's layout
    tokens, call_flops, unit = workload_call(args.workload)
    s = OracleBlock(spec)
    for _ in range(args.warmup):
        s.run_sampled()
    t0 = time.perf_counter()
    times = [s.run() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    t_step = statistics.mean(times)
    single = call_flops == block_flops(s.T) and tokens == s.T
    line_unit = unit if single else UNIT_ONE_BLOCK
    value = s.T / t_step
    sample = s.describe(args.steps) + f"; warm-up: {args.warmup} sampled block(s) ({s.rows_n} query rows)"
    line = {"metric": METRIC, "value": value, "unit": line_unit, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "T": s.T, "unit_of_work": "one joint block, measured in full"},
            "cpu_baseline": {"value": value, "unit": line_unit, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": line_unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s_timed_region": wall}
    if not single:
        call_s = t_step * call_flops / block_flops(s.T)
        line["call_extrapolation"] = {"value": tokens / call_s, "unit": unit, "ms_per_call": 1e3 * call_s,
                                      "how": f"the measured block scaled to one call of the workload by "
                                             f"algorithmic FLOPs x{call_flops / block_flops(s.T):.2f}"}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def dist_setup():
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    return rank, world, local, dev


def max_over_ranks(v, world, dev):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank, step_ms, world, dev):
    """Whole-job throughput of `world` independent replicas: every rank
    processes `units_per_rank` units per step; the job's step time is the
    slowest rank's.  Returns (units per second, the max step time in ms)."""
    slowest = max_over_ranks(step_ms, world, dev)
    return world * units_per_rank / (slowest * 1e-3), slowest


def timed_graphs(step_fn, n_events, steps, stream):
    """Captures `steps` CUDA graphs of step_fn(events), each with its own
    event-record nodes; returns (graphs, events)."""
    import torch
    graphs, evs = [], []
    for _ in range(steps):
        e = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n_events)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step_fn(e)
        graphs.append(g)
        evs.append(e)
    torch.cuda.synchronize()
    return graphs, evs


def run_ours(args):
    import torch
    import torch.distributed as dist

    import diffusion_transformer_block_fwd_b300 as F3
    import synth

    rank, world, local, dev = dist_setup()
    F3.lib()   # fail loudly if the library is missing
    wl = synth.WORKLOADS[args.workload]
    if wl.get("stage") == "modes":
        return run_modes(args, rank, world, local, dev)
    if wl.get("stage") == "model":
        return run_model(args, rank, world, local, dev)
    if wl.get("stage") == "cfg":
        return run_cfg(args, rank, world, local, dev)
    if wl["blocks"] > 1:
        return run_stack(args, rank, world, local, dev)
    spec = wl["spec"]
    lay = synth.build_layout(spec)
    T = lay.T
    w = synth.block_weights(1, 0, device=dev)
    blocks = F3.Flux3Blocks([w], max_tokens=T)
    x = synth.activations(1, T, device=dev)
    mods = synth.modulation(1, device=dev)
    pos = torch.from_numpy(lay.pos).to(dev)
    sid = torch.empty(T, dtype=torch.uint8, device=dev)
    cs = torch.empty((T, 64), device=dev)
    sn = torch.empty((T, 64), device=dev)
    h = torch.empty((T, 3072), dtype=torch.bfloat16, device=dev)
    qkv = torch.empty((T, 9216), dtype=torch.bfloat16, device=dev)
    cat = torch.empty((T, 12288), dtype=torch.bfloat16, device=dev)
    split = torch.empty(F3.FLUX3_SPLIT_BYTES // 4, dtype=torch.float32, device=dev)   # out-projection K split
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    cfg = blocks.cfg

    names = ["prep", "ln_modulate", "in_projection", "attention", "out_projection"]

    def step_api(evs):
        # the public call, one block: its kernels are launched back to back, each
        # a programmatic dependent of the one before (set-up overlaps the tail)
        evs[0].record(stream)
        blocks.forward(x, lay.segments, pos, mods, stream=stream)
        evs[1].record(stream)

    def step_kernels(evs=None):
        # the same launch sequence through the step entry points, an event
        # around each kernel (the events serialise the kernels)
        if evs is not None:
            evs[0].record(stream)
        F3.flux3_prepare(lay.segments, T, pos.data_ptr(), cfg.rope_theta, sid.data_ptr(), cs.data_ptr(),
                         sn.data_ptr(), sp)
        if evs is not None:
            evs[1].record(stream)
        F3.flux3_ln_modulate(x.data_ptr(), T, sid.data_ptr(), mods.data_ptr(), cfg.eps_ln, h.data_ptr(), sp)
        if evs is not None:
            evs[2].record(stream)
        F3.flux3_in_projection(blocks.handle, 0, h.data_ptr(), T, cs.data_ptr(), sn.data_ptr(), qkv.data_ptr(),
                               cat.data_ptr(), sp)
        if evs is not None:
            evs[3].record(stream)
        F3.flux3_attention(qkv.data_ptr(), T, cat.data_ptr(), sp, split.data_ptr(), F3.FLUX3_SPLIT_BYTES)
        if evs is not None:
            evs[4].record(stream)
        F3.flux3_out_projection(blocks.handle, 0, cat.data_ptr(), T, sid.data_ptr(), mods.data_ptr(), x.data_ptr(),
                                sp, split.data_ptr(), F3.FLUX3_SPLIT_BYTES)
        if evs is not None:
            evs[5].record(stream)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    launches_per_step = 5 + merges(T, sms)
    torch.cuda.synchronize(dev)          # inputs were made on the default stream
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step_kernels()
            blocks.forward(x, lay.segments, pos, mods, stream=stream)
        st = F3.flux3_check_error(sp)
        assert st == 0, F3.status_string(st)
        graphs, events = timed_graphs(step_api, 2, args.steps, stream)
        kgraphs, kevents = timed_graphs(step_kernels, 6, args.steps, stream)
        # every captured graph is replayed once before timing: a graph's first
        # replay uploads it from the host (milliseconds each), which inside the
        # timed loop would leave the GPU idle between steps
        for g in graphs + kgraphs:
            g.replay()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(local)
        sampler.start()
        t_wall0 = time.perf_counter()
        for g in graphs:
            flush.zero_()
            g.replay()
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        clocks = sampler.stop()
        if world > 1:
            dist.barrier()
        # the kernel breakdown: the same number of replays of the instrumented graph
        torch.cuda.synchronize(dev)
        for g in kgraphs:
            flush.zero_()
            g.replay()
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    st = F3.flux3_check_error(sp)
    assert st == 0, F3.status_string(st)

    per_kernel = {n: statistics.mean(kevents[i][k].elapsed_time(kevents[i][k + 1]) for i in range(args.steps))
                  for k, n in enumerate(names)}
    kernels_step_ms = statistics.mean(kevents[i][0].elapsed_time(kevents[i][5]) for i in range(args.steps))
    step_ms = statistics.mean(events[i][0].elapsed_time(events[i][1]) for i in range(args.steps))
    value, step_ms = replica_throughput(T, step_ms, world, dev)
    tflops = world * block_flops(T) / (step_ms * 1e-3) / 1e12

    # ---- end to end through the public call, host buffers, copies inside the timed region.
    # Each step copies its inputs in from pinned host memory, runs flux3_block_forward and
    # copies the result out; copies run on their own streams and three device buffers let
    # step i+1's upload and step i-1's download overlap step i's compute.  (With two, the
    # upload of step i+2 waits for the download of step i, which waits for step i's
    # compute: every two steps would carry an upload, a compute and a download in series.)
    nbuf = 3
    x_hosts = [synth.activations(2 + b, T, device="cpu").pin_memory() for b in range(nbuf)]
    pos_host = torch.from_numpy(lay.pos.copy()).pin_memory()
    mod_host = synth.modulation(2).pin_memory()
    out_hosts = [torch.empty_like(x_hosts[0]).pin_memory() for _ in range(nbuf)]
    xd = [torch.empty_like(x_hosts[0], device=dev) for _ in range(nbuf)]
    posd = [torch.empty_like(pos_host, device=dev) for _ in range(nbuf)]
    modd = [torch.empty_like(mod_host, device=dev) for _ in range(nbuf)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    torch.cuda.synchronize(dev)

    def e2e_step(i):
        b = i % nbuf
        s_in.wait_event(ev_out[b])                 # the last download of buffer b has read it
        with torch.cuda.stream(s_in):
            xd[b].copy_(x_hosts[b], non_blocking=True)
            posd[b].copy_(pos_host, non_blocking=True)
            modd[b].copy_(mod_host, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        blocks.forward(xd[b], lay.segments, posd[b], modd[b], stream=stream)
        ev_comp[b].record(stream)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            out_hosts[b].copy_(xd[b], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(max(nbuf, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e0.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_value, e2e_ms = replica_throughput(T, e0.elapsed_time(e1) / args.steps, world, dev)
    h2d = x_hosts[0].numel() * 4 + pos_host.numel() * 4 + mod_host.numel() * 4
    d2h = out_hosts[0].numel() * 4
    st = F3.flux3_check_error(sp)
    assert st == 0, F3.status_string(st)

    # ---- LayerNorm + modulation as it runs in a graph: a chain of launches
    # back to back in one CUDA graph (no event between them), rotating over
    # enough input / output sets that each launch's set was last touched more
    # than 2 x L2 bytes earlier; one event pair around the graph.
    set_bytes = T * 3072 * (4 + 2)
    n_sets = max(4, -(-256 * 1024 * 1024 // set_bytes) + 1)
    n_chain = max(20, n_sets)
    ln_x = [synth.activations(10 + k, T, device=dev) for k in range(n_sets)]
    ln_h = [torch.empty((T, 3072), dtype=torch.bfloat16, device=dev) for _ in range(n_sets)]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        F3.flux3_prepare(lay.segments, T, pos.data_ptr(), cfg.rope_theta, sid.data_ptr(), cs.data_ptr(),
                         sn.data_ptr(), sp)
        ln_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ln_graph, stream=stream):
            for j in range(n_chain):
                F3.flux3_ln_modulate(ln_x[j % n_sets].data_ptr(), T, sid.data_ptr(), mods.data_ptr(), cfg.eps_ln,
                                     ln_h[j % n_sets].data_ptr(), sp)
        ln_graph.replay()
        ln_ms = []
        for _ in range(3):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ln_graph.replay()
            b.record(stream)
            b.synchronize()
            ln_ms.append(a.elapsed_time(b) / n_chain)
    st = F3.flux3_check_error(sp)
    assert st == 0, F3.status_string(st)
    del ln_x, ln_h, ln_graph

    hbm, bf16_burst, bf16_sust, peak_src = load_peaks()
    kf = kernel_flops(T)
    dominant = max(("in_projection", "attention", "out_projection"), key=lambda n: per_kernel[n])
    achieved = kf[dominant] / (per_kernel[dominant] * 1e-3) / 1e12
    tr = TRAFFIC.get(dominant)
    traffic = None
    if tr and tr.get("src_sha") == src_sha(tr["src"]) and tr.get("T") == T:
        traffic = tr["bytes_per_launch"]
    roofline = {"kernel": dominant, "bound": "tensor", "achieved": achieved, "peak": bf16_burst,
                "unit": "TFLOP/s", "frac": achieved / bf16_burst, "traffic": traffic,
                "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)" if peak_src == "measured"
                else "fallback 1.8 PFLOP/s"}
    kernels = {}
    for n in names:
        d = {"ms": per_kernel[n]}
        if n in kf:
            d["tflops"] = kf[n] / (per_kernel[n] * 1e-3) / 1e12
            d["frac_of_bf16_peak"] = d["tflops"] / bf16_burst
        if n == "ln_modulate":
            d["gbs"] = kernel_bytes(T)["ln_modulate"] / (per_kernel[n] * 1e-3) / 1e9
            d["frac_of_hbm"] = d["gbs"] / hbm
            g_ms = statistics.mean(ln_ms)
            d["in_graph"] = {"ms": g_ms, "gbs": kernel_bytes(T)["ln_modulate"] / (g_ms * 1e-3) / 1e9,
                             "frac_of_hbm": kernel_bytes(T)["ln_modulate"] / (g_ms * 1e-3) / 1e9 / hbm,
                             "method": f"{n_chain} launches back to back in one CUDA graph over {n_sets} rotating "
                                       "input/output sets (each set untouched for more than 2x L2 bytes), L2 "
                                       "flushed before the graph, one event pair around it"}
        kernels[n] = d

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init N(0,0.02) bf16 weights)",
            "config": {"workload": args.workload, "T": T, "segments": lay.segments,
                       "l2": L2_NOTE,
                       "launch": "one CUDA graph replay of flux3_block_forward per step (events at the graph's "
                                 "ends); kernel breakdown: as many replays of the same launch sequence through the "
                                 "step entry points with an event around each kernel, after the timed region",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "tflops": tflops, "frac_of_bf16_peak": tflops / world / bf16_burst,
            "frac_of_bf16_spec_2250": tflops / world / 2250.0,
            "kernels": kernels, "roofline": roofline,
            "e2e": {"value": e2e_value, "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "api": "flux3_block_forward with pinned host x/pos/mod, H2D + D2H inside the timed region "
                           "(copy streams, three device buffers)"},
            "kernels_step_ms": kernels_step_ms,
            "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
            "wall_s_timed_region": t_wall}
    blocks.close()
    if not args.no_stack_target:
        line["stack28_1024sq_ref1_t8704"] = stack_target(dev, local, world)
    if world > 1:
        dist.barrier()
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_baseline(spec, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_stack(name, steps, warmup, dev, local, world):
    """Times a 28-block stack workload: a step is `calls` stack calls (one per
    sampler step, each with its own modulation vectors) over the whole token
    sequence, bf16 or NVFP4 / fp8r weights (quantised on the device); L2 is
    flushed between steps; CUDA events on the launching stream; nvidia-smi
    clock samples over the timed region.  Returns the figures of the
    workload's line."""
    import torch
    import torch.distributed as dist

    import diffusion_transformer_block_fwd_b300 as F3
    import synth

    wl = synth.WORKLOADS[name]
    lay = synth.build_layout(wl["spec"])
    T, nb, calls = lay.T, wl["blocks"], wl["calls"]
    fp4, fp8 = wl["wfmt"] == "nvfp4", wl["wfmt"] == "fp8r"
    ws = []
    for b in range(nb):
        w = synth.block_weights(1, b, device=dev)
        if fp4 or fp8:
            quant = F3.quantize_nvfp4 if fp4 else F3.quantize_fp8r
            q = {k: quant(w[k]) for k in F3.NVFP4_MATRICES}
            q.update({k: w[k] for k in ("query_norm", "key_norm")})
            w = q
        ws.append(w)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    torch.cuda.synchronize(dev)          # weights were made (and quantised) on the default stream
    with torch.cuda.stream(stream):
        blocks = F3.Flux3Blocks(ws, max_tokens=T, wfmt=wl["wfmt"], stream=stream)
    del ws
    torch.cuda.synchronize(dev)
    x0 = synth.activations(1, T, device=dev)
    x = x0.clone()
    mods = [synth.modulation(1, call=c, device=dev) for c in range(calls)]
    pos = torch.from_numpy(lay.pos).to(dev)
    flush = L2Flush(dev)
    torch.cuda.synchronize(dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        for c in range(calls):
            blocks.forward(x, lay.segments, pos, mods[c], stream=stream)
        if evs is not None:
            evs[1].record(stream)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    expand = (fp4 or fp8) and T > 128   # up to 128 tokens the codes are expanded inside the GEMMs
    per_call_launches = 1 + nb * (4 + (1 if expand else 0) + merges(T, sms))
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            x.copy_(x0)
            step()
        st = F3.flux3_check_error(sp)
        assert st == 0, F3.status_string(st)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(local)
        sampler.start()
        t_wall0 = time.perf_counter()
        for i in range(steps):
            x.copy_(x0)
            flush.zero_()
            step(events[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        clocks = sampler.stop()
    st = F3.flux3_check_error(sp)
    assert st == 0, F3.status_string(st)
    blocks.close()
    value, step_ms = replica_throughput(T * calls, statistics.mean(e[0].elapsed_time(e[1]) for e in events), world,
                                        dev)
    flops = calls * nb * block_flops(T)
    hbm, bf16_burst, bf16_sust, peak_src = load_peaks()
    tflops = world * flops / (step_ms * 1e-3) / 1e12
    return {"T": T, "blocks": nb, "calls": calls, "segments": lay.segments, "fp4": fp4, "fp8": fp8,
            "value": value, "ms_per_step": step_ms, "tflops": tflops, "bf16_burst": bf16_burst,
            "bf16_sust": bf16_sust, "launches": per_call_launches * calls * steps, "clocks": clocks,
            "wall_s_timed_region": t_wall}


def run_stack(args, rank, world, local, dev):
    """A 28-block stack workload's line (see measure_stack)."""
    import torch.distributed as dist

    m = measure_stack(args.workload, args.steps, args.warmup, dev, local, world)
    fp4, fp8, tflops, calls, nb = m["fp4"], m["fp8"], m["tflops"], m["calls"], m["blocks"]
    bf16_burst, bf16_sust, step_ms = m["bf16_burst"], m["bf16_sust"], m["ms_per_step"]
    small = m["T"] <= 128          # one-CTA GEMMs, bound by the weight stream
    if small:
        # weight bytes one block streams: bf16 [27648 + 3072 rows]; NVFP4 e2m1 codes + e4m3 scales
        wbytes = (27648 * 3072 + 3072 * 12288) * (9 / 16 if fp4 else 1 if fp8 else 2)
        gbs = world * wbytes * nb * calls / (step_ms * 1e-3) / 1e9
        hbm = load_peaks()[0]
        roof = {"kernel": "whole stack (weight stream)", "bound": "hbm", "achieved": gbs / world, "peak": hbm,
                "unit": "GB/s", "frac": gbs / world / hbm, "traffic": None,
                "algorithmic_bytes_per_block": wbytes, "peak_source": "measured copy (MEASURED_PEAKS.json)"}
    else:
        roof = {"kernel": "whole stack", "bound": "tensor", "achieved": tflops / world,
                "peak": bf16_sust or bf16_burst, "unit": "TFLOP/s",
                "frac": tflops / world / (bf16_sust or bf16_burst), "traffic": None,
                "peak_source": "measured bf16 sustained (MEASURED_PEAKS.json)"}
    line = {"metric": METRIC, "value": m["value"], "unit": UNIT_STACK,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" + ((" (NVFP4 weights expanded inside the GEMMs)" if small else
                                " (NVFP4 weights dequantised per block)") if fp4 else
                               (" (fp8r weights expanded inside the GEMMs)" if small else
                                " (fp8r weights expanded per block)") if fp8 else ""),
            "data": "synthetic (random-init N(0,0.02) weights" + (", NVFP4-quantised on the device)" if fp4 else
                                                                    ", fp8r-quantised on the device)" if fp8 else ")"),
            "config": {"workload": args.workload, "T": m["T"], "blocks": nb, "calls_per_step": calls,
                       "segments": m["segments"], "l2": L2_NOTE,
                       "launch": "stream launches through flux3_stack_forward"},
            "ms_per_stack_call": step_ms / calls, "ms_per_block": step_ms / calls / nb,
            "tflops": tflops, "frac_of_bf16_peak": tflops / world / bf16_burst,
            "frac_of_bf16_sustained": (tflops / world / bf16_sust) if bf16_sust else None,
            "frac_of_bf16_spec_2250": tflops / world / 2250.0,
            "roofline": roof,
            "gpu_launches": m["launches"], "clocks": m["clocks"], "wall_s_timed_region": m["wall_s_timed_region"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def stack_target(dev, local, world, steps=5, warmup=2):
    """The 28-block stack at 1024x1024 + one 1024x1024 reference (8704 tokens),
    timed on its own (own events and clock record) for the line of the
    single-block workload: ms per stack call and TFLOP/s against the dense
    bf16 spec (2.25 PFLOP/s) and the measured burst and sustained peaks."""
    name = "stack28_1024sq_ref1_t8704"
    m = measure_stack(name, steps, warmup, dev, local, world)
    t = m["tflops"] / world
    return {"workload": name, "T": m["T"], "blocks": m["blocks"], "steps": steps, "warmup": warmup,
            "ms_per_stack_call": m["ms_per_step"] / m["calls"], "ms_per_block": m["ms_per_step"] / m["calls"] / m["blocks"],
            "tokens_per_s": m["value"], "tflops": t, "frac_of_bf16_spec_2250": t / 2250.0,
            "frac_of_bf16_peak": t / m["bf16_burst"],
            "frac_of_bf16_sustained": (t / m["bf16_sust"]) if m["bf16_sust"] else None,
            "gpu_launches": m["launches"], "clocks": m["clocks"],
            "timing": "CUDA events around each stack call (flux3_stack_forward), L2 flushed between calls"}


def run_modes(args, rank, world, local, dev):
    """The per-mode blocks: a step is one flux3_mode_blocks_forward call (each
    mode's tokens through that mode's own `blocks` blocks, attending only among
    themselves).  FLOPs are the per-mode blocks' algorithmic FLOPs, i.e. the
    block formula at each mode's own token count."""
    import torch
    import torch.distributed as dist

    import diffusion_transformer_block_fwd_b300 as F3
    from diffusion_transformer_block_fwd_b300.model import mode_blocks_forward
    import synth

    wl = synth.WORKLOADS[args.workload]
    lay = synth.build_layout(wl["spec"])
    T, nb = lay.T, wl["blocks"]
    counts = [int((lay.stream_id == m).sum()) for m in range(3)]
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    mb = []
    for m in range(3):
        ws = [synth.block_weights(1 + m, b, device=dev) for b in range(nb)]
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            mb.append(F3.Flux3Blocks(ws, max_tokens=max(1, counts[m]), stream=stream) if counts[m] else None)
        del ws
    torch.cuda.synchronize(dev)
    x0 = synth.activations(1, T, device=dev)
    x = x0.clone()
    mods = synth.modulation(1, device=dev)
    pos = torch.from_numpy(lay.pos).to(dev)
    flush = L2Flush(dev)
    torch.cuda.synchronize(dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        mode_blocks_forward(mb, x, lay.segments, pos, mods, stream=stream)
        if evs is not None:
            evs[1].record(stream)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    launches = sum(1 + nb * (4 + merges(c, sms)) for c in counts if c)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            x.copy_(x0)
            step()
        st = F3.flux3_check_error(sp)
        assert st == 0, F3.status_string(st)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(local)
        sampler.start()
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            x.copy_(x0)
            flush.zero_()
            step(events[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        clocks = sampler.stop()
    st = F3.flux3_check_error(sp)
    assert st == 0, F3.status_string(st)
    value, step_ms = replica_throughput(T, statistics.mean(e[0].elapsed_time(e[1]) for e in events), world, dev)
    flops = nb * sum(block_flops(c) for c in counts if c)
    hbm, bf16_burst, bf16_sust, peak_src = load_peaks()
    tflops = world * flops / (step_ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT_MODES,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random-init N(0,0.02) weights, one set per mode)",
            "config": {"workload": args.workload, "T": T, "tokens_per_mode": counts, "blocks_per_mode": nb,
                       "segments": lay.segments, "l2": L2_NOTE,
                       "launch": "stream launches through flux3_mode_blocks_forward"},
            "tflops": tflops, "frac_of_bf16_peak": tflops / world / bf16_burst,
            "frac_of_bf16_sustained": (tflops / world / bf16_sust) if bf16_sust else None,
            "roofline": {"kernel": "per-mode blocks", "bound": "tensor", "achieved": tflops / world,
                         "peak": bf16_burst, "unit": "TFLOP/s", "frac": tflops / world / bf16_burst,
                         "traffic": None, "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)"},
            "gpu_launches": launches * args.steps, "clocks": clocks, "wall_s_timed_region": t_wall}
    if rank == 0:
        print(json.dumps(line), flush=True)
    for b in mb:
        if b is not None:
            b.close()
    if world > 1:
        dist.destroy_process_group()


def model_call_flops(counts, n_mode_blocks, n_joint):
    """Algorithmic FLOPs of one transformer call: embedders, the per-mode
    blocks at each mode's token count, the joint blocks, the output linear
    (the conditioning linears are ~0.2 GFLOP and not counted)."""
    T = sum(counts)
    emb = 2 * 3072 * ((counts[0] + counts[1]) * 128 + counts[2] * 20480)
    modes = n_mode_blocks * sum(block_flops(c) for c in counts if c)
    return emb + modes + n_joint * block_flops(T) + 2 * counts[0] * 3072 * 128


def cfg_call_flops(counts, n_mode_blocks, n_joint):
    """Algorithmic FLOPs of one batched call on a pack (counts per sample):
    per sample the embedders, per-mode blocks and output linear; the joint
    blocks with attention within each sample."""
    return (sum(model_call_flops(c, n_mode_blocks, 0) for c in counts)
            + n_joint * sum(block_flops(sum(c)) for c in counts))


def workload_call(name):
    """What a step of `name` repeats: (tokens, algorithmic FLOPs, unit) of one
    call, the unit being that of the workload's JSON line.  The value of a
    line is tokens per call / seconds per call."""
    import synth
    wl = synth.WORKLOADS[name]
    stage, nb = wl.get("stage"), wl["blocks"]
    if stage == "cfg":
        pack = synth.build_pack(wl["specs"])
        counts = [[int((lay.stream_id == m).sum()) for m in range(3)] for lay in pack.layouts]
        return pack.T, cfg_call_flops(counts, wl["mode_blocks"], nb), UNIT_CFG
    lay = synth.build_layout(wl["spec"])
    counts = [int((lay.stream_id == m).sum()) for m in range(3)]
    if stage == "model":
        return lay.T, model_call_flops(counts, wl["mode_blocks"], nb), UNIT_MODEL
    if stage == "modes":
        return lay.T, nb * sum(block_flops(c) for c in counts if c), UNIT_MODES
    if nb > 1:
        return lay.T, nb * block_flops(lay.T), UNIT_STACK
    return lay.T, block_flops(lay.T), UNIT


def run_model(args, rank, world, local, dev):
    """The flow-map sampler: a step is `calls` sampler steps, each one
    transformer call (flux3_transformer_forward: conditioning, embedders, the
    per-mode blocks, the joint blocks, the output layer) and the Euler update
    of the image latents (flux3_euler_step)."""
    import torch
    import torch.distributed as dist

    import diffusion_transformer_block_fwd_b300 as F3
    import synth

    wl = synth.WORKLOADS[args.workload]
    lay = synth.build_layout(wl["spec"])
    T, nb, steps, nm = lay.T, wl["blocks"], wl["calls"], wl["mode_blocks"]
    counts = [int((lay.stream_id == m).sum()) for m in range(3)]
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        cw = synth.cond_weights(1, device=dev)
        stream.synchronize()
        cond = F3.Flux3Conditioning(cw, stream=stream)
        del cw
        mb = []
        for m in range(3):
            if counts[m] == 0:
                mb.append(None)
                continue
            ws = [synth.block_weights(10 + m, b, device=dev) for b in range(nm)]
            stream.synchronize()
            mb.append(F3.Flux3Blocks(ws, max_tokens=counts[m], stream=stream))
            del ws
        ws = [synth.block_weights(1, b, device=dev) for b in range(nb)]
        stream.synchronize()
        joint = F3.Flux3Blocks(ws, max_tokens=T, stream=stream)
        del ws
    torch.cuda.synchronize(dev)
    model = F3.Flux3Transformer(cond, mb, joint)
    ins = synth.stream_inputs(1, lay, device=dev)
    noise = ins[0].float()
    lat = noise.clone()
    pos = torch.from_numpy(lay.pos).to(dev)
    flush = L2Flush(dev)
    torch.cuda.synchronize(dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        model.sample(lat, ins, lay.segments, pos, steps=steps, stream=stream)
        if evs is not None:
            evs[1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            lat.copy_(noise)
            step()
        st = F3.flux3_check_error(sp)
        assert st == 0, F3.status_string(st)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(local)
        sampler.start()
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            lat.copy_(noise)
            flush.zero_()
            step(events[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        clocks = sampler.stop()
    st = F3.flux3_check_error(sp)
    assert st == 0, F3.status_string(st)
    assert torch.isfinite(lat).all()
    value, step_ms = replica_throughput(T * steps, statistics.mean(e[0].elapsed_time(e[1]) for e in events), world,
                                        dev)
    flops = steps * model_call_flops(counts, nm, nb)
    hbm, bf16_burst, bf16_sust, peak_src = load_peaks()
    tflops = world * flops / (step_ms * 1e-3) / 1e12
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    per_call_launches = (15 + sum(1 + nm * (4 + merges(c, sms)) for c in counts if c)
                         + 1 + nb * (4 + merges(T, sms)) + 1
                         + sum(1 for s_ in lay.segments) + 2 + 1)
    line = {"metric": METRIC, "value": value, "unit": UNIT_MODEL,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random-init N(0,0.02) weights, N(0,1) latents and text features)",
            "config": {"workload": args.workload, "T": T, "tokens_per_mode": counts, "sampler_steps": steps,
                       "mode_blocks": nm, "joint_blocks": nb, "segments": lay.segments,
                       "l2": L2_NOTE,
                       "launch": "stream launches through flux3_transformer_forward and flux3_euler_step"},
            "ms_per_image": step_ms, "ms_per_call": step_ms / steps,
            "tflops": tflops, "frac_of_bf16_peak": tflops / world / bf16_burst,
            "frac_of_bf16_sustained": (tflops / world / bf16_sust) if bf16_sust else None,
            "roofline": {"kernel": "whole sampler", "bound": "tensor", "achieved": tflops / world,
                         "peak": bf16_sust or bf16_burst, "unit": "TFLOP/s",
                         "frac": tflops / world / (bf16_sust or bf16_burst), "traffic": None,
                         "peak_source": "measured bf16 sustained (MEASURED_PEAKS.json)"},
            "gpu_launches": per_call_launches * steps * args.steps, "clocks": clocks, "wall_s_timed_region": t_wall}
    if rank == 0:
        print(json.dumps(line), flush=True)
    for b in mb + [joint]:
        if b is not None:
            b.close()
    cond.close()
    if world > 1:
        dist.destroy_process_group()


def run_cfg(args, rank, world, local, dev):
    """The base model's sampler: a step is `calls` sampler steps, each one
    batched transformer call on the two-sample pack [unconditional,
    conditional] (flux3_transformer_forward_batch: joint blocks over both
    samples at once, attention per sample) and the guided Euler update
    (flux3_cfg_euler_step, guidance 3.5)."""
    import torch
    import torch.distributed as dist

    import diffusion_transformer_block_fwd_b300 as F3
    import synth

    wl = synth.WORKLOADS[args.workload]
    pack = synth.build_pack(wl["specs"])
    T, nb, steps, nm = pack.T, wl["blocks"], wl["calls"], wl["mode_blocks"]
    counts = [[int((lay.stream_id == m).sum()) for m in range(3)] for lay in pack.layouts]
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        cw = synth.cond_weights(1, device=dev, flow=False)
        stream.synchronize()
        cond = F3.Flux3Conditioning(cw, stream=stream)
        del cw
        mb = []
        for m in range(3):
            mx = max(c[m] for c in counts)
            if mx == 0:
                mb.append(None)
                continue
            ws = [synth.block_weights(10 + m, b, device=dev) for b in range(nm)]
            stream.synchronize()
            mb.append(F3.Flux3Blocks(ws, max_tokens=mx, stream=stream))
            del ws
        ws = [synth.block_weights(1, b, device=dev) for b in range(nb)]
        stream.synchronize()
        joint = F3.Flux3Blocks(ws, max_tokens=T, stream=stream)
        del ws
    torch.cuda.synchronize(dev)
    model = F3.Flux3Transformer(cond, mb, joint)
    ins = [synth.stream_inputs(1 + b, lay, device=dev) for b, lay in enumerate(pack.layouts)]
    noise = ins[1][0].float()
    lat = noise.clone()
    pos = torch.from_numpy(pack.pos).to(dev)
    flush = L2Flush(dev)
    torch.cuda.synchronize(dev)

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        model.sample_cfg(lat, ins[0], ins[1], pack.segments, pack.sample_start, pos, steps=steps, stream=stream)
        if evs is not None:
            evs[1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            lat.copy_(noise)
            step()
        st = F3.flux3_check_error(sp)
        assert st == 0, F3.status_string(st)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(local)
        sampler.start()
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            lat.copy_(noise)
            flush.zero_()
            step(events[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        clocks = sampler.stop()
    st = F3.flux3_check_error(sp)
    assert st == 0, F3.status_string(st)
    assert torch.isfinite(lat).all()
    value, step_ms = replica_throughput(T * steps, statistics.mean(e[0].elapsed_time(e[1]) for e in events), world,
                                        dev)
    # per call: per-sample embedders, per-mode blocks and output layers; joint blocks over the pack
    per_call = cfg_call_flops(counts, nm, nb)
    # our kernels per call: per sample ~13 conditioning launches, one embedder GEMM per segment, the per-mode
    # blocks (2 + 4 per block per present mode), the output layer (LayerNorm + GEMM); the joint blocks
    # (2 + 4 per block, one more attention launch per block for each further sample); the guided update
    n_s = len(counts)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    launches = (sum(13 + len(lay.segments) + sum(1 + nm * (4 + merges(c[m], sms))
                                                  for m in range(3) if c[m]) + 2
                    for c, lay in zip(counts, pack.layouts))
                + 1 + nb * (4 + (out_proj_splits(pack.T, sms) > 1)
                            + sum(1 + (attn_splits(l.T, sms) > 1) for l in pack.layouts) - 1) + 1)
    flops = steps * per_call
    hbm, bf16_burst, bf16_sust, peak_src = load_peaks()
    tflops = world * flops / (step_ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT_CFG,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random-init N(0,0.02) weights, N(0,1) latents and text features)",
            "config": {"workload": args.workload, "T": T, "sample_start": pack.sample_start,
                       "tokens_per_mode_per_sample": counts, "sampler_steps": steps, "guidance": 3.5,
                       "mode_blocks": nm, "joint_blocks": nb, "segments": pack.segments,
                       "l2": L2_NOTE,
                       "launch": "stream launches through flux3_transformer_forward_batch and flux3_cfg_euler_step"},
            "ms_per_image": step_ms, "ms_per_call": step_ms / steps,
            "tflops": tflops, "frac_of_bf16_peak": tflops / world / bf16_burst,
            "frac_of_bf16_sustained": (tflops / world / bf16_sust) if bf16_sust else None,
            "roofline": {"kernel": "whole sampler", "bound": "tensor", "achieved": tflops / world,
                         "peak": bf16_sust or bf16_burst, "unit": "TFLOP/s",
                         "frac": tflops / world / (bf16_sust or bf16_burst), "traffic": None,
                         "peak_source": "measured bf16 sustained (MEASURED_PEAKS.json)"},
            "gpu_launches": launches * steps * args.steps, "clocks": clocks, "wall_s_timed_region": t_wall}
    if rank == 0:
        print(json.dumps(line), flush=True)
    for b in mb + [joint]:
        if b is not None:
            b.close()
    cond.close()
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="block_1024sq_t4608")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stack-target", action="store_true",
                    help="skip the 28-block 8704-token stack timed beside the single-block workload")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
