"""Benchmark of the sink + window KV attention hot path on GB300.

Default workload (N=1): the windowed-layer decode step -- B=32 sequences, H_q=32,
H_kv=8, d_h=r=128, theta=5e5, bf16, S=4 sinks + W=4092 ring (C=4096), positions
U[4096, 32768] with the ring wrapped at a random head; each step rotates and appends
one new token per sequence and runs split-K decode attention over the 4096 visible
keys.  The metric is the KV bytes the attention must read per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload window|hybrid|rerotate|prefill]

For N > 1 (torchrun, one rank per GPU) every rank runs its own replica: the path
shards by sequence with no exchange step, so scaling is weak.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sink+window decode attn KV-read GB/s (frac of HBM peak), tokens/s, keys/s"


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a kernel from one
# ncu capture, stated here with the sha256 of every source the captured build came from.
# A row reports it only while those sources are unchanged, else null.  "scale": the capture
# ran a smaller case of the same kernel; the traffic grows in proportion to the units
# processed and is scaled by that factor to one launch of the full workload.
DECODE_SOURCES = {"decode.cu": "e6c7c2686de1a89eeb4a8c18ed6f37b833011124de96333c41c2fea3ae08a2b3",
                  "decode_kernels.cuh": "ca32eb46afc019674dcaf78784becae5d1234f61e3683aec9364237854cca0cf",
                  "rope_lane.cuh": "92cd7898465a1776e0e3f9e32707943dca4d074e80246d99524d949885102532",
                  "common.cuh": "b851c4f7d4f058ac8da61a6434a86b4bf5523a2512acac6795794a145dcd4fa0"}
NCU_TRAFFIC = {
    "decode_window_b32": dict(
        bytes=542240000, scale=1,
        capture="ncu --set full -k regex:decode_split -s 3 -c 1, python bench.py --no-rows --no-cpu-baseline "
                "--steps 5 --warmup 3 (split kernel only)",
        sources=DECODE_SOURCES),
    "decode_paged_window_b32_bs16": dict(
        bytes=540921088, scale=1,
        capture="ncu --set full -k regex:decode_split -s 3 -c 1, python bench.py --workload paged "
                "--steps 5 --warmup 3 (split kernel only)",
        sources=DECODE_SOURCES),
    "decode_window_b32_int8": dict(
        bytes=410360032, scale=1,
        capture="ncu --set full -k regex:decode_split -s 3 -c 1, python bench.py --workload window_i8 "
                "--steps 5 --warmup 3 (split kernel only)",
        sources=DECODE_SOURCES),
    "decode_step_window_b32": dict(
        bytes=541355520, scale=1,
        capture="ncu --set full -k regex:decode_split -s 3 -c 1, python bench.py --workload window_step "
                "--steps 5 --warmup 3 (fused split kernel only)",
        sources=dict(DECODE_SOURCES, **{"decode_step.cu": "ccf687b9b226f8b64abc0f4dc079d32f1dbdcc27c072859308f1e00ad42dff18"})),
    "prefill_attn_t32768": dict(
        bytes=633978880, scale=1,
        capture="ncu --set full -k regex:prefill_attn -s 2 -c 1, python bench.py --workload prefill "
                "--steps 3 --warmup 2",
        sources={"prefill.cu": "bf63f0ca63cd9186c7cb6bee43620de94930b33e1d74b6e801213dd5b5d633b1",
                 "tcgen05.cuh": "351b9597267c8e6efeb86d6fc37090095dc2b99a351b47884061cba635ae854d"}),
    "rerotate_bf16_48l": dict(
        bytes=2358400000, scale=12,
        capture="ncu --set full -k regex:rerotate_bf16 -s 2 -c 1, python bench.py --workload rerotate_bf16 "
                "--layers 4 --steps 3 --warmup 2 (4 of 48 layers, x12)",
        sources={"rerotate.cu": "d3577ee983e461c227d117bf96e81fbb3eb4d59417b4704116cc72c317f3b411"}),
    "rerotate_i8_48l": dict(
        bytes=2421800000, scale=12,
        capture="ncu --set full -k regex:rerotate_i8 -s 2 -c 1, python bench.py --workload rerotate_i8 "
                "--layers 4 --steps 3 --warmup 2 (4 of 48 layers, x12)",
        sources={"rerotate.cu": "d3577ee983e461c227d117bf96e81fbb3eb4d59417b4704116cc72c317f3b411"}),
}


def _traffic(name):
    """Per-launch DRAM bytes of NCU_TRAFFIC[name] while its sources are unchanged, else None."""
    import hashlib
    ent = NCU_TRAFFIC.get(name)
    if ent is None:
        return None
    for fname, digest in ent["sources"].items():
        try:
            with open(os.path.join(ROOT, "sink_kv_attention_gb300", "csrc", fname), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return int(ent["bytes"] * ent["scale"])


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.06 <= r[0] <= (self.t1 or 1e30) + 0.06]
        used = inside if inside else [min(rows, key=lambda r: abs(r[0] - (self.t1 or r[0])))]
        sm = [float(p[1]) for _, p in used if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in used if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, p in used for n, v in zip(names, p[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(used), "in_region": bool(inside)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------

def _dist_init(n_gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world, device="cuda"):
    """Slowest rank's time: the whole job is as fast as its slowest replica."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed_base(rank):
    """Each replica draws its own synthetic inputs (independent sequences per GPU)."""
    return 100 * rank


def weak_scaling_value(bytes_per_rank, ms_per_step_max, world):
    """Whole-job GB/s: every rank moved bytes_per_rank per step; time is the slowest rank's."""
    return world * bytes_per_rank / (ms_per_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# windowed decode workload
# ---------------------------------------------------------------------------

def window_setup(seed_base=0, steps=1):
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    tbl = sk.RopeTable(D, c["r"], c["theta"], c["pos_hi"] + steps + 64)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 11 + seed_base)
    synth.fill_normal_(layer.v, 12 + seed_base)
    pos, head, count = synth.window_state(13 + seed_base, B, W, c["pos_lo"], c["pos_hi"])
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    return tbl, layer, c


def _learned_sinks(args, n_q_heads):
    """Per-head learned sink logits for --learned-sink runs (float32 on the device),
    spread over the clamp range; None otherwise."""
    import torch
    if not args.learned_sink:
        return None
    return torch.linspace(-12.0, 17.0, n_q_heads, device="cuda").contiguous()


def bench_window(args, rank, world):
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    steps, warm = args.steps, args.warmup
    tbl, layer, c = window_setup(seed_base=replica_seed_base(rank), steps=2 * steps + warm + 2)
    B, Hq, Hkv, D, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["W"]
    n = steps + warm
    # one fresh token per sequence per step, resident in HBM before timing
    qs = synth.normal((n, B, 1, Hq, D), 14, torch.bfloat16, device="cuda")
    ks = synth.normal((n, B, 1, Hkv, D), 15, torch.bfloat16, device="cuda")
    vs = synth.normal((n, B, 1, Hkv, D), 16, torch.bfloat16, device="cuda")
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(sk.decode_workspace_bytes(layer, Hq), sk.decode_step_workspace_bytes(layer, Hq)),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    zl = _learned_sinks(args, Hq)

    def step(i):
        sk.kv_append(tbl, layer, qs[i], ks[i], vs[i])
        sk.decode_attention(layer, qs[i, :, 0], out=out, workspace=ws, sink_logits=zl)

    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    # The timed steps run as one captured CUDA graph, the way a serving loop runs decode
    # (the library's calls keep all state on the device, so they capture).  The graph is
    # replayed until the timed region lasts at least TARGET_MS; after every replay the
    # ring counters are put back, so every replay makes the same appends and reads.
    reset = _state_saver([layer])
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    if args.eager:
        graph = None
        per = []
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
        _barrier(world)
        torch.cuda.synchronize()
        clocks.mark("start")
        t0 = time.perf_counter()
        for a, b in ev:
            a.record(stream)
            for i in range(steps):
                step(warm + i)
            b.record(stream)
            reset()
        torch.cuda.synchronize()
        clocks.mark("end")
        per = [a.elapsed_time(b) / steps for a, b in ev]
        region_ms, R = (time.perf_counter() - t0) * 1e3, len(ev)
    else:
        graph = _capture(step, warm, steps)
        per, region_ms, R = _replays(graph, steps, TARGET_MS, reset=reset, clocks=clocks, world=world)
    if rank == 0:
        clocks.stop()
    assert layer.error_bits() == 0
    ms_step = _max_over_ranks(statistics.median(per), world)
    # the same steps as the decode step (sk_decode_step: the append folded into the
    # attention's two kernels), on the same state
    ms_fused = None
    if graph is not None:
        def step_fused(i):
            sk.decode_step(tbl, layer, qs[i, :, 0], ks[i, :, 0], vs[i, :, 0], out=out, workspace=ws, sink_logits=zl)
        g_f = _capture(step_fused, warm, steps)
        per_f, _, _ = _replays(g_f, steps, TARGET_MS / 2, reset=reset, world=world)
        assert layer.error_bits() == 0
        ms_fused = _max_over_ranks(statistics.median(per_f), world)

    L = c["S"] + W  # visible keys per sequence (ring full)
    kv_bytes = B * Hkv * L * D * 2 * 2
    alg_bytes_decode = kv_bytes + 2 * (B * Hq * D * 2)          # + q read, out write
    value = weak_scaling_value(kv_bytes, ms_step, world)
    # the dominant kernel, decode attention: its launches back to back in one graph
    roof = _launch_roofline(lambda i: sk.decode_attention(layer, qs[i, :, 0], out=out, workspace=ws, sink_logits=zl),
                            steps, alg_bytes_decode, "decode_window_b32",
                            "decode attention (split-K + combine); its launches back to back in one graph",
                            "K+V of 4096 visible rows x 32 sequences x 8 kv heads + q + out")

    # end to end through the public API with host buffers: pinned inputs copied in,
    # the output copied out, every step.  A serving loop overlaps the copies of the next
    # step with the current step's kernels: the device inputs and outputs are double
    # buffered and the copies run on a second stream, ordered by events.
    hq = torch.empty((steps, B, 1, Hq, D), dtype=torch.bfloat16).pin_memory()
    hk = torch.empty((steps, B, 1, Hkv, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty((steps, B, 1, Hkv, D), dtype=torch.bfloat16).pin_memory()
    hq.copy_(qs[:steps].cpu()); hk.copy_(ks[:steps].cpu()); hv.copy_(vs[:steps].cpu())
    hout = torch.empty((steps, B, Hq, D), dtype=torch.bfloat16).pin_memory()
    dq = [torch.empty_like(qs[0]) for _ in range(2)]
    dk = [torch.empty_like(ks[0]) for _ in range(2)]
    dv = [torch.empty_like(vs[0]) for _ in range(2)]
    dout = [torch.empty_like(out) for _ in range(2)]
    tbl2, layer2, _ = window_setup(seed_base=100 * rank + 7, steps=steps + 2)
    copy_stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def e2e_steps():
        comp = torch.cuda.current_stream()
        # event lists per step: inputs landed, step computed, output read back
        landed = [torch.cuda.Event() for _ in range(steps)]
        computed = [torch.cuda.Event() for _ in range(steps)]
        read = [torch.cuda.Event() for _ in range(steps)]

        def h2d(i):
            j = i % 2
            copy_stream.wait_stream(comp) if i == 0 else None
            if i >= 2:
                copy_stream.wait_event(computed[i - 2])   # buffers j free again
            with torch.cuda.stream(copy_stream):
                dq[j].copy_(hq[i], non_blocking=True)
                dk[j].copy_(hk[i], non_blocking=True)
                dv[j].copy_(hv[i], non_blocking=True)
                landed[i].record(copy_stream)

        h2d(0)
        for i in range(steps):
            j = i % 2
            if i + 1 < steps:
                h2d(i + 1)
            comp.wait_event(landed[i])
            if i >= 2:
                comp.wait_event(read[i - 2])   # out buffer j read back
            sk.kv_append(tbl2, layer2, dq[j], dk[j], dv[j])
            sk.decode_attention(layer2, dq[j][:, 0], out=dout[j], workspace=ws, sink_logits=zl)
            computed[i].record(comp)
            copy_stream.wait_event(computed[i])
            with torch.cuda.stream(copy_stream):
                hout[i].copy_(dout[j], non_blocking=True)
                read[i].record(copy_stream)
        comp.wait_stream(copy_stream)

    reset2 = _state_saver([layer2])
    if graph is not None:  # the same calls, host copies included, as one captured graph
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_steps()
        torch.cuda.synchronize()
        per_e, _, _ = _replays(g_e2e, steps, TARGET_MS / 2, reset=reset2, world=world)
    else:
        per_e = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_steps()
            e1.record(stream)
            torch.cuda.synchronize()
            reset2()
            per_e.append(e0.elapsed_time(e1) / steps)
    e2e_ms = _max_over_ranks(statistics.median(per_e), world)
    if layer2.error_bits() != 0:  # a skipped append would make the timed pass do less work
        raise RuntimeError(f"end-to-end pass set device error bits {layer2.error_bits():#x}")
    h2d_bytes = (hq[0].numel() + hk[0].numel() + hv[0].numel()) * 2
    e2e = {"value": round(world * kv_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": hout[0].numel() * 2,
           "ms_per_step": round(e2e_ms, 5),
           "overlap": "next step's inputs copied in on a second stream during this step"}

    hbm, _, _, peak_kind = _peaks()
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "windowed-layer decode step (RoPE + append + split-K attention)",
                   "batch_per_gpu": B, "H_q": Hq, "H_kv": Hkv, "d_h": D, "rotary_dim": c["r"],
                   "theta": c["theta"], "sinks": c["S"], "window": W, "visible_keys": L,
                   "positions": "U[4096, 32768], ring wrapped at random head",
                   "learned_sink_logits": bool(args.learned_sink),
                   "l2": f"inputs larger than L2 (KV {kv_bytes / 1e6:.0f} MB per step > 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "frac_of_hbm_peak": round(value / world / hbm, 4),
        "tokens_per_s": round(world * B / (ms_step * 1e-3), 1),
        "keys_per_s": round(world * B * L / (ms_step * 1e-3), 1),
        "roofline": roof,
        "e2e": e2e,
        "decode_step": None if ms_fused is None else {
            "ms_per_step": round(ms_fused, 5), "gbs": round(world * kv_bytes / (ms_fused * 1e-3) / 1e9, 2),
            "calls": "sk_decode_step: the same steps in two launches (split with the token's RoPE + append, "
                     "combine), same state; not the headline, which times sk_kv_append + sk_decode_attention"},
        "timing": {"replays": R, "steps_per_replay": steps, "timed_steps": R * steps,
                   "timed_ms": round(region_ms, 2), "ms_per_step": "median over replays",
                   "ms_per_step_mean": round(statistics.fmean(per), 5),
                   "ms_per_step_min": round(min(per), 5), "ms_per_step_max": round(max(per), 5)},
        "gpu_launches": R * steps * 3,
        "launch": "eager" if graph is None else "cuda graph of the steps, replayed",
    }
    if rank == 0:
        result["clocks"] = clocks.summary()
    return result


# ---------------------------------------------------------------------------
# other rows of the hot path (measured with --workload)
# ---------------------------------------------------------------------------

TARGET_MS = 300.0        # the shortest timed region: replays of a captured graph of the steps
MAX_REPLAYS = 2000


def _capture(fn, first, n):
    """One CUDA graph of fn(first) .. fn(first + n - 1) (the library's calls keep all
    state on the device, so they capture)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fn(first + i)
    torch.cuda.synchronize()
    return g


def _replays(graph, n_steps, target_ms=TARGET_MS, reset=None, clocks=None, world=1, max_replays=MAX_REPLAYS):
    """Replay a captured graph of n_steps steps until the timed region lasts at least
    target_ms: one untimed replay first (it also uploads the graph), then R timed
    replays, each between two events on the launching stream.  reset(), when given,
    runs after every replay, outside the per-replay events (it puts back state such as
    a ring's counters).  Returns the per-step times of the replays (ms), the whole
    region's time (ms) and R."""
    import torch
    stream = torch.cuda.current_stream()
    graph.replay()
    if reset is not None:
        reset()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    if reset is not None:
        reset()
    torch.cuda.synchronize()
    est = max(e0.elapsed_time(e1), 1e-3)
    R = int(min(max_replays, max(3, -(-target_ms // est))))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(R)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark("start")
    t0.record(stream)
    for a, b in ev:
        a.record(stream)
        graph.replay()
        b.record(stream)
        if reset is not None:
            reset()
    t1.record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark("end")
    _barrier(world)
    per_step = [a.elapsed_time(b) / n_steps for a, b in ev]
    return per_step, t0.elapsed_time(t1), R


def _timed(fn, steps, warm, target_ms=TARGET_MS, reset=None):
    """Run fn(i) warm times, capture fn(warm) .. fn(warm + steps - 1) as one CUDA graph
    and replay it until at least target_ms are timed; returns the median time per step
    (ms), the clocks sampled over the timed region and the timing record."""
    import torch
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    if reset is not None:
        reset()
    g = _capture(fn, warm, steps)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    per, total, R = _replays(g, steps, target_ms, reset=reset, clocks=clocks)
    clocks.stop()
    ms = statistics.median(per)
    return ms, clocks.summary(), {"replays": R, "steps_per_replay": steps, "timed_ms": round(total, 2),
                                  "ms_per_step_mean": round(statistics.fmean(per), 5),
                                  "ms_per_step_min": round(min(per), 5), "ms_per_step_max": round(max(per), 5)}


def _state_saver(layers):
    """reset() that puts back the layers' pos (and ring head/count) as they are now,
    with device-to-device copies (no kernels)."""
    saved = []
    for L in layers:
        for t in (L.pos, L.head, L.count):
            if t is not None:
                saved.append((t, t.clone()))

    def reset():
        for t, s0 in saved:
            t.copy_(s0)
    return reset


def _launch_roofline(fn, n, alg_bytes, name, kernel, unit_note, target_ms=TARGET_MS / 2, reset=None):
    """Roofline of an HBM-bound kernel: fn(i) for i < n (launches of that kernel alone,
    back to back in one graph, programmatic dependent launch between them, as in a
    decode loop over layers) replayed for target_ms; achieved = algorithmic bytes per
    launch / median time per launch.  reset() (outside the timed replays) puts back
    state the launches advance."""
    hbm, _, _, peak_kind = _peaks()
    g = _capture(fn, 0, n)
    per, total, R = _replays(g, n, target_ms, reset=reset)
    ms = statistics.median(per)
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "traffic": _traffic(name) if name else None,
            "kernel": kernel, "algorithmic_bytes_per_launch": int(alg_bytes), "algorithmic_bytes": unit_note,
            "launch_ms": round(ms, 5), "launches_timed": R * n, "peak_source": f"{peak_kind} hbm_gbs (of measured)"
            if peak_kind == "measured" else f"{peak_kind} hbm_gbs"}


def bench_hybrid(args):
    """Llama-3-8B-shaped hybrid decode: 32 layers (every 4th global with a 131072-token
    prefix, the rest S=4 + W=4096 rings), B=16; one step = RoPE + append + attention on
    all 32 layers as sk_kv_append + sk_decode_attention; the decode step (sk_decode_step)
    timed beside it on the same state.  The layers' counters are put back after every
    replay of the captured steps, so each replay makes the same appends and reads."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.HYBRID
    B, Hq, Hkv, D, S, W, prefix = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"], c["prefix"]
    steps, warm = args.steps, args.warmup
    tbl = sk.RopeTable(D, c["r"], c["theta"], prefix + steps + warm + 8)
    layers = []
    for i in range(c["layers"]):
        if synth.hybrid_layer_is_global(i):
            L = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=prefix + steps + warm + 4)
        else:
            L = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
            L.count.fill_(W)
            L.head.copy_(synth.randint((B,), 900 + i, 0, W).to(torch.int32))
        synth.fill_normal_(L.k, 1000 + i)
        synth.fill_normal_(L.v, 2000 + i)
        L.pos.fill_(prefix)
        layers.append(L)
    n = steps + warm
    nl = c["layers"]
    # fresh q/k/v per layer and step, resident in HBM before timing
    qs = synth.normal((n, nl, B, 1, Hq, D), 3, torch.bfloat16, device="cuda")
    ks = synth.normal((n, nl, B, 1, Hkv, D), 4, torch.bfloat16, device="cuda")
    vs = synth.normal((n, nl, B, 1, Hkv, D), 5, torch.bfloat16, device="cuda")
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(max(sk.decode_workspace_bytes(L, Hq), sk.decode_step_workspace_bytes(L, Hq))
                         for L in layers), dtype=torch.uint8, device="cuda")
    zl = _learned_sinks(args, Hq)

    def step(i):  # rotates q and k in place
        for j, L in enumerate(layers):
            sk.kv_append(tbl, L, qs[i, j], ks[i, j], vs[i, j])
            sk.decode_attention(L, qs[i, j, :, 0], out=out, workspace=ws, sink_logits=zl)

    def step_fused(i):  # q, k, v are read only
        for j, L in enumerate(layers):
            sk.decode_step(tbl, L, qs[i, j, :, 0], ks[i, j, :, 0], vs[i, j, :, 0], out=out, workspace=ws,
                           sink_logits=zl)

    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    reset = _state_saver(layers)
    ms, clk, rec = _timed(lambda i: step(warm + i), steps, 0, reset=reset)
    assert all(L.error_bits() == 0 for L in layers)
    n_glob = sum(1 for i in range(c["layers"]) if synth.hybrid_layer_is_global(i))
    n_slid = c["layers"] - n_glob
    # visible rows grow by one per step on global layers; use the mean over the captured steps
    mean_glob = prefix + 1 + warm + (steps - 1) / 2
    kv_bytes = (n_glob * mean_glob + n_slid * (S + W)) * B * Hkv * D * 2 * 2
    hbm, _, _, peak_kind = _peaks()
    value = kv_bytes / (ms * 1e-3) / 1e9
    # the dominant kernel: decode attention over a global layer (131,073+ visible rows per
    # (sequence, kv head)), the 8 global layers' calls back to back
    glob = [L for L in layers if L.kind == sk.SK_LAYER_GLOBAL]
    rows_g = int(glob[0].pos[0])
    alg = B * Hkv * rows_g * D * 2 * 2 + 2 * B * Hq * D * 2
    roof = _launch_roofline(lambda i: sk.decode_attention(glob[i % len(glob)], qs[0, 0, :, 0], out=out, workspace=ws,
                                                          sink_logits=zl),
                            len(glob), alg, None, "decode attention over a global layer (split-K + combine), "
                            "8 launches back to back", f"K+V of {rows_g} rows x 16 sequences x 8 kv heads + q + out")
    reset()
    ms_fused, _, rec_fused = _timed(lambda i: step_fused(warm + i), steps, 0, reset=reset)
    assert all(L.error_bits() == 0 for L in layers)
    return {"metric": "hybrid decode step KV-read GB/s (frac of HBM peak), tokens/s", "value": round(value, 2),
            "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": warm, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "Llama-3-8B-shaped hybrid decode: 32 layers 3:1 sliding:global, B=16, "
                                   "H_q=32, H_kv=8, d_h=128, W=4096+4 sinks, global prefix 131072",
                       "l2": f"inputs larger than L2 ({kv_bytes / 1e9:.1f} GB per step)",
                       "learned_sink_logits": bool(args.learned_sink)},
            "frac_of_hbm_peak": round(value / hbm, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
            "decode_step": {"ms_per_step": round(ms_fused, 4), "gbs": round(kv_bytes / (ms_fused * 1e-3) / 1e9, 2),
                            "calls": "sk_decode_step, two launches per layer, same state", "timing": rec_fused},
            "roofline": roof, "timing": rec,
            "peak_source": f"{peak_kind} hbm_gbs", "gpu_launches": rec["replays"] * steps * c["layers"] * 3,
            "clocks": clk}


def bench_rerotate(args, kdt):
    """Cached-key rerotation: 1 sequence, 48 layers, H_kv=4, d_h=128 with r=64,
    524288 cached positions, YaRN L0=262144, factor 1 <-> 2 (alternating so the keys
    stay well scaled); bf16 keys or int8 keys with one fp32 scale per row."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.REROTATE
    D, r, Hkv, N = c["D"], c["r"], c["Hkv"], c["positions"]
    nl = args.layers or c["layers"]   # fewer layers only for small profiling captures
    t0 = time.perf_counter()
    tA = sk.RopeTable(D, r, c["theta"], N, yarn_factor=c["factor_a"], yarn_orig_ctx=c["orig_ctx"])
    table_ms = (time.perf_counter() - t0) * 1e3
    tB = sk.RopeTable(D, r, c["theta"], N, yarn_factor=c["factor_b"], yarn_orig_ctx=c["orig_ctx"])
    t0 = time.perf_counter()
    tB.rebuild(c["factor_b"])
    rebuild_ms = (time.perf_counter() - t0) * 1e3
    kdtype = torch.bfloat16 if kdt == "bf16" else torch.int8
    layers = []
    for l in range(nl):
        L = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, Hkv, D, capacity=N, k_dtype=kdtype, with_v=False)
        L.pos.fill_(N)
        if kdt == "bf16":
            synth.fill_uniform_(L.k, 500 + l, -1.0, 1.0)
        else:
            L.k.copy_(synth.randint(L.k.shape, 600 + l, -127, 128, device="cuda").to(torch.int8))
            synth.fill_uniform_(L.k_scale, 700 + l, 1.0 / 127, 2.0 / 127)
        layers.append(L)

    def step(i):
        if i % 2 == 0:
            sk.kv_rerotate(layers, tA, tB)
        else:
            sk.kv_rerotate(layers, tB, tA)

    steps = args.steps + (args.steps % 2)     # an even number of turns: the keys come back
    ms, clk, rec = _timed(step, steps, args.warmup)
    rows = nl * Hkv * N
    alg = rows * (r * 2 * 2 if kdt == "bf16" else (D + 4) * 2)
    hbm, _, _, peak_kind = _peaks()
    value = alg / (ms * 1e-3) / 1e9
    assert all(L.error_bits() == 0 for L in layers)
    traffic = _traffic(f"rerotate_{kdt}_48l") if nl == 48 else None
    roof = {"bound": "hbm", "achieved": round(value, 2), "peak": hbm, "unit": "GB/s", "frac": round(value / hbm, 4),
            "traffic": traffic, "kernel": f"rerotate_{kdt}_kernel, one launch per step (all layers)",
            "algorithmic_bytes_per_launch": alg,
            "algorithmic_bytes": ("rows x r x 2 B, read and written (only the rotary half)" if kdt == "bf16" else
                                  "rows x (d_h codes + 4 B scale), read and written"),
            "launch_ms": round(ms, 5), "peak_source": f"{peak_kind} hbm_gbs"}
    return {"metric": f"cached-key rerotation ({kdt}) GB/s (frac of HBM peak), keys/s", "value": round(value, 2),
            "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "dtype": kdt, "data": "synthetic",
            "config": {"workload": f"{nl} layers x 4 kv heads x 524288 positions, d_h=128, r=64, YaRN 1<->2",
                       "algorithmic_bytes": alg, "l2": "inputs larger than L2"},
            "frac_of_hbm_peak": round(value / hbm, 4), "keys_per_s": round(rows / (ms * 1e-3), 1),
            "table_build_ms": round(table_ms, 1), "table_rebuild_ms": round(rebuild_ms, 1),
            "roofline": roof, "timing": rec,
            "peak_source": f"{peak_kind} hbm_gbs", "gpu_launches": rec["replays"] * steps, "clocks": clk}


def bench_rope(args):
    """Standalone RoPE (sk_rope_apply), as a chunk prefilled over a cached prefix uses it:
    the queries and keys of the prefill chunk (T=32768, H_q=32, H_kv=8, d_h=r=128,
    theta 5e5) rotated in place, one call for Q and one for K per step; positions
    p0 .. p0+T-1 with p0 = 32768."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.PREFILL
    T, Hq, Hkv, D = c["T"], c["Hq"], c["Hkv"], c["D"]
    p0 = 32768
    tbl = sk.RopeTable(D, c["r"], c["theta"], p0 + T)
    q = synth.normal((T, Hq, D), 31, torch.bfloat16, device="cuda")
    k = synth.normal((T, Hkv, D), 32, torch.bfloat16, device="cuda")
    posn = torch.arange(p0, p0 + T, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step(i):
        sk.rope_apply(tbl, q, posn, err=err)
        sk.rope_apply(tbl, k, posn, err=err)

    ms, clk, rec = _timed(step, args.steps, args.warmup)
    assert int(err.item()) == 0
    half = c["r"] // 2
    # rows read and written in place, plus each call's table rows (one per token)
    alg = 2 * T * (Hq + Hkv) * D * 2 + 2 * T * half * 8
    hbm, _, _, peak_kind = _peaks()
    value = alg / (ms * 1e-3) / 1e9
    return {"metric": "RoPE apply GB/s (frac of HBM peak), rows/s", "value": round(value, 2), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"Q and K of a {T}-token chunk at positions {p0}.. (H_q={Hq}, H_kv={Hkv}, "
                                   f"d_h=r={D}), rotated in place", "algorithmic_bytes": alg,
                       "l2": "inputs larger than L2"},
            "frac_of_hbm_peak": round(value / hbm, 4), "rows_per_s": round(T * (Hq + Hkv) / (ms * 1e-3), 1),
            "timing": rec, "peak_source": f"{peak_kind} hbm_gbs", "gpu_launches": 2 * args.steps * rec["replays"],
            "clocks": clk}


def bench_paged(args):
    """The windowed-layer decode step on a paged cache: B=32, H_q=32, H_kv=8,
    d_h=r=128, request sinks S=4, window W=4092, 16-token blocks scattered over a
    shared pool (only the sink block, the window's blocks and the blocks the timed
    steps will fill are allocated); one step = RoPE + paged append + paged split-K
    attention, the timed steps captured as one CUDA graph."""
    import numpy as np_
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W, bs = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"], 16
    steps, warm = args.steps, args.warmup
    n = 2 * steps + warm
    pos = synth.window_state(13, B, W, c["pos_lo"], c["pos_hi"])[0]
    end = pos + n + 1                                  # lengths after the last step
    max_blocks = int((int(end.max()) + bs - 1) // bs)
    needed = []
    for b in range(B):
        first = max(0, int(pos[b]) + 1 - W) // bs      # oldest block the first step's window reads
        last = (int(end[b]) - 1) // bs
        needed.append(sorted({0} | set(range(first, last + 1))))
    n_blocks = sum(len(x) for x in needed)
    layer = sk.PagedLayer.allocate(B, Hkv, D, block_size=bs, n_blocks=n_blocks, max_blocks=max_blocks,
                                   sinks=S, window=W)
    synth.fill_normal_(layer.k_pool, 11)
    synth.fill_normal_(layer.v_pool, 12)
    perm = np_.random.default_rng(17).permutation(n_blocks)
    table = np_.full((B, max_blocks), -1, dtype=np_.int32)
    k_ = 0
    for b in range(B):
        for j in needed[b]:
            table[b, j] = perm[k_]
            k_ += 1
    layer.block_table.copy_(torch.from_numpy(table))
    layer.seq_lens.copy_(pos)
    tbl = sk.RopeTable(D, c["r"], c["theta"], int(end.max()) + 64)
    qs = synth.normal((n, B, 1, Hq, D), 14, torch.bfloat16, device="cuda")
    ks = synth.normal((n, B, 1, Hkv, D), 15, torch.bfloat16, device="cuda")
    vs = synth.normal((n, B, 1, Hkv, D), 16, torch.bfloat16, device="cuda")
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(sk.paged_decode_workspace_bytes(layer, Hq), dtype=torch.uint8, device="cuda")
    zl = _learned_sinks(args, Hq)

    def step(i):
        sk.paged_append(tbl, layer, qs[i], ks[i], vs[i])
        sk.paged_decode_attention(layer, qs[i, :, 0], out=out, workspace=ws, sink_logits=zl)

    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    lens0 = layer.seq_lens.clone()

    def reset():  # the lengths put back: every replay appends the same tokens into the same blocks
        layer.seq_lens.copy_(lens0)

    ms, clk, rec = _timed(lambda i: step(warm + i), steps, 0, reset=reset)
    assert layer.error_bits() == 0
    L = S + W
    kv_bytes = B * Hkv * L * D * 2 * 2
    alg_decode = kv_bytes + 2 * (B * Hq * D * 2)
    hbm, _, _, peak_kind = _peaks()
    value = kv_bytes / (ms * 1e-3) / 1e9
    roof = _launch_roofline(lambda i: sk.paged_decode_attention(layer, qs[i, :, 0], out=out, workspace=ws,
                                                                sink_logits=zl), steps, alg_decode,
                            "decode_paged_window_b32_bs16",
                            "paged decode attention (split-K + combine); its launches back to back in one graph",
                            "K+V of 4096 visible rows x 32 sequences x 8 kv heads + q + out")
    return {"metric": METRIC + " (paged cache)", "value": round(value, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": steps, "warmup": warm, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "windowed-layer decode step on a paged cache (RoPE + paged append + paged "
                                   "split-K attention)", "batch": B, "H_q": Hq, "H_kv": Hkv, "d_h": D, "sinks": S,
                       "window": W, "block_size": bs, "pool_blocks": n_blocks,
                       "learned_sink_logits": bool(args.learned_sink),
                       "l2": f"inputs larger than L2 (KV {kv_bytes / 1e6:.0f} MB per step)"},
            "frac_of_hbm_peak": round(value / hbm, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
            "roofline": roof, "timing": rec,
            "gpu_launches": steps * 3 * rec["replays"], "clocks": clk}


def bench_window_i8(args):
    """The windowed-layer decode step on an int8 K cache: the same shapes as the default
    line (B=32, H_q=32, H_kv=8, d_h=r=128, S=4, W=4092, rings full at random heads);
    K rows are 128 int8 codes plus one fp32 scale, V and queries bf16.  One step = RoPE +
    append (K quantised per row) + split-K attention, the steps captured as one CUDA
    graph and replayed (ring counters put back after each replay)."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    steps, warm = args.steps, args.warmup
    n = steps + warm
    tbl = sk.RopeTable(D, c["r"], c["theta"], c["pos_hi"] + n + 64)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=torch.int8)
    layer.k.copy_(synth.randint(layer.k.shape, 11, -127, 128, device="cuda").to(torch.int8))
    synth.fill_uniform_(layer.k_scale, 12, 0.5 / 127, 2.0 / 127)
    synth.fill_normal_(layer.v, 13)
    pos, head, count = synth.window_state(13, B, W, c["pos_lo"], c["pos_hi"])
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    qs = synth.normal((n, B, 1, Hq, D), 14, torch.bfloat16, device="cuda")
    ks = synth.normal((n, B, 1, Hkv, D), 15, torch.bfloat16, device="cuda")
    vs = synth.normal((n, B, 1, Hkv, D), 16, torch.bfloat16, device="cuda")
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(sk.decode_workspace_bytes(layer, Hq), dtype=torch.uint8, device="cuda")
    zl = _learned_sinks(args, Hq)

    def step(i):
        sk.kv_append(tbl, layer, qs[i], ks[i], vs[i])
        sk.decode_attention(layer, qs[i, :, 0], out=out, workspace=ws, sink_logits=zl)

    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    ms, clk, rec = _timed(lambda i: step(warm + i), steps, 0, reset=_state_saver([layer]))
    assert layer.error_bits() == 0
    L = S + W
    kv_bytes = B * Hkv * L * (D + 4 + D * 2)     # int8 K row + its scale, bf16 V row
    alg_decode = kv_bytes + 2 * (B * Hq * D * 2)
    hbm, _, _, peak_kind = _peaks()
    value = kv_bytes / (ms * 1e-3) / 1e9
    roof = _launch_roofline(lambda i: sk.decode_attention(layer, qs[i, :, 0], out=out, workspace=ws,
                                                          sink_logits=zl), steps, alg_decode, "decode_window_b32_int8",
                            "decode attention over int8 keys (split-K + combine); its launches back to back in "
                            "one graph", "int8 K + fp32 scale + bf16 V of 4096 rows x 32 sequences x 8 kv heads "
                                         "+ q + out")
    return {"metric": METRIC + " (int8 K cache)", "value": round(value, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": steps, "warmup": warm, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "dtype": "bf16 q/v, int8 K + fp32 scale", "data": "synthetic",
            "config": {"workload": "windowed-layer decode step on an int8 K cache (RoPE + quantising append + "
                                   "split-K attention)", "batch": B, "H_q": Hq, "H_kv": Hkv, "d_h": D, "sinks": S,
                       "window": W, "learned_sink_logits": bool(args.learned_sink),
                       "l2": f"inputs larger than L2 (KV {kv_bytes / 1e6:.0f} MB per step)"},
            "frac_of_hbm_peak": round(value / hbm, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
            "roofline": roof, "timing": rec,
            "gpu_launches": steps * 3 * rec["replays"], "clocks": clk}


def bench_shift(args, kdt):
    """Local-position window slide: the recent keys of the windowed decode workload's
    cache (B=32, H_kv=8, d_h=r=128, S=4, W=4092, every ring full) turned by one
    position per step (alternately -1 and +1 so the keys stay put), sinks untouched.
    --layers N turns N such layers in one call (a model slides all its windowed layers
    at once); default 1."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hkv, D, r, S, W = c["B"], c["Hkv"], c["D"], c["r"], c["S"], c["W"]
    table = sk.RopeTable(D, r, c["theta"], 64)
    kdtype = torch.bfloat16 if kdt == "bf16" else torch.int8
    nl = args.layers or 1
    pos, head, count = synth.window_state(13, B, W, c["pos_lo"], c["pos_hi"])
    layers = []
    for l in range(nl):
        layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=kdtype, with_v=False)
        if kdt == "bf16":
            synth.fill_normal_(layer.k, 11 + 100 * l)
        else:
            layer.k.copy_(synth.randint(layer.k.shape, 11 + 100 * l, -127, 128, device="cuda").to(torch.int8))
            synth.fill_uniform_(layer.k_scale, 12 + 100 * l, 1.0 / 127, 2.0 / 127)
        layer.pos.copy_(pos)
        layer.head.copy_(head)
        layer.count.copy_(count)
        layers.append(layer)

    def step(i):
        sk.kv_shift_recent(layers, table, -1 if i % 2 == 0 else 1)

    steps = args.steps + (args.steps % 2)     # as many -1 as +1 turns per replay
    ms, clk, rec = _timed(step, steps, args.warmup)
    rows = nl * B * Hkv * W
    alg = rows * (r * 2 * 2 if kdt == "bf16" else (D + 4) * 2)
    hbm, _, _, peak_kind = _peaks()
    value = alg / (ms * 1e-3) / 1e9
    assert all(l.error_bits() == 0 for l in layers)
    return {"metric": f"recent-key shift ({kdt}) GB/s (frac of HBM peak)", "value": round(value, 2),
            "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "dtype": kdt, "data": "synthetic",
            "config": {"workload": f"windowed decode cache x {nl} layer(s): B=32, H_kv=8, d_h=r=128, S=4, "
                                   "W=4092, rings full; recent keys turned by one position", "layers": nl,
                       "algorithmic_bytes": alg, "l2": "inputs larger than L2" if alg > 129e6 else "fits L2"},
            "frac_of_hbm_peak": round(value / hbm, 4), "keys_per_s": round(rows / (ms * 1e-3), 1),
            "timing": rec, "peak_source": f"{peak_kind} hbm_gbs", "gpu_launches": steps * rec["replays"],
            "clocks": clk}


DYNAMIC_CHAIN = (1.125, 1.25, 1.5, 1.625, 1.75, 1.875, 2.0)


def bench_dynamic(args, kdt):
    """Dynamic YaRN switches on the rerotation workload (48 layers x 4 kv heads x
    524288 cached positions, L0 = 262144): one step drives a growing dialog through the
    seven switches 1 -> 1.125 -> 1.25 -> 1.5 -> 1.625 -> 1.75 -> 1.875 -> 2 and back
    to 1; each switch = host build of the new table + turning every cached key + the
    in-place table copy, timed on the host clock around the public call (which
    synchronises its stream)."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.REROTATE
    D, r, Hkv, N, L0 = c["D"], c["r"], c["Hkv"], c["positions"], c["orig_ctx"]
    nl = args.layers or c["layers"]
    dyn = sk.DynamicRope(D, r, c["theta"], N, L0, cap=2.0)
    kdtype = torch.bfloat16 if kdt == "bf16" else torch.int8
    layers = []
    for l in range(nl):
        L = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, Hkv, D, capacity=N, k_dtype=kdtype, with_v=False)
        L.pos.fill_(N)
        if kdt == "bf16":
            synth.fill_uniform_(L.k, 500 + l, -1.0, 1.0)
        else:
            L.k.copy_(synth.randint(L.k.shape, 600 + l, -127, 128, device="cuda").to(torch.int8))
            synth.fill_uniform_(L.k_scale, 700 + l, 1.0 / 127, 2.0 / 127)
        layers.append(L)
    lengths = [int(L0 * (f - 0.125)) + 1 for f in DYNAMIC_CHAIN]
    lengths[2] = int(L0 * 1.375) + 1            # the page's chain steps over 1.375
    targets = lengths + [L0]                    # ... and a dialog below L0 again

    def one_chain(times):
        for n in targets:
            t0 = time.perf_counter()
            f, switched = dyn.update(n, layers)
            times.append((time.perf_counter() - t0) * 1e3)
            assert switched

    for _ in range(max(1, args.warmup)):
        one_chain([])
    torch.cuda.synchronize()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    clocks.mark("start")
    times = []
    for _ in range(args.steps):
        one_chain(times)
    clocks.mark("end")
    clocks.stop()
    # the host table build alone, at the same size and thread count
    t0 = time.perf_counter()
    sk.rope_table_fill_host(D, r, c["theta"], N, yarn_factor=2.0, yarn_orig_ctx=L0)
    build_ms = (time.perf_counter() - t0) * 1e3
    assert all(L.error_bits() == 0 for L in layers)
    rows = nl * Hkv * N
    alg = rows * (r * 2 * 2 if kdt == "bf16" else (D + 4) * 2)
    ms = statistics.mean(times)
    return {"metric": f"dynamic YaRN switch ({kdt} keys): ms per switch (table build + key rotation)",
            "value": round(ms, 3), "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms * len(targets), 3), "higher_is_better": False, "dtype": kdt,
            "data": "synthetic",
            "config": {"workload": f"{nl} layers x 4 kv heads x 524288 positions, d_h=128, r=64, L0=262144; "
                                   "chain 1->1.125->1.25->1.5->1.625->1.75->1.875->2->1",
                       "switches_per_step": len(targets), "rotated_bytes_per_switch": alg},
            "switch_ms_min": round(min(times), 3), "switch_ms_max": round(max(times), 3),
            "table_build_ms": round(build_ms, 2), "keys_per_switch": rows,
            "gpu_launches": args.steps * len(targets), "clocks": clocks.summary()}


def _prefill_heads_per_cta(n_rep):
    """q heads of one GQA group packed into a prefill CTA: the largest power of two
    dividing n_rep, at most 8 (the library's choice)."""
    nh = 1
    while nh < 8 and n_rep % (2 * nh) == 0:
        nh *= 2
    return nh


PREFILL_SINK_STRIP = 16   # keys of the strip a sink tile below the window is visited as


def _prefill_tiles(T, S, W, n_rep, p0=0, qoff=0, BM=128, BN=64, strips=False):
    """(128-row x 64-key) tiles the prefill kernel visits per (sequence, group of nh q
    heads), and nh: the kernel's plan (blocks of BM / nh queries of nh heads; per block
    the sink tiles below the window, then the window's tiles).  qoff > 0: a chunk over
    a prior cache; its qoff keys come first, padded to a multiple of BN (the padding is
    never visible), then the chunk's keys.  strips=True also returns how many of those
    tiles are visited as a 16-key sink strip (a single sink tile below the window whose
    sinks fit in the strip)."""
    nh = _prefill_heads_per_cta(n_rep)
    qpb = BM // nh
    qpad = -(-qoff // BN) * BN
    Tk = T + qpad
    chunk_sinks = max(0, S - p0)
    if qoff > 0:
        nsk = min(S, p0)
        nskc = qpad + min(T, chunk_sinks)
        sink_end = nskc if chunk_sinks > 0 else nsk
    else:
        nsk = sink_end = min(T, chunk_sinks)
    n_total = n_strip = 0
    for q0 in range(0, T, qpb):
        q_last = min(q0 + qpb, T) - 1 + qpad
        win_lo = 0
        if W > 0:
            prior_lo = q0 + qoff - W + 1
            win_lo = max(0, prior_lo) if prior_lo < qoff else q0 + qpad - W + 1
        first, last = win_lo // BN, q_last // BN
        sink_keys = min(Tk, sink_end) if W > 0 else 0
        n_sink = min(first, (sink_keys + BN - 1) // BN)
        n_total += n_sink + (last - first + 1)
        n_strip += 1 if (n_sink == 1 and nsk <= PREFILL_SINK_STRIP) else 0
    return (n_total, nh, n_strip) if strips else (n_total, nh)


def bench_prefill(args):
    """Prefill chunk: B=1, T=32768, H_q=32, H_kv=8, d_h=r=128, bf16, S=4, W=4092: RoPE +
    ring append of the chunk, then masked attention of the chunk over itself.  The
    appends of a replay go into one fresh ring per captured step; the rings are
    emptied again after every replay."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.PREFILL
    B, T, Hq, Hkv, D, S, W = c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    steps, warm = args.steps, args.warmup
    tbl = sk.RopeTable(D, c["r"], c["theta"], T + 8)
    layers = [sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W) for _ in range(steps + warm)]
    q0 = synth.normal((B, T, Hq, D), 63, torch.bfloat16, device="cuda")
    k0 = synth.normal((B, T, Hkv, D), 64, torch.bfloat16, device="cuda")
    v = synth.normal((B, T, Hkv, D), 65, torch.bfloat16, device="cuda")
    q, k = q0.clone(), k0.clone()
    out = torch.empty_like(q)
    ws = torch.empty(sk.prefill_workspace_bytes(B, T, Hkv, D), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    zl = _learned_sinks(args, Hq)

    def append(i):
        sk.kv_append(tbl, layers[i], q, k, v)

    def attend(i):
        sk.prefill_attention(q, k, v, 0, S, W, out=out, workspace=ws, err=err, sink_logits=zl)

    empty = _state_saver(layers)            # every ring as allocated: empty
    ms_append, clk_a, rec_a = _timed(append, steps, warm, reset=empty)
    ms_attn, clk, rec = _timed(attend, steps, warm)
    assert int(err.item()) == 0 and all(L.error_bits() == 0 for L in layers)
    _, bf16_peak, bf16_sust, peak_kind = _peaks()
    hbm = _peaks()[0]
    vis_pairs = sum(min(t + 1, S + W) for t in range(T))      # (query, key) pairs per head
    alg_flops = vis_pairs * Hq * B * 4 * D
    tiles, nh, strips = _prefill_tiles(T, S, W, Hq // Hkv, strips=True)
    # visited tiles at 64 keys each, the sink strips at 16
    tile_keys = (tiles - strips) * 64 + strips * PREFILL_SINK_STRIP
    tile_flops = tile_keys * (Hq // nh) * B * 4 * 128 * D
    append_bytes = B * T * (Hq + 2 * Hkv) * D * 2 + B * T * (Hq + Hkv) * D * 2 + B * Hkv * (S + W) * D * 2 * 2
    tf = tile_flops / (ms_attn * 1e-3) / 1e12
    tf_alg = alg_flops / (ms_attn * 1e-3) / 1e12
    append_gbs = append_bytes / (ms_append * 1e-3) / 1e9
    # The peak: the sustained bf16 figure (a seconds-long matmul loop under the power cap)
    # when the clock record shows the power cap active over this region, else the burst
    # figure; both fractions are reported.
    capped = "sw_power_cap" in (clk.get("reasons") or []) and bool(bf16_sust)
    peak = bf16_sust if capped else bf16_peak
    roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(tf / peak, 4), "frac_burst": round(tf / bf16_peak, 4),
            "frac_sustained": round(tf / bf16_sust, 4) if bf16_sust else None,
            "traffic": _traffic("prefill_attn_t32768"),
            "kernel": "prefill_attn_kernel (tcgen05, one launch per step)",
            "flops_per_launch": tile_flops, "flops": "4 d_h x 128 x 64 per visited (128-row, 64-key) tile and "
                                                     "group of q heads (the tiles the mask does not rule out), "
                                                     "x 16 for a sink strip",
            "algorithmic": {"achieved": round(tf_alg, 1), "frac": round(tf_alg / peak, 4),
                            "flops_per_launch": alg_flops,
                            "flops": "4 d_h per visible (query, key) pair and q head"},
            "launch_ms": round(ms_attn, 5),
            "peak_source": (f"{peak_kind} bf16_tflops_sustained: the region ran under the power cap" if capped
                            else f"{peak_kind} bf16_tflops (burst)")}
    append_roof = {"bound": "hbm", "achieved": round(append_gbs, 1), "peak": hbm, "unit": "GB/s",
                   "frac": round(append_gbs / hbm, 4), "traffic": None,
                   "kernel": "kv_append_kernel (RoPE on Q and K + ring write of the chunk's last W rows)",
                   "algorithmic_bytes_per_launch": append_bytes,
                   "algorithmic_bytes": "read Q, K, V + write Q_rot, K_rot + write the ring's S + W rows of K and V",
                   "launch_ms": round(ms_append, 5), "peak_source": f"{peak_kind} hbm_gbs"}
    return {"metric": "prefill attention TFLOP/s on visited tiles (frac of dense bf16 peak); append GB/s",
            "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": steps, "warmup": warm,
            "ms_per_step": round(ms_attn, 4), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "prefill chunk: B=1, T=32768, H_q=32, H_kv=8, d_h=128, S=4, W=4092",
                       "l2": "inputs larger than L2 (Q, K, V 403 MB per call)",
                       "visited_tiles_per_head_group": tiles, "sink_strips_per_head_group": strips,
                       "heads_per_cta": nh,
                       "tile": f"128 rows ({nh} heads x {128 // nh} queries) x 64 keys",
                       "learned_sink_logits": bool(args.learned_sink)},
            "frac_of_bf16_peak": round(tf / peak, 4),
            "algorithmic_tflops": round(tf_alg, 1), "algorithmic_frac_of_bf16_peak": round(tf_alg / peak, 4),
            "algorithmic_flops": alg_flops, "tile_flops": tile_flops,
            "append_ms": round(ms_append, 4), "append_gbs": round(append_gbs, 1),
            "append_frac_of_hbm_peak": round(append_gbs / hbm, 4),
            "roofline": roof, "append_roofline": append_roof, "timing": rec, "append_timing": rec_a,
            "peak_source": f"{peak_kind} bf16_tflops {bf16_peak} / hbm_gbs {hbm}",
            "gpu_launches": steps * rec["replays"], "clocks": clk, "append_clocks": clk_a}


def bench_prefill_chunk(args):
    """A later chunk of a long prompt: B=1, T=8192 new tokens at p0=32768 attending over
    the full, wrapped ring a first chunk left (S=4, W=4092) and over themselves;
    H_q=32, H_kv=8, d_h=128, bf16.  One step = the gather of the prior's keys and
    values and the attention (sk_prefill_attention with a prior), which reads the chunk's
    own keys and values in place."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.PREFILL
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    T, p0 = 8192, 32768
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 66)
    synth.fill_normal_(layer.v, 67)
    layer.pos.fill_(p0)
    layer.count.fill_(W)
    layer.head.fill_(1234)
    # three sets of chunk inputs and outputs in rotation (168 MB each): a call's inputs
    # have left L2 by the time they come round again
    n_sets = 3
    qs = [synth.normal((B, T, Hq, D), 68 + 10 * j, torch.bfloat16, device="cuda") for j in range(n_sets)]
    ks = [synth.normal((B, T, Hkv, D), 69 + 10 * j, torch.bfloat16, device="cuda") for j in range(n_sets)]
    vs = [synth.normal((B, T, Hkv, D), 70 + 10 * j, torch.bfloat16, device="cuda") for j in range(n_sets)]
    outs = [torch.empty_like(qs[0]) for _ in range(n_sets)]
    qoff = sk.prefill_prior_keys(p0, S, W)
    ws = torch.empty(sk.prefill_workspace_bytes(B, T, Hkv, D, qoff), dtype=torch.uint8, device="cuda")
    zl = _learned_sinks(args, Hq)

    def attend(i):
        j = i % n_sets
        sk.prefill_attention(qs[j], ks[j], vs[j], p0, S, W, out=outs[j], workspace=ws, err=layer.err,
                             sink_logits=zl, prior=layer)

    ms, clk, rec = _timed(attend, args.steps, args.warmup)
    assert layer.error_bits() == 0
    _, bf16_peak, _, peak_kind = _peaks()
    alg_flops = T * (S + W) * Hq * B * 4 * D          # every query sees S + W keys here
    tiles, nh, strips = _prefill_tiles(T, S, W, Hq // Hkv, p0=p0, qoff=qoff, strips=True)
    tile_keys = (tiles - strips) * 64 + strips * PREFILL_SINK_STRIP
    tile_flops = tile_keys * (Hq // nh) * B * 4 * 128 * D
    tf = tile_flops / (ms * 1e-3) / 1e12
    return {"metric": "chunked prefill attention over a prior ring, TFLOP/s on visited tiles (frac of dense bf16 "
                      "peak)",
            "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "prompt chunk over a prior ring: B=1, T=8192 at p0=32768, H_q=32, H_kv=8, "
                                   "d_h=128, S=4, W=4092 (ring full, wrapped)",
                       "l2": "inputs larger than L2: three sets of q, k, v and out (168 MB each) in rotation",
                       "prior_keys": qoff, "visited_tiles_per_head_group": tiles, "heads_per_cta": nh,
                       "learned_sink_logits": bool(args.learned_sink)},
            "frac_of_bf16_peak": round(tf / bf16_peak, 4),
            "algorithmic_tflops": round(alg_flops / (ms * 1e-3) / 1e12, 1),
            "algorithmic_flops": alg_flops, "tile_flops": tile_flops,
            "peak_source": f"{peak_kind} bf16_tflops {bf16_peak}", "timing": rec,
            "gpu_launches": args.steps * 2 * rec["replays"], "clocks": clk}


# ---------------------------------------------------------------------------
# the configurations beside the headline: the tiny case and single-stream decode
# ---------------------------------------------------------------------------

def bench_tiny(args):
    """The tiny case: 1 sequence, H_q=8, H_kv=4, d_h=r=64, theta=1e4, fp32, C=6 with S=2
    sinks, 10 tokens decoded one at a time (RoPE + append + attention per token, as the
    decode step sk_decode_step; sk_kv_append + sk_decode_attention timed beside it).  A
    replay of the captured graph decodes the 10 tokens; the ring is emptied after it."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.TINY
    T, Hq, Hkv, D = c["T"], c["Hq"], c["Hkv"], c["D"]
    tbl = sk.RopeTable(D, c["r"], c["theta"], 64)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, Hkv, D, sinks=c["S"], window=c["W"], k_dtype=torch.float32,
                                v_dtype=torch.float32)
    q_all = synth.normal((1, T, Hq, D), 0)
    k_all = synth.normal((1, T, Hkv, D), 1)
    v_all = synth.normal((1, T, Hkv, D), 2)
    qs = [q_all[:, t:t + 1].contiguous().cuda() for t in range(T)]
    ks = [k_all[:, t:t + 1].contiguous().cuda() for t in range(T)]
    vs = [v_all[:, t:t + 1].contiguous().cuda() for t in range(T)]
    out = torch.empty(1, Hq, D, device="cuda")
    ws = torch.empty(max(sk.decode_workspace_bytes(layer, Hq), sk.decode_step_workspace_bytes(layer, Hq)),
                     dtype=torch.uint8, device="cuda")
    empty = _state_saver([layer])

    def step(t):  # q, k, v are read only
        sk.decode_step(tbl, layer, qs[t % T][:, 0], ks[t % T][:, 0], vs[t % T][:, 0], out=out, workspace=ws)

    def step_two_calls(t):  # rotates q and k in place
        sk.kv_append(tbl, layer, qs[t % T], ks[t % T], vs[t % T])
        sk.decode_attention(layer, qs[t % T][:, 0], out=out, workspace=ws)

    for t in range(T):
        step(t)
    torch.cuda.synchronize()
    empty()

    # Each timed step starts with L2 flushed: a 512 MB buffer rewritten (longer than the host needs
    # to queue the step behind it, so the step's launches run back to back) precedes the
    # step, outside its events; the ring is emptied after every T steps, also outside.
    flush = torch.empty(128 * 1024 * 1024, dtype=torch.float32, device="cuda")

    def flushed(fn, n_iter):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_iter)]
        for it in range(n_iter):
            if it % T == 0:
                empty()
            flush.add_(1.0)
            ev[it][0].record()
            fn(it % T)
            ev[it][1].record()
        torch.cuda.synchronize()
        empty()
        return [a.elapsed_time(b) for a, b in ev]

    flushed(step, 2 * T)  # warm-up
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    clocks.mark("start")
    per = flushed(step, 120 * T)  # synchronizes before it returns
    clocks.mark("end")
    wall = time.perf_counter() - t0
    clocks.stop()
    assert layer.error_bits() == 0
    us = statistics.median(per) * 1e3
    per2 = flushed(step_two_calls, 30 * T)
    assert layer.error_bits() == 0
    # beside it: the same steps back to back in one captured graph, L2 warm
    g = _capture(step, 0, T)
    per_w, _, _ = _replays(g, T, TARGET_MS / 6, reset=empty)
    assert layer.error_bits() == 0
    return {"metric": "tiny case: microseconds per decode step (RoPE + append + attention of one token)",
            "value": round(us, 3), "unit": "us/step", "higher_is_better": False, "dtype": "f32",
            "config": {"workload": "tiny: 1 sequence, H_q=8, H_kv=4, d_h=r=64, theta=1e4, fp32, C=6, S=2, "
                                   "10 tokens one at a time",
                       "l2": "flushed before every timed step (a 512 MB buffer rewritten between steps, outside "
                             "the events)"},
            "roofline": {"bound": "latency", "achieved": round(us, 3), "unit": "us/step", "peak": None,
                         "frac": None, "kernel": "split (with the token's RoPE + append) + combine per token "
                                                 "(2 launches)",
                         "note": "a parity case: 3 KB of cache, far from any throughput roofline"},
            "timing": {"steps_timed": len(per), "us_per_step": "median of per-step CUDA events",
                       "us_per_step_min": round(min(per) * 1e3, 3), "wall_s": round(wall, 2)},
            "two_calls": {"us_per_step": round(statistics.median(per2) * 1e3, 3),
                          "calls": "sk_kv_append + sk_decode_attention, three launches per token"},
            "warm_graph": {"us_per_step": round(statistics.median(per_w) * 1e3, 3),
                           "how": "the 10 steps back to back in one captured graph, replayed, L2 warm"},
            "gpu_launches": 2 * len(per), "clocks": clocks.summary()}


def bench_window_step(args):
    """The windowed decode step (B=32, H_q=32, H_kv=8, d_h=r=128, S=4, W=4092, rings full at
    random heads) through sk_decode_step: the token's RoPE + append folded into the split
    kernel, two launches per step; sk_kv_append + sk_decode_attention (the headline's
    calls) timed beside it on the same state.  Roofline: the step's launches back to back
    (split with the token, combine), the counters put back after every replay."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    steps, warm = args.steps, args.warmup
    tbl, layer, c = window_setup(seed_base=0, steps=2 * steps + warm + 2)
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    n = steps + warm
    qs = synth.normal((n, B, 1, Hq, D), 14, torch.bfloat16, device="cuda")
    ks = synth.normal((n, B, 1, Hkv, D), 15, torch.bfloat16, device="cuda")
    vs = synth.normal((n, B, 1, Hkv, D), 16, torch.bfloat16, device="cuda")
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(sk.decode_workspace_bytes(layer, Hq), sk.decode_step_workspace_bytes(layer, Hq)),
                     dtype=torch.uint8, device="cuda")

    def step(i):  # q, k, v are read only
        sk.decode_step(tbl, layer, qs[i, :, 0], ks[i, :, 0], vs[i, :, 0], out=out, workspace=ws)

    def step_two_calls(i):  # rotates q and k in place
        sk.kv_append(tbl, layer, qs[i], ks[i], vs[i])
        sk.decode_attention(layer, qs[i, :, 0], out=out, workspace=ws)

    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    reset = _state_saver([layer])
    ms, clk, rec = _timed(lambda i: step(warm + i), steps, 0, reset=reset)
    assert layer.error_bits() == 0
    kv_bytes = B * Hkv * (S + W) * D * 2 * 2
    hbm, _, _, peak_kind = _peaks()
    value = kv_bytes / (ms * 1e-3) / 1e9
    alg = kv_bytes + 2 * B * Hq * D * 2 + 4 * B * Hkv * D * 2
    roof = _launch_roofline(lambda i: step(i % n), steps, alg, "decode_step_window_b32",
                            "decode step (split-K with the token's RoPE + append, combine); its launches back "
                            "to back in one graph",
                            "K+V of 4096 visible rows x 32 sequences x 8 kv heads + q + out + the token's k, v "
                            "in and out", reset=reset)
    reset()
    ms_two, _, rec_two = _timed(lambda i: step_two_calls(warm + i), steps, 0, reset=reset)
    assert layer.error_bits() == 0
    return {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
            "higher_is_better": True, "dtype": "bf16",
            "config": {"workload": "windowed-layer decode step (RoPE + append + split-K attention) through "
                                   "sk_decode_step, B=32, H_q=32, H_kv=8, d_h=r=128, S=4, W=4092",
                       "l2": f"inputs larger than L2 (KV {kv_bytes / 1e6:.0f} MB per step)"},
            "frac_of_hbm_peak": round(value / hbm, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
            "two_calls": {"ms_per_step": round(ms_two, 5), "gbs": round(kv_bytes / (ms_two * 1e-3) / 1e9, 2),
                          "calls": "sk_kv_append + sk_decode_attention (the headline's), same state",
                          "timing": rec_two},
            "roofline": roof, "timing": rec, "peak_source": f"{peak_kind} hbm_gbs",
            "gpu_launches": 2 * steps * rec["replays"], "clocks": clk}


def bench_window_b1(args):
    """Single-stream decode: one sequence through 32 windowed layers (each H_q=32,
    H_kv=8, d_h=r=128, S=4, W=4092, ring full at a random head), one token per step:
    RoPE + append + split-K attention over 4096 visible keys on every layer, as the
    decode step (sk_decode_step: the append folded into the attention's two kernels).
    The same steps as sk_kv_append + sk_decode_attention (three launches per layer) are
    timed beside it on the same state.  The 32 layers' caches (537 MB) exceed L2, as a
    model's layers do."""
    import torch
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    Hq, Hkv, D, S, W = c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    nl = 32
    steps, warm = args.steps, args.warmup
    tbl = sk.RopeTable(D, c["r"], c["theta"], c["pos_hi"] + steps + warm + 8)
    pos, head, count = synth.window_state(43, nl, W, c["pos_lo"], c["pos_hi"])
    layers = []
    for j in range(nl):
        L = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, Hkv, D, sinks=S, window=W)
        synth.fill_normal_(L.k, 4100 + j)
        synth.fill_normal_(L.v, 4200 + j)
        L.pos.fill_(int(pos[0]))
        L.head.fill_(int(head[j]))
        L.count.fill_(W)
        layers.append(L)
    n = steps + warm
    qs = synth.normal((n, nl, 1, 1, Hq, D), 44, torch.bfloat16, device="cuda")
    ks = synth.normal((n, nl, 1, 1, Hkv, D), 45, torch.bfloat16, device="cuda")
    vs = synth.normal((n, nl, 1, 1, Hkv, D), 46, torch.bfloat16, device="cuda")
    out = torch.empty(1, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(sk.decode_workspace_bytes(layers[0], Hq), sk.decode_step_workspace_bytes(layers[0], Hq)),
                     dtype=torch.uint8, device="cuda")
    reset = _state_saver(layers)

    def step(i):  # q, k, v are read only
        for j, L in enumerate(layers):
            sk.decode_step(tbl, L, qs[i, j, :, 0], ks[i, j, :, 0], vs[i, j, :, 0], out=out, workspace=ws)

    def step_two_calls(i):  # rotates q and k in place
        for j, L in enumerate(layers):
            sk.kv_append(tbl, L, qs[i, j], ks[i, j], vs[i, j])
            sk.decode_attention(L, qs[i, j, :, 0], out=out, workspace=ws)

    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    ms, clk, rec = _timed(lambda i: step(warm + i), steps, 0, reset=reset)
    assert all(L.error_bits() == 0 for L in layers)
    kv_layer = Hkv * (S + W) * D * 2 * 2
    hbm, _, _, peak_kind = _peaks()
    value = nl * kv_layer / (ms * 1e-3) / 1e9
    tok_bytes = 4 * Hkv * D * 2  # the token's k and v read, then written to the cache
    roof = _launch_roofline(lambda i: sk.decode_step(tbl, layers[i % nl], qs[0, i % nl, :, 0], ks[0, i % nl, :, 0],
                                                     vs[0, i % nl, :, 0], out=out, workspace=ws), nl,
                            kv_layer + 2 * Hq * D * 2 + tok_bytes, None,
                            "decode step at batch 1 (split-K with the token's RoPE + append, combine); the 32 "
                            "layers' launches back to back in one graph",
                            "K+V of 4096 visible rows x 8 kv heads + q + out + the token's k, v in and out, "
                            "per layer", reset=reset)
    reset()
    ms_two, _, rec_two = _timed(lambda i: step_two_calls(warm + i), steps, 0, reset=reset)
    assert all(L.error_bits() == 0 for L in layers)
    return {"metric": "single-stream decode over 32 windowed layers: us per token, tokens/s, KV-read GB/s",
            "value": round(ms * 1e3, 2), "unit": "us/token", "higher_is_better": False, "dtype": "bf16",
            "config": {"workload": "batch 1 through 32 windowed layers (H_q=32, H_kv=8, d_h=r=128, S=4, W=4092, "
                                   "rings full): RoPE + append + attention per layer (sk_decode_step)",
                       "l2": f"inputs larger than L2 (KV {nl * kv_layer / 1e6:.0f} MB per step)"},
            "tokens_per_s": round(1.0 / (ms * 1e-3), 1), "gbs": round(value, 2),
            "frac_of_hbm_peak": round(value / hbm, 4), "us_per_layer": round(ms * 1e3 / nl, 3),
            "two_calls": {"us_per_token": round(ms_two * 1e3, 2), "calls": "sk_kv_append + sk_decode_attention, "
                          "three launches per layer, same state", "timing": rec_two},
            "roofline": roof, "timing": rec, "gpu_launches": 2 * nl * steps * rec["replays"], "clocks": clk}


# ---------------------------------------------------------------------------
# CPU oracle baseline (single thread, in a subprocess)
# ---------------------------------------------------------------------------

def cpu_oracle_window(n_seq: int, seed_base: int = 0, first: int = 0):
    """Time the float64 oracle on sequences first .. first + n_seq - 1 of the windowed
    decode step (RoPE + append + attention) and return (seconds, kv_bytes)."""
    import numpy as np
    import torch
    from oracle.sinkkv_oracle import RingCache, RopeSpec, decode_attention, rope_rotate
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    pos, head, count = synth.window_state(13 + seed_base, B, W, c["pos_lo"], c["pos_hi"])
    spec = RopeSpec(D, c["r"], c["theta"])
    omega = spec.omega()
    total = 0.0
    for b in range(first, first + n_seq):
        kb = synth.normal((Hkv, S + W, D), 1000 + b, torch.bfloat16).double().numpy()
        vb = synth.normal((Hkv, S + W, D), 2000 + b, torch.bfloat16).double().numpy()
        q = synth.normal((1, Hq, D), 3000 + b, torch.bfloat16).double().numpy()
        k = synth.normal((1, Hkv, D), 4000 + b, torch.bfloat16).double().numpy()
        v = synth.normal((Hkv, D), 5000 + b, torch.bfloat16).double().numpy()
        t0 = time.perf_counter()
        ring = RingCache(S, W)
        ring.pos, ring.head, ring.count = int(pos[b]), int(head[b]), int(count[b])
        for s in range(S + W):
            ring.slots[s] = (kb[:, s], vb[:, s])
        P = int(pos[b])
        qr = rope_rotate(q, [P], omega, 1.0, D)
        kr = rope_rotate(k, [P], omega, 1.0, D)
        ring.append([(kr[0], v)])
        decode_attention(ring, qr[0])
        total += time.perf_counter() - t0
    return total, n_seq * Hkv * (S + W) * D * 2 * 2


CPU_SAMPLE_SECS = 10.0   # CPU work the oracle baselines aim for
CPU_SAMPLE_REPS = 12      # steps of the all-cores sample (about 10 s of CPU work on a Neoverse-V2)


def _cpu_worker(n_seq):
    """Whole steps (n_seq sequences each, fresh inputs per step) until about
    CPU_SAMPLE_SECS of oracle time, at most 24 steps."""
    secs, kv, reps = 0.0, 0, 0
    while reps < 24 and (reps == 0 or secs < CPU_SAMPLE_SECS):
        s, b = cpu_oracle_window(n_seq, seed_base=reps)
        secs, kv, reps = secs + s, kv + b, reps + 1
    print(json.dumps({"secs": secs, "kv_bytes": kv, "steps": reps}))


def _cpu_model():
    """The host CPU's name from /proc/cpuinfo (Arm cores report implementer and part)."""
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    arm_parts = {("0x41", "0xd4f"): "Arm Neoverse-V2", ("0x41", "0xd40"): "Arm Neoverse-V1",
                 ("0x41", "0xd0c"): "Arm Neoverse-N1", ("0x41", "0xd49"): "Arm Neoverse-N2"}
    key = (fields.get("cpu implementer", ""), fields.get("cpu part", ""))
    if key in arm_parts:
        return arm_parts[key]
    import platform
    return f"{platform.machine()} implementer {key[0]} part {key[1]}".strip()


def _cpu_mt_part(args):
    """One process of the all-cores oracle run: sequences [lo, hi) of every sampled step."""
    lo, hi, reps = args
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    secs = 0.0
    for rep in range(reps):
        for b in range(lo, hi):
            secs += cpu_oracle_window_one(b, rep)
    return secs


def cpu_oracle_window_one(b: int, seed_base: int = 0) -> float:
    """Oracle seconds for sequence b of the windowed decode step."""
    return cpu_oracle_window(1, seed_base=seed_base, first=b)[0]


def _cpu_worker_mt(n_seq):
    import multiprocessing as mp
    n = os.cpu_count() or 1
    parts = [(n_seq * i // n, n_seq * (i + 1) // n, CPU_SAMPLE_REPS) for i in range(n)]
    parts = [x for x in parts if x[1] > x[0]]
    with mp.get_context("spawn").Pool(len(parts)) as pool:
        secs = pool.map(_cpu_mt_part, parts)
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    kv = CPU_SAMPLE_REPS * n_seq * c["Hkv"] * (c["S"] + c["W"]) * c["D"] * 2 * 2
    print(json.dumps({"secs": max(secs), "cpu_secs": sum(secs), "kv_bytes": kv, "procs": len(parts),
                      "steps": CPU_SAMPLE_REPS}))


def cpu_baseline_all_cores(n_seq=32):
    """The same oracle sample spread over every host core (one process per core): the
    parallel time is the slowest process's oracle time."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker-mt", str(n_seq)],
                       capture_output=True, text=True, env=env, timeout=600)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    gbs = d["kv_bytes"] / d["secs"] / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": d["procs"], "kind": "oracle",
            "cpu": _cpu_model(),
            "sample": f"{d['steps']} windowed decode steps of {n_seq} sequences over {d['procs']} processes "
                      f"(float64 numpy, one thread each, {d['cpu_secs']:.1f} s of CPU work, slowest "
                      f"process {d['secs']:.2f} s)"}


# ---------------------------------------------------------------------------
# oracle baselines of the other configurations (float64 numpy, single thread, in a
# subprocess); where the whole configuration would take minutes, a bounded sample is
# timed and the configuration's time extrapolated from it (said so in "sample")
# ---------------------------------------------------------------------------

def _cpu_tiny():
    import numpy as np
    from oracle.sinkkv_oracle import RingCache, RopeSpec, decode_attention, rope_rotate
    from sink_kv_attention_gb300 import synth
    c = synth.TINY
    T, D = c["T"], c["D"]
    om = RopeSpec(D, c["r"], c["theta"]).omega()
    q = synth.normal((T, c["Hq"], D), 0).double().numpy()
    k = synth.normal((T, c["Hkv"], D), 1).double().numpy()
    v = synth.normal((T, c["Hkv"], D), 2).double().numpy()
    secs, steps = 0.0, 0
    while secs < 2.0:
        t0 = time.perf_counter()
        ring = RingCache(c["S"], c["W"])
        for t in range(T):
            qr = rope_rotate(q[t:t + 1], [t], om, 1.0, c["r"])
            kr = rope_rotate(k[t:t + 1], [t], om, 1.0, c["r"])
            ring.append([(kr[0], v[t])])
            decode_attention(ring, qr[0])
        secs += time.perf_counter() - t0
        steps += T
    return {"value": round(secs / steps * 1e6, 2), "unit": "us/step",
            "sample": f"the whole case, {steps // T} times ({steps} decode steps, {secs:.2f} s)"}


def _cpu_window_b1():
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    secs, reps = 0.0, 0
    while secs < 5.0:
        s_, _ = cpu_oracle_window(1, seed_base=reps)
        secs, reps = secs + s_, reps + 1
    per_layer = secs / reps
    kv = c["Hkv"] * (c["S"] + c["W"]) * c["D"] * 2 * 2
    return {"value": round(per_layer * 32 * 1e6, 1), "unit": "us/token", "gbs": round(kv / per_layer / 1e9, 4),
            "sample": f"{reps} single-sequence windowed decode steps of one layer ({secs:.2f} s), x 32 layers "
                      "(extrapolated)"}


def _cpu_hybrid():
    import numpy as np
    from oracle.sinkkv_oracle import GlobalCache, RingCache, RopeSpec, decode_attention, rope_rotate
    from sink_kv_attention_gb300 import synth
    c = synth.HYBRID
    B, Hq, Hkv, D, S, W, prefix = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"], c["prefix"]
    om = RopeSpec(D, c["r"], c["theta"]).omega()
    t_glob, t_slid = [], []
    for b, kind in [(0, "g"), (1, "g")] + [(b, "s") for b in range(8)]:
        n = prefix if kind == "g" else S + W
        kb = synth.normal((n, Hkv, D), 7000 + b, torch_dtype()).double().numpy()
        vb = synth.normal((n, Hkv, D), 7100 + b, torch_dtype()).double().numpy()
        q = synth.normal((1, Hq, D), 7200 + b, torch_dtype()).double().numpy()
        k = synth.normal((1, Hkv, D), 7300 + b, torch_dtype()).double().numpy()
        v = synth.normal((Hkv, D), 7400 + b, torch_dtype()).double().numpy()
        t0 = time.perf_counter()
        if kind == "g":
            cache = GlobalCache(prefix + 1)
            cache.append([(kb[s], vb[s]) for s in range(prefix)])
        else:
            cache = RingCache(S, W)
            cache.pos, cache.head, cache.count = prefix, (97 * b) % W, W
            for s in range(S + W):
                cache.slots[s] = (kb[s], vb[s])
        qr = rope_rotate(q, [prefix], om, 1.0, D)
        kr = rope_rotate(k, [prefix], om, 1.0, D)
        cache.append([(kr[0], v)])
        decode_attention(cache, qr[0])
        (t_glob if kind == "g" else t_slid).append(time.perf_counter() - t0)
    tg, ts = sum(t_glob) / len(t_glob), sum(t_slid) / len(t_slid)
    step_s = B * (8 * tg + 24 * ts)
    kv = (8 * (prefix + 1) + 24 * (S + W)) * B * Hkv * D * 2 * 2
    return {"value": round(kv / step_s / 1e9, 4), "unit": "GB/s", "ms_per_step": round(step_s * 1e3, 1),
            "sample": f"one global layer for {len(t_glob)} sequences ({sum(t_glob):.2f} s) and one sliding layer "
                      f"for {len(t_slid)} sequences ({sum(t_slid):.2f} s); the 32-layer, 16-sequence step "
                      "extrapolated as 16 x (8 global + 24 sliding)"}


def torch_dtype():
    import torch
    return torch.bfloat16


def _cpu_prefill():
    import numpy as np
    from oracle.sinkkv_oracle import prefill_attention
    from sink_kv_attention_gb300 import synth
    c = synth.PREFILL
    T, Hq, Hkv, D, S, W = c["T"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    q = synth.normal((T, Hq, D), 63, torch_dtype()).double().numpy()
    k = synth.normal((T, Hkv, D), 64, torch_dtype()).double().numpy()
    v = synth.normal((T, Hkv, D), 65, torch_dtype()).double().numpy()
    rows = sorted(np.random.default_rng(5).choice(T, 256, replace=False).tolist())
    t0 = time.perf_counter()
    prefill_attention(q, k, v, 0, S, W, rows=rows)
    secs = time.perf_counter() - t0
    pairs = lambda ts: sum(min(t + 1, S + W) for t in ts)
    full_s = secs * pairs(range(T)) / pairs(rows)
    flops = pairs(range(T)) * Hq * 4 * D
    return {"value": round(flops / full_s / 1e12, 6), "unit": "TFLOP/s", "ms_per_step": round(full_s * 1e3, 1),
            "sample": f"256 sampled query rows, all 32 heads ({secs:.2f} s); the chunk's time extrapolated by "
                      "its visible (query, key) pairs"}


def _cpu_rerotate(kdt):
    import numpy as np
    from oracle.sinkkv_oracle import RopeSpec, rerotate, rerotate_int8
    c = synth_cfg("REROTATE")
    D, r, Hkv, N = c["D"], c["r"], c["Hkv"], c["positions"]
    a = RopeSpec(D, r, c["theta"], True, c["factor_a"], c["orig_ctx"])
    b = a.with_factor(c["factor_b"])
    rng = np.random.default_rng(6)
    secs, rows = 0.0, 0
    while secs < 6.0:
        pos = rng.integers(0, N, 16384)
        if kdt == "bf16":
            x = rng.uniform(-1, 1, (len(pos), Hkv, D))
            t0 = time.perf_counter()
            rerotate(x, pos, a, b)
        else:
            codes = rng.integers(-127, 128, (len(pos), Hkv, D)).astype(np.int8)
            sc = rng.uniform(1 / 127, 2 / 127, (len(pos), Hkv))
            t0 = time.perf_counter()
            rerotate_int8(codes, sc, pos, a, b)
        secs += time.perf_counter() - t0
        rows += len(pos) * Hkv
    per_row = r * 2 * 2 if kdt == "bf16" else (D + 4) * 2
    total_rows = c["layers"] * Hkv * N
    return {"value": round(rows * per_row / secs / 1e9, 4), "unit": "GB/s",
            "ms_per_step": round(secs / rows * total_rows * 1e3, 1),
            "sample": f"{rows} key rows at random positions ({secs:.2f} s); the 48-layer step "
                      f"({total_rows} rows) extrapolated by the row count"}


CPU_ROW_SECS = 5.0  # oracle time of the single-sequence samples below


def _cpu_window_step():
    """The decode step's arithmetic is the windowed line's (RoPE + append + attention):
    single sequences of that workload, about 5 s of oracle time."""
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    secs, n = 0.0, 0
    while n == 0 or secs < CPU_ROW_SECS:
        s_, _ = cpu_oracle_window(1, seed_base=0, first=n % c["B"])
        secs, n = secs + s_, n + 1
    kv = c["Hkv"] * (c["S"] + c["W"]) * c["D"] * 2 * 2
    return {"value": round(n * kv / secs / 1e9, 4), "unit": "GB/s",
            "ms_per_step": round(secs / n * c["B"] * 1e3, 1),
            "sample": f"{n} single-sequence windowed decode steps ({secs:.2f} s); the {c['B']}-sequence step "
                      "extrapolated by the sequence count"}


def _cpu_window_i8():
    """The windowed step over int8 keys: the cached codes dequantized (code x row
    scale), the new key rotated and quantized by the int8 rule, then attention over the
    dequantized keys; single sequences, about 5 s of oracle time."""
    import numpy as np
    from oracle.sinkkv_oracle import (RingCache, RopeSpec, decode_attention, dequantize_int8_rows,
                                      quantize_int8_rows, rope_rotate)
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    pos, head, count = synth.window_state(13, B, W, c["pos_lo"], c["pos_hi"])
    om = RopeSpec(D, c["r"], c["theta"]).omega()
    rng = np.random.default_rng(8)
    secs, n = 0.0, 0
    while n == 0 or secs < CPU_ROW_SECS:
        b = n % B
        codes = rng.integers(-127, 128, (Hkv, S + W, D)).astype(np.int8)
        scale = rng.uniform(0.5 / 127, 2.0 / 127, (Hkv, S + W))
        vb = synth.normal((Hkv, S + W, D), 2000 + b, torch_dtype()).double().numpy()
        q = synth.normal((1, Hq, D), 3000 + b, torch_dtype()).double().numpy()
        k = synth.normal((1, Hkv, D), 4000 + b, torch_dtype()).double().numpy()
        v = synth.normal((Hkv, D), 5000 + b, torch_dtype()).double().numpy()
        t0 = time.perf_counter()
        kb = dequantize_int8_rows(codes, scale)
        ring = RingCache(S, W)
        ring.pos, ring.head, ring.count = int(pos[b]), int(head[b]), int(count[b])
        for s_ in range(S + W):
            ring.slots[s_] = (kb[:, s_], vb[:, s_])
        P = int(pos[b])
        qr = rope_rotate(q, [P], om, 1.0, D)
        kr = rope_rotate(k, [P], om, 1.0, D)
        kc, ks = quantize_int8_rows(kr[0])
        ring.append([(dequantize_int8_rows(kc, ks), v)])
        decode_attention(ring, qr[0])
        secs += time.perf_counter() - t0
        n += 1
    kv = Hkv * (S + W) * (D + 4 + 2 * D)  # codes + scale + bf16 V per row
    return {"value": round(n * kv / secs / 1e9, 4), "unit": "GB/s", "ms_per_step": round(secs / n * B * 1e3, 1),
            "sample": f"{n} single-sequence windowed decode steps over int8 keys ({secs:.2f} s); the "
                      f"{B}-sequence step extrapolated by the sequence count"}


def _cpu_paged():
    """The windowed step over a paged cache (16-token blocks): the token's rotated key
    and value written at its block and offset, then paged decode attention over the
    sink block and the window's blocks (every other table entry -1); single sequences,
    about 5 s of oracle time."""
    import numpy as np
    from oracle.sinkkv_oracle import RopeSpec, paged_decode_attention, rope_rotate
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    bs = 16
    pos = synth.window_state(13, B, W, c["pos_lo"], c["pos_hi"])[0]
    om = RopeSpec(D, c["r"], c["theta"]).omega()
    rng = np.random.default_rng(9)
    secs, n = 0.0, 0
    while n == 0 or secs < CPU_ROW_SECS:
        b = n % B
        P = int(pos[b])
        first_win = P - W + 1   # the oldest recent key the new token's query sees
        logical = sorted({0} | set(range(first_win // bs, P // bs + 1)))
        perm = rng.permutation(len(logical))
        table = np.full(P // bs + 1, -1, dtype=np.int64)
        for j, lb in enumerate(logical):
            table[lb] = perm[j]
        kp = rng.standard_normal((len(logical), Hkv, bs, D))
        vp = rng.standard_normal((len(logical), Hkv, bs, D))
        q = synth.normal((1, Hq, D), 3000 + b, torch_dtype()).double().numpy()
        k = synth.normal((1, Hkv, D), 4000 + b, torch_dtype()).double().numpy()
        v = synth.normal((Hkv, D), 5000 + b, torch_dtype()).double().numpy()
        t0 = time.perf_counter()
        qr = rope_rotate(q, [P], om, 1.0, D)
        kr = rope_rotate(k, [P], om, 1.0, D)
        blk = int(table[P // bs])
        kp[blk, :, P % bs] = kr[0]
        vp[blk, :, P % bs] = v
        paged_decode_attention(qr[0], kp, vp, table, P + 1, bs, S, W)
        secs += time.perf_counter() - t0
        n += 1
    kv = Hkv * (S + W) * D * 2 * 2
    return {"value": round(n * kv / secs / 1e9, 4), "unit": "GB/s", "ms_per_step": round(secs / n * B * 1e3, 1),
            "sample": f"{n} single-sequence windowed decode steps over 16-token blocks ({secs:.2f} s); the "
                      f"{B}-sequence step extrapolated by the sequence count"}


def synth_cfg(name):
    from sink_kv_attention_gb300 import synth
    return getattr(synth, name)


CPU_ROWS = {"tiny": _cpu_tiny, "window_b1": _cpu_window_b1, "hybrid": _cpu_hybrid, "prefill": _cpu_prefill,
            "rerotate_bf16": lambda: _cpu_rerotate("bf16"), "rerotate_i8": lambda: _cpu_rerotate("i8"),
            "window_i8": _cpu_window_i8, "paged": _cpu_paged, "window_step": _cpu_window_step}


def cpu_row(name):
    """The oracle baseline of configuration `name`, single-threaded in a subprocess."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-row", name],
                       capture_output=True, text=True, env=env, timeout=900)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d.update({"cores": 1, "kind": "oracle", "cpu": _cpu_model()})
    return d


def cpu_baseline(n_seq=32):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", str(n_seq)],
                       capture_output=True, text=True, env=env, timeout=600)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    gbs = d["kv_bytes"] / d["secs"] / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu": _cpu_model(),
            "sample": f"{d['steps']} windowed decode steps of {n_seq} sequences, fresh inputs each "
                      f"(float64 numpy, single thread, {d['secs']:.2f} s)"}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

ROWS = (("tiny", bench_tiny), ("window_b1", bench_window_b1), ("hybrid", bench_hybrid),
        ("prefill", bench_prefill), ("rerotate_bf16", lambda a: bench_rerotate(a, "bf16")),
        ("rerotate_i8", lambda a: bench_rerotate(a, "i8")), ("window_i8", bench_window_i8),
        ("paged", bench_paged), ("window_step", bench_window_step))


def bench_rows(args):
    """Every other configuration of the path on this GPU, each with its roofline and
    its oracle baseline: the tiny case, single-stream decode, the hybrid 32-layer step,
    the prefill chunk and the two rerotations; then the windowed step over int8 keys,
    over a paged cache and through sk_decode_step."""
    import gc
    import torch
    rows = {}
    for name, fn in ROWS:
        try:
            r = fn(args)
            for key in ("n_gpus", "data", "peak_source"):
                r.pop(key, None)
        except Exception as e:  # reported, never fatal to the headline
            r = {"error": f"{type(e).__name__}: {str(e)[:300]}"}
        gc.collect()
        torch.cuda.empty_cache()
        if not args.no_cpu_baseline and name in CPU_ROWS:
            try:
                r["cpu_baseline"] = cpu_row(name)
            except Exception as e:
                r["cpu_baseline"] = {"value": None, "error": str(e)[:200]}
        rows[name] = r
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="window",
                    choices=["window", "window_i8", "hybrid", "rerotate_bf16", "rerotate_i8", "prefill",
                             "prefill_chunk", "dynamic_bf16", "dynamic_i8", "shift_bf16", "shift_i8", "paged",
                             "rope", "tiny", "window_b1", "window_step"])
    ap.add_argument("--cpu-worker", type=int, default=0)
    ap.add_argument("--cpu-row", default="", choices=[""] + sorted(CPU_ROWS))
    ap.add_argument("--no-rows", action="store_true",
                    help="the headline line only, without the other configurations")
    ap.add_argument("--cpu-worker-mt", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0, help="rerotate: layer count (default 48)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--learned-sink", action="store_true",
                    help="window/hybrid/prefill: add per-head learned sink logits to the attention")
    ap.add_argument("--eager", action="store_true", help="launch each step from Python instead of a CUDA graph")
    args = ap.parse_args()

    if args.cpu_worker:
        _cpu_worker(args.cpu_worker)
        return
    if args.cpu_row:
        print(json.dumps(CPU_ROWS[args.cpu_row]()))
        return
    if args.cpu_worker_mt:
        _cpu_worker_mt(args.cpu_worker_mt)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        # The reference arm is the float64 CPU oracle, on rank 0 only, one thread (set
        # before numpy loads its BLAS).
        if rank != 0:
            return
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        steps, warm = args.steps, args.warmup
        per_step = 2  # sequences of the 32 per step: a bounded sample
        n = min(steps, 20)
        for _ in range(min(warm, 2)):
            cpu_oracle_window(1)
        secs, kv = 0.0, 0
        for i in range(n):
            s, b = cpu_oracle_window(per_step, seed_base=i)
            secs += s
            kv += b
        value = kv / secs / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
                "n_gpus": args.gpus, "steps": n, "warmup": min(warm, 2),
                "ms_per_step": round(1e3 * secs / n, 3), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": "windowed-layer decode step (RoPE + append + split-K attention)",
                           "sample_per_step": f"{per_step} of 32 sequences"},
                "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": f"{per_step} of 32 sequences per step, {n} steps"},
                "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    _, world_, _ = _dist_init(args.gpus)
    if args.workload != "window":
        if rank == 0:
            if args.workload == "hybrid":
                print(json.dumps(bench_hybrid(args)))
            elif args.workload == "prefill":
                print(json.dumps(bench_prefill(args)))
            elif args.workload == "prefill_chunk":
                print(json.dumps(bench_prefill_chunk(args)))
            elif args.workload.startswith("dynamic"):
                print(json.dumps(bench_dynamic(args, args.workload.split("_")[1])))
            elif args.workload == "paged":
                print(json.dumps(bench_paged(args)))
            elif args.workload == "window_i8":
                print(json.dumps(bench_window_i8(args)))
            elif args.workload.startswith("shift"):
                print(json.dumps(bench_shift(args, args.workload.split("_")[1])))
            elif args.workload == "rope":
                print(json.dumps(bench_rope(args)))
            elif args.workload == "tiny":
                print(json.dumps(bench_tiny(args)))
            elif args.workload == "window_b1":
                print(json.dumps(bench_window_b1(args)))
            elif args.workload == "window_step":
                print(json.dumps(bench_window_step(args)))
            else:
                print(json.dumps(bench_rerotate(args, args.workload.split("_")[1])))
        return
    result = bench_window(args, rank, world_)
    if rank == 0:
        if not args.no_rows and world_ == 1:
            result["rows"] = bench_rows(args)
        if not args.no_cpu_baseline and world_ == 1:
            try:
                result["cpu_baseline"] = cpu_baseline()
            except Exception as e:  # reported, never fatal
                result["cpu_baseline"] = {"value": None, "error": str(e)[:200]}
            try:
                result["cpu_baseline_all_cores"] = cpu_baseline_all_cores()
            except Exception as e:  # reported, never fatal
                result["cpu_baseline_all_cores"] = {"value": None, "error": str(e)[:200]}
        print(json.dumps(result))
    if world_ > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
