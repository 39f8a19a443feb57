"""Benchmark: batch-1 decode tokens/s and achieved HBM GB/s as a fraction of the GB300 roofline.

One bench step is one decode step (one token: embedding, every layer, final norm, LM head) of the
SmolLM-135M-shaped decoder (30 layers, hidden 576, 9/3 heads, vocab 49152, static 128-entry KV
cache), teacher-forced over seeded uniform token ids at positions 0..127 (cycling), random-init
bf16 weights ~N(0, 0.02).  `--config` picks another decoder shape.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Our arm times K back-to-back steps with CUDA events on the launching stream (inputs resident in
HBM; the 270 MB of weights read per step exceed the 129 MB L2, and weights stream with an
evict-first L2 policy).  `e2e` repeats the measurement through the C ABI with host buffers: each
step passes the token id from the host and copies the logits back into pinned host memory.  The
reference arm (`--impl reference`) is the CPU oracle timed on this machine's cores.
With N > 1 (torchrun), every rank runs an independent replica: the decode does not shard.
"""
from __future__ import annotations

import argparse
import json
import re
import os
import statistics
import subprocess
import sys
import time

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

PAGES_TOKS = {"smollm-135m": 912.0, "qwen2-0.5b": 759.0, "smollm-1.7b": 419.0}  # H200 MIG 60-SM slice, context only
METRIC = "batch-1 decode tokens/s and achieved HBM GB/s as fraction of GB300 roofline"


def algorithmic_bytes(shape, positions, fp8: bool = False) -> float:
    """Bytes a decode step must move, averaged over `positions`: every weight once (tied E as the LM
    head), the norm gains, the token's embedding row, K/V rows 0..p read once, one K/V row written.
    fp8: the projections and the LM head as one byte per weight plus a 4-byte scale per row."""
    s = shape
    H, I, d = s.hidden, s.intermediate, s.head_dim
    qd, kvd = s.n_heads * d, s.n_kv_heads * d
    wb = 1 if fp8 else 2
    proj = qd * H + 2 * kvd * H + H * qd + 3 * H * I
    per_layer = proj * wb + 2 * H * 2
    if fp8:
        per_layer += (qd + 2 * kvd + H + 2 * I + H) * 4
    if s.qkv_bias:
        per_layer += (qd + 2 * kvd) * 2
    fixed = s.n_layers * per_layer + s.vocab * H * wb + (s.vocab * 4 if fp8 else 0) + H * 2 + H * 2
    kv_row = s.n_layers * 2 * kvd * 2
    kv = statistics.fmean([(p + 1) * kv_row + kv_row for p in positions])
    return fixed + kv


def steps_per_call(steps: int, positions: int) -> int:
    """Largest power of two dividing both the requested steps and the workload's positions that still
    leaves at least 5 timed launches (1 when none does)."""
    best, spc = 1, 1
    while spc <= positions:
        if positions % spc == 0 and steps % spc == 0 and steps // spc >= 5:
            best = spc
        spc *= 2
    return best


NOMINAL_HBM_GBS = 8000.0  # HBM3e nominal, GB300


def load_peaks():
    p = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="mbk_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, bus_id: str | None):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if bus_id:
            mine = [r for r in rows if r[1].lower().endswith(bus_id.lower()[-12:])]
            rows = mine or rows
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower().startswith("active")})
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if os.environ.get("MBK_BENCH_BACKEND", "nccl") == "nccl" else "gloo")
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_oracle(wl, budget_s: float, max_steps: int, fp8: bool = False):
    """Oracle decode steps of `wl` for about budget_s seconds; returns (tokens/s, steps, threads).
    fp8: the oracle on the FP8 copies of the weights (quantized before the timed steps)."""
    from oracle import OracleDecoder
    orc = OracleDecoder(wl, fp8=fp8)
    s = wl.shape
    n, t0 = 0, time.perf_counter()
    while n < max_steps:
        orc.step(int(wl.tokens[n % s.steps]), s.pos0 + (n % s.steps))
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, orc.lib.orc_max_threads()


def run_reference(args, shape_name):
    from persistent_decode_megakernel_gb300 import workloads
    world, rank, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    wl = workloads.generate(shape_name, seed=0)
    s = wl.shape
    budget = float(os.environ.get("MBK_REF_BUDGET_S", "60"))
    # warm-up steps (untimed), then the timed sample
    from oracle import OracleDecoder
    fp8 = args.weights == "fp8"
    warm = OracleDecoder(wl, fp8=fp8)
    for i in range(min(args.warmup, 3)):
        warm.step(int(wl.tokens[i]), s.pos0 + i)
    tps, n, cores = time_oracle(wl, budget, args.steps, fp8)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tps, 3), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 / tps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{shape_name} batch-1 teacher-forced decode", "positions": f"{s.pos0}..{s.pos0 + s.steps - 1}",
                   "kv_capacity": s.kv_capacity},
        "cpu_baseline": {"value": round(tps, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {args.steps} decode steps (time-bounded to {budget:.0f} s)"},
        "e2e": {"value": round(tps, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, shape_name):
    import torch

    from persistent_decode_megakernel_gb300 import build, mbk, workloads

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    build.build()
    wl = workloads.generate(shape_name, seed=0)
    s = wl.shape
    fp8 = getattr(args, "weights", "bf16") == "fp8"
    dec = mbk.Decoder(wl, device=local, fp8=fp8)
    stream = torch.cuda.current_stream()
    # one call decodes `spc` consecutive teacher-forced positions (mbk_decode_steps; 1 = mbk_decode_step):
    # exactly --steps steps are timed, in at least 5 launches when --steps allows it
    spc = args.steps_per_call if args.steps_per_call > 0 else steps_per_call(args.steps, s.steps)
    if s.steps % spc:
        raise SystemExit(f"--steps-per-call must divide the workload's {s.steps} positions")
    steps = (args.steps + spc - 1) // spc * spc
    warm = (args.warmup + spc - 1) // spc * spc
    toks = [int(wl.tokens[i % s.steps]) for i in range(steps + warm)]
    poss = [s.pos0 + (i % s.steps) for i in range(steps + warm)]
    out = dec.logits if spc == 1 else torch.empty((spc, s.vocab), dtype=torch.float32, device=dec.device)

    def call(i):  # the call that decodes steps i .. i + spc - 1
        if spc == 1:
            dec.step(toks[i], poss[i], out)
        else:
            dec.steps(toks[i:i + spc], poss[i], out)

    for i in range(0, warm, spc):
        call(i)
    torch.cuda.synchronize()

    ncalls = steps // spc
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ncalls)]
    sampler = ClockSampler()
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(ncalls):
        ev[k][0].record(stream)
        call(warm + k * spc)
        ev[k][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(local).pci_bus_id
    except Exception:
        pass
    clocks = sampler.stop(bus)
    assert dec.status() == 0, "device-side wait timed out during the benchmark"
    total_ms = max_over_ranks(start.elapsed_time(end), world, torch.device("cuda", local))
    kern_ms = [a.elapsed_time(b) / spc for a, b in ev]  # per decode step
    kernel_avg_ms = statistics.fmean(kern_ms)
    ks = sorted(kern_ms)
    spread = {"median_us": round(1e3 * ks[len(ks) // 2], 3), "p10_us": round(1e3 * ks[len(ks) // 10], 3),
              "p90_us": round(1e3 * ks[min(len(ks) - 1, (9 * len(ks)) // 10)], 3), "launches": len(ks)}

    # the same workload one step per launch (mbk_decode_step), for reference
    single_tps = None
    if spc > 1:
        n1 = min(steps, 1024)
        for i in range(8):
            dec.step(toks[i], poss[i], dec.logits)
        torch.cuda.synchronize()
        a1, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a1.record(stream)
        for i in range(n1):
            dec.step(toks[warm + i], poss[warm + i], dec.logits)
        b1.record(stream)
        torch.cuda.synchronize()
        single_tps = n1 / (a1.elapsed_time(b1) * 1e-3)

    # greedy decoding over the same positions (mbk_decode_greedy: each step's argmax is the next
    # token, inside one launch per run of positions; tokens only, no logits), for reference
    greedy_tps = None
    if spc > 1:
        for _ in range(2):
            dec.greedy(toks[0], spc, s.pos0, want_logits=False)
        torch.cuda.synchronize()
        ng = max(1, min(ncalls, 8))
        a1, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a1.record(stream)
        for _ in range(ng):
            dec.greedy(toks[0], spc, s.pos0, want_logits=False)
        b1.record(stream)
        torch.cuda.synchronize()
        assert dec.status() == 0, "device-side wait timed out during greedy decoding"
        greedy_tps = ng * spc / (a1.elapsed_time(b1) * 1e-3)

    # end to end through the C ABI with host buffers: token ids from the host, every step's logits
    # back to pinned host memory, the stream synchronised after each call
    host = torch.empty((spc, s.vocab), dtype=torch.float32, pin_memory=True)
    e2e_steps = min(steps, 2048 // spc * spc if spc <= 2048 else spc)

    def call_host(i):
        if spc == 1:
            rc = mbk.mbk_decode_step_host(dec.handle, toks[i], poss[i], host.data_ptr(), stream.cuda_stream)
            assert rc == 0, mbk.mbk_error_string(rc)
        else:
            dec.steps(toks[i:i + spc], poss[i], out)
            host.copy_(out, non_blocking=True)
            stream.synchronize()

    for i in range(0, min(warm, 2 * spc), spc):
        call_host(i)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(0, e2e_steps, spc):
        call_host(warm + i)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, torch.device("cuda", local))

    positions = [poss[warm + i] for i in range(steps)]
    algo = algorithmic_bytes(s, positions, fp8)
    peak, peak_kind = load_peaks()
    achieved = algo / (kernel_avg_ms * 1e-3) / 1e9
    tps = steps * world / (total_ms * 1e-3)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        budget = float(os.environ.get("MBK_CPU_BUDGET_S", "15"))
        ctps, cn, cores = time_oracle(wl, budget, s.steps, fp8)
        cpu = {"value": round(ctps, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{cn} teacher-forced decode steps of the same workload (time-bounded to {budget:.0f} s)"}
    traffic = profiled_traffic(shape_name) if not fp8 else None
    others = measure_others(shape_name, fp8, local, peak) if (rank == 0 and not args.no_others) else None
    prefill = measure_prefill(local) if (rank == 0 and not args.no_others and not fp8) else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(tps, 2), "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": round(total_ms / steps, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": round(tps / PAGES_TOKS[shape_name], 3) if shape_name in PAGES_TOKS else None,
            "dtype": "fp8-e4m3 weights, f32 math" if fp8 else "bf16", "data": "synthetic",
            "config": {"workload": f"{shape_name} batch-1 teacher-forced decode, random-init weights",
                       "positions": f"{s.pos0}..{s.pos0 + s.steps - 1} cycling", "kv_capacity": s.kv_capacity,
                       "parallelism": "replicas" if world > 1 else "single-gpu",
                       "l2": "inputs larger than L2 (weights stream evict-first)",
                       "steps_per_call": spc,
                       "single_step_tokens_per_s": round(single_tps, 2) if single_tps else None,
                       "greedy_tokens_per_s": round(greedy_tps, 2) if greedy_tps else None,
                       "per_step_time_over_launches": spread,
                       "e2e_path": "mbk_decode_step_host (C ABI, host logits) per step" if spc == 1 else
                                   "mbk_decode_steps per launch, then the launch's logits copied to pinned host memory",
                       "others": others,
                       "prefill": prefill,
                       "vs_baseline_note": "pages' H200 MIG 60-SM number, context only",
                       "weights": "fp8 (E4M3, per-row fp32 scales, quantized by the library)" if fp8 else "bf16"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_kind": peak_kind,
                         "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                         "algorithmic_bytes_per_step": round(algo), "kernel_avg_us_per_step": round(kernel_avg_ms * 1e3, 3),
                         "per": "decode step (a launch of n steps moves n times the bytes in n times the time)",
                         "kernel": "mbk::decode_kernel"},
            "e2e": {"value": round(e2e_steps * world / e2e_s, 2), "unit": "tokens/s", "h2d_bytes_per_step": 4,
                    "d2h_bytes_per_step": s.vocab * 4},
            "gpu_launches": ncalls,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    dec.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_others(main: str, fp8: bool, device: int, peak: float):
    """The other decoder shapes, a few launches each (one launch = the workload's teacher-forced
    positions): tokens/s, roofline fraction of the measured and of the nominal HBM peak."""
    import torch

    from persistent_decode_megakernel_gb300 import mbk, workloads
    out = []
    for name in ("tiny", "smollm-135m", "qwen2-0.5b", "smollm-135m-long", "smollm-1.7b"):
        if name == main:
            continue
        wl = workloads.generate(name, seed=0)
        s = wl.shape
        dec = mbk.Decoder(wl, device=device, fp8=fp8)
        toks = [int(t) for t in wl.tokens[:s.steps]]
        logits = torch.empty((s.steps, s.vocab), dtype=torch.float32, device=dec.device)
        for _ in range(2):
            dec.steps(toks, s.pos0, logits)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
        for a, b in ev:
            a.record(stream)
            dec.steps(toks, s.pos0, logits)
            b.record(stream)
        torch.cuda.synchronize()
        assert dec.status() == 0, f"device-side wait timed out ({name})"
        per_step = sorted(a.elapsed_time(b) * 1e-3 / s.steps for a, b in ev)
        med = per_step[len(per_step) // 2]
        algo = algorithmic_bytes(s, [s.pos0 + i for i in range(s.steps)], fp8)
        ach = algo / med / 1e9
        fits_l2 = algo < 100e6  # the tiny decoder's working set stays in the 129 MB L2
        out.append({"workload": name, "tokens_per_s": round(1.0 / med, 1), "us_per_step_median": round(med * 1e6, 2),
                    "launches": len(ev), "steps_per_launch": s.steps, "algorithmic_bytes_per_step": round(algo),
                    "achieved_gbs": round(ach, 1), "frac": None if fits_l2 else round(ach / peak, 4),
                    "frac_of_nominal_8tbs": None if fits_l2 else round(ach / NOMINAL_HBM_GBS, 4),
                    "note": "fits in L2: no HBM roofline" if fits_l2 else None})
        dec.close()
        del dec, logits, wl
    return out


def load_tensor_peak():
    p = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    return 1900.0, "fallback (burst)"


def measure_prefill(device: int, n: int = 4096):
    """A prompt of n tokens through mbk_prefill on the 135M shape with an 8,192-row cache (the long-
    context shape's cache, positions 0..n-1), last-row logits: time, tokens/s, and the algorithmic work
    against the bf16 tensor peak.  Work = 2 x the projection MACs of every token (the LM head for the
    last token only) + the causal attention's 4 nq d (t + 1) flops per token and layer; the tensor cores
    execute the projections twice (the bf16 high/low pair of each input), counted as overhead."""
    import torch

    from persistent_decode_megakernel_gb300 import mbk, workloads
    wl = workloads.generate("smollm-135m-long", seed=0)
    s = wl.shape
    g = torch.Generator().manual_seed(1)
    toks = [int(t) for t in torch.randint(0, s.vocab, (n,), generator=g)]
    dec = mbk.Decoder(wl, device=device)
    out = torch.empty(s.vocab, dtype=torch.float32, device=dec.device)
    dec.prefill(toks, 0, logits="last", out=out)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
    for a, b in ev:
        a.record(stream)
        dec.prefill(toks, 0, logits="last", out=out)
        b.record(stream)
    torch.cuda.synchronize()
    assert dec.status() == 0, "device-side wait timed out in the prefill"
    dec.close()
    ms = sorted(a.elapsed_time(b) for a, b in ev)[1]
    H, I, d = s.hidden, s.intermediate, s.head_dim
    proj = s.n_layers * (H * s.n_heads * d + 2 * H * s.n_kv_heads * d + s.n_heads * d * H + 3 * H * I)
    gemm = 2.0 * proj * n + 2.0 * s.vocab * H
    attn = 4.0 * s.n_heads * d * s.n_layers * n * (n + 1) / 2
    peak, kind = load_tensor_peak()
    tf = (gemm + attn) / (ms * 1e-3) / 1e12
    return {"workload": f"prefill of {n} tokens, SmolLM-135M shape, last-row logits", "ms_median_of_3": round(ms, 3),
            "tokens_per_s": round(n / (ms * 1e-3), 1), "gemm_tflop": round(gemm / 1e12, 3),
            "attention_tflop": round(attn / 1e12, 3), "achieved_tflops": round(tf, 2),
            "peak_tflops": peak, "peak_kind": kind, "frac": round(tf / peak, 4),
            "note": "tensor cores run the projections twice (bf16 high/low input pair): overhead, not work; "
                    "the causal attention runs on the tensor cores as well (mma.sync, fp32 operands as bf16 pairs)"}


def profiled_traffic(shape_name: str):
    """DRAM bytes per launch from the committed ncu summary of this workload, or None when the
    summary is missing or was taken on different kernel sources."""
    tp = os.path.join(_ROOT, "profiles", f"decode_kernel_{shape_name.replace('-', '').replace('.', '')}.md")
    if not os.path.exists(tp):
        return None
    with open(tp) as f:
        text = f.read()
    mh = re.search(r"kernel_source_hash: `([0-9a-f]+)`", text)
    mb = re.search(r"dram_bytes_per_launch: (\d+)", text)
    if not mh or not mb or mh.group(1) != _kernel_hash():
        return None
    return int(mb.group(1))


def _kernel_hash() -> str:
    """Hash of the decode kernel's code: its sources with comments and whitespace removed, so that a
    comment-only edit keeps the committed ncu counters."""
    import hashlib
    h = hashlib.sha256()
    for f in ("mbk_kernel.cu", "mbk_plan.h", "mbk_device.h", "mbk_sched.cpp"):
        with open(os.path.join(_ROOT, "persistent_decode_megakernel_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)                # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="smollm-135m")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip config.others (the other decoder shapes) and config.prefill")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "fp8"],
                    help="fp8: stream the library's FP8 (E4M3, per-row scale) copies of the weights")
    ap.add_argument("--steps-per-call", type=int, default=0,
                    help="teacher-forced steps per launch (default: the workload's positions; 1 = one launch per step)")
    ap.add_argument("--prefill-only", type=int, default=0, metavar="N",
                    help="diagnostics: time one N-token prefill (as config.prefill does) and print its line only")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.prefill_only > 0:
        print(json.dumps(measure_prefill(0, args.prefill_only)))
        return
    if args.impl == "reference":
        run_reference(args, args.config)
    else:
        run_ours(args, args.config)


if __name__ == "__main__":
    main()
