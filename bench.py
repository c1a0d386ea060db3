"""Benchmark of the inverse-RoPE + block-FP8 quant hot path on one or more GPUs.

One step = one pass of the whole hot path over one batch of seeded synthetic
input resident in HBM:
  1. inverse RoPE + block-FP8 quant of the DeepSeek-V4-Flash TP2 prefill shape
     (x [16384, 32, 512] bf16, heads_per_group 8, positions 0..16383,
     cos/sin cache [65536, 64]),
  2. forward RoPE + FP8 quant + paged insert of kv [16384, 512] into a
     512-block x 64-slot cache (slots: a seeded permutation of the 32768 slots).
``value`` = algorithmic bytes of the step (every tensor read or written once)
/ step time, in GB/s, summed over ranks (each rank runs its own full copy:
weak scaling, no collective on the data path).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (the plain C statement of the op)
on the host cores over a bounded sample of the same workload.
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "µs and achieved HBM GB/s (% of B300 peak) at N=16384,H=32,D=512"
INV_SPEC = W.PREFILL16K
INS_SPEC = W.INSERT16K
INV_BYTES = W.inverse_bytes(INV_SPEC.n_tokens, INV_SPEC.n_heads)
INS_BYTES = W.insert_bytes(INS_SPEC.n_tokens)
STEP_BYTES = INV_BYTES + INS_BYTES
L2_BYTES = 126 * 2 ** 20
FALLBACK_HBM_GBS = 6400.0
# the kernel the default (auto) variant launches at the benchmarked shape
INV_KERNEL_NAME = "inv_rope_fp8_quant_kernel"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=12000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the host-buffer end-to-end leg (default min(steps, 20))")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunk", type=int, default=512,
                    help="tokens per chunk of the host-buffer pipeline in the e2e leg")
    ap.add_argument("--mode-launches", type=int, default=300,
                    help="launches timed per extra output kind / layout (0 skips them)")
    ap.add_argument("--ref-budget-s", type=float, default=60.0,
                    help="host seconds the reference arm's timed + warm-up steps aim to take")
    ap.add_argument("--inv-tokens", type=int, default=None,
                    help="tokens of the inverse op (default 16384; smaller cases are for "
                         "profiling captures and are not bench lines)")
    ap.add_argument("--profile-op", choices=sorted(PROFILE_OPS), default=None,
                    help="run only this op, 3 times, on --inv-tokens tokens (default 4096), "
                         "then exit: the small case an ncu capture runs; prints no bench line")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak_fp8():
    """Dense fp8 tensor peak: the measured cuBLAS bf16 burst figure times the
    nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s = 2)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return round(2.0 * float(d["bf16_tflops"]), 1), "measured bf16 burst x 2 (nominal ratio)"
    except Exception:
        return 3600.0, "fallback 1.8 PFLOP/s bf16 x 2"


class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons of one GPU during
    the timed region: through NVML when pynvml imports, else by running
    ``nvidia-smi --query-gpu=... -lms 50`` (both only read the settings)."""

    REASON_BITS = {
        0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
    }
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.02):
        self.period = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.bus_id = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            self.bus_id = "{:08X}:{:02X}:{:02X}.0".format(
                getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
        except Exception:
            self.bus_id = None
        self.nv = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.h = (pynvml.nvmlDeviceGetHandleByPciBusId(self.bus_id) if self.bus_id
                      else pynvml.nvmlDeviceGetHandleByIndex(device_index))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.nv = pynvml
        except Exception as e:
            self.error = f"nvml: {type(e).__name__}: {e}"

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                bits = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                self.reasons |= {n for b, n in self.REASON_BITS.items() if bits & b}
            except Exception as e:
                self.error = f"{type(e).__name__}: {e}"
                return
            self._stop.wait(self.period)

    def __enter__(self):
        if self.nv is not None:
            self._thread = threading.Thread(target=self._run_nvml, daemon=True)
            self._thread.start()
        else:
            import subprocess
            cmd = ["nvidia-smi", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", str(int(self.period * 1000))]
            if self.bus_id:
                cmd += ["-i", self.bus_id]
            try:
                self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                              text=True)
                self._thread = threading.Thread(target=self._read_smi, daemon=True)
                self._thread.start()
            except Exception as e:
                self.error = (self.error or "") + f"; nvidia-smi: {type(e).__name__}: {e}"
        return self

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            f = [v.strip() for v in line.split(",")]
            if len(f) < 8:
                continue
            try:
                self.samples.append(float(f[0]))
                self.max_mhz = float(f[1])
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    self.reasons.add(name)

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread:
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "error": self.error or "no samples"}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "nvml" if self.nv is not None else "nvidia-smi"}


# ------------------------------------------------------------------ our arm

def make_inputs(inv_tokens=None):
    cache = W.rope_cache(INV_SPEC.cache_rows)
    spec = INV_SPEC
    if inv_tokens:
        spec = W.InverseSpec(f"prefill{inv_tokens}", inv_tokens, INV_SPEC.n_heads,
                             INV_SPEC.heads_per_group, INV_SPEC.cache_rows, "arange", True)
    inv = W.inverse_inputs(spec, cache=cache)
    ins = W.insert_inputs(INS_SPEC, cache=cache)
    return inv, ins


def oracle_step_rate(inv, ins, tokens, steps, warmup, threads):
    """Warm mean of `steps` oracle steps (after `warmup` untimed ones) over the
    first `tokens` tokens of both ops: (GB/s of the step's algorithmic bytes,
    seconds per step). The one method behind cpu_baseline and the reference arm."""
    import oracle
    oracle.build()
    xi, pi = inv["x"][:tokens].contiguous(), inv["positions"][:tokens].contiguous()
    kv, kp, sl = (ins["kv"][:tokens].contiguous(), ins["positions"][:tokens].contiguous(),
                  ins["slot_mapping"][:tokens].contiguous())
    cache = inv["cos_sin_cache"]
    sample_bytes = W.inverse_bytes(tokens, inv["x"].shape[1]) + W.insert_bytes(tokens)

    def step():
        oracle.inv_rope_fp8_quant(xi, pi, cache, inv["heads_per_group"], threads=threads)
        oracle.rope_fp8_quant_insert(kv, kp, cache, sl, ins["k_cache"], ins["block_size"],
                                     threads=threads)

    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = (time.perf_counter() - t0) / steps
    return sample_bytes / dt / 1e9, dt


def cpu_baseline(inv, ins):
    """The oracle, as it stands, on all host cores: the warm mean of 3 full
    steps after one untimed step (the reference arm's method), plus the inverse
    alone on one core over a quarter of the tokens (warm)."""
    import oracle
    threads = os.cpu_count() or 1
    tokens = inv["x"].shape[0]
    gbs, dt = oracle_step_rate(inv, ins, tokens, steps=3, warmup=1, threads=threads)
    q = tokens // 4
    xq, pq = inv["x"][:q].contiguous(), inv["positions"][:q].contiguous()
    oracle.inv_rope_fp8_quant(xq[:256], pq[:256], inv["cos_sin_cache"], inv["heads_per_group"],
                              threads=1)
    t1 = time.perf_counter()
    oracle.inv_rope_fp8_quant(xq, pq, inv["cos_sin_cache"], inv["heads_per_group"], threads=1)
    dt1 = time.perf_counter() - t1
    one_bytes = W.inverse_bytes(q, inv["x"].shape[1])
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds_per_step": round(dt, 4),
            "sample": f"one full step (inverse {tokens} tok x {inv['x'].shape[1]} heads + insert "
                      f"{tokens} tok), warm mean of 3 steps after 1 untimed; oracle with "
                      f"{threads} threads",
            "single_thread": {"value": round(one_bytes / dt1 / 1e9, 4), "unit": "GB/s",
                              "cores": 1, "seconds": round(dt1, 3),
                              "sample": f"inverse only, {q} tokens x {inv['x'].shape[1]} heads, "
                                        "after a warm call"}}


def block_stream(stream, ms: float):
    """Keep `stream` busy for about `ms` milliseconds (a spinning kernel), so
    that the host enqueues the launches that follow before the device reaches
    them: events recorded after it then time device work only, not the host's
    launch rate (the blocking-kernel method of GPU benchmark harnesses)."""
    clock_hz = 2.0e9
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 1e-3 * clock_hz))


def host_us_per_call(fn, calls: int = 3) -> float:
    t0 = time.perf_counter()
    for _ in range(calls):
        fn()
    return (time.perf_counter() - t0) / calls * 1e6


def run_ours(args, world, rank, local):
    import rope_block_fp8_inverse_b300 as rq
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inv_h, ins_h = make_inputs(args.inv_tokens)
    inv_bytes = W.inverse_bytes(inv_h["x"].shape[0], inv_h["x"].shape[1])
    step_bytes = inv_bytes + INS_BYTES
    peak, peak_src = measured_peaks()

    # device-resident inputs and caller-owned outputs
    x = inv_h["x"].to(dev)
    pos = inv_h["positions"].to(dev)
    cache = inv_h["cos_sin_cache"].to(dev)
    hpg = inv_h["heads_per_group"]
    n, h = x.shape[0], x.shape[1]
    out = torch.empty((n, h // hpg, hpg * 512), dtype=torch.uint8, device=dev)
    scales = torch.empty((n, h // hpg, hpg * 4), dtype=torch.float32, device=dev)
    kv = ins_h["kv"].to(dev)
    kpos = ins_h["positions"].to(dev)
    slots = ins_h["slot_mapping"].to(dev)
    k_cache = ins_h["k_cache"].to(dev)
    bs = ins_h["block_size"]
    stream = torch.cuda.current_stream(dev)

    def inverse_call():
        rq.inv_rope_fp8_quant(x, pos, cache, hpg, out=out, scales=scales)

    def insert_call():
        rq.rope_fp8_quant_insert(kv, kpos, cache, slots, k_cache, bs)

    def step():
        inverse_call()
        insert_call()

    enqueue = {}

    def held(name, body, est_host_ms, launches):
        """Run `body` (it enqueues launches and records events on `stream`)
        behind a spinning kernel that holds the stream until the host has
        enqueued all of it, so the events time device work only. The host's
        enqueue time is measured: if it outlasted the block, the device may
        have waited on the host inside the timed region, so the run is
        repeated with a longer block (up to three times; a loop with more
        launches than the launch queue holds cannot be covered, and says so
        in `enqueue`)."""
        block = max(2.0, 2.0 * est_host_ms + 1.0)
        tries = 3 if launches <= 1024 else 1
        for attempt in range(tries):
            torch.cuda.synchronize(dev)
            block_stream(stream, block)
            t0 = time.perf_counter()
            body()
            host_ms = (time.perf_counter() - t0) * 1e3
            torch.cuda.synchronize(dev)
            covered = host_ms < 0.9 * block
            if covered:
                break
            block = min(4000.0, 2.0 * host_ms + 5.0)
        enqueue[name] = {"host_ms": round(host_ms, 2), "block_ms": round(block, 2),
                         "covered": covered, "tries": attempt + 1}

    def span_us(fn, launches, name):
        """Mean µs per launch of `launches` back-to-back calls: one event pair
        around all of them on the launching stream, after 3 warm calls, with
        the stream held by a spinning kernel while the host enqueues them."""
        host = host_us_per_call(fn, 3)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def body():
            a.record(stream)
            for _ in range(launches):
                fn()
            b.record(stream)
        held(name, body, host * launches * 1e-3, launches)
        return a.elapsed_time(b) * 1e3 / launches

    # clocks are sampled (read only) from before the warm-up to the end of the
    # last GPU leg, so every leg, the timed steps included, lies inside
    sampler = ClockSampler(local)
    with sampler:
        warm = max(3, args.warmup)
        t_w = time.perf_counter()
        for _ in range(warm):
            step()
        torch.cuda.synchronize(dev)
        # at least ~0.25 s of steps before timing (bounded), so clocks and
        # power settle; the count above is the contract's minimum
        extra = 0
        while time.perf_counter() - t_w < 0.25 and extra < 4000:
            for _ in range(20):
                step()
            extra += 20
            torch.cuda.synchronize(dev)
        host_step_us = host_us_per_call(step, 3)
        torch.cuda.synchronize(dev)

        # the timed steps: one event pair around all of them, nothing between
        # the launches (the insert may start while the inverse drains), and the
        # launches enqueued while a spinning kernel holds the stream
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def timed_steps():
            start.record(stream)
            for _ in range(args.steps):
                step()
            end.record(stream)
        barrier(world)
        held("timed_steps", timed_steps, host_step_us * args.steps * 1e-3, 2 * args.steps)
        barrier(world)
        total_ms = max_over_ranks(start.elapsed_time(end), world)
        ms_step = total_ms / args.steps

        # the dominant kernel back to back (its mean launch duration in a
        # stream of launches: the roofline's figure), and the insert alone
        span_launches = max(50, min(300, args.steps))
        inv_span = span_us(inverse_call, span_launches, "inverse_span")
        ins_span = span_us(insert_call, span_launches, "insert_span")

        # the same steps with an event pair around each launch: the per-launch
        # durations including each launch's own start-up and drain (no overlap
        # with a neighbour), their percentiles
        ev_steps = max(10, min(args.steps, 200))
        inv_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(ev_steps)]
        ins_ev = [torch.cuda.Event(enable_timing=True) for _ in range(ev_steps)]

        def event_pairs():
            for i in range(ev_steps):
                inv_ev[i][0].record(stream)
                inverse_call()
                inv_ev[i][1].record(stream)
                insert_call()
                ins_ev[i].record(stream)
        held("event_pairs", event_pairs, 2.0 * host_step_us * ev_steps * 1e-3, 2 * ev_steps)
        inv_all = sorted(a.elapsed_time(b) for a, b in inv_ev)
        inv_ms_ev = statistics.fmean(inv_all)
        inv_pct = {f"p{q}": round(inv_all[min(len(inv_all) - 1, int(len(inv_all) * q / 100))] * 1e3, 2)
                   for q in (10, 50, 90, 99)}
        inv_pct["max"] = round(inv_all[-1] * 1e3, 2)
        ins_ms_ev = statistics.fmean(inv_ev[i][1].elapsed_time(ins_ev[i]) for i in range(ev_steps))

        secondary = {}
        if world == 1 and args.mode_launches > 0:
            secondary = run_secondary(args, rq, dev, stream, inv_h, x, pos, cache, hpg, out, scales,
                                      kv, kpos, slots, k_cache, bs, span_us, peak)

        e2e = run_e2e(args, rq, dev, stream, world, inv_h, ins_h, cache, hpg, out, scales, kv,
                      kpos, slots, k_cache, bs)

    achieved = inv_bytes / (inv_span * 1e-6) / 1e9
    achieved_ev = inv_bytes / (inv_ms_ev * 1e-3) / 1e9
    traffic = _committed_traffic()
    target_gbs = 6400.0  # 80% of the nominal ~8 TB/s
    result = {
        "metric": METRIC,
        "value": round(world * step_bytes / (ms_step * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": warm,
        "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "inverse_span_us": round(inv_span, 2),
        "inverse_span_GBs": round(achieved, 1),
        "inverse_span_frac_of_measured_peak": round(achieved / peak, 4),
        "inverse_span_frac_of_6400_target": round(achieved / target_gbs, 4),
        "insert_span_us": round(ins_span, 2),
        "insert_span_frac_of_measured_peak": round(INS_BYTES / ins_span / 1e3 / peak, 4),
        "span_launches": span_launches,
        "inverse_us_event_pair": round(inv_ms_ev * 1e3, 2),
        "inverse_us_event_pair_percentiles": inv_pct,
        "insert_us_event_pair": round(ins_ms_ev * 1e3, 2),
        "timing": "value / ms_per_step: the K timed steps under one event pair, enqueued while "
                  "a spinning kernel held the stream; *_span_us: mean per launch of back-to-back "
                  "launches under one event pair (same enqueue method); *_event_pair: an event "
                  "pair around every launch (each launch's own start-up and drain, no overlap)",
        "frac_of_nominal_8tbs": round(step_bytes / (ms_step * 1e-3) / 8e12, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in, fp32 math, e4m3 out",
        "data": "synthetic (seeded: randn + 1% x50 outliers, bf16)",
        "config": {
            "workload": "prefill16k inverse RoPE+FP8 quant (N=16384,H=32,hpg=8,D=512) "
                        "+ insert16k forward RoPE+FP8 paged insert (N=16384, 512x64 slots)",
            "bytes_per_step": step_bytes,
            "inverse_bytes": inv_bytes,
            "insert_bytes": INS_BYTES,
            "l2": f"inputs larger than L2: {step_bytes / 2**20:.0f} MiB streamed per step "
                  f"vs {L2_BYTES / 2**20:.0f} MiB L2",
            "parallelism": f"replicas x{world} (each rank its own full step)",
        },
        "roofline": {
            "kernel": INV_KERNEL_NAME,
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                           else "fallback 6.4 TB/s",
            "algorithmic_bytes_per_launch": inv_bytes,
            "duration": f"mean launch duration of {span_launches} back-to-back launches "
                        "(inverse_span_us)",
            "event_pair_per_launch": {"achieved": round(achieved_ev, 1),
                                      "frac": round(achieved_ev / peak, 4)},
        },
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(),
        "enqueue": enqueue,
    }
    result.update(secondary)
    if args.inv_tokens and args.inv_tokens != INV_SPEC.n_tokens:
        result["config"]["workload"] = (f"profiling case: inverse N={args.inv_tokens},H=32,hpg=8 "
                                        "+ insert16k (not the benchmarked configuration)")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inv_h, ins_h)
    return result


def run_secondary(args, rq, dev, stream, inv_h, x, pos, cache, hpg, out, scales, kv, kpos, slots,
                  k_cache, bs, span_us, peak):
    """The other configurations and the "next" rows of the path, each timed
    outside the step: config 4 (irregular grouping), the output kinds and
    layouts, the fused q/kv op, the indexer q op, the consumer GEMMs, decode
    latency and the L2-resident configurations cold. One GPU only."""
    n, h = x.shape[0], x.shape[1]
    res = {"secondary_timing": "back-to-back launches under one event pair, mean per launch "
                               "(span_us), unless a leg says otherwise"}

    # config 4: irregular grouping (N=8192, H=24, heads_per_group=6)
    ii = W.inverse_inputs(W.IRREGULAR)
    ix, ip, ic = ii["x"].to(dev), ii["positions"].to(dev), ii["cos_sin_cache"].to(dev)
    ihpg = ii["heads_per_group"]
    io = torch.empty((ix.shape[0], ix.shape[1] // ihpg, ihpg * 512), dtype=torch.uint8, device=dev)
    isc = torch.empty((ix.shape[0], ix.shape[1] // ihpg, ihpg * 4), dtype=torch.float32, device=dev)
    us = span_us(lambda: rq.inv_rope_fp8_quant(ix, ip, ic, ihpg, out=io, scales=isc),
                 args.mode_launches, "irregular")
    ib = W.inverse_bytes(ix.shape[0], ix.shape[1])
    res["irregular"] = {"kernel": INV_KERNEL_NAME, "workload": "irregular (N=8192, H=24, "
                        "heads_per_group=6, positions U[0,32768), cache 32768 rows)",
                        "us": round(us, 2), "bytes": ib, "GBs": round(ib / us / 1e3, 1),
                        "frac_of_measured_peak": round(ib / us / 1e3 / peak, 4),
                        "frac_of_6400_target": round(ib / us / 1e3 / 6400.0, 4),
                        "launches": args.mode_launches}
    del ix, ip, ic, io, isc

    # the "next" rows of the path: other output kinds and layouts
    modes = {}
    for name, mode, gm in (("fp8_group_major", "fp8", True), ("ue8m0", "ue8m0", False),
                           ("ue8m0_group_major", "ue8m0", True), ("bf16", "bf16", False),
                           ("fp8_scales_transposed", "fp8", False),
                           ("ue8m0_scales_transposed", "ue8m0", False)):
        mo, ms = rq.empty_outputs(n, h // hpg, hpg, mode, group_major=gm, device=dev)
        if name.endswith("scales_transposed"):  # scales stored [G, hpg*4, N]
            ms = torch.empty((h // hpg, ms.shape[2], n), dtype=ms.dtype, device=dev).permute(2, 0, 1)
        us = span_us(lambda: rq.inv_rope_quant(x, pos, cache, hpg, mode=mode, out=mo, scales=ms),
                     args.mode_launches, name)
        mb = W.inverse_bytes(n, h, mode)
        modes[name] = {"us": round(us, 2), "bytes": mb, "GBs": round(mb / us / 1e3, 1),
                       "frac_of_measured_peak": round(mb / us / 1e3 / peak, 4)}
        del mo, ms
    res["output_modes"] = {"call": "rq_inv_rope_quant_layout (heads_per_group 8): warp-rows kernel "
                                   "(token-major and contiguous group-major rows), token-tiled "
                                   "layout kernel (fp32 scales stored transposed, [G, hpg*4, N]), "
                                   "warp-rows layout kernel (bf16; UE8M0 words stored transposed, "
                                   "[G, hpg, N])",
                           "launches_each": args.mode_launches, "results": modes}

    # the fused q/kv op (q RMS norm + RoPE into a padded q_out, with the kv insert)
    fi = W.fused_inputs(W.FUSED16K, cache=inv_h["cos_sin_cache"])
    fq, fkv = fi["q"].to(dev), fi["kv"].to(dev)
    fpos, fsl, fkc = fi["positions"].to(dev), fi["slot_mapping"].to(dev), fi["k_cache"].to(dev)
    fqo = torch.empty((fq.shape[0], fi["q_head_padded"], 512), dtype=torch.bfloat16, device=dev)
    fw = W.norm_weight(W.FUSED16K.seed).to(dev)
    us = span_us(lambda: rq.qnorm_rope_kv_rope_quant_insert(
        fq, fkv, fpos, cache, fsl, fkc, fi["block_size"], fi["q_head_padded"], q_out=fqo),
        args.mode_launches, "fused_qkv")
    us_w = span_us(lambda: rq.qnorm_rope_kv_rope_quant_insert(
        fq, fkv, fpos, cache, fsl, fkc, fi["block_size"], fi["q_head_padded"], q_out=fqo,
        norm_weight=fw), args.mode_launches, "fused_qkv_weighted")
    fb = W.fused_bytes(W.FUSED16K.n_tokens, W.FUSED16K.n_heads_q, W.FUSED16K.q_head_padded)
    res["fused_qkv"] = {"kernel": "qnorm_rope_kv_insert_kernel", "workload": "fused16k (N=16384, "
                        "Hq=32 padded to 64, kv into 512x64 slots)", "us": round(us, 2),
                        "bytes": fb, "GBs": round(fb / us / 1e3, 1),
                        "frac_of_measured_peak": round(fb / us / 1e3 / peak, 4),
                        "with_norm_weight": {"us": round(us_w, 2),
                                             "frac_of_measured_peak":
                                                 round(fb / us_w / 1e3 / peak, 4),
                                             "what": "synthetic bf16 RMSNorm weight [512] on q"},
                        "launches": args.mode_launches}
    del fq, fkv, fpos, fsl, fkc, fqo, fw

    # the indexer q op (RoPE through bf16 + per-head FP8 + scale fold)
    xi = W.indexer_inputs(W.INDEXER16K, cache=inv_h["cos_sin_cache"])
    iq, iw, ipos = xi["q"].to(dev), xi["weights"].to(dev), xi["positions"].to(dev)
    ico = torch.empty((iq.shape[0], iq.shape[1], 128), dtype=torch.uint8, device=dev)
    iwo = torch.empty((iq.shape[0], iq.shape[1]), dtype=torch.float32, device=dev)
    indexer = {}
    ib = W.indexer_bytes(W.INDEXER16K.n_tokens, W.INDEXER16K.n_heads)
    for style in ("neox", "gptj"):
        us = span_us(lambda: rq.indexer_q_rope_quant(iq, ipos, cache, iw, xi["softmax_scale"],
                                                     xi["head_scale"], rope_style=style, out=ico,
                                                     weights_out=iwo), args.mode_launches,
                     f"indexer_{style}")
        indexer[style] = {"us": round(us, 2), "bytes": ib, "GBs": round(ib / us / 1e3, 1),
                          "frac_of_measured_peak": round(ib / us / 1e3 / peak, 4)}
    res["indexer_q"] = {"kernel": "indexer_q_rope_quant_fixed_kernel", "workload": "indexer16k "
                        "(N=16384, H=64, head 128, dims 0..63 rotary)",
                        "launches_each": args.mode_launches, "results": indexer}
    del iq, iw, ipos, ico, iwo

    res["consumer_gemm"] = gemm_leg(args, rq, dev, x, pos, cache, hpg, out, scales, span_us)
    res["consumer_gemm"]["decode"] = decode_gemm_leg(rq, dev, stream, inv_h, cache)
    res["decode_latency"] = decode_leg(rq, dev, stream, inv_h, cache)
    res["small_configs_cold"] = cold_leg(rq, dev, stream, inv_h, cache, kv, kpos, slots, k_cache, bs)
    return res


def gemm_leg(args, rq, dev, x, pos, cache, hpg, out, scales, span_us):
    """The consumer of the op's output: grouped FP8 GEMM (wo_a-style), 4 groups
    x K = 4096, n_out = 1024 per group, on the tensor cores (tcgen05). The
    measured path of the row is the op's UE8M0 mode followed by the
    block-scaled GEMM; the fp32-scale GEMM and the fused kernel are reported
    beside it."""
    n, h = x.shape[0], x.shape[1]
    g_out = 1024
    gen = torch.Generator().manual_seed(7)
    wc = torch.randint(0, 256, (h // hpg, g_out, hpg * 512), generator=gen,
                       dtype=torch.int32).to(torch.uint8)
    wc[(wc & 0x7F) == 0x7F] = 0x38
    wc = wc.to(dev)
    ws = (2.0 ** torch.randint(-10, -6, (h // hpg, g_out // 128, hpg * 4), generator=gen)
          .float()).to(dev)
    gy = torch.empty((n, h // hpg, g_out), dtype=torch.bfloat16, device=dev)
    gl = max(10, args.mode_launches // 6)
    flop = 2.0 * n * h * 512 * g_out
    fp8_peak, fp8_src = measured_tensor_peak_fp8()

    def roof(us):
        return {"bound": "tensor", "achieved": round(flop / us / 1e6, 1), "peak": fp8_peak,
                "unit": "TFLOP/s", "frac": round(flop / us / 1e6 / fp8_peak, 4),
                "peak_source": fp8_src}

    # the row's path: the op writes token-major codes + packed UE8M0 words,
    # the block-scaled MMA reads them as they are
    mx_codes = torch.empty_like(out)
    mx_words = torch.empty((n, h // hpg, hpg), dtype=torch.int32, device=dev)
    w_sf = (torch.log2(ws).round().to(torch.int32) + 127).to(torch.uint8)

    def op_ue8m0():
        rq.inv_rope_quant(x, pos, cache, hpg, mode="ue8m0", out=mx_codes, scales=mx_words)

    def mx_call():
        rq.grouped_fp8_gemm_ue8m0(mx_codes, mx_words, wc, w_sf, out=gy)

    op_ue8m0()
    us_op = span_us(op_ue8m0, gl, "gemm_path_op")
    us_mx = span_us(mx_call, gl, "gemm_ue8m0")
    us_pair = span_us(lambda: (op_ue8m0(), mx_call()), gl, "gemm_path_pair")

    rq.inv_rope_fp8_quant(x, pos, cache, hpg, out=out, scales=scales)
    us = span_us(lambda: rq.grouped_fp8_gemm(out, scales, wc, ws, out=gy), gl, "gemm_fp32")
    us_fused = span_us(lambda: rq.inv_rope_fp8_quant_gemm(x, pos, cache, hpg, wc, ws, out=gy),
                       max(5, gl // 4), "gemm_fused")
    del mx_codes, mx_words, wc, ws, gy
    return {"workload": f"grouped FP8 GEMM: M={n}, G={h // hpg}, K={hpg * 512}, n_out={g_out} "
                        "per group, block scales 1x128 (A) / 128x128 (W)", "flop": flop,
            "launches": gl,
            "path": {"what": "the row's measured path: rq_inv_rope_quant_layout in UE8M0 mode "
                             "(token-major) then rq_grouped_fp8_gemm_ue8m0 on its output",
                     "op_us": round(us_op, 2), "gemm_us": round(us_mx, 2),
                     "op_then_gemm_us": round(us_pair, 2)},
            "ue8m0": {"kernel": "grouped_fp8_gemm_ue8m0_kernel",
                      "what": "UE8M0 block scales (the op's packed-scale output) applied inside "
                              "the block-scaled MMA (tcgen05 kind::mxf8f6f4)",
                      "us": round(us_mx, 2), "roofline": roof(us_mx)},
            "fp32_scales": {"kernel": "grouped_fp8_gemm_kernel",
                            "what": "fp32 block scales folded per K tile in registers",
                            "us": round(us, 2), "roofline": roof(us)},
            "fused": {"kernel": "fused_inv_rope_quant_gemm_kernel",
                      "what": "inverse RoPE + block-FP8 quant produced inside the fp32-scale GEMM "
                              "from bf16 x (not the default: slower than op + GEMM)",
                      "us": round(us_fused, 2), "roofline": roof(us_fused)}}


def decode_leg(rq, dev, stream, inv_h, cache):
    """Decode-sized calls (N tokens x 32 heads), hot: device time per call from
    CUDA-graph replays of 100 back-to-back calls (host launch cost excluded)."""
    decode = {}
    for nt in W.DECODE_TOKENS:
        di = W.inverse_inputs(W.decode_spec(nt), cache=inv_h["cos_sin_cache"])
        dx, dp = di["x"].to(dev), di["positions"].to(dev)
        do = torch.empty((nt, 4, 4096), dtype=torch.uint8, device=dev)
        ds = torch.empty((nt, 4, 32), dtype=torch.float32, device=dev)
        rq.inv_rope_fp8_quant(dx, dp, cache, 8, out=do, scales=ds)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            with torch.cuda.graph(g, stream=gs):
                for _ in range(100):
                    rq.inv_rope_fp8_quant(dx, dp, cache, 8, out=do, scales=ds)
        g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        decode[str(nt)] = round(e0.elapsed_time(e1) * 1e3 / 500, 2)
    return {"workload": "decode: N tokens x 32 heads, heads_per_group 8, positions U[0,65536); "
                        "graph of 100 calls, 5 replays", "us_per_call": decode}


def decode_gemm_leg(rq, dev, stream, inv_h, cache, reps=20, rounds=9):
    """The consumer at decode sizes: N = 1, 16, 64 tokens x 32 heads through
    the op's UE8M0 mode and the block-scaled GEMM (4 groups, K 4096, 1024
    outputs per group; up to 64 tokens the GEMM runs its split-K kernel).
    Device time per call from CUDA graphs of `reps` calls: hot (replayed back
    to back) and cold (each call after a 160 MiB write that evicts L2, minus a
    graph of the writes alone, paired replays, median over `rounds`)."""
    gen = torch.Generator().manual_seed(11)
    wc = torch.randint(0, 256, (4, 1024, 4096), generator=gen, dtype=torch.int32).to(torch.uint8)
    wc[(wc & 0x7F) == 0x7F] = 0x38
    wc = wc.to(dev)
    w_sf = torch.randint(118, 124, (4, 8, 32), generator=gen, dtype=torch.int32).to(torch.uint8).to(dev)
    w32 = torch.ldexp(torch.ones((), device=dev), (w_sf.to(torch.int32) - 127).float())
    flush = torch.empty(160 << 20, dtype=torch.uint8, device=dev)

    def graph_of(fn, with_flush):
        g = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            if fn is not None:
                fn()
            with torch.cuda.graph(g, stream=gs):
                for r in range(reps):
                    if with_flush:
                        flush.fill_(r & 0xFF)
                    if fn is not None:
                        fn()
        torch.cuda.synchronize(dev)
        return g

    def once(g):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e3

    base = graph_of(None, True)
    base.replay()
    out = {}
    for nt in (1, 16, 64):
        di = W.inverse_inputs(W.decode_spec(nt), cache=inv_h["cos_sin_cache"])
        dx, dp = di["x"].to(dev), di["positions"].to(dev)
        codes = torch.empty((nt, 4, 4096), dtype=torch.uint8, device=dev)
        words = torch.empty((nt, 4, 8), dtype=torch.int32, device=dev)
        s32 = torch.empty((nt, 4, 32), dtype=torch.float32, device=dev)
        y = torch.empty((nt, 4, 1024), dtype=torch.bfloat16, device=dev)
        op = lambda: rq.inv_rope_quant(dx, dp, cache, 8, mode="ue8m0", out=codes, scales=words)
        gemm = lambda: rq.grouped_fp8_gemm_ue8m0(codes, words, wc, w_sf, out=y)
        pair = lambda: (op(), gemm())
        # the op's default output (fp32 scales) into the fp32-scale GEMM
        op32 = lambda: rq.inv_rope_fp8_quant(dx, dp, cache, 8, out=codes, scales=s32)
        gemm32 = lambda: rq.grouped_fp8_gemm(codes, s32, wc, w32, out=y)
        pair32 = lambda: (op32(), gemm32())
        row = {}
        for name, fn in (("gemm", gemm), ("op_then_gemm", pair), ("gemm_fp32", gemm32),
                         ("op_then_gemm_fp32", pair32)):
            g = graph_of(fn, False)
            g.replay()
            row[name + "_hot"] = round(once(g) / reps, 2)
            g = graph_of(fn, True)
            g.replay()
            diffs = []
            for _ in range(rounds):
                t1 = once(g)
                diffs.append(t1 - once(base))
            row[name + "_cold"] = round(statistics.median(diffs) / reps, 2)
            del g
        out[str(nt)] = row
    del flush, base, wc
    return {"what": "decode: N tokens x 32 heads -> op (UE8M0 words; *_fp32: the default fp32 "
                    "scales) -> grouped GEMM (4 groups, K 4096, 1024 outputs per group), device "
                    "us per call; hot: graphs of "
                    f"{reps} calls back to back; cold: each call after a 160 MiB write, minus "
                    "the writes alone", "kernel": "grouped_fp8_gemm_ue8m0_small_kernel / "
                    "grouped_fp8_gemm_f32_small_kernel (split K over 8-CTA clusters)", "us": out}


def cold_leg(rq, dev, stream, inv_h, cache, kv, kpos, slots, k_cache, bs, reps=20, rounds=15):
    """The configurations that fit in L2, cold. Two CUDA graphs: `reps` x
    (a 160 MiB write that evicts L2, then the call), and the same writes
    alone; they are replayed alternately under event pairs, `rounds` times,
    and the cold time of one call is the median over rounds of (with calls -
    without) / reps (pairing the two replays cancels drift between rounds).
    Launch overhead inside a graph is that of a graph node, so the figure is
    device time."""
    flush = torch.empty(160 << 20, dtype=torch.uint8, device=dev)

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            if fn is not None:
                fn()
            with torch.cuda.graph(g, stream=gs):
                for r in range(reps):
                    flush.fill_(r & 0xFF)
                    if fn is not None:
                        fn()
        torch.cuda.synchronize(dev)
        return g

    def once(g):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e3

    base = graph_of(None)
    base.replay()
    cases = {}
    ti = W.inverse_inputs(W.TINY)
    tx, tp, tc = ti["x"].to(dev), ti["positions"].to(dev), ti["cos_sin_cache"].to(dev)
    cases["tiny (N=64, H=8)"] = lambda: rq.inv_rope_fp8_quant(tx, tp, tc, ti["heads_per_group"])
    dec = {}
    for nt in W.DECODE_TOKENS:
        di = W.inverse_inputs(W.decode_spec(nt), cache=inv_h["cos_sin_cache"])
        dec[nt] = (di["x"].to(dev), di["positions"].to(dev))
    for nt in W.DECODE_TOKENS:
        dx, dp = dec[nt]
        cases[f"decode N={nt}"] = (lambda dx=dx, dp=dp: rq.inv_rope_fp8_quant(dx, dp, cache, 8))
    cases["insert16k"] = lambda: rq.rope_fp8_quant_insert(kv, kpos, cache, slots, k_cache, bs)
    us = {}
    flush_us = []
    for name, fn in cases.items():
        g = graph_of(fn)
        g.replay()
        diffs = []
        for _ in range(rounds):
            t1 = once(g)
            t0 = once(base)
            diffs.append(t1 - t0)
            flush_us.append(t0)
        us[name] = round(statistics.median(diffs) / reps, 2)
        del g
    del flush, base
    return {"what": "device us per call after a 160 MiB write evicts L2: CUDA graphs of "
                    f"{reps} x (write, call) and {reps} x (write) replayed alternately, median "
                    f"over {rounds} rounds of the difference / {reps}",
            "flush_us": round(statistics.median(flush_us) / reps, 2), "us": us}


def run_e2e(args, rq, dev, stream, world, inv_h, ins_h, cache, hpg, out, scales, kv, kpos, slots,
            k_cache, bs):
    """The same step end to end through the public API from pinned host buffers."""
    e2e_steps = args.e2e_steps or min(args.steps, 20)
    x_host = inv_h["x"].pin_memory()
    pos_host = inv_h["positions"].pin_memory()
    kv_host = ins_h["kv"].pin_memory()
    kpos_host = ins_h["positions"].pin_memory()
    slots_host = ins_h["slot_mapping"].pin_memory()
    out_host = torch.empty(out.shape, dtype=torch.uint8).pin_memory()
    scales_host = torch.empty(scales.shape, dtype=torch.float32).pin_memory()
    kc_host = torch.empty(k_cache.shape, dtype=torch.uint8).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (x_host, pos_host, kv_host, kpos_host, slots_host))
    d2h = sum(t.numel() * t.element_size() for t in (out_host, scales_host, kc_host))
    step_bytes = W.inverse_bytes(inv_h["x"].shape[0], inv_h["x"].shape[1]) + INS_BYTES

    # the inverse op goes through the host-buffer C-ABI call (chunked copy-in /
    # kernel / copy-out pipeline inside the library); the insert's inputs are
    # copied in and the paged cache read back around its device call
    ws = torch.empty(rq.host_workspace_bytes(inv_h["x"].shape[1], args.e2e_chunk),
                     dtype=torch.uint8, device=dev)

    # the insert (its copies, kernel and cache readback) runs on a second
    # stream, overlapping the inverse pipeline's transfers; both join the
    # timed stream at the end of every step
    side = torch.cuda.Stream(device=dev)

    def e2e_step():
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            kv.copy_(kv_host, non_blocking=True)
            kpos.copy_(kpos_host, non_blocking=True)
            slots.copy_(slots_host, non_blocking=True)
            rq.rope_fp8_quant_insert(kv, kpos, cache, slots, k_cache, bs)
            kc_host.copy_(k_cache, non_blocking=True)
        rq.inv_rope_fp8_quant_host(x_host, pos_host, cache, hpg, out=out_host, scales=scales_host,
                                   workspace=ws, chunk_tokens=args.e2e_chunk)
        stream.wait_stream(side)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    del ws
    return {
        "value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 3),
        "unit": "GB/s",
        "ms_per_step": round(e2e_ms, 3),
        "h2d_bytes_per_step": h2d,
        "d2h_bytes_per_step": d2h,
        "steps": e2e_steps,
        "path": "inverse: rq_inv_rope_fp8_quant_host (pinned host buffers; chunked copy-in / "
                "kernels / copy-out pipeline over a device workspace, "
                f"{args.e2e_chunk} tokens per chunk); insert, on a second stream: pinned "
                "host -> device copies, the device call, paged cache -> pinned host",
    }


def _committed_traffic():
    """dram bytes per launch of the inverse kernel from the committed ncu summary
    (profiles/inv_rope_fp8_quant_prefill16k.md), or None when absent or taken
    on another kernel than the one the bench times."""
    path = os.path.join(ROOT, "profiles", "inv_rope_fp8_quant_prefill16k.md")
    kernel, value = None, None
    try:
        with open(path) as f:
            for line in f:
                if line.startswith("traffic_kernel:"):
                    kernel = line.split(":", 1)[1].strip()
                if line.startswith("traffic_bytes_per_launch:"):
                    v = line.split(":", 1)[1].strip()
                    value = None if v in ("", "null") else int(float(v))
    except OSError:
        return None
    return value if kernel == INV_KERNEL_NAME else None


# ------------------------------------------------------------------ reference arm

def run_reference(args, world, rank):
    """The CPU oracle timed on the host cores, on a bounded sample per step
    (the same warm-mean method as cpu_baseline)."""
    threads = os.cpu_count() or 1
    inv_h, ins_h = make_inputs()
    warm = max(3, args.warmup)
    total_steps = args.steps + warm
    # ~13 us of CPU per (token, head) row: size the sample to the time budget
    budget_rows = args.ref_budget_s * threads / 13e-6 / max(1, total_steps)
    tokens = int(max(1, min(INV_SPEC.n_tokens, budget_rows // (INV_SPEC.n_heads + 1))))
    value, dt = oracle_step_rate(inv_h, ins_h, tokens, args.steps, warm, threads)
    value = round(value, 4)
    sample_bytes = W.inverse_bytes(tokens, INV_SPEC.n_heads) + W.insert_bytes(tokens)
    sample = (f"first {tokens} tokens of each op per step (inverse {tokens}x32 heads, "
              f"insert {tokens}); warm mean of {args.steps} steps after {warm} untimed; "
              f"oracle with {threads} threads")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": warm,
        "ms_per_step": round(dt * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in, fp32 math, e4m3 out",
        "data": "synthetic (seeded: randn + 1% x50 outliers, bf16)",
        "config": {"workload": "prefill16k + insert16k (bounded sample, see cpu_baseline)",
                   "sample_tokens": tokens, "bytes_per_step": sample_bytes},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ops --profile-op can run alone (kernel each one launches at these sizes)
PROFILE_OPS = {
    "inverse": "inv_rope_fp8_quant_kernel (warp rows)",
    "inverse_stream": "inv_rope_fp8_quant_stream_kernel (RQ_INV_STREAM)",
    "gemm": "grouped_fp8_gemm_kernel (M = tokens, G 4, K 4096, n_out 1024)",
    "gemm_ue8m0": "grouped_fp8_gemm_ue8m0_kernel (same shape)",
    "gemm_fused": "fused_inv_rope_quant_gemm_kernel (same shape, A produced from x in the kernel)",
    "indexer": "indexer_q_rope_quant_kernel (tokens x 64 heads of 128, NeoX)",
    "fused_qkv": "qnorm_rope_kv_insert_kernel (tokens x 32 q heads padded to 64 + kv)",
    "insert": "rope_fp8_quant_insert_kernel (tokens into 512 x 64 slots)",
    "gemm_decode": "grouped_fp8_gemm_ue8m0_small_kernel after the op's UE8M0 mode (tokens x 32 "
                   "heads, at most 64 tokens; default 1)",
    "layout_transposed": "the layout kernel for fp32 scales stored [G, hpg*4, N] (token-tiled "
                         "from 8192 tokens x 32 heads, fixed-head below)",
}


def run_profile_op(args):
    """One op, 3 launches, nothing else: the small case of an ncu capture."""
    import rope_block_fp8_inverse_b300 as rq
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    op = args.profile_op
    n = args.inv_tokens or (1 if op == "gemm_decode" else 4096)
    spec = W.InverseSpec(f"profile{n}", n, INV_SPEC.n_heads, INV_SPEC.heads_per_group,
                         INV_SPEC.cache_rows, "arange", True)
    if op in ("inverse", "inverse_stream", "gemm", "gemm_ue8m0", "gemm_fused"):
        inp = W.inverse_inputs(spec)
        x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
        hpg = spec.heads_per_group
        variant = rq.VARIANT_STREAM if op == "inverse_stream" else rq.VARIANT_AUTO
        if op.startswith("inverse"):
            call = lambda: rq.inv_rope_fp8_quant(x, pos, cache, hpg, variant=variant)
        else:
            g = spec.n_heads // hpg
            gen = torch.Generator().manual_seed(7)
            wc = torch.randint(0, 256, (g, 1024, hpg * 512), generator=gen, dtype=torch.int32)
            wc = wc.to(torch.uint8)
            wc[(wc & 0x7F) == 0x7F] = 0x38
            wc = wc.to(dev)
            e = torch.randint(117, 121, (g, 8, hpg * 4), generator=gen, dtype=torch.int32)
            if op == "gemm":
                codes, scales = rq.inv_rope_fp8_quant(x, pos, cache, hpg)
                ws = torch.ldexp(torch.ones(()), (e - 127).float()).float().to(dev)
                call = lambda: rq.grouped_fp8_gemm(codes, scales, wc, ws)
            elif op == "gemm_fused":
                ws = torch.ldexp(torch.ones(()), (e - 127).float()).float().to(dev)
                call = lambda: rq.inv_rope_fp8_quant_gemm(x, pos, cache, hpg, wc, ws)
            else:
                codes, words = rq.inv_rope_quant(x, pos, cache, hpg, mode="ue8m0")
                wsf = e.to(torch.uint8).to(dev)
                call = lambda: rq.grouped_fp8_gemm_ue8m0(codes, words, wc, wsf)
    elif op == "gemm_decode":
        if n > 64:
            raise SystemExit("gemm_decode takes at most 64 tokens")
        inp = W.inverse_inputs(spec)
        x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
        gen = torch.Generator().manual_seed(7)
        wc = torch.randint(0, 256, (4, 1024, 4096), generator=gen, dtype=torch.int32).to(torch.uint8)
        wc[(wc & 0x7F) == 0x7F] = 0x38
        wc = wc.to(dev)
        wsf = torch.randint(117, 121, (4, 8, 32), generator=gen, dtype=torch.int32).to(torch.uint8).to(dev)
        codes = torch.empty((n, 4, 4096), dtype=torch.uint8, device=dev)
        words = torch.empty((n, 4, 8), dtype=torch.int32, device=dev)

        def call():
            rq.inv_rope_quant(x, pos, cache, 8, mode="ue8m0", out=codes, scales=words)
            rq.grouped_fp8_gemm_ue8m0(codes, words, wc, wsf)
    elif op == "insert":
        ii = W.insert_inputs(W.InsertSpec(f"profile{n}", n, 65536, 512, 64))
        kv, kpos, cache, slots, kc = (ii[k].to(dev) for k in
                                      ("kv", "positions", "cos_sin_cache", "slot_mapping",
                                       "k_cache"))
        call = lambda: rq.rope_fp8_quant_insert(kv, kpos, cache, slots, kc, ii["block_size"])
    elif op == "layout_transposed":
        inp = W.inverse_inputs(spec)
        x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
        hpg = spec.heads_per_group
        g = spec.n_heads // hpg
        mo, _ = rq.empty_outputs(n, g, hpg, "fp8", device=dev)
        ms = torch.empty((g, hpg * 4, n), dtype=torch.float32, device=dev).permute(2, 0, 1)
        call = lambda: rq.inv_rope_quant(x, pos, cache, hpg, mode="fp8", out=mo, scales=ms)
    elif op == "indexer":
        ii = W.indexer_inputs(W.IndexerSpec(f"profile{n}", n, 64, 65536))
        q, w, pos, cache = (ii[k].to(dev) for k in ("q", "weights", "positions", "cos_sin_cache"))
        call = lambda: rq.indexer_q_rope_quant(q, pos, cache, w, ii["softmax_scale"],
                                               ii["head_scale"], rope_style="neox")
    else:
        fi = W.fused_inputs(W.FusedSpec(f"profile{n}", n, 32, 64, 65536, 512, 64))
        fq, fkv, fpos, cache, fsl, fkc = (fi[k].to(dev) for k in
                                          ("q", "kv", "positions", "cos_sin_cache",
                                           "slot_mapping", "k_cache"))
        call = lambda: rq.qnorm_rope_kv_rope_quant_insert(fq, fkv, fpos, cache, fsl, fkc,
                                                          fi["block_size"], fi["q_head_padded"])
    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    print(f"profile-op {op}: 3 launches of {PROFILE_OPS[op]} at {n} tokens", flush=True)
    return 0


def main():
    args = parse()
    if args.profile_op:
        return run_profile_op(args)
    if args.impl == "reference":
        # CPU arm: rank 0 alone times the oracle; other ranks exit without work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, world, rank)), flush=True)
        return 0
    world, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    res = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
