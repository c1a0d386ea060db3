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
            self.error = f"nvml: {type(e).__name__}"

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
                self.error = f"nvidia-smi: {type(e).__name__}"
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


def cpu_baseline(inv, ins):
    """The oracle, as it stands, on the host cores over one full step of the workload."""
    import oracle
    threads = os.cpu_count() or 1
    oracle.build()
    t0 = time.perf_counter()
    oracle.inv_rope_fp8_quant(inv["x"], inv["positions"], inv["cos_sin_cache"],
                              inv["heads_per_group"], threads=threads)
    oracle.rope_fp8_quant_insert(ins["kv"], ins["positions"], ins["cos_sin_cache"],
                                 ins["slot_mapping"], ins["k_cache"], ins["block_size"],
                                 threads=threads)
    dt = time.perf_counter() - t0
    # single-threaded on a quarter of the inverse's tokens (bytes scaled to match)
    q = inv["x"].shape[0] // 4
    t1 = time.perf_counter()
    oracle.inv_rope_fp8_quant(inv["x"][:q], inv["positions"][:q], inv["cos_sin_cache"],
                              inv["heads_per_group"], threads=1)
    dt1 = time.perf_counter() - t1
    one_bytes = W.inverse_bytes(q, inv["x"].shape[1])
    return {"value": round(STEP_BYTES / dt / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": "one full step: inverse 16384 tok x 32 heads + insert 16384 tok",
            "single_thread": {"value": round(one_bytes / dt1 / 1e9, 3), "unit": "GB/s",
                              "cores": 1, "seconds": round(dt1, 3),
                              "sample": f"inverse only, {q} tokens x 32 heads"}}


def run_ours(args, world, rank, local):
    import rope_block_fp8_inverse_b300 as rq
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inv_h, ins_h = make_inputs(args.inv_tokens)
    inv_bytes = W.inverse_bytes(inv_h["x"].shape[0], inv_h["x"].shape[1])
    step_bytes = inv_bytes + INS_BYTES

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

    def step():
        rq.inv_rope_fp8_quant(x, pos, cache, hpg, out=out, scales=scales)
        rq.rope_fp8_quant_insert(kv, kpos, cache, slots, k_cache, bs)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)

    # per-launch timing of the dominant kernel (events on the launching stream)
    inv_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    ins_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    with sampler:
        # the timed steps: one event pair around all of them, so nothing sits
        # between the launches (the insert may start while the inverse drains)
        start.record(stream)
        for i in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        # the same steps again with an event pair around each launch: the
        # per-kernel durations (roofline, percentiles, insert time)
        for i in range(args.steps):
            inv_ev[i][0].record(stream)
            rq.inv_rope_fp8_quant(x, pos, cache, hpg, out=out, scales=scales)
            inv_ev[i][1].record(stream)
            rq.rope_fp8_quant_insert(kv, kpos, cache, slots, k_cache, bs)
            ins_ev[i].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    total_ms = max_over_ranks(start.elapsed_time(end), world)
    inv_ms = statistics.fmean(a.elapsed_time(b) for a, b in inv_ev)
    inv_all = sorted(a.elapsed_time(b) for a, b in inv_ev)
    inv_ms_med = statistics.median(inv_all)
    inv_pct = {f"p{q}": round(inv_all[min(len(inv_all) - 1, int(len(inv_all) * q / 100))] * 1e3, 2)
               for q in (10, 50, 90, 99)}
    inv_pct["max"] = round(inv_all[-1] * 1e3, 2)
    ins_ms = statistics.fmean(inv_ev[i][1].elapsed_time(ins_ev[i]) for i in range(args.steps))
    ms_step = total_ms / args.steps

    def span_us(fn, launches):
        """Mean µs per launch of `launches` back-to-back calls, one event pair
        around all of them on the launching stream (after 3 warm calls)."""
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(launches):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e3 / launches

    # the "next" rows of the path (other output kinds and layouts), outside the
    # step's timed region, each as back-to-back launches
    modes = {}
    for name, mode, gm in ((("fp8_group_major", "fp8", True), ("ue8m0", "ue8m0", False),
                            ("ue8m0_group_major", "ue8m0", True), ("bf16", "bf16", False))
                           if args.mode_launches > 0 else ()):
        mo, ms = rq.empty_outputs(n, h // hpg, hpg, mode, group_major=gm, device=dev)
        us = span_us(lambda: rq.inv_rope_quant(x, pos, cache, hpg, mode=mode, out=mo, scales=ms),
                     args.mode_launches)
        mb = W.inverse_bytes(n, h, mode)
        modes[name] = {"us": round(us, 2), "bytes": mb, "GBs": round(mb / us / 1e3, 1),
                       "frac_of_measured_peak": round(mb / us / 1e3 / measured_peaks()[0], 4)}
        del mo, ms

    # the fused q/kv op (q RMS norm + RoPE into a padded q_out, with the kv insert)
    fused = None
    if args.mode_launches > 0:
        fi = W.fused_inputs(W.FUSED16K, cache=inv_h["cos_sin_cache"])
        fq, fkv = fi["q"].to(dev), fi["kv"].to(dev)
        fpos, fsl, fkc = fi["positions"].to(dev), fi["slot_mapping"].to(dev), fi["k_cache"].to(dev)
        fqo = torch.empty((fq.shape[0], fi["q_head_padded"], 512), dtype=torch.bfloat16, device=dev)

        def fused_call():
            rq.qnorm_rope_kv_rope_quant_insert(fq, fkv, fpos, cache, fsl, fkc, fi["block_size"],
                                               fi["q_head_padded"], q_out=fqo)
        us = span_us(fused_call, args.mode_launches)
        fw = W.norm_weight(W.FUSED16K.seed).to(dev)

        def fused_weighted_call():
            rq.qnorm_rope_kv_rope_quant_insert(fq, fkv, fpos, cache, fsl, fkc, fi["block_size"],
                                               fi["q_head_padded"], q_out=fqo, norm_weight=fw)
        us_w = span_us(fused_weighted_call, args.mode_launches)
        fb = W.fused_bytes(W.FUSED16K.n_tokens, W.FUSED16K.n_heads_q, W.FUSED16K.q_head_padded)
        fused = {"kernel": "qnorm_rope_kv_insert_kernel", "workload": "fused16k (N=16384, Hq=32 "
                 "padded to 64, kv into 512x64 slots)", "us": round(us, 2), "bytes": fb,
                 "GBs": round(fb / us / 1e3, 1),
                 "frac_of_measured_peak": round(fb / us / 1e3 / measured_peaks()[0], 4),
                 "with_norm_weight": {"us": round(us_w, 2),
                                      "frac_of_measured_peak":
                                          round(fb / us_w / 1e3 / measured_peaks()[0], 4),
                                      "what": "synthetic bf16 RMSNorm weight [512] on q"},
                 "launches": args.mode_launches}
        del fq, fkv, fpos, fsl, fkc, fqo, fw

    # the indexer q op (RoPE through bf16 + per-head FP8 + scale fold)
    indexer = None
    if args.mode_launches > 0:
        ii = W.indexer_inputs(W.INDEXER16K, cache=inv_h["cos_sin_cache"])
        iq, iw, ipos = ii["q"].to(dev), ii["weights"].to(dev), ii["positions"].to(dev)
        ico = torch.empty((iq.shape[0], iq.shape[1], 128), dtype=torch.uint8, device=dev)
        iwo = torch.empty((iq.shape[0], iq.shape[1]), dtype=torch.float32, device=dev)
        indexer = {}
        for style in ("neox", "gptj"):
            def idx_call():
                rq.indexer_q_rope_quant(iq, ipos, cache, iw, ii["softmax_scale"], ii["head_scale"],
                                        rope_style=style, out=ico, weights_out=iwo)
            us = span_us(idx_call, args.mode_launches)
            ib = W.indexer_bytes(W.INDEXER16K.n_tokens, W.INDEXER16K.n_heads)
            indexer[style] = {"us": round(us, 2), "bytes": ib, "GBs": round(ib / us / 1e3, 1),
                              "frac_of_measured_peak": round(ib / us / 1e3 / measured_peaks()[0], 4)}
        indexer = {"kernel": "indexer_q_rope_quant_kernel", "workload": "indexer16k (N=16384, "
                   "H=64, head 128, dims 0..63 rotary)", "launches_each": args.mode_launches,
                   "results": indexer}
        del iq, iw, ipos, ico, iwo

    # the consumer: grouped FP8 GEMM (wo_a-style) on the inverse op's own output,
    # 4 groups x K = 4096, n_out = 1024 per group, tensor cores (tcgen05)
    gemm = None
    if args.mode_launches > 0:
        g_out = 1024
        gen = torch.Generator().manual_seed(7)
        wc = torch.randint(0, 256, (h // hpg, g_out, hpg * 512), generator=gen,
                           dtype=torch.int32).to(torch.uint8)
        wc[(wc & 0x7F) == 0x7F] = 0x38
        wc = wc.to(dev)
        ws = (2.0 ** torch.randint(-10, -6, (h // hpg, g_out // 128, hpg * 4), generator=gen)
              .float()).to(dev)
        gy = torch.empty((n, h // hpg, g_out), dtype=torch.bfloat16, device=dev)
        rq.inv_rope_fp8_quant(x, pos, cache, hpg, out=out, scales=scales)

        def gemm_call():
            rq.grouped_fp8_gemm(out, scales, wc, ws, out=gy)
        gl = max(10, args.mode_launches // 6)
        us = span_us(gemm_call, gl)

        def fused_gemm_call():
            rq.inv_rope_fp8_quant_gemm(x, pos, cache, hpg, wc, ws, out=gy)
        us_fused = span_us(fused_gemm_call, gl)

        # the same GEMM on the block-scaled MMA, fed by the op's UE8M0 mode
        # (token-major packed words) and the weight scales as UE8M0 codes
        mx_codes = torch.empty_like(out)
        mx_words = torch.empty((n, h // hpg, hpg), dtype=torch.int32, device=dev)
        rq.inv_rope_quant(x, pos, cache, hpg, mode="ue8m0", out=mx_codes, scales=mx_words)
        w_sf = (torch.log2(ws).round().to(torch.int32) + 127).to(torch.uint8)

        def mx_call():
            rq.grouped_fp8_gemm_ue8m0(mx_codes, mx_words, wc, w_sf, out=gy)
        us_mx = span_us(mx_call, gl)
        del mx_codes, mx_words
        flop = 2.0 * n * h * 512 * g_out
        tf = flop / us / 1e6
        fp8_peak, fp8_src = measured_tensor_peak_fp8()
        gemm = {"kernel": "grouped_fp8_gemm_kernel", "workload": f"grouped FP8 GEMM: M={n}, "
                f"G={h // hpg}, K={hpg * 512}, n_out={g_out} per group, block scales 1x128 / "
                "128x128", "us": round(us, 2), "flop": flop,
                "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": fp8_peak,
                             "unit": "TFLOP/s", "frac": round(tf / fp8_peak, 4),
                             "peak_source": fp8_src},
                "fused": {"kernel": "fused_inv_rope_quant_gemm_kernel",
                          "what": "inverse RoPE + block-FP8 quant produced inside the GEMM "
                                  "from bf16 x (codes never reach HBM)",
                          "us": round(us_fused, 2),
                          "tflops": round(flop / us_fused / 1e6, 1),
                          "frac": round(flop / us_fused / 1e6 / fp8_peak, 4),
                          "unfused_op_plus_gemm_us": round(inv_ms * 1e3 + us, 2)},
                "ue8m0": {"kernel": "grouped_fp8_gemm_ue8m0_kernel",
                          "what": "UE8M0 block scales (the op's packed-scale output) applied "
                                  "inside the block-scaled MMA (tcgen05 kind::mxf8f6f4)",
                          "us": round(us_mx, 2),
                          "roofline": {"bound": "tensor", "achieved": round(flop / us_mx / 1e6, 1),
                                       "peak": fp8_peak, "unit": "TFLOP/s",
                                       "frac": round(flop / us_mx / 1e6 / fp8_peak, 4),
                                       "peak_source": fp8_src}},
                "launches": gl}
        del wc, ws, gy

    # decode-sized calls (N tokens x 32 heads): device time per call, taken from
    # CUDA-graph replays of 100 back-to-back calls (host launch cost excluded)
    decode = None
    if args.mode_launches > 0:
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
        decode = {"workload": "decode: N tokens x 32 heads, heads_per_group 8, positions "
                  "U[0,65536); graph of 100 calls, 5 replays", "us_per_call": decode}

    # the configurations that fit in L2, cold: each call after a 256 MiB write
    # that evicts L2, one event pair around the call (median of 20); the hot
    # figures are the graph replays above and the in-step insert
    small_cold = None
    if args.mode_launches > 0:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def cold_us(fn, reps=20):
            fn()
            ts = []
            for r in range(reps):
                flush.fill_(r & 0xFF)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize(dev)
                ts.append(a.elapsed_time(b) * 1e3)
            return round(statistics.median(ts), 2)
        small_cold = {}
        ti = W.inverse_inputs(W.TINY)
        tx, tp, tc = ti["x"].to(dev), ti["positions"].to(dev), ti["cos_sin_cache"].to(dev)
        small_cold["tiny (N=64, H=8)"] = cold_us(
            lambda: rq.inv_rope_fp8_quant(tx, tp, tc, ti["heads_per_group"]))
        for nt in (1, 8, 64):
            di = W.inverse_inputs(W.decode_spec(nt), cache=inv_h["cos_sin_cache"])
            dx, dp = di["x"].to(dev), di["positions"].to(dev)
            small_cold[f"decode N={nt}"] = cold_us(lambda: rq.inv_rope_fp8_quant(dx, dp, cache, 8))
        small_cold["insert16k"] = cold_us(
            lambda: rq.rope_fp8_quant_insert(kv, kpos, cache, slots, k_cache, bs))
        small_cold = {"what": "median us per call after evicting L2 (cold); event pair around "
                              "the call", "us": small_cold}
        del flush

    # end to end through the public API from pinned host buffers
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

    # the inverse op goes through the host-buffer C-ABI call (chunked copy-in /
    # kernel / copy-out pipeline inside the library); the insert's inputs are
    # copied in and the paged cache read back around its device call
    ws = torch.empty(rq.host_workspace_bytes(h, args.e2e_chunk), dtype=torch.uint8, device=dev)

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

    peak, peak_src = measured_peaks()
    achieved = inv_bytes / (inv_ms * 1e-3) / 1e9
    traffic = _committed_traffic()
    result = {
        "metric": METRIC,
        "value": round(world * step_bytes / (ms_step * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "inverse_us": round(inv_ms * 1e3, 2),
        "inverse_us_median": round(inv_ms_med * 1e3, 2),
        "inverse_us_percentiles": inv_pct,
        "insert_us": round(ins_ms * 1e3, 2),
        "per_launch_timing": "inverse_us, insert_us, percentiles and roofline.achieved come from "
                             "a second pass of the same steps with an event pair around each "
                             "launch; value and ms_per_step from the timed steps (one event pair "
                             "around all of them)",
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
        },
        "e2e": {
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
        },
        "gpu_launches": 2 * args.steps,
        "secondary_timing": "output_modes, fused_qkv, indexer_q and consumer_gemm: one event pair "
                            "around N back-to-back launches, mean per launch",
        "output_modes": {"kernel": "rq_inv_rope_quant_layout (heads_per_group 8): "
                                   "inv_rope_fp8_quant_kernel for token-major UE8M0, "
                                   "inv_rope_fp8_quant_stream_kernel for group-major fp8 / "
                                   "UE8M0, inv_rope_quant_layout_kernel<1> for bf16",
                         "launches_each": args.mode_launches,
                         "results": modes},
        "fused_qkv": fused,
        "indexer_q": indexer,
        "decode_latency": decode,
        "small_configs_cold": small_cold,
        "consumer_gemm": gemm,
        "clocks": sampler.summary(),
    }
    if args.inv_tokens and args.inv_tokens != INV_SPEC.n_tokens:
        result["config"]["workload"] = (f"profiling case: inverse N={args.inv_tokens},H=32,hpg=8 "
                                        "+ insert16k (not the benchmarked configuration)")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inv_h, ins_h)
    return result


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
    """The CPU oracle timed on the host cores, on a bounded sample per step."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    inv_h, ins_h = make_inputs()
    total_steps = args.steps + max(3, args.warmup)
    # ~13 us of CPU per (token, head) row: size the sample to the time budget
    budget_rows = args.ref_budget_s * threads / 13e-6 / max(1, total_steps)
    tokens = int(max(1, min(INV_SPEC.n_tokens, budget_rows // (INV_SPEC.n_heads + 1))))
    xi, pi = inv_h["x"][:tokens].contiguous(), inv_h["positions"][:tokens].contiguous()
    kv, kp, sl = (ins_h["kv"][:tokens].contiguous(), ins_h["positions"][:tokens].contiguous(),
                  ins_h["slot_mapping"][:tokens].contiguous())
    cache = inv_h["cos_sin_cache"]
    sample_bytes = W.inverse_bytes(tokens, INV_SPEC.n_heads) + W.insert_bytes(tokens)

    def step():
        oracle.inv_rope_fp8_quant(xi, pi, cache, inv_h["heads_per_group"], threads=threads)
        oracle.rope_fp8_quant_insert(kv, kp, cache, sl, ins_h["k_cache"], ins_h["block_size"],
                                     threads=threads)

    for _ in range(max(3, args.warmup)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = round(sample_bytes / dt / 1e9, 4)
    sample = (f"first {tokens} tokens of each op per step (inverse {tokens}x32 heads, "
              f"insert {tokens}); oracle with {threads} threads")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
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
    "indexer": "indexer_q_rope_quant_kernel (tokens x 64 heads of 128, NeoX)",
    "fused_qkv": "qnorm_rope_kv_insert_kernel (tokens x 32 q heads padded to 64 + kv)",
}


def run_profile_op(args):
    """One op, 3 launches, nothing else: the small case of an ncu capture."""
    import rope_block_fp8_inverse_b300 as rq
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = args.inv_tokens or 4096
    spec = W.InverseSpec(f"profile{n}", n, INV_SPEC.n_heads, INV_SPEC.heads_per_group,
                         INV_SPEC.cache_rows, "arange", True)
    op = args.profile_op
    if op in ("inverse", "inverse_stream", "gemm", "gemm_ue8m0"):
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
            else:
                codes, words = rq.inv_rope_quant(x, pos, cache, hpg, mode="ue8m0")
                wsf = e.to(torch.uint8).to(dev)
                call = lambda: rq.grouped_fp8_gemm_ue8m0(codes, words, wc, wsf)
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
