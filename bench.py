"""Benchmark of the MXFP4 latent-MoE layer on one GB300 (one JSON line).

One step = one pass of the whole layer (route, group, quantise, stage-1 GEMM
+ GLU + requant, stage-2 GEMM, combine) over one batch of synthetic tokens of
the chosen workload. The headline is the largest workload,
prefill_outlier_t32768 (T=32768, d=3584, E=896, k=16, I=3072, 1% of the rows
scaled by 64); the other full-size workloads are measured in the same run and
reported under per_workload.

  value      tokens/s, device-timed with CUDA events around K moe_forward
             calls, inputs resident in HBM.
  e2e        the same metric through the layer's HostPipeline: every step's
             inputs copied from pinned host memory and its output read back,
             the copies on two copy streams overlapping the neighbouring
             steps' forwards (e2e_serial: the same in one stream; e2e_graph:
             serial copies around a replayed CUDA graph of the step).
  roofline   the dominant kernel: algorithmic bytes (HBM-bound workloads) or
             FLOPs (tensor-bound) per launch / its mean event-timed duration,
             against MEASURED_PEAKS.json.
  cpu_baseline  the CPU oracle (test infrastructure) timed on the host cores on
             a bounded sample of the headline workload.

The layer runs on one GPU; --gpus other than 1 is refused before any GPU
work. --impl reference runs the oracle itself as the reference arm.
"""
import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and % roofline (HBM GB/s decode, tensor TFLOP/s prefill), 1xGB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 4.5 / 2.25   # nominal dense ratio: kind::mxf8f6f4 runs at the FP8 rate
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio: kind::mxf4 (A4W4 stage 1) runs at the FP4 rate
# Measured on GB300 with a tensor-rate probe: an M=128, N=256 MMA issues every
# 128 cycles in both kind::mxf8f6f4 (K=32) and kind::mxf4 (K=64), i.e. the
# MXFP4 x MXFP4 rate is 2x the MXFP8 x MXFP4 rate, bf16 x 4 (not the nominal 6).
FP4_MMA_OVER_BF16 = 2 * FP8_OVER_BF16


# The other full-size workloads, measured in the same run as the headline:
# the two decode batches, the skewed prefill, and the A4W4 stage 1 at prefill.
DEFAULT_PER_WORKLOAD = ("decode_t64,decode_t512,prefill_skewed_t8192,"
                        "prefill_skewed_t8192:a4w4,prefill_outlier_t32768:a4w4")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill_outlier_t32768",
                    help="headline workload (default: the largest, T=32768)")
    ap.add_argument("--per-workload", default=DEFAULT_PER_WORKLOAD,
                    help="comma list of further workloads measured in the same run "
                         "(name or name:a4w4; 'none' for none)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override: T tokens at the full layer dims, uniform routing")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=0, help="oracle tokens (0 = automatic)")
    ap.add_argument("--gemm-kernel", default="auto", choices=["auto", "token", "weight", "pair"],
                    help="grouped-GEMM family (auto = the library's default for the shape)")
    ap.add_argument("--step", default="", choices=["", "router", "latent_down", "latent_up",
                                                   "shared_experts", "block"],
                    help="time one neighbouring BF16 step at the workload's T instead of the layer")
    ap.add_argument("--a4w4", action="store_true",
                    help="MXFP4 stage-1 activations (moe_forward_a4w4); the family is stage 2's")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Clocks over [t0, t1] (wall-clock seconds; default: the first to the
        last mark), padded by one sampling period on each side."""
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        if t0 is None:
            t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, 1e30)
        rows = [r for t, r in self.rows if t0 - 0.25 <= t <= t1 + 0.25] or [r for _, r in self.rows]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# Kernel source files per GEMM family: a committed traffic figure is only used
# while these files are unchanged since its capture.
FAMILY_SOURCES = {
    "token_tiles": ["mxfp4_latent_moe_gb300/csrc/gemm.cu",
                    "mxfp4_latent_moe_gb300/csrc/gemm_token_pair.cu",
                    "mxfp4_latent_moe_gb300/csrc/common.cuh"],
    "weight_tiles": ["mxfp4_latent_moe_gb300/csrc/gemm_decode.cu",
                     "mxfp4_latent_moe_gb300/csrc/common.cuh"],
    "pair_tiles": ["mxfp4_latent_moe_gb300/csrc/gemm_pair.cu",
                   "mxfp4_latent_moe_gb300/csrc/common.cuh"],
}


def profiled_traffic(kernel, workload, family):
    """DRAM bytes per launch of `kernel` (GEMM family `family`) from the
    committed ncu summary, if it was taken on the current kernel source; None
    otherwise."""
    src_hash = source_hash(FAMILY_SOURCES[family])
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("kernel_family") != family or e.get("source_hash") != src_hash:
        return None
    return e.get("dram_bytes_per_launch")


def oracle_inputs(L, n_tokens):
    """Host copies of the first n_tokens of the workload and of all weights."""
    from mxfp4_latent_moe_gb300 import synth
    xb = synth.bf16_bits(L["x"][:n_tokens])
    lg = L["logits"][:n_tokens].cpu().numpy()
    W = [L[n].cpu().numpy() for n in ("w13", "w13_s", "w2", "w2_s")]
    return xb, lg, W


def cpu_model():
    """The host CPU's name (x86 `model name`; Arm implementer/part codes)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
    except OSError:
        return platform.machine()
    for line in info:
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    fields = {}
    for line in info:
        if ":" in line:
            key, val = (x.strip() for x in line.split(":", 1))
            fields.setdefault(key, val)
    if "CPU part" in fields:
        return "%s (implementer %s, part %s)" % (platform.machine(),
                                                fields.get("CPU implementer", "?"),
                                                fields["CPU part"])
    return platform.machine()


def oracle_seconds(wl, host, threads, a4w4=False):
    """Time the CPU oracle, as it stands, on the prepared token sample."""
    import oracle
    xb, lg, W = host
    t0 = time.perf_counter()
    oracle.moe_forward(xb, lg, wl.k, *W, threads=threads, a4w4=a4w4)
    return time.perf_counter() - t0


def run_reference(args, wl):
    if int(os.environ.get("RANK", "0")) != 0:
        return   # under torchrun only rank 0 runs the (CPU) reference arm
    import torch
    from mxfp4_latent_moe_gb300 import synth
    import oracle
    oracle.build_oracle()
    cores = os.cpu_count() or 1
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    L = synth.make_layer(wl, seed=args.seed, device=dev)
    if args.cpu_sample:
        n = args.cpu_sample
    else:  # size the per-step sample so the whole run takes about 150 s
        n0 = min(wl.T, cores)
        per_token = oracle_seconds(wl, oracle_inputs(L, n0), cores, args.a4w4) / n0
        n = max(1, min(wl.T, int(150.0 / (args.steps + args.warmup) / per_token)))
    host = oracle_inputs(L, n)
    del L
    times = []
    for i in range(args.warmup + args.steps):
        dt = oracle_seconds(wl, host, cores, args.a4w4)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = n * len(times) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k, "I": wl.I,
                   "a4w4": bool(args.a4w4)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "first %d tokens of the workload per step, full layer" % n,
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# The neighbouring BF16 steps at the layer's sizes: (name, [(N, K, epilogue)] per GEMM call),
# hidden 7,168, latent 3,584, 896 experts; shared experts: 2 x (7,168 -> 3,072 -> 7,168).
HIDDEN, LATENT, SHARED_I, N_SHARED = 7168, 3584, 3072, 2
BF16_STEPS = {
    "router": [(896, HIDDEN, 0)],
    "latent_down": [(LATENT, HIDDEN, 1)],
    "latent_up": [(HIDDEN, LATENT, 1)],
    "shared_experts": [(2 * SHARED_I, HIDDEN, 2), (HIDDEN, SHARED_I, 1)] * N_SHARED,
}


def run_step(args, wl):
    """Times one neighbouring BF16 step (moe_gemm_bf16 calls) on T tokens."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_latent_moe_gb300 import abi
    dev = torch.device("cuda", 0)
    T = wl.T
    calls = BF16_STEPS[args.step]
    g = torch.Generator(device=dev).manual_seed(args.seed)
    bufs = []
    for i, (N, K, epi) in enumerate(calls):
        a_rows = T
        a = (torch.randn(a_rows, K, generator=g, device=dev)).to(torch.bfloat16)
        b = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
        n_out = N // 2 if epi == 2 else N
        c = torch.empty(T, n_out, dtype=torch.float32 if epi == 0 else torch.bfloat16, device=dev)
        bufs.append((a, b, c, N, K, epi))
    ws = torch.zeros(max(abi.moe_gemm_bf16_workspace_size(T, N, K, epi)
                         for _, _, _, N, K, epi in bufs), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        for a, b, c, N, K, epi in bufs:
            abi.moe_gemm_bf16(a, b, T, N, K, epi, c, ws)

    sampler = ClockSampler(0)
    sampler.start()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    sampler.mark()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[2 * i].record(stream)
        step()
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    if abi.moe_check_device_status(ws) != abi.OK:
        raise RuntimeError("device status error")
    total_ms = sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps))
    ms = total_ms / args.steps
    flops = sum(2.0 * T * N * K for _, _, _, N, K, _ in bufs)
    w_bytes = sum(N * K * 2 for _, _, _, N, K, _ in bufs)
    io_bytes = sum(T * K * 2 + T * (N // 2 if epi == 2 else N) * (4 if epi == 0 else 2)
                   for _, _, _, N, K, epi in bufs)
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    t_mem = (w_bytes + io_bytes) / (hbm * 1e9)
    t_math = flops / (bf16 * 1e12)
    bound = "hbm" if t_mem >= t_math else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": (w_bytes + io_bytes) / (ms / 1e3) / 1e9, "peak": hbm,
                "unit": "GB/s", "algorithmic_bytes": w_bytes + io_bytes}
    else:
        roof = {"bound": "tensor", "achieved": flops / (ms / 1e3) / 1e12, "peak": bf16,
                "unit": "TFLOP/s", "algorithmic_flops": flops}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = peak_src
    roof["traffic"] = None
    # oracle on a bounded sample of rows
    import oracle
    oracle.build_oracle()
    n = 2
    t0 = time.perf_counter()
    for a, b, c, N, K, epi in bufs:
        ab = a[:n].cpu().view(torch.int16).numpy().view("uint16")
        bb = b.cpu().view(torch.int16).numpy().view("uint16")
        (oracle.gemm_bf16_swiglu if epi == 2 else oracle.gemm_bf16)(ab, bb)
    dt = time.perf_counter() - t0
    splits = [abi.moe_gemm_bf16_workspace_size(T, N, K, epi) > 256 for _, _, _, N, K, epi in bufs]
    line = {
        "metric": "BF16 %s step tokens/s (neighbouring step of the MoE layer), 1xGB300" % args.step,
        "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16xbf16->f32", "data": "synthetic (seeded N(0,1) "
        "activations, N(0,0.02) weights)",
        "config": {"workload": "%s_t%d" % (args.step, T), "T": T,
                   "gemms": [[N, K, ["f32", "bf16", "swiglu_bf16"][epi]] for _, _, _, N, K, epi in bufs],
                   "split_k": splits,
                   "l2": "L2 flushed between steps (256 MB write)"},
        "roofline": roof, "gpu_launches": (len(bufs) + sum(splits)) * args.steps,
        "tflops": flops / (ms / 1e3) / 1e12,
        "cpu_baseline": {"value": n / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "%d tokens, all GEMMs of the step (%.1f s)" % (n, dt),
                         "cpu_model": cpu_model()},
        "clocks": sampler.summary(),
    }
    print(json.dumps(line))


def run_block(args, wl):
    """Times the composed block (moe_block_forward) at the workload's T and
    full dims: shared experts on a second stream, the same call on one stream,
    and each part alone; reports the overlap gain."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_latent_moe_gb300 import abi, synth
    from mxfp4_latent_moe_gb300.layer import MoeBlock
    dev = torch.device("cuda", 0)
    T = wl.T
    bw = synth.block_shape("block_t%d" % T, T=T, hidden=2 * wl.d, d=wl.d, E=wl.E, k=wl.k, I=wl.I,
                           shared_I=2 * wl.I)
    B = synth.make_block(bw, seed=args.seed, device=dev)
    blk = MoeBlock(B["w_down"], B["w_router"], B["w_shared13"], B["w_out"], B["w13"], B["w13_s"],
                   B["w2"], B["w2_s"], k=bw.k)
    ws = blk.workspace(T)
    out = torch.empty(T, bw.hidden, dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream(dev)
    stream = torch.cuda.current_stream()
    L = blk.layer
    # the parts, on their own buffers
    x = torch.empty(T, bw.d, dtype=torch.bfloat16, device=dev)
    logits = torch.empty(T, bw.E, dtype=torch.float32, device=dev)
    ylat = torch.empty(T, bw.d, dtype=torch.bfloat16, device=dev)
    hs = torch.empty(T, bw.shared_I, dtype=torch.bfloat16, device=dev)
    gws = torch.zeros(max(abi.moe_gemm_bf16_workspace_size(T, n, kk, e) for n, kk, e in (
        (bw.d, bw.hidden, 1), (bw.E, bw.hidden, 0), (2 * bw.shared_I, bw.hidden, 2),
        (bw.hidden, bw.d + bw.shared_I, 1))), dtype=torch.uint8, device=dev)
    lws = L.workspace(T)
    blk.forward(B["h"], ws=ws, out=out, shared_stream=side)
    abi.moe_gemm_bf16(B["h"], B["w_down"], T, bw.d, bw.hidden, 1, x, gws)
    abi.moe_gemm_bf16(B["h"], B["w_router"], T, bw.E, bw.hidden, 0, logits, gws)
    parts = {
        "down_and_router": lambda: (
            abi.moe_gemm_bf16(B["h"], B["w_down"], T, bw.d, bw.hidden, 1, x, gws),
            abi.moe_gemm_bf16(B["h"], B["w_router"], T, bw.E, bw.hidden, 0, logits, gws)),
        "routed_experts": lambda: L.forward(x, logits, ws=lws, y=ylat),
        "shared_experts": lambda: abi.moe_gemm_bf16(B["h"], B["w_shared13"], T,
                                                    2 * bw.shared_I, bw.hidden, 2, hs, gws),
        "output_gemm": lambda: abi.moe_gemm_bf16_cat(ylat, bw.d, hs, bw.shared_I, B["w_out"], T,
                                                     bw.hidden, 1, out, gws),
        "block_one_stream": lambda: blk.forward(B["h"], ws=ws, out=out),
        "block_two_streams": lambda: blk.forward(B["h"], ws=ws, out=out, shared_stream=side),
    }
    sampler = ClockSampler(0)
    sampler.start()
    ms = {}
    for name, fn in parts.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if name == "block_two_streams":
            sampler.mark()
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if name == "block_two_streams":
            sampler.mark()
        ms[name] = e0.elapsed_time(e1) / args.steps
    sampler.stop()
    for w_ in (ws, gws, lws):
        if abi.moe_check_device_status(w_) != abi.OK:
            raise RuntimeError("device status error in the block benchmark")
    serial_parts = sum(ms[n] for n in ("down_and_router", "routed_experts", "shared_experts",
                                       "output_gemm"))
    two = ms["block_two_streams"]
    line = {
        "metric": "latent-MoE block tokens/s (routed MXFP4 experts with BF16 latent projections, "
                  "router and two shared experts on a second stream), 1xGB300",
        "value": T / (two / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": two, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 dense steps, mxfp8(e4m3)xmxfp4(e2m1)->f32 routed",
        "data": "synthetic (seeded; power-of-two grid inputs, see synth.make_block)",
        "config": {"workload": bw.name, "T": T, "hidden": bw.hidden, "d": bw.d, "E": bw.E,
                   "k": bw.k, "I": bw.I, "shared_I": bw.shared_I,
                   "gemm_kernel": "weight_tiles" if L.kernel_for(T) == abi.GEMM_WEIGHT_TILES
                   else "token_tiles",
                   "l2": "inputs larger than L2 (routed weights)"},
        "parts_ms": ms, "sum_of_parts_ms": serial_parts,
        "overlap_gain_vs_one_stream": ms["block_one_stream"] / two,
        "saved_ms_vs_sum_of_parts": serial_parts - two,
        "gpu_launches": None,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line))


def _free(*objs):
    import torch
    for o in objs:
        del o
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def measure_layer(args, wl, dev, sampler, a4w4=False):
    """Builds the workload's layer on `dev` and times it: K moe_forward calls on
    device-resident inputs (one CUDA-event pair), then the same kernels through
    the step entry points with events between them. Returns (entry, state):
    the per-workload JSON entry and the device objects the headline reuses."""
    import torch
    from mxfp4_latent_moe_gb300 import abi, synth
    from mxfp4_latent_moe_gb300.layer import MoeLayer

    L = synth.make_layer(wl, seed=args.seed, device=dev)
    kernel_arg = {"auto": abi.GEMM_AUTO, "token": abi.GEMM_TOKEN_TILES,
                  "weight": abi.GEMM_WEIGHT_TILES, "pair": abi.GEMM_PAIR_TILES}[args.gemm_kernel]
    layer = MoeLayer(L["w13"], L["w13_s"], L["w2"], L["w2_s"], k=wl.k, kernel=kernel_arg)
    T, d, E, k, I = wl.T, wl.d, wl.E, wl.k, wl.I
    x, logits = L["x"], L["logits"]
    ws = layer.workspace(T)
    y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def fwd():
        layer.forward(x, logits, ws=ws, y=y, topk_ids=ids, topk_w=w, a4w4=a4w4)

    # routing statistics for the roofline (outside any timed region)
    fwd()
    if abi.moe_check_device_status(ws) != abi.OK:
        raise RuntimeError("device status error in the first forward (%s)" % wl.name)
    counts = torch.bincount(ids.reshape(-1).long(), minlength=E)
    U = int((counts > 0).sum())
    valid_rows = T * k
    kernel = layer.kernel_for(T)      # both stages, or stage 2 under a4w4
    pad = 32 if kernel == abi.GEMM_WEIGHT_TILES and not a4w4 else 128
    layout = abi.SCALES_GROUP32 if kernel == abi.GEMM_WEIGHT_TILES else abi.SCALES_TILED128
    xs_layout = abi.SCALES_TILED128 if a4w4 else layout
    rows_cap = abi.moe_rows_capacity(T, E, k, pad)
    padded_rows = int(((counts + pad - 1) // pad * pad).sum())
    expert_bytes = layer.weight_bytes_per_expert()
    w13_bytes = 2 * I * d // 2 + 2 * I * d // 32
    flops = 6.0 * T * k * d * I
    l2_note = "inputs larger than L2 (touched weights %.2f GB)" % (U * expert_bytes / 1e9)
    flush = None
    if U * expert_bytes < 512e6:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        l2_note = "L2 flushed between steps (256 MB write)"

    for _ in range(max(3, args.warmup)):
        fwd()
    torch.cuda.synchronize()

    # ---- timed region: K moe_forward calls on device-resident inputs
    torch.cuda.synchronize()
    t_wall0 = time.time()
    sampler.mark()
    if flush is None:
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            fwd()
        t_end.record(stream)
        torch.cuda.synchronize()
        total_ms = t_start.elapsed_time(t_end)
    else:  # time each step between its L2 flush and the next
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ev[2 * i].record(stream)
            fwd()
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        total_ms = sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps))
    sampler.mark()
    t_wall1 = time.time()
    if abi.moe_check_device_status(ws) != abi.OK:
        raise RuntimeError("device status error in the timed forwards (%s)" % wl.name)
    # this library's kernels per forward: route, grouping (one kernel for a
    # one-chunk batch of T <= 256 tokens, else count + scan + scatter),
    # quantisation, the two GEMMs, combine; a token-tile GEMM stage is two
    # launches (the heavy experts' CTA pairs of m-tiles, then the rest)
    token_stages = (2 if kernel == abi.GEMM_TOKEN_TILES else
                    1 if a4w4 else 0)   # A4W4 stage 1 always runs token tiles
    launches_per_step = (6 if T <= 256 else 8) + token_stages

    # ---- per-kernel breakdown: the same kernels through the step entry points
    rc = rows_cap
    counts_d = torch.empty(E, dtype=torch.int32, device=dev)
    offsets_d = torch.empty(E + 1, dtype=torch.int32, device=dev)
    s2r = torch.empty(T * k, dtype=torch.int32, device=dev)
    r2s = torch.empty(rc, dtype=torch.int32, device=dev)
    pws = torch.zeros(abi.moe_permute_workspace_size(T, E), dtype=torch.uint8, device=dev)
    xq = torch.empty(rc, d // 2 if a4w4 else d, dtype=torch.uint8, device=dev)
    xs = torch.empty(abi.moe_activation_scale_bytes(rc, d, xs_layout), dtype=torch.uint8,
                     device=dev)
    hq = torch.empty(rc, I, dtype=torch.uint8, device=dev)
    hs = torch.empty(abi.moe_activation_scale_bytes(rc, I, layout), dtype=torch.uint8, device=dev)
    yp = torch.empty(rc, d, dtype=torch.bfloat16, device=dev)
    gws = torch.zeros(256, dtype=torch.uint8, device=dev)
    names = ["route_topk", "permute", "quant_mxfp4" if a4w4 else "quant_mxfp8",
             "gemm_w13_glu", "gemm_w2", "combine"]
    if a4w4:
        quant_call = lambda: abi.moe_quant_mxfp4(x, T, d, s2r, k, xq, xs, rc, xs_layout)
        w13_call = lambda: abi.moe_grouped_gemm_w13_glu_a4w4(
            xq, xs, counts_d, offsets_d, E, d, I, layout, layer.w13, layer.w13_sf, hq, hs, rc, gws)
    else:
        quant_call = lambda: abi.moe_quant_mxfp8(x, T, d, s2r, k, xq, xs, rc, layout)
        w13_call = lambda: abi.moe_grouped_gemm_w13_glu(xq, xs, counts_d, offsets_d, E, d, I,
                                                        kernel, layer.w13, layer.w13_sf, hq, hs,
                                                        rc, gws)
    calls = [
        lambda: abi.moe_route_topk(logits, T, E, k, ids, w),
        lambda: abi.moe_permute(ids, T, E, k, pad, counts_d, offsets_d, s2r, r2s, rc, pws),
        quant_call,
        w13_call,
        lambda: abi.moe_grouped_gemm_w2(hq, hs, counts_d, offsets_d, E, I, d, kernel, layer.w2,
                                        layer.w2_sf, yp, rc, gws),
        lambda: abi.moe_unpermute_combine(yp, s2r, w, T, k, d, y),
    ]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
           for _ in range(args.steps)]
    for i in range(max(3, args.warmup // 2)):
        for c in calls:
            c()
    torch.cuda.synchronize()
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        kev[i][0].record(stream)
        for j, c in enumerate(calls):
            c()
            kev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    kms = {n: statistics.mean(kev[i][j].elapsed_time(kev[i][j + 1]) for i in range(args.steps))
           for j, n in enumerate(names)}
    if abi.moe_check_device_status(gws) != abi.OK or abi.moe_check_device_status(pws) != abi.OK:
        raise RuntimeError("device status error in the kernel breakdown (%s)" % wl.name)

    # ---- the step as one CUDA graph, replayed back to back (device-resident):
    # graph time minus the two GEMMs' event times bounds what folding the
    # other kernels into the GEMMs (a single-launch layer) could save
    graph, _, _ = layer.capture(x, logits, ws=ws, y=y, a4w4=a4w4)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if flush is None:
        g0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1) / args.steps
    else:
        gev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            gev[2 * i].record(stream)
            graph.replay()
            gev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        graph_ms = sum(gev[2 * i].elapsed_time(gev[2 * i + 1]) for i in range(args.steps)) / args.steps
    del graph
    if abi.moe_check_device_status(ws) != abi.OK:
        raise RuntimeError("device status error in the graph replays (%s)" % wl.name)

    peaks, peak_src = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bf16_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    bf16_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    # The tensor peak of the regime the timed region ran in: the sustained
    # (power-capped) bf16 figure when the GPU reported sw_power_cap during the
    # timed steps, the burst figure otherwise. Both fractions are reported.
    clocks = sampler.summary(t_wall0, t_wall1)
    capped = "sw_power_cap" in clocks.get("reasons", [])
    bf16_peak = bf16_sus if capped else bf16_burst
    regime = "sustained (sw_power_cap during the timed steps)" if capped else "burst"
    w13_ratio = FP4_OVER_BF16 if a4w4 else FP8_OVER_BF16

    def math_time(bf16):
        return (4.0 * T * k * d * I / (bf16 * w13_ratio * 1e12) +
                2.0 * T * k * d * I / (bf16 * FP8_OVER_BF16 * 1e12))

    w13_peak = bf16_peak * w13_ratio
    t_mem = U * expert_bytes / (hbm_peak * 1e9)
    t_math = math_time(bf16_peak)
    bound = "hbm" if t_mem >= t_math else "tensor"
    ms_per_step = total_ms / args.steps
    layer_frac = max(t_mem, t_math) / (ms_per_step / 1e3)
    family = {abi.GEMM_WEIGHT_TILES: "weight_tiles", abi.GEMM_PAIR_TILES: "pair_tiles"}.get(
        kernel, "token_tiles")
    dom = "gemm_w13_glu"
    dom_s = kms[dom] / 1e3
    x_row_bytes = (d // 2 if a4w4 else d) + d // 32
    if bound == "hbm":
        dom_bytes = U * w13_bytes + valid_rows * x_row_bytes + valid_rows * (I + I // 32)
        roof = {"kernel": dom, "bound": "hbm", "achieved": dom_bytes / dom_s / 1e9,
                "peak": hbm_peak, "unit": "GB/s", "frac": dom_bytes / dom_s / 1e9 / hbm_peak,
                "traffic": profiled_traffic(dom, wl.name, family) if not a4w4 else None,
                "algorithmic_bytes": dom_bytes,
                "algorithmic_bytes_how": "touched experts x w13 bytes (codes + scales) + "
                                         "T*k x-code rows in + T*k h-code rows out",
                "mean_ms": kms[dom], "peak_source": peak_src + " hbm_gbs (copy)"}
    else:
        dom_flops = 4.0 * T * k * d * I
        ratio, what = (FP4_OVER_BF16, "fp4") if a4w4 else (FP8_OVER_BF16, "fp8")
        roof = {"kernel": dom, "bound": "tensor", "achieved": dom_flops / dom_s / 1e12,
                "peak": w13_peak, "unit": "TFLOP/s",
                "frac": dom_flops / dom_s / 1e12 / w13_peak,
                "frac_of_burst": dom_flops / dom_s / 1e12 / (bf16_burst * ratio),
                "frac_of_sustained": dom_flops / dom_s / 1e12 / (bf16_sus * ratio),
                "traffic": profiled_traffic(dom, wl.name, family) if not a4w4 else None,
                "algorithmic_flops": dom_flops,
                "algorithmic_flops_how": "4*T*k*d*I (gate and up products of the routed rows; "
                                         "padding rows not credited)",
                "mean_ms": kms[dom],
                "peak_source": "%s bf16 %s x %.1f (nominal %s / bf16 dense ratio)"
                               % (peak_src, regime, ratio, what)}
        if a4w4:
            mma_peak = bf16_peak * FP4_MMA_OVER_BF16
            roof["frac_of_measured_mma_rate"] = dom_flops / dom_s / 1e12 / mma_peak
            roof["measured_mma_rate_peak"] = mma_peak
    entry = {
        "workload": wl.name, "a4w4": bool(a4w4),
        "value": T * args.steps / (total_ms / 1e3), "unit": "tokens/s",
        "ms_per_step": ms_per_step, "steps": args.steps,
        "gemm_kernel": family, "touched_experts": U, "padded_rows": padded_rows,
        "layer_roofline": {"bound": bound, "time_ms": 1e3 * max(t_mem, t_math),
                           "frac": layer_frac,
                           "frac_of_burst": max(t_mem, math_time(bf16_burst))
                           / (ms_per_step / 1e3),
                           "frac_of_sustained": max(t_mem, math_time(bf16_sus))
                           / (ms_per_step / 1e3),
                           "tensor_peak_regime": regime,
                           "tflops": flops / (ms_per_step / 1e3) / 1e12,
                           "weight_gbs": U * expert_bytes / (ms_per_step / 1e3) / 1e9,
                           "how": "max(touched experts x 17,547,264 B / hbm_gbs, 4TkdI FLOP / "
                                  "stage-1 peak + 2TkdI FLOP / (bf16 peak x 2)), bf16 peak of "
                                  "the regime"},
        "roofline": roof,
        "kernels_ms": kms,
        "graph_ms_per_step": graph_ms,
        "outside_gemms_ms": graph_ms - kms["gemm_w13_glu"] - kms["gemm_w2"],
        "outside_gemms_how": "step replayed as one CUDA graph minus the two GEMMs' mean event "
                             "times: the most a single-launch layer could save",
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "l2": l2_note,
    }
    state = dict(L=L, layer=layer, ws=ws, y=y, flush=flush, stream=stream)
    return entry, state


def measure_e2e(args, wl, st, a4w4=False):
    """The headline's end-to-end legs through the public API: every step's x and
    logits copied from pinned host memory and y copied back (HostPipeline, the
    copies on copy streams; serial, in one stream; graph-replayed)."""
    import torch
    from mxfp4_latent_moe_gb300 import abi
    from mxfp4_latent_moe_gb300.layer import HostPipeline
    L, layer, ws, y, flush, stream = (st[n] for n in ("L", "layer", "ws", "y", "flush", "stream"))
    T, d = wl.T, wl.d
    x, logits = L["x"], L["logits"]
    x_h = x.cpu().pin_memory()
    lg_h = logits.cpu().pin_memory()
    y_h = torch.empty(T, d, dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(x)
    lg_d = torch.empty_like(logits)
    for _ in range(3):
        x_d.copy_(x_h, non_blocking=True)
        lg_d.copy_(lg_h, non_blocking=True)
        layer.forward(x_d, lg_d, ws=ws, y=y, a4w4=a4w4)
        y_h.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        x_d.copy_(x_h, non_blocking=True)
        lg_d.copy_(lg_h, non_blocking=True)
        layer.forward(x_d, lg_d, ws=ws, y=y, a4w4=a4w4)
        y_h.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = e0.elapsed_time(e1)

    pipe = HostPipeline(layer, T, a4w4=a4w4)
    for _ in range(3):
        pipe.submit(x_h, lg_h, y_h)
    pipe.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    pipe.h2d.wait_event(p0)
    last = None
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)   # on the compute stream, between forwards
        last = pipe.submit(x_h, lg_h, y_h)
    stream.wait_event(last)
    p1.record(stream)
    torch.cuda.synchronize()
    if abi.moe_check_device_status(pipe.ws) != abi.OK:
        raise RuntimeError("device status error in the pipelined end-to-end steps")
    e2e_ms = p0.elapsed_time(p1)
    del pipe

    graph, y_g, _ = layer.capture(x_d, lg_d, ws=ws, a4w4=a4w4)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        x_d.copy_(x_h, non_blocking=True)
        lg_d.copy_(lg_h, non_blocking=True)
        graph.replay()
        y_h.copy_(y_g, non_blocking=True)
    g1.record(stream)
    torch.cuda.synchronize()
    e2e_graph_ms = g0.elapsed_time(g1)
    if abi.moe_check_device_status(ws) != abi.OK:
        raise RuntimeError("device status error in the graph replays")
    del graph
    rate = lambda ms: T * args.steps / (ms / 1e3)
    return {
        "e2e": {"value": rate(e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": T * d * 2 + T * wl.E * 4,
                "d2h_bytes_per_step": T * d * 2,
                "how": "HostPipeline: pinned host batches, copies on two copy streams "
                       "overlapping the neighbouring batches' forwards"},
        "e2e_serial": {"value": rate(e2e_serial_ms), "unit": "tokens/s",
                       "how": "same copies and forwards in one stream"},
        "e2e_graph": {"value": rate(e2e_graph_ms), "unit": "tokens/s",
                      "how": "same copies, the step replayed as one CUDA graph "
                             "(MoeLayer.capture)"},
    }


def cpu_baseline_leg(args, wl, L, a4w4=False, budget_s=15.0):
    """The oracle, as it stands, on the host cores, on the first n tokens of
    the workload, n sized for about budget_s seconds of CPU work."""
    cores = os.cpu_count() or 1
    if args.cpu_sample:
        n = args.cpu_sample
    else:
        n0 = min(wl.T, cores)
        per_token = oracle_seconds(wl, oracle_inputs(L, n0), cores, a4w4) / n0
        n = max(1, min(wl.T, int(budget_s / per_token)))
    dt = oracle_seconds(wl, oracle_inputs(L, n), cores, a4w4=a4w4)
    return {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "first %d of %d tokens of the workload, full layer (%.1f s)" % (n, wl.T, dt),
            "cpu_model": cpu_model()}


def parse_per_workload(spec):
    out = []
    for item in (spec or "").split(","):
        item = item.strip()
        if not item or item == "none":
            continue
        name, _, mode = item.partition(":")
        out.append((name, mode == "a4w4"))
    return out


def main():
    args = parse()
    from mxfp4_latent_moe_gb300 import synth
    wl = synth.workload(args.workload) if args.tokens <= 0 else synth.full_dims(args.tokens)
    if args.impl == "reference":
        return run_reference(args, wl)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != 1 or world != 1:
        # libmoe.so is single-GPU code: its prefill GEMMs multicast TMA loads
        # inside 2-CTA clusters, which may only run in one-GPU programs.
        sys.stderr.write("bench.py: this layer runs on one GPU only (--gpus 1); "
                         "got --gpus %d, WORLD_SIZE %d\n" % (args.gpus, world))
        sys.exit(2)
    if args.step == "block":
        return run_block(args, wl)
    if args.step:
        return run_step(args, wl)

    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()

    sampler = ClockSampler(0)
    sampler.start()
    head, st = measure_layer(args, wl, dev, sampler, a4w4=args.a4w4)
    e2e = measure_e2e(args, wl, st, a4w4=args.a4w4)
    cpu = None if args.no_cpu_baseline else cpu_baseline_leg(args, wl, st["L"], a4w4=args.a4w4)
    st.clear()
    _free()
    per = {}
    for name, a4 in parse_per_workload(args.per_workload):
        if name == wl.name and a4 == bool(args.a4w4):
            continue
        entry, st2 = measure_layer(args, synth.workload(name), dev, sampler, a4w4=a4)
        st2.clear()
        _free()
        per[name + (":a4w4" if a4 else "")] = entry
    sampler.stop()

    line = {
        "metric": METRIC,
        "value": head["value"], "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("stage1 mxfp4(e2m1)xmxfp4(e2m1)->f32, stage2 mxfp8(e4m3)xmxfp4(e2m1)->f32"
                  if args.a4w4 else "mxfp8(e4m3)xmxfp4(e2m1)->f32"),
        "data": "synthetic (seeded; x~N(0,1) bf16, logits~N(0,1), uniform E2M1 codes, "
                "E8M0 scales 118..122)",
        "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k, "I": wl.I,
                   "gemm_kernel": head["gemm_kernel"], "a4w4": bool(args.a4w4),
                   "touched_experts": head["touched_experts"],
                   "padded_rows": head["padded_rows"], "parallelism": "single",
                   "l2": head["l2"]},
        "layer_roofline": head["layer_roofline"],
        "roofline": head["roofline"],
        "kernels_ms": head["kernels_ms"],
        "graph_ms_per_step": head["graph_ms_per_step"],
        "outside_gemms_ms": head["outside_gemms_ms"],
        "gpu_launches": head["gpu_launches"],
        "e2e": e2e["e2e"],
        "e2e_serial": e2e["e2e_serial"],
        "e2e_graph": e2e["e2e_graph"],
        "cpu_baseline": cpu,
        "clocks": head["clocks"],
        "per_workload": per,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
