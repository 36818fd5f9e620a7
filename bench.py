"""Benchmark of the chunked low-precision MoE layer on GB300.

One step = the whole hot path on one batch of synthetic input, device
resident: Cayley map of the adapter parameters, router top-k, grouping of
the pairs by expert, the chunked forward (rotation, dequantized grouped
GEMMs with SwiGLU, weighted un-permute), the backward-data pass (dX,
d_topk_w, adapter gradients) and the Cayley gradient.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  The default workload is the Kimi-K2-shaped
INT4 layer (T=8192, d=7168, E=384, top-8, inter=2048, OFT block 64,
chunk C=32, Zipf-skewed router).  For N > 1 (torchrun), every rank runs its
own replica of the workload (the layer's tokens are independent): weak
scaling, no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from precision_moe_adapter_gb300 import inputs as gi  # noqa: E402


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="kimi_k2", choices=sorted(gi.CONFIGS))
    ap.add_argument("--mode", default="fused", choices=["fused", "scratch"])
    ap.add_argument("--chunk", type=int, default=0, help="experts per chunk (0: the config's C)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (0: the config's T)")
    ap.add_argument("--experts", type=int, default=0, help="override E (0: the config's E)")
    ap.add_argument("--sweep-chunks", default="",
                    help="comma-separated chunk sizes (0: all active experts): after the main "
                         "line, one line per C with the step time in --mode and its dequant "
                         "scratch bytes")
    ap.add_argument("--decode", action="store_true",
                    help="decode sweep on the Kimi-K2 shape (forward only): one line per "
                         "(T, weight format, C) with the achieved HBM bandwidth")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# of the GEMM classes on the default workload, from one ncu capture, keyed
# by the digest of the GEMM sources it was taken with: once those sources
# change the figure no longer describes the kernel and is reported as null.
TRAFFIC = {"digest": "80a4dc6f4381af7e", "bytes": {
    ("kimi_k2", "fused", "gemm_gate_up"): 9.234523e9,
    ("kimi_k2", "fused", "gemm_down"): 5.281668e9,
    ("kimi_k2", "fused", "gemm_bwd_g"): 5.070333e9,
    ("kimi_k2", "fused", "gemm_bwd_dx"): 9.113973e9}}


def gemm_digest() -> str:
    """SHA-256 (first 16 hex digits) of the grouped GEMM's sources."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "precision_moe_adapter_gb300", "csrc")
    for f in ("gemm_tc.cuh", "gemm_tc_host.cuh", "gemm_tc.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(cfg_name: str, mode: str, kernel: str, default_load: bool):
    if not default_load or TRAFFIC["digest"] != gemm_digest():
        return None
    return TRAFFIC["bytes"].get((cfg_name, mode, kernel))


def pick_peak(pk, clocks):
    """The dense BF16 denominator: the measured burst figure when the timed
    region ran at the maximum SM clock with no power cap, else the measured
    sustained (power-capped) one."""
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    at_max = sm is not None and smax is not None and sm >= 0.97 * smax
    if at_max and not capped:
        return pk["bf16"], f"{pk['src']} bf16 burst (timed region at {sm:.0f} MHz, no power cap)"
    return pk["bf16_sus"], f"{pk['src']} bf16 sustained (timed region at {sm} MHz, reasons {clocks.get('reasons')})"


def max_over_ranks(x: float) -> float:
    """The largest x over all ranks (x itself outside a process group):
    every rank times its own replica and the job takes the slowest."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = (torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl"
           else torch.device("cpu"))
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, steps: int, ms: float, world: int) -> float:
    """Units per second of the whole job: every rank processed
    units_per_rank per step, and the job took ms (max over ranks)."""
    return world * units_per_rank * steps / (ms / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return dict(hbm=m["hbm_gbs"], bf16=m["bf16_tflops"],
                    bf16_sus=m.get("bf16_tflops_sustained", m["bf16_tflops"]), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def flops_of(cfg, P):
    """Algorithmic FLOPs of one step (forward + backward-data)."""
    d, I, b = cfg.d, cfg.I, cfg.b
    fwd = 2 * 3 * d * I * P + 2 * (d + I) * b * P + 2 * cfg.T * d * cfg.E
    bwd = 2 * 3 * d * I * P + 4 * (d + I) * b * P
    return fwd, bwd


def bytes_of(cfg, counts):
    """Algorithmic HBM bytes of one step: quantized weights + scales +
    adapters of the active experts (each read once per pass), activations."""
    d, I, b = cfg.d, cfg.I, cfg.b
    na = int((counts > 0).sum())
    if cfg.fmt == gi.FP8:
        wq = 3 * d * I + 3 * (d // 128) * (I // 128) * 4
    else:
        wq = 3 * d * I // 2 + 3 * d * (I // 32) * (2 if cfg.fmt == gi.INT4 else 1)
    adp = (d + I) * b * 2 if cfg.adapter == "per_expert" else 0
    act_f = cfg.T * d * 2 * 2 + d * cfg.E * 4          # X, Y, Wr
    act_b = cfg.T * d * 2 * 3 + cfg.P * I * 12         # X, dY, dX, ctx (g, u f32; h, h~ bf16)
    return na * (wq + adp) * 2 + act_f + act_b


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- CPU side

def oracle_sample(cfg, host, n_tok):
    """Run the oracle on a bounded sample of the workload: router, forward
    and backward-data for the first n_tok tokens.  Returns (seconds, threads)."""
    import oracle
    toks = list(range(n_tok))
    t0 = time.perf_counter()
    _, idx, w = oracle.route(host["X"], host["Wr"], host["bias"], cfg.k, toks=toks)
    L = oracle.Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b, cfg.fmt, host["w13"], host["s13"],
                     host["w2"], host["s2"], R_up=host["Ru_bits"], R_down=host["Rd_bits"])
    L.forward(host["X"], idx, w, toks=toks)
    L.backward(host["X"], host["dY"], idx, w, toks=toks)
    return time.perf_counter() - t0, oracle.num_threads()


def host_inputs(cfg, with_rbits):
    X, dY = gi.gen_x(cfg), gi.gen_dy(cfg)
    w13, s13, w2, s2 = gi.gen_weights(cfg)
    Wr, bias = gi.gen_router(cfg)
    Su, Sd = gi.gen_adapter_params(cfg)
    h = dict(X=X, dY=dY, w13=w13, s13=s13, w2=w2, s2=s2, Wr=Wr, bias=bias, Su=Su, Sd=Sd,
             Ru_bits=None, Rd_bits=None)
    if with_rbits and Su is not None:
        import oracle
        rb = lambda S: gi.f32_to_bf16_bits(
            oracle.cayley(S.reshape(-1, cfg.b, cfg.b)).astype(np.float32)).reshape(S.shape)
        h["Ru_bits"], h["Rd_bits"] = rb(Su), rb(Sd)
    return h


def sample_tokens(cfg, threads):
    """Tokens of the CPU-baseline sample: about 10-30 s of oracle work."""
    return max(1, min(cfg.T, (8 * threads) // cfg.k))


def run_reference(args, cfg, rank):
    """The oracle as the reference arm: each step is the oracle on a bounded
    sample of the workload, on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    host = host_inputs(cfg, with_rbits=True)
    n_tok = max(1, min(cfg.T, oracle.num_threads() // cfg.k))
    for _ in range(args.warmup):
        oracle_sample(cfg, host, n_tok)
    total, thr = 0.0, 1
    for _ in range(args.steps):
        dt, thr = oracle_sample(cfg, host, n_tok)
        total += dt
    v = n_tok * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload(cfg, args),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                             "sample": f"first {n_tok} tokens of the workload per step "
                                       f"(router + forward + backward-data)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


METRIC = "MoE-layer tokens/s (forward + backward-data), INT4 Kimi-K2 shape, 1 GB300"


def workload(cfg, args):
    fmt = gi.FMT_NAMES[cfg.fmt]
    return {"workload": f"{cfg.name}: {fmt} MoE layer forward + backward-data, T={cfg.T} d={cfg.d} "
                        f"E={cfg.E} top-{cfg.k} inter={cfg.I} OFT b={cfg.b} C={cfg.C} "
                        f"router={cfg.router}",
            "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "inter": cfg.I, "block": cfg.b,
            "chunk_C": cfg.C, "mode": args.mode, "weights": fmt,
            "l2": "inputs larger than L2 (quantized experts alone exceed 129 MB)"}


# ---------------------------------------------------------------- GPU side

def decode_bytes(cfg, counts):
    """Algorithmic HBM bytes of one decode forward: the packed weights,
    scales and adapter blocks of the active experts (each read once), the
    router weights, X and Y."""
    d, I, b = cfg.d, cfg.I, cfg.b
    na = int((counts > 0).sum())
    if cfg.fmt == gi.FP8:
        wq = 3 * d * I + 3 * (d // 128) * (I // 128) * 4
    else:
        wq = 3 * d * I // 2 + 3 * d * (I // 32) * (2 if cfg.fmt == gi.INT4 else 1)
    adp = (d + I) * b * 2
    return na * (wq + adp) + d * cfg.E * 4 + 2 * cfg.T * d * 2


def run_decode(args):
    """Decode-sized forward on the Kimi-K2 shape, T in {1, 8, 64, 512}, INT4
    and FP8 weights, C in {8, 32, all active}: latency of router + grouping
    + forward (CUDA events, a 256 MB L2-flush write between iterations) and
    the achieved bandwidth against the measured HBM copy rate."""
    import torch
    from precision_moe_adapter_gb300 import build as pbuild
    from precision_moe_adapter_gb300 import pmoe
    from precision_moe_adapter_gb300.layer import DeviceLayer
    pbuild.build()
    pmoe.lib()
    pk = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for fmt in (gi.INT4, gi.FP8):
        base = gi.decode_config(1, fmt)
        if fmt == gi.FP8:
            w13, s13 = gi.gen_fp8_matrix_on_device(base.E, 2 * base.I, base.d, base.seed, "w13", "s13",
                                                   "cuda")
            w2, s2 = gi.gen_fp8_matrix_on_device(base.E, base.d, base.I, base.seed, "w2", "s2", "cuda")
        else:
            w13, s13, w2, s2 = gi.gen_weights(base)
        Su, Sd = gi.gen_adapter_params(base)
        for T in (1, 8, 64, 512):
            cfg = gi.decode_config(T, fmt)
            Wr, bias = gi.gen_router(cfg)
            L = DeviceLayer(cfg, w13, s13, w2, s2, Wr=Wr, bias=bias, S_up=Su, S_down=Sd)
            X = torch.from_numpy(gi.gen_x(cfg)).view(torch.int16).cuda()
            Y = torch.empty_like(X)
            rt = L.new_routing()
            L.route(X, rt)
            L.permute(rt)
            torch.cuda.synchronize()
            counts = rt.counts.cpu().numpy()
            na = int((counts > 0).sum())
            B = decode_bytes(cfg, counts)
            for C in (8, 32, na):
                def once():
                    L.route(X, rt)
                    L.permute(rt)
                    L.forward(X, rt, Y, C=C)
                for _ in range(max(args.warmup, 3)):
                    once()
                times = []
                for _ in range(args.steps):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    once()
                    e1.record()
                    torch.cuda.synchronize()
                    times.append(e0.elapsed_time(e1))
                ms = statistics.median(times)
                gbs = B / (ms / 1e3) / 1e9
                print(json.dumps({
                    "metric": "decode forward latency and HBM bandwidth (router + grouping + forward)",
                    "workload": cfg.name, "T": T, "weights": gi.FMT_NAMES[fmt], "C": C,
                    "active_experts": na, "ms": ms, "tokens_per_s": T / (ms / 1e3),
                    "bytes": B, "achieved_gbs": gbs, "peak_gbs": pk["hbm"],
                    "frac": gbs / pk["hbm"], "bound": "hbm", "peak_source": f"{pk['src']} HBM copy",
                    "timing": f"median of {args.steps}, 256 MB L2 flush between iterations"}), flush=True)
            st = L.status()
            if st != pmoe.PMOE_OK:
                raise RuntimeError(f"device error: {pmoe.status_string(st)}")
            del L
            torch.cuda.empty_cache()
        del w13, w2
        torch.cuda.empty_cache()


def main():
    args = parse()
    cfg = gi.CONFIGS[args.config]
    if args.tokens:
        cfg = cfg.with_(T=args.tokens)
    if args.experts:
        cfg = cfg.with_(E=args.experts)
    if args.chunk:
        cfg = cfg.with_(C=args.chunk)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return
    if args.decode:
        run_decode(args)
        return

    import torch
    import torch.distributed as dist
    from precision_moe_adapter_gb300 import build as pbuild
    from precision_moe_adapter_gb300 import pmoe
    from precision_moe_adapter_gb300.layer import DeviceLayer

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        pbuild.build()
    if world > 1:
        dist.barrier()
    pmoe.lib()

    host = host_inputs(cfg, with_rbits=(rank == 0 and world == 1 and not args.no_cpu_baseline))
    L = DeviceLayer(cfg, host["w13"], host["s13"], host["w2"], host["s2"], Wr=host["Wr"],
                    bias=host["bias"], S_up=host["Su"], S_down=host["Sd"])
    mode = pmoe.MODE_FUSED if args.mode == "fused" else pmoe.MODE_SCRATCH
    dev = L.device
    X = torch.from_numpy(host["X"]).view(torch.int16).to(dev)
    dY = torch.from_numpy(host["dY"]).view(torch.int16).to(dev)
    rt = L.new_routing()
    Y = torch.empty_like(X)
    dX = torch.empty_like(X)
    ctx = L.new_ctx()
    dtw = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    dRu, dRd = L.grads()
    dSu = None if L.S_up is None else torch.empty_like(L.S_up)
    dSd = None if L.S_down is None else torch.empty_like(L.S_down)
    b = cfg.b

    PHASES = ("cayley", "route", "permute", "forward", "backward", "cayley_grad")
    phase_ms = {p_: 0.0 for p_ in PHASES}
    phase_ev = []

    def mark(name, timed):
        if timed:
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            phase_ev.append((name, e))

    def step(Xs, dYs, timed=False, Yo=None, dXo=None, C=None):
        Yo = Y if Yo is None else Yo
        dXo = dX if dXo is None else dXo
        C = C or cfg.C
        mark("cayley", timed)
        if L.S_up is not None:   # R = Cayley(S) for the adapter of this step
            pmoe.adapter_cayley(L.S_up.numel() // (b * b), b, L.S_up, L.R_up, L.Rf_up)
            pmoe.adapter_cayley(L.S_down.numel() // (b * b), b, L.S_down, L.R_down, L.Rf_down)
        mark("route", timed)
        L.route(Xs, rt)
        mark("permute", timed)
        L.permute(rt)
        mark("forward", timed)
        L.forward(Xs, rt, Yo, C=C, mode=mode, ctx=ctx)
        mark("backward", timed)
        L.backward(Xs, dYs, ctx, rt, dXo, dtw, dRu, dRd, C=C)
        mark("cayley_grad", timed)
        if L.S_up is not None:
            pmoe.adapter_cayley_grad(L.S_up.numel() // (b * b), b, L.S_up, L.Rf_up, dRu, dSu)
            pmoe.adapter_cayley_grad(L.S_down.numel() // (b * b), b, L.S_down, L.Rf_down, dRd, dSd)
        mark("end", timed)

    for _ in range(args.warmup):
        step(X, dY)
    torch.cuda.synchronize()
    st = L.status()
    if st != pmoe.PMOE_OK:
        raise RuntimeError(f"device error after warm-up: {pmoe.status_string(st)}")
    counts = rt.counts.cpu().numpy()

    # ---- device-resident timed region
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    pmoe.pmoe_kernel_timing(True)
    n0 = pmoe.pmoe_launch_count()
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step(X, dY)
        ev1.record(stream)
        torch.cuda.synchronize()
    launches = pmoe.pmoe_launch_count() - n0
    ms = ev0.elapsed_time(ev1)
    # per-launch device times of the timed region only
    kt = {name: pmoe.pmoe_kernel_time(i) for i, name in enumerate(
        ("gemm_gate_up", "gemm_down", "gemm_bwd_g", "gemm_bwd_dx", "router"))}
    pmoe.pmoe_kernel_timing(False)
    # one extra step with events between the calls: where the step's time goes
    phase_ev.clear()
    step(X, dY, timed=True)
    torch.cuda.synchronize()
    for (n_, e_), (_, f_) in zip(phase_ev[:-1], phase_ev[1:]):
        phase_ms[n_] += e_.elapsed_time(f_)
    ms = max_over_ranks(ms)
    ms_step = ms / args.steps
    tokens_per_s = whole_job_rate(cfg.T, args.steps, ms, world)
    P = cfg.P
    f_fwd, f_bwd = flops_of(cfg, P)
    pk = peaks()
    tflops = (f_fwd + f_bwd) / (ms_step / 1e3) / 1e12
    B = bytes_of(cfg, counts)
    clocks = clk.summary()
    peak_tf, peak_src = pick_peak(pk, clocks)
    t_roof = max((f_fwd + f_bwd) / (peak_tf * 1e12), B / (pk["hbm"] * 1e9))

    # dominant kernel: the timed class with the largest share of device time
    dom = max(kt, key=lambda k_: kt[k_][0])
    dom_ms, dom_n = kt[dom]
    dom_flops = {"gemm_gate_up": 2 * P * cfg.d * 2 * cfg.I, "gemm_down": 2 * P * cfg.I * cfg.d,
                 "gemm_bwd_g": 2 * P * cfg.d * cfg.I, "gemm_bwd_dx": 2 * P * 2 * cfg.I * cfg.d,
                 "router": 2 * cfg.T * cfg.d * cfg.E}[dom]
    dom_avg_ms = dom_ms / max(dom_n, 1)
    dom_tf = dom_flops / (dom_avg_ms / 1e3) / 1e12
    default_load = not (args.tokens or args.experts or args.chunk)
    traffic = traffic_of(cfg.name, args.mode, dom, default_load)
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(dom_tf, 3),
                "peak": peak_tf, "unit": "TFLOP/s", "frac": round(dom_tf / peak_tf, 5),
                "traffic": traffic, "peak_source": peak_src,
                "frac_of_sustained": round(dom_tf / pk["bf16_sus"], 5),
                "launch_ms": round(dom_avg_ms, 4), "launches": dom_n,
                "algorithmic_flops_per_launch": dom_flops}

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        # every step copies its X and dY in from pinned host memory and its Y
        # and dX back out; the copies run on their own stream, double-buffered,
        # so step i's copies overlap the compute of steps i-1 and i+1
        Xh = torch.from_numpy(host["X"]).view(torch.int16).pin_memory()
        dYh = torch.from_numpy(host["dY"]).view(torch.int16).pin_memory()
        Yh = [torch.empty_like(Xh).pin_memory() for _ in range(2)]
        dXh = [torch.empty_like(Xh).pin_memory() for _ in range(2)]
        Xd = [torch.empty_like(X) for _ in range(2)]
        dYd = [torch.empty_like(dY) for _ in range(2)]
        Yd = [torch.empty_like(Y) for _ in range(2)]
        dXd = [torch.empty_like(dX) for _ in range(2)]
        cs = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            Xd[0].copy_(Xh, non_blocking=True)
            dYd[0].copy_(dYh, non_blocking=True)
            ev_in[0].record(cs)
        for i in range(args.steps):
            bi = i % 2
            stream.wait_event(ev_in[bi])
            if i >= 2:
                stream.wait_event(ev_out[bi])      # step i-2's outputs are out
            step(Xd[bi], dYd[bi], Yo=Yd[bi], dXo=dXd[bi])
            ev_done[bi].record(stream)
            with torch.cuda.stream(cs):
                if i + 1 < args.steps:             # buffer (i+1)%2 was freed by step i-1
                    nb_ = (i + 1) % 2
                    Xd[nb_].copy_(Xh, non_blocking=True)
                    dYd[nb_].copy_(dYh, non_blocking=True)
                    ev_in[nb_].record(cs)
                cs.wait_event(ev_done[bi])
                Yh[bi].copy_(Yd[bi], non_blocking=True)
                dXh[bi].copy_(dXd[bi], non_blocking=True)
                ev_out[bi].record(cs)
        stream.wait_stream(cs)
        ev1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(ev0.elapsed_time(ev1))
        nb = X.numel() * 2
        e2e = {"value": whole_job_rate(cfg.T, args.steps, e_ms, world), "unit": "tokens/s",
               "h2d_bytes_per_step": 2 * nb, "d2h_bytes_per_step": 2 * nb,
               "ms_per_step": e_ms / args.steps}

    st = L.status()
    if st != pmoe.PMOE_OK:
        raise RuntimeError(f"device error: {pmoe.status_string(st)}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        n_tok = sample_tokens(cfg, oracle.num_threads())
        dt, thr = oracle_sample(cfg, host, n_tok)
        cpu = {"value": n_tok / dt, "unit": "tokens/s", "cores": thr, "kind": "oracle",
               "sample": f"first {n_tok} of {cfg.T} tokens (router + forward + backward-data), "
                         f"{dt:.1f} s"}

    sweep = []
    if args.sweep_chunks:
        for c_ in [int(v) for v in args.sweep_chunks.split(",")]:
            C_ = c_ if c_ > 0 else cfg.E
            for _ in range(args.warmup):
                step(X, dY, C=C_)
            torch.cuda.synchronize()
            f0 = torch.cuda.mem_get_info()[0]
            ev0.record(stream)
            for _ in range(args.steps):
                step(X, dY, C=C_)
            ev1.record(stream)
            torch.cuda.synchronize()
            sms = ev0.elapsed_time(ev1) / args.steps
            sweep.append({"sweep": "chunk", "mode": args.mode, "C": C_,
                          "active_experts": int((counts > 0).sum()),
                          "chunks": int(np.ceil((counts > 0).sum() / C_)),
                          "ms_per_step": sms, "tokens_per_s": cfg.T / (sms / 1e3),
                          "scratch_bytes_per_chunk": pmoe.moe_scratch_bytes(L.dims, C_, mode),
                          "workspace_bytes_forward": pmoe.moe_workspace_bytes(
                              L.dims, pmoe.OP_FORWARD, C_, mode),
                          "device_bytes_in_use": torch.cuda.mem_get_info()[1] - f0})
        st = L.status()
        if st != pmoe.PMOE_OK:
            raise RuntimeError(f"device error in the sweep: {pmoe.status_string(st)}")

    if rank == 0:
        line = {"metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": workload(cfg, args),
                "tflops": tflops, "step_roofline": {
                    "time_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms_step,
                    "flops": f_fwd + f_bwd, "bytes": B,
                    "peaks": f"{peak_src}: {peak_tf} TF/s; HBM {pk['hbm']} GB/s ({pk['src']})",
                    "note": "the layer-level fraction the >= 0.6 target is judged on"},
                "roofline": roofline, "kernel_ms_per_step": {k_: v[0] / args.steps for k_, v in kt.items()},
                "phase_ms": {k_: round(v, 3) for k_, v in phase_ms.items()},
                "clocks": clocks, "e2e": e2e, "gpu_launches": launches,
                "cpu_baseline": cpu,
                "scratch_bytes_per_chunk": pmoe.moe_scratch_bytes(L.dims, cfg.C, mode)}
        print(json.dumps(line), flush=True)
        for sl in sweep:
            print(json.dumps(sl), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
