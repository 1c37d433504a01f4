"""Benchmark of chunked causal linear attention (forward + backward) on GB300.

One step = the whole hot path over one batch: linattn_fwd (segment aggregates,
state scan, chunked forward) then linattn_bwd (forward states recomputed,
reverse states, dq / dv / dk passes) on the synthetic workload
B=2, H=16, T=65536, d=128, bf16, lambda=1 (seeded; q, k, v ~ N(0, 0.125^2),
dO ~ N(0, 1)).  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 3]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the reference arm of this benchmark: there is no upstream code).
Under torchrun each rank runs an independent replica (weak scaling); only
rank 0 prints.
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
sys.path.insert(0, ROOT)

METRIC = "causal linear-attn fwd+bwd tokens/s & TFLOP/s @H16 d128 T16K–1M; % roofline"
# algorithmic work per token per head at d = 128 (chunk 64): forward 4d(C+d) FLOP and
# q,k,v read + o written; backward 8d(C+d) FLOP and q,k,v,dO read + dq,dk,dv written.
FLOP_FWD, FLOP_BWD = 98304, 196608
BYTES_FWD, BYTES_BWD = 1024, 1792
# algorithmic bytes per token-head of one launch of each tensor-core kernel kind:
# the chunked kernel reads three bf16 sequence tensors and writes one (with the
# fused group aggregates of the dq pass it reads a fourth); the dual reverse-time
# kernel reads four (k, q, dO, v) and writes two (dk, dv); the aggregate kernel
# reads two.  Group states are overhead, not credited.
KIND_BYTES_PER_TOKEN_HEAD = {"tc_chunked_fwd": 1024, "tc_chunked_fwd_agg": 1280,
                             "tc_dual_rev": 1536, "tc_segment_aggregate": 512}
CHUNKED_KINDS = ("tc_chunked_fwd", "tc_chunked_fwd_agg", "tc_dual_rev")


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_max(x: float, device=None) -> float:
    """Maximum of x over the ranks of the default process group (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(units_per_rank: float, ms_per_step_max: float, world: int) -> float:
    """Units all ranks processed per second, timed by the slowest rank (weak scaling)."""
    return units_per_rank * world / (ms_per_step_max * 1e-3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _gpu_uuid(dev):
    import torch
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def _profile_traffic():
    """(DRAM bytes per token-head per step, launches per step) of the chunked kernels from the
    committed ncu summary of the current kernels, if any."""
    path = os.path.join(ROOT, "profiles", "chunked_kernels_traffic_B2H16T64K.md")
    vals = {}
    try:
        with open(path) as f:
            for ln in f:
                if "=" in ln and ln.split("=")[0].strip() in ("dram_bytes_per_token_head_per_step",
                                                             "chunked_launches_per_step"):
                    k, v = ln.split("=")
                    vals[k.strip()] = float(v)
    except OSError:
        return None
    if len(vals) != 2:
        return None
    return vals["dram_bytes_per_token_head_per_step"], vals["chunked_launches_per_step"]


# ---------------------------------------------------------------------------------- reference arm
def workload_config(cfg, ws_n):
    """The `config` object of the JSON line, the same for both arms."""
    from chunked_state_scan_causal_gb300 import inputs
    lam = inputs.workload_decay(cfg)
    gated = cfg.get("gates") is not None
    return {"workload": cfg["name"], "B": cfg["B"], "H": cfg["H"], "T": cfg["T"], "d": cfg["d"], "chunk": 64,
            "decay": "per-head" if lam is not None else ("per-token gates" if gated else "none"),
            "l2": "inputs 512 MiB per tensor > L2 (no flush)",
            "step": "linattn_fwd_ckpt + linattn_bwd_ckpt", "parallelism": f"replicas x{ws_n}"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from chunked_state_scan_causal_gb300 import inputs
    cfg = inputs.WORKLOADS[args.workload]
    oracle.build()
    T = cfg["T"]
    heads = list(range(min(cfg["H"], args.ref_heads)))
    lam = inputs.workload_decay(cfg)
    lam_s = None if lam is None else lam[heads]
    x = {w: np.stack([inputs.make_head64(cfg, w, 0, h) for h in heads])[None] for w in ("q", "k", "v", "dO")}
    gates = None
    if cfg.get("gates") is not None:
        gates = np.stack([inputs.gate_head(cfg, 0, h) for h in heads])[None].astype(np.float64)

    def run(n):
        xs = [x[w][:, :, :n] for w in ("q", "k", "v", "dO")]
        if gates is not None:
            oracle.fwd_gated(*xs[:3], gates[:, :, :n])
            oracle.bwd_gated(*xs, gates[:, :, :n])
            return
        oracle.fwd_recurrent(*xs[:3], lam=lam_s)
        oracle.bwd_recurrent(*xs, lam=lam_s)

    # each step is the first T_s tokens of every sampled head, T_s sized so that the
    # whole run (warm-up + timed steps) takes about --ref-budget seconds
    n_cal = min(T, 2048)
    t0 = time.perf_counter()
    run(n_cal)
    per_token = (time.perf_counter() - t0) / n_cal
    T_s = int(args.ref_budget / (args.warmup + args.steps) / per_token) // 64 * 64
    T_s = max(64, min(T, T_s))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        run(T_s)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    tokens = T_s * len(heads) / cfg["H"]  # token equivalents of the full-head workload
    value = tokens / sec
    sample = (f"batch row 0, heads 0..{len(heads) - 1} of {cfg['H']}, first {T_s} of T={T} tokens: "
              f"fwd+bwd fp64 recurrence")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, ws),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads_used(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import chunked_state_scan_causal_gb300 as la
    from chunked_state_scan_causal_gb300 import build, inputs

    ws_n, rank, local = _dist()
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    cfg = dict(inputs.WORKLOADS[args.workload])
    if args.B:
        cfg["B"] = args.B
    if args.T:
        cfg["T"] = args.T
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    lam = inputs.workload_decay(cfg)

    # inputs: seeded on the host, pinned, copied once (the device-resident leg)
    gated = cfg.get("gates") is not None
    host = {w: inputs.make(cfg, w).pin_memory() for w in ("q", "k", "v", "dO")}
    if gated:
        host["log_gate"] = inputs.make_gates(cfg).pin_memory()
    x = {w: t.to(dev, non_blocking=True) for w, t in host.items()}
    decay = None if lam is None else torch.from_numpy(lam).to(dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    def buffers():
        """Outputs, workspaces and the forward's checkpoint of one step."""
        b = dict(o=torch.empty_like(x["q"]), g=[torch.empty_like(x["q"]) for _ in range(3)])
        if gated:
            b.update(wsf=la.workspace(x["q"], la.OP_FWD_GATED), wsb=la.workspace(x["q"], la.OP_BWD_GATED),
                     ck=la.checkpoint_gated(x["q"]), dlg=torch.empty_like(x["log_gate"]))
        else:
            b.update(wsf=la.workspace(x["q"], la.OP_FWD, decay), wsb=la.workspace(x["q"], la.OP_BWD, decay),
                     ck=la.checkpoint(x["q"], decay))
        return b

    def layer(xs, b):
        # a training step of the layer: forward keeping its group states, then backward
        if gated:
            la.fwd_gated(xs["q"], xs["k"], xs["v"], xs["log_gate"], b["ck"], out=b["o"], ws=b["wsf"])
            la.bwd_gated(xs["q"], xs["k"], xs["v"], xs["dO"], xs["log_gate"], b["ck"], outs=b["g"], ws=b["wsb"],
                         dlg_out=b["dlg"])
        else:
            la.fwd(xs["q"], xs["k"], xs["v"], decay=decay, out=b["o"], ws=b["wsf"], ckpt=b["ck"])
            la.bwd(xs["q"], xs["k"], xs["v"], xs["dO"], decay=decay, outs=b["g"], ws=b["wsb"], ckpt=b["ck"])

    main_buf = buffers()

    def step():
        layer(x, main_buf)

    def barrier():
        if ws_n > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if la.device_status(main_buf["wsb"]) != la.OK or la.device_status(main_buf["wsf"]) != la.OK:
        raise RuntimeError("device-side error during warm-up")

    # ---- timed region (inputs are 512 MiB per tensor, 4x larger than L2: no flush needed)
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(_gpu_uuid(dev)) as clk:
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    la.linattn_timing_enable(False)
    kernels = la.linattn_timing_collect()
    ms = dist_max(e0.elapsed_time(e1) / args.steps, dev)
    tokens_step = B * T * ws_n
    value = whole_job_throughput(B * T, ms, ws_n)
    flops = (FLOP_FWD + FLOP_BWD) * B * H * T
    # gates add a 4-byte log-gate read to each pass and the 4-byte gate gradient written
    bytes_ = (BYTES_FWD + BYTES_BWD + (12 if gated else 0)) * B * H * T
    hbm, tf, peak_src = _peaks()

    # ---- dominant kernels' roofline: the chunked tensor-core kernels (the forward-time
    # chunked kernel for o and dq, the dual reverse-time kernel for dk and dv); achieved =
    # their algorithmic bytes over their summed CUDA-event time on the launching stream
    launches = sum(n for n, _ in kernels.values())
    tok_heads = B * H * T
    main = {k: kernels[k] for k in CHUNKED_KINDS if k in kernels}
    n_main = sum(n for n, _ in main.values())
    ms_main = sum(t for _, t in main.values())
    bytes_main = sum(KIND_BYTES_PER_TOKEN_HEAD[k] * tok_heads * n for k, (n, _) in main.items())
    achieved = bytes_main / (ms_main * 1e-3) / 1e9 if n_main else None
    traffic_tok = _profile_traffic()
    roofline = {
        "kernel": "chunked tensor-core kernels: " + ", ".join(f"{k} x{n // args.steps}" for k, (n, _) in main.items()),
        "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
        "frac": (achieved / hbm) if achieved else None,
        # measured for the benchmark workload with lambda = 1 (null for other workloads)
        "traffic": (traffic_tok[0] * tok_heads / traffic_tok[1]) if (
            traffic_tok and args.workload == 3 and not args.B and not args.T) else None,
        "peak_source": f"{peak_src} hbm_gbs",
        "launches_per_step": n_main / args.steps,
        "share_of_step": ms_main / (ms * args.steps) if ms else None,
    }
    # token-heads per step that the aggregate launches cover: the forward's, plus
    # the backward's for the heads whose dq pass does not accumulate them itself
    # (gates, or a per-head decay below 0.8, where the chunked kernels switch
    # to their weighted-operand form)
    if gated:
        agg_units = 2 * tok_heads
    elif lam is not None:
        agg_units = tok_heads * (1 + float((lam < 0.8).mean()))
    else:
        agg_units = tok_heads
    breakdown = {}
    for k, (n, t) in kernels.items():
        e = {"launches_per_step": n / args.steps, "ms_per_step": t / args.steps}
        if k in KIND_BYTES_PER_TOKEN_HEAD and t > 0:
            units = agg_units * args.steps if k == "tc_segment_aggregate" else tok_heads * n
            e["algorithmic_gbs"] = KIND_BYTES_PER_TOKEN_HEAD[k] * units / (t * 1e-3) / 1e9
        breakdown[k] = e

    # ---- end to end through the public API with host buffers: every step copies its
    # inputs host->device from pinned memory and its results (o, dq, dk, dv) device->host.
    # Steps are pipelined over two buffer sets on three streams (copy-in, compute,
    # copy-out), so step i+1's inputs arrive while step i computes.
    ms_e2e, h2d, d2h = None, 0, 0
    if not args.no_e2e:
        slots = []
        for _ in range(2):
            xin = {w: torch.empty_like(x[w]) for w in x}
            b = buffers()
            outs = [b["o"]] + b["g"] + ([b["dlg"]] if gated else [])
            hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
            ev = {n: torch.cuda.Event() for n in ("in", "comp", "out")}
            slots.append(dict(x=xin, b=b, o=outs, h=hout, ev=ev, used=False))
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in slots[0]["h"])

        def e2e_step(i):
            sl = slots[i % 2]
            with torch.cuda.stream(s_in):
                if sl["used"]:
                    s_in.wait_event(sl["ev"]["comp"])      # compute done reading this slot's inputs
                for w in x:
                    sl["x"][w].copy_(host[w], non_blocking=True)
                sl["ev"]["in"].record(s_in)
            stream.wait_event(sl["ev"]["in"])
            if sl["used"]:
                stream.wait_event(sl["ev"]["out"])         # previous results of this slot copied out
            layer(sl["x"], sl["b"])
            sl["ev"]["comp"].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(sl["ev"]["comp"])
                for hbuf, t in zip(sl["h"], sl["o"]):
                    hbuf.copy_(t, non_blocking=True)
                sl["ev"]["out"].record(s_out)
            sl["used"] = True

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        n_e2e = max(6, args.steps // 4)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(s_in)                                   # all streams are idle here
        for i in range(n_e2e):
            e2e_step(i)
        ev1.record(s_out)                                  # after the last copy-out, which waits for all else
        torch.cuda.synchronize()
        ms_e2e = dist_max(ev0.elapsed_time(ev1) / n_e2e, dev)

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        import numpy as np
        import oracle
        oracle.build()
        heads = list(range(min(H, args.cpu_heads)))
        xs = {w: np.stack([inputs.make_head64(cfg, w, 0, h) for h in heads])[None]
              for w in ("q", "k", "v", "dO")}
        lam_s = None if lam is None else lam[heads]
        t0 = time.perf_counter()
        if gated:
            gs = np.stack([inputs.gate_head(cfg, 0, h) for h in heads])[None].astype(np.float64)
            oracle.fwd_gated(xs["q"], xs["k"], xs["v"], gs)
            oracle.bwd_gated(xs["q"], xs["k"], xs["v"], xs["dO"], gs)
        else:
            oracle.fwd_recurrent(xs["q"], xs["k"], xs["v"], lam=lam_s)
            oracle.bwd_recurrent(xs["q"], xs["k"], xs["v"], xs["dO"], lam=lam_s)
        sec = time.perf_counter() - t0
        cpu = {"value": T * len(heads) / H / sec, "unit": "tokens/s", "cores": oracle.threads_used(),
               "kind": "oracle",
               "sample": f"batch row 0, heads 0..{len(heads) - 1} of {H}, T={T}, fwd+bwd fp64 recurrence, "
                         f"{sec:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal; no dataset)",
            "config": workload_config(cfg, ws_n),
            "tflops": flops / (ms * 1e-3) / 1e12,
            "algorithmic_gbs": bytes_ / (ms * 1e-3) / 1e9,
            "path_roofline_frac": max(flops / (tf * 1e12), bytes_ / (hbm * 1e9)) / (ms * 1e-3),
            "roofline": roofline,
            "kernels": breakdown,
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "e2e": None if ms_e2e is None else {
                "value": whole_job_throughput(B * T, ms_e2e, ws_n), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------------- decode
def run_decode(args):
    """Recurrent decode (constant-memory inference): one new token per sequence per call
    for decode_batch x 16 heads at d = 128, the fp32 states resident on the device.  Bound
    by the state traffic: 2 d^2 fp32 (read + write) per sequence per call."""
    import torch
    import chunked_state_scan_causal_gb300 as la
    from chunked_state_scan_causal_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    B, H, d, T = args.decode_batch, 16, 128, 1
    g = torch.Generator(device="cpu").manual_seed(9)
    q, k, v = [(torch.randn(B, H, T, d, generator=g) / d ** 0.5).to(torch.bfloat16).to(dev) for _ in range(3)]
    state = torch.zeros(B, H, d, d, dtype=torch.float32, device=dev)
    o = torch.empty_like(q)
    decay = torch.full((H,), 0.99, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        la.decode(q, k, v, state, decay=decay, out=o)
    torch.cuda.synchronize()
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        la.decode(q, k, v, state, decay=decay, out=o)
    e1.record()
    torch.cuda.synchronize()
    la.linattn_timing_enable(False)
    kern = la.linattn_timing_collect().get("decode", (0, 0.0))
    ms = e0.elapsed_time(e1) / args.steps
    seq = B * H
    bytes_call = seq * (2 * d * d * 4 + 4 * T * d * 2)  # states in and out, q, k, v read, o written
    hbm, _, src = _peaks()
    kms = kern[1] / max(kern[0], 1)
    print(json.dumps({
        "metric": "recurrent decode tokens/s (one token per sequence per call)", "value": B * T / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16 (fp32 state)", "data": "synthetic",
        "config": {"workload": f"decode-B{B}H{H}-d{d}", "B": B, "H": H, "T_per_call": T, "d": d},
        "roofline": {"kernel": "decode_kernel", "bound": "hbm", "achieved": bytes_call / (kms * 1e-3) / 1e9,
                     "peak": hbm, "unit": "GB/s", "frac": bytes_call / (kms * 1e-3) / 1e9 / hbm,
                     "peak_source": f"{src} hbm_gbs"},
        "gpu_launches": kern[0]}), flush=True)


# ---------------------------------------------------------------------------------- sequence split
def run_sp(args):
    """The sequence split across ranks (sp.forward + sp.backward) with N ranks as threads of
    this process on one GPU, each holding T/N tokens of every sequence of the workload; the
    ranks share the GPU, so this measures the split's total cost (its extra passes over the
    segments and the exchanges) against the unsplit step, not scaling."""
    import threading
    import torch
    import chunked_state_scan_causal_gb300 as la
    from chunked_state_scan_causal_gb300 import build, inputs, sp
    build.build()
    dev = torch.device("cuda", 0)
    cfg = dict(inputs.WORKLOADS[args.workload])
    B, H, T = cfg["B"], cfg["H"], cfg["T"]
    N = args.sp
    L = T // N
    x = {w: inputs.make(cfg, w).to(dev) for w in ("q", "k", "v", "dO")}
    torch.cuda.synchronize()

    def split_step():
        group = sp.ThreadExchange.Group(N, timeout=60)
        errs = []

        def rank(r):
            ex = group.rank(r)
            try:
                seg = {w: t[:, :, r * L:(r + 1) * L] for w, t in x.items()}
                _, _, ctx = sp.forward(seg["q"], seg["k"], seg["v"], ex)
                sp.backward(seg["q"], seg["k"], seg["v"], seg["dO"], ctx, ex)
            except Exception as e:
                errs.append(e)
                ex.abort()

        th = [threading.Thread(target=rank, args=(r,)) for r in range(N)]
        for t in th:
            t.start()
        for t in th:
            t.join()
        if errs:
            raise errs[0]

    ck = la.checkpoint(x["q"])

    def whole_step():
        la.fwd(x["q"], x["k"], x["v"], ckpt=ck)
        la.bwd(x["q"], x["k"], x["v"], x["dO"], ckpt=ck)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    ms_split, ms_whole = timed(split_step), timed(whole_step)
    print(json.dumps({
        "metric": f"sequence-split fwd+bwd tokens/s ({N} ranks as threads on one GPU)",
        "value": B * T / (ms_split * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_split, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg["name"], "ranks": N, "segment": L},
        "unsplit_ms_per_step": ms_whole, "split_over_unsplit": ms_split / ms_whole}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--ref-heads", type=int, default=16, help="heads per step of the reference arm")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds for the whole reference arm")
    ap.add_argument("--cpu-heads", type=int, default=16, help="heads of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--B", type=int, default=0, help="override the batch size (profiling cases)")
    ap.add_argument("--T", type=int, default=0, help="override the sequence length (profiling cases)")
    ap.add_argument("--decode", action="store_true", help="measure the recurrent decode instead")
    ap.add_argument("--decode-batch", type=int, default=512, help="sequences per head for --decode")
    ap.add_argument("--sp", type=int, default=0, help="measure the sequence split with this many thread ranks")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.decode:
        run_decode(args)
    elif args.sp:
        run_sp(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
