"""Benchmark of chunked causal linear attention on GB300.

A "step" is one pass of the whole hot path over one batch of synthetic input:

  workload 3 (default): B=2 H=16 T=65536 d=128 bf16, lambda=1; step = the
      checkpointed forward (linattn_fwd_ckpt) then the backward
      (linattn_bwd_ckpt); q, k, v ~ N(0, 0.125^2), dO ~ N(0, 1), seeded;
  workload 2: B=4 H=16 T=16384 forward only (linattn_fwd);
  workload 4: B=1 H=32 T=131072 with per-head decays, forward + backward;
  workload 5: B=1 H=16 T=2^20 as 64 segments of 16384 tokens: segment states
      (linattn_chunk_states) -> exclusive scan (linattn_state_scan) ->
      per-segment forward from those states; the single unsegmented forward of
      the same sequence is timed in the same run (`single_fwd`);
  workload 6: B=1 H=32 T=131072 with per-token gates, forward + backward.
  workload 7: B=2 H=16 T=65536 d=64 bf16, forward + backward (the d = 128 kernels
    as the zero-padded problem).

Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 3]

The timed region runs with the library's per-kernel event timing off; the
per-kernel breakdown (`kernels`) comes from a separate pass afterwards.
--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the reference arm of this benchmark: there is no upstream code).
Under torchrun each rank runs an independent replica (weak scaling); only
rank 0 prints.
"""
from __future__ import annotations

import argparse
import ctypes
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
# Algorithmic work per token per head at d = 128 (chunk 64): forward 4d(C+d) FLOP,
# q, k, v read once and o written once; backward 8d(C+d) FLOP, q, k, v, dO read
# once and dq, dk, dv written once.  The segment pipeline reads k, v once more
# for the segment states (1536 B).  Group states, recomputation and re-reads
# are not credited.
FLOP_FWD, FLOP_BWD = 98304, 196608
BYTES_FWD, BYTES_BWD = 1024, 1792
BYTES_SEGMENTS = 1536
# Bytes each kernel kind moves per token-head and launch by its own inputs and
# outputs (sequence tensors only): an I/O figure per kernel, not the method's
# algorithmic bytes.
KIND_IO_BYTES_PER_TOKEN_HEAD = {"tc_chunked_fwd": 1024, "tc_chunked_fwd_agg": 1280,
                                "tc_dual_rev": 1536, "tc_segment_aggregate": 512}
# The tensor-core kernels run 128-token blocks (two chunks of 64): the chunked
# form equals the definition for any chunk length, only the rounding order changes.
BLOCK = 128
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


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


class _Nvml:
    """Read-only NVML queries through ctypes (clocks and clock-event reasons)."""
    SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, uuid: str | None, index: int):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        if uuid:
            ok = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) == 0
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
            raise OSError("no NVML device handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self):
        v = ctypes.c_uint()
        return v.value if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, ctypes.byref(v)) == 0 else None

    def max_sm_mhz(self):
        v = ctypes.c_uint()
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, ctypes.byref(v)) == 0 else None

    def reasons(self):
        v = ctypes.c_ulonglong()
        if self.reasons_fn(self.h, ctypes.byref(v)) != 0:
            return set()
        return {n for bit, n in self.REASONS.items() if v.value & bit}


class ClockSampler:
    """SM clock and throttle-reason samples while the timed region runs: NVML every
    2 ms (read-only queries), else nvidia-smi every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None, index: int = 0):
        self.gpu_id, self.index = gpu_id, index
        self.proc = None
        self.nvml = None
        self.lines = []
        self.samples = []   # (sm MHz, reasons)
        self.max_mhz = None
        self.stop = threading.Event()

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.gpu_id, self.index)
            self.max_mhz = self.nvml.max_sm_mhz()
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return self
        except Exception:
            self.nvml = None
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

    def _poll(self):
        while not self.stop.is_set():
            mhz = self.nvml.sm_mhz()
            if mhz is not None:
                self.samples.append((float(mhz), self.nvml.reasons()))
            self.stop.wait(0.002)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        self.stop.set()
        if self.nvml is not None:
            self.t.join(timeout=2)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], self.max_mhz, set()
        for mhz, rs in self.samples:
            sm.append(mhz)
            reasons |= rs
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
                "samples": len(sm), "source": "nvml" if self.samples else "nvidia-smi"}


def _gpu_uuid(dev):
    import torch
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def _traffic(workload_name: str):
    """DRAM bytes per token-head of one step of this workload, from profiles/traffic.json
    (written by `bench.py --traffic-from` out of an ncu capture), or None."""
    try:
        with open(TRAFFIC_JSON) as f:
            t = json.load(f)
        return t["workloads"][workload_name]
    except (OSError, KeyError, ValueError):
        return None


def traffic_from_ncu(csv_path: str, workload_name: str, units: float, note: str) -> dict:
    """Sum dram__bytes_read.sum + dram__bytes_write.sum over every captured launch of an
    `ncu --csv --metrics dram__bytes_read.sum,dram__bytes_write.sum` capture of whole steps,
    divide by the token-heads the captured steps processed (`units`) and store the result
    under the workload's name in profiles/traffic.json."""
    import csv
    per_kernel = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(ln for ln in f if not ln.startswith("=="))]
    head = rows[0]
    ik, im, iv, iu = head.index("Kernel Name"), head.index("Metric Name"), head.index("Metric Value"), \
        head.index("Metric Unit")
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
    for r in rows[1:]:
        if len(r) <= max(ik, im, iv, iu) or r[im] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        name = r[ik].split("(")[0].split("::")[-1].strip()
        v = float(r[iv].replace(",", "")) * scale.get(r[iu], 1)
        per_kernel[name] = per_kernel.get(name, 0.0) + v
    total = sum(per_kernel.values())
    try:
        with open(TRAFFIC_JSON) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        doc = {}
    doc.setdefault("workloads", {})[workload_name] = {
        "dram_bytes_per_token_head_per_step": total / units,
        "per_kernel": {k: v / units for k, v in sorted(per_kernel.items())},
        "note": note}
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(doc, f, indent=1)
    return doc["workloads"][workload_name]


# ---------------------------------------------------------------------------------- workloads
def passes(cfg) -> str:
    return cfg["passes"]


def step_units(cfg):
    """(algorithmic FLOP, algorithmic bytes) per token-head of one step of the workload.

    The constants above are for d = 128; bytes scale with d (bf16 rows of d), and
    FLOPs are 4 C d (the masked intra-chunk products) + 4 d^2 (the state products)
    per pass, the backward twice the forward."""
    gated = cfg.get("gates") is not None
    p = passes(cfg)
    d = cfg["d"]
    fs = (4 * 64 * d + 4 * d * d) / FLOP_FWD  # 1 at d = 128
    bs = d / 128
    if p == "fwd":
        return FLOP_FWD * fs, BYTES_FWD * bs
    if p == "segments":
        return FLOP_FWD * fs, BYTES_SEGMENTS * bs
    # gates add a 4-byte log-gate read to each pass and the 4-byte gate gradient written
    return (FLOP_FWD + FLOP_BWD) * fs, (BYTES_FWD + BYTES_BWD) * bs + (12 if gated else 0)


def step_name(cfg) -> str:
    p = passes(cfg)
    if p == "fwd":
        return "linattn_fwd"
    if p == "segments":
        return "linattn_chunk_states -> linattn_state_scan -> linattn_fwd(init) over 64 segments"
    if cfg.get("gates") is not None:
        return "linattn_fwd_gated + linattn_bwd_gated"
    return "linattn_fwd_ckpt + linattn_bwd_ckpt"


def workload_config(cfg, ws_n):
    """The `config` object of the JSON line, the same for both arms."""
    from chunked_state_scan_causal_gb300 import inputs
    lam = inputs.workload_decay(cfg)
    gated = cfg.get("gates") is not None
    c = {"workload": cfg["name"], "B": cfg["B"], "H": cfg["H"], "T": cfg["T"], "d": cfg["d"], "chunk": 64,
         "block": BLOCK,
         "decay": "per-head" if lam is not None else ("per-token gates" if gated else "none"),
         "l2": f"inputs {cfg['B'] * cfg['H'] * cfg['T'] * cfg['d'] * 2 >> 20} MiB per tensor > L2 (no flush)",
         "step": step_name(cfg), "parallelism": f"replicas x{ws_n}"}
    if passes(cfg) == "segments":
        c["segments"] = cfg["T"] // cfg["seg_len"]
        c["seg_len"] = cfg["seg_len"]
    return c


# ---------------------------------------------------------------------------------- reference arm
def _oracle_step(oracle, cfg, xs, lam_s, gates):
    p = passes(cfg)
    if gates is not None:
        oracle.fwd_gated(*xs[:3], gates)
        oracle.bwd_gated(*xs, gates)
    elif p in ("fwd", "segments"):
        oracle.fwd_recurrent(*xs[:3], lam=lam_s)
    else:
        oracle.fwd_recurrent(*xs[:3], lam=lam_s)
        oracle.bwd_recurrent(*xs, lam=lam_s)


def _oracle_label(cfg):
    return "fwd fp64 recurrence" if passes(cfg) in ("fwd", "segments") else "fwd+bwd fp64 recurrence"


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
    # at most the first 2^18 tokens of every sampled head are drawn (bounded host memory)
    T_max = min(T, 1 << 18)
    x = {w: np.stack([inputs.make_head64(cfg, w, 0, h, T=T_max) for h in heads])[None]
         for w in ("q", "k", "v", "dO")}
    gates = None
    if cfg.get("gates") is not None:
        gates = np.stack([inputs.gate_head(cfg, 0, h) for h in heads])[None].astype(np.float64)

    def run(n):
        xs = [x[w][:, :, :n] for w in ("q", "k", "v", "dO")]
        _oracle_step(oracle, cfg, xs, lam_s, None if gates is None else gates[:, :, :n])

    # each step is the first T_s tokens of every sampled head, T_s sized so that the
    # whole run (warm-up + timed steps) takes about --ref-budget seconds
    n_cal = min(T_max, 2048)
    t0 = time.perf_counter()
    run(n_cal)
    per_token = (time.perf_counter() - t0) / n_cal
    T_s = int(args.ref_budget / (args.warmup + args.steps) / per_token) // 64 * 64
    T_s = max(64, min(T_max, T_s))
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
              f"{_oracle_label(cfg)}")
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
def _cpu_baseline(cfg, args, lam):
    """The oracle, as it stands, on a bounded sample of the workload (rank 0, N = 1)."""
    import numpy as np
    import oracle
    from chunked_state_scan_causal_gb300 import inputs
    oracle.build()
    H, T = cfg["H"], cfg["T"]
    heads = list(range(min(H, args.cpu_heads)))
    T_s = min(T, args.cpu_tokens)
    xs = {w: np.stack([inputs.make_head64(cfg, w, 0, h, T=T_s) for h in heads])[None]
          for w in ("q", "k", "v", "dO")}
    lam_s = None if lam is None else lam[heads]
    gs = None
    if cfg.get("gates") is not None:
        gs = np.stack([inputs.gate_head(cfg, 0, h, T=T_s) for h in heads])[None].astype(np.float64)
    t0 = time.perf_counter()
    _oracle_step(oracle, cfg, [xs[w] for w in ("q", "k", "v", "dO")], lam_s, gs)
    sec = time.perf_counter() - t0
    extra = "" if T_s == T else f", first {T_s} of T={T} tokens (extrapolated linearly in tokens)"
    return {"value": T_s * len(heads) / H / sec, "unit": "tokens/s", "cores": oracle.threads_used(),
            "kind": "oracle",
            "sample": f"batch row 0, heads 0..{len(heads) - 1} of {H}{extra}, {_oracle_label(cfg)}, {sec:.1f} s"}


def _link_rates(dev, nbytes=1 << 29):
    """Host<->device copy rates (GB/s) of one pinned buffer, measured with CUDA events."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    rates = {}
    for name, (dst, src) in (("h2d_gbs", (d, h)), ("d2h_gbs", (h, d))):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        rates[name] = 3 * nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9
    return rates


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
    mode = passes(cfg)
    if mode not in ("fwd", "fwd+bwd", "segments"):
        raise SystemExit(f"workload {args.workload} ({mode}) is a parity case, not a bench workload")
    gated = cfg.get("gates") is not None

    # inputs: seeded on the host, pinned, copied once (the device-resident leg)
    names = ("q", "k", "v", "dO") if mode == "fwd+bwd" else ("q", "k", "v")
    host = {w: inputs.make(cfg, w).pin_memory() for w in names}
    if gated:
        host["log_gate"] = inputs.make_gates(cfg).pin_memory()
    x = {w: t.to(dev, non_blocking=True) for w, t in host.items()}
    decay = None if lam is None else torch.from_numpy(lam).to(dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    if mode == "segments":
        L = cfg["seg_len"]
        S = T // L

        def seg(t):  # [1, H, T, d] -> [S, H, L, d] view (segments as a batch, by strides)
            return t[0].view(H, S, L, d).permute(1, 0, 2, 3)

    def buffers():
        """Outputs, workspaces and checkpoints of one step."""
        b = dict(o=torch.empty_like(x["q"]))
        if mode == "fwd+bwd":
            b["g"] = [torch.empty_like(x["q"]) for _ in range(3)]
            if gated:
                b.update(wsf=la.workspace(x["q"], la.OP_FWD_GATED), wsb=la.workspace(x["q"], la.OP_BWD_GATED),
                         ck=la.checkpoint_gated(x["q"]), dlg=torch.empty_like(x["log_gate"]))
            else:
                b.update(wsf=la.workspace(x["q"], la.OP_FWD, decay), wsb=la.workspace(x["q"], la.OP_BWD, decay),
                         ck=la.checkpoint(x["q"], decay))
        elif mode == "fwd":
            b["wsf"] = la.workspace(x["q"], la.OP_FWD, decay)
        else:
            qs = seg(x["q"])
            b.update(U=torch.empty((S, 1, H, d, d), dtype=torch.float32, device=dev),
                     init=torch.empty((S, H, d, d), dtype=torch.float32, device=dev),
                     wsc=la.workspace(x["k"], la.OP_CHUNK_STATES, None, L),
                     wsf=la.workspace(qs, la.OP_FWD))
            st, n = la.linattn_state_scan_workspace_size(S, H, d, d)
            b["wss"] = torch.empty(n, dtype=torch.uint8, device=dev)
        return b

    def layer(xs, b):
        if mode == "fwd+bwd" and gated:
            la.fwd_gated(xs["q"], xs["k"], xs["v"], xs["log_gate"], b["ck"], out=b["o"], ws=b["wsf"])
            la.bwd_gated(xs["q"], xs["k"], xs["v"], xs["dO"], xs["log_gate"], b["ck"], outs=b["g"], ws=b["wsb"],
                         dlg_out=b["dlg"])
        elif mode == "fwd+bwd":
            # a training step of the layer: forward keeping its group states, then backward
            la.fwd(xs["q"], xs["k"], xs["v"], decay=decay, out=b["o"], ws=b["wsf"], ckpt=b["ck"])
            la.bwd(xs["q"], xs["k"], xs["v"], xs["dO"], decay=decay, outs=b["g"], ws=b["wsb"], ckpt=b["ck"])
        elif mode == "fwd":
            la.fwd(xs["q"], xs["k"], xs["v"], decay=decay, out=b["o"], ws=b["wsf"])
        else:
            la.chunk_states(xs["k"], xs["v"], L, out=b["U"], ws=b["wsc"])
            la.state_scan(b["U"].view(S, H, d, d), out=b["init"], ws=b["wss"])
            la.fwd(seg(xs["q"]), seg(xs["k"]), seg(xs["v"]), init_state=b["init"], out=seg(b["o"]), ws=b["wsf"])

    def outputs_of(b):
        outs = [b["o"]]
        if mode == "fwd+bwd":
            outs += b["g"] + ([b["dlg"]] if gated else [])
        return outs

    def status_ok(b):
        return all(la.device_status(b[k]) == la.OK for k in ("wsf", "wsb", "wsc", "wss") if k in b)

    main_buf = buffers()

    def step():
        layer(x, main_buf)

    def barrier():
        if ws_n > 1:
            import torch.distributed as dist
            dist.barrier()

    def timed(fn, n):
        """ms per call of fn over n calls, CUDA events on the launching stream."""
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return e0.elapsed_time(e1) / n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if not status_ok(main_buf):
        raise RuntimeError("device-side error during warm-up")

    # ---- timed region: per-kernel event timing off; inputs are larger than L2 (no flush)
    la.linattn_timing_enable(False)
    with ClockSampler(_gpu_uuid(dev), local) as clk:
        ms_local = timed(step, args.steps)
    ms = dist_max(ms_local, dev)
    if not status_ok(main_buf):
        raise RuntimeError("device-side error during the timed steps")

    # ---- per-kernel breakdown: a separate pass with the library's event timing on
    n_break = max(1, min(args.steps, 50))
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    timed(step, n_break)
    la.linattn_timing_enable(False)
    kernels = la.linattn_timing_collect()

    tok_heads = B * H * T
    flop_th, bytes_th = step_units(cfg)
    flops, bytes_ = flop_th * tok_heads, bytes_th * tok_heads
    hbm, tf, peak_src = _peaks()
    value = whole_job_throughput(B * T, ms, ws_n)
    launches = sum(n for n, _ in kernels.values())
    breakdown = {}
    for k, (n, t) in kernels.items():
        e = {"launches_per_step": n / n_break, "ms_per_step": t / n_break}
        if k in KIND_IO_BYTES_PER_TOKEN_HEAD and t > 0 and k != "tc_segment_aggregate":
            # bytes the kernel's own sequence-tensor inputs and outputs take per token-head
            io = KIND_IO_BYTES_PER_TOKEN_HEAD[k] * d / 128
            e["io_bytes_per_token_head"] = io
            e["io_gbs"] = io * tok_heads * n / (t * 1e-3) / 1e9
        breakdown[k] = e
    ms_kernels = sum(t for _, t in kernels.values()) / n_break
    traffic = _traffic(cfg["name"]) if not (args.B or args.T) else None
    # The roofline unit is the whole step (every launch of the hot path): achieved =
    # the step's algorithmic bytes / the step's device time; frac = achieved / peak.
    roofline = {
        "kernel": "whole step: " + ", ".join(f"{k} x{n / n_break:g}" for k, (n, _) in sorted(kernels.items())),
        "bound": "hbm", "achieved": bytes_ / (ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
        "frac": bytes_ / (ms * 1e-3) / 1e9 / hbm,
        "traffic": None if traffic is None else traffic["dram_bytes_per_token_head_per_step"] * tok_heads,
        "algorithmic_bytes": bytes_,
        "peak_source": f"{peak_src} hbm_gbs (of {peak_src})",
        "kernel_time_share": ms_kernels / ms if ms else None,
    }

    # ---- single unsegmented forward of the segment workload (same sequence, same run)
    single = None
    if mode == "segments":
        ob = torch.empty_like(x["q"])
        wso = la.workspace(x["q"], la.OP_FWD)

        def one():
            la.fwd(x["q"], x["k"], x["v"], out=ob, ws=wso)

        for _ in range(args.warmup):
            one()
        ms1 = dist_max(timed(one, args.steps), dev)
        if la.device_status(wso) != la.OK:
            raise RuntimeError("device-side error in the single forward")
        single = {"ms_per_step": ms1, "tokens_per_s": whole_job_throughput(B * T, ms1, ws_n),
                  "tflops": FLOP_FWD * tok_heads / (ms1 * 1e-3) / 1e12,
                  "algorithmic_gbs": BYTES_FWD * tok_heads / (ms1 * 1e-3) / 1e9,
                  "path_roofline_frac": BYTES_FWD * tok_heads / (ms1 * 1e-3) / 1e9 / hbm}

    # ---- end to end through the public API with host buffers: every step copies its
    # inputs host->device from pinned memory and its results device->host.  Steps are
    # pipelined over two buffer sets on three streams (copy-in, compute, copy-out), so
    # step i+1's inputs arrive while step i computes.
    ms_e2e, h2d, d2h, link = None, 0, 0, None
    if not args.no_e2e:
        slots = []
        for _ in range(2):
            xin = {w: torch.empty_like(x[w]) for w in x}
            b = buffers()
            outs = outputs_of(b)
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
        del slots
        link = _link_rates(dev)

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        cpu = _cpu_baseline(cfg, args, lam)

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
            "gpu_launches": launches * args.steps // n_break,
            "clocks": clk.summary(),
            "e2e": None if ms_e2e is None else {
                "value": whole_job_throughput(B * T, ms_e2e, ws_n), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "link": link,
                # the host link alone, both directions overlapped at their one-way rates
                "link_min_ms": max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9)) * 1e3},
            "cpu_baseline": cpu,
        }
        if single is not None:
            line["single_fwd"] = single
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


# ---------------------------------------------------------------------------------- softmax segment
def run_softmax_segment(args):
    """The softmax-attention segment of the hybrid variant: the last Tq = 16384 positions
    (one rank's segment of four) of a B1 H16 prefix of Tk = 65536 tokens attend causally
    over the gathered prefix, d = 128, bf16.  Tensor-bound: algorithmic FLOPs are
    4 d per (query, visible key) pair (Q K^T and P V)."""
    import numpy as np
    import torch
    import chunked_state_scan_causal_gb300 as la
    from chunked_state_scan_causal_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    B, H, Tk, Tq, d = 1, 16, args.sm_tk, args.sm_tq, 128
    g = torch.Generator(device="cpu").manual_seed(11)
    q = torch.randn(B, H, Tq, d, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(B, H, Tk, d, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(B, H, Tk, d, generator=g).to(torch.bfloat16).to(dev)
    o = torch.empty_like(q)
    ws = la.workspace(q, la.OP_SOFTMAX_SEGMENT)
    bwd = args.sm_bwd
    if bwd:
        # the backward alone, from the forward's o and lse
        dO = torch.randn(B, H, Tq, d, generator=g).to(torch.bfloat16).to(dev)
        _, lse = la.softmax_segment_fwd(q, k, v, out=o, want_lse=True, ws=ws)
        wsb = la.workspace(q, la.OP_SOFTMAX_SEGMENT_BWD)
        outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        step = lambda: la.softmax_segment_bwd(q, k, v, o, dO, lse, outs=outs, ws=wsb)
    else:
        wsb = ws
        step = lambda: la.softmax_segment_fwd(q, k, v, out=o, ws=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if la.device_status(wsb) != la.OK:
        raise RuntimeError("device-side error during warm-up")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(_gpu_uuid(dev), 0) as clk:
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    # per-kernel times from a separate pass (the library's event timing stays off above)
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    for _ in range(min(args.steps, 10)):
        step()
    torch.cuda.synchronize()
    kern = {name: round(t / n, 4) for name, (n, t) in la.linattn_timing_collect().items()}
    la.linattn_timing_enable(False)
    off = Tk - Tq
    pairs = Tq * off + Tq * (Tq + 1) // 2
    # forward: Q K^T and P V (4 d per visible pair); backward: the five products of the
    # usual count, Q K^T (recomputed), dO V^T, P^T dO, dS^T Q, dS K (10 d per pair)
    flops = (10 if bwd else 4) * d * pairs * B * H
    bytes_ = ((4 * Tq + 4 * Tk) if bwd else (2 * Tq + 2 * Tk)) * d * 2 * B * H  # each tensor once
    p = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(p.get("bf16_tflops", 1900.0))
    src = "measured bf16_tflops (burst, of measured)" if "bf16_tflops" in p else "fallback 1900 TFLOP/s"
    tf = flops / (ms * 1e-3) / 1e12
    cpu = None
    if not args.no_cpu_baseline and not bwd:
        import oracle
        rows = list(range(0, Tq, max(1, Tq // 16)))[:16]
        qn, kn, vn = (x[0:1, 0:4].double().cpu().numpy() for x in (q, k, v))
        t0 = time.perf_counter()
        oracle.softmax_segment_fwd(qn, kn, vn, rows=rows)
        sec = time.perf_counter() - t0
        rp = sum(off + r + 1 for r in rows) * 4
        cpu = {"value": 4 * d * rp / sec / 1e12, "unit": "TFLOP/s", "cores": oracle.threads_used(), "kind": "oracle",
               "sample": f"heads 0..3, {len(rows)} query rows spread over the segment, fp64 numpy, {sec:.2f} s"}
    if bwd and not args.no_cpu_baseline:
        # the last 128 queries of head 0 over the whole prefix (the same positions as in the
        # workload: its queries are the prefix's last Tq)
        import oracle
        n_s = min(128, Tq)
        qs, dOs = (x[0:1, 0:1, Tq - n_s:].double().cpu().numpy() for x in (q, dO))
        ks, vs = (x[0:1, 0:1].double().cpu().numpy() for x in (k, v))
        t0 = time.perf_counter()
        oracle.softmax_segment_bwd(qs, ks, vs, dOs)
        sec = time.perf_counter() - t0
        sp = n_s * (Tk - n_s) + n_s * (n_s + 1) // 2
        cpu = {"value": 10 * d * sp / sec / 1e12, "unit": "TFLOP/s", "cores": oracle.threads_used(), "kind": "oracle",
               "sample": f"head 0, the last {n_s} queries over the {Tk}-token prefix, fp64 numpy, {sec:.2f} s"}
    print(json.dumps({
        "metric": "causal softmax-attention segment " + ("backward " if bwd else "") +
                  "TFLOP/s (hybrid layers, prefix gathered)", "value": tf,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded normal)",
        "config": {"workload": f"softmax-segment-B{B}H{H}-Tq{Tq}-Tk{Tk}-d{d}", "B": B, "H": H, "Tq": Tq, "Tk": Tk,
                   "d": d, "causal": True, "scale": "1/sqrt(d)"},
        "tokens_per_s": B * Tq / (ms * 1e-3), "algorithmic_gbs": bytes_ / (ms * 1e-3) / 1e9,
        "roofline": {"kernel": "softmax_bwd_kernel (dK/dV and dQ)" if bwd else "softmax_segment_kernel",
                     "bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                     "traffic": None, "peak_source": src},
        "kernels_ms": kern, "gpu_launches": args.steps * (3 if bwd else 1), "clocks": clk.summary(),
        "cpu_baseline": cpu}), flush=True)


# ---------------------------------------------------------------------------------- per-dimension gates
def run_gated_vec(args):
    """The per-dimension gated step (fwd_gated_vec + bwd_gated_vec, the backward taking
    the forward's group states from its checkpoint) on workload 8 (B1 H32 T131072 d128
    bf16, log-gates U(-1/16, 0) per token, head and key dimension).  CUDA-core kernels
    walking chunk groups: bound by the fp32 pipe.  Algorithmic FLOPs per state element and
    token: the sequential recurrence's own arithmetic, forward 5 (the update a s + k v, 3;
    the output's q s, 2) and backward 12 (the forward states again, 3, with dq's S dO, 2;
    the reverse update, 3, with dk's R v and dv's R^T k, 2 each).  The group split's extra
    passes (the forward's group states from zero and the backward's reverse aggregates,
    2.5 each: two tokens folded into one update of 5 FLOP) are executed but not credited."""
    import torch
    import chunked_state_scan_causal_gb300 as la
    from chunked_state_scan_causal_gb300 import build, inputs
    build.build()
    dev = torch.device("cuda", 0)
    cfg = dict(inputs.WORKLOADS[8])
    B, H, d = cfg["B"], cfg["H"], cfg["d"]
    T = args.T or cfg["T"]  # --T: a shorter case of the same kernels (profiling)
    q, k, v, dO = (inputs.make(cfg, w, T=T).to(dev) for w in ("q", "k", "v", "dO"))
    lg = inputs.make_gates(cfg, T=T, device=dev)
    wsf, wsb = la.workspace(q, la.OP_FWD_GATED_VEC), la.workspace(q, la.OP_BWD_GATED_VEC)
    ck = la.checkpoint_gated_vec(q)
    o = torch.empty_like(q)
    outs = [torch.empty_like(q) for _ in range(3)]

    def step():
        la.fwd_gated_vec(q, k, v, lg, out=o, ws=wsf, ckpt=ck)
        la.bwd_gated_vec(q, k, v, dO, lg, outs=outs, ws=wsb, ckpt=ck)

    steps = args.steps
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if la.device_status(wsf) != la.OK or la.device_status(wsb) != la.OK:
        raise RuntimeError("device-side error during warm-up")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(_gpu_uuid(dev), 0) as clk:
        torch.cuda.synchronize()
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    la.linattn_timing_enable(True)
    la.linattn_timing_collect()
    for _ in range(min(steps, 5)):
        step()
    torch.cuda.synchronize()
    timing = la.linattn_timing_collect()
    la.linattn_timing_enable(False)
    kern = {name: round(t / n, 4) for name, (n, t) in timing.items()}
    launches = sum(n for n, _ in timing.values()) // min(steps, 5)
    units = B * H * T
    flops = 17 * d * d * units
    executed = 22 * d * d * units  # with the split's two extra passes
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = 2070.0
    peak = sm * 128 * 2 * mhz * 1e6 / 1e12  # FP32 FMA lanes x 2 FLOP x the maximum SM clock
    tf = flops / (ms * 1e-3) / 1e12
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        n_s = min(T, 1 << 17)  # about 10 s
        qs, ks, vs, ds = (x[0:1, 0:1, :n_s].double().cpu().numpy() for x in (q, k, v, dO))
        gs = lg[0:1, 0:1, :n_s].double().cpu().numpy()
        t0 = time.perf_counter()
        oracle.fwd_gated_vec(qs, ks, vs, gs)
        oracle.bwd_gated_vec(qs, ks, vs, ds, gs)
        sec = time.perf_counter() - t0
        cpu = {"value": 17 * d * d * n_s / sec / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"batch row 0, head 0, the first {n_s} tokens, fp64 C recurrence, {sec:.2f} s"}
    print(json.dumps({
        "metric": "per-dimension gated fwd+bwd token-heads/s", "value": units / (ms * 1e-3),
        "unit": "token-heads/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16 (fp32 state)", "data": "synthetic (seeded normal; uniform log-gates)",
        "config": {"workload": cfg["name"] if T == cfg["T"] else f"{cfg['name']} at T={T}", "B": B, "H": H, "T": T,
                   "d": d, "gates": "per token, head and key dim",
                   "step": "linattn_fwd_gated_vec_ckpt + linattn_bwd_gated_vec_ckpt"},
        "roofline": {"kernel": "gated_vec_fwd + gated_vec_bwd (whole step)", "bound": "alu", "achieved": tf,
                     "peak": peak, "unit": "TFLOP/s", "frac": tf / peak, "traffic": None,
                     "executed_tflops": executed / (ms * 1e-3) / 1e12,
                     "peak_source": f"{sm} SMs x 128 fp32 lanes x 2 FLOP x {mhz:.0f} MHz (nominal unit counts)"},
        "kernels_ms": kern, "gpu_launches": launches * steps, "clocks": clk.summary(), "cpu_baseline": cpu}),
        flush=True)


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
    ap.add_argument("--cpu-tokens", type=int, default=1 << 17, help="tokens per head of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--B", type=int, default=0, help="override the batch size (profiling cases)")
    ap.add_argument("--T", type=int, default=0, help="override the sequence length (profiling cases)")
    ap.add_argument("--decode", action="store_true", help="measure the recurrent decode instead")
    ap.add_argument("--decode-batch", type=int, default=512, help="sequences per head for --decode")
    ap.add_argument("--sp", type=int, default=0, help="measure the sequence split with this many thread ranks")
    ap.add_argument("--softmax-segment", action="store_true", help="measure the softmax-attention segment instead")
    ap.add_argument("--sm-tq", type=int, default=16384, help="queries of the softmax segment")
    ap.add_argument("--sm-tk", type=int, default=65536, help="gathered prefix length of the softmax segment")
    ap.add_argument("--sm-bwd", action="store_true", help="with --softmax-segment: time the backward")
    ap.add_argument("--gated-vec", action="store_true", help="measure the per-dimension gated step instead "
                    "(workload 8; pass --steps 20)")
    ap.add_argument("--traffic-from", default="", help="ncu CSV of whole steps (dram__bytes_read/write.sum): "
                    "store DRAM bytes per token-head in profiles/traffic.json and exit")
    ap.add_argument("--traffic-steps", type=int, default=1, help="steps the --traffic-from capture covers")
    ap.add_argument("--traffic-note", default="", help="how the --traffic-from capture was taken")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.traffic_from:
        from chunked_state_scan_causal_gb300 import inputs
        cfg = dict(inputs.WORKLOADS[args.workload])
        B, T = args.B or cfg["B"], args.T or cfg["T"]
        units = B * cfg["H"] * T * args.traffic_steps
        print(json.dumps(traffic_from_ncu(args.traffic_from, cfg["name"], units, args.traffic_note)))
    elif args.decode:
        run_decode(args)
    elif args.softmax_segment:
        run_softmax_segment(args)
    elif args.gated_vec:
        run_gated_vec(args)
    elif args.sp:
        run_sp(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
