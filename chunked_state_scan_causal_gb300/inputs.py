"""Seeded synthetic workloads (shared by the tests, the smoke check and the benchmark).

This module holds no arithmetic of the attention method: it only draws random
tensors, rounds them to the workload's element type and lists the workload
shapes.  Both the CUDA path and the CPU oracle receive exactly these values.

Recipe (one stream per tensor and head, so any head can be regenerated alone):
  rng = numpy PCG64(SeedSequence([seed, tensor_id, b, h]))   tensor_id: q=0 k=1 v=2 dO=3
  x   = rng.standard_normal((T, d), float32)
  scale by the workload's sigma, for "unit_k" divide every key row by its fp32
  L2 norm, then round to the element type with torch (round-to-nearest-even).
Decays (the per-head decay workload): lambda_h = 1 - 2^-(5 + 8h/32) evaluated
in float64 and rounded once to float32.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

TENSOR_ID = {"q": 0, "k": 1, "v": 2, "dO": 3}  # 4: the log-gates of a gated workload

# The workloads.  "sigma" is the std-dev of q, k, v; dO is always N(0, 1).
WORKLOADS = {
    1: dict(name="tiny-fp32-fwd-B1H2T1K-d64", B=1, H=2, T=1024, d=64, dtype="f32",
            decay=None, dist="normal", sigma=0.125, seed=0, passes="fwd+chunk_states"),
    2: dict(name="fwd-B4H16T16K-d128", B=4, H=16, T=16384, d=128, dtype="bf16",
            decay=None, dist="unit_k", sigma=1.0 / math.sqrt(128), seed=1, passes="fwd"),
    3: dict(name="fwdbwd-B2H16T64K-d128", B=2, H=16, T=65536, d=128, dtype="bf16",
            decay=None, dist="normal", sigma=0.125, seed=2, passes="fwd+bwd"),
    4: dict(name="fwdbwd-decay-B1H32T128K-d128", B=1, H=32, T=131072, d=128, dtype="bf16",
            decay="per_head", dist="normal", sigma=1.0 / math.sqrt(128), seed=3, passes="fwd+bwd"),
    5: dict(name="segmented-B1H16T1M-d128-64x16K", B=1, H=16, T=1 << 20, d=128, dtype="bf16",
            decay=None, dist="normal", sigma=1.0 / math.sqrt(128), seed=4, passes="segments",
            seg_len=16384),
    # data-dependent gates: log_gate ~ U(-1/16, 0) per token and head (gates in [0.94, 1])
    6: dict(name="fwdbwd-gated-B1H32T128K-d128", B=1, H=32, T=131072, d=128, dtype="bf16",
            decay=None, dist="normal", sigma=1.0 / math.sqrt(128), seed=5, passes="fwd+bwd",
            gates=(-1.0 / 16, 0.0)),
    # the benchmark's shape with heads of 64 (bf16: the d = 128 tensor-core kernels as the
    # zero-padded problem)
    7: dict(name="fwdbwd-B2H16T64K-d64", B=2, H=16, T=65536, d=64, dtype="bf16", decay=None,
            dist="normal", sigma=1.0 / math.sqrt(64), seed=6, passes="fwd+bwd"),
    # per-dimension gates: log_gate ~ U(-1/16, 0) per token, head and key dimension
    8: dict(name="fwdbwd-gatedvec-B1H32T128K-d128", B=1, H=32, T=131072, d=128, dtype="bf16",
            decay=None, dist="normal", sigma=1.0 / math.sqrt(128), seed=7, passes="fwd+bwd",
            gates=(-1.0 / 16, 0.0), gate_per_dim=True),
}


def decay_per_head(H: int) -> np.ndarray:
    """lambda_h = 1 - 2^-(5 + 8h/32) for h = 0..H-1 (float64 math, one rounding to float32)."""
    h = np.arange(H, dtype=np.float64)
    return (1.0 - np.power(2.0, -(5.0 + 8.0 * h / 32.0))).astype(np.float32)


def gate_head(cfg: dict, b: int, h: int, T: int | None = None) -> np.ndarray:
    """log-gates of one head, float32 [T] (or [T, d] with a gate per key dimension; uniform
    in cfg["gates"]), or None without gates."""
    if cfg.get("gates") is None:
        return None
    T = cfg["T"] if T is None else T
    lo, hi = cfg["gates"]
    ss = np.random.SeedSequence([cfg["seed"], 4, b, h])
    shape = (T, cfg["d"]) if cfg.get("gate_per_dim") else T
    return np.random.Generator(np.random.PCG64(ss)).uniform(lo, hi, shape).astype(np.float32)


def make_gates(cfg: dict, T: int | None = None, B: int | None = None, H: int | None = None, device=None):
    """log-gates [B, H, T] (or [B, H, T, d]) float32 of a gated workload (None without gates)."""
    if cfg.get("gates") is None:
        return None
    B = cfg["B"] if B is None else B
    H = cfg["H"] if H is None else H
    g = np.stack([np.stack([gate_head(cfg, b, h, T) for h in range(H)]) for b in range(B)])
    return torch.from_numpy(g).to(device) if device is not None else torch.from_numpy(g)


def workload_decay(cfg: dict):
    return decay_per_head(cfg["H"]) if cfg.get("decay") == "per_head" else None


def _torch_dtype(name: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def head(seed: int, which: str, b: int, h: int, T: int, d: int, dist: str, sigma: float) -> np.ndarray:
    """One head of one tensor as float32 (before the element-type rounding)."""
    ss = np.random.SeedSequence([seed, TENSOR_ID[which], b, h])
    x = np.random.Generator(np.random.PCG64(ss)).standard_normal((T, d), dtype=np.float32)
    if which == "dO":
        return x
    x *= np.float32(sigma)
    if dist == "unit_k" and which == "k":
        n = np.sqrt(np.sum(x * x, axis=1, dtype=np.float32), dtype=np.float32)
        x /= n[:, None]
    return x


def make(cfg: dict, which: str, T: int | None = None, B: int | None = None, H: int | None = None,
         device=None, threads: int = 16) -> torch.Tensor:
    """Tensor [B, H, T, d] of the workload's element type (optionally with a smaller B/H/T)."""
    B = cfg["B"] if B is None else B
    H = cfg["H"] if H is None else H
    T = cfg["T"] if T is None else T
    d = cfg["d"]
    dt = _torch_dtype(cfg["dtype"])
    out = torch.empty((B, H, T, d), dtype=dt, device=device)

    def one(bh):
        b, h = divmod(bh, H)
        x = head(cfg["seed"], which, b, h, T, d, cfg["dist"], cfg["sigma"])
        out[b, h].copy_(torch.from_numpy(x).to(dt))

    with ThreadPoolExecutor(max_workers=max(1, min(threads, B * H))) as ex:
        list(ex.map(one, range(B * H)))
    return out


def make_head64(cfg: dict, which: str, b: int, h: int, T: int | None = None) -> np.ndarray:
    """One head, rounded to the workload's element type, widened to float64 ([T, d])."""
    T = cfg["T"] if T is None else T
    x = head(cfg["seed"], which, b, h, T, cfg["d"], cfg["dist"], cfg["sigma"])
    dt = _torch_dtype(cfg["dtype"])
    return torch.from_numpy(x).to(dt).to(torch.float64).numpy()


def random_case(seed: int, B: int, H: int, T: int, d: int, dtype: str = "bf16", sigma: float = 0.125,
                dv: int | None = None, with_dO: bool = True):
    """Small ad-hoc case (tests): dict of float64 numpy arrays holding element-type-rounded values."""
    cfg = dict(B=B, H=H, T=T, d=d, dtype=dtype, dist="normal", sigma=sigma, seed=seed)
    out = {}
    for w in ("q", "k", "v", "dO") if with_dO else ("q", "k", "v"):
        dd = d if w in ("q", "k") or dv is None else dv
        arr = np.empty((B, H, T, dd))
        for b in range(B):
            for h in range(H):
                x = head(seed, w, b, h, T, dd, "normal", sigma)
                arr[b, h] = torch.from_numpy(x).to(_torch_dtype(dtype)).to(torch.float64).numpy()
        out[w] = arr
    return out
