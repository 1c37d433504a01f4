"""Chunked causal linear attention for GB300 (sm_103a): Python binding of liblinattn.

Argument marshalling only: every step of the computation runs in the CUDA
library (``_lib/liblinattn.so``, built in-tree by ``build.py``).  PyTorch is
used to allocate outputs and workspaces and to supply the current stream.
There is no fallback: if the library is missing, every call raises.

Low-level functions carry the C names (``linattn_fwd`` ...) and take raw
pointers; the helpers ``fwd``, ``bwd``, ``chunk_states`` and ``state_scan``
take torch tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "liblinattn.so")

OK = 0
ERR_INVALID = -1
ERR_UNSUPPORTED = -2
ERR_ALIGN = -3
ERR_WORKSPACE = -4
ERR_CUDA = -5
ERR_DEVICE_TIMEOUT = -6
ERR_DEVICE = -7
ERR_SCRATCH_LIMIT = -8
NOALLOC_MAX_TILES = 65536
BF16, F32 = 0, 1
OP_FWD, OP_BWD, OP_CHUNK_STATES, OP_CHECKPOINT = 1, 2, 3, 4
OP_FWD_GATED, OP_BWD_GATED, OP_CHECKPOINT_GATED = 5, 6, 7
OP_SOFTMAX_SEGMENT, OP_SOFTMAX_SEGMENT_BWD = 8, 9
OP_FWD_GATED_VEC, OP_BWD_GATED_VEC, OP_CHECKPOINT_GATED_VEC = 10, 11, 12
ABI_VERSION = 2


class LinattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


class Shape(ctypes.Structure):
    """Mirror of ``linattn_shape`` in include/linattn.h."""
    _fields_ = [
        ("abi_version", ctypes.c_int32), ("B", ctypes.c_int32), ("H", ctypes.c_int32),
        ("T", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
        ("chunk", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64), ("stride_t", ctypes.c_int64),
        ("decay", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None
_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_SIGS = {
    "linattn_abi_version": ([], _i32),
    "linattn_status_string": ([_i32], ctypes.c_char_p),
    "linattn_workspace_size": ([ctypes.POINTER(Shape), _i32, _i32, ctypes.POINTER(_sz)], _i32),
    "linattn_fwd": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "linattn_bwd": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "linattn_fwd_ckpt": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp], _i32),
    "linattn_bwd_ckpt": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp, _vp, _vp, _vp,
                          _sz, _vp], _i32),
    "linattn_chunk_states": ([ctypes.POINTER(Shape), _i32, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "linattn_chunk_states_rev": ([ctypes.POINTER(Shape), _i32, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "linattn_fwd_gated": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp], _i32),
    "linattn_bwd_gated": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp, _vp, _vp,
                           _vp, _vp, _sz, _vp], _i32),
    "linattn_fwd_gated_vec": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "linattn_bwd_gated_vec": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                               _vp, _sz, _vp], _i32),
    "linattn_fwd_gated_vec_ckpt": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz,
                                    _vp], _i32),
    "linattn_bwd_gated_vec_ckpt": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp,
                                    _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "linattn_decode": ([ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "linattn_state_scan_workspace_size": ([_i32, _i32, _i32, _i32, ctypes.POINTER(_sz)], _i32),
    "linattn_state_scan": ([_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "linattn_device_status": ([_vp, _vp], _i32),
    "linattn_state_scan_noalloc": ([_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "linattn_diag_mma": ([_i32, _vp, _vp, _vp, _vp], _i32),
    "linattn_segment_decay": ([_vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "linattn_softmax_segment_fwd": ([ctypes.POINTER(Shape), ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp,
                                     ctypes.c_float, _vp, _sz, _vp], _i32),
    "linattn_softmax_segment_bwd": ([ctypes.POINTER(Shape), ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _vp, ctypes.c_float, _vp, _sz, _vp], _i32),
    "linattn_diag_scan_withhold": ([_i32, _i32, _i32, _i32, _vp, _vp, _i32, ctypes.c_double, _vp, _sz, _vp],
                                   _i32),
    "linattn_timing_enable": ([_i32], _i32),
    "linattn_timing_collect": ([_i32, ctypes.POINTER(_i32), ctypes.POINTER(ctypes.c_float)], _i32),
    "linattn_kernel_name": ([_i32], ctypes.c_char_p),
}
KERNEL_KINDS = 20


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m chunked_state_scan_causal_gb300.build`")
            l = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                f = getattr(l, name)
                f.argtypes = args
                f.restype = res
            _lib = l
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().linattn_status_string(status).decode()
    except RuntimeError:
        return "?"


# ------------------------------------------------------------------ C names (raw pointers)
def linattn_status_string(status: int) -> str:
    return lib().linattn_status_string(status).decode()


def linattn_abi_version() -> int:
    return lib().linattn_abi_version()


def linattn_workspace_size(shape: Shape, op: int, seg_len: int = 0) -> tuple[int, int]:
    n = _sz(0)
    st = lib().linattn_workspace_size(ctypes.byref(shape), op, seg_len, ctypes.byref(n))
    return st, n.value


def linattn_fwd(shape, q, k, v, o, init_state, final_state, chunk_states, ws, ws_bytes, stream) -> int:
    return lib().linattn_fwd(ctypes.byref(shape), q, k, v, o, init_state, final_state, chunk_states,
                             ws, ws_bytes, stream)


def linattn_bwd(shape, q, k, v, dO, init_state, d_final, dq, dk, dv, d_init, ws, ws_bytes, stream) -> int:
    return lib().linattn_bwd(ctypes.byref(shape), q, k, v, dO, init_state, d_final, dq, dk, dv, d_init,
                             ws, ws_bytes, stream)


def linattn_decode(shape, q, k, v, o, state, stream) -> int:
    return lib().linattn_decode(ctypes.byref(shape), q, k, v, o, state, stream)


def linattn_fwd_ckpt(shape, q, k, v, o, init_state, final_state, ckpt, ckpt_bytes, ws, ws_bytes, stream) -> int:
    return lib().linattn_fwd_ckpt(ctypes.byref(shape), q, k, v, o, init_state, final_state, ckpt, ckpt_bytes,
                                  ws, ws_bytes, stream)


def linattn_bwd_ckpt(shape, q, k, v, dO, init_state, d_final, ckpt, ckpt_bytes, dq, dk, dv, d_init, ws, ws_bytes,
                     stream) -> int:
    return lib().linattn_bwd_ckpt(ctypes.byref(shape), q, k, v, dO, init_state, d_final, ckpt, ckpt_bytes, dq, dk,
                                  dv, d_init, ws, ws_bytes, stream)


def linattn_chunk_states(shape, seg_len, k, v, out, ws, ws_bytes, stream) -> int:
    return lib().linattn_chunk_states(ctypes.byref(shape), seg_len, k, v, out, ws, ws_bytes, stream)


def linattn_fwd_gated(shape, q, k, v, log_gate, o, init_state, final_state, ckpt, ckpt_bytes, ws, ws_bytes,
                      stream) -> int:
    return lib().linattn_fwd_gated(ctypes.byref(shape), q, k, v, log_gate, o, init_state, final_state, ckpt,
                                   ckpt_bytes, ws, ws_bytes, stream)


def linattn_bwd_gated(shape, q, k, v, dO, log_gate, init_state, d_final, ckpt, ckpt_bytes, dq, dk, dv, d_log_gate,
                      d_init, ws, ws_bytes, stream) -> int:
    return lib().linattn_bwd_gated(ctypes.byref(shape), q, k, v, dO, log_gate, init_state, d_final, ckpt,
                                   ckpt_bytes, dq, dk, dv, d_log_gate, d_init, ws, ws_bytes, stream)


def linattn_fwd_gated_vec(shape, q, k, v, log_gate, o, init_state, final_state, ws, ws_bytes, stream) -> int:
    return lib().linattn_fwd_gated_vec(ctypes.byref(shape), q, k, v, log_gate, o, init_state, final_state, ws,
                                       ws_bytes, stream)


def linattn_bwd_gated_vec(shape, q, k, v, dO, log_gate, init_state, d_final, dq, dk, dv, d_log_gate, d_init, ws,
                          ws_bytes, stream) -> int:
    return lib().linattn_bwd_gated_vec(ctypes.byref(shape), q, k, v, dO, log_gate, init_state, d_final, dq, dk, dv,
                                       d_log_gate, d_init, ws, ws_bytes, stream)


def linattn_fwd_gated_vec_ckpt(shape, q, k, v, log_gate, o, init_state, final_state, ckpt, ckpt_bytes, ws, ws_bytes,
                               stream) -> int:
    return lib().linattn_fwd_gated_vec_ckpt(ctypes.byref(shape), q, k, v, log_gate, o, init_state, final_state, ckpt,
                                            ckpt_bytes, ws, ws_bytes, stream)


def linattn_bwd_gated_vec_ckpt(shape, q, k, v, dO, log_gate, init_state, d_final, ckpt, ckpt_bytes, dq, dk, dv,
                               d_log_gate, d_init, ws, ws_bytes, stream) -> int:
    return lib().linattn_bwd_gated_vec_ckpt(ctypes.byref(shape), q, k, v, dO, log_gate, init_state, d_final, ckpt,
                                            ckpt_bytes, dq, dk, dv, d_log_gate, d_init, ws, ws_bytes, stream)


def linattn_chunk_states_rev(shape, seg_len, q, dO, out, ws, ws_bytes, stream) -> int:
    return lib().linattn_chunk_states_rev(ctypes.byref(shape), seg_len, q, dO, out, ws, ws_bytes, stream)


def linattn_state_scan_workspace_size(G, BH, dk, dv) -> tuple[int, int]:
    n = _sz(0)
    st = lib().linattn_state_scan_workspace_size(G, BH, dk, dv, ctypes.byref(n))
    return st, n.value


def linattn_state_scan(G, BH, dk, dv, seg_decay, local, init, out, total, ws, ws_bytes, stream) -> int:
    return lib().linattn_state_scan(G, BH, dk, dv, seg_decay, local, init, out, total, ws, ws_bytes, stream)


def linattn_state_scan_noalloc(G, BH, dk, dv, seg_decay, local, init, out, total, device_status, stream) -> int:
    """Allocation-free scan: no workspace; the library's fixed device scratch is used instead."""
    return lib().linattn_state_scan_noalloc(G, BH, dk, dv, seg_decay, local, init, out, total, device_status,
                                            stream)


def linattn_device_status(ws, stream) -> int:
    return lib().linattn_device_status(ws, stream)


def linattn_softmax_segment_fwd(q_shape, kv_shape, q, k, v, o, lse, softmax_scale, ws, ws_bytes, stream) -> int:
    return lib().linattn_softmax_segment_fwd(ctypes.byref(q_shape), ctypes.byref(kv_shape), q, k, v, o, lse,
                                             softmax_scale, ws, ws_bytes, stream)


def linattn_softmax_segment_bwd(q_shape, kv_shape, q, k, v, o, dO, lse, dq, dk, dv, softmax_scale, ws, ws_bytes,
                                stream) -> int:
    return lib().linattn_softmax_segment_bwd(ctypes.byref(q_shape), ctypes.byref(kv_shape), q, k, v, o, dO, lse, dq,
                                             dk, dv, softmax_scale, ws, ws_bytes, stream)


def linattn_segment_decay(decay, B, H, seg_len, out, stream) -> int:
    return lib().linattn_segment_decay(decay, B, H, seg_len, out, stream)


def linattn_diag_scan_withhold(G, BH, dk, dv, local, out, withhold_tile, wait_limit_ms, ws, ws_bytes,
                               stream) -> int:
    return lib().linattn_diag_scan_withhold(G, BH, dk, dv, local, out, withhold_tile, wait_limit_ms, ws,
                                            ws_bytes, stream)


def linattn_diag_mma(mode, A, B, D, stream) -> int:
    return lib().linattn_diag_mma(mode, A, B, D, stream)


def linattn_timing_enable(on: bool) -> int:
    return lib().linattn_timing_enable(1 if on else 0)


def linattn_timing_collect() -> dict:
    """{kernel name: (launches, total ms)} of the launches recorded since the last collect."""
    n = (_i32 * KERNEL_KINDS)()
    ms = (ctypes.c_float * KERNEL_KINDS)()
    st = lib().linattn_timing_collect(KERNEL_KINDS, n, ms)
    if st < 0:
        raise LinattnError(st, "linattn_timing_collect")
    return {linattn_kernel_name(k): (n[k], ms[k]) for k in range(KERNEL_KINDS) if n[k]}


def linattn_kernel_name(kind: int) -> str:
    return lib().linattn_kernel_name(kind).decode()


# ------------------------------------------------------------------ torch helpers
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(dev, stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return s.cuda_stream


def shape_of(q, decay=None, chunk: int = 64) -> Shape:
    """linattn_shape for a [B, H, T, d] tensor (last dim contiguous)."""
    import torch
    if q.dim() != 4 or q.stride(-1) != 1:
        raise ValueError("sequence tensors must be [B, H, T, d] with a contiguous last dimension")
    B, H, T, d = q.shape
    dt = {torch.bfloat16: BF16, torch.float32: F32}.get(q.dtype)
    if dt is None:
        raise ValueError(f"unsupported dtype {q.dtype}")
    s = Shape()
    s.abi_version, s.B, s.H, s.T, s.dk, s.dv, s.chunk, s.dtype = ABI_VERSION, B, H, T, d, d, chunk, dt
    s.stride_b, s.stride_h, s.stride_t = q.stride(0), q.stride(1), q.stride(2)
    s.decay = _ptr(decay)
    return s


def _same_layout(ref, *ts):
    for t in ts:
        if t is not None and (t.shape != ref.shape or t.stride() != ref.stride() or t.dtype != ref.dtype
                              or t.device != ref.device):
            raise ValueError("q, k, v (and dO, outputs) must share shape, strides, dtype and device")


def _check(st, what):
    if st != OK:
        raise LinattnError(st, what)


def workspace(q, op: int, decay=None, seg_len: int = 0):
    import torch
    st, n = linattn_workspace_size(shape_of(q, decay), op, seg_len)
    _check(st, "linattn_workspace_size")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def checkpoint(q, decay=None):
    """Buffer for the forward group states kept by fwd(..., ckpt=...) for bwd(..., ckpt=...)."""
    import torch
    st, n = linattn_workspace_size(shape_of(q, decay), OP_CHECKPOINT)
    _check(st, "linattn_workspace_size")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def fwd(q, k, v, decay=None, init_state=None, want_final=False, want_chunk_states=False,
        out=None, ws=None, stream=None, ckpt=None):
    """o (, final_state) (, chunk_states) for q, k, v [B, H, T, d] (bf16 or fp32).

    With ``ckpt`` (from ``checkpoint``) the forward group states are also stored for ``bwd(..., ckpt=)``."""
    import torch
    _same_layout(q, k, v, out)
    B, H, T, d = q.shape
    o = out if out is not None else torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    fin = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device) if want_final else None
    nch = (T + 63) // 64
    cs = torch.empty((B, H, nch, d, d), dtype=torch.float32, device=q.device) if want_chunk_states else None
    shape = shape_of(q, decay)
    if ws is None:
        ws = workspace(q, OP_FWD, decay)
    if ckpt is not None:
        if cs is not None:
            raise ValueError("per-chunk states are not offered together with a checkpoint")
        st = linattn_fwd_ckpt(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(init_state), _ptr(fin),
                              _ptr(ckpt), ckpt.numel(), _ptr(ws), ws.numel(), _stream(q.device, stream))
        _check(st, "linattn_fwd_ckpt")
        return o, fin, cs
    st = linattn_fwd(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(init_state), _ptr(fin), _ptr(cs),
                     _ptr(ws), ws.numel(), _stream(q.device, stream))
    _check(st, "linattn_fwd")
    return o, fin, cs


def bwd(q, k, v, dO, decay=None, init_state=None, want_dinit=False, outs=None, ws=None, stream=None, ckpt=None,
        d_final=None):
    """(dq, dk, dv, d_init or None) for the upstream gradient dO (forward states from ``ckpt`` if given).

    ``d_final`` [B, H, d, d] fp32: gradient arriving at the final state (None: zero)."""
    import torch
    _same_layout(q, k, v, dO)
    B, H, T, d = q.shape
    if outs is None:
        outs = [torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device) for _ in range(3)]
    dq, dk, dv = outs
    dinit = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device) if want_dinit else None
    shape = shape_of(q, decay)
    if ws is None:
        ws = workspace(q, OP_BWD, decay)
    if ckpt is not None:
        st = linattn_bwd_ckpt(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(init_state), _ptr(d_final),
                              _ptr(ckpt), ckpt.numel(),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dinit), _ptr(ws), ws.numel(),
                              _stream(q.device, stream))
        _check(st, "linattn_bwd_ckpt")
        return dq, dk, dv, dinit
    st = linattn_bwd(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(init_state), _ptr(d_final), _ptr(dq), _ptr(dk),
                     _ptr(dv), _ptr(dinit), _ptr(ws), ws.numel(), _stream(q.device, stream))
    _check(st, "linattn_bwd")
    return dq, dk, dv, dinit


def decode(q, k, v, state, decay=None, out=None, stream=None):
    """o for T new tokens [B, H, T, d]; `state` [B, H, d, d] fp32 is updated in place."""
    import torch
    _same_layout(q, k, v, out)
    if state.dtype != torch.float32 or not state.is_contiguous():
        raise ValueError("state must be contiguous fp32 [B, H, d, d]")
    o = out if out is not None else torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    st = linattn_decode(shape_of(q, decay), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(state),
                        _stream(q.device, stream))
    _check(st, "linattn_decode")
    return o


def chunk_states(k, v, seg_len: int, decay=None, out=None, ws=None, stream=None):
    """Segment-local states [G, B, H, d, d] (fp32) for G = T / seg_len segments."""
    import torch
    _same_layout(k, v)
    B, H, T, d = k.shape
    G = T // seg_len if seg_len > 0 else 0
    out = out if out is not None else torch.empty((G, B, H, d, d), dtype=torch.float32, device=k.device)
    if ws is None:
        ws = workspace(k, OP_CHUNK_STATES, decay, seg_len)
    st = linattn_chunk_states(shape_of(k, decay), seg_len, _ptr(k), _ptr(v), _ptr(out), _ptr(ws), ws.numel(),
                              _stream(k.device, stream))
    _check(st, "linattn_chunk_states")
    return out


def chunk_states_rev(q, dO, seg_len: int, decay=None, out=None, ws=None, stream=None):
    """Segment-local gradient states [G, B, H, d, d] (fp32): sum_s lambda^{s - start + 1} q_s dO_s^T."""
    import torch
    _same_layout(q, dO)
    B, H, T, d = q.shape
    G = T // seg_len if seg_len > 0 else 0
    out = out if out is not None else torch.empty((G, B, H, d, d), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(q, OP_CHUNK_STATES, decay, seg_len)
    st = linattn_chunk_states_rev(shape_of(q, decay), seg_len, _ptr(q), _ptr(dO), _ptr(out), _ptr(ws), ws.numel(),
                                  _stream(q.device, stream))
    _check(st, "linattn_chunk_states_rev")
    return out


def checkpoint_gated(q):
    """Checkpoint buffer of fwd_gated for bwd_gated (group states and the final state)."""
    import torch
    st, n = linattn_workspace_size(shape_of(q, None), OP_CHECKPOINT_GATED)
    _check(st, "linattn_workspace_size")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def _gate_tensor(log_gate, q):
    import torch
    B, H, T, _ = q.shape
    if log_gate.dtype != torch.float32 or not log_gate.is_contiguous() or tuple(log_gate.shape) != (B, H, T):
        raise ValueError("log_gate must be contiguous fp32 [B, H, T]")
    return log_gate


def fwd_gated(q, k, v, log_gate, ckpt, init_state=None, want_final=False, out=None, ws=None, stream=None):
    """(o, final_state or None) with a gate per token: S_t = exp(log_gate_t) S_{t-1} + k_t v_t^T.
    ``ckpt`` (from checkpoint_gated) receives what bwd_gated needs."""
    import torch
    _same_layout(q, k, v, out)
    _gate_tensor(log_gate, q)
    B, H, T, d = q.shape
    o = out if out is not None else torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    fin = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device) if want_final else None
    shape = shape_of(q, None)
    if ws is None:
        ws = workspace(q, OP_FWD_GATED)
    st = linattn_fwd_gated(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(log_gate), _ptr(o), _ptr(init_state), _ptr(fin),
                           _ptr(ckpt), ckpt.numel(), _ptr(ws), ws.numel(), _stream(q.device, stream))
    _check(st, "linattn_fwd_gated")
    return o, fin


def bwd_gated(q, k, v, dO, log_gate, ckpt, init_state=None, d_final=None, want_dinit=False, outs=None, ws=None,
              stream=None, dlg_out=None):
    """(dq, dk, dv, d_log_gate, d_init or None) of fwd_gated for the upstream gradient dO."""
    import torch
    _same_layout(q, k, v, dO)
    _gate_tensor(log_gate, q)
    B, H, T, d = q.shape
    if outs is None:
        outs = [torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device) for _ in range(3)]
    dq, dk, dv = outs
    dlg = dlg_out if dlg_out is not None else torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    dinit = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device) if want_dinit else None
    shape = shape_of(q, None)
    if ws is None:
        ws = workspace(q, OP_BWD_GATED)
    st = linattn_bwd_gated(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(log_gate), _ptr(init_state),
                           _ptr(d_final), _ptr(ckpt), ckpt.numel(), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dlg),
                           _ptr(dinit), _ptr(ws), ws.numel(), _stream(q.device, stream))
    _check(st, "linattn_bwd_gated")
    return dq, dk, dv, dlg, dinit


def _gate_tensor_vec(log_gate, q):
    import torch
    B, H, T, d = q.shape
    if log_gate.dtype != torch.float32 or not log_gate.is_contiguous() or tuple(log_gate.shape) != (B, H, T, d):
        raise ValueError("log_gate must be contiguous fp32 [B, H, T, d]")
    return log_gate


def checkpoint_gated_vec(q):
    """Checkpoint buffer of fwd_gated_vec(..., ckpt=) for bwd_gated_vec(..., ckpt=) (the chunk
    groups' entering states and log-gate sums)."""
    import torch
    st, n = linattn_workspace_size(shape_of(q, None), OP_CHECKPOINT_GATED_VEC)
    _check(st, "linattn_workspace_size")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def fwd_gated_vec(q, k, v, log_gate, init_state=None, want_final=False, out=None, ws=None, stream=None, ckpt=None):
    """(o, final_state or None) with a gate per token and key dimension:
    S_t = diag(exp(log_gate_t)) S_{t-1} + k_t v_t^T (log_gate [B, H, T, d] fp32).  With ``ckpt``
    (from checkpoint_gated_vec) the groups' states are also kept for bwd_gated_vec(..., ckpt=)."""
    import torch
    _same_layout(q, k, v, out)
    _gate_tensor_vec(log_gate, q)
    B, H, T, d = q.shape
    o = out if out is not None else torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    fin = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device) if want_final else None
    if ws is None:
        ws = workspace(q, OP_FWD_GATED_VEC)
    if ckpt is not None:
        st = linattn_fwd_gated_vec_ckpt(shape_of(q, None), _ptr(q), _ptr(k), _ptr(v), _ptr(log_gate), _ptr(o),
                                        _ptr(init_state), _ptr(fin), _ptr(ckpt), ckpt.numel(), _ptr(ws), ws.numel(),
                                        _stream(q.device, stream))
        _check(st, "linattn_fwd_gated_vec_ckpt")
        return o, fin
    st = linattn_fwd_gated_vec(shape_of(q, None), _ptr(q), _ptr(k), _ptr(v), _ptr(log_gate), _ptr(o),
                               _ptr(init_state), _ptr(fin), _ptr(ws), ws.numel(), _stream(q.device, stream))
    _check(st, "linattn_fwd_gated_vec")
    return o, fin


def bwd_gated_vec(q, k, v, dO, log_gate, init_state=None, d_final=None, want_dinit=False, outs=None, ws=None,
                  stream=None, ckpt=None):
    """(dq, dk, dv, d_log_gate [B, H, T, d], d_init or None) of fwd_gated_vec for the upstream gradient dO
    (the forward's group states from ``ckpt`` if given)."""
    import torch
    _same_layout(q, k, v, dO)
    _gate_tensor_vec(log_gate, q)
    B, H, T, d = q.shape
    if outs is None:
        outs = [torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device) for _ in range(3)]
    dq, dk, dv = outs
    dlg = torch.empty((B, H, T, d), dtype=torch.float32, device=q.device)
    dinit = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device) if want_dinit else None
    if ws is None:
        ws = workspace(q, OP_BWD_GATED_VEC)
    if ckpt is not None:
        st = linattn_bwd_gated_vec_ckpt(shape_of(q, None), _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(log_gate),
                                        _ptr(init_state), _ptr(d_final), _ptr(ckpt), ckpt.numel(), _ptr(dq), _ptr(dk),
                                        _ptr(dv), _ptr(dlg), _ptr(dinit), _ptr(ws), ws.numel(),
                                        _stream(q.device, stream))
        _check(st, "linattn_bwd_gated_vec_ckpt")
        return dq, dk, dv, dlg, dinit
    st = linattn_bwd_gated_vec(shape_of(q, None), _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(log_gate),
                               _ptr(init_state), _ptr(d_final), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dlg), _ptr(dinit),
                               _ptr(ws), ws.numel(), _stream(q.device, stream))
    _check(st, "linattn_bwd_gated_vec")
    return dq, dk, dv, dlg, dinit


def state_scan(local, seg_decay=None, init=None, want_total=False, out=None, ws=None, stream=None):
    """Exclusive scan over the leading axis of local [G, *BH, dk, dv] (fp32)."""
    import torch
    G, dk, dv = local.shape[0], local.shape[-2], local.shape[-1]
    BH = local[0].numel() // (dk * dv)
    if not local.is_contiguous() or local.dtype != torch.float32:
        raise ValueError("local states must be contiguous fp32")
    out = out if out is not None else torch.empty_like(local)
    total = torch.empty(local.shape[1:], dtype=torch.float32, device=local.device) if want_total else None
    if ws is None:
        st, n = linattn_state_scan_workspace_size(G, BH, dk, dv)
        _check(st, "linattn_state_scan_workspace_size")
        ws = torch.empty(n, dtype=torch.uint8, device=local.device)
    st = linattn_state_scan(G, BH, dk, dv, _ptr(seg_decay), _ptr(local), _ptr(init), _ptr(out), _ptr(total),
                            _ptr(ws), ws.numel(), _stream(local.device, stream))
    _check(st, "linattn_state_scan")
    return out, total


def segment_decay(decay, B: int, seg_len: int, out=None, stream=None):
    """Per-(b, h) scan multiplier decay[h]^seg_len, [B*H] fp32 (None for decay None)."""
    import torch
    if decay is None:
        return None
    H = decay.numel()
    out = out if out is not None else torch.empty(B * H, dtype=torch.float32, device=decay.device)
    st = linattn_segment_decay(_ptr(decay), B, H, seg_len, _ptr(out), _stream(decay.device, stream))
    _check(st, "linattn_segment_decay")
    return out


def softmax_segment_fwd(q, k, v, scale: float = 0.0, want_lse: bool = False, out=None, ws=None, stream=None):
    """(o, lse or None): causal softmax attention of q [B,H,Tq,128] (the last Tq positions)
    over the prefix k, v [B,H,Tk,128] (bf16; scale 0 means 1/sqrt(128))."""
    import torch
    _same_layout(q, out)
    _same_layout(k, v)
    B, H, Tq, d = q.shape
    o = out if out is not None else torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device) if want_lse else None
    if ws is None:
        ws = workspace(q, OP_SOFTMAX_SEGMENT)
    st = linattn_softmax_segment_fwd(shape_of(q), shape_of(k), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), scale,
                                     _ptr(ws), ws.numel(), _stream(q.device, stream))
    _check(st, "linattn_softmax_segment_fwd")
    return o, lse


def softmax_segment_bwd(q, k, v, o, dO, lse, scale: float = 0.0, outs=None, ws=None, stream=None):
    """(dq, dk, dv): gradients of the causal softmax attention segment for the output
    gradient dO, from the forward's o and lse (bf16 q, o, dO, dq with q's layout; k, v,
    dk, dv with k's layout; scale 0 means 1/sqrt(128))."""
    import torch
    _same_layout(q, o)
    _same_layout(q, dO)
    _same_layout(k, v)
    if outs is None:
        outs = (torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device),
                torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device),
                torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, device=v.device))
    dq, dk, dv = outs
    _same_layout(q, dq)
    _same_layout(k, dk)
    _same_layout(k, dv)
    if ws is None:
        ws = workspace(q, OP_SOFTMAX_SEGMENT_BWD)
    st = linattn_softmax_segment_bwd(shape_of(q), shape_of(k), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO),
                                     _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), scale, _ptr(ws), ws.numel(),
                                     _stream(q.device, stream))
    _check(st, "linattn_softmax_segment_bwd")
    return dq, dk, dv


def device_status(ws, stream=None) -> int:
    return linattn_device_status(_ptr(ws), _stream(ws.device, stream))
