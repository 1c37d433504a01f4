"""Sequence parallelism across ranks: every rank holds one contiguous segment of
each sequence, and the only exchange is one gather of fixed-size fp32 states.

Forward (the All-Scan of the ZeCO page; the gather-then-combine of
length-independent states of the LASP-2 page):
  1. each rank sums its segment into a local state
         U_r = sum_{s in segment r} lambda^{end_r - s} k_s v_s^T      (linattn_chunk_states)
  2. the ranks gather all U_r (B*H*d*d fp32 each, independent of the length)
  3. each rank runs the exclusive scan S_r = a S_{r-1} + U_{r-1}, a = lambda^{T_seg},
     S_0 = the initial state                                          (linattn_state_scan)
     and keeps its own entering state S_r (the scan total is the final state)
  4. each rank runs its chunked forward from S_r                      (linattn_fwd_ckpt)
Backward (the same exchange run in reverse):
  1. each rank sums its segment into a local gradient state
         W_r = sum_{s in segment r} lambda^{s - start_r + 1} q_s dO_s^T (linattn_chunk_states_rev)
  2. the ranks gather all W_r (in reverse rank order)
  3. each rank runs the reverse exclusive scan D_r = sum_{r' > r} a^{r'-r-1} W_r'
     (+ a^{N-1-r} d_final), the gradient arriving at its final state; the scan
     total is the gradient of the initial state               (linattn_state_scan)
  4. each rank runs its backward with d_final_state = D_r     (linattn_bwd_ckpt)

The arithmetic runs in this package's kernels; this module only moves the
states between ranks.  The exchange is pluggable: ``TorchDistExchange`` uses a
torch.distributed process group (NCCL between GPUs, gloo between CPU
processes); ``ThreadExchange`` connects ranks that are threads of one process.
Every wait is bounded: an exchange that does not complete in ``timeout``
seconds (a rank that died, hung or never joined) raises
``SequenceParallelError`` on the ranks that are waiting, instead of hanging.

All ranks must hold segments of the same length and the same B, H, d.
"""
from __future__ import annotations

import datetime
import threading
from dataclasses import dataclass


class SequenceParallelError(RuntimeError):
    """An exchange between ranks failed or timed out."""


# ----------------------------------------------------------------------------- exchanges
class TorchDistExchange:
    """All-gather over a torch.distributed process group with a bounded wait."""

    def __init__(self, group=None, timeout: float = 60.0):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.timeout = timeout

    def all_gather(self, local, reverse: bool = False):
        """[world, *local.shape]; row i is rank i's tensor (rank world-1-i's when reverse)."""
        import torch
        out = torch.empty((self.world, *local.shape), dtype=local.dtype, device=local.device)
        views = [out[self.world - 1 - i] if reverse else out[i] for i in range(self.world)]
        try:
            work = self.dist.all_gather(views, local.contiguous(), group=self.group, async_op=True)
            ok = work.wait(timeout=datetime.timedelta(seconds=self.timeout))
        except Exception as e:  # peer gone, connection reset, backend timeout
            raise SequenceParallelError(f"rank {self.rank}: state exchange failed: {e}") from e
        if ok is False:
            raise SequenceParallelError(f"rank {self.rank}: state exchange timed out after {self.timeout} s")
        return out


class ThreadExchange:
    """Ranks that are threads of one process (a rendezvous per exchange).

    Build one ``ThreadExchange.Group(world)`` and give every thread
    ``group.rank(r)``.  A thread that does not arrive within ``timeout`` breaks
    the rendezvous and every waiting thread raises ``SequenceParallelError``.
    """

    class Group:
        def __init__(self, world: int, timeout: float = 60.0):
            self.world, self.timeout = world, timeout
            self.slots = [None] * world
            self.barrier = threading.Barrier(world)

        def rank(self, r: int) -> "ThreadExchange":
            return ThreadExchange(self, r)

    def __init__(self, group: "ThreadExchange.Group", rank: int):
        self.group, self.rank, self.world = group, rank, group.world
        self.timeout = group.timeout

    def _wait(self):
        try:
            self.group.barrier.wait(timeout=self.timeout)
        except threading.BrokenBarrierError as e:
            raise SequenceParallelError(f"rank {self.rank}: a peer did not reach the exchange") from e

    def abort(self):
        """Break the rendezvous (a rank that fails calls this so its peers stop waiting)."""
        self.group.barrier.abort()

    def all_gather(self, local, reverse: bool = False):
        import torch
        self.group.slots[self.rank] = local
        self._wait()
        rows = list(self.group.slots)
        self._wait()  # every rank has read the slots before they are reused
        return torch.stack(rows[::-1] if reverse else rows)


# ----------------------------------------------------------------------------- local operations
class KernelOps:
    """The per-rank steps, on this package's CUDA kernels (the product path)."""

    def __init__(self):
        import chunked_state_scan_causal_gb300 as la
        self.la = la

    def chunk_states(self, k, v, seg_len, decay):
        return self.la.chunk_states(k, v, seg_len, decay=decay)

    def chunk_states_rev(self, q, dO, seg_len, decay):
        return self.la.chunk_states_rev(q, dO, seg_len, decay=decay)

    def state_scan(self, local, seg_decay, init):
        return self.la.state_scan(local, seg_decay=seg_decay, init=init, want_total=True)

    def checkpoint(self, q, decay):
        return self.la.checkpoint(q, decay)

    def fwd(self, q, k, v, decay, init_state, ckpt):
        o, _, _ = self.la.fwd(q, k, v, decay=decay, init_state=init_state, ckpt=ckpt)
        return o

    def bwd(self, q, k, v, dO, decay, init_state, ckpt, d_final):
        dq, dk, dv, _ = self.la.bwd(q, k, v, dO, decay=decay, init_state=init_state, ckpt=ckpt, d_final=d_final)
        return dq, dk, dv

    def seg_decay(self, decay, B, seg_len):
        """Per-(b, h) multiplier lambda_h^seg_len for the scan, [B*H] fp32 (None for lambda = 1)."""
        return self.la.segment_decay(decay, B, seg_len)


@dataclass
class Context:
    """What a rank keeps from its forward for its backward."""
    init_state: object      # the state entering this rank's segment, [B, H, d, d] fp32
    checkpoint: object      # the forward's group states (or None)
    seg_len: int


def _check_segment(q, world):
    if q.dim() != 4:
        raise ValueError("segments are [B, H, T_segment, d]")
    if q.shape[2] < 1:
        raise ValueError("every rank needs at least one token")


def forward(q, k, v, exchange, decay=None, init_state=None, ops=None):
    """This rank's outputs for its segment, the whole sequence's final state, and a Context.

    ``init_state`` is the state before the first token of the whole sequence (the
    same tensor on every rank, or None)."""
    ops = ops or KernelOps()
    _check_segment(q, exchange.world)
    B, H, L, d = q.shape
    U = ops.chunk_states(k, v, L, decay)                         # [1, B, H, d, d]
    allU = exchange.all_gather(U[0])                              # [N, B, H, d, d]
    S, total = ops.state_scan(allU, ops.seg_decay(decay, B, L), init_state)
    s_in = S[exchange.rank].contiguous()
    ckpt = ops.checkpoint(q, decay)
    o = ops.fwd(q, k, v, decay, s_in, ckpt)
    return o, total, Context(s_in, ckpt, L)


def backward(q, k, v, dO, ctx: Context, exchange, decay=None, d_final=None, ops=None):
    """This rank's (dq, dk, dv) and the whole sequence's gradient of the initial state.

    ``d_final`` is the gradient arriving at the whole sequence's final state (the
    same tensor on every rank, or None)."""
    ops = ops or KernelOps()
    B, H, L, d = q.shape
    W = ops.chunk_states_rev(q, dO, L, decay)                     # [1, B, H, d, d]
    allW = exchange.all_gather(W[0], reverse=True)                # row i = rank N-1-i
    D, d_init = ops.state_scan(allW, ops.seg_decay(decay, B, L), d_final)
    d_fin = D[exchange.world - 1 - exchange.rank].contiguous()
    dq, dk, dv = ops.bwd(q, k, v, dO, decay, ctx.init_state, ctx.checkpoint, d_fin)
    return dq, dk, dv, d_init
