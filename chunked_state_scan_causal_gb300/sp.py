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

The standard-attention layers of the hybrid model (LASP-2H on the same page)
split the same way with one gather of keys and values instead of states
(``softmax_forward`` / ``softmax_backward``): every rank gathers the k, v of all
segments, its queries attend causally over segments 0..rank
(linattn_softmax_segment_fwd), and in the backward the gradients of the
gathered k, v go back to their owners, summed over the ranks that used them,
by one reduce-scatter (linattn_softmax_segment_bwd for the local gradients).

The arithmetic runs in this package's kernels; this module only moves the
states (and, for the softmax layers, keys, values and their gradients)
between ranks.  The exchange is pluggable: ``TorchDistExchange`` uses a
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

    def reduce_scatter(self, parts):
        """The sum over ranks of parts[this rank], for parts [world, ...] on every rank
        (NCCL's reduce-scatter; other backends reduce the whole stack and keep the row)."""
        import torch
        parts = parts.contiguous()
        try:
            if self.dist.get_backend(self.group) == "nccl":
                out = torch.empty_like(parts[0])
                work = self.dist.reduce_scatter_tensor(out, parts, group=self.group, async_op=True)
            else:
                out = parts.clone()
                work = self.dist.all_reduce(out, group=self.group, async_op=True)
            ok = work.wait(timeout=datetime.timedelta(seconds=self.timeout))
        except Exception as e:  # peer gone, connection reset, backend timeout
            raise SequenceParallelError(f"rank {self.rank}: gradient exchange failed: {e}") from e
        if ok is False:
            raise SequenceParallelError(f"rank {self.rank}: gradient exchange timed out after {self.timeout} s")
        return out if out.dim() == parts.dim() - 1 else out[self.rank]


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

    def reduce_scatter(self, parts):
        """The sum over ranks of parts[this rank] (in rank order)."""
        self.group.slots[self.rank] = parts
        self._wait()
        rows = list(self.group.slots)
        out = rows[0][self.rank].clone()
        for x in rows[1:]:
            out += x[self.rank]
        self._wait()
        return out


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

    def softmax_fwd(self, q, k, v, scale):
        return self.la.softmax_segment_fwd(q, k, v, scale=scale, want_lse=True)

    def softmax_bwd(self, q, k, v, o, dO, lse, scale):
        return self.la.softmax_segment_bwd(q, k, v, o, dO, lse, scale=scale)


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


# ----------------------------------------------------------------------------- softmax layers (LASP-2H)
@dataclass
class SoftmaxContext:
    """What a rank keeps from a softmax layer's forward for its backward."""
    k_prefix: object   # [B, H, (rank + 1) L, d]: the gathered keys of segments 0..rank
    v_prefix: object
    o: object          # this rank's outputs
    lse: object        # [B, H, L] fp32 log-sum-exp of this rank's rows
    scale: float


def softmax_forward(q, k, v, exchange, scale=0.0, ops=None):
    """This rank's outputs of causal softmax attention and a SoftmaxContext.

    One gather hands every rank the keys and values of all segments; the rank's
    queries, the last L positions of the prefix that ends with its own segment,
    attend over segments 0..rank.  ``scale`` 0 means 1/sqrt(d)."""
    import torch
    ops = ops or KernelOps()
    _check_segment(q, exchange.world)
    allK = exchange.all_gather(k.contiguous())                    # [N, B, H, L, d]
    allV = exchange.all_gather(v.contiguous())
    r = exchange.rank
    kp = torch.cat(list(allK[:r + 1]), dim=2)                     # [B, H, (r + 1) L, d]
    vp = torch.cat(list(allV[:r + 1]), dim=2)
    o, lse = ops.softmax_fwd(q, kp, vp, scale)
    return o, SoftmaxContext(kp, vp, o, lse, scale)


def softmax_backward(q, dO, ctx: SoftmaxContext, exchange, ops=None):
    """This rank's (dq, dk, dv).  The gradients of the gathered keys and values are
    returned to their owners, summed over the ranks whose queries saw them (one
    reduce-scatter)."""
    import torch
    ops = ops or KernelOps()
    dq, dkp, dvp = ops.softmax_bwd(q, ctx.k_prefix, ctx.v_prefix, ctx.o, dO, ctx.lse, ctx.scale)
    N, r = exchange.world, exchange.rank
    B, H, L, d = q.shape

    def spread(x):
        # this rank's contribution to every segment's gradient: [N, B, H, L, d], zero past
        # rank r, summed in fp32 (or the inputs' own type when that is wider)
        acc = torch.float64 if x.dtype == torch.float64 else torch.float32
        out = torch.zeros((N, B, H, L, x.shape[3]), dtype=acc, device=x.device)
        out[:r + 1] = x.to(acc).reshape(B, H, r + 1, L, x.shape[3]).permute(2, 0, 1, 3, 4)
        return out

    dk = exchange.reduce_scatter(spread(dkp)).to(q.dtype)
    dv = exchange.reduce_scatter(spread(dvp)).to(q.dtype)
    return dq, dk, dv
