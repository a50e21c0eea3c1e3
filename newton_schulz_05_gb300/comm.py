"""Data-parallel gradient reduction overlapped with backward, feeding the
Muon step.

Paddle PR "Support Muon sharding optimizer comm overlap" gives the Muon
sharding optimizer a stage-1 overlap: backward hooks hand each parameter's
gradient to a communication buffer as soon as it is accumulated, a buffer
whose gradients are all in starts its reduction while backward goes on, and
the optimizer waits for the reductions before it steps.  Its review adds
three rules, kept here:
  * matrix parameters (the Muon path) and the others (1-D biases and norm
    scales, the AdamW path) go to separate buffers;
  * a parameter whose gradient is not complete when its hook fires (a weight
    shared with another stage, or one the caller names) goes to a buffer
    without hooks, reduced synchronously when backward is over;
  * a loss scaler may unscale and check the gradients only after every
    buffer, the synchronous ones included, has been reduced.

GradReduceOverlap does this with torch.distributed: flat buffers per
(class, dtype) of about `bucket_bytes`, filled in the reverse order of the
parameter list (the order backward produces gradients in), each reduced by
one asynchronous all_reduce when its last gradient arrives.  finish() reduces
the synchronous buckets, waits for every handle, scales to the mean and
returns the reduced gradients as views into the buffers, in parameter order,
ready for MuonWithAdamW.step or muon_step_amp.  The reduction moves bytes
only; every arithmetic step of the optimizer stays in libmuon's kernels.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Sequence

import torch

__all__ = ["GradReduceOverlap"]


class _Bucket:
    def __init__(self, kind: str, dtype: torch.dtype, device, members: List[int],
                 numels: List[int], sync_only: bool):
        self.kind = kind
        self.sync_only = sync_only
        self.members = members                     # parameter indices
        self.offsets = {}
        off = 0
        for i, n in zip(members, numels):
            self.offsets[i] = (off, n)
            off += n
        self.buffer = torch.zeros(off, dtype=dtype, device=device)
        self.pending = set(members)
        self.handle = None
        self.launched_early = False                # started while backward still ran

    def view(self, i: int, shape) -> torch.Tensor:
        off, n = self.offsets[i]
        return self.buffer[off:off + n].view(shape)

    def reset(self):
        self.pending = set(self.members)
        self.handle = None
        self.launched_early = False


class GradReduceOverlap:
    """Backward-overlapped all_reduce of a data-parallel model's gradients.

    params       the model's parameters, in model order (every rank the same)
    group        torch.distributed process group (None: the default group)
    bucket_bytes target bytes of one reduction buffer
    sync_only    parameters whose gradient is complete only after backward
                 (shared across stages, or accumulated outside autograd):
                 reduced synchronously in finish(), never from a hook
    Use: call begin() before each backward of an optimizer step (with
    last_micro_batch=False for the gradient-accumulation micro-batches that
    precede the last one: their hooks only accumulate), run backward, then
    grads = finish()."""

    def __init__(self, params: Sequence[torch.Tensor], group=None, bucket_bytes: int = 25 << 20,
                 sync_only: Iterable[torch.Tensor] = ()):
        import torch.distributed as dist
        self.dist = dist
        self.params = list(params)
        self.group = group
        self.world = dist.get_world_size(group) if dist.is_initialized() else 1
        ids = {id(p) for p in sync_only}
        self.sync_only = [i for i, p in enumerate(self.params) if id(p) in ids]
        self.kind = ["matrix" if p.dim() in (2, 3) else "other" for p in self.params]
        self.buckets: List[_Bucket] = []
        self.where: Dict[int, _Bucket] = {}
        # reverse parameter order: the gradients of the last layers arrive first
        order = list(range(len(self.params)))[::-1]
        for sync in (False, True):
            for kind in ("matrix", "other"):
                by_dtype: Dict[torch.dtype, List[int]] = {}
                for i in order:
                    if self.kind[i] == kind and ((i in self.sync_only) == sync):
                        by_dtype.setdefault(self.params[i].dtype, []).append(i)
                for dt, idx in by_dtype.items():
                    cur, cur_bytes = [], 0
                    for i in idx:
                        nb = self.params[i].numel() * self.params[i].element_size()
                        if cur and cur_bytes + nb > bucket_bytes:
                            self._add_bucket(kind, dt, cur, sync)
                            cur, cur_bytes = [], 0
                        cur.append(i)
                        cur_bytes += nb
                    if cur:
                        self._add_bucket(kind, dt, cur, sync)
        self._hooks = []
        for i, p in enumerate(self.params):
            if i not in self.sync_only and p.requires_grad:
                self._hooks.append(p.register_post_accumulate_grad_hook(self._make_hook(i)))
        self._last = True
        self._in_backward = False
        self._finished = False

    def _add_bucket(self, kind, dtype, members, sync):
        b = _Bucket(kind, dtype, self.params[members[0]].device, members,
                    [self.params[i].numel() for i in members], sync)
        self.buckets.append(b)
        for i in members:
            self.where[i] = b

    def _make_hook(self, i: int):
        def hook(p: torch.Tensor):
            if not self._in_backward:
                raise RuntimeError("GradReduceOverlap: begin() was not called before backward")
            b = self.where[i]
            v = b.view(i, p.shape)
            v.add_(p.grad)          # micro-batches accumulate into the buffer
            p.grad = None
            if not self._last:
                return
            b.pending.discard(i)
            if not b.pending:
                b.launched_early = any(bb.pending for bb in self.buckets if not bb.sync_only)
                b.handle = self.dist.all_reduce(b.buffer, group=self.group, async_op=True) \
                    if self.world > 1 else None
        return hook

    def begin(self, last_micro_batch: bool = True) -> None:
        """Arm the hooks for one backward; the first call of an optimizer
        step also clears the buffers."""
        if self._finished or not self._in_backward:
            for b in self.buckets:
                b.buffer.zero_()
                b.reset()
            self._finished = False
        self._in_backward = True
        self._last = last_micro_batch

    def finish(self) -> List[torch.Tensor]:
        """Reduce the synchronous buckets, wait for every reduction, scale to
        the mean; returns the reduced gradient of every parameter (views
        into the buffers, in parameter order).  Call it before a loss scaler
        unscales or checks the gradients."""
        if not self._in_backward:
            raise RuntimeError("GradReduceOverlap: finish() without begin() and backward")
        for i in self.sync_only:
            p = self.params[i]
            if p.grad is not None:
                self.where[i].view(i, p.shape).add_(p.grad)
                p.grad = None
        for b in self.buckets:
            if b.pending and not b.sync_only:
                raise RuntimeError("GradReduceOverlap: backward produced no gradient for "
                                   "parameters %s" % sorted(b.pending))
            if b.sync_only and self.world > 1:
                self.dist.all_reduce(b.buffer, group=self.group)
        for b in self.buckets:
            if b.handle is not None:
                b.handle.wait()
                b.handle = None
            if self.world > 1:
                b.buffer.div_(self.world)
        self._in_backward = False
        self._finished = True
        return [self.where[i].view(i, p.shape) for i, p in enumerate(self.params)]

    def overlapped_buckets(self) -> int:
        """Buckets of the last step whose reduction started while backward
        still had gradients to produce."""
        return sum(1 for b in self.buckets if b.launched_early)

    def remove(self) -> None:
        for h in self._hooks:
            h.remove()
        self._hooks = []
