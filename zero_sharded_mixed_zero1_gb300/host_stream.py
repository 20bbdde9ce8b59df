"""The fused step fed from gradients in pinned host memory, with explicit
copies overlapping the computation.

The range is cut into chunks.  Each chunk's M gradient slices are copied to
a device staging slot on a copy stream (one cudaMemcpyAsync per slice) while
the step runs on the previous chunk (zero1_step_bucket, the fused step on an
element range); two slots alternate.  The updated bf16 parameters can be
copied back to a pinned host buffer chunk by chunk.  The step is
element-wise, so the result is bit for bit that of one fused step.  The
streams and events are PyTorch's; every step of the arithmetic runs in the
library's kernels.
"""
from __future__ import annotations

import torch

from . import _lib


class HostStreamedStep:
    """The fused step over shards [shard_begin, shard_end) with the M
    replicas' gradients in pinned host memory (each host_grads[r] holds the
    range's nv real elements), fp32 state and bf16 parameters on the device.

    chunk_elems sets the copy granularity (rounded up to a multiple of 8);
    the staging memory is 2 x M x chunk_elems bf16 on the device.  If
    params_host (pinned, nv elements) is given, the updated parameters are
    copied back into it.  Launches go to `stream` (default: the current
    stream at construction); the copies go to a second stream."""

    def __init__(self, plan: _lib.Plan, shard_begin: int, shard_end: int, host_grads, master, m, v, params,
                 chunk_elems: int = 1 << 24, params_host=None, overflow_flag=None, stream=None):
        _lib._replicas(plan, host_grads, "host_grads")
        base, L, nv = _lib._range(plan, shard_begin, shard_end)
        if L == 0:
            raise ValueError("empty or invalid shard range")
        for i, g in enumerate(host_grads):
            if g.device.type != "cpu" or not g.is_pinned() or g.dtype != torch.bfloat16 or g.numel() < nv:
                raise ValueError(f"host_grads[{i}] must be a pinned bf16 host tensor of at least {nv} elements")
        if params_host is not None and (not params_host.is_pinned() or params_host.numel() < nv):
            raise ValueError("params_host must be a pinned host tensor of at least nv elements")
        self.plan, self.base, self.L, self.nv = plan, base, L, nv
        self.host_grads, self.master, self.m, self.v, self.params = host_grads, master, m, v, params
        self.params_host, self.flag = params_host, overflow_flag
        dev = master.device
        self.chunk = max(8, (int(chunk_elems) + 7) // 8 * 8)
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        self.copy_stream = torch.cuda.Stream(device=dev)
        size = min(self.chunk, max(nv, 8))
        self.slots = [[torch.empty(size, dtype=torch.bfloat16, device=dev) for _ in range(plan.M)]
                      for _ in range(2)]
        self.copied = [torch.cuda.Event() for _ in range(2)]
        self.consumed = [torch.cuda.Event() for _ in range(2)]
        cuts = list(range(0, L, self.chunk)) + [L]
        self.pieces = list(zip(cuts[:-1], cuts[1:]))

    def __call__(self, hp: _lib.AdamW) -> None:
        st, cs = self.stream, self.copy_stream
        cs.wait_stream(st)                      # state from earlier work is ready
        for k, (e0, e1) in enumerate(self.pieces):
            slot = k % 2
            real = max(0, min(self.nv, e1) - e0)
            if k >= 2:
                cs.wait_event(self.consumed[slot])
            with torch.cuda.stream(cs):
                for r in range(self.plan.M):
                    if real:
                        self.slots[slot][r][:real].copy_(self.host_grads[r][e0:e0 + real], non_blocking=True)
                self.copied[slot].record(cs)
            st.wait_event(self.copied[slot])
            grads = [s[:max(real, 1)] for s in self.slots[slot]]
            params = self.params[e0:] if e0 < self.nv else self.params[:0]
            _lib.zero1_step_bucket(self.plan, self.base + e0, self.base + e1, grads, self.master[e0:],
                                   self.m[e0:], self.v[e0:], params, hp, self.flag, stream=st)
            self.consumed[slot].record(st)
            if self.params_host is not None and real:
                with torch.cuda.stream(st):
                    self.params_host[e0:e0 + real].copy_(self.params[e0:e0 + real], non_blocking=True)
