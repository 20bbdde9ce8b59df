"""The fused step over buffers in pinned host memory, staged through HBM by
the copy engines while the computation runs.

The range is cut into chunks.  For each chunk, the inputs that live in host
memory (the M gradient slices, the fp32 master/m/v) are copied into a device
staging slot on an inbound copy stream (one cudaMemcpyAsync per slice); the
step runs on the slot (zero1_step_bucket, the fused step on an element
range); the outputs that live in host memory (master/m/v, and the bf16
parameters if a host copy is wanted) are copied back on an outbound copy
stream.  Three slots rotate, so the inbound copy of chunk k + 1, the step on
chunk k and the outbound copy of chunk k - 1 run at the same time: with
optimizer state in host memory both directions of the host link are busy
(the ZeRO-Offload placement of the fp32 state in CPU memory, with the update
itself on the GPU).  The step is element-wise, so the result is bit for bit
that of one fused step on device buffers.  The streams and events are
PyTorch's; every step of the arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import torch

from . import _lib

_SLOTS = 3


def _pinned(t: torch.Tensor) -> bool:
    return t.device.type == "cpu" and t.is_pinned()


class HostStreamedStep:
    """The fused step over shards [shard_begin, shard_end).

    grads: M bf16 tensors holding the range's nv real elements, either all
    pinned host tensors (staged chunk by chunk) or all CUDA tensors (read in
    place).  master/m/v: the range's L fp32 elements, either all pinned host
    tensors (staged in, updated, copied back) or all CUDA tensors (updated in
    place).  params: a CUDA bf16 tensor of nv elements, written by the step;
    if params_host (pinned, nv elements) is given, the updated parameters are
    also copied into it.  At least one of grads, master/m/v and params_host
    must be in host memory, or there is nothing to stream.

    chunk_elems sets the copy granularity (rounded up to a multiple of 8);
    the staging memory is 3 x chunk_elems x (2M bytes if the gradients are
    staged + 12 bytes if the state is).  Launches go to `stream` (default:
    the current stream at construction); the copies go to two more streams.
    When a call returns, work enqueued later on `stream` sees the whole
    step, including the copies back to host memory."""

    def __init__(self, plan: _lib.Plan, shard_begin: int, shard_end: int, grads, master, m, v, params,
                 chunk_elems: int = 1 << 24, params_host=None, overflow_flag=None, stream=None):
        _lib._replicas(plan, grads, "grads")
        base, L, nv = _lib._range(plan, shard_begin, shard_end)
        if L == 0:
            raise ValueError("empty or invalid shard range")
        self.grads_on_host = _pinned(grads[0])
        for i, g in enumerate(grads):
            if g.dtype != torch.bfloat16 or g.numel() < nv or _pinned(g) != self.grads_on_host or \
                    not (_pinned(g) or g.device.type == "cuda"):
                raise ValueError(f"grads[{i}] must be a bf16 tensor of at least {nv} elements, all of them "
                                 "pinned host tensors or all CUDA tensors")
        self.state_on_host = _pinned(master)
        for name, x in (("master", master), ("m", m), ("v", v)):
            if x.dtype != torch.float32 or x.numel() < L or _pinned(x) != self.state_on_host or \
                    not (_pinned(x) or x.device.type == "cuda"):
                raise ValueError(f"{name} must be an fp32 tensor of at least {L} elements; master, m and v "
                                 "all pinned host tensors or all CUDA tensors")
        if params.device.type != "cuda":
            raise ValueError("params must be a CUDA tensor")
        if params_host is not None and (not _pinned(params_host) or params_host.numel() < nv):
            raise ValueError("params_host must be a pinned host tensor of at least nv elements")
        if not (self.grads_on_host or self.state_on_host or params_host is not None):
            raise ValueError("no buffer in host memory: call the fused step directly")
        self.plan, self.base, self.L, self.nv = plan, base, L, nv
        self.grads, self.master, self.m, self.v, self.params = grads, master, m, v, params
        self.params_host, self.flag = params_host, overflow_flag
        dev = params.device
        self.chunk = max(8, (int(chunk_elems) + 7) // 8 * 8)
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        self.in_stream = torch.cuda.Stream(device=dev)
        self.out_stream = torch.cuda.Stream(device=dev)
        gsize = min(self.chunk, max(nv, 8))
        ssize = min(self.chunk, L)
        self.gslots = [[torch.empty(gsize, dtype=torch.bfloat16, device=dev) for _ in range(plan.M)]
                       for _ in range(_SLOTS)] if self.grads_on_host else None
        self.sslots = [[torch.empty(ssize, dtype=torch.float32, device=dev) for _ in range(3)]
                       for _ in range(_SLOTS)] if self.state_on_host else None
        self.copied_in = [torch.cuda.Event() for _ in range(_SLOTS)]
        self.computed = [torch.cuda.Event() for _ in range(_SLOTS)]
        self.copied_out = [torch.cuda.Event() for _ in range(_SLOTS)]
        cuts = list(range(0, L, self.chunk)) + [L]
        self.pieces = list(zip(cuts[:-1], cuts[1:]))

    def __call__(self, hp: _lib.AdamW) -> None:
        st, cin, cout = self.stream, self.in_stream, self.out_stream
        has_out = self.state_on_host or self.params_host is not None
        cin.wait_stream(st)                     # earlier work on the buffers is done
        for k, (e0, e1) in enumerate(self.pieces):
            slot = k % _SLOTS
            real = max(0, min(self.nv, e1) - e0)
            if k >= _SLOTS:                     # the slot's previous chunk is out of it
                cin.wait_event(self.copied_out[slot] if has_out else self.computed[slot])
            with torch.cuda.stream(cin):
                if self.grads_on_host and real:
                    for s, g in zip(self.gslots[slot], self.grads):
                        s[:real].copy_(g[e0:e0 + real], non_blocking=True)
                if self.state_on_host:
                    for s, x in zip(self.sslots[slot], (self.master, self.m, self.v)):
                        s[:e1 - e0].copy_(x[e0:e1], non_blocking=True)
                self.copied_in[slot].record(cin)
            st.wait_event(self.copied_in[slot])
            if self.grads_on_host:
                grads = [s[:max(real, 1)] for s in self.gslots[slot]]
            else:
                grads = [g[e0:e0 + real] for g in self.grads]
            state = self.sslots[slot] if self.state_on_host else [x[e0:] for x in (self.master, self.m, self.v)]
            params = self.params[e0:] if e0 < self.nv else self.params[:0]
            _lib.zero1_step_bucket(self.plan, self.base + e0, self.base + e1, grads, *state, params, hp,
                                   self.flag, stream=st)
            self.computed[slot].record(st)
            if has_out:
                cout.wait_event(self.computed[slot])
                with torch.cuda.stream(cout):
                    if self.state_on_host:
                        for s, x in zip(self.sslots[slot], (self.master, self.m, self.v)):
                            x[e0:e1].copy_(s[:e1 - e0], non_blocking=True)
                    if self.params_host is not None and real:
                        self.params_host[e0:e0 + real].copy_(self.params[e0:e0 + real], non_blocking=True)
                    self.copied_out[slot].record(cout)
        if has_out:
            st.wait_stream(cout)                # the copies back are part of the step
