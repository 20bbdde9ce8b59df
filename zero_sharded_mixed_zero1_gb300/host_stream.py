"""The fused step over buffers in pinned host memory, staged through HBM by
the copy engines while the computation runs: the binding of the staged-step
handle (zero1_staged_create / zero1_staged_step / zero1_staged_destroy).

The library cuts the range into chunks; for each chunk an inbound copy
stream moves the host-resident inputs (gradients, fp32 master/m/v) into one
of three device slots, the fused step runs on the slot on the caller's
stream, and an outbound copy stream moves the host-resident outputs back
(master/m/v, and the bf16 parameters when a host copy is wanted).  This is
the ZeRO-Offload placement of the fp32 state in host memory with the update
itself on the GPU.  The results are bit for bit those of one fused step on
device buffers.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib


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
    must be in host memory, or there is nothing to stage.

    chunk_elems sets the copy granularity (rounded up to a multiple of 8; the
    default 8M elements measured faster than 4M and 16M on GB300);
    the library allocates 3 x chunk_elems x (2M bytes if the gradients are
    staged + 12 bytes if the state is) of device memory for the slots, and
    two copy streams.  Launches go to `stream` (default: the current stream
    at each call); when the stream reaches work enqueued after a call, the
    step and its copies back to host memory are complete."""

    def __init__(self, plan: _lib.Plan, shard_begin: int, shard_end: int, grads, master, m, v, params,
                 chunk_elems: int = 1 << 23, params_host=None, overflow_flag=None, stream=None,
                 timeline: bool = False):
        _lib._replicas(plan, grads, "grads")
        base, L, nv = _lib._range(plan, shard_begin, shard_end)
        if L == 0:
            raise ValueError("empty or invalid shard range")
        grads_on_host = _pinned(grads[0])
        for i, g in enumerate(grads):
            if _pinned(g) != grads_on_host:
                raise ValueError("grads: all pinned host tensors or all CUDA tensors")
        state_on_host = _pinned(master)
        if _pinned(m) != state_on_host or _pinned(v) != state_on_host:
            raise ValueError("master, m and v: all pinned host tensors or all CUDA tensors")
        if params.device.type != "cuda":
            raise ValueError("params must be a CUDA tensor")
        if params_host is not None and not _pinned(params_host):
            raise ValueError("params_host must be a pinned host tensor")
        what = ((_lib.ZERO1_STAGE_GRADS if grads_on_host else 0) |
                (_lib.ZERO1_STAGE_STATE if state_on_host else 0) |
                (_lib.ZERO1_STAGE_PARAMS if params_host is not None else 0))
        if what == 0:
            raise ValueError("no buffer in host memory: call the fused step directly")
        if timeline:
            what |= _lib.ZERO1_STAGE_TIMELINE
        self.plan, self.nv, self.L = plan, nv, L
        self.chunk = max(8, (int(chunk_elems) + 7) // 8 * 8)
        # keep the tensors alive for as long as the handle holds their addresses
        self._tensors = (list(grads), master, m, v, params, params_host, overflow_flag)
        self._grads = _lib._ptrs(grads, torch.bfloat16, nv, "grads")
        self._state = [_lib._dev(x, torch.float32, L, name) for x, name in ((master, "master"), (m, "m"), (v, "v"))]
        self._params = _lib._dev(params, torch.bfloat16, nv, "params")
        self._params_host = _lib._dev(params_host, torch.bfloat16, nv, "params_host") if params_host is not None \
            else None
        self._flag = _lib._dev(overflow_flag, torch.int32, 1, "overflow_flag") if overflow_flag is not None \
            else None
        self._stream = stream
        self._device = params.device
        self._lib = _lib.load()
        handle = ctypes.c_void_p()
        with torch.cuda.device(self._device):
            _lib._check_rc(self._lib.zero1_staged_create(ctypes.byref(plan), shard_begin, shard_end, what,
                                                         self.chunk, ctypes.byref(handle)))
        self._handle = handle
        count = ctypes.c_int32()
        _lib._check_rc(self._lib.zero1_staged_chunks(handle, None, 0, ctypes.byref(count)))
        cuts = (ctypes.c_int64 * count.value)()
        _lib._check_rc(self._lib.zero1_staged_chunks(handle, cuts, count.value, ctypes.byref(count)))
        self.pieces = list(zip(cuts[:-1], cuts[1:]))   # the library's chunk boundaries

    def __call__(self, hp: _lib.AdamW) -> None:
        if self._handle is None:
            raise ValueError("the staged step has been closed")
        with torch.cuda.device(self._device):
            _lib._check_rc(self._lib.zero1_staged_step(
                self._handle, self._grads, *self._state, self._params, self._params_host,
                ctypes.byref(hp.c_struct()), self._flag, _lib._stream(self._stream)))

    def dynamic(self, hp: _lib.AdamW, scaler: torch.Tensor, policy: _lib.LossScalePolicy) -> None:
        """One attempt with dynamic loss scaling (zero1_staged_step_dynamic):
        S and t come from the device scaler, an overflow pass decides the skip
        before any chunk is updated, and the scaler advances afterwards.  The
        overflow_flag given at construction is not used."""
        if self._handle is None:
            raise ValueError("the staged step has been closed")
        with torch.cuda.device(self._device):
            _lib._check_rc(self._lib.zero1_staged_step_dynamic(
                self._handle, self._grads, *self._state, self._params, self._params_host,
                ctypes.byref(hp.c_struct()), _lib._scaler_ptr(scaler), ctypes.byref(policy.c_struct()),
                _lib._stream(self._stream)))

    def timeline(self):
        """Per-chunk timeline of the last step (created with timeline=True):
        a (chunks, 6) float32 array of milliseconds since the step started -
        inbound copies start/end, kernel start/end, outbound copies start/end
        (-1 when nothing is copied back).  Waits for the step to finish."""
        import numpy as np
        if self._handle is None:
            raise ValueError("the staged step has been closed")
        count = ctypes.c_int32()
        _lib._check_rc(self._lib.zero1_staged_timeline(self._handle, None, 0, ctypes.byref(count)))
        out = np.zeros((count.value, 6), np.float32)
        _lib._check_rc(self._lib.zero1_staged_timeline(self._handle, out.ctypes.data, out.size, ctypes.byref(count)))
        return out

    def close(self) -> None:
        """Wait for the handle's queued work and free its staging memory."""
        if getattr(self, "_handle", None) is not None:
            with torch.cuda.device(self._device):
                self._lib.zero1_staged_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
