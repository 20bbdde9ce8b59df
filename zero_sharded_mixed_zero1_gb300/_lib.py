"""ctypes binding of libzero1.so (include/zero1.h).

Argument marshalling only: every step of the optimizer path runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current CUDA
stream.  The binding checks what a C caller would have to guarantee (device,
dtype, contiguity and that each tensor is long enough) so that a wrong tensor
raises here instead of reaching the GPU.  There is no fallback: if the
library is not built, loading fails.
"""
from __future__ import annotations

import ctypes
import os
import struct
from dataclasses import dataclass

import torch

from . import build as _build

ZERO1_OK, ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ERANGE, ZERO1_ECUDA = 0, -1, -2, -3, -4
ZERO1_MAX_REPLICAS = 64
ZERO1_DTYPE_BF16, ZERO1_DTYPE_F32 = 0, 1
ZERO1_STAGE_GRADS, ZERO1_STAGE_STATE, ZERO1_STAGE_PARAMS, ZERO1_STAGE_TIMELINE = 1, 2, 4, 8

_lib = None


class Zero1Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


# zero1_abi_version() of the library this binding is written for.
ABI_VERSION = 3


class Plan(ctypes.Structure):
    """zero1_plan_t: n real parameters padded to P = multiple of M*align,
    shard size s = P/M."""
    _fields_ = [("n", ctypes.c_int64), ("padded_n", ctypes.c_int64), ("shard", ctypes.c_int64),
                ("M", ctypes.c_int32), ("align", ctypes.c_int32), ("n_tensors", ctypes.c_int32)]

    def shard_range(self, shard_begin: int, shard_end: int) -> tuple[int, int, int]:
        """(base element, length L, real elements nv) of shards [begin, end)."""
        base = shard_begin * self.shard
        L = (shard_end - shard_begin) * self.shard
        return base, L, max(0, min(self.n - base, L))

    def __repr__(self):
        return (f"Plan(n={self.n}, padded_n={self.padded_n}, shard={self.shard}, "
                f"M={self.M}, align={self.align}, n_tensors={self.n_tensors})")


class _AdamWStruct(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("loss_scale", ctypes.c_float), ("global_batch", ctypes.c_int64),
                ("step", ctypes.c_int64)]


@dataclass(frozen=True)
class AdamW:
    """zero1_adamw_t: AdamW hyperparameters, global batch B, loss scale S and
    step t of one optimizer step."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    loss_scale: float = 1.0
    global_batch: int = 1
    step: int = 1

    def c_struct(self) -> _AdamWStruct:
        return _AdamWStruct(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay,
                            self.loss_scale, self.global_batch, self.step)


class _PolicyStruct(ctypes.Structure):
    _fields_ = [("initial_scale", ctypes.c_float), ("factor", ctypes.c_float), ("window", ctypes.c_int32),
                ("hysteresis", ctypes.c_int32), ("min_scale", ctypes.c_float)]


@dataclass(frozen=True)
class LossScalePolicy:
    """zero1_loss_scale_policy_t: initial scale (2^initial_scale_power),
    growth/back-off factor, loss_scale_window, hysteresis, min_loss_scale."""
    initial_scale: float = 2.0 ** 12
    factor: float = 2.0
    window: int = 1000
    hysteresis: int = 2
    min_scale: float = 1.0

    def c_struct(self) -> _PolicyStruct:
        return _PolicyStruct(self.initial_scale, self.factor, self.window, self.hysteresis, self.min_scale)


SCALER_BYTES = 56
_SCALER_FMT = "<ffffqqqiiII"


def new_scaler(device) -> torch.Tensor:
    """Device storage for one zero1_scaler_t (56 bytes)."""
    return torch.zeros(SCALER_BYTES, dtype=torch.uint8, device=device)


def scaler_state(scaler: torch.Tensor) -> dict:
    """Read a zero1_scaler_t back to the host (synchronises with its stream)."""
    raw = bytes(scaler.cpu().numpy().tobytes())
    k = ["scale", "inv", "bc1", "bc2", "step", "attempts", "skipped", "good_steps", "hysteresis_left",
         "overflow", "current"]
    return dict(zip(k, struct.unpack(_SCALER_FMT, raw)))


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libzero1.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"libzero1.so is not built ({path}); run zero_sharded_mixed_zero1_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    P = ctypes.POINTER(Plan)
    A = ctypes.POINTER(_AdamWStruct)
    sig = {
        "zero1_plan": [i64, i32, i32, vp, i32, P],
        "zero1_plan_segments": [P, vp, i32, vp, vp, vp, i32, vp],
        "zero1_plan_memory": [P, vp, vp],
        "zero1_reduce_scatter_adamw_allgather": [P, i32, i32, vp, vp, vp, vp, vp, A, vp, i32, vp],
        "zero1_overflow_check": [P, i32, i32, vp, vp, vp],
        "dp_allreduce": [P, vp, vp, f32, i32, vp],
        "zero1_reduce_scatter": [P, i32, i32, vp, f32, i32, vp, vp, vp],
        "zero1_adamw_update": [P, i32, i32, vp, vp, vp, vp, A, vp],
        "zero1_all_gather": [P, i32, i32, vp, vp, vp],
        "zero1_all_gather_shards": [P, vp, vp, vp],
        "zero1_scaler_init": [vp, ctypes.POINTER(_PolicyStruct), A, vp],
        "zero1_step_bucket": [P, i64, i64, vp, vp, vp, vp, vp, A, vp, vp],
        "zero1_step_tma": [P, i32, i32, vp, vp, vp, vp, vp, A, vp, i32, vp],
        "zero1_device_status": [vp, i32],
        "zero1_bounded_wait_selftest": [ctypes.c_uint32, vp, vp],
        "zero1_checksum": [vp, i64, vp, vp],
        "zero1_step_dynamic": [P, i32, i32, vp, vp, vp, vp, vp, A, vp, ctypes.POINTER(_PolicyStruct), vp, vp],
        "zero1_step_dynamic_noalloc": [P, i32, i32, vp, vp, vp, vp, vp, A, vp, ctypes.POINTER(_PolicyStruct), vp],
        "zero1_step_dynamic_pingpong": [P, i32, i32, vp, vp, vp, vp, vp, A, vp, ctypes.POINTER(_PolicyStruct), vp],
        "zero1_pingpong_bucket": [P, i64, i64, vp, vp, vp, vp, vp, A, vp, vp],
        "zero1_pingpong_finish": [P, i32, i32, vp, vp, A, vp, ctypes.POINTER(_PolicyStruct), vp],
        "zero1_staged_create": [P, i32, i32, i32, i64, ctypes.POINTER(vp)],
        "zero1_staged_step": [vp, vp, vp, vp, vp, vp, vp, A, vp, vp],
        "zero1_staged_destroy": [vp],
        "zero1_staged_chunks": [vp, vp, i32, vp],
        "zero1_staged_timeline": [vp, vp, i32, vp],
        "zero1_staged_step_dynamic": [vp, vp, vp, vp, vp, vp, vp, A, vp, ctypes.POINTER(_PolicyStruct), vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.zero1_strerror.argtypes = [ctypes.c_int]
    lib.zero1_strerror.restype = ctypes.c_char_p
    lib.zero1_last_error.argtypes = []
    lib.zero1_last_error.restype = ctypes.c_char_p
    lib.zero1_abi_version.argtypes = []
    lib.zero1_abi_version.restype = ctypes.c_int
    lib.zero1_debug_last_launch.argtypes = [ctypes.POINTER(ctypes.c_char_p), vp, vp, vp, vp]
    lib.zero1_debug_last_launch.restype = ctypes.c_int
    if lib.zero1_abi_version() != ABI_VERSION:
        raise ImportError(f"libzero1.so has ABI version {lib.zero1_abi_version()}, the binding expects "
                          f"{ABI_VERSION}; rebuild it")
    _lib = lib
    return lib


def _check_rc(rc: int) -> None:
    if rc != ZERO1_OK:
        lib = load()
        raise Zero1Error(rc, f"{lib.zero1_strerror(rc).decode()}: {lib.zero1_last_error().decode()}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtype: torch.dtype, min_numel: int, what: str) -> int:
    """Pointer of a tensor the GPU can address: a CUDA tensor, or a pinned
    host tensor (mapped at the same address; the kernels reach it over the
    host link)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: expected a torch.Tensor")
    if t.device.type != "cuda" and not (t.device.type == "cpu" and t.is_pinned()):
        raise ValueError(f"{what}: must be a CUDA tensor or a pinned host tensor")
    if t.dtype != dtype:
        raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    if t.numel() < min_numel:
        raise ValueError(f"{what}: has {t.numel()} elements, needs at least {min_numel}")
    return t.data_ptr()


def _ptrs(tensors, dtype, min_numel, what) -> ctypes.Array:
    return (ctypes.c_void_p * len(tensors))(*[_dev(t, dtype, min_numel, f"{what}[{i}]")
                                              for i, t in enumerate(tensors)])


def _range(plan: Plan, shard_begin: int, shard_end: int) -> tuple[int, int, int]:
    """(base, L, nv) of a shard range, or zeros for an invalid range (which
    the library then rejects with its own message)."""
    if 0 <= shard_begin < shard_end <= plan.M:
        return plan.shard_range(shard_begin, shard_end)
    return 0, 0, 0


def _replicas(plan: Plan, tensors, what: str) -> None:
    if len(tensors) != plan.M:
        raise ValueError(f"{what}: expected M = {plan.M} tensors, got {len(tensors)}")


# -- plan ---------------------------------------------------------------------

def zero1_plan(n: int, M: int, align: int = 1, tensor_numels=None) -> Plan:
    """The shard plan; tensor_numels (optional) lists the tensors the flat
    buffer concatenates, for zero1_plan_segments."""
    p = Plan()
    if tensor_numels is None:
        _check_rc(load().zero1_plan(n, M, align, None, 0, ctypes.byref(p)))
    else:
        nums = (ctypes.c_int64 * len(tensor_numels))(*tensor_numels)
        _check_rc(load().zero1_plan(n, M, align, nums, len(tensor_numels), ctypes.byref(p)))
    return p


def zero1_plan_segments(plan: Plan, tensor_numels, shard_index: int):
    """[(tensor index, first element inside the tensor, length)] of one
    shard, in shard order; the plan must have been built with the list."""
    nums = (ctypes.c_int64 * len(tensor_numels))(*tensor_numels)
    cap = len(tensor_numels) + 1
    outs = [(ctypes.c_int64 * cap)() for _ in range(3)]
    count = ctypes.c_int32()
    _check_rc(load().zero1_plan_segments(ctypes.byref(plan), nums, shard_index, *outs, cap, ctypes.byref(count)))
    return [tuple(int(o[i]) for o in outs) for i in range(count.value)]


def debug_last_launch() -> dict:
    """The last kernel launched by a library call on this host thread: its
    (mangled) name, grid, the resident blocks per SM the grid was sized from,
    the threads per block, and whether the vector body moved fp32 in 32-byte
    accesses."""
    name = ctypes.c_char_p()
    grid, per_sm, block, w32 = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check_rc(load().zero1_debug_last_launch(ctypes.byref(name), ctypes.byref(grid), ctypes.byref(per_sm),
                                             ctypes.byref(block), ctypes.byref(w32)))
    return {"kernel": name.value.decode(), "grid": grid.value, "blocks_per_sm": per_sm.value,
            "block": block.value, "w32": bool(w32.value)}


def zero1_plan_memory(plan: Plan) -> tuple[int, int]:
    """(naive data-parallel bytes per rank, ZeRO-1 bytes per rank)."""
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check_rc(load().zero1_plan_memory(ctypes.byref(plan), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


# -- the step -----------------------------------------------------------------

def zero1_reduce_scatter_adamw_allgather(plan: Plan, shard_begin: int, shard_end: int, grads,
                                         master, m, v, params, hp: AdamW, overflow_flag=None,
                                         skip_if_flag: bool = False, stream=None) -> None:
    """Fused ZeRO-1 step over shards [shard_begin, shard_end).  grads[r] and
    params start at the range's first global element; master/m/v hold the
    range's fp32 state (L elements)."""
    _replicas(plan, grads, "grads")
    _, L, nv = _range(plan, shard_begin, shard_end)
    g = _ptrs(grads, torch.bfloat16, nv, "grads")
    flag = 0 if overflow_flag is None else _dev(overflow_flag, torch.int32, 1, "overflow_flag")
    _check_rc(load().zero1_reduce_scatter_adamw_allgather(
        ctypes.byref(plan), shard_begin, shard_end, g,
        _dev(master, torch.float32, L, "master"), _dev(m, torch.float32, L, "m"),
        _dev(v, torch.float32, L, "v"), _dev(params, torch.bfloat16, nv, "params"),
        ctypes.byref(hp.c_struct()), flag or None, int(bool(skip_if_flag)), _stream(stream)))


def zero1_step_tma(plan: Plan, shard_begin: int, shard_end: int, grads, master, m, v, params, hp: AdamW,
                   overflow_flag=None, skip_if_flag: bool = False, stream=None) -> None:
    """The fused step with shared-memory staging by bulk copies (same
    arguments and bits as zero1_reduce_scatter_adamw_allgather; device
    memory only)."""
    _replicas(plan, grads, "grads")
    _, L, nv = _range(plan, shard_begin, shard_end)
    flag = 0 if overflow_flag is None else _dev(overflow_flag, torch.int32, 1, "overflow_flag")
    _check_rc(load().zero1_step_tma(
        ctypes.byref(plan), shard_begin, shard_end, _ptrs(grads, torch.bfloat16, nv, "grads"),
        _dev(master, torch.float32, L, "master"), _dev(m, torch.float32, L, "m"), _dev(v, torch.float32, L, "v"),
        _dev(params, torch.bfloat16, nv, "params"), ctypes.byref(hp.c_struct()), flag or None,
        int(bool(skip_if_flag)), _stream(stream)))


def zero1_bounded_wait_selftest(limit_us: int, gave_up: torch.Tensor, stream=None) -> None:
    """Launch the bounded-wait self-test: a wait that cannot complete must give
    up after limit_us, write 1 to gave_up (device int32) and set bit 0 of the
    device status word."""
    _check_rc(load().zero1_bounded_wait_selftest(int(limit_us), _dev(gave_up, torch.int32, 1, "gave_up"),
                                                 _stream(stream)))


def zero1_checksum(t: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Consistency checksum of a tensor's bytes as 16-bit units: a device
    int64 tensor of two words (sum of units, sum of (index + 1) * unit, both
    mod 2^64; read them as unsigned)."""
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise ValueError("checksum: expected a contiguous tensor")
    if t.device.type != "cuda" and not (t.device.type == "cpu" and t.is_pinned()):
        raise ValueError("checksum: must be a CUDA tensor or a pinned host tensor")
    nbytes = t.numel() * t.element_size()
    if out is None:
        dev = t.device if t.device.type == "cuda" else torch.device("cuda", torch.cuda.current_device())
        out = torch.empty(2, dtype=torch.int64, device=dev)
    _check_rc(load().zero1_checksum(t.data_ptr() if nbytes else None, nbytes,
                                    _dev(out, torch.int64, 2, "out"), _stream(stream)))
    return out


def zero1_device_status(clear: bool = True) -> int:
    """The library's device status word (bit 0: a bounded wait ran out)."""
    out = ctypes.c_uint32()
    _check_rc(load().zero1_device_status(ctypes.byref(out), int(bool(clear))))
    return out.value


def zero1_step_bucket(plan: Plan, elem_begin: int, elem_end: int, grads, master, m, v, params, hp: AdamW,
                      overflow_flag=None, stream=None) -> None:
    """The fused step on the element range [elem_begin, elem_end) of the
    padded flat buffer (one gradient bucket).  grads[r]: the bucket's
    gradients; master/m/v/params: tensors starting at element elem_begin."""
    _replicas(plan, grads, "grads")
    L = max(0, elem_end - elem_begin)
    nv = max(0, min(plan.n - elem_begin, L))
    flag = 0 if overflow_flag is None else _dev(overflow_flag, torch.int32, 1, "overflow_flag")
    _check_rc(load().zero1_step_bucket(
        ctypes.byref(plan), elem_begin, elem_end, _ptrs(grads, torch.bfloat16, nv, "grads"),
        _dev(master, torch.float32, L, "master"), _dev(m, torch.float32, L, "m"), _dev(v, torch.float32, L, "v"),
        _dev(params, torch.bfloat16, nv, "params"), ctypes.byref(hp.c_struct()), flag or None, _stream(stream)))


def zero1_overflow_check(plan: Plan, shard_begin: int, shard_end: int, grads, flag, stream=None) -> None:
    _replicas(plan, grads, "grads")
    _, _, nv = _range(plan, shard_begin, shard_end)
    _check_rc(load().zero1_overflow_check(ctypes.byref(plan), shard_begin, shard_end,
                                          _ptrs(grads, torch.bfloat16, nv, "grads"),
                                          _dev(flag, torch.int32, 1, "flag"), _stream(stream)))


def dp_allreduce(plan: Plan, grads_in, outs, scale: float = 1.0, stream=None) -> None:
    """Naive All-Reduce; output dtype (bf16 or fp32) from outs."""
    _replicas(plan, grads_in, "grads_in")
    _replicas(plan, outs, "outs")
    dt = outs[0].dtype
    code = {torch.bfloat16: ZERO1_DTYPE_BF16, torch.float32: ZERO1_DTYPE_F32}.get(dt)
    if code is None:
        raise TypeError("outs must be bfloat16 or float32")
    _check_rc(load().dp_allreduce(ctypes.byref(plan), _ptrs(grads_in, torch.bfloat16, plan.n, "grads_in"),
                                  _ptrs(outs, dt, plan.n, "outs"), scale, code, _stream(stream)))


def zero1_reduce_scatter(plan: Plan, shard_begin: int, shard_end: int, grads, scale: float, out,
                         flag=None, stream=None) -> None:
    _replicas(plan, grads, "grads")
    _, L, nv = _range(plan, shard_begin, shard_end)
    code = {torch.bfloat16: ZERO1_DTYPE_BF16, torch.float32: ZERO1_DTYPE_F32}.get(out.dtype)
    if code is None:
        raise TypeError("out must be bfloat16 or float32")
    f = 0 if flag is None else _dev(flag, torch.int32, 1, "flag")
    _check_rc(load().zero1_reduce_scatter(ctypes.byref(plan), shard_begin, shard_end,
                                          _ptrs(grads, torch.bfloat16, nv, "grads"), scale, code,
                                          _dev(out, out.dtype, L, "out"), f or None, _stream(stream)))


def zero1_adamw_update(plan: Plan, shard_begin: int, shard_end: int, g, master, m, v, hp: AdamW,
                       stream=None) -> None:
    _, L, _ = _range(plan, shard_begin, shard_end)
    _check_rc(load().zero1_adamw_update(ctypes.byref(plan), shard_begin, shard_end,
                                        _dev(g, torch.float32, L, "g"), _dev(master, torch.float32, L, "master"),
                                        _dev(m, torch.float32, L, "m"), _dev(v, torch.float32, L, "v"),
                                        ctypes.byref(hp.c_struct()), _stream(stream)))


def zero1_all_gather(plan: Plan, shard_begin: int, shard_end: int, master, params, stream=None) -> None:
    _, L, nv = _range(plan, shard_begin, shard_end)
    _check_rc(load().zero1_all_gather(ctypes.byref(plan), shard_begin, shard_end,
                                      _dev(master, torch.float32, nv, "master"),
                                      _dev(params, torch.bfloat16, nv, "params"), _stream(stream)))


def zero1_all_gather_shards(plan: Plan, shards, outs, stream=None) -> None:
    _replicas(plan, outs, "outs")
    _check_rc(load().zero1_all_gather_shards(ctypes.byref(plan), _dev(shards, torch.bfloat16, plan.n, "shards"),
                                             _ptrs(outs, torch.bfloat16, plan.n, "outs"), _stream(stream)))


# -- dynamic loss scaling -------------------------------------------------------

def _scaler_ptr(scaler: torch.Tensor) -> int:
    if scaler.dtype != torch.uint8 or scaler.numel() < SCALER_BYTES or scaler.device.type != "cuda":
        raise ValueError("scaler must be a CUDA uint8 tensor of at least 56 bytes (new_scaler)")
    return scaler.data_ptr()


def zero1_scaler_init(scaler: torch.Tensor, policy: LossScalePolicy, hp: AdamW, stream=None) -> None:
    """Start a device-resident scaler: S = policy.initial_scale, t = hp.step."""
    _check_rc(load().zero1_scaler_init(_scaler_ptr(scaler), ctypes.byref(policy.c_struct()),
                                       ctypes.byref(hp.c_struct()), _stream(stream)))


def zero1_step_dynamic(plan: Plan, shard_begin: int, shard_end: int, grads, master, m, v, params, hp: AdamW,
                       scaler: torch.Tensor, policy: LossScalePolicy, sums, stream=None) -> None:
    """One dynamically scaled attempt (S and t from the device scaler);
    sums: fp32 workspace of at least L elements."""
    _replicas(plan, grads, "grads")
    _, L, nv = _range(plan, shard_begin, shard_end)
    _check_rc(load().zero1_step_dynamic(
        ctypes.byref(plan), shard_begin, shard_end, _ptrs(grads, torch.bfloat16, nv, "grads"),
        _dev(master, torch.float32, L, "master"), _dev(m, torch.float32, L, "m"), _dev(v, torch.float32, L, "v"),
        _dev(params, torch.bfloat16, nv, "params"), ctypes.byref(hp.c_struct()), _scaler_ptr(scaler),
        ctypes.byref(policy.c_struct()), _dev(sums, torch.float32, L, "sums"), _stream(stream)))


def zero1_step_dynamic_pingpong(plan: Plan, shard_begin: int, shard_end: int, grads, master, m, v, params,
                                hp: AdamW, scaler: torch.Tensor, policy: LossScalePolicy, stream=None) -> None:
    """One dynamically scaled attempt with ping-pong state: master, m, v are
    pairs of fp32 tensors (two copies of the state; the scaler's `current`
    field names the one holding the current state, see current_state)."""
    _replicas(plan, grads, "grads")
    _, L, nv = _range(plan, shard_begin, shard_end)
    pairs = [_pair(name, pair, L) for name, pair in (("master", master), ("m", m), ("v", v))]
    _check_rc(load().zero1_step_dynamic_pingpong(
        ctypes.byref(plan), shard_begin, shard_end, _ptrs(grads, torch.bfloat16, nv, "grads"), *pairs,
        _dev(params, torch.bfloat16, nv, "params"), ctypes.byref(hp.c_struct()), _scaler_ptr(scaler),
        ctypes.byref(policy.c_struct()), _stream(stream)))


def _pair(name, pair, numel):
    if len(pair) != 2:
        raise ValueError(f"{name}: expected two tensors (the two copies of the state)")
    return (ctypes.c_void_p * 2)(*[_dev(t, torch.float32, numel, f"{name}[{k}]") for k, t in enumerate(pair)])


def zero1_pingpong_bucket(plan: Plan, elem_begin: int, elem_end: int, grads, master, m, v, params, hp: AdamW,
                          scaler: torch.Tensor, stream=None) -> None:
    """The ping-pong kernel on one bucket [elem_begin, elem_end): master, m,
    v are pairs of tensors and params a tensor, all starting at element
    elem_begin; grads[r] the bucket's gradients."""
    _replicas(plan, grads, "grads")
    L = max(0, elem_end - elem_begin)
    nv = max(0, min(plan.n - elem_begin, L))
    _check_rc(load().zero1_pingpong_bucket(
        ctypes.byref(plan), elem_begin, elem_end, _ptrs(grads, torch.bfloat16, nv, "grads"),
        _pair("master", master, L), _pair("m", m, L), _pair("v", v, L), _dev(params, torch.bfloat16, nv, "params"),
        ctypes.byref(hp.c_struct()), _scaler_ptr(scaler), _stream(stream)))


def zero1_pingpong_finish(plan: Plan, shard_begin: int, shard_end: int, master, params, hp: AdamW,
                          scaler: torch.Tensor, policy: LossScalePolicy, stream=None) -> None:
    """End of a bucketed ping-pong attempt over shards [shard_begin,
    shard_end): params restored if any bucket overflowed, scaler advanced."""
    _, L, nv = _range(plan, shard_begin, shard_end)
    _check_rc(load().zero1_pingpong_finish(
        ctypes.byref(plan), shard_begin, shard_end, _pair("master", master, L),
        _dev(params, torch.bfloat16, nv, "params"), ctypes.byref(hp.c_struct()), _scaler_ptr(scaler),
        ctypes.byref(policy.c_struct()), _stream(stream)))


class PingPongBuckets:
    """One ping-pong attempt fed bucket by bucket over shards [shard_begin,
    shard_end), with the copies (pairs of L-element fp32 tensors) and params
    (nv elements) of the whole range.  bucket() takes offsets relative to the
    range; finish() checks on the host that the attempt's buckets covered the
    range once, then ends the attempt."""

    def __init__(self, plan: Plan, shard_begin: int, shard_end: int, master, m, v, params, scaler: torch.Tensor,
                 policy: LossScalePolicy, stream=None):
        self.plan, self.sb, self.se = plan, shard_begin, shard_end
        self.base, self.L, self.nv = _range(plan, shard_begin, shard_end)
        if self.L == 0:
            raise ValueError("empty or invalid shard range")
        self.master, self.m, self.v, self.params = master, m, v, params
        self.scaler, self.policy, self.stream = scaler, policy, stream
        self._done = []

    def bucket(self, begin: int, end: int, grads, hp: AdamW) -> None:
        if not 0 <= begin < end <= self.L:
            raise ValueError(f"bucket [{begin}, {end}) not inside the range [0, {self.L})")
        params = self.params[begin:] if begin < self.nv else self.params[:0]
        zero1_pingpong_bucket(self.plan, self.base + begin, self.base + end, grads,
                              [x[begin:] for x in self.master], [x[begin:] for x in self.m],
                              [x[begin:] for x in self.v], params, hp, self.scaler, self.stream)
        self._done.append((begin, end))

    def finish(self, hp: AdamW) -> None:
        cover = sorted(self._done)
        edge = 0
        for b, e in cover:
            if b != edge:
                raise ValueError(f"the attempt's buckets do not cover the range once (at element {edge})")
            edge = e
        if edge != self.L:
            raise ValueError(f"the attempt's buckets end at element {edge}, not {self.L}")
        zero1_pingpong_finish(self.plan, self.sb, self.se, self.master, self.params, hp, self.scaler, self.policy,
                              self.stream)
        self._done = []


def current_state(scaler: torch.Tensor, master, m, v):
    """(master, m, v) of the copy holding the current state after ping-pong
    attempts (reads the scaler back: synchronises with its stream)."""
    k = scaler_state(scaler)["current"] & 1
    return master[k], m[k], v[k]


# -- the dynamically scaled step with the library's own workspace --------------

ZERO1_NOALLOC_MAX_ELEMS = 16 * 1024 * 1024


def zero1_step_dynamic_noalloc(plan: Plan, shard_begin: int, shard_end: int, grads, master, m, v, params,
                               hp: AdamW, scaler: torch.Tensor, policy: LossScalePolicy, stream=None) -> None:
    """zero1_step_dynamic without a caller-provided workspace (the library's
    built-in 64 MiB array; ranges of at most ZERO1_NOALLOC_MAX_ELEMS
    elements).  For callers that cannot allocate device memory."""
    fn = load().zero1_step_dynamic_noalloc
    _replicas(plan, grads, "grads")
    _, L, nv = _range(plan, shard_begin, shard_end)
    _check_rc(fn(ctypes.byref(plan), shard_begin, shard_end, _ptrs(grads, torch.bfloat16, nv, "grads"),
                 _dev(master, torch.float32, L, "master"), _dev(m, torch.float32, L, "m"),
                 _dev(v, torch.float32, L, "v"), _dev(params, torch.bfloat16, nv, "params"),
                 ctypes.byref(hp.c_struct()), _scaler_ptr(scaler), ctypes.byref(policy.c_struct()),
                 _stream(stream)))


# -- a step bound to fixed buffers ---------------------------------------------

class FusedStep:
    """The fused ZeRO-1 step bound to fixed buffers, for training loops.

    The tensors are validated and their addresses marshalled once, here; each
    call then only fills in the step's hyperparameters and calls
    zero1_reduce_scatter_adamw_allgather, so the host cost per step is a few
    microseconds (the one-shot function re-checks every tensor each time,
    which dominates on small problems).  The tensors must stay alive and in
    place while the object is used.  Launches go to `stream` (default: the
    stream current when the object is made)."""

    def __init__(self, plan: Plan, shard_begin: int, shard_end: int, grads, master, m, v, params,
                 overflow_flag=None, skip_if_flag: bool = False, stream=None):
        _replicas(plan, grads, "grads")
        _, L, nv = _range(plan, shard_begin, shard_end)
        self._plan = plan
        # a copy of the list: the cached addresses stay valid even if the
        # caller later replaces an element of its own list
        self._keep = (tuple(grads), master, m, v, params, overflow_flag)
        self._grads = _ptrs(grads, torch.bfloat16, nv, "grads")
        flag = 0 if overflow_flag is None else _dev(overflow_flag, torch.int32, 1, "overflow_flag")
        self._args = (ctypes.byref(plan), shard_begin, shard_end, self._grads,
                      _dev(master, torch.float32, L, "master"), _dev(m, torch.float32, L, "m"),
                      _dev(v, torch.float32, L, "v"), _dev(params, torch.bfloat16, nv, "params"))
        self._hp = _AdamWStruct()
        self._tail = (flag or None, int(bool(skip_if_flag)), _stream(stream))
        self._fn = load().zero1_reduce_scatter_adamw_allgather

    def __call__(self, hp: AdamW) -> None:
        h = self._hp
        h.lr, h.beta1, h.beta2, h.eps, h.weight_decay = hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay
        h.loss_scale, h.global_batch, h.step = hp.loss_scale, hp.global_batch, hp.step
        rc = self._fn(*self._args, ctypes.byref(h), *self._tail)
        if rc != ZERO1_OK:
            _check_rc(rc)
