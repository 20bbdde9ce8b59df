"""CPU oracle of the ZeRO Stage-1 optimizer step (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes it, and this package
imports nothing from the product.

The arithmetic lives in ``zero1_oracle.c`` (plain C99, single-threaded, built
with ``-ffp-contract=off``); this module only compiles it with the host C
compiler and marshals numpy arrays.  Every function follows a passage of the
pages, cited in the C source:

* "CS336 Lecture 7: Parallelism 1" - naive data parallelism (the SGD equation
  with the 1/B mean), the five collectives and All-Reduce == Reduce-Scatter +
  All-Gather, the 16 bytes/parameter table, and the four steps of ZeRO Stage 1.
* "第2章 软件程序与专用硬件的结合" section 2.3.4 - each of N GPUs keeps 1/N of the
  optimizer state.
* "五维并行实战" sections 3.2 and 4.2 - AdamW hyperparameters and the fp16
  loss-scale / overflow behaviour.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero1_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler; returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cc = os.environ.get("CC", "gcc")
        subprocess.run([cc, *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        # ZERO1_ORACLE_LIB lets the mutation test load a deliberately broken
        # build of this same source, to show the pins catch each mistake.
        lib = ctypes.CDLL(os.environ.get("ZERO1_ORACLE_LIB") or build())
        i64, i32 = ctypes.c_int64, ctypes.c_int32
        f32, vp = ctypes.c_float, ctypes.c_void_p
        lib.orc_bf16_to_f32_array.argtypes = [vp, vp, i64]
        lib.orc_f32_to_bf16_array.argtypes = [vp, vp, i64]
        lib.orc_plan.argtypes = [i64, i32, i32, vp, vp]
        lib.orc_plan.restype = ctypes.c_int
        lib.orc_segments.argtypes = [vp, i32, i64, i32, i32, vp, vp, vp, vp]
        lib.orc_segments.restype = ctypes.c_int
        lib.orc_memory.argtypes = [i64, i64, vp, vp]
        lib.orc_adamw_constants.argtypes = [f32, f32, f32, f32, i64, f32, i64, vp]
        lib.orc_pow_int.argtypes = [ctypes.c_double, i64]
        lib.orc_pow_int.restype = ctypes.c_double
        lib.orc_reduce_scatter.argtypes = [i32, vp, i64, i64, f32, vp, vp]
        lib.orc_adamw.argtypes = [i64, vp, vp, vp, vp, f32, f32, f32, f32, vp]
        lib.orc_all_gather.argtypes = [i64, vp, vp]
        lib.orc_zero1_step.argtypes = [i32, vp, i64, i64, vp, vp, vp, vp,
                                       f32, f32, f32, f32, f32, f32, i64, i64, vp, i32]
        lib.orc_zero1_step.restype = ctypes.c_int
        lib.orc_allreduce.argtypes = [i32, vp, i64, f32, i32, vp]
        lib.orc_checksum16.argtypes = [vp, i64, vp]
        lib.orc_scaler_init.argtypes = [vp, f32, i32, i64]
        lib.orc_scaler_update.argtypes = [vp, ctypes.c_uint32, f32, i32, i32, f32]
        lib.orc_zero1_dynamic_attempt.argtypes = [i32, vp, i64, i64, vp, vp, vp, vp, f32, f32, f32, f32, f32,
                                                  i64, vp, f32, i32, i32, f32, vp]
        lib.orc_zero1_dynamic_attempt.restype = ctypes.c_int
        lib.orc_overflow_check.argtypes = [i32, vp, i64, vp]
        _lib = lib
    return _lib


@dataclass(frozen=True)
class AdamW:
    """Hyperparameters of one step, as the pages name them: learning rate,
    betas, eps, weight decay ("五维并行实战" section 4.2), global batch B (the 1/B
    of the naive data-parallel SGD equation), loss scale S and step t."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    loss_scale: float = 1.0
    global_batch: int = 1
    step: int = 1


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _ptr_array(arrays) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrays))(*[_ptr(a) for a in arrays])


def _check(a: np.ndarray, dtype) -> None:
    if a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"expected a contiguous {np.dtype(dtype)} array, got {a.dtype}")


# -- bf16 -------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float32)
    _L().orc_bf16_to_f32_array(_ptr(bits), _ptr(out), bits.size)
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _L().orc_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


# -- plan ---------------------------------------------------------------------

def plan(n: int, M: int, align: int) -> tuple[int, int]:
    """(padded length P, shard size s)."""
    P = ctypes.c_int64()
    s = ctypes.c_int64()
    if _L().orc_plan(n, M, align, ctypes.byref(P), ctypes.byref(s)) != 0:
        raise ValueError("invalid plan arguments")
    return P.value, s.value


def segments(numels, shard: int, idx: int) -> list[tuple[int, int, int, int]]:
    """[(tensor, offset in tensor, offset in shard, length)] for shard idx."""
    nums = np.ascontiguousarray(numels, dtype=np.int64)
    cap = len(nums) + 1
    outs = [np.zeros(cap, np.int64) for _ in range(4)]
    c = _L().orc_segments(_ptr(nums), len(nums), shard, idx, cap, *[_ptr(o) for o in outs])
    if c < 0:
        raise RuntimeError("segment capacity exceeded")
    return [tuple(int(o[i]) for o in outs) for i in range(c)]


def memory(n: int, shard: int) -> tuple[int, int]:
    """(naive data-parallel bytes per rank, ZeRO-1 bytes per rank)."""
    a = ctypes.c_int64()
    b = ctypes.c_int64()
    _L().orc_memory(n, shard, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def pow_int(b: float, t: int) -> float:
    """b^t in double by square-and-multiply (the bias-correction power)."""
    return _L().orc_pow_int(b, t)


def adamw_constants(hp: AdamW) -> dict:
    c = np.zeros(6, np.float32)
    _L().orc_adamw_constants(hp.lr, hp.beta1, hp.beta2, hp.weight_decay,
                             hp.global_batch, hp.loss_scale, hp.step, _ptr(c))
    return dict(zip(["inv", "omb1", "omb2", "bc1", "bc2", "cdec"], [np.float32(x) for x in c]))


# -- the step and its phases -------------------------------------------------

def reduce_scatter(grads, n_valid: int, length: int, scale: float):
    """(fp32 scaled rank-order sums over `length` elements, overflow flag)."""
    for g in grads:
        _check(g, np.uint16)
        assert g.size >= n_valid
    out = np.empty(length, np.float32)
    flag = np.zeros(1, np.uint32)
    _L().orc_reduce_scatter(len(grads), _ptr_array(grads), length, n_valid, scale,
                            _ptr(out), _ptr(flag))
    return out, int(flag[0])


def adamw(g, master, m, v, hp: AdamW) -> None:
    """In-place AdamW on fp32 arrays given the fp32 scaled gradient g."""
    for a in (g, master, m, v):
        _check(a, np.float32)
    c = np.zeros(6, np.float32)
    _L().orc_adamw_constants(hp.lr, hp.beta1, hp.beta2, hp.weight_decay,
                             hp.global_batch, hp.loss_scale, hp.step, _ptr(c))
    _L().orc_adamw(master.size, _ptr(g), _ptr(master), _ptr(m), _ptr(v),
                   hp.lr, hp.beta1, hp.beta2, hp.eps, _ptr(c))


def all_gather(master, n_valid: int, params) -> None:
    _check(master, np.float32)
    _check(params, np.uint16)
    _L().orc_all_gather(n_valid, _ptr(master), _ptr(params))


def zero1_step(grads, n_valid: int, master, m, v, params, hp: AdamW,
               flag: np.ndarray | None = None, skip_if_flag: bool = False) -> None:
    """One ZeRO-1 step over a shard range, in place on master/m/v/params.

    grads: M uint16 (bf16 bit) arrays, each at least n_valid long, starting at
    the range's first element; master/m/v: fp32 state of the range; params:
    uint16 array (at least n_valid long) receiving the bf16 parameters; flag: a
    uint32 array of one element, OR-ed (or, with skip_if_flag, only read)."""
    for g in grads:
        _check(g, np.uint16)
        assert g.size >= n_valid
    for a in (master, m, v):
        _check(a, np.float32)
        assert a.size == master.size
    _check(params, np.uint16)
    assert params.size >= n_valid and n_valid <= master.size
    if flag is not None:
        _check(flag, np.uint32)
    rc = _L().orc_zero1_step(len(grads), _ptr_array(grads), master.size, n_valid,
                             _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                             hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay,
                             hp.loss_scale, hp.global_batch, hp.step,
                             None if flag is None else _ptr(flag), int(skip_if_flag))
    if rc != 0:
        raise MemoryError("oracle step could not allocate its gradient buffer")


def allreduce(grads, n: int, scale: float = 1.0, out_bf16: bool = True, outs=None):
    """Naive All-Reduce; returns the M outputs (new arrays unless given)."""
    for g in grads:
        _check(g, np.uint16)
    if outs is None:
        outs = [np.empty(n, np.uint16 if out_bf16 else np.float32) for _ in grads]
    _L().orc_allreduce(len(grads), _ptr_array(grads), n, scale, int(out_bf16), _ptr_array(outs))
    return outs


def overflow_check(grads, n_valid: int) -> int:
    for g in grads:
        _check(g, np.uint16)
    flag = np.zeros(1, np.uint32)
    _L().orc_overflow_check(len(grads), _ptr_array(grads), n_valid, _ptr(flag))
    return int(flag[0])


# -- dynamic loss scaling ("五维并行实战" 4.2, fp16 block) ---------------------

@dataclass(frozen=True)
class LossScalePolicy:
    """The fp16 block's keys: the initial scale (2^initial_scale_power), the
    growth/back-off factor, loss_scale_window, hysteresis, min_loss_scale."""
    initial_scale: float = 2.0 ** 12
    factor: float = 2.0
    window: int = 1000
    hysteresis: int = 2
    min_scale: float = 1.0


class Scaler(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("good", ctypes.c_int32), ("hyst_left", ctypes.c_int32),
                ("step", ctypes.c_int64), ("attempts", ctypes.c_int64), ("skipped", ctypes.c_int64)]

    @classmethod
    def start(cls, policy: LossScalePolicy, first_step: int = 1) -> "Scaler":
        sc = cls()
        _L().orc_scaler_init(ctypes.byref(sc), policy.initial_scale, policy.hysteresis, first_step)
        return sc

    def update(self, overflow: int, policy: LossScalePolicy) -> None:
        _L().orc_scaler_update(ctypes.byref(self), int(overflow), policy.factor, policy.window,
                               policy.hysteresis, policy.min_scale)


def zero1_dynamic_attempt(grads, n_valid: int, master, m, v, params, hp: AdamW, scaler: Scaler,
                          policy: LossScalePolicy) -> int:
    """One attempt of the dynamically scaled step over a whole range (hp's
    loss_scale and step are ignored: the scaler's are used).  Returns the
    attempt's overflow flag."""
    for g in grads:
        _check(g, np.uint16)
    for a in (master, m, v):
        _check(a, np.float32)
    _check(params, np.uint16)
    f = ctypes.c_uint32()
    rc = _L().orc_zero1_dynamic_attempt(len(grads), _ptr_array(grads), master.size, n_valid, _ptr(master),
                                        _ptr(m), _ptr(v), _ptr(params), hp.lr, hp.beta1, hp.beta2, hp.eps,
                                        hp.weight_decay, hp.global_batch, ctypes.byref(scaler),
                                        policy.factor, policy.window, policy.hysteresis, policy.min_scale,
                                        ctypes.byref(f))
    if rc != 0:
        raise MemoryError("oracle step could not allocate its gradient buffer")
    return int(f.value)


def checksum16(buf: np.ndarray) -> tuple[int, int]:
    """(sum of the 16-bit units, sum of (index + 1) * unit), both mod 2^64."""
    b = np.ascontiguousarray(buf)
    if b.nbytes % 2:
        raise ValueError("buffer length must be a whole number of 16-bit units")
    u = b.view(np.uint16).reshape(-1)
    out = np.zeros(2, np.uint64)
    _L().orc_checksum16(_ptr(u), u.size, _ptr(out))
    return int(out[0]), int(out[1])
