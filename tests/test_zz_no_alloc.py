"""The dynamically scaled step that needs no device allocation from its
caller (for programs whose pool allocator owns the device memory, or that
must not call cudaMalloc/cudaFree because those can synchronise the device).

It is called through the C ABI (ctypes on libzero1.so) and must give the same
bits as zero1_step_dynamic with a caller-provided workspace, and as the CPU
oracle's dynamically scaled attempt, on two calls in a row.  This file is
collected last so that a run stopping at the first failure has run every
other test first; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import _lib
from zero_sharded_mixed_zero1_gb300 import synth
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, u16

pytestmark = pytest.mark.gpu


def _c_noalloc(lib):
    fn = lib.zero1_step_dynamic_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(z.Plan), i32, i32, vp, vp, vp, vp, vp, ctypes.POINTER(_lib._AdamWStruct), vp,
                   ctypes.POINTER(_lib._PolicyStruct), vp]
    fn.restype = ctypes.c_int
    return fn


def _state(n, P, dev, seed):
    master = torch.zeros(P, dtype=torch.float32, device=dev)
    master[:n] = synth.normal_f32(n, 0.02, synth.seed_of(seed, 1), dev)
    return master, torch.zeros(P, dtype=torch.float32, device=dev), torch.zeros(P, dtype=torch.float32, device=dev)


def test_no_alloc_step_matches_workspace_step_on_two_calls(cuda_device):
    dev = cuda_device
    lib = z.load()
    fn = _c_noalloc(lib)
    M, n, align = 8, 1_000_003, 128
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    assert P <= lib_max() and P > 0
    policy = z.LossScalePolicy(initial_scale=1024.0, factor=2.0, window=2, hysteresis=1, min_scale=1.0)
    hp = z.AdamW(global_batch=512, step=1)
    a = _state(n, P, dev, 5)
    b = [t.clone() for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    sa, sb = z.new_scaler(dev), z.new_scaler(dev)
    z.zero1_scaler_init(sa, policy, hp)
    z.zero1_scaler_init(sb, policy, hp)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    # the oracle's copy of the state, its scaler and its parameters
    o = [f32(t).copy() for t in a]
    o_params = np.zeros(n, np.uint16)
    o_policy = oracle.LossScalePolicy(initial_scale=policy.initial_scale, factor=policy.factor,
                                      window=policy.window, hysteresis=policy.hysteresis, min_scale=policy.min_scale)
    o_scaler = oracle.Scaler.start(o_policy, hp.step)
    o_hp = oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay,
                        global_batch=hp.global_batch)
    for call in range(2):
        grads = [synth.normal_bf16(n, 1e-3 * 1024, synth.seed_of(6, call, r), dev) for r in range(M)]
        if call == 1:
            grads[2][777] = float("inf")          # second call: an overflow, skipped on the device
        z.zero1_step_dynamic(plan, 0, M, grads, *a, pa, hp, sa, policy, sums)
        gp = (ctypes.c_void_p * M)(*[g.data_ptr() for g in grads])
        rc = fn(ctypes.byref(plan), 0, M, gp, b[0].data_ptr(), b[1].data_ptr(), b[2].data_ptr(), pb.data_ptr(),
                ctypes.byref(hp.c_struct()), sb.data_ptr(), ctypes.byref(policy.c_struct()), stream)
        assert rc == 0, lib.zero1_last_error()
        torch.cuda.synchronize()
        flag = oracle.zero1_dynamic_attempt([u16(g) for g in grads], n, *o, o_params, o_hp, o_scaler, o_policy)
        assert flag == call
        for x, y, want, what in zip(a, b, o, ("master", "m", "v")):
            assert_f32_bits(f32(y), f32(x), f"{what} call {call}")
            assert_f32_bits(f32(y), want, f"{what} call {call} against the oracle")
        assert_bf16_bits(u16(pb), u16(pa), f"params call {call}")
        assert_bf16_bits(u16(pb), o_params, f"params call {call} against the oracle")
        st = z.scaler_state(sb)
        assert z.scaler_state(sa) == st
        assert (st["scale"], st["step"], st["attempts"], st["skipped"]) == \
            (o_scaler.scale, o_scaler.step, o_scaler.attempts, o_scaler.skipped)
    st = z.scaler_state(sb)
    assert st["attempts"] == 2 and st["skipped"] == 1 and st["step"] == 2


def lib_max() -> int:
    return _lib.ZERO1_NOALLOC_MAX_ELEMS


def test_no_alloc_step_rejects_ranges_beyond_its_workspace(cuda_device):
    """A range longer than the built-in array is refused before any launch."""
    dev = cuda_device
    lib = z.load()
    fn = _c_noalloc(lib)
    M = 2
    plan = z.zero1_plan(lib_max() * 2 + 16, M, 8)
    hp = z.AdamW(global_batch=8)
    policy = z.LossScalePolicy()
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    before = z.scaler_state(scaler)
    one = torch.zeros(8, dtype=torch.float32, device=dev)
    gp = (ctypes.c_void_p * M)(*[one.data_ptr()] * M)
    rc = fn(ctypes.byref(plan), 0, M, gp, one.data_ptr(), one.data_ptr(), one.data_ptr(), one.data_ptr(),
            ctypes.byref(hp.c_struct()), scaler.data_ptr(), ctypes.byref(policy.c_struct()), None)
    assert rc == -3
    assert b"exceeds the built-in workspace" in lib.zero1_last_error()
    torch.cuda.synchronize()
    # nothing was launched: the scaler (S, t, counters) is exactly as before
    assert z.scaler_state(scaler) == before
    # the binding refuses tensors shorter than the range before reaching the library
    g16 = torch.zeros(8, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        z.zero1_step_dynamic_noalloc(plan, 0, 1, [g16] * M, one, one, one, g16, hp, scaler, policy)


def test_no_alloc_step_at_its_maximum_range(cuda_device):
    """A range of exactly ZERO1_NOALLOC_MAX_ELEMS elements fills the built-in
    array and is accepted; the result is the workspace step's and the
    oracle's, bit for bit."""
    dev = cuda_device
    lib = z.load()
    fn = _c_noalloc(lib)
    M, n = 2, lib_max() - 5
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    assert P == lib_max()
    policy = z.LossScalePolicy(initial_scale=64.0, factor=2.0, window=1000, hysteresis=2, min_scale=1.0)
    hp = z.AdamW(global_batch=64, step=1)
    a = _state(n, P, dev, 8)
    b = [t.clone() for t in a]
    o = [f32(t).copy() for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    sa, sb = z.new_scaler(dev), z.new_scaler(dev)
    z.zero1_scaler_init(sa, policy, hp)
    z.zero1_scaler_init(sb, policy, hp)
    grads = [synth.normal_bf16(n, 1e-3 * 64, synth.seed_of(9, r), dev) for r in range(M)]
    z.zero1_step_dynamic(plan, 0, M, grads, *a, pa, hp, sa, policy, torch.empty(P, dtype=torch.float32, device=dev))
    gp = (ctypes.c_void_p * M)(*[g.data_ptr() for g in grads])
    rc = fn(ctypes.byref(plan), 0, M, gp, b[0].data_ptr(), b[1].data_ptr(), b[2].data_ptr(), pb.data_ptr(),
            ctypes.byref(hp.c_struct()), sb.data_ptr(), ctypes.byref(policy.c_struct()),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.zero1_last_error()
    torch.cuda.synchronize()
    o_policy = oracle.LossScalePolicy(initial_scale=64.0, factor=2.0, window=1000, hysteresis=2, min_scale=1.0)
    o_sc = oracle.Scaler.start(o_policy, 1)
    o_p = np.zeros(n, np.uint16)
    o_hp = oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay,
                        global_batch=hp.global_batch)
    assert oracle.zero1_dynamic_attempt([u16(g) for g in grads], n, *o, o_p, o_hp, o_sc, o_policy) == 0
    for x, y, want, what in zip(a, b, o, ("master", "m", "v")):
        assert_f32_bits(f32(y), f32(x), what)
        assert_f32_bits(f32(y), want, what + " against the oracle")
    assert_bf16_bits(u16(pb), u16(pa), "params")
    assert_bf16_bits(u16(pb), o_p, "params against the oracle")
    assert z.scaler_state(sb) == z.scaler_state(sa)
