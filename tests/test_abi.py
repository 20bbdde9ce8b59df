"""The C-ABI library without a GPU: it loads, exports every function that
include/zero1.h declares, its host-only plan logic equals the oracle's, and
every invalid argument is rejected before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import build as zbuild
from zero_sharded_mixed_zero1_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    zbuild.build()
    return z.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "zero1.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^(?:int|const char \*)\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for required in ["zero1_plan", "zero1_reduce_scatter_adamw_allgather", "dp_allreduce",
                     "zero1_overflow_check"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in zero1.h but not exported"
    assert lib.zero1_abi_version() == 3


@pytest.mark.parametrize("n", [1, 2, 7, 8, 9, 1000, 4099, 10**6 + 3, 1_300_000_000, 7_500_000_000])
def test_plan_equals_oracle(lib, n):
    for M in [1, 2, 3, 4, 5, 7, 8, 16, 63, 64]:
        for a in [1, 8, 128, 1024]:
            p = z.zero1_plan(n, M, a)
            assert (p.padded_n, p.shard) == oracle.plan(n, M, a)
            assert z.zero1_plan_memory(p) == oracle.memory(n, p.shard)


def test_segments_equal_oracle(lib):
    rng = np.random.default_rng(3)
    cases = [list(W.LLAMA4.tensor_numels)]
    for _ in range(40):
        cases.append([int(x) for x in rng.integers(1, 50, int(rng.integers(1, 8)))])
    for numels in cases:
        n = sum(numels)
        for M in [1, 3, 8]:
            p = z.zero1_plan(n, M, int(rng.choice([1, 8, 128])), tensor_numels=numels)
            assert p.n_tensors == len(numels)
            for i in range(M):
                want = oracle.segments(numels, p.shard, i)
                assert z.zero1_plan_segments(p, numels, i) == [(k, toff, ln) for k, toff, _, ln in want]
                # the pieces tile the shard from its first element: the
                # oracle's offsets inside the shard are the running lengths
                assert [soff for _, _, soff, _ in want] == list(np.cumsum([0] + [ln for *_, ln in want])[:-1])


def test_plan_tensor_list_validation(lib):
    """The tensor list given to zero1_plan must sum to n; segments need it."""
    p = z.Plan()
    nums = (ctypes.c_int64 * 3)(5, 7, 11)
    assert lib.zero1_plan(23, 2, 4, nums, 3, ctypes.byref(p)) == 0 and p.n_tensors == 3
    assert lib.zero1_plan(24, 2, 4, nums, 3, ctypes.byref(p)) == -1     # sizes sum to 23, not 24
    assert lib.zero1_plan(23, 2, 4, nums, 0, ctypes.byref(p)) == -1     # a list needs n_tensors >= 1
    assert lib.zero1_plan(23, 2, 4, None, 2, ctypes.byref(p)) == -1     # no list: n_tensors must be 0
    neg = (ctypes.c_int64 * 3)(30, -7, 0)
    assert lib.zero1_plan(23, 2, 4, neg, 3, ctypes.byref(p)) == -1
    flat = z.zero1_plan(23, 2, 4)
    assert flat.n_tensors == 0
    with pytest.raises(z.Zero1Error):
        z.zero1_plan_segments(flat, [5, 7, 11], 0)                    # built without the list


# --------------------------------------------------------- validation ------
# Fake device addresses: every call below must fail validation on the host,
# before any CUDA call.  Skipped where a GPU exists (the GPU tests cover the
# real paths there).

no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="host-validation test uses fake pointers")

A = 0x100000  # 16-byte aligned fake address


def _ptr_array(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def _hp(**kw):
    base = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, loss_scale=1.0,
                global_batch=8, step=1)
    base.update(kw)
    return z.AdamW(**base).c_struct()


def _fused(lib, plan, sb=0, se=None, grads=None, master=A, m=A + 4096, v=A + 8192, params=A + 12288,
           hp=None, flag=None, skip=0):
    se = plan.M if se is None else se
    grads = _ptr_array([A + 65536 * (r + 1) for r in range(plan.M)]) if grads is None else grads
    return lib.zero1_reduce_scatter_adamw_allgather(ctypes.byref(plan), sb, se, grads, master, m, v, params,
                                                    ctypes.byref(hp or _hp()), flag, skip, None)


@no_gpu
def test_plan_rejects_bad_arguments(lib):
    p = z.Plan()
    assert lib.zero1_plan(0, 4, 1, None, 0, ctypes.byref(p)) == -1
    assert lib.zero1_plan(10, 0, 1, None, 0, ctypes.byref(p)) == -1
    assert lib.zero1_plan(10, 4, 0, None, 0, ctypes.byref(p)) == -1
    assert lib.zero1_plan(10, 65, 1, None, 0, ctypes.byref(p)) == -3
    assert lib.zero1_plan(2**63 - 6, 64, 1024, None, 0, ctypes.byref(p)) == -3  # padding overflows int64
    assert lib.zero1_plan(10, 4, 1, None, 0, None) == -1


@no_gpu
def test_fused_step_rejects_bad_arguments(lib):
    plan = z.zero1_plan(1000, 4, 8)
    assert _fused(lib, plan, sb=0, se=5) == -1            # range beyond M
    assert _fused(lib, plan, sb=2, se=2) == -1            # empty range
    assert _fused(lib, plan, sb=-1, se=2) == -1
    assert _fused(lib, plan, grads=_ptr_array([A, A, None, A])) == -1
    assert _fused(lib, plan, master=None) == -1
    # buffers the step writes must not overlap each other or the gradients
    assert _fused(lib, plan, m=A) == -1                             # m is master
    assert _fused(lib, plan, v=A + 4096 + 2048) == -1               # v starts inside m
    assert _fused(lib, plan, params=A + 8192 + 4000) == -1          # params runs into v's end
    assert _fused(lib, plan, grads=_ptr_array([A + 65536] * 3 + [A + 12288 + 1000])) == -1  # a gradient inside params
    assert "overlap" in lib.zero1_last_error().decode()
    # gradient buffers may alias one another, and neighbours may touch: this
    # call passes the host checks (it fails later only because the addresses
    # are fake, when the pointer kind is looked up or the launch is made)
    assert _fused(lib, plan, grads=_ptr_array([A + 65536] * 4)) in (-4, 0)
    assert _fused(lib, plan, master=A + 2) == -2          # fp32 not 4-byte aligned
    assert _fused(lib, plan, params=A + 1) == -2          # bf16 odd address
    assert _fused(lib, plan, grads=_ptr_array([A, A + 3, A, A])) == -2
    assert _fused(lib, plan, hp=_hp(global_batch=2)) == -1  # B < M
    assert _fused(lib, plan, hp=_hp(step=0)) == -1
    assert _fused(lib, plan, hp=_hp(loss_scale=0.0)) == -1
    assert _fused(lib, plan, hp=_hp(beta1=1.0)) == -1
    assert _fused(lib, plan, hp=_hp(eps=-1.0)) == -1
    assert _fused(lib, plan, hp=_hp(lr=float("nan"))) == -1
    assert _fused(lib, plan, flag=None, skip=1) == -1     # skip needs a flag
    assert _fused(lib, plan, flag=A + 2, skip=0) == -2
    bad = z.zero1_plan(1000, 4, 8)
    bad.shard += 1
    assert _fused(lib, bad) == -1                         # plan not built by zero1_plan
    assert b"inconsistent" in lib.zero1_last_error()


@no_gpu
def test_other_entry_points_reject_bad_arguments(lib):
    plan = z.zero1_plan(1000, 2, 8)
    g = _ptr_array([A, A + 4096])
    o = _ptr_array([A + 8192, A + 16384])
    P = ctypes.byref(plan)
    assert lib.dp_allreduce(P, g, o, 1.0, 7, None) == -1                      # unknown dtype
    assert lib.dp_allreduce(P, g, o, float("inf"), 0, None) == -1
    assert lib.dp_allreduce(P, g, _ptr_array([A + 8193, A]), 1.0, 0, None) == -2
    assert lib.dp_allreduce(P, g, _ptr_array([A, A + 8192]), 1.0, 1, None) == -1  # fp32 out overlaps input
    assert lib.zero1_overflow_check(P, 0, 2, g, None, None) == -1
    assert lib.zero1_overflow_check(P, 0, 3, g, A, None) == -1
    assert lib.zero1_overflow_check(P, 0, 2, g, A + 1, None) == -2
    assert lib.zero1_reduce_scatter(P, 0, 2, g, 1.0, 5, A, None, None) == -1
    assert lib.zero1_reduce_scatter(P, 0, 2, g, 1.0, 1, A + 2, None, None) == -2
    assert lib.zero1_adamw_update(P, 0, 2, None, A, A, A, ctypes.byref(_hp()), None) == -1
    assert lib.zero1_adamw_update(P, 0, 2, A, A + 8192, A + 8192, A + 16384, ctypes.byref(_hp()), None) == -1
    assert lib.zero1_reduce_scatter(P, 0, 2, g, 1.0, 1, A + 2048, None, None) == -1     # out inside grads[0]
    assert lib.zero1_all_gather(P, 0, 2, A, A + 2048, None) == -1                      # params inside master
    assert lib.zero1_all_gather_shards(P, A, _ptr_array([A + 1024, A + 65536]), None) == -1
    assert lib.zero1_all_gather(P, 1, 1, A, A, None) == -1
    assert lib.zero1_all_gather_shards(P, A + 1, o, None) == -2
    assert lib.zero1_strerror(-2) == b"misaligned device pointer"


def test_staged_handle_rejects_bad_arguments(lib):
    """The staged-step handle validates the plan, range, stage bits and chunk
    size before any CUDA call; a NULL handle is rejected and destroying NULL
    is a no-op."""
    plan = z.zero1_plan(1000, 4, 8)
    P = ctypes.byref(plan)
    h = ctypes.c_void_p()
    assert lib.zero1_staged_create(P, 0, 4, 0, 1024, ctypes.byref(h)) == -1        # nothing staged
    assert lib.zero1_staged_create(P, 0, 4, 8, 1024, ctypes.byref(h)) == -1        # tracing alone stages nothing
    assert lib.zero1_staged_create(P, 0, 4, 16 | 2, 1024, ctypes.byref(h)) == -1   # unknown bit
    assert lib.zero1_staged_create(P, 0, 4, z.ZERO1_STAGE_STATE, 0, ctypes.byref(h)) == -1
    assert lib.zero1_staged_create(P, 2, 2, z.ZERO1_STAGE_STATE, 64, ctypes.byref(h)) == -1   # empty range
    assert lib.zero1_staged_create(P, 0, 5, z.ZERO1_STAGE_STATE, 64, ctypes.byref(h)) == -1
    assert lib.zero1_staged_create(P, 0, 4, z.ZERO1_STAGE_STATE, 64, None) == -1
    assert h.value is None
    assert lib.zero1_staged_step(None, None, None, None, None, None, None, ctypes.byref(_hp()), None, None) == -1
    assert lib.zero1_staged_destroy(None) == 0
    cnt = ctypes.c_int32()
    assert lib.zero1_staged_timeline(None, None, 0, ctypes.byref(cnt)) == -1
    pol = ctypes.byref(z.LossScalePolicy().c_struct())
    assert lib.zero1_staged_step_dynamic(None, None, None, None, None, None, None, ctypes.byref(_hp()), None, pol,
                                         None) == -1                    # no scaler
    assert lib.zero1_staged_step_dynamic(None, None, None, None, None, None, None, ctypes.byref(_hp()), A, pol,
                                         None) == -1                    # no handle
    assert lib.zero1_bounded_wait_selftest(0, A, None) == -1          # limit out of range
    assert lib.zero1_bounded_wait_selftest(100, None, None) == -1
    assert lib.zero1_bounded_wait_selftest(100, A + 2, None) == -2    # misaligned result word


@no_gpu
def test_pingpong_entries_reject_bad_arguments(lib):
    """The ping-pong step, bucket and finish validate the two state copies,
    the policy, the range and the hyperparameters before any CUDA call."""
    plan = z.zero1_plan(1000, 2, 8)
    P = ctypes.byref(plan)
    g = _ptr_array([A + 65536, A + 131072])
    two = lambda a, b: _ptr_array([a, b])
    pol = ctypes.byref(z.LossScalePolicy().c_struct())
    hp = ctypes.byref(_hp(global_batch=64))
    sc = A + (1 << 22)
    w, m, v = two(A, A + 8192), two(A + 16384, A + 24576), two(A + 32768, A + 40960)
    step = lambda *a: lib.zero1_step_dynamic_pingpong(P, 0, 2, g, *a)
    assert step(two(A, A), m, v, A + 49152, hp, sc, pol, None) == -1             # one buffer for both copies
    assert step(two(A, A + 2048), m, v, A + 49152, hp, sc, pol, None) == -1      # copy 1 inside copy 0
    assert step(w, m, v, A + 65536 + 1024, hp, sc, pol, None) == -1             # params inside grads[0]
    assert step(w, m, v, A + 49152, hp, A + 40960 + 512, pol, None) == -1       # scaler inside v[1]
    assert b"overlap" in lib.zero1_last_error()
    dyn = lambda sums, mm=A + 16384: lib.zero1_step_dynamic(P, 0, 2, g, A, mm, A + 32768, A + 49152, hp, sc, pol,
                                                            sums, None)
    assert dyn(A) == -1                                                         # sums is master
    assert dyn(A + 24576, mm=A + 2048) == -1                                    # m inside master
    assert step(two(A, A + 8194), m, v, A + 49152, hp, sc, pol, None) == -2      # copy 1 misaligned
    assert step(None, m, v, A + 49152, hp, sc, pol, None) == -1
    assert step(w, m, v, A + 49152, hp, sc + 4, pol, None) == -2                # scaler not 8-byte aligned
    bad_pol = ctypes.byref(z.LossScalePolicy(factor=1.0).c_struct())
    assert step(w, m, v, A + 49152, hp, sc, bad_pol, None) == -1
    assert lib.zero1_pingpong_bucket(P, 500, 2000, g, w, m, v, A + 49152, hp, sc, None) == -1   # past P
    assert lib.zero1_pingpong_bucket(P, 10, 10, g, w, m, v, A + 49152, hp, sc, None) == -1     # empty
    bad_hp = ctypes.byref(_hp(beta1=1.0, global_batch=64))
    assert lib.zero1_pingpong_finish(P, 0, 2, w, A + 49152, bad_hp, sc, pol, None) == -1
    assert lib.zero1_pingpong_finish(P, 0, 2, two(A, A), A + 49152, hp, sc, pol, None) == -1
    assert lib.zero1_pingpong_finish(P, 0, 3, w, A + 49152, hp, sc, pol, None) == -1         # bad range


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import zero_sharded_mixed_zero1_gb300._lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        L.load()


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "zero1.h"

int main(void)
{
    zero1_plan_t p;
    int64_t naive = 0, z1 = 0;
    int64_t numels[3] = {5, 7, 11};
    int64_t t[4], toff[4], len[4];
    int32_t count = 0;
    if (zero1_plan(1300000000LL, 8, 128, NULL, 0, &p) != ZERO1_OK) return 1;
    if (p.padded_n != 1300000768LL || p.shard != 162500096LL || p.n_tensors != 0) return 2;
    if (zero1_plan_memory(&p, &naive, &z1) != ZERO1_OK || naive != 16LL * 1300000000LL) return 3;
    if (zero1_plan(23, 2, 4, numels, 3, &p) != ZERO1_OK || p.n_tensors != 3) return 4;
    if (zero1_plan_segments(&p, numels, 1, t, toff, len, 4, &count) != ZERO1_OK) return 5;
    printf("%lld %lld %d", (long long)p.padded_n, (long long)p.shard, count);
    for (int i = 0; i < count; ++i) printf(" (%lld,%lld,%lld)", (long long)t[i], (long long)toff[i], (long long)len[i]);
    if (zero1_plan(10, 65, 1, NULL, 0, &p) != ZERO1_ERANGE) return 6;
    if (strcmp(zero1_strerror(ZERO1_ERANGE), "size or replica count out of the supported range") != 0) return 7;
    printf(" | %s\n", zero1_last_error());
    return zero1_abi_version() == 3 ? 0 : 8;
}
"""


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/zero1.h compiles as C99 and a C program links libzero1.so and
    calls its host-only functions."""
    import subprocess
    src = tmp_path / "use_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(zbuild.LIB)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-l:libzero1.so", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    head, _, err = r.stdout.partition(" | ")
    P, s, count, *segs = head.split(" ")
    assert (int(P), int(s)) == oracle.plan(23, 2, 4)
    want = oracle.segments([5, 7, 11], int(s), 1)
    assert int(count) == len(want) and segs == [f"({a},{b},{d})" for a, b, c, d in want]
    assert "M = 65" in err
