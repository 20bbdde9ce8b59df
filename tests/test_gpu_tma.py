"""The shared-memory staged form of the fused step (bulk copies into a ring
of stages, mbarrier-counted): bit for bit the fused step and the oracle,
every wait finished in time (device status 0)."""
import numpy as np
import pytest
import torch

import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, oracle_hp, u16
from test_gpu_parity import make_grads, make_state, oracle_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [1, 2, 4, 7, 8, 9, 16, 64])
@pytest.mark.parametrize("n,align", [(1, 1), (9, 1), (1024 * 5 + 24, 8), (100_003, 1), (300_000, 128)])
def test_staged_step_matches_oracle(cuda_device, M, n, align):
    dev = cuda_device
    z.zero1_device_status(clear=True)
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    master, m, v = make_state(n, P, 700 + M, dev, nonzero_moments=True)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    o = [f32(master), f32(m), f32(v)]
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    for t in (1, 2):
        hp = z.AdamW(global_batch=max(M, 32), step=t)
        grads = make_grads(M, n, 1e-2, 710 + M, t, dev)
        if t == 1:
            z.zero1_step_tma(plan, 0, M, grads, master, m, v, params, hp, flag)
        else:         # shard by shard: per-element heads where shard sizes are odd
            for i in range(M):
                base, L, nv = plan.shard_range(i, i + 1)
                z.zero1_step_tma(plan, i, i + 1, [g[base:] if base < n else g[:0] for g in grads],
                                 master[base:base + L], m[base:base + L], v[base:base + L],
                                 params[base:] if base < n else params[:0], hp, flag)
        torch.cuda.synchronize()
        want = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp))
        assert_f32_bits(f32(master), o[0], f"master t={t}")
        assert_f32_bits(f32(m), o[1], f"m t={t}")
        assert_f32_bits(f32(v), o[2], f"v t={t}")
        assert_bf16_bits(u16(params), want, f"params t={t}")
    assert int(flag.item()) == 0
    assert z.zero1_device_status() == 0


@pytest.mark.parametrize("M", [8, 64])
def test_staged_step_equals_fused_step_at_size(cuda_device, M):
    dev = cuda_device
    n = 124_439_808 if M == 8 else 20_000_003
    plan = z.zero1_plan(n, M, 1)
    a = make_state(n, plan.padded_n, 720, dev, nonzero_moments=True)
    b = [t.clone() for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    for t in (1, 2):
        grads = make_grads(M, n, 1e-3, 721, t, dev)
        hp = z.AdamW(global_batch=512, step=t)
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *a, pa, hp)
        z.zero1_step_tma(plan, 0, M, grads, *b, pb, hp)
        del grads
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))
    assert z.zero1_device_status() == 0
    del a, b, pa, pb
    torch.cuda.empty_cache()


def test_staged_step_skips_and_rejects_host_memory(cuda_device):
    dev = cuda_device
    M, n = 4, 40_000
    plan = z.zero1_plan(n, M, 8)
    grads = make_grads(M, n, 1e-3, 730, 1, dev)
    grads[1][123] = float("inf")
    master, m, v = make_state(n, plan.padded_n, 731, dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    snap = [x.clone() for x in (master, m, v)]
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    z.zero1_overflow_check(plan, 0, M, grads, flag)
    z.zero1_step_tma(plan, 0, M, grads, master, m, v, params, z.AdamW(global_batch=64), flag, skip_if_flag=True)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    for x, y in zip((master, m, v), snap):
        assert torch.equal(x, y)
    with pytest.raises(z.Zero1Error):
        z.zero1_step_tma(plan, 0, M, [g.cpu().pin_memory() for g in grads], master, m, v, params,
                         z.AdamW(global_batch=64))


@pytest.mark.parametrize("limit_us", [200, 5000])
def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable(cuda_device, limit_us):
    """Failure detection without a fault: a wait that can never complete (a
    barrier that expects two arrivals and gets one) gives up after its limit,
    reports through the device status word and returns; the context then
    runs the staged step correctly with a clean status."""
    import time
    dev = cuda_device
    assert z.zero1_device_status(clear=True) in (0, 1)
    gave_up = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    z.zero1_bounded_wait_selftest(limit_us, gave_up)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(gave_up.item()) == 1
    assert elapsed >= limit_us * 1e-6
    assert z.zero1_device_status(clear=True) == 1
    assert z.zero1_device_status(clear=True) == 0
    M, n = 4, 50_003
    plan = z.zero1_plan(n, M, 8)
    a = make_state(n, plan.padded_n, 11, dev, nonzero_moments=True)
    b = [t.clone() for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grads = make_grads(M, n, 1e-2, 12, 1, dev)
    hp = z.AdamW(global_batch=64)
    z.zero1_step_tma(plan, 0, M, grads, *a, pa, hp)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *b, pb, hp)
    torch.cuda.synchronize()
    for x, y, what in zip(a, b, ("master", "m", "v")):
        assert_f32_bits(f32(x), f32(y), what)
    assert_bf16_bits(u16(pa), u16(pb), "params")
    assert z.zero1_device_status(clear=True) == 0


def test_bounded_wait_selftest_validates(cuda_device):
    gave_up = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for bad in (0, 1_000_001):
        with pytest.raises(z.Zero1Error):
            z.zero1_bounded_wait_selftest(bad, gave_up)
