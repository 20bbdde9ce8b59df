"""Launch shapes the library picks: each kernel's grid is one resident wave
sized from that kernel's own occupancy, whatever ran before it in the
process, and the vector body moves fp32 in 32-byte accesses whenever the
buffers allow it.  (Results are checked bit for bit elsewhere; this checks
the shapes that the measured rooflines rely on.)"""
import pytest
import torch

import zero_sharded_mixed_zero1_gb300 as z
from test_gpu_parity import make_grads, make_state

pytestmark = pytest.mark.gpu


def _sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def _fused(dev, n, M, state_offset=0):
    plan = z.zero1_plan(n, M, 1)
    P = plan.padded_n
    grads = make_grads(M, n, 1e-3, 7, 1, dev)
    master, m, v = (torch.cat([torch.zeros(state_offset, device=dev), t])[state_offset:]
                    for t in make_state(n, P, 8, dev))
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, z.AdamW(global_batch=64))
    torch.cuda.synchronize()
    return z.debug_last_launch()


def test_each_kernel_gets_its_own_occupancy(cuda_device):
    """The fused kernel on a small range (its full occupancy, blocks of 256)
    and on a large one (the launch shape of its table: five blocks of 128
    per SM at M = 8) keep their own grids whatever ran before."""
    dev = cuda_device
    sms = _sms()
    big, small = 8 << 20, 1 << 16            # 8M elements: the table's shape; 64K: full occupancy
    first_big = _fused(dev, big, 8)
    first_small = _fused(dev, small, 8)
    again_big = _fused(dev, big, 8)
    assert "k_fused_step" in first_big["kernel"] and "k_fused_step" in first_small["kernel"]
    assert first_big == again_big
    assert (first_big["blocks_per_sm"], first_big["block"]) == (5, 128)
    assert first_big["grid"] == sms * 5
    assert first_small["block"] == 256 and first_small["blocks_per_sm"] >= 4
    # the small range needs fewer blocks than a wave: one vector of 8 per thread
    assert first_small["grid"] == min(sms * first_small["blocks_per_sm"], -(-small // 8 // 256))


def test_large_range_shapes_per_replica_count(cuda_device):
    """On a large range the fused step runs 20 warps per SM (five blocks of
    128) for M = 1 and 6..8, 18 (three blocks of 192) for M = 2, 3 and 16 (two
    blocks of 256) for M = 4, 5, the measured faster shape for each M; the
    grid is one wave."""
    dev = cuda_device
    sms = _sms()
    big = 8 << 20
    for M, per_sm, block in ((1, 5, 128), (2, 3, 192), (3, 3, 192), (4, 2, 256), (5, 2, 256), (6, 5, 128),
                             (8, 5, 128)):
        d = _fused(dev, big, M)
        assert "k_fused_step" in d["kernel"] and "grouped" not in d["kernel"], (M, d)
        assert (d["blocks_per_sm"], d["block"]) == (per_sm, block) and d["grid"] == per_sm * sms, (M, d)
    # M > 8: the grouped kernel at its occupancy
    d = _fused(dev, 1 << 20, 9)
    assert "k_fused_step_grouped" in d["kernel"] and d["block"] == 256, d


def test_allreduce_and_update_shapes(cuda_device):
    """All-reduce grids follow their per-M table (one vector per thread, the
    blocks per SM and block size of the table); the dynamic step's update from
    the sums runs one vector per thread at two blocks per SM."""
    dev = cuda_device
    sms = _sms()
    n = 4 << 20
    for M, per_sm, block, one_vector in ((1, 3, 256, True), (2, 5, 128, True), (3, 2, 256, True),
                                         (4, 5, 128, True), (5, 3, 192, True), (6, 2, 256, True),
                                         (8, 3, 128, True)):
        plan = z.zero1_plan(n, M, 1)
        grads = make_grads(M, n, 1e-3, 5, 1, dev)
        outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
        z.dp_allreduce(plan, grads, outs, 1.0)
        d = z.debug_last_launch()
        assert "k_allreduce" in d["kernel"], d
        # the depth is the kernel's last template argument (mangled: ...ELi<D>EEE)
        assert ("Li1EEE" if one_vector else "Li2EEE") in d["kernel"], (M, d)
        assert (d["blocks_per_sm"], d["block"]) == (per_sm, block) and d["grid"] == per_sm * sms, (M, d)
    M = 8
    plan = z.zero1_plan(n, M, 1)
    P = plan.padded_n
    grads = make_grads(M, n, 1e-3, 6, 1, dev)
    master, m, v = make_state(n, P, 9, dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    policy = z.LossScalePolicy()
    hp = z.AdamW(global_batch=64)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    z.zero1_step_dynamic(plan, 0, M, grads, master, m, v, params, hp, scaler, policy, sums)
    torch.cuda.synchronize()
    d = z.debug_last_launch()
    assert "k_apply_sums" in d["kernel"] and d["blocks_per_sm"] == 2 and d["grid"] == 2 * sms, d
    assert "k_apply_sumsILi1E" in d["kernel"], d
    # state in host memory: the two-deep update at its occupancy
    host_state = [t.cpu().pin_memory() for t in (master, m, v)]
    z.zero1_step_dynamic(plan, 0, M, grads, *host_state, params, hp, scaler, policy, sums)
    torch.cuda.synchronize()
    d = z.debug_last_launch()
    assert "k_apply_sumsILi2E" in d["kernel"] and d["grid"] == d["blocks_per_sm"] * sms, d
    # the unfused update: one vector per thread, three blocks of 192 per SM
    z.zero1_adamw_update(plan, 0, M, sums, master, m, v, hp)
    d = z.debug_last_launch()
    assert "k_adamw" in d["kernel"] and "Li1E" in d["kernel"] and (d["grid"], d["block"]) == (3 * sms, 192), d
    # the overflow check at M = 8: three blocks per SM
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    z.zero1_overflow_check(plan, 0, M, grads, flag)
    d = z.debug_last_launch()
    assert "k_overflow" in d["kernel"] and d["blocks_per_sm"] == 3 and d["grid"] == 3 * sms, d
    # the ping-pong step ends with the parameter restore at four blocks per SM
    pairs = [[x, x.clone()] for x in (master, m, v)]
    z.zero1_step_dynamic_pingpong(plan, 0, M, grads, *pairs, params, hp, scaler, policy)
    torch.cuda.synchronize()
    d = z.debug_last_launch()
    assert "k_restore_params" in d["kernel"] and d["blocks_per_sm"] == 4 and d["grid"] == 4 * sms, d


def test_pingpong_shape_depends_on_where_the_state_lives(cuda_device):
    """The ping-pong kernel runs the HBM table's shape (one vector per thread,
    five blocks of 128 per SM at M = 8) on device state and two vectors in
    flight per thread at its occupancy when both copies are in host memory."""
    dev = cuda_device
    sms = _sms()
    M, n = 8, 4 << 20
    plan = z.zero1_plan(n, M, 1)
    P = plan.padded_n
    grads = make_grads(M, n, 1e-3, 12, 1, dev)
    policy = z.LossScalePolicy()
    hp = z.AdamW(global_batch=64)
    for on_host in (False, True):
        state = make_state(n, P, 13, dev)
        if on_host:
            state = [t.cpu().pin_memory() for t in state]
        pairs = [[x, torch.empty(x.shape, dtype=x.dtype, pin_memory=True) if on_host else torch.empty_like(x)]
                 for x in state]
        params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
        scaler = z.new_scaler(dev)
        z.zero1_scaler_init(scaler, policy, hp)
        z.PingPongBuckets(plan, 0, M, *pairs, params, scaler, policy).bucket(0, P, grads, hp)
        torch.cuda.synchronize()
        d = z.debug_last_launch()
        assert "k_fused_step_pingpong" in d["kernel"], d
        if on_host:
            assert "Li2EEE" in d["kernel"] and d["block"] == 256 and d["grid"] == d["blocks_per_sm"] * sms, d
        else:
            assert "Li1EEE" in d["kernel"] and (d["blocks_per_sm"], d["block"]) == (5, 128), d


def test_grouped_allreduce_runs_two_blocks_per_sm(cuda_device):
    """M > 8: the all-reduce's grouped loop runs at two blocks per SM (below
    its occupancy of three, measured faster)."""
    dev = cuda_device
    sms = _sms()
    n, M = 1 << 20, 16
    plan = z.zero1_plan(n, M, 1)
    grads = make_grads(M, n, 1e-3, 8, 1, dev)
    outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    z.dp_allreduce(plan, grads, outs, 1.0)
    d = z.debug_last_launch()
    assert "k_allreduce" in d["kernel"] and d["blocks_per_sm"] == 2 and d["grid"] == 2 * sms, d


def test_fp32_arrays_move_in_32_byte_accesses_when_aligned(cuda_device):
    """torch's allocations are 32-byte aligned: the vector body uses 32-byte
    fp32 accesses; state starting 16 bytes past a 32-byte boundary falls back
    to 16-byte accesses (same bits, checked by the parity tests)."""
    dev = cuda_device
    assert _fused(dev, 1 << 20, 4)["w32"] is True
    # master/m/v shifted by 4 floats (16 bytes) against the gradients
    assert _fused(dev, 1 << 20, 4, state_offset=4)["w32"] is False
