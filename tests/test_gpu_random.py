"""Seeded random configurations against the oracle, bit for bit: replica
count, size, alignment unit, shard sub-range, the element phase of every
buffer (so the vector head, 32- and 16-byte fp32 accesses, the per-element
fallback and the ragged tail all occur), hyperparameters and step, and every entry point that computes the
step (one-shot, prepared, bucketed, shared-memory staged, dynamic, ping-pong
whole and in buckets, and the copy-engine staged step with state or
gradients in pinned host memory, with and without dynamic loss scaling)."""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, oracle_hp, u16

pytestmark = pytest.mark.gpu

ENTRIES = ["fused", "prepared", "bucket", "tma", "dynamic", "pingpong", "pingpong_buckets", "staged_state",
           "staged_grads", "staged_dynamic", "offload", "pingpong_host"]


def _buf(numel, dtype, phase, dev):
    """A tensor of `numel` elements starting `phase` elements into a fresh
    allocation (varies the 16-byte phase of the pointer)."""
    return torch.zeros(numel + 8, dtype=dtype, device=dev)[phase:phase + numel]


def _pinned_like(t, phase):
    """A pinned host copy of t starting `phase` elements into its allocation."""
    h = torch.zeros(t.numel() + 8, dtype=t.dtype).pin_memory()[phase:phase + t.numel()]
    h.copy_(t.cpu())
    return h


def _cuts(rng, L):
    return sorted({0, L, *[int(x) for x in rng.integers(0, L + 1, int(rng.integers(1, 6)))]})


@pytest.mark.parametrize("case", range(168))
def test_random_configuration(cuda_device, case):
    dev = cuda_device
    rng = np.random.default_rng(20_000 + case)
    M = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 11, 16, 31, 64]))
    n = int(np.exp(rng.uniform(0, np.log(400_000))))
    align = int(rng.choice([1, 2, 4, 8, 64, 128, 1024]))
    plan = z.zero1_plan(n, M, align)
    sb = int(rng.integers(0, M))
    se = int(rng.integers(sb + 1, M + 1))
    base, L, nv = plan.shard_range(sb, se)
    entry = ENTRIES[case % len(ENTRIES)]
    # buffer phases: all at the allocation's start (32-byte accesses); fp32
    # buffers 16 bytes in (the vector body moves fp32 in 16-byte accesses);
    # or every buffer at a random element phase (mostly the per-element path)
    mode = str(rng.choice(["same", "state16", "mixed"], p=[0.45, 0.2, 0.35]))
    if mode == "mixed":
        ph = ph32 = lambda: int(rng.integers(0, 8))
    else:
        ph = lambda: 0
        ph32 = (lambda: 4) if mode == "state16" else ph
    g_np = [(rng.standard_normal(nv) * 10 ** rng.uniform(-4, -1)).astype(np.float32) for _ in range(M)]
    g_np = [oracle.f32_to_bf16(x) for x in g_np]
    grads = []
    for x in g_np:
        t = _buf(nv, torch.bfloat16, ph(), dev)
        t.copy_(torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16))
        grads.append(t)
    w_np = np.zeros(L, np.float32)
    w_np[:nv] = rng.standard_normal(nv) * 0.02
    m_np = (rng.standard_normal(L) * 1e-4).astype(np.float32)
    v_np = (rng.random(L) * 1e-7).astype(np.float32)
    m_np[nv:] = 0
    v_np[nv:] = 0
    state = []
    for a in (w_np, m_np, v_np):
        t = _buf(L, torch.float32, ph32(), dev)
        t.copy_(torch.from_numpy(a))
        state.append(t)
    params = _buf(nv, torch.bfloat16, ph(), dev)
    S = float(2 ** int(rng.integers(0, 17)))
    hp = z.AdamW(lr=float(10 ** rng.uniform(-5, -2)), beta1=float(rng.uniform(0, 0.99)),
                 beta2=float(rng.uniform(0.5, 0.9999)), eps=float(10 ** rng.uniform(-10, -3)),
                 weight_decay=float(rng.uniform(0, 0.3)), loss_scale=S,
                 global_batch=int(M * rng.integers(1, 64)), step=int(rng.integers(1, 2000)))
    if entry == "fused":
        z.zero1_reduce_scatter_adamw_allgather(plan, sb, se, grads, *state, params, hp)
    elif entry == "prepared":
        z.FusedStep(plan, sb, se, grads, *state, params)(hp)
    elif entry == "tma":
        z.zero1_step_tma(plan, sb, se, grads, *state, params, hp)
    elif entry == "dynamic":
        policy = z.LossScalePolicy(initial_scale=S, window=1000, hysteresis=2)
        scaler = z.new_scaler(dev)
        z.zero1_scaler_init(scaler, policy, hp)
        sums = _buf(L, torch.float32, ph32(), dev)
        z.zero1_step_dynamic(plan, sb, se, grads, *state, params, hp, scaler, policy, sums)
    elif entry == "offload":
        # master/m/v in pinned host memory, read and written by the offload kernel
        state = [_pinned_like(t, ph32()) for t in state]
        z.zero1_reduce_scatter_adamw_allgather(plan, sb, se, grads, *state, params, hp)
    elif entry in ("pingpong", "pingpong_buckets", "pingpong_host"):
        policy = z.LossScalePolicy(initial_scale=S, window=1000, hysteresis=2)
        scaler = z.new_scaler(dev)
        z.zero1_scaler_init(scaler, policy, hp)
        if entry == "pingpong_host":
            # both copies in pinned host memory, at one phase
            p32 = ph32()
            state = [_pinned_like(t, p32) for t in state]
            pairs = [[t, _pinned_like(torch.full((L,), float("nan")), p32)] for t in state]
        else:
            pairs = [[t, _buf(L, torch.float32, ph32(), dev).fill_(float("nan"))] for t in state]
        if entry in ("pingpong", "pingpong_host"):
            z.zero1_step_dynamic_pingpong(plan, sb, se, grads, *pairs, params, hp, scaler, policy)
        else:
            attempt = z.PingPongBuckets(plan, sb, se, *pairs, params, scaler, policy)
            cuts = _cuts(rng, L)
            for i in rng.permutation(len(cuts) - 1):
                e0, e1 = cuts[i], cuts[i + 1]
                k = max(0, min(nv, e1) - e0)
                attempt.bucket(e0, e1, [g[e0:e0 + k] for g in grads], hp)
            attempt.finish(hp)
        state = list(z.current_state(scaler, *pairs))
    elif entry in ("staged_state", "staged_dynamic"):
        state = [_pinned_like(t, ph32()) for t in state]
        step = z.HostStreamedStep(plan, sb, se, grads, *state, params, chunk_elems=int(rng.integers(1, 6000)))
        if entry == "staged_dynamic":
            policy = z.LossScalePolicy(initial_scale=S, window=1000, hysteresis=2)
            scaler = z.new_scaler(dev)
            z.zero1_scaler_init(scaler, policy, hp)
            step.dynamic(hp, scaler, policy)
        else:
            step(hp)
    elif entry == "staged_grads":
        grads = [_pinned_like(g, ph()) for g in grads]
        host_p = _pinned_like(params, ph())
        z.HostStreamedStep(plan, sb, se, grads, *state, params, chunk_elems=int(rng.integers(1, 6000)),
                           params_host=host_p)(hp)
        torch.cuda.synchronize()
        assert_bf16_bits(u16(host_p), u16(params), f"case {case}: params copied to host")
    else:  # buckets over [base, base + L) in global element coordinates
        cuts = _cuts(rng, L)
        for e0, e1 in zip(cuts[:-1], cuts[1:]):
            k = max(0, min(nv, e1) - e0)
            z.zero1_step_bucket(plan, base + e0, base + e1, [g[e0:e0 + k] for g in grads],
                                *[t[e0:] for t in state], params[e0:] if e0 < nv else params[:0], hp)
    torch.cuda.synchronize()
    want_p = np.zeros(nv, np.uint16)
    oracle.zero1_step(g_np, nv, w_np, m_np, v_np, want_p, oracle_hp(hp))
    what = f"case {case}: {entry} M={M} n={n} align={align} shards=[{sb},{se}) phases={mode}"
    assert_f32_bits(f32(state[0]), w_np, "master " + what)
    assert_f32_bits(f32(state[1]), m_np, "m " + what)
    assert_f32_bits(f32(state[2]), v_np, "v " + what)
    assert_bf16_bits(u16(params), want_p, "params " + what)
    assert z.zero1_device_status() == 0
