"""GPU parity of the dynamically scaled step ("五维并行实战" 4.2 fp16 block):
every attempt's master/m/v/params bit for bit against the oracle's attempt,
and the device-resident scaler (S, t, counters, derived constants) against
the oracle's scaler and constants."""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth
from zero_sharded_mixed_zero1_gb300 import workloads as W
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, u16
from test_gpu_parity import make_state

pytestmark = pytest.mark.gpu


def oracle_policy(p: z.LossScalePolicy) -> oracle.LossScalePolicy:
    return oracle.LossScalePolicy(initial_scale=p.initial_scale, factor=p.factor, window=p.window,
                                  hysteresis=p.hysteresis, min_scale=p.min_scale)


def check_scaler(dev_state: dict, sc: oracle.Scaler, hp: z.AdamW):
    assert dev_state["scale"] == sc.scale
    assert dev_state["step"] == sc.step
    assert dev_state["attempts"] == sc.attempts and dev_state["skipped"] == sc.skipped
    assert dev_state["good_steps"] == sc.good and dev_state["hysteresis_left"] == sc.hyst_left
    assert dev_state["overflow"] == 0
    c = oracle.adamw_constants(oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, weight_decay=hp.weight_decay,
                                            global_batch=hp.global_batch, loss_scale=sc.scale, step=sc.step))
    for k in ("inv", "bc1", "bc2"):
        assert np.float32(dev_state[k]).view(np.uint32) == np.float32(c[k]).view(np.uint32), k


@pytest.mark.parametrize("M,n,align", [(1, 1000, 1), (2, 40_001, 8), (4, 2048 * 3 + 37, 128), (5, 30_011, 1),
                                       (7, 20_003, 128), (8, 100_003, 1), (9, 5000, 8), (64, 3001, 1)])
def test_dynamic_attempts_match_oracle(cuda_device, M, n, align):
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=2.0 ** 10, factor=2.0, window=3, hysteresis=2, min_scale=1.0)
    hp = z.AdamW(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, global_batch=max(M, 64), step=1)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    sc = oracle.Scaler.start(oracle_policy(policy), 1)
    check_scaler(z.scaler_state(scaler), sc, hp)
    master, m, v = make_state(n, P, 900 + M, dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    o = [f32(master), f32(m), f32(v)]
    o_params = np.zeros(n, np.uint16)
    overflow_at = {2, 3, 6}
    for attempt in range(9):
        S = sc.scale
        grads = [synth.normal_bf16(n, 1e-3 * S, synth.seed_of(M, attempt, r), dev) for r in range(M)]
        if attempt in overflow_at:
            grads[attempt % M][(37 * attempt) % n] = float("inf")
        g_np = [u16(g) for g in grads]
        z.zero1_step_dynamic(plan, 0, M, grads, master, m, v, params, hp, scaler, policy, sums)
        torch.cuda.synchronize()
        ohp = oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay,
                           global_batch=hp.global_batch)
        f = oracle.zero1_dynamic_attempt(g_np, n, *o, o_params, ohp, sc, oracle_policy(policy))
        assert f == (1 if attempt in overflow_at else 0)
        check_scaler(z.scaler_state(scaler), sc, hp)
        assert_f32_bits(f32(master), o[0], f"master attempt {attempt}")
        assert_f32_bits(f32(m), o[1], f"m attempt {attempt}")
        assert_f32_bits(f32(v), o[2], f"v attempt {attempt}")
        assert_bf16_bits(u16(params), o_params, f"params attempt {attempt}")
    assert sc.skipped == len(overflow_at)


@pytest.mark.parametrize("design", ["two_pass", "pingpong"])
def test_scaler_growth_refills_hysteresis_like_the_oracle(cuda_device, design):
    """A sequence that grows the scale with hysteresis left below its full
    count, then overflows right after the growth: the device scaler follows
    the oracle's rule (growth refills the hysteresis) attempt by attempt,
    and the state stays the oracle's."""
    dev = cuda_device
    M, n = 2, 4099
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=64.0, factor=2.0, window=2, hysteresis=2, min_scale=1.0)
    hp = z.AdamW(global_batch=64, step=1)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    sc = oracle.Scaler.start(oracle_policy(policy), 1)
    master, m, v = make_state(n, P, 77, dev)
    o = [f32(master), f32(m), f32(v)]
    # parameters consistent with the master weights, as after any earlier
    # step (the ping-pong design restores them from the master on a skip)
    o_params = oracle.f32_to_bf16(o[0][:n])
    params = torch.from_numpy(o_params.view(np.int16).copy()).view(torch.bfloat16).to(dev)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    pairs = [[x, torch.zeros_like(x)] for x in (master, m, v)]
    ohp = oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay,
                       global_batch=hp.global_batch)
    pattern = [1, 0, 0, 1, 1, 0, 0, 1, 0, 0]
    for attempt, over in enumerate(pattern):
        grads = [synth.normal_bf16(n, 1e-3 * sc.scale, synth.seed_of(78, attempt, r), dev) for r in range(M)]
        if over:
            grads[attempt % M][(13 * attempt) % n] = float("-inf")
        g_np = [u16(g) for g in grads]
        if design == "two_pass":
            z.zero1_step_dynamic(plan, 0, M, grads, master, m, v, params, hp, scaler, policy, sums)
        else:
            z.zero1_step_dynamic_pingpong(plan, 0, M, grads, *pairs, params, hp, scaler, policy)
        torch.cuda.synchronize()
        assert oracle.zero1_dynamic_attempt(g_np, n, *o, o_params, ohp, sc, oracle_policy(policy)) == over
        check_scaler(z.scaler_state(scaler), sc, hp)
        state = [master, m, v] if design == "two_pass" else z.current_state(scaler, *pairs)
        for x, want, what in zip(state, o, ("master", "m", "v")):
            assert_f32_bits(f32(x), want, f"{design} {what} attempt {attempt}")
        assert_bf16_bits(u16(params), o_params, f"{design} params attempt {attempt}")
    # growth after attempts 1-2 refilled the hysteresis, so attempt 3 did not
    # back off and attempt 4 did (64 -> 128 -> 64); then 128 and 256
    assert sc.scale == 256.0 and sc.skipped == 4


def test_clean_dynamic_step_equals_fused_step(cuda_device):
    """Without overflow the three-kernel dynamic step is bit for bit the
    fused step with the scaler's S and t."""
    dev = cuda_device
    M, n = 8, 300_007
    plan = z.zero1_plan(n, M, 128)
    policy = z.LossScalePolicy(initial_scale=65536.0, window=1000, hysteresis=2)
    hp = z.AdamW(global_batch=1024, step=5)
    a = make_state(n, plan.padded_n, 77, dev, nonzero_moments=True)
    b = [t.clone() for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    sums = torch.empty(plan.padded_n, dtype=torch.float32, device=dev)
    for t in range(5, 8):
        grads = [synth.normal_bf16(n, 1e-3 * 65536, synth.seed_of(78, t, r), dev) for r in range(M)]
        z.zero1_step_dynamic(plan, 0, M, grads, *a, pa, hp, scaler, policy, sums)
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *b, pb, z.AdamW(global_batch=1024, step=t,
                                                                                  loss_scale=65536.0))
    torch.cuda.synchronize()
    for x, y, what in zip(a, b, ("master", "m", "v")):
        assert_f32_bits(f32(x), f32(y), what)
    assert_bf16_bits(u16(pa), u16(pb), "params")
    st = z.scaler_state(scaler)
    assert st["step"] == 8 and st["skipped"] == 0 and st["scale"] == 65536.0


def test_llama_layers_dynamic_with_pages_policy(cuda_device):
    """Four Llama-style layers, the pages' fp16 block (hysteresis 2): the
    overflowing third attempt is skipped on the device, S is kept (one
    overflow is tolerated), t does not advance; checked on samples."""
    w = W.LLAMA4
    dev = cuda_device
    plan = z.zero1_plan(w.n, w.M, w.align)
    n, P = plan.n, plan.padded_n
    policy = z.LossScalePolicy(initial_scale=w.S, factor=2.0, window=1000, hysteresis=2, min_scale=1.0)
    hp = z.AdamW(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, global_batch=w.B)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    sc = oracle.Scaler.start(oracle_policy(policy), 1)
    master = torch.zeros(P, dtype=torch.float32, device=dev)
    master[:n] = synth.normal_f32(n, w.master_std, synth.seed_of(w.seed, 1), dev)
    m = torch.zeros(P, dtype=torch.float32, device=dev)
    v = torch.zeros(P, dtype=torch.float32, device=dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    grads = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(w.M)]
    rng = np.random.default_rng(2)
    idx_np = np.unique(np.concatenate([rng.integers(0, n, 1 << 15), np.arange(n - 64, n)]))
    idx = torch.from_numpy(idx_np).to(dev)
    o = [f32(master[idx]), f32(m[idx]), f32(v[idx])]
    o_params = np.zeros(idx_np.size, np.uint16)
    for attempt in range(1, 5):
        injected = 0
        for r, g in enumerate(grads):
            g.copy_(synth.normal_bf16(n, w.grad_std * sc.scale, synth.seed_of(w.seed, 100 + attempt, r), dev))
            if attempt == w.inf_attempt:
                injected += synth.set_inf(g, w.inf_prob, synth.seed_of(w.seed, 900 + attempt, r))
        g_s = [u16(g[idx]) for g in grads]
        z.zero1_step_dynamic(plan, 0, w.M, grads, master, m, v, params, hp, scaler, policy, sums)
        torch.cuda.synchronize()
        # the global flag is known from the draws: +inf was injected on this attempt only
        expect = 1 if attempt == w.inf_attempt else 0
        assert (injected > 0) == bool(expect)
        f = np.array([expect], np.uint32)
        ohp = oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay,
                           global_batch=hp.global_batch, loss_scale=sc.scale, step=sc.step)
        oracle.zero1_step(g_s, idx_np.size, *o, o_params, ohp, flag=f, skip_if_flag=True)
        sc.update(expect, oracle_policy(policy))
        check_scaler(z.scaler_state(scaler), sc, hp)
        assert_f32_bits(f32(master[idx]), o[0], f"master attempt {attempt}")
        assert_f32_bits(f32(v[idx]), o[2], f"v attempt {attempt}")
        assert_bf16_bits(u16(params[idx]), o_params, f"params attempt {attempt}")
    st = z.scaler_state(scaler)
    assert st["step"] == 4 and st["skipped"] == 1 and st["scale"] == w.S and st["hysteresis_left"] == 1
    del grads, master, m, v, params, sums
    torch.cuda.empty_cache()


def test_dynamic_step_replays_from_a_cuda_graph(cuda_device):
    """S and t live on the device, so one dynamically scaled attempt can be
    captured once and replayed each iteration (new gradients written into
    the same buffers); the replays give the eager calls' bits, overflow
    skips included."""
    dev = cuda_device
    M, n = 4, 70_001
    plan = z.zero1_plan(n, M, 128)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=512.0, window=2, hysteresis=1, min_scale=1.0)
    hp = z.AdamW(global_batch=64, step=1)
    eager = make_state(n, P, 61, dev)
    graphed = [t.clone() for t in eager]
    pe = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pg = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    se, sg = z.new_scaler(dev), z.new_scaler(dev)
    z.zero1_scaler_init(se, policy, hp)
    z.zero1_scaler_init(sg, policy, hp)
    sums_e = torch.empty(P, dtype=torch.float32, device=dev)
    sums_g = torch.empty(P, dtype=torch.float32, device=dev)
    gbuf = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    torch.cuda.synchronize()
    # warm up on a side stream (occupancy queries are cached), then capture
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        spare = z.new_scaler(dev)
        z.zero1_scaler_init(spare, policy, hp)
        z.zero1_step_dynamic(plan, 0, M, gbuf, *[t.clone() for t in graphed], pg.clone(), hp, spare, policy, sums_g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        z.zero1_step_dynamic(plan, 0, M, gbuf, *graphed, pg, hp, sg, policy, sums_g)
    for k in range(7):
        fresh = [synth.normal_bf16(n, 1e-3 * 512, synth.seed_of(62, k, r), dev) for r in range(M)]
        if k in (2, 5):
            fresh[k % M][100 + k] = float("inf")
        for g, f in zip(gbuf, fresh):
            g.copy_(f)
        graph.replay()
        z.zero1_step_dynamic(plan, 0, M, fresh, *eager, pe, hp, se, policy, sums_e)
    torch.cuda.synchronize()
    for x, y, what in zip(eager, graphed, ("master", "m", "v")):
        assert_f32_bits(f32(y), f32(x), what)
    assert_bf16_bits(u16(pg), u16(pe), "params")
    assert z.scaler_state(sg) == z.scaler_state(se)
    assert z.scaler_state(sg)["skipped"] == 2 and z.scaler_state(sg)["step"] == 6
