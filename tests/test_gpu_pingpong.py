"""GPU parity of the dynamically scaled step with ping-pong state ("五维并行实战"
4.2 fp16 block; "CS336 Lecture 7: Parallelism 1", ZeRO Stage 1): every
attempt's current master/m/v and the parameters bit for bit against the
oracle's attempt and against the two-pass dynamic step, skipped attempts
included (the first attempt, consecutive ones, M > 8), and replayed from a
CUDA graph."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, u16
from test_gpu_dynamic import check_scaler, oracle_policy
from test_gpu_parity import make_state

pytestmark = pytest.mark.gpu


def bf16_of(master: torch.Tensor, n: int) -> torch.Tensor:
    """params = bf16(master[:n]), rounded by the oracle (the state a skipped
    first attempt must leave unchanged)."""
    bits = oracle.f32_to_bf16(f32(master[:n]))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(master.device)


def two_copies(n, P, seed, dev, nonzero_moments=False):
    """Copy 0 holds the state; copy 1 starts as garbage (NaN), which no
    attempt may read."""
    cur = make_state(n, P, seed, dev, nonzero_moments=nonzero_moments)
    other = [torch.full_like(t, float("nan")) for t in cur]
    return [[a, b] for a, b in zip(cur, other)]


@pytest.mark.parametrize("M,n,align", [(1, 1000, 1), (3, 40_001, 8), (4, 2048 * 3 + 37, 128), (5, 30_011, 1),
                                       (6, 20_003, 128), (8, 100_003, 1), (9, 5000, 8), (64, 3001, 1), (8, 7, 1)])
def test_pingpong_attempts_match_oracle(cuda_device, M, n, align):
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=2.0 ** 10, factor=2.0, window=3, hysteresis=2, min_scale=1.0)
    hp = z.AdamW(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, global_batch=max(M, 64), step=1)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    sc = oracle.Scaler.start(oracle_policy(policy), 1)
    masters, ms, vs = two_copies(n, P, 700 + M, dev, nonzero_moments=True)
    params = bf16_of(masters[0], n)
    o = [f32(masters[0]), f32(ms[0]), f32(vs[0])]
    o_params = u16(params).copy()
    overflow_at = {0, 3, 4, 7}
    for attempt in range(10):
        S = sc.scale
        grads = [synth.normal_bf16(n, 1e-3 * S, synth.seed_of(M, 50 + attempt, r), dev) for r in range(M)]
        if attempt in overflow_at:
            grads[attempt % M][(37 * attempt) % n] = float("inf") if attempt != 4 else float("nan")
        g_np = [u16(g) for g in grads]
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads, masters, ms, vs, params, hp, scaler, policy)
        torch.cuda.synchronize()
        ohp = oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay,
                           global_batch=hp.global_batch)
        f = oracle.zero1_dynamic_attempt(g_np, n, *o, o_params, ohp, sc, oracle_policy(policy))
        assert f == (1 if attempt in overflow_at else 0)
        st = z.scaler_state(scaler)
        check_scaler(st, sc, hp)
        assert st["current"] == (attempt + 1 - len([a for a in overflow_at if a <= attempt])) % 2
        cm, cmo, cv = z.current_state(scaler, masters, ms, vs)
        assert_f32_bits(f32(cm), o[0], f"master attempt {attempt}")
        assert_f32_bits(f32(cmo), o[1], f"m attempt {attempt}")
        assert_f32_bits(f32(cv), o[2], f"v attempt {attempt}")
        assert_bf16_bits(u16(params), o_params, f"params attempt {attempt}")
    assert sc.skipped == len(overflow_at)


@pytest.mark.parametrize("M,n,align,shards", [(8, 300_007, 128, None), (13, 20_011, 8, (3, 9)),
                                              (2, 50_000, 1, (1, 2))])
def test_pingpong_equals_two_pass_dynamic_step(cuda_device, M, n, align, shards):
    """Same inputs through the two-pass dynamic step and the ping-pong step:
    the same bits after every attempt, on a shard range too."""
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    sb, se = shards or (0, M)
    base, L, nv = plan.shard_range(sb, se)
    policy = z.LossScalePolicy(initial_scale=4096.0, factor=2.0, window=2, hysteresis=1, min_scale=1.0)
    hp = z.AdamW(global_batch=1024, step=3)
    a = [t[base:base + L].clone() for t in make_state(n, plan.padded_n, 31, dev, nonzero_moments=True)]
    pairs = [[t.clone(), torch.zeros_like(t)] for t in a]
    pa = bf16_of(a[0], nv) if nv else torch.zeros(1, dtype=torch.bfloat16, device=dev)
    pb = pa.clone()
    s_a, s_b = z.new_scaler(dev), z.new_scaler(dev)
    z.zero1_scaler_init(s_a, policy, hp)
    z.zero1_scaler_init(s_b, policy, hp)
    sums = torch.empty(L, dtype=torch.float32, device=dev)
    for k in range(6):
        grads = [synth.normal_bf16(max(nv, 1), 1e-3 * 4096, synth.seed_of(32, k, r), dev)[:nv] for r in range(M)]
        if k in (1, 2) and nv:
            grads[k % M][nv // 2] = float("-inf")
        z.zero1_step_dynamic(plan, sb, se, grads, *a, pa, hp, s_a, policy, sums)
        z.zero1_step_dynamic_pingpong(plan, sb, se, grads, *pairs, pb, hp, s_b, policy)
        torch.cuda.synchronize()
        cur = z.current_state(s_b, *pairs)
        for x, y, what in zip(a, cur, ("master", "m", "v")):
            assert_f32_bits(f32(y), f32(x), f"{what} attempt {k}")
        assert_bf16_bits(u16(pb[:nv]), u16(pa[:nv]), f"params attempt {k}")
        sa, sb_ = z.scaler_state(s_a), z.scaler_state(s_b)
        sa.pop("current"), sb_.pop("current")
        assert sa == sb_


def test_pingpong_copies_at_different_phases(cuda_device):
    """Copies whose 16-byte phases differ run per element, with the same
    bits."""
    dev = cuda_device
    M, n = 4, 10_003
    plan = z.zero1_plan(n, M, 1)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=256.0, window=1000, hysteresis=2)
    hp = z.AdamW(global_batch=64, step=1)
    a = make_state(n, P, 41, dev, nonzero_moments=True)
    raw = [torch.zeros(P + 1, dtype=torch.float32, device=dev) for _ in range(3)]
    pairs = [[t.clone(), r[1:]] for t, r in zip(a, raw)]     # copy 1 four bytes off the 16-byte phase
    pa = bf16_of(a[0], n)
    pb = pa.clone()
    s_a, s_b = z.new_scaler(dev), z.new_scaler(dev)
    z.zero1_scaler_init(s_a, policy, hp)
    z.zero1_scaler_init(s_b, policy, hp)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    for k in range(3):
        grads = [synth.normal_bf16(n, 1e-3 * 256, synth.seed_of(42, k, r), dev) for r in range(M)]
        z.zero1_step_dynamic(plan, 0, M, grads, *a, pa, hp, s_a, policy, sums)
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads, *pairs, pb, hp, s_b, policy)
    torch.cuda.synchronize()
    for x, y, what in zip(a, z.current_state(s_b, *pairs), ("master", "m", "v")):
        assert_f32_bits(f32(y), f32(x), what)
    assert_bf16_bits(u16(pb), u16(pa), "params")


def test_pingpong_replays_from_a_cuda_graph(cuda_device):
    """The copy to read is decided on the device, so one captured attempt
    replays correctly whichever copy is current, skips included."""
    dev = cuda_device
    M, n = 8, 90_001
    plan = z.zero1_plan(n, M, 128)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=512.0, window=2, hysteresis=1, min_scale=1.0)
    hp = z.AdamW(global_batch=64, step=1)
    eager = make_state(n, P, 71, dev, nonzero_moments=True)
    pairs = [[t.clone(), torch.zeros_like(t)] for t in eager]
    pe = bf16_of(eager[0], n)
    pg = pe.clone()
    se, sg = z.new_scaler(dev), z.new_scaler(dev)
    z.zero1_scaler_init(se, policy, hp)
    z.zero1_scaler_init(sg, policy, hp)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    gbuf = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm-up on spare buffers (occupancy queries are cached)
        spare = z.new_scaler(dev)
        z.zero1_scaler_init(spare, policy, hp)
        z.zero1_step_dynamic_pingpong(plan, 0, M, gbuf, *[[x.clone() for x in p] for p in pairs], pg.clone(), hp,
                                      spare, policy)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        z.zero1_step_dynamic_pingpong(plan, 0, M, gbuf, *pairs, pg, hp, sg, policy)
    for k in range(8):
        fresh = [synth.normal_bf16(n, 1e-3 * 512, synth.seed_of(72, k, r), dev) for r in range(M)]
        if k in (2, 3, 6):
            fresh[k % M][200 + k] = float("inf")
        for g, f in zip(gbuf, fresh):
            g.copy_(f)
        graph.replay()
        z.zero1_step_dynamic(plan, 0, M, fresh, *eager, pe, hp, se, policy, sums)
    torch.cuda.synchronize()
    for x, y, what in zip(eager, z.current_state(sg, *pairs), ("master", "m", "v")):
        assert_f32_bits(f32(y), f32(x), what)
    assert_bf16_bits(u16(pg), u16(pe), "params")
    a, b = z.scaler_state(sg), z.scaler_state(se)
    assert a.pop("current") == (8 - 3) % 2
    b.pop("current")
    assert a == b and a["skipped"] == 3


def test_pingpong_rejects_bad_arguments(cuda_device):
    dev = cuda_device
    M, n = 2, 1000
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    policy = z.LossScalePolicy()
    hp = z.AdamW(global_batch=64)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    st = make_state(n, P, 1, dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grads = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    with pytest.raises(z.Zero1Error) as e:       # both copies the same buffer
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads, [st[0], st[0]], [st[1], st[1].clone()],
                                      [st[2], st[2].clone()], params, hp, scaler, policy)
    assert e.value.code == -1
    with pytest.raises(ValueError):              # not a pair
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads, [st[0]], [st[1], st[1]], [st[2], st[2]], params, hp,
                                      scaler, policy)
    with pytest.raises(z.Zero1Error) as e:       # a policy the rule cannot use
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads, [st[0], st[0].clone()], [st[1], st[1].clone()],
                                      [st[2], st[2].clone()], params, hp, scaler, z.LossScalePolicy(factor=1.0))
    assert e.value.code == -1
    # a copy that is not 4-byte aligned, through the C ABI (the binding's
    # fp32 tensors cannot express it)
    raw = torch.zeros(P + 1, dtype=torch.float32, device=dev)
    odd = raw.view(torch.uint8)[2:2 + 4 * P]
    pair = lambda a, b: (ctypes.c_void_p * 2)(a, b)
    m1, v1 = st[1].clone(), st[2].clone()
    rc = z.load().zero1_step_dynamic_pingpong(
        ctypes.byref(plan), 0, M, (ctypes.c_void_p * M)(*[g.data_ptr() for g in grads]),
        pair(st[0].data_ptr(), odd.data_ptr()), pair(st[1].data_ptr(), m1.data_ptr()),
        pair(st[2].data_ptr(), v1.data_ptr()), params.data_ptr(), ctypes.byref(hp.c_struct()),
        scaler.data_ptr(), ctypes.byref(policy.c_struct()), torch.cuda.current_stream().cuda_stream)
    assert rc == -2


def random_cover(L, rng, max_bucket):
    """Random bucket boundaries over [0, L), multiples of 8 but the last."""
    cuts = [0]
    while cuts[-1] < L:
        step = int(rng.integers(1, max_bucket // 8 + 1)) * 8
        cuts.append(min(L, cuts[-1] + step))
    return list(zip(cuts[:-1], cuts[1:]))


@pytest.mark.parametrize("M,n,align,shards,max_bucket", [(8, 200_003, 128, None, 50_000),
                                                         (13, 30_011, 8, (2, 11), 4096),
                                                         (3, 9_999, 1, (1, 2), 800)])
def test_bucketed_pingpong_equals_whole_attempt(cuda_device, M, n, align, shards, max_bucket):
    """Buckets in random order and sizes, their gradient buffers recycled,
    then the finish: bit for bit the whole-range ping-pong attempt, including
    attempts skipped because one bucket overflowed."""
    dev = cuda_device
    rng = np.random.default_rng(M)
    plan = z.zero1_plan(n, M, align)
    sb, se = shards or (0, M)
    base, L, nv = plan.shard_range(sb, se)
    policy = z.LossScalePolicy(initial_scale=1024.0, factor=2.0, window=2, hysteresis=1, min_scale=1.0)
    hp = z.AdamW(global_batch=1024, step=1)
    start = [t[base:base + L].clone() for t in make_state(n, plan.padded_n, 51, dev, nonzero_moments=True)]
    whole = [[t.clone(), torch.zeros_like(t)] for t in start]
    bucketed = [[t.clone(), torch.full_like(t, float("nan"))] for t in start]
    pw = bf16_of(start[0], nv) if nv else torch.zeros(1, dtype=torch.bfloat16, device=dev)
    pb = pw.clone()
    s_w, s_b = z.new_scaler(dev), z.new_scaler(dev)
    z.zero1_scaler_init(s_w, policy, hp)
    z.zero1_scaler_init(s_b, policy, hp)
    attempt = z.PingPongBuckets(plan, sb, se, *bucketed, pb, s_b, policy)
    recycled = [torch.empty(max_bucket, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    for k in range(5):
        grads = [synth.normal_bf16(max(nv, 1), 1e-3 * 1024, synth.seed_of(52, k, r), dev)[:nv] for r in range(M)]
        if k in (1, 3) and nv:
            grads[k % M][nv - 1 - k] = float("inf")          # in the range's last bucket
        z.zero1_step_dynamic_pingpong(plan, sb, se, grads, *whole, pw, hp, s_w, policy)
        cover = random_cover(L, rng, max_bucket)
        for i in rng.permutation(len(cover)):
            b, e = cover[i]
            real = max(0, min(nv, e) - b)
            for buf, g in zip(recycled, grads):
                buf[:real].copy_(g[b:b + real])
            attempt.bucket(b, e, [buf[:real] for buf in recycled], hp)
        attempt.finish(hp)
        torch.cuda.synchronize()
        for x, y, what in zip(z.current_state(s_w, *whole), z.current_state(s_b, *bucketed), ("master", "m", "v")):
            assert_f32_bits(f32(y), f32(x), f"{what} attempt {k}")
        assert_bf16_bits(u16(pb[:nv]), u16(pw[:nv]), f"params attempt {k}")
        assert z.scaler_state(s_b) == z.scaler_state(s_w)
    assert z.scaler_state(s_b)["skipped"] == 2


def test_bucketed_pingpong_checks_coverage(cuda_device):
    dev = cuda_device
    M, n = 2, 4096
    plan = z.zero1_plan(n, M, 8)
    policy = z.LossScalePolicy()
    hp = z.AdamW(global_batch=64)
    sc = z.new_scaler(dev)
    z.zero1_scaler_init(sc, policy, hp)
    st = make_state(n, plan.padded_n, 1, dev)
    pairs = [[t, torch.zeros_like(t)] for t in st]
    params = bf16_of(st[0], n)
    grads = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    attempt = z.PingPongBuckets(plan, 0, M, *pairs, params, sc, policy)
    attempt.bucket(0, 1024, [g[:1024] for g in grads], hp)
    attempt.bucket(2048, 4096, [g[2048:] for g in grads], hp)
    with pytest.raises(ValueError):          # [1024, 2048) missing
        attempt.finish(hp)
    with pytest.raises(ValueError):
        attempt.bucket(4000, 4100, [g[4000:] for g in grads], hp)


def test_llama_layers_pingpong_with_pages_policy(cuda_device):
    """Full size: the four Llama-style layers (872,448,000 parameters, M = 8,
    S = 65536), the pages' fp16 block (hysteresis 2), +inf injected on the
    third attempt: the ping-pong step skips it on the device, keeps S, does
    not advance t, restores params; sampled elements of the current copy and
    of params equal the oracle after every attempt."""
    from zero_sharded_mixed_zero1_gb300 import workloads as W
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
    pairs = [[master, torch.empty_like(master)], [torch.zeros_like(master), torch.empty_like(master)],
             [torch.zeros_like(master), torch.empty_like(master)]]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grads = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(w.M)]
    rng = np.random.default_rng(3)
    idx_np = np.unique(np.concatenate([rng.integers(0, n, 1 << 15), np.arange(n - 64, n)]))
    idx = torch.from_numpy(idx_np).to(dev)
    o = [f32(pairs[0][0][idx]), f32(pairs[1][0][idx]), f32(pairs[2][0][idx])]
    o_params = np.zeros(idx_np.size, np.uint16)
    for attempt in range(1, 5):
        injected = 0
        for r, g in enumerate(grads):
            g.copy_(synth.normal_bf16(n, w.grad_std * sc.scale, synth.seed_of(w.seed, 100 + attempt, r), dev))
            if attempt == w.inf_attempt:
                injected += synth.set_inf(g, w.inf_prob, synth.seed_of(w.seed, 900 + attempt, r))
        g_s = [u16(g[idx]) for g in grads]
        z.zero1_step_dynamic_pingpong(plan, 0, w.M, grads, *pairs, params, hp, scaler, policy)
        torch.cuda.synchronize()
        expect = 1 if attempt == w.inf_attempt else 0           # known from the draws
        assert (injected > 0) == bool(expect)
        ohp = oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay,
                           global_batch=hp.global_batch, loss_scale=sc.scale, step=sc.step)
        oracle.zero1_step(g_s, idx_np.size, *o, o_params, ohp, flag=np.array([expect], np.uint32),
                          skip_if_flag=True)
        sc.update(expect, oracle_policy(policy))
        check_scaler(z.scaler_state(scaler), sc, hp)
        cm, cmo, cv = z.current_state(scaler, *pairs)
        assert_f32_bits(f32(cm[idx]), o[0], f"master attempt {attempt}")
        assert_f32_bits(f32(cmo[idx]), o[1], f"m attempt {attempt}")
        assert_f32_bits(f32(cv[idx]), o[2], f"v attempt {attempt}")
        assert_bf16_bits(u16(params[idx]), o_params, f"params attempt {attempt}")
    st = z.scaler_state(scaler)
    assert st["step"] == 4 and st["skipped"] == 1 and st["scale"] == w.S and st["current"] == 1
    del grads, pairs, params, master
    torch.cuda.empty_cache()
