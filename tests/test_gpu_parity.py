"""GPU parity at small sizes: every output element of the CUDA path against
the CPU oracle on the same seeded inputs, bit for bit.

Sizes span several blocks (a block walks 256 x 8 = 2048 elements per
iteration) plus ragged tails; replica counts cover the compile-time paths
(M = 1..8) and the grouped path (M > 8); shard ranges cover one call over all
shards, one call per shard on slices of full buffers (head + vector body +
tail), one call per shard on separately allocated state (per-element path
when the element phases differ) and a sub-range of shards.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, oracle_hp, u16

pytestmark = pytest.mark.gpu

SIZES = [(1, 1), (7, 1), (8, 8), (9, 1), (2048 * 3 + 37, 1), (2048 * 3 + 37, 128), (100_003, 8)]
REPLICAS = [1, 2, 3, 4, 5, 7, 8, 9, 16, 64]


def make_state(n, P, seed, device, nonzero_moments=False):
    master = torch.zeros(P, dtype=torch.float32, device=device)
    master[:n] = synth.normal_f32(n, 0.02, synth.seed_of(seed, 1), device)
    m = torch.zeros(P, dtype=torch.float32, device=device)
    v = torch.zeros(P, dtype=torch.float32, device=device)
    if nonzero_moments:
        m[:n] = synth.normal_f32(n, 1e-5, synth.seed_of(seed, 2), device)
        v[:n] = synth.normal_f32(n, 1e-5, synth.seed_of(seed, 3), device).square_()
    return master, m, v


def make_grads(M, n, std, seed, step, device):
    return [synth.normal_bf16(n, std, synth.seed_of(seed, 100 + step, r), device) for r in range(M)]


def oracle_step(plan, grads_np, master_np, m_np, v_np, hp, flag=None):
    """Oracle over all shards, one shard at a time (as M ranks would)."""
    params = np.zeros(plan.n, np.uint16)
    for i in range(plan.M):
        lo, hi = i * plan.shard, (i + 1) * plan.shard
        nv = max(0, min(hi, plan.n) - lo)
        sub = [np.ascontiguousarray(g[lo:lo + nv]) for g in grads_np]
        w, mm, vv = master_np[lo:hi].copy(), m_np[lo:hi].copy(), v_np[lo:hi].copy()
        pp = np.zeros(nv, np.uint16)
        oracle.zero1_step(sub, nv, w, mm, vv, pp, hp, flag=flag)
        master_np[lo:hi], m_np[lo:hi], v_np[lo:hi] = w, mm, vv
        params[lo:lo + nv] = pp
    return params


@pytest.mark.parametrize("M", REPLICAS)
@pytest.mark.parametrize("n,align", SIZES)
@pytest.mark.parametrize("mode", ["whole", "per_shard_sliced", "per_shard_separate", "sub_range"])
def test_fused_step_matches_oracle(cuda_device, M, n, align, mode):
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    P, s = plan.padded_n, plan.shard
    seed = synth.seed_of(M, n, align)
    master, m, v = make_state(n, P, seed, dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    o_master, o_m, o_v = f32(master), f32(m), f32(v)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    sb, se = (1, M - 1) if mode == "sub_range" else (0, M)
    if mode == "sub_range" and M < 3:
        pytest.skip("needs three shards")
    sep = None
    if mode == "per_shard_separate":
        sep = [[t[i * s:(i + 1) * s].clone() for t in (master, m, v)] for i in range(M)]
    for t in range(1, 4):
        hp = z.AdamW(global_batch=max(M, 32), step=t)
        grads = make_grads(M, n, 1e-2, seed, t, dev)
        g_np = [u16(g) for g in grads]
        if mode == "whole":
            z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp, flag)
        elif mode == "sub_range":
            base, L, nv = plan.shard_range(sb, se)
            z.zero1_reduce_scatter_adamw_allgather(plan, sb, se, [g[base:] for g in grads], master[base:base + L],
                                                   m[base:base + L], v[base:base + L], params[base:], hp, flag)
        else:
            for i in range(M):
                base, L, nv = plan.shard_range(i, i + 1)
                if sep is None:
                    st = (master[base:base + L], m[base:base + L], v[base:base + L])
                else:
                    st = sep[i]
                gi = [g[base:] if base < n else g[:0] for g in grads]
                pi = params[base:] if base < n else params[:0]
                z.zero1_reduce_scatter_adamw_allgather(plan, i, i + 1, gi, *st, pi, hp, flag)
        torch.cuda.synchronize()
        ohp = oracle_hp(hp)
        if mode == "sub_range":
            base, L, nv = plan.shard_range(sb, se)
            o_params_full = u16(params).copy()
            sub = [np.ascontiguousarray(g[base:base + nv]) for g in g_np]
            w, mm, vv = o_master[base:base + L].copy(), o_m[base:base + L].copy(), o_v[base:base + L].copy()
            pp = np.zeros(nv, np.uint16)
            oracle.zero1_step(sub, nv, w, mm, vv, pp, ohp)
            o_master[base:base + L], o_m[base:base + L], o_v[base:base + L] = w, mm, vv
            want_params = pp
            got_params = o_params_full[base:base + nv]
        else:
            want_params = oracle_step(plan, g_np, o_master, o_m, o_v, ohp)
            got_params = u16(params)
        if sep is not None:
            got = [np.concatenate([f32(sep[i][k]) for i in range(M)]) for k in range(3)]
        else:
            got = [f32(master), f32(m), f32(v)]
        assert_f32_bits(got[0], o_master, f"master t={t}")
        assert_f32_bits(got[1], o_m, f"m t={t}")
        assert_f32_bits(got[2], o_v, f"v t={t}")
        assert_bf16_bits(got_params, want_params, f"params t={t}")
        # padding stays +0
        assert not got[0][n:].view(np.uint32).any()
    assert int(flag.item()) == 0


@pytest.mark.parametrize("M", [1, 4, 8, 13])
def test_unaligned_pointers_run_the_per_element_path(cuda_device, M):
    """Pointers that are naturally but not 16-byte aligned at any common
    element phase: every element goes through the per-element path."""
    dev = cuda_device
    n = 5000
    plan = z.zero1_plan(n, M, 1)
    P = plan.padded_n
    seed = synth.seed_of(77, M)
    raw = [synth.normal_bf16(n + 1, 1e-2, synth.seed_of(seed, r), dev) for r in range(M)]
    grads = [g[1:] for g in raw]                       # 2-byte phase
    store = torch.zeros(3 * (P + 3), dtype=torch.float32, device=dev)
    master, m, v = (store[k * (P + 3) + 2: k * (P + 3) + 2 + P] for k in range(3))  # 8-byte phase
    master[:n] = synth.normal_f32(n, 0.02, seed, dev)
    pbuf = torch.zeros(n + 3, dtype=torch.bfloat16, device=dev)
    params = pbuf[3:3 + n]
    o_master, o_m, o_v = f32(master), f32(m), f32(v)
    hp = z.AdamW(global_batch=64, step=2)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp)
    want = oracle_step(plan, [u16(g) for g in grads], o_master, o_m, o_v, oracle_hp(hp))
    assert_f32_bits(f32(master), o_master, "master")
    assert_f32_bits(f32(m), o_m, "m")
    assert_f32_bits(f32(v), o_v, "v")
    assert_bf16_bits(u16(params), want, "params")
    assert not f32(store[:2]).any() and not u16(pbuf[:3]).any()   # nothing written outside


def test_moments_and_hyperparameters_sweep(cuda_device):
    """Nonzero moments, several hyperparameter sets incl. beta = 0, eps = 0,
    weight decay 0, a large loss scale, the pages' DeepSpeed block."""
    dev = cuda_device
    M, n = 8, 20_000
    plan = z.zero1_plan(n, M, 8)
    for k, hp in enumerate([
        z.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, global_batch=1024, step=5),
        z.AdamW(lr=2.0 ** -10, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.0, global_batch=8, step=1),
        z.AdamW(lr=3e-4, beta1=0.8, beta2=0.9, eps=1e-6, weight_decay=0.1, loss_scale=65536.0,
                global_batch=1024, step=1000),
        z.AdamW(lr=1e-2, beta1=0.5, beta2=0.7, eps=1e-3, weight_decay=-0.5, global_batch=12, step=3),
    ]):
        master, m, v = make_state(n, plan.padded_n, 900 + k, dev, nonzero_moments=True)
        params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
        grads = make_grads(M, n, 1e-3 * hp.loss_scale, 900 + k, 1, dev)
        o = [f32(master), f32(m), f32(v)]
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp)
        want = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp))
        assert_f32_bits(f32(master), o[0], f"master hp{k}")
        assert_f32_bits(f32(m), o[1], f"m hp{k}")
        assert_f32_bits(f32(v), o[2], f"v hp{k}")
        assert_bf16_bits(u16(params), want, f"params hp{k}")


def test_special_values_and_flag(cuda_device):
    """inf, -inf, NaN, inf + -inf, bf16 max + bf16 max (fp32 overflow), -0,
    subnormal bf16 gradients: the flag and every output against the oracle
    (the step is not skipped, so non-finite values propagate)."""
    dev = cuda_device
    M, n = 3, 4099
    plan = z.zero1_plan(n, M, 1)
    base = [u16(synth.normal_bf16(n, 1e-2, synth.seed_of(55, r), dev)) for r in range(M)]
    specials = {10: (0x7F80, 0x3F80, 0x3F80), 2000: (0xFF80, 0, 0), 3001: (0x7FC0, 0, 0),
                3002: (0x7F80, 0xFF80, 0), 4050: (0x7F7F, 0x7F7F, 0), 4051: (0x8000, 0x8000, 0x8000),
                4052: (0x0001, 0x0001, 0x8001), 4098: (0x0040, 0x0000, 0x0000)}
    for j, vals in specials.items():
        for r in range(M):
            base[r][j] = vals[r]
    grads = [torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(dev) for b in base]
    master, m, v = make_state(n, plan.padded_n, 56, dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    o = [f32(master), f32(m), f32(v)]
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    hp = z.AdamW(global_batch=3, step=1)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp, flag)
    oflag = np.zeros(1, np.uint32)
    want = oracle_step(plan, base, *o, oracle_hp(hp), flag=oflag)
    assert int(flag.item()) == int(oflag[0]) == 1
    assert_f32_bits(f32(master), o[0], "master")
    assert_f32_bits(f32(m), o[1], "m")
    assert_f32_bits(f32(v), o[2], "v")
    assert_bf16_bits(u16(params), want, "params")
    # the standalone check agrees, per shard and over all shards
    for sb, se in [(0, M), (0, 1), (1, 2), (2, 3)]:
        f = torch.zeros(1, dtype=torch.int32, device=dev)
        b0, L, nv = plan.shard_range(sb, se)
        z.zero1_overflow_check(plan, sb, se, [g[b0:] for g in grads], f)
        want_f = oracle.overflow_check([np.ascontiguousarray(b[b0:b0 + nv]) for b in base], nv)
        assert int(f.item()) == want_f


@pytest.mark.parametrize("entry", ["fused", "dynamic", "pingpong"])
@pytest.mark.parametrize("M", [1, 3, 8, 9])
def test_subnormal_moments_are_kept(cuda_device, M, entry):
    """Gradients near 1e-20 give v' = (1 - beta2) g^2 around 1e-41, below the
    smallest normal fp32, and the state also starts with subnormal m and v:
    no step may flush them to zero (the oracle keeps them), over the vector
    body and the per-element tail."""
    dev = cuda_device
    n = 20_011
    plan = z.zero1_plan(n, M, 1)
    P = plan.padded_n
    grads = [synth.normal_bf16(n, 1e-20, synth.seed_of(91, r), dev) for r in range(M)]
    master, m, v = make_state(n, P, 92, dev)
    m[:n] = synth.normal_f32(n, 1e-39, synth.seed_of(93, 1), dev)
    v[:n] = synth.normal_f32(n, 1e-39, synth.seed_of(93, 2), dev).abs_()
    assert bool(((v[:n] > 0) & (v[:n] < 1.1754944e-38)).any())       # subnormal state present
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    o = [f32(master), f32(m), f32(v)]
    hp = z.AdamW(global_batch=M, step=1, eps=1e-30)
    if entry == "fused":
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp)
    else:
        # S = 1 and t = 1 from the device scaler: the same constants as hp
        policy = z.LossScalePolicy(initial_scale=1.0)
        scaler = z.new_scaler(dev)
        z.zero1_scaler_init(scaler, policy, hp)
        if entry == "dynamic":
            sums = torch.empty(P, dtype=torch.float32, device=dev)
            z.zero1_step_dynamic(plan, 0, M, grads, master, m, v, params, hp, scaler, policy, sums)
        else:
            pairs = [[x, torch.empty_like(x)] for x in (master, m, v)]
            z.zero1_step_dynamic_pingpong(plan, 0, M, grads, *pairs, params, hp, scaler, policy)
            master, m, v = z.current_state(scaler, *pairs)
    want = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp))
    vv = f32(v)[:n]
    assert ((vv > 0) & (vv < np.float32(1.1754944e-38))).any()          # subnormal results produced
    assert_f32_bits(f32(master), o[0], "master")
    assert_f32_bits(f32(m), o[1], "m")
    assert_f32_bits(f32(v), o[2], "v")
    assert_bf16_bits(u16(params), want, "params")


@pytest.mark.parametrize("entry", ["fused", "dynamic", "pingpong"])
def test_squared_gradient_overflow_without_a_flag(cuda_device, entry):
    """Finite gradient sums near 1e20 whose squares overflow fp32: the flag
    stays clear (the sums are finite), v becomes +inf and the update of those
    elements reduces to the decay; every output against the oracle."""
    dev = cuda_device
    M, n = 4, 9_001
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    grads = [synth.normal_bf16(n, 1e-3 * M, synth.seed_of(94, r), dev) for r in range(M)]
    for r in range(M):
        grads[r][::97] = 3.0e19 * (1 if r % 2 == 0 else 0.5)
    master, m, v = make_state(n, P, 95, dev, nonzero_moments=True)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    o = [f32(master), f32(m), f32(v)]
    hp = z.AdamW(global_batch=M, step=3)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    if entry == "fused":
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp, flag)
        assert int(flag.item()) == 0
    else:
        policy = z.LossScalePolicy(initial_scale=1.0)
        scaler = z.new_scaler(dev)
        z.zero1_scaler_init(scaler, policy, hp)
        if entry == "dynamic":
            sums = torch.empty(P, dtype=torch.float32, device=dev)
            z.zero1_step_dynamic(plan, 0, M, grads, master, m, v, params, hp, scaler, policy, sums)
        else:
            pairs = [[x, torch.empty_like(x)] for x in (master, m, v)]
            z.zero1_step_dynamic_pingpong(plan, 0, M, grads, *pairs, params, hp, scaler, policy)
            master, m, v = z.current_state(scaler, *pairs)
        st = z.scaler_state(scaler)
        assert st["skipped"] == 0 and st["step"] == 4
    oflag = np.zeros(1, np.uint32)
    want = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp), flag=oflag)
    assert int(oflag[0]) == 0
    assert np.isinf(f32(v)[:n:97]).all()
    assert_f32_bits(f32(master), o[0], "master")
    assert_f32_bits(f32(m), o[1], "m")
    assert_f32_bits(f32(v), o[2], "v")
    assert_bf16_bits(u16(params), want, "params")


def test_skip_if_flag_writes_nothing(cuda_device):
    dev = cuda_device
    M, n = 8, 30_011
    plan = z.zero1_plan(n, M, 128)
    grads = make_grads(M, n, 1e-3, 31, 1, dev)
    grads[5][12345] = float("inf")
    master, m, v = make_state(n, plan.padded_n, 32, dev, nonzero_moments=True)
    params = synth.normal_bf16(n, 0.02, 33, dev)
    snap = [t.clone() for t in (master, m, v, params)]
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    z.zero1_overflow_check(plan, 0, M, grads, flag)
    hp = z.AdamW(global_batch=64, step=4)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp, flag, skip_if_flag=True)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    for a, b in zip((master, m, v, params), snap):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
    # clean gradients: the check leaves the flag at 0 and the step runs
    grads[5][12345] = 0.0
    flag.zero_()
    z.zero1_overflow_check(plan, 0, M, grads, flag)
    o = [f32(master), f32(m), f32(v)]
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp, flag, skip_if_flag=True)
    want = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp))
    assert int(flag.item()) == 0
    assert_f32_bits(f32(master), o[0], "master")
    assert_bf16_bits(u16(params), want, "params")


@pytest.mark.parametrize("M,n", [(1, 17), (1, 70_001), (2, 9_999), (3, 20_003), (4, 10_000), (5, 12_345), (6, 8_191),
                                 (7, 30_001), (8, 2048 * 3 + 5), (9, 4099), (64, 3000)])
def test_allreduce_matches_oracle_and_equals_rs_plus_ag(cuda_device, M, n):
    """Naive All-Reduce vs the oracle, and All-Reduce == Reduce-Scatter +
    All-Gather on the GPU, bitwise."""
    dev = cuda_device
    plan = z.zero1_plan(n, M, 8)
    grads = make_grads(M, n, 1.0, 41, M, dev)
    g_np = [u16(g) for g in grads]
    scale = 1.0 / 256
    outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    z.dp_allreduce(plan, grads, outs, scale)
    want = oracle.allreduce(g_np, n, scale=scale)
    for r in range(M):
        assert_bf16_bits(u16(outs[r]), want[r], f"AR bf16 out {r}")
    outs32 = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(M)]
    z.dp_allreduce(plan, grads, outs32, scale)
    want32 = oracle.allreduce(g_np, n, scale=scale, out_bf16=False)
    for r in range(M):
        assert_f32_bits(f32(outs32[r]), want32[r], f"AR f32 out {r}")
    # RS over all shards into one P-buffer, then AG into M outputs
    shards = torch.empty(plan.padded_n, dtype=torch.bfloat16, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    z.zero1_reduce_scatter(plan, 0, M, grads, scale, shards, flag)
    gathered = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    z.zero1_all_gather_shards(plan, shards, gathered)
    for r in range(M):
        assert torch.equal(gathered[r].view(torch.int16), outs[r].view(torch.int16))
    assert not u16(shards[n:]).any()
    # separate outputs run the instance that reads the gradients through the
    # read-only path
    z.dp_allreduce(plan, grads, outs, scale)
    last = z.debug_last_launch()
    assert "k_allreduce" in last["kernel"] and "k_allreduce_inplace" not in last["kernel"]
    # in place: outputs alias the inputs, so the coherent-load instance runs
    z.dp_allreduce(plan, grads, grads, scale)
    last = z.debug_last_launch()
    assert "k_allreduce_inplace" in last["kernel"], last
    for r in range(M):
        assert_bf16_bits(u16(grads[r]), want[r], f"AR in place {r}")


@pytest.mark.parametrize("M,n,align", [(4, 10_000, 8), (8, 2048 * 5 + 3, 1), (16, 4099, 128)])
def test_unfused_phases_equal_fused_step(cuda_device, M, n, align):
    """Reduce-scatter to fp32, AdamW, all-gather: the same bits as the fused
    kernel, and the fp32 reduce-scatter equals the oracle's."""
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    grads = make_grads(M, n, 1e-3, 61, 1, dev)
    hp = z.AdamW(global_batch=256, step=2)
    a = make_state(n, P, 62, dev, nonzero_moments=True)
    b = [t.clone() for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *a, pa, hp)
    g = torch.empty(P, dtype=torch.float32, device=dev)
    inv = float(oracle.adamw_constants(oracle_hp(hp))["inv"])
    z.zero1_reduce_scatter(plan, 0, M, grads, inv, g)
    want_g, _ = oracle.reduce_scatter([u16(x) for x in grads], n, P, inv)
    assert_f32_bits(f32(g), want_g, "reduce-scatter fp32")
    z.zero1_adamw_update(plan, 0, M, g, *b, hp)
    z.zero1_all_gather(plan, 0, M, b[0], pb)
    for x, y, what in zip(a, b, ("master", "m", "v")):
        assert_f32_bits(f32(y), f32(x), what)
    assert_bf16_bits(u16(pb), u16(pa), "params")


def test_prepared_step_equals_one_shot_calls(cuda_device):
    """FusedStep (buffers validated once) gives the one-shot call's bits."""
    dev = cuda_device
    M, n = 8, 50_003
    plan = z.zero1_plan(n, M, 8)
    a = make_state(n, plan.padded_n, 71, dev, nonzero_moments=True)
    b = [t.clone() for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grads = make_grads(M, n, 1e-3, 72, 1, dev)
    fa = torch.zeros(1, dtype=torch.int32, device=dev)
    step = z.FusedStep(plan, 0, M, grads, *b, pb)
    for t in range(1, 5):
        for g, g2 in zip(grads, make_grads(M, n, 1e-3, 72, t, dev)):
            g.copy_(g2)
        hp = z.AdamW(global_batch=512, step=t)
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *a, pa, hp, fa)
        step(hp)
    torch.cuda.synchronize()
    for x, y, what in zip(a, b, ("master", "m", "v")):
        assert_f32_bits(f32(y), f32(x), what)
    assert_bf16_bits(u16(pb), u16(pa), "params")


@pytest.mark.parametrize("M", [1, 2, 3, 5, 7, 8])
def test_pipelined_kernel_above_the_small_range_threshold(cuda_device, M):
    """Ranges above 2^21 elements run the two-deep pipelined kernel (smaller
    ones the wide kernel): every M it is compiled for, a ragged tail, a
    per-element head (a range starting at element 3), every element against
    the oracle."""
    dev = cuda_device
    n = 2 ** 21 + 2 ** 17 + 37
    plan = z.zero1_plan(n, M, 1)
    P, s = plan.padded_n, plan.shard
    master, m, v = make_state(n, P, 500 + M, dev, nonzero_moments=True)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    o = [f32(master), f32(m), f32(v)]
    for t in (1, 2):
        hp = z.AdamW(global_batch=max(M, 16), step=t)
        grads = make_grads(M, n, 1e-2, 510 + M, t, dev)
        if t == 1:
            z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp)
        else:        # a large range starting at element 3: a per-element head, then vectors
            z.zero1_step_bucket(plan, 0, 3, grads, master, m, v, params, hp)
            z.zero1_step_bucket(plan, 3, P, [g[3:] for g in grads], master[3:], m[3:], v[3:], params[3:], hp)
        torch.cuda.synchronize()
        want = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp))
        assert_f32_bits(f32(master), o[0], f"master t={t}")
        assert_f32_bits(f32(m), o[1], f"m t={t}")
        assert_f32_bits(f32(v), o[2], f"v t={t}")
        assert_bf16_bits(u16(params), want, f"params t={t}")


@pytest.mark.parametrize("M,n,align,S", [(8, 2048 * 11 + 5, 128, 65536.0), (4, 30_001, 1, 1.0)])
def test_pages_deepspeed_optimizer_block(cuda_device, M, n, align, S):
    """The AdamW block of the pages' DeepSpeed configuration ("五维并行实战" 4.2:
    lr 0.001, betas (0.9, 0.999), eps 1e-8, weight_decay 0.01), over ten
    steps with and without the fp16 block's loss scale: bit for bit the
    oracle at every step."""
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    state = make_state(n, plan.padded_n, 600 + M, dev)
    o = [f32(t) for t in state]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    for t in range(1, 11):
        hp = z.AdamW(lr=0.001, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=S,
                     global_batch=1024, step=t)
        grads = make_grads(M, n, 1e-3 * S, 601 + M, t, dev)
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *state, params, hp)
        torch.cuda.synchronize()
        want_p = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp))
        for x, y, what in zip(state, o, ("master", "m", "v")):
            assert_f32_bits(f32(x), y, f"{what} t={t}")
        assert_bf16_bits(u16(params), want_p, f"params t={t}")


@pytest.mark.parametrize("M", [1, 2, 3, 8, 13])
def test_state_at_16_byte_phase_matches_oracle(cuda_device, M):
    """fp32 buffers 16 bytes past a 32-byte boundary (the gradients at one):
    every vector kernel moves the state in 16-byte accesses instead of 32,
    with the same bits - the fused step (both store widths), the dynamic
    step, the ping-pong step and the unfused chain."""
    dev = cuda_device
    n = 3 * 4096 + 37
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n

    def shifted(t):
        """t's values in a fresh buffer that starts 4 floats into its allocation."""
        out = torch.zeros(t.numel() + 4, dtype=t.dtype, device=dev)[4:]
        out.copy_(t)
        return out

    grads = make_grads(M, n, 1e-2, 70 + M, 1, dev)
    g_np = [u16(g) for g in grads]
    hp = z.AdamW(global_batch=max(M, 64), step=3)
    base_state = make_state(n, P, 71 + M, dev, nonzero_moments=True)

    # the oracle, once
    o = [f32(t).copy() for t in base_state]
    want_p = oracle_step(plan, g_np, *o, oracle_hp(hp))

    # fused step
    st = [shifted(t) for t in base_state]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *st, params, hp)
    assert z.debug_last_launch()["w32"] is False
    torch.cuda.synchronize()
    for x, want, what in zip(st, o, ("master", "m", "v")):
        assert_f32_bits(f32(x), want, f"fused {what} M={M}")
    assert_bf16_bits(u16(params), want_p, f"fused params M={M}")

    # dynamic step and ping-pong step with the scaler at S = 1 and t = 3
    policy = z.LossScalePolicy(initial_scale=1.0, window=1000, hysteresis=2)
    for design in ("dynamic", "pingpong"):
        st = [shifted(t) for t in base_state]
        params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
        scaler = z.new_scaler(dev)
        z.zero1_scaler_init(scaler, policy, hp)
        if design == "dynamic":
            sums = shifted(torch.zeros(P, dtype=torch.float32, device=dev))
            z.zero1_step_dynamic(plan, 0, M, grads, *st, params, hp, scaler, policy, sums)
        else:
            pairs = [[t, shifted(torch.full_like(t, float("nan")))] for t in st]
            z.zero1_step_dynamic_pingpong(plan, 0, M, grads, *pairs, params, hp, scaler, policy)
            st = list(z.current_state(scaler, *pairs))
        torch.cuda.synchronize()
        for x, want, what in zip(st, o, ("master", "m", "v")):
            assert_f32_bits(f32(x), want, f"{design} {what} M={M}")
        assert_bf16_bits(u16(params), want_p, f"{design} params M={M}")

    # unfused chain: reduce-scatter to fp32, AdamW, all-gather
    st = [shifted(t) for t in base_state]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    g = shifted(torch.zeros(P, dtype=torch.float32, device=dev))
    inv = float(oracle.adamw_constants(oracle_hp(hp))["inv"])
    z.zero1_reduce_scatter(plan, 0, M, grads, inv, g)
    z.zero1_adamw_update(plan, 0, M, g, *st, hp)
    z.zero1_all_gather(plan, 0, M, st[0], params)
    torch.cuda.synchronize()
    for x, want, what in zip(st, o, ("master", "m", "v")):
        assert_f32_bits(f32(x), want, f"unfused {what} M={M}")
    assert_bf16_bits(u16(params), want_p, f"unfused params M={M}")
