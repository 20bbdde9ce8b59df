"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's formula: they check closed forms, special
cases that reduce to something exact, figures the pages print, library
routines (torch's CPU bf16 cast) and brute force on tiny inputs.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import AdamW

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


def bf16_bits(values) -> np.ndarray:
    """Exact bf16 codes of values that are exactly representable in bf16."""
    f = np.asarray(values, np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def f32(x) -> np.float32:
    return np.float32(x)


# ---------------------------------------------------------------- bf16 -----

def _stratified_f32_bits(rng, per_exp=64):
    """Every exponent (incl. subnormal and inf/NaN), random mantissas, both
    signs, plus the exact rounding ties and the overflow boundary."""
    out = []
    for e in range(256):
        mant = rng.integers(0, 1 << 23, per_exp, dtype=np.uint32)
        for s in (0, 1):
            out.append((s << 31) | (e << 23) | mant)
        # ties: low 16 bits exactly 0x8000, both parities of bit 16
        out.append(np.array([(e << 23) | 0x8000, (e << 23) | 0x18000,
                             (1 << 31) | (e << 23) | 0x8000, (e << 23) | 0x7FFF,
                             (e << 23) | 0x8001], np.uint32))
    out.append(np.array([0, 0x80000000, 0x7F7F7FFF, 0x7F7F8000, 0x7F7F8001, 0x7F7FFFFF,
                         0x00000001, 0x00008000, 0x00018000, 0x007FFFFF], np.uint32))
    return np.concatenate(out).astype(np.uint32)


def test_bf16_rne_matches_torch_cast():
    """The oracle's round-to-nearest-even equals torch's CPU float->bfloat16
    cast (a library routine) on a stratified sample of every exponent."""
    rng = np.random.default_rng(1)
    u = _stratified_f32_bits(rng)
    x = u.view(np.float32)
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN with its sign
    back = oracle.bf16_to_f32(ours[nan])
    assert np.all(np.isnan(back))
    assert np.array_equal(ours[nan] >> 15, (u[nan] >> 31).astype(np.uint16))


def test_bf16_rne_ties_and_overflow():
    one_tie = f32(1.0 + 2.0 ** -8)          # halfway between 1 and 1+2^-7
    odd_tie = f32(1.0 + 3 * 2.0 ** -8)      # halfway between 1+2^-7 and 1+2^-6
    r = oracle.bf16_to_f32(oracle.f32_to_bf16(np.array([one_tie, odd_tie, -one_tie], np.float32)))
    assert r.tolist() == [1.0, 1.0 + 2.0 ** -6, -1.0]
    big = np.array([3.3895314e38, 3.40282e38], np.float32)  # bf16 max, beyond half ulp
    codes = oracle.f32_to_bf16(big)
    assert codes.tolist() == [0x7F7F, 0x7F80]


def test_bf16_to_f32_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f32(codes)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ---------------------------------------------------------------- plan -----

@pytest.mark.parametrize("n,M,align,P,s", [
    (1_048_576, 4, 128, 1_048_576, 262_144),            # tiny: shards of 262,144
    (124_439_808, 8, 1, 124_439_808, 15_554_976),        # GPT-2-small-sized, equal shards
    (1_300_000_000, 8, 128, 1_300_000_768, 162_500_096),  # 1.3B padded to a multiple of 8*128
    (7_500_000_000, 64, 1, 7_500_000_000, 117_187_500),  # 7.5B over 64 ranks
    (872_448_000, 8, 128, 872_448_000, 109_056_000),     # 4 Llama-style layers
])
def test_plan_workloads(n, M, align, P, s):
    assert oracle.plan(n, M, align) == (P, s)


def test_plan_invariants_sweep():
    for n in [1, 2, 7, 8, 9, 63, 64, 65, 1000, 4099, 10**6 + 3]:
        for M in [1, 2, 3, 4, 5, 7, 8, 16, 64]:
            for a in [1, 8, 128]:
                P, s = oracle.plan(n, M, a)
                assert P % (M * a) == 0 and 0 <= P - n < M * a and s * M == P
    with pytest.raises(ValueError):
        oracle.plan(0, 4, 1)


def llama_layer_numels(d=4096, kv=1024, ffn=14336):
    return [d, d * d, d * kv, d * kv, d * d, d, d * ffn, d * ffn, ffn * d]


def test_segments_llama_layers_cover_exactly():
    numels = llama_layer_numels() * 4
    n = sum(numels)
    assert n == 872_448_000 and sum(llama_layer_numels()) == 218_112_000
    P, s = oracle.plan(n, 8, 128)
    starts = np.cumsum([0] + numels[:-1])
    covered = 0
    for i in range(8):
        segs = oracle.segments(numels, s, i)
        pos = 0
        for (k, toff, soff, ln) in segs:
            assert soff == pos and ln > 0 and toff + ln <= numels[k]
            assert starts[k] + toff == i * s + soff
            pos += ln
        assert pos == min(s, n - i * s)
        covered += pos
    assert covered == n
    # shard cuts cross tensors: shard 0 ends strictly inside a tensor
    k, toff, _, ln = oracle.segments(numels, s, 0)[-1]
    assert toff + ln < numels[k]


def test_segments_brute_force_tiny():
    rng = np.random.default_rng(5)
    for _ in range(50):
        nt = int(rng.integers(1, 6))
        numels = [int(x) for x in rng.integers(1, 20, nt)]
        n = sum(numels)
        M = int(rng.integers(1, 6))
        P, s = oracle.plan(n, M, int(rng.choice([1, 2, 4])))
        owner = [(k, o) for k, ne in enumerate(numels) for o in range(ne)]
        for i in range(M):
            got = []
            for (k, toff, soff, ln) in oracle.segments(numels, s, i):
                got += [(k, toff + q) for q in range(ln)]
            assert got == owner[i * s: min((i + 1) * s, n)]


# -------------------------------------------------------------- memory -----

def test_memory_matches_pages_table_and_example():
    g = json.load(open(GOLDEN))
    t = g["bytes_per_param_table"]
    assert t["bf16_param"] + t["bf16_grad"] + t["fp32_master"] + t["adam_m"] + t["adam_v"] == t["total"] == 16
    naive, _ = oracle.memory(1, 1)
    assert naive == t["total"]
    ex = g["naive_dp_7p5b_on_64"]
    P, s = oracle.plan(ex["params"], ex["gpus"], 1)
    naive, z1 = oracle.memory(ex["params"], s)
    assert naive == 120 * 10**9 and naive / 1e9 == pytest.approx(ex["approx_gb_per_gpu"])
    assert naive / 1e9 > ex["a100_gb"]
    assert z1 == 4 * 7_500_000_000 + 12 * 117_187_500 == 31_406_250_000
    # optimizer state per rank is 1/M of the unsharded 12 bytes/param
    for M in [1, 2, 8, 64]:
        P, s = oracle.plan(10**6, M, 1)
        naive, z1 = oracle.memory(10**6, s)
        assert z1 - 4 * 10**6 == 12 * 10**6 // M


# ------------------------------------------------------ reduce + scale -----

@pytest.mark.parametrize("B,M,S", [(32, 4, 1.0), (64, 8, 1.0), (32, 4, 65536.0), (8, 8, 4096.0)])
def test_reduce_scale_is_the_batch_mean(B, M, S):
    """Naive DP SGD equation: (1/B) * sum over all B samples.  M replicas each
    hold the sum of their B/M per-sample gradients (times the loss scale S);
    the reduce-scatter output must be exactly the batch mean."""
    rng = np.random.default_rng(B * M)
    n = 257
    per_sample = rng.integers(-8, 9, size=(B, n)) * Fraction(1, 16)
    replica_sums = [per_sample[r * (B // M):(r + 1) * (B // M)].sum(axis=0) for r in range(M)]
    grads = [bf16_bits([float(x * int(S)) for x in rs]) for rs in replica_sums]
    inv = oracle.adamw_constants(AdamW(global_batch=B, loss_scale=S))["inv"]
    got, flag = oracle.reduce_scatter(grads, n, n, float(inv))
    mean = per_sample.sum(axis=0) / B
    assert flag == 0
    assert [Fraction(float(x)) for x in got] == list(mean)


def test_reduce_order_is_rank_order_left_fold():
    """The chosen reading: fp32 left fold starting from rank 0.  2^24 + 1 + 1
    gives 2^24 in that order (each +1 is a tie that rounds to even)."""
    grads = [bf16_bits([2.0 ** 24]), bf16_bits([1.0]), bf16_bits([1.0])]
    got, _ = oracle.reduce_scatter(grads, 1, 1, 1.0)
    assert got[0] == 2.0 ** 24
    got, _ = oracle.reduce_scatter(grads[::-1], 1, 1, 1.0)
    assert got[0] == 2.0 ** 24 + 2


def test_allreduce_order_is_rank_order_left_fold():
    """The All-Reduce sums in the same order as the reduce-scatter: an fp32
    left fold from rank 0, so 2^24 + 1 + 1 stays 2^24 and the reverse order
    gives 2^24 + 2 (fp32 outputs keep the difference visible)."""
    grads = [bf16_bits([2.0 ** 24]), bf16_bits([1.0]), bf16_bits([1.0])]
    got = oracle.allreduce(grads, 1, scale=1.0, out_bf16=False)
    assert all(float(o[0]) == 2.0 ** 24 for o in got)
    got = oracle.allreduce(grads[::-1], 1, scale=1.0, out_bf16=False)
    assert all(float(o[0]) == 2.0 ** 24 + 2 for o in got)


def test_reduce_padding_is_zero():
    grads = [bf16_bits([1.0, 2.0, 3.0])] * 2
    got, _ = oracle.reduce_scatter(grads, 2, 5, 0.5)
    assert got.tolist() == [1.0, 2.0, 0.0, 0.0, 0.0]
    assert not np.signbit(got[2:]).any()


# --------------------------------------------------------------- AdamW -----

def _state(n, seed):
    rng = np.random.default_rng(seed)
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    return master, np.zeros(n, np.float32), np.zeros(n, np.float32)


def test_adamw_sign_descent_special_case():
    """beta1 = beta2 = 0, eps = 0, wd = 0: m' = g, v' = g^2, no bias
    correction, u = g / sqrt(g^2) = sign(g) exactly, so w' = w - lr*sign(g)."""
    rng = np.random.default_rng(2)
    n = 4096
    master, m, v = _state(n, 2)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[g == 0] = 1e-3
    hp = AdamW(lr=2.0 ** -10, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.0)
    w0 = master.copy()
    oracle.adamw(g, master, m, v, hp)
    expect = (w0.astype(np.float64) - 2.0 ** -10 * np.sign(g)).astype(np.float32)
    assert np.array_equal(master, expect)
    assert np.array_equal(m, g) and np.array_equal(v, g * g)


def test_adamw_zero_gradient_is_pure_decoupled_decay():
    """g = 0 from m = v = 0: m, v stay 0, the Adam term is 0/(0+eps) = 0 and
    the weight only decays, w' = round(w * (1 - lr*wd)); lr*wd chosen so that
    1 - lr*wd = 1 - 2^-14 is exact and the product is exact in double."""
    n = 2048
    master, m, v = _state(n, 3)
    hp = AdamW(lr=2.0 ** -10, weight_decay=2.0 ** -4, eps=1e-8)
    w = master.copy()
    for t in range(1, 6):
        oracle.adamw(np.zeros(n, np.float32), master, m, v, AdamW(**{**hp.__dict__, "step": t}))
        w = (w.astype(np.float64) * (1.0 - 2.0 ** -14)).astype(np.float32)
        assert np.array_equal(master, w)
        assert not m.any() and not v.any()


def test_adamw_constant_gradient_closed_form():
    """With a constant gradient g from m = v = 0, bias correction makes
    m-hat = g and v-hat = g^2 at every step t (exact arithmetic), so
    w_t = c w_{t-1} - lr * g / (|g| + eps), c = 1 - lr*wd.  A missing or
    shifted bias correction, or swapped betas, is off by O(1)."""
    n = 1024
    rng = np.random.default_rng(4)
    master, m, v = _state(n, 4)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    hp = AdamW(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    w = master.astype(np.float64)
    c = 1.0 - 1e-3 * 0.1
    u = g.astype(np.float64) / (np.abs(g.astype(np.float64)) + 1e-8)
    for t in range(1, 11):
        oracle.adamw(g, master, m, v, AdamW(**{**hp.__dict__, "step": t}))
        w = c * w - hp.lr * u
        assert np.max(np.abs(master - w)) < 1e-8 + 2e-6 * hp.lr * t


def test_adamw_gradient_then_zero_separates_the_betas():
    """Step 1 with g, step 2 with 0: m-hat_2 = beta1 g/(1+beta1),
    v-hat_2 = beta2 g^2/(1+beta2).  beta1 != beta2, so swapping them fails."""
    n = 512
    rng = np.random.default_rng(6)
    master, m, v = _state(n, 6)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    b1, b2, lr, eps, wd = 0.9, 0.95, 1e-3, 1e-8, 0.0
    hp = AdamW(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wd)
    w0 = master.astype(np.float64)
    oracle.adamw(g, master, m, v, AdamW(**{**hp.__dict__, "step": 1}))
    oracle.adamw(np.zeros(n, np.float32), master, m, v, AdamW(**{**hp.__dict__, "step": 2}))
    b1f, b2f = float(f32(b1)), float(f32(b2))
    gd = g.astype(np.float64)
    u1 = gd / (np.abs(gd) + eps)
    u2 = (b1f / (1 + b1f)) * gd / (math.sqrt(b2f / (1 + b2f)) * np.abs(gd) + eps)
    expect = w0 - lr * u1 - lr * u2
    assert np.max(np.abs(master - expect)) < 1e-8 + 4e-6 * lr
    swapped = w0 - lr * u1 - lr * (b2f / (1 + b2f)) * gd / (math.sqrt(b1f / (1 + b1f)) * np.abs(gd) + eps)
    assert np.max(np.abs(master - swapped)) > 1e-5 * lr


def test_adamw_eps_is_added_after_the_square_root():
    """t = 1 from zero state: u = g/(|g| + eps) exactly in real arithmetic;
    with eps comparable to |g| the eps-inside-sqrt variant differs by O(1)."""
    n = 256
    g = np.linspace(-2e-3, 2e-3, n).astype(np.float32)
    master, m, v = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    eps, lr = 1e-3, 1.0
    oracle.adamw(g, master, m, v, AdamW(lr=lr, eps=eps, weight_decay=0.0, step=1))
    gd = g.astype(np.float64)
    expect = -lr * gd / (np.abs(gd) + float(f32(eps)))
    assert np.max(np.abs(master - expect)) < 4e-7
    inside = -lr * gd / np.sqrt(gd * gd + float(f32(eps)))
    assert np.max(np.abs(master - inside)) > 0.1


def test_adamw_general_within_fp64_evaluation():
    """Random state and gradients: each output within a few fp32 ulps of an
    fp64 evaluation of the AdamW update."""
    rng = np.random.default_rng(7)
    n = 20000
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = (rng.random(n) * 1e-7).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    hp = AdamW(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=7)
    b1, b2 = float(f32(hp.beta1)), float(f32(hp.beta2))
    gd, md, vd, wd_ = (a.astype(np.float64) for a in (g, m, v, master))
    m1 = b1 * md + (1 - b1) * gd
    v1 = b2 * vd + (1 - b2) * gd * gd
    u = (m1 / (1 - b1 ** 7)) / (np.sqrt(v1 / (1 - b2 ** 7)) + float(f32(hp.eps)))
    w1 = wd_ * (1 - float(f32(hp.lr)) * float(f32(hp.weight_decay))) - float(f32(hp.lr)) * u
    oracle.adamw(g, master, m, v, hp)
    # bounds scale with the terms' magnitudes (the m sum can cancel)
    assert np.all(np.abs(m - m1) <= 2.0 ** -22 * (b1 * np.abs(md) + (1 - b1) * np.abs(gd)))
    assert np.all(np.abs(v - v1) <= 2.0 ** -22 * np.abs(v1))
    assert np.all(np.abs(master - w1) <= 2.0 ** -22 * np.abs(wd_) + 1e-6 * hp.lr * np.abs(u))


# ------------------------------------------------ sharding and identity ----

def _unsharded_numpy_reference(grads, n, P, master, m, v, hp):
    """Independent brute force: all P elements at once in numpy float32 (no
    shards), for checking the partition, padding and assembly."""
    f = [np.zeros(P, np.float32) for _ in grads]
    for r, g in enumerate(grads):
        f[r][:n] = (g.astype(np.uint32) << 16).view(np.float32)
    s = f[0].copy()
    for r in range(1, len(grads)):
        s = s + f[r]
    c = oracle.adamw_constants(hp)
    g = s * c["inv"]
    b1, b2 = f32(hp.beta1), f32(hp.beta2)
    m1 = b1 * m + c["omb1"] * g
    v1 = b2 * v + c["omb2"] * (g * g)
    u = (m1 / c["bc1"]) / (np.sqrt(v1 / c["bc2"]) + f32(hp.eps))
    w = master * c["cdec"] - f32(hp.lr) * u
    return w, m1, v1


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8, 64])
def test_sharded_equals_unsharded_brute_force(M):
    rng = np.random.default_rng(M)
    for n in sorted({1, 7, 8, 9, max(M - 1, 1), M + 1, 1000, 4099}):
        for align in (1, 8, 128):
            P, s = oracle.plan(n, M, align)
            grads = [oracle.f32_to_bf16((rng.standard_normal(n) * 1e-2).astype(np.float32))
                     for _ in range(M)]
            master = np.zeros(P, np.float32)
            master[:n] = rng.standard_normal(n) * 0.02
            m = np.zeros(P, np.float32)
            v = np.zeros(P, np.float32)
            hp = AdamW(global_batch=max(M, 4), step=1)
            w_ref, m_ref, v_ref = _unsharded_numpy_reference(grads, n, P, master.copy(), m.copy(), v.copy(), hp)
            params = np.zeros(n, np.uint16)
            for i in range(M):
                lo, hi = i * s, (i + 1) * s
                nv = max(0, min(hi, n) - lo)
                sub = [np.ascontiguousarray(g[lo:lo + nv]) for g in grads]
                mm, mv, mw = m[lo:hi].copy(), v[lo:hi].copy(), master[lo:hi].copy()
                pp = np.zeros(nv, np.uint16)
                oracle.zero1_step(sub, nv, mw, mm, mv, pp, hp)
                master[lo:hi], m[lo:hi], v[lo:hi] = mw, mm, mv
                params[lo:lo + nv] = pp
            assert np.array_equal(master.view(np.uint32), w_ref.view(np.uint32))
            assert np.array_equal(m.view(np.uint32), m_ref.view(np.uint32))
            assert np.array_equal(v.view(np.uint32), v_ref.view(np.uint32))
            assert np.array_equal(params, oracle.f32_to_bf16(w_ref[:n]))
            # padding stays exactly +0
            assert not master[n:].view(np.uint32).any() and not m[n:].any() and not v[n:].any()


def test_allreduce_equals_reduce_scatter_then_all_gather():
    """All-Reduce == Reduce-Scatter + All-Gather, bitwise, for bf16 outputs."""
    rng = np.random.default_rng(11)
    for M, n, align in [(4, 1000, 8), (8, 4099, 1), (3, 17, 128)]:
        P, s = oracle.plan(n, M, align)
        grads = [oracle.f32_to_bf16((rng.standard_normal(n)).astype(np.float32)) for _ in range(M)]
        ar = oracle.allreduce(grads, n, scale=0.25)
        gathered = np.zeros(n, np.uint16)
        for i in range(M):
            lo = i * s
            nv = max(0, min(lo + s, n) - lo)
            shard, _ = oracle.reduce_scatter([np.ascontiguousarray(g[lo:lo + nv]) for g in grads], nv, nv, 0.25)
            gathered[lo:lo + nv] = oracle.f32_to_bf16(shard)
        for out in ar:
            assert np.array_equal(out, gathered)


def test_zero1_step_equals_allreduce_then_unsharded_adamw():
    """ZeRO-1 changes where the state lives, not the values: the sharded
    step equals a fp32 All-Reduce followed by one unsharded AdamW."""
    rng = np.random.default_rng(12)
    M, n, align = 8, 5000, 128
    P, s = oracle.plan(n, M, align)
    grads = [oracle.f32_to_bf16((rng.standard_normal(n) * 1e-3).astype(np.float32)) for _ in range(M)]
    hp = AdamW(global_batch=512, step=3)
    master0 = np.zeros(P, np.float32)
    master0[:n] = rng.standard_normal(n) * 0.02
    m0 = (rng.standard_normal(P) * 1e-5).astype(np.float32)
    v0 = (rng.random(P) * 1e-9).astype(np.float32)
    m0[n:] = 0
    v0[n:] = 0
    inv = float(oracle.adamw_constants(hp)["inv"])
    g = np.zeros(P, np.float32)
    g[:n] = oracle.allreduce(grads, n, scale=inv, out_bf16=False)[0]
    wa, ma, va = master0.copy(), m0.copy(), v0.copy()
    oracle.adamw(g, wa, ma, va, hp)
    pa = np.zeros(n, np.uint16)
    oracle.all_gather(wa, n, pa)
    wb, mb, vb = master0.copy(), m0.copy(), v0.copy()
    pb = np.zeros(n, np.uint16)
    for i in range(M):
        lo, hi = i * s, (i + 1) * s
        nv = max(0, min(hi, n) - lo)
        sw, sm, sv = wb[lo:hi].copy(), mb[lo:hi].copy(), vb[lo:hi].copy()
        pp = np.zeros(nv, np.uint16)
        oracle.zero1_step([np.ascontiguousarray(x[lo:lo + nv]) for x in grads], nv, sw, sm, sv, pp, hp)
        wb[lo:hi], mb[lo:hi], vb[lo:hi] = sw, sm, sv
        pb[lo:lo + nv] = pp
    for a, b in [(wa, wb), (ma, mb), (va, vb)]:
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.array_equal(pa, pb)


# ------------------------------------------------------------ overflow -----

BF16_MAX = 0x7F7F
INF, NINF, NAN = 0x7F80, 0xFF80, 0x7FC0


@pytest.mark.parametrize("codes,expect", [
    ([INF, 0x3F80], 1),
    ([NINF, 0x3F80], 1),
    ([NAN, 0x3F80], 1),
    ([INF, NINF], 1),                 # inf + -inf = NaN
    ([BF16_MAX, BF16_MAX], 1),        # finite bf16s whose fp32 sum overflows
    ([0x8000, 0x8000], 0),            # -0 + -0
    ([BF16_MAX, 0xFF7F], 0),          # max + -max = 0
    ([0x7F00, 0x7F00], 1),            # 2^127 + 2^127 overflows fp32
    ([0x7E80, 0x7E80], 0),            # 2^126 + 2^126 = 2^127, finite
])
def test_overflow_special_cases(codes, expect):
    grads = [np.array([0x3F80, c, 0x3F80], np.uint16) for c in codes]
    assert oracle.overflow_check(grads, 3) == expect
    _, f = oracle.reduce_scatter(grads, 3, 4, 1.0)
    assert f == expect


def test_overflow_ignores_padding_and_skip_writes_nothing():
    grads = [np.array([0x3F80, 0x3F80, INF], np.uint16)] * 2
    assert oracle.overflow_check(grads, 2) == 0
    assert oracle.overflow_check(grads, 3) == 1
    master, m, v = _state(3, 9)
    m[:] = 1e-4
    v[:] = 1e-8
    params = np.full(3, 0x1234, np.uint16)
    snap = [a.copy() for a in (master, m, v, params)]
    flag = np.array([oracle.overflow_check(grads, 3)], np.uint32)
    oracle.zero1_step(grads, 3, master, m, v, params, AdamW(step=3), flag=flag, skip_if_flag=True)
    for a, b in zip((master, m, v, params), snap):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert flag[0] == 1
    # flag clear + skip requested: the step runs and the flag is only read
    flag[0] = 0
    oracle.zero1_step([g[:2].copy() for g in grads], 2, master, m, v, params, AdamW(step=3), flag=flag,
                      skip_if_flag=True)
    assert flag[0] == 0 and not np.array_equal(master, snap[0])


def _nearest_f32(x: Fraction) -> np.float32:
    """The float32 nearest to the exact rational x (ties to the even code)."""
    c = np.float32(float(x))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = min(abs(Fraction(float(y)) - x) for y in cands)
    near = [y for y in cands if abs(Fraction(float(y)) - x) == best]
    return min(near, key=lambda y: int(np.array(y, np.float32).view(np.uint32)) & 1)


def test_inverse_batch_scale_is_rounded_once():
    """1/(B*S), evaluated in double and then rounded to fp32, equals the exact
    quotient rounded once to fp32 on these cases, also where B*S itself has
    no fp32 representation (2^24 + 1, 3 * (2^24 + 1) * 2^10)."""
    for B, S in [(2 ** 24 + 1, 1.0), (3 * (2 ** 24 + 1), 1024.0), (1000, 3.0), (1024, 65536.0)]:
        got = np.float32(oracle.adamw_constants(AdamW(global_batch=B, loss_scale=S))["inv"])
        want = _nearest_f32(Fraction(1, B) / Fraction(S))
        assert got.view(np.uint32) == want.view(np.uint32), (B, S)


def test_bias_correction_power():
    """beta^t: exact for powers of two, t = 0 and t = 1; otherwise within the
    square-and-multiply error bound of the exact rational power: each squaring
    doubles the relative error, so it is at most about (t + 2 log2 t) units
    of 2^-53."""
    for t in [0, 1, 2, 3, 7, 64, 1000, 1023, 10**6]:
        assert oracle.pow_int(0.5, t) == math.ldexp(1.0, -t)
    assert oracle.pow_int(0.9, 0) == 1.0 and oracle.pow_int(0.9, 1) == 0.9
    for b in [float(f32(0.9)), float(f32(0.95)), float(f32(0.999))]:
        for t in [2, 3, 5, 10, 17, 100, 999, 1000, 4097]:
            exact = Fraction(b) ** t
            got = Fraction(oracle.pow_int(b, t))
            rounds = t + 2 * t.bit_length() + 1
            assert abs(got - exact) <= exact * Fraction(rounds, 2 ** 53)
            assert abs(got - exact) > 0 or t < 3      # not trivially exact


def test_deepspeed_hyperparameters_from_the_pages():
    """The pages' AdamW block (lr 1e-3, betas 0.9/0.999, eps 1e-8, wd 0.01)
    runs through the constants: 1-beta^t in fp32 and the decay factor."""
    g = json.load(open(GOLDEN))["deepspeed_adamw"]
    hp = AdamW(lr=g["lr"], beta1=g["betas"][0], beta2=g["betas"][1], eps=g["eps"],
               weight_decay=g["weight_decay"], global_batch=1024, step=1)
    c = oracle.adamw_constants(hp)
    assert c["bc1"] == f32(1 - float(f32(0.9)))
    assert c["bc2"] == f32(1 - float(f32(0.999)))
    assert c["cdec"] == f32(1 - float(f32(1e-3)) * float(f32(0.01)))
    assert c["inv"] == f32(2.0 ** -10)
