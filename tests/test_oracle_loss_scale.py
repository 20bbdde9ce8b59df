"""Pins of the oracle's dynamic loss scaler against the fp16 block the pages
print ("五维并行实战" section 4.2: loss_scale 0 = dynamic, initial_scale_power 12,
loss_scale_window 1000, hysteresis 2, min_loss_scale 1) and the invariants of
the reading taken (skipped attempts write nothing and do not advance t)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import AdamW, LossScalePolicy, Scaler

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


def pages_policy() -> LossScalePolicy:
    g = json.load(open(GOLDEN))["deepspeed_fp16"]
    assert g["loss_scale"] == 0          # 0 selects the dynamic scaler
    return LossScalePolicy(initial_scale=2.0 ** g["initial_scale_power"], factor=2.0,
                           window=g["loss_scale_window"], hysteresis=g["hysteresis"],
                           min_scale=float(g["min_loss_scale"]))


def run(seq, pol, first_step=1):
    sc = Scaler.start(pol, first_step)
    for f in seq:
        sc.update(f, pol)
    return sc


def test_pages_config_grows_after_a_full_window():
    pol = pages_policy()
    assert Scaler.start(pol).scale == 4096.0
    assert run([0] * 999, pol).scale == 4096.0
    sc = run([0] * 1000, pol)
    assert sc.scale == 8192.0 and sc.step == 1001 and sc.good == 0
    assert run([0] * 3000, pol).scale == 4096.0 * 8


def test_hysteresis_two_tolerates_one_overflow():
    pol = pages_policy()
    sc = run([1], pol)
    assert sc.scale == 4096.0 and sc.hyst_left == 1 and sc.step == 1 and sc.skipped == 1
    sc = run([1, 0, 0, 0, 1], pol)                   # clean attempts do not refill it
    assert sc.scale == 2048.0 and sc.hyst_left == 2 and sc.step == 4 and sc.skipped == 2
    sc = run([1, 1, 1, 1], pol)
    assert sc.scale == 1024.0


def test_growth_refills_the_hysteresis():
    """After a full window the scale grows and the hysteresis is back to its
    full count: one overflow right after growth only uses one unit of it."""
    pol = LossScalePolicy(initial_scale=16.0, window=2, hysteresis=2)
    sc = run([1, 0, 0], pol)
    assert sc.scale == 32.0 and sc.hyst_left == 2 and sc.good == 0
    sc = run([1, 0, 0, 1], pol)
    assert sc.scale == 32.0 and sc.hyst_left == 1
    sc = run([1, 0, 0, 1, 1], pol)
    assert sc.scale == 16.0 and sc.hyst_left == 2


def test_overflow_restarts_the_window():
    pol = LossScalePolicy(initial_scale=16.0, window=4, hysteresis=2)
    assert run([0, 0, 0, 1, 0, 0, 0], pol).scale == 16.0
    assert run([0, 0, 0, 1, 0, 0, 0, 0], pol).scale == 32.0


def test_min_scale_and_fp32_ceiling():
    pol = LossScalePolicy(initial_scale=2.0, window=1000, hysteresis=1, min_scale=1.0)
    assert run([1, 1, 1], pol).scale == 1.0
    top = LossScalePolicy(initial_scale=2.0 ** 127, window=1, hysteresis=1)
    assert run([0, 0], top).scale == 2.0 ** 127     # 2^128 is not finite: no growth


def test_invariants_on_random_sequences():
    rng = np.random.default_rng(3)
    for k in range(20):
        pol = LossScalePolicy(initial_scale=2.0 ** int(rng.integers(0, 20)), window=int(rng.integers(1, 30)),
                              hysteresis=int(rng.integers(1, 4)), min_scale=2.0 ** int(rng.integers(-2, 3)))
        seq = (rng.random(500) < rng.random() * 0.3).astype(int)
        sc = run(seq, pol, first_step=7)
        assert sc.attempts == 500 and sc.skipped == seq.sum() and sc.step == 7 + (500 - seq.sum())
        e = np.log2(sc.scale)
        assert e == int(e) and sc.scale >= min(pol.min_scale, pol.initial_scale)


def test_dynamic_attempt_skips_or_equals_the_plain_step():
    rng = np.random.default_rng(4)
    M, n = 4, 3001
    pol = LossScalePolicy(initial_scale=1024.0, window=2, hysteresis=1)
    sc = Scaler.start(pol, 1)
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    params = np.zeros(n, np.uint16)
    hp = AdamW(global_batch=64)
    for attempt in range(6):
        grads = [oracle.f32_to_bf16((rng.standard_normal(n) * 1e-3 * sc.scale).astype(np.float32))
                 for _ in range(M)]
        if attempt in (2, 3):
            grads[attempt % M][100 * attempt] = 0x7F80
        before = [a.copy() for a in (master, m, v, params)]
        S, t = sc.scale, sc.step
        f = oracle.zero1_dynamic_attempt(grads, n, master, m, v, params, hp, sc, pol)
        assert f == (1 if attempt in (2, 3) else 0)
        if f:
            for a, b in zip((master, m, v, params), before):
                assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
            assert sc.step == t
        else:
            w2, m2, v2, p2 = (b.copy() for b in before)
            oracle.zero1_step(grads, n, w2, m2, v2, p2, AdamW(global_batch=64, loss_scale=S, step=t))
            assert np.array_equal(master, w2) and np.array_equal(params, p2)
            assert sc.step == t + 1
    assert sc.skipped == 2
