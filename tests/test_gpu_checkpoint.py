"""Checkpoint and resume: the optimizer state of a shard is its fp32
master/m/v, the step counter and (for the dynamic path) the scaler.  Ten
steps in a row must equal five steps, a save to disk, a load into fresh
buffers and five more steps, bit for bit ("CS336 Lecture 7: Parallelism 1"
case studies: long runs are interrupted and resumed), and both must be the
oracle's run."""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, oracle_hp, u16
from test_gpu_parity import make_grads, make_state, oracle_step

pytestmark = pytest.mark.gpu


def test_ten_steps_equal_five_save_load_five(cuda_device, tmp_path):
    dev = cuda_device
    M, n = 8, 200_003
    plan = z.zero1_plan(n, M, 128)
    P = plan.padded_n
    grads = [make_grads(M, n, 1e-3, 41, t, dev) for t in range(1, 11)]
    run = make_state(n, P, 40, dev)
    ref = [t.clone() for t in run]
    o = [f32(t).copy() for t in run]
    p_ref = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    for t in range(1, 11):
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads[t - 1], *ref, p_ref, z.AdamW(global_batch=512, step=t))
    p = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    for t in range(1, 6):
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads[t - 1], *run, p, z.AdamW(global_batch=512, step=t))
    torch.save({"master": run[0].cpu(), "m": run[1].cpu(), "v": run[2].cpu(), "params": p.cpu(), "next_step": 6,
                "plan": (plan.n, plan.M, plan.align)}, tmp_path / "shard.pt")
    del run, p
    ck = torch.load(tmp_path / "shard.pt")
    plan2 = z.zero1_plan(*ck["plan"])
    state = [ck[k].to(dev) for k in ("master", "m", "v")]
    p2 = ck["params"].to(dev)
    for t in range(ck["next_step"], 11):
        z.zero1_reduce_scatter_adamw_allgather(plan2, 0, M, grads[t - 1], *state, p2, z.AdamW(global_batch=512, step=t))
    torch.cuda.synchronize()
    for a, b in zip(state, ref):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(p2.view(torch.int16), p_ref.view(torch.int16))
    # and both are the oracle's ten steps
    for t in range(1, 11):
        o_p = oracle_step(plan, [u16(g) for g in grads[t - 1]], *o, oracle_hp(z.AdamW(global_batch=512, step=t)))
    for a, want, what in zip(state, o, ("master", "m", "v")):
        assert_f32_bits(f32(a), want, f"resumed {what} against the oracle")
    assert_bf16_bits(u16(p2), o_p, "resumed params against the oracle")


def test_dynamic_scaler_resumes(cuda_device, tmp_path):
    dev = cuda_device
    M, n = 4, 50_000
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=256.0, window=3, hysteresis=1)
    hp = z.AdamW(global_batch=64, step=1)
    grads = [make_grads(M, n, 1e-3 * 256, 51, t, dev) for t in range(8)]
    grads[2][1][7] = float("inf")
    grads[6][0][9] = float("inf")

    def fresh():
        st = make_state(n, P, 50, dev)
        sc = z.new_scaler(dev)
        z.zero1_scaler_init(sc, policy, hp)
        return st, sc, torch.zeros(n, dtype=torch.bfloat16, device=dev), torch.empty(P, dtype=torch.float32,
                                                                                      device=dev)

    ref, sref, pref, sums = fresh()
    for k in range(8):
        z.zero1_step_dynamic(plan, 0, M, grads[k], *ref, pref, hp, sref, policy, sums)
    run, srun, prun, sums2 = fresh()
    for k in range(4):
        z.zero1_step_dynamic(plan, 0, M, grads[k], *run, prun, hp, srun, policy, sums2)
    torch.save({"state": [x.cpu() for x in run], "scaler": srun.cpu(), "params": prun.cpu()}, tmp_path / "dyn.pt")
    ck = torch.load(tmp_path / "dyn.pt")
    state = [x.to(dev) for x in ck["state"]]
    sc = ck["scaler"].to(dev)
    p = ck["params"].to(dev)
    for k in range(4, 8):
        z.zero1_step_dynamic(plan, 0, M, grads[k], *state, p, hp, sc, policy, sums2)
    torch.cuda.synchronize()
    for a, b in zip(state, ref):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(p.view(torch.int16), pref.view(torch.int16))
    assert z.scaler_state(sc) == z.scaler_state(sref)
    assert z.scaler_state(sc)["skipped"] == 2
    # and the oracle's eight attempts give the same state, parameters and scaler
    o = [f32(t).copy() for t in make_state(n, P, 50, dev)]
    o_p = np.zeros(n, np.uint16)
    o_pol = oracle.LossScalePolicy(initial_scale=policy.initial_scale, factor=policy.factor, window=policy.window,
                                   hysteresis=policy.hysteresis, min_scale=policy.min_scale)
    o_sc = oracle.Scaler.start(o_pol, 1)
    for k in range(8):
        oracle.zero1_dynamic_attempt([u16(g) for g in grads[k]], n, *o, o_p, oracle_hp(hp), o_sc, o_pol)
    for a, want, what in zip(state, o, ("master", "m", "v")):
        assert_f32_bits(f32(a), want, f"resumed {what} against the oracle")
    assert_bf16_bits(u16(p), o_p, "resumed params against the oracle")
    st = z.scaler_state(sc)
    assert (st["scale"], st["step"], st["skipped"]) == (o_sc.scale, o_sc.step, o_sc.skipped)


def test_pingpong_resumes_from_the_current_copy(cuda_device, tmp_path):
    """A ping-pong checkpoint is the scaler (its `current` field included) and
    the copy it names; the other copy is not saved.  On load the state goes
    into the copy the saved scaler names, and the run continues bit for bit
    as if never interrupted, skipped attempts included."""
    dev = cuda_device
    M, n = 8, 70_001
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=512.0, window=2, hysteresis=1)
    hp = z.AdamW(global_batch=64, step=1)
    grads = [make_grads(M, n, 1e-3 * 512, 61, t, dev) for t in range(9)]
    grads[3][2][11] = float("inf")
    grads[7][5][13] = float("nan")

    def fresh():
        st = make_state(n, P, 60, dev, nonzero_moments=True)
        pairs = [[x, torch.zeros_like(x)] for x in st]
        sc = z.new_scaler(dev)
        z.zero1_scaler_init(sc, policy, hp)
        return pairs, sc, st[0][:n].to(torch.bfloat16)

    ref, sref, pref = fresh()
    for k in range(9):
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads[k], *ref, pref, hp, sref, policy)
    run, srun, prun = fresh()
    for k in range(5):
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads[k], *run, prun, hp, srun, policy)
    cur = z.current_state(srun, *run)
    torch.save({"state": [x.cpu() for x in cur], "scaler": srun.cpu(), "params": prun.cpu()}, tmp_path / "pp.pt")
    ck = torch.load(tmp_path / "pp.pt")
    sc = ck["scaler"].to(dev)
    k_cur = z.scaler_state(sc)["current"]
    pairs = [[torch.full((P,), float("nan"), device=dev) for _ in range(2)] for _ in range(3)]
    for pair, saved in zip(pairs, ck["state"]):
        pair[k_cur].copy_(saved)
    p = ck["params"].to(dev)
    for k in range(5, 9):
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads[k], *pairs, p, hp, sc, policy)
    torch.cuda.synchronize()
    for a, b in zip(z.current_state(sc, *pairs), z.current_state(sref, *ref)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(p.view(torch.int16), pref.view(torch.int16))
    assert z.scaler_state(sc) == z.scaler_state(sref)
    assert z.scaler_state(sc)["skipped"] == 2
