"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (one call over the workload's shard range).

The oracle cannot run 1.3e9 elements in seconds, but the step is element-wise:
a sample of indices (random, plus every shard edge, the end of the real
parameters and the ragged tail) is gathered before each step, the oracle
runs on that compact sample, and the GPU's outputs at the same indices must
match bit for bit.  The overflow flag is checked through properties that
hold at any size (finite draws cannot overflow; an injected +inf must set
it), and a skipped step must leave every byte of state unchanged.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth
from zero_sharded_mixed_zero1_gb300 import workloads as W
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, oracle_hp, u16

pytestmark = pytest.mark.gpu


def sample_indices(plan, sb, se, L, nv, k=1 << 16, seed=0):
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, L, k)]
    edges = [0, L, nv] + [(i - sb) * plan.shard for i in range(sb, se + 1)]
    for e in edges:
        idx.append(np.arange(e - 64, e + 64))
    idx = np.unique(np.concatenate(idx))
    idx = idx[(idx >= 0) & (idx < L)]
    return idx[idx < nv], idx[idx >= nv]


class Run:
    """Device buffers of one workload over its shard range, plus the oracle's
    copy of the sampled elements."""

    def __init__(self, w: W.Workload, device, sample_seed=1):
        self.w = w
        self.dev = device
        self.plan = z.zero1_plan(w.n, w.M, w.align, tensor_numels=list(w.tensor_numels) or None)
        self.sb, self.se = w.shards
        self.base, self.L, self.nv = self.plan.shard_range(self.sb, self.se)
        L, nv = self.L, self.nv
        self.master = torch.zeros(L, dtype=torch.float32, device=device)
        self.master[:nv] = synth.normal_f32(nv, w.master_std, synth.seed_of(w.seed, 1), device)
        self.m = torch.zeros(L, dtype=torch.float32, device=device)
        self.v = torch.zeros(L, dtype=torch.float32, device=device)
        self.params = torch.zeros(nv, dtype=torch.bfloat16, device=device)
        self.grads = [torch.empty(nv, dtype=torch.bfloat16, device=device) for _ in range(w.M)]
        self.flag = torch.zeros(1, dtype=torch.int32, device=device)
        real, pad = sample_indices(self.plan, self.sb, self.se, L, nv, seed=sample_seed)
        self.real, self.pad = real, pad
        self.idx = torch.from_numpy(np.concatenate([real, pad])).to(device)
        self.idx_real = torch.from_numpy(real).to(device)
        self.o_master = f32(self.master[self.idx])
        self.o_m = f32(self.m[self.idx])
        self.o_v = f32(self.v[self.idx])
        self.o_params = np.zeros(self.real.size, np.uint16)    # params start at zero

    def fill_grads(self, attempt: int) -> int:
        w = self.w
        injected = 0
        for r, g in enumerate(self.grads):
            g.copy_(synth.normal_bf16(self.nv, w.grad_std * w.S, synth.seed_of(w.seed, 100 + attempt, r), self.dev))
            if attempt == w.inf_attempt:
                injected += synth.set_inf(g, w.inf_prob, synth.seed_of(w.seed, 900 + attempt, r))
        return injected

    def hp(self, t: int) -> z.AdamW:
        w = self.w
        return z.AdamW(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                       loss_scale=w.S, global_batch=w.B, step=t)

    def step(self, t: int, skip_check: bool, expect_flag: int = 0) -> None:
        """One GPU step and the oracle on the samples.  The oracle's flag is
        the expected one (known from how the gradients were drawn), never
        the GPU's."""
        hp = self.hp(t)
        g_s = [u16(g[self.idx_real]) for g in self.grads]
        self.flag.zero_()
        if skip_check:
            z.zero1_overflow_check(self.plan, self.sb, self.se, self.grads, self.flag)
        z.zero1_reduce_scatter_adamw_allgather(self.plan, self.sb, self.se, self.grads, self.master, self.m,
                                               self.v, self.params, hp, self.flag, skip_if_flag=skip_check)
        torch.cuda.synchronize()
        oflag = np.array([expect_flag if skip_check else 0], np.uint32)
        oracle.zero1_step(g_s, self.real.size, self.o_master, self.o_m, self.o_v, self.o_params,
                          oracle_hp(hp), flag=oflag, skip_if_flag=skip_check)
        assert int(self.flag.item()) == expect_flag

    def check(self, what: str) -> None:
        assert_f32_bits(f32(self.master[self.idx]), self.o_master, f"{what} master")
        assert_f32_bits(f32(self.m[self.idx]), self.o_m, f"{what} m")
        assert_f32_bits(f32(self.v[self.idx]), self.o_v, f"{what} v")
        assert_bf16_bits(u16(self.params[self.idx_real]), self.o_params, f"{what} params")


def free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", [W.TINY, W.GPT2_SMALL, W.FLAT_1P3B, W.RANK_7P5B_M64],
                         ids=lambda w: w.name)
def test_workload_steps_match_oracle_on_samples(cuda_device, w):
    run = Run(w, cuda_device)
    if w is W.TINY:        # small enough to compare every element
        run.idx = torch.arange(run.L, device=cuda_device)
        run.idx_real = torch.arange(run.nv, device=cuda_device)
        run.real, run.pad = np.arange(run.nv), np.arange(run.nv, run.L)
        run.o_master, run.o_m, run.o_v = f32(run.master), f32(run.m), f32(run.v)
        run.o_params = np.zeros(run.nv, np.uint16)
    for t in range(1, w.steps + 1):
        run.fill_grads(t)
        run.step(t, skip_check=False, expect_flag=0)   # finite normal draws cannot overflow
        run.check(f"{w.name} t={t}")
    if run.L > run.nv:       # padding stays exactly +0
        assert not torch.any(run.master[run.nv:].view(torch.int32) != 0)
    del run
    free()


def test_llama_layers_with_skipped_overflow_step(cuda_device):
    """Four Llama-style layers flattened with shard cuts crossing tensors,
    loss scale 65536: steps t = 1, 2; the third attempt's gradients hold
    +inf entries, so the check sets the flag and the step writes nothing; the
    fourth attempt runs t = 3."""
    w = W.LLAMA4
    run = Run(w, cuda_device)
    # the per-tensor segments tile the processed range exactly
    covered = 0
    for i in range(run.sb, run.se):
        segs = z.zero1_plan_segments(run.plan, list(w.tensor_numels), i)
        covered += sum(s[2] for s in segs)
        if i < run.se - 1:
            k, toff, ln = segs[-1]
            assert toff + ln <= w.tensor_numels[k]
    assert covered == run.nv
    t = 1
    for attempt in range(1, 5):
        injected = run.fill_grads(attempt)
        if attempt == w.inf_attempt:
            assert injected > 0
            snap = [x.clone() for x in (run.master, run.m, run.v, run.params)]
            run.step(t, skip_check=True, expect_flag=1)    # an injected +inf makes a sum non-finite
            for a, b in zip((run.master, run.m, run.v), snap[:3]):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32))
            assert torch.equal(run.params.view(torch.int16), snap[3].view(torch.int16))
            run.check(f"attempt {attempt} (skipped)")
            del snap
            continue                        # t is not advanced
        run.step(t, skip_check=True, expect_flag=0)
        run.check(f"attempt {attempt} t={t}")
        t += 1
    assert t == 4
    del run
    free()


def test_flat_1p3b_allreduce_equals_reduce_scatter_plus_all_gather(cuda_device):
    """The 1.3B flat buffer: naive All-Reduce of the eight replicas' gradients
    equals Reduce-Scatter + All-Gather bit for bit, and matches the oracle on
    samples."""
    w = W.FLAT_1P3B
    dev = cuda_device
    plan = z.zero1_plan(w.n, w.M, w.align)
    n = plan.n
    grads = [synth.normal_bf16(n, w.grad_std, synth.seed_of(w.seed, 500, r), dev) for r in range(w.M)]
    scale = 1.0 / w.B
    outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(w.M)]
    z.dp_allreduce(plan, grads, outs, scale)
    shards = torch.empty(plan.padded_n, dtype=torch.bfloat16, device=dev)
    z.zero1_reduce_scatter(plan, 0, w.M, grads, scale, shards)
    for r in range(w.M):
        assert torch.equal(outs[r].view(torch.int16), shards[:n].view(torch.int16))
    real, _ = sample_indices(plan, 0, w.M, plan.padded_n, n)
    idx = torch.from_numpy(real).to(dev)
    want = oracle.allreduce([u16(g[idx]) for g in grads], real.size, scale=scale)
    for r in (0, w.M - 1):
        assert_bf16_bits(u16(outs[r][idx]), want[r], f"AR out {r}")
    del outs
    gathered = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(w.M)]
    z.zero1_all_gather_shards(plan, shards, gathered)
    for r in range(w.M):
        assert torch.equal(gathered[r].view(torch.int16), shards[:n].view(torch.int16))
    del grads, gathered, shards
    free()


def test_buffers_beyond_two_to_the_31_elements(cuda_device):
    """One flat buffer longer than 2^31 elements (ragged, M = 2): 64-bit
    element indices and byte offsets above 8 GB in the fused step, the
    overflow check and a bucket crossing 2^31; checked on samples around
    2^31, the end and at random."""
    dev = cuda_device
    M, n, align = 2, 2 ** 31 + 2 ** 20 + 13, 8
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    grads = [synth.normal_bf16(n, 1e-3, synth.seed_of(31, r), dev) for r in range(M)]
    master = torch.zeros(P, dtype=torch.float32, device=dev)
    master[:n] = synth.normal_f32(n, 0.02, synth.seed_of(31, 9), dev)
    m = torch.zeros(P, dtype=torch.float32, device=dev)
    v = torch.zeros(P, dtype=torch.float32, device=dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    rng = np.random.default_rng(31)
    idx_np = np.unique(np.concatenate([rng.integers(0, n, 1 << 14), np.arange(2 ** 31 - 64, 2 ** 31 + 64),
                                       np.arange(n - 64, n), np.arange(plan.shard - 32, plan.shard + 32)]))
    idx = torch.from_numpy(idx_np).to(dev)
    g_s = [u16(g[idx]) for g in grads]
    o = [f32(t[idx]) for t in (master, m, v)]
    op = np.zeros(idx_np.size, np.uint16)
    hp = z.AdamW(global_batch=64, step=1)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    z.zero1_overflow_check(plan, 0, M, grads, flag)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    oracle.zero1_step(g_s, idx_np.size, *o, op, oracle_hp(hp))
    assert_f32_bits(f32(master[idx]), o[0], "master")
    assert_f32_bits(f32(v[idx]), o[2], "v")
    assert_bf16_bits(u16(params[idx]), op, "params")
    # a bucket across 2^31 (second step), against the oracle on the samples inside it
    e0, e1 = 2 ** 31 - 1000, 2 ** 31 + 1003
    hp2 = z.AdamW(global_batch=64, step=2)
    z.zero1_step_bucket(plan, e0, e1, [g[e0:e1] for g in grads], master[e0:], m[e0:], v[e0:], params[e0:], hp2)
    torch.cuda.synchronize()
    inside = (idx_np >= e0) & (idx_np < e1)
    sel = np.flatnonzero(inside)
    w2, m2, v2 = (a[sel].copy() for a in o)
    p2 = np.zeros(sel.size, np.uint16)
    oracle.zero1_step([g[sel].copy() for g in g_s], sel.size, w2, m2, v2, p2, oracle_hp(hp2))
    assert_f32_bits(f32(master[idx][torch.from_numpy(sel).to(dev)]), w2, "master in the bucket")
    assert_bf16_bits(u16(params[idx][torch.from_numpy(sel).to(dev)]), p2, "params in the bucket")
    del grads, master, m, v, params
    free()
