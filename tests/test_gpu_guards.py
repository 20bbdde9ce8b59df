"""Out-of-bounds write detection: every buffer a call writes sits between
guard words (a fixed byte pattern before and after the view handed to the
call), and the guards must read back unchanged after the call.  The parity
tests compare the elements inside each range; these tests check that nothing
outside it was written.  Covered: every kernel shape of the fused step (wide,
pipelined, grouped, offload), buckets, the shared-memory staged kernel, the
dynamic and ping-pong steps (whole and in buckets), the copy-engine staged
step, the unfused phases, the All-Reduce, the overflow flag and the
checksum, with ragged tails and mixed 16-byte phases."""
import numpy as np
import pytest
import torch

import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 40          # elements on each side
PATTERN = 0xA5      # byte value of every guard byte


class Guarded:
    """A view of `numel` elements with GUARD elements of PATTERN bytes on
    each side (plus `phase` elements of shift), on the device or in pinned
    host memory."""

    def __init__(self, numel, dtype, dev, phase=0, pinned=False):
        total = numel + 2 * GUARD + phase
        if pinned:
            self.raw = torch.empty(total, dtype=dtype).pin_memory()
        else:
            self.raw = torch.empty(total, dtype=dtype, device=dev)
        self.raw.view(torch.uint8).fill_(PATTERN)
        self.lo = GUARD + phase
        self.view = self.raw[self.lo:self.lo + numel]

    def check(self, what):
        b = self.raw.detach().view(torch.uint8).cpu().numpy()
        es = self.raw.element_size()
        before = b[:self.lo * es]
        after = b[(self.lo + self.view.numel()) * es:]
        bad_b = np.flatnonzero(before != PATTERN)
        bad_a = np.flatnonzero(after != PATTERN)
        assert bad_b.size == 0, f"{what}: {bad_b.size} guard bytes before the buffer overwritten"
        assert bad_a.size == 0, f"{what}: {bad_a.size} guard bytes after the buffer overwritten (first at +{bad_a[0]})"


def _state(L, nv, dev, ph, pinned=False):
    out = []
    for k in range(3):
        g = Guarded(L, torch.float32, dev, ph(), pinned)
        g.view.zero_()
        if k == 0:
            g.view[:nv].copy_(synth.normal_f32(nv, 0.02, synth.seed_of(5, k), dev))
        out.append(g)
    return out


def _grads(M, nv, dev, ph, S=1.0, pinned=False):
    out = []
    for r in range(M):
        g = Guarded(nv, torch.bfloat16, dev, ph(), pinned)
        g.view.copy_(synth.normal_bf16(nv, 1e-3 * S, synth.seed_of(6, r), dev))
        out.append(g)
    return out


def _phases(rng, mixed):
    return (lambda: int(rng.integers(0, 8))) if mixed else (lambda: 0)


# (M, n, align, shards): the wide kernel (small ranges), the pipelined kernel
# (more than 2^18 vectors), the grouped kernel (M > 8), ragged tails
CASES = [(1, 1003, 1, None), (3, 5000, 8, (1, 3)), (8, 100_003, 128, None), (2, 2_100_003, 1, None),
         (9, 20_001, 1, (2, 7)), (64, 7001, 8, None), (8, 7, 1, None)]


@pytest.mark.parametrize("M,n,align,shards", CASES)
@pytest.mark.parametrize("mixed", [False, True])
def test_fused_entries_stay_in_bounds(cuda_device, M, n, align, shards, mixed):
    dev = cuda_device
    rng = np.random.default_rng(M * 1000 + n % 997 + mixed)
    ph = _phases(rng, mixed)
    plan = z.zero1_plan(n, M, align)
    sb, se = shards or (0, M)
    base, L, nv = plan.shard_range(sb, se)
    hp = z.AdamW(global_batch=max(M, 64), step=3)
    for entry in ("fused", "prepared", "bucket", "tma"):
        grads = _grads(M, nv, dev, ph)
        state = _state(L, nv, dev, ph)
        params = Guarded(nv, torch.bfloat16, dev, ph())
        flag = Guarded(1, torch.int32, dev, 0)
        flag.view.zero_()
        gv, sv = [g.view for g in grads], [s.view for s in state]
        if entry == "fused":
            z.zero1_reduce_scatter_adamw_allgather(plan, sb, se, gv, *sv, params.view, hp, flag.view)
        elif entry == "prepared":
            z.FusedStep(plan, sb, se, gv, *sv, params.view, flag.view)(hp)
        elif entry == "tma":
            z.zero1_step_tma(plan, sb, se, gv, *sv, params.view, hp, flag.view)
        else:
            cuts = sorted({0, L, *[int(x) for x in rng.integers(0, L + 1, 4)]})
            for e0, e1 in zip(cuts[:-1], cuts[1:]):
                k = max(0, min(nv, e1) - e0)
                z.zero1_step_bucket(plan, base + e0, base + e1, [g[e0:e0 + k] for g in gv],
                                    *[s[e0:] for s in sv], params.view[e0:] if e0 < nv else params.view[:0], hp,
                                    flag.view)
        torch.cuda.synchronize()
        for i, b in enumerate(grads + state + [params, flag]):
            b.check(f"{entry} M={M} n={n} buffer {i}")
        assert int(flag.view.item()) == 0
    assert z.zero1_device_status() == 0


@pytest.mark.parametrize("M,n,align,shards", [(4, 50_003, 8, None), (9, 20_001, 1, (2, 7)), (2, 2_100_003, 1, None)])
def test_offload_and_staged_steps_stay_in_bounds(cuda_device, M, n, align, shards):
    """Host-resident state through the offload kernel and through the
    copy-engine staged step, host-resident gradients and a host copy of
    params: guards on both sides of every host and device buffer."""
    dev = cuda_device
    rng = np.random.default_rng(M + n)
    ph = _phases(rng, True)
    plan = z.zero1_plan(n, M, align)
    sb, se = shards or (0, M)
    base, L, nv = plan.shard_range(sb, se)
    hp = z.AdamW(global_batch=max(M, 64), step=2)
    for entry in ("offload_kernel", "staged_state", "staged_grads", "staged_dynamic"):
        grads = _grads(M, nv, dev, ph, pinned=(entry == "staged_grads"))
        state = _state(L, nv, dev, ph, pinned=(entry != "staged_grads"))
        params = Guarded(nv, torch.bfloat16, dev, ph())
        host_p = Guarded(nv, torch.bfloat16, dev, ph(), pinned=True)
        gv, sv = [g.view for g in grads], [s.view for s in state]
        if entry == "offload_kernel":
            z.zero1_reduce_scatter_adamw_allgather(plan, sb, se, gv, *sv, params.view, hp)
        else:
            step = z.HostStreamedStep(plan, sb, se, gv, *sv, params.view, chunk_elems=int(rng.integers(500, 70_000)),
                                      params_host=host_p.view)
            if entry == "staged_dynamic":
                policy = z.LossScalePolicy(initial_scale=64.0, window=1000, hysteresis=2)
                scaler = z.new_scaler(dev)
                z.zero1_scaler_init(scaler, policy, hp)
                step.dynamic(hp, scaler, policy)
            else:
                step(hp)
            step.close()
        torch.cuda.synchronize()
        for i, b in enumerate(grads + state + [params, host_p]):
            b.check(f"{entry} M={M} n={n} buffer {i}")


@pytest.mark.parametrize("M,n,align,shards", [(4, 50_003, 8, None), (9, 20_001, 1, (2, 7)), (8, 100_003, 128, None),
                                              (64, 7001, 8, None)])
@pytest.mark.parametrize("overflow", [False, True])
def test_dynamic_and_pingpong_steps_stay_in_bounds(cuda_device, M, n, align, shards, overflow):
    """The two-pass dynamic step (with its sums workspace), the ping-pong
    step (both copies) and the bucketed ping-pong attempt, clean and with an
    overflow (the restore path)."""
    dev = cuda_device
    rng = np.random.default_rng(M * 7 + n)
    ph = _phases(rng, True)
    plan = z.zero1_plan(n, M, align)
    sb, se = shards or (0, M)
    base, L, nv = plan.shard_range(sb, se)
    policy = z.LossScalePolicy(initial_scale=1024.0, window=1000, hysteresis=2)
    hp = z.AdamW(global_batch=max(M, 64), step=1)
    for entry in ("dynamic", "pingpong", "pingpong_buckets"):
        grads = _grads(M, nv, dev, ph, S=1024.0)
        if overflow and nv:
            grads[M // 2].view[nv // 3] = float("inf")
        state = _state(L, nv, dev, ph)
        other = _state(L, nv, dev, ph)
        params = Guarded(nv, torch.bfloat16, dev, ph())
        params.view.copy_(state[0].view[:nv].to(torch.bfloat16))
        sums = Guarded(L, torch.float32, dev, ph())
        scaler = z.new_scaler(dev)
        z.zero1_scaler_init(scaler, policy, hp)
        gv, sv, ov = [g.view for g in grads], [s.view for s in state], [s.view for s in other]
        pairs = [[a, b] for a, b in zip(sv, ov)]
        if entry == "dynamic":
            z.zero1_step_dynamic(plan, sb, se, gv, *sv, params.view, hp, scaler, policy, sums.view)
        elif entry == "pingpong":
            z.zero1_step_dynamic_pingpong(plan, sb, se, gv, *pairs, params.view, hp, scaler, policy)
        else:
            attempt = z.PingPongBuckets(plan, sb, se, *pairs, params.view, scaler, policy)
            cuts = sorted({0, L, *[int(x) for x in rng.integers(0, L + 1, 4)]})
            for i in rng.permutation(len(cuts) - 1):
                e0, e1 = cuts[i], cuts[i + 1]
                k = max(0, min(nv, e1) - e0)
                attempt.bucket(e0, e1, [g[e0:e0 + k] for g in gv], hp)
            attempt.finish(hp)
        torch.cuda.synchronize()
        for i, b in enumerate(grads + state + other + [params, sums]):
            b.check(f"{entry} M={M} n={n} overflow={overflow} buffer {i}")
        assert z.scaler_state(scaler)["skipped"] == (1 if overflow and nv else 0)


@pytest.mark.parametrize("M,n,align", [(4, 50_003, 8), (9, 20_001, 1), (2, 2_100_003, 1)])
def test_phases_allreduce_flag_and_checksum_stay_in_bounds(cuda_device, M, n, align):
    dev = cuda_device
    rng = np.random.default_rng(M + 3 * n)
    ph = _phases(rng, True)
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    hp = z.AdamW(global_batch=max(M, 64), step=4)
    grads = _grads(M, n, dev, ph)
    gv = [g.view for g in grads]
    checked = list(grads)
    for dt in (torch.bfloat16, torch.float32):
        rs = Guarded(P, dt, dev, ph())
        flag = Guarded(1, torch.int32, dev, 0)
        flag.view.zero_()
        z.zero1_reduce_scatter(plan, 0, M, gv, 1.0 / (hp.global_batch * hp.loss_scale), rs.view, flag.view)
        outs = [Guarded(n, dt, dev, ph()) for _ in range(M)]
        z.dp_allreduce(plan, gv, [o.view for o in outs], 1.0 / 64)
        checked += [rs, flag] + outs
    g32 = Guarded(P, torch.float32, dev, ph())
    z.zero1_reduce_scatter(plan, 0, M, gv, 1.0 / 64, g32.view)
    state = _state(P, n, dev, ph)
    z.zero1_adamw_update(plan, 0, M, g32.view, *[s.view for s in state], hp)
    params = Guarded(n, torch.bfloat16, dev, ph())
    z.zero1_all_gather(plan, 0, M, state[0].view, params.view)
    shards = Guarded(P, torch.bfloat16, dev, ph())
    z.zero1_reduce_scatter(plan, 0, M, gv, 1.0 / 64, shards.view)
    gathered = [Guarded(n, torch.bfloat16, dev, ph()) for _ in range(M)]
    z.zero1_all_gather_shards(plan, shards.view, [o.view for o in gathered])
    flag = Guarded(1, torch.int32, dev, 0)
    flag.view.zero_()
    z.zero1_overflow_check(plan, 0, M, gv, flag.view)
    ck = Guarded(2, torch.int64, dev, 0)
    z.zero1_checksum(params.view, ck.view)
    torch.cuda.synchronize()
    checked += [g32, params, shards, flag, ck] + state + gathered
    for i, b in enumerate(checked):
        b.check(f"phases M={M} n={n} buffer {i}")
