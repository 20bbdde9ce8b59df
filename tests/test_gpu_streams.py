"""Stream discipline: every entry point enqueues its work on the stream it is
given.  Each call goes to a side stream right after a long busy kernel and
the writes of that call's gradients on the same stream; an entry that
launched on another stream would read the gradients before they exist and
fail the comparison with the same call made on the default stream."""
import pytest
import torch

import zero_sharded_mixed_zero1_gb300 as z
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, u16
from test_gpu_parity import make_grads, make_state

pytestmark = pytest.mark.gpu

SPIN_CYCLES = 20_000_000   # about 10 ms at 2 GHz


def _call(entry, plan, M, P, n, grads, state, params, hp, policy, scaler, pairs, sums, step, stream):
    if entry in ("dynamic", "pingpong", "staged_dynamic"):
        z.zero1_scaler_init(scaler, policy, hp, stream=stream)
    if entry == "fused":
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *state, params, hp, stream=stream)
    elif entry == "bucket":
        for e0, e1 in ((0, 100_000), (100_000, P)):
            k = max(0, min(n, e1) - e0)
            z.zero1_step_bucket(plan, e0, e1, [g[e0:e0 + k] for g in grads], *[s[e0:] for s in state],
                                params[e0:], hp, stream=stream)
    elif entry == "dynamic":
        z.zero1_step_dynamic(plan, 0, M, grads, *state, params, hp, scaler, policy, sums, stream=stream)
    elif entry == "pingpong":
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads, *pairs, params, hp, scaler, policy, stream=stream)
    elif entry == "staged_dynamic":
        step.dynamic(hp, scaler, policy)
    else:
        step(hp)


def _buffers(entry, plan, M, P, n, src, state0, dev, stream):
    grads = [torch.zeros_like(g) for g in src]
    state = [t.clone() for t in state0]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    step = None
    if entry.startswith("staged"):
        state = [t.cpu().pin_memory() for t in state]
        step = z.HostStreamedStep(plan, 0, M, grads, *state, params, chunk_elems=65536, stream=stream)
    pairs = [[t, torch.zeros_like(t)] for t in state] if entry == "pingpong" else None
    return grads, state, params, z.new_scaler(dev), pairs, torch.empty(P, dtype=torch.float32, device=dev), step


@pytest.mark.parametrize("entry", ["fused", "bucket", "dynamic", "pingpong", "staged", "staged_dynamic"])
def test_entry_points_run_on_the_given_stream(cuda_device, entry):
    dev = cuda_device
    M, n = 8, 300_007
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    hp = z.AdamW(global_batch=64, step=1)
    policy = z.LossScalePolicy(initial_scale=1.0, window=1000, hysteresis=2)
    src = make_grads(M, n, 1e-2, 77, 1, dev)
    state0 = make_state(n, P, 78, dev, nonzero_moments=True)
    ref_state = [t.clone() for t in state0]
    ref_p = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, src, *ref_state, ref_p, hp)   # default stream, grads ready
    side = torch.cuda.Stream(device=dev)
    # warm-up on scratch buffers: every kernel of the entry is loaded before the
    # delay starts (loading a module on first use can wait for the device)
    warm = _buffers(entry, plan, M, P, n, src, state0, dev, side)
    _call(entry, plan, M, P, n, warm[0], warm[1], warm[2], hp, policy, warm[3], warm[4], warm[5], warm[6], side)
    grads, state, params, scaler, pairs, sums, step = _buffers(entry, plan, M, P, n, src, state0, dev, side)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        torch.cuda._sleep(SPIN_CYCLES)
        for o, g in zip(grads, src):
            o.copy_(g, non_blocking=True)
    assert not side.query(), "the delay must still be running when the call is made"
    _call(entry, plan, M, P, n, grads, state, params, hp, policy, scaler, pairs, sums, step, side)
    assert not side.query(), "the call returned after the gradients it reads were written"
    side.synchronize()
    torch.cuda.synchronize()
    if entry == "pingpong":
        state = list(z.current_state(scaler, *pairs))
    for x, y, what in zip(state, ref_state, ("master", "m", "v")):
        assert_f32_bits(f32(x), f32(y), f"{entry}: {what}")
    assert_bf16_bits(u16(params), u16(ref_p), f"{entry}: params")
