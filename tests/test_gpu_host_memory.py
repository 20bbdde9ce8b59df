"""Pinned host buffers passed straight to the kernels (read and written over
the host link, no staging copy): the results must be bit-identical to the
same step on HBM buffers, and to the oracle.

Covers gradients streamed from host memory (the end-to-end path), bf16
parameters written to host memory, and fp32 master/m/v kept in host memory
(optimizer-state offload, "五维并行实战" section 4.2 offload_optimizer)."""
import warnings

import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, oracle_hp, u16
from test_gpu_parity import make_grads, make_state, oracle_step

pytestmark = pytest.mark.gpu


def pinned(t: torch.Tensor) -> torch.Tensor:
    return t.cpu().pin_memory()


@pytest.mark.parametrize("M,n,align", [(8, 100_003, 128), (4, 2048 * 5 + 3, 1), (64, 20_000, 8), (13, 4099, 1)])
@pytest.mark.parametrize("where", ["grads", "grads_params", "state", "everything"])
def test_host_buffers_match_hbm(cuda_device, M, n, align, where):
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    a_state = make_state(n, P, 800 + M, dev, nonzero_moments=True)
    b_state = [t.clone() for t in a_state]
    o_state = [f32(t) for t in a_state]
    if where in ("state", "everything"):
        b_state = [pinned(t) for t in b_state]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    if where in ("grads_params", "everything"):
        pb = pinned(pb)
    fa = torch.zeros(1, dtype=torch.int32, device=dev)
    fb = torch.zeros(1, dtype=torch.int32, device=dev)
    for t in (1, 2):
        hp = z.AdamW(global_batch=max(M, 64), step=t)
        grads = make_grads(M, n, 1e-2, 810 + M, t, dev)
        gb = [pinned(g) for g in grads] if where != "state" else grads
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *a_state, pa, hp, fa)
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, gb, *b_state, pb, hp, fb)
        torch.cuda.synchronize()
        want_p = oracle_step(plan, [u16(g) for g in grads], *o_state, oracle_hp(hp))
        for x, y, o, what in zip(a_state, b_state, o_state, ("master", "m", "v")):
            assert_f32_bits(f32(y), f32(x), f"{where}: {what} t={t}")
            assert_f32_bits(f32(x), o, f"{what} t={t} vs oracle")
        assert_bf16_bits(u16(pb), u16(pa), f"{where}: params t={t}")
        assert_bf16_bits(u16(pa), want_p, f"params t={t} vs oracle")
    assert int(fa.item()) == int(fb.item()) == 0


def test_overflow_check_reads_host_gradients(cuda_device):
    dev = cuda_device
    M, n = 8, 50_000
    plan = z.zero1_plan(n, M, 8)
    grads = [pinned(g) for g in make_grads(M, n, 1e-3, 820, 1, dev)]
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    z.zero1_overflow_check(plan, 0, M, grads, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    grads[3][40_000] = float("inf")
    z.zero1_overflow_check(plan, 0, M, grads, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1


def test_pageable_host_tensor_is_rejected(cuda_device):
    plan = z.zero1_plan(100, 1, 1)
    master, m, v = make_state(100, plan.padded_n, 1, cuda_device)
    params = torch.zeros(100, dtype=torch.bfloat16, device=cuda_device)
    grads = [torch.zeros(100, dtype=torch.bfloat16)]       # pageable: not accepted
    with pytest.raises(ValueError):
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, 1, grads, master, m, v, params, z.AdamW())


@pytest.mark.parametrize("M,n,align,chunk,shards", [(8, 100_003, 128, 4096, None), (4, 50_000, 1, 1000, (1, 3)),
                                                    (13, 9_999, 8, 777, None), (2, 20, 128, 8, (1, 2)),
                                                    (13, 9_999, 8, 1024, None), (3, 70_001, 1, 8192, (0, 2))])
@pytest.mark.parametrize("where", ["grads", "state", "grads_state", "params"])
def test_host_streamed_step_equals_fused_step(cuda_device, M, n, align, chunk, shards, where):
    """Buffers in pinned host memory, staged chunk by chunk through HBM by
    copy streams while the step runs on another chunk (three slots: copy in,
    step, copy back): the fused step's bits on device buffers, and the
    parameters copied back to host memory."""
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    sb, se = shards or (0, M)
    base, L, nv = plan.shard_range(sb, se)
    a = [t[base:base + L].clone() for t in make_state(n, plan.padded_n, 90 + M, dev, nonzero_moments=True)]
    b = [pinned(t) for t in a] if where in ("state", "grads_state") else [t.clone() for t in a]
    pa = torch.zeros(max(nv, 1), dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(max(nv, 1), dtype=torch.bfloat16, device=dev)
    grads_on_host = where in ("grads", "grads_state")
    gb = [torch.zeros(max(nv, 1), dtype=torch.bfloat16, device=dev) for _ in range(M)]
    if grads_on_host:
        gb = [pinned(g) for g in gb]
    host_p = torch.zeros(max(nv, 1), dtype=torch.bfloat16).pin_memory()
    step = z.HostStreamedStep(plan, sb, se, gb, *b, pb, chunk_elems=chunk, params_host=host_p)
    o = [f32(t).copy() for t in a]                 # the oracle's copy of the range's state
    for t in (1, 2, 3, 4):
        grads = [g[base:base + nv] for g in make_grads(M, n, 1e-2, 91 + M, t, dev)]
        for x, g in zip(gb, grads):
            x[:nv].copy_(g)
        torch.cuda.synchronize()
        hp = z.AdamW(global_batch=max(M, 64), step=t)
        z.zero1_reduce_scatter_adamw_allgather(plan, sb, se, grads, *a, pa, hp)
        step(hp)
        torch.cuda.synchronize()
        o_p = np.zeros(nv, np.uint16)
        oracle.zero1_step([np.ascontiguousarray(u16(g)) for g in grads], nv, *o, o_p, oracle_hp(hp))
        for x, y, want, what in zip(a, b, o, ("master", "m", "v")):
            assert_f32_bits(f32(y), f32(x), f"{where}: {what} t={t}")
            assert_f32_bits(f32(y), want, f"{where}: {what} t={t} vs oracle")
        assert_bf16_bits(u16(pb[:nv]), u16(pa[:nv]), f"{where}: params t={t}")
        assert_bf16_bits(u16(host_p[:nv]), u16(pa[:nv]), f"{where}: params on host t={t}")
        assert_bf16_bits(u16(host_p[:nv]), o_p, f"{where}: params on host t={t} vs oracle")


def test_host_streamed_step_is_ordered_on_its_stream(cuda_device):
    """Work enqueued on the step's stream after a call sees the host state the
    call copied back, and the next call sees work enqueued before it."""
    dev = cuda_device
    M, n = 4, 40_000
    plan = z.zero1_plan(n, M, 8)
    L = plan.padded_n
    dev_state = make_state(n, L, 5, dev, nonzero_moments=True)
    ref = [t.clone() for t in dev_state]
    host_state = [pinned(t) for t in dev_state]
    grads = make_grads(M, n, 1e-2, 6, 1, dev)
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    st = torch.cuda.Stream(device=dev)
    step = z.HostStreamedStep(plan, 0, M, grads, *host_state, pb, chunk_elems=4096, stream=st)
    snap = torch.empty(L, dtype=torch.float32, device=dev)
    for t in (1, 2):
        hp = z.AdamW(global_batch=64, step=t)
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *ref, pa, hp)
        with torch.cuda.stream(st):
            step(hp)
            snap.copy_(host_state[0], non_blocking=True)     # ordered after the copies back
        st.synchronize()
        torch.cuda.synchronize()
        assert_f32_bits(f32(snap), f32(ref[0]), f"master seen on the stream t={t}")


def test_host_streamed_step_rejects_mixed_placement(cuda_device):
    dev = cuda_device
    M, n = 2, 1000
    plan = z.zero1_plan(n, M, 1)
    state = make_state(n, plan.padded_n, 1, dev)
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grads = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    with pytest.raises(ValueError):      # nothing in host memory
        z.HostStreamedStep(plan, 0, M, grads, *state, params)
    with pytest.raises(ValueError):      # master on the host, m and v on the device
        z.HostStreamedStep(plan, 0, M, grads, pinned(state[0]), state[1], state[2], params)
    with pytest.raises(ValueError):      # one replica's gradients on the host
        z.HostStreamedStep(plan, 0, M, [grads[0], pinned(grads[1])], *state, params)


def test_staged_step_rejects_misplaced_buffers(cuda_device):
    """Through the C ABI: a handle that stages the state refuses device-memory
    state and a params_host it was not created for, and a capturing stream is
    refused before anything is enqueued."""
    import ctypes
    dev = cuda_device
    M, n = 2, 4096
    plan = z.zero1_plan(n, M, 8)
    lib = z.load()
    h = ctypes.c_void_p()
    assert lib.zero1_staged_create(ctypes.byref(plan), 0, M, z.ZERO1_STAGE_STATE, 1000, ctypes.byref(h)) == 0
    try:
        dev_state = make_state(n, plan.padded_n, 3, dev)
        host_state = [pinned(t) for t in dev_state]
        grads = make_grads(M, n, 1e-2, 4, 1, dev)
        g = (ctypes.c_void_p * M)(*[x.data_ptr() for x in grads])
        params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
        hp = ctypes.byref(z.AdamW(global_batch=64).c_struct())
        st = torch.cuda.current_stream().cuda_stream
        rc = lib.zero1_staged_step(h, g, *[t.data_ptr() for t in dev_state], params.data_ptr(), None, hp, None, st)
        assert rc == -1 and b"pinned host memory" in lib.zero1_last_error()
        host_p = torch.zeros(n, dtype=torch.bfloat16).pin_memory()
        rc = lib.zero1_staged_step(h, g, *[t.data_ptr() for t in host_state], params.data_ptr(), host_p.data_ptr(),
                                   hp, None, st)
        assert rc == -1 and b"ZERO1_STAGE_PARAMS" in lib.zero1_last_error()
        graph = torch.cuda.CUDAGraph()
        with warnings.catch_warnings():          # the refused call leaves the capture empty, as intended
            warnings.simplefilter("ignore", UserWarning)
            with torch.cuda.graph(graph):
                rc = lib.zero1_staged_step(h, g, *[t.data_ptr() for t in host_state], params.data_ptr(), None,
                                           hp, None, torch.cuda.current_stream().cuda_stream)
        assert rc == -1 and b"capturing" in lib.zero1_last_error()
        rc = lib.zero1_staged_step(h, g, *[t.data_ptr() for t in host_state], params.data_ptr(), None, hp, None, st)
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.count_nonzero(params).item() > 0
    finally:
        assert lib.zero1_staged_destroy(h) == 0


@pytest.mark.parametrize("L_n,M,chunk", [(100_003, 8, 4096), (9_999, 13, 1024), (1 << 20, 2, 1 << 16),
                                         (5000, 1, 1000), (20, 2, 8), (3 * 1024 + 5, 1, 1021)])
def test_staged_chunk_boundaries(cuda_device, L_n, M, chunk):
    """The handle's chunks cover [0, L) in order with chunk_elems (rounded up
    to a multiple of 8) elements each, the last one shorter."""
    plan = z.zero1_plan(L_n, M, 8)
    base, L, nv = plan.shard_range(0, M)
    master, m, v = (pinned(t) for t in make_state(L_n, plan.padded_n, 1, cuda_device))
    params = torch.zeros(L_n, dtype=torch.bfloat16, device=cuda_device)
    grads = [torch.zeros(L_n, dtype=torch.bfloat16, device=cuda_device) for _ in range(M)]
    step = z.HostStreamedStep(plan, 0, M, grads, master, m, v, params, chunk_elems=chunk)
    cuts = [a for a, _ in step.pieces] + [step.pieces[-1][1]]
    step.close()
    c = (chunk + 7) // 8 * 8
    assert cuts == list(range(0, L, c)) + [L]


def test_staged_step_close(cuda_device):
    """close() waits for the queued work and frees the handle; a second close
    is a no-op and a call after it raises."""
    dev = cuda_device
    M, n = 2, 10_000
    plan = z.zero1_plan(n, M, 8)
    state = [pinned(t) for t in make_state(n, plan.padded_n, 3, dev)]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grads = make_grads(M, n, 1e-2, 4, 1, dev)
    step = z.HostStreamedStep(plan, 0, M, grads, *state, params, chunk_elems=1024)
    step(z.AdamW(global_batch=64))
    step.close()
    torch.cuda.synchronize()
    assert torch.count_nonzero(params).item() > 0
    step.close()
    with pytest.raises(ValueError):
        step(z.AdamW(global_batch=64, step=2))


@pytest.mark.parametrize("M,n,align,chunk", [(8, 100_003, 128, 8192), (13, 9_999, 8, 1000), (3, 50_000, 1, 7000)])
@pytest.mark.parametrize("where", ["state", "grads_state", "state_params"])
def test_staged_dynamic_step_equals_device_dynamic_step(cuda_device, M, n, align, chunk, where):
    """Dynamic loss scaling with the optimizer state in pinned host memory
    (the fp16 block with offload_optimizer): every attempt bit for bit the
    two-pass dynamic step on device buffers, overflowing attempts included
    (consecutive ones that halve S), and the same scaler."""
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=1024.0, factor=2.0, window=2, hysteresis=1, min_scale=1.0)
    hp = z.AdamW(global_batch=max(M, 64), step=1)
    a = make_state(n, P, 130 + M, dev, nonzero_moments=True)
    b = [pinned(t) for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    host_p = torch.zeros(n, dtype=torch.bfloat16).pin_memory() if where == "state_params" else None
    gb = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    if where == "grads_state":
        gb = [pinned(g) for g in gb]
    s_a, s_b = z.new_scaler(dev), z.new_scaler(dev)
    z.zero1_scaler_init(s_a, policy, hp)
    z.zero1_scaler_init(s_b, policy, hp)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    step = z.HostStreamedStep(plan, 0, M, gb, *b, pb, chunk_elems=chunk, params_host=host_p)
    # the oracle's attempts on its own copy of the state
    o = [f32(t).copy() for t in a]
    o_p = np.zeros(n, np.uint16)
    o_policy = oracle.LossScalePolicy(initial_scale=policy.initial_scale, factor=policy.factor,
                                      window=policy.window, hysteresis=policy.hysteresis, min_scale=policy.min_scale)
    o_sc = oracle.Scaler.start(o_policy, hp.step)
    o_hp = oracle_hp(hp)
    for k in range(7):
        S = z.scaler_state(s_a)["scale"]
        assert S == o_sc.scale
        grads = make_grads(M, n, 1e-3 * S, 140 + M, k, dev)
        if k in (2, 3, 5):
            grads[k % M][(97 * k) % n] = float("inf") if k != 3 else float("nan")
        for x, g in zip(gb, grads):
            x.copy_(g)
        torch.cuda.synchronize()
        z.zero1_step_dynamic(plan, 0, M, grads, *a, pa, hp, s_a, policy, sums)
        step.dynamic(hp, s_b, policy)
        torch.cuda.synchronize()
        flag = oracle.zero1_dynamic_attempt([u16(g) for g in grads], n, *o, o_p, o_hp, o_sc, o_policy)
        assert flag == (1 if k in (2, 3, 5) else 0)
        for x, y, want, what in zip(a, b, o, ("master", "m", "v")):
            assert_f32_bits(f32(y), f32(x), f"{where}: {what} attempt {k}")
            assert_f32_bits(f32(y), want, f"{where}: {what} attempt {k} vs oracle")
        assert_bf16_bits(u16(pb), u16(pa), f"{where}: params attempt {k}")
        assert_bf16_bits(u16(pb), o_p, f"{where}: params attempt {k} vs oracle")
        if host_p is not None:
            assert_bf16_bits(u16(host_p), u16(pa), f"{where}: params on host attempt {k}")
        st = z.scaler_state(s_b)
        assert st == z.scaler_state(s_a)
        assert (st["scale"], st["step"], st["attempts"], st["skipped"]) == \
            (o_sc.scale, o_sc.step, o_sc.attempts, o_sc.skipped)
    st = z.scaler_state(s_b)
    assert st["skipped"] == 3 and st["step"] == 5
    step.close()


@pytest.mark.parametrize("where", ["grads_params", "state"])
def test_staged_timeline_is_ordered_and_changes_no_bit(cuda_device, where):
    """With tracing on, the handle reports per-chunk times of its last step:
    each chunk's stages in order (copies in, kernel, copies out), the inbound
    copies of successive chunks one after another on their stream, no kernel
    before its copies; and the step's results are the untraced step's bits."""
    dev = cuda_device
    M, n, chunk = 4, 200_003, 16384
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    a = make_state(n, P, 31, dev, nonzero_moments=True)
    b = [t.clone() for t in a]
    on_host = where == "state"
    if on_host:
        a, b = [pinned(t) for t in a], [pinned(t) for t in b]
    grads = make_grads(M, n, 1e-2, 32, 1, dev)
    host_g = [pinned(g) for g in grads]
    gsrc = grads if on_host else host_g
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    ha = None if on_host else torch.zeros(n, dtype=torch.bfloat16).pin_memory()
    hb = None if on_host else torch.zeros(n, dtype=torch.bfloat16).pin_memory()
    plain = z.HostStreamedStep(plan, 0, M, gsrc, *a, pa, chunk_elems=chunk, params_host=ha)
    traced = z.HostStreamedStep(plan, 0, M, gsrc, *b, pb, chunk_elems=chunk, params_host=hb, timeline=True)
    with pytest.raises(z.Zero1Error):
        traced.timeline()                            # no step yet
    for t in (1, 2):
        hp = z.AdamW(global_batch=64, step=t)
        plain(hp)
        traced(hp)
        torch.cuda.synchronize()
        tl = traced.timeline()
        assert tl.shape == (len(traced.pieces), 6)
        eps = 0.005                                  # event timestamps resolve to about half a microsecond
        for k in range(tl.shape[0]):
            i0, i1, c0, c1, o0, o1 = tl[k]
            assert -eps <= i0 <= i1 + eps and i1 <= c0 + eps and c0 <= c1 + eps
            assert c1 <= o0 + eps and o0 <= o1 + eps
            if k:
                assert tl[k - 1][1] <= i0 + eps      # one inbound stream: chunk after chunk
        for x, y, what in zip(a, b, ("master", "m", "v")):
            assert_f32_bits(f32(y), f32(x), f"traced {what} t={t}")
        assert_bf16_bits(u16(pb), u16(pa), f"traced params t={t}")
        if ha is not None:
            assert_bf16_bits(u16(hb), u16(ha), f"traced host params t={t}")
    with pytest.raises(z.Zero1Error):
        plain.timeline()                             # created without tracing
    plain.close()
    traced.close()


@pytest.mark.parametrize("M,n,align", [(8, 100_003, 128), (2, 30_001, 1), (13, 9_999, 8)])
def test_pingpong_with_host_state_matches_oracle(cuda_device, M, n, align):
    """The dynamically scaled ping-pong step with both copies of master/m/v in
    pinned host memory (offload with one pass over the data): every attempt
    bit for bit the oracle's, overflowing ones included."""
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=1024.0, factor=2.0, window=2, hysteresis=1, min_scale=1.0)
    hp = z.AdamW(global_batch=max(M, 64), step=1)
    state = [pinned(t) for t in make_state(n, P, 150 + M, dev, nonzero_moments=True)]
    o = [f32(t).copy() for t in state]
    pairs = [[t, torch.full((P,), float("nan"), dtype=torch.float32).pin_memory()] for t in state]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    o_p = np.zeros(n, np.uint16)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    o_policy = oracle.LossScalePolicy(initial_scale=policy.initial_scale, factor=policy.factor,
                                      window=policy.window, hysteresis=policy.hysteresis, min_scale=policy.min_scale)
    o_sc = oracle.Scaler.start(o_policy, hp.step)
    for k in range(5):
        grads = make_grads(M, n, 1e-3 * o_sc.scale, 160 + M, k, dev)
        if k in (1, 2):
            grads[k % M][(31 * k) % n] = float("inf")
        z.zero1_step_dynamic_pingpong(plan, 0, M, grads, *pairs, params, hp, scaler, policy)
        torch.cuda.synchronize()
        flag = oracle.zero1_dynamic_attempt([u16(g) for g in grads], n, *o, o_p, oracle_hp(hp), o_sc, o_policy)
        assert flag == (1 if k in (1, 2) else 0)
        cur = z.current_state(scaler, *pairs)
        for x, want, what in zip(cur, o, ("master", "m", "v")):
            assert_f32_bits(f32(x), want, f"{what} attempt {k}")
        assert_bf16_bits(u16(params), o_p, f"params attempt {k}")
    st = z.scaler_state(scaler)
    assert (st["step"], st["skipped"]) == (o_sc.step, o_sc.skipped) == (4, 2)


@pytest.mark.parametrize("M,n,align", [(8, 100_003, 128), (3, 30_001, 1), (13, 9_999, 8)])
def test_two_pass_dynamic_step_with_host_state_matches_oracle(cuda_device, M, n, align):
    """The two-pass dynamically scaled step (reduce-scatter into HBM sums,
    then the update from the sums) with master/m/v in pinned host memory,
    updated over the link in place: every attempt bit for bit the oracle's,
    overflowing ones included."""
    dev = cuda_device
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    policy = z.LossScalePolicy(initial_scale=1024.0, factor=2.0, window=2, hysteresis=1, min_scale=1.0)
    hp = z.AdamW(global_batch=max(M, 64), step=1)
    state = [pinned(t) for t in make_state(n, P, 170 + M, dev, nonzero_moments=True)]
    o = [f32(t).copy() for t in state]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    o_p = np.zeros(n, np.uint16)
    sums = torch.empty(P, dtype=torch.float32, device=dev)
    scaler = z.new_scaler(dev)
    z.zero1_scaler_init(scaler, policy, hp)
    o_policy = oracle.LossScalePolicy(initial_scale=policy.initial_scale, factor=policy.factor,
                                      window=policy.window, hysteresis=policy.hysteresis, min_scale=policy.min_scale)
    o_sc = oracle.Scaler.start(o_policy, hp.step)
    for k in range(5):
        grads = make_grads(M, n, 1e-3 * o_sc.scale, 180 + M, k, dev)
        if k in (1, 3):
            grads[k % M][(29 * k) % n] = float("inf")
        z.zero1_step_dynamic(plan, 0, M, grads, *state, params, hp, scaler, policy, sums)
        torch.cuda.synchronize()
        flag = oracle.zero1_dynamic_attempt([u16(g) for g in grads], n, *o, o_p, oracle_hp(hp), o_sc, o_policy)
        assert flag == (1 if k in (1, 3) else 0)
        for x, want, what in zip(state, o, ("master", "m", "v")):
            assert_f32_bits(f32(x), want, f"{what} attempt {k}")
        assert_bf16_bits(u16(params), o_p, f"params attempt {k}")
    st = z.scaler_state(scaler)
    assert (st["step"], st["skipped"]) == (o_sc.step, o_sc.skipped) == (4, 2)
