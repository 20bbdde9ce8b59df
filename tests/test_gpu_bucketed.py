"""Bucketed (streaming) steps: gradients arrive bucket by bucket and each
bucket is reduced and applied at once, its buffers then reused ("五维并行实战"
4.2: reduce_bucket_size, contiguous_gradients, overlap_comm; "CS336 Lecture 7:
Parallelism 1", ZeRO Stage 2: hand gradients off as they are produced).  Any
cover of [0, P) by disjoint buckets must give the fused step's bits."""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth
from zero_sharded_mixed_zero1_gb300 import workloads as W
from gpu_helpers import assert_bf16_bits, assert_f32_bits, f32, oracle_hp, u16
from test_gpu_parity import make_grads, make_state, oracle_step

pytestmark = pytest.mark.gpu


def random_buckets(P, rng, max_bucket):
    cuts = [0]
    while cuts[-1] < P:
        cuts.append(min(P, cuts[-1] + int(rng.integers(1, max_bucket + 1))))
    return list(zip(cuts[:-1], cuts[1:]))


@pytest.mark.parametrize("M,n,align,max_bucket", [(4, 10_001, 8, 3000), (8, 2048 * 7 + 13, 1, 5000),
                                                  (13, 4099, 128, 700), (64, 3001, 1, 1000), (1, 777, 1, 7)])
def test_buckets_equal_the_whole_step(cuda_device, M, n, align, max_bucket):
    dev = cuda_device
    rng = np.random.default_rng(M * 7 + n)
    plan = z.zero1_plan(n, M, align)
    P = plan.padded_n
    a = make_state(n, P, 300 + M, dev, nonzero_moments=True)
    b = [t.clone() for t in a]
    o = [f32(t) for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pool = [[torch.empty(max_bucket, dtype=torch.bfloat16, device=dev) for _ in range(M)] for _ in range(2)]
    for t in (1, 2):
        hp = z.AdamW(global_batch=max(M, 64), step=t)
        grads = make_grads(M, n, 1e-2, 310 + M, t, dev)
        z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, *a, pa, hp)
        for k, (e0, e1) in enumerate(random_buckets(P, rng, max_bucket)):
            nv = max(0, min(n, e1) - e0)
            slot = pool[k % 2]                        # recycled bucket buffers
            for r in range(M):
                if nv:
                    slot[r][:nv].copy_(grads[r][e0:e0 + nv])
            z.zero1_step_bucket(plan, e0, e1, [s[:max(nv, 1)] for s in slot], b[0][e0:], b[1][e0:], b[2][e0:],
                                pb[e0:] if e0 < n else pb[:0], hp)
        torch.cuda.synchronize()
        want = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp))
        for x, y, oo, what in zip(a, b, o, ("master", "m", "v")):
            assert_f32_bits(f32(y), f32(x), f"{what} t={t} buckets vs whole")
            assert_f32_bits(f32(y), oo, f"{what} t={t} buckets vs oracle")
        assert_bf16_bits(u16(pb), u16(pa), f"params t={t}")
        assert_bf16_bits(u16(pb), want, f"params t={t} vs oracle")


def test_bucket_range_is_validated(cuda_device):
    plan = z.zero1_plan(1000, 4, 8)
    master, m, v = make_state(1000, plan.padded_n, 1, cuda_device)
    params = torch.zeros(1000, dtype=torch.bfloat16, device=cuda_device)
    grads = make_grads(4, 1000, 1e-2, 2, 1, cuda_device)
    # the library rejects bad ranges; a range longer than the tensors is
    # already refused by the binding's length check
    for e0, e1 in [(-1, 10), (10, 10), (0, plan.padded_n + 1)]:
        with pytest.raises((z.Zero1Error, ValueError)):
            z.zero1_step_bucket(plan, e0, e1, grads, master, m, v, params, z.AdamW(global_batch=8))


def test_llama_layers_in_pages_sized_buckets(cuda_device):
    """Four Llama-style layers stepped in buckets of 5e7 elements (the pages'
    reduce_bucket_size) equal one fused step, bit for bit on the device; the
    oracle checks samples."""
    w = W.LLAMA4
    dev = cuda_device
    plan = z.zero1_plan(w.n, w.M, w.align)
    n, P = plan.n, plan.padded_n
    hp = z.AdamW(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                 loss_scale=w.S, global_batch=w.B, step=1)
    master = torch.zeros(P, dtype=torch.float32, device=dev)
    master[:n] = synth.normal_f32(n, w.master_std, synth.seed_of(w.seed, 1), dev)
    a = [master, torch.zeros_like(master), torch.zeros_like(master)]
    b = [t.clone() for t in a]
    pa = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    pb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grads = [synth.normal_bf16(n, w.grad_std * w.S, synth.seed_of(w.seed, 101, r), dev) for r in range(w.M)]
    rng = np.random.default_rng(9)
    idx_np = np.unique(np.concatenate([rng.integers(0, n, 1 << 15), np.arange(n - 64, n)]))
    idx = torch.from_numpy(idx_np).to(dev)
    o = [f32(t[idx]) for t in a]
    g_s = [u16(g[idx]) for g in grads]
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, w.M, grads, *a, pa, hp)
    bucket = 50_000_000
    nb = 0
    for e0 in range(0, P, bucket):
        e1 = min(P, e0 + bucket)
        nv = max(0, min(n, e1) - e0)
        z.zero1_step_bucket(plan, e0, e1, [g[e0:e0 + nv] for g in grads], b[0][e0:], b[1][e0:], b[2][e0:],
                            pb[e0:], hp)
        nb += 1
    torch.cuda.synchronize()
    assert nb == (P + bucket - 1) // bucket == 18
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))
    op = np.zeros(idx_np.size, np.uint16)
    oracle.zero1_step(g_s, idx_np.size, *o, op, oracle_hp(hp))
    assert_f32_bits(f32(b[0][idx]), o[0], "master samples vs oracle")
    assert_bf16_bits(u16(pb[idx]), op, "params samples vs oracle")
    del grads, a, b
    torch.cuda.empty_cache()


def test_per_tensor_weight_decay_through_buckets(cuda_device):
    """Weight decay chosen per tensor (none on the norm vectors), done as one
    bucket per tensor with that tensor's hyperparameters: each tensor's
    elements equal the oracle's step over that tensor's range with its own
    weight decay; the padding after the last tensor takes the last call's."""
    dev = cuda_device
    d, f = 64, 224          # a small Llama-style layer: norms, attention and MLP matrices
    numels = [d, d * d, d * d // 4, d * d // 4, d * d, d, d * f, d * f, f * d, d]
    norms = {0, 5, 9}
    n = sum(numels)
    M = 4
    plan = z.zero1_plan(n, M, 8)
    P = plan.padded_n
    state = make_state(n, P, 401, dev, nonzero_moments=True)
    o = [f32(t) for t in state]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    want_p = np.zeros(n, np.uint16)
    offsets = np.concatenate([[0], np.cumsum(numels)])
    start = [x.copy() for x in o]
    for t in (1, 2, 3):
        grads = make_grads(M, n, 1e-2, 402, t, dev)
        g_np = [u16(g) for g in grads]
        ranges = [(int(offsets[i]), int(offsets[i + 1]), i in norms) for i in range(len(numels))]
        ranges[-1] = (ranges[-1][0], P, ranges[-1][2])          # the last call also covers the padding
        for b, e, is_norm in ranges:
            hp = z.AdamW(global_batch=64, step=t, weight_decay=0.0 if is_norm else 0.1)
            k = max(0, min(n, e) - b)
            z.zero1_step_bucket(plan, b, e, [g[b:b + k] for g in grads], *[s[b:] for s in state], params[b:], hp)
            seg = [x[b:b + k] for x in g_np]
            o_seg = [x[b:e].copy() for x in o]
            p_seg = np.zeros(k, np.uint16)
            oracle.zero1_step(seg, k, *o_seg, p_seg, oracle_hp(hp))
            for x, y in zip(o, o_seg):
                x[b:e] = y
            want_p[b:b + k] = p_seg
        torch.cuda.synchronize()
        for x, y, what in zip(state, o, ("master", "m", "v")):
            assert_f32_bits(f32(x), y, f"{what} t={t}")
        assert_bf16_bits(u16(params), want_p, f"params t={t}")
        if t == 1:
            # the choice mattered: the first norm under the uniform decay differs
            b, e = int(offsets[0]), int(offsets[1])
            uni = [x[b:e].copy() for x in start]
            oracle.zero1_step([x[b:e] for x in g_np], e - b, *uni, np.zeros(e - b, np.uint16),
                              oracle_hp(z.AdamW(global_batch=64, step=1, weight_decay=0.1)))
            assert not np.array_equal(uni[0], o[0][b:e])
