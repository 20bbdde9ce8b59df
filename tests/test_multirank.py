"""Multi-rank host logic on the CPU with world-size-2 gloo process groups.

1. bench.py's timing reduction: the slowest rank's time counts, and the
   barrier brackets the timed region.
2. The distributed form of the step on CPU ranks: rank i owns shard i of the
   plan, reduce-scatters by reading every replica's shard-i slice, updates its
   own fp32 state, the overflow flag is a MAX all-reduce, and an all-gather
   of the bf16 shards rebuilds the full parameters ("CS336 Lecture 7:
   Parallelism 1", ZeRO Stage 1 steps).  The assembled result must equal one
   process running every shard.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        out = {}
        # 1. max over ranks
        out["max"] = bench.max_over_ranks(float(10 + rank), world)
        bench.barrier(world)
        # 2. distributed ZeRO-1 on CPU ranks, M = world
        M, n, align = world, 1003, 8
        P, s = oracle.plan(n, M, align)
        rng = np.random.default_rng(0)               # same draws on every rank
        grads = [oracle.f32_to_bf16((rng.standard_normal(n) * 1e-2).astype(np.float32)) for _ in range(M)]
        master = np.zeros(P, np.float32)
        master[:n] = rng.standard_normal(n) * 0.02
        if rank == 1:
            grads[1][700] = 0x7F80                    # +inf on rank 1's replica, inside shard 1
        lo, hi = rank * s, (rank + 1) * s
        nv = max(0, min(hi, n) - lo)
        mine = [np.ascontiguousarray(g[lo:lo + nv]) for g in grads]   # reduce-scatter input
        flag = oracle.overflow_check(mine, nv)
        t = torch.tensor([flag], dtype=torch.int32)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)       # the only global value
        hp = oracle.AdamW(global_batch=8, step=1)
        w, m, v = master[lo:hi].copy(), np.zeros(s, np.float32), np.zeros(s, np.float32)
        shard_params = np.zeros(s, np.uint16)
        f = np.array([int(t.item())], np.uint32)
        oracle.zero1_step(mine, nv, w, m, v, shard_params, hp, flag=f, skip_if_flag=True)
        gathered = [torch.zeros(s, dtype=torch.int32) for _ in range(world)]   # gloo: no 16-bit gather
        dist.all_gather(gathered, torch.from_numpy(shard_params.astype(np.int32)))
        full = np.concatenate([g.numpy().astype(np.uint16) for g in gathered])[:n]
        out["flag"] = int(t.item())
        out["full"] = full
        out["skipped_equal_input"] = bool(np.array_equal(w, master[lo:hi]))
        q.put((rank, out))
    except Exception as e:  # surface the failure to the parent instead of hanging it
        q.put((rank, f"error: {e!r}"))
        raise
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert not any(isinstance(v, str) for v in res.values()), res
    assert all(p.exitcode == 0 for p in procs)
    assert res[0]["max"] == res[1]["max"] == 11.0
    # rank 1's +inf sets the global flag on both ranks; the step is skipped everywhere
    assert res[0]["flag"] == res[1]["flag"] == 1
    assert res[0]["skipped_equal_input"] and res[1]["skipped_equal_input"]
    assert np.array_equal(res[0]["full"], res[1]["full"])
    assert not res[0]["full"].any()                 # params untouched (still zero)


def _worker_clean(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        M, n, align = world, 4099, 1
        P, s = oracle.plan(n, M, align)
        rng = np.random.default_rng(1)
        grads = [oracle.f32_to_bf16((rng.standard_normal(n) * 1e-2).astype(np.float32)) for _ in range(M)]
        master = np.zeros(P, np.float32)
        master[:n] = rng.standard_normal(n) * 0.02
        lo, hi = rank * s, (rank + 1) * s
        nv = max(0, min(hi, n) - lo)
        hp = oracle.AdamW(global_batch=16, step=2)
        w, m, v = master[lo:hi].copy(), np.zeros(s, np.float32), np.zeros(s, np.float32)
        sp = np.zeros(s, np.uint16)
        oracle.zero1_step([np.ascontiguousarray(g[lo:lo + nv]) for g in grads], nv, w, m, v, sp, hp)
        gathered = [torch.zeros(s, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(gathered, torch.from_numpy(sp.astype(np.int32)))
        full = np.concatenate([g.numpy().astype(np.uint16) for g in gathered])[:n]
        # single-process reference: one call over the whole range
        W_, Mm, Vv = master.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
        pp = np.zeros(n, np.uint16)
        oracle.zero1_step(grads, n, W_, Mm, Vv, pp, hp)
        q.put((rank, bool(np.array_equal(full, pp)) and bool(np.array_equal(w, W_[lo:hi]))))
    except Exception as e:
        q.put((rank, f"error: {e!r}"))
        raise
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_assemble_the_single_process_result():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker_clean, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: True, 1: True}
    assert all(p.exitcode == 0 for p in procs)


def _worker_dies(rank, world, port, q):
    import datetime
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        os._exit(3)                       # a rank that fails between steps, no collective in flight
    t0 = time.time()
    try:
        out = [torch.zeros(4, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(out, torch.ones(4, dtype=torch.int32))
        q.put((rank, "no error"))
    except Exception as e:                # the survivor learns of it from its next collective
        q.put((rank, f"detected after {time.time() - t0:.1f}s: {type(e).__name__}"))


def test_a_failed_rank_is_detected_not_waited_for():
    """A rank that dies between steps: the surviving rank's next collective
    ends with an error within the process group's short timeout instead of
    hanging (the pages' NCCL-timeout trap, exercised on CPU ranks)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker_dies, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    rank, msg = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
    assert rank == 0 and msg.startswith("detected"), msg
    assert procs[1].exitcode == 3


def _worker_sdc(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        rng = np.random.default_rng(0)                       # the same parameters on every rank
        params = rng.integers(0, 1 << 16, 10_007).astype(np.uint16)
        if rank == 1:
            params[4321] ^= np.uint16(1 << 3)                 # one silently corrupted bit
        mine = torch.tensor([oracle.checksum16(params)[0] & 0x7FFFFFFFFFFFFFFF,
                             oracle.checksum16(params)[1] & 0x7FFFFFFFFFFFFFFF], dtype=torch.int64)
        all_sums = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(all_sums, mine)
        q.put((rank, all(torch.equal(all_sums[0], s) for s in all_sums)))
    except Exception as e:
        q.put((rank, f"error: {e!r}"))
        raise
    finally:
        dist.destroy_process_group()


def test_ranks_compare_parameter_checksums():
    """After the all-gather every rank holds the same parameters: ranks
    exchange their checksums (two words each) and all see the one rank whose
    copy has a flipped bit."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker_sdc, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: False, 1: False}
