"""The consistency checksum on the GPU against the oracle's, exactly."""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z
from zero_sharded_mixed_zero1_gb300 import synth
from gpu_helpers import oracle_hp, u16
from test_gpu_parity import make_grads, make_state, oracle_step

pytestmark = pytest.mark.gpu


def words(t):
    return tuple(int(x) for x in t.cpu().numpy().view(np.uint64))


@pytest.mark.parametrize("units", [0, 1, 7, 8, 9, 4097, 1_000_003, 300_000_017])
@pytest.mark.parametrize("phase", [0, 3])
def test_checksum_matches_oracle(cuda_device, units, phase):
    dev = cuda_device
    buf = torch.randint(-32768, 32767, (units + phase,), dtype=torch.int16, device=dev)[phase:]
    got = words(z.zero1_checksum(buf))
    assert got == oracle.checksum16(buf.cpu().numpy())


def test_checksum_of_fp32_and_a_flipped_bit(cuda_device):
    dev = cuda_device
    x = synth.normal_f32(123_457, 1.0, 5, dev)
    c = words(z.zero1_checksum(x))
    assert c == oracle.checksum16(x.cpu().numpy())
    x.view(torch.int32)[77_777] ^= 1 << 9
    assert words(z.zero1_checksum(x))[0] != c[0]


def test_checksum_guards_the_gathered_parameters(cuda_device):
    """After a step the parameters' checksum equals the checksum of the
    oracle's parameters: what ranks compare to catch silent corruption."""
    dev = cuda_device
    M, n = 8, 200_003
    plan = z.zero1_plan(n, M, 128)
    master, m, v = make_state(n, plan.padded_n, 15, dev)
    o = [t.cpu().numpy().copy() for t in (master, m, v)]
    params = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grads = make_grads(M, n, 1e-3, 16, 1, dev)
    hp = z.AdamW(global_batch=512, step=1)
    z.zero1_reduce_scatter_adamw_allgather(plan, 0, M, grads, master, m, v, params, hp)
    want = oracle_step(plan, [u16(g) for g in grads], *o, oracle_hp(hp))
    assert words(z.zero1_checksum(params)) == oracle.checksum16(want)
