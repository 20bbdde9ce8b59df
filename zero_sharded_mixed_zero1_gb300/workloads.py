"""The five synthetic workloads of the optimizer step.

Sizes follow the workloads the method is stated on: a tiny flat buffer, a
GPT-2-small-sized flat buffer, a 1.3B flat buffer, one rank's shard of a 7.5B
model over 64 replicas, and four Llama-style decoder layers flattened with
shard cuts crossing tensors.  All values are synthetic draws (synth.py); no
weights or datasets are involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field


def llama_layer_numels(d: int = 4096, kv: int = 1024, ffn: int = 14336) -> list[int]:
    """One decoder layer's tensors in order: attn RMSNorm, Wq, Wk, Wv, Wo,
    ffn RMSNorm, W_gate, W_up, W_down (32 query / 8 key-value heads x 128)."""
    return [d, d * d, d * kv, d * kv, d * d, d, d * ffn, d * ffn, ffn * d]


@dataclass(frozen=True)
class Workload:
    name: str
    n: int                      # |theta| of the whole model
    M: int                      # replicas
    align: int                  # shard alignment (elements)
    B: int                      # global batch
    S: float                    # loss scale
    steps: int                  # optimizer steps t = 1..steps
    grad_std: float
    master_std: float = 0.02
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    shard_begin: int = 0        # the shards this GPU processes
    shard_end: int | None = None
    tensor_numels: tuple = field(default=())
    inf_attempt: int = 0        # 1-based attempt whose gradients get +inf (0: none)
    inf_prob: float = 0.0
    seed: int = 0

    @property
    def shards(self) -> tuple[int, int]:
        return self.shard_begin, self.M if self.shard_end is None else self.shard_end


TINY = Workload("tiny_1M_M4", n=1_048_576, M=4, align=128, B=32, S=1.0, steps=1, grad_std=1e-2, seed=1)
GPT2_SMALL = Workload("gpt2_small_124M_M8", n=124_439_808, M=8, align=1, B=512, S=1.0, steps=10,
                      grad_std=1e-3, seed=2)
FLAT_1P3B = Workload("flat_1.3B_M8", n=1_300_000_000, M=8, align=128, B=1024, S=1.0, steps=3,
                     grad_std=1e-3, seed=3)
RANK_7P5B_M64 = Workload("7.5B_over_64_one_shard", n=7_500_000_000, M=64, align=1, B=2048, S=1.0,
                         steps=5, grad_std=1e-3, shard_begin=0, shard_end=1, seed=4)
LLAMA4 = Workload("llama_4_layers_872M_M8", n=4 * sum(llama_layer_numels()), M=8, align=128, B=1024,
                  S=65536.0, steps=3, grad_std=1e-3, tensor_numels=tuple(llama_layer_numels() * 4),
                  inf_attempt=3, inf_prob=1e-6, seed=5)

ALL = [TINY, GPT2_SMALL, FLAT_1P3B, RANK_7P5B_M64, LLAMA4]

# A reduced GPT-2-small-like case for profiler captures: 705 MB of traffic
# per launch (well above L2) but about 1 GB on the device.
PROFILE = Workload("prof_16M_M8", n=16_777_216, M=8, align=1, B=512, S=1.0, steps=10, grad_std=1e-3, seed=6)

BY_NAME = {w.name: w for w in ALL + [PROFILE]}
