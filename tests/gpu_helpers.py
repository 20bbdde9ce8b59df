"""Helpers for the GPU parity tests: move tensors to numpy, convert
hyperparameters, compare bit patterns (NaN compared by NaN-ness only)."""
import numpy as np
import torch

import oracle
import zero_sharded_mixed_zero1_gb300 as z


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.float32, copy=False)


def bf16_from_u16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)


def oracle_hp(hp: z.AdamW) -> oracle.AdamW:
    return oracle.AdamW(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                        weight_decay=hp.weight_decay, loss_scale=hp.loss_scale,
                        global_batch=hp.global_batch, step=hp.step)


def assert_f32_bits(got: np.ndarray, want: np.ndarray, what: str) -> None:
    """Bit-exact fp32 (the fixed operation order makes the result unique);
    NaN payloads are not compared."""
    got = np.ascontiguousarray(got, np.float32)
    want = np.ascontiguousarray(want, np.float32)
    assert got.shape == want.shape, what
    gn, wn = np.isnan(got), np.isnan(want)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    ok = got.view(np.uint32) == want.view(np.uint32)
    ok |= gn
    if not ok.all():
        bad = np.flatnonzero(~ok)
        j = bad[0]
        rel = np.max(np.abs(got[bad].astype(np.float64) - want[bad]) / (np.abs(want[bad]) + 1e-45))
        raise AssertionError(f"{what}: {bad.size} of {got.size} differ; first at {j}: "
                             f"{got[j]!r} vs {want[j]!r}; max rel {rel:.3g}")


def assert_bf16_bits(got: np.ndarray, want: np.ndarray, what: str) -> None:
    got = np.ascontiguousarray(got, np.uint16)
    want = np.ascontiguousarray(want, np.uint16)
    assert got.shape == want.shape, what
    gn = ((got & 0x7FFF) > 0x7F80)
    wn = ((want & 0x7FFF) > 0x7F80)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    ok = (got == want) | gn
    if not ok.all():
        bad = np.flatnonzero(~ok)
        raise AssertionError(f"{what}: {bad.size} of {got.size} bf16 values differ; first at {bad[0]}: "
                             f"{got[bad[0]]:#06x} vs {want[bad[0]]:#06x}")
