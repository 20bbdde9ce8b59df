"""Plant plausible mistakes in the oracle (on the CPU) and check that the pin
suite catches every one: a dropped term, a wrong sign or index, a transposed
operand, a wrong constant, a wrong rounding rule."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero1_oracle.c")

MUTANTS = {
    "drop_bias_correction_1": ("float mh = m1 / bc1;", "float mh = m1;"),
    "bias_correction_off_by_one": ("orc_pow_int((double)beta1, t)", "orc_pow_int((double)beta1, t + 1)"),
    "power_skips_a_bit": ("        if (t & 1) r = r * x;", "        if ((t & 1) && t > 1) r = r * x;"),
    "betas_swapped_in_m": ("float m1 = beta1 * m[j] + omb1 * gj;", "float m1 = beta2 * m[j] + omb2 * gj;"),
    "eps_inside_sqrt": ("float u = mh / (sqrtf(vh) + eps);", "float u = mh / sqrtf(vh + eps);"),
    "decay_without_lr": ("out[5] = (float)(1.0 - (double)lr * (double)weight_decay);",
                         "out[5] = (float)(1.0 - (double)weight_decay);"),
    "update_sign": ("float w = master[j] * cdec - lr * u;", "float w = master[j] * cdec + lr * u;"),
    "loss_scale_ignored": ("out[0] = (float)(1.0 / ((double)B * (double)S));", "out[0] = (float)(1.0 / ((double)B));"),
    "rank0_dropped": ("s = orc_bf16_to_f32(grads[0][j]);\n            for (int32_t r = 1;",
                      "s = 0.0f;\n            for (int32_t r = 1;"),
    "v_not_squared": ("float v1 = beta2 * v[j] + omb2 * (gj * gj);", "float v1 = beta2 * v[j] + omb2 * gj;"),
    "ties_round_up": ("else mag = (lo & 1u) ? hi : lo;", "else mag = hi;"),
    "plan_overpads": ("int64_t P = ((n + unit - 1) / unit) * unit;", "int64_t P = (n / unit) * unit + unit;"),
    "gather_not_from_master": ("params[j] = orc_f32_to_bf16(master[j]);",
                               "params[j] = orc_f32_to_bf16(master[j] * 1.0000001f);"),
    "sqrt_of_m": ("float u = mh / (sqrtf(vh) + eps);", "float u = vh / (sqrtf(mh) + eps);"),
    "scaler_ignores_hysteresis": ("        sc->hyst_left -= 1;", "        sc->hyst_left -= 2;"),
    "scaler_window_off_by_one": ("        if (sc->good >= window) {", "        if (sc->good > window) {"),
    "skip_advances_t": ("        sc->skipped += 1;", "        sc->skipped += 1;\n        sc->step += 1;"),
    "checksum_index_from_zero": ("        s2 += (uint64_t)(i + 1) * (uint64_t)u[i];", "        s2 += (uint64_t)i * (uint64_t)u[i];"),
    "checksum_drops_units": ("        s1 += (uint64_t)u[i];", "        s1 += (uint64_t)(u[i] & 0xFFFEu);"),
    "scaler_no_floor": ("            sc->scale = down < min_scale ? min_scale : down;", "            sc->scale = down;"),
    "scaler_growth_keeps_hysteresis": ("            sc->good = 0;\n            sc->hyst_left = hysteresis;\n        }\n    }",
                                       "            sc->good = 0;\n        }\n    }"),
    "skip_still_writes": ("weight_decay, sc->scale, B, sc->step, &f, 1);", "weight_decay, sc->scale, B, sc->step, &f, 0);"),
    "allreduce_reverse_order": ("        float s = orc_bf16_to_f32(in[0][j]);\n        for (int32_t r = 1; r < M; ++r) s = s + orc_bf16_to_f32(in[r][j]);",
                                "        float s = orc_bf16_to_f32(in[M - 1][j]);\n        for (int32_t r = M - 2; r >= 0; --r) s = s + orc_bf16_to_f32(in[r][j]);"),
    "allreduce_unscaled": ("        float y = s * scale;", "        float y = s;"),
    "inv_rounded_in_fp32": ("out[0] = (float)(1.0 / ((double)B * (double)S));", "out[0] = 1.0f / ((float)B * S);"),
    "sum_in_double": ("            for (int32_t r = 1; r < M; ++r) s = s + orc_bf16_to_f32(grads[r][j]);\n            if (!isfinite(s)) f = 1;",
                      "            double sd = s;\n            for (int32_t r = 1; r < M; ++r) sd = sd + orc_bf16_to_f32(grads[r][j]);\n            s = (float)sd;\n            if (!isfinite(s)) f = 1;"),
    "flag_ignores_nan": ("            if (!isfinite(s)) f = 1;\n        }\n        g_out[j]", "            if (isinf(s)) f = 1;\n        }\n        g_out[j]"),
    "mhat_uses_bc2": ("float mh = m1 / bc1;", "float mh = m1 / bc2;"),
    "decay_after_update": ("float w = master[j] * cdec - lr * u;", "float w = (master[j] - lr * u) * cdec;"),
    "subnormal_ulp": ("double ulp = ldexp(1.0, (e == 0 ? 1 : e) - 127 - 7);", "double ulp = ldexp(1.0, e - 127 - 7);"),
    "segments_shard_offset_from_tensor": ("seg_shard_off[count] = x0 - lo;", "seg_shard_off[count] = x0 - a;"),
    "memory_state_unsharded": ("*zero1_bytes = 2 * n + 2 * n + 12 * shard;", "*zero1_bytes = 2 * n + 2 * n + 12 * n;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    a, b = MUTANTS[name]
    src = open(SRC).read()
    assert a in src, "mutation anchor missing: the oracle changed, update the mutant"
    c = tmp_path / "mutant.c"
    c.write_text(src.replace(a, b))
    so = tmp_path / "mutant.so"
    subprocess.run([os.environ.get("CC", "gcc"), *oracle.CFLAGS, "-o", str(so), str(c), "-lm"], check=True)
    env = dict(os.environ, ZERO1_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_loss_scale.py"),
                        os.path.join(ROOT, "tests", "test_oracle_checksum.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins"
