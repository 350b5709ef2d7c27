"""Plant plausible mistakes in copies of the oracle's C source; each must fail a pin.

This shows the pins constrain every part of the oracle: a dropped term, a wrong sign,
a wrong index, a transposed operand or a swapped constant all get caught. The mistakes
are planted only in temporary copies on the CPU; the committed oracle is untouched.
"""
import os

import pytest

import oracle
from oracle import build as obuild
from pins import PINS

SRC = open(obuild.SRC).read()

# (name, text in the oracle source, replacement, occurrence index)
MUTANTS = [
    ("drop_worker_error", "zw[i] = p + ew[i];", "zw[i] = p;", 0),
    ("sign_zero_negative", "return z >= 0.0f;", "return z > 0.0f;", 0),
    ("momentum_minus", "float p = old_part + new_part;", "float p = old_part - new_part;", 0),
    ("momentum_swap_b1_c1", "float old_part = b1 * m[i];", "float old_part = c1 * m[i];", 0),
    ("scale_wrong_divisor", "return (float)sqrt(sum / (double)C);",
     "return (float)sqrt(sum / (double)(C + 1));", 0),
    ("scale_no_sqrt", "return (float)sqrt(sum / (double)C);", "return (float)(sum / (double)C);", 0),
    ("server_sum_not_mean", "float avg = acc / (float)W;", "float avg = acc;", 0),
    ("warmup_mean_descending",
     "for (int32_t w = 0; w < W; ++w) acc = acc + ora_grad(grads, dtype, (int64_t)w * n + i);",
     "for (int32_t w = W - 1; w >= 0; --w) acc = acc + ora_grad(grads, dtype, (int64_t)w * n + i);", 0),
    ("loco_mean_descending",
     "for (int32_t w = 0; w < W; ++w) {\n            float deq",
     "for (int32_t w = W - 1; w >= 0; --w) {\n            float deq", 0),
    ("server_sum_descending", "for (int32_t w = 0; w < W; ++w) {\n            float sent;",
     "for (int32_t w = W - 1; w >= 0; --w) {\n            float sent;", 0),
    ("drop_server_error", "y[i] = avg + server_err[i];", "y[i] = avg;", 0),
    ("residual_reversed", "resid[i] = z[i] - ora_signed(scales[i / C], ora_sign_bit(z[i]));",
     "resid[i] = ora_signed(scales[i / C], ora_sign_bit(z[i])) - z[i];", 0),
    ("mask_ignored", "mi = mi * keep;", "mi = mi * 1.0f + 0.0f * keep;", 0),
    ("eps_inside_sqrt", "float denom = sqrtf(v) + eps;", "float denom = sqrtf(v + eps);", 0),
    ("bit_order_reversed", "word |= (uint32_t)1 << t;", "word |= (uint32_t)1 << (31 - t);", 0),
    ("f16_exponent_bias", "expo - 25", "expo - 24", 0),
    ("unpack_wrong_chunk", "out[i] = ora_signed(scales[i / C], bit);",
     "out[i] = ora_signed(scales[(i / C + 1) % (n / C)], bit);", 0),
    ("worker_row_transposed", "float g = ora_grad(grads, dtype, (int64_t)w * n + i);",
     "float g = ora_grad(grads, dtype, (int64_t)i * W + w);", 0),
    ("warmup_v_not_squared", "float v_new = c2 * sq;", "float v_new = c2 * gbar;", 0),
    ("warmup_mean_not_divided", "float gbar = acc / (float)W;", "float gbar = acc;", 0),
    ("weight_decay_sign", "u = u + decay;", "u = u - decay;", 0),
    ("compressed_drops_weight_decay", "x[i] = ora_apply_update(x[i], mi, v[i], eps, lr, wd);",
     "x[i] = ora_apply_update(x[i], mi, v[i], eps, lr, 0.0f);", 0),
    ("loco_truncate", "float r = rintf(c[i] / s);", "float r = truncf(c[i] / s);", 0),
    ("loco_nibbles_swapped",
     "cw[j] = (uint8_t)(((uint8_t)qw[2 * j] & 0x0f) | (((uint8_t)qw[2 * j + 1] & 0x0f) << 4));",
     "cw[j] = (uint8_t)(((uint8_t)qw[2 * j + 1] & 0x0f) | (((uint8_t)qw[2 * j] & 0x0f) << 4));", 0),
    ("loco_no_average", "float new_part = keep * e;", "float new_part = e;", 0),
    ("loco_scale_levels", "float s = amax / flevels;", "float s = amax / (flevels + 1.0f);", 0),
    ("loco_drop_compensation",
     "c[i] = ora_grad(grads, dtype, (int64_t)w * n + i) + comp;",
     "c[i] = ora_grad(grads, dtype, (int64_t)w * n + i);", 0),
    ("loco_ratio_ignored", "float comp = ratio * et[i];", "float comp = et[i];", 0),
    ("loco_momentum_b2", "float m_old = b1 * m[i];", "float m_old = b2 * m[i];", 1),
    ("loco_variance_b1", "float v_old = b2 * v[i];", "float v_old = b1 * v[i];", 1),
    ("loco_dequant_first_chunk_scale",
     "float deq = (float)q[(int64_t)w * n + i] * scales[(int64_t)w * nchunks + i / C];",
     "float deq = (float)q[(int64_t)w * n + i] * scales[(int64_t)w * nchunks];", 0),
    ("loco_8bit_codes_shifted", "for (int64_t i = 0; i < n; ++i) cw[i] = (uint8_t)qw[i];",
     "for (int64_t i = 0; i < n; ++i) cw[i] = (uint8_t)(qw[i] + 1);", 0),
    ("loco_levels_off_by_one", "const int levels = (1 << (bits - 1)) - 1;",
     "const int levels = bits == 8 ? 128 : (1 << (bits - 1)) - 1;", 0),
    ("loco_ratio_on_average", "float old_part = beta * et[i];", "float old_part = beta * ratio * et[i];", 0),
]


def _mutate(src, old, new, occurrence):
    parts = src.split(old)
    assert len(parts) > occurrence + 1, "mutation target not found: %r" % old
    return old.join(parts[:occurrence + 1]) + new + old.join(parts[occurrence + 1:])


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    src = tmp_path / ("mutant_%s.c" % name)
    src.write_text(_mutate(SRC, old, new, occ))
    lib = obuild.build(str(src), str(tmp_path / ("libmutant_%s.so" % name)), force=True)
    ora = oracle.Oracle(lib)
    caught = []
    for pin_name, pin in PINS.items():
        try:
            pin(ora)
        except (AssertionError, ValueError):
            caught.append(pin_name)
    assert caught, "planted mistake %s passed every pin" % name
