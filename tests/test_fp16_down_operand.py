"""The fp16 operand format of the down projection, checked on the host over
every bf16 bit pattern: bf16 -> fp16 (round to nearest even) is exact from
2^-14 (fp16's smallest normal) up to fp16's largest value, within 2^-25 of
the value below 2^-14, and overflows only beyond 65504.  These are the facts
the library's fp16 down weights rest on."""
import numpy as np


def _all_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    return vals[np.isfinite(vals)]


def test_normal_range_converts_exactly():
    v = _all_bf16()
    sel = (np.abs(v) >= 2.0 ** -14) & (np.abs(v) <= 65504.0)
    h = v[sel].astype(np.float16)
    assert np.array_equal(h.astype(np.float32), v[sel])
    assert sel.sum() == 30 * 128 * 2  # binades 2^-14 .. 2^15, 7 stored bits, two signs


def test_small_values_err_at_most_half_a_subnormal_step():
    v = _all_bf16()
    sel = np.abs(v) < 2.0 ** -14
    err = np.abs(v[sel].astype(np.float16).astype(np.float64) - v[sel].astype(np.float64))
    assert err.max() <= 2.0 ** -25


def test_overflow_only_beyond_the_fp16_range():
    v = _all_bf16()
    with np.errstate(over="ignore"):
        inf = np.isinf(v.astype(np.float16))
    assert np.array_equal(inf, np.abs(v) > 65504.0)


def test_weight_scale_values_are_in_the_exact_range():
    """N(0, 0.02) weights (the synthetic and Qwen3-like scale): the share
    below 2^-14 is tiny, so almost every weight converts exactly."""
    rng = np.random.default_rng(0)
    w = (0.02 * rng.standard_normal(1 << 20)).astype(np.float32)
    assert np.mean(np.abs(w) < 2.0 ** -14) < 0.005
