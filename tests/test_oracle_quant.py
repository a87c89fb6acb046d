"""Pins of the low-bit KV oracle (per-row symmetric quantization, quantizing
append, attention over the quantized cache) and planted mistakes that must
fail one of them.

Pinned against the notebook's own definition (``fake_quantize_rows``,
float64 scale): with the scale stored as float32, every dequantized value
stays within one quantization step of the notebook's and nearly all codes
agree; against closed forms (the row maximum maps to +-limit, a zero row has
scale 1 and zero codes, every value is within half a step of its code);
and against the notebook's experiment (attention over 8-bit K/V is closer to
the exact attention than over 3-bit K/V).
"""

import numpy as np
import pytest

import oracle.quant as Q
from oracle import attention as OA


def page_fake_quantize_rows(x, bits):
    """The notebook's definition, float64 throughout (the pin's reference)."""
    limit = 2 ** (bits - 1) - 1
    scale = np.max(np.abs(x), axis=-1, keepdims=True) / limit
    scale = np.where(scale == 0, 1.0, scale)
    codes = np.clip(np.rint(x / scale), -limit, limit)
    return codes * scale, scale, codes


def pin_against_page_definition():
    x = np.random.default_rng(1).standard_normal((4000, 128)).astype(np.float32).astype(np.float64)
    for bits in (8, 3):
        c, s = Q.quantize_rows(x, bits)
        ours = Q.dequantize_rows(c, s)
        page, ps, pc = page_fake_quantize_rows(x, bits)
        assert np.all(np.abs(ours - page) <= 1.0001 * ps)       # within one step everywhere
        assert np.mean(c != pc) < 1e-3                         # and the same code nearly everywhere


def pin_closed_forms():
    rows = np.array([[1.0, -2.0, 4.0, 0.5], [0.0, 0.0, 0.0, 0.0], [-3.0, 1.5, 0.0, 2.9]])
    c, s = Q.quantize_rows(rows, 8)
    assert c[0, 2] == 127 and c[2, 0] == -127              # the row maximum maps to +-limit
    assert s[1] == 1.0 and np.all(c[1] == 0)                # zero row
    assert s.dtype == np.float32 and c.dtype == np.int8
    assert s[0] == np.float32(np.float32(4.0) / np.float32(127.0))
    c3, _ = Q.quantize_rows(rows, 3)
    assert c3.min() >= -3 and c3.max() <= 3 and c3[0, 2] == 3
    x = np.random.default_rng(2).standard_normal((500, 64)) * np.random.default_rng(3).uniform(1e-3, 1e3, (500, 1))
    c, s = Q.quantize_rows(x, 8)
    assert np.all(np.abs(x - Q.dequantize_rows(c, s)) <= 0.5 * s.astype(np.float64)[:, None] * (1 + 1e-12))


def pin_append():
    rng = np.random.default_rng(4)
    kc = np.zeros((6, 2, 16, 8), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((6, 2, 16), np.float32)
    vs = np.zeros_like(ks)
    kn = rng.standard_normal((3, 2, 8))
    vn = rng.standard_normal((3, 2, 8))
    Q.append_tokens_q8(kc, vc, ks, vs, kn, vn, [5 * 16 + 3, -1, 17])
    c, s = Q.quantize_rows(kn)
    assert np.array_equal(kc[5, :, 3], c[0]) and np.array_equal(kc[1, :, 1], c[2]) and np.array_equal(ks[5, :, 3], s[0])
    c, s = Q.quantize_rows(vn)
    assert np.array_equal(vc[1, :, 1], c[2]) and np.array_equal(vs[1, :, 1], s[2])
    assert np.count_nonzero(ks) == 4                     # the skipped token wrote nothing


def pin_attention_over_quantized_cache():
    rng = np.random.default_rng(5)
    nb, hkv, G, d = 12, 2, 4, 64
    kp = rng.standard_normal((nb, hkv, 16, d)).astype(np.float32)
    vp = rng.standard_normal((nb, hkv, 16, d)).astype(np.float32)
    q = rng.standard_normal((3, hkv * G, d)).astype(np.float32)
    tables = np.array([[3, 7, 1, 0], [5, 2, 9, 11], [4, 6, 8, 10]])
    lens = np.array([50, 64, 17])
    exact = OA.decode_attention(q, kp, vp, tables, lens, 0.125, hkv, "f32")
    errs = {}
    for bits in (8, 3):
        kc, ks = Q.quantize_rows(kp, bits)
        vc, vs = Q.quantize_rows(vp, bits)
        got = Q.decode_attention_q8(q, kc, vc, ks, vs, tables, lens, 0.125, hkv, "f32")
        ref = OA.decode_attention(q, Q.dequantize_rows(kc, ks), Q.dequantize_rows(vc, vs), tables, lens, 0.125,
                                  hkv, "f64")
        assert np.max(np.abs(got - ref)) < 1e-12
        errs[bits] = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert errs[8] < 0.02 and errs[8] < errs[3]


PINS = [pin_against_page_definition, pin_closed_forms, pin_append, pin_attention_over_quantized_cache]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ------------------------------------------------------------------ mutants
_orig_q = Q.quantize_rows
_orig_dq = Q.dequantize_rows


def _scale_per_tensor(x, bits=8):
    limit = 2 ** (bits - 1) - 1
    x = np.asarray(x, dtype=np.float64)
    amax = np.float32(np.max(np.abs(x)))
    s = np.full(x.shape[:-1], np.float32(amax / np.float32(limit)), np.float32)
    return np.clip(np.rint(x / s.astype(np.float64)[..., None]), -limit, limit).astype(np.int8), s


def _floor_codes(x, bits=8):
    c, s = _orig_q(x, bits)
    return np.clip(np.floor(np.asarray(x, np.float64) / s.astype(np.float64)[..., None]), -127, 127).astype(np.int8), s


def _limit_off_by_one(x, bits=8):
    limit = 2 ** (bits - 1)
    x = np.asarray(x, dtype=np.float64)
    s = (np.max(np.abs(x), axis=-1).astype(np.float32) / np.float32(limit)).astype(np.float32)
    s = np.where(s == 0, np.float32(1), s).astype(np.float32)
    return np.clip(np.rint(x / s.astype(np.float64)[..., None]), -limit, limit - 1).astype(np.int8), s


def _dequant_without_scale(codes, scale):
    return codes.astype(np.float64)


MUTANTS = {
    "scale_per_tensor": ("quantize_rows", _scale_per_tensor),
    "floor_instead_of_round": ("quantize_rows", _floor_codes),
    "limit_off_by_one": ("quantize_rows", _limit_off_by_one),
    "dequant_without_scale": ("dequantize_rows", _dequant_without_scale),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_quant_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(Q, attr, fn)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError, OverflowError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
