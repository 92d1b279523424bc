"""Pins of the oracle's weight-only int4 format (oracle/quant.py).

The format: W(n, k) = bf16(s(n, k // 64) * (u(n, k) - 8)), codes two per byte
(low nibble = even input index). Checked here against a hand-decoded example,
against exact rational arithmetic with an independently written rounding rule,
and through a round-to-nearest quantiser whose reconstruction must lie within
half a scale step.
"""
from fractions import Fraction

import numpy as np
import pytest

import fixtures as FX
from oracle import model as OM
from oracle import quant as OQ


def test_hand_decoded_bytes():
    # row 0: bytes 0x9F, 0x80 then zeros (code 0 -> -8); row 1: all 0x88 (zero weights)
    codes = np.zeros((2, 32), np.uint8)
    codes[0, 0], codes[0, 1] = 0x9F, 0x80
    codes[1, :] = 0x88
    scales = np.array([[0.5], [3.0]], np.float32)
    w = OQ.dequantize(codes, scales)
    assert w.shape == (2, 64)
    # 0x9F: low nibble 15 -> +7, high nibble 9 -> +1; 0x80: low 0 -> -8, high 8 -> 0
    assert w[0, :4].tolist() == [3.5, 0.5, -4.0, 0.0]
    assert (w[0, 4:] == -4.0).all()
    assert (w[1] == 0.0).all()


def _nearest_bf16(q: Fraction) -> float:
    """Nearest bfloat16 to an exact rational (ties to an even significand), by enumeration."""
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    # a in [1, 2): significand with 7 fraction bits
    lo = int(a * 128)
    frac = a * 128 - lo
    if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * float(Fraction(lo, 128) * Fraction(2) ** e)


def test_every_code_against_exact_products():
    rng = np.random.default_rng(3)
    # bf16 scales over many exponents with random 8-bit significands
    sig = rng.integers(128, 256, 40)
    exp = rng.integers(-20, 4, 40)
    scales = np.array([float(Fraction(int(m), 128) * Fraction(2) ** int(e)) for m, e in zip(sig, exp)], np.float32)
    assert (OQ.bf16_round(scales) == scales).all()
    codes = np.zeros((40, 32), np.uint8)
    for c in range(16):   # codes 0..15 at inputs 2c (low nibble) and 2c + 1 (high nibble, code 15 - c)
        codes[:, c] = c | ((15 - c) << 4)
    w = OQ.dequantize(codes, scales[:, None])
    for n in range(40):
        s = Fraction(float(scales[n]))
        for k in range(64):
            # byte k // 2 < 16 holds codes (k // 2, 15 - k // 2); bytes 16.. are zero (code 0)
            u = 0 if k >= 32 else (k // 2 if k % 2 == 0 else 15 - k // 2)
            assert w[n, k] == _nearest_bf16(s * (u - 8)), (n, k, u, float(s), w[n, k])


def test_round_to_nearest_quantiser_reconstructs_within_half_a_step():
    rng = np.random.default_rng(8)
    W = OQ.bf16_round((rng.standard_normal((16, 256)) * 0.02).astype(np.float32))
    g = W.reshape(16, 4, 64)
    s = OQ.bf16_round((np.abs(g).max(-1) / 7.0).astype(np.float32))   # bf16 scale per group
    u = np.clip(np.rint(g / s[..., None]) + 8, 0, 15).astype(np.uint8).reshape(16, 256)
    codes = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    R = OQ.dequantize(codes, s)
    step = np.repeat(s, 64, axis=1)
    # half a step for the code, plus one bf16 rounding of the result and of the scale's clipping
    assert (np.abs(R - W) <= 0.5 * step * (1 + 2 ** -7) + np.abs(W) * 2 ** -8 + 1e-12).all()


def test_fixture_codes_and_scales():
    m = FX.TINY.reduced(weight_bits=4)
    c = FX.int4_codes(m, 0, "wq")
    s = FX.int4_scales(m, 0, "wq")
    assert c.shape == (m.q_dim, m.d // 2) and s.shape == (m.q_dim, m.d // 64)
    u = OQ.unpack_codes(c)
    assert u.min() >= 1 and u.max() <= 15 and len(np.unique(u)) == 15
    base = FX.int4_scale_base(m)
    assert (s >= 0.74 * base).all() and (s <= 1.26 * base).all()
    w = OQ.dequantize(c, s)
    assert abs(float(w.std()) - m.init_std) < 0.1 * m.init_std
    # the element index of a code is row * K + input: a different row range gives a different stream
    assert not np.array_equal(c[0], c[1])


def test_int4_model_uses_dequantised_projections_only():
    m4 = FX.TINY.reduced(weight_bits=4, n_layers=1, ffn=704)   # int4 needs every K % 64 == 0
    M = OM.build_model(m4, 64)
    M16 = OM.build_model(FX.TINY.reduced(n_layers=1, ffn=704), 64)
    np.testing.assert_array_equal(M.layers[0].wd, OQ.dequantize(FX.int4_codes(m4, 0, "wd"), FX.int4_scales(m4, 0, "wd")))
    np.testing.assert_array_equal(M.embed, M16.embed)
    np.testing.assert_array_equal(M.lm_head, M16.lm_head)
    np.testing.assert_array_equal(M.head_layer.wq, M16.head_layer.wq)


def test_int4_target_speculative_decoding_is_lossless():
    from oracle import decode as OD
    import dataclasses
    m4 = FX.TINY.reduced(weight_bits=4, ffn=704)
    w = dataclasses.replace(FX.WORKLOADS["tiny_static"], model=m4, max_new=16)
    cap = FX.kv_capacity(w)
    M = OM.build_model(m4, cap)
    p = FX.prompts(m4, 1, w.prompt_len)[0]
    assert OD.speculative_generate(M, p, w, cap=cap).out == OD.vanilla_greedy(M, p, 16, cap)
