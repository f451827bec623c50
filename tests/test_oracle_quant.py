"""Pins of the oracle's Q8_0 and Q4_0 weight quantisers (no GPU).

"opus-mtp-turbo: Track 1 report", item 3: the Q8_0 column of its
quantisation-error table (GEMV output rel-RMSE 0.58 %-1.18 % on the real MTP
tensors).  The format follows ggml's rule: blocks of 32 weights, scale
max|w| / 127 stored as binary16, codes round(w / scale).  Pinned by the
binary16 scales against numpy's float16 conversion, exact reconstruction of
weights that are code multiples of a binary16 scale, the per-element error
bound, the extreme code at the block maximum, zero blocks, and the GEMV error
on Gaussian data against the magnitude the page prints.
"""
import numpy as np
import pytest

import oracle
import synth


def test_scales_are_numpys_float16_of_the_fp32_scale():
    rng = np.random.default_rng(3)
    # block maxima over many binades, subnormal and overflowing scales included
    amax = np.concatenate([10.0 ** rng.uniform(-9, 7, 600), [0.0, 1e-30, 65504 * 127.0, 3e9]]).astype(np.float32)
    w = np.zeros((amax.size, 32), dtype=np.float32)
    w[:, 5] = amax
    w[:, 9] = -amax / 3
    _, d = oracle.quantize_q8_0(w)
    with np.errstate(over="ignore"):   # scales past binary16's range become infinity
        want = (amax / np.float32(127)).astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(d[:, 0], want)


def test_code_multiples_of_a_float16_scale_reconstruct_exactly():
    d = np.float32(2.0 ** -4)
    k = np.arange(-127, 128, dtype=np.float32)
    rows = []
    for r in range(8):
        blk = np.resize(np.roll(k, 37 * r), 32).astype(np.float32)
        blk[0] = 127.0   # the block maximum gives the scale exactly
        rows.append(blk * d)
    w = np.concatenate(rows).reshape(2, 128)
    q, s = oracle.quantize_q8_0(w)
    np.testing.assert_array_equal(s, np.full_like(s, np.float16(d).view(np.uint16)))
    np.testing.assert_array_equal(oracle.dequantize_q8_0(q, s), w)
    np.testing.assert_array_equal(q.astype(np.float32) * d, w)


def test_error_bound_and_extreme_code():
    w = synth.normal(7, "q8w", (64, 256), std=0.02)
    q, s = oracle.quantize_q8_0(w)
    dq = oracle.dequantize_q8_0(q, s)
    d = s.view(np.float16).astype(np.float64)                    # [64, 8] scales as stored
    scale = np.repeat(d, 32, axis=1)
    err = np.abs(dq.astype(np.float64) - w.astype(np.float64))
    # |w - d q| <= d / 2 for the fp32 scale; the binary16 scale moves d q by at most 127 |d16 - d|
    assert np.all(err <= scale * (0.5 + 127 * 2.0 ** -11) + 1e-12)
    blocks = w.reshape(64, 8, 32)
    at = np.abs(blocks).argmax(axis=2)
    qb = q.reshape(64, 8, 32)
    top = np.take_along_axis(qb, at[..., None], axis=2)[..., 0]
    assert np.all(np.abs(top) == 127)
    assert np.all(np.abs(q) <= 127)


def test_zero_block():
    w = np.zeros((1, 64), dtype=np.float32)
    w[0, 40] = 1.0
    q, s = oracle.quantize_q8_0(w)
    assert s[0, 0] == 0 and np.all(q[0, :32] == 0)
    assert q[0, 40] == 127


def test_gemv_error_matches_the_reports_magnitude():
    """rel-RMSE of W x with Q8_0 weights on Gaussian data: the page measures
    0.58-1.18 % on real tensors; Gaussian weights give about 0.5-0.6 %."""
    w = synth.normal(8, "q8g", (256, 1024), std=0.02)
    x = synth.normal(8, "q8x", (1024,)).astype(np.float64)
    q, s = oracle.quantize_q8_0(w)
    y = w.astype(np.float64) @ x
    yq = oracle.dequantize_q8_0(q, s).astype(np.float64) @ x
    rel = np.sqrt(np.mean((yq - y) ** 2) / np.mean(y ** 2))
    assert 0.003 < rel < 0.0125


def test_rejects_ragged_rows():
    with pytest.raises(ValueError):
        oracle.quantize_q8_0(np.zeros((2, 48), dtype=np.float32))


# ----------------------------------------------------------------------------
# Q4_0 ("opus-mtp-turbo: Track 1 report", item 3, the Q4_0 column; ggml's
# scale rule d = m / -8 with m the block's weight of largest magnitude)
# ----------------------------------------------------------------------------

def test_q4_scales_are_numpys_float16_of_the_signed_extreme_over_minus_eight():
    rng = np.random.default_rng(4)
    m = (rng.choice([-1.0, 1.0], 500) * 10.0 ** rng.uniform(-9, 5, 500)).astype(np.float32)
    w = np.zeros((m.size, 32), dtype=np.float32)
    w[:, 3] = m
    w[:, 20] = -m / 2          # smaller magnitude, opposite sign: m stays the extreme
    _, d = oracle.quantize_q4_0(w)
    with np.errstate(over="ignore"):
        want = (m / np.float32(-8)).astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(d[:, 0], want)


def test_q4_codes_and_nibble_layout_on_a_worked_block():
    """A block whose extreme is -8: d = 1, so each weight q - 8 gets code q;
    byte j holds the code of weight j (low four bits) and of weight j + 16
    (high four)."""
    codes = np.array([0, 15, 3, 8, 9, 1, 14, 7, 2, 12, 5, 10, 6, 13, 4, 11,
                      11, 4, 13, 6, 10, 5, 12, 2, 7, 14, 1, 9, 8, 3, 15, 0], dtype=np.int64)
    w = (codes - 8).astype(np.float32).reshape(1, 32)
    q, d = oracle.quantize_q4_0(w)
    assert d[0, 0] == np.float16(1.0).view(np.uint16)
    want = (codes[:16] | (codes[16:] << 4)).astype(np.uint8)
    np.testing.assert_array_equal(q[0], want)
    np.testing.assert_array_equal(oracle.dequantize_q4_0(q, d), w)
    # the same block scaled by 2^-5: the same codes, the scale 2^-5, exact again
    q2, d2 = oracle.quantize_q4_0(w * np.float32(2.0 ** -5))
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(oracle.dequantize_q4_0(q2, d2), w * np.float32(2.0 ** -5))


def test_q4_error_bound_extreme_code_and_clamp():
    w = synth.normal(9, "q4w", (64, 256), std=0.02)
    q, s = oracle.quantize_q4_0(w)
    dq = oracle.dequantize_q4_0(q, s).astype(np.float64)
    d = np.abs(np.repeat(s.view(np.float16).astype(np.float64), 32, axis=1))
    err = np.abs(dq - w.astype(np.float64))
    # nearest code: |d| / 2; a weight at +|m| clamps to code 15: |d|; plus the binary16 scale's rounding
    assert np.all(err <= d * (1.0 + 16 * 2.0 ** -11) + 1e-12)
    assert np.mean(err <= d * (0.5 + 8 * 2.0 ** -11) + 1e-12) > 0.99
    blocks = w.reshape(64, 8, 32)
    at = np.abs(blocks).argmax(axis=2)            # the first extreme of each block
    lo = (q & 15).reshape(64, 8, 16)
    hi = (q >> 4).reshape(64, 8, 16)
    codes = np.concatenate([lo, hi], axis=2)
    assert np.all(np.take_along_axis(codes, at[..., None], axis=2) == 0)
    assert codes.max() <= 15
    # an opposite extreme of the same magnitude clamps to 15
    blk = np.zeros((1, 32), dtype=np.float32)
    blk[0, 0], blk[0, 9] = -2.0, 2.0
    qc, _ = oracle.quantize_q4_0(blk)
    assert (qc[0, 0] & 15) == 0 and (qc[0, 9] & 15) == 15


def test_q4_zero_block():
    q, d = oracle.quantize_q4_0(np.zeros((1, 64), dtype=np.float32))
    assert np.all((d & 0x7FFF) == 0) and np.all(q == 0x88)   # 0 / -8 is a negative zero
    np.testing.assert_array_equal(oracle.dequantize_q4_0(q, d), np.zeros((1, 64), dtype=np.float32))


def test_q4_gemv_error_matches_the_reports_magnitude():
    """rel-RMSE of W x with Q4_0 weights on Gaussian data: the page measures
    5.8-10.7 % on real tensors with its Lloyd quantiser; ggml's rule on
    Gaussian weights gives about 8-9 %."""
    w = synth.normal(8, "q4g", (256, 1024), std=0.02)
    x = synth.normal(8, "q4x", (1024,)).astype(np.float64)
    q, s = oracle.quantize_q4_0(w)
    y = w.astype(np.float64) @ x
    yq = oracle.dequantize_q4_0(q, s).astype(np.float64) @ x
    rel = np.sqrt(np.mean((yq - y) ** 2) / np.mean(y ** 2))
    assert 0.05 < rel < 0.13


def test_q4_rejects_ragged_rows():
    with pytest.raises(ValueError):
        oracle.quantize_q4_0(np.zeros((2, 48), dtype=np.float32))
