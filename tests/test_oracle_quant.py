"""Pins of the oracle's Q8_0 weight quantiser (no GPU).

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
