"""Pins of the oracle's building blocks against library routines, closed forms
and brute force (no GPU).  Every check here is independent of the oracle's own
formula text: a library computes the expected value, or a closed form /
invariant fixes it."""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def test_philox_known_answers():
    """Random123's published KAT vectors for Philox-4x32-10."""
    n = 0
    for line in open(os.path.join(HERE, "golden", "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(x, 16) for x in line.split()]
        assert list(oracle.philox4x32_10(v[0:4], v[4:6])) == v[6:]
        n += 1
    assert n == 3


def test_uniform_range_and_counter_layout():
    us = [oracle.uniform(7, 3, b, i, p) for b in range(4) for i in range(4) for p in range(4)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert len(set(us)) == len(us)
    # u = (word0 >> 8) * 2^-24 of philox(ctr = (b, 4 i + purpose, off lo, off hi), key = (seed lo, seed hi))
    seed, off = 0x123456789ABCDEF0, 0x0FEDCBA987654321
    o = oracle.philox4x32_10([5, 4 * 2 + 3, off & 0xFFFFFFFF, off >> 32], [seed & 0xFFFFFFFF, seed >> 32])
    assert oracle.uniform(seed, off, 5, 2, 3) == (int(o[0]) >> 8) / 2.0 ** 24


@pytest.mark.parametrize("n", [1, 7, 256, 1000])
def test_rmsnorm_matches_torch(n):
    rng = np.random.default_rng(n)
    x = rng.standard_normal(n)
    g = (1 + 0.02 * rng.standard_normal(n)).astype(np.float32)
    ref = F.rms_norm(torch.from_numpy(x), (n,), weight=torch.from_numpy(g.astype(np.float64)), eps=1e-6)
    assert np.allclose(oracle.rmsnorm(x, g, 1e-6), ref.numpy(), rtol=1e-13, atol=1e-13)


def test_rmsnorm_of_zero_is_zero():
    assert np.all(oracle.rmsnorm(np.zeros(16), None, 1e-6) == 0.0)


@pytest.mark.parametrize("bf16", [False, True])
def test_matvec_matches_torch(bf16):
    rng = np.random.default_rng(3)
    W32 = rng.standard_normal((37, 129)).astype(np.float32)
    W = synth.f32_to_bf16_bits(W32) if bf16 else W32
    Wd = (synth.bf16_bits_to_f32(W) if bf16 else W32).astype(np.float64)
    x = rng.standard_normal(129)
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(Wd)).numpy()
    assert np.allclose(oracle.matvec(W, x, bf16), ref, rtol=1e-12, atol=1e-12)


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.0078125, 1.01171875, -2.5, 3.0e-39, np.inf], dtype=np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even mantissa (1.0); 1 + 3*2^-8 ties up to 1 + 2^-6
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(vals))
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0078125 and got[3] == 1.015625
    assert got[4] == -2.5 and np.isinf(got[6])
    t = torch.from_numpy(vals).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got[:6], t[:6])


def test_gelu_tanh_matches_torch():
    x = np.linspace(-6, 6, 101)
    ref = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(oracle.gelu_tanh(x), ref, rtol=1e-13, atol=1e-14)


def test_rope_closed_forms():
    rng = np.random.default_rng(0)
    hd = 32
    q = rng.standard_normal(hd)
    # position 0 is the identity; every position preserves the norm
    assert np.allclose(oracle.rope_neox(q, 0, 1e4), q, atol=0)
    for pos in (1, 17, 8191):
        r = oracle.rope_neox(q, pos, 1e4)
        assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-12
    # the NeoX pairing is multiplication of (q_i + j q_{i+hd/2}) by exp(j pos theta^(-2i/hd))
    pos, theta = 123, 1e6
    z = q[: hd // 2] + 1j * q[hd // 2:]
    ang = pos * theta ** (-2.0 * np.arange(hd // 2) / hd)
    zr = z * np.exp(1j * ang)
    r = oracle.rope_neox(q, pos, theta)
    assert np.allclose(r[: hd // 2], zr.real, atol=1e-12) and np.allclose(r[hd // 2:], zr.imag, atol=1e-12)


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    a = oracle.rope_neox(q, 100, 1e4) @ oracle.rope_neox(k, 90, 1e4)
    b = oracle.rope_neox(q, 1010, 1e4) @ oracle.rope_neox(k, 1000, 1e4)
    assert abs(a - b) < 1e-9


def test_argmax_ties_and_nan():
    assert oracle.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax([np.nan, 1.0, np.nan, 1.0]) == 1
    assert oracle.argmax([np.nan, np.nan]) == 0
    assert oracle.argmax([-np.inf, -np.inf, -5.0]) == 2
    assert oracle.argmax([np.nan, -np.inf, -np.inf]) == 1


def _kv(rng, B, H, cap, hd):
    return rng.standard_normal((B, H, cap, hd)).astype(np.float32), rng.standard_normal((B, H, cap, hd)).astype(np.float32)


@pytest.mark.parametrize("kv_len,window,cap", [(1, 0, 8), (40, 0, 40), (40, 16, 24), (100, 7, 7), (5, 16, 16)])
def test_attention_matches_sdpa(kv_len, window, cap):
    """Ring-buffer, windowed, GQA cross-attention vs torch SDPA on the gathered keys."""
    rng = np.random.default_rng(kv_len * 31 + window)
    B, Hq, Hkv, hd = 2, 4, 2, 16
    k, v = _kv(rng, B, Hkv, cap, hd)
    q = rng.standard_normal((Hq, hd))
    lo = max(0, kv_len - window) if window else 0
    slots = np.arange(lo, kv_len) % cap
    for b in range(B):
        Kt = torch.from_numpy(k[b][:, slots, :].astype(np.float64)).repeat_interleave(Hq // Hkv, dim=0)
        Vt = torch.from_numpy(v[b][:, slots, :].astype(np.float64)).repeat_interleave(Hq // Hkv, dim=0)
        ref = F.scaled_dot_product_attention(torch.from_numpy(q)[:, None, :], Kt, Vt)[:, 0, :].numpy()
        for h in range(Hq):
            got = oracle.attend_head(q[h], k, v, b, h // (Hq // Hkv), kv_len, window)
            assert np.allclose(got, ref[h], rtol=1e-11, atol=1e-11)


def test_attention_brute_force_bf16():
    rng = np.random.default_rng(9)
    k32, v32 = _kv(rng, 1, 1, 12, 8)
    kb, vb = synth.f32_to_bf16_bits(k32), synth.f32_to_bf16_bits(v32)
    K, Vv = synth.bf16_bits_to_f32(kb).astype(np.float64), synth.bf16_bits_to_f32(vb).astype(np.float64)
    q = rng.standard_normal(8)
    s = np.array([(q @ K[0, 0, t]) / math.sqrt(8) for t in range(12)])
    w = np.exp(s - s.max())
    ref = sum(w[t] * Vv[0, 0, t] for t in range(12)) / w.sum()
    assert np.allclose(oracle.attend_head(q, kb, vb, 0, 0, 12, 0, bf16=True), ref, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(5)
    k, v = _kv(rng, 1, 1, 32, 16)
    q = rng.standard_normal(16)
    # one key: the output is that key's value row
    assert np.allclose(oracle.attend_head(q, k, v, 0, 0, 1), v[0, 0, 0], atol=1e-12)
    # identical keys: the output is the mean of the values
    ke = np.repeat(k[:, :, :1, :], 32, axis=2)
    assert np.allclose(oracle.attend_head(q, ke, v, 0, 0, 20), v[0, 0, :20].mean(0), atol=1e-12)
    # window 1: the newest position's value
    assert np.allclose(oracle.attend_head(q, k, v, 0, 0, 20, window=1), v[0, 0, 19], atol=1e-12)
    # a window at least as long as the context is full attention
    assert np.allclose(oracle.attend_head(q, k, v, 0, 0, 20, window=20),
                       oracle.attend_head(q, k, v, 0, 0, 20, window=0), atol=0)
    assert np.allclose(oracle.attend_head(q, k, v, 0, 0, 20, window=64),
                       oracle.attend_head(q, k, v, 0, 0, 20, window=0), atol=0)


def test_attention_ignores_poisoned_slots():
    """Slots outside [kv_len - W, kv_len) hold NaN and must not reach the output."""
    rng = np.random.default_rng(6)
    k, v = _kv(rng, 1, 1, 16, 8)
    kv_len, W = 21, 6
    mask = synth.view_valid_mask(16, W, kv_len)
    k[0, 0, ~mask] = np.nan
    v[0, 0, ~mask] = np.nan
    out = oracle.attend_head(rng.standard_normal(8), k, v, 0, 0, kv_len, W)
    assert np.all(np.isfinite(out))


# ----------------------------------------------------------------------------
# sink + window ("opus-mtp-turbo: Track 1 report", item 2): the draft
# attention reads the first `sink` positions beside the window; position t is
# stored in slot t below the sink and in a ring over the other slots above it
# ----------------------------------------------------------------------------

def _plain_attention(q, keys, vals):
    s = keys @ q / np.sqrt(q.size)
    p = np.exp(s - s.max())
    return (p[:, None] * vals).sum(0) / p.sum()


@pytest.mark.parametrize("kv_len,W,S,cap", [(100, 40, 8, 48), (45, 40, 8, 48), (30, 40, 8, 48),
                                             (200, 16, 16, 40), (9, 4, 4, 8)])
def test_sink_window_brute_force(kv_len, W, S, cap):
    """The key set enumerated by hand: [0, min(S, lo)) then [lo, kv_len),
    gathered from their slots; every other slot holds NaN."""
    rng = np.random.default_rng(kv_len + S)
    hd = 16
    k = np.full((1, 1, cap, hd), np.nan, dtype=np.float32)
    v = np.full((1, 1, cap, hd), np.nan, dtype=np.float32)
    lo = max(0, kv_len - W)
    pos = list(range(min(S, lo))) + list(range(lo, kv_len))
    slot = [t if t < S else S + (t - S) % (cap - S) for t in pos]
    assert len(set(slot)) == len(slot)      # every read position has its own slot
    kk = rng.standard_normal((len(pos), hd)).astype(np.float32)
    vv = rng.standard_normal((len(pos), hd)).astype(np.float32)
    k[0, 0, slot] = kk
    v[0, 0, slot] = vv
    q = rng.standard_normal(hd)
    got = oracle.attend_head(q, k, v, 0, 0, kv_len, W, sink=S)
    assert np.allclose(got, _plain_attention(q, kk.astype(np.float64), vv.astype(np.float64)), atol=1e-12)


def test_sink_zero_is_the_plain_window_and_a_wide_sink_the_full_view():
    rng = np.random.default_rng(11)
    cap, hd = 64, 8
    k = rng.standard_normal((1, 1, cap, hd)).astype(np.float32)
    v = rng.standard_normal((1, 1, cap, hd)).astype(np.float32)
    q = rng.standard_normal(hd)
    assert np.array_equal(oracle.attend_head(q, k, v, 0, 0, 50, 20, sink=0),
                          oracle.attend_head(q, k, v, 0, 0, 50, 20))
    # kv_len - W <= sink and cap >= kv_len: every position in slot t, all read
    assert np.allclose(oracle.attend_head(q, k, v, 0, 0, 40, 24, sink=16),
                       oracle.attend_head(q, k, v, 0, 0, 40, 0), atol=0)


def test_synth_sink_layout_matches_the_read_set():
    m = synth.ModelSpec(d_t=32, d_a=32, n_blocks=1, n_q_heads=2, head_dim=16, n_kv_heads=1, d_ff=64,
                        vocab=64, dtype="f32", block_view=(0,))
    vs = synth.ViewSpec(cap=48, window=40, rope_theta=1e4, sink=8)
    view = synth.make_kv_view(m, vs, np.array([100, 45, 23], dtype=np.int32), 3, "s")
    for b, L in enumerate((100, 45, 23)):
        finite = np.isfinite(view["k"][b, 0, :, 0])
        assert finite.sum() == len(synth.view_positions(40, L, 8))
