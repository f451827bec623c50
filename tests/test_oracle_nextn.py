"""Pins of the oracle's dense NextN drafter (no GPU).

"MTP decoding (--mtp)": "Requirements" (the NextN block: enorm / hnorm /
eh_proj, the shared head with its norm), "How it is wired" (draft from the
head, verify, let the draft context catch up on the accepted prefix) and "The
catch-up runs on the accepted prefix" (accepting first and catching up on
[confirmed token, accepted drafts] leaves the same drafter state as catching up
on the whole batch and rolling the tail back); "Fused NextN draft graph", "The
two MTP lanes" (NextN keeps its own KV).

The building blocks (RMSNorm, the matrix-vector product, NeoX RoPE, the
attention of one head) are pinned in test_oracle.py.  Here: SiLU's closed
forms, the one-time bf16 rounding of the stored keys and values, and
properties of the chain that a slip in it would break -- a single key makes
the attention ignore the queries, a zero block reduces the drafter to eh_proj
and the head, permuting KV heads together with their query groups changes
nothing, one call equals two calls that carry the KV and the hidden state
over, and the page's accept-first claim.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def tiny(dtype="f32", B=2, N=3, M=2, kv_len=(0, 5), n_cu=(0, 2), seed=7, d=64, Hq=4, Hkv=2, hd=32, V=500):
    m = synth.NextnSpec(d=d, n_q_heads=Hq, head_dim=hd, n_kv_heads=Hkv, d_ff=128, vocab=V, dtype=dtype,
                        rope_theta=1e4)
    return synth.make_nextn_workload("tiny-nextn", m, B, N, M, list(kv_len)[:B], list(n_cu)[:B], seed)


def with_weights(w, **repl):
    """A copy of the workload with some weights replaced."""
    import copy
    w2 = copy.copy(w)
    w2.weights = dict(w.weights)
    w2.weights.update(repl)
    return w2


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    # x sigma(x): sigma(ln 3) = 3 / 4
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    xs = np.linspace(-9, 9, 37)
    # silu(x) - silu(-x) = x (sigma(x) + sigma(-x) = 1)
    np.testing.assert_allclose(oracle.silu(xs) - oracle.silu(-xs), xs, rtol=0, atol=1e-14)
    assert abs(oracle.silu(60.0) - 60.0) < 1e-20 * 60 + 1e-12
    assert abs(oracle.silu(-60.0)) < 1e-24


def test_bf16_rounding_once_to_nearest_even():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(2000) * 10.0 ** rng.uniform(-30, 30, 2000)).astype(np.float32)
    # values exact in fp32: the same as rounding the fp32 value
    np.testing.assert_array_equal(oracle.to_bf16(x.astype(np.float64)), synth.f32_to_bf16_bits(x))
    one = 1.0
    assert oracle.to_bf16(one + 2.0 ** -8) == 0x3F80          # tie -> even (1.0)
    assert oracle.to_bf16(one + 3 * 2.0 ** -8) == 0x3F82      # tie -> even (1 + 2^-6)
    assert oracle.to_bf16(-(one + 2.0 ** -8)) == 0xBF80
    # just above the tie: rounds up; an fp32 detour would land on the tie and round down
    assert oracle.to_bf16(one + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert oracle.to_bf16(2.0 ** -130) == 0x0008               # subnormal, exact
    assert oracle.to_bf16(float("inf")) == 0x7F80
    assert oracle.to_bf16(3.5e38) == 0x7F80                    # past the largest bf16
    assert oracle.to_bf16(float("nan")) == 0x7FC0
    assert oracle.to_bf16(0.0) == 0 and oracle.to_bf16(-0.0) == 0x8000


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_key_attention_ignores_the_queries(dtype):
    """An empty drafter KV and no catch-up: the first draft step attends to its
    own key only, so its output is the value whatever the queries are; with
    earlier rows in the KV the queries matter."""
    w = tiny(dtype, B=1, N=1, kv_len=(0,), n_cu=(0,))
    r0 = oracle.nextn_draft(w)
    g = w.weights["q_norm"]
    r1 = oracle.nextn_draft(with_weights(w, q_norm=(g * 3.0 + 0.5).astype(np.float32)))
    np.testing.assert_array_equal(r0["logits"], r1["logits"])
    np.testing.assert_array_equal(r0["h_last"], r1["h_last"])
    # the key norm changes the stored key but not this step's output either
    gk = w.weights["k_norm"]
    r2 = oracle.nextn_draft(with_weights(w, k_norm=(gk * -2.0).astype(np.float32)))
    np.testing.assert_array_equal(r0["logits"], r2["logits"])
    assert not np.array_equal(r0["k"][0, :, 0], r2["k"][0, :, 0])
    np.testing.assert_array_equal(r0["v"][0, :, 0], r2["v"][0, :, 0])
    # with 5 rows before it, the queries decide the weights
    w5 = tiny(dtype, B=1, N=1, kv_len=(5,), n_cu=(0,))
    a = oracle.nextn_draft(w5)
    b = oracle.nextn_draft(with_weights(w5, q_norm=(g * 3.0 + 0.5).astype(np.float32)))
    assert np.max(np.abs(a["h_last"] - b["h_last"])) > 1e-6


def test_zero_block_reduces_to_eh_proj_and_the_head():
    """w_o = 0 and w_down = 0: the block adds nothing, so the step's output is
    eh_proj [enorm(e); hnorm(h)] (embedding scale 1) and its logits the tied
    table against head_norm of it."""
    w = tiny("f32", B=2, N=1, kv_len=(3, 0), n_cu=(1, 0))
    w = with_weights(w, w_o=np.zeros_like(w.weights["w_o"]), w_down=np.zeros_like(w.weights["w_down"]))
    r = oracle.nextn_draft(w)
    W = w.weights
    eps = w.model.rms_eps

    def rms(x, g):
        x = x.astype(np.float64)
        return x / np.sqrt(np.mean(x * x) + eps) * g.astype(np.float64)

    for b in range(w.B):
        e = W["tok_embd"][w.last_tok[b]].astype(np.float64)
        u = np.concatenate([rms(e, W["enorm"]), rms(w.h_prev[b], W["hnorm"])])
        x = W["eh_proj"].astype(np.float64) @ u
        np.testing.assert_allclose(r["h_last"][b], x, rtol=1e-12, atol=1e-12)
        z = W["tok_embd"].astype(np.float64) @ rms(x, W["head_norm"])
        np.testing.assert_allclose(r["logits"][b, 0], z, rtol=1e-11, atol=1e-11)
        assert r["drafts"][b, 0] == int(np.argmax(z))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kv_head_permutation_changes_nothing(dtype):
    """Swap KV heads 0 and 1 together with their query groups (rows of w_qkv,
    columns of w_o) and the rows already in the KV: same drafts, logits and
    hidden state.  A query head read against the wrong KV head breaks it."""
    w = tiny(dtype, B=2, N=3, kv_len=(4, 7), n_cu=(2, 1), Hq=4, Hkv=2)
    m = w.model
    hd, Hq, Hkv, grp = m.head_dim, m.n_q_heads, m.n_kv_heads, m.n_q_heads // m.n_kv_heads
    perm_kv = np.array([1, 0])
    perm_q = np.concatenate([np.arange(perm_kv[g] * grp, perm_kv[g] * grp + grp) for g in range(Hkv)])
    rows = lambda heads, base: np.concatenate([np.arange((base + h) * hd, (base + h + 1) * hd) for h in heads])
    qkv = w.weights["w_qkv"]
    new_rows = np.concatenate([rows(perm_q, 0), rows(perm_kv, Hq), rows(perm_kv, Hq + Hkv)])
    wp = with_weights(w, w_qkv=np.ascontiguousarray(qkv[new_rows]),
                      w_o=np.ascontiguousarray(w.weights["w_o"][:, rows(perm_q, 0)]))
    dkv = dict(w.dkv, k=np.ascontiguousarray(w.dkv["k"][:, perm_kv]), v=np.ascontiguousarray(w.dkv["v"][:, perm_kv]))
    a = oracle.nextn_draft(w)
    b = oracle.nextn_draft(wp, dkv=dkv)
    np.testing.assert_array_equal(a["drafts"], b["drafts"])
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a["h_last"], b["h_last"], rtol=0, atol=1e-12)
    # and the stored rows are the same rows under the permutation
    np.testing.assert_array_equal(a["k"][:, perm_kv], b["k"])


def _replace(w, **kw):
    import copy
    w2 = copy.copy(w)
    for k, v in kw.items():
        setattr(w2, k, v)
    return w2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_call_equals_two_calls(dtype):
    """N = 3 drafts in one call, against N = 1 followed by a call that starts
    from the first call's KV (one row longer than it was plus the catch-up
    rows), its draft and its hidden state (fp32, as a caller holds it)."""
    w = tiny(dtype, B=2, N=3, kv_len=(3, 6), n_cu=(2, 0))
    one = oracle.nextn_draft(w)
    first = oracle.nextn_draft(_replace(w, N=1))
    second = oracle.nextn_draft(
        _replace(w, N=2, kv_len=(w.kv_len + w.n_cu + 1).astype(np.int32), n_cu=np.zeros(w.B, np.int32),
                 last_tok=first["drafts"][:, 0].copy(), h_prev=first["h_last"].astype(np.float32)),
        dkv=dict(w.dkv, k=first["k"], v=first["v"]))
    np.testing.assert_array_equal(one["drafts"][:, :1], first["drafts"])
    for b in range(w.B):
        rms = float(np.sqrt(np.mean(one["logits"][b, 1:] ** 2)))
        np.testing.assert_allclose(second["logits"][b], one["logits"][b, 1:], rtol=0, atol=1e-5 * rms)
        for k in range(2):
            if one["margin"][b, k + 1] > 1e-4:
                assert second["drafts"][b, k] == one["drafts"][b, k + 1]
    # the catch-up rows and the first step's row are the same in both
    for b in range(w.B):
        hi = int(w.kv_len[b] + w.n_cu[b] + 1)
        np.testing.assert_array_equal(one["k"][b, :, :hi], first["k"][b, :, :hi])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_accept_first_equals_catch_up_on_the_whole_batch(dtype):
    """The previous window drafted d1 d2 d3 and the target accepted two.
    Accept-first: catch up on (H0, d1), (H1, d2), then draft from (H2, bonus).
    Whole batch: catch up on all three rows, (H2', d3) included, then roll the
    drafter's KV back to the accepted rows and draft from (H2, bonus).  Same
    drafts and logits: the rejected row sits where the bonus row is written."""
    w = tiny(dtype, B=2, N=3, M=3, kv_len=(4, 9), n_cu=(2, 2))
    acc = oracle.nextn_draft(w)
    rej_tok = synth.uniform_int(99, "rejected", (w.B, 1), 0, w.model.vocab)
    rej_h = synth.normal(99, "rejected.h", (w.B, 1, w.model.d))
    full = _replace(w, N=1, n_cu=np.full(w.B, 3, np.int32), cu_tok=np.concatenate([w.cu_tok[:, :2], rej_tok], 1),
                    cu_h=np.concatenate([w.cu_h[:, :2], rej_h], 1))
    batch = oracle.nextn_draft(full)
    after = oracle.nextn_draft(_replace(w, kv_len=(w.kv_len + 2).astype(np.int32), n_cu=np.zeros(w.B, np.int32)),
                               dkv=dict(w.dkv, k=batch["k"], v=batch["v"]))
    np.testing.assert_array_equal(acc["drafts"], after["drafts"])
    np.testing.assert_array_equal(acc["logits"], after["logits"])
    np.testing.assert_array_equal(acc["h_last"], after["h_last"])


def test_rows_beyond_the_call_stay_unwritten_and_unread():
    """The drafter KV's unwritten slots are NaN: a read of one would make the
    logits NaN.  After the call the rows up to kv_len + n_cu + N - 1 are
    written, the rest are still NaN."""
    w = tiny("bf16", B=2, N=3, kv_len=(0, 5), n_cu=(0, 2))
    r = oracle.nextn_draft(w)
    assert np.isfinite(r["logits"]).all()
    for b in range(w.B):
        hi = int(w.kv_len[b] + w.n_cu[b] + w.N)
        k = synth.bf16_bits_to_f32(r["k"][b])
        assert np.isfinite(k[:, :hi]).all() and np.isnan(k[:, hi:]).all()


def test_rejects_out_of_range_inputs():
    w = tiny("f32", B=1, N=3, kv_len=(5,), n_cu=(2,))
    with pytest.raises(ValueError):
        oracle.nextn_draft(_replace(w, kv_len=np.array([w.dkv["cap"] - 3], np.int32)))   # no room for the rows
    with pytest.raises(ValueError):
        oracle.nextn_draft(_replace(w, n_cu=np.array([3], np.int32)))                     # above M
    with pytest.raises(ValueError):
        oracle.nextn_draft(_replace(w, last_tok=np.array([w.model.vocab], np.int32)))


def test_self_attention_closed_form_with_null_prefix():
    """Queries equal to the keys (the query rows of each head copy its KV
    head's key rows, q_norm = k_norm) and n earlier rows whose keys and values
    are zero: head h's output is e^s / (e^s + n) times the row's own value,
    s = attn_scale * |k|^2 of its own stored key (RoPE keeps the norm, and a
    query and key rotated at the same position meet at angle 0).  With the
    feed-forward zeroed the block output minus the eh_proj output is w_o times
    those head outputs."""
    n = 3
    w = tiny("f32", B=1, N=1, kv_len=(n,), n_cu=(0,), Hq=4, Hkv=2)
    m = w.model
    hd, Hq, Hkv, grp = m.head_dim, m.n_q_heads, m.n_kv_heads, m.n_q_heads // m.n_kv_heads
    qkv = w.weights["w_qkv"].copy()
    for h in range(Hq):
        g = h // grp
        qkv[h * hd:(h + 1) * hd] = qkv[(Hq + g) * hd:(Hq + g + 1) * hd]
    k0 = w.dkv["k"].copy()
    v0 = w.dkv["v"].copy()
    k0[:, :, :n] = 0.0
    v0[:, :, :n] = 0.0
    dkv = dict(w.dkv, k=k0, v=v0)
    base = dict(w_qkv=qkv, q_norm=w.weights["k_norm"].copy(), w_down=np.zeros_like(w.weights["w_down"]))
    ra = oracle.nextn_draft(with_weights(w, w_o=np.zeros_like(w.weights["w_o"]), **base), dkv=dkv)
    rb = oracle.nextn_draft(with_weights(w, **base), dkv=dkv)
    K = rb["k"][0, :, n].astype(np.float64)   # [Hkv, hd]: the row's own stored key and value
    V = rb["v"][0, :, n].astype(np.float64)
    o = np.zeros(Hq * hd)
    for h in range(Hq):
        g = h // grp
        s = m.attn_scale * float(K[g] @ K[g])
        o[h * hd:(h + 1) * hd] = math.exp(s) / (math.exp(s) + n) * V[g]
    want = w.weights["w_o"].astype(np.float64) @ o
    # the stored key is the fp32 rounding of the one the attention used
    np.testing.assert_allclose(rb["h_last"][0] - ra["h_last"][0], want, rtol=1e-5,
                               atol=1e-6 * float(np.max(np.abs(want))))


def test_stored_key_is_rotated_at_its_row_position():
    """The same (token, hidden state) stored at position 0 and at position 5:
    RoPE at position 0 is the identity, so the key at 5 is the key at 0
    rotated by 5 positions (NeoX RoPE, pinned on its own); the value is the
    same in both."""
    w0 = tiny("f32", B=1, N=1, kv_len=(0,), n_cu=(0,))
    w5 = tiny("f32", B=1, N=1, kv_len=(5,), n_cu=(0,))
    w5 = _replace(w5, last_tok=w0.last_tok, h_prev=w0.h_prev)
    r0, r5 = oracle.nextn_draft(w0), oracle.nextn_draft(w5)
    for g in range(w0.model.n_kv_heads):
        k0 = r0["k"][0, g, 0].astype(np.float64)
        np.testing.assert_allclose(r5["k"][0, g, 5], oracle.rope_neox(k0, 5, w0.dkv["rope_theta"]), rtol=1e-6,
                                   atol=1e-6)
        np.testing.assert_array_equal(r5["v"][0, g, 5], r0["v"][0, g, 0])


def test_value_rows_feed_the_stored_value_only():
    """Doubling the value rows of w_qkv doubles the stored value and leaves the
    stored key as it was (exact in fp32: a power of two); doubling the key rows
    leaves the stored value as it was."""
    w = tiny("f32", B=2, N=2, kv_len=(2, 5), n_cu=(1, 2))
    m = w.model
    hd, Hq, Hkv = m.head_dim, m.n_q_heads, m.n_kv_heads
    vrows = slice((Hq + Hkv) * hd, (Hq + 2 * Hkv) * hd)
    krows = slice(Hq * hd, (Hq + Hkv) * hd)
    r = oracle.nextn_draft(w)
    qv = w.weights["w_qkv"].copy()
    qv[vrows] *= 2
    rv = oracle.nextn_draft(with_weights(w, w_qkv=qv))
    qk = w.weights["w_qkv"].copy()
    qk[krows] *= 2
    rk = oracle.nextn_draft(with_weights(w, w_qkv=qk))
    for b in range(w.B):
        lo, hi = int(w.kv_len[b]), int(w.kv_len[b] + w.n_cu[b] + 1)   # catch-up rows and the first step's row
        np.testing.assert_array_equal(rv["v"][b, :, lo:hi], 2 * r["v"][b, :, lo:hi])
        np.testing.assert_array_equal(rv["k"][b, :, lo:hi], r["k"][b, :, lo:hi])
        np.testing.assert_array_equal(rk["v"][b, :, lo:hi], r["v"][b, :, lo:hi])


def test_feed_forward_gate_identities():
    """Attention switched off (w_o = 0).  With the gate rows negated the
    feed-forward's two outputs differ by w_down (g * u) and sum to
    w_down (g tanh(g / 2) * u), g = w_gate n, u = w_up n, n the ffn_norm of the
    eh_proj output: silu(g) - silu(-g) = g and silu(g) + silu(-g) =
    g tanh(g / 2).  (A gate and up swapped, or another activation, breaks the
    second.)"""
    w = tiny("f32", B=1, N=1, kv_len=(4,), n_cu=(0,))
    off = dict(w_o=np.zeros_like(w.weights["w_o"]))
    x = oracle.nextn_draft(with_weights(w, w_down=np.zeros_like(w.weights["w_down"]), **off))["h_last"][0]
    ya = oracle.nextn_draft(with_weights(w, **off))["h_last"][0] - x
    yb = oracle.nextn_draft(with_weights(w, w_gate=-w.weights["w_gate"], **off))["h_last"][0] - x
    W = w.weights
    n = x / np.sqrt(np.mean(x * x) + w.model.rms_eps) * W["ffn_norm"].astype(np.float64)
    g = W["w_gate"].astype(np.float64) @ n
    u = W["w_up"].astype(np.float64) @ n
    Wd = W["w_down"].astype(np.float64)
    scale = float(np.max(np.abs(ya))) + 1e-30
    np.testing.assert_allclose(ya - yb, Wd @ (g * u), rtol=0, atol=1e-10 * scale)
    np.testing.assert_allclose(ya + yb, Wd @ (g * np.tanh(g / 2) * u), rtol=0, atol=1e-10 * scale)
