"""Pins of the oracle's draft step and draft chain (no GPU).

The step is checked against a composition of torch library routines
(F.rms_norm, F.linear, F.scaled_dot_product_attention, F.gelu) wired in the
order the Gemma-4 MTP page gives (sec. 4 "Per-step MTP graph": embed from the
target's table scaled by sqrt(n_embd), concat with h_prev and pre-project, then
per block RMSNorm -> Q proj -> Q-norm -> RoPE -> cross-attention into the
target KV -> residual + post-norm -> GELU FFN + post-FFN norm; final RMSNorm ->
post-projection -> tied LM head -> optional softcap), with the NextN input
norms of the embedding and hidden state ("MTP decoding", Requirements).  The
chain is checked by invariants: greedy picks are the argmax of the step's
logits, the step after consumes the previous pick, sequences are independent,
and the fused steps only read the frozen KV prefix.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth


def tiny_workload(dtype="f32", B=2, N=3, softcap=0.0, seed=11, kv=(37, 23)):
    m = synth.ModelSpec(d_t=48, d_a=32, n_blocks=2, n_q_heads=4, head_dim=8, n_kv_heads=2,
                        d_ff=40, vocab=97, dtype=dtype, block_view=(0, 1), logit_softcap=softcap)
    views = [synth.ViewSpec(cap=12, window=9, rope_theta=1e4),
             synth.ViewSpec(cap=40, window=0, rope_theta=1e6)]
    return synth.make_draft_workload("tiny-test", m, views, B, N, list(kv)[:B], seed, hist_len=8)


def _t(a, dtype):
    if dtype == "bf16" and a.dtype == np.uint16:
        a = synth.bf16_bits_to_f32(a)
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def torch_step(w, b, step, tok, h):
    """The step composed from torch library routines (fp64)."""
    m = w.model
    W = {k: _t(v, m.dtype) for k, v in w.weights.items()}
    eps = m.rms_eps
    e = W["tok_embd"][tok] * math.sqrt(m.d_t)
    u = torch.cat([F.rms_norm(e, (m.d_t,), W["norm_e"], eps),
                   F.rms_norm(torch.as_tensor(h, dtype=torch.float64), (m.d_t,), W["norm_h"], eps)])
    x = F.linear(u, W["w_pre"])
    grp = m.n_q_heads // m.n_kv_heads
    for l in range(m.n_blocks):
        p = f"blk{l}."
        vd = w.views[m.block_view[l]]
        q = F.linear(F.rms_norm(x, (m.d_a,), W[p + "attn_norm"], eps), W[p + "w_q"]).view(m.n_q_heads, m.head_dim)
        q = F.rms_norm(q, (m.head_dim,), W[p + "q_norm"], eps)
        half = m.head_dim // 2
        pos = int(w.kv_len[b]) + step
        ang = pos * vd["rope_theta"] ** (-2.0 * torch.arange(half, dtype=torch.float64) / m.head_dim)
        zc = torch.complex(q[:, :half], q[:, half:]) * torch.polar(torch.ones_like(ang), ang)
        q = torch.cat([zc.real, zc.imag], dim=1)
        kv_len = int(w.kv_len[b])
        lo = max(0, kv_len - vd["window"]) if vd["window"] else 0
        slots = torch.arange(lo, kv_len) % vd["cap"]
        K = _t(vd["k"][b], m.dtype)[:, slots, :].repeat_interleave(grp, dim=0)
        V = _t(vd["v"][b], m.dtype)[:, slots, :].repeat_interleave(grp, dim=0)
        o = F.scaled_dot_product_attention(q[:, None, :], K, V)[:, 0, :].reshape(-1)
        x = x + F.rms_norm(F.linear(o, W[p + "w_o"]), (m.d_a,), W[p + "post_attn_norm"], eps)
        n = F.rms_norm(x, (m.d_a,), W[p + "pre_ffn_norm"], eps)
        mm = F.gelu(F.linear(n, W[p + "w_gate"]), approximate="tanh") * F.linear(n, W[p + "w_up"])
        x = x + F.rms_norm(F.linear(mm, W[p + "w_down"]), (m.d_a,), W[p + "post_ffn_norm"], eps)
    hn = F.linear(F.rms_norm(x, (m.d_a,), W["final_norm"], eps), W["w_post"])
    z = F.linear(hn, W["tok_embd"])
    if m.logit_softcap > 0:
        z = m.logit_softcap * torch.tanh(z / m.logit_softcap)
    return hn.numpy(), z.numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("softcap", [0.0, 7.5])
def test_step_matches_library_composition(dtype, softcap):
    w = tiny_workload(dtype, softcap=softcap)
    for b in range(w.B):
        for step in (0, 2):
            tok = int(w.last_tok[b]) if step == 0 else 5
            h = w.h_prev[b].astype(np.float64)
            hn, z = oracle.draft_step(w, b, step, tok, h)
            rh, rz = torch_step(w, b, step, tok, h)
            assert np.allclose(hn, rh, rtol=1e-10, atol=1e-10)
            assert np.allclose(z, rz, rtol=1e-10, atol=1e-10)


def test_step_output_is_finite_despite_poisoned_kv():
    w = tiny_workload("bf16")
    hn, z = oracle.draft_step(w, 1, 0, 3, w.h_prev[1])
    assert np.all(np.isfinite(hn)) and np.all(np.isfinite(z))


def test_block_greedy_chain_invariants():
    w = tiny_workload("f32", B=2, N=4)
    r = oracle.draft_block(w)
    for b in range(w.B):
        h = w.h_prev[b].astype(np.float64)
        tok = int(w.last_tok[b])
        for k in range(w.N):
            hn, z = oracle.draft_step(w, b, k, tok, h)
            assert np.array_equal(z, r["logits"][b, k])
            assert r["drafts"][b, k] == int(np.argmax(z))
            srt = np.sort(z)
            assert abs(r["margin"][b, k] - (srt[-1] - srt[-2])) < 1e-12
            tok, h = int(r["drafts"][b, k]), hn
        assert np.array_equal(h, r["h_last"][b])


def test_block_sequences_are_independent():
    w = tiny_workload("bf16", B=2, N=3)
    both = oracle.draft_block(w)
    one = oracle.draft_block(w, seqs=[1])
    assert np.array_equal(both["drafts"][1], one["drafts"][0])
    assert np.array_equal(both["logits"][1], one["logits"][0])


def test_block_teacher_forcing():
    w = tiny_workload("f32", B=1, N=3)
    force = np.array([[7, 8, 9]], dtype=np.int32)
    r = oracle.draft_block(w, force=force)
    h = w.h_prev[0].astype(np.float64)
    tok = int(w.last_tok[0])
    for k in range(3):
        hn, z = oracle.draft_step(w, 0, k, tok, h)
        assert np.array_equal(z, r["logits"][0, k])
        tok, h = int(force[0, k]), hn


def test_frozen_prefix_only():
    """Changing KV outside every view's readable range changes nothing; changing a
    readable slot changes the logits (the chain reads the prefix, never drafts)."""
    w = tiny_workload("f32", B=1, N=2, kv=(30,))
    base = oracle.draft_block(w)
    vd = w.views[1]
    vd["k"][0, :, 35, :] = 1e3   # beyond kv_len in the full view (never read)
    vd["v"][0, :, 35, :] = -1e3
    same = oracle.draft_block(w)
    assert np.array_equal(base["logits"], same["logits"])
    vd["k"][0, :, 29, :] += 1.0  # newest readable position
    diff = oracle.draft_block(w)
    assert not np.array_equal(base["logits"], diff["logits"])


def test_step_position_is_kv_len_plus_step():
    """Step k's query RoPE position is kv_len + k: the same token and hidden state
    at two steps give different logits, each equal to the library composition at
    its own position."""
    w = tiny_workload("f32", B=1, N=2)
    h = w.h_prev[0].astype(np.float64)
    _, z0 = oracle.draft_step(w, 0, 0, 3, h)
    _, z1 = oracle.draft_step(w, 0, 1, 3, h)
    assert not np.allclose(z0, z1)
    for step, z in ((0, z0), (1, z1)):
        _, rz = torch_step(w, 0, step, 3, h)
        assert np.allclose(z, rz, rtol=1e-10, atol=1e-10)


# ----------------------------------------------------------------------------
# the per-step confidence ("MTP decoding (--mtp)", "Stopping early when the
# head is unsure"): the top-1 softmax probability of the step's logits
# ----------------------------------------------------------------------------

def test_top1_prob_closed_forms():
    import math
    assert abs(oracle.top1_prob(np.zeros(4096)) - 1.0 / 4096) < 1e-15
    a, n = 3.0, 1000
    z = np.zeros(n)
    z[17] = a
    assert abs(oracle.top1_prob(z) - math.exp(a) / (math.exp(a) + n - 1)) < 1e-15
    assert abs(oracle.top1_prob(np.array([2.0, 2.0, -np.inf])) - 0.5) < 1e-15
    assert abs(oracle.top1_prob(np.array([1.0, np.nan, 1.0])) - 0.5) < 1e-15


def test_top1_prob_is_softmax_max():
    from scipy.special import softmax
    rng = np.random.default_rng(4)
    for scale in (0.1, 1.0, 5.0):
        z = scale * rng.standard_normal(3001)
        assert abs(oracle.top1_prob(z) - softmax(z).max()) < 1e-12


def test_draft_block_confidence_matches_its_logits():
    w = synth.make_draft_inputs(0)
    ref = oracle.draft_block(w)
    for k in range(w.N):
        assert ref["conf"][0, k] == oracle.top1_prob(ref["logits"][0, k])
        assert 1.0 / w.model.vocab <= ref["conf"][0, k] <= 1.0
