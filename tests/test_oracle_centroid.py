"""Pins of the oracle's centroid-routed LM head (no GPU).

"Gemma 4 MTP -- Multi-Token Prediction speculative decoding", sec. 3
"Centroid / ordered-embeddings LM head": centroid logits C h, the top_k
centroids, their lists of vocab / n_centroids candidate ids out of
token_ordering, the candidates' logits E[t] h, scattered into a row that is
-1e30 everywhere else.  Pinned by a hand-worked tiny case whose two readings
of the ordering layout give different rows, the tie rule, the special case
top_k = n_centroids (every token a candidate: the dense head, checked against
numpy's matmul), and the draft chain with that special case equal to the
dense-head model's chain.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth

FILL = -1e30


@dataclasses.dataclass
class _M:
    d_t: int
    vocab: int
    n_centroids: int
    centroid_top_k: int
    dtype: str = "f32"
    logit_softcap: float = 0.0
    d_a: int = 1
    n_blocks: int = 0
    n_q_heads: int = 1
    head_dim: int = 1
    n_kv_heads: int = 1
    d_ff: int = 1
    rms_eps: float = 1e-6
    attn_scale: float = 1.0
    emb_scale: float = 1.0


def _tiny():
    # V = 8 tokens, 2 centroids, lists of 4; E[t] = (t, 1), centroid j = unit vector j
    E = np.array([[t, 1.0] for t in range(8)], dtype=np.float32)
    C = np.eye(2, dtype=np.float32)
    order = np.array([3, 0, 6, 5, 1, 7, 2, 4], dtype=np.int32)
    return E, C, order


def test_hand_case_lists_are_contiguous():
    """h = (0.25, 0.5): centroid 1 wins; its list is order[4:8] = {1, 7, 2, 4}, each
    with logit 0.25 t + 0.5.  (Reading the view with n_centroids as the
    contiguous dimension would pick {0, 5, 7, 4} instead.)"""
    E, C, order = _tiny()
    z = oracle.centroid_head(_M(d_t=2, vocab=8, n_centroids=2, centroid_top_k=1), C, order, E,
                             np.array([0.25, 0.5]))
    want = np.full(8, FILL)
    for t in (1, 7, 2, 4):
        want[t] = 0.25 * t + 0.5
    np.testing.assert_array_equal(z, want)
    assert int(np.argmax(z)) == 7


def test_hand_case_tie_takes_lower_centroid():
    E, C, order = _tiny()
    z = oracle.centroid_head(_M(d_t=2, vocab=8, n_centroids=2, centroid_top_k=1), C, order, E,
                             np.array([0.5, 0.5]))
    want = np.full(8, FILL)
    for t in (3, 0, 6, 5):
        want[t] = 0.5 * t + 0.5
    np.testing.assert_array_equal(z, want)


def test_hand_case_softcap_applies_to_candidates_only():
    E, C, order = _tiny()
    cap = 1.5
    z = oracle.centroid_head(_M(d_t=2, vocab=8, n_centroids=2, centroid_top_k=1, logit_softcap=cap), C,
                             order, E, np.array([0.25, 0.5]))
    for t in range(8):
        if t in (1, 7, 2, 4):
            assert z[t] == pytest.approx(cap * np.tanh((0.25 * t + 0.5) / cap), rel=1e-15)
        else:
            assert z[t] == FILL


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_all_centroids_is_the_dense_head(dtype, softcap):
    """top_k = n_centroids with a permutation ordering: every token is a
    candidate and the row is the dense tied head's, E h (softcapped)."""
    V, d, nc = 512, 64, 16
    m = _M(d_t=d, vocab=V, n_centroids=nc, centroid_top_k=nc, dtype=dtype, logit_softcap=softcap)
    E32 = synth.normal(5, "E", (V, d))
    C32 = synth.normal(5, "C", (nc, d))
    order = synth.permutation(5, "order", V)
    h = synth.normal(5, "h", (d,)).astype(np.float64)
    E = synth.f32_to_bf16_bits(E32) if dtype == "bf16" else E32
    C = synth.f32_to_bf16_bits(C32) if dtype == "bf16" else C32
    z, gap, _ = oracle.centroid_head(m, C, order, E, h, full=True)
    assert gap == np.inf
    Ew = synth.bf16_bits_to_f32(E).astype(np.float64) if dtype == "bf16" else E32.astype(np.float64)
    dense = Ew @ h
    if softcap:
        dense = softcap * np.tanh(dense / softcap)
    np.testing.assert_allclose(z, dense, rtol=1e-12, atol=1e-12)


def test_candidate_set_is_the_top_centroids_lists():
    """Exactly top_k * vsc finite entries: the lists of the top_k centroids by
    C h (brute force: sorted by value desc, id asc)."""
    V, d, nc, kc = 1024, 32, 64, 5
    m = _M(d_t=d, vocab=V, n_centroids=nc, centroid_top_k=kc)
    E = synth.normal(6, "E", (V, d))
    C = synth.normal(6, "C", (nc, d))
    order = synth.permutation(6, "order", V)
    h = synth.normal(6, "h", (d,)).astype(np.float64)
    z, gap, clo = oracle.centroid_head(m, C, order, E, h, full=True)
    cl = C.astype(np.float64) @ h
    np.testing.assert_allclose(clo, cl, rtol=1e-12, atol=1e-12)
    top = sorted(range(nc), key=lambda j: (-cl[j], j))[:kc]
    srt = np.sort(cl)[::-1]
    assert gap == pytest.approx((srt[kc - 1] - srt[kc]) / np.std(cl), rel=1e-9)
    vsc = V // nc
    cand = set(int(t) for j in top for t in order[j * vsc:(j + 1) * vsc])
    assert set(np.flatnonzero(z > FILL).tolist()) == cand
    assert len(cand) == kc * vsc
    for t in cand:
        assert z[t] == pytest.approx(float(E[t].astype(np.float64) @ h), rel=1e-12, abs=1e-12)


def test_rejects_bad_sizes():
    E, C, order = _tiny()
    with pytest.raises(ValueError):
        oracle.centroid_head(_M(d_t=2, vocab=8, n_centroids=3, centroid_top_k=1), C, order, E, np.zeros(2))
    with pytest.raises(ValueError):
        oracle.centroid_head(_M(d_t=2, vocab=8, n_centroids=2, centroid_top_k=3), C, order, E, np.zeros(2))
    bad = order.copy()
    bad[5] = 8
    with pytest.raises(ValueError):
        oracle.centroid_head(_M(d_t=2, vocab=8, n_centroids=2, centroid_top_k=2), C, bad, E, np.zeros(2))


def _chain_workload(nc, kc, softcap=0.0):
    m = synth.ModelSpec(d_t=48, d_a=32, n_blocks=2, n_q_heads=4, head_dim=8, n_kv_heads=2, d_ff=40, vocab=96,
                        dtype="f32", block_view=(0, 1), logit_softcap=softcap, n_centroids=nc, centroid_top_k=kc)
    views = [synth.ViewSpec(cap=12, window=9, rope_theta=1e4), synth.ViewSpec(cap=40, window=0, rope_theta=1e6)]
    return synth.make_draft_workload("tiny-centroid", m, views, 2, 3, [37, 23], 11, hist_len=8)


def test_draft_chain_all_centroids_equals_dense_chain():
    wc = _chain_workload(12, 12, softcap=20.0)
    wd = _chain_workload(0, 0, softcap=20.0)
    for n in wd.weights:   # same tensors apart from the centroid head's own
        np.testing.assert_array_equal(wd.weights[n], wc.weights[n])
    rc, rd = oracle.draft_block(wc), oracle.draft_block(wd)
    np.testing.assert_array_equal(rc["drafts"], rd["drafts"])
    np.testing.assert_array_equal(rc["logits"], rd["logits"])
    np.testing.assert_array_equal(rc["h_last"], rd["h_last"])


def test_draft_chain_picks_a_candidate():
    w = _chain_workload(12, 3)
    r = oracle.draft_block(w)
    z = r["logits"]
    assert np.all((z > FILL).sum(axis=2) == 3 * 8)
    for b in range(w.B):
        for k in range(w.N):
            assert z[b, k, r["drafts"][b, k]] > FILL
            assert r["drafts"][b, k] == int(np.argmax(z[b, k]))
