"""GPU parity of the centroid-routed LM head inside mtp_draft_block ("Gemma 4
MTP -- Multi-Token Prediction speculative decoding", sec. 3 "Centroid /
ordered-embeddings LM head").

Rules, per step:
  * structure (exact): the row holds -1e30 (fp32) everywhere but on exactly
    top_k whole candidate lists of token_ordering;
  * the draft is the argmax of the step's own row (lowest index on ties);
  * against the oracle chain (teacher-forced with the GPU's tokens): the
    logits on the candidates both rows hold match within the dtype tolerance
    (1e-3 fp32, 2e-2 bf16, relative to the rms of the oracle's candidate
    logits); where the oracle's set margin (the top_k-th minus the next
    centroid logit, over their standard deviation) exceeds 0.2 the sets are
    equal, and where the token margin exceeds 1e-2 of the candidates'
    standard deviation as well, so are the drafts;
  * the last step's head against the oracle's head on the GPU's own h (the
    h_last output is that step's head input): equal sets where the set
    margin exceeds 1e-3, candidate logits within 1e-4 (fp32 accumulation of
    the same products), the draft equal where its margin exceeds 1e-4.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import run_gpu_draft, tol_for

pytestmark = pytest.mark.gpu

FILL32 = np.float32(-1e30)
SP = synth.SampleParams()


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mtp_speculative_decoding_gb300 import build
    build.build()


def tiny_centroid(B=2, N=3, nc=64, kc=8, softcap=30.0, dtype="f32", seed=21):
    m = synth.ModelSpec(d_t=256, d_a=128, n_blocks=1, n_q_heads=4, head_dim=32, n_kv_heads=1, d_ff=512,
                        vocab=4096, dtype=dtype, block_view=(0,), logit_softcap=softcap, n_centroids=nc,
                        centroid_top_k=kc)
    views = [synth.ViewSpec(cap=128, window=0, rope_theta=1e6)]
    kv = np.random.default_rng(seed).integers(1, 129, size=B)
    return synth.make_draft_workload("tiny-centroid", m, views, B, N, kv, seed, hist_len=8)


def _lists(w):
    m = w.model
    return w.weights["token_ordering"].reshape(m.n_centroids, m.vocab // m.n_centroids)


def check_structure(w, zg, draft):
    m = w.model
    lists = _lists(w)
    cand = zg > -1e29
    assert np.all(zg[~cand] == FILL32)
    assert int(cand.sum()) == m.centroid_top_k * lists.shape[1]
    assert int(cand[lists].all(axis=1).sum()) == m.centroid_top_k   # whole lists
    assert np.all(np.isfinite(zg[cand]))
    assert draft == int(np.argmax(zg))
    return cand


def check_centroid_parity(w, g_drafts, g_h, g_logits, seqs):
    m = w.model
    tol = tol_for(w)
    ref = oracle.draft_block(w, seqs=seqs, force=g_drafts)
    stable = 0
    for j, b in enumerate(seqs):
        for k in range(w.N):
            zg, zo = g_logits[b, k], ref["logits"][j, k]
            cg = check_structure(w, zg, int(g_drafts[b, k]))
            co = zo > -1e29
            vals = zo[co]
            rms = float(np.sqrt(np.mean(vals * vals)))
            both = cg & co
            assert both.any()
            err = float(np.max(np.abs(zg[both] - zo[both])))
            assert err <= tol * rms, f"b={b} k={k}: max|dz| {err:.3g} > {tol} * {rms:.3g}"
            if ref["cgap"][j, k] > 0.2:
                stable += 1
                assert np.array_equal(cg, co), f"b={b} k={k}: candidate sets differ (gap {ref['cgap'][j, k]:.3g})"
                srt = np.sort(vals)
                if srt[-1] - srt[-2] > 1e-2 * np.std(vals):
                    assert g_drafts[b, k] == int(np.argmax(zo))
        ho = ref["h_last"][j]
        assert np.max(np.abs(g_h[b] - ho)) <= tol * float(np.sqrt(np.mean(ho * ho)))
        # the last step's head on the GPU's own input
        zl, gap, _ = oracle.centroid_head(m, w.weights["centroids"], w.weights["token_ordering"],
                                          w.weights["tok_embd"], g_h[b].astype(np.float64), full=True)
        zg = g_logits[b, w.N - 1]
        if gap > 1e-3:
            cand = zl > -1e29
            assert np.array_equal(zg > -1e29, cand), f"b={b}: last-step sets differ (gap {gap:.3g})"
            v = zl[cand]
            assert float(np.max(np.abs(zg[cand] - v))) <= 1e-4 * float(np.sqrt(np.mean(v * v)))
            srt = np.sort(v)
            if srt[-1] - srt[-2] > 1e-4 * np.std(v):
                assert g_drafts[b, w.N - 1] == int(np.argmax(zl))
    return stable


@pytest.mark.parametrize("dtype,softcap", [("f32", 30.0), ("f32", 0.0), ("bf16", 30.0)])
def test_tiny_centroid_parity(dtype, softcap):
    w = tiny_centroid(B=3, dtype=dtype, softcap=softcap)
    _, d, h, z = run_gpu_draft(w)
    check_centroid_parity(w, d, h, z, range(w.B))


def test_tiny_single_sequence_and_odd_sizes():
    # one sequence (every CTA serves it), 48 lists of 64 (a non-power-of-two
    # sort), top_k 5
    m = synth.ModelSpec(d_t=256, d_a=128, n_blocks=1, n_q_heads=4, head_dim=32, n_kv_heads=1, d_ff=512,
                        vocab=3072, dtype="f32", block_view=(0,), n_centroids=48, centroid_top_k=5)
    views = [synth.ViewSpec(cap=64, window=0, rope_theta=1e6)]
    w = synth.make_draft_workload("tiny-centroid-1", m, views, 1, 4, [50], 4, hist_len=4)
    _, d, h, z = run_gpu_draft(w)
    check_centroid_parity(w, d, h, z, [0])


def test_all_centroids_equals_dense_head_on_gpu():
    """top_k = n_centroids: every token is a candidate, and the GPU's row is
    the GPU's dense-head row up to fp32 summation order."""
    wc = tiny_centroid(B=2, nc=32, kc=32, seed=8)
    md = synth.ModelSpec(**{**wc.model.__dict__, "n_centroids": 0, "centroid_top_k": 0})
    wd = synth.make_draft_workload("tiny-dense", md, wc.views_spec, wc.B, wc.N, wc.kv_len, 8, hist_len=8)
    _, dc, hc, zc = run_gpu_draft(wc)
    _, dd, hd, zd = run_gpu_draft(wd)
    assert np.all(zc > -1e29)
    np.testing.assert_allclose(zc, zd, rtol=2e-5, atol=2e-5 * float(np.sqrt(np.mean(zd * zd))))
    np.testing.assert_array_equal(dc, dd)


def test_many_sequences_share_the_grid():
    # B = 20: groups of CTAs per sequence, bf16 weights (CUDA-core variant)
    w = tiny_centroid(B=20, N=2, dtype="bf16", seed=3)
    _, d, h, z = run_gpu_draft(w)
    check_centroid_parity(w, d, h, z, [0, 7, 13, 19])


def test_timed_path_without_logits_matches():
    w = tiny_centroid(B=3, seed=9)
    dev, d1, h1, z1 = run_gpu_draft(w)
    _, d2, h2, _ = run_gpu_draft(w, want_logits=False, dev=dev)
    np.testing.assert_array_equal(d1, d2)
    np.testing.assert_array_equal(h1, h2)


def test_confidence_over_candidates():
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import upload_draft
    w = tiny_centroid(B=3, seed=12)
    dev = upload_draft(w)
    B, N, V = w.B, w.N, w.model.vocab
    drafts = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    conf = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    logits = torch.full((B, N, V), float("nan"), dtype=torch.float32, device="cuda")
    dev.run(drafts, out_logits=logits, out_conf=conf)
    torch.cuda.synchronize()
    assert mtp.last_error(dev.ws) == 0
    d, c, z = drafts.cpu().numpy(), conf.cpu().numpy(), logits.cpu().numpy()
    ref = oracle.draft_block(w, force=d, want_logits=False)
    for b in range(B):
        for k in range(N):
            own = oracle.top1_prob(z[b, k].astype(np.float64))   # -1e30 entries add nothing
            assert abs(c[b, k] - own) <= 1e-4 * own
            assert abs(c[b, k] - ref["conf"][b, k]) <= 1e-3 * ref["conf"][b, k]


def test_sampled_drafts_stay_in_the_candidates():
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import upload_draft
    w = tiny_centroid(B=3, seed=14, softcap=0.0)
    dev = upload_draft(w)
    B, N, V = w.B, w.N, w.model.vocab
    drafts = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    logits = torch.full((B, N, V), float("nan"), dtype=torch.float32, device="cuda")
    sp = (SP.temp, SP.top_p, SP.min_p, SP.rep_penalty, SP.presence_penalty, SP.top_k)
    dev.run(drafts, out_logits=logits, sample=sp, seed=77, offset=2)
    torch.cuda.synchronize()
    assert mtp.last_error(dev.ws) == 0
    d, z = drafts.cpu().numpy(), logits.cpu().numpy()
    ref = oracle.draft_block(w, sample=SP, seed=77, offset=2, force=d)
    same = 0
    for b in range(B):
        for k in range(N):
            assert z[b, k, d[b, k]] > -1e29   # a draw from the candidates
            cg = z[b, k] > -1e29
            zo = ref["logits"][b, k]
            both = cg & (zo > -1e29)
            vals = zo[zo > -1e29]
            assert float(np.max(np.abs(z[b, k][both] - zo[both]))) <= 1e-3 * float(np.sqrt(np.mean(vals * vals)))
            if d[b, k] == ref["drafts"][b, k]:
                same += 1
            else:
                assert ref["margin"][b, k] < 1e-3 or ref["cgap"][b, k] < 0.2
    assert same >= B * N - max(1, (B * N) // 10)


def test_out_of_range_ordering_sets_status():
    """An ordering entry outside [0, vocab) is skipped with MTP_ERR_ARG in the
    status word (host-checked bounds: the kernel never dereferences it)."""
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import upload_draft
    w = tiny_centroid(B=1, nc=4, kc=4, seed=2)   # every list is scored
    w.weights = dict(w.weights)
    bad = w.weights["token_ordering"].copy()
    bad[17] = w.model.vocab + 5
    w.weights["token_ordering"] = bad
    dev = upload_draft(w)
    drafts = torch.full((1, w.N), -7, dtype=torch.int32, device="cuda")
    dev.run(drafts)
    torch.cuda.synchronize()
    assert mtp.last_error(dev.ws) == mtp.MTP_ERR_ARG


@pytest.mark.slow
def test_edge_workload():
    w = synth.make_draft_inputs(5)
    _, d, h, z = run_gpu_draft(w)
    check_centroid_parity(w, d, h, z, [0])


@pytest.mark.slow
def test_edge_workload_batch4_without_logits():
    w = synth.make_draft_inputs(5, B=4)
    dev, d, h, z = run_gpu_draft(w)
    check_centroid_parity(w, d, h, z, range(4))
    _, d2, h2, _ = run_gpu_draft(w, want_logits=False, dev=dev)
    np.testing.assert_array_equal(d, d2)
