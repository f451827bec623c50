"""Pins of the oracle's verify-accept step (no GPU).

Greedy verify ("MTP decoding", How it is wired): planted accept lengths are
recovered exactly, and greedy speculative decoding reproduces plain argmax
decoding for every draft width and every drafter on a toy language model.

Exact sampling ("opus-mtp-turbo: Track 1 report", item 4): sample_dist is
checked on hand-computed closed forms; the verifier is checked by its
reductions (min-p = 1 gives greedy verify, q = p accepts everything, a unit
penalty ignores the history) and by the Monte Carlo total-variation test the
page describes, including the greedy-match negative control.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------------------
# greedy verify
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seed", range(6))
def test_planted_accept_length_recovered(dtype, seed):
    inp = synth.make_verify_greedy_inputs(0, seed=seed, B=8, N=4, V=1000, dtype=dtype)
    out, n_acc = oracle.verify_greedy(inp.logits, inp.dtype, inp.drafts)
    assert np.array_equal(n_acc, inp.planted)
    vals = synth.bf16_bits_to_f32(inp.logits) if dtype == "bf16" else inp.logits
    for b in range(8):
        k = int(inp.planted[b])
        assert np.array_equal(out[b, :k], inp.drafts[b, :k])
        assert out[b, k] == int(np.argmax(vals[b, k]))
        assert np.all(out[b, k + 1:] == -1)


def test_verify_greedy_ties_and_nan_rows():
    V = 8
    logits = np.zeros((1, 3, V), dtype=np.float32)
    logits[0, 0, [2, 5]] = 3.0          # tie: lowest index (2) is the argmax
    logits[0, 1, :] = np.nan
    logits[0, 1, 6] = 1.0               # NaN never wins
    drafts = np.array([[2, 6]], dtype=np.int32)
    out, n = oracle.verify_greedy(logits, "f32", drafts)
    assert n[0] == 2 and list(out[0]) == [2, 6, 0]
    drafts = np.array([[5, 6]], dtype=np.int32)
    out, n = oracle.verify_greedy(logits, "f32", drafts)
    assert n[0] == 0 and list(out[0]) == [2, -1, -1]


class ToyLM:
    """Deterministic toy target: logits depend on the last two tokens."""

    def __init__(self, V, seed):
        rng = np.random.default_rng(seed)
        self.V = V
        self.t1 = rng.standard_normal((V, V)).astype(np.float32)
        self.t2 = rng.standard_normal((V, V)).astype(np.float32)

    def logits(self, ctx):
        return (self.t1[ctx[-1]] + 0.5 * self.t2[ctx[-2]]).astype(np.float32)


@pytest.mark.parametrize("N", [1, 2, 3, 4])
@pytest.mark.parametrize("drafter", ["perfect", "random", "adversarial", "mixed"])
def test_greedy_speculation_equals_plain_greedy(N, drafter):
    lm = ToyLM(11, 3)
    rng = np.random.default_rng(N)
    T = 20
    plain = [4, 7]
    while len(plain) < 2 + T:
        plain.append(int(np.argmax(lm.logits(plain))))
    ctx = [4, 7]
    rounds = 0
    while len(ctx) < 2 + T:
        d, c = [], list(ctx)
        for i in range(N):
            g = int(np.argmax(lm.logits(c)))
            if drafter == "perfect":
                x = g
            elif drafter == "random":
                x = int(rng.integers(0, 11))
            elif drafter == "adversarial":
                x = (g + 1) % 11
            else:
                x = g if rng.random() < 0.6 else int(rng.integers(0, 11))
            d.append(x)
            c.append(x)
        rows = np.stack([lm.logits(ctx + d[:i]) for i in range(N + 1)])[None]
        out, n = oracle.verify_greedy(rows, "f32", np.array([d], dtype=np.int32))
        ctx += [int(t) for t in out[0, :n[0] + 1]]
        rounds += 1
    assert ctx[:2 + T] == plain
    if drafter == "perfect":
        assert rounds <= math.ceil(T / (N + 1))


# ----------------------------------------------------------------------------
# sample_dist closed forms
# ----------------------------------------------------------------------------

def P(**kw):
    base = dict(temp=1.0, top_p=1.0, min_p=0.0, rep_penalty=1.0, presence_penalty=0.0, top_k=0)
    base.update(kw)
    return synth.SampleParams(**base)


def probs(z, pen=(), **kw):
    ids, w, ws, _ = oracle.sample_dist(np.asarray(z, dtype=np.float64), list(pen), P(**kw))
    return list(ids), list(np.asarray(w) / ws)


def test_sample_dist_softmax_min_p_top_p():
    z = [2.0, 1.0, 0.0, -1.0]
    ids, p = probs(z)
    e = np.exp(np.array(z) - 2.0)
    assert ids == [0, 1, 2, 3] and np.allclose(p, e / e.sum(), rtol=2e-6)
    # min-p 0.2 keeps p >= 0.2 p_max: e^-1 = 0.368 stays, e^-2 = 0.135 goes
    ids, p = probs(z, min_p=0.2)
    assert ids == [0, 1] and np.allclose(p, [1 / (1 + math.e ** -1), math.e ** -1 / (1 + math.e ** -1)], rtol=2e-6)
    # top-p keeps the shortest prefix whose mass reaches top_p (0.731 >= 0.7)
    assert probs(z, min_p=0.2, top_p=0.7)[0] == [0]
    assert probs(z, min_p=0.2, top_p=0.75)[0] == [0, 1]
    # temperature 0.5 doubles every logit gap
    ids, p = probs(z, temp=0.5)
    e2 = np.exp(2 * (np.array(z) - 2.0))
    assert np.allclose(p, e2 / e2.sum(), rtol=2e-6)


def test_sample_dist_penalties():
    # repetition: positive logits divided by r, negative multiplied; presence subtracted;
    # each distinct token once, out-of-range ids ignored
    z = [2.0, -1.0, 0.5, 0.1]
    ids, p = probs(z, pen=[0, 1, 1, 1, -1, 99], rep_penalty=2.0, presence_penalty=0.1)
    l = np.array([2.0 / 2 - 0.1, -1.0 * 2 - 0.1, 0.5, 0.1])
    e = np.exp(l - l.max())
    order = [0, 2, 3, 1]
    assert ids == order and np.allclose(p, e[order] / e.sum(), rtol=2e-6)
    # a unit penalty is a no-op
    assert probs(z, pen=[0, 1], rep_penalty=1.0) == probs(z)


def test_sample_dist_top_k_and_ties():
    z = [3.0, 5.0, 5.0, 1.0]
    assert probs(z, top_k=2)[0] == [1, 2]
    assert probs(z, top_k=1)[0] == [1]
    ids, p = probs(z, top_k=3)
    assert ids == [1, 2, 0]


def test_pick_inverse_cdf():
    ids, w = [7, 3, 9], [0.5, 0.3, 0.2]
    assert oracle.pick(ids, w, 1.0, 0.0)[0] == 7
    assert oracle.pick(ids, w, 1.0, 0.49)[0] == 7
    assert oracle.pick(ids, w, 1.0, 0.5)[0] == 3
    assert oracle.pick(ids, w, 1.0, 0.99)[0] == 9


# ----------------------------------------------------------------------------
# exact sampling verify: reductions
# ----------------------------------------------------------------------------

def _cont_inputs(B, N, V, seed):
    rng = np.random.default_rng(seed)
    tgt = (2 * rng.standard_normal((B, N + 1, V))).astype(np.float32)
    dft = (0.8 * tgt[:, :N] + 0.6 * 2 * rng.standard_normal((B, N, V))).astype(np.float32)
    drafts = np.argmax(dft, axis=2).astype(np.int32)
    drafts[::3, 0] = rng.integers(0, V, size=drafts[::3, 0].shape)
    hist = rng.integers(0, V, size=(B, 16)).astype(np.int32)
    return tgt, dft, drafts, hist


def test_min_p_one_reduces_to_greedy():
    tgt, dft, drafts, hist = _cont_inputs(64, 3, 300, 0)
    sp = P(min_p=1.0, temp=0.7)
    out, n, _ = oracle.verify_sample(tgt, dft, "f32", drafts, hist, sp, 5, 0)
    g_out, g_n = oracle.verify_greedy(tgt, "f32", drafts)
    assert np.array_equal(n, g_n) and np.array_equal(out, g_out)


def test_identical_draft_distribution_accepts_everything():
    tgt, _, drafts, hist = _cont_inputs(64, 3, 300, 1)
    sp = P(temp=0.6, top_p=0.95, min_p=0.05, rep_penalty=1.08)
    dft = np.ascontiguousarray(tgt[:, :3])
    # drafts inside q's support: the row argmax after the same penalties
    for b in range(64):
        pen = list(hist[b])
        for i in range(3):
            ids, _, _, _ = oracle.sample_dist(dft[b, i].astype(np.float64), pen, sp)
            drafts[b, i] = ids[0]
            pen.append(int(ids[0]))
    out, n, _ = oracle.verify_sample(tgt, dft, "f32", drafts, hist, sp, 9, 0)
    assert np.all(n == 3)
    assert np.array_equal(out[:, :3], drafts)


def test_unit_penalty_ignores_history():
    tgt, dft, drafts, hist = _cont_inputs(32, 2, 200, 2)
    sp = P(temp=0.8, top_p=0.9, min_p=0.02, rep_penalty=1.0)
    a = oracle.verify_sample(tgt, dft, "f32", drafts, hist, sp, 1, 2)
    b = oracle.verify_sample(tgt, dft, "f32", drafts, -np.ones_like(hist), sp, 1, 2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bf16_inputs_equal_their_fp32_widening():
    tgt, dft, drafts, hist = _cont_inputs(16, 3, 500, 3)
    tb, db = synth.f32_to_bf16_bits(tgt), synth.f32_to_bf16_bits(dft)
    sp = P(temp=0.6, top_p=0.95, min_p=0.05, rep_penalty=1.08)
    a = oracle.verify_sample(tb, db, "bf16", drafts, hist, sp, 4, 0)
    b = oracle.verify_sample(synth.bf16_bits_to_f32(tb), synth.bf16_bits_to_f32(db), "f32", drafts, hist, sp, 4, 0)
    assert np.array_equal(a[0], b[0])


# ----------------------------------------------------------------------------
# Monte Carlo total variation
# ----------------------------------------------------------------------------

class ToySampler:
    """6-token toy model with history-dependent logits and a distinct drafter."""

    def __init__(self, sp, seed=42):
        rng = np.random.default_rng(seed)
        self.V = 6
        self.t1 = 1.5 * rng.standard_normal((6, 6))
        self.t2 = 0.8 * rng.standard_normal((6, 6))
        self.d1 = 1.0 * rng.standard_normal((6, 6))
        self.sp = sp
        self._cache = {}

    def z_target(self, ctx):
        return self.t1[ctx[-1]] + self.t2[ctx[-2]]

    def z_draft(self, ctx):
        return 0.7 * self.z_target(ctx) + self.d1[ctx[-1]]

    def dist(self, ctx, which):
        key = (tuple(ctx), which)
        if key not in self._cache:
            z = self.z_target(ctx) if which == "t" else self.z_draft(ctx)
            ids, w, ws, _ = oracle.sample_dist(z, list(ctx), self.sp)
            p = np.zeros(6)
            p[ids] = w / ws
            self._cache[key] = (ids, np.cumsum(w / ws), p)
        return self._cache[key]


def _exact_3(toy, h0):
    P3 = np.zeros((6, 6, 6))
    p1 = toy.dist(h0, "t")[2]
    for a in range(6):
        if p1[a] == 0:
            continue
        p2 = toy.dist(h0 + [a], "t")[2]
        for b in range(6):
            if p2[b] == 0:
                continue
            p3 = toy.dist(h0 + [a, b], "t")[2]
            P3[a, b] = p1[a] * p2[b] * p3
    return P3.reshape(-1)


def _draw(toy, ctxs, which, rng):
    """Sample one token for each context from toy.dist(ctx, which)."""
    out = np.empty(len(ctxs), dtype=np.int32)
    groups = {}
    for j, c in enumerate(ctxs):
        groups.setdefault(tuple(c), []).append(j)
    for c, js in groups.items():
        ids, cdf, _ = toy.dist(list(c), which)
        u = rng.random(len(js)) * cdf[-1]
        out[js] = np.asarray(ids)[np.minimum(np.searchsorted(cdf, u, side="right"), len(ids) - 1)]
    return out


def _speculate(toy, h0, S, N, rng, seed, rule="exact", greedy_drafter=False, verify=None):
    """Generate 3 tokens per sequence by rounds of N drafts + verify (the
    oracle's exact verifier unless `verify` is given, with its signature)."""
    verify = verify or oracle.verify_sample
    gen = [[] for _ in range(S)]
    rnd = 0
    tokens_per_round = []
    while True:
        act = [s for s in range(S) if len(gen[s]) < 3]
        if not act:
            break
        ctx = [h0 + gen[s] for s in act]
        drafts = np.empty((len(act), N), dtype=np.int32)
        cur = [list(c) for c in ctx]
        for i in range(N):
            if greedy_drafter:
                d = np.array([int(np.argmax(toy.z_target(c))) for c in cur], dtype=np.int32)
            else:
                d = _draw(toy, cur, "d", rng)
            drafts[:, i] = d
            for j in range(len(act)):
                cur[j].append(int(d[j]))
        tgt = np.empty((len(act), N + 1, 6), dtype=np.float32)
        dft = np.empty((len(act), N, 6), dtype=np.float32)
        H = len(h0) + 3
        hist = -np.ones((len(act), H), dtype=np.int32)
        for j, c in enumerate(ctx):
            full = c + list(drafts[j])
            for i in range(N + 1):
                tgt[j, i] = toy.z_target(full[:len(c) + i])
            for i in range(N):
                if greedy_drafter:
                    dft[j, i] = -1e4
                    dft[j, i, drafts[j, i]] = 0.0
                else:
                    dft[j, i] = toy.z_draft(full[:len(c) + i])
            hist[j, H - len(c):] = c
        if rule == "exact":
            out, n, _ = verify(tgt, dft, "f32", drafts, hist, toy.sp, seed, rnd)
        else:
            # the old rule: keep drafts while they equal the unpenalised target argmax,
            # then sample the stop row from the penalised target distribution
            out = -np.ones((len(act), N + 1), dtype=np.int32)
            n = np.zeros(len(act), dtype=np.int32)
            stop_ctx = []
            for j in range(len(act)):
                k = 0
                while k < N and drafts[j, k] == int(np.argmax(tgt[j, k])):
                    k += 1
                n[j] = k
                out[j, :k] = drafts[j, :k]
                stop_ctx.append(ctx[j] + list(drafts[j, :k]))
            last = _draw(toy, stop_ctx, "t", rng)
            for j in range(len(act)):
                out[j, n[j]] = last[j]
        for j, s in enumerate(act):
            gen[s] += [int(t) for t in out[j, :n[j] + 1]]
        tokens_per_round.append(float(np.mean(n + 1)))
        rnd += 1
    seqs = np.array([g[:3] for g in gen])
    idx = seqs[:, 0] * 36 + seqs[:, 1] * 6 + seqs[:, 2]
    return np.bincount(idx, minlength=216) / S, tokens_per_round[0]


def _tv(a, b):
    return 0.5 * float(np.abs(a - b).sum())


@pytest.mark.slow
def test_monte_carlo_tv_exact_vs_greedy_match():
    g = json.load(open(os.path.join(HERE, "golden", "spec_sample_tv.json")))
    st = g["setup"]
    sp = P(temp=st["temp"], top_p=st["top_p"], min_p=st["min_p"], rep_penalty=st["rep_penalty"],
           presence_penalty=st["presence_penalty"])
    S = st["sequences"]
    toy = ToySampler(sp)
    h0 = [1, 4, 2, 0]
    exact = _exact_3(toy, h0)
    assert abs(exact.sum() - 1.0) < 1e-6   # fp32 sampler probabilities
    exact = exact / exact.sum()
    rng = np.random.default_rng(2024)
    direct = np.bincount(rng.choice(216, size=S, p=exact / exact.sum()), minlength=216) / S
    tv_noise = _tv(direct, exact)
    spec, tpr = _speculate(toy, h0, S, 2, rng, seed=77)
    tv_exact = _tv(spec, exact)
    greedy, _ = _speculate(toy, h0, S, 2, rng, seed=78, rule="greedy-match")
    tv_greedy = _tv(greedy, exact)
    print(f"TV noise {tv_noise:.4f} exact {tv_exact:.4f} greedy-match {tv_greedy:.4f}; tokens/round {tpr:.2f}")
    # the pages: exact sits at the noise floor, greedy-match an order of magnitude above
    assert tv_exact < 1.5 * tv_noise + 0.002
    assert tv_greedy > 5 * tv_noise and tv_greedy > 0.02
    # chi-square goodness of fit of the speculative sample against the exact law
    from scipy.stats import chisquare
    keep = exact * S >= 5
    obs, exp_ = spec[keep] * S, exact[keep] * S
    if exact[~keep].sum() > 0:
        obs = np.append(obs, spec[~keep].sum() * S)
        exp_ = np.append(exp_, exact[~keep].sum() * S)
    exp_ = exp_ * (obs.sum() / exp_.sum())
    assert chisquare(obs, exp_).pvalue > 1e-3


@pytest.mark.slow
def test_monte_carlo_tv_deterministic_drafter():
    """q one-hot (the drafter's own greedy chain): accept with p(x), still exact."""
    sp = P(temp=0.6, top_p=0.95, min_p=0.05, rep_penalty=1.08, presence_penalty=0.4)
    toy = ToySampler(sp, seed=7)
    h0 = [3, 5, 1, 2]
    exact = _exact_3(toy, h0)
    S = 200000
    rng = np.random.default_rng(5)
    direct = np.bincount(rng.choice(216, size=S, p=exact / exact.sum()), minlength=216) / S
    spec, tpr = _speculate(toy, h0, S, 2, rng, seed=3, greedy_drafter=True)
    print(f"TV noise {_tv(direct, exact):.4f} exact {_tv(spec, exact):.4f}; tokens/round {tpr:.2f}")
    assert _tv(spec, exact) < 1.5 * _tv(direct, exact) + 0.002
    assert 1.0 < tpr <= 3.0


# ----------------------------------------------------------------------------
# the sampling drafter's draws
# ----------------------------------------------------------------------------

def test_sample_drafts_min_p_one_is_penalised_argmax_chain():
    """min-p 1 keeps only the largest penalised logit, so every draw is the
    row's argmax after penalties over the history and the earlier draws."""
    rng = np.random.default_rng(7)
    B, N, V = 6, 4, 50
    dft = rng.standard_normal((B, N, V)).astype(np.float32)
    hist = rng.integers(0, V, size=(B, 5)).astype(np.int32)
    # make the raw argmax of every row a penalised token, so penalties matter
    for b in range(B):
        for i in range(N):
            dft[b, i, hist[b, 0]] = 10.0
            dft[b, i, (hist[b, 0] + 1) % V] = 9.5
    sp = P(min_p=1.0, temp=0.9, rep_penalty=2.0)
    d, _ = oracle.sample_drafts(dft, "f32", hist, sp, 3, 0)
    for b in range(B):
        pen = set(int(x) for x in hist[b])
        for i in range(N):
            l = dft[b, i].astype(np.float64).copy()
            for x in pen:
                l[x] = l[x] / 2.0 if l[x] > 0 else l[x] * 2.0
            assert d[b, i] == int(np.argmax(l))
            pen.add(int(d[b, i]))


def test_sample_drafts_are_picks_of_their_rows():
    """Each draw is the inverse-CDF pick of sample_dist of its row with the
    penalty set grown by the earlier draws and the uniform of (b, i, 0)."""
    rng = np.random.default_rng(8)
    B, N, V = 5, 3, 300
    dft = (2 * rng.standard_normal((B, N, V))).astype(np.float32)
    hist = rng.integers(0, V, size=(B, 9)).astype(np.int32)
    sp = P(temp=0.6, top_p=0.95, min_p=0.05, rep_penalty=1.08)
    d, _ = oracle.sample_drafts(dft, "f32", hist, sp, 12, 34)
    for b in range(B):
        pen = list(hist[b])
        for i in range(N):
            ids, w, ws, _ = oracle.sample_dist(dft[b, i].astype(np.float64), pen, sp)
            u = oracle.uniform(12, 34, b, i, 0)
            assert d[b, i] == oracle.pick(ids, w, ws, u)[0]
            pen.append(int(d[b, i]))


def test_sample_drafts_follow_q():
    """Over many offsets the first draw's frequencies match q_0 (chi-square)."""
    from scipy.stats import chisquare
    z = np.array([[[1.0, 0.3, -0.2, 0.8, -1.5, 0.0, 0.5]]], dtype=np.float32)
    sp = P(temp=0.8, top_p=0.97, min_p=0.02, rep_penalty=1.0)
    ids, w, ws, _ = oracle.sample_dist(z[0, 0].astype(np.float64), [], sp)
    q = np.zeros(7)
    q[ids] = np.asarray(w) / ws
    T = 20000
    zz = np.repeat(z, T, axis=0)
    d, _ = oracle.sample_drafts(zz, "f32", np.zeros((T, 0), dtype=np.int32), sp, 5, 0)
    cnt = np.bincount(d[:, 0], minlength=7)
    keep = q > 0
    assert np.all(cnt[~keep] == 0)
    exp_ = q[keep] * cnt[keep].sum() / q[keep].sum()
    assert chisquare(cnt[keep], exp_).pvalue > 1e-3


def test_exact_min_p_boundary_has_zero_margin():
    """A weight exactly at the min-p cut is kept (w >= min_p) and reported
    with margin 0: another exp could round it to either side."""
    l1 = np.float32(-0.6931472)
    mp = float(np.float32(np.exp(np.float64(l1))))
    ids, w, ws, mg = oracle.sample_dist(np.array([0.0, float(l1), -3.0]), [], P(min_p=mp))
    assert list(ids) == [0, 1] and mg == 0.0
