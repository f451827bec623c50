"""GPU parity of mtp_verify_greedy and mtp_verify_sample against the oracle."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mtp_speculative_decoding_gb300 import build
    build.build()


def gpu_greedy(logits, dtype, drafts, ws=None):
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import to_device
    B, R, V = logits.shape
    lg = to_device(logits, dtype)
    dr = torch.from_numpy(np.ascontiguousarray(drafts, dtype=np.int32)).cuda()
    out = torch.full((B, R), -9, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ws = ws if ws is not None else mtp.alloc_workspace(mtp.workspace_size(None, B, R - 1, V))
    mtp.verify_greedy(lg, dr, out, n, ws)
    torch.cuda.synchronize()
    assert mtp.last_error(ws) == 0
    return out.cpu().numpy(), n.cpu().numpy()


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_greedy_parity_workloads(cfg):
    inp = synth.make_verify_greedy_inputs(cfg)
    go, gn = gpu_greedy(inp.logits, inp.dtype, inp.drafts)
    oo, on = oracle.verify_greedy(inp.logits, inp.dtype, inp.drafts)
    assert np.array_equal(gn, on) and np.array_equal(go, oo)
    assert np.array_equal(gn, inp.planted)


@pytest.mark.parametrize("V,dtype", [(1, "f32"), (7, "bf16"), (1001, "f32"), (4099, "bf16"), (300001, "bf16")])
def test_greedy_ragged_vocab(V, dtype):
    inp = synth.make_verify_greedy_inputs(0, seed=V, B=5, N=3, V=V, dtype=dtype)
    go, gn = gpu_greedy(inp.logits, inp.dtype, inp.drafts)
    oo, on = oracle.verify_greedy(inp.logits, inp.dtype, inp.drafts)
    assert np.array_equal(go, oo) and np.array_equal(gn, on)


def test_greedy_edge_rows():
    V = 4099
    rng = np.random.default_rng(1)
    lg = rng.standard_normal((4, 3, V)).astype(np.float32)
    lg[0, 0, :] = np.nan              # all-NaN row -> token 0
    lg[1, 0, [5, 4000]] = 50.0         # tie -> lowest index
    lg[2, :, :] = -np.inf
    lg[2, 1, 77] = np.nan
    lg[3, 0, :] = 0.0
    lg[3, 0, 3] = -0.0
    drafts = np.array([[0, 1], [5, 2], [0, 0], [0, 9]], dtype=np.int32)
    go, gn = gpu_greedy(lg, "f32", drafts)
    oo, on = oracle.verify_greedy(lg, "f32", drafts)
    assert np.array_equal(go, oo) and np.array_equal(gn, on)


def test_greedy_no_drafts_and_max_batch():
    inp = synth.make_verify_greedy_inputs(0, seed=3, B=64, N=0, V=5000, dtype="bf16")
    go, gn = gpu_greedy(inp.logits, inp.dtype, inp.drafts.reshape(64, 0))
    oo, on = oracle.verify_greedy(inp.logits, inp.dtype, inp.drafts.reshape(64, 0))
    assert np.array_equal(go, oo) and np.all(gn == 0)


# ----------------------------------------------------------------------------
# exact sampling: both sides take every decision in IEEE fp32 with weights
# exp(l - lmax) rounded once to fp32, so draws agree bit for bit.  A decision
# the oracle finds within BOUNDARY (relative) of its threshold could still go
# either way under a last-bit difference; such sequences are counted, checked
# for validity only, and may be at most 1 % of the sequences (at least one).
# ----------------------------------------------------------------------------

BOUNDARY = 1e-6


def _boundary_budget(n):
    return max(1, n // 100)


def with_oracle_drafts(inp):
    """The drafter's tokens: draws from q_i = sample_dist(draft row i) (oracle)."""
    d, mg = oracle.sample_drafts(inp.draft, inp.dtype, inp.hist, inp.params, inp.seed, inp.offset)
    inp.drafts = d
    return inp, mg


def gpu_sample(inp, seed, offset, ws=None):
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import to_device
    B, R, V = inp.target.shape
    tg, df = to_device(inp.target, inp.dtype), to_device(inp.draft, inp.dtype)
    dr = torch.from_numpy(np.ascontiguousarray(inp.drafts, dtype=np.int32)).cuda()
    hi = torch.from_numpy(np.ascontiguousarray(inp.hist, dtype=np.int32)).cuda()
    out = torch.full((B, R), -9, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ws = ws if ws is not None else mtp.alloc_workspace(mtp.workspace_size(None, B, R - 1, V))
    mtp.verify_sample(tg, df, dr, hi, inp.params, seed, offset, out, n, ws)
    torch.cuda.synchronize()
    assert mtp.last_error(ws) == 0
    return out.cpu().numpy(), n.cpu().numpy()


def gpu_draws(inp, seed, offset):
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import to_device
    B, N, V = inp.draft.shape
    df = to_device(inp.draft, inp.dtype)
    hi = torch.from_numpy(np.ascontiguousarray(inp.hist, dtype=np.int32)).cuda()
    out = torch.full((B, N), -9, dtype=torch.int32, device="cuda")
    ws = mtp.alloc_workspace(mtp.workspace_size(None, B, N, V))
    mtp.sample_drafts(df, hi, inp.params, seed, offset, out, ws)
    torch.cuda.synchronize()
    assert mtp.last_error(ws) == 0
    return out.cpu().numpy()


def _valid_window(out, n, drafts, V):
    B, R = out.shape
    for b in range(B):
        k = int(n[b])
        assert 0 <= k <= R - 1
        assert np.array_equal(out[b, :k], drafts[b, :k])
        assert 0 <= out[b, k] < V
        assert np.all(out[b, k + 1:] == -1)


def compare_sample(inp, seed, offset):
    go, gn = gpu_sample(inp, seed, offset)
    oo, on, mg = oracle.verify_sample(inp.target, inp.draft, inp.dtype, inp.drafts, inp.hist, inp.params,
                                      seed, offset)
    near = mg < BOUNDARY
    print(f"closest decision margin {mg.min():.2e}; sequences within {BOUNDARY}: {near.sum()} of {mg.size}")
    assert near.sum() <= _boundary_budget(mg.size)
    bad = np.nonzero(((go != oo).any(1) | (gn != on)) & ~near)[0]
    assert bad.size == 0, f"sequences {bad} differ; their margins {mg[bad]}"
    _valid_window(go, gn, inp.drafts, inp.target.shape[2])
    return gn


def compare_draws(inp, seed, offset):
    gd = gpu_draws(inp, seed, offset)
    od, mg = oracle.sample_drafts(inp.draft, inp.dtype, inp.hist, inp.params, seed, offset)
    near = mg < BOUNDARY
    assert near.sum() <= _boundary_budget(mg.size)
    bad = np.nonzero((gd != od).any(1) & ~near)[0]
    assert bad.size == 0, f"sequences {bad} differ; their margins {mg[bad]}"
    assert np.all((gd >= 0) & (gd < inp.draft.shape[2]))
    return gd


def test_sample_parity_workload4():
    """Workload 4 at full size: the drafter's draws and the verification."""
    inp = synth.make_verify_sample_inputs()
    compare_draws(inp, inp.seed, inp.offset)
    inp, _ = with_oracle_drafts(inp)
    n = compare_sample(inp, seed=inp.seed, offset=inp.offset)
    assert 0 < n.mean() < 3


@pytest.mark.parametrize("seed", [1, 2])
def test_sample_parity_small_penalties(seed):
    p = synth.SampleParams(temp=0.8, top_p=0.9, min_p=0.02, rep_penalty=1.3, presence_penalty=0.5)
    inp = synth.make_verify_sample_inputs(seed=seed, B=16, N=4, V=6007, H=24, dtype="f32", params=p)
    inp.offset = seed * 1000
    compare_draws(inp, inp.seed, inp.offset)
    inp, _ = with_oracle_drafts(inp)
    compare_sample(inp, seed=seed, offset=inp.offset)


@pytest.mark.parametrize("V,dtype", [(1, "f32"), (6, "bf16"), (33, "f32"), (4097, "bf16"), (70001, "f32")])
def test_sample_ragged_vocab(V, dtype):
    """Vocabularies below, at and across the piece and vector sizes, ragged tails."""
    p = synth.SampleParams(temp=0.7, top_p=0.9, min_p=0.01, rep_penalty=1.1)
    inp = synth.make_verify_sample_inputs(seed=V, B=5, N=3, V=V, H=7, dtype=dtype, params=p)
    inp, _ = with_oracle_drafts(inp)
    compare_sample(inp, seed=11, offset=V)


def test_sample_overflow_rescan():
    """Early pieces of flat logits overflow the survivor buffers; a spike later
    in the row sets the true maximum, so the rows are rescanned exactly."""
    p = synth.SampleParams(temp=1.0, top_p=0.93, min_p=0.05, rep_penalty=1.0)
    inp = synth.make_verify_sample_inputs(seed=9, B=3, N=2, V=100000, H=4, dtype="f32", params=p)
    inp.target[:, :, :60000] = 0.0
    inp.draft[:, :, :60000] = 0.0
    inp.target[:, :, 99000:99010] = 12.0
    inp.draft[:, :, 99000:99020] = 11.0
    inp, _ = with_oracle_drafts(inp)
    compare_sample(inp, seed=3, offset=0)


def test_sample_capacity_status():
    """A min-p set of more than 4096 candidates sets MTP_ERR_CAPACITY."""
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    p = synth.SampleParams(temp=1.0, top_p=1.0, min_p=0.5, rep_penalty=1.0)
    inp = synth.make_verify_sample_inputs(seed=2, B=1, N=1, V=9000, H=0, dtype="f32", params=p)
    inp.target[:] = 0.0
    inp.drafts = np.zeros((1, 1), dtype=np.int32)
    from mtp_speculative_decoding_gb300.device import to_device
    tg, df = to_device(inp.target, "f32"), to_device(inp.draft, "f32")
    dr = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    hi = torch.zeros((1, 0), dtype=torch.int32, device="cuda")
    out = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    n = torch.empty((1,), dtype=torch.int32, device="cuda")
    ws = mtp.alloc_workspace(mtp.workspace_size(None, 1, 1, 9000))
    mtp.verify_sample(tg, df, dr, hi, p, 1, 0, out, n, ws)
    assert mtp.last_error(ws) == mtp.MTP_ERR_CAPACITY


def test_sample_min_p_one_is_greedy():
    p = synth.SampleParams(temp=0.7, top_p=1.0, min_p=1.0, rep_penalty=1.0)
    inp = synth.make_verify_sample_inputs(seed=4, B=8, N=3, V=5000, dtype="f32", params=p)
    inp, _ = with_oracle_drafts(inp)
    so, sn = gpu_sample(inp, 3, 0)
    go, gn = gpu_greedy(inp.target, inp.dtype, inp.drafts)
    assert np.array_equal(so, go) and np.array_equal(sn, gn)


@pytest.mark.slow
def test_monte_carlo_tv_on_gpu():
    """The Monte Carlo check of exact sampling ("opus-mtp-turbo: Track 1
    report", CPU-verified table), with every verification window taken by
    mtp_verify_sample on the GPU: 400k sequences of 3 tokens from a 6-token
    toy model; the speculative sample's total variation from the exact law
    stays at the noise floor of direct sampling, and the greedy-match rule
    (host) stays far above it."""
    import json
    import os
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from test_oracle_verify import HERE, P, ToySampler, _exact_3, _speculate, _tv
    g = json.load(open(os.path.join(HERE, "golden", "spec_sample_tv.json")))
    st = g["setup"]
    sp = P(temp=st["temp"], top_p=st["top_p"], min_p=st["min_p"], rep_penalty=st["rep_penalty"],
           presence_penalty=st["presence_penalty"])
    S = st["sequences"]
    chunk = mtp.MTP_MAX_VERIFY_BATCH
    ws = mtp.alloc_workspace(mtp.workspace_size(None, chunk, 2, 6))

    def gpu_verify(tgt, dft, dtype, drafts, hist, params, seed, offset):
        B = tgt.shape[0]
        out = np.empty((B, tgt.shape[1]), dtype=np.int32)
        n = np.empty(B, dtype=np.int32)
        for c0 in range(0, B, chunk):
            c1 = min(B, c0 + chunk)
            # each chunk is its own call: the Philox sequence word is the row in the call,
            # so chunks take distinct offsets
            tg = torch.from_numpy(np.ascontiguousarray(tgt[c0:c1])).cuda()
            df = torch.from_numpy(np.ascontiguousarray(dft[c0:c1])).cuda()
            dr = torch.from_numpy(np.ascontiguousarray(drafts[c0:c1])).cuda()
            hi = torch.from_numpy(np.ascontiguousarray(hist[c0:c1])).cuda()
            o = torch.empty((c1 - c0, tgt.shape[1]), dtype=torch.int32, device="cuda")
            nn = torch.empty((c1 - c0,), dtype=torch.int32, device="cuda")
            mtp.verify_sample(tg, df, dr, hi, params, seed, offset * 4096 + c0 // chunk, o, nn, ws)
            out[c0:c1] = o.cpu().numpy()
            n[c0:c1] = nn.cpu().numpy()
        assert mtp.last_error(ws) == 0
        return out, n, None

    toy = ToySampler(sp)
    h0 = [1, 4, 2, 0]
    exact = _exact_3(toy, h0)
    exact = exact / exact.sum()
    rng = np.random.default_rng(2025)
    direct = np.bincount(rng.choice(216, size=S, p=exact), minlength=216) / S
    tv_noise = _tv(direct, exact)
    spec, tpr = _speculate(toy, h0, S, 2, rng, seed=91, verify=gpu_verify)
    tv_exact = _tv(spec, exact)
    greedy, _ = _speculate(toy, h0, S, 2, rng, seed=92, rule="greedy-match")
    tv_greedy = _tv(greedy, exact)
    print(f"GPU: TV noise {tv_noise:.4f} exact {tv_exact:.4f} greedy-match {tv_greedy:.4f}; tokens/round {tpr:.2f}")
    assert tv_exact < 1.5 * tv_noise + 0.002
    assert tv_greedy > 5 * tv_noise and tv_greedy > 0.02
