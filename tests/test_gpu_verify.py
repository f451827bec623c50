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


def compare_sample(inp, seed, offset):
    """Bit-exact: both sides take the sampler's decisions in IEEE fp32 with the
    same steps, so every sequence must match.  The oracle's margins (distance
    of each decision to its threshold) are printed for the record."""
    go, gn = gpu_sample(inp, seed, offset)
    oo, on, mg = oracle.verify_sample(inp.target, inp.draft, inp.dtype, inp.drafts, inp.hist, inp.params,
                                      seed, offset)
    print(f"closest decision margin {mg.min():.2e}; sequences within 1e-6: {(mg < 1e-6).sum()} of {mg.size}")
    bad = np.nonzero((go != oo).any(1) | (gn != on))[0]
    assert bad.size == 0, f"sequences {bad} differ; their margins {mg[bad]}"
    return gn


def test_sample_parity_workload4():
    inp = synth.make_verify_sample_inputs()
    n = compare_sample(inp, seed=inp.seed, offset=0)
    assert 0 < n.mean() < 3


@pytest.mark.parametrize("seed", [1, 2])
def test_sample_parity_small_penalties(seed):
    p = synth.SampleParams(temp=0.8, top_p=0.9, min_p=0.02, rep_penalty=1.3, presence_penalty=0.5)
    inp = synth.make_verify_sample_inputs(seed=seed, B=16, N=4, V=6007, H=24, dtype="f32", params=p)
    compare_sample(inp, seed=seed, offset=seed * 1000)


def test_sample_min_p_one_is_greedy():
    p = synth.SampleParams(temp=0.7, top_p=1.0, min_p=1.0, rep_penalty=1.0)
    inp = synth.make_verify_sample_inputs(seed=4, B=8, N=3, V=5000, dtype="f32", params=p)
    so, sn = gpu_sample(inp, 3, 0)
    go, gn = gpu_greedy(inp.target, inp.dtype, inp.drafts)
    assert np.array_equal(so, go) and np.array_equal(sn, gn)
