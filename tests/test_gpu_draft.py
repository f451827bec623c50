"""GPU parity of mtp_draft_block against the oracle (through the C ABI)."""
import numpy as np
import pytest

import synth
from gpu_common import check_draft_parity, run_gpu_draft

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mtp_speculative_decoding_gb300 import build
    build.build()


def small_workload(dtype, B=3, N=3, seed=5, kv=(37, 23, 100), softcap=0.0, V=1000, hd=32, sink=0):
    """Several tiles of every phase plus ragged tails: V not a multiple of the
    row split, a sliding ring view with stale (NaN) slots, ragged kv_len."""
    m = synth.ModelSpec(d_t=96, d_a=64, n_blocks=2, n_q_heads=4, head_dim=hd, n_kv_heads=2, d_ff=136,
                        vocab=V, dtype=dtype, block_view=(0, 1), logit_softcap=softcap)
    views = [synth.ViewSpec(cap=48 + sink, window=40, rope_theta=1e4, sink=sink),
             synth.ViewSpec(cap=128, window=0, rope_theta=1e6)]
    return synth.make_draft_workload("small", m, views, B, N, list(kv)[:B], seed, hist_len=8)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_parity(dtype):
    w = small_workload(dtype)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=range(w.B))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_single_sequence(dtype):
    """B = 1 streams every weight share and the LM head through bulk copies;
    few rows per CTA here, so rows are split across warps."""
    w = small_workload(dtype, B=1, kv=(77,), V=3001)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0])


def test_single_sequence_split_and_paired_rows():
    """B = 1 with rows that take the split-row GEMV (fewer rows than half the
    grid's warps: pre/post-projection, O, FFN2; 250 chunks split unevenly
    over CTAs of 8 rows) and the paired-row GEMV (4096 query rows of 125
    chunks, more rows than warps, a ragged second row)."""
    m = synth.ModelSpec(d_t=1000, d_a=1000, n_blocks=1, n_q_heads=16, head_dim=256, n_kv_heads=4, d_ff=1200,
                        vocab=3001, dtype="bf16", block_view=(0,))
    views = [synth.ViewSpec(cap=160, window=0, rope_theta=1e6)]
    w = synth.make_draft_workload("wide_b1", m, views, 1, 2, [150], 21, hist_len=4)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_sink_and_window(dtype):
    """Attention sink + window ("opus-mtp-turbo", item 2): the sliding view
    keeps 8 sink positions in slots 0..7 and a 40-slot ring after them; the
    lengths cover a window past the sink with a ring wrap (100), a window
    overlapping the sink (45) and no window cut (23)."""
    w = small_workload(dtype, kv=(100, 45, 23), sink=8)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=range(w.B))


@pytest.mark.slow
def test_workload2_with_sink_64():
    """Workload 2 with the page's default of 64 sink positions beside the
    1024-position sliding window."""
    w = synth.make_draft_inputs(2, sink=64)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0, 5, 11, 15])


def test_small_softcap_and_head_dim_64():
    w = small_workload("bf16", softcap=5.0, hd=64, kv=(1, 64, 127))
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=range(w.B))


def test_small_batch_needs_global_activations():
    # B = 40 does not fit the shared-memory activation stage at this width
    m = synth.ModelSpec(d_t=1024, d_a=256, n_blocks=1, n_q_heads=4, head_dim=64, n_kv_heads=1, d_ff=512,
                        vocab=2048, dtype="bf16", block_view=(0,))
    views = [synth.ViewSpec(cap=96, window=0, rope_theta=1e6)]
    rng = np.random.default_rng(0)
    kv = rng.integers(1, 97, size=40)
    w = synth.make_draft_workload("batch40", m, views, 40, 2, kv, 9, hist_len=4)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0, 17, 39])


def test_tensor_core_head_ragged_vocab_softcap():
    """Smallest tensor-core batch (B = 9): the head's 256-row table tiles end
    in a partial tile (V = 3001), logits are soft-capped and stored, and the
    batch block is zero past B."""
    m = synth.ModelSpec(d_t=1024, d_a=256, n_blocks=1, n_q_heads=4, head_dim=64, n_kv_heads=1, d_ff=512,
                        vocab=3001, dtype="bf16", block_view=(0,), logit_softcap=8.0)
    views = [synth.ViewSpec(cap=96, window=0, rope_theta=1e6)]
    rng = np.random.default_rng(3)
    kv = rng.integers(1, 97, size=9)
    w = synth.make_draft_workload("tc_head_v3001", m, views, 9, 2, kv, 13, hist_len=4)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0, 4, 8])


def test_workload0_tiny_fp32():
    w = synth.make_draft_inputs(0)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0])


def test_deterministic_and_workspace_reuse():
    import torch
    w = small_workload("bf16")
    dev, d1, h1, z1 = run_gpu_draft(w)
    _, d2, h2, z2 = run_gpu_draft(w, dev=dev)
    assert np.array_equal(d1, d2) and np.array_equal(h1, h2) and np.array_equal(z1, z2)


def test_default_scales_are_the_documented_ones():
    """attn_scale = emb_scale = 0 selects 1/sqrt(head_dim) and sqrt(d_t): the
    same outputs, bit for bit, as the explicit values."""
    import ctypes
    w = small_workload("f32", softcap=3.0)
    dev, d1, h1, z1 = run_gpu_draft(w)
    dev.cfg.attn_scale = 0.0
    dev.cfg.emb_scale = 0.0
    _, d2, h2, z2 = run_gpu_draft(w, dev=dev)
    assert np.array_equal(d1, d2) and np.array_equal(h1, h2) and np.array_equal(z1, z2)
    assert ctypes.c_float(w.model.attn_scale).value == ctypes.c_float(1.0 / np.sqrt(w.model.head_dim)).value


@pytest.mark.slow
def test_workload1_gemma_b1():
    w = synth.make_draft_inputs(1)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0])


# Sequences of a 64-row batch spread over the tensor-core LM head's four
# epilogue warps: accumulator row b sits in lane b % 16 of warp b / 16.
SPREAD64 = [16 * q + i for q in range(4) for i in (0, 5, 10, 15)]


@pytest.mark.slow
def test_workload2_ragged_b16_every_sequence():
    w = synth.make_draft_inputs(2)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=range(w.B))


@pytest.mark.slow
def test_workload3_b64_spread_sequences():
    w = synth.make_draft_inputs(3)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=SPREAD64)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [1, 3])
def test_timed_path_without_logits(cfg):
    """The configuration the benchmark times (no logits output) gives the
    same drafts and h_last, bit for bit, as the run that stores the logits,
    and matches the oracle."""
    w = synth.make_draft_inputs(cfg)
    dev, d0, h0, _ = run_gpu_draft(w, want_logits=False)
    _, d1, h1, z1 = run_gpu_draft(w, dev=dev)
    assert np.array_equal(d0, d1) and np.array_equal(h0, h1)
    check_draft_parity(w, d0, h0, None, seqs=[0] if w.B == 1 else SPREAD64[::2])


# ----------------------------------------------------------------------------
# sampled drafting (temperature > 0)
# ----------------------------------------------------------------------------

SP = synth.SampleParams()


def run_sampled(w, seed, offset, want_logits=True):
    import torch
    from mtp_speculative_decoding_gb300.device import upload_draft
    import mtp_speculative_decoding_gb300 as mtp
    dev = upload_draft(w)
    B, N, V = w.B, w.N, w.model.vocab
    drafts = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    h_last = torch.full((B, w.model.d_t), float("nan"), dtype=torch.float32, device="cuda")
    logits = torch.full((B, N, V), float("nan"), dtype=torch.float32, device="cuda") if want_logits else None
    sp = (SP.temp, SP.top_p, SP.min_p, SP.rep_penalty, SP.presence_penalty, SP.top_k)
    dev.run(drafts, h_last, logits, sample=sp, seed=seed, offset=offset)
    torch.cuda.synchronize()
    assert mtp.last_error(dev.ws) == 0
    return drafts.cpu().numpy(), h_last.cpu().numpy(), (logits.cpu().numpy() if want_logits else None)


def check_sampled(w, seed, offset, g_drafts, g_h, g_logits, seqs, margin_min=1e-3):
    """The oracle follows the GPU's tokens (teacher forcing).  Each step's
    logits match within the dtype tolerance.  The draws are the same except
    where a sampler decision (a min-p or top-p cut, the order of two
    candidates, the inverse-CDF pick) lies within margin_min (relative) of its
    threshold -- there the last-bit differences of the logits may move it --
    and such draws are at most a tenth of all.  Returns the matching draws."""
    from gpu_common import tol_for
    import oracle
    tol = tol_for(w)
    ref = oracle.draft_block(w, sample=SP, seed=seed, offset=offset, seqs=seqs, force=g_drafts)
    same, total = 0, 0
    for j, b in enumerate(seqs):
        for k in range(w.N):
            assert 0 <= g_drafts[b, k] < w.model.vocab
            if g_logits is not None:
                zo, zg = ref["logits"][j, k], g_logits[b, k]
                rms = float(np.sqrt(np.mean(zo * zo)))
                assert float(np.max(np.abs(zg - zo))) <= tol * rms
            total += 1
            if g_drafts[b, k] == ref["drafts"][j, k]:
                same += 1
            else:
                assert ref["margin"][j, k] < margin_min, f"b={b} k={k}: {g_drafts[b, k]} != {ref['drafts'][j, k]}"
        ho = ref["h_last"][j]
        assert np.max(np.abs(g_h[b] - ho)) <= tol * float(np.sqrt(np.mean(ho * ho)))
    assert total - same <= max(1, total // 10), f"{total - same} of {total} draws differ"
    return same


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_sampled_drafts(dtype):
    w = small_workload(dtype)
    d, h, z = run_sampled(w, seed=1234, offset=7)
    check_sampled(w, 1234, 7, d, h, z, seqs=range(w.B))
    d2, _, _ = run_sampled(w, seed=1234, offset=7)
    assert np.array_equal(d, d2)   # same Philox stream -> same draws
    d3, _, _ = run_sampled(w, seed=1235, offset=7)
    assert not np.array_equal(d, d3) or w.model.vocab < 4


def test_small_sampled_tensor_core_batch():
    # B = 40 runs the tensor-core head and projections, then the sampler
    m = synth.ModelSpec(d_t=1024, d_a=256, n_blocks=1, n_q_heads=4, head_dim=64, n_kv_heads=1, d_ff=512,
                        vocab=2048, dtype="bf16", block_view=(0,))
    views = [synth.ViewSpec(cap=96, window=0, rope_theta=1e6)]
    rng = np.random.default_rng(1)
    kv = rng.integers(1, 97, size=40)
    w = synth.make_draft_workload("batch40s", m, views, 40, 2, kv, 11, hist_len=4)
    d, h, z = run_sampled(w, seed=99, offset=3)
    check_sampled(w, 99, 3, d, h, z, seqs=[0, 21, 39])


@pytest.mark.slow
def test_workload1_sampled():
    w = synth.make_draft_inputs(1)
    d, h, z = run_sampled(w, seed=5, offset=0)
    check_sampled(w, 5, 0, d, h, z, seqs=[0])


# ----------------------------------------------------------------------------
# per-step confidence output ("MTP decoding (--mtp)", "Stopping early when the
# head is unsure"): the top-1 softmax probability of each step's logits
# ----------------------------------------------------------------------------

def run_conf(w, sample=None):
    import torch
    from mtp_speculative_decoding_gb300.device import upload_draft
    import mtp_speculative_decoding_gb300 as mtp
    dev = upload_draft(w)
    B, N, V = w.B, w.N, w.model.vocab
    drafts = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    conf = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    logits = torch.full((B, N, V), float("nan"), dtype=torch.float32, device="cuda")
    kw = {}
    if sample is not None:
        kw = dict(sample=(SP.temp, SP.top_p, SP.min_p, SP.rep_penalty, SP.presence_penalty, SP.top_k), seed=3)
    dev.run(drafts, out_logits=logits, out_conf=conf, **kw)
    torch.cuda.synchronize()
    assert mtp.last_error(dev.ws) == 0
    # the confidence output leaves the drafts unchanged
    d2 = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    dev.run(d2, **kw)
    torch.cuda.synchronize()
    assert torch.equal(drafts, d2)
    return drafts.cpu().numpy(), conf.cpu().numpy(), logits.cpu().numpy()


def check_conf(w, d, c, z, seqs, sample=None):
    """The reduction is checked against the GPU's own logits: the softmax
    probability of their largest entry, within 1e-4 (relative; fp32 sums
    over the vocabulary).  Against the oracle's top-1 probability of the same
    step (the oracle follows the GPU's tokens) the bound is the logits' own:
    1e-3 with fp32 weights; 1e-2 with bf16 weights, since the batched head
    multiplies bf16(h) and every logit moves by up to ~2^-8 of its size."""
    import oracle
    tol = 1e-3 if w.model.dtype == "f32" else 1e-2
    ref = oracle.draft_block(w, sample=sample, seed=3, seqs=seqs, force=d, want_logits=False)
    for j, b in enumerate(seqs):
        for k in range(w.N):
            own = oracle.top1_prob(z[b, k].astype(np.float64))
            assert abs(c[b, k] - own) <= 1e-4 * own, f"b={b} k={k}: conf {c[b, k]} vs its logits' {own}"
            o = ref["conf"][j, k]
            assert abs(c[b, k] - o) <= tol * o, f"b={b} k={k}: conf {c[b, k]} vs oracle {o}"


@pytest.mark.parametrize("dtype,B", [("f32", 3), ("bf16", 3), ("bf16", 1)])
def test_confidence_small(dtype, B):
    """CUDA-core heads: the generic GEMV head (B = 3) and the single-sequence
    bulk-copy head (B = 1)."""
    w = small_workload(dtype, B=B, kv=(37, 23, 100)[:B], V=3001, softcap=4.0)
    d, c, z = run_conf(w)
    check_conf(w, d, c, z, range(B))


def test_confidence_tensor_core_head_sampled():
    """The tensor-core head (B = 9) with sampled drafting: the confidence is
    the top-1 probability of the raw logits either way."""
    m = synth.ModelSpec(d_t=1024, d_a=256, n_blocks=1, n_q_heads=4, head_dim=64, n_kv_heads=1, d_ff=512,
                        vocab=3001, dtype="bf16", block_view=(0,))
    views = [synth.ViewSpec(cap=96, window=0, rope_theta=1e6)]
    kv = np.random.default_rng(5).integers(1, 97, size=9)
    w = synth.make_draft_workload("conf_tc", m, views, 9, 2, kv, 17, hist_len=4)
    d, c, z = run_conf(w, sample=SP)
    check_conf(w, d, c, z, range(9), sample=SP)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [1, 3])
def test_confidence_workloads(cfg):
    w = synth.make_draft_inputs(cfg)
    d, c, z = run_conf(w)
    check_conf(w, d, c, z, [0] if w.B == 1 else SPREAD64[::4])


@pytest.mark.parametrize("dtype,B", [("bf16", 1), ("bf16", 3), ("f32", 2)])
def test_head_dim_512(dtype, B):
    """head_dim 512 (two 16-byte chunks per lane per key row in bf16, four in
    fp32; two query heads per attention pass) on a sliding and a full view,
    one sequence (CUDA-core head) and a batch (bf16: tensor-core head)."""
    m = synth.ModelSpec(d_t=1024, d_a=512, n_blocks=2, n_q_heads=4, head_dim=512, n_kv_heads=2, d_ff=1024,
                        vocab=2000, dtype=dtype, block_view=(0, 1))
    views = [synth.ViewSpec(cap=64, window=48, rope_theta=1e4), synth.ViewSpec(cap=300, window=0, rope_theta=1e6)]
    w = synth.make_draft_workload("hd512", m, views, B, 3, [70, 200, 33][:B], 51 + B, hist_len=4)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=range(B))


@pytest.mark.parametrize("dtype,B", [("f32", 1), ("bf16", 2)])
def test_api_limits(dtype, B):
    """The largest shapes the header allows in one call: N = 16 draft steps,
    MTP_MAX_BLOCKS = 8 blocks over MTP_MAX_VIEWS = 4 views, 16 query heads per
    KV head."""
    import mtp_speculative_decoding_gb300 as mtp
    m = synth.ModelSpec(d_t=256, d_a=128, n_blocks=mtp.MTP_MAX_BLOCKS, n_q_heads=16, head_dim=32, n_kv_heads=1,
                        d_ff=256, vocab=1500, dtype=dtype, block_view=(0, 1, 2, 3, 3, 2, 1, 0))
    views = [synth.ViewSpec(cap=40, window=24, rope_theta=1e4), synth.ViewSpec(cap=90, window=0, rope_theta=1e6),
             synth.ViewSpec(cap=32, window=16, rope_theta=5e3, sink=4), synth.ViewSpec(cap=120, window=0, rope_theta=2e5)]
    assert len(views) == mtp.MTP_MAX_VIEWS
    w = synth.make_draft_workload("limits", m, views, B, 16, [77, 30][:B], 70 + B, hist_len=4)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=range(B))


def test_sampled_sixteen_steps_small_batch():
    """Sampled drafting over N = 16 steps (the penalty set grows to the history
    plus 15 drafts) at B = 3, bf16: the tensor-core head with the sampler."""
    w = small_workload("bf16", N=16, seed=17)
    d, h, z = run_sampled(w, seed=4321, offset=2)
    check_sampled(w, 4321, 2, d, h, z, seqs=range(w.B))
