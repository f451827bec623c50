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


def small_workload(dtype, B=3, N=3, seed=5, kv=(37, 23, 100), softcap=0.0, V=1000, hd=32):
    """Several tiles of every phase plus ragged tails: V not a multiple of the
    row split, a sliding ring view with stale (NaN) slots, ragged kv_len."""
    m = synth.ModelSpec(d_t=96, d_a=64, n_blocks=2, n_q_heads=4, head_dim=hd, n_kv_heads=2, d_ff=136,
                        vocab=V, dtype=dtype, block_view=(0, 1), logit_softcap=softcap)
    views = [synth.ViewSpec(cap=48, window=40, rope_theta=1e4), synth.ViewSpec(cap=128, window=0, rope_theta=1e6)]
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


@pytest.mark.slow
def test_workload1_gemma_b1():
    w = synth.make_draft_inputs(1)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0])


@pytest.mark.slow
def test_workload2_ragged_b16_sampled_sequences():
    w = synth.make_draft_inputs(2)
    _, d, h, z = run_gpu_draft(w)
    shortest, longest = int(np.argmin(w.kv_len)), int(np.argmax(w.kv_len))
    check_draft_parity(w, d, h, z, seqs=sorted({shortest, longest, 7}))


@pytest.mark.slow
def test_workload3_b64_sampled_sequences():
    w = synth.make_draft_inputs(3)
    _, d, h, z = run_gpu_draft(w)
    check_draft_parity(w, d, h, z, seqs=[0, 63])
