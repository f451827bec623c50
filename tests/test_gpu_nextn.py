"""GPU parity of the dense NextN drafter (mtp_nextn_draft) against the oracle.

"MTP decoding (--mtp)", "Requirements" and "How it is wired" (the NextN block
drafts from its own KV; the draft context catches up on the accepted rows) and
"The catch-up runs on the accepted prefix".  Rules, as for the assistant
(tests/gpu_common.py): logits and the last hidden state within tol x rms of
the oracle's row (1e-3 fp32, 2e-2 bf16), the oracle teacher-forced with the
GPU's tokens, drafts equal where the oracle's top-1 / top-2 margin exceeds
1e-2 of the row's standard deviation.  The drafter's KV rows the call writes
(catch-up rows and every step's row) match the oracle's within the same
tolerance of the row's rms, and every slot past them is still the NaN the
inputs put there (written nowhere, and never read: a read NaN would make the
logits NaN).
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mtp_speculative_decoding_gb300 import build
    build.build()


def tiny(dtype="f32", B=3, N=3, M=2, kv_len=(0, 5, 9), n_cu=(0, 1, 2), seed=11, d=256, Hq=4, Hkv=2, hd=64,
         V=3000, softcap=0.0):
    m = synth.NextnSpec(d=d, n_q_heads=Hq, head_dim=hd, n_kv_heads=Hkv, d_ff=512, vocab=V, dtype=dtype,
                        rope_theta=1e4, logit_softcap=softcap)
    kv = list(np.resize(np.asarray(kv_len), B))
    nc = list(np.resize(np.asarray(n_cu), B))
    return synth.make_nextn_workload("tiny-nextn", m, B, N, M, kv, nc, seed)


def run(w, dev=None, want_logits=True, conf=False):
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import upload_nextn
    dev = dev or upload_nextn(w)
    B, N, V, d = w.B, w.N, w.model.vocab, w.model.d
    drafts = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    h = torch.full((B, d), float("nan"), dtype=torch.float32, device="cuda")
    z = torch.full((B, N, V), float("nan"), dtype=torch.float32, device="cuda") if want_logits else None
    c = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda") if conf else None
    dev.run(drafts, h, z, out_conf=c)
    torch.cuda.synchronize()
    assert mtp.last_error(dev.ws) == 0
    out = dict(dev=dev, drafts=drafts.cpu().numpy(), h=h.cpu().numpy(), z=None if z is None else z.cpu().numpy(),
               conf=None if c is None else c.cpu().numpy())
    out["k"], out["v"] = dev.k.float().cpu().numpy(), dev.v.float().cpu().numpy()   # the drafter KV, as fp32
    return out


def _widen(a, w):
    return synth.bf16_bits_to_f32(a) if w.model.dtype == "bf16" else np.asarray(a, dtype=np.float32)


def tol_for(w):
    return 1e-3 if w.model.dtype == "f32" else 2e-2


def check(w, g, seqs=None):
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    tol = tol_for(w)
    ref = oracle.nextn_draft(w, force=g["drafts"], seqs=seqs)
    ok_tokens = 0
    for j, b in enumerate(seqs):
        for k in range(w.N):
            zo = ref["logits"][j, k]
            rms = float(np.sqrt(np.mean(zo * zo)))
            if g["z"] is not None:
                zg = g["z"][b, k]
                assert np.all(np.isfinite(zg)), f"b={b} k={k}: non-finite logits"
                err = float(np.max(np.abs(zg - zo)))
                assert err <= tol * rms, f"b={b} k={k}: max|dz| {err:.3g} > {tol} * {rms:.3g}"
            if ref["margin"][j, k] > 1e-2 * float(np.std(zo)):
                assert g["drafts"][b, k] == ref["drafts"][j, k], f"b={b} k={k}"
                ok_tokens += 1
        ho = ref["h_last"][j]
        assert np.max(np.abs(g["h"][b] - ho)) <= tol * float(np.sqrt(np.mean(ho * ho)))
        # the rows this call wrote, and nothing past them
        lo, hi = int(w.kv_len[b]), int(w.kv_len[b] + w.n_cu[b] + w.N)
        for name in ("k", "v"):
            want = _widen(ref[name][b], w)[:, lo:hi].astype(np.float64)
            got = g[name][b][:, lo:hi].astype(np.float64)
            scale = float(np.sqrt(np.mean(want * want)))
            assert np.max(np.abs(got - want)) <= tol * scale, f"b={b} {name} rows"
            assert np.isnan(g[name][b][:, hi:]).all(), f"b={b}: {name} written past its rows"
            np.testing.assert_array_equal(g[name][b][:, :lo], _widen(w.dkv[name][b], w)[:, :lo])
    return ok_tokens


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiny_parity(dtype):
    """Three sequences: an empty KV with no catch-up, 5 rows + 1 catch-up row,
    9 rows + 2 (the catch-up iterations right-aligned over the ragged counts)."""
    w = tiny(dtype)
    g = run(w)
    assert check(w, g) >= w.B * w.N // 2


def test_softcap_and_head_dims():
    for hd, d in ((128, 512), (256, 512), (32, 128)):
        w = tiny("bf16", B=2, kv_len=(7, 3), n_cu=(2, 0), hd=hd, d=d, softcap=20.0)
        check(w, run(w))


def test_batch_sixteen_and_twenty():
    """B >= 2, bf16: the tensor-core LM head (the projections stay on CUDA
    cores at these small widths: their inputs fit in shared memory)."""
    for B in (16, 20):
        w = tiny("bf16", B=B, N=2, M=3, kv_len=tuple(range(0, 3 * B, 3)), n_cu=tuple(i % 4 for i in range(B)),
                 seed=B)
        check(w, run(w), seqs=[0, 5, B - 1])


@pytest.mark.parametrize("B", [9, 24])
def test_tensor_core_paths(B):
    """Width 1024, SwiGLU 4096, bf16: at B = 9 the inputs still fit in shared
    memory (tensor-core head, CUDA-core projections); at B = 24 they do not,
    and the projections run as split-K tensor-core GEMMs (the stored keys and
    values summed from the fused projection's partials, the block output from
    the down projection's)."""
    m = synth.NextnSpec(d=1024, n_q_heads=8, head_dim=128, n_kv_heads=2, d_ff=4096, vocab=5000, dtype="bf16",
                        rope_theta=1e4)
    w = synth.make_nextn_workload("tc-nextn", m, B, 3, 2, [1 + 7 * i for i in range(B)], [i % 3 for i in range(B)],
                                  40 + B)
    check(w, run(w), seqs=[0, B // 2, B - 1])


def test_without_logits_and_confidence():
    w = tiny("f32", seed=3)
    a = run(w)
    b = run(w, want_logits=False, conf=True)
    np.testing.assert_array_equal(a["drafts"], b["drafts"])
    np.testing.assert_array_equal(a["h"], b["h"])
    ref = oracle.nextn_draft(w, force=a["drafts"])
    np.testing.assert_allclose(b["conf"], ref["conf"], rtol=1e-3)
    for bb in range(w.B):
        for k in range(w.N):
            assert abs(b["conf"][bb, k] - oracle.top1_prob(a["z"][bb, k].astype(np.float64))) <= 1e-4 * b["conf"][bb, k]


def test_two_calls_carry_the_kv():
    """N = 3 in one call against N = 1, then a call on the first call's KV
    starting one row after its catch-up rows with its draft and hidden state
    (the library's own chain, on the device between calls)."""
    import copy
    import torch
    w = tiny("f32", seed=5)
    one = run(w)
    w1 = copy.copy(w)
    w1.N = 1
    first = run(w1)
    w2 = copy.copy(w)
    w2.N = 2
    w2.kv_len = (w.kv_len + w.n_cu + 1).astype(np.int32)
    w2.n_cu = np.zeros(w.B, np.int32)
    w2.last_tok = first["drafts"][:, 0].astype(np.int32)
    w2.h_prev = first["h"].astype(np.float32)
    w2.dkv = dict(w.dkv, k=first["k"], v=first["v"])
    second = run(w2)
    for b in range(w.B):
        rms = float(np.sqrt(np.mean(one["z"][b, 1:] ** 2)))
        assert np.max(np.abs(second["z"][b] - one["z"][b, 1:])) <= 1e-4 * rms
        np.testing.assert_array_equal(second["drafts"][b], one["drafts"][b, 1:])


def test_out_of_range_rows_set_the_status():
    """kv_len + n_cu + N past the KV capacity, n_cu above M, a catch-up token
    outside the vocabulary: the status word says MTP_ERR_ARG and the kernel
    writes nothing (checked before any work)."""
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import upload_nextn
    w = tiny("bf16", B=2, kv_len=(3, 4), n_cu=(1, 2))
    cap = w.dkv["cap"]
    for what in ("cap", "ncu", "tok"):
        dev = upload_nextn(w)
        if what == "cap":
            dev.kv_len[1] = cap - w.N - 1   # + n_cu 2 + N > cap
        elif what == "ncu":
            dev.n_cu[0] = w.M + 1
        else:
            dev.cu_tok[1, 0] = w.model.vocab
        k0 = dev.k.clone()
        d = torch.full((w.B, w.N), -7, dtype=torch.int32, device="cuda")
        dev.run(d)
        torch.cuda.synchronize()
        assert mtp.last_error(dev.ws) == mtp.MTP_ERR_ARG, what
        assert torch.equal(dev.k.view(torch.int16), k0.view(torch.int16)), what


def test_host_rejections():
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import upload_nextn
    w = tiny("f32", B=1, kv_len=(2,), n_cu=(1,))
    dev = upload_nextn(w)
    d = torch.empty((1, w.N), dtype=torch.int32, device="cuda")

    def call(**kw):
        cfg = kw.pop("cfg", dev.cfg)
        weights = kw.pop("weights", dev.weights)
        view = kw.pop("view", dev.view)
        mtp.nextn_draft(cfg, weights, view, dev.kv_len, dev.last_tok, dev.h_prev, kw.pop("out", d), dev.ws,
                        n_cu=dev.n_cu, cu_tok=kw.pop("cu_tok", dev.cu_tok), cu_h=dev.cu_h)

    call()
    torch.cuda.synchronize()
    m = w.model
    bad_cfg = mtp.make_config(m.d, m.d // 2, 1, m.n_q_heads, m.head_dim, m.n_kv_heads, m.d_ff, m.vocab, wdtype="f32")
    with pytest.raises(mtp.MTPError) as e:
        call(cfg=bad_cfg)                                    # d_a != d_t
    assert e.value.code == mtp.MTP_ERR_ARG
    two = mtp.make_config(m.d, m.d, 2, m.n_q_heads, m.head_dim, m.n_kv_heads, m.d_ff, m.vocab, wdtype="f32")
    with pytest.raises(mtp.MTPError) as e:
        call(cfg=two)                                        # one block only
    assert e.value.code == mtp.MTP_ERR_UNSUPPORTED
    vw = mtp.make_view(dev.k, dev.v, w.dkv["cap"], 4, 1e4)
    with pytest.raises(mtp.MTPError):
        call(view=vw)                                        # a window
    wk = mtp.make_nextn_weights(dev.tensors)
    wk.blk[0].k_norm = None
    with pytest.raises(mtp.MTPError):
        call(weights=wk)                                     # no key norm
    with pytest.raises(mtp.MTPError):
        call(cu_tok=torch.zeros((1, mtp.MTP_MAX_CATCHUP + 1), dtype=torch.int32, device="cuda"))


@pytest.mark.slow
def test_qwen_shaped_workload():
    w = synth.make_nextn_inputs(7)
    g = run(w)
    check(w, g)


@pytest.mark.slow
def test_qwen_shaped_batch_of_sixteen():
    w = synth.make_nextn_inputs(7, B=16)
    g = run(w, want_logits=False)
    check(w, g, seqs=[0, 15])


def test_maximum_catch_up_and_a_full_kv():
    """M = MTP_MAX_CATCHUP rows (ragged 0..16), and a sequence whose last draft
    row lands in the KV's last slot (kv_len + n_cu + N == cap)."""
    import mtp_speculative_decoding_gb300 as mtp
    M = mtp.MTP_MAX_CATCHUP
    m = synth.NextnSpec(d=256, n_q_heads=4, head_dim=64, n_kv_heads=2, d_ff=512, vocab=3000, dtype="bf16",
                        rope_theta=1e4)
    kv, nc, N = [3, 40, 0, 17], [16, 0, 7, 16], 3
    cap = max(k + c for k, c in zip(kv, nc)) + N
    w = synth.make_nextn_workload("max-catchup", m, 4, N, M, kv, nc, 77, cap=cap)
    assert int((w.kv_len + w.n_cu).max()) + N == w.dkv["cap"]
    check(w, run(w))


def test_batch_of_sixty_four():
    w = tiny("bf16", B=64, N=2, M=2, kv_len=tuple(range(0, 128, 2)), n_cu=tuple(i % 3 for i in range(64)), seed=64)
    check(w, run(w, want_logits=False), seqs=[0, 17, 34, 63])


def test_null_counts_mean_no_catch_up():
    """n_cu NULL with catch-up arrays given: no catch-up rows (the header's
    "NULL: all 0"), the same as counts of zero."""
    import copy
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import upload_nextn
    w = tiny("f32", B=2, kv_len=(4, 6), n_cu=(2, 1), seed=19)
    w0 = copy.copy(w)
    w0.n_cu = np.zeros(w.B, np.int32)
    ref = run(w0)
    dev = upload_nextn(w)
    d = torch.full((w.B, w.N), -7, dtype=torch.int32, device="cuda")
    h = torch.empty((w.B, w.model.d), dtype=torch.float32, device="cuda")
    mtp.nextn_draft(dev.cfg, dev.weights, dev.view, dev.kv_len, dev.last_tok, dev.h_prev, d, dev.ws, n_cu=None,
                    cu_tok=dev.cu_tok, cu_h=dev.cu_h, out_h_last=h)
    torch.cuda.synchronize()
    assert mtp.last_error(dev.ws) == 0
    np.testing.assert_array_equal(d.cpu().numpy(), ref["drafts"])
    np.testing.assert_array_equal(h.cpu().numpy(), ref["h"])


@pytest.mark.parametrize("wquant", ["q8_0", "q4_0"])
@pytest.mark.parametrize("B", [1, 4])
def test_quantised_projections(wquant, B):
    """Q8_0 and Q4_0 projections (eh_proj, the fused query / key / value
    projection with the catch-up rows' key and value rows at their row and
    scale offsets, w_o, the SwiGLU matrices) beside the bf16 table and KV; the
    oracle runs on the weights the codes stand for."""
    m = synth.NextnSpec(d=512, n_q_heads=4, head_dim=64, n_kv_heads=2, d_ff=1024, vocab=3000, dtype="bf16",
                        rope_theta=1e4, wquant=wquant)
    kv, nc = [0, 5, 9, 2][:B], [1, 0, 2, 2][:B]
    w = synth.make_nextn_workload("q-nextn", m, B, 3, 2, kv, nc, 50 + B)
    check(w, run(w))


def test_head_dim_512():
    m = synth.NextnSpec(d=1024, n_q_heads=4, head_dim=512, n_kv_heads=2, d_ff=1024, vocab=2000, dtype="bf16",
                        rope_theta=1e4)
    for B in (1, 3):
        w = synth.make_nextn_workload("hd512-nextn", m, B, 3, 2, [9, 0, 30][:B], [2, 1, 0][:B], 60 + B)
        check(w, run(w))


def test_sixteen_drafts_and_sixteen_heads_per_kv_head():
    m = synth.NextnSpec(d=256, n_q_heads=16, head_dim=32, n_kv_heads=1, d_ff=512, vocab=1500, dtype="bf16",
                        rope_theta=1e4)
    w = synth.make_nextn_workload("limits-nextn", m, 2, 16, 3, [5, 0], [3, 1], 81)
    check(w, run(w))


def test_maximum_catch_up_on_the_tensor_core_path():
    """Sixteen catch-up iterations through the split-K tensor-core projections
    (width 1024, SwiGLU 4096, B = 24 bf16: the inputs outgrow shared memory)."""
    import mtp_speculative_decoding_gb300 as mtp
    m = synth.NextnSpec(d=1024, n_q_heads=8, head_dim=128, n_kv_heads=2, d_ff=4096, vocab=3000, dtype="bf16",
                        rope_theta=1e4)
    B, M = 24, mtp.MTP_MAX_CATCHUP
    w = synth.make_nextn_workload("tc-catchup", m, B, 2, M, [3 * i for i in range(B)], [(5 * i) % (M + 1) for i in range(B)],
                                  91)
    check(w, run(w, want_logits=False), seqs=[0, 3, 16, B - 1])
