"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding and compare with the oracle under the parity rules.

Parity rules (logits and hidden state): max |gpu - oracle| <= tol * rms(oracle
row), tol = 1e-3 for fp32 weights and 2e-2 for bf16 weights; draft tokens must
equal the oracle's argmax wherever the oracle's top-1 / top-2 margin exceeds
1e-2 of the row's standard deviation.  The oracle is teacher-forced with the
GPU's tokens, so a flipped near-tie does not derail the later steps.
"""
import numpy as np

import oracle


def tol_for(w):
    return 1e-3 if w.model.dtype == "f32" else 2e-2


def run_gpu_draft(w, want_logits=True, dev=None):
    import torch
    from mtp_speculative_decoding_gb300.device import upload_draft
    import mtp_speculative_decoding_gb300 as mtp
    dev = dev or upload_draft(w)
    B, N, V, d_t = w.B, w.N, w.model.vocab, w.model.d_t
    drafts = torch.full((B, N), -7, dtype=torch.int32, device="cuda")
    h_last = torch.full((B, d_t), float("nan"), dtype=torch.float32, device="cuda")
    logits = torch.full((B, N, V), float("nan"), dtype=torch.float32, device="cuda") if want_logits else None
    dev.run(drafts, h_last, logits)
    torch.cuda.synchronize()
    assert mtp.last_error(dev.ws) == 0
    return dev, drafts.cpu().numpy(), h_last.cpu().numpy(), (logits.cpu().numpy() if want_logits else None)


def check_draft_parity(w, g_drafts, g_h, g_logits, seqs):
    """g_logits may be None (a run without the diagnostic logits output):
    then the tokens and h_last are checked against the oracle alone."""
    tol = tol_for(w)
    seqs = list(seqs)
    ref = oracle.draft_block(w, seqs=seqs, force=g_drafts)
    worst = 0.0
    flips = 0
    for j, b in enumerate(seqs):
        for k in range(w.N):
            zo = ref["logits"][j, k]
            rms = float(np.sqrt(np.mean(zo * zo)))
            if g_logits is not None:
                zg = g_logits[b, k]
                assert np.all(np.isfinite(zg)), f"non-finite GPU logits (b={b}, k={k})"
                err = float(np.max(np.abs(zg - zo)))
                worst = max(worst, err / rms)
                assert err <= tol * rms, f"b={b} k={k}: max|dz| {err:.3g} > {tol} * rms {rms:.3g}"
            srt = np.sort(zo)
            margin = srt[-1] - srt[-2]
            if margin > 1e-2 * np.std(zo):
                assert g_drafts[b, k] == int(np.argmax(zo)), f"b={b} k={k}: draft {g_drafts[b, k]} != {int(np.argmax(zo))}"
            elif g_drafts[b, k] != int(np.argmax(zo)):
                flips += 1
        ho = ref["h_last"][j]
        hr = float(np.sqrt(np.mean(ho * ho)))
        assert np.max(np.abs(g_h[b] - ho)) <= tol * hr
    return worst, flips
