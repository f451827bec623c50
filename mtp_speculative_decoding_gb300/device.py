"""Device-side containers: upload host arrays (numpy, bf16 as uint16 bits) to
CUDA tensors and keep the C structs that point into them alive together."""
from __future__ import annotations

import dataclasses

import numpy as np

from . import (Config, KVView, Weights, alloc_workspace, draft_block, make_config, make_nextn_weights, make_view,
               make_weights, nextn_draft, quantize, workspace_size)


def to_device(a: np.ndarray, dtype: str | None = None, device="cuda"):
    """numpy -> CUDA tensor; uint16 arrays (or dtype='bf16') become bfloat16."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16 or dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.to(device, non_blocking=False)


@dataclasses.dataclass
class DeviceDraft:
    cfg: Config
    weights: Weights
    views: list
    tensors: dict
    kv_len: object
    last_tok: object
    h_prev: object
    hist: object
    B: int
    N: int
    V: int
    d_t: int
    ws: object

    def run(self, out_drafts, out_h_last=None, out_logits=None, sample=None, seed=0, offset=0, stream=None,
            out_conf=None):
        draft_block(self.cfg, self.weights, self.views, self.kv_len, self.last_tok, self.h_prev, out_drafts,
                    self.ws, out_h_last=out_h_last, out_logits=out_logits, sample=sample, seed=seed,
                    offset=offset, hist=self.hist if sample is not None else None, stream=stream,
                    out_conf=out_conf)


def upload_draft(w, device="cuda", extra_ws_for=None, reuse: "DeviceDraft | None" = None) -> DeviceDraft:
    """Upload a ``synth.DraftWorkload`` (or anything with the same fields).

    ``extra_ws_for`` = (B, N, V) of verify calls that will share the workspace.
    ``reuse``: an earlier upload of the same model whose weight tensors are
    shared instead of uploaded again (its views and workspace are not).
    """
    import torch
    m = w.model
    cfg = make_config(m.d_t, m.d_a, m.n_blocks, m.n_q_heads, m.head_dim, m.n_kv_heads, m.d_ff, m.vocab,
                      wdtype=m.dtype, rms_eps=m.rms_eps, attn_scale=m.attn_scale, emb_scale=m.emb_scale,
                      logit_softcap=m.logit_softcap, n_centroids=getattr(m, "n_centroids", 0),
                      centroid_top_k=getattr(m, "centroid_top_k", 0), wquant=getattr(m, "wquant", "none"))
    same = (reuse is not None and bytes(reuse.cfg) == bytes(cfg) and
            all(n in reuse.tensors and tuple(reuse.tensors[n].shape) == a.shape for n, a in w.weights.items()))
    if same:
        tensors = {n: reuse.tensors[n] for n in w.weights}
        reuse.tensors.pop("_views", None)   # the old views go with the old workload
    elif getattr(m, "wquant", "none") in ("q8_0", "q4_0"):
        # Q8_0 / Q4_0 projections: quantised here by the library's host
        # quantiser, codes and block scales uploaded side by side
        tensors = {}
        for n, a in w.weights.items():
            if a.dtype == np.float32 and a.ndim == 2 and n.split(".")[-1].startswith("w_"):
                q, d = quantize(a, m.wquant)
                tensors[n] = torch.from_numpy(q).to(device)
                tensors[n + ".scale"] = torch.from_numpy(d.view(np.int16)).to(device)
            else:
                tensors[n] = to_device(a, device=device)
    else:
        tensors = {n: to_device(a, device=device) for n, a in w.weights.items()}
    views, keep = [], []
    for vd in w.views:
        k, v = to_device(vd["k"], device=device), to_device(vd["v"], device=device)
        keep += [k, v]
        views.append(make_view(k, v, vd["cap"], vd["window"], vd["rope_theta"], vd.get("sink", 0)))
    tensors["_views"] = keep
    weights = make_weights(tensors, m.n_blocks, m.block_view)
    kv_len = torch.from_numpy(np.ascontiguousarray(w.kv_len, dtype=np.int32)).to(device)
    last_tok = torch.from_numpy(np.ascontiguousarray(w.last_tok, dtype=np.int32)).to(device)
    h_prev = torch.from_numpy(np.ascontiguousarray(w.h_prev, dtype=np.float32)).to(device)
    hist = torch.from_numpy(np.ascontiguousarray(w.hist, dtype=np.int32)).to(device) if w.hist.size else None
    nbytes = workspace_size(cfg, w.B, w.N, m.vocab)
    if extra_ws_for is not None:
        nbytes = max(nbytes, workspace_size(None, *extra_ws_for))
    ws = alloc_workspace(nbytes, device)
    return DeviceDraft(cfg, weights, views, tensors, kv_len, last_tok, h_prev, hist, w.B, w.N, m.vocab, m.d_t, ws)


@dataclasses.dataclass
class DeviceNextn:
    """A NextN drafter on the device: weights, its own KV (k, v tensors, written
    by every run), the catch-up rows and the step inputs of one call."""
    cfg: Config
    weights: Weights
    tensors: dict
    k: object
    v: object
    view: KVView
    kv_len: object
    n_cu: object
    cu_tok: object
    cu_h: object
    last_tok: object
    h_prev: object
    B: int
    N: int
    V: int
    d: int
    ws: object

    def run(self, out_drafts, out_h_last=None, out_logits=None, out_conf=None, stream=None):
        nextn_draft(self.cfg, self.weights, self.view, self.kv_len, self.last_tok, self.h_prev, out_drafts, self.ws,
                    n_cu=self.n_cu, cu_tok=self.cu_tok, cu_h=self.cu_h, out_h_last=out_h_last,
                    out_logits=out_logits, out_conf=out_conf, stream=stream)


def upload_nextn(w, device="cuda") -> DeviceNextn:
    """Upload a ``synth.NextnWorkload``: the weights, a copy of its drafter KV
    and the call's inputs."""
    import torch
    m = w.model
    cfg = make_config(m.d, m.d, 1, m.n_q_heads, m.head_dim, m.n_kv_heads, m.d_ff, m.vocab, wdtype=m.dtype,
                      rms_eps=m.rms_eps, attn_scale=m.attn_scale, emb_scale=m.emb_scale,
                      logit_softcap=m.logit_softcap, wquant=m.wquant)
    tensors = {}
    for n, a in w.weights.items():
        if m.wquant != "none" and a.dtype == np.float32 and a.ndim == 2:
            # a quantised projection: codes and block scales by the library's host quantiser
            q, d = quantize(a, m.wquant)
            tensors[n] = torch.from_numpy(q).to(device)
            tensors[n + ".scale"] = torch.from_numpy(d.view(np.int16)).to(device)
        else:
            tensors[n] = to_device(a, device=device)
    weights = make_nextn_weights(tensors)
    k, v = to_device(w.dkv["k"], device=device), to_device(w.dkv["v"], device=device)
    view = make_view(k, v, w.dkv["cap"], 0, w.dkv["rope_theta"])
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
    M = w.M
    cu_tok = i32(w.cu_tok) if M > 0 else None
    cu_h = f32(w.cu_h) if M > 0 else None
    ws = alloc_workspace(workspace_size(cfg, w.B, w.N, m.vocab), device)
    return DeviceNextn(cfg, weights, tensors, k, v, view, i32(w.kv_len), i32(w.n_cu), cu_tok, cu_h,
                       i32(w.last_tok), f32(w.h_prev), w.B, w.N, m.vocab, m.d, ws)
