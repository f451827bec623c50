"""Seeded synthetic inputs for the MTP draft block and the verify-accept step.

This module only draws random numbers and arranges them into the shapes the
draft chain and the verifiers consume.  It holds none of the method's
arithmetic: the CPU oracle (``oracle/``) and the CUDA library
(``mtp_speculative_decoding_gb300``) both take their inputs from here and from
nowhere else, and neither side is imported by this module.

Shapes follow the model the pages describe (Gemma-4 assistant drafter, "Gemma 4
MTP -- Multi-Token Prediction speculative decoding", sections 3-5): a token
embedding table shared with the target, a pre-projection of the concatenated
[token embedding; target hidden state], L assistant blocks that cross-attend into
the target's last full-attention and last sliding-window KV layers, a
post-projection back to the backbone width and the tied LM head.  The dense
NextN drafter ("MTP decoding (--mtp)", "Requirements") is one block at the
backbone width with its own KV, fed through eh_proj, and the shared head.

Conventions
-----------
* bf16 tensors are returned as ``np.uint16`` bit patterns, rounded from fp32
  with round-to-nearest-even.  fp32 tensors are ``np.float32``.
* RMSNorm gains are always fp32 and are drawn as ``1 + N(0, 0.02)``.
* KV views are ``[B, n_kv_heads, cap, head_dim]`` ring buffers: position ``t``
  lives in slot ``t % cap``.  Every slot that does not hold a position the
  drafter may read (beyond ``kv_len`` or before the sliding window) is filled
  with NaN, so an over-read shows up as a NaN in the output.
* Every tensor gets its own random stream, keyed by (seed, tensor name, chunk),
  so its values do not depend on which other tensors were generated or on the
  number of worker threads.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os
import zlib

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
_CHUNK = 1 << 22  # elements per independent random stream


# ----------------------------------------------------------------------------
# random streams and bf16 rounding
# ----------------------------------------------------------------------------

def _stream(seed: int, name: str, chunk: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF, zlib.crc32(name.encode()), int(chunk)])
    return np.random.Generator(np.random.SFC64(ss))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    out = np.empty(a.shape, dtype=np.uint16)
    flat_u = u.reshape(-1)
    flat_o = out.reshape(-1)
    n = flat_u.size

    def conv(lo: int, hi: int) -> None:
        x = flat_u[lo:hi]
        bias = ((x >> 16) & 1) + np.uint32(0x7FFF)
        r = ((x + bias) >> 16).astype(np.uint16)
        nan = (x & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
        if nan.any():
            r[nan] = BF16_NAN
        flat_o[lo:hi] = r

    step = 1 << 24
    if n <= step:
        conv(0, n)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(lambda lo: conv(lo, min(n, lo + step)), range(0, n, step)))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """fp32 array of N(mean, std^2) values, one independent stream per chunk."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = _stream(seed, name, c)
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)
        if mean != 0.0:
            out[lo:hi] += np.float32(mean)

    nch = (n + _CHUNK - 1) // _CHUNK
    if nch <= 1:
        for c in range(nch):
            fill(c)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nch)))
    return out.reshape(shape)


def uniform_int(seed: int, name: str, shape, lo: int, hi: int) -> np.ndarray:
    """int32 array uniform in [lo, hi)."""
    g = _stream(seed, name, 0)
    return g.integers(lo, hi, size=shape, dtype=np.int64).astype(np.int32)


def permutation(seed: int, name: str, n: int) -> np.ndarray:
    """int32 uniformly random permutation of 0..n-1."""
    return _stream(seed, name, 0).permutation(n).astype(np.int32)


def _as_dtype(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(a)
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# model / workload description
# ----------------------------------------------------------------------------

BLOCK_TENSORS = ("attn_norm", "w_q", "q_norm", "w_o", "post_attn_norm",
                 "pre_ffn_norm", "w_gate", "w_up", "w_down", "post_ffn_norm")


@dataclasses.dataclass
class ModelSpec:
    d_t: int           # backbone (target) width
    d_a: int           # assistant width
    n_blocks: int
    n_q_heads: int
    head_dim: int
    n_kv_heads: int
    d_ff: int
    vocab: int
    dtype: str = "bf16"          # weights and KV: "f32" or "bf16"
    block_view: tuple = (0,)     # per block: index of the KV view it cross-attends
    rms_eps: float = 1e-6
    logit_softcap: float = 0.0
    n_centroids: int = 0         # > 0: centroid-routed LM head over n_centroids lists of vocab / n_centroids ids
    centroid_top_k: int = 0      # centroids whose lists are scored per step
    wquant: str = "none"         # "q8_0" / "q4_0": the projections are quantised (generated here in fp32, unrounded)

    @property
    def emb_scale(self) -> float:
        return math.sqrt(self.d_t)

    @property
    def attn_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def params(self) -> int:
        d_t, d_a, q, F = self.d_t, self.d_a, self.n_q_heads * self.head_dim, self.d_ff
        per_block = 2 * q * d_a + 3 * F * d_a
        return self.vocab * d_t + 2 * d_t * d_a + self.n_blocks * per_block + d_t * d_a


@dataclasses.dataclass
class ViewSpec:
    cap: int             # slots per (sequence, kv head)
    window: int          # 0 = full attention over [0, kv_len); W > 0 = last W positions
    rope_theta: float
    sink: int = 0        # with a window: positions [0, sink) kept beside it (slots 0..sink-1)


@dataclasses.dataclass
class DraftWorkload:
    name: str
    model: ModelSpec
    views_spec: list
    B: int
    N: int
    weights: dict        # name -> array; per-block tensors as "blk{i}.{name}"
    views: list          # list of dict(k, v, cap, window, rope_theta)
    kv_len: np.ndarray   # int32 [B]
    last_tok: np.ndarray  # int32 [B]
    h_prev: np.ndarray   # float32 [B, d_t]
    hist: np.ndarray     # int32 [B, H] (may be H = 0)

    def weight_bytes(self) -> int:
        return sum(int(a.nbytes) for a in self.weights.values())


def projection_names(m: ModelSpec) -> tuple:
    """The drafter's projection matrices (the ones a quantised model quantises)."""
    return ("w_pre", "w_post") + tuple(f"blk{i}.{n}" for i in range(m.n_blocks)
                                       for n in ("w_q", "w_o", "w_gate", "w_up", "w_down"))


def make_model_weights(m: ModelSpec, seed: int, std: float = 0.02) -> dict:
    q = m.n_q_heads * m.head_dim
    shapes = {
        "tok_embd": (m.vocab, m.d_t),
        "w_pre": (m.d_a, 2 * m.d_t),
        "w_post": (m.d_t, m.d_a),
    }
    norms = {"norm_e": m.d_t, "norm_h": m.d_t, "final_norm": m.d_a}
    for i in range(m.n_blocks):
        shapes[f"blk{i}.w_q"] = (q, m.d_a)
        shapes[f"blk{i}.w_o"] = (m.d_a, q)
        shapes[f"blk{i}.w_gate"] = (m.d_ff, m.d_a)
        shapes[f"blk{i}.w_up"] = (m.d_ff, m.d_a)
        shapes[f"blk{i}.w_down"] = (m.d_a, m.d_ff)
        norms[f"blk{i}.attn_norm"] = m.d_a
        norms[f"blk{i}.q_norm"] = m.head_dim
        norms[f"blk{i}.post_attn_norm"] = m.d_a
        norms[f"blk{i}.pre_ffn_norm"] = m.d_a
        norms[f"blk{i}.post_ffn_norm"] = m.d_a
    if m.n_centroids:
        shapes["centroids"] = (m.n_centroids, m.d_t)
    w = {}
    for name, shp in shapes.items():
        vals = normal(seed, name, shp, std=std)
        w[name] = vals if m.wquant != "none" and name in projection_names(m) else _as_dtype(vals, m.dtype)
    for name, n in norms.items():
        w[name] = normal(seed, name, (n,), std=std, mean=1.0)
    if m.n_centroids:
        # ordered embeddings: every token in exactly one centroid's list
        w["token_ordering"] = permutation(seed, "token_ordering", m.vocab)
    return w


def view_positions(window: int, kv_len: int, sink: int = 0) -> np.ndarray:
    """The positions a drafter reads: the window [lo, kv_len) and, with a
    window, the sink [0, min(sink, lo))."""
    lo = max(0, kv_len - window) if window > 0 else 0
    s0 = min(sink, lo) if window > 0 else 0
    return np.concatenate([np.arange(0, s0), np.arange(lo, kv_len)])


def view_slot(t: np.ndarray, cap: int, sink: int = 0) -> np.ndarray:
    """Slot of position t: t below the sink, then a ring over cap - sink slots."""
    t = np.asarray(t)
    return np.where(t < sink, t, sink + (t - sink) % max(1, cap - sink))


def view_valid_mask(cap: int, window: int, kv_len: int, sink: int = 0) -> np.ndarray:
    """bool [cap]: which slots hold a position the drafter may read."""
    mask = np.zeros(cap, dtype=bool)
    mask[view_slot(view_positions(window, kv_len, sink), cap, sink if window > 0 else 0)] = True
    return mask


def make_kv_view(m: ModelSpec, vs: ViewSpec, kv_len: np.ndarray, seed: int, tag: str) -> dict:
    B = kv_len.shape[0]
    shape = (B, m.n_kv_heads, vs.cap, m.head_dim)
    out = {}
    for which in ("k", "v"):
        vals = normal(seed, f"{tag}.{which}", shape, std=1.0)
        arr = _as_dtype(vals, m.dtype)
        for b in range(B):
            bad = ~view_valid_mask(vs.cap, vs.window, int(kv_len[b]), vs.sink)
            if m.dtype == "bf16":
                arr[b][:, bad, :] = BF16_NAN
            else:
                arr[b][:, bad, :] = np.nan
        out[which] = arr
    out.update(cap=vs.cap, window=vs.window, rope_theta=vs.rope_theta, sink=vs.sink)
    return out


_WEIGHT_CACHE: dict = {}


def cached_model_weights(m: ModelSpec, seed: int) -> dict:
    """make_model_weights, memoised for the last model (several workloads share one model)."""
    key = (dataclasses.astuple(m), seed)
    if key not in _WEIGHT_CACHE:
        _WEIGHT_CACHE.clear()
        _WEIGHT_CACHE[key] = make_model_weights(m, seed)
    return _WEIGHT_CACHE[key]


def make_draft_workload(name: str, m: ModelSpec, views_spec: list, B: int, N: int,
                        kv_len, seed: int, hist_len: int = 0, model_seed: int | None = None) -> DraftWorkload:
    kv_len = np.asarray(kv_len, dtype=np.int32).reshape(B)
    for vs in views_spec:
        need = vs.window + vs.sink if vs.window > 0 else int(kv_len.max())
        if need > vs.cap:
            raise ValueError(f"view cap {vs.cap} too small for {need} positions")
    weights = cached_model_weights(m, seed if model_seed is None else model_seed)
    views = [make_kv_view(m, vs, kv_len, seed, f"view{j}") for j, vs in enumerate(views_spec)]
    last_tok = uniform_int(seed, "last_tok", (B,), 0, m.vocab)
    h_prev = normal(seed, "h_prev", (B, m.d_t))
    hist = uniform_int(seed, "hist", (B, hist_len), 0, m.vocab)
    if hist_len:
        hist[:, -1] = last_tok  # the newest history entry is the token being consumed
    return DraftWorkload(name, m, views_spec, B, N, weights, views, kv_len, last_tok, h_prev, hist)


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

def _gemma_assistant(dtype: str = "bf16") -> ModelSpec:
    return ModelSpec(d_t=5120, d_a=1024, n_blocks=4, n_q_heads=16, head_dim=256, n_kv_heads=4,
                     d_ff=4096, vocab=262144, dtype=dtype, block_view=(0, 0, 0, 1))


def _edge_assistant() -> ModelSpec:
    """An Edge-shaped assistant with the centroid-routed head (synthetic sizes:
    the pages give the head's steps, not an Edge model's dimensions): 2048-wide
    backbone, 512-wide assistant, 4 blocks, 8 query heads x 256 against 2 KV
    heads, GeGLU 2048, the 262144-token table in 2048 lists of 128 ids, 32
    lists scored per step."""
    return ModelSpec(d_t=2048, d_a=512, n_blocks=4, n_q_heads=8, head_dim=256, n_kv_heads=2, d_ff=2048,
                     vocab=262144, dtype="bf16", block_view=(0, 0, 0, 1), n_centroids=2048, centroid_top_k=32)


def _gemma_views(full_cap: int) -> list:
    # view 0: the target's last sliding-window layer (bounded ring of 1536 cells, window 1024)
    # view 1: the target's last full-attention layer
    return [ViewSpec(cap=1536, window=1024, rope_theta=10000.0),
            ViewSpec(cap=full_cap, window=0, rope_theta=1000000.0)]


WORKLOADS = {
    0: "tiny-fp32-b1-n3",
    1: "gemma-assistant-bf16-b1-n3-ctx8192",
    2: "gemma-assistant-bf16-b16-n4-ragged2k-32k",
    3: "gemma-assistant-bf16-b64-n2-ctx4096",
    4: "verify-sample-b32-n3-v248320",
    5: "edge-centroid-bf16-b1-n3-ctx4096",
    6: "gemma-assistant-q8-b1-n3-ctx8192",
    7: "nextn-qwen-dense-bf16-b1-n3-kv4096-catchup2",
    8: "gemma-assistant-q4-b1-n3-ctx8192",
}


def workload_seed(cfg_id: int) -> int:
    return 1000 + int(cfg_id)


def make_draft_inputs(cfg_id: int, seed: int | None = None, B: int | None = None, sink: int = 0) -> DraftWorkload:
    """Draft-block inputs of one of the named workloads (0-3, 5).

    Workload 5 is the Edge-shaped model with the centroid-routed head, batch
    1, N = 3, a sliding layer (window 512) and a full layer of 4096 positions.
    Workload 6 is workload 1 with Q8_0 projections (the table and KV bf16),
    workload 8 the same with Q4_0 projections.

    ``B`` may shrink the batch (the first B sequences' lengths are kept) for
    parity runs at full model size.  ``sink`` > 0 keeps that many attention-
    sink positions beside the sliding window (workloads 1-3).
    """
    seed = workload_seed(cfg_id) if seed is None else seed
    name = WORKLOADS[cfg_id]
    if cfg_id == 0:
        m = ModelSpec(d_t=256, d_a=128, n_blocks=1, n_q_heads=4, head_dim=32, n_kv_heads=1,
                      d_ff=512, vocab=4096, dtype="f32", block_view=(0,))
        views = [ViewSpec(cap=128, window=0, rope_theta=1000000.0)]
        Bf, N, kv = 1, 3, np.array([128])
    elif cfg_id == 1:
        m, views = _gemma_assistant(), _gemma_views(8192)
        Bf, N, kv = 1, 3, np.array([8192])
    elif cfg_id == 2:
        m, views = _gemma_assistant(), _gemma_views(32768)
        Bf, N = 16, 4
        kv = uniform_int(seed, "kv_len", (Bf,), 2048, 32769)
    elif cfg_id == 3:
        m, views = _gemma_assistant(), _gemma_views(4096)
        Bf, N, kv = 64, 2, np.full(64, 4096)
    elif cfg_id in (6, 8):
        q = "q8_0" if cfg_id == 6 else "q4_0"
        m, views = dataclasses.replace(_gemma_assistant(), wquant=q), _gemma_views(8192)
        Bf, N, kv = 1, 3, np.array([8192])
    elif cfg_id == 5:
        m = _edge_assistant()
        views = [ViewSpec(cap=768, window=512, rope_theta=10000.0), ViewSpec(cap=4096, window=0, rope_theta=1000000.0)]
        Bf, N, kv = 1, 3, np.array([4096])
    else:
        raise ValueError("workload 4 has no draft block")
    B = Bf if B is None else B
    kv = np.resize(np.asarray(kv, dtype=np.int32), B) if B != Bf else kv
    if cfg_id == 2:
        views = [views[0], ViewSpec(cap=int(kv.max()), window=0, rope_theta=1e6)]
    if sink and cfg_id in (1, 2, 3):
        views = [ViewSpec(cap=views[0].cap, window=views[0].window, rope_theta=views[0].rope_theta, sink=sink)] + views[1:]
    # workloads 1-3 share one model ("same model as config 1"): its weights use seed 1001;
    # workloads 6 and 8 quantise that model's projections (the same fp32 draws)
    model_seed = workload_seed(1) if cfg_id in (1, 2, 3, 6, 8) else seed
    return make_draft_workload(name, m, views, B, N, kv, seed, hist_len=64, model_seed=model_seed)


# ----------------------------------------------------------------------------
# the dense NextN drafter ("MTP decoding (--mtp)", "Requirements"; "Fused
# NextN draft graph", "The two MTP lanes": its own block and its own KV)
# ----------------------------------------------------------------------------

NEXTN_TENSORS = ("tok_embd", "enorm", "hnorm", "eh_proj", "head_norm", "attn_norm", "w_qkv", "q_norm",
                 "k_norm", "w_o", "ffn_norm", "w_gate", "w_up", "w_down")
NEXTN_PROJECTIONS = ("eh_proj", "w_qkv", "w_o", "w_gate", "w_up", "w_down")


@dataclasses.dataclass
class NextnSpec:
    """A dense NextN drafter: one attention + SwiGLU block at the backbone width
    d with its own KV, fed [enorm(embedding); hnorm(hidden state)] through
    eh_proj, and the shared head (the tied table after head_norm)."""
    d: int
    n_q_heads: int
    head_dim: int
    n_kv_heads: int
    d_ff: int
    vocab: int
    dtype: str = "bf16"
    rms_eps: float = 1e-6
    logit_softcap: float = 0.0
    rope_theta: float = 1e7
    wquant: str = "none"         # "q8_0" / "q4_0": the projections quantised (generated here in fp32, unrounded)

    # the shapes the oracle's model record shares with the assistant
    @property
    def d_t(self) -> int:
        return self.d

    @property
    def d_a(self) -> int:
        return self.d

    n_blocks = 1
    n_centroids = 0
    centroid_top_k = 0

    @property
    def emb_scale(self) -> float:
        return 1.0

    @property
    def attn_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def params(self) -> int:
        d, F, hq = self.d, self.d_ff, self.n_q_heads * self.head_dim
        return self.vocab * d + 2 * d * d + self.qkv_rows * d + d * hq + 3 * F * d


@dataclasses.dataclass
class NextnWorkload:
    name: str
    model: NextnSpec
    B: int
    N: int
    M: int               # catch-up rows a sequence may bring (the width of cu_tok / cu_h)
    weights: dict        # NEXTN_TENSORS -> array
    dkv: dict            # the drafter's KV: k, v [B, Hkv, cap, hd], cap, rope_theta
    kv_len: np.ndarray   # int32 [B]: rows already in the drafter's KV
    n_cu: np.ndarray     # int32 [B]: catch-up rows of this call, 0..M
    cu_tok: np.ndarray   # int32 [B, M]: their tokens (rows j < n_cu[b] used)
    cu_h: np.ndarray     # float32 [B, M, d]: the target's hidden states paired with them
    last_tok: np.ndarray  # int32 [B]: the token the first draft step consumes
    h_prev: np.ndarray   # float32 [B, d]: the target's hidden state paired with it

    def weight_bytes(self) -> int:
        return sum(int(a.nbytes) for a in self.weights.values())


def make_nextn_weights(m: NextnSpec, seed: int, std: float = 0.02) -> dict:
    d, F, hq = m.d, m.d_ff, m.n_q_heads * m.head_dim
    shapes = {"tok_embd": (m.vocab, d), "eh_proj": (d, 2 * d), "w_qkv": (m.qkv_rows, d), "w_o": (d, hq),
              "w_gate": (F, d), "w_up": (F, d), "w_down": (d, F)}
    norms = {"enorm": d, "hnorm": d, "head_norm": d, "attn_norm": d, "ffn_norm": d,
             "q_norm": m.head_dim, "k_norm": m.head_dim}
    w = {}
    for name, shp in shapes.items():
        vals = normal(seed, "nextn." + name, shp, std=std)
        w[name] = vals if m.wquant != "none" and name in NEXTN_PROJECTIONS else _as_dtype(vals, m.dtype)
    for name, n in norms.items():
        w[name] = normal(seed, "nextn." + name, (n,), std=std, mean=1.0)
    return w


def make_nextn_workload(name: str, m: NextnSpec, B: int, N: int, M: int, kv_len, n_cu, seed: int,
                        cap: int | None = None, model_seed: int | None = None) -> NextnWorkload:
    """The drafter's KV holds kv_len[b] rows of N(0, 1) keys and values (what
    earlier calls wrote); every slot from kv_len[b] on is NaN, so a read of a
    row this call has not written shows up as a NaN."""
    kv_len = np.asarray(kv_len, dtype=np.int32).reshape(B)
    n_cu = np.asarray(n_cu, dtype=np.int32).reshape(B)
    need = int((kv_len + n_cu).max()) + N
    cap = need if cap is None else cap
    if need > cap or n_cu.min() < 0 or n_cu.max() > M:
        raise ValueError("drafter KV capacity or catch-up rows out of range")
    key = ("nextn", dataclasses.astuple(m), seed if model_seed is None else model_seed)
    if key not in _WEIGHT_CACHE:
        _WEIGHT_CACHE.clear()
        _WEIGHT_CACHE[key] = make_nextn_weights(m, seed if model_seed is None else model_seed)
    weights = _WEIGHT_CACHE[key]
    shape = (B, m.n_kv_heads, cap, m.head_dim)
    dkv = {}
    for which in ("k", "v"):
        arr = _as_dtype(normal(seed, "nextn.dkv." + which, shape), m.dtype)
        for b in range(B):
            arr[b][:, int(kv_len[b]):, :] = BF16_NAN if m.dtype == "bf16" else np.nan
        dkv[which] = arr
    dkv.update(cap=cap, rope_theta=m.rope_theta)
    cu_tok = uniform_int(seed, "nextn.cu_tok", (B, max(M, 1)), 0, m.vocab)[:, :M].copy()
    cu_h = normal(seed, "nextn.cu_h", (B, max(M, 1), m.d))[:, :M].copy()
    last_tok = uniform_int(seed, "nextn.last_tok", (B,), 0, m.vocab)
    h_prev = normal(seed, "nextn.h_prev", (B, m.d))
    return NextnWorkload(name, m, B, N, M, weights, dkv, kv_len, n_cu, cu_tok, cu_h, last_tok, h_prev)


def _qwen_nextn() -> NextnSpec:
    """A Qwen3.5-9B-shaped dense NextN block (synthetic sizes: the pages name
    the model family and its tensors, not their dimensions): width 4096, 16
    query heads x 256 against 4 KV heads, SwiGLU 12288, a 248320-token table."""
    return NextnSpec(d=4096, n_q_heads=16, head_dim=256, n_kv_heads=4, d_ff=12288, vocab=248320, dtype="bf16")


def make_nextn_inputs(cfg_id: int = 7, seed: int | None = None, B: int | None = None) -> NextnWorkload:
    """Workload 7: the Qwen-shaped NextN drafter, batch 1, N = 3 drafts, 4096
    rows already in its KV, two catch-up rows (the accepted drafts of the
    previous window) before the drafts."""
    if cfg_id != 7:
        raise ValueError("workload 7 is the NextN drafter")
    seed = workload_seed(cfg_id) if seed is None else seed
    B = 1 if B is None else B
    return make_nextn_workload(WORKLOADS[7], _qwen_nextn(), B, 3, 3, np.full(B, 4096), np.full(B, 2), seed)


# ----------------------------------------------------------------------------
# verify inputs
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class VerifyGreedyInputs:
    logits: np.ndarray   # [B, 1+N, V] float32 or uint16 (bf16 bits)
    dtype: str
    drafts: np.ndarray   # int32 [B, N]
    planted: np.ndarray  # int32 [B]: the accept length the inputs were built for


def plant_greedy_logits(logits32: np.ndarray, drafts: np.ndarray, planted: np.ndarray,
                        dtype: str) -> np.ndarray:
    """Make row i's largest value sit at drafts[i] for i < k, and not at drafts[k].

    Works on the values as stored (after bf16 rounding), so the planted rows'
    maxima are exact in the stored dtype.
    """
    B, R, V = logits32.shape
    N = R - 1
    store = _as_dtype(logits32, dtype)
    vals = bf16_bits_to_f32(store) if dtype == "bf16" else store
    for b in range(B):
        k = int(planted[b])
        for i in range(min(k, N)):
            top = float(np.nanmax(vals[b, i]))
            new = np.float32(top + 1.0)
            if dtype == "bf16":
                bits = f32_to_bf16_bits(np.array([new], dtype=np.float32))[0]
                store[b, i, drafts[b, i]] = bits
            else:
                store[b, i, drafts[b, i]] = new
        if k < N:
            row = vals[b, k]
            d = drafts[b, k]
            low = np.float32(float(np.nanmin(row)) - 1.0)
            if dtype == "bf16":
                store[b, k, d] = f32_to_bf16_bits(np.array([low], dtype=np.float32))[0]
            else:
                store[b, k, d] = low
    return store


def make_verify_greedy_inputs(cfg_id: int, seed: int | None = None, B: int | None = None,
                              N: int | None = None, V: int | None = None,
                              dtype: str | None = None) -> VerifyGreedyInputs:
    seed = workload_seed(cfg_id) if seed is None else seed
    defaults = {0: (1, 3, 4096, "f32"), 1: (1, 3, 262144, "bf16"), 2: (16, 4, 262144, "bf16"),
                3: (64, 2, 262144, "bf16"), 5: (1, 3, 262144, "bf16"), 6: (1, 3, 262144, "bf16"),
                7: (1, 3, 248320, "bf16"), 8: (1, 3, 262144, "bf16")}
    Bd, Nd, Vd, dd = defaults[cfg_id]
    B = Bd if B is None else B
    N = Nd if N is None else N
    V = Vd if V is None else V
    dtype = dd if dtype is None else dtype
    logits = normal(seed, "verify.logits", (B, N + 1, V))
    drafts = uniform_int(seed, "verify.drafts", (B, N), 0, V)
    planted = uniform_int(seed, "verify.planted", (B,), 0, N + 1)
    store = plant_greedy_logits(logits, drafts, planted, dtype)
    return VerifyGreedyInputs(store, dtype, drafts, planted)


@dataclasses.dataclass
class SampleParams:
    temp: float = 0.6
    top_p: float = 0.95
    min_p: float = 0.05
    rep_penalty: float = 1.08
    presence_penalty: float = 0.0
    top_k: int = 0


@dataclasses.dataclass
class VerifySampleInputs:
    target: np.ndarray   # [B, 1+N, V] (bf16 bits or fp32)
    draft: np.ndarray    # [B, N, V]
    dtype: str
    hist: np.ndarray     # int32 [B, H]; newest token last
    params: SampleParams
    seed: int
    offset: int
    drafts: np.ndarray | None = None   # int32 [B, N]: filled in by the caller's drafter


def make_verify_sample_inputs(seed: int | None = None, B: int = 32, N: int = 3, V: int = 248320,
                              H: int = 64, rho: float = 0.8, std: float = 2.0,
                              dtype: str = "bf16", params: SampleParams | None = None
                              ) -> VerifySampleInputs:
    """Target logits ~N(0, std^2); draft logits rho-correlated with the target rows.

    The drafted tokens are not part of these inputs: a sampling drafter draws
    them from its own distribution q_i = sample_dist(draft row i), which is
    arithmetic of the method, so the caller fills ``drafts`` in (the oracle's
    draws in the tests, the library's on the GPU).
    """
    seed = workload_seed(4) if seed is None else seed
    tgt = normal(seed, "vs.target", (B, N + 1, V), std=std)
    eps = normal(seed, "vs.eps", (B, N, V), std=std)
    dft = (np.float32(rho) * tgt[:, :N, :] + np.float32(math.sqrt(1 - rho * rho)) * eps)
    tgt_s, dft_s = _as_dtype(tgt, dtype), _as_dtype(dft, dtype)
    hist = uniform_int(seed, "vs.hist", (B, H), 0, V)
    return VerifySampleInputs(tgt_s, dft_s, dtype, hist, params or SampleParams(), seed=seed, offset=0)
