"""Python access to the plain CPU oracle (``mtp_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg use it; the CUDA library never does.  The oracle
is compiled with gcc on first use (``build()``) and loaded through ctypes.  It
shares no code with the CUDA path; both take their inputs from ``synth``.
"""
from __future__ import annotations

import ctypes as C
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mtp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", platform.machine(), "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-D_DEFAULT_SOURCE", "-shared", "-fPIC", "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


class Model(C.Structure):
    _fields_ = [("d_t", C.c_int32), ("d_a", C.c_int32), ("n_blocks", C.c_int32),
                ("n_q_heads", C.c_int32), ("head_dim", C.c_int32), ("n_kv_heads", C.c_int32),
                ("d_ff", C.c_int32), ("vocab", C.c_int32), ("wbf16", C.c_int32), ("n_centroids", C.c_int32),
                ("centroid_top_k", C.c_int32), ("kv_bf16", C.c_int32),
                ("rms_eps", C.c_double), ("attn_scale", C.c_double), ("emb_scale", C.c_double),
                ("logit_softcap", C.c_double)]


class View(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("stride_b", C.c_int64),
                ("stride_h", C.c_int64), ("stride_t", C.c_int64), ("cap", C.c_int32),
                ("window", C.c_int32), ("sink", C.c_int32), ("pad_", C.c_int32), ("rope_theta", C.c_double)]


class SampleParams(C.Structure):
    _fields_ = [("temp", C.c_double), ("top_p", C.c_double), ("min_p", C.c_double),
                ("rep_penalty", C.c_double), ("presence_penalty", C.c_double),
                ("top_k", C.c_int32), ("pad_", C.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _declare(_lib)
    return _lib


def _declare(L):
    P, I, D, U64 = C.c_void_p, C.c_int, C.c_double, C.c_uint64
    L.orc_rmsnorm.argtypes = [P, I, P, D, P]
    L.orc_matvec.argtypes = [P, I, I, I, P, P]
    L.orc_gelu_tanh.argtypes = [D]
    L.orc_gelu_tanh.restype = D
    L.orc_rope_neox.argtypes = [P, I, C.c_int64, D]
    L.orc_argmax_f64.argtypes = [P, C.c_int64]
    L.orc_argmax_f64.restype = C.c_int64
    L.orc_attend_head.argtypes = [P, P, I, I, I, I, D, I, P]
    L.orc_philox4x32_10.argtypes = [P, P, P]
    L.orc_uniform.argtypes = [U64, U64, C.c_uint32, C.c_uint32, C.c_uint32]
    L.orc_uniform.restype = D
    L.orc_sample_dist.argtypes = [P, I, P, I, P, P, P, P, P]
    L.orc_sample_dist.restype = I
    L.orc_pick.argtypes = [P, P, I, D, D, P]
    L.orc_pick.restype = C.c_int32
    L.orc_draft_step.argtypes = [P, P, P, P, I, I, P, I, P, P, P, P, P]
    L.orc_draft_step.restype = I
    L.orc_draft_block.argtypes = [P, P, P, P, I, I, I, P, P, P, P, U64, U64, I, P, I, P, P, P, P, P, P, P]
    L.orc_centroid_head.argtypes = [P, P, P, P, P, P, P, P]
    L.orc_centroid_head.restype = I
    L.orc_quantize_q8_0.argtypes = [P, C.c_int64, C.c_int64, P, P]
    L.orc_dequantize_q8_0.argtypes = [P, P, C.c_int64, C.c_int64, P]
    L.orc_quantize_q4_0.argtypes = [P, C.c_int64, C.c_int64, P, P]
    L.orc_dequantize_q4_0.argtypes = [P, P, C.c_int64, C.c_int64, P]
    L.orc_top1_prob.argtypes = [P, C.c_int64]
    L.orc_top1_prob.restype = D
    L.orc_draft_block.restype = I
    L.orc_verify_greedy.argtypes = [P, I, I, I, I, P, P, P]
    L.orc_verify_sample.argtypes = [P, P, I, I, I, I, P, P, I, P, U64, U64, P, P, P]
    L.orc_sample_drafts.argtypes = [P, I, I, I, I, P, I, P, U64, U64, P, P]
    L.orc_silu.argtypes = [D]
    L.orc_silu.restype = D
    L.orc_to_bf16.argtypes = [D]
    L.orc_to_bf16.restype = C.c_uint16
    L.orc_nextn_draft.argtypes = [P, P, P, I, I, P, I, P, P, P, P, P, P, P, P, P, P, P]
    L.orc_nextn_draft.restype = I
    L.orc_set_threads.argtypes = [I]
    L.orc_num_threads.restype = I


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on (the CPU baseline's single-core run)."""
    lib().orc_set_threads(int(n))


# ----------------------------------------------------------------------------
# building blocks (exposed for the pins)
# ----------------------------------------------------------------------------

def rmsnorm(x, g=None, eps=1e-6):
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = None if g is None else np.ascontiguousarray(g, dtype=np.float32)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), x.size, _p(g), eps, _p(y))
    return y


def matvec(W, x, bf16=False):
    W = np.ascontiguousarray(W)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(W.shape[0], dtype=np.float64)
    lib().orc_matvec(_p(W), W.shape[0], W.shape[1], int(bf16), _p(x), _p(y))
    return y


def gelu_tanh(x):
    return np.array([lib().orc_gelu_tanh(float(v)) for v in np.ravel(x)]).reshape(np.shape(x))


def rope_neox(q, pos, theta):
    q = np.array(q, dtype=np.float64, copy=True)
    lib().orc_rope_neox(_p(q), q.size, int(pos), float(theta))
    return q


def argmax(z):
    z = np.ascontiguousarray(z, dtype=np.float64)
    return int(lib().orc_argmax_f64(_p(z), z.size))


def attend_head(q, k, v, b, g, kv_len, window=0, scale=None, bf16=False, sink=0):
    """k, v: [B, Hkv, cap, hd] arrays (fp32, or uint16 bf16 bits with bf16=True)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    B, H, cap, hd = k.shape
    vw = View(_p(k).value, _p(v).value, H * cap * hd, cap * hd, hd, cap, window, sink, 0, 0.0)
    out = np.empty(hd, dtype=np.float64)
    sc = 1.0 / np.sqrt(hd) if scale is None else scale
    lib().orc_attend_head(_p(q), C.byref(vw), b, g, hd, kv_len, sc, int(bf16), _p(out))
    return out


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    o = np.empty(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(o))
    return o


def uniform(seed, offset, b, i, purpose):
    return float(lib().orc_uniform(seed, offset, b, i, purpose))


def make_params(sp) -> SampleParams:
    return SampleParams(float(sp.temp), float(sp.top_p), float(sp.min_p), float(sp.rep_penalty),
                        float(getattr(sp, "presence_penalty", 0.0)), int(getattr(sp, "top_k", 0)), 0)


def sample_dist(z, pen, sp):
    """Returns (ids, weights, wsum, margin) of sample_dist(z) in (weight desc, id asc) order."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    pen = np.ascontiguousarray(np.asarray(pen, dtype=np.int32).reshape(-1))
    V = z.size
    ids = np.empty(V, dtype=np.int32)
    w = np.empty(V, dtype=np.float64)
    ws = C.c_double()
    mg = C.c_double()
    prm = make_params(sp)
    n = lib().orc_sample_dist(_p(z), V, _p(pen), pen.size, C.byref(prm), _p(ids), _p(w),
                              C.byref(ws), C.byref(mg))
    return ids[:n].copy(), w[:n].copy(), ws.value, mg.value


def quantize_q8_0(w):
    """Q8_0 codes (int8 [rows, cols]) and block scales (binary16 bits [rows, cols / 32]) of an fp32 matrix."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    if cols % 32:
        raise ValueError("Q8_0 needs a multiple of 32 columns")
    q = np.empty((rows, cols), dtype=np.int8)
    d = np.empty((rows, cols // 32), dtype=np.uint16)
    lib().orc_quantize_q8_0(_p(w), rows, cols, _p(q), _p(d))
    return q, d


def dequantize_q8_0(q, d):
    """The fp32 weights Q8_0 codes and scales stand for."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = np.ascontiguousarray(d, dtype=np.uint16)
    rows, cols = q.shape
    w = np.empty((rows, cols), dtype=np.float32)
    lib().orc_dequantize_q8_0(_p(q), _p(d), rows, cols, _p(w))
    return w


def quantize_q4_0(w):
    """Q4_0 codes (uint8 [rows, cols / 2], two per byte) and block scales
    (binary16 bits [rows, cols / 32]) of an fp32 matrix (ggml's scale rule)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    if cols % 32:
        raise ValueError("Q4_0 needs a multiple of 32 columns")
    q = np.empty((rows, cols // 2), dtype=np.uint8)
    d = np.empty((rows, cols // 32), dtype=np.uint16)
    lib().orc_quantize_q4_0(_p(w), rows, cols, _p(q), _p(d))
    return q, d


def dequantize_q4_0(q, d):
    """The fp32 weights Q4_0 codes and scales stand for."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    d = np.ascontiguousarray(d, dtype=np.uint16)
    rows, cols = q.shape[0], q.shape[1] * 2
    w = np.empty((rows, cols), dtype=np.float32)
    lib().orc_dequantize_q4_0(_p(q), _p(d), rows, cols, _p(w))
    return w


def top1_prob(z):
    """The softmax probability of the largest logit (NaN entries left out)."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    return float(lib().orc_top1_prob(_p(z), z.size))


def pick(ids, w, wsum, u):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    mg = C.c_double()
    r = lib().orc_pick(_p(ids), _p(w), ids.size, float(wsum), float(u), C.byref(mg))
    return int(r), mg.value


# ----------------------------------------------------------------------------
# draft block
# ----------------------------------------------------------------------------

GLOBAL_ORDER = ("tok_embd", "norm_e", "norm_h", "w_pre", "final_norm", "w_post", "centroids", "token_ordering")
BLOCK_ORDER = ("attn_norm", "w_q", "q_norm", "w_o", "post_attn_norm", "pre_ffn_norm",
               "w_gate", "w_up", "w_down", "post_ffn_norm")


def _model(m) -> Model:
    bf = 1 if m.dtype == "bf16" else 0
    return Model(m.d_t, m.d_a, m.n_blocks, m.n_q_heads, m.head_dim, m.n_kv_heads, m.d_ff, m.vocab,
                 bf, getattr(m, "n_centroids", 0), getattr(m, "centroid_top_k", 0), bf,
                 m.rms_eps, m.attn_scale, m.emb_scale, m.logit_softcap)


def centroid_head(m, centroids, ordering, tok_embd, h, full=False):
    """The centroid-routed head's full logit row [V] (f64) for one hidden state h [d_t];
    with ``full``, (row, cgap, centroid logits [n_c]), cgap the set margin
    relative to the centroid logits' standard deviation.

    ``m``: a model spec with n_centroids / centroid_top_k / vocab / d_t / dtype /
    logit_softcap; matrices fp32, or uint16 bf16 bits when m.dtype == 'bf16'."""
    c = np.ascontiguousarray(centroids)
    o = np.ascontiguousarray(ordering, dtype=np.int32)
    e = np.ascontiguousarray(tok_embd)
    h = np.ascontiguousarray(h, dtype=np.float64)
    z = np.empty(m.vocab, dtype=np.float64)
    mdl = _model(m)
    gap = C.c_double()
    cl = np.empty(max(1, m.n_centroids), dtype=np.float64)
    if lib().orc_centroid_head(C.byref(mdl), _p(c), _p(o), _p(e), _p(h), _p(z), C.byref(gap), _p(cl)) != 0:
        raise ValueError("oracle centroid head rejected its inputs")
    return (z, gap.value, cl) if full else z


def _projection_names(m):
    return ("w_pre", "w_post") + tuple(f"blk{i}.{n}" for i in range(m.n_blocks)
                                       for n in ("w_q", "w_o", "w_gate", "w_up", "w_down"))


_DERIVED: dict = {}   # id(source array) -> (source, derived): widened or dequantised copies, reused


def _derived(a, kind):
    hit = _DERIVED.get((id(a), kind))
    if hit is not None and hit[0] is a:
        return hit[1]
    if kind == "widen":
        out = np.ascontiguousarray((a.astype(np.uint32) << 16).view(np.float32)) if a.dtype == np.uint16 else a
    elif kind == "q4_0":
        out = dequantize_q4_0(*quantize_q4_0(a))
    else:
        out = dequantize_q8_0(*quantize_q8_0(a))
    if len(_DERIVED) > 64:
        _DERIVED.clear()
    _DERIVED[(id(a), kind)] = (a, out)
    return out


def _widen(a):
    """bf16 bit patterns (uint16) to fp32, exactly; other arrays unchanged."""
    return _derived(a, "widen")


class _Bound:
    """ctypes views of one workload, restricted to one sequence b (or all)."""

    def __init__(self, w, b=None):
        m = w.model
        self.keep = []
        self.model = _model(m)
        names = list(GLOBAL_ORDER) + [f"blk{i}.{n}" for i in range(m.n_blocks) for n in BLOCK_ORDER]
        # the centroid head's tensors exist only for centroid-head models (NULL otherwise)
        arrs = [np.ascontiguousarray(w.weights[n]) if n in w.weights else None for n in names]
        quant = getattr(m, "wquant", "none")
        q8 = quant in ("q8_0", "q4_0")
        if q8:
            # Q8_0 / Q4_0 projections: the weights the codes stand for (exact in
            # fp32); the table and the KV widened from bf16 exactly, and the step
            # run in fp32
            proj = set(_projection_names(m))
            arrs = [None if a is None else
                    _derived(a, quant) if n in proj else
                    _widen(a) for n, a in zip(names, arrs)]
            self.model.wbf16 = 0
        self.keep += [a for a in arrs if a is not None]
        self.tensors = (C.c_void_p * len(arrs))(*[None if a is None else a.ctypes.data for a in arrs])
        self.block_view = np.ascontiguousarray(np.asarray(m.block_view, dtype=np.int32))
        views = []
        esz = 2 if m.dtype == "bf16" and not q8 else 4
        for vd in w.views:
            k, v = (_widen(vd["k"]), _widen(vd["v"])) if q8 else (vd["k"], vd["v"])
            Bv, H, cap, hd = k.shape
            off = 0 if b is None else b * H * cap * hd * esz
            views.append(View(k.ctypes.data + off, v.ctypes.data + off, H * cap * hd, cap * hd, hd,
                              cap, vd["window"], vd.get("sink", 0), 0, vd["rope_theta"]))
            self.keep += [k, v]
        self.views = (View * len(views))(*views)
        self.n_views = len(views)
        sl = slice(None) if b is None else slice(b, b + 1)
        self.B = w.B if b is None else 1
        self.kv_len = np.ascontiguousarray(w.kv_len[sl], dtype=np.int32)
        self.last_tok = np.ascontiguousarray(w.last_tok[sl], dtype=np.int32)
        self.h_prev = np.ascontiguousarray(w.h_prev[sl], dtype=np.float32)
        self.hist = np.ascontiguousarray(w.hist[sl], dtype=np.int32)


def draft_block(w, sample=None, seed=0, offset=0, force=None, seqs=None, want_logits=True):
    """Run the oracle draft block over sequences ``seqs`` (default: all).

    ``force`` ([B, N] int32, optional) teacher-forces the token consumed at
    step k+1 to force[b, k] instead of the oracle's own pick.
    Returns dict(drafts [S,N] int32, h_last [S,d_t] f64, logits [S,N,V] f64 or
    None, margin [S,N] f64, conf [S,N] f64: each step's top-1 softmax
    probability, cgap [S,N] f64: the centroid-routed head's set margin, +inf
    for the dense head) for the S selected sequences, in ``seqs`` order.
    """
    L = lib()
    m = w.model
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    S, N, V = len(seqs), w.N, m.vocab
    out_d = np.empty((S, N), dtype=np.int32)
    out_h = np.empty((S, m.d_t), dtype=np.float64)
    out_z = np.empty((S, N, V), dtype=np.float64) if want_logits else None
    out_m = np.empty((S, N), dtype=np.float64)
    out_c = np.empty((S, N), dtype=np.float64)
    out_g = np.empty((S, N), dtype=np.float64)
    prm = make_params(sample) if sample is not None else None
    for j, b in enumerate(seqs):
        bd = _Bound(w, b)
        f = None if force is None else np.ascontiguousarray(force[b:b + 1], dtype=np.int32)
        d = np.empty((1, N), dtype=np.int32)
        h = np.empty((1, m.d_t), dtype=np.float64)
        z = np.empty((1, N, V), dtype=np.float64) if want_logits else None
        mg = np.empty((1, N), dtype=np.float64)
        cf = np.empty((1, N), dtype=np.float64)
        cg = np.empty((1, N), dtype=np.float64)
        rc = L.orc_draft_block(C.byref(bd.model), bd.tensors, _p(bd.block_view), bd.views, bd.n_views,
                               1, N, _p(bd.kv_len), _p(bd.last_tok), _p(bd.h_prev),
                               C.byref(prm) if prm is not None else None, seed, offset, b,
                               _p(bd.hist), bd.hist.shape[1], _p(f), _p(d), _p(h), _p(z), _p(mg), _p(cf), _p(cg))
        if rc != 0:
            raise ValueError(f"oracle draft block rejected its inputs (rc={rc})")
        out_d[j], out_h[j], out_m[j], out_c[j], out_g[j] = d[0], h[0], mg[0], cf[0], cg[0]
        if want_logits:
            out_z[j] = z[0]
    return dict(drafts=out_d, h_last=out_h, logits=out_z, margin=out_m, conf=out_c, cgap=out_g)


def draft_step(w, b, step, tok, h_prev):
    """One oracle step for sequence b: returns (h_next [d_t] f64, logits [V] f64)."""
    L = lib()
    bd = _Bound(w, b)
    m = w.model
    tk = np.array([tok], dtype=np.int32)
    h = np.ascontiguousarray(np.asarray(h_prev, dtype=np.float64).reshape(1, m.d_t))
    hn = np.empty((1, m.d_t), dtype=np.float64)
    z = np.empty((1, m.vocab), dtype=np.float64)
    rc = L.orc_draft_step(C.byref(bd.model), bd.tensors, _p(bd.block_view), bd.views, bd.n_views, 1,
                          _p(bd.kv_len), step, _p(tk), _p(h), _p(hn), _p(z), None)
    if rc != 0:
        raise ValueError("oracle draft step rejected its inputs")
    return hn[0], z[0]


# ----------------------------------------------------------------------------
# the dense NextN drafter
# ----------------------------------------------------------------------------

NEXTN_ORDER = ("tok_embd", "enorm", "hnorm", "eh_proj", "head_norm", "attn_norm", "w_qkv", "q_norm",
               "k_norm", "w_o", "ffn_norm", "w_gate", "w_up", "w_down")
NEXTN_PROJECTIONS = ("eh_proj", "w_qkv", "w_o", "w_gate", "w_up", "w_down")


def silu(x):
    return np.array([lib().orc_silu(float(v)) for v in np.ravel(x)]).reshape(np.shape(x))


def to_bf16(x):
    """Real values rounded once to bf16 (nearest, ties to even): uint16 bit patterns."""
    return np.array([lib().orc_to_bf16(float(v)) for v in np.ravel(x)], dtype=np.uint16).reshape(np.shape(x))


def nextn_draft(w, force=None, seqs=None, want_logits=True, dkv=None):
    """One drafting call of the NextN drafter over sequences ``seqs`` (default:
    all): the catch-up rows, then w.N draft steps (see orc_nextn_draft).

    ``force`` ([B, N] int32) teacher-forces the token consumed at step k+1.
    ``dkv`` (optional dict with k, v) replaces the workload's drafter KV as the
    starting state.  The workload's arrays are never modified: the call works
    on a copy of the KV and returns it.  Returns dict(drafts [S,N], h_last
    [S,d] f64, logits [S,N,V] f64 or None, margin [S,N], conf [S,N], k, v (the
    drafter KV after the call, [B, Hkv, cap, hd], all sequences)).
    """
    L = lib()
    m = w.model
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    S, N, V, d = len(seqs), w.N, m.vocab, m.d
    src = w.dkv if dkv is None else dkv
    k = np.array(src["k"], copy=True, order="C")
    v = np.array(src["v"], copy=True, order="C")
    Bv, H, cap, hd = k.shape
    arrs = [np.ascontiguousarray(w.weights[n]) for n in NEXTN_ORDER]
    mdl = _model(m)
    quant = getattr(m, "wquant", "none")
    if quant in ("q8_0", "q4_0"):
        # quantised projections: the weights the codes stand for, the table
        # widened, the step in fp32; the drafter's KV stays bf16
        proj = set(NEXTN_PROJECTIONS)
        arrs = [_derived(a, quant) if n in proj else _widen(a) for n, a in zip(NEXTN_ORDER, arrs)]
        mdl.wbf16 = 0
    tensors = (C.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    esz = k.itemsize
    out = dict(drafts=np.empty((S, N), dtype=np.int32), h_last=np.empty((S, d)), margin=np.empty((S, N)),
               conf=np.empty((S, N)), logits=np.empty((S, N, V)) if want_logits else None)
    M = max(1, w.M)
    cu_tok = np.zeros((w.B, M), dtype=np.int32)
    cu_h = np.zeros((w.B, M, d), dtype=np.float32)
    cu_tok[:, :w.M] = w.cu_tok
    cu_h[:, :w.M] = w.cu_h
    for j, b in enumerate(seqs):
        off = b * H * cap * hd * esz
        vw = View(k.ctypes.data + off, v.ctypes.data + off, H * cap * hd, cap * hd, hd, cap, 0, 0, 0,
                  float(w.dkv["rope_theta"]))
        f = None if force is None else np.ascontiguousarray(force[b:b + 1], dtype=np.int32)
        dd = np.empty((1, N), dtype=np.int32)
        h = np.empty((1, d))
        z = np.empty((1, N, V)) if want_logits else None
        mg, cf = np.empty((1, N)), np.empty((1, N))
        rc = L.orc_nextn_draft(C.byref(mdl), tensors, C.byref(vw), 1, N,
                               _p(np.ascontiguousarray(w.kv_len[b:b + 1], dtype=np.int32)), M,
                               _p(np.ascontiguousarray(w.n_cu[b:b + 1], dtype=np.int32)),
                               _p(np.ascontiguousarray(cu_tok[b:b + 1])), _p(np.ascontiguousarray(cu_h[b:b + 1])),
                               _p(np.ascontiguousarray(w.last_tok[b:b + 1], dtype=np.int32)),
                               _p(np.ascontiguousarray(w.h_prev[b:b + 1], dtype=np.float32)), _p(f), _p(dd), _p(h),
                               _p(z), _p(mg), _p(cf))
        if rc != 0:
            raise ValueError(f"oracle NextN drafter rejected its inputs (rc={rc})")
        out["drafts"][j], out["h_last"][j], out["margin"][j], out["conf"][j] = dd[0], h[0], mg[0], cf[0]
        if want_logits:
            out["logits"][j] = z[0]
    out["k"], out["v"] = k, v
    return out


# ----------------------------------------------------------------------------
# verify
# ----------------------------------------------------------------------------

def verify_greedy(logits, dtype, drafts):
    logits = np.ascontiguousarray(logits)
    drafts = np.ascontiguousarray(drafts, dtype=np.int32)
    B, R, V = logits.shape
    N = R - 1
    out = np.empty((B, N + 1), dtype=np.int32)
    n_acc = np.empty(B, dtype=np.int32)
    lib().orc_verify_greedy(_p(logits), 1 if dtype == "bf16" else 0, B, N, V, _p(drafts), _p(out), _p(n_acc))
    return out, n_acc


def verify_sample(target, draft, dtype, drafts, hist, params, seed, offset):
    """Returns (out_tokens [B,1+N], n_accept [B], margin [B])."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    drafts = np.ascontiguousarray(drafts, dtype=np.int32)
    hist = np.ascontiguousarray(hist, dtype=np.int32)
    B, R, V = target.shape
    N = R - 1
    H = hist.shape[1] if hist.ndim == 2 else 0
    out = np.empty((B, N + 1), dtype=np.int32)
    n_acc = np.empty(B, dtype=np.int32)
    mg = np.empty(B, dtype=np.float64)
    prm = make_params(params)
    lib().orc_verify_sample(_p(target), _p(draft), 1 if dtype == "bf16" else 0, B, N, V, _p(drafts),
                            _p(hist), H, C.byref(prm), seed, offset, _p(out), _p(n_acc), _p(mg))
    return out, n_acc, mg


def sample_drafts(draft, dtype, hist, params, seed, offset):
    """Draws of a sampling drafter: drafts[b, i] ~ sample_dist(draft row (b, i)) with
    penalty set hist[b] + drafts[b, :i] and the uniform of (b, i, purpose 0).
    Returns (drafts [B, N] int32, margin [B])."""
    draft = np.ascontiguousarray(draft)
    hist = np.ascontiguousarray(hist, dtype=np.int32)
    B, N, V = draft.shape
    H = hist.shape[1] if hist.ndim == 2 else 0
    out = np.empty((B, N), dtype=np.int32)
    mg = np.empty(B, dtype=np.float64)
    prm = make_params(params)
    lib().orc_sample_drafts(_p(draft), 1 if dtype == "bf16" else 0, B, N, V, _p(hist), H, C.byref(prm),
                            seed, offset, _p(out), _p(mg))
    return out, mg
