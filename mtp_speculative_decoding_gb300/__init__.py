"""Thin Python binding of libmtp.so (the C ABI declared in include/mtp.h).

Argument marshalling only: every step of the draft block and the verifiers
runs in the library's CUDA kernels.  PyTorch supplies device memory and the
current stream.  There is no fallback: if the compiled library is missing or
no CUDA device is present, the calls raise.
"""
from __future__ import annotations

import ctypes as C
import os
import platform
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", platform.machine(), "libmtp.so")

MTP_OK = 0
MTP_ERR_ARG = -1
MTP_ERR_UNSUPPORTED = -2
MTP_ERR_WORKSPACE = -3
MTP_ERR_CUDA = -4
MTP_ERR_TIMEOUT = -5
MTP_ERR_CAPACITY = -6
MTP_DTYPE_F32 = 0
MTP_DTYPE_BF16 = 1
MTP_WQ_NONE = 0
MTP_WQ_Q8_0 = 1
MTP_WQ_Q4_0 = 2
MTP_MAX_BLOCKS = 8
MTP_MAX_VIEWS = 4
MTP_MAX_BATCH = 64
MTP_MAX_VERIFY_BATCH = 65536
MTP_MAX_CATCHUP = 16

# every entry point include/mtp.h declares
EXPORTS = ("mtp_workspace_size", "mtp_draft_block", "mtp_verify_greedy", "mtp_verify_sample",
           "mtp_sample_drafts", "mtp_quantize_q8_0", "mtp_last_error", "mtp_strerror", "mtp_debug_barrier_timeout",
           "mtp_verify_greedy_noalloc", "mtp_nextn_draft", "mtp_quantize_q4_0")


class MTPError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


class Config(C.Structure):
    _fields_ = [("d_t", C.c_int32), ("d_a", C.c_int32), ("n_blocks", C.c_int32), ("n_q_heads", C.c_int32),
                ("head_dim", C.c_int32), ("n_kv_heads", C.c_int32), ("d_ff", C.c_int32), ("vocab", C.c_int32),
                ("wdtype", C.c_int32), ("rms_eps", C.c_float), ("attn_scale", C.c_float),
                ("emb_scale", C.c_float), ("logit_softcap", C.c_float), ("n_centroids", C.c_int32),
                ("centroid_top_k", C.c_int32), ("wquant", C.c_int32), ("pad_", C.c_int32)]


class BlockWeights(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("w_q", C.c_void_p), ("q_norm", C.c_void_p), ("w_o", C.c_void_p),
                ("post_attn_norm", C.c_void_p), ("pre_ffn_norm", C.c_void_p), ("w_gate", C.c_void_p),
                ("w_up", C.c_void_p), ("w_down", C.c_void_p), ("post_ffn_norm", C.c_void_p),
                ("kv_view", C.c_int32), ("pad_", C.c_int32), ("w_q_scale", C.c_void_p), ("w_o_scale", C.c_void_p),
                ("w_gate_scale", C.c_void_p), ("w_up_scale", C.c_void_p), ("w_down_scale", C.c_void_p),
                ("k_norm", C.c_void_p)]


class Weights(C.Structure):
    _fields_ = [("tok_embd", C.c_void_p), ("norm_e", C.c_void_p), ("norm_h", C.c_void_p), ("w_pre", C.c_void_p),
                ("final_norm", C.c_void_p), ("w_post", C.c_void_p), ("blk", BlockWeights * MTP_MAX_BLOCKS),
                ("centroids", C.c_void_p), ("token_ordering", C.c_void_p), ("w_pre_scale", C.c_void_p),
                ("w_post_scale", C.c_void_p)]


class KVView(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("stride_b", C.c_int64), ("stride_h", C.c_int64),
                ("stride_t", C.c_int64), ("cap", C.c_int32), ("window", C.c_int32), ("rope_theta", C.c_float),
                ("sink", C.c_int32)]


class SampleParams(C.Structure):
    _fields_ = [("temp", C.c_float), ("top_p", C.c_float), ("min_p", C.c_float), ("rep_penalty", C.c_float),
                ("presence_penalty", C.c_float), ("top_k", C.c_int32)]


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "or python -m mtp_speculative_decoding_gb300.build")
            L = C.CDLL(LIB_PATH)
            P, I, Z = C.c_void_p, C.c_int, C.c_size_t
            L.mtp_workspace_size.argtypes = [P, I, I, I]
            L.mtp_workspace_size.restype = Z
            L.mtp_draft_block.argtypes = [P, P, P, I, P, I, I, P, P, P, C.c_uint64, C.c_uint64, P, I, P, P, P, P, P, Z,
                                          P]
            L.mtp_draft_block.restype = I
            L.mtp_verify_greedy.argtypes = [P, I, I, I, I, P, P, P, P, Z, P]
            L.mtp_verify_greedy.restype = I
            L.mtp_verify_sample.argtypes = [P, P, I, I, I, I, P, P, I, P, C.c_uint64, C.c_uint64, P, P, P, Z, P]
            L.mtp_verify_sample.restype = I
            L.mtp_last_error.argtypes = [P, P]
            L.mtp_last_error.restype = I
            L.mtp_strerror.argtypes = [I]
            L.mtp_strerror.restype = C.c_char_p
            L.mtp_debug_barrier_timeout.argtypes = [P, Z, I, P]
            L.mtp_debug_barrier_timeout.restype = I
            L.mtp_sample_drafts.argtypes = [P, I, I, I, I, P, I, P, C.c_uint64, C.c_uint64, P, P, Z, P]
            L.mtp_sample_drafts.restype = I
            L.mtp_verify_greedy_noalloc.argtypes = [P, I, I, I, I, P, P, P, P]
            L.mtp_verify_greedy_noalloc.restype = I
            L.mtp_nextn_draft.argtypes = [P, P, P, P, I, I, P, P, P, I, P, P, P, P, P, P, P, Z, P]
            L.mtp_nextn_draft.restype = I
            L.mtp_quantize_q8_0.argtypes = [P, C.c_int64, C.c_int64, P, P]
            L.mtp_quantize_q4_0.argtypes = [P, C.c_int64, C.c_int64, P, P]
            L.mtp_quantize_q4_0.restype = I
            L.mtp_quantize_q8_0.restype = I
            _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().mtp_strerror(int(code)).decode()
    except Exception:  # library not loadable: still give a readable message
        return f"error {code}"


def _check(rc: int, what: str) -> None:
    if rc != MTP_OK:
        raise MTPError(rc, what)


def _ptr(t):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _require_cuda(*tensors):
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError("every tensor argument must live on the CUDA device")


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return MTP_DTYPE_BF16
    if t.dtype == torch.float32:
        return MTP_DTYPE_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


# ----------------------------------------------------------------------------
# configuration
# ----------------------------------------------------------------------------

def make_config(d_t, d_a, n_blocks, n_q_heads, head_dim, n_kv_heads, d_ff, vocab, wdtype="bf16",
                rms_eps=1e-6, attn_scale=None, emb_scale=None, logit_softcap=0.0, n_centroids=0,
                centroid_top_k=0, wquant="none") -> Config:
    # None -> 0: the library's documented defaults (1/sqrt(head_dim), sqrt(d_t))
    return Config(d_t, d_a, n_blocks, n_q_heads, head_dim, n_kv_heads, d_ff, vocab,
                  MTP_DTYPE_BF16 if wdtype == "bf16" else MTP_DTYPE_F32, rms_eps,
                  0.0 if attn_scale is None else attn_scale, 0.0 if emb_scale is None else emb_scale,
                  logit_softcap, n_centroids, centroid_top_k,
                  {"q8_0": MTP_WQ_Q8_0, "q4_0": MTP_WQ_Q4_0}.get(wquant, MTP_WQ_NONE), 0)


def quantize_q8_0(w):
    """Q8_0 codes (int8 [rows, cols]) and block scales (binary16 bits, uint16
    [rows, cols / 32]) of an fp32 matrix, by mtp_quantize_q8_0 (host)."""
    import numpy as np
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    q = np.empty((rows, cols), dtype=np.int8)
    d = np.empty((rows, cols // 32 if cols % 32 == 0 else 0), dtype=np.uint16)
    rc = lib().mtp_quantize_q8_0(w.ctypes.data_as(C.c_void_p), rows, cols, q.ctypes.data_as(C.c_void_p),
                                 d.ctypes.data_as(C.c_void_p))
    if rc != MTP_OK:
        raise MTPError(rc, "mtp_quantize_q8_0")
    return q, d


def quantize_q4_0(w):
    """Q4_0 codes (uint8 [rows, cols / 2], two per byte) and block scales
    (binary16 bits, uint16 [rows, cols / 32]) of an fp32 matrix, by
    mtp_quantize_q4_0 (host)."""
    import numpy as np
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    q = np.empty((rows, cols // 2), dtype=np.uint8)
    d = np.empty((rows, cols // 32 if cols % 32 == 0 else 0), dtype=np.uint16)
    rc = lib().mtp_quantize_q4_0(w.ctypes.data_as(C.c_void_p), rows, cols, q.ctypes.data_as(C.c_void_p),
                                 d.ctypes.data_as(C.c_void_p))
    if rc != MTP_OK:
        raise MTPError(rc, "mtp_quantize_q4_0")
    return q, d


def quantize(w, wquant: str):
    """Codes and block scales of an fp32 projection in the format wquant names."""
    if wquant == "q8_0":
        return quantize_q8_0(w)
    if wquant == "q4_0":
        return quantize_q4_0(w)
    raise ValueError(wquant)


def workspace_size(cfg: Config | None, B: int, N: int, V: int) -> int:
    n = lib().mtp_workspace_size(C.byref(cfg) if cfg is not None else None, B, N, V)
    if n == 0:
        raise MTPError(MTP_ERR_ARG, "mtp_workspace_size")
    return int(n)


def alloc_workspace(nbytes: int, device="cuda"):
    """A device buffer usable as workspace (PyTorch allocations are 256-byte aligned)."""
    import torch
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------
# draft block
# ----------------------------------------------------------------------------

GLOBAL_TENSORS = ("tok_embd", "norm_e", "norm_h", "w_pre", "final_norm", "w_post")
BLOCK_TENSORS = ("attn_norm", "w_q", "q_norm", "w_o", "post_attn_norm", "pre_ffn_norm",
                 "w_gate", "w_up", "w_down", "post_ffn_norm")


def make_weights(tensors: dict, n_blocks: int, block_view) -> Weights:
    """Pack device tensors (keys: GLOBAL_TENSORS, 'blk{i}.<name>' and, for a
    centroid-routed head, 'centroids' and 'token_ordering') into mtp_weights."""
    w = Weights()
    for n in GLOBAL_TENSORS:
        setattr(w, n, tensors[n].data_ptr())
    for n in ("centroids", "token_ordering"):
        if n in tensors:
            setattr(w, n, tensors[n].data_ptr())
    for n in ("w_pre", "w_post"):   # Q8_0 block scales, when the model has them
        if n + ".scale" in tensors:
            setattr(w, n + "_scale", tensors[n + ".scale"].data_ptr())
    for i in range(n_blocks):
        b = w.blk[i]
        for n in BLOCK_TENSORS:
            setattr(b, n, tensors[f"blk{i}.{n}"].data_ptr())
            if f"blk{i}.{n}.scale" in tensors:
                setattr(b, n + "_scale", tensors[f"blk{i}.{n}.scale"].data_ptr())
        b.kv_view = int(block_view[i])
    return w


def make_view(k, v, cap: int, window: int, rope_theta: float, sink: int = 0) -> KVView:
    """k, v: [B, n_kv_heads, cap, head_dim] device tensors (head_dim contiguous);
    sink: attention-sink positions read with a window (see mtp_kv_view)."""
    assert k.shape == v.shape and k.stride() == v.stride() and k.stride(-1) == 1
    sb, sh, st, _ = k.stride()
    return KVView(k.data_ptr(), v.data_ptr(), sb, sh, st, cap, window, rope_theta, sink)


def draft_block(cfg: Config, weights: Weights, views, kv_len, last_tok, h_prev, out_drafts, ws,
                out_h_last=None, out_logits=None, sample=None, seed: int = 0, offset: int = 0, hist=None,
                stream=None, out_conf=None) -> None:
    """Launch mtp_draft_block on the current stream (asynchronous).  out_conf
    [B, N] fp32 (optional) receives each step's top-1 softmax probability."""
    _require_cuda(kv_len, last_tok, h_prev, out_drafts, ws, out_h_last, out_logits, hist, out_conf)
    B, N = out_drafts.shape
    arr = (KVView * len(views))(*views)
    sp = SampleParams(*sample) if sample is not None else None
    H = 0 if hist is None else int(hist.shape[1])
    rc = lib().mtp_draft_block(C.byref(cfg), C.byref(weights), arr, len(views), _ptr(kv_len), B, N,
                               _ptr(last_tok), _ptr(h_prev), C.byref(sp) if sp is not None else None,
                               seed, offset, _ptr(hist), H, _ptr(out_drafts), _ptr(out_h_last),
                               _ptr(out_logits), _ptr(out_conf), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "mtp_draft_block")


# ----------------------------------------------------------------------------
# the dense NextN drafter
# ----------------------------------------------------------------------------

# NextN tensor names -> the mtp_weights / mtp_block_weights fields they fill
NEXTN_FIELDS = {"tok_embd": "tok_embd", "enorm": "norm_e", "hnorm": "norm_h", "eh_proj": "w_pre",
                "head_norm": "final_norm"}
NEXTN_BLOCK_FIELDS = {"attn_norm": "attn_norm", "w_qkv": "w_q", "q_norm": "q_norm", "k_norm": "k_norm",
                      "w_o": "w_o", "ffn_norm": "pre_ffn_norm", "w_gate": "w_gate", "w_up": "w_up",
                      "w_down": "w_down"}


def make_nextn_weights(tensors: dict) -> Weights:
    """Pack the NextN drafter's device tensors (keys: NEXTN_FIELDS and
    NEXTN_BLOCK_FIELDS, plus '<name>.scale' for quantised projections) into
    mtp_weights: eh_proj is w_pre, head_norm is final_norm, the fused query /
    key / value projection is blk[0].w_q."""
    w = Weights()
    for n, f in NEXTN_FIELDS.items():
        setattr(w, f, tensors[n].data_ptr())
        if n + ".scale" in tensors:
            setattr(w, f + "_scale", tensors[n + ".scale"].data_ptr())
    for n, f in NEXTN_BLOCK_FIELDS.items():
        setattr(w.blk[0], f, tensors[n].data_ptr())
        if n + ".scale" in tensors:
            setattr(w.blk[0], f + "_scale", tensors[n + ".scale"].data_ptr())
    return w


def nextn_draft(cfg: Config, weights: Weights, dkv: KVView, kv_len, last_tok, h_prev, out_drafts, ws,
                n_cu=None, cu_tok=None, cu_h=None, out_h_last=None, out_logits=None, out_conf=None,
                stream=None) -> None:
    """Launch mtp_nextn_draft on the current stream (asynchronous): the
    catch-up rows (cu_tok [B, M] int32, cu_h [B, M, d] fp32, n_cu [B] int32),
    then out_drafts.shape[1] draft steps; writes the drafter's KV in dkv."""
    _require_cuda(kv_len, last_tok, h_prev, out_drafts, ws, n_cu, cu_tok, cu_h, out_h_last, out_logits, out_conf)
    B, N = out_drafts.shape
    M = 0 if cu_tok is None else int(cu_tok.shape[1])
    rc = lib().mtp_nextn_draft(C.byref(cfg), C.byref(weights), C.byref(dkv), _ptr(kv_len), B, N, _ptr(n_cu),
                               _ptr(cu_tok), _ptr(cu_h), M, _ptr(last_tok), _ptr(h_prev), _ptr(out_drafts),
                               _ptr(out_h_last), _ptr(out_logits), _ptr(out_conf), _ptr(ws), ws.numel(),
                               _stream(stream))
    _check(rc, "mtp_nextn_draft")


# ----------------------------------------------------------------------------
# verify
# ----------------------------------------------------------------------------

def verify_greedy(logits, drafts, out_tokens, out_n_accept, ws, stream=None) -> None:
    """logits [B, 1+N, V] (bf16 or fp32), drafts [B, N] int32 -> out_tokens [B, 1+N], out_n_accept [B]."""
    _require_cuda(logits, drafts, out_tokens, out_n_accept, ws)
    B, R, V = logits.shape
    rc = lib().mtp_verify_greedy(_ptr(logits), _dtype_code(logits), B, R - 1, V, _ptr(drafts),
                                 _ptr(out_tokens), _ptr(out_n_accept), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "mtp_verify_greedy")


def verify_greedy_noalloc(logits, drafts, out_tokens, out_n_accept, stream=None) -> None:
    """Greedy verify through the library's built-in scratch (no workspace, no
    allocation): for callers that may not allocate device memory.  Calls on
    overlapping streams race; B * (1 + N) <= 480."""
    _require_cuda(logits, drafts, out_tokens, out_n_accept)
    B, R, V = logits.shape
    rc = lib().mtp_verify_greedy_noalloc(_ptr(logits), _dtype_code(logits), B, R - 1, V, _ptr(drafts),
                                         _ptr(out_tokens), _ptr(out_n_accept), _stream(stream))
    _check(rc, "mtp_verify_greedy_noalloc")


def verify_sample(tgt_logits, dft_logits, drafts, hist, params, seed: int, offset: int, out_tokens,
                  out_n_accept, ws, stream=None) -> None:
    """params: (temp, top_p, min_p, rep_penalty, presence_penalty, top_k) or an object with those fields."""
    _require_cuda(tgt_logits, dft_logits, drafts, hist, out_tokens, out_n_accept, ws)
    B, R, V = tgt_logits.shape
    sp = _sample_params(params)
    H = 0 if hist is None else int(hist.shape[1])
    rc = lib().mtp_verify_sample(_ptr(tgt_logits), _ptr(dft_logits), _dtype_code(tgt_logits), B, R - 1, V,
                                 _ptr(drafts), _ptr(hist), H, C.byref(sp), seed, offset, _ptr(out_tokens),
                                 _ptr(out_n_accept), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "mtp_verify_sample")


def _sample_params(params) -> SampleParams:
    if hasattr(params, "temp"):
        params = (params.temp, params.top_p, params.min_p, params.rep_penalty,
                  getattr(params, "presence_penalty", 0.0), getattr(params, "top_k", 0))
    return SampleParams(*params)


def sample_drafts(dft_logits, hist, params, seed: int, offset: int, out_drafts, ws, stream=None) -> None:
    """Draws of a sampling drafter: out_drafts[b, i] ~ sample_dist(dft_logits[b, i]) (mtp_sample_drafts)."""
    _require_cuda(dft_logits, hist, out_drafts, ws)
    B, N, V = dft_logits.shape
    sp = _sample_params(params)
    H = 0 if hist is None else int(hist.shape[1])
    rc = lib().mtp_sample_drafts(_ptr(dft_logits), _dtype_code(dft_logits), B, N, V, _ptr(hist), H, C.byref(sp),
                                 seed, offset, _ptr(out_drafts), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "mtp_sample_drafts")


def last_error(ws, stream=None) -> int:
    """Device status word of the last call on `ws` (synchronizes the stream)."""
    return int(lib().mtp_last_error(_ptr(ws), _stream(stream)))


def debug_barrier_timeout(ws, timeout_us: int, stream=None) -> None:
    _check(lib().mtp_debug_barrier_timeout(_ptr(ws), ws.numel(), int(timeout_us), _stream(stream)),
           "mtp_debug_barrier_timeout")
