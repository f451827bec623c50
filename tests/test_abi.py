"""The C-ABI library builds for sm_103a, loads, and exports every entry point
include/mtp.h declares (no GPU needed: nothing is called)."""
import ctypes
import os
import re
import subprocess

import pytest

import mtp_speculative_decoding_gb300 as mtp
from mtp_speculative_decoding_gb300 import build as mtp_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mtp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(mtp_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(mtp.EXPORTS)


def test_library_builds_and_exports_every_symbol():
    path = mtp_build.build()
    L = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(L, name), name


def test_binding_loads_library():
    mtp_build.build()
    L = mtp.lib()
    assert mtp.strerror(mtp.MTP_ERR_TIMEOUT) == "grid barrier timed out"
    assert mtp.strerror(0) == "ok"


_STRUCTS = (("mtp_config", "Config"), ("mtp_block_weights", "BlockWeights"), ("mtp_weights", "Weights"),
            ("mtp_kv_view", "KVView"), ("mtp_sample_params", "SampleParams"))


def test_struct_layouts_match_header(tmp_path):
    """Every binding struct has the size and field offsets the C compiler gives
    the header's struct of the same name."""
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "mtp.h"', "int main(void) {"]
    for cname, pname in _STRUCTS:
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in getattr(mtp, pname)._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for ln in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        *key, val = ln.split()
        got[tuple(key)] = int(val)
    for cname, pname in _STRUCTS:
        S = getattr(mtp, pname)
        assert got[(cname, "size")] == ctypes.sizeof(S), cname
        for f, _ in S._fields_:
            assert got[(cname, f)] == getattr(S, f).offset, (cname, f)


def test_workspace_size_host_only():
    mtp_build.build()
    cfg = mtp.make_config(5120, 1024, 4, 16, 256, 4, 4096, 262144)
    n = mtp.workspace_size(cfg, 1, 3, 262144)
    assert n > 0 and n % 256 == 0
    assert mtp.workspace_size(None, 32, 3, 248320) > 0
    with pytest.raises(mtp.MTPError):
        mtp.workspace_size(cfg, 65, 3, 262144)
    assert mtp.workspace_size(mtp.make_config(5120, 1024, 4, 16, 256, 4, 4096, 262144, attn_scale=0.0,
                                              emb_scale=0.0), 1, 3, 262144) == n   # 0: the defaults
    with pytest.raises(mtp.MTPError):
        mtp.workspace_size(mtp.make_config(5120, 1024, 4, 16, 256, 4, 4096, 262144, attn_scale=-1.0), 1, 3, 262144)
    bad = mtp.make_config(5120, 1024, 4, 16, 96, 4, 4096, 262144)   # head_dim 96 unsupported
    with pytest.raises(mtp.MTPError):
        mtp.workspace_size(bad, 1, 3, 262144)


def test_host_q8_0_quantiser_matches_the_oracle():
    """mtp_quantize_q8_0 (host code of the library) and the oracle's
    quantiser give the same codes and scales bit for bit (integer output of
    the same fp32 rule), over Gaussian rows, exact code multiples, zero
    blocks and extreme ranges."""
    import numpy as np
    import oracle
    import synth
    mtp_build.build()
    rng = np.random.default_rng(11)
    w = synth.normal(12, "hostq8", (96, 512), std=0.02)
    w[3, :32] = 0.0
    w[4] *= 1e-6
    w[5] *= 1e4
    w[6, :64] = np.arange(-32, 32, dtype=np.float32) * np.float32(2.0 ** -5)
    w[7] = rng.standard_normal(512).astype(np.float32) * 3e-8   # binary16 subnormal scales
    q1, d1 = mtp.quantize_q8_0(w)
    q2, d2 = oracle.quantize_q8_0(w)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(d1, d2)
    with pytest.raises(mtp.MTPError):
        mtp.quantize_q8_0(np.zeros((2, 48), dtype=np.float32))


def test_host_q4_0_quantiser_matches_the_oracle():
    """mtp_quantize_q4_0 (host code of the library) and the oracle's
    quantiser give the same codes and scales bit for bit, over Gaussian rows,
    code multiples of a power-of-two scale, zero blocks, opposite extremes of
    one magnitude (the clamp to 15), ties of the extreme, and extreme ranges."""
    import numpy as np
    import oracle
    import synth
    mtp_build.build()
    rng = np.random.default_rng(13)
    w = synth.normal(14, "hostq4", (96, 512), std=0.02)
    w[3, :32] = 0.0
    w[4] *= 1e-6
    w[5] *= 1e4
    w[6, :32] = (np.arange(32, dtype=np.float32) % 16 - 8) * np.float32(2.0 ** -5)
    w[7] = rng.standard_normal(512).astype(np.float32) * 3e-8
    w[8, :32] = 0.0
    w[8, 2], w[8, 30] = 0.5, -0.5                  # equal magnitudes: the first is the extreme
    q1, d1 = mtp.quantize_q4_0(w)
    q2, d2 = oracle.quantize_q4_0(w)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(d1, d2)
    with pytest.raises(mtp.MTPError):
        mtp.quantize_q4_0(np.zeros((2, 48), dtype=np.float32))


def test_nextn_host_checks_reject_before_any_device_work():
    """mtp_nextn_draft's argument checks return before the first CUDA call, so
    they run without a GPU: a NextN config needs d_a == d_t and one block, the
    drafter KV a plain view (window 0), at most MTP_MAX_CATCHUP catch-up rows,
    catch-up arrays when M > 0, and no sampling.  (Placeholder addresses: none
    is dereferenced.)"""
    import ctypes as C
    mtp_build.build()
    L = mtp.lib()
    fake = 1 << 20   # 16-byte aligned, never dereferenced

    def call(cfg, view, M=2, cu=True, kv_len=fake):
        w = mtp.Weights()
        w.tok_embd = w.norm_e = w.norm_h = w.w_pre = w.final_norm = fake
        b = w.blk[0]
        b.attn_norm = b.w_q = b.q_norm = b.k_norm = b.w_o = b.pre_ffn_norm = b.w_gate = b.w_up = b.w_down = fake
        return L.mtp_nextn_draft(C.byref(cfg), C.byref(w), C.byref(view), kv_len, 1, 3, fake,
                                 fake if cu else None, fake if cu else None, M, fake, fake, fake, None, None, None,
                                 fake, 1 << 30, None)

    good_view = mtp.KVView(fake, fake, 4 * 64 * 64, 64 * 64, 64, 64, 0, 1e4, 0)
    cfg = mtp.make_config(256, 256, 1, 4, 64, 2, 512, 1000)
    assert call(mtp.make_config(256, 128, 1, 4, 64, 2, 512, 1000), good_view) == mtp.MTP_ERR_ARG      # d_a != d_t
    assert call(mtp.make_config(256, 256, 2, 4, 64, 2, 512, 1000), good_view) == mtp.MTP_ERR_UNSUPPORTED
    assert call(cfg, mtp.KVView(fake, fake, 4 * 64 * 64, 64 * 64, 64, 64, 16, 1e4, 0)) == mtp.MTP_ERR_ARG  # window
    assert call(cfg, good_view, M=mtp.MTP_MAX_CATCHUP + 1) == mtp.MTP_ERR_ARG
    assert call(cfg, good_view, M=2, cu=False) == mtp.MTP_ERR_ARG                                      # no rows
    assert call(cfg, good_view, kv_len=None) == mtp.MTP_ERR_ARG                                        # no kv_len
