"""The C-ABI library builds for sm_103a, loads, and exports every entry point
include/mtp.h declares (no GPU needed: nothing is called)."""
import ctypes
import os
import re

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


def test_struct_layouts_match_header_sizes():
    # sizes the C compiler gives the header's structs (x86-64 and aarch64 agree)
    assert ctypes.sizeof(mtp.Config) == 13 * 4
    assert ctypes.sizeof(mtp.BlockWeights) == 10 * 8 + 8
    assert ctypes.sizeof(mtp.Weights) == 6 * 8 + mtp.MTP_MAX_BLOCKS * (10 * 8 + 8)
    assert ctypes.sizeof(mtp.KVView) == 2 * 8 + 3 * 8 + 4 * 4
    assert ctypes.sizeof(mtp.SampleParams) == 6 * 4


def test_workspace_size_host_only():
    mtp_build.build()
    cfg = mtp.make_config(5120, 1024, 4, 16, 256, 4, 4096, 262144)
    n = mtp.workspace_size(cfg, 1, 3, 262144)
    assert n > 0 and n % 256 == 0
    assert mtp.workspace_size(None, 32, 3, 248320) > 0
    with pytest.raises(mtp.MTPError):
        mtp.workspace_size(cfg, 65, 3, 262144)
    bad = mtp.make_config(5120, 1024, 4, 16, 96, 4, 4096, 262144)   # head_dim 96 unsupported
    with pytest.raises(mtp.MTPError):
        mtp.workspace_size(bad, 1, 3, 262144)
