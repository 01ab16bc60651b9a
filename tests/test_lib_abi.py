"""The C-ABI library builds, loads and exports every entry point declared in include/gla.h.

CPU only: no call here launches device work.  Argument checks that fail before
any CUDA call are exercised with null / misaligned pointers.
"""
import ctypes
import os
import re

import pytest

from gated_linear_rnn_gb300 import build as B
from gated_linear_rnn_gb300 import gla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gla.h")


@pytest.fixture(scope="module")
def lib():
    B.build_library()
    return gla.load()


def declared_entry_points():
    text = open(HEADER).read()
    return re.findall(r"GLA_API\s+[\w\s\*]*?\b(gla_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for required in ("gla_chunk_fwd", "gla_decode_step", "gla_last_device_status", "gla_status_str"):
        assert required in names
    assert len(names) == len(set(names))


def test_every_declared_symbol_is_exported(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name
        assert name in gla.SIGNATURES, f"binding lacks {name}"


def test_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gla.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_entry_points())


def test_status_strings_and_version(lib):
    assert gla.gla_version() >= 100
    for code, name in gla.STATUS.items():
        s = gla.gla_status_str(code)
        assert isinstance(s, str) and s and s != "unknown status", name
    assert gla.gla_status_str(12345) == "unknown status"


def test_null_arguments_rejected_on_the_host(lib):
    P = ctypes.c_void_p
    rc = lib.gla_chunk_fwd(None, None, None, None, None, None, None, 1, 1, 1, 16, 16, 128, None, None)
    assert rc == -1
    rc = lib.gla_chunk_fwd_f32(None, None, None, None, None, None, None, 1, 1, 1, 16, 16, 64, None, None)
    assert rc == -1
    rc = lib.gla_decode_step(None, None, None, None, None, None, 1, 1, 16, 16, None)
    assert rc == -1
    # non-positive sizes with non-null (never dereferenced) pointers
    fake = P(4096)
    rc = lib.gla_chunk_fwd(fake, fake, fake, fake, None, fake, None, 0, 1, 1, 16, 16, 128, None, None)
    assert rc == -1
    rc = lib.gla_decode_step(fake, fake, fake, fake, fake, fake, 1, -1, 16, 16, None)
    assert rc == -1


def test_unsupported_shapes_and_alignment_rejected_on_the_host(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    # dk not a multiple of 8
    assert lib.gla_chunk_fwd(fake, fake, fake, fake, None, fake, None, 1, 8, 1, 20, 64, 128, None, None) == -2
    # dv beyond the decode limit
    assert lib.gla_decode_step(fake, fake, fake, fake, fake, fake, 1, 1, 16, 2048, None) == -2
    # misaligned pointer
    odd = P(4096 + 8)
    assert lib.gla_chunk_fwd(odd, fake, fake, fake, None, fake, None, 1, 8, 1, 16, 16, 128, None, None) == -3
    assert lib.gla_decode_step(fake, fake, fake, fake, odd, fake, 1, 1, 16, 16, None) == -3


def test_host_entry_rejects_bad_arguments_before_any_copy(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    # null inputs, non-positive sizes, unsupported head sizes and chunk lengths
    assert lib.gla_chunk_fwd_host(None, fake, fake, fake, None, fake, None, 1, 1, 1, 16, 16, 128, None) == -1
    assert lib.gla_chunk_fwd_host(fake, fake, fake, None, None, fake, None, 1, 1, 1, 16, 16, 128, None) == -1
    assert lib.gla_chunk_fwd_host(fake, fake, fake, fake, None, fake, None, 1, 0, 1, 16, 16, 128, None) == -1
    assert lib.gla_chunk_fwd_host(fake, fake, fake, fake, None, fake, None, 1, 8, 1, 20, 64, 128, None) == -2
    assert lib.gla_chunk_fwd_host(fake, fake, fake, fake, None, fake, None, 1, 8, 1, 64, 64, 48, None) == -2


def test_chunk_kernel_query_rejects_bad_arguments_on_the_host(lib):
    # unknown operation or dtype, then sizes no entry point takes; on a host without an sm_103 device
    # every valid query answers GLA_ERR_UNSUPPORTED
    assert lib.gla_chunk_kernel(3, 0, 96, 192, 128) == -1
    assert lib.gla_chunk_kernel(0, 2, 96, 192, 128) == -1
    assert lib.gla_chunk_kernel(0, 0, 20, 192, 128) == -2
    assert lib.gla_chunk_kernel(2, 0, 96, 192, 48) == -2
