"""The C ABI without a GPU: the library loads, exports every symbol that
include/kda.h declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_41_gb300 as kda
from gated_delta_rule_41_gb300 import build as kbuild
from gated_delta_rule_41_gb300.kda import KdaDims

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "kda_chunk_fwd" in names and "kda_recurrent_step" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/kda.h but not exported"


def test_status_strings(lib):
    for code in range(8):
        s = lib.kda_status_str(code)
        assert s and s != b"unknown status"
    assert lib.kda_status_str(99) == b"unknown status"
    assert lib.kda_version() >= 10000


def dims(**kw):
    base = dict(B=2, T=128, H=2, HV=4, K=64, V=64, chunk_size=64, scale=0.125, dtype=1, impl=0)
    base.update(kw)
    return KdaDims(**base)


def test_workspace_sizes(lib):
    d = dims()
    fwd = lib.kda_chunk_workspace_bytes(ctypes.byref(d), 0)
    bwd = lib.kda_chunk_workspace_bytes(ctypes.byref(d), 1)
    assert 0 < fwd < bwd
    assert fwd % 256 == 0 and bwd % 256 == 0
    # chunk 128: the SIMT kernels (AUTO or SIMT), not the tensor cores
    c128 = dims(T=256, chunk_size=128)
    assert lib.kda_chunk_workspace_bytes(ctypes.byref(c128), 1) > 0
    assert lib.kda_chunk_workspace_bytes(ctypes.byref(dims(T=256, chunk_size=128, impl=1)), 0) > 0
    assert lib.kda_chunk_workspace_bytes(ctypes.byref(dims(T=256, chunk_size=128, impl=2)), 0) == 0
    for bad in (dims(T=100), dims(HV=3), dims(K=256), dims(chunk_size=48), dims(dtype=7),
                dims(impl=9)):
        assert lib.kda_chunk_workspace_bytes(ctypes.byref(bad), 0) == 0


FAKE = ctypes.c_void_p(1 << 20)       # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p((1 << 20) + 1)


def fwd(lib, d, ptrs=None, ws=None, nws=0, final=0, ht=None):
    p = ptrs or [FAKE] * 6
    return lib.kda_chunk_fwd(ctypes.byref(d), p[0], p[1], p[2], p[3], p[4], None, p[5], final,
                             ht, ws, nws, None)


def test_validation_errors(lib):
    assert fwd(lib, dims(T=100)) == 2                   # T % chunk
    assert fwd(lib, dims(HV=3)) == 2                    # HV % H
    assert fwd(lib, dims(K=256)) == 3                   # K > 128
    assert fwd(lib, dims(chunk_size=8)) == 3            # chunk size
    assert fwd(lib, dims(impl=5)) == 1
    assert fwd(lib, dims(), ptrs=[FAKE, None, FAKE, FAKE, FAKE, FAKE]) == 1
    assert fwd(lib, dims(), ptrs=[FAKE, MISALIGNED, FAKE, FAKE, FAKE, FAKE]) == 4
    assert fwd(lib, dims(), final=1, ht=None) == 1      # final state requested, no buffer
    assert fwd(lib, dims()) == 5                        # workspace missing
    assert fwd(lib, dims(K=48, impl=1)) == 3            # SIMT needs K | 256
    d = dims()
    bwd = lib.kda_chunk_bwd(ctypes.byref(d), *([FAKE] * 5), None, FAKE, None,
                            *([FAKE] * 5), None, None, 0, None)
    assert bwd == 5
    st = lib.kda_recurrent_step(ctypes.byref(dims(HV=3)), *([FAKE] * 7), None)
    assert st == 2


def test_size_limits(lib):
    """B * HV * T at 2^30 (32-bit tile coordinates) is refused before any
    pointer is looked at; just below it only the workspace is missing."""
    big = dims(B=8192, HV=4, T=32768)                   # 2^13 * 4 * 2^15 = 2^30
    assert fwd(lib, big, ptrs=[None] * 6) == 3
    assert lib.kda_chunk_workspace_bytes(ctypes.byref(big), 0) == 0
    assert fwd(lib, dims(B=8192, HV=4, T=16384)) == 5
    assert lib.kda_chunk_workspace_bytes(ctypes.byref(dims(B=8192, HV=4, T=16384)), 0) > 0
    # packed sequences count their padded chunk slots
    vl = dims(B=1, HV=4, T=(1 << 28) - 64 * 1000)
    assert lib.kda_chunk_workspace_bytes_varlen(ctypes.byref(vl), 1000, 0) == 0
    assert lib.kda_chunk_workspace_bytes_varlen(ctypes.byref(vl), 999, 0) > 0
    assert lib.kda_chunk_workspace_bytes(ctypes.byref(dims(B=65536, HV=1, H=1, T=64)), 0) == 0


def test_build_flags_target_sm103a():
    assert "arch=compute_103a,code=sm_103a" in kbuild.ARCH
