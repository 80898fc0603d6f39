"""The allocation-free forward (kda_chunk_fwd_noalloc) against the regular
workspace forward (kda_chunk_fwd with the SIMT kernels) and against the
float64 oracle, through the C ABI.

It exists for callers that cannot allocate device memory where they run the
scan (graph capture, fixed memory pools); its scratch is a 32 MiB device
array inside the library.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

import gated_delta_rule_41_gb300 as kda
from gated_delta_rule_41_gb300 import inputs as I
from gated_delta_rule_41_gb300.kda import _ptr, _stream, make_dims, KdaDims
from parity_util import assert_close, oracle_chunk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_41_gb300 import build
    build.build()
    lib = kda.load_library()
    P = ctypes.c_void_p
    lib.kda_chunk_fwd_noalloc.argtypes = [ctypes.POINTER(KdaDims), P, P, P, P, P, P, P,
                                          ctypes.c_int, P, P]
    lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
    return lib


def _noalloc(lib, t, chunk):
    dims = make_dims(t["q"], t["v"], chunk, None, "simt")
    o = torch.empty_like(t["v"])
    ht = torch.empty(dims.B, dims.HV, dims.K, dims.V, dtype=torch.float32, device="cuda")
    st = lib.kda_chunk_fwd_noalloc(ctypes.byref(dims), _ptr(t["q"]), _ptr(t["k"]), _ptr(t["v"]),
                                   _ptr(t["g"]), _ptr(t["beta"]), _ptr(t["h0"]), _ptr(o), 1,
                                   _ptr(ht), _stream(None))
    assert st == 0, f"kda_chunk_fwd_noalloc returned {st}"
    return o, ht


def test_noalloc_forward_matches_workspace_forward_twice(lib):
    w = I.SMALL_BF16  # B=4, T=512, H=HV=8, K=V=64, bf16, h0: 28 MiB of scratch
    for seed in (11, 12):  # two calls in a row, different inputs
        t = {n: (x.cuda() if x is not None else None)
             for n, x in I.make_chunk_inputs(w, seed=seed).items()}
        o_ref, ht_ref = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                          initial_state=t["h0"], output_final_state=True,
                                          chunk_size=w.chunk, impl="simt")
        o, ht = _noalloc(lib, t, w.chunk)
        torch.cuda.synchronize()
        kda.check()
        assert_close("o", o, o_ref.double().cpu().numpy(), w.dtype)
        assert_close("ht", ht, ht_ref.double().cpu().numpy(), w.dtype)
        ref = oracle_chunk({n: (x.cpu() if x is not None else None) for n, x in t.items()},
                           False)
        assert_close("o vs oracle", o, ref["o"], w.dtype)
        assert_close("ht vs oracle", ht, ref["ht"], w.dtype)


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    w = I.TRAIN_BF16  # about 1.3 GiB of scratch: over the 32 MiB limit
    dims = KdaDims(w.B, w.T, w.H, w.HV, w.K, w.V, w.chunk, w.K ** -0.5, 1, 1)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected before any launch
    st = lib.kda_chunk_fwd_noalloc(ctypes.byref(dims), fake, fake, fake, fake, fake, None, fake,
                                   0, None, None)
    assert st == 5  # KDA_ERR_WORKSPACE
