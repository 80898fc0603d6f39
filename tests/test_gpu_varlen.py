"""Packed variable-length sequences (kda_chunk_fwd_varlen / _bwd_varlen)
through the C ABI, against the float64 oracle run on each sequence on its
own: packing must not let one sequence see another, and each sequence's last
chunk may be partial."""
import numpy as np
import pytest
import torch

import gated_delta_rule_41_gb300 as kda
from gated_delta_rule_41_gb300 import inputs as I
from parity_util import assert_close, oracle_chunk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_41_gb300 import build
    build.build()


def packed_inputs(lengths, H, HV, K, V, dtype, seed, with_h0=True, with_dht=True,
                  normalize_qk=True):
    T = int(sum(lengths))
    w = I.Workload("varlen", 1, T, H, HV, K, V, 64, dtype, g_sigma=2.0, dht=False, seed=seed)
    inp = I.make_chunk_inputs(w, normalize_qk=normalize_qk)
    gen = torch.Generator().manual_seed(seed + 1000)
    n = len(lengths)
    inp["h0"] = 0.2 * torch.randn(n, HV, K, V, generator=gen) if with_h0 else None
    inp["dht"] = torch.randn(n, HV, K, V, generator=gen) if with_dht else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return inp, cu


def oracle_packed(inp, cu, want_bwd, qk_l2norm=False):
    """The oracle on every sequence alone, outputs and gradients put back in
    place (empty sequences: final state = initial state, dh0 = dht)."""
    T = inp["q"].shape[1]
    HV, V, K = inp["v"].shape[2], inp["v"].shape[3], inp["q"].shape[3]
    n = len(cu) - 1
    out = dict(o=np.zeros((1, T, HV, V)), ht=np.zeros((n, HV, K, V)))
    if want_bwd:
        for name, x in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta")):
            out[name] = np.zeros(tuple(inp[x].shape))
        out["dh0"] = np.zeros((n, HV, K, V))
    for s in range(n):
        a, e = int(cu[s]), int(cu[s + 1])
        h0 = None if inp["h0"] is None else inp["h0"][s:s + 1]
        dht = None if inp["dht"] is None else inp["dht"][s:s + 1]
        if e == a:
            out["ht"][s] = 0.0 if h0 is None else h0[0].double().numpy()
            if want_bwd:
                out["dh0"][s] = 0.0 if dht is None else dht[0].double().numpy()
            continue
        sl = {n_: inp[n_][:, a:e] for n_ in ("q", "k", "v", "g", "beta", "do")}
        r = oracle_chunk(dict(sl, h0=h0, dht=dht), want_bwd, qk_l2norm=qk_l2norm)
        out["o"][:, a:e] = r["o"]
        out["ht"][s] = r["ht"][0]
        if want_bwd:
            for name in ("dq", "dk", "dv", "dg", "dbeta"):
                out[name][:, a:e] = r[name]
            if h0 is not None:
                out["dh0"][s] = r["dh0"][0]
            elif dht is not None:
                out["dh0"][s] = 0.0
    return out


def run_packed(inp, cu, chunk, impl="auto", qk_l2norm=False):
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    cu_d = torch.from_numpy(cu).cuda()
    o, ht = kda.chunk_kda_fwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], cu_d,
                                     initial_state=t["h0"], output_final_state=True,
                                     chunk_size=chunk, impl=impl,
                                     use_qk_l2norm_in_kernel=qk_l2norm)
    res = dict(o=o, ht=ht)
    res.update(kda.chunk_kda_bwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], cu_d,
                                        dht=t["dht"], initial_state=t["h0"], chunk_size=chunk,
                                        impl=impl, use_qk_l2norm_in_kernel=qk_l2norm))
    torch.cuda.synchronize()
    kda.check()
    return res


def compare(res, ref, dtype, with_h0=True):
    for n in ("o", "ht", "dq", "dk", "dv", "dg", "dbeta"):
        assert_close(n, res[n], ref[n], dtype)
    if with_h0:
        assert_close("dh0", res["dh0"], ref["dh0"], dtype)


@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_varlen_fp32_gva_ragged_and_empty_sequences(chunk):
    lengths = [1, 37, 64, 100, 0, 130]
    inp, cu = packed_inputs(lengths, 2, 4, 32, 32, torch.float32, seed=61 + chunk)
    compare(run_packed(inp, cu, chunk), oracle_packed(inp, cu, True), torch.float32)


def test_varlen_bf16_k128():
    lengths = [200, 64, 7, 0, 129]
    inp, cu = packed_inputs(lengths, 2, 2, 128, 128, torch.bfloat16, seed=65, with_dht=False)
    compare(run_packed(inp, cu, 64), oracle_packed(inp, cu, True), torch.bfloat16)


def test_varlen_with_qk_l2norm_in_kernel():
    lengths = [50, 14, 77]
    inp, cu = packed_inputs(lengths, 1, 2, 64, 64, torch.float32, seed=66, normalize_qk=False)
    compare(run_packed(inp, cu, 32, qk_l2norm=True),
            oracle_packed(inp, cu, True, qk_l2norm=True), torch.float32)


def test_one_sequence_equals_the_fixed_length_scan():
    w = I.Workload("one_seq", 1, 256, 2, 2, 64, 64, 64, torch.float32, g_sigma=2.0, h0_std=0.2,
                   dht=True, seed=67)
    inp = I.make_chunk_inputs(w)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    cu = np.array([0, 256], dtype=np.int32)
    res = run_packed(inp, cu, 64, impl="simt")
    o, ht = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                              output_final_state=True, impl="simt")
    gr = kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], dht=t["dht"],
                           initial_state=t["h0"], impl="simt")
    torch.cuda.synchronize()
    assert torch.equal(res["o"], o) and torch.equal(res["ht"], ht)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert torch.equal(res[n], gr[n]), n


def test_all_sequences_empty():
    HV, K, V = 2, 32, 32
    q = torch.empty(1, 0, 2, K, device="cuda")
    v = torch.empty(1, 0, HV, V, device="cuda")
    g = torch.empty(1, 0, HV, K, device="cuda")
    beta = torch.empty(1, 0, HV, device="cuda")
    h0 = torch.randn(3, HV, K, V, device="cuda")
    cu = torch.zeros(4, dtype=torch.int32, device="cuda")
    o, ht = kda.chunk_kda_fwd_varlen(q, q, v, g, beta, cu, initial_state=h0,
                                     output_final_state=True, chunk_size=32)
    torch.cuda.synchronize()
    kda.check()
    assert torch.equal(ht, h0)


def test_invalid_cu_seqlens_reported_by_check():
    """A decreasing cu_seqlens is caught by the table kernel's own check: no
    sequence is scanned (final state = initial state) and kda_check reports
    KDA_ERR_SHAPE."""
    inp, _ = packed_inputs([40, 40], 1, 1, 32, 32, torch.float32, seed=68)
    bad = np.array([0, 60, 20, 80], dtype=np.int32)   # sequence 1 has negative length
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    kda.check()
    h0 = torch.zeros(3, 1, 32, 32, device="cuda")
    kda.chunk_kda_fwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"],
                             torch.from_numpy(bad).cuda(), initial_state=h0,
                             output_final_state=True, chunk_size=32)
    with pytest.raises(kda.KdaError) as ei:
        kda.check()
    assert ei.value.status == 2
    kda.check()   # the error word was cleared
    _, ht = kda.chunk_kda_fwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                     torch.from_numpy(bad).cuda(), initial_state=h0 + 1.0,
                                     output_final_state=True, chunk_size=32)
    with pytest.raises(kda.KdaError):
        kda.check()
    assert torch.equal(ht, h0 + 1.0)


@pytest.mark.parametrize("H,HV,K,lengths,with_h0,with_dht,qkn", [
    (2, 4, 128, [200, 64, 7, 0, 129, 1, 300], True, True, False),
    (2, 2, 64, [65, 127, 64, 3], True, False, False),
    (1, 2, 128, [100, 28, 250], True, False, True),
])
def test_varlen_tcgen05(H, HV, K, lengths, with_h0, with_dht, qkn):
    """Packed sequences on the tensor cores: each sequence's chunks are
    64-token tiles from its first token (the last one partial, its rows past
    the end masked on load and not written), the state passes run one CTA per
    (sequence, value head).  GVA, K = V = 64 and 128, empty and one-token
    sequences, an upstream final-state gradient (the two-term backward) and
    the in-kernel q/k normalisation.  (The normalisation with an O(1) dht is
    left to the fixed-length test: the kernels' bf16 rounding of the
    normalised q, k alone can move a small dbeta element to the bar.)"""
    inp, cu = packed_inputs(lengths, H, HV, K, K, torch.bfloat16, seed=71 + K + len(lengths),
                            with_h0=with_h0, with_dht=with_dht, normalize_qk=not qkn)
    res = run_packed(inp, cu, 64, impl="tcgen05", qk_l2norm=qkn)
    compare(res, oracle_packed(inp, cu, True, qk_l2norm=qkn), torch.bfloat16, with_h0=with_h0)


@pytest.mark.parametrize("saved", [False, True])
def test_varlen_tcgen05_many_sequences(saved):
    """64 packed sequences (seeded lengths 0 to 200, a few empty and
    one-token ones) at HV = 4: the state passes run 256 CTAs, more than one
    wave, and the persistent kernels walk about 300 chunk slots.  Stateless
    (the recomputed forward state pass beside the reverse pass) and saved."""
    rng = np.random.default_rng(4242)
    lengths = [int(x) for x in rng.integers(0, 201, size=64)]
    lengths[3], lengths[10], lengths[20], lengths[41] = 0, 1, 0, 1
    inp, cu = packed_inputs(lengths, 2, 4, 128, 128, torch.bfloat16, seed=83, with_dht=False)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    cu_d = torch.from_numpy(cu).cuda()
    out = kda.chunk_kda_fwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], cu_d,
                                   initial_state=t["h0"], output_final_state=True,
                                   impl="tcgen05", save_for_backward=saved)
    res = dict(o=out[0], ht=out[1])
    res.update(kda.chunk_kda_bwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], cu_d,
                                        initial_state=t["h0"], impl="tcgen05",
                                        saved=out[2] if saved else None))
    torch.cuda.synchronize()
    kda.check()
    compare(res, oracle_packed(inp, cu, True), torch.bfloat16)


def test_varlen_tcgen05_one_sequence_equals_the_fixed_length_scan():
    w = I.Workload("one_seq_tc", 1, 256, 2, 2, 128, 128, 64, torch.bfloat16, g_sigma=2.0,
                   h0_std=0.2, dht=True, seed=74)
    inp = I.make_chunk_inputs(w)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    res = run_packed(inp, np.array([0, 256], dtype=np.int32), 64, impl="tcgen05")
    o, ht = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                              output_final_state=True, impl="tcgen05")
    gr = kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], dht=t["dht"],
                           initial_state=t["h0"], impl="tcgen05")
    torch.cuda.synchronize()
    assert torch.equal(res["o"], o) and torch.equal(res["ht"], ht)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert torch.equal(res[n], gr[n]), n


def test_varlen_tcgen05_invalid_cu_seqlens_and_empty_batch():
    """On the tensor-core dims: an invalid cu_seqlens leaves every final
    state at its initial value and is reported by kda_check; an empty packed
    batch (T = 0) returns the initial states."""
    inp, _ = packed_inputs([70, 58], 2, 2, 128, 128, torch.bfloat16, seed=75)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    bad = torch.tensor([0, 90, 40, 128], dtype=torch.int32, device="cuda")
    h0 = torch.randn(3, 2, 128, 128, device="cuda")
    kda.check()
    _, ht = kda.chunk_kda_fwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], bad,
                                     initial_state=h0, output_final_state=True, impl="tcgen05")
    with pytest.raises(kda.KdaError) as ei:
        kda.check()
    assert ei.value.status == 2
    assert torch.equal(ht, h0)
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(3, dtype=torch.int32, device="cuda")
    _, ht = kda.chunk_kda_fwd_varlen(e(1, 0, 2, 128), e(1, 0, 2, 128), e(1, 0, 2, 128),
                                     e(1, 0, 2, 128), e(1, 0, 2), cu, initial_state=h0[:2],
                                     output_final_state=True)
    torch.cuda.synchronize()
    kda.check()
    assert torch.equal(ht, h0[:2])


@pytest.mark.parametrize("impl,K,dtype,with_dht", [("tcgen05", 128, torch.bfloat16, False),
                                                   ("tcgen05", 64, torch.bfloat16, True),
                                                   ("simt", 32, torch.float32, True)])
def test_varlen_saved_forward_backward(impl, K, dtype, with_dht):
    """A saving packed forward, then the backward from its workspace (the
    tensor cores skip the recompute unless dht is given; the SIMT kernels
    always recompute): the oracle's outputs and gradients per sequence."""
    lengths = [130, 0, 64, 9, 190]
    inp, cu = packed_inputs(lengths, 2, 2, K, K, dtype, seed=77 + K, with_dht=with_dht)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    cu_d = torch.from_numpy(cu).cuda()
    o, ht, sv = kda.chunk_kda_fwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], cu_d,
                                         initial_state=t["h0"], output_final_state=True,
                                         impl=impl, save_for_backward=True)
    res = dict(o=o, ht=ht)
    res.update(kda.chunk_kda_bwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], cu_d,
                                        dht=t["dht"], initial_state=t["h0"], impl=impl, saved=sv))
    torch.cuda.synchronize()
    kda.check()
    compare(res, oracle_packed(inp, cu, True), dtype)
