"""Parity of the CUDA chunk scan (forward and backward) with the float64
oracle, on the seeded workloads and on edge cases.  All calls go through the
C ABI via the ctypes binding."""
import dataclasses

import numpy as np
import pytest
import torch

import gated_delta_rule_41_gb300 as kda
from gated_delta_rule_41_gb300 import inputs as I
from gated_delta_rule_41_gb300.inputs import to_f64
import oracle
from parity_util import assert_close, oracle_chunk

pytestmark = pytest.mark.gpu

IMPLS = ["simt", "tcgen05"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_41_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def run_gpu(inp, w, impl, backward=True):
    dev = "cuda"
    t = {n: (x.to(dev) if x is not None else None) for n, x in inp.items()}
    try:
        o, ht = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                  initial_state=t["h0"], output_final_state=True,
                                  chunk_size=w.chunk, impl=impl)
    except kda.KdaError as e:
        if e.status == 3 and impl != "simt":
            pytest.skip(f"{impl} does not support this shape")
        raise
    res = dict(o=o, ht=ht)
    if backward:
        res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                     dht=t["dht"], initial_state=t["h0"], chunk_size=w.chunk,
                                     impl=impl))
    torch.cuda.synchronize()
    kda.check()
    return res


GRADS = ["dq", "dk", "dv", "dg", "dbeta"]


def compare_all(res, ref, w, backward=True, with_h0=False):
    assert_close("o", res["o"], ref["o"], w.dtype)
    assert_close("ht", res["ht"], ref["ht"], w.dtype)
    if backward:
        for n in GRADS:
            assert_close(n, res[n], ref[n], w.dtype)
        if with_h0:
            assert_close("dh0", res["dh0"], ref["dh0"], w.dtype)


@pytest.mark.parametrize("impl", IMPLS)
def test_tiny_gva_fp32(impl):
    w = I.TINY_GVA_F32
    inp = I.make_chunk_inputs(w)
    res = run_gpu(inp, w, impl)
    ref = oracle_chunk(inp, True)
    compare_all(res, ref, w)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_fp32_gva_chunks_with_h0(impl, chunk):
    w = I.Workload("fp32_gva", 2, 128, 2, 4, 32, 32, chunk, torch.float32, g_sigma=2.0,
                   h0_std=0.3, dht=True, seed=21)
    inp = I.make_chunk_inputs(w)
    res = run_gpu(inp, w, impl)
    compare_all(res, oracle_chunk(inp, True), w, with_h0=True)


@pytest.mark.parametrize("dtype,K,H,HV,qkn", [(torch.float32, 32, 2, 2, False),
                                              (torch.float32, 16, 1, 2, False),
                                              (torch.bfloat16, 64, 2, 4, False),
                                              (torch.bfloat16, 128, 2, 2, False),
                                              (torch.bfloat16, 128, 1, 2, True)])
def test_chunk_128(dtype, K, H, HV, qkn):
    """Chunks of 128 rows (the K3 README's 关键约束 / 风险点 table, row
    chunk_size: 64 by default, 128 on a large-memory GPU) on the CUDA-core
    kernels, whose C x C matrices then live in the workspace: three chunks
    with an initial state and an upstream final-state gradient, with GVA and
    the in-kernel q/k normalisation; every output and gradient against the
    oracle, through AUTO (which picks those kernels) and the saving forward."""
    w = I.Workload("chunk128", 2, 384, H, HV, K, K, 128, dtype, g_sigma=2.0, h0_std=0.1,
                   dht=True, seed=81 + K + H)
    inp = I.make_chunk_inputs(w, normalize_qk=not qkn)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    out = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                            output_final_state=True, chunk_size=128, save_for_backward=True,
                            use_qk_l2norm_in_kernel=qkn)
    res = dict(o=out[0], ht=out[1])
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                 dht=t["dht"], initial_state=t["h0"], chunk_size=128,
                                 saved=out[2], use_qk_l2norm_in_kernel=qkn))
    torch.cuda.synchronize()
    kda.check()
    compare_all(res, oracle_chunk(inp, True, qk_l2norm=qkn), w, with_h0=True)


def test_chunk_128_refused_on_tensor_cores():
    w = I.Workload("chunk128_tc", 1, 256, 1, 1, 128, 128, 128, torch.bfloat16, seed=85)
    t = {n: (x.cuda() if x is not None else None) for n, x in I.make_chunk_inputs(w).items()}
    with pytest.raises(kda.KdaError) as ei:
        kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], chunk_size=128,
                          impl="tcgen05")
    assert ei.value.status == 3


@pytest.mark.parametrize("impl", IMPLS)
def test_small_bf16_full(impl):
    """bf16 B4 T512 H8 K = V = 64 with an initial state and an upstream
    final-state gradient; on the tensor cores K = V = 64 runs at 128 with
    zero-filled upper channels, and dht takes the two-term backward."""
    w = I.SMALL_BF16
    inp = I.make_chunk_inputs(w)
    res = run_gpu(inp, w, impl)
    compare_all(res, oracle_chunk(inp, True), w, with_h0=True)


@pytest.mark.parametrize("impl", IMPLS)
def test_fp32_k128_full_tile(impl):
    w = I.Workload("fp32_k128", 1, 192, 2, 2, 128, 128, 64, torch.float32, g_sigma=2.0,
                   h0_std=0.1, dht=True, seed=22)
    inp = I.make_chunk_inputs(w)
    res = run_gpu(inp, w, impl)
    compare_all(res, oracle_chunk(inp, True), w, with_h0=True)


@pytest.mark.parametrize("impl,with_dht", [("simt", True), ("auto", True), ("simt", False),
                                           ("tcgen05", False), ("tcgen05", True)])
def test_bf16_gva_k128(impl, with_dht):
    """K = V = 128 with GVA, with and without an O(1) upstream final-state
    gradient (on the tensor cores, dht takes the two-term backward)."""
    w = I.Workload("bf16_gva_k128", 2, 256, 2, 4, 128, 128, 64, torch.bfloat16, g_sigma=2.0,
                   dht=with_dht, seed=23)
    inp = I.make_chunk_inputs(w)
    res = run_gpu(inp, w, impl)
    compare_all(res, oracle_chunk(inp, True), w)


@pytest.mark.parametrize("impl,wl", [
    ("tcgen05", I.Workload("saved_k128", 2, 256, 2, 4, 128, 128, 64, torch.bfloat16,
                           g_sigma=2.0, h0_std=0.1, seed=27)),
    ("auto", I.Workload("saved_k128_dht", 1, 192, 2, 2, 128, 128, 64, torch.bfloat16,
                        g_sigma=2.0, h0_std=0.1, dht=True, seed=28)),
    ("tcgen05", I.Workload("saved_k64_dht", 2, 192, 2, 4, 64, 64, 64, torch.bfloat16,
                           g_sigma=2.0, h0_std=0.1, dht=True, seed=30)),
    ("simt", I.Workload("saved_simt", 2, 128, 2, 4, 32, 32, 32, torch.float32, g_sigma=2.0,
                        h0_std=0.3, dht=True, seed=29)),
])
def test_saved_forward_backward(impl, wl):
    """A saving forward followed by the backward from its workspace gives the
    oracle's outputs and gradients (the tensor cores skip the recompute unless
    dht is given; the SIMT kernels always recompute)."""
    t = {n: (x.cuda() if x is not None else None) for n, x in I.make_chunk_inputs(wl).items()}
    o, ht, saved = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                     initial_state=t["h0"], output_final_state=True,
                                     chunk_size=wl.chunk, impl=impl, save_for_backward=True)
    # another call in between must not matter: it uses its own workspace
    kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], chunk_size=wl.chunk, impl=impl)
    res = dict(o=o, ht=ht)
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], dht=t["dht"],
                                 initial_state=t["h0"], chunk_size=wl.chunk, impl=impl,
                                 saved=saved))
    torch.cuda.synchronize()
    kda.check()
    compare_all(res, oracle_chunk(I.make_chunk_inputs(wl), True), wl, with_h0=True)


def test_saved_backward_rejects_other_dims():
    w = I.Workload("saved_dims", 1, 128, 1, 1, 128, 128, 64, torch.bfloat16, seed=30)
    t = {n: (x.cuda() if x is not None else None) for n, x in I.make_chunk_inputs(w).items()}
    _, _, saved = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                    save_for_backward=True)
    with pytest.raises(kda.KdaError):
        kda.chunk_kda_bwd(t["q"][:, :64], t["k"][:, :64], t["v"][:, :64], t["g"][:, :64],
                          t["beta"][:, :64], t["do"][:, :64], saved=saved)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("saved", [False, True])
@pytest.mark.parametrize("B,T,H,HV", [(1, 64, 1, 1), (1, 128, 1, 1), (2, 192, 1, 4),
                                      (1, 256, 1, 2), (1, 320, 2, 2)])
def test_tcgen05_chunk_counts_and_groups(B, T, H, HV, saved, D):
    """Tensor-core path on one chunk, odd and even chunk counts (the state
    passes alternate two state tiles and two stages) and GVA groups of 2 and
    4, with an initial state and the final state, stateless and saved
    backward; K = V = 128, and 64 (zero-filled upper channels)."""
    w = I.Workload("tc_shapes", B, T, H, HV, D, D, 64, torch.bfloat16, g_sigma=2.0,
                   h0_std=0.1, seed=31 + T + HV + D)
    inp = I.make_chunk_inputs(w)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    if saved:
        o, ht, sv = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                      initial_state=t["h0"], output_final_state=True,
                                      impl="tcgen05", save_for_backward=True)
    else:
        o, ht = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                  initial_state=t["h0"], output_final_state=True, impl="tcgen05")
        sv = None
    res = dict(o=o, ht=ht)
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                 initial_state=t["h0"], impl="tcgen05", saved=sv))
    torch.cuda.synchronize()
    kda.check()
    compare_all(res, oracle_chunk(inp, True), w, with_h0=True)


@pytest.mark.parametrize("vl", [False, True])
def test_recompute_backward_on_a_side_stream(vl):
    """The recomputing tensor-core backward runs its reverse state pass on a
    second stream beside the forward state pass and joins the caller's stream
    before the contractions over V.  Called on a non-default stream, with the
    results copied on that stream right after the call (no host
    synchronisation in between), every output equals the default-stream run
    bit for bit (the kernels use no atomics) and is within the bar of the
    oracle.  Also for packed sequences."""
    w = I.Workload("side_stream", 2, 1024, 2, 2, 128, 128, 64, torch.bfloat16, g_sigma=2.0,
                   h0_std=0.1, seed=77)
    inp = I.make_chunk_inputs(w)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    if vl:
        lens = [700, 1348]   # one packed batch of the same 2048 tokens
        cu = torch.tensor([0, lens[0], sum(lens)], dtype=torch.int32, device="cuda")
        pk = {n: t[n].reshape(1, -1, *t[n].shape[2:]) for n in ("q", "k", "v", "g", "beta", "do")}

    def step():
        if vl:
            o, ht = kda.chunk_kda_fwd_varlen(pk["q"], pk["k"], pk["v"], pk["g"], pk["beta"], cu,
                                             output_final_state=True, impl="tcgen05")
            grads = kda.chunk_kda_bwd_varlen(pk["q"], pk["k"], pk["v"], pk["g"], pk["beta"],
                                             pk["do"], cu, impl="tcgen05")
        else:
            o, ht = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                      initial_state=t["h0"], output_final_state=True,
                                      impl="tcgen05")
            grads = kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                      initial_state=t["h0"], impl="tcgen05")
        out = dict(o=o, ht=ht, **grads)
        return {n: x.clone() for n, x in out.items() if x is not None}

    ref = step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        got = step()
    torch.cuda.synchronize()
    kda.check()
    assert set(got) == set(ref)
    for n in ref:
        assert torch.equal(got[n], ref[n]), n
    if not vl:
        compare_all(got, oracle_chunk(inp, True), w, with_h0=True)


@pytest.mark.parametrize("B,T,H,HV,D,saved,h0", [
    (2, 256, 2, 4, 128, False, True), (2, 256, 2, 4, 128, True, True),
    (1, 512, 2, 2, 128, False, True), (2, 1024, 1, 1, 128, False, True),
    (1, 64, 1, 1, 128, False, False), (1, 320, 3, 3, 64, True, True),
    (3, 192, 1, 2, 64, False, False)])
def test_tcgen05_final_state_gradient(B, T, H, HV, D, saved, h0):
    """An O(1) upstream final-state gradient on the tensor cores (the two-term
    backward: U, Kb, delta and dS split into bf16 high and low parts), with
    GVA, K = V = 64 and 128, one to sixteen chunks, with and without h0 and a
    saving forward: every output and gradient within the bf16 bar."""
    w = I.Workload("tc_dht", B, T, H, HV, D, D, 64, torch.bfloat16, g_sigma=2.0,
                   h0_std=0.1 if h0 else None, dht=True, seed=26 + T + D)
    inp = I.make_chunk_inputs(w)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    out = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                            output_final_state=True, impl="tcgen05", save_for_backward=saved)
    res = dict(o=out[0], ht=out[1])
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                 dht=t["dht"], initial_state=t["h0"], impl="tcgen05",
                                 saved=out[2] if saved else None))
    torch.cuda.synchronize()
    kda.check()
    compare_all(res, oracle_chunk(inp, True), w, with_h0=h0)


@pytest.mark.parametrize("impl", IMPLS)
def test_clamp_active_below_minus_five(impl):
    """Gates far below -5 reach the kernel: it must clamp them and pass no
    gradient through them (g == -5 exactly still passes)."""
    w = I.Workload("clamp", 2, 128, 2, 2, 64, 64, 64, torch.bfloat16, g_mu=3.0, g_sigma=3.0,
                   h0_std=0.2, dht=True, seed=24)
    inp = I.make_chunk_inputs(w, g_floor=None)
    g = inp["g"].float()
    g[:, :8] = -5.0  # exact boundary values
    inp["g"] = g.to(w.dtype)
    assert (inp["g"].float() < -5).float().mean() > 0.2
    res = run_gpu(inp, w, impl)
    ref = oracle_chunk(inp, True)
    compare_all(res, ref, w, with_h0=True)
    assert torch.all(res["dg"].float().cpu()[inp["g"].float() < -5] == 0)


@pytest.mark.parametrize("saved", [False, True])
def test_tcgen05_clamp_below_minus_five(saved):
    """The tensor-core kernels at K = V = 128 on gates far below -5 (down to
    about -15) plus a block of exact -5 values: the in-kernel clamp must hold
    every in-chunk decay factor in range, and dg must vanish where g < -5
    (the K3 README's lower bound of -5 on the log-decay, row "exp 下溢")."""
    w = I.Workload("clamp_tc", 1, 256, 2, 2, 128, 128, 64, torch.bfloat16, g_mu=3.0,
                   g_sigma=3.0, h0_std=0.1, seed=24)
    inp = I.make_chunk_inputs(w, g_floor=None)
    g = inp["g"].float()
    g[:, 64:72] = -5.0  # exact boundary values, inside the second chunk
    inp["g"] = g.to(w.dtype)
    below = inp["g"].float() < -5
    assert below.float().mean() > 0.2 and inp["g"].float().min() < -12
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    out = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                            output_final_state=True, impl="tcgen05", save_for_backward=saved)
    o, ht = out[0], out[1]
    res = dict(o=o, ht=ht)
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                 initial_state=t["h0"], impl="tcgen05",
                                 saved=out[2] if saved else None))
    torch.cuda.synchronize()
    kda.check()
    compare_all(res, oracle_chunk(inp, True), w, with_h0=True)
    assert torch.all(res["dg"].float().cpu()[below] == 0)


@pytest.mark.parametrize("impl,saved,D", [("simt", False, 128), ("tcgen05", False, 128),
                                          ("tcgen05", True, 128), ("tcgen05", True, 64)])
@pytest.mark.parametrize("H,HV", [(2, 2), (1, 2)])
def test_qk_l2norm_in_kernel(impl, saved, D, H, HV):
    """The kernels L2-normalise raw q and k themselves (the K3 README's "q/k
    L2-norm" variant): outputs are the scan of the normalised q, k, and dq, dk
    are gradients with respect to the raw q, k (after the GVA group sum)."""
    w = I.Workload("qkn", 2, 192, H, HV, D, D, 64, torch.bfloat16, g_sigma=2.0, h0_std=0.1,
                   seed=51 + H + HV + D)
    inp = I.make_chunk_inputs(w, normalize_qk=False)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    out = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                            output_final_state=True, impl=impl, save_for_backward=saved,
                            use_qk_l2norm_in_kernel=True)
    res = dict(o=out[0], ht=out[1])
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                 initial_state=t["h0"], impl=impl,
                                 saved=out[2] if saved else None, use_qk_l2norm_in_kernel=True))
    torch.cuda.synchronize()
    kda.check()
    compare_all(res, oracle_chunk(inp, True, qk_l2norm=True), w, with_h0=True)


@pytest.mark.parametrize("saved", [False, True])
def test_qk_l2norm_in_kernel_tcgen05_with_final_state_gradient(saved):
    """q/k L2 normalisation in the kernels together with an upstream
    final-state gradient on the tensor cores (GVA, K = V = 128)."""
    w = I.Workload("qkn_dht", 2, 192, 2, 4, 128, 128, 64, torch.bfloat16, g_sigma=2.0,
                   h0_std=0.1, dht=True, seed=57)
    inp = I.make_chunk_inputs(w, normalize_qk=False)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    out = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                            output_final_state=True, impl="tcgen05", save_for_backward=saved,
                            use_qk_l2norm_in_kernel=True)
    res = dict(o=out[0], ht=out[1])
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                 dht=t["dht"], initial_state=t["h0"], impl="tcgen05",
                                 saved=out[2] if saved else None, use_qk_l2norm_in_kernel=True))
    torch.cuda.synchronize()
    kda.check()
    compare_all(res, oracle_chunk(inp, True, qk_l2norm=True), w, with_h0=True)


def test_qk_l2norm_in_kernel_fp32_gva_with_final_state_gradient():
    w = I.Workload("qkn_fp32", 2, 64, 2, 4, 16, 16, 16, torch.float32, g_sigma=2.0, h0_std=0.3,
                   dht=True, seed=55)
    inp = I.make_chunk_inputs(w, normalize_qk=False)
    t = {n: (x.cuda() if x is not None else None) for n, x in inp.items()}
    o, ht = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                              output_final_state=True, chunk_size=w.chunk,
                              use_qk_l2norm_in_kernel=True)
    res = dict(o=o, ht=ht)
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                 dht=t["dht"], initial_state=t["h0"], chunk_size=w.chunk,
                                 use_qk_l2norm_in_kernel=True))
    torch.cuda.synchronize()
    kda.check()
    compare_all(res, oracle_chunk(inp, True, qk_l2norm=True), w, with_h0=True)


@pytest.mark.parametrize("B,T,H,HV,D", [(1, 4096, 2, 4, 128), (2, 3072, 1, 1, 64),
                                        (1, 8192, 4, 4, 128)])
def test_tcgen05_segmented_forward(B, T, H, HV, D):
    """Few heads and long sequences: the plain forward cuts the state pass into
    segments (segment 0 in full; later ones from zero and as K x K transitions,
    combined, then rerun in full), which must give the oracle's outputs and
    final state exactly as the single pass does."""
    w = I.Workload("segmented", B, T, H, HV, D, D, 64, torch.bfloat16, g_mu=-3.0, g_sigma=1.0,
                   h0_std=0.1, seed=71 + T + D)
    inp = I.make_chunk_inputs(w)
    res = run_gpu(inp, w, "tcgen05", backward=False)
    ref = oracle_chunk(inp, False)
    assert_close("o", res["o"], ref["o"], w.dtype)
    assert_close("ht", res["ht"], ref["ht"], w.dtype)


def test_ragged_value_width_simt():
    """V not a multiple of the 32-column tile, small K."""
    w = I.Workload("ragged_v", 1, 64, 1, 2, 16, 40, 32, torch.float32, h0_std=0.5, dht=True,
                   seed=25)
    inp = I.make_chunk_inputs(w)
    res = run_gpu(inp, w, "simt")
    compare_all(res, oracle_chunk(inp, True), w, with_h0=True)


def test_empty_sequence_and_batch():
    w = I.Workload("empty", 2, 0, 1, 1, 64, 64, 64, torch.bfloat16, h0_std=1.0, dht=True)
    inp = I.make_chunk_inputs(w, device="cuda")
    o, ht = kda.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              initial_state=inp["h0"], output_final_state=True)
    gr = kda.chunk_kda_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["do"],
                           dht=inp["dht"], initial_state=inp["h0"])
    torch.cuda.synchronize()
    assert o.numel() == 0
    assert torch.equal(ht, inp["h0"])
    assert torch.equal(gr["dh0"], inp["dht"])
    w0 = I.Workload("empty_b", 0, 64, 1, 1, 64, 64, 64, torch.bfloat16)
    inp0 = I.make_chunk_inputs(w0, device="cuda")
    o0, _ = kda.chunk_kda_fwd(inp0["q"], inp0["k"], inp0["v"], inp0["g"], inp0["beta"])
    assert o0.numel() == 0


# ---- full-size workloads: sampled heads against the oracle ----

def _sampled(w, heads, impl, backward):
    inp = I.make_chunk_inputs(w, device="cuda")
    res = run_gpu(inp, w, impl, backward=backward)
    refs = oracle_chunk(inp, backward, heads=heads)
    for (b, hv), ref in zip(heads, refs):
        sl = lambda x: x[b:b + 1, :, hv:hv + 1]
        assert_close(f"o[{b},{hv}]", sl(res["o"]), ref["o"], w.dtype)
        assert_close(f"ht[{b},{hv}]", res["ht"][b:b + 1, hv:hv + 1], ref["ht"], w.dtype)
        if backward:
            for n in GRADS:
                assert_close(f"{n}[{b},{hv}]", sl(res[n]), ref[n], w.dtype)
    return res


@pytest.mark.parametrize("impl", IMPLS)
def test_train_shape_full_size_sampled_heads(impl):
    w = I.TRAIN_BF16
    heads = [(0, 0), (0, 9), (1, 3), (1, 14), (2, 6), (2, 11), (3, 1), (3, 15)]
    res = _sampled(w, heads, impl, backward=True)
    for n in ["o"] + GRADS:
        assert torch.isfinite(res[n].float()).all(), n


def test_train_shape_full_size_saved_sampled_heads():
    """The configuration the benchmark times: a saving forward, then the
    backward from its workspace, at the full training size (AUTO takes the
    tensor cores), on sampled heads against the oracle."""
    w = I.TRAIN_BF16
    heads = [(0, 3), (0, 12), (1, 8), (2, 0), (2, 12), (3, 7)]
    inp = I.make_chunk_inputs(w, device="cuda")
    o, ht, sv = kda.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  initial_state=inp["h0"], output_final_state=True,
                                  chunk_size=w.chunk, save_for_backward=True)
    res = dict(o=o, ht=ht)
    res.update(kda.chunk_kda_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["do"],
                                 dht=inp["dht"], initial_state=inp["h0"], chunk_size=w.chunk,
                                 saved=sv))
    torch.cuda.synchronize()
    kda.check()
    refs = oracle_chunk(inp, True, heads=heads)
    for (b, hv), ref in zip(heads, refs):
        sl = lambda x: x[b:b + 1, :, hv:hv + 1]
        assert_close(f"o[{b},{hv}]", sl(res["o"]), ref["o"], w.dtype)
        assert_close(f"ht[{b},{hv}]", res["ht"][b:b + 1, hv:hv + 1], ref["ht"], w.dtype)
        for n in GRADS:
            assert_close(f"{n}[{b},{hv}]", sl(res[n]), ref[n], w.dtype)


def test_train_shape_full_size_final_state_gradient_sampled_heads():
    """The training size with an initial state and an O(1) upstream
    final-state gradient on the tensor cores (the two-term backward, which
    recomputes even after a saving forward), on sampled heads against the
    oracle."""
    w = dataclasses.replace(I.TRAIN_BF16, h0_std=0.1, dht=True, seed=33)
    heads = [(0, 10), (1, 5), (2, 2), (3, 14)]
    inp = I.make_chunk_inputs(w, device="cuda")
    o, ht, sv = kda.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  initial_state=inp["h0"], output_final_state=True,
                                  impl="tcgen05", save_for_backward=True)
    res = dict(o=o, ht=ht)
    res.update(kda.chunk_kda_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["do"],
                                 dht=inp["dht"], initial_state=inp["h0"], impl="tcgen05",
                                 saved=sv))
    torch.cuda.synchronize()
    kda.check()
    refs = oracle_chunk(inp, True, heads=heads)
    for (b, hv), ref in zip(heads, refs):
        sl = lambda x: x[b:b + 1, :, hv:hv + 1]
        assert_close(f"o[{b},{hv}]", sl(res["o"]), ref["o"], w.dtype)
        assert_close(f"ht[{b},{hv}]", res["ht"][b:b + 1, hv:hv + 1], ref["ht"], w.dtype)
        for n in GRADS:
            assert_close(f"{n}[{b},{hv}]", sl(res[n]), ref[n], w.dtype)
        assert_close(f"dh0[{b},{hv}]", res["dh0"][b:b + 1, hv:hv + 1], ref["dh0"], w.dtype)


@pytest.mark.parametrize("impl", IMPLS)
def test_long_context_full_size_sampled_heads(impl):
    _sampled(I.LONG_BF16, [(0, h) for h in (0, 4, 9, 13, 18, 22, 27, 31)], impl, backward=False)


@pytest.mark.parametrize("impl,K,dtype", [("simt", 64, torch.bfloat16), ("simt", 64, torch.float32),
                                           ("tcgen05", 64, torch.bfloat16),
                                           ("tcgen05", 128, torch.bfloat16)])
def test_96_heads_sampled(impl, K, dtype):
    """H = HV = 96 heads, head dim 64 (CUDA-core path) and 128 (tensor cores),
    with an initial state, on sampled heads against the oracle."""
    w = I.Workload("heads96", 1, 256, 96, 96, K, K, 64, dtype, g_sigma=2.0, h0_std=0.1,
                   seed=41 + K)
    inp = I.make_chunk_inputs(w, device="cuda")
    res = run_gpu(inp, w, impl)
    heads = [(0, 0), (0, 47), (0, 95)]
    refs = oracle_chunk(inp, True, heads=heads)
    for (b, hv), ref in zip(heads, refs):
        sl = lambda x: x[b:b + 1, :, hv:hv + 1]
        assert_close(f"o[{hv}]", sl(res["o"]), ref["o"], w.dtype)
        assert_close(f"ht[{hv}]", res["ht"][b:b + 1, hv:hv + 1], ref["ht"], w.dtype)
        for n in GRADS:
            assert_close(f"{n}[{hv}]", sl(res[n]), ref[n], w.dtype)


@pytest.mark.parametrize("saved", [False, True])
def test_tcgen05_more_heads_than_sms(saved):
    """B = 2 x 96 heads: 192 (batch, head) pairs, so the one-CTA-per-SM state
    passes run in two waves; heads from both waves (bh 0, 95, 150, 191) on
    the oracle, with an initial state, stateless and saved."""
    w = I.Workload("heads192", 2, 192, 96, 96, 128, 128, 64, torch.bfloat16, g_sigma=2.0,
                   h0_std=0.1, seed=57)
    inp = I.make_chunk_inputs(w, device="cuda")
    t = inp
    out = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], initial_state=t["h0"],
                            output_final_state=True, impl="tcgen05", save_for_backward=saved)
    res = dict(o=out[0], ht=out[1])
    res.update(kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"],
                                 initial_state=t["h0"], impl="tcgen05",
                                 saved=out[2] if saved else None))
    torch.cuda.synchronize()
    kda.check()
    heads = [(0, 0), (0, 95), (1, 54), (1, 95)]
    refs = oracle_chunk(inp, True, heads=heads)
    for (b, hv), ref in zip(heads, refs):
        sl = lambda x: x[b:b + 1, :, hv:hv + 1]
        assert_close(f"o[{b},{hv}]", sl(res["o"]), ref["o"], w.dtype)
        assert_close(f"ht[{b},{hv}]", res["ht"][b:b + 1, hv:hv + 1], ref["ht"], w.dtype)
        assert_close(f"dh0[{b},{hv}]", res["dh0"][b:b + 1, hv:hv + 1], ref["dh0"], w.dtype)
        for n in GRADS:
            assert_close(f"{n}[{b},{hv}]", sl(res[n]), ref[n], w.dtype)


def test_impls_agree_train_shape_subset():
    """The SIMT and tensor-core paths agree with each other on a slice of the
    training workload (T = 1024)."""
    w = I.TRAIN_BF16
    inp = I.make_chunk_inputs(w, device="cuda", T=1024)
    a = run_gpu(inp, w, "simt")
    b = run_gpu(inp, w, "tcgen05")
    for n in ["o", "ht"] + GRADS:
        assert_close(n, b[n], a[n].double().cpu().numpy(), w.dtype)
