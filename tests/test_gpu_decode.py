"""Parity of the CUDA decode step with the float64 oracle (single-token
recurrence applied in place to the [B,HV,K,V] state), through the C ABI."""
import numpy as np
import pytest
import torch

import gated_delta_rule_41_gb300 as kda
from gated_delta_rule_41_gb300 import inputs as I
from gated_delta_rule_41_gb300.inputs import to_f64
import oracle
from parity_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_41_gb300 import build
    build.build()


def run_steps(inp, steps, rows=None):
    """GPU: all steps in place; oracle: the same steps on the sampled rows."""
    state = inp["state"].cuda().contiguous()
    d = {n: inp[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    rows = list(range(state.shape[0])) if rows is None else rows
    ref_state = to_f64(inp["state"])[rows].copy()
    for s in range(steps):
        o = kda.recurrent_step(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s], state)
        sel = lambda n: to_f64(inp[n][s])[rows]
        o_ref = oracle.step(sel("q"), sel("k"), sel("v"), sel("g"), sel("beta"), ref_state)
        assert_close(f"o step {s}", o[rows], o_ref, inp["q"].dtype)
    torch.cuda.synchronize()
    kda.check()
    assert_close("state", state[rows], ref_state, inp["q"].dtype)


def test_decode_full_size_sampled_rows():
    w = I.DECODE_BF16
    inp = I.make_decode_inputs(w, device="cuda")
    run_steps(inp, w.steps, rows=list(range(0, 256, 17)))


@pytest.mark.parametrize("K,V,H,HV", [(64, 64, 2, 4), (8, 8, 2, 4), (32, 48, 1, 3),
                                      (128, 128, 4, 4)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_shapes(K, V, H, HV, dtype):
    w = I.DecodeWorkload("dec", 3, H, HV, K, V, 16, dtype, seed=31)
    run_steps(I.make_decode_inputs(w), 16)


def test_decode_matches_chunk_scan():
    """Decoding token by token from h0 equals the chunk scan's outputs and
    final state (both on the GPU, fp32)."""
    w = I.Workload("dec_vs_chunk", 2, 64, 2, 2, 64, 64, 64, torch.float32, h0_std=0.2, seed=32)
    inp = I.make_chunk_inputs(w, device="cuda")
    o, ht = kda.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              initial_state=inp["h0"], output_final_state=True, impl="simt")
    state = inp["h0"].clone()
    outs = []
    for t in range(w.T):
        outs.append(kda.recurrent_step(inp["q"][:, t].contiguous(), inp["k"][:, t].contiguous(),
                                       inp["v"][:, t].contiguous(), inp["g"][:, t].contiguous(),
                                       inp["beta"][:, t].contiguous(), state))
    torch.cuda.synchronize()
    torch.testing.assert_close(torch.stack(outs, 1), o, atol=1e-4, rtol=0)
    torch.testing.assert_close(state, ht, atol=1e-4, rtol=0)


@pytest.mark.parametrize("K,V,H,HV,dtype", [(128, 128, 2, 4, torch.bfloat16),
                                             (64, 64, 2, 2, torch.float32),
                                             (32, 48, 1, 3, torch.float32)])
def test_decode_qk_l2norm_in_kernel(K, V, H, HV, dtype):
    """Raw q and k, L2-normalised by the decode kernel (fast and generic
    paths) against the oracle step on the normalised q, k."""
    w = I.DecodeWorkload("dec_qkn", 3, H, HV, K, V, 8, dtype, seed=33)
    inp = I.make_decode_inputs(w, normalize_qk=False)
    state = inp["state"].cuda().contiguous()
    d = {n: inp[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    ref_state = to_f64(inp["state"]).copy()
    for s in range(w.steps):
        o = kda.recurrent_step(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s], state,
                               use_qk_l2norm_in_kernel=True)
        o_ref = oracle.step(oracle.l2norm(to_f64(inp["q"][s])), oracle.l2norm(to_f64(inp["k"][s])),
                            to_f64(inp["v"][s]), to_f64(inp["g"][s]), to_f64(inp["beta"][s]),
                            ref_state)
        assert_close(f"o step {s}", o, o_ref, dtype)
    torch.cuda.synchronize()
    kda.check()
    assert_close("state", state, ref_state, dtype)
