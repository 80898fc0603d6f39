"""Shared helpers for the parity tests: tolerances, comparison, and running
the float64 oracle on the same (dtype-rounded) inputs, whole or per head."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from gated_delta_rule_41_gb300.inputs import to_f64

# Tolerances: fp32 inputs 1e-4 absolute; bf16 inputs 1e-2 absolute plus 2e-2
# relative, per element, against the float64 oracle fed the same values.
TOL = {torch.float32: (1e-4, 0.0), torch.bfloat16: (1e-2, 2e-2)}


def assert_close(name, got, ref, dtype):
    """|got - ref| <= atol + rtol*|ref| elementwise; reports the worst case."""
    atol, rtol = TOL[dtype]
    g = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    fro = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    if os.environ.get("KDA_PARITY_REPORT"):
        # worst error as a fraction of its bound: the margin left in the bar
        print(f"[parity] {name}: worst err/bound {float(np.max(err / bound)):.3f}, "
              f"max abs err {float(err.max()):.3g}, rel fro err {fro:.3g}")
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{name}: {bad.sum()} / {bad.size} elements out of tolerance "
            f"(atol {atol}, rtol {rtol}); worst at {idx}: got {g[idx]:.6g} ref {ref[idx]:.6g}; "
            f"max abs err {err.max():.3g}, rel fro err {fro:.3g}")
    return float(err.max()), float(fro)


def oracle_chunk(inp, want_bwd, heads=None, qk_l2norm=False):
    """Run the oracle on the inputs dict (torch, any device).

    heads=None: all heads.  Otherwise a list of (b, hv); results are returned
    per head as dicts of arrays shaped like the one-head slices [1,T,1,X].
    Only valid per head when H == HV (no GVA group sums needed).
    qk_l2norm: q and k are L2-normalised first (oracle.l2norm) and dq, dk are
    mapped back to the raw q, k (oracle.l2norm_bwd).
    """
    if qk_l2norm:
        qr, kr = to_f64(inp["q"]), to_f64(inp["k"])
        normed = dict(inp, q=torch.from_numpy(oracle.l2norm(qr)),
                      k=torch.from_numpy(oracle.l2norm(kr)))
        res = oracle_chunk(normed, want_bwd, heads)
        if want_bwd and heads is None:
            res["dq"], res["dk"] = oracle.l2norm_bwd(qr, res["dq"]), oracle.l2norm_bwd(kr, res["dk"])
        elif want_bwd:
            for (b, hv), r in zip(heads, res):
                sl = lambda x: x[b:b + 1, :, hv:hv + 1]
                r["dq"], r["dk"] = (oracle.l2norm_bwd(sl(qr), r["dq"]),
                                    oracle.l2norm_bwd(sl(kr), r["dk"]))
        return res
    q, k, v, g, beta = (to_f64(inp[n]) for n in ("q", "k", "v", "g", "beta"))
    h0 = to_f64(inp.get("h0"))
    do = to_f64(inp.get("do"))
    dht = to_f64(inp.get("dht"))
    if heads is None:
        o, ht = oracle.fwd_recurrent(q, k, v, g, beta, h0=h0)
        res = dict(o=o, ht=ht)
        if want_bwd:
            res.update(oracle.bwd_recurrent(q, k, v, g, beta, do, h0=h0, dht=dht))
        return res
    assert q.shape[2] == v.shape[2], "per-head oracle runs need H == HV"
    # the sampled heads side by side as the heads of one batch row, so that
    # one oracle call runs them in parallel (the heads are independent)
    cat = lambda x: None if x is None else np.concatenate(
        [x[b:b + 1, :, hv:hv + 1] for b, hv in heads], axis=2)
    cst = lambda x: None if x is None else np.concatenate(
        [x[b:b + 1, hv:hv + 1] for b, hv in heads], axis=1)
    qs, ks, vs, gs, bs = cat(q), cat(k), cat(v), cat(g), cat(beta)
    o, ht = oracle.fwd_recurrent(qs, ks, vs, gs, bs, h0=cst(h0))
    allr = dict(o=o, ht=ht)
    if want_bwd:
        allr.update(oracle.bwd_recurrent(qs, ks, vs, gs, bs, cat(do), h0=cst(h0), dht=cst(dht)))
    out = []
    for i in range(len(heads)):
        r = {}
        for n_, x in allr.items():
            if x is None:
                r[n_] = None
            elif n_ in ("ht", "dh0"):
                r[n_] = x[:, i:i + 1]
            else:
                r[n_] = x[:, :, i:i + 1]
        out.append(r)
    return out
