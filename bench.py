#!/usr/bin/env python
"""Benchmark of the KDA chunk scan: forward + backward tokens/s on the KDA layer
training shape of a 1.7B KDA:GQA hybrid (B=4, T=8192, H=HV=16, K=V=128, bf16,
chunk 64), one GPU per rank, inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--path auto|simt|tcgen05]

Prints ONE JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on a bounded sample of the same workload instead.  Under torchrun each
rank runs its own replica of the workload (the scan is independent per head,
so ranks share no data; only the timing is reduced with a max).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunk_kda fwd+bwd tokens/s (B=4,T=8192,H=16,K=V=128 bf16); % roofline"
# Algorithmic bytes per head-token of the fused forward and backward (bf16 I/O,
# K = V = 128, chunk 64): forward reads q, k, v, g (4 x 256 B) and beta (2 B)
# and writes o (256 B); backward reads q, k, v, g, beta, do (1282 B), writes
# dq, dk, dv, dg, dbeta (1026 B) and writes + reads the fp32 chunk-boundary
# states (2 x 128*128*4 / 64 = 2048 B).
FWD_BYTES_PER_HEAD_TOKEN = 1282
BWD_BYTES_PER_HEAD_TOKEN = 4356


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _src_hash(name):
    """Hash of a CUDA source's code: comments and whitespace are removed
    first, so that an edit of comments alone keeps a capture valid."""
    path = os.path.join(ROOT, "gated_delta_rule_41_gb300", "csrc", name)
    if not os.path.exists(path):
        return ""
    code = re.sub(r"/\*.*?\*/", " ", open(path).read(), flags=re.S)
    code = re.sub(r"//[^\n]*", " ", code)
    return hashlib.sha256(" ".join(code.split()).encode()).hexdigest()[:12]


# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture
# of that kernel alone (-k, one launch), keyed by kernel name: (bytes per
# launch, head-tokens B*T*HV of the captured launch, the source file, the
# hash of that file's code when captured).  A kernel whose source code has
# changed since (comments aside) reports traffic null.  The step's kernels were captured at B=1, T=8192, HV=16 (2048
# chunks, inputs and workspace above L2), the plain forward's state pass at
# B=4 (at B=1 the plain forward cuts its state pass into segments); traffic
# grows with the chunk count, so a launch at another size reports the bytes
# scaled by its head-tokens.
NCU_TRAFFIC = {
    "tc_local_bwd": (434779904, 1 * 8192 * 16, "kda_tc.cu", "7d87e21548ab"),
    "tc_intra": (276193536, 1 * 8192 * 16, "kda_tc.cu", "7d87e21548ab"),
    "tc_grad_v": (485224192, 1 * 8192 * 16, "kda_tc.cu", "7d87e21548ab"),
    "tc_chain_fwd_save": (247514112, 1 * 8192 * 16, "kda_tc.cu", "7d87e21548ab"),
    "tc_chain_bwd": (220022528, 1 * 8192 * 16, "kda_tc.cu", "7d87e21548ab"),
    "tc_chain_fwd": (726314752, 4 * 8192 * 16, "kda_tc.cu", "7d87e21548ab"),
}
# decode_kernel: dram read + write per launch at the decode workload (B=256,
# HV=16, K=V=128), its source file and the hash of its code when captured
NCU_DECODE_TRAFFIC = (272652544 + 205543936, "kda_decode.cu", "fc013c481cc7")


def ncu_traffic(name, w):
    """Measured DRAM bytes per launch of kernel `name` at workload w, or None
    when there is no capture of its current source."""
    if name not in NCU_TRAFFIC:
        return None
    tb, ht, src, h = NCU_TRAFFIC[name]
    if _src_hash(src) != h:
        return None
    return int(round(tb * (w.B * w.T * w.HV) / ht))


def kernel_algo_bytes(name, w):
    """Algorithmic bytes one launch of kernel `name` must move at workload w.

    Inputs are counted once at their dtype, outputs once, fp32 workspace
    intermediates once each way."""
    B, T, H, HV, K, V, C = w.B, w.T, w.H, w.HV, w.K, w.V, w.chunk
    e = 2 if str(w.dtype).endswith("bfloat16") else 4
    BH, NT = B * HV, T // C
    tok_in = B * T * (2 * H * K * e + HV * (V * e + K * e + e))   # q, k, v, g, beta
    o = BH * T * V * e
    f32 = 4
    WQK = 3 * BH * T * K * f32      # W, Qh, Kb
    U = BH * T * V * f32
    CC = BH * NT * C * C * f32      # one C x C matrix per chunk
    gam = BH * NT * K * f32
    hs = BH * NT * K * V * f32
    if name == "simt_intra":
        return tok_in + WQK + U + 2 * CC + gam
    if name == "simt_state_fwd":
        return WQK + U + CC + gam + max(o, hs + U)
    if name == "simt_state_bwd":
        return WQK + CC + gam + o + hs + U
    if name == "simt_vgrad":
        return 2 * hs + 2 * U + 2 * o + CC + WQK + 2 * CC + o
    if name == "simt_kgrad":
        return tok_in + WQK + 3 * CC + 2 * B * T * HV * K * f32 + BH * T * K * e
    if name == "simt_group_sum":
        return 2 * B * T * HV * K * f32 + 2 * B * T * H * K * e
    # tensor-core path (K = V = 128, chunk 64): per head-token bytes of the
    # kernel's own inputs and outputs, bf16 operand arrays at 2 B/element,
    # fp32 workspace arrays at 4 B; q and k are read once per query head.
    if K == 128 and V == 128 and C == 64 and e == 2:
        G = HV // H
        qk = 2 * K * e // G                      # q, k per value head
        ops = 4 * K * 2                          # W, Qh, U, Kb (bf16)
        cc = C * 2                               # one bf16 C x C row per token
        per = {
            # T out as bf16 high and low parts, like Aqk one C-row each
            "tc_intra": qk + 2 * K * e + e + ops + 3 * cc + K * 4 // C,
            "tc_chain_fwd": ops + cc + K * 4 // C + V * e,
            "tc_chain_fwd_save": ops + cc + K * 4 // C + V * e + K * V * 2 // C + V * 2,
            "tc_chain_states": ops + cc + K * 4 // C + K * V * 2 // C + V * 2,
            "tc_chain_bwd": V * e + 3 * K * 2 + cc + K * 4 // C + K * V * 2 // C + V * 2,
            # out: dv, dQh and dK (fp32), dW (bf16), dgam, dAqk (bf16), dTv (fp32), d(beta v)
            "tc_grad_v": (2 * K * V * 2 // C + V * e + 2 * V * 2 + V * e + cc + e)
                         + (V * e + 2 * K * 4 + K * 2 + K * 4 // C + cc + C * 4 + 4),
            # in: T (hi, lo), dW (bf16), dQh, dK (fp32), dAqk (bf16), dTv (fp32), ...
            "tc_local_bwd": (2 * cc + K * 2 + 2 * K * 4 + cc + C * 4 + K * 4 // C + 4 + qk +
                             K * e + e)
                            + (2 * K * (e if G == 1 else 4) + K * e + e),
        }
        if name in per:
            return BH * T * per[name]
    return None


def kernel_method_bytes(name, w):
    """The method's own bytes (the per-head-token budget of the fused path)
    that one launch of kernel `name` moves: the tensors of the method it
    reads or writes, each counted once at its dtype, and the fp32
    chunk-boundary states at the budget's one write and one read.  Workspace
    intermediates of this design do not count.  Summed over a step's kernels
    this is exactly the step's budget (1282 + 4356 B per head-token at
    K = V = 128, bf16, one value head per key head)."""
    B, T, H, HV, K, V, C = w.B, w.T, w.H, w.HV, w.K, w.V, w.chunk
    e = 2 if str(w.dtype).endswith("bfloat16") else 4
    G = HV // H
    qk = K * e // G                      # q or k, per value head
    states = K * V * 4 // C              # fp32 chunk-boundary state, per head-token
    per = {
        "tc_intra": 2 * qk + V * e + K * e + e,          # q, k, v, g, beta in
        "tc_chain_fwd": V * e,                           # o out
        "tc_chain_fwd_save": V * e + states,             # o out, states written
        "tc_chain_bwd": V * e,                           # do in
        "tc_grad_v": V * e + states + V * e,             # v in, states read, dv out
        "tc_local_bwd": 2 * (2 * qk + K * e + e),        # q, k, g, beta in; dq, dk, dg, dbeta out
    }
    return B * HV * T * per[name] if name in per else None


def kernel_entry(name, total_ms, launches, total_k, w, hbm):
    """Per-kernel line: launches, time, share; the method's bytes it moves and
    their rate against the copy peak; its own design bytes (inputs and outputs
    including workspace intermediates) and their rate; and the measured DRAM
    bytes per launch."""
    per = total_ms / launches
    e = {"launches": launches, "ms_per_launch": per, "share": total_ms / total_k}
    method = kernel_method_bytes(name, w)
    if method:
        e["method_bytes"] = method
        e["method_gbs"] = method / (per / 1e3) / 1e9
        e["frac"] = e["method_gbs"] / hbm
    design = kernel_algo_bytes(name, w)
    if design:
        e["design_bytes"] = design
        e["design_gbs"] = design / (per / 1e3) / 1e9
    if name in NCU_TRAFFIC:
        e["traffic"] = ncu_traffic(name, w)
    return e


def start_clock_sampler():
    f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    try:
        p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                              "-lms", "50"], stdout=f, stderr=subprocess.DEVNULL)
    except OSError:
        p = None
    return p, f.name


def stop_clock_sampler(p, path, gpu_index):
    if p is None:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    p.terminate()
    try:
        p.wait(timeout=5)
    except subprocess.TimeoutExpired:
        p.kill()
    sms, smax, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in open(path):
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9 or not parts[0].isdigit() or int(parts[0]) != gpu_index:
            continue
        try:
            sms.append(float(parts[1]))
            smax = float(parts[2])
        except ValueError:
            continue
        for n, val in zip(names, parts[5:9]):
            if val.lower().startswith("active"):
                reasons.add(n)
    os.unlink(path)
    return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": smax,
            "reasons": sorted(reasons), "samples": len(sms)}


# --------------------------------------------------------------------------
# CPU oracle on a bounded sample (reference arm and cpu_baseline)
# --------------------------------------------------------------------------

def oracle_sample(w, inp_cpu, nheads, tsample, head0=0):
    """Time the float64 oracle (forward + backward) on the first `tsample`
    tokens of heads head0 .. head0 + nheads - 1 of the workload; return the
    throughput scaled to the metric's unit (whole-workload tokens/s: the
    oracle's cost is linear in heads and in tokens), the seconds taken and
    the threads used."""
    import oracle
    from gated_delta_rule_41_gb300.inputs import to_f64
    heads = [(i // w.HV, i % w.HV) for i in range(head0, head0 + nheads)]
    # gather the sampled heads into one [1, T, n, X] problem (H == HV here)
    take = lambda x: to_f64(torch.stack([x[b, :tsample, hv] for b, hv in heads], dim=1)[None])
    q, k, v, g, do = (take(inp_cpu[n]) for n in ("q", "k", "v", "g", "do"))
    beta = to_f64(torch.stack([inp_cpu["beta"][b, :tsample, hv] for b, hv in heads],
                              dim=1)[None])
    t0 = time.perf_counter()
    oracle.fwd_recurrent(q, k, v, g, beta)
    oracle.bwd_recurrent(q, k, v, g, beta, do)
    dt = time.perf_counter() - t0
    frac = (nheads / (w.B * w.HV)) * (tsample / w.T)
    return w.tokens * frac / dt, dt, oracle.num_threads()


def oracle_whole(w, inp_cpu, min_seconds=10.0, max_passes=4):
    """The oracle over the whole workload (every head, all T tokens), in
    groups of one head per thread, repeated until at least `min_seconds` of
    work (at most `max_passes` passes).  Returns (tokens/s, seconds, passes,
    threads)."""
    import oracle
    group = max(1, oracle.num_threads())
    nh = w.B * w.HV
    total, passes = 0.0, 0
    while passes < max_passes and (passes == 0 or total < min_seconds):
        for h0 in range(0, nh, group):
            _, dt, cores = oracle_sample(w, inp_cpu, min(group, nh - h0), w.T, head0=h0)
            total += dt
        passes += 1
    return passes * w.tokens / total, total, passes, cores


def reference_arm(args, w):
    """The oracle as it stands, timed on the host cores: each step runs it
    (forward + backward) on a bounded sample of the workload -- the first
    `tsample` tokens of `nheads` heads -- and the line's value scales that
    sample's throughput to whole-workload tokens/s (the oracle's cost is
    linear in heads and in tokens).  ms_per_step is the time a sample step
    actually took."""
    import torch as _t  # noqa: F401
    from gated_delta_rule_41_gb300 import inputs as I
    import oracle
    oracle.build()
    inp = I.make_chunk_inputs(w, device="cpu")
    nheads = min(w.B * w.HV, max(1, oracle.num_threads()))
    tsample = 1024
    for _ in range(args.warmup):
        oracle_sample(w, inp, nheads, tsample)
    vals, secs = [], []
    for _ in range(args.steps):
        v, dt, cores = oracle_sample(w, inp, nheads, tsample)
        vals.append(v)
        secs.append(dt)
    value = statistics.median(vals)
    sample = (f"per step: the first {tsample} of T={w.T} tokens of {nheads} of {w.B * w.HV} "
              f"heads, forward+backward ({nheads * tsample} head-tokens of "
              f"{w.B * w.HV * w.T}); value = that throughput scaled to the whole workload")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(secs) * 1e3,
            "ms_per_step_note": "seconds of one sample step as timed (not the whole workload)",
            "whole_workload_ms_extrapolated": w.tokens / value * 1e3,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, "oracle"),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w, path, bwd="saved"):
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.HV, "K": w.K, "V": w.V,
            "chunk": w.chunk, "pass": "fwd+bwd", "path": path, "backward": bwd,
            "l2": f"inputs larger than L2 (q, k, v, g = {4 * w.B * w.T * w.HV * w.K * 2 >> 20} MiB "
                  f"bf16; no flush needed)",
            "parallelism": "one independent replica per rank"}


def fwd_method_bytes(w, final_state):
    """The forward's own bytes for workload w: q, k (once per key head), v, g,
    beta read and o written, at the input dtype; plus the fp32 final state
    when it is returned."""
    e = 2 if str(w.dtype).endswith("bfloat16") else 4
    per = 2 * w.K * e // (w.HV // w.H) + w.V * e + w.K * e + e + w.V * e
    b = w.B * w.T * w.HV * per
    if final_state:
        b += w.B * w.HV * w.K * w.V * 4
    return b


def measure_forward(kda, w, dev, hbm, steps, warmup, path):
    """Forward only (kda_chunk_fwd, nothing kept for a backward) on workload
    w, inputs resident, timed with CUDA events on the launching stream; its
    HBM roofline on the method's bytes and the per-kernel split."""
    from gated_delta_rule_41_gb300 import inputs as I
    inp = I.make_chunk_inputs(w, device=dev)
    q, k, v, g, beta = (inp[n] for n in ("q", "k", "v", "g", "beta"))
    dims = kda.kda.make_dims(q, v, w.chunk, None, path)
    ws = torch.empty(max(1, kda.workspace_bytes(dims, False)), dtype=torch.uint8, device=dev)
    o = torch.empty_like(v)
    ht = (torch.empty(w.B, w.HV, w.K, w.V, dtype=torch.float32, device=dev)
          if w.final_state else None)
    stream = torch.cuda.current_stream()

    def fwd():
        kda.chunk_kda_fwd(q, k, v, g, beta, chunk_size=w.chunk, impl=path, workspace=ws, out=o,
                          output_final_state=w.final_state, final_state=ht)

    for _ in range(max(warmup, 3)):
        fwd()
    torch.cuda.synchronize()
    kda.check()
    kda.timing_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fwd()
    e1.record(stream)
    torch.cuda.synchronize()
    kernels = kda.timing_read()
    kda.timing_enable(False)
    kda.check()
    ms = e0.elapsed_time(e1) / steps
    method = fwd_method_bytes(w, w.final_state)
    gbs = method / (ms / 1e3) / 1e9
    total_k = sum(t for t, _ in kernels.values()) or 1.0
    l2 = 4 * w.B * w.T * w.HV * w.K * 2 >> 20
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.HV, "K": w.K, "V": w.V,
            "chunk": w.chunk, "final_state": w.final_state, "tokens_per_s": w.tokens / (ms / 1e3),
            "ms_per_step": ms, "steps": steps, "method_bytes": method, "achieved_gbs": gbs,
            "peak_gbs": hbm, "frac": gbs / hbm, "bound": "hbm",
            "gpu_launches_per_step": sum(n for _, n in kernels.values()) / steps,
            "l2": f"inputs larger than L2 (q, k, v, g = {l2} MiB); no flush needed",
            "kernels": {n: {"ms_per_launch": t / c, "launches": c, "share": t / total_k}
                        for n, (t, c) in sorted(kernels.items(), key=lambda x: -x[1][0])}}


def measure_chunk_sizes(kda, dev, steps=10, warmup=3):
    """The fwd+bwd step (stateless forward with the final state, backward
    with dht and dh0) at the K = V = 64 shape with an initial state
    (B=4, T=512, H=HV=8, bf16) for chunk 64 (AUTO: the tensor cores) and
    chunk 128 (AUTO: the CUDA-core kernels, the only ones with 128-row
    tiles), timed with CUDA events.  A small, launch-bound shape: tokens/s
    only, no roofline."""
    from gated_delta_rule_41_gb300 import inputs as I
    w = I.SMALL_BF16
    t = I.make_chunk_inputs(w, device=dev)
    out = {}
    for chunk in (64, 128):
        def step():
            o, ht = kda.chunk_kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                      initial_state=t["h0"], output_final_state=True,
                                      chunk_size=chunk)
            kda.chunk_kda_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], dht=t["dht"],
                              initial_state=t["h0"], chunk_size=chunk)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        kda.check()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        kda.check()
        ms = e0.elapsed_time(e1) / steps
        out[f"chunk_{chunk}"] = {"ms_per_step": ms, "tokens_per_s": w.tokens / (ms / 1e3),
                                 "path": "tcgen05" if chunk == 64 else "simt"}
    out["workload"] = w.name
    out["pass"] = "fwd+bwd, dht and h0, stateless backward"
    return out


def measure_varlen(kda, dev, steps=5, warmup=3):
    """Packed variable-length sequences at the training head shape (H=HV=16,
    K=V=128, bf16): 32768 tokens cut into seeded lengths of 512 to 4096,
    fwd+bwd through kda_chunk_fwd_varlen / _bwd_varlen on the tensor cores
    (saving forward + saved backward, and stateless) and on the CUDA-core
    kernels, timed with CUDA events."""
    from gated_delta_rule_41_gb300 import inputs as I
    gen = torch.Generator().manual_seed(91)
    lengths, total = [], 32768
    while total > 0:
        n = min(total, int(torch.randint(512, 4097, (1,), generator=gen)))
        lengths.append(n)
        total -= n
    w = I.Workload("varlen_32k", 1, 32768, 16, 16, 128, 128, 64, torch.bfloat16, g_sigma=2.0,
                   seed=92)
    t = I.make_chunk_inputs(w, device=dev)
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32, device=dev)
    out = {"sequences": len(lengths), "tokens": w.T, "min_len": min(lengths),
           "max_len": max(lengths)}
    for name in ("tcgen05_saved", "tcgen05", "simt"):
        impl = name.split("_")[0]

        def step():
            if name.endswith("_saved"):   # saving forward, backward from its workspace
                _, _, sv = kda.chunk_kda_fwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                                    cu, impl=impl, save_for_backward=True)
            else:
                sv = None
                kda.chunk_kda_fwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], cu, impl=impl)
            kda.chunk_kda_bwd_varlen(t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], cu,
                                     impl=impl, saved=sv)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        kda.check()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        kda.check()
        ms = e0.elapsed_time(e1) / steps
        out[name] = {"ms_per_step": ms, "tokens_per_s": w.T / (ms / 1e3)}
    out["pass"] = ("fwd+bwd, no h0; tcgen05_saved: saving forward and the backward from its "
                   "workspace; tcgen05, simt: stateless backward")
    return out


def measure_decode(kda, dev, hbm):
    """Decode step at B=256, HV=16, K=V=128 (state 256 MiB fp32), 64 steps,
    timed with CUDA events; HBM roofline of the step."""
    from gated_delta_rule_41_gb300 import inputs as I
    w = I.DECODE_BF16
    d = I.make_decode_inputs(w, device=dev)
    state = d["state"]
    o = torch.empty(w.B, w.HV, w.V, dtype=w.dtype, device=dev)
    args = [(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s]) for s in range(w.steps)]
    for s in range(4):
        kda.recurrent_step(*args[s], state, out=o)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(w.steps):
        kda.recurrent_step(*args[s], state, out=o)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / w.steps
    el = 2 if w.dtype == torch.bfloat16 else 4
    io = w.B * (2 * w.H * w.K + w.HV * (w.V + w.K + 1) + w.HV * w.V) * el
    bytes_ = 2 * state.numel() * 4 + io
    gbs = bytes_ / (ms / 1e3) / 1e9
    tb, src, h = NCU_DECODE_TRAFFIC
    return {"workload": w.name, "ms_per_step": ms, "bytes_per_step": bytes_,
            "traffic": tb if _src_hash(src) == h else None,
            "achieved_gbs": gbs, "peak_gbs": hbm, "frac": gbs / hbm, "bound": "hbm",
            "note": "state read once and written once per step; state (256 MiB) > L2"}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------


def slowest_rank_ms(ms, world, device=None):
    """The job's step time: every rank timed the same steps between barriers,
    and the job runs as fast as its slowest rank (max over ranks)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms):
    """Whole-job throughput: the tokens all ranks processed (each runs its own
    replica of the workload) over the job's step time."""
    return world * tokens_per_rank / (ms / 1e3)

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "tcgen05"])
    ap.add_argument("--bwd", default="saved", choices=["saved", "recompute"],
                    help="saved: the backward starts from the forward's saved intermediates; "
                         "recompute: stateless backward")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--B", type=int, default=None,
                    help="override the batch (profiling / sweeps; default: the workload's)")
    ap.add_argument("--T", type=int, default=None,
                    help="override the sequence length (profiling / sweeps)")
    ap.add_argument("--part", default="all", choices=["all", "step", "fwd", "long", "decode"],
                    help="profiling: run only the fwd+bwd step, the forward-only line, the "
                         "long-context forward or the decode leg (default: all, one JSON line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    global torch
    import torch
    from gated_delta_rule_41_gb300 import inputs as I

    w = I.TRAIN_BF16
    if args.B is not None or args.T is not None:
        import dataclasses
        B = w.B if args.B is None else args.B
        T = w.T if args.T is None else args.T
        w = dataclasses.replace(w, B=B, T=T, name=f"kda_layer_B{B}_T{T}_H16_K128")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, w)
        return

    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from gated_delta_rule_41_gb300 import build as kbuild
    kbuild.build()
    import gated_delta_rule_41_gb300 as kda

    hbm, tf, tf_sus, peak_src = _peaks()
    if args.part in ("fwd", "long", "decode"):
        # one part alone (for a profiler): its own line, no step
        if args.part == "decode":
            part = measure_decode(kda, dev, hbm)
        else:
            pw = w if args.part == "fwd" else I.LONG_BF16
            part = measure_forward(kda, pw, dev, hbm, args.steps, args.warmup, args.path)
        if rank == 0:
            print(json.dumps({"part": args.part, **part}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    inp = I.make_chunk_inputs(w, device=dev, seed=w.seed + rank)
    q, k, v, g, beta, do = (inp[n] for n in ("q", "k", "v", "g", "beta", "do"))
    dims_f = kda.kda.make_dims(q, v, w.chunk, None, args.path)
    ws_f = torch.empty(max(1, kda.workspace_bytes(dims_f, False)), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(1, kda.workspace_bytes(dims_f, True)), dtype=torch.uint8, device=dev)
    saving = args.bwd == "saved"
    o = torch.empty_like(v)
    grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                 dg=torch.empty_like(g), dbeta=torch.empty_like(beta), dh0=None)
    stream = torch.cuda.current_stream()

    def fwd_bwd(q, k, v, g, beta, do):
        # saved: the forward keeps its intermediates for the backward (as an
        # autograd function saves tensors); recompute: a stateless backward
        if saving:
            _, _, sv = kda.chunk_kda_fwd(q, k, v, g, beta, chunk_size=w.chunk, impl=args.path,
                                         workspace=ws_b, out=o, save_for_backward=True)
            kda.chunk_kda_bwd(q, k, v, g, beta, do, chunk_size=w.chunk, impl=args.path,
                              grads=grads, saved=sv)
        else:
            kda.chunk_kda_fwd(q, k, v, g, beta, chunk_size=w.chunk, impl=args.path,
                              workspace=ws_f, out=o)
            kda.chunk_kda_bwd(q, k, v, g, beta, do, chunk_size=w.chunk, impl=args.path,
                              workspace=ws_b, grads=grads)

    def step():
        fwd_bwd(q, k, v, g, beta, do)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    kda.check()

    # ---- timed region: device-resident inputs ----
    sampler, spath = start_clock_sampler() if rank == 0 else (None, None)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    kda.timing_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    kernels = kda.timing_read()
    kda.timing_enable(False)
    clocks = stop_clock_sampler(sampler, spath, local) if rank == 0 else None
    kda.check()
    ms = slowest_rank_ms(ev0.elapsed_time(ev1) / args.steps, world, dev)
    value = job_tokens_per_s(w.tokens, world, ms)

    # ---- end to end: pinned host buffers, copies inside the timed region ----
    # Each step copies its inputs host -> device and its outputs device -> host.
    # The copies run on their own streams, double-buffered on the device, so
    # that step i's inputs arrive and step i-1's outputs leave while step i-1
    # (i) computes; events order every reuse of a buffer.
    names_in = ("q", "k", "v", "g", "beta", "do")
    h_in = {n: inp[n].cpu().pin_memory() for n in names_in}
    outs = (("o", v), ("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))
    h_out = {n: torch.empty_like(x, device="cpu").pin_memory() for n, x in outs}
    d_in = [{n: torch.empty_like(inp[n]) for n in names_in} for _ in range(2)]
    d_out = [{n: torch.empty_like(x) for n, x in outs} for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in h_in.values())
    d2h = sum(x.numel() * x.element_size() for x in h_out.values())
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    ev_in, ev_comp, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e_ in ev_comp + ev_out:
        e_.record(stream)

    def e2e_step(i):
        j = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[j])            # step i-2 has read this input set
            for n in names_in:
                d_in[j][n].copy_(h_in[n], non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])               # step i-2's outputs have left
        x, y = d_in[j], d_out[j]
        if saving:
            _, _, sv = kda.chunk_kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                         chunk_size=w.chunk, impl=args.path, workspace=ws_b,
                                         out=y["o"], save_for_backward=True)
            kda.chunk_kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"],
                              chunk_size=w.chunk, impl=args.path, grads=y, saved=sv)
        else:
            kda.chunk_kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], chunk_size=w.chunk,
                              impl=args.path, workspace=ws_f, out=y["o"])
            kda.chunk_kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"],
                              chunk_size=w.chunk, impl=args.path, workspace=ws_b, grads=y)
        ev_comp[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[j])
            for n in h_out:
                h_out[n].copy_(y[n], non_blocking=True)
            ev_out[j].record(s_out)

    # the host link alone: the same copies, both directions at once, no
    # compute (the floor of the end-to-end step).  The host's memory and link
    # are shared with the machine's other GPUs, so the floor is taken before
    # and after the end-to-end loop and the lower one kept.
    def copy_floor(reps=3):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        c0.record(stream)
        s_in.wait_event(c0)
        s_out.wait_event(c0)
        for i in range(reps):
            with torch.cuda.stream(s_in):
                for n in names_in:
                    d_in[i & 1][n].copy_(h_in[n], non_blocking=True)
            with torch.cuda.stream(s_out):
                for n in h_out:
                    h_out[n].copy_(d_out[i & 1][n], non_blocking=True)
        e_in, e_out = torch.cuda.Event(), torch.cuda.Event()
        e_in.record(s_in)
        e_out.record(s_out)
        stream.wait_event(e_in)
        stream.wait_event(e_out)
        c1.record(stream)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / reps

    for i in range(2):
        e2e_step(i)
    copy_ms = copy_floor()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_event(ev_out[(args.steps - 1) & 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = slowest_rank_ms(e0.elapsed_time(e1) / args.steps, world, dev)
    e2e_value = job_tokens_per_s(w.tokens, world, e2e_ms)
    copy_ms = min(copy_ms, copy_floor())

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel, on the method's bytes ----
    # The numerator is what the method itself must move through this kernel
    # (kernel_method_bytes: its share of the 5638 B per head-token budget),
    # not the design's workspace intermediates (reported as design_bytes).
    total_k = sum(t for t, _ in kernels.values()) or 1.0
    dom = max(kernels, key=lambda n: kernels[n][0])
    dom_ms, dom_n = kernels[dom]
    per_launch_ms = dom_ms / dom_n
    method = kernel_method_bytes(dom, w)
    achieved = method / (per_launch_ms / 1e3) / 1e9 if method else None
    traffic = ncu_traffic(dom, w)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": (achieved / hbm) if achieved else None,
                "traffic": traffic, "peak_source": f"{peak_src} (hbm_gbs, copy bandwidth)",
                "method_bytes_per_launch": method, "design_bytes_per_launch":
                kernel_algo_bytes(dom, w), "ms_per_launch": per_launch_ms,
                "note": "achieved = the method's bytes this kernel moves (its share of the "
                        "per-head-token budget) / its CUDA-event time; traffic = ncu DRAM "
                        "bytes per launch (null if its source changed since the capture)"}
    step_bytes = w.B * w.T * w.HV * (FWD_BYTES_PER_HEAD_TOKEN + BWD_BYTES_PER_HEAD_TOKEN)
    step_roof_ms = step_bytes / (hbm * 1e9) * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(w, args.path, args.bwd),
        "roofline": roofline,
        "step_roofline": {"bytes": step_bytes, "roofline_ms": step_roof_ms,
                          "achieved_gbs": step_bytes / (ms / 1e3) / 1e9,
                          "frac": step_roof_ms / ms, "peak": hbm,
                          "note": "whole fwd+bwd step: 5638 B per head-token at the copy peak"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copy_floor_ms": copy_ms, "frac_of_copy_floor": copy_ms / e2e_ms,
                "via": "the Python binding (kda.chunk_kda_fwd / chunk_kda_bwd); torch copies "
                       "pinned host buffers to and from the device, the C ABI takes device "
                       "pointers"},
        "gpu_launches": int(sum(n for _, n in kernels.values())),
        "kernels": {n: kernel_entry(n, t, c, total_k, w, hbm)
                    for n, (t, c) in sorted(kernels.items(), key=lambda x: -x[1][0])},
        "clocks": clocks,
    }
    if world == 1 and args.part == "all":
        # forward only (inference): the training shape, and the long-context
        # forward with its final state
        line["forward"] = measure_forward(kda, w, dev, hbm, max(5, args.steps), 3, args.path)
        line["long_context_forward"] = measure_forward(kda, I.LONG_BF16, dev, hbm, 3, 3,
                                                       args.path)
    if world == 1 and args.part == "all":
        line["decode"] = measure_decode(kda, dev, hbm)
        line["chunk_sizes"] = measure_chunk_sizes(kda, dev)
        line["varlen"] = measure_varlen(kda, dev)
    if world == 1 and not args.no_cpu_baseline and args.part == "all":
        import oracle
        oracle.build()
        inp_cpu = {n: inp[n].cpu() for n in ("q", "k", "v", "g", "beta", "do")}
        cv, cdt, passes, cores = oracle_whole(w, inp_cpu)
        line["cpu_baseline"] = {"value": cv, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"the whole workload ({w.B * w.HV} heads x T={w.T}, "
                                          f"forward+backward) {passes} time(s), {cdt:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
