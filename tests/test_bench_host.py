"""Host logic of bench.py: the algorithmic bytes per launch (the roofline
numerators) and the scaling of the measured DRAM traffic.  No GPU."""
import dataclasses
import importlib.util
import os

import pytest

from gated_delta_rule_41_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


# bytes per head-token of each tensor-core kernel's own inputs and outputs at
# K = V = 128, chunk 64, bf16, one value head per key head
PER_HEAD_TOKEN = {
    "tc_intra": 2442,
    "tc_chain_fwd": 1416,
    "tc_chain_fwd_save": 2184,
    "tc_chain_states": 1928,
    "tc_chain_bwd": 1928,
    "tc_grad_v": 4110,
    "tc_local_bwd": 3472,
}


@pytest.mark.parametrize("name", sorted(PER_HEAD_TOKEN))
def test_tc_algorithmic_bytes_per_head_token(bench, name):
    w = I.TRAIN_BF16
    head_tokens = w.B * w.T * w.HV
    assert bench.kernel_algo_bytes(name, w) == PER_HEAD_TOKEN[name] * head_tokens


def test_tc_algorithmic_bytes_scale_with_the_workload(bench):
    w = I.TRAIN_BF16
    half = dataclasses.replace(w, B=w.B // 2)
    for name in PER_HEAD_TOKEN:
        assert 2 * bench.kernel_algo_bytes(name, half) == bench.kernel_algo_bytes(name, w)


def test_measured_traffic_scales_with_head_tokens(bench):
    w = I.TRAIN_BF16
    for name, (tb, ht, src, h) in bench.NCU_TRAFFIC.items():
        got = bench.ncu_traffic(name, w)
        if bench._src_hash(src) != h:
            assert got is None   # source changed since the capture
            continue
        assert got == round(tb * w.B * w.T * w.HV / ht)
        # the captured launch itself reports its own bytes
        cap = dataclasses.replace(w, B=ht // (w.T * w.HV))
        assert bench.ncu_traffic(name, cap) == tb
    assert bench.ncu_traffic("no_such_kernel", w) is None


def test_source_hash_ignores_comments_only(bench, tmp_path, monkeypatch):
    """A capture stays valid across edits of comments and whitespace, and is
    dropped when the code itself changes."""
    d = tmp_path / "gated_delta_rule_41_gb300" / "csrc"
    d.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = d / "k.cu"
    f.write_text("__global__ void k(int* p) { p[0] = 1; }  // one\n/* block\n comment */\n")
    h = bench._src_hash("k.cu")
    f.write_text("// another comment\n__global__ void k(int* p)\n{\n    p[0] = 1;\n}\n")
    assert bench._src_hash("k.cu") == h
    f.write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench._src_hash("k.cu") != h
    assert bench._src_hash("missing.cu") == ""


def test_measured_traffic_is_dropped_for_a_changed_source(bench, monkeypatch):
    monkeypatch.setattr(bench, "_src_hash", lambda src: "0" * 12)
    assert all(bench.ncu_traffic(n, I.TRAIN_BF16) is None for n in bench.NCU_TRAFFIC)


def test_method_bytes_of_a_step_sum_to_the_budget(bench):
    """The method bytes attributed to the kernels of one fwd+bwd step (saving
    forward + backward from its workspace) add up to the per-head-token
    budget: 1282 B forward + 4356 B backward at K = V = 128, bf16."""
    w = I.TRAIN_BF16
    step = ["tc_intra", "tc_chain_fwd_save", "tc_chain_bwd", "tc_grad_v", "tc_local_bwd"]
    total = sum(bench.kernel_method_bytes(n, w) for n in step)
    assert total == (1282 + 4356) * w.B * w.T * w.HV
    assert bench.kernel_method_bytes("tc_local_bwd", w) == 1540 * w.B * w.T * w.HV


def test_forward_method_bytes(bench):
    w = I.TRAIN_BF16
    assert bench.fwd_method_bytes(w, False) == 1282 * w.B * w.T * w.HV
    lw = I.LONG_BF16
    assert bench.fwd_method_bytes(lw, True) == (1282 * lw.B * lw.T * lw.HV
                                                + lw.B * lw.HV * lw.K * lw.V * 4)
    # GVA: q and k are read once per key head
    g = dataclasses.replace(w, H=w.HV // 2)
    assert bench.fwd_method_bytes(g, False) == (1282 - 256) * w.B * w.T * w.HV


def test_two_ranks_take_the_slowest_rank_and_count_every_rank():
    """bench.py under torchrun (here: two gloo ranks on the CPU): the job's
    step time is the slowest rank's, and the value counts the tokens of
    every rank's replica."""
    import multiprocessing as mp
    import socket

    import dist_worker
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    ms_by_rank, tokens = [2.0, 3.0], 131072
    procs = [ctx.Process(target=dist_worker.timing_rank,
                         args=(r, 2, port, ms_by_rank, tokens, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(out.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r for r, _, _ in got] == [0, 1]
    for _, ms, value in got:
        assert ms == 3.0
        assert value == pytest.approx(2 * tokens / 3e-3)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the oracle arm runs and prints on rank 0 alone; any
    other rank exits 0 without work or output."""
    import subprocess
    import sys
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
