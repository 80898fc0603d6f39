"""The tensor-core building blocks (TMA into 128B-swizzled tiles, tcgen05.mma
with shared-memory descriptors, TMEM accumulator read back by tcgen05.ld)
against a plain fp32 product of the same bf16 operands."""
import pytest
import torch

import gated_delta_rule_41_gb300 as kda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_41_gb300 import build
    build.build()


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("use_tma", [True, False])
def test_mma_chain_matches_fp32_product(N, use_tma):
    g = torch.Generator(device="cpu").manual_seed(N + use_tma)
    A = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    B = torch.randn(N, 64, generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    D = kda.kda.selftest_mma(A.cuda(), B.cuda(), use_tma=use_tma)
    torch.testing.assert_close(D.double().cpu(), ref, atol=1e-3, rtol=1e-4)


def _mn_case(N, a_mn, b_mn):
    g = torch.Generator(device="cpu").manual_seed(100 + N + 2 * a_mn + 4 * b_mn)
    A = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    B = torch.randn(N, 64, generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    Ain = A.T.contiguous() if a_mn else A
    Bin = B.T.contiguous() if b_mn else B
    D = kda.kda.selftest_mma(Ain.cuda(), Bin.cuda(), a_mn=a_mn, b_mn=b_mn)
    return (D.double().cpu() - ref).abs().max().item()


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("a_mn,b_mn", [(True, False), (False, True), (True, True)])
def test_mn_major_operands(N, a_mn, b_mn):
    """MN-major operands (M/N contiguous): 64-element M/N blocks 8 KB apart,
    8-row K groups 1 KB apart."""
    assert _mn_case(N, a_mn, b_mn) < 1e-3


def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    """A wait on an mbarrier that nothing arrives at gives up after its limit
    (here about 1 ms at 2 GHz), records the error word, and kda_check reports
    KDA_ERR_TIMEOUT once; the next calls run normally."""
    lib = kda.load_library()
    kda.check()
    st = lib.kda_selftest_wait_timeout(2_000_000, kda.kda._stream(None))
    assert st == 0
    with pytest.raises(kda.KdaError) as ei:
        kda.check()
    assert ei.value.status == 7
    kda.check()   # cleared
    # the tensor cores still run and agree with a plain product
    g = torch.Generator(device="cpu").manual_seed(5)
    A = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    B = torch.randn(64, 64, generator=g).to(torch.bfloat16)
    D = kda.kda.selftest_mma(A.cuda(), B.cuda())
    torch.testing.assert_close(D.double().cpu(), A.double() @ B.double().T, atol=1e-3, rtol=1e-4)
