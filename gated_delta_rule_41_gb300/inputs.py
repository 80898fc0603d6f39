"""Seeded synthetic inputs for the KDA chunk scan and decode step.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It draws random numbers and shapes them into the input distributions
of the workloads; it holds none of the method's own arithmetic (no decay, no
delta-rule write, no chunk algebra).

Recipe (one torch generator per call, seeded with ``seed``; float32 draws in
this order: q, k, v, beta-logit, g-logit, h0, do, dht):

* q, k ~ N(0,1), L2-normalised over the key dimension in float32, then cast.
* v ~ N(0,1).
* beta = sigmoid(N(0,1))  -- one scalar per token and value head.
* g = max(-softplus(N(mu, sigma)), g_floor) -- a per-key-channel log-decay.
  The workloads fix g_floor = -5; tests that exercise the kernel's own clamp
  pass ``g_floor=None`` so that values below -5 reach it.
* h0 ~ h0_std * N(0,1) in float32 (the recurrent state is always float32).
* do, dht ~ N(0,1) (upstream gradients).

Workload shapes come from the "DM-KDAGQA-1.7B-SD" model card (KDA layers of
16 heads x 128, context 8192) and the K3 README test-shape rows (tiny GVA
shape T=16, B=2, H=2, HV=4, K=V=8).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    HV: int
    K: int
    V: int
    chunk: int
    dtype: torch.dtype
    g_mu: float = 0.0
    g_sigma: float = 1.0
    h0_std: Optional[float] = None     # None: zero initial state (h0 omitted)
    final_state: bool = False
    backward: bool = True
    dht: bool = False                  # upstream gradient on the final state
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The five workloads.  Names describe what each one is.
TINY_GVA_F32 = Workload("tiny_gva_fp32_B2_T16_H2_HV4_K8", 2, 16, 2, 4, 8, 8, 16, torch.float32,
                        dht=True, seed=0)
SMALL_BF16 = Workload("bf16_B4_T512_H8_K64_h0", 4, 512, 8, 8, 64, 64, 64, torch.bfloat16,
                      h0_std=0.1, final_state=True, dht=True, seed=1)
TRAIN_BF16 = Workload("kda_layer_1p7b_train_B4_T8192_H16_K128", 4, 8192, 16, 16, 128, 128, 64,
                      torch.bfloat16, g_sigma=2.0, seed=2)
LONG_BF16 = Workload("long_ctx_fwd_B1_T65536_H32_K128", 1, 65536, 32, 32, 128, 128, 64,
                     torch.bfloat16, g_mu=-3.0, g_sigma=1.0, final_state=True, backward=False,
                     seed=3)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    HV: int
    K: int
    V: int
    steps: int
    dtype: torch.dtype
    g_mu: float = 0.0
    g_sigma: float = 2.0
    state_std: float = 0.1
    seed: int = 4


DECODE_BF16 = DecodeWorkload("decode_B256_HV16_K128_64steps", 256, 16, 16, 128, 128, 64,
                             torch.bfloat16)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _l2norm(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make_chunk_inputs(w: Workload, device="cpu", g_floor: Optional[float] = -5.0,
                      T: Optional[int] = None, seed: Optional[int] = None,
                      normalize_qk: bool = True) -> dict:
    """Draw q, k, v, g, beta (w.dtype), h0 (float32 or None), do (w.dtype), dht.

    ``T`` and ``seed`` override the workload's (used for ragged / scaled cases).
    ``normalize_qk=False`` leaves q and k as raw N(0,1) draws (for the kernels'
    own L2 normalisation).
    """
    T = w.T if T is None else T
    gen = _gen(w.seed if seed is None else seed, device)
    f32 = dict(dtype=torch.float32, device=device, generator=gen)
    B, H, HV, K, V = w.B, w.H, w.HV, w.K, w.V
    nrm = _l2norm if normalize_qk else (lambda x: x)
    q = nrm(torch.randn(B, T, H, K, **f32))
    k = nrm(torch.randn(B, T, H, K, **f32))
    v = torch.randn(B, T, HV, V, **f32)
    beta = torch.sigmoid(torch.randn(B, T, HV, **f32))
    g = -torch.nn.functional.softplus(torch.randn(B, T, HV, K, **f32) * w.g_sigma + w.g_mu)
    if g_floor is not None:
        g = g.clamp_min(g_floor)
    h0 = torch.randn(B, HV, K, V, **f32) * w.h0_std if w.h0_std is not None else None
    do = torch.randn(B, T, HV, V, **f32)
    dht = torch.randn(B, HV, K, V, **f32) if w.dht else None
    cast = lambda x: x.to(w.dtype).contiguous()
    return dict(q=cast(q), k=cast(k), v=cast(v), g=cast(g), beta=cast(beta), h0=h0,
                do=cast(do), dht=dht)


def make_decode_inputs(w: DecodeWorkload, device="cpu", steps: Optional[int] = None,
                       B: Optional[int] = None, normalize_qk: bool = True) -> dict:
    """Per-step q,k [S,B,H,K]; v [S,B,HV,V]; g [S,B,HV,K]; beta [S,B,HV]; state0."""
    steps = w.steps if steps is None else steps
    B = w.B if B is None else B
    gen = _gen(w.seed, device)
    f32 = dict(dtype=torch.float32, device=device, generator=gen)
    H, HV, K, V = w.H, w.HV, w.K, w.V
    state = torch.randn(B, HV, K, V, **f32) * w.state_std
    nrm = _l2norm if normalize_qk else (lambda x: x)
    q = nrm(torch.randn(steps, B, H, K, **f32))
    k = nrm(torch.randn(steps, B, H, K, **f32))
    v = torch.randn(steps, B, HV, V, **f32)
    beta = torch.sigmoid(torch.randn(steps, B, HV, **f32))
    g = (-torch.nn.functional.softplus(torch.randn(steps, B, HV, K, **f32) * w.g_sigma
                                       + w.g_mu)).clamp_min(-5.0)
    cast = lambda x: x.to(w.dtype).contiguous()
    return dict(q=cast(q), k=cast(k), v=cast(v), g=cast(g), beta=cast(beta), state=state)


def to_f64(x: Optional[torch.Tensor]):
    """Exact widening to a float64 numpy array (bf16 and fp32 embed in fp64)."""
    if x is None:
        return None
    return x.detach().to("cpu", torch.float64).numpy()
