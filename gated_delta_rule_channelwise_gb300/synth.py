"""Seeded synthetic inputs for the channelwise gated delta rule.

This module only draws random numbers and shapes their distributions; it
holds none of the method's arithmetic (no decay, no state update).  Where a
workload states "q, k L2-normalised", q and k rows are drawn N(0,1), scaled to
unit length in fp32 and then cast to the input dtype: that shapes the input
distribution, and the library still L2-normalises them itself (idempotent up
to eps and the cast).  Both the GPU path and the CPU oracle consume exactly the
tensors it returns (the oracle upcasts them exactly to fp64), so the two sides
see identical inputs.

Workloads (named by what they are):

=================  ===================================================================
``tiny_f32``       B=1, H=2, dk=dv=32, T=50, chunk 16 (ragged last chunk of 2), fp32
``gdn_decode_b1``  fused GatedDeltaNet decode, B=1, 16 k-heads -> 32 v-heads,
                   dk=dv=128, packed bf16 q|k|v row of width 8192, 256 steps
``decode_b64``     channelwise decode, B=64, H=32, dk=dv=128, bf16, 128 steps
``prefill_t4000``  channelwise chunked prefill, B=1, H=32, dk=dv=128, T=4000,
                   chunk 64 (ragged 32), bf16, zero initial state
``prefill_long``   B=4, H=32, dk=dv=128, T=16411, chunk 64 (ragged 27), bf16,
                   stronger decay g = -softplus(N(1,1)); then 64 decode steps
=================  ===================================================================

Distributions: q, k, v ~ N(0,1), with q and k rows scaled to unit length in
fp32 before the cast (all but the packed fused-decode row, whose projection is
raw; the library L2-normalises q and k itself either way);
per-channel log-decay g = -softplus(N(mu,1)) * scale; beta = sigmoid(N(0,1));
GatedDeltaNet gate inputs A_log ~ U(-1,1), dt_bias ~ N(0,1), a, b ~ N(0,1);
initial state ~ 0.1 * N(0,1) (std 0.1).  Draw order per seed: S0, then
(A_log, dt_bias), then q, k, v (or the packed row), then the gate noise.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    T: int                 # sequence length (prefill) or number of decode steps
    dtype: str             # "f32" or "bf16"
    gate: str              # "channel" or "gdn"
    chunk: int = 64
    packed: bool = False   # q|k|v in one packed row (fused decode)
    g_mu: float = 0.0
    g_scale: float = 0.5
    s0_std: float = 0.1
    seed: int = 0
    tail_steps: int = 0    # decode steps that follow a prefill
    qk_unit: bool = True   # q, k rows drawn at unit L2 length (fp32, before the cast); not for packed rows

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", B=1, Hk=2, Hv=2, dk=32, dv=32, T=50, dtype="f32",
                         gate="channel", chunk=16, seed=1001),
    "gdn_decode_b1": Workload("gdn_decode_b1", B=1, Hk=16, Hv=32, dk=128, dv=128, T=256,
                              dtype="bf16", gate="gdn", packed=True, seed=1002),
    "decode_b64": Workload("decode_b64", B=64, Hk=32, Hv=32, dk=128, dv=128, T=128,
                           dtype="bf16", gate="channel", seed=1003),
    "prefill_t4000": Workload("prefill_t4000", B=1, Hk=32, Hv=32, dk=128, dv=128, T=4000,
                              dtype="bf16", gate="channel", chunk=64, s0_std=0.0, seed=1004),
    "prefill_long": Workload("prefill_long", B=4, Hk=32, Hv=32, dk=128, dv=128, T=16411,
                             dtype="bf16", gate="channel", chunk=64, g_mu=1.0, g_scale=1.0,
                             seed=1005, tail_steps=64),
}


def make_inputs(w: Workload, *, T: Optional[int] = None, B: Optional[int] = None,
                device="cpu", seed: Optional[int] = None):
    """Draw one sequence of inputs for workload ``w``.

    Returns a dict with ``q, k [B,T,Hk,dk]``, ``v [B,T,Hv,dv]`` (views into one
    packed ``qkv [B,T,Hk*dk*2+Hv*dv]`` row when ``w.packed``), the gate
    (``g [B,T,Hv,dk]`` fp32 and ``beta [B,T,Hv]`` fp32, or ``a, b [B,T,Hv]`` in
    the input dtype with ``A_log, dt_bias [Hv]`` fp32) and ``S0 [B,Hv,dk,dv]``
    fp32.  For decode workloads token t is decode step t.
    """
    T = w.T if T is None else T
    B = w.B if B is None else B
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    dt = w.torch_dtype
    f32 = torch.float32

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=f32)

    out = {}
    out["S0"] = (randn(B, w.Hv, w.dk, w.dv) * w.s0_std) if w.s0_std > 0 else torch.zeros(
        B, w.Hv, w.dk, w.dv, device=device, dtype=f32)
    if w.gate == "gdn":
        out["A_log"] = torch.rand(w.Hv, generator=gen, device=device, dtype=f32) * 2.0 - 1.0
        out["dt_bias"] = randn(w.Hv)
    if w.packed:
        width = 2 * w.Hk * w.dk + w.Hv * w.dv
        qkv = randn(B, T, width).to(dt)
        out["qkv"] = qkv
        nq = w.Hk * w.dk
        out["q"] = qkv[..., :nq].unflatten(-1, (w.Hk, w.dk))
        out["k"] = qkv[..., nq:2 * nq].unflatten(-1, (w.Hk, w.dk))
        out["v"] = qkv[..., 2 * nq:].unflatten(-1, (w.Hv, w.dv))
    else:
        def qk_rows():
            x = randn(B, T, w.Hk, w.dk)
            if w.qk_unit:
                x = x / torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-12)
            return x.to(dt)
        out["q"] = qk_rows()
        out["k"] = qk_rows()
        out["v"] = randn(B, T, w.Hv, w.dv).to(dt)
    if w.gate == "gdn":
        out["a"] = randn(B, T, w.Hv).to(dt)
        out["b"] = randn(B, T, w.Hv).to(dt)
    else:
        noise = randn(B, T, w.Hv, w.dk) + w.g_mu
        out["g"] = -torch.nn.functional.softplus(noise) * w.g_scale
        out["beta"] = torch.sigmoid(randn(B, T, w.Hv))
    return out


def gate_kwargs(inp: dict) -> dict:
    """The gate entries of an input dict, as keyword arguments."""
    keys = ("g", "beta") if "g" in inp else ("a", "b", "A_log", "dt_bias")
    return {k: inp[k] for k in keys}
