"""Shared helpers for the parity tests: run the oracle on host copies of the
very tensors the GPU consumed, optionally on a sample of (batch, v-head)
units, and measure errors the way the tolerance is stated (max abs error
relative to the RMS of the reference)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel_err(got, ref) -> float:
    got = np.asarray(got.detach().cpu().double() if isinstance(got, torch.Tensor) else got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(got - ref)) / max(rms, 1e-30))


def select_units(inp: dict, units, rep: int):
    """Gather the inputs of (b, h) units into a batch of single-head problems."""
    def take(x, b, h):
        return x[b:b + 1, :, h:h + 1]
    sel = {}
    for key in ("q", "k"):
        sel[key] = torch.cat([take(inp[key], b, h // rep) for b, h in units]).cpu()
    for key in ("v", "g", "beta", "a", "b"):
        if key in inp:
            sel[key] = torch.cat([take(inp[key], b, h) for b, h in units]).cpu()
    if "A_log" in inp:
        # one head per problem: gate parameters of that head, as a length-1 vector;
        # all problems share the same head index only if units do, so run per unit head
        sel["A_log"] = [inp["A_log"][h:h + 1].cpu() for _, h in units]
        sel["dt_bias"] = [inp["dt_bias"][h:h + 1].cpu() for _, h in units]
    sel["S0"] = torch.cat([inp["S0"][b:b + 1, h:h + 1] for b, h in units]).cpu()
    return sel


def oracle_run(inp: dict, *, units=None, rep: int = 1, S0=None, l2norm=True, q_scale=None):
    """Oracle on the whole input dict, or on the listed (b, h) units.

    Returns (o, S) with o [B', T, H', dv] and S [B', H', dk, dv]; for units,
    B' = len(units) and H' = 1, in the order given.
    """
    if units is None:
        kw = {k: inp[k].cpu() for k in ("g", "beta", "a", "b", "A_log", "dt_bias") if k in inp}
        s0 = inp["S0"].cpu() if S0 is None else S0
        return oracle.recurrence(inp["q"].cpu(), inp["k"].cpu(), inp["v"].cpu(), S0=s0,
                                 l2norm=l2norm, q_scale=q_scale, **kw)
    sel = select_units(inp, units, rep)
    s0 = sel["S0"] if S0 is None else S0
    if "g" in sel:
        return oracle.recurrence(sel["q"], sel["k"], sel["v"], g=sel["g"], beta=sel["beta"], S0=s0,
                                 l2norm=l2norm, q_scale=q_scale)
    # scalar gate: parameters differ per head, so run unit by unit in one process
    os_, Ss = [], []
    for i in range(len(units)):
        o, S = oracle.recurrence(sel["q"][i:i + 1], sel["k"][i:i + 1], sel["v"][i:i + 1],
                                 a=sel["a"][i:i + 1], b=sel["b"][i:i + 1], A_log=sel["A_log"][i],
                                 dt_bias=sel["dt_bias"][i], S0=s0[i:i + 1], l2norm=l2norm, q_scale=q_scale)
        os_.append(o)
        Ss.append(S)
    return np.concatenate(os_), np.concatenate(Ss)


def gather_units(x: torch.Tensor, units, head_dim: int):
    """x[b, ..., h, ...] for each unit, stacked along a new batch dim, head dim kept (size 1)."""
    out = []
    for b, h in units:
        sl = x[b:b + 1].narrow(head_dim, h, 1)
        out.append(sl)
    return torch.cat(out).cpu()


def decode_steps(cg, inp: dict, steps: int, state: torch.Tensor, *, l2norm=True, q_scale=None,
                 o_dtype=torch.float32):
    """Run `steps` decode calls over the token axis of `inp`; returns o [B, steps, Hv, dv]."""
    B, _, Hv, dv = inp["v"].shape
    o = torch.empty(B, steps, Hv, dv, dtype=o_dtype, device=inp["v"].device)
    for t in range(steps):
        kw = {}
        if "g" in inp:
            kw = dict(g=inp["g"][:, t], beta=inp["beta"][:, t])
        else:
            kw = dict(a=inp["a"][:, t], b=inp["b"][:, t], A_log=inp["A_log"], dt_bias=inp["dt_bias"])
        cg.decode(inp["q"][:, t], inp["k"][:, t], inp["v"][:, t], state, o[:, t], l2norm=l2norm,
                  q_scale=q_scale, **kw)
    return o
