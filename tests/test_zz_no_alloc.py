"""The allocation-free prefill entry point (cgdr_prefill_noalloc).

Some callers cannot allocate device memory while they run: runtimes that plan
every buffer ahead of time, or latency paths where a cudaMalloc could
synchronise the device.  cgdr_prefill_noalloc serves them by taking its
scratch from a static device array inside the library.  This file checks,
through the C ABI, that two calls in a row give the same results as the
regular entry point with a caller workspace, within the bf16-input tolerance
the parity tests use.  It is collected last on purpose.
"""
import ctypes

import pytest
import torch

import gated_delta_rule_channelwise_gb300 as cg
from gated_delta_rule_channelwise_gb300.synth import Workload, gate_kwargs, make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).abs().max() / b.pow(2).mean().sqrt().clamp_min(1e-30))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_channelwise_gb300 import build
    build.build()
    cg.lib()


@pytest.mark.parametrize("gate", ["channel", "gdn"])
def test_noalloc_matches_workspace_entry_point_twice(gate):
    w = Workload("noalloc", B=2, Hk=2, Hv=4, dk=128, dv=128, T=150, dtype="bf16", gate=gate, seed=61)
    inp = make_inputs(w, device="cuda")
    kw = gate_kwargs(inp)
    ref_state = inp["S0"].clone()
    ref_o = cg.prefill(inp["q"], inp["k"], inp["v"], ref_state, chunk=64, **kw)
    torch.cuda.synchronize()
    lib = cg.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):                      # two calls in a row share the static scratch
        state = inp["S0"].clone()
        o = torch.full(inp["v"].shape, float("nan"), dtype=torch.float32, device="cuda")
        A = cg.make_args(inp["q"], inp["k"], inp["v"], state, o, T=w.T, chunk=64, **kw)
        assert lib.cgdr_prefill_noalloc(ctypes.byref(A), stream) == cg.OK
        torch.cuda.synchronize()
        assert torch.isfinite(o).all()
        assert _rel(o, ref_o) <= TOL
        assert _rel(state, ref_state) <= TOL


def test_noalloc_rejects_bad_arguments():
    A = cg.CgdrArgs()
    A.B, A.T, A.Hk, A.Hv, A.dk, A.dv = 1, 4, 1, 1, 96, 128
    assert cg.lib().cgdr_prefill_noalloc(ctypes.byref(A), None) == cg.ERR_UNSUPPORTED
