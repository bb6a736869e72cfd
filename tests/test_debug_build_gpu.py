"""The index-checking build (libcgdr_debug.so) on the GPU.

libcgdr_debug.so is built from the same sources with every global-memory access of the kernels
tested against its tensor's footprint; a failed test records CGDR_ERR_BOUNDS in the status
words and skips the access (no trap, no fault).  Here it runs the small parity cases through
every kernel path -- the tiny fp32 workload (chunk 16, CUDA-core kernel), T in {1, 2, 3, 17}
on the token recurrence, the per-head and the cluster tensor-core kernels and the CUDA-core
kernel, both gates, and decode steps -- and each call must report CGDR_OK and match the
oracle.  A decode whose checked o footprint is shrunk shows that the checks fire: the last o
stores are skipped (their sentinel stays) and CGDR_ERR_BOUNDS is reported.
"""
import ctypes

import pytest
import torch

import gated_delta_rule_channelwise_gb300 as cg
from gated_delta_rule_channelwise_gb300 import build as cbuild
from gated_delta_rule_channelwise_gb300.synth import WORKLOADS, Workload, gate_kwargs, make_inputs
from harness import TOL, oracle_run, rel_err

pytestmark = pytest.mark.gpu

P = ctypes.POINTER(cg.CgdrArgs)


@pytest.fixture(scope="module")
def dlib():
    cbuild.build_all()
    L = ctypes.CDLL(cbuild.LIB_DEBUG)
    for name, res, args in [
        ("cgdr_decode", ctypes.c_int, [P, ctypes.c_void_p]),
        ("cgdr_prefill", ctypes.c_int, [P, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
        ("cgdr_prefill_workspace_size", ctypes.c_size_t, [P]),
        ("cgdr_workspace_status", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
        ("cgdr_debug_decode_shrunk_o", ctypes.c_int, [P, ctypes.c_int64, ctypes.c_void_p]),
    ]:
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    return L


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _prefill(L, inp, chunk, path):
    state = inp["S0"].clone()
    o = torch.empty(inp["v"].shape, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    A = cg.make_args(inp["q"], inp["k"], inp["v"], state, o, T=inp["q"].shape[1], chunk=chunk, path=path,
                     status=st, **gate_kwargs(inp))
    n = int(L.cgdr_prefill_workspace_size(ctypes.byref(A)))
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    assert L.cgdr_prefill(ctypes.byref(A), ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(ws.numel()), _stream()) == cg.OK
    torch.cuda.synchronize()
    assert int(st.item()) == cg.OK
    assert L.cgdr_workspace_status(ctypes.c_void_p(ws.data_ptr()), _stream()) == cg.OK
    return o, state


def test_tiny_f32_chunk16(dlib):
    w = WORKLOADS["tiny_f32"]
    inp = make_inputs(w, device="cuda")
    o, s = _prefill(dlib, inp, 16, cg.PREFILL_AUTO)
    o_ref, S_ref = oracle_run(inp)
    assert rel_err(o, o_ref) <= TOL[torch.float32] and rel_err(s, S_ref) <= TOL[torch.float32]


@pytest.mark.parametrize("T", [1, 2, 3, 17])
@pytest.mark.parametrize("path", [cg.PREFILL_AUTO, cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_SIMT])
@pytest.mark.parametrize("gate", ["channel", "gdn"])
def test_small_prefills_every_path(dlib, T, path, gate):
    w = Workload("dbg", B=2, Hk=1, Hv=2, dk=128, dv=128, T=T, dtype="bf16", gate=gate, seed=70 + T)
    inp = make_inputs(w, device="cuda")
    o, s = _prefill(dlib, inp, 64, path)
    o_ref, S_ref = oracle_run(inp, rep=2)
    assert rel_err(o, o_ref) <= TOL[torch.bfloat16] and rel_err(s, S_ref) <= TOL[torch.bfloat16]


def _decode_args(inp, state, o, st):
    u = lambda t: t[:, 0].unsqueeze(1)
    kw = {"g": u(inp["g"]), "beta": u(inp["beta"])} if "g" in inp else \
        {"a": u(inp["a"]), "b": u(inp["b"]), "A_log": inp["A_log"], "dt_bias": inp["dt_bias"]}
    return cg.make_args(u(inp["q"]), u(inp["k"]), u(inp["v"]), state, o.unsqueeze(1), T=1, status=st, **kw)


@pytest.mark.parametrize("gate", ["channel", "gdn"])
def test_decode_step(dlib, gate):
    w = Workload("dbgd", B=3, Hk=2, Hv=4, dk=128, dv=64, T=1, dtype="bf16", gate=gate, seed=9)
    inp = make_inputs(w, device="cuda")
    state = inp["S0"].clone()
    o = torch.empty(inp["v"][:, 0].shape, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    A = _decode_args(inp, state, o, st)
    assert dlib.cgdr_decode(ctypes.byref(A), _stream()) == cg.OK
    torch.cuda.synchronize()
    assert int(st.item()) == cg.OK
    o_ref, S_ref = oracle_run(inp, rep=2)
    assert rel_err(o, o_ref[:, 0]) <= TOL[torch.bfloat16] and rel_err(state, S_ref) <= TOL[torch.bfloat16]


def test_checks_fire_on_a_shrunk_footprint(dlib):
    """o's checked footprint 4 elements short: the last 4 o values of the last (batch, head) are
    skipped and CGDR_ERR_BOUNDS is reported; everything else matches a normal decode."""
    w = Workload("dbgs", B=2, Hk=2, Hv=2, dk=64, dv=64, T=1, dtype="f32", gate="channel", seed=10)
    inp = make_inputs(w, device="cuda")
    sentinel = -12345.0
    outs = []
    for shrink in (0, 4):
        state = inp["S0"].clone()
        o = torch.full(inp["v"][:, 0].shape, sentinel, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        A = _decode_args(inp, state, o, st)
        assert dlib.cgdr_debug_decode_shrunk_o(ctypes.byref(A), shrink, _stream()) == cg.OK
        torch.cuda.synchronize()
        outs.append((o, state, int(st.item())))
    (o0, s0, st0), (o4, s4, st4) = outs
    assert st0 == cg.OK and st4 == cg.ERR_BOUNDS
    assert torch.equal(s0, s4)
    flat0, flat4 = o0.reshape(-1), o4.reshape(-1)
    assert torch.equal(flat4[:-4], flat0[:-4])
    assert torch.all(flat4[-4:] == sentinel) and not torch.any(flat0[-4:] == sentinel)
