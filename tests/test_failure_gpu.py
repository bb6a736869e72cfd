"""Failure detection of the bounded device waits, exercised without faulting the GPU.

Every wait in the kernels on data the kernel itself requested (a TMA tile, a
tensor-core commit) polls a bounded number of times; a wait that gives up
records CGDR_ERR_TIMEOUT in a status word, the kernel waits (with the full
limit) for its copies still in flight and returns, and the context stays
usable.  These tests make a wait give up on purpose through the library's
test hook (a negative ``wait_polls``: the first such wait of every block
targets a barrier that nothing ever completes, for a few polls -- a flag that
nothing sets), and inject the status word from the host.  Nothing here traps,
hangs or faults: the real copies of the abandoned step are still waited for
before each block exits.

The prefill workspace plays the part of the scratch arena of "Add parallel
chunked prefill for channelwise gated delta rule" (Summary); its first word
is the status word.
"""
import pytest
import torch

import gated_delta_rule_channelwise_gb300 as cg
from gated_delta_rule_channelwise_gb300.synth import Workload, gate_kwargs, make_inputs
from harness import TOL, decode_steps, oracle_run, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_channelwise_gb300 import build
    build.build()
    cg.lib()


def _inputs(T, B=1, H=1, gate="channel", seed=4):
    w = Workload("fail", B=B, Hk=H, Hv=H, dk=128, dv=128, T=T, dtype="bf16", gate=gate, seed=seed)
    return w, make_inputs(w, device="cuda")


def test_workspace_status_round_trip():
    """A status word written from the host reads back through cgdr_workspace_status, and the
    next prefill with that workspace clears it (each call starts from CGDR_OK)."""
    w, inp = _inputs(70)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ws.view(torch.int32)[0] = cg.ERR_TIMEOUT
    assert cg.workspace_status(ws) == cg.ERR_TIMEOUT
    state = inp["S0"].clone()
    cg.prefill(inp["q"], inp["k"], inp["v"], state, chunk=64, path=cg.PREFILL_PER_HEAD, workspace=ws,
               **gate_kwargs(inp))
    assert cg.workspace_status(ws) == cg.OK


def test_caller_status_word_is_never_cleared():
    """The optional caller status word: untouched by calls that succeed (so a code set earlier
    stays), zero after a clean call on a zeroed word."""
    w, inp = _inputs(1, B=2, H=2)
    st = torch.full((1,), cg.ERR_TIMEOUT, dtype=torch.int32, device="cuda")
    state = inp["S0"].clone()
    cg.decode(inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0], state, g=inp["g"][:, 0], beta=inp["beta"][:, 0],
              status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == cg.ERR_TIMEOUT
    st.zero_()
    cg.decode(inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0], state, g=inp["g"][:, 0], beta=inp["beta"][:, 0],
              status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == cg.OK


def test_decode_wait_gives_up():
    """The first tile wait of every block gives up (test hook).  The call reports
    CGDR_ERR_TIMEOUT, every unit has NaN in o and its state untouched, and a normal decode
    afterwards on the same context matches the oracle."""
    w, inp = _inputs(1, B=2, H=3)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = inp["S0"].clone()
    o = torch.zeros(inp["v"][:, 0].shape, dtype=torch.float32, device="cuda")
    cg.decode(inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0], state, o, g=inp["g"][:, 0], beta=inp["beta"][:, 0],
              status=st, wait_polls=-4)
    torch.cuda.synchronize()
    assert int(st.item()) == cg.ERR_TIMEOUT
    good_state = inp["S0"].clone()
    good_o = decode_steps(cg, inp, 1, good_state)[:, 0]
    torch.cuda.synchronize()
    assert torch.isnan(o).all()
    assert torch.equal(state, inp["S0"])
    o_ref, S_ref = oracle_run(inp)
    assert rel_err(good_o, o_ref[:, 0]) <= TOL[torch.bfloat16]
    assert rel_err(good_state, S_ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("path", [cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_COOP])
@pytest.mark.parametrize("gate", ["channel", "gdn"])
def test_prefill_wait_gives_up(gate, path):
    """A tensor-core prefill on one chunk of one head: the staging wait for the chunk's rows
    gives up (test hook) while those rows are still being copied in, and with it (cluster and
    cooperative kernels) the state CTA's wait for the chunk's hand-off; both status words read
    CGDR_ERR_TIMEOUT, the state is untouched, and a normal call afterwards on the same context
    and workspace matches the oracle."""
    w, inp = _inputs(64, gate=gate, seed=12)
    n = cg.prefill_workspace_size(inp["q"], inp["k"], inp["v"], inp["S0"], torch.empty(inp["v"].shape, device="cuda"),
                                  path=path, chunk=64, **gate_kwargs(inp))
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = inp["S0"].clone()
    cg.prefill(inp["q"], inp["k"], inp["v"], state, chunk=64, path=path, workspace=ws, status=st,
               wait_polls=-4, **gate_kwargs(inp))
    assert cg.workspace_status(ws) == cg.ERR_TIMEOUT
    assert int(st.item()) == cg.ERR_TIMEOUT
    assert torch.equal(state, inp["S0"])
    o = cg.prefill(inp["q"], inp["k"], inp["v"], state, chunk=64, path=path, workspace=ws, **gate_kwargs(inp))
    assert cg.workspace_status(ws) == cg.OK
    o_ref, S_ref = oracle_run(inp)
    assert rel_err(o, o_ref) <= TOL[torch.bfloat16]
    assert rel_err(state, S_ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("path", [cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_COOP])
def test_fp16_operand_range(path):
    """The tensor-core kernels carry some products in fp16 operands.  Inputs well inside the
    fp16 range report CGDR_OK; a v of magnitude 1e5 (a valid bf16 value beyond the largest
    fp16, 65504) reports CGDR_ERR_RANGE through both status words, and the fp32 CUDA-core
    kernel -- the remedy the header names -- runs the same call to the oracle's result."""
    w, inp = _inputs(200, H=2, seed=12)
    ref_ws = None
    for big in (False, True):
        v = inp["v"].clone()
        if big:
            v[0, 100, 1, 7] = 1.0e5
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.zeros(cg.prefill_workspace_size(inp["q"], inp["k"], v, inp["S0"],
                                                   torch.empty(v.shape, device="cuda"), path=path, chunk=64,
                                                   **gate_kwargs(inp)) + 256, dtype=torch.uint8, device="cuda")
        state = inp["S0"].clone()
        cg.prefill(inp["q"], inp["k"], v, state, chunk=64, path=path, workspace=ws, status=st, **gate_kwargs(inp))
        torch.cuda.synchronize()
        want = cg.ERR_RANGE if big else cg.OK
        assert int(st.item()) == want and cg.workspace_status(ws) == want
        if big:
            state = inp["S0"].clone()
            o = cg.prefill(inp["q"], inp["k"], v, state, chunk=64, path=cg.PREFILL_SIMT, **gate_kwargs(inp))
            o_ref, S_ref = oracle_run(dict(inp, v=v))
            assert rel_err(o, o_ref) <= TOL[torch.bfloat16] and rel_err(state, S_ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("path", [cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_COOP])
def test_growing_gate_range(path):
    """A positive log-decay (a gate that grows the state) scales keys by e^(sum of g); 64 tokens of
    g = +0.5 reach e^32, beyond fp16: CGDR_ERR_RANGE, not a silent overflow."""
    w, inp = _inputs(128, H=1, seed=13)
    g = torch.full_like(inp["g"], 0.5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = inp["S0"].clone()
    cg.prefill(inp["q"], inp["k"], inp["v"], state, chunk=64, path=path, status=st, g=g, beta=inp["beta"])
    torch.cuda.synchronize()
    assert int(st.item()) == cg.ERR_RANGE
