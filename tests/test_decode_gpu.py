"""GPU parity of cgdr_decode against the fp64 oracle (token recurrence).

Tolerance (max abs error / RMS of the reference): 1e-4 for fp32 inputs,
2e-2 for bf16 inputs, on o over every step and on the final state."""
import numpy as np
import pytest
import torch

import gated_delta_rule_channelwise_gb300 as cg
from gated_delta_rule_channelwise_gb300.synth import WORKLOADS, Workload, make_inputs
from harness import TOL, decode_steps, oracle_run, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_channelwise_gb300 import build
    build.build()
    cg.lib()


def _run_and_compare(w: Workload, steps: int, units=None, l2norm=True, q_scale=None, inp=None):
    inp = inp or make_inputs(w, T=steps, device="cuda")
    state = inp["S0"].clone()
    o = decode_steps(cg, inp, steps, state, l2norm=l2norm, q_scale=q_scale)
    torch.cuda.synchronize()
    rep = w.Hv // w.Hk
    o_ref, S_ref = oracle_run(inp, units=units, rep=rep, l2norm=l2norm, q_scale=q_scale)
    if units is not None:
        o = torch.cat([o[b:b + 1, :, h:h + 1] for b, h in units])
        state = torch.cat([state[b:b + 1, h:h + 1] for b, h in units])
    tol = TOL[w.torch_dtype]
    eo, es = rel_err(o, o_ref), rel_err(state, S_ref)
    print("[parity] %s steps=%d dk=%d dv=%d err_o=%.3e err_S=%.3e" % (w.name, steps, w.dk, w.dv, eo, es))
    assert eo <= tol, ("o", eo)
    assert es <= tol, ("state", es)
    return eo, es


def test_tiny_f32_as_decode_steps():
    """The tiny fp32 workload run as 50 consecutive decode calls."""
    _run_and_compare(WORKLOADS["tiny_f32"], 50)


@pytest.mark.parametrize("dk", [32, 64, 128])
@pytest.mark.parametrize("dv", [32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("gate", ["channel", "gdn"])
def test_shapes_dtypes_gates(dk, dv, dtype, gate):
    w = Workload("shape", B=3, Hk=2, Hv=4, dk=dk, dv=dv, T=6, dtype=dtype, gate=gate, seed=dk * 7 + dv)
    _run_and_compare(w, 6)


def test_gdn_packed_decode_b1_full():
    """Fused GatedDeltaNet decode: packed bf16 q|k|v row, 16 k-heads -> 32 v-heads, 256 steps."""
    w = WORKLOADS["gdn_decode_b1"]
    inp = make_inputs(w, device="cuda")
    assert inp["q"].data_ptr() == inp["qkv"].data_ptr()          # zero-copy split
    _run_and_compare(w, w.T, inp=inp)


def test_gdn_decode_b1_cuda_graph_sequence():
    """The fused decode at B=1 as the benchmark times it: 256 consecutive steps captured once
    as a CUDA graph and replayed from the initial state (the kernel-count reduction of "Add
    fused GatedDeltaNet decode Triton kernel", description).  Every step's o and the final
    state are checked against the oracle."""
    w = WORKLOADS["gdn_decode_b1"]
    inp = make_inputs(w, device="cuda")
    st = inp["S0"].clone()
    o = torch.empty(w.T, 1, w.Hv, w.dv, dtype=torch.float32, device="cuda")

    def steps():
        for t in range(w.T):
            cg.decode(inp["q"][:, t], inp["k"][:, t], inp["v"][:, t], st, o[t], a=inp["a"][:, t], b=inp["b"][:, t],
                      A_log=inp["A_log"], dt_bias=inp["dt_bias"])

    steps()                                   # eager first: per-device set-up happens outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        steps()
    st.copy_(inp["S0"])
    o.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    o_ref, S_ref = oracle_run(inp, rep=w.Hv // w.Hk)
    got_o = o.permute(1, 0, 2, 3)             # [1, 256, 32, 128]
    eo, es = rel_err(got_o, o_ref), rel_err(st, S_ref)
    print("[parity] gdn_decode_b1 graph err_o=%.3e err_S=%.3e" % (eo, es))
    assert eo <= TOL[torch.bfloat16] and es <= TOL[torch.bfloat16]


def test_decode_b64_full_size_sampled():
    """B=64, H=32, 128 steps on the GPU; the oracle checks 24 sampled (b, h) units."""
    w = WORKLOADS["decode_b64"]
    rng = np.random.default_rng(0)
    units = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 24), rng.integers(0, 32, 24))})
    units += [(0, 0), (63, 31)]
    _run_and_compare(w, w.T, units=units)


def test_no_l2norm_custom_scale():
    """l2norm off with pre-normalised q, k and an explicit q scale."""
    w = Workload("nonorm", B=2, Hk=1, Hv=2, dk=64, dv=64, T=8, dtype="f32", gate="channel", seed=5)
    inp = make_inputs(w, device="cuda")
    for key in ("q", "k"):
        x = inp[key]
        inp[key] = x / x.norm(dim=-1, keepdim=True)
    _run_and_compare(w, 8, l2norm=False, q_scale=0.3, inp=inp)


def test_zero_batch_is_noop():
    z = torch.empty(0, 2, 128, device="cuda", dtype=torch.bfloat16)
    v = torch.empty(0, 2, 128, device="cuda", dtype=torch.bfloat16)
    s = torch.empty(0, 2, 128, 128, device="cuda")
    g = torch.empty(0, 2, 128, device="cuda")
    be = torch.empty(0, 2, device="cuda")
    cg.decode(z, z, v, s, g=g, beta=be)


def test_identity_gate_keeps_state_exactly():
    """alpha = 1, beta = 0 leaves every state element bit-identical (both sweeps)."""
    w = Workload("ident", B=4, Hk=4, Hv=4, dk=128, dv=128, T=1, dtype="bf16", gate="channel", seed=11)
    inp = make_inputs(w, device="cuda")
    state = inp["S0"].clone()
    cg.decode(inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0], state,
              g=torch.zeros_like(inp["g"][:, 0]), beta=torch.zeros_like(inp["beta"][:, 0]))
    torch.cuda.synchronize()
    assert torch.equal(state, inp["S0"])


@pytest.mark.parametrize("dk,dv", [(128, 128), (32, 64)])
def test_bf16_output_is_the_rounded_fp32_output(dk, dv):
    """o in bf16 is exactly the fp32 result rounded to nearest (same kernel, same inputs)."""
    w = Workload("obf", B=5, Hk=2, Hv=4, dk=dk, dv=dv, T=3, dtype="bf16", gate="channel", seed=19)
    inp = make_inputs(w, device="cuda")
    s1, s2 = inp["S0"].clone(), inp["S0"].clone()
    o32 = decode_steps(cg, inp, 3, s1)
    o16 = decode_steps(cg, inp, 3, s2, o_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(s1, s2)
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_scalar_gate_equals_broadcast_channel_gate():
    """Decode: the scalar gate is the channelwise gate with one g broadcast over dk."""
    import torch.nn.functional as F
    w = Workload("gbd", B=3, Hk=2, Hv=4, dk=128, dv=64, T=4, dtype="bf16", gate="gdn", seed=321)
    inp = make_inputs(w, device="cuda")
    g1 = -torch.exp(inp["A_log"])[None, None, :] * F.softplus(inp["a"].float() + inp["dt_bias"][None, None, :])
    chan = {k: inp[k] for k in ("q", "k", "v", "S0")}
    chan["g"] = g1[..., None].expand(-1, -1, -1, w.dk).contiguous()
    chan["beta"] = torch.sigmoid(inp["b"].float()).contiguous()
    s1, s2 = inp["S0"].clone(), inp["S0"].clone()
    o1 = decode_steps(cg, inp, 4, s1)
    o2 = decode_steps(cg, chan, 4, s2)
    torch.cuda.synchronize()
    assert rel_err(o1, o2.double().cpu().numpy()) <= 1e-4
    assert rel_err(s1, s2.double().cpu().numpy()) <= 1e-4
