"""GPU parity of cgdr_prefill (chunked WY/UT form) against the fp64 oracle.

The oracle is the token recurrence; the chunked form must reach the same
result for every chunk length and tail position ("Add parallel chunked
prefill for channelwise gated delta rule", Summary).  Tolerance: 1e-4 for
fp32 inputs, 2e-2 for bf16 inputs (max abs error / RMS of the reference),
on o and on the final state."""
import numpy as np
import pytest
import torch

import gated_delta_rule_channelwise_gb300 as cg
from gated_delta_rule_channelwise_gb300.synth import WORKLOADS, Workload, gate_kwargs, make_inputs
from harness import TOL, decode_steps, oracle_run, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_channelwise_gb300 import build
    build.build()
    cg.lib()


TC_PATHS = [pytest.param(cg.PREFILL_PER_HEAD, id="per_head"), pytest.param(cg.PREFILL_CLUSTER, id="cluster"),
            pytest.param(cg.PREFILL_COOP, id="coop")]


def _ws_bytes(path, units):
    """Workspace of each tensor-core kernel: the status word, then (cluster) nine 82432-byte
    hand-off slots per (batch, v-head), or (cooperative) 16 sequence numbers and eight slots."""
    if path == cg.PREFILL_PER_HEAD:
        return 256
    if path == cg.PREFILL_CLUSTER:
        return 256 + units * 9 * 82432
    return 256 + (64 * units + 255) // 256 * 256 + units * 8 * 82432


@pytest.fixture(params=TC_PATHS)
def tc_path(request):
    """Runs the test once per tensor-core prefill kernel (the choice is passed with each call)."""
    return request.param


@pytest.fixture
def simt_path():
    """The chunked CUDA-core kernel (a small T would otherwise run the token recurrence)."""
    return cg.PREFILL_SIMT


def _expect_path(inp, expected, path=cg.PREFILL_AUTO):
    o = torch.empty(inp["v"].shape, device=inp["v"].device)
    got = cg.prefill_path_for(inp["q"], inp["k"], inp["v"], inp["S0"], o, chunk=64, path=path, **gate_kwargs(inp))
    assert got == expected


def _prefill(inp, chunk, state=None, path=cg.PREFILL_AUTO, **kw):
    state = inp["S0"].clone() if state is None else state
    o = cg.prefill(inp["q"], inp["k"], inp["v"], state, chunk=chunk, path=path, **gate_kwargs(inp), **kw)
    torch.cuda.synchronize()
    return o, state


def _check(w, inp, o, state, units=None, tol=None):
    o_ref, S_ref = oracle_run(inp, units=units, rep=w.Hv // w.Hk)
    if units is not None:
        o = torch.cat([o[b:b + 1, :, h:h + 1] for b, h in units])
        state = torch.cat([state[b:b + 1, h:h + 1] for b, h in units])
    tol = tol or TOL[w.torch_dtype]
    eo, es = rel_err(o, o_ref), rel_err(state, S_ref)
    print("[parity] %s T=%d dv=%d err_o=%.3e err_S=%.3e" % (w.name, o.shape[1], w.dv, eo, es))
    assert eo <= tol, ("o", eo)
    assert es <= tol, ("state", es)
    return eo, es


def test_tiny_f32_chunk16():
    """B=1, H=2, dk=dv=32, T=50, chunk 16 (ragged 2), fp32: the CUDA-core chunked path."""
    w = WORKLOADS["tiny_f32"]
    inp = make_inputs(w, device="cuda")
    o, s = _prefill(inp, 16)
    _check(w, inp, o, s)


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("T", [1, 2, 17, 64, 100])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 32), (128, 64)])
def test_fp32_chunk_sizes_and_tails(chunk, T, dk, dv, simt_path):
    w = Workload("f32", B=2, Hk=1, Hv=2, dk=dk, dv=dv, T=T, dtype="f32", gate="channel", seed=T + chunk)
    inp = make_inputs(w, device="cuda")
    _expect_path(inp, cg.PREFILL_SIMT, simt_path)
    o, s = _prefill(inp, chunk, path=simt_path)
    _check(w, inp, o, s)


@pytest.mark.parametrize("T", [1, 2, 31, 63, 64, 65, 127, 200])
@pytest.mark.parametrize("dv", [32, 64, 128])
@pytest.mark.parametrize("gate", ["channel", "gdn"])
def test_tensor_core_path_tails(T, dv, gate, tc_path):
    if dv != 128 and tc_path != cg.PREFILL_PER_HEAD:
        pytest.skip("dv < 128 runs the CUDA-core kernel whatever the choice")
    w = Workload("tc", B=2, Hk=1, Hv=2, dk=128, dv=dv, T=T, dtype="bf16", gate=gate, seed=T * 3 + dv)
    inp = make_inputs(w, device="cuda")
    _expect_path(inp, tc_path if dv == 128 else cg.PREFILL_SIMT, tc_path)
    o, s = _prefill(inp, 64, path=tc_path)
    _check(w, inp, o, s)


@pytest.mark.parametrize("chunk", [16, 32])
def test_bf16_cuda_core_chunks_agree(chunk):
    """bf16 inputs with chunk 16/32 run the CUDA-core kernel; both paths match the oracle."""
    w = Workload("bfc", B=1, Hk=2, Hv=2, dk=128, dv=128, T=150, dtype="bf16", gate="channel", seed=chunk)
    inp = make_inputs(w, device="cuda")
    o1, s1 = _prefill(inp, chunk)
    o2, s2 = _prefill(inp, 64)
    _check(w, inp, o1, s1)
    _check(w, inp, o2, s2)


def test_strong_decay_anchoring(tc_path):
    """Log-decay near -3 per token (-190 per chunk): e^-gamma would overflow fp32 without anchoring."""
    w = Workload("strong", B=1, Hk=2, Hv=2, dk=128, dv=128, T=300, dtype="bf16", gate="channel",
                 g_mu=3.0, g_scale=1.0, seed=77)
    inp = make_inputs(w, device="cuda")
    o, s = _prefill(inp, 64, path=tc_path)
    _check(w, inp, o, s)


def test_head_repeat_prefill(tc_path):
    w = Workload("rep", B=2, Hk=2, Hv=8, dk=128, dv=128, T=90, dtype="bf16", gate="channel", seed=3)
    inp = make_inputs(w, device="cuda")
    o, s = _prefill(inp, 64, path=tc_path)
    _check(w, inp, o, s)


def test_prefill_t4000_full(tc_path):
    """B=1, H=32, dk=dv=128, T=4000, chunk 64 (ragged 32), zero initial state: every unit checked."""
    w = WORKLOADS["prefill_t4000"]
    inp = make_inputs(w, device="cuda")
    _expect_path(inp, tc_path, tc_path)
    o, s = _prefill(inp, 64, path=tc_path)
    _check(w, inp, o, s)


def test_prefill_t4000_as_benchmarked_bf16_o():
    """The configuration the benchmark times -- T = 4000, 32 heads, automatic kernel choice,
    o in bf16 -- gives exactly the bf16 rounding of the fp32-o result (whose parity with the
    oracle test_prefill_t4000_full checks) and the same final state."""
    w = WORKLOADS["prefill_t4000"]
    inp = make_inputs(w, device="cuda")
    o32, s32 = _prefill(inp, 64)
    s16 = inp["S0"].clone()
    o16 = torch.empty(inp["v"].shape, dtype=torch.bfloat16, device="cuda")
    cg.prefill(inp["q"], inp["k"], inp["v"], s16, o16, chunk=64, **gate_kwargs(inp))
    torch.cuda.synchronize()
    assert torch.equal(s16, s32)
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_prefill_long_then_decode_sampled(tc_path):
    """B=4, H=32, T=16411 (ragged 27), strong decay; then 64 decode steps from the final state.
    Eight sampled (b, h) units are checked against the oracle over all T + 64 tokens."""
    w = WORKLOADS["prefill_long"]
    inp = make_inputs(w, device="cuda")
    o, s = _prefill(inp, 64, path=tc_path)
    units = [(0, 0), (0, 31), (1, 7), (2, 16), (3, 3), (3, 30), (1, 22), (2, 9)]
    tail = make_inputs(w, T=w.tail_steps, device="cuda", seed=w.seed + 1)
    o_tail = decode_steps(cg, tail, w.tail_steps, s)
    torch.cuda.synchronize()
    # oracle: prefill units, then continue the same units over the decode tail
    o_ref, S_ref = oracle_run(inp, units=units)
    tail_ref_o, tail_ref_S = oracle_run(tail, units=units, S0=S_ref)
    got_o = torch.cat([o[b:b + 1, :, h:h + 1] for b, h in units])
    got_t = torch.cat([o_tail[b:b + 1, :, h:h + 1] for b, h in units])
    got_S = torch.cat([s[b:b + 1, h:h + 1] for b, h in units])
    tol = TOL[torch.bfloat16]
    print("[parity] prefill_long err_o=%.3e tail_o=%.3e S=%.3e" % (
        rel_err(got_o, o_ref), rel_err(got_t, tail_ref_o), rel_err(got_S, tail_ref_S)))
    assert rel_err(got_o, o_ref) <= tol
    assert rel_err(got_t, tail_ref_o) <= tol
    assert rel_err(got_S, tail_ref_S) <= tol
    assert torch.isfinite(s).all()


@pytest.mark.parametrize("path", [cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_AUTO])
def test_more_heads_than_sms(path):
    """B=3 x 64 v-heads over 32 k-heads = 192 (batch, head) units, more than the GPU's SMs: the
    per-head kernel runs in two waves, the cluster kernel in several rounds of clusters, and the
    automatic choice takes one of them (the cooperative kernel needs a CTA per head at once).
    Sampled units from every wave against the oracle; the kernels agree with each other within
    the sum of their distances from the oracle (each ~6e-3 of the RMS here, rounded differently:
    TF32 state products in the per-head kernel, fp16 in the cluster kernel)."""
    w = Workload("waves", B=3, Hk=32, Hv=64, dk=128, dv=128, T=150, dtype="bf16", gate="channel", seed=63)
    inp = make_inputs(w, device="cuda")
    if path != cg.PREFILL_AUTO:
        _expect_path(inp, path, path)
    o, s = _prefill(inp, 64, path=path)
    _check(w, inp, o, s, units=[(0, 0), (0, 63), (1, 20), (2, 0), (2, 55), (2, 63)])
    o_ph, s_ph = _prefill(inp, 64, path=cg.PREFILL_PER_HEAD)
    assert rel_err(o, o_ph.double().cpu().numpy()) <= 1e-2 and rel_err(s, s_ph.double().cpu().numpy()) <= 1e-2


def test_prefill_T1_matches_decode():
    w = Workload("t1", B=3, Hk=2, Hv=4, dk=128, dv=128, T=1, dtype="bf16", gate="gdn", seed=8)
    inp = make_inputs(w, device="cuda")
    o_p, s_p = _prefill(inp, 64)
    s_d = inp["S0"].clone()
    o_d = decode_steps(cg, inp, 1, s_d)
    torch.cuda.synchronize()
    assert rel_err(o_p, o_d.double().cpu().numpy()) <= 1e-2
    assert rel_err(s_p, s_d.double().cpu().numpy()) <= 1e-2


def test_prefill_continuation(tc_path):
    """prefill(T1) then prefill(T2) from the carried state equals the oracle over T1 + T2."""
    w = Workload("cont", B=2, Hk=2, Hv=2, dk=128, dv=128, T=230, dtype="bf16", gate="channel", seed=21)
    inp = make_inputs(w, device="cuda")
    first = {k: (v[:, :100] if v.dim() >= 2 and v.shape[1] == 230 else v) for k, v in inp.items()}
    second = {k: (v[:, 100:] if v.dim() >= 2 and v.shape[1] == 230 else v) for k, v in inp.items()}
    o1, s = _prefill(first, 64, path=tc_path)
    o2, s = _prefill(second, 64, state=s, path=tc_path)
    _check(w, inp, torch.cat([o1, o2], dim=1), s)


def test_zero_length_is_noop():
    w = Workload("z", B=1, Hk=1, Hv=1, dk=128, dv=128, T=0, dtype="bf16", gate="channel", seed=1)
    inp = make_inputs(w, device="cuda")
    s = inp["S0"].clone()
    _prefill(inp, 64, state=s)
    assert torch.equal(s, inp["S0"])


@pytest.mark.parametrize("dtype,chunk", [("bf16", 64), ("bf16", 32), ("f32", 16)])
def test_bf16_output_is_the_rounded_fp32_output(dtype, chunk, tc_path):
    w = Workload("obf", B=1, Hk=2, Hv=2, dk=128, dv=128, T=77, dtype=dtype, gate="channel", seed=23)
    inp = make_inputs(w, device="cuda")
    o32, s1 = _prefill(inp, chunk, path=tc_path)
    o16 = torch.empty(o32.shape, dtype=torch.bfloat16, device="cuda")
    s2 = inp["S0"].clone()
    cg.prefill(inp["q"], inp["k"], inp["v"], s2, o16, chunk=chunk, path=tc_path, **gate_kwargs(inp))
    torch.cuda.synchronize()
    assert torch.equal(s1, s2)
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_tensor_core_path_reports_ok_status(tc_path):
    """The tensor-core prefill leaves CGDR_OK in its workspace status word."""
    w = Workload("st", B=1, Hk=1, Hv=1, dk=128, dv=128, T=70, dtype="bf16", gate="channel", seed=4)
    inp = make_inputs(w, device="cuda")
    state = inp["S0"].clone()
    n = cg.prefill_workspace_size(inp["q"], inp["k"], inp["v"], state, torch.empty(inp["v"].shape, device="cuda"),
                                  path=tc_path, **gate_kwargs(inp))
    assert n == _ws_bytes(tc_path, 1)
    ws = torch.full((n,), 0x7F, dtype=torch.uint8, device="cuda")
    cg.prefill(inp["q"], inp["k"], inp["v"], state, chunk=64, path=tc_path, workspace=ws, **gate_kwargs(inp))
    assert cg.workspace_status(ws) == cg.OK


def test_mixed_wide_and_narrow_chunks(tc_path):
    """Decay that switches between mild and extreme across chunks (both A/P paths in one call)."""
    w = Workload("mix", B=1, Hk=2, Hv=2, dk=128, dv=128, T=260, dtype="bf16", gate="channel", seed=31)
    inp = make_inputs(w, device="cuda")
    g = inp["g"].clone()
    g[:, 64:128] *= 12.0          # second chunk: ~ -5 per token on average
    inp["g"] = g
    o, s = _prefill(inp, 64, path=tc_path)
    _check(w, inp, o, s)


def test_tensor_core_kernels_agree():
    """The three tensor-core kernels run the same chunk algorithm; the cluster and the
    cooperative kernel also run the very same per-chunk code (only the hand-off between their
    CTAs differs), so those two agree bit for bit, and with the per-head kernel (TF32 state
    products where they use fp16) far inside the oracle tolerance."""
    w = Workload("agree", B=1, Hk=2, Hv=4, dk=128, dv=128, T=700, dtype="bf16", gate="channel", seed=55)
    inp = make_inputs(w, device="cuda")
    (o1, s1), (o2, s2), (o3, s3) = [_prefill(inp, 64, path=path)
                                    for path in (cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_COOP)]
    eo, es = rel_err(o2, o1.double().cpu().numpy()), rel_err(s2, s1.double().cpu().numpy())
    print("[kernels] o %.3e S %.3e" % (eo, es))
    assert eo <= 5e-3 and es <= 5e-3
    assert torch.equal(o3, o2) and torch.equal(s3, s2)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("dtype,gate,dk,dv", [("bf16", "channel", 128, 128), ("bf16", "gdn", 128, 128),
                                              ("f32", "channel", 32, 64), ("f32", "gdn", 64, 32)])
def test_recurrent_small_T(T, dtype, gate, dk, dv):
    """1 <= T <= 8 runs the token recurrence (the decode kernel stepping through the tokens with
    the state tile held on chip): parity with the oracle, and the result of T
    single-token decode calls (up to the compiler's choice of fused multiply-adds)."""
    w = Workload("rec", B=3, Hk=2, Hv=4, dk=dk, dv=dv, T=T, dtype=dtype, gate=gate, seed=40 + T)
    inp = make_inputs(w, device="cuda")
    _expect_path(inp, cg.PREFILL_RECURRENT)
    o, s = _prefill(inp, 64)
    _check(w, inp, o, s, tol=TOL[torch.float32])
    s_d = inp["S0"].clone()
    o_d = decode_steps(cg, inp, T, s_d)
    torch.cuda.synchronize()
    # the same per-token arithmetic in both launches (the compiler may contract it differently)
    assert rel_err(s, s_d.double().cpu().numpy()) <= 1e-5
    assert rel_err(o, o_d.double().cpu().numpy()) <= 1e-5


def test_recurrent_matches_chunked_kernels():
    """T = 8 by the token recurrence and by each chunked kernel: the same result up to rounding."""
    w = Workload("rec8", B=2, Hk=2, Hv=2, dk=128, dv=128, T=8, dtype="bf16", gate="channel", seed=77)
    inp = make_inputs(w, device="cuda")
    o_r, s_r = _prefill(inp, 64)
    for path in (cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_COOP, cg.PREFILL_SIMT):
        _expect_path(inp, path, path)
        o_c, s_c = _prefill(inp, 64, path=path)
        assert rel_err(o_c, o_r.double().cpu().numpy()) <= 2e-2
        assert rel_err(s_c, s_r.double().cpu().numpy()) <= 2e-2


@pytest.mark.parametrize("T", [5, 200])
def test_packed_gdn_prefill(T, tc_path):
    """The fused GatedDeltaNet layout in prefill: q | k | v views into one packed bf16 row per
    token (16 k-heads repeated to 32 v-heads), scalar gate; the tensor maps take the row's
    strides.  T = 5 is one ragged chunk, T = 200 four chunks."""
    w = Workload("pk", B=2, Hk=16, Hv=32, dk=128, dv=128, T=T, dtype="bf16", gate="gdn", packed=True, seed=90 + T)
    inp = make_inputs(w, device="cuda")
    assert inp["q"].stride(1) == 16 * 128 * 2 + 32 * 128          # a view into the packed row
    o, s = _prefill(inp, 64, path=tc_path)
    _check(w, inp, o, s, units=[(0, 0), (0, 1), (1, 17), (1, 31)])


def test_packed_gdn_prefill_recurrent():
    """The same packed layout with T = 5 under the automatic choice: the token recurrence."""
    w = Workload("pkr", B=2, Hk=16, Hv=32, dk=128, dv=128, T=5, dtype="bf16", gate="gdn", packed=True, seed=97)
    inp = make_inputs(w, device="cuda")
    _expect_path(inp, cg.PREFILL_RECURRENT)
    o, s = _prefill(inp, 64)
    _check(w, inp, o, s, units=[(0, 0), (0, 1), (1, 17), (1, 31)], tol=TOL[torch.float32])


@pytest.mark.parametrize("path", [cg.PREFILL_PER_HEAD, cg.PREFILL_CLUSTER, cg.PREFILL_SIMT, cg.PREFILL_RECURRENT])
def test_scalar_gate_equals_broadcast_channel_gate(path):
    """The scalar GatedDeltaNet gate is the channelwise gate with one g broadcast over dk: the
    same call with g = -exp(A_log) softplus(a + dt_bias) expanded to every channel and
    beta = sigmoid(b) gives the same result (up to the rounding of the gate itself, computed
    by torch here and on the device there), on every prefill kernel."""
    import torch.nn.functional as F
    T = 5 if path == cg.PREFILL_RECURRENT else 150
    w = Workload("gb", B=2, Hk=2, Hv=4, dk=128, dv=128, T=T, dtype="bf16", gate="gdn", seed=123)
    inp = make_inputs(w, device="cuda")
    g1 = -torch.exp(inp["A_log"])[None, None, :] * F.softplus(inp["a"].float() + inp["dt_bias"][None, None, :])
    chan = dict(inp)
    chan["g"] = g1[..., None].expand(-1, -1, -1, w.dk).contiguous()
    chan["beta"] = torch.sigmoid(inp["b"].float()).contiguous()
    for key in ("a", "b", "A_log", "dt_bias"):
        chan.pop(key)
    o1, s1 = _prefill(inp, 64, path=path)
    o2, s2 = _prefill(chan, 64, path=path)
    eo = rel_err(o1, o2.double().cpu().numpy())
    es = rel_err(s1, s2.double().cpu().numpy())
    print("[gate] path %d o %.3e S %.3e" % (path, eo, es))
    assert eo <= 1e-3 and es <= 1e-3
