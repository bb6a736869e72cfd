"""Pins for the fp64 oracle, independent of the oracle itself.

Each test checks the oracle against something the pages or plain mathematics
fix: a hand-worked example, closed forms of special cases, invariants of the
recurrence, a brute-force dense-matrix restatement, and the chunked WY/UT
form of "Add parallel chunked prefill for channelwise gated delta rule"
(executorch PR #21061), which must agree with the token recurrence.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(12345)


def _rand_case(B=2, T=7, Hk=1, Hv=2, dk=5, dv=3, g_scale=0.5, s0=True, seed=0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, Hk, dk))
    k = r.standard_normal((B, T, Hk, dk))
    v = r.standard_normal((B, T, Hv, dv))
    g = -np.log1p(np.exp(r.standard_normal((B, T, Hv, dk)))) * g_scale
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, Hv))))
    S0 = r.standard_normal((B, Hv, dk, dv)) * 0.3 if s0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0)


def _unit(x, eps=0.0):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def test_golden_worked_example():
    """Hand-worked two-token example (tests/golden/worked_example_dk2.json)."""
    d = json.load(open(os.path.join(HERE, "golden", "worked_example_dk2.json")))
    i = {k: np.array(v) if isinstance(v, list) else v for k, v in d["inputs"].items()}
    o, S = oracle.recurrence(i["q"], i["k"], i["v"], g=i["g"], beta=i["beta"], S0=i["S0"],
                             eps=i["eps"], q_scale=i["q_scale"])
    np.testing.assert_allclose(o, np.array(d["expected"]["o"]), atol=1e-12)
    np.testing.assert_allclose(S, np.array(d["expected"]["S"]), atol=1e-12)


def test_identity_when_no_decay_and_no_write():
    """alpha = 1, beta = 0: S unchanged and o_t = S0^T qn_t exactly."""
    c = _rand_case(T=9, Hk=2, Hv=4, dk=6, dv=4)
    g = np.zeros_like(c["g"])
    beta = np.zeros_like(c["beta"])
    o, S = oracle.recurrence(c["q"], c["k"], c["v"], g=g, beta=beta, S0=c["S0"])
    np.testing.assert_array_equal(S, c["S0"])
    qn = np.repeat(_unit(c["q"], 1e-6), 2, axis=2) / math.sqrt(6)
    expect = np.einsum("bthi,bhij->bthj", qn, c["S0"])
    np.testing.assert_allclose(o, expect, rtol=1e-13, atol=1e-14)


def test_reconstruction_beta_one_unit_key():
    """beta = 1 and a unit key: after the update S^T kn = v (delta-rule write).

    Reading with q = k and q_scale = 1 makes o_t = S_t^T kn_t, which must equal v_t
    for any decay and any prior state.
    """
    c = _rand_case(T=12, Hk=1, Hv=1, dk=8, dv=5, g_scale=1.0)
    beta = np.ones_like(c["beta"])
    o, _ = oracle.recurrence(c["k"], c["k"], c["v"], g=c["g"], beta=beta, S0=c["S0"], eps=0.0,
                             q_scale=1.0)
    np.testing.assert_allclose(o, c["v"], rtol=1e-12, atol=1e-12)


def test_decay_only_closed_form():
    """beta = 0: S_t = Diag(exp(sum_{s<=t} g_s)) S0 (closed form), o_t reads it."""
    c = _rand_case(T=10, Hk=1, Hv=3, dk=4, dv=6, g_scale=0.7)
    beta = np.zeros_like(c["beta"])
    o, S = oracle.recurrence(c["q"], c["k"], c["v"], g=c["g"], beta=beta, S0=c["S0"])
    cum = np.exp(np.cumsum(c["g"], axis=1))                # [B,T,H,dk]
    St = cum[..., None] * c["S0"][:, None]                 # [B,T,H,dk,dv]
    np.testing.assert_allclose(S, St[:, -1], rtol=1e-12, atol=1e-15)
    qn = np.repeat(_unit(c["q"], 1e-6), 3, axis=2) / 2.0
    np.testing.assert_allclose(o, np.einsum("bthi,bthij->bthj", qn, St), rtol=1e-11, atol=1e-14)


def test_scalar_case_dk_dv_one():
    """dk = dv = 1: kn = sign(k), S <- (1 - beta) alpha S + beta kn v, o = sign(q) S."""
    T = 25
    q = rng.standard_normal((1, T, 1, 1))
    k = rng.standard_normal((1, T, 1, 1))
    v = rng.standard_normal((1, T, 1, 1))
    g = -rng.random((1, T, 1, 1))
    beta = rng.random((1, T, 1))
    S0 = np.array([[[[0.7]]]])
    o, S = oracle.recurrence(q, k, v, g=g, beta=beta, S0=S0, eps=0.0)
    s = 0.7
    for t in range(T):
        kn = math.copysign(1.0, k[0, t, 0, 0])
        s = (1.0 - beta[0, t, 0]) * math.exp(g[0, t, 0, 0]) * s + beta[0, t, 0] * kn * v[0, t, 0, 0]
        assert abs(o[0, t, 0, 0] - math.copysign(1.0, q[0, t, 0, 0]) * s) < 1e-13
    assert abs(S[0, 0, 0, 0] - s) < 1e-13


def test_orthonormal_keys_store_values():
    """alpha = 1, beta = 1, S0 = 0, keys e_1..e_n: afterwards S^T e_i = v_i."""
    dk, dv, n = 6, 4, 5
    k = np.zeros((1, n, 1, dk))
    for i in range(n):
        k[0, i, 0, i] = 1.0
    q = rng.standard_normal((1, n, 1, dk))
    v = rng.standard_normal((1, n, 1, dv))
    o, S = oracle.recurrence(q, k, v, g=np.zeros((1, n, 1, dk)), beta=np.ones((1, n, 1)), eps=0.0)
    for i in range(n):
        np.testing.assert_allclose(S[0, 0, i], v[0, i, 0], atol=1e-14)
    np.testing.assert_allclose(S[0, 0, n:], 0.0, atol=0)


def test_linearity_in_values_and_state():
    """With q, k, g, beta fixed, (V, S0) -> (O, S_T) is linear."""
    c1 = _rand_case(seed=1)
    c2 = _rand_case(seed=2)
    a, b = 0.75, -1.5
    fx = lambda v, s: oracle.recurrence(c1["q"], c1["k"], v, g=c1["g"], beta=c1["beta"], S0=s)
    o1, S1 = fx(c1["v"], c1["S0"])
    o2, S2 = fx(c2["v"], c2["S0"])
    o3, S3 = fx(a * c1["v"] + b * c2["v"], a * c1["S0"] + b * c2["S0"])
    np.testing.assert_allclose(o3, a * o1 + b * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S3, a * S1 + b * S2, rtol=1e-11, atol=1e-12)


def test_brute_force_dense_transitions():
    """Dense restatement: S_t = (I - beta kn kn^T) Diag(alpha) S_{t-1} + beta kn v^T."""
    c = _rand_case(B=1, T=8, Hk=1, Hv=1, dk=4, dv=3, g_scale=0.9)
    o, S = oracle.recurrence(c["q"], c["k"], c["v"], g=c["g"], beta=c["beta"], S0=c["S0"])
    St = c["S0"][0, 0].copy()
    for t in range(8):
        kn = _unit(c["k"][0, t, 0], 1e-6)
        qn = _unit(c["q"][0, t, 0], 1e-6) / 2.0
        be = c["beta"][0, t, 0]
        M = (np.eye(4) - be * np.outer(kn, kn)) @ np.diag(np.exp(c["g"][0, t, 0]))
        St = M @ St + be * np.outer(kn, c["v"][0, t, 0])
        np.testing.assert_allclose(o[0, t, 0], St.T @ qn, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S[0, 0], St, rtol=1e-12, atol=1e-13)


def test_continuation_equals_one_pass():
    """recurrence(T1) then recurrence(T2) from the carried state == recurrence(T1+T2)."""
    c = _rand_case(T=15, Hk=2, Hv=2, dk=5, dv=5)
    o, S = oracle.recurrence(c["q"], c["k"], c["v"], g=c["g"], beta=c["beta"], S0=c["S0"])
    sl = lambda x, a, b: x[:, a:b]
    oa, Sa = oracle.recurrence(sl(c["q"], 0, 6), sl(c["k"], 0, 6), sl(c["v"], 0, 6),
                               g=sl(c["g"], 0, 6), beta=sl(c["beta"], 0, 6), S0=c["S0"])
    ob, Sb = oracle.recurrence(sl(c["q"], 6, 15), sl(c["k"], 6, 15), sl(c["v"], 6, 15),
                               g=sl(c["g"], 6, 15), beta=sl(c["beta"], 6, 15), S0=Sa)
    np.testing.assert_array_equal(np.concatenate([oa, ob], axis=1), o)
    np.testing.assert_array_equal(Sb, S)


@pytest.mark.parametrize("chunk", [1, 2, 3, 4, 5, 11, 16])
def test_chunkwise_equals_recurrence(chunk):
    """The chunked WY/UT form equals the recurrence for every chunk size and tail."""
    c = _rand_case(B=2, T=11, Hk=1, Hv=2, dk=5, dv=3, g_scale=0.8)
    o, S = oracle.recurrence(c["q"], c["k"], c["v"], g=c["g"], beta=c["beta"], S0=c["S0"])
    oc, Sc = oracle.chunkwise(c["q"], c["k"], c["v"], chunk=chunk, g=c["g"], beta=c["beta"], S0=c["S0"])
    scale = np.sqrt(np.mean(o ** 2))
    assert np.max(np.abs(oc - o)) / scale < 1e-12
    assert np.max(np.abs(Sc - S)) / np.sqrt(np.mean(S ** 2)) < 1e-12


def test_chunkwise_strong_decay_and_ragged_tail_positions():
    """Strong decay (log-decay near -5 per token) and every tail length 1..C-1."""
    for T in range(9, 17):
        c = _rand_case(B=1, T=T, Hk=1, Hv=1, dk=4, dv=4, g_scale=4.0, seed=T)
        o, S = oracle.recurrence(c["q"], c["k"], c["v"], g=c["g"], beta=c["beta"], S0=c["S0"])
        oc, Sc = oracle.chunkwise(c["q"], c["k"], c["v"], chunk=8, g=c["g"], beta=c["beta"], S0=c["S0"])
        assert np.max(np.abs(oc - o)) <= 1e-12 * max(1.0, np.abs(o).max())
        assert np.max(np.abs(Sc - S)) <= 1e-12 * max(1.0, np.abs(S).max())


def test_gdn_gate_special_points():
    """Scalar GatedDeltaNet gate at points where softplus and sigmoid are known.

    a = -dt_bias gives softplus(0) = ln 2, so g = -exp(A_log) ln 2; b = 0 gives
    beta = 1/2.  a + dt_bias = 30 is past the softplus threshold (softplus = 30
    to 1e-13).  The result must equal channel mode with that g broadcast over
    dk (the scalar gate is the broadcast special case of the channelwise one).
    """
    B, T, Hk, Hv, dk, dv = 1, 6, 1, 3, 4, 3
    r = np.random.default_rng(7)
    q = r.standard_normal((B, T, Hk, dk))
    k = r.standard_normal((B, T, Hk, dk))
    v = r.standard_normal((B, T, Hv, dv))
    S0 = r.standard_normal((B, Hv, dk, dv))
    A_log = np.array([0.0, 0.5, -0.25])
    dt_bias = np.array([0.3, -1.2, 2.0])
    a = np.tile(-dt_bias, (B, T, 1))
    a[0, 3, 1] = 30.0 - dt_bias[1]
    b = np.zeros((B, T, Hv))
    o, S = oracle.recurrence(q, k, v, a=a, b=b, A_log=A_log, dt_bias=dt_bias, S0=S0)
    sp = np.full((B, T, Hv), math.log(2.0))
    sp[0, 3, 1] = 30.0
    g = np.repeat((-np.exp(A_log) * sp)[..., None], dk, axis=-1)
    oc, Sc = oracle.recurrence(q, k, v, g=g, beta=np.full((B, T, Hv), 0.5), S0=S0)
    np.testing.assert_allclose(o, oc, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, Sc, rtol=1e-12, atol=1e-13)


def test_gdn_gate_generic_points():
    """The scalar gate at points that are not symmetric, so that a flipped sigmoid or a
    softplus of the negated argument fails ("Add fused GatedDeltaNet decode Triton kernel",
    description, gating: g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)).

    b = ln 3 gives beta = 3/4 exactly (1/(1+e^b) would give 1/4); a + dt_bias = ln(e - 1)
    gives softplus = 1 (softplus(-x) there is 1 - ln(e - 1) = 0.459), so g = -e^A_log; with
    A_log = 0.7 and -0.4 the factor e^A_log is not 1.  The result must equal the channel
    gate with those closed-form g and beta broadcast over dk.
    """
    B, T, Hk, Hv, dk, dv = 1, 5, 1, 2, 4, 3
    r = np.random.default_rng(17)
    q = r.standard_normal((B, T, Hk, dk))
    k = r.standard_normal((B, T, Hk, dk))
    v = r.standard_normal((B, T, Hv, dv))
    S0 = r.standard_normal((B, Hv, dk, dv))
    A_log = np.array([0.7, -0.4])
    dt_bias = np.array([0.25, -1.5])
    a = np.tile(math.log(math.e - 1.0) - dt_bias, (B, T, 1))
    b = np.full((B, T, Hv), math.log(3.0))
    o, S = oracle.recurrence(q, k, v, a=a, b=b, A_log=A_log, dt_bias=dt_bias, S0=S0)
    g = np.broadcast_to((-np.exp(A_log))[None, None, :, None], (B, T, Hv, dk)).copy()
    oc, Sc = oracle.recurrence(q, k, v, g=g, beta=np.full((B, T, Hv), 0.75), S0=S0)
    np.testing.assert_allclose(o, oc, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, Sc, rtol=1e-12, atol=1e-13)
    # the flipped readings give a different result on this case (the pin can fail)
    of, _ = oracle.recurrence(q, k, v, g=g, beta=np.full((B, T, Hv), 0.25), S0=S0)
    gs = np.broadcast_to((-np.exp(A_log) * (1.0 - math.log(math.e - 1.0)))[None, None, :, None],
                         (B, T, Hv, dk)).copy()
    os_, _ = oracle.recurrence(q, k, v, g=gs, beta=np.full((B, T, Hv), 0.75), S0=S0)
    assert np.max(np.abs(of - o)) > 1e-3 and np.max(np.abs(os_ - o)) > 1e-3


def test_gdn_chunkwise_equals_recurrence():
    r = np.random.default_rng(9)
    B, T, Hk, Hv, dk, dv = 1, 13, 2, 4, 4, 3
    q, k = r.standard_normal((B, T, Hk, dk)), r.standard_normal((B, T, Hk, dk))
    v = r.standard_normal((B, T, Hv, dv))
    a, b = r.standard_normal((B, T, Hv)), r.standard_normal((B, T, Hv))
    A_log, dt_bias = r.uniform(-1, 1, Hv), r.standard_normal(Hv)
    S0 = r.standard_normal((B, Hv, dk, dv))
    kw = dict(a=a, b=b, A_log=A_log, dt_bias=dt_bias, S0=S0)
    o, S = oracle.recurrence(q, k, v, **kw)
    oc, Sc = oracle.chunkwise(q, k, v, chunk=4, **kw)
    np.testing.assert_allclose(oc, o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Sc, S, rtol=1e-10, atol=1e-12)


def test_head_repeat_convention():
    """v-head h reads q/k head h // (Hv/Hk) (repeat-interleave).

    The pages say only "head repeat"; this pins the oracle to the convention
    the library documents, by comparing with single-head runs.
    """
    c = _rand_case(B=1, T=5, Hk=2, Hv=4, dk=3, dv=2)
    o, S = oracle.recurrence(c["q"], c["k"], c["v"], g=c["g"], beta=c["beta"], S0=c["S0"])
    for h in range(4):
        hk = h // 2
        o1, S1 = oracle.recurrence(c["q"][:, :, hk:hk + 1], c["k"][:, :, hk:hk + 1], c["v"][:, :, h:h + 1],
                                   g=c["g"][:, :, h:h + 1], beta=c["beta"][:, :, h:h + 1],
                                   S0=c["S0"][:, h:h + 1])
        np.testing.assert_array_equal(o[:, :, h:h + 1], o1)
        np.testing.assert_array_equal(S[:, h:h + 1], S1)


def test_thread_count_and_empty_sequence():
    c = _rand_case(B=3, T=6, Hk=1, Hv=3, dk=4, dv=4)
    o1, S1 = oracle.recurrence(c["q"], c["k"], c["v"], g=c["g"], beta=c["beta"], S0=c["S0"], threads=1)
    o4, S4 = oracle.recurrence(c["q"], c["k"], c["v"], g=c["g"], beta=c["beta"], S0=c["S0"], threads=4)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(S1, S4)
    z = lambda x: x[:, :0]
    o0, S0 = oracle.recurrence(z(c["q"]), z(c["k"]), z(c["v"]), g=z(c["g"]), beta=z(c["beta"]), S0=c["S0"])
    assert o0.shape == (3, 0, 3, 4)
    np.testing.assert_array_equal(S0, c["S0"])


def test_bf16_inputs_are_upcast_exactly():
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, 4, 1, 8, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 4, 1, 8, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 4, 1, 8, generator=g).to(torch.bfloat16)
    gg = -torch.rand(1, 4, 1, 8, generator=g)
    be = torch.rand(1, 4, 1, generator=g)
    o1, S1 = oracle.recurrence(q, k, v, g=gg, beta=be)
    o2, S2 = oracle.recurrence(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                               g=gg.double().numpy(), beta=be.double().numpy())
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)
