"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics, not by the oracle itself.

Every check below would fail for a plausible slip in the oracle (a dropped
term, decay after the write instead of before the probe, a readout taken
before the write, a transposed state, a wrong tap order, a wrong epsilon
placement, a leak across sequence boundaries).

Sources, by page title and section:
  * "Kimi K3 / Architecture", panels "Kimi Delta Attention . one head at token t"
    and "KDA short convolution . one channel c at token t";
  * "Animated Kimi K3 architecture diagram", section "LOCAL MEMORY: A FIXED
    MATRIX THAT PREDICTS, FORGETS, AND CORRECTS" (four moves, notebook trace).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from kimi_delta_attention_16_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unit_rows(rng, L, d):
    x = rng.standard_normal((L, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _core_inputs(rng, L, Dk, Dv, g_lo=-5.0, g_hi=0.0, s0=True):
    q = _unit_rows(rng, L, Dk)
    k = _unit_rows(rng, L, Dk)
    v = rng.standard_normal((L, Dv))
    g = rng.uniform(g_lo, g_hi, (L, Dk))
    beta = rng.uniform(0.0, 1.0, L)
    S0 = 0.3 * rng.standard_normal((Dk, Dv)) if s0 else None
    return q, k, v, g, beta, S0


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------- recurrence

def test_hand_worked_scalar_example():
    """Dk = Dv = 1, worked by hand from the four moves and the readout after the write.

    t=1: S0=0, alpha=1, k=1, v=2, beta=0.5, q=1:
         S_bar=0, e=2-0=2, S=0+0.5*1*2=1, o=1*1=1
    t=2: alpha=0.5, k=1, v=3, beta=1, q=2:
         S_bar=0.5, e=3-0.5=2.5, S=0.5+1*1*2.5=3, o=3*2=6
    """
    q = np.array([[1.0], [2.0]])
    k = np.array([[1.0], [1.0]])
    v = np.array([[2.0], [3.0]])
    g = np.array([[0.0], [math.log(0.5)]])
    beta = np.array([0.5, 1.0])
    o, S = oracle.recurrence(q, k, v, g, beta)
    np.testing.assert_allclose(o[:, 0], [1.0, 6.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(S, [[3.0]], rtol=0, atol=1e-15)


def test_hand_worked_two_channel_example():
    """Dk = 2, Dv = 1: the decay is per key channel, the probe reads the decayed state.

    S0 = [1, 2]^T, alpha = (0.5, 0.25), k = (1, 0), v = 4, beta = 1, q = (0, 1):
      S_bar = (0.5, 0.5); e = 4 - (0.5*1 + 0.5*0) = 3.5;
      S = S_bar + k e = (4, 0.5); o = q . S = 0.5
    """
    S0 = np.array([[1.0], [2.0]])
    o, S = oracle.recurrence(np.array([[0.0, 1.0]]), np.array([[1.0, 0.0]]), np.array([[4.0]]),
                             np.array([[math.log(0.5), math.log(0.25)]]), np.array([1.0]), S0)
    np.testing.assert_allclose(S[:, 0], [4.0, 0.5], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[0, 0], 0.5, rtol=0, atol=1e-15)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("L", [1, 5, 63, 64, 65, 130])
@pytest.mark.parametrize("g_lo", [-5.0, -0.05])
def test_sequential_equals_chunkwise(C, L, g_lo):
    """Notebook trace: 'sequential ~ chunkwise'.  Two independent fp64 forms agree to 1e-12.

    g_lo = -0.05 keeps memory over many chunks so the carry across chunks matters.
    """
    rng = np.random.default_rng(1000 * C + L)
    q, k, v, g, beta, S0 = _core_inputs(rng, L, 16, 8, g_lo=g_lo)
    o1, S1 = oracle.recurrence(q, k, v, g, beta, S0, scale=0.7)
    o2, S2 = oracle.chunkwise(q, k, v, g, beta, S0, chunk=C, scale=0.7)
    assert _rel(o2, o1) < 1e-12
    assert _rel(S2, S1) < 1e-12


def test_chunk_states_are_the_sequential_states():
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = _core_inputs(rng, 40, 8, 8, g_lo=-0.2)
    _, _, st = oracle.chunkwise(q, k, v, g, beta, S0, chunk=16, return_chunk_states=True)
    for n, t in enumerate([0, 16, 32]):
        S = S0.copy() if t == 0 else oracle.recurrence(q[:t], k[:t], v[:t], g[:t], beta[:t], S0)[1]
        assert _rel(st[n], S) < 1e-12


def test_no_decay_no_write_keeps_state():
    """alpha = 1, beta = 0: S_t = S0 and o_t = scale * S0^T q_t for every t."""
    rng = np.random.default_rng(1)
    q, k, v, _, _, S0 = _core_inputs(rng, 20, 12, 7)
    o, S = oracle.recurrence(q, k, v, np.zeros((20, 12)), np.zeros(20), S0, scale=1.5)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, 1.5 * q @ S0, rtol=1e-14, atol=1e-14)


def test_pure_decay():
    """beta = 0: S_T = Diag(exp(sum_t g_t)) S0 (decay acts on key rows)."""
    rng = np.random.default_rng(2)
    q, k, v, g, _, S0 = _core_inputs(rng, 9, 6, 5)
    _, S = oracle.recurrence(q, k, v, g, np.zeros(9), S0)
    np.testing.assert_allclose(S, np.exp(g.sum(0))[:, None] * S0, rtol=1e-13, atol=0)


@pytest.mark.parametrize("g_lo", [-5.0, -0.5])
def test_full_strength_write_recalls_value(g_lo):
    """beta = 1 and |k_t| = 1: the write makes S_t^T k_t = v_t exactly, for any alpha.

    This pins the order decay -> probe -> write (a decay applied after the
    write would break the identity whenever alpha != 1).
    """
    rng = np.random.default_rng(3)
    q, k, v, g, _, S0 = _core_inputs(rng, 12, 10, 6, g_lo=g_lo)
    S = S0.copy()
    for t in range(12):
        _, S = oracle.recurrence(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], np.ones(1), S)
        np.testing.assert_allclose(S.T @ k[t], v[t], rtol=0, atol=1e-13)


def test_orthonormal_keys_recall_every_value():
    """alpha = 1, beta = 1, orthonormal keys (T <= dk): S_T^T k_i = v_i for all i."""
    rng = np.random.default_rng(4)
    dk, T = 16, 11
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:T]
    v = rng.standard_normal((T, 5))
    S0 = rng.standard_normal((dk, 5))
    _, S = oracle.recurrence(rng.standard_normal((T, dk)), k, v, np.zeros((T, dk)), np.ones(T), S0)
    np.testing.assert_allclose(k @ S, v, rtol=0, atol=1e-12)


def test_linear_in_values_and_initial_state():
    """For fixed q, k, g, beta the map (V, S0) -> (o, S_T) is linear."""
    rng = np.random.default_rng(5)
    q, k, v1, g, beta, S1 = _core_inputs(rng, 30, 8, 6, g_lo=-1.0)
    v2 = rng.standard_normal(v1.shape)
    S2 = rng.standard_normal(S1.shape)
    a, b = 0.75, -1.25
    o1, T1 = oracle.recurrence(q, k, v1, g, beta, S1)
    o2, T2 = oracle.recurrence(q, k, v2, g, beta, S2)
    o3, T3 = oracle.recurrence(q, k, a * v1 + b * v2, g, beta, a * S1 + b * S2)
    np.testing.assert_allclose(o3, a * o1 + b * o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(T3, a * T1 + b * T2, rtol=1e-12, atol=1e-12)


def test_value_columns_are_independent():
    """Decay acts on key rows and k k^T mixes only keys: permuting value columns
    (of V and S0) permutes the columns of o and S_T, nothing else."""
    rng = np.random.default_rng(6)
    q, k, v, g, beta, S0 = _core_inputs(rng, 25, 8, 7, g_lo=-1.0)
    perm = rng.permutation(7)
    o1, T1 = oracle.recurrence(q, k, v, g, beta, S0)
    o2, T2 = oracle.recurrence(q, k, v[:, perm], g, beta, S0[:, perm])
    np.testing.assert_allclose(o2, o1[:, perm], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(T2, T1[:, perm], rtol=1e-13, atol=1e-13)


def test_notebook_trace_golden():
    """Notebook trace: miniature output [2,16,64]; sequential ~ chunkwise; state shape fixed."""
    gold = json.load(open(os.path.join(GOLDEN, "notebook_trace.json")))
    B, T, D = gold["output_shape"]
    inp = synth.make_prefill("tiny_fp32", seed=11, lengths=[T] * B, H=1, D=D)
    res = oracle.forward(synth.to_f32_numpy(inp.q), synth.to_f32_numpy(inp.k),
                         synth.to_f32_numpy(inp.v), synth.to_f32_numpy(inp.conv_w),
                         inp.cu_seqlens, synth.to_f32_numpy(inp.g), synth.to_f32_numpy(inp.beta),
                         gate=synth.to_f32_numpy(inp.gate), want_o_pre=True)
    assert res["out"].reshape(B, T, D).shape == tuple(gold["output_shape"])
    assert res["final_state"].shape == (B, 1, D, D)
    # sequential (whole layer) ~ chunkwise on the same convolved inputs
    x = np.concatenate([synth.to_f32_numpy(t).reshape(B * T, D) for t in (inp.q, inp.k, inp.v)], 1)
    y, _ = oracle.conv_silu(x, synth.to_f32_numpy(inp.conv_w).reshape(3 * D, 4), inp.cu_seqlens)
    qc, kc, vc = oracle.l2norm(y[:, :D]), oracle.l2norm(y[:, D:2 * D]), y[:, 2 * D:]
    g = synth.to_f32_numpy(inp.g).reshape(B * T, D)
    b = synth.to_f32_numpy(inp.beta).reshape(B * T)
    for n in range(B):
        s = slice(n * T, (n + 1) * T)
        o_c, S_c = oracle.chunkwise(qc[s], kc[s], vc[s], g[s], b[s], chunk=4)
        assert _rel(o_c, res["o_pre"][s, 0]) < 1e-12
        assert _rel(S_c, res["final_state"][n, 0]) < 1e-12
    # the state shape does not grow with T
    for T2 in (1, 3, 40):
        r = oracle.recurrence(qc[:T2], kc[:T2], vc[:T2], g[:T2], b[:T2])
        assert r[1].shape == (D, D)


def test_page_constants_golden():
    gold = json.load(open(os.path.join(GOLDEN, "kda_shapes.json")))
    H, D = gold["heads"], gold["head_dim"]
    assert 3 * H * D == gold["rolling_state_channels"]
    assert [H * D, 1, gold["conv_width"]] == gold["filter_bank_shape"]
    assert gold["conv_width"] - 1 == gold["rolling_state_per_channel"]
    assert synth.WORKLOADS["layer_8k"]["H"] == H and synth.WORKLOADS["layer_8k"]["D"] == D


# --------------------------------------------------------------------------- conv / norms

def test_conv_matches_numpy_convolve():
    """Tap w[3] multiplies x[t], w[0] multiplies x[t-3]; zero left padding; length kept."""
    rng = np.random.default_rng(8)
    lengths = [1, 2, 3, 4, 9]
    cu = synth.cu_from_lengths(lengths)
    x = rng.standard_normal((cu[-1], 5)).astype(np.float32)
    w = rng.standard_normal((5, 4)).astype(np.float32)
    y, so = oracle.conv_silu(x, w, cu, apply_silu=False)
    for n, L in enumerate(lengths):
        for c in range(5):
            xs = x[cu[n]:cu[n + 1], c].astype(np.float64)
            ref = np.convolve(xs, w[c, ::-1].astype(np.float64))[:L]
            np.testing.assert_allclose(y[cu[n]:cu[n + 1], c], ref, rtol=1e-14, atol=1e-14)
            last = np.concatenate([np.zeros(3), xs])[-3:]
            np.testing.assert_array_equal(so[n, c], last)


def test_conv_state_in_equals_concatenated_stream():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((10, 3)).astype(np.float32)
    w = rng.standard_normal((3, 4)).astype(np.float32)
    whole, s_whole = oracle.conv_silu(x, w, [0, 10])
    a, s_a = oracle.conv_silu(x[:4], w, [0, 4])
    b, s_b = oracle.conv_silu(x[4:], w, [0, 6], state_in=s_a.astype(np.float32))
    np.testing.assert_array_equal(np.concatenate([a, b]), whole)
    np.testing.assert_array_equal(s_b, s_whole)


def test_conv_is_causal_and_channel_isolated():
    """'Only time is mixed': a bump in channel c at token t changes only channel c, tokens t..t+3."""
    rng = np.random.default_rng(10)
    x = rng.standard_normal((12, 6)).astype(np.float32)
    w = rng.standard_normal((6, 4)).astype(np.float32)
    y0, _ = oracle.conv_silu(x, w, [0, 12])
    x2 = x.copy()
    x2[5, 2] += 1.0
    y1, _ = oracle.conv_silu(x2, w, [0, 12])
    changed = np.argwhere(y1 != y0)
    assert set(map(tuple, changed)) == {(t, 2) for t in range(5, 9)}


def test_conv_sequences_do_not_see_each_other():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((8, 2)).astype(np.float32)
    w = rng.standard_normal((2, 4)).astype(np.float32)
    packed, _ = oracle.conv_silu(x, w, [0, 3, 8])
    solo, _ = oracle.conv_silu(x[3:], w, [0, 5])
    np.testing.assert_array_equal(packed[3:], solo)


def test_silu_special_values():
    """SiLU(x) = x sigmoid(x): sigmoid(0)=1/2, sigmoid(ln 3)=3/4, sigmoid(-ln 3)=1/4."""
    vals = np.array([0.0, math.log(3.0), -math.log(3.0), 30.0], np.float32)
    x = np.zeros((7, 1), np.float32)
    x[3:, 0] = vals
    y, _ = oracle.conv_silu(x, np.array([[0, 0, 0, 1]], np.float32), [0, 7])
    xv = vals.astype(np.float64)
    expect = [0.0, 0.75 * xv[1], 0.25 * xv[2], xv[3]]
    np.testing.assert_allclose(y[3:, 0], expect, rtol=2e-7, atol=1e-12)
    np.testing.assert_array_equal(y[:3, 0], 0.0)


def test_l2norm_closed_form():
    np.testing.assert_allclose(oracle.l2norm([[3.0, 4.0]], eps=0.0), [[0.6, 0.8]], rtol=1e-15, atol=0)
    np.testing.assert_allclose(oracle.l2norm([[3.0, 4.0]], eps=11.0), [[0.5, 2.0 / 3.0]], rtol=1e-15)


def test_rmsnorm_gate_closed_form():
    o = np.array([[2.0, -2.0, 2.0, -2.0]])
    np.testing.assert_allclose(oracle.rmsnorm_gate(o, eps=0.0), [[1, -1, 1, -1]], atol=1e-15)
    # mean(o^2) + eps = 4 + 5 = 9 -> divide by 3; weight; sigmoid(0) = 1/2
    y = oracle.rmsnorm_gate(o, gate=np.zeros((1, 4)), w=np.array([1.0, 2.0, 3.0, 4.0]), eps=5.0)
    np.testing.assert_allclose(y, [[1 / 3, -2 / 3, 1.0, -4 / 3]], rtol=1e-15)


# --------------------------------------------------------------------------- whole layer

def _np_inputs(inp):
    f = synth.to_f32_numpy
    return dict(q=f(inp.q), k=f(inp.k), v=f(inp.v), conv_w=f(inp.conv_w), cu_seqlens=inp.cu_seqlens,
                g=f(inp.g), beta=f(inp.beta), gate=f(inp.gate), rms_w=f(inp.rms_w),
                initial_state=f(inp.initial_state), conv_state_in=f(inp.conv_state_in))


def test_forward_composes_its_pieces():
    """The threaded whole-layer oracle equals conv+SiLU -> L2 -> recurrence -> RMSNorm+gate."""
    inp = synth.make_prefill("tiny_fp32", seed=3, lengths=[7, 20], H=2, D=16, rms_w="random",
                             s0_std=0.5, conv_state=True)
    a = _np_inputs(inp)
    res = oracle.forward(**a, eps_l2=1e-3, eps_rms=1e-2, scale=0.9, want_o_pre=True)
    H, D, T = 2, 16, inp.T
    x = np.concatenate([a["q"].reshape(T, H * D), a["k"].reshape(T, H * D), a["v"].reshape(T, H * D)], 1)
    y, so = oracle.conv_silu(x, a["conv_w"].reshape(3 * H * D, 4), inp.cu_seqlens,
                             state_in=a["conv_state_in"])
    np.testing.assert_array_equal(res["conv_state_out"], so)
    y = y.reshape(T, 3, H, D)
    for n in range(2):
        s = slice(inp.cu_seqlens[n], inp.cu_seqlens[n + 1])
        for h in range(H):
            qh = oracle.l2norm(y[s, 0, h], 1e-3)
            kh = oracle.l2norm(y[s, 1, h], 1e-3)
            o, S = oracle.recurrence(qh, kh, y[s, 2, h], a["g"][s, h], a["beta"][s, h],
                                     a["initial_state"][n, h], scale=0.9)
            assert _rel(res["o_pre"][s, h], o) < 1e-13
            assert _rel(res["final_state"][n, h], S) < 1e-13
            yy = oracle.rmsnorm_gate(o, a["gate"][s, h], a["rms_w"], 1e-2)
            assert _rel(res["out"][s, h], yy) < 1e-13


def test_packed_equals_solo():
    inp = synth.make_prefill("tiny_fp32", seed=4, lengths=[5, 1, 33], H=2, D=16, s0_std=0.1,
                             conv_state=True)
    a = _np_inputs(inp)
    res = oracle.forward(**a)
    cu = inp.cu_seqlens
    for n in range(3):
        s = slice(cu[n], cu[n + 1])
        solo = oracle.forward(q=a["q"][s], k=a["k"][s], v=a["v"][s], conv_w=a["conv_w"],
                              cu_seqlens=[0, cu[n + 1] - cu[n]], g=a["g"][s], beta=a["beta"][s],
                              gate=a["gate"][s], rms_w=a["rms_w"],
                              initial_state=a["initial_state"][n:n + 1],
                              conv_state_in=a["conv_state_in"][n:n + 1])
        np.testing.assert_array_equal(solo["out"], res["out"][s])
        np.testing.assert_array_equal(solo["final_state"][0], res["final_state"][n])
        np.testing.assert_array_equal(solo["conv_state_out"][0], res["conv_state_out"][n])


def test_handoff_prefill_prefill_and_decode():
    """prefill(T1+T2) == prefill(T1) -> prefill(T2) == prefill(T1) -> T2 single-token steps."""
    inp = synth.make_prefill("tiny_fp32", seed=5, lengths=[29], H=2, D=16, s0_std=0.2)
    a = _np_inputs(inp)
    whole = oracle.forward(**a)
    T1 = 17

    def part(s, state, cstate):
        return oracle.forward(q=a["q"][s], k=a["k"][s], v=a["v"][s], conv_w=a["conv_w"],
                              cu_seqlens=[0, s.stop - s.start], g=a["g"][s], beta=a["beta"][s],
                              gate=a["gate"][s], rms_w=a["rms_w"], initial_state=state,
                              conv_state_in=cstate)

    p1 = part(slice(0, T1), a["initial_state"], None)
    p2 = part(slice(T1, 29), p1["final_state"], p1["conv_state_out"].astype(np.float32))
    np.testing.assert_array_equal(np.concatenate([p1["out"], p2["out"]]), whole["out"])
    np.testing.assert_array_equal(p2["final_state"], whole["final_state"])
    st, cs = p1["final_state"], p1["conv_state_out"]
    for t in range(T1, 29):
        step = part(slice(t, t + 1), st, cs.astype(np.float32))
        st, cs = step["final_state"], step["conv_state_out"]
        np.testing.assert_array_equal(step["out"][0], whole["out"][t])
    np.testing.assert_array_equal(st, whole["final_state"])
    np.testing.assert_array_equal(cs, whole["conv_state_out"])


# --------------------------------------------------------------------------- projections around the layer

def test_linear_is_the_brute_force_sum():
    """x W^T by three nested loops on a tiny case, and the identity weight returns x."""
    rng = np.random.default_rng(11)
    x, w = rng.standard_normal((3, 5)), rng.standard_normal((4, 5))
    ref = np.zeros((3, 4))
    for m in range(3):
        for n in range(4):
            for kk in range(5):
                ref[m, n] += x[m, kk] * w[n, kk]
    np.testing.assert_allclose(oracle.linear(x, w), ref, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(oracle.linear(x, np.eye(5)), x)


def test_bounded_decay_and_strength_activations():
    """g = -5 sigmoid(z): -2.5 at 0, the ends of (-5, 0) at the tails, g(z) + g(-z) = -5,
    increasing towards 0 as z falls; beta = sigmoid(z): 1/2 at 0, beta(z) + beta(-z) = 1,
    the logistic 1 / (1 + e^-z) at hand-chosen points."""
    assert oracle.decay_from_logits(0.0) == -2.5
    z = np.linspace(-30, 30, 121)  # beyond |z| ~ 37 sigmoid(z) rounds to 0 or 1 in fp64
    g = oracle.decay_from_logits(z)
    assert np.all(g > -5) and np.all(g < 0)
    np.testing.assert_allclose(g + oracle.decay_from_logits(-z), -5.0, rtol=0, atol=1e-13)
    assert np.all(np.diff(g) < 0)
    assert oracle.decay_from_logits(-800.0) == 0.0 and oracle.decay_from_logits(800.0) == -5.0
    b = oracle.strength_from_logits(z)
    np.testing.assert_allclose(b + oracle.strength_from_logits(-z), 1.0, rtol=0, atol=1e-15)
    for zz in (-3.0, -0.5, 0.0, 1.25, 7.0):
        assert math.isclose(float(oracle.strength_from_logits(zz)), 1.0 / (1.0 + math.exp(-zz)), rel_tol=1e-15)
    assert oracle.strength_from_logits(0.0) == 0.5


def test_round_bf16_ties_to_even_and_matches_torch():
    """Hand-worked cases (1 + 2^-8 is a tie -> 1; 1 + 3 * 2^-8 -> 1 + 2^-6; 1 + 2^-7 is exact),
    and agreement with torch's bf16 cast on random values of every magnitude."""
    import torch
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    assert oracle.round_bf16(1 + 2 ** -7) == 1 + 2 ** -7
    assert oracle.round_bf16(-(1 + 2 ** -8 + 2 ** -20)) == -(1 + 2 ** -7)
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(4096) * np.exp(rng.uniform(-60, 60, 4096))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), ref)


def test_projected_layer_composes_its_stages():
    """The layer with its projections is the plain layer fed the activated projections: g and
    beta from the bounded activations, the gate rounded to bf16, and out = bf16(y) W_o^T."""
    inp = synth.make_prefill("tiny_fp32", seed=13, lengths=[19, 6], H=2, D=16)
    a = _np_inputs(inp)
    T, H, D, dm = 25, 2, 16, 24
    rng = np.random.default_rng(14)
    x = rng.standard_normal((T, dm)).astype(np.float32)
    wa, wb, wg = (rng.standard_normal((n, dm)) / math.sqrt(dm) for n in (H * D, H, H * D))
    wo = rng.standard_normal((40, H * D)) / math.sqrt(H * D)
    res = oracle.projected_layer(x, wa, wb, wg, wo, a["q"], a["k"], a["v"], a["conv_w"],
                                 a["cu_seqlens"], rms_w=a["rms_w"])
    g = (-5.0 / (1.0 + np.exp(-(x.astype(np.float64) @ wa.T)))).reshape(T, H, D)
    np.testing.assert_allclose(res["g"], g, rtol=1e-13, atol=1e-15)
    assert np.all(res["g"] > -5) and np.all(res["g"] < 0)
    ref = oracle.forward(q=a["q"], k=a["k"], v=a["v"], conv_w=a["conv_w"], cu_seqlens=a["cu_seqlens"],
                         g=res["g"].astype(np.float32), beta=res["beta"].astype(np.float32),
                         gate=res["gate"].astype(np.float32), rms_w=a["rms_w"])
    np.testing.assert_array_equal(res["y"], ref["out"])
    np.testing.assert_array_equal(res["gate"], oracle.round_bf16(res["gate"]))
    np.testing.assert_allclose(res["out"], oracle.round_bf16(ref["out"]).reshape(T, H * D) @ wo.T,
                               rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------- backward pass

def _fd_case(seed=17, g_range=(-1.0, 0.0)):
    """A tiny two-sequence case with every optional input present, all values exact in fp32."""
    inp = synth.make_prefill("tiny_fp32", seed=seed, lengths=[5, 3], H=2, D=4, s0_std=0.5,
                             conv_state=True, rms_w="random", g_range=g_range)
    a = _np_inputs(inp)
    rng = np.random.default_rng(seed + 1)
    dy = rng.standard_normal(a["q"].shape)
    dsf = rng.standard_normal(a["initial_state"].shape)
    return a, dy, dsf


def _loss(a, dy, dsf):
    res = oracle.forward(**a, n_threads=1)
    return float(np.sum(dy * res["out"]) + np.sum(dsf * res["final_state"]))


@pytest.mark.parametrize("g_range", [(-1.0, 0.0), (-5.0, -4.0)])
def test_backward_matches_central_differences_of_the_forward(g_range):
    """Every element of every input: central differences of the forward at steps h = 2^-12 and
    h / 4 (the perturbed values stay exact in fp32, so the forward itself is unchanged),
    combined by Richardson extrapolation (16 D(h/4) - D(h)) / 15 to remove the h^2 term,
    against the backward's gradient; loss = sum dy . out + sum dS . final_state.  (With strong
    decay the RMSNorm of small outputs makes the third derivatives large: plain differences at
    h = 2^-12 are off by ~1e-4 there, the extrapolated ones by ~1e-8.)"""
    a, dy, dsf = _fd_case(g_range=g_range)
    grads = oracle.backward(**a, dy=dy, d_final_state=dsf, n_threads=1)
    names = {"q": "dq", "k": "dk", "v": "dv", "conv_w": "dconv_w", "g": "dg", "beta": "dbeta",
             "gate": "dgate", "rms_w": "drms_w", "initial_state": "dinitial_state",
             "conv_state_in": "dconv_state_in"}
    def central(x, idx, h):
        keep = x[idx]
        x[idx] = keep + h
        lp = _loss(a, dy, dsf)
        x[idx] = keep - h
        lm = _loss(a, dy, dsf)
        x[idx] = keep
        return (lp - lm) / (2 * h)

    h = 2.0 ** -12
    worst = 0.0
    for name, gname in names.items():
        x = a[name]
        gr = grads[gname].reshape(x.shape)
        for idx in np.ndindex(x.shape):
            fd = (16.0 * central(x, idx, h / 4) - central(x, idx, h)) / 15.0
            err = abs(fd - gr[idx])
            worst = max(worst, err / (1.0 + abs(fd)))
            assert err <= 1e-6 * (1.0 + abs(fd)), f"{name}{idx}: backward {gr[idx]:.9e}, differences {fd:.9e}"
    assert worst > 0.0


def test_backward_is_linear_in_the_upstream_gradients():
    a, dy, dsf = _fd_case(seed=19)
    g1 = oracle.backward(**a, dy=dy, d_final_state=None)
    g2 = oracle.backward(**a, dy=np.zeros_like(dy), d_final_state=dsf)
    g12 = oracle.backward(**a, dy=dy, d_final_state=dsf)
    for key in g12:
        np.testing.assert_allclose(g12[key], g1[key] + g2[key], rtol=1e-12, atol=1e-12)


def test_backward_closed_form_without_decay_or_write():
    """alpha = 1, beta = 0: the state never changes, o_t = scale S0^T q_t, so the initial
    state's gradient is sum_t scale q_t do_t^T (do_t the readout's gradient, here with no
    RMSNorm weight or gate: do = r dy - r^3 o (dy . o) / D), and the log-decay's gradient is
    dg_t[c] = sum_j dS_t[c][j] S0[c][j] with dS_t = sum_{s >= t} scale q_s do_s^T."""
    inp = synth.make_prefill("tiny_fp32", seed=23, lengths=[6], H=1, D=4, s0_std=0.5, gate=False,
                             rms_w=None, g_range=(0.0, 0.0))
    inp.beta.zero_()
    a = _np_inputs(inp)
    dy = np.random.default_rng(24).standard_normal(a["q"].shape)
    grads = oracle.backward(**a, dy=dy)
    res = oracle.forward(**a, want_o_pre=True)
    # q after conv + SiLU + L2, from the oracle's pinned pieces
    x = a["q"].reshape(6, 4)
    cq, _ = oracle.conv_silu(x, a["conv_w"][0].reshape(4, 4), a["cu_seqlens"])
    qh = oracle.l2norm(cq)
    o = res["o_pre"][:, 0]
    r = 1.0 / np.sqrt(np.mean(o * o, axis=1) + 1e-6)
    do = r[:, None] * dy[:, 0] - (r ** 3)[:, None] * o * np.sum(dy[:, 0] * o, axis=1)[:, None] / 4
    np.testing.assert_allclose(grads["dinitial_state"][0, 0], qh.T @ do, rtol=1e-10, atol=1e-12)
    S0 = a["initial_state"][0, 0]
    for t in range(6):
        dSt = qh[t:].T @ do[t:]
        np.testing.assert_allclose(grads["dg"][t, 0], np.sum(dSt * S0, axis=1), rtol=1e-10, atol=1e-12)
