"""GPU parity at the method's edge cases, on every path of the library.

The log-decay is bounded below by -5 ("Kimi K3 / Architecture", KDA panel:
channel-wise retention with a bounded log-decay), and the tensor-core path
splits each decay factor e^{G_r - G_i} through anchors that are safe exactly up
to that bound: within a 32-token half a factor reaches e^{80} when g = -5 on
every token.  These tests drive the decay to its two ends (g = -5 everywhere,
g = 0 everywhere, and a per-channel mix of the two) and the write strength to
its two ends (beta = 0, beta = 1), across several full 64-token chunks plus a
ragged tail, through:

  * the tensor-core path with one segment per sequence and with 3 segments,
  * the fp32 SIMT path (bf16 and fp32 inputs),
  * the recurrent path for batches of short sequences,
  * the single-token decode step,

and compare element by element with the fp64 oracle at the layer's
tolerances (fp32 outputs under the plain bound, bf16 outputs with their own
rounding allowance).  Two closed forms that need no recurrence at all are
asserted on the GPU as well ("Animated Kimi K3 architecture diagram", LOCAL
MEMORY section: decay, probe, correct, write):

  * alpha = 1 (g = 0) and beta = 0: nothing is forgotten and nothing written,
    so the final state equals the initial state and o_t = S_0^T q_t;
  * beta = 1 with a unit-norm key: the write makes S_t^T k_t = v_t exactly,
    for any decay; with q_t = k_t (equal raw q and k and equal filters) the
    readout o_t is v_t itself, so y_t = v_t / rms(v_t).
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_16_gb300 as kda
from kimi_delta_attention_16_gb300 import _lib, synth
from kda_testlib import (TOL_FP32, TOL_OUT_BF16, TOL_STATE_BF16, check_out, head_slice_inputs,
                         oracle_prefill, per_head_rel, to_np)
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"

# path name -> (flags, segments, lengths, io, expected plan)
PATHS = {
    "tc_p1": (_lib.KDA_FLAG_NO_RECURRENT, 1, [64 * 3 + 17, 130], "bf16", ("tc", 1)),
    "tc_p3": (_lib.KDA_FLAG_NO_RECURRENT, 3, [64 * 12 + 29], "bf16", ("tc", 3)),
    "simt_bf16": (_lib.KDA_FLAG_FORCE_SIMT, 0, [200, 70], "bf16", ("simt", 1)),
    "simt_fp32": (_lib.KDA_FLAG_FORCE_SIMT, 0, [200, 70], "fp32", ("simt", 1)),
    "recurrent": (0, 0, [8, 5, 8, 1], "bf16", ("recurrent", 1)),
}
G_MODES = ["min", "zero", "mix"]
BETA_MODES = ["rand", "zero", "one"]


def _set_g(g: torch.Tensor, mode: str, seed: int) -> None:
    """g [..., H, D] in place: -5 everywhere, 0 everywhere, or a fixed per-(head, channel)
    mix of the two (about half the channels forget at the bound, the others never)."""
    if mode == "min":
        g.fill_(-5.0)
    elif mode == "zero":
        g.zero_()
    else:
        gen = torch.Generator(device="cpu")
        gen.manual_seed(seed)
        mask = torch.rand(g.shape[-2:], generator=gen) < 0.5
        g.copy_(torch.where(mask, -5.0, 0.0).to(g.device).expand_as(g))


def _set_beta(beta: torch.Tensor, mode: str) -> None:
    if mode == "zero":
        beta.zero_()
    elif mode == "one":
        beta.fill_(1.0)


def _inputs(path, g_mode, beta_mode, seed):
    flags, segments, lengths, io, plan = PATHS[path]
    inp = synth.make_prefill("layer_8k", seed=seed, device=DEV, lengths=lengths, H=2, io=io,
                             s0_std=0.02, conv_state=True, rms_w="random")
    _set_g(inp.g, g_mode, seed)
    _set_beta(inp.beta, beta_mode)
    assert kda.kda_prefill_plan(inp.T, inp.H, inp.D, N=inp.N, io=inp.q.dtype, flags=flags,
                                segments=segments, cu_seqlens=inp.cu_seqlens) == plan
    return inp, flags, segments


def _run(inp, flags, segments, out_dtype, **kw):
    cso = torch.empty((inp.N, 3 * inp.H * inp.D, 3), dtype=inp.q.dtype, device=DEV)
    out, fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens,
                               chunk=inp.chunk, gate=inp.gate, rms_w=inp.rms_w,
                               initial_state=inp.initial_state, conv_state_in=inp.conv_state_in,
                               conv_state_out=cso, out_dtype=out_dtype, flags=flags,
                               segments=segments, **kw)
    torch.cuda.synchronize()
    return out, fin, cso


@pytest.mark.parametrize("beta_mode", BETA_MODES)
@pytest.mark.parametrize("g_mode", G_MODES)
@pytest.mark.parametrize("path", list(PATHS))
def test_prefill_decay_and_strength_extremes(path, g_mode, beta_mode):
    """Every path against the oracle with the decay and the write strength at their ends."""
    seed = 300 + 10 * G_MODES.index(g_mode) + BETA_MODES.index(beta_mode)
    inp, flags, segments = _inputs(path, g_mode, beta_mode, seed)
    ref = oracle_prefill(inp)
    fp32_io = inp.io == "fp32"
    for out_dtype in (torch.float32, torch.bfloat16):
        out, fin, cso = _run(inp, flags, segments, out_dtype)
        assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(fin).all())
        tol_o = TOL_FP32 if fp32_io and out_dtype == torch.float32 else TOL_OUT_BF16
        tol_s = TOL_FP32 if fp32_io else TOL_STATE_BF16
        check_out(to_np(out), ref["out"], 1, tol_o, bf16_out=out_dtype == torch.bfloat16)
        err = per_head_rel(to_np(fin), ref["final_state"], 1)
        assert err.max() <= tol_s, f"final state err {err.max():.3e} > {tol_s:.1e}"
        np.testing.assert_array_equal(synth.to_f32_numpy(cso), ref["conv_state_out"].astype(np.float32))


def _conv_qkv(inp):
    """Convolved, activated q, k, v of the given inputs from the oracle's conv piece, with q
    and k L2-normalised: [T, H, D] each, fp64."""
    a = head_slice_inputs(inp, range(inp.H))
    T, H, D = inp.T, inp.H, inp.D
    x = np.concatenate([a["q"].reshape(T, -1), a["k"].reshape(T, -1), a["v"].reshape(T, -1)], 1)
    y, _ = oracle.conv_silu(x, a["conv_w"].reshape(-1, 4), inp.cu_seqlens, state_in=a["conv_state_in"])
    y = y.reshape(T, 3, H, D)
    return oracle.l2norm(y[:, 0]), oracle.l2norm(y[:, 1]), y[:, 2]


@pytest.mark.parametrize("path", list(PATHS))
def test_closed_form_no_decay_no_write_keeps_state(path):
    """alpha = 1, beta = 0: S_T = S_0 to fp32 rounding, and o_t = S_0^T q_t at every token."""
    inp, flags, segments = _inputs(path, "zero", "zero", 401)
    out, fin, _ = _run(inp, flags, segments, torch.float32)
    err = per_head_rel(to_np(fin), to_np(inp.initial_state), 1)
    assert err.max() <= 1e-5, f"state moved by {err.max():.3e} with alpha = 1, beta = 0"
    q, _, _ = _conv_qkv(inp)
    S0 = to_np(inp.initial_state)                     # [N, H, D, D]
    o = np.zeros_like(q)
    cu = inp.cu_seqlens
    for n in range(inp.N):
        s = slice(int(cu[n]), int(cu[n + 1]))
        o[s] = np.einsum("thc,hcj->thj", q[s], S0[n])
    y = oracle.rmsnorm_gate(o, synth.to_f32_numpy(inp.gate), synth.to_f32_numpy(inp.rms_w))
    tol = TOL_FP32 if inp.io == "fp32" else TOL_OUT_BF16
    check_out(to_np(out), y, 1, tol, bf16_out=False)


@pytest.mark.parametrize("g_mode", ["min", "zero", "rand"])
@pytest.mark.parametrize("path", list(PATHS))
def test_closed_form_full_write_recalls_value(path, g_mode):
    """beta = 1, q = k: the readout after the write is the token's own value, for any decay,
    so without a gate y_t = v_t / sqrt(mean(v_t^2) + eps) * w."""
    inp, flags, segments = _inputs(path, "zero" if g_mode == "rand" else g_mode, "one", 402)
    if g_mode == "rand":
        inp.g.uniform_(-5.0, 0.0)
    inp.k.copy_(inp.q)
    H, D = inp.H, inp.D
    inp.conv_w.view(3, H * D, 4)[1].copy_(inp.conv_w.view(3, H * D, 4)[0])
    if inp.conv_state_in is not None:
        cs = inp.conv_state_in.view(inp.N, 3, H * D, 3)
        cs[:, 1].copy_(cs[:, 0])
    inp.gate = None
    # eps_l2 = 0 makes |k| = 1 exactly in the closed form
    out, fin, _ = _run(inp, flags, segments, torch.float32, eps_l2=0.0)
    _, _, v = _conv_qkv(inp)
    y = oracle.rmsnorm_gate(v, None, synth.to_f32_numpy(inp.rms_w))
    tol = TOL_FP32 if inp.io == "fp32" else TOL_OUT_BF16
    check_out(to_np(out), y, 1, tol, bf16_out=False)


@pytest.mark.parametrize("beta_mode", BETA_MODES)
@pytest.mark.parametrize("g_mode", G_MODES)
def test_decode_decay_and_strength_extremes(g_mode, beta_mode):
    """The single-token decode step over 70 steps (more than a chunk) at the ends of the decay
    and write-strength ranges, against the oracle over the whole stream."""
    N, H, D, steps = 3, 2, 128, 70
    seed = 500 + 10 * G_MODES.index(g_mode) + BETA_MODES.index(beta_mode)
    dec = synth.make_decode(seed=seed, device=DEV, N=N, H=H, D=D, ring=steps, rms_w="random")
    _set_g(dec.g, g_mode, seed)
    _set_beta(dec.beta, beta_mode)
    st0 = dec.state.clone()
    cs0 = dec.conv_state.clone()
    outs = []
    for i in range(steps):
        outs.append(kda.kda_decode_step(dec.q[i], dec.k[i], dec.v[i], dec.g[i], dec.beta[i],
                                        dec.conv_w, dec.state, dec.conv_state, gate=dec.gate[i],
                                        rms_w=dec.rms_w, out_dtype=torch.float32).clone())
    torch.cuda.synchronize()
    o = torch.stack(outs, 1).reshape(N * steps, H, D)

    def seq_major(t):
        return t.transpose(0, 1).reshape(N * steps, *t.shape[2:])

    inp = synth.PrefillInputs(N=N, H=H, D=D, chunk=64, io="bf16",
                              cu_seqlens=synth.cu_from_lengths([steps] * N), q=seq_major(dec.q),
                              k=seq_major(dec.k), v=seq_major(dec.v), conv_w=dec.conv_w,
                              g=seq_major(dec.g), beta=seq_major(dec.beta), gate=seq_major(dec.gate),
                              rms_w=dec.rms_w, initial_state=st0, conv_state_in=cs0)
    ref = oracle_prefill(inp)
    check_out(to_np(o), ref["out"], 1, TOL_OUT_BF16, bf16_out=False)
    err = per_head_rel(to_np(dec.state), ref["final_state"], 1)
    assert err.max() <= TOL_STATE_BF16, f"final state err {err.max():.3e}"
    if g_mode == "zero" and beta_mode == "zero":
        assert per_head_rel(to_np(dec.state), to_np(st0), 1).max() <= 1e-6
    np.testing.assert_array_equal(synth.to_f32_numpy(dec.conv_state),
                                  ref["conv_state_out"].astype(np.float32))
