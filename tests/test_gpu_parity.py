"""GPU parity: libkda.so (called through its C ABI) against the fp64 oracle.

Tolerances are the ones stated for the layer: per-head max relative error
<= 2e-3 on outputs and <= 1e-3 on final states with bf16 inputs and an fp32
state, <= 1e-5 with fp32 I/O; the rolling conv state is copied data and
must match bit for bit; cu_seqlens indexing is checked bit-exactly through
packed-vs-solo runs.  Sizes range from a few tokens to the full workloads the
benchmark times (there on sampled heads / sequences, which is exact because
every (sequence, head) unit is independent).
"""
import ctypes

import numpy as np
import pytest
import torch

import kimi_delta_attention_16_gb300 as kda
from kimi_delta_attention_16_gb300 import _lib, synth
from kda_testlib import (TOL_FP32, TOL_OUT_BF16, TOL_STATE_BF16, check_out, oracle_prefill,
                         per_head_rel, to_np)
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _prefill(inp, flags=0, out_dtype=None, conv_out=False, **kw):
    cso = None
    if conv_out:
        cso = torch.empty((inp.N, 3 * inp.H * inp.D, 3), dtype=inp.q.dtype, device=DEV)
    out, fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta,
                               inp.cu_seqlens, chunk=inp.chunk, gate=inp.gate, rms_w=inp.rms_w,
                               initial_state=inp.initial_state,
                               conv_state_in=inp.conv_state_in, conv_state_out=cso,
                               out_dtype=out_dtype, flags=flags, **kw)
    torch.cuda.synchronize()
    return out, fin, cso


def _check_prefill(inp, out, fin, ref, out_tol, state_tol, bf16_out, heads=None):
    o = to_np(out)
    f = to_np(fin)
    if heads is not None:
        o = o[:, heads]
        f = f[:, heads]
    check_out(o, ref["out"], 1, out_tol, bf16_out)
    err_s = per_head_rel(f, ref["final_state"], 1)
    assert err_s.max() <= state_tol, f"final state err {err_s.max():.3e} > {state_tol:.1e}"


# --------------------------------------------------------------------------- short conv

@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("D", [16, 128])
def test_short_conv_parity(io, D):
    inp = synth.make_prefill("tiny_fp32", seed=21, device=DEV, lengths=[1, 2, 5, 40, 33], H=3, D=D,
                             io=io, conv_state=True)
    T, H = inp.T, inp.H
    # a fused, row-strided buffer: [T, 3*H*D + pad]
    pad = 8
    buf = torch.zeros((T, 3 * H * D + pad), dtype=inp.q.dtype, device=DEV)
    x = buf[:, :3 * H * D]
    x.copy_(torch.cat([inp.q.reshape(T, -1), inp.k.reshape(T, -1), inp.v.reshape(T, -1)], 1))
    cso = torch.empty_like(inp.conv_state_in)
    y = kda.kda_short_conv(x, inp.conv_w.reshape(-1, 4), inp.cu_seqlens, H=H, D=D,
                           conv_state_in=inp.conv_state_in, conv_state_out=cso)
    torch.cuda.synchronize()
    yr, sor = oracle.conv_silu(synth.to_f32_numpy(x), synth.to_f32_numpy(inp.conv_w).reshape(-1, 4),
                               inp.cu_seqlens, state_in=synth.to_f32_numpy(inp.conv_state_in))
    yr = yr.reshape(T, 3, H, D)
    yr[:, 0] = oracle.l2norm(yr[:, 0])
    yr[:, 1] = oracle.l2norm(yr[:, 1])
    yg = to_np(y).reshape(T, 3, H, D)
    if io == "fp32":
        assert np.abs(yg - yr).max() <= 1e-6 * max(1.0, np.abs(yr).max())
    else:
        assert np.all(np.abs(yg - yr) <= 2.0 ** -8 * np.abs(yr) + 1e-6)
    np.testing.assert_array_equal(synth.to_f32_numpy(cso), sor.astype(np.float32))


# --------------------------------------------------------------------------- fp32 path

@pytest.mark.parametrize("gate,rms", [(True, "ones"), (False, None), (True, "random")])
def test_prefill_tiny_fp32(gate, rms):
    """B=1, T=64, H=2, d=16, chunk 16, fp32 I/O, zero initial state: <= 1e-5."""
    inp = synth.make_prefill("tiny_fp32", seed=0, device=DEV, gate=gate, rms_w=rms)
    out, fin, _ = _prefill(inp)
    ref = oracle_prefill(inp)
    _check_prefill(inp, out, fin, ref, TOL_FP32, TOL_FP32, bf16_out=False)


@pytest.mark.parametrize("D,chunk", [(16, 32), (32, 16), (64, 64), (128, 32)])
def test_prefill_fp32_shapes(D, chunk):
    inp = synth.make_prefill("tiny_fp32", seed=D + chunk, device=DEV, lengths=[1, 3, 70, 129],
                             H=2, D=D, chunk=chunk, s0_std=0.05, conv_state=True, rms_w="random")
    out, fin, cso = _prefill(inp, conv_out=True, eps_l2=1e-4, eps_rms=1e-3, scale=0.8)
    ref = oracle_prefill(inp, eps_l2=1e-4, eps_rms=1e-3, scale=0.8)
    _check_prefill(inp, out, fin, ref, TOL_FP32, TOL_FP32, bf16_out=False)
    np.testing.assert_array_equal(synth.to_f32_numpy(cso), ref["conv_state_out"].astype(np.float32))


# --------------------------------------------------------------------------- bf16, D = 128

# the last entry is the multi-token continuation shape (8 sequences x 4 new tokens from carried
# states and conv states, as in speculative verification)
SMALL_LENGTHS = [[1], [2], [3], [5], [63], [64], [65], [127], [130], [1, 64, 3, 200, 65], [4] * 8]


# flags: 0 = the library's own choice (the recurrent path when every sequence has at most 8
# tokens, else the tensor-core path), NO_RECURRENT = the tensor-core path, FORCE_SIMT
@pytest.mark.parametrize("lengths", SMALL_LENGTHS)
@pytest.mark.parametrize("flags", [0, _lib.KDA_FLAG_NO_RECURRENT, _lib.KDA_FLAG_FORCE_SIMT])
def test_prefill_bf16_small(lengths, flags):
    inp = synth.make_prefill("layer_8k", seed=sum(lengths), device=DEV, lengths=lengths, H=4,
                             s0_std=0.02, conv_state=True, rms_w="random")
    ref = oracle_prefill(inp)
    for out_dtype in (torch.float32, torch.bfloat16):
        out, fin, cso = _prefill(inp, flags=flags, out_dtype=out_dtype, conv_out=True)
        _check_prefill(inp, out, fin, ref, TOL_OUT_BF16, TOL_STATE_BF16,
                       bf16_out=out_dtype == torch.bfloat16)
        np.testing.assert_array_equal(synth.to_f32_numpy(cso),
                                      ref["conv_state_out"].astype(np.float32))


def test_prefill_empty_sequences_and_zero_tokens():
    inp = synth.make_prefill("layer_8k", seed=5, device=DEV, lengths=[0, 7, 0], H=2, s0_std=0.1)
    out, fin, _ = _prefill(inp)
    ref = oracle_prefill(inp)
    _check_prefill(inp, out, fin, ref, TOL_OUT_BF16, TOL_STATE_BF16, bf16_out=True)
    # an empty sequence hands its initial state through unchanged
    torch.testing.assert_close(fin[0], inp.initial_state[0], rtol=0, atol=0)
    torch.testing.assert_close(fin[2], inp.initial_state[2], rtol=0, atol=0)


@pytest.mark.parametrize("flags,lengths", [
    (_lib.KDA_FLAG_NO_RECURRENT, [70, 1, 128, 5, 64]),
    (_lib.KDA_FLAG_FORCE_SIMT, [70, 1, 128, 5, 64]),
    (0, [1, 8, 3, 0, 5]),  # all short: the recurrent path for the batch and for each solo run
])
def test_packed_equals_solo_bitwise(flags, lengths):
    """cu_seqlens indexing: each sequence of a packed batch equals its solo run bit for bit
    (both through the same path)."""
    inp = synth.make_prefill("layer_8k", seed=9, device=DEV, lengths=lengths, H=3, s0_std=0.02,
                             conv_state=True)
    out, fin, _ = _prefill(inp, flags=flags)
    cu = inp.cu_seqlens
    for n in range(len(lengths)):
        s = slice(int(cu[n]), int(cu[n + 1]))
        o1, f1 = kda.kda_prefill(inp.q[s], inp.k[s], inp.v[s], inp.conv_w, inp.g[s], inp.beta[s],
                                 [0, lengths[n]], chunk=64, gate=inp.gate[s], rms_w=inp.rms_w,
                                 initial_state=inp.initial_state[n:n + 1].contiguous(),
                                 conv_state_in=inp.conv_state_in[n:n + 1].contiguous(),
                                 flags=flags)
        torch.cuda.synchronize()
        assert torch.equal(o1, out[s])
        assert torch.equal(f1[0], fin[n])


@pytest.mark.parametrize("T1", [64, 37])
def test_prefill_handoff(T1):
    """prefill(T1+T2) == prefill(T1) -> prefill(T2) with the state and conv-state hand-off."""
    inp = synth.make_prefill("layer_8k", seed=T1, device=DEV, lengths=[200], H=2, s0_std=0.02)
    out, fin, _ = _prefill(inp)
    s1, s2 = slice(0, T1), slice(T1, 200)
    cs = torch.empty((1, 3 * 2 * 128, 3), dtype=torch.bfloat16, device=DEV)
    o1, f1 = kda.kda_prefill(inp.q[s1], inp.k[s1], inp.v[s1], inp.conv_w, inp.g[s1], inp.beta[s1],
                             [0, T1], gate=inp.gate[s1], rms_w=inp.rms_w,
                             initial_state=inp.initial_state, conv_state_out=cs)
    o2, f2 = kda.kda_prefill(inp.q[s2], inp.k[s2], inp.v[s2], inp.conv_w, inp.g[s2], inp.beta[s2],
                             [0, 200 - T1], gate=inp.gate[s2], rms_w=inp.rms_w, initial_state=f1,
                             conv_state_in=cs)
    torch.cuda.synchronize()
    ref = oracle_prefill(inp)
    both = torch.cat([o1, o2])
    check_out(to_np(both), ref["out"], 1, TOL_OUT_BF16, True)
    assert per_head_rel(to_np(f2)[0], ref["final_state"][0], 0).max() <= TOL_STATE_BF16


def test_prefill_then_decode_handoff():
    """prefill(T1) -> decode steps == the oracle over the whole stream."""
    T, T1, H = 20, 13, 2
    inp = synth.make_prefill("layer_8k", seed=33, device=DEV, lengths=[T], H=H, s0_std=0.02)
    cs = torch.empty((1, 3 * H * 128, 3), dtype=torch.bfloat16, device=DEV)
    o1, st = kda.kda_prefill(inp.q[:T1], inp.k[:T1], inp.v[:T1], inp.conv_w, inp.g[:T1],
                             inp.beta[:T1], [0, T1], gate=inp.gate[:T1], rms_w=inp.rms_w,
                             initial_state=inp.initial_state, conv_state_out=cs)
    outs = [o1]
    for t in range(T1, T):
        s = slice(t, t + 1)
        outs.append(kda.kda_decode_step(inp.q[s], inp.k[s], inp.v[s], inp.g[s], inp.beta[s],
                                        inp.conv_w, st, cs, gate=inp.gate[s], rms_w=inp.rms_w))
    torch.cuda.synchronize()
    ref = oracle_prefill(inp)
    check_out(to_np(torch.cat(outs)), ref["out"], 1, TOL_OUT_BF16, True)
    assert per_head_rel(to_np(st)[0], ref["final_state"][0], 0).max() <= TOL_STATE_BF16


def test_device_side_cu_check_flags_status():
    """An inconsistent device cu_seqlens (no host copy) is reported via d_status; all
    indices stay clamped inside the buffers, so nothing faults."""
    inp = synth.make_prefill("layer_8k", seed=2, device=DEV, lengths=[30, 34], H=2)
    bad = torch.tensor([0, 50, 30], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    a = kda.api._prefill_args(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, bad,
                              np.array([0, 30, 64], np.int32), chunk=64, gate=None, rms_w=None,
                              eps_l2=1e-6, eps_rms=1e-6, scale=1.0, initial_state=None,
                              final_state=None, conv_state_in=None, conv_state_out=None,
                              out=torch.empty_like(inp.q), workspace=None, d_status=status,
                              flags=0, check_cu_on_host=False)
    n = ctypes.c_size_t()
    lib = _lib.load()
    assert lib.kda_prefill_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    ws = torch.empty(max(n.value, 1), dtype=torch.uint8, device=DEV)
    a.workspace, a.workspace_bytes = ws.data_ptr(), n.value
    assert lib.kda_prefill(ctypes.byref(a), None) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == _lib.KDA_ERR_DEVICE_ARG


def test_dropped_staging_times_out_and_reports():
    """Failure detection without a fault: with KDA_FLAG_TEST_DROP_STAGING the tensor-core
    kernel never issues its first q/k row staging, its bounded mbarrier wait runs out, and it
    writes KDA_ERR_TIMEOUT to d_status and returns.  The context stays usable: the same call
    without the flag then matches the oracle."""
    inp = synth.make_prefill("layer_8k", seed=3, device=DEV, N=1, T=200, H=1, s0_std=0.02)
    assert kda.kda_prefill_plan(inp.T, inp.H, inp.D, N=inp.N)[0] == "tc"
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens, gate=inp.gate,
                    rms_w=inp.rms_w, initial_state=inp.initial_state, d_status=status,
                    flags=_lib.KDA_FLAG_TEST_DROP_STAGING)
    torch.cuda.synchronize()
    assert int(status.item()) == _lib.KDA_ERR_TIMEOUT
    status.zero_()
    out, fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens,
                               gate=inp.gate, rms_w=inp.rms_w, initial_state=inp.initial_state,
                               d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle_prefill(inp)
    check_out(to_np(out), ref["out"], 1, TOL_OUT_BF16, True)
    assert per_head_rel(to_np(fin), ref["final_state"], 1).max() <= TOL_STATE_BF16


def _guarded(shape, dtype, guard, fill):
    """A tensor of `shape` inside a 1-D buffer with `guard` elements of `fill` on each side."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * guard,), fill, dtype=dtype, device=DEV)
    return buf, buf[guard:guard + n].view(shape)


@pytest.mark.parametrize("case", ["tensor_core_segments", "simt_fp32", "recurrent"])
def test_guard_bands_and_poisoned_workspace(case):
    """Every output lives inside guard bands that must come back untouched, and the workspace
    is filled with NaN bytes (0xFF) first: a write out of bounds changes a guard, a read of
    scratch the call did not write puts a NaN into the result."""
    if case == "tensor_core_segments":
        inp = synth.make_prefill("layer_8k", seed=81, device=DEV, N=1, T=64 * 20 + 13, H=2, s0_std=0.02,
                                 conv_state=True, g_range=(-0.05, 0.0))
        segments, path = 3, "tc"
    elif case == "simt_fp32":
        inp = synth.make_prefill("layer_8k", seed=82, device=DEV, lengths=[70, 1, 130], H=2, io="fp32",
                                 s0_std=0.02, conv_state=True)
        segments, path = 0, "simt"
    else:
        inp = synth.make_prefill("layer_8k", seed=83, device=DEV, lengths=[3, 8, 1], H=2, s0_std=0.02,
                                 conv_state=True)
        segments, path = 0, "recurrent"
    assert kda.kda_prefill_plan(inp.T, inp.H, inp.D, N=inp.N, io=inp.q.dtype, segments=segments,
                                cu_seqlens=inp.cu_seqlens)[0] == path
    G = 4096
    dt = inp.q.dtype
    out_buf, out = _guarded((inp.T, inp.H, inp.D), dt, G, -7.0)
    fin_buf, fin = _guarded((inp.N, inp.H, inp.D, inp.D), torch.float32, G, -7.0)
    cso_buf, cso = _guarded((inp.N, 3 * inp.H * inp.D, 3), dt, G, -7.0)
    n_ws = kda.kda_prefill_workspace_size(inp.T, inp.H, inp.D, N=inp.N, io=dt, segments=segments)
    ws_buf = torch.full((n_ws + 2 * G,), 0xFF, dtype=torch.uint8, device=DEV)
    ws = ws_buf[G:G + n_ws]
    kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens, chunk=inp.chunk,
                    gate=inp.gate, rms_w=inp.rms_w, initial_state=inp.initial_state, final_state=fin,
                    conv_state_in=inp.conv_state_in, conv_state_out=cso, out=out, workspace=ws,
                    segments=segments)
    torch.cuda.synchronize()
    for buf in (out_buf, fin_buf, cso_buf):
        assert bool((buf[:G] == -7.0).all()) and bool((buf[-G:] == -7.0).all())
    assert bool((ws_buf[:G] == 0xFF).all()) and bool((ws_buf[-G:] == 0xFF).all())
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(fin).all())
    ref = oracle_prefill(inp)
    tol_o, tol_s = (TOL_FP32, TOL_FP32) if dt == torch.float32 else (TOL_OUT_BF16, TOL_STATE_BF16)
    check_out(to_np(out), ref["out"], 1, tol_o, bf16_out=dt == torch.bfloat16)
    assert per_head_rel(to_np(fin), ref["final_state"], 1).max() <= tol_s
    np.testing.assert_array_equal(synth.to_f32_numpy(cso), ref["conv_state_out"].astype(np.float32))


# --------------------------------------------------------------------------- decode

@pytest.mark.parametrize("D,io", [(128, "bf16"), (64, "bf16"), (16, "fp32"), (32, "fp32")])
def test_decode_small(D, io):
    N, H, steps = 5, 3, 6
    dec = synth.make_decode(seed=D, device=DEV, N=N, H=H, D=D, ring=steps, io=io, rms_w="random")
    st0 = dec.state.clone()
    cs0 = dec.conv_state.clone()
    outs = []
    for i in range(steps):
        outs.append(kda.kda_decode_step(dec.q[i], dec.k[i], dec.v[i], dec.g[i], dec.beta[i],
                                        dec.conv_w, dec.state, dec.conv_state, gate=dec.gate[i],
                                        rms_w=dec.rms_w, out_dtype=torch.float32).clone())
    torch.cuda.synchronize()
    o = torch.stack(outs, 1).reshape(N * steps, H, D)  # sequence-major stream
    inp = synth.PrefillInputs(N=N, H=H, D=D, chunk=16, io=io,
                              cu_seqlens=synth.cu_from_lengths([steps] * N),
                              q=dec.q.transpose(0, 1).reshape(N * steps, H, D),
                              k=dec.k.transpose(0, 1).reshape(N * steps, H, D),
                              v=dec.v.transpose(0, 1).reshape(N * steps, H, D),
                              conv_w=dec.conv_w, g=dec.g.transpose(0, 1).reshape(N * steps, H, D),
                              beta=dec.beta.transpose(0, 1).reshape(N * steps, H),
                              gate=dec.gate.transpose(0, 1).reshape(N * steps, H, D),
                              rms_w=dec.rms_w, initial_state=st0, conv_state_in=cs0)
    ref = oracle_prefill(inp)
    tol_o, tol_s = (TOL_FP32, TOL_FP32) if io == "fp32" else (TOL_OUT_BF16, TOL_STATE_BF16)
    check_out(to_np(o), ref["out"], 1, tol_o, False)
    err = per_head_rel(to_np(dec.state), ref["final_state"], 1)
    assert err.max() <= tol_s
    np.testing.assert_array_equal(synth.to_f32_numpy(dec.conv_state),
                                  ref["conv_state_out"].astype(np.float32))
