"""Shared helpers for the KDA tests: run the oracle on (a head slice of) a
synthetic batch, and the error metrics the tolerances are stated in.

Tolerances (bf16 inputs, fp32 state): outputs <= 2e-3 and final states <=
1e-3 in max relative error, measured per head as max|gpu - ref| / max|ref|
over that head's tokens and channels; <= 1e-5 for fp32 I/O.  A bf16 output
is additionally allowed its own rounding, 2^-8 |ref| per element (the unit
roundoff of bf16: the correctly rounded value can be that far from the fp64
one), since no kernel can store a bf16 result closer than that.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kimi_delta_attention_16_gb300 import synth

TOL_OUT_BF16 = 2e-3
TOL_STATE_BF16 = 1e-3
TOL_FP32 = 1e-5
BF16_U = 2.0 ** -8


def head_slice_inputs(inp: synth.PrefillInputs, heads):
    """Host fp32 copies of the inputs of the given heads only (exact values)."""
    hs = torch.as_tensor(list(heads), dtype=torch.long, device=inp.q.device)
    H, D, N = inp.H, inp.D, inp.N
    f = synth.to_f32_numpy

    def sel(t, axis):
        return None if t is None else f(torch.index_select(t, axis, hs))

    cw = inp.conv_w.view(3, H, D, 4)
    cs = None
    if inp.conv_state_in is not None:
        cs = f(torch.index_select(inp.conv_state_in.view(N, 3, H, D, 3), 2, hs)).reshape(N, -1, 3)
    return dict(q=sel(inp.q, 1), k=sel(inp.k, 1), v=sel(inp.v, 1),
                conv_w=f(torch.index_select(cw, 1, hs)).reshape(3, -1, 4),
                cu_seqlens=inp.cu_seqlens, g=sel(inp.g, 1), beta=sel(inp.beta, 1),
                gate=sel(inp.gate, 1), rms_w=f(inp.rms_w),
                initial_state=sel(inp.initial_state, 1), conv_state_in=cs)


def oracle_prefill(inp: synth.PrefillInputs, heads=None, eps_l2=1e-6, eps_rms=1e-6, scale=1.0,
                   want_o_pre=False):
    heads = list(range(inp.H)) if heads is None else list(heads)
    a = head_slice_inputs(inp, heads)
    return oracle.forward(**a, eps_l2=eps_l2, eps_rms=eps_rms, scale=scale, want_o_pre=want_o_pre)


def per_head_rel(gpu: np.ndarray, ref: np.ndarray, head_axis: int) -> np.ndarray:
    """max|gpu-ref| / max|ref| for every index of head_axis."""
    g = np.moveaxis(np.asarray(gpu, np.float64), head_axis, 0).reshape(gpu.shape[head_axis], -1)
    r = np.moveaxis(np.asarray(ref, np.float64), head_axis, 0).reshape(ref.shape[head_axis], -1)
    den = np.maximum(np.abs(r).max(1), 1e-30)
    return np.abs(g - r).max(1) / den


def check_out(gpu, ref, head_axis, tol, bf16_out):
    """Per-head max relative error; a bf16 result also gets its own rounding allowance.

    Returns the worst per-head error with the rounding allowance removed."""
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    if not bf16_out:
        err = per_head_rel(g, r, head_axis)
        assert err.max() <= tol, f"max per-head rel err {err.max():.3e} > {tol:.1e}"
        return float(err.max())
    gm = np.moveaxis(g, head_axis, 0).reshape(g.shape[head_axis], -1)
    rm = np.moveaxis(r, head_axis, 0).reshape(r.shape[head_axis], -1)
    scale = np.maximum(np.abs(rm).max(1, keepdims=True), 1e-30)
    excess = np.maximum(np.abs(gm - rm) - BF16_U * np.abs(rm), 0.0) / scale
    worst = float(excess.max())
    assert worst <= tol, f"max per-head rel err beyond bf16 rounding {worst:.3e} > {tol:.1e}"
    return worst


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()
