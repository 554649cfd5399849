"""kda_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Some callers have no way to allocate device memory at call time -- a plugin
inside a host application that owns every device allocation and hands over
only input and output buffers, a service that reserved its memory budget at
start-up, or a latency-critical loop that cannot afford cudaMalloc's
device-wide synchronisation.  kda_prefill_noalloc serves them: it takes the
same arguments as kda_prefill minus the workspace, and runs the fp32 SIMT
path with its scratch in a fixed array inside the library.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.  It passes on its own in a fresh
process too: nothing here depends on state left by earlier tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import kimi_delta_attention_16_gb300 as kda
from kimi_delta_attention_16_gb300 import _lib, api, synth
from kda_testlib import TOL_OUT_BF16, TOL_STATE_BF16, check_out, oracle_prefill, per_head_rel, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc_call(inp, out, fin, cs_out):
    """One kda_prefill_noalloc call through the C ABI (no workspace passed)."""
    cu_dev = torch.from_numpy(inp.cu_seqlens).to(DEV)
    a = api._prefill_args(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, cu_dev,
                          inp.cu_seqlens, chunk=inp.chunk, gate=inp.gate, rms_w=inp.rms_w,
                          eps_l2=1e-6, eps_rms=1e-6, scale=1.0, initial_state=inp.initial_state,
                          final_state=fin, conv_state_in=inp.conv_state_in,
                          conv_state_out=cs_out, out=out, workspace=None, d_status=None, flags=0,
                          check_cu_on_host=True)
    st = _lib.load().kda_prefill_noalloc(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    return st


def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    """Two consecutive calls (different inputs, the second reusing the fixed scratch the
    first one filled) each match the regular entry point and the fp64 oracle within the
    parity tolerances (fp32 outputs, so the plain bound applies)."""
    for call, lengths in enumerate(([100, 37, 200], [65, 1, 129, 64])):
        inp = synth.make_prefill("layer_8k", seed=200 + call, device=DEV, lengths=lengths, H=4,
                                 s0_std=0.02, conv_state=True, rms_w="random")
        ref_cs = torch.empty_like(inp.conv_state_in)
        ref_out, ref_fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta,
                                           inp.cu_seqlens, chunk=64, gate=inp.gate,
                                           rms_w=inp.rms_w, initial_state=inp.initial_state,
                                           conv_state_in=inp.conv_state_in,
                                           conv_state_out=ref_cs, out_dtype=torch.float32)
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        cs = torch.zeros_like(ref_cs)
        assert _noalloc_call(inp, out, fin, cs) == 0, _lib.load().kda_last_error()
        torch.cuda.synchronize()
        assert per_head_rel(to_np(out), to_np(ref_out), 1).max() <= TOL_OUT_BF16
        assert per_head_rel(to_np(fin), to_np(ref_fin), 1).max() <= TOL_STATE_BF16
        assert torch.equal(cs, ref_cs)
        ref = oracle_prefill(inp)
        check_out(to_np(out), ref["out"], 1, TOL_OUT_BF16, bf16_out=False)
        assert per_head_rel(to_np(fin), ref["final_state"], 1).max() <= TOL_STATE_BF16
        np.testing.assert_array_equal(synth.to_f32_numpy(cs), ref["conv_state_out"].astype(np.float32))


def test_noalloc_rejects_problems_beyond_its_fixed_scratch():
    """16 * T * H * D bytes above the fixed size: a clear error, nothing launched."""
    H, D = 96, 128
    T = _lib.NOALLOC_SCRATCH_BYTES // (16 * H * D) + 1
    inp = synth.make_prefill("layer_8k", seed=3, device=DEV, lengths=[T], H=H)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    st = _noalloc_call(inp, out, None, None)
    assert st == _lib.KDA_ERR_WORKSPACE
    assert b"fixed scratch" in _lib.load().kda_last_error()
