"""GPU parity of the segment-parallel scan of the tensor-core prefill.

A sequence cut into P segments is computed as: segment 0 from the initial
state, every later segment twice (from S = 0, and from S = I with v = 0), an
in-order composition of the segments' affine state maps, and a fix-up of the
outputs.  The result must meet the same tolerances against the fp64 oracle as
the single-pass path.  Most cases use a slow log-decay (g ~ U[-0.05, 0]) so
that the state carried across a segment boundary is large and a wrong
composition or fix-up shows; with the workloads' g ~ U[-5, 0] the state
forgets within a chunk.
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_16_gb300 as kda
from kimi_delta_attention_16_gb300 import synth
from kda_testlib import TOL_OUT_BF16, TOL_STATE_BF16, check_out, oracle_prefill, per_head_rel, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
MILD = (-0.05, 0.0)


def _run(inp, segments, out_dtype=None, final_state=None, initial_state="inp"):
    s0 = inp.initial_state if initial_state == "inp" else initial_state
    out, fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens,
                               chunk=inp.chunk, gate=inp.gate, rms_w=inp.rms_w, initial_state=s0,
                               final_state=final_state, conv_state_in=inp.conv_state_in,
                               out_dtype=out_dtype, segments=segments)
    torch.cuda.synchronize()
    return out, fin


def _check(inp, out, fin, ref, bf16_out=True):
    check_out(to_np(out), ref["out"], 1, TOL_OUT_BF16, bf16_out=bf16_out)
    err = per_head_rel(to_np(fin), ref["final_state"], 1)
    assert err.max() <= TOL_STATE_BF16, f"final state err {err.max():.3e}"


def _plan(inp, segments=0):
    return kda.kda_prefill_plan(inp.T, inp.H, inp.D, N=inp.N, chunk=inp.chunk, segments=segments)


@pytest.mark.parametrize("P", [2, 3, 5, 16])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_segments_parity_slow_decay(P, out_dtype):
    """One ragged sequence (37 full chunks + 29 tokens), nonzero initial and conv states,
    random RMSNorm weight, gate on."""
    inp = synth.make_prefill("layer_8k", seed=40 + P, device=DEV, N=1, T=64 * 37 + 29, H=3, s0_std=0.02,
                             conv_state=True, rms_w="random", g_range=MILD)
    assert _plan(inp, P) == ("tc", P)
    out, fin = _run(inp, P, out_dtype=out_dtype)
    _check(inp, out, fin, oracle_prefill(inp), bf16_out=out_dtype == torch.bfloat16)


@pytest.mark.parametrize("gate", [True, False])
def test_segments_varlen_with_short_and_empty_sequences(gate):
    """Packed sequences of 1, 70, 0, 640, 1900 and 129 tokens cut into 4 segments each:
    short sequences leave trailing segments empty (identity maps)."""
    inp = synth.make_prefill("layer_8k", seed=50, device=DEV, lengths=[1, 70, 0, 640, 1900, 129], H=2,
                             s0_std=0.02, gate=gate, g_range=MILD)
    out, fin = _run(inp, 4)
    _check(inp, out, fin, oracle_prefill(inp))


def test_segments_agree_with_single_pass():
    """The same batch through 1 and 6 segments: both within tolerance of the oracle and of
    each other."""
    inp = synth.make_prefill("layer_8k", seed=51, device=DEV, N=2, T=2 * 64 * 30, H=2, s0_std=0.02,
                             g_range=MILD)
    ref = oracle_prefill(inp)
    o1, f1 = _run(inp, 1)
    o6, f6 = _run(inp, 6)
    _check(inp, o1, f1, ref)
    _check(inp, o6, f6, ref)
    assert per_head_rel(to_np(o6), to_np(o1), 1).max() <= 2 * TOL_OUT_BF16
    assert per_head_rel(to_np(f6), to_np(f1), 1).max() <= 2 * TOL_STATE_BF16


def test_segments_workload_decay():
    """The workloads' own log-decay law, U[-5, 0], through 3 segments."""
    inp = synth.make_prefill("layer_8k", seed=52, device=DEV, N=1, T=64 * 50, H=4)
    out, fin = _run(inp, 3)
    _check(inp, out, fin, oracle_prefill(inp))


def test_segments_in_place_state():
    """final_state may be the initial_state buffer: the composition writes it only after every
    segment has read its start."""
    inp = synth.make_prefill("layer_8k", seed=53, device=DEV, N=2, T=3000, H=2, s0_std=0.02, g_range=MILD)
    ref = oracle_prefill(inp)
    st = inp.initial_state.clone()
    out, fin = _run(inp, 3, final_state=st, initial_state=st)
    assert fin.data_ptr() == st.data_ptr()
    _check(inp, out, fin, ref)


def test_auto_plan_fills_the_sms():
    """The automatic choice: batches with fewer (sequence, head) units than SMs are cut into
    segments (at most 16), others are not; `segments` forces a count."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for name in ("long_1m", "layer_8k"):
        w = synth.WORKLOADS[name]
        path, P = kda.kda_prefill_plan(w["T"], w["H"], w["D"], N=w["N"])
        assert path == "tc"
        if w["N"] * w["H"] < sms:
            assert 2 <= P <= 16, (name, P)
    assert kda.kda_prefill_plan(73000, 96, 128, N=16) == ("tc", 1)       # 1,536 units
    assert kda.kda_prefill_plan(8192, sms, 128) == ("tc", 1)             # units = SMs
    assert kda.kda_prefill_plan(1 << 20, 24, 128, segments=1) == ("tc", 1)
    assert kda.kda_prefill_plan(1 << 20, 24, 128, segments=5) == ("tc", 5)
    assert kda.kda_prefill_plan(1 << 20, 24, 128, io=torch.float32)[0] == "simt"
    assert kda.kda_prefill_plan(256, 4, 128)[1] == 1                      # 4 chunks: too short


def test_auto_plan_unequal_segments_parity():
    """The automatic plan on a batch with fewer units than SMs (unequal segments: a long first
    segment, short later ones) against the oracle, slow decay."""
    inp = synth.make_prefill("layer_8k", seed=55, device=DEV, N=1, T=64 * 100 + 17, H=48,
                             s0_std=0.02, conv_state=True, g_range=MILD)
    assert _plan(inp)[1] >= 2
    out, fin = _run(inp, 0)
    heads = [0, 17, 47]
    ref = oracle_prefill(inp, heads=heads)
    check_out(to_np(out[:, heads]), ref["out"], 1, TOL_OUT_BF16, bf16_out=True)
    assert per_head_rel(to_np(fin[:, heads]), ref["final_state"], 1).max() <= TOL_STATE_BF16


@pytest.mark.slow
def test_segments_long_slow_decay_sampled_heads():
    """T = 262,144 (4096 chunks), H = 24 in the automatic plan, slow decay: two sampled heads
    over the full length."""
    inp = synth.make_prefill("long_1m", seed=54, device=DEV, T=1 << 18, g_range=MILD)
    path, P = _plan(inp)
    assert path == "tc"
    out, fin = _run(inp, 0)
    heads = [3, 20]
    ref = oracle_prefill(inp, heads=heads)
    check_out(to_np(out[:, heads]), ref["out"], 1, TOL_OUT_BF16, bf16_out=True)
    err = per_head_rel(to_np(fin[:, heads]), ref["final_state"], 1)
    assert err.max() <= TOL_STATE_BF16
