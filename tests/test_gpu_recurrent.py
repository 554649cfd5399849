"""GPU parity of the recurrent prefill path: batches whose sequences all have at
most 8 tokens (multi-token decode, speculative verification of drafted
tokens), continuing from carried states and rolling conv states.

Against the fp64 oracle with the layer's tolerances, in both I/O dtypes; the
multi-token steps of a stream must equal the oracle over the whole stream, and
a full-size batch (256 sequences x 4 tokens, 96 heads) is checked on sampled
(sequence, head) pairs.
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_16_gb300 as kda
from kimi_delta_attention_16_gb300 import _lib, synth
from kda_testlib import (TOL_FP32, TOL_OUT_BF16, TOL_STATE_BF16, check_out, oracle_prefill,
                         per_head_rel, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(inp, flags=0, out_dtype=None, final_state=None, conv_out=False, initial_state="inp"):
    s0 = inp.initial_state if initial_state == "inp" else initial_state
    cso = torch.empty((inp.N, 3 * inp.H * inp.D, 3), dtype=inp.q.dtype, device=DEV) if conv_out else None
    out, fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens,
                               chunk=inp.chunk, gate=inp.gate, rms_w=inp.rms_w, initial_state=s0,
                               final_state=final_state, conv_state_in=inp.conv_state_in,
                               conv_state_out=cso, out_dtype=out_dtype, flags=flags)
    torch.cuda.synchronize()
    return out, fin, cso


# (7 tokens at most: the largest batch whose fp32 rows and states still fit the pipelined kernel's
# shared memory; 8 with fp32 inputs takes the plainer kernel)
LENGTHS = [[1], [2], [4] * 8, [7, 2, 6, 7], [8] * 5, [1, 8, 0, 3, 5, 7]]


@pytest.mark.parametrize("lengths", LENGTHS)
@pytest.mark.parametrize("io", ["bf16", "fp32"])
def test_recurrent_parity(lengths, io):
    inp = synth.make_prefill("layer_8k", seed=60 + sum(lengths), device=DEV, lengths=lengths, H=3,
                             io=io, s0_std=0.02, conv_state=True, rms_w="random")
    assert kda.kda_prefill_plan(inp.T, inp.H, inp.D, cu_seqlens=inp.cu_seqlens, io=inp.q.dtype)[0] == "recurrent"
    ref = oracle_prefill(inp)
    for out_dtype in (torch.float32, torch.bfloat16):
        out, fin, cso = _run(inp, out_dtype=out_dtype, conv_out=True)
        if io == "fp32" and out_dtype == torch.float32:
            check_out(to_np(out), ref["out"], 1, TOL_FP32, bf16_out=False)
            assert per_head_rel(to_np(fin), ref["final_state"], 1).max() <= TOL_FP32
        else:
            check_out(to_np(out), ref["out"], 1, TOL_OUT_BF16, bf16_out=out_dtype == torch.bfloat16)
            assert per_head_rel(to_np(fin), ref["final_state"], 1).max() <= TOL_STATE_BF16
        np.testing.assert_array_equal(synth.to_f32_numpy(cso), ref["conv_state_out"].astype(np.float32))


def test_recurrent_without_initial_state_gate_or_rms():
    inp = synth.make_prefill("layer_8k", seed=71, device=DEV, lengths=[3, 8, 1], H=2, gate=False,
                             rms_w=None)
    assert inp.initial_state is None and inp.conv_state_in is None
    out, fin, _ = _run(inp)
    ref = oracle_prefill(inp)
    check_out(to_np(out), ref["out"], 1, TOL_OUT_BF16, bf16_out=True)
    assert per_head_rel(to_np(fin), ref["final_state"], 1).max() <= TOL_STATE_BF16


def test_recurrent_matches_tensor_core_path():
    """The same short batch through the recurrent and the tensor-core path."""
    inp = synth.make_prefill("layer_8k", seed=72, device=DEV, lengths=[5, 8, 2, 7], H=4,
                             s0_std=0.02, conv_state=True)
    o_r, f_r, _ = _run(inp)
    o_t, f_t, _ = _run(inp, flags=_lib.KDA_FLAG_NO_RECURRENT)
    assert per_head_rel(to_np(o_r), to_np(o_t), 1).max() <= 2 * TOL_OUT_BF16
    assert per_head_rel(to_np(f_r), to_np(f_t), 1).max() <= 2 * TOL_STATE_BF16


@pytest.mark.parametrize("step", [2, 4, 8])
def test_multi_token_stream(step):
    """A 100-token prompt (tensor-core path), then 24 tokens in steps of `step` through the
    recurrent path with the state updated in place and the conv state handed on: equal to the
    oracle over the whole 124-token stream."""
    T0, T = 100, 124
    H = 2
    inp = synth.make_prefill("layer_8k", seed=73 + step, device=DEV, lengths=[T], H=H, s0_std=0.02)
    st = inp.initial_state.clone()
    cs = torch.empty((1, 3 * H * 128, 3), dtype=torch.bfloat16, device=DEV)
    o0, _ = kda.kda_prefill(inp.q[:T0], inp.k[:T0], inp.v[:T0], inp.conv_w, inp.g[:T0], inp.beta[:T0],
                            [0, T0], gate=inp.gate[:T0], rms_w=inp.rms_w, initial_state=st,
                            final_state=st, conv_state_out=cs)
    outs = [o0]
    for t in range(T0, T, step):
        s = slice(t, t + step)
        assert kda.kda_prefill_plan(step, H, 128, cu_seqlens=[0, step])[0] == "recurrent"
        cs2 = torch.empty_like(cs)
        o, _ = kda.kda_prefill(inp.q[s], inp.k[s], inp.v[s], inp.conv_w, inp.g[s], inp.beta[s],
                               [0, step], gate=inp.gate[s], rms_w=inp.rms_w, initial_state=st,
                               final_state=st, conv_state_in=cs, conv_state_out=cs2)
        cs = cs2
        outs.append(o)
    torch.cuda.synchronize()
    ref = oracle_prefill(inp)
    check_out(to_np(torch.cat(outs)), ref["out"], 1, TOL_OUT_BF16, True)
    assert per_head_rel(to_np(st)[0], ref["final_state"][0], 0).max() <= TOL_STATE_BF16


@pytest.mark.slow
def test_verify_256x4_sampled_pairs():
    """256 sequences x 4 new tokens, H = 96, states ~N(0, 0.02^2), conv states ~N(0, 1): the
    full-size multi-token step, sampled (sequence, head) pairs against the oracle."""
    inp = synth.make_prefill("verify_256x4", seed=74, device=DEV)
    assert inp.N == 256 and inp.T == 1024
    out, fin, cso = _run(inp, conv_out=True)
    x = torch.stack([inp.q, inp.k, inp.v])  # [3, T, H, D]
    for n in (0, 37, 255):  # 4 tokens per sequence: the rolled window is its last 3 raw values
        assert torch.equal(cso.view(256, 3, 96, 128, 3)[n], x[:, 4 * n + 1:4 * n + 4].permute(0, 2, 3, 1))
    for n, h in [(0, 0), (37, 11), (128, 50), (255, 95)]:
        sub = synth.PrefillInputs(
            N=1, H=1, D=128, chunk=64, io="bf16", cu_seqlens=synth.cu_from_lengths([4]),
            q=inp.q[4 * n:4 * n + 4, h:h + 1], k=inp.k[4 * n:4 * n + 4, h:h + 1],
            v=inp.v[4 * n:4 * n + 4, h:h + 1],
            conv_w=inp.conv_w.view(3, 96, 128, 4)[:, h].contiguous(),
            g=inp.g[4 * n:4 * n + 4, h:h + 1], beta=inp.beta[4 * n:4 * n + 4, h:h + 1],
            gate=inp.gate[4 * n:4 * n + 4, h:h + 1], rms_w=inp.rms_w,
            initial_state=inp.initial_state[n:n + 1, h:h + 1],
            conv_state_in=inp.conv_state_in.view(256, 3, 96, 128, 3)[n:n + 1, :, h].reshape(1, 3 * 128, 3))
        ref = oracle_prefill(sub)
        check_out(to_np(out[4 * n:4 * n + 4, h:h + 1]), ref["out"], 1, TOL_OUT_BF16, True)
        assert per_head_rel(to_np(fin[n, h])[None], ref["final_state"][0], 0).max() <= TOL_STATE_BF16


def test_recurrent_fallback_kernel_for_unaligned_conv_state():
    """A conv state that is not 16-byte aligned (a view one element into its buffer) cannot be
    staged by the TMA engine: the plain recurrent kernel takes the call, with the same results."""
    inp = synth.make_prefill("layer_8k", seed=72, device=DEV, lengths=[4, 1, 8, 3], H=3, s0_std=0.02,
                             conv_state=True, rms_w="random")
    buf = torch.empty(inp.conv_state_in.numel() + 1, dtype=inp.conv_state_in.dtype, device=DEV)
    cs_in = buf[1:].view_as(inp.conv_state_in)
    cs_in.copy_(inp.conv_state_in)
    assert cs_in.data_ptr() % 16 != 0
    cso = torch.empty_like(inp.conv_state_in)
    out, fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens,
                               gate=inp.gate, rms_w=inp.rms_w, initial_state=inp.initial_state,
                               conv_state_in=cs_in, conv_state_out=cso, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle_prefill(inp)
    check_out(to_np(out), ref["out"], 1, TOL_OUT_BF16, bf16_out=False)
    assert per_head_rel(to_np(fin), ref["final_state"], 1).max() <= TOL_STATE_BF16
    np.testing.assert_array_equal(synth.to_f32_numpy(cso), ref["conv_state_out"].astype(np.float32))


def test_recurrent_batch_of_empty_sequences_hands_states_through():
    """Every sequence empty (T_total = 0): final states equal the initial ones and the conv
    states pass through unchanged."""
    inp = synth.make_prefill("layer_8k", seed=73, device=DEV, lengths=[0, 0, 0], H=2, s0_std=0.02,
                             conv_state=True)
    cso = torch.empty_like(inp.conv_state_in)
    out, fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens,
                               gate=inp.gate, rms_w=inp.rms_w, initial_state=inp.initial_state,
                               conv_state_in=inp.conv_state_in, conv_state_out=cso)
    torch.cuda.synchronize()
    assert out.shape[0] == 0
    assert torch.equal(fin, inp.initial_state)
    assert torch.equal(cso, inp.conv_state_in)
