"""GPU parity of the layer's backward pass (kda_backward) against the fp64 oracle's gradients.

The oracle's backward is pinned to central differences of the fp64 forward (see the oracle pin
tests); here every gradient the library returns is compared with it on the same seeded inputs.

Tolerance.  The library recomputes the forward and runs its adjoint in fp32 (IEEE exp for the
decays and the gate sigmoid, the fast exponential and reciprocal for the recomputed SiLU and its
derivative, a few ulp; bf16 inputs are exact in fp32; the chunk products on the tensor cores as
three TF32 terms of hi/lo splits, about 2^-21 relative per product), so the errors are fp32-level
roundoff carried through the recurrence.  Each step is a contraction of the state and of its adjoint (0 < e^g <= 1,
|k| = 1 after the L2 norm, 0 <= beta <= 1), so roundoff does not grow from step to step; it
accumulates over the D = 128 terms of each dot product and over the tokens of a sequence.
With the fp32 unit roundoff 6e-8 and a few hundred tokens that is ~1e-6 of the tensor's scale
typically, and the bound is set well above that: every gradient tensor is held to
max|gpu - ref| <= TOL_BWD * max|ref|, TOL_BWD = 1e-4.  A wrong term of the adjoint (a dropped
product, a transposed operand, a wrong sign) moves the result by O(1) of max|ref|.
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_16_gb300 as kda
from kimi_delta_attention_16_gb300 import synth
from kda_testlib import head_slice_inputs, to_np
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_BWD = 1e-4


def _draw(shape, std, seed, dtype=torch.float32):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    return (torch.randn(shape, generator=gen, device=DEV) * std).to(dtype)


def _gpu_backward(inp, dy, dsf, *, use_gate=True, use_rms=True, use_s0=True, use_cs=True,
                  scale=1.0, eps_l2=1e-6, eps_rms=1e-6):
    res = kda.kda_backward(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens, dy,
                           gate=inp.gate if use_gate else None, rms_w=inp.rms_w if use_rms else None,
                           eps_l2=eps_l2, eps_rms=eps_rms, scale=scale,
                           initial_state=inp.initial_state if use_s0 else None,
                           conv_state_in=inp.conv_state_in if use_cs else None, d_final_state=dsf)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in res.items()}


def _oracle_backward(inp, dy, dsf, heads=None, *, use_gate=True, use_rms=True, use_s0=True,
                     use_cs=True, scale=1.0, eps_l2=1e-6, eps_rms=1e-6):
    heads = list(range(inp.H)) if heads is None else list(heads)
    a = head_slice_inputs(inp, heads)
    hs = torch.as_tensor(heads, dtype=torch.long, device=DEV)
    dyh = synth.to_f32_numpy(torch.index_select(dy, 1, hs))
    dsh = None if dsf is None else synth.to_f32_numpy(torch.index_select(dsf, 1, hs))
    return oracle.backward(a["q"], a["k"], a["v"], a["conv_w"], a["cu_seqlens"], a["g"], a["beta"], dyh,
                           gate=a["gate"] if use_gate else None, rms_w=a["rms_w"] if use_rms else None,
                           eps_l2=eps_l2, eps_rms=eps_rms, scale=scale,
                           initial_state=a["initial_state"] if use_s0 else None,
                           conv_state_in=a["conv_state_in"] if use_cs else None, d_final_state=dsh)


def _check(gpu, ref, names=None):
    names = names or sorted(ref)
    assert set(gpu) >= set(names), f"missing gradients {set(names) - set(gpu)}"
    worst = {}
    for n in names:
        g, r = np.asarray(gpu[n], np.float64), np.asarray(ref[n], np.float64)
        assert g.shape == r.shape, f"{n}: shape {g.shape} vs {r.shape}"
        assert np.isfinite(g).all(), f"{n}: non-finite values"
        scale = max(np.abs(r).max(), 1e-30)
        worst[n] = np.abs(g - r).max() / scale
    bad = {n: e for n, e in worst.items() if e > TOL_BWD}
    assert not bad, f"relative errors above {TOL_BWD:g}: {bad} (all: {worst})"
    return worst


def _case(io, lengths, H=2, seed=0, g_range=(-5.0, 0.0), beta_one=False, out_dt=None):
    inp = synth.make_prefill("layer_8k", seed=seed, device=DEV, lengths=lengths, H=H, io=io,
                             s0_std=0.05, conv_state=True, rms_w="random", g_range=g_range)
    if beta_one:
        inp.beta.fill_(1.0)
    T = inp.q.shape[0]
    out_dt = out_dt or (torch.bfloat16 if io == "bf16" else torch.float32)
    dy = _draw((T, H, 128), 1.0, seed + 1, out_dt)
    dsf = _draw((len(lengths), H, 128, 128), 0.05, seed + 2)
    return inp, dy, dsf


@pytest.mark.parametrize("io", ["bf16", "fp32"])
def test_backward_parity_varlen_all_inputs(io):
    """Ragged batch (64-token checkpoint segments and 8-token staging blocks cut mid-sequence, a
    1-token and an empty sequence), every optional input given: gate, RMSNorm weight, initial
    state, conv state, dS_fin."""
    inp, dy, dsf = _case(io, [70, 1, 0, 33, 130], seed=11)
    _check(_gpu_backward(inp, dy, dsf), _oracle_backward(inp, dy, dsf))


@pytest.mark.parametrize("io,pad", [("bf16", 0), ("bf16", 8), ("fp32", 4)])
def test_backward_parity_fused_qkv_rows(io, pad):
    """q, k and v as views of one [T, 3 H D + pad] buffer (a fused projection, padded rows within
    the ABI's row rules: 16-byte multiples), read by the recompute's staged row copies; against the
    oracle."""
    inp, dy, dsf = _case(io, [70, 1, 33], seed=41)
    T, H, D = inp.q.shape
    HD = H * D
    buf = torch.zeros((T, 3 * HD + pad), dtype=inp.q.dtype, device=DEV)
    views = []
    for i, x in enumerate((inp.q, inp.k, inp.v)):
        buf[:, i * HD:(i + 1) * HD] = x.reshape(T, HD)
        views.append(buf[:, i * HD:(i + 1) * HD].unflatten(1, (H, D)))
    res = kda.kda_backward(views[0], views[1], views[2], inp.conv_w, inp.g, inp.beta, inp.cu_seqlens, dy,
                           gate=inp.gate, rms_w=inp.rms_w, initial_state=inp.initial_state,
                           conv_state_in=inp.conv_state_in, d_final_state=dsf)
    torch.cuda.synchronize()
    _check({k: to_np(v) for k, v in res.items()}, _oracle_backward(inp, dy, dsf))


def test_backward_parity_chunk_and_segment_boundaries():
    """Lengths on either side of every 16-token chunk and 64-token checkpoint segment boundary in
    one batch: partial last chunks, segments of one to four chunks, a segment of a single token."""
    lengths = [15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 193]
    inp, dy, dsf = _case("bf16", lengths, seed=61)
    _check(_gpu_backward(inp, dy, dsf), _oracle_backward(inp, dy, dsf))


def test_backward_parity_without_optional_inputs():
    """No gate, no RMSNorm weight, zero initial and conv states, no dS_fin: the returned
    dinitial_state is still the gradient at the (zero) start state."""
    inp, dy, _ = _case("bf16", [45, 96], seed=21)
    kw = dict(use_gate=False, use_rms=False, use_s0=False, use_cs=False)
    gpu = _gpu_backward(inp, dy, None, **kw)
    assert "dgate" not in gpu and "drms_w" not in gpu and "dconv_state_in" not in gpu
    _check(gpu, _oracle_backward(inp, dy, None, **kw))


def test_backward_parity_fp32_dy_for_bf16_inputs_and_scale():
    """dy in fp32 (a bf16-input layer whose out was fp32) and a readout scale of 1/sqrt(D)."""
    inp, dy, dsf = _case("bf16", [64, 17], seed=31, out_dt=torch.float32)
    s = 128 ** -0.5
    _check(_gpu_backward(inp, dy, dsf, scale=s), _oracle_backward(inp, dy, dsf, scale=s))


@pytest.mark.parametrize("g_range,beta_one", [((0.0, 0.0), True), ((-5.0, -5.0), False),
                                              ((-0.05, 0.0), True)])
def test_backward_parity_decay_extremes(g_range, beta_one):
    """The ends of the decay range (no forgetting, strongest forgetting), and full-strength
    writes with almost no forgetting (the state carries every token to the end)."""
    inp, dy, dsf = _case("bf16", [100, 29], seed=41, g_range=g_range, beta_one=beta_one)
    _check(_gpu_backward(inp, dy, dsf), _oracle_backward(inp, dy, dsf))


def test_backward_parity_long_sequence():
    """One sequence of 1000 tokens (16 checkpoint segments, the last one partial) and one head."""
    inp, dy, dsf = _case("bf16", [1000], H=1, seed=51, g_range=(-0.5, 0.0))
    _check(_gpu_backward(inp, dy, dsf), _oracle_backward(inp, dy, dsf))


def test_backward_all_empty_sequences():
    """T = 0: only the state gradients are defined (dS0 = dS_fin, dconv_state_in = 0)."""
    inp, dy, dsf = _case("bf16", [0, 0], seed=61)
    gpu = _gpu_backward(inp, dy, dsf)
    assert np.array_equal(gpu["dinitial_state"], to_np(dsf))
    assert not gpu["dconv_state_in"].any() and not gpu["dconv_w"].any()


def test_backward_full_size_sampled_heads():
    """The 8192-token, 96-head workload with every input: all heads on the GPU, three of them
    (first, middle, last) against the oracle.  drms_w sums over every head, so it is checked
    at the small sizes above only."""
    H = 96
    inp = synth.make_prefill("layer_8k", seed=71, device=DEV, s0_std=0.05, conv_state=True,
                             rms_w="random", g_range=(-1.0, 0.0))
    T, N = inp.q.shape[0], inp.N
    dy = _draw((T, H, 128), 1.0, 72, torch.bfloat16)
    dsf = _draw((N, H, 128, 128), 0.05, 73)
    gpu = _gpu_backward(inp, dy, dsf)
    heads = [0, 47, 95]
    ref = _oracle_backward(inp, dy, dsf, heads)
    sel = {"dq": 1, "dk": 1, "dv": 1, "dg": 1, "dbeta": 1, "dgate": 1, "dinitial_state": 1}
    got = {n: np.take(gpu[n], heads, axis=ax) for n, ax in sel.items()}
    # dconv_w [3, H*D, 4] and dconv_state_in [N, 3*H*D, 3]: the channels of the sampled heads
    ch = np.concatenate([np.arange(h * 128, (h + 1) * 128) for h in heads])
    got["dconv_w"] = gpu["dconv_w"][:, ch, :]
    cs = gpu["dconv_state_in"].reshape(N, 3, H * 128, 3)[:, :, ch, :]
    got["dconv_state_in"] = cs.reshape(N, 3 * len(ch), 3)
    _check(got, ref, names=sorted(sel) + ["dconv_w", "dconv_state_in"])


def test_backward_rejects_unsupported_shapes():
    inp = synth.make_prefill("tiny_fp32", seed=1, device=DEV)  # D < 128
    dy = torch.zeros_like(inp.q)
    with pytest.raises(kda.KDAError) as e:
        kda.kda_backward(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens, dy)
    assert e.value.status == 2


def test_backward_reports_a_device_cu_seqlens_that_disagrees_with_the_host_copy():
    """The checkpoint layout is planned from the host copy of cu_seqlens; a device copy with other
    sequence lengths (same total) must be reported through d_status (KDA_ERR_DEVICE_ARG), with no
    access outside the planned checkpoint slots, and the next correct call on the same context
    must still match the oracle."""
    inp, dy, dsf = _case("bf16", [64, 64], seed=81)
    host = np.array([0, 64, 128], np.int32)
    bad_dev = torch.tensor([0, 100, 128], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_backward(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, (bad_dev, host), dy, gate=inp.gate,
                     rms_w=inp.rms_w, initial_state=inp.initial_state, conv_state_in=inp.conv_state_in,
                     d_final_state=dsf, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6  # KDA_ERR_DEVICE_ARG
    _check(_gpu_backward(inp, dy, dsf), _oracle_backward(inp, dy, dsf))


def test_autograd_layer_matches_the_oracle_gradients():
    """kda_layer (kda_prefill forward, kda_backward backward) under torch.autograd: every input's
    .grad equals the oracle's gradient of loss = sum(dy . out) + sum(dS_fin . final_state).
    fp32 inputs, so the gradients are not rounded to a narrower dtype."""
    inp, dy, dsf = _case("fp32", [50, 21], seed=91)
    leaves = {name: getattr(inp, name).clone().requires_grad_(True)
              for name in ("q", "k", "v", "conv_w", "g", "beta", "gate", "rms_w", "initial_state", "conv_state_in")}
    out, fin = kda.kda_layer(leaves["q"], leaves["k"], leaves["v"], leaves["conv_w"], leaves["g"], leaves["beta"],
                             inp.cu_seqlens, gate=leaves["gate"], rms_w=leaves["rms_w"],
                             initial_state=leaves["initial_state"], conv_state_in=leaves["conv_state_in"])
    loss = (out * dy).sum() + (fin * dsf).sum()
    loss.backward()
    torch.cuda.synchronize()
    ref = _oracle_backward(inp, dy, dsf)
    got = {"d" + n: to_np(t.grad).reshape(ref["d" + n].shape) for n, t in leaves.items()}
    _check(got, ref)


def test_autograd_layer_bf16_gradients_have_the_input_dtypes():
    """bf16 inputs: each .grad is the fp32 gradient rounded to bf16 (within the bf16 unit roundoff
    of the oracle's value, plus the fp32 tolerance), and inputs that do not require a gradient get
    none."""
    inp, dy, dsf = _case("bf16", [40], seed=93)
    q = inp.q.clone().requires_grad_(True)
    g = inp.g.clone().requires_grad_(True)
    out, fin = kda.kda_layer(q, inp.k, inp.v, inp.conv_w, g, inp.beta, inp.cu_seqlens, gate=inp.gate,
                             rms_w=inp.rms_w, initial_state=inp.initial_state, conv_state_in=inp.conv_state_in)
    ((out.float() * dy.float()).sum() + (fin * dsf).sum()).backward()
    torch.cuda.synchronize()
    assert q.grad.dtype == torch.bfloat16 and g.grad.dtype == torch.float32
    ref = _oracle_backward(inp, dy, dsf)
    dq, rq = to_np(q.grad), ref["dq"]
    assert np.all(np.abs(dq - rq) <= 2.0 ** -8 * np.abs(rq) + TOL_BWD * np.abs(rq).max())
    _check({"dg": to_np(g.grad)}, ref, names=["dg"])
