"""GPU parity of the projections around the layer (kda_gemm) and of the layer with them.

C = epilogue(A W^T) on the tensor cores against the fp64 oracle.  The operands are
bf16 values, so every product is exact in fp32 and the only errors are the fp32
accumulation over K and the final rounding: an fp32 result is held to 1e-4 of the
largest |C| (a few units of fp32 roundoff times sqrt(K) at K = 12288), a bf16 result
to that plus its own rounding, 2^-8 |C| per element.  Shapes cover ragged tiles in M
and N, the single tile, K from one 64-block to the model's 12288, and every epilogue.

The projected layer (x -> g, beta, gate -> KDA prefill -> y -> y W_o) is compared with
the oracle's composition ("Kimi K3 / Architecture", KDA panel: projections to
alpha_t / beta_t with the log-decay bounded below by -5, the sigmoid gate, y_t W_o).
"""
import math

import numpy as np
import pytest
import torch

import kimi_delta_attention_16_gb300 as kda
from kimi_delta_attention_16_gb300 import synth
from kda_testlib import BF16_U, TOL_OUT_BF16, TOL_STATE_BF16, check_out, per_head_rel, to_np
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_GEMM = 1e-4
EPI_FN = {"none": lambda z: z, "decay": oracle.decay_from_logits, "sigmoid": oracle.strength_from_logits}


def _operands(M, N, K, seed, w_std=None):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    A = torch.randn(M, K, generator=gen, device=DEV).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=gen, device=DEV) * (w_std or 1.0 / math.sqrt(K))).to(torch.bfloat16)
    return A, W


def _check(C, ref, out_dtype):
    """max |C - ref| <= TOL_GEMM max |ref| (+ a bf16 result's own rounding per element)."""
    c = to_np(C)
    scale = max(np.abs(ref).max(), 1e-30)
    allow = TOL_GEMM * scale + (BF16_U * np.abs(ref) if out_dtype == torch.bfloat16 else 0.0)
    excess = np.abs(c - ref) - allow
    assert excess.max() <= 0, f"max excess {excess.max():.3e} (scale {scale:.3e})"


@pytest.mark.parametrize("epilogue", ["none", "decay", "sigmoid"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(1, 16, 64), (130, 96, 64), (256, 512, 128), (300, 1000, 192),
                                   (129, 257, 640)])
def test_gemm_parity(M, N, K, epilogue, out_dtype):
    A, W = _operands(M, N, K, seed=M + N + K)
    C = kda.kda_gemm(A, W, epilogue=epilogue, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = EPI_FN[epilogue](oracle.linear(to_np(A), to_np(W)))
    _check(C, ref, out_dtype)


def test_gemm_into_strided_rows_leaves_the_rest_untouched():
    """C as a column slice of a wider buffer (ldc > N): the columns outside stay as they were."""
    A, W = _operands(200, 136, 128, seed=5)
    buf = torch.full((200, 160), -7.0, dtype=torch.float32, device=DEV)
    view = buf[:, 8:144]
    kda.kda_gemm(A, W, epilogue="none", out=view)
    torch.cuda.synchronize()
    assert bool((buf[:, :8] == -7).all()) and bool((buf[:, 144:] == -7).all())
    _check(view, oracle.linear(to_np(A), to_np(W)), torch.float32)


@pytest.mark.parametrize("which", ["alpha", "gate", "w_out"])
def test_gemm_full_size_sampled_rows(which):
    """The model's projection shapes at T = 8192 (d_model 7168, 96 heads of 128): every
    column of 64 rows spread over M (each output row depends only on its own A row)."""
    M, dm, HD = 8192, 7168, 12288
    N, K, epi, odt = {"alpha": (HD, dm, "decay", torch.float32), "gate": (HD, dm, "none", torch.bfloat16),
                      "w_out": (dm, HD, "none", torch.bfloat16)}[which]
    A, W = _operands(M, N, K, seed=77)
    C = kda.kda_gemm(A, W, epilogue=epi, out_dtype=odt)
    torch.cuda.synchronize()
    rows = torch.linspace(0, M - 1, 64, device=DEV).long()
    ref = EPI_FN[epi](oracle.linear(to_np(A[rows]), to_np(W)))
    _check(C[rows], ref, odt)


def test_gemm_rejects_bad_shapes():
    A, W = _operands(64, 64, 96, seed=1)  # K = 96 is not a multiple of 64
    with pytest.raises(kda.KDAError) as e:
        kda.kda_gemm(A, W)
    assert e.value.status == 2


def _layer_weights(dm, H, D, d_out, seed):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)

    def w(n, k):
        return (torch.randn(n, k, generator=gen, device=DEV) / math.sqrt(k)).to(torch.bfloat16)
    return w(H * D, dm), w(H, dm), w(H * D, dm), w(d_out, H * D)


def test_projected_layer_end_to_end():
    """x -> (g, beta, gate) by kda_gemm -> kda_prefill -> y -> y W_o by kda_gemm, against
    the oracle's composition: g and beta (fp32) within 1e-5 of their range, the gate and y
    with their bf16 rounding, y and the final state at the layer's tolerances, and out."""
    dm, H, D, d_out = 256, 2, 128, 192
    inp = synth.make_prefill("layer_8k", seed=91, device=DEV, lengths=[200, 77], H=H, s0_std=0.02,
                             rms_w="random")
    T = inp.T
    gen = torch.Generator(device=DEV)
    gen.manual_seed(92)
    x = torch.randn(T, dm, generator=gen, device=DEV).to(torch.bfloat16)
    wa, wb, wg, wo = _layer_weights(dm, H, D, d_out, 93)
    g = kda.kda_gemm(x, wa, epilogue="decay").view(T, H, D)
    beta = kda.kda_gemm(x, wb, epilogue="sigmoid")
    gate = kda.kda_gemm(x, wg, epilogue="none").view(T, H, D)
    y, fin = kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, g, beta, inp.cu_seqlens, gate=gate,
                             rms_w=inp.rms_w, initial_state=inp.initial_state)
    out = kda.kda_gemm(y.view(T, H * D), wo, epilogue="none", out_dtype=torch.float32)
    torch.cuda.synchronize()
    f = synth.to_f32_numpy
    ref = oracle.projected_layer(f(x), f(wa), f(wb), f(wg), f(wo), f(inp.q), f(inp.k), f(inp.v),
                                 f(inp.conv_w), inp.cu_seqlens, rms_w=f(inp.rms_w),
                                 initial_state=f(inp.initial_state))
    assert np.abs(to_np(g) - ref["g"]).max() <= 5e-5
    assert np.abs(to_np(beta) - ref["beta"]).max() <= 1e-5
    # the gate is a bf16 rounding of the fp32-accumulated pre-activation: one bf16 step at most
    assert np.all(np.abs(to_np(gate) - ref["gate"]) <= 2 * BF16_U * np.abs(ref["gate"]) + 1e-6)
    check_out(to_np(y), ref["y"], 1, TOL_OUT_BF16, bf16_out=True)
    assert per_head_rel(to_np(fin), ref["final_state"], 1).max() <= TOL_STATE_BF16
    # out = bf16(y) W_o^T: y differs from the oracle's by the layer tolerance plus its rounding;
    # through W_o (entries ~ 1/sqrt(H D), random signs) that stays within a few 1e-3 of max|out|
    o = to_np(out)
    assert np.abs(o - ref["out"]).max() <= 1e-2 * np.abs(ref["out"]).max()
