"""Seeded synthetic inputs for the KDA layer.

This module is shared by the tests, the benchmark and the oracle harness.  It
holds none of the layer's arithmetic: only shapes, value distributions, the
varlen length mix and dtype casts (bf16 by round-to-nearest-even).

Workloads (shapes from "Kimi K3 / Architecture", panels "Kimi Delta
Attention . one head at token t" -- 96 heads of 128 -- and "KDA short
convolution" -- width-4 taps, rolling state of 3 values per channel):

  tiny_fp32     N=1, T=64, H=2, D=16, chunk 16, fp32 I/O
  layer_8k      N=1, T=8192, H=96, D=128, chunk 64, bf16 I/O
  varlen_16     16 sequences, lengths round(exp(U[ln 512, ln 16384])), H=96,
                D=128, bf16 I/O, initial states ~N(0, 0.02^2)
  long_1m       N=1, T=1,048,576, H=24, D=128, chunk 64, bf16 I/O
  decode_256    256 sequences x 1 token per step, H=96, D=128, states
                ~N(0, 0.02^2), rolling conv state ~N(0,1) bf16
  verify_256x4  256 sequences x 4 new tokens (a multi-token decode or
                speculative-verification step), H=96, D=128, states
                ~N(0, 0.02^2), rolling conv states ~N(0,1) bf16

Value laws (all workloads): raw q, k, v ~ N(0,1); conv taps ~ N(0, 0.5^2);
log-decay g ~ U[-5, 0] per (token, head, key channel); beta ~ U[0, 1) per
(token, head); gate pre-activations ~ N(0,1) (the law of x.W_g for x ~ N(0,1)
at d_model = 7168 with W_g ~ N(0, 1/7168)); RMSNorm weight = 1.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

WORKLOADS = {
    "tiny_fp32": dict(N=1, T=64, H=2, D=16, chunk=16, io="fp32", s0_std=0.0),
    "layer_8k": dict(N=1, T=8192, H=96, D=128, chunk=64, io="bf16", s0_std=0.0),
    "varlen_16": dict(N=16, T=None, H=96, D=128, chunk=64, io="bf16", s0_std=0.02,
                      len_lo=512, len_hi=16384),
    "long_1m": dict(N=1, T=1_048_576, H=24, D=128, chunk=64, io="bf16", s0_std=0.0),
    "decode_256": dict(N=256, H=96, D=128, io="bf16", s0_std=0.02, steps=1000, ring=32),
    "verify_256x4": dict(N=256, T=1024, H=96, D=128, chunk=64, io="bf16", s0_std=0.02,
                         conv_state=True),
}

_TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """n lengths round(exp(U[ln lo, ln hi])), seeded."""
    rng = np.random.default_rng(seed)
    return [int(round(math.exp(u))) for u in rng.uniform(math.log(lo), math.log(hi), size=n)]


def cu_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, np.int64))
    return cu


@dataclasses.dataclass
class PrefillInputs:
    """One prefill batch.  Tensors live on ``device``; cu_seqlens also on host."""
    N: int
    H: int
    D: int
    chunk: int
    io: str
    cu_seqlens: np.ndarray          # [N+1] int32, host
    q: torch.Tensor                 # [T, H, D] io dtype (raw, before the conv)
    k: torch.Tensor
    v: torch.Tensor
    conv_w: torch.Tensor            # [3, H*D, 4] fp32
    g: torch.Tensor                 # [T, H, D] fp32 log-decay
    beta: torch.Tensor              # [T, H] fp32
    gate: Optional[torch.Tensor]    # [T, H, D] io dtype or None
    rms_w: Optional[torch.Tensor]   # [D] fp32 or None
    initial_state: Optional[torch.Tensor]  # [N, H, D, D] fp32 or None
    conv_state_in: Optional[torch.Tensor]  # [N, 3*H*D, 3] io dtype or None

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])


def _gen(seed: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return gen


def _normal(shape, std, gen, device, dtype):
    """N(0, std^2) drawn in fp32, then cast to ``dtype`` (RNE for bf16)."""
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def _uniform(shape, lo, hi, gen, device):
    x = torch.rand(*shape, generator=gen, device=device, dtype=torch.float32)
    return x.mul_(hi - lo).add_(lo)


def make_prefill(name: str = "tiny_fp32", seed: int = 0, device="cpu", *, N=None, T=None,
                 lengths=None, H=None, D=None, chunk=None, io=None, gate=True, rms_w="ones",
                 s0_std=None, conv_state=None, g_range=(-5.0, 0.0)) -> PrefillInputs:
    """Seeded prefill inputs for a named workload, with optional overrides.

    ``lengths`` (a list) overrides N/T with an explicit varlen mix.
    ``g_range``: the log-decay law U[lo, hi]; a range near 0 (slow forgetting)
    makes the state carry information across many chunks.
    ``rms_w``: "ones", "random" (1 + 0.1 N(0,1)) or None (no RMSNorm weight).
    ``conv_state``: also draw a rolling conv state ~N(0,1) per sequence.
    """
    w = dict(WORKLOADS[name])
    H = H or w["H"]
    D = D or w["D"]
    chunk = chunk or w.get("chunk", 64)
    io = io or w["io"]
    s0_std = w.get("s0_std", 0.0) if s0_std is None else s0_std
    conv_state = w.get("conv_state", False) if conv_state is None else conv_state
    if lengths is None:
        if N is None and T is None and w.get("T") is None:
            lengths = varlen_lengths(w["N"], w["len_lo"], w["len_hi"], seed)
        else:
            N = N or w["N"]
            T = T if T is not None else w["T"]
            base, rem = divmod(T, N)
            lengths = [base + (1 if i < rem else 0) for i in range(N)]
    cu = cu_from_lengths(lengths)
    N = len(lengths)
    Tt = int(cu[-1])
    dt = _TORCH_DT[io]
    gen = _gen(seed, device)
    q = _normal((Tt, H, D), 1.0, gen, device, dt)
    k = _normal((Tt, H, D), 1.0, gen, device, dt)
    v = _normal((Tt, H, D), 1.0, gen, device, dt)
    conv_w = _normal((3, H * D, 4), 0.5, gen, device, torch.float32)
    g = _uniform((Tt, H, D), float(g_range[0]), float(g_range[1]), gen, device)
    beta = _uniform((Tt, H), 0.0, 1.0, gen, device)
    gt = _normal((Tt, H, D), 1.0, gen, device, dt) if gate else None
    if rms_w == "ones":
        rw = torch.ones(D, device=device, dtype=torch.float32)
    elif rms_w == "random":
        rw = 1.0 + _normal((D,), 0.1, gen, device, torch.float32)
    else:
        rw = None
    s0 = _normal((N, H, D, D), s0_std, gen, device, torch.float32) if s0_std else None
    cs = _normal((N, 3 * H * D, 3), 1.0, gen, device, dt) if conv_state else None
    return PrefillInputs(N=N, H=H, D=D, chunk=chunk, io=io, cu_seqlens=cu, q=q, k=k, v=v,
                         conv_w=conv_w, g=g, beta=beta, gate=gt, rms_w=rw, initial_state=s0,
                         conv_state_in=cs)


@dataclasses.dataclass
class DecodeInputs:
    """Batched decode: a ring of per-step inputs plus the two rolling states."""
    N: int
    H: int
    D: int
    io: str
    conv_w: torch.Tensor        # [3, H*D, 4] fp32
    rms_w: Optional[torch.Tensor]
    state: torch.Tensor         # [N, H, D, D] fp32 (updated in place by decode)
    conv_state: torch.Tensor    # [N, 3*H*D, 3] io dtype (rolled in place)
    q: torch.Tensor             # [R, N, H, D] io dtype, R = ring size
    k: torch.Tensor
    v: torch.Tensor
    gate: torch.Tensor
    g: torch.Tensor             # [R, N, H, D] fp32
    beta: torch.Tensor          # [R, N, H] fp32

    @property
    def ring(self) -> int:
        return int(self.q.shape[0])


def make_decode(seed: int = 0, device="cpu", *, N=None, H=None, D=None, ring=None,
                io=None, rms_w="ones") -> DecodeInputs:
    """Seeded decode inputs; step i uses ring entry i mod ring."""
    w = WORKLOADS["decode_256"]
    N = N or w["N"]
    H = H or w["H"]
    D = D or w["D"]
    R = ring or w["ring"]
    io = io or w["io"]
    dt = _TORCH_DT[io]
    gen = _gen(seed, device)
    conv_w = _normal((3, H * D, 4), 0.5, gen, device, torch.float32)
    state = _normal((N, H, D, D), w["s0_std"], gen, device, torch.float32)
    cs = _normal((N, 3 * H * D, 3), 1.0, gen, device, dt)
    q = _normal((R, N, H, D), 1.0, gen, device, dt)
    k = _normal((R, N, H, D), 1.0, gen, device, dt)
    v = _normal((R, N, H, D), 1.0, gen, device, dt)
    gt = _normal((R, N, H, D), 1.0, gen, device, dt)
    g = _uniform((R, N, H, D), -5.0, 0.0, gen, device)
    beta = _uniform((R, N, H), 0.0, 1.0, gen, device)
    if rms_w == "ones":
        rw = torch.ones(D, device=device, dtype=torch.float32)
    elif rms_w == "random":
        rw = 1.0 + _normal((D,), 0.1, gen, device, torch.float32)
    else:
        rw = None
    return DecodeInputs(N=N, H=H, D=D, io=io, conv_w=conv_w, rms_w=rw, state=state,
                        conv_state=cs, q=q, k=k, v=v, gate=gt, g=g, beta=beta)


def to_f32_numpy(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Exact fp32 host copy of a bf16/fp32 tensor (bf16 -> fp32 is exact)."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float32).contiguous().numpy()
