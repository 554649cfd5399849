"""PyTorch-facing binding of libkda.so: argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; these functions
only turn tensors into pointers, sizes and the current stream, allocate
outputs and workspace with PyTorch (device memory is plumbing), and raise
``KDAError`` when the library returns a status.  There is no CPU fallback:
calling these without the built library or without a CUDA device fails.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import numpy as np
import torch

from . import _lib

_DT = {torch.bfloat16: _lib.KDA_BF16, torch.float32: _lib.KDA_FP32}
_TORCH = {_lib.KDA_BF16: torch.bfloat16, _lib.KDA_FP32: torch.float32}


class KDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _lib.load()
        msg = lib.kda_last_error().decode() or lib.kda_status_string(status).decode()
        super().__init__(f"{where}: status {status} ({lib.kda_status_string(status).decode()}): {msg}")
        self.status = status


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _same_cuda_device(**tensors) -> None:
    """Every given tensor must live on one CUDA device: the library dereferences
    these pointers only on the GPU, and a host pointer there would fault."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} is on {t.device}; every tensor must be on a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, other tensors on {dev}")
    if dev is not None and dev.index is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"tensors are on {dev} but the current device is cuda:{torch.cuda.current_device()}")


def _row_stride(t: torch.Tensor, H: int, D: int) -> int:
    """Row stride (elements) of a [T, H, D] view whose (H, D) block is dense."""
    if t.dim() != 3 or t.shape[1] != H or t.shape[2] != D:
        raise ValueError(f"expected [T, {H}, {D}], got {tuple(t.shape)}")
    if t.shape[0] > 0 and (t.stride(2) != 1 or t.stride(1) != D):
        raise ValueError("the (H, D) block of each token row must be contiguous")
    return t.stride(0) if t.shape[0] > 0 else H * D


def _cu_pair(cu_seqlens, device) -> Tuple[torch.Tensor, np.ndarray]:
    """(device int32 tensor, host int32 array) for cu_seqlens given as a tensor, a
    host sequence, or an already prepared (device tensor, host array) pair (no copy)."""
    if isinstance(cu_seqlens, tuple):
        dev, host = cu_seqlens
        return dev, np.ascontiguousarray(host, dtype=np.int32)
    if isinstance(cu_seqlens, torch.Tensor):
        host = cu_seqlens.detach().to("cpu", torch.int32).numpy()
        dev = cu_seqlens.to(device=device, dtype=torch.int32)
    else:
        host = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        dev = torch.from_numpy(host).to(device)
    return dev.contiguous(), np.ascontiguousarray(host)


def kda_short_conv(x: torch.Tensor, w: torch.Tensor, cu_seqlens, *, H: int, D: int,
                   conv_state_in: Optional[torch.Tensor] = None,
                   conv_state_out: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                   l2norm_qk: bool = True, eps_l2: float = 1e-6, d_status=None,
                   check_cu_on_host: bool = True, stream=None) -> torch.Tensor:
    """Causal width-4 short conv + SiLU (+ L2 on q, k) of [T, 3*H*D] rows (q | k | v)."""
    lib = _lib.load()
    io = _DT[x.dtype]
    T = x.shape[0]
    if y is None:
        y = torch.empty((T, 3 * H * D), dtype=x.dtype, device=x.device)
    cu_dev, cu_host = _cu_pair(cu_seqlens, x.device)
    _same_cuda_device(x=x, w=w, cu_seqlens=cu_dev, conv_state_in=conv_state_in,
                      conv_state_out=conv_state_out, y=y, d_status=d_status)
    N = cu_host.shape[0] - 1
    st = lib.kda_short_conv(_p(x), x.stride(0) if T else 3 * H * D, _p(w), _p(cu_dev),
                            cu_host.ctypes.data_as(ctypes.c_void_p) if check_cu_on_host else None,
                            N, T, H, D, _p(conv_state_in), _p(conv_state_out), _p(y),
                            y.stride(0) if T else 3 * H * D, int(l2norm_qk), float(eps_l2), io,
                            _p(d_status), _stream(stream))
    if st:
        raise KDAError(st, "kda_short_conv")
    return y


def _prefill_args(q, k, v, conv_w, g, beta, cu_dev, cu_host, *, chunk, gate, rms_w, eps_l2,
                  eps_rms, scale, initial_state, final_state, conv_state_in, conv_state_out, out,
                  workspace, d_status, flags, check_cu_on_host, segments=0):
    T, H, D = q.shape
    _same_cuda_device(q=q, k=k, v=v, conv_w=conv_w, g=g, beta=beta, cu_seqlens=cu_dev, gate=gate,
                      rms_w=rms_w, initial_state=initial_state, final_state=final_state,
                      conv_state_in=conv_state_in, conv_state_out=conv_state_out, out=out,
                      workspace=workspace, d_status=d_status)
    xs = _row_stride(q, H, D)
    if _row_stride(k, H, D) != xs or _row_stride(v, H, D) != xs:
        raise ValueError("q, k and v must share one row stride")
    a = _lib.PrefillArgs()
    a.N = cu_host.shape[0] - 1
    a.H, a.D, a.chunk, a.T_total = H, D, int(chunk), T
    a.io = _DT[q.dtype]
    a.out_dtype = _DT[out.dtype] if out is not None else a.io
    a.cu_seqlens = cu_dev.data_ptr()
    a.cu_seqlens_host = cu_host.ctypes.data if check_cu_on_host else None
    a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.qkv_row_stride = xs
    a.conv_w = conv_w.data_ptr()
    a.conv_state_in = conv_state_in.data_ptr() if conv_state_in is not None else None
    a.conv_state_out = conv_state_out.data_ptr() if conv_state_out is not None else None
    a.g, a.beta = g.data_ptr(), beta.data_ptr()
    a.gate = gate.data_ptr() if gate is not None else None
    a.rms_w = rms_w.data_ptr() if rms_w is not None else None
    a.eps_l2, a.eps_rms, a.scale = float(eps_l2), float(eps_rms), float(scale)
    a.initial_state = initial_state.data_ptr() if initial_state is not None else None
    a.final_state = final_state.data_ptr() if final_state is not None else None
    a.out = out.data_ptr() if out is not None else None
    a.workspace = workspace.data_ptr() if workspace is not None else None
    a.workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    a.d_status = d_status.data_ptr() if d_status is not None else None
    a.flags = int(flags)
    a.segments = int(segments)
    return a


def kda_prefill_workspace_size(T_total: int, H: int, D: int, *, N: int = 1, chunk: int = 64,
                               io=torch.bfloat16, flags: int = 0, segments: int = 0) -> int:
    """Workspace bytes kda_prefill needs for N packed sequences of T_total tokens
    in all (on the current device: the segment choice depends on its SM count)."""
    lib = _lib.load()
    a = _lib.PrefillArgs()
    a.N, a.H, a.D, a.chunk, a.T_total = N, H, D, chunk, T_total
    a.io = _DT[io]
    a.out_dtype = a.io
    a.flags = flags
    a.segments = segments
    n = ctypes.c_size_t(0)
    st = lib.kda_prefill_workspace_size(ctypes.byref(a), ctypes.byref(n))
    if st:
        raise KDAError(st, "kda_prefill_workspace_size")
    return int(n.value)


_PATH_NAMES = {_lib.KDA_PATH_SIMT: "simt", _lib.KDA_PATH_TENSOR_CORE: "tc",
               _lib.KDA_PATH_RECURRENT: "recurrent"}


def kda_prefill_plan(T_total: int, H: int, D: int, *, N: int = 1, chunk: int = 64,
                     io=torch.bfloat16, flags: int = 0, segments: int = 0, cu_seqlens=None):
    """(path, segments) kda_prefill takes on the current device: path is "tc" (tcgen05
    chunkwise), "simt" (fp32 chunkwise) or "recurrent" (token by token, for batches whose
    sequences all have at most 8 tokens; needs ``cu_seqlens`` to decide); segments per
    sequence (1 = none)."""
    lib = _lib.load()
    a = _lib.PrefillArgs()
    a.N, a.H, a.D, a.chunk, a.T_total = N, H, D, chunk, T_total
    a.io = _DT[io]
    a.out_dtype = a.io
    a.flags = flags
    a.segments = segments
    host = None
    if cu_seqlens is not None:
        host = np.ascontiguousarray(np.asarray(
            cu_seqlens.detach().cpu() if isinstance(cu_seqlens, torch.Tensor) else cu_seqlens,
            dtype=np.int32))
        a.N = host.shape[0] - 1
        a.cu_seqlens_host = host.ctypes.data
    path, seg = ctypes.c_int(0), ctypes.c_int(1)
    st = lib.kda_prefill_plan(ctypes.byref(a), ctypes.byref(path), ctypes.byref(seg))
    if st:
        raise KDAError(st, "kda_prefill_plan")
    return _PATH_NAMES[path.value], int(seg.value)


def kda_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, conv_w: torch.Tensor,
                g: torch.Tensor, beta: torch.Tensor, cu_seqlens, *, chunk: int = 64,
                gate: Optional[torch.Tensor] = None, rms_w: Optional[torch.Tensor] = None,
                eps_l2: float = 1e-6, eps_rms: float = 1e-6, scale: float = 1.0,
                initial_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
                final_state: Optional[torch.Tensor] = None,
                conv_state_in: Optional[torch.Tensor] = None,
                conv_state_out: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                out_dtype=None, workspace: Optional[torch.Tensor] = None, d_status=None,
                flags: int = 0, check_cu_on_host: bool = True, stream=None, segments: int = 0):
    """The whole KDA layer over packed sequences; returns (out, final_state or None).

    segments: tensor-core path only -- 0 lets the library cut long sequences into
    parallel segments when the batch has too few (sequence, head) units to fill the
    GPU, 1 disables that, 2..16 forces that many segments per sequence.

    q, k, v: [T, H, D] raw projections (bf16 or fp32; rows may be strided views of
    one fused buffer); conv_w [3, H*D, 4] fp32; g [T, H, D] fp32; beta [T, H] fp32;
    cu_seqlens [N+1] (tensor or sequence); gate [T, H, D] like q or None;
    initial_state / final_state [N, H, D, D] fp32; conv states [N, 3*H*D, 3] like q.
    """
    lib = _lib.load()
    T, H, D = q.shape
    cu_dev, cu_host = _cu_pair(cu_seqlens, q.device)
    N = cu_host.shape[0] - 1
    if out is None:
        out = torch.empty((T, H, D), dtype=out_dtype or q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, D, D), dtype=torch.float32, device=q.device)
    a = _prefill_args(q, k, v, conv_w, g, beta, cu_dev, cu_host, chunk=chunk, gate=gate,
                      rms_w=rms_w, eps_l2=eps_l2, eps_rms=eps_rms, scale=scale,
                      initial_state=initial_state, final_state=final_state,
                      conv_state_in=conv_state_in, conv_state_out=conv_state_out, out=out,
                      workspace=workspace, d_status=d_status, flags=flags,
                      check_cu_on_host=check_cu_on_host, segments=segments)
    if workspace is None:
        n = ctypes.c_size_t(0)
        st = lib.kda_prefill_workspace_size(ctypes.byref(a), ctypes.byref(n))
        if st:
            raise KDAError(st, "kda_prefill_workspace_size")
        if n.value:
            workspace = torch.empty(n.value, dtype=torch.uint8, device=q.device)
            a.workspace = workspace.data_ptr()
            a.workspace_bytes = n.value
    st = lib.kda_prefill(ctypes.byref(a), _stream(stream))
    if st:
        raise KDAError(st, "kda_prefill")
    return out, final_state


def kda_prefill_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, conv_w: torch.Tensor,
                        g: torch.Tensor, beta: torch.Tensor, cu_seqlens, *, chunk: int = 64,
                        gate: Optional[torch.Tensor] = None, rms_w: Optional[torch.Tensor] = None,
                        eps_l2: float = 1e-6, eps_rms: float = 1e-6, scale: float = 1.0,
                        initial_state: Optional[torch.Tensor] = None,
                        final_state: Optional[torch.Tensor] = None,
                        conv_state_in: Optional[torch.Tensor] = None,
                        conv_state_out: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None, d_status=None, stream=None):
    """kda_prefill for callers that cannot allocate device memory at call time.

    The caller passes every input and output buffer (``out`` and, if wanted,
    ``final_state`` are required); the library takes its scratch from a fixed
    array of ``NOALLOC_SCRATCH_BYTES`` per device and allocates nothing.
    Problems needing more scratch than that raise KDAError (status 3).

    ``cu_seqlens`` must already be a prepared pair (int32 CUDA tensor, int32 host
    array): turning a list or a CPU tensor into a device tensor here would allocate
    device memory, and reading a device tensor back would synchronise.
    """
    lib = _lib.load()
    if out is None:
        raise ValueError("kda_prefill_noalloc allocates nothing: pass `out`")
    if not (isinstance(cu_seqlens, tuple) and len(cu_seqlens) == 2
            and isinstance(cu_seqlens[0], torch.Tensor) and cu_seqlens[0].is_cuda
            and cu_seqlens[0].dtype == torch.int32 and cu_seqlens[0].is_contiguous()):
        raise ValueError("kda_prefill_noalloc needs cu_seqlens as a prepared "
                         "(int32 CUDA tensor, int32 host array) pair")
    cu_dev, cu_host = cu_seqlens
    cu_host = np.asarray(cu_host)
    if cu_host.dtype != np.int32 or not cu_host.flags.c_contiguous:
        raise ValueError("the host half of cu_seqlens must be a contiguous int32 array")
    a = _prefill_args(q, k, v, conv_w, g, beta, cu_dev, cu_host, chunk=chunk, gate=gate,
                      rms_w=rms_w, eps_l2=eps_l2, eps_rms=eps_rms, scale=scale,
                      initial_state=initial_state, final_state=final_state,
                      conv_state_in=conv_state_in, conv_state_out=conv_state_out, out=out,
                      workspace=None, d_status=d_status, flags=0, check_cu_on_host=True)
    st = lib.kda_prefill_noalloc(ctypes.byref(a), _stream(stream))
    if st:
        raise KDAError(st, "kda_prefill_noalloc")
    return out, final_state


def kda_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                    beta: torch.Tensor, conv_w: torch.Tensor, state: torch.Tensor,
                    conv_state: torch.Tensor, *, gate: Optional[torch.Tensor] = None,
                    rms_w: Optional[torch.Tensor] = None, eps_l2: float = 1e-6,
                    eps_rms: float = 1e-6, scale: float = 1.0, out: Optional[torch.Tensor] = None,
                    out_dtype=None, d_status=None, stream=None) -> torch.Tensor:
    """One decode step for N sequences; state [N,H,D,D] fp32 and conv_state
    [N,3*H*D,3] are updated in place.  q, k, v, gate: [N, H, D]; g [N,H,D]; beta [N,H]."""
    lib = _lib.load()
    N, H, D = q.shape
    if out is None:
        out = torch.empty((N, H, D), dtype=out_dtype or q.dtype, device=q.device)
    _same_cuda_device(q=q, k=k, v=v, g=g, beta=beta, conv_w=conv_w, state=state,
                      conv_state=conv_state, gate=gate, rms_w=rms_w, out=out, d_status=d_status)
    a = _lib.DecodeArgs()
    a.N, a.H, a.D = N, H, D
    a.io = _DT[q.dtype]
    a.out_dtype = _DT[out.dtype]
    xs = _row_stride(q, H, D)
    if _row_stride(k, H, D) != xs or _row_stride(v, H, D) != xs:
        raise ValueError("q, k and v must share one row stride")
    a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.qkv_row_stride = xs
    a.gate = gate.data_ptr() if gate is not None else None
    a.g, a.beta, a.conv_w = g.data_ptr(), beta.data_ptr(), conv_w.data_ptr()
    a.rms_w = rms_w.data_ptr() if rms_w is not None else None
    a.eps_l2, a.eps_rms, a.scale = float(eps_l2), float(eps_rms), float(scale)
    a.state, a.conv_state, a.out = state.data_ptr(), conv_state.data_ptr(), out.data_ptr()
    a.d_status = d_status.data_ptr() if d_status is not None else None
    st = lib.kda_decode_step(ctypes.byref(a), _stream(stream))
    if st:
        raise KDAError(st, "kda_decode_step")
    return out


_EPI = {"none": _lib.KDA_EPI_NONE, "decay": _lib.KDA_EPI_DECAY, "sigmoid": _lib.KDA_EPI_SIGMOID}


def kda_gemm(A: torch.Tensor, W: torch.Tensor, *, epilogue: str = "none",
             out: Optional[torch.Tensor] = None, out_dtype=None, d_status=None,
             stream=None) -> torch.Tensor:
    """C = epilogue(A @ W^T) on the tensor cores: A [M, K] bf16, W [N, K] bf16 (a linear
    layer's [out, in] weight), K a multiple of 64.  epilogue: "none" (C = A W^T), "decay"
    (C = -5 sigmoid(A W^T): the bounded log-decay g), "sigmoid" (the write strength beta).
    C is [M, N] in out_dtype (default bf16 for "none", fp32 otherwise); its rows may be a
    strided view."""
    lib = _lib.load()
    if A.dim() != 2 or W.dim() != 2 or A.shape[1] != W.shape[1]:
        raise ValueError(f"expected A [M, K] and W [N, K], got {tuple(A.shape)} and {tuple(W.shape)}")
    if A.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise ValueError("A and W must be bf16")
    if A.stride(1) != 1 or W.stride(1) != 1:
        raise ValueError("A and W rows must be contiguous")
    M, K = A.shape
    N = W.shape[0]
    if out is None:
        dt = out_dtype or (torch.bfloat16 if epilogue == "none" else torch.float32)
        out = torch.empty((M, N), dtype=dt, device=A.device)
    if out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError(f"out must be [{M}, {N}] with contiguous rows")
    _same_cuda_device(A=A, W=W, out=out, d_status=d_status)
    g = _lib.GemmArgs()
    g.M, g.N, g.K = M, N, K
    g.A, g.lda = A.data_ptr(), A.stride(0) if M else K
    g.W, g.ldw = W.data_ptr(), W.stride(0) if N else K
    g.C, g.ldc = out.data_ptr(), out.stride(0) if M else N
    g.c_dtype = _DT[out.dtype]
    g.epilogue = _EPI[epilogue]
    g.d_status = d_status.data_ptr() if d_status is not None else None
    st = lib.kda_gemm(ctypes.byref(g), _stream(stream))
    if st:
        raise KDAError(st, "kda_gemm")
    return out


def kda_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, conv_w: torch.Tensor,
                 g: torch.Tensor, beta: torch.Tensor, cu_seqlens, dy: torch.Tensor, *,
                 gate: Optional[torch.Tensor] = None, rms_w: Optional[torch.Tensor] = None,
                 eps_l2: float = 1e-6, eps_rms: float = 1e-6, scale: float = 1.0,
                 initial_state: Optional[torch.Tensor] = None,
                 conv_state_in: Optional[torch.Tensor] = None,
                 d_final_state: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 d_status=None, stream=None) -> dict:
    """Gradients of sum(dy * out) + sum(d_final_state * final_state) of one kda_prefill call
    (same inputs) with respect to its inputs.  Returns a dict of fp32 tensors: dq, dk, dv
    [T, H, D]; dconv_w [3, H*D, 4]; dg [T, H, D]; dbeta [T, H]; dgate (when gate is given);
    drms_w (when rms_w is given); dinitial_state [N, H, D, D]; dconv_state_in [N, 3*H*D, 3]
    (when conv_state_in is given).
    dy has the dtype of the forward's out.  D must be 128."""
    lib = _lib.load()
    T, H, D = q.shape
    cu_dev, cu_host = _cu_pair(cu_seqlens, q.device)
    N = cu_host.shape[0] - 1
    if dy.shape != (T, H, D) or not dy.is_contiguous():
        raise ValueError(f"dy must be a contiguous [{T}, {H}, {D}] tensor")
    if d_final_state is not None and (d_final_state.dtype != torch.float32 or not d_final_state.is_contiguous()):
        raise ValueError("d_final_state must be a contiguous fp32 tensor")
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    res = {"dq": torch.empty((T, H, D), **f32), "dk": torch.empty((T, H, D), **f32),
           "dv": torch.empty((T, H, D), **f32), "dconv_w": torch.empty((3, H * D, 4), **f32),
           "dg": torch.empty((T, H, D), **f32), "dbeta": torch.empty((T, H), **f32)}
    if gate is not None:
        res["dgate"] = torch.empty((T, H, D), **f32)
    if rms_w is not None:
        res["drms_w"] = torch.empty((D,), **f32)
    res["dinitial_state"] = torch.empty((N, H, D, D), **f32)
    if conv_state_in is not None:
        res["dconv_state_in"] = torch.empty((N, 3 * H * D, 3), **f32)
    _same_cuda_device(dy=dy, d_final_state=d_final_state, **res)
    b = _lib.BackwardArgs()
    b.fwd = _prefill_args(q, k, v, conv_w, g, beta, cu_dev, cu_host, chunk=64, gate=gate,
                          rms_w=rms_w, eps_l2=eps_l2, eps_rms=eps_rms, scale=scale,
                          initial_state=initial_state, final_state=None,
                          conv_state_in=conv_state_in, conv_state_out=None, out=None,
                          workspace=workspace, d_status=d_status, flags=0, check_cu_on_host=True)
    b.fwd.out_dtype = _DT[dy.dtype]
    b.dy = dy.data_ptr()
    b.d_final_state = _p(d_final_state)
    for name in ("dq", "dk", "dv", "dconv_w", "dg", "dbeta", "dgate", "drms_w", "dinitial_state",
                 "dconv_state_in"):
        setattr(b, name, res[name].data_ptr() if name in res else None)
    if workspace is None:
        n = ctypes.c_size_t(0)
        st = lib.kda_backward_workspace_size(ctypes.byref(b), ctypes.byref(n))
        if st:
            raise KDAError(st, "kda_backward_workspace_size")
        if n.value:
            workspace = torch.empty(n.value, dtype=torch.uint8, device=dev)
            b.fwd.workspace = workspace.data_ptr()
            b.fwd.workspace_bytes = n.value
    st = lib.kda_backward(ctypes.byref(b), _stream(stream))
    if st:
        raise KDAError(st, "kda_backward")
    return res


def kda_backward_workspace_size(cu_seqlens, H: int, D: int = 128) -> int:
    """Workspace bytes kda_backward needs for these sequences and heads."""
    lib = _lib.load()
    host = np.ascontiguousarray(np.asarray(
        cu_seqlens.detach().cpu() if isinstance(cu_seqlens, torch.Tensor) else cu_seqlens, dtype=np.int32))
    b = _lib.BackwardArgs()
    b.fwd.N, b.fwd.H, b.fwd.D, b.fwd.T_total = host.shape[0] - 1, H, D, int(host[-1]) if host.size else 0
    b.fwd.cu_seqlens_host = host.ctypes.data
    n = ctypes.c_size_t(0)
    st = lib.kda_backward_workspace_size(ctypes.byref(b), ctypes.byref(n))
    if st:
        raise KDAError(st, "kda_backward_workspace_size")
    return int(n.value)


class _KDALayer(torch.autograd.Function):
    """kda_prefill forward, kda_backward backward (marshalling only; both run in libkda)."""

    @staticmethod
    def forward(ctx, q, k, v, conv_w, g, beta, gate, rms_w, initial_state, conv_state_in, cu_pair,
                eps_l2, eps_rms, scale):
        out, fin = kda_prefill(q, k, v, conv_w, g, beta, cu_pair, gate=gate, rms_w=rms_w, eps_l2=eps_l2,
                               eps_rms=eps_rms, scale=scale, initial_state=initial_state,
                               conv_state_in=conv_state_in)
        ctx.save_for_backward(q, k, v, conv_w, g, beta, gate, rms_w, initial_state, conv_state_in)
        ctx.cu_pair = cu_pair
        ctx.hp = (eps_l2, eps_rms, scale)
        return out, fin

    @staticmethod
    def backward(ctx, dout, dfin):
        q, k, v, conv_w, g, beta, gate, rms_w, initial_state, conv_state_in = ctx.saved_tensors
        eps_l2, eps_rms, scale = ctx.hp
        if dout is None:
            dout = torch.zeros(q.shape, dtype=q.dtype, device=q.device)
        gr = kda_backward(q, k, v, conv_w, g, beta, ctx.cu_pair, dout.contiguous(), gate=gate, rms_w=rms_w,
                          eps_l2=eps_l2, eps_rms=eps_rms, scale=scale, initial_state=initial_state,
                          conv_state_in=conv_state_in,
                          d_final_state=None if dfin is None else dfin.contiguous())

        def cast(name, like):
            if like is None or not ctx.needs_input_grad[names.index(name)]:
                return None
            return gr[name].to(like.dtype).view(like.shape)

        names = ["dq", "dk", "dv", "dconv_w", "dg", "dbeta", "dgate", "drms_w", "dinitial_state",
                 "dconv_state_in"]
        ins = [q, k, v, conv_w, g, beta, gate, rms_w, initial_state, conv_state_in]
        return (*(cast(n, t) for n, t in zip(names, ins)), None, None, None, None)


def kda_layer(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, conv_w: torch.Tensor, g: torch.Tensor,
              beta: torch.Tensor, cu_seqlens, *, gate: Optional[torch.Tensor] = None,
              rms_w: Optional[torch.Tensor] = None, eps_l2: float = 1e-6, eps_rms: float = 1e-6,
              scale: float = 1.0, initial_state: Optional[torch.Tensor] = None,
              conv_state_in: Optional[torch.Tensor] = None):
    """The KDA layer as a differentiable PyTorch operation: returns (out, final_state) from
    kda_prefill, and on backward runs kda_backward (D = 128) for every input that requires a
    gradient (q, k, v, conv_w, g, beta, gate, rms_w, initial_state, conv_state_in).  The
    gradients are those of the exact layer in fp32, cast to each input's dtype."""
    cu_pair = _cu_pair(cu_seqlens, q.device)
    return _KDALayer.apply(q, k, v, conv_w, g, beta, gate, rms_w, initial_state, conv_state_in, cu_pair,
                           float(eps_l2), float(eps_rms), float(scale))
