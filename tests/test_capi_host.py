"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments with a status before anything is launched.

No GPU is needed: every call below fails host validation, so no CUDA call is
made.  The pointers are never dereferenced on the host.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from kimi_delta_attention_16_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x7f0000000000  # a 256-byte aligned address that is never dereferenced on the host


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    lib = _lib.load()
    names = _declared_functions()
    assert set(names) == set(_lib.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version():
    lib = _lib.load()
    assert lib.kda_status_string(0) == b"ok"
    assert b"workspace" in lib.kda_status_string(_lib.KDA_ERR_WORKSPACE)
    assert lib.kda_version() >= _lib.ABI_VERSION


def test_header_constants_match_the_binding():
    """Every #define and enum value of kda.h that the binding mirrors has the same value."""
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    defines = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(KDA_[A-Z_0-9]+)\s+(\d+)", src)}
    enums = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(KDA_[A-Z_0-9]+)\s*=\s*(\d+)", src)}
    consts = {**enums, **defines}
    mirrored = [n for n in dir(_lib) if n.startswith("KDA_") and isinstance(getattr(_lib, n), int)]
    assert "KDA_FLAG_TEST_DROP_STAGING" in mirrored
    for n in mirrored:
        if n in consts:
            assert getattr(_lib, n) == consts[n], n


def _args(**kw):
    a = _lib.PrefillArgs()
    a.N, a.H, a.D, a.chunk, a.T_total = 1, 2, 128, 64, 64
    a.io = a.out_dtype = _lib.KDA_BF16
    cu = np.array([0, 64], np.int32)
    a.cu_seqlens = FAKE
    a.cu_seqlens_host = cu.ctypes.data
    a.q, a.k, a.v = FAKE, FAKE + 0x100000, FAKE + 0x200000
    a.qkv_row_stride = 0
    a.conv_w = FAKE + 0x300000
    a.g, a.beta, a.out = FAKE + 0x400000, FAKE + 0x500000, FAKE + 0x600000
    a.eps_l2 = a.eps_rms = 1e-6
    a.scale = 1.0
    a.workspace = FAKE + 0x10000000
    a.workspace_bytes = 1 << 40
    for k, v in kw.items():
        setattr(a, k, v)
    return a, cu


def _prefill(a):
    lib = _lib.load()
    return lib.kda_prefill(ctypes.byref(a), None)


@pytest.mark.parametrize("field,value,code", [
    ("D", 48, _lib.KDA_ERR_UNSUPPORTED),
    ("chunk", 128, _lib.KDA_ERR_UNSUPPORTED),
    ("io", 7, _lib.KDA_ERR_INVALID_ARG),
    ("H", 0, _lib.KDA_ERR_INVALID_ARG),
    ("T_total", 65, _lib.KDA_ERR_INVALID_ARG),       # cu[N] != T_total
    ("q", None, _lib.KDA_ERR_INVALID_ARG),
    ("g", None, _lib.KDA_ERR_INVALID_ARG),
    ("q", FAKE + 2, _lib.KDA_ERR_INVALID_ARG),       # misaligned
    ("qkv_row_stride", 100, _lib.KDA_ERR_INVALID_ARG),  # < H*D
    ("qkv_row_stride", 260, _lib.KDA_ERR_INVALID_ARG),  # not a multiple of 8
    ("workspace", None, _lib.KDA_ERR_WORKSPACE),
    ("workspace_bytes", 16, _lib.KDA_ERR_WORKSPACE),
    ("workspace", FAKE + 0x10000010, _lib.KDA_ERR_WORKSPACE),  # not 256-byte aligned
    ("out", FAKE, _lib.KDA_ERR_INVALID_ARG),         # out aliases q
])
def test_prefill_rejects_bad_arguments(field, value, code):
    a, cu = _args(**{field: value})
    assert _prefill(a) == code
    assert _lib.load().kda_last_error()


def test_prefill_rejects_bad_host_cu_seqlens():
    a, _ = _args(N=2)
    for bad in ([1, 30, 64], [0, 40, 30], [0, 30, 63]):
        cu = np.array(bad, np.int32)
        a.cu_seqlens_host = cu.ctypes.data
        assert _prefill(a) == _lib.KDA_ERR_INVALID_ARG


def test_prefill_rejects_aliased_conv_states():
    a, cu = _args(conv_state_in=FAKE + 0x800000, conv_state_out=FAKE + 0x800000 + 64)
    assert _prefill(a) == _lib.KDA_ERR_INVALID_ARG


def test_prefill_rejects_partially_overlapping_states():
    a, cu = _args(initial_state=FAKE + 0x20000000, final_state=FAKE + 0x20000000 + 4096)
    assert _prefill(a) == _lib.KDA_ERR_INVALID_ARG


def test_workspace_size_matches_layout():
    lib = _lib.load()
    for T, H, D, chunk, flags in [(8192, 96, 128, 64, 1), (64, 2, 16, 16, 0), (0, 4, 32, 32, 0)]:
        a, cu = _args(T_total=T, H=H, D=D, chunk=chunk, flags=flags)
        n = ctypes.c_size_t()
        assert lib.kda_prefill_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
        if flags & _lib.KDA_FLAG_FORCE_SIMT or D != 128:
            r = lambda x: (x + 255) // 256 * 256  # noqa: E731
            assert n.value == r(T * 3 * H * D * 4) + r(T * H * D * 4)


def test_segments_argument_is_range_checked():
    lib = _lib.load()
    for seg, want in [(-1, _lib.KDA_ERR_INVALID_ARG), (_lib.KDA_MAX_SEGMENTS + 1, _lib.KDA_ERR_INVALID_ARG),
                      (0, 0), (1, 0), (_lib.KDA_MAX_SEGMENTS, 0)]:
        a, cu = _args(T_total=8192, H=4, D=128, chunk=64, cu_seqlens_host=None)
        a.segments = seg
        n = ctypes.c_size_t()
        assert lib.kda_prefill_workspace_size(ctypes.byref(a), ctypes.byref(n)) == want
        path, p = ctypes.c_int(-1), ctypes.c_int(-1)
        assert lib.kda_prefill_plan(ctypes.byref(a), ctypes.byref(path), ctypes.byref(p)) == want
        if seg < 0 or seg > _lib.KDA_MAX_SEGMENTS:
            assert _prefill(a) == _lib.KDA_ERR_INVALID_ARG


def test_plan_without_a_tensor_core_device_is_simt():
    """With no sm_103 device current (this host has none) every call plans the SIMT path."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = _lib.load()
    a, cu = _args(T_total=1 << 20, H=24, D=128, chunk=64, cu_seqlens_host=None)
    path, p = ctypes.c_int(-1), ctypes.c_int(-1)
    assert lib.kda_prefill_plan(ctypes.byref(a), ctypes.byref(path), ctypes.byref(p)) == 0
    assert (path.value, p.value) == (_lib.KDA_PATH_SIMT, 1)


def test_plan_takes_the_recurrent_path_for_short_batches():
    """Every sequence of at most 8 tokens (host cu_seqlens given), D = 128: the recurrent
    path, whatever the chunk; one longer sequence, D != 128, no host copy or the opt-out flag:
    a chunkwise path."""
    lib = _lib.load()

    def plan(lengths, **kw):
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        a, _ = _args(T_total=int(cu[-1]), H=4, D=kw.pop("D", 128), chunk=kw.pop("chunk", 64), **kw)
        a.N = len(lengths)
        a.cu_seqlens_host = cu.ctypes.data
        path, p = ctypes.c_int(-1), ctypes.c_int(-1)
        assert lib.kda_prefill_plan(ctypes.byref(a), ctypes.byref(path), ctypes.byref(p)) == 0
        return path.value

    assert plan([4] * 8) == _lib.KDA_PATH_RECURRENT
    assert plan([1, 8, 0, 3]) == _lib.KDA_PATH_RECURRENT
    assert plan([1, 8, 0, 3], chunk=16) == _lib.KDA_PATH_RECURRENT
    assert plan([1, 9]) != _lib.KDA_PATH_RECURRENT
    assert plan([4] * 8, D=64) != _lib.KDA_PATH_RECURRENT
    assert plan([4] * 8, flags=_lib.KDA_FLAG_NO_RECURRENT) != _lib.KDA_PATH_RECURRENT
    assert plan([4] * 8, flags=_lib.KDA_FLAG_FORCE_SIMT) == _lib.KDA_PATH_SIMT


def test_short_conv_rejects_bad_arguments():
    lib = _lib.load()
    cu = np.array([0, 10], np.int32)
    base = dict(x=FAKE, xs=3 * 2 * 16, w=FAKE + 0x1000, cu=FAKE + 0x2000, cuh=cu.ctypes.data, N=1,
                T=10, H=2, D=16, csi=None, cso=None, y=FAKE + 0x100000, ys=96, l2=1, eps=1e-6,
                io=_lib.KDA_BF16)

    def call(**kw):
        b = dict(base, **kw)
        return lib.kda_short_conv(b["x"], b["xs"], b["w"], b["cu"], b["cuh"], b["N"], b["T"], b["H"],
                                  b["D"], b["csi"], b["cso"], b["y"], b["ys"], b["l2"], b["eps"],
                                  b["io"], None, None)

    assert call(D=24) == _lib.KDA_ERR_UNSUPPORTED
    assert call(xs=90) == _lib.KDA_ERR_INVALID_ARG
    assert call(y=FAKE + 8) == _lib.KDA_ERR_INVALID_ARG   # misaligned and overlapping
    assert call(T=11) == _lib.KDA_ERR_INVALID_ARG         # cu[N] != T
    assert call(w=None) == _lib.KDA_ERR_INVALID_ARG
    assert call(csi=FAKE + 0x200000, cso=FAKE + 0x200000) == _lib.KDA_ERR_INVALID_ARG


def test_decode_rejects_bad_arguments():
    lib = _lib.load()

    def call(**kw):
        a = _lib.DecodeArgs()
        a.N, a.H, a.D = 4, 2, 128
        a.io = a.out_dtype = _lib.KDA_BF16
        a.q, a.k, a.v = FAKE, FAKE + 0x1000, FAKE + 0x2000
        a.g, a.beta, a.conv_w = FAKE + 0x3000, FAKE + 0x4000, FAKE + 0x5000
        a.state, a.conv_state, a.out = FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000
        for k, v in kw.items():
            setattr(a, k, v)
        return lib.kda_decode_step(ctypes.byref(a), None)

    assert call(D=100) == _lib.KDA_ERR_UNSUPPORTED
    assert call(state=None) == _lib.KDA_ERR_INVALID_ARG
    assert call(state=FAKE + 0x100004) == _lib.KDA_ERR_INVALID_ARG
    assert call(qkv_row_stride=10) == _lib.KDA_ERR_INVALID_ARG
    assert call(out=FAKE + 0x100000) == _lib.KDA_ERR_INVALID_ARG
    assert call(N=-1) == _lib.KDA_ERR_INVALID_ARG


def test_binding_rejects_host_tensors_before_any_call():
    """Host tensors never reach the library: it would hand their pointers to a kernel."""
    import torch
    import kimi_delta_attention_16_gb300 as kda
    from kimi_delta_attention_16_gb300 import synth
    inp = synth.make_prefill("tiny_fp32", seed=0)  # host tensors
    with pytest.raises(ValueError, match="CUDA device"):
        kda.kda_prefill(inp.q, inp.k, inp.v, inp.conv_w, inp.g, inp.beta, inp.cu_seqlens,
                        chunk=inp.chunk, gate=inp.gate, rms_w=inp.rms_w)
    x = torch.zeros((inp.T, 3 * inp.H * inp.D))
    with pytest.raises(ValueError, match="CUDA device"):
        kda.kda_short_conv(x, inp.conv_w.reshape(-1, 4), inp.cu_seqlens, H=inp.H, D=inp.D)
    dec = synth.make_decode(seed=0, N=2, H=2, D=16, ring=1)
    with pytest.raises(ValueError, match="CUDA device"):
        kda.kda_decode_step(dec.q[0], dec.k[0], dec.v[0], dec.g[0], dec.beta[0], dec.conv_w,
                            dec.state, dec.conv_state, gate=dec.gate[0], rms_w=dec.rms_w)


def _gemm_args(**kw):
    g = _lib.GemmArgs()
    g.M, g.N, g.K = 128, 256, 128
    g.A, g.lda = FAKE, 128
    g.W, g.ldw = FAKE + (1 << 24), 128
    g.C, g.ldc = FAKE + (1 << 26), 256
    g.c_dtype = _lib.KDA_BF16
    g.epilogue = _lib.KDA_EPI_NONE
    for k, v in kw.items():
        setattr(g, k, v)
    return g


@pytest.mark.parametrize("field,value,code", [
    ("K", 96, _lib.KDA_ERR_UNSUPPORTED),          # not a multiple of 64
    ("K", 0, _lib.KDA_ERR_INVALID_ARG),
    ("M", -1, _lib.KDA_ERR_INVALID_ARG),
    ("lda", 64, _lib.KDA_ERR_INVALID_ARG),        # < K
    ("ldw", 132, _lib.KDA_ERR_INVALID_ARG),       # not a multiple of 8 elements
    ("ldc", 200, _lib.KDA_ERR_INVALID_ARG),       # < N
    ("A", FAKE + 8, _lib.KDA_ERR_INVALID_ARG),    # misaligned
    ("A", None, _lib.KDA_ERR_INVALID_ARG),
    ("C", FAKE + 64, _lib.KDA_ERR_INVALID_ARG),   # overlaps A
    ("epilogue", 7, _lib.KDA_ERR_INVALID_ARG),
    ("c_dtype", 5, _lib.KDA_ERR_INVALID_ARG),
])
def test_gemm_rejects_bad_arguments(field, value, code):
    lib = _lib.load()
    assert lib.kda_gemm(ctypes.byref(_gemm_args(**{field: value})), None) == code
    assert lib.kda_last_error()


def test_gemm_empty_problem_is_a_no_op_and_no_device_is_unsupported():
    lib = _lib.load()
    assert lib.kda_gemm(ctypes.byref(_gemm_args(M=0)), None) == _lib.KDA_OK
    # valid arguments without an sm_103 device in this process: unsupported, nothing launched
    import torch
    if not torch.cuda.is_available():
        assert lib.kda_gemm(ctypes.byref(_gemm_args()), None) == _lib.KDA_ERR_UNSUPPORTED


def _bwd_args(**kw):
    """kda_backward arguments for N = 2 sequences (40 + 24 tokens), H = 2, D = 128."""
    b = _lib.BackwardArgs()
    a, _ = _args()
    cu = np.array([0, 40, 64], np.int32)
    a.N, a.cu_seqlens_host = 2, cu.ctypes.data
    a.out = None
    b.fwd = a
    b._keep = cu
    b.dy = FAKE + 0x700000
    base = FAKE + 0x1000000
    for i, n in enumerate(("dq", "dk", "dv", "dconv_w", "dg", "dbeta")):
        setattr(b, n, base + i * 0x100000)
    for k, v in kw.items():
        if k.startswith("fwd."):
            setattr(b.fwd, k[4:], v)
        else:
            setattr(b, k, v)
    return b


@pytest.mark.parametrize("field,value,code", [
    ("fwd.D", 64, _lib.KDA_ERR_UNSUPPORTED),
    ("fwd.io", 9, _lib.KDA_ERR_INVALID_ARG),
    ("fwd.cu_seqlens_host", None, _lib.KDA_ERR_INVALID_ARG),   # the layout is planned on the host
    ("fwd.T_total", 63, _lib.KDA_ERR_INVALID_ARG),              # cu[N] != T_total
    ("fwd.q", None, _lib.KDA_ERR_INVALID_ARG),
    ("dy", None, _lib.KDA_ERR_INVALID_ARG),
    ("dbeta", None, _lib.KDA_ERR_INVALID_ARG),
    ("dconv_w", None, _lib.KDA_ERR_INVALID_ARG),
    ("dq", FAKE + 0x1000004, _lib.KDA_ERR_INVALID_ARG),         # misaligned
    ("dk", FAKE + 0x1000000 + 4096, _lib.KDA_ERR_INVALID_ARG),  # overlaps dq
    ("dg", FAKE + 0x400000, _lib.KDA_ERR_INVALID_ARG),          # aliases the input g
    ("dgate", FAKE + 0x10000000, _lib.KDA_ERR_INVALID_ARG),     # inside the workspace
    ("fwd.workspace", None, _lib.KDA_ERR_WORKSPACE),
    ("fwd.workspace_bytes", 1024, _lib.KDA_ERR_WORKSPACE),
])
def test_backward_rejects_bad_arguments(field, value, code):
    lib = _lib.load()
    b = _bwd_args(**{field: value})
    assert lib.kda_backward(ctypes.byref(b), None) == code
    assert lib.kda_last_error()


def test_backward_workspace_size_matches_the_stated_layout():
    """36 T H D + 8 T H + 8 slots D^2 + 8 slots D + 16 slots (49 D + 784) + 4 N H D + 8 (N + 1)
    bytes, each part rounded up to 256 (in the header's order), slots = H * sum over sequences of
    ceil(len / 64)."""
    lib = _lib.load()
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for lengths, H in [([40, 24], 2), ([0, 1, 65, 0, 128], 3), ([8192], 96), ([], 4)]:
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        b = _bwd_args(**{"fwd.N": len(lengths), "fwd.H": H, "fwd.T_total": int(cu[-1]),
                         "fwd.cu_seqlens_host": cu.ctypes.data})
        n = ctypes.c_size_t()
        assert lib.kda_backward_workspace_size(ctypes.byref(b), ctypes.byref(n)) == 0
        T, D, N = int(cu[-1]), 128, len(lengths)
        slots = H * sum((L + 63) // 64 for L in lengths)
        want = (r(T * 3 * H * D * 4) + r(T * H * 2 * 4) + r(T * H * D * 4) + r(T * 3 * H * D * 4)
                + r(T * H * D * 4) + r(T * H * D * 4)
                + 2 * r(slots * D * D * 4) + 2 * r(slots * D * 4) + r(16 * slots * (49 * D + 784))
                + r(N * H * D * 4) + r((N + 1) * 8))
        assert n.value == want, (lengths, H)


def test_backward_with_no_sequences_is_a_no_op():
    lib = _lib.load()
    cu = np.array([0], np.int32)
    b = _bwd_args(**{"fwd.N": 0, "fwd.T_total": 0, "fwd.cu_seqlens_host": cu.ctypes.data})
    assert lib.kda_backward(ctypes.byref(b), None) == _lib.KDA_OK
