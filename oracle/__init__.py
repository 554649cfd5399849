"""fp64 CPU oracle for the Kimi Delta Attention (KDA) layer -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does: the
oracle and the CUDA path share no code, header, helper or constant.  The
arithmetic lives in ``kda_oracle.c`` (plain C, fp64); this module only builds
it with gcc and marshals numpy arrays into it.

Sources, by page title and section:
  * "Kimi K3 / Architecture" -- panels "Kimi Delta Attention . one head at
    token t" and "KDA short convolution . one channel c at token t";
  * "Animated Kimi K3 architecture diagram" -- section "LOCAL MEMORY: A FIXED
    MATRIX THAT PREDICTS, FORGETS, AND CORRECTS" (the four moves and the
    notebook trace).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_dbl = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``_build/libkda_oracle.so`` (gcc, -O2, IEEE fp64)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.kda_oracle_conv_silu.restype = _int
            lib.kda_oracle_conv_silu.argtypes = [_i64, _int, _f32p, _i64, _f32p, _i32p, _int, _vp,
                                                 _vp, _i64, _vp, _int]
            lib.kda_oracle_l2norm.restype = None
            lib.kda_oracle_l2norm.argtypes = [_i64, _int, _f64p, _i64, _dbl]
            lib.kda_oracle_rmsnorm_gate.restype = None
            lib.kda_oracle_rmsnorm_gate.argtypes = [_i64, _int, _f64p, _vp, _vp, _dbl, _f64p]
            core = [_i64, _int, _int, _f64p, _i64, _f64p, _i64, _f64p, _i64, _f64p, _i64, _f64p,
                    _i64, _dbl, _f64p, _f64p, _i64]
            lib.kda_oracle_recurrence.restype = _int
            lib.kda_oracle_recurrence.argtypes = core
            lib.kda_oracle_chunkwise.restype = _int
            lib.kda_oracle_chunkwise.argtypes = core[:3] + [_int] + core[3:] + [_vp]
            lib.kda_oracle_forward.restype = _int
            lib.kda_oracle_forward.argtypes = [_i64, _int, _int, _int, _i32p, _f32p, _f32p, _f32p,
                                               _f32p, _vp, _f32p, _f32p, _vp, _vp, _dbl, _dbl,
                                               _dbl, _vp, _vp, _vp, _vp, _vp, _int]
            lib.kda_oracle_backward.restype = _int
            lib.kda_oracle_backward.argtypes = [_i64, _int, _int, _int, _i32p, _f32p, _f32p, _f32p,
                                                _f32p, _vp, _f32p, _f32p, _vp, _vp, _dbl, _dbl,
                                                _dbl, _vp, _f64p, _vp, _f64p, _f64p, _f64p, _f64p,
                                                _vp, _f64p, _f64p, _vp, _vp, _vp, _int]
            lib.kda_oracle_num_cores.restype = _int
            _lib = lib
    return _lib


def num_cores() -> int:
    return int(_load().kda_oracle_num_cores())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _exact_f32(a, name):
    """fp32 container for input values; refuses anything fp32 cannot hold exactly."""
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype == np.float32:
        return np.ascontiguousarray(a)
    b = np.ascontiguousarray(a.astype(np.float32))
    if not np.array_equal(b.astype(a.dtype), a):
        raise ValueError(f"oracle input {name} is not exactly representable in fp32")
    return b


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# --------------------------------------------------------------------------- pieces

def conv_silu(x, w, cu_seqlens, state_in=None, apply_silu=True):
    """Causal width-4 depthwise conv (+ SiLU) of every channel.

    x: [T_total, n_ch]; w: [n_ch, 4] (w[:, 3] multiplies x[t]); cu_seqlens: [N+1];
    state_in: [N, n_ch, 3] oldest first, or None (zero left padding).
    Returns (y [T_total, n_ch] fp64, state_out [N, n_ch, 3] fp64).
    """
    x = _exact_f32(x, "x")
    w = _exact_f32(w, "w")
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, n_ch = x.shape
    N = cu.shape[0] - 1
    si = _exact_f32(state_in, "state_in")
    y = np.zeros((T, n_ch), np.float64)
    so = np.zeros((N, n_ch, 3), np.float64)
    rc = _load().kda_oracle_conv_silu(T, n_ch, x, n_ch, w, cu, N, _ptr(si), _ptr(y), n_ch,
                                      _ptr(so), int(bool(apply_silu)))
    if rc:
        raise ValueError("kda_oracle_conv_silu rejected its arguments")
    return y, so


def l2norm(x, eps=1e-6):
    """Rows of x (last axis) scaled to x / sqrt(sum x^2 + eps)."""
    x = _f64(x).copy()
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    _load().kda_oracle_l2norm(flat.shape[0], d, flat, d, float(eps))
    return flat.reshape(x.shape)


def rmsnorm_gate(o, gate=None, w=None, eps=1e-6):
    """y = o / sqrt(mean o^2 + eps) * w * sigmoid(gate) over the last axis."""
    o = _f64(o)
    d = o.shape[-1]
    of = o.reshape(-1, d)
    gf = None if gate is None else _f64(gate).reshape(-1, d)
    wf = None if w is None else _f64(w).reshape(d)
    y = np.zeros_like(of)
    _load().kda_oracle_rmsnorm_gate(of.shape[0], d, of, _ptr(gf), _ptr(wf), float(eps), y)
    return y.reshape(o.shape)


def _core_args(q, k, v, g, beta, S0):
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    L, Dk = q.shape
    Dv = v.shape[1]
    assert k.shape == (L, Dk) and g.shape == (L, Dk) and v.shape == (L, Dv) and beta.shape == (L,)
    S = np.zeros((Dk, Dv)) if S0 is None else _f64(S0).copy()
    assert S.shape == (Dk, Dv)
    return q, k, v, g, beta, S, L, Dk, Dv


def recurrence(q, k, v, g, beta, S0=None, scale=1.0):
    """Token-sequential gated delta rule on convolved, normalised inputs.

    q, k, g: [L, Dk]; v: [L, Dv]; beta: [L]; S0: [Dk, Dv] or None (zeros).
    Returns (o [L, Dv], S_L [Dk, Dv]).
    """
    q, k, v, g, beta, S, L, Dk, Dv = _core_args(q, k, v, g, beta, S0)
    o = np.zeros((L, Dv))
    rc = _load().kda_oracle_recurrence(L, Dk, Dv, q, Dk, k, Dk, v, Dv, g, Dk, beta, 1,
                                       float(scale), S, o, Dv)
    if rc:
        raise MemoryError("kda_oracle_recurrence")
    return o, S


def chunkwise(q, k, v, g, beta, S0=None, chunk=64, scale=1.0, return_chunk_states=False):
    """The chunkwise form of the same recurrence (independent fp64 code path).

    Returns (o, S_L) or (o, S_L, states at every chunk start [n_chunks, Dk, Dv]).
    """
    q, k, v, g, beta, S, L, Dk, Dv = _core_args(q, k, v, g, beta, S0)
    o = np.zeros((L, Dv))
    n_chunks = (L + chunk - 1) // chunk
    st = np.zeros((max(n_chunks, 1), Dk, Dv)) if return_chunk_states else None
    rc = _load().kda_oracle_chunkwise(L, Dk, Dv, int(chunk), q, Dk, k, Dk, v, Dv, g, Dk, beta, 1,
                                      float(scale), S, o, Dv, _ptr(st))
    if rc:
        raise ValueError("kda_oracle_chunkwise")
    if return_chunk_states:
        return o, S, st[:n_chunks]
    return o, S


# --------------------------------------------------------------------------- whole layer

def forward(q, k, v, conv_w, cu_seqlens, g, beta, gate=None, rms_w=None, eps_l2=1e-6,
            eps_rms=1e-6, scale=1.0, initial_state=None, conv_state_in=None, heads=None,
            want_o_pre=False, n_threads=0):
    """Whole KDA layer (conv + SiLU + L2 -> gated delta rule -> RMSNorm + gate).

    Shapes (all host numpy; input values must be exact in fp32, e.g. bf16 or fp32 data):
      q, k, v, g, gate: [T_total, H, D]; beta: [T_total, H]; conv_w: [3, H*D, 4];
      cu_seqlens: [N+1]; initial_state: [N, H, D, D]; conv_state_in: [N, 3*H*D, 3].
    heads: optional list of head indices; the result then covers only those heads
    (in that order), and the head axis of every output has len(heads).
    Returns a dict with out [T, Hs, D], final_state [N, Hs, D, D], conv_state_out
    [N, 3*Hs*D, 3] (fp64) and, if want_o_pre, o_pre [T, Hs, D] (o before RMSNorm/gate).
    """
    q = np.asarray(q)
    T, H, D = q.shape
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    sel = np.arange(H) if heads is None else np.asarray(heads, dtype=np.int64)
    Hs = len(sel)

    def pick(a, axis):
        return None if a is None else np.take(np.asarray(a), sel, axis=axis)

    qs, ks, vs = (_exact_f32(pick(a, 1), n) for a, n in ((q, "q"), (k, "k"), (v, "v")))
    gs = _exact_f32(pick(g, 1), "g")
    bs = _exact_f32(pick(beta, 1), "beta")
    gts = _exact_f32(pick(gate, 1), "gate")
    cw = np.asarray(conv_w).reshape(3, H, D, 4)
    cws = _exact_f32(np.take(cw, sel, axis=1).reshape(3, Hs * D, 4), "conv_w")
    csi = None
    if conv_state_in is not None:
        c = np.asarray(conv_state_in).reshape(N, 3, H, D, 3)
        csi = _exact_f32(np.take(c, sel, axis=2).reshape(N, 3 * Hs * D, 3), "conv_state_in")
    s0 = None if initial_state is None else _f64(pick(initial_state, 1))
    rw = _exact_f32(rms_w, "rms_w")
    out = np.zeros((T, Hs, D))
    fin = np.zeros((N, Hs, D, D))
    cso = np.zeros((N, 3 * Hs * D, 3))
    opre = np.zeros((T, Hs, D)) if want_o_pre else None
    rc = _load().kda_oracle_forward(T, N, Hs, D, cu, qs, ks, vs, cws, _ptr(csi), gs, bs,
                                    _ptr(gts), _ptr(rw), float(eps_l2), float(eps_rms),
                                    float(scale), _ptr(s0), _ptr(out), _ptr(opre), _ptr(fin),
                                    _ptr(cso), int(n_threads))
    if rc:
        raise ValueError(f"kda_oracle_forward failed ({rc})")
    res = {"out": out, "final_state": fin, "conv_state_out": cso}
    if want_o_pre:
        res["o_pre"] = opre
    return res


def backward(q, k, v, conv_w, cu_seqlens, g, beta, dy, gate=None, rms_w=None, eps_l2=1e-6,
             eps_rms=1e-6, scale=1.0, initial_state=None, conv_state_in=None,
             d_final_state=None, n_threads=0):
    """Gradients of loss = sum(dy * out) + sum(d_final_state * final_state) through the whole
    layer, with respect to every input of ``forward`` (the same shapes; values exact in fp32).

    Returns a dict of fp64 arrays: dq, dk, dv (raw projections, [T, H, D]), dconv_w [3, H*D, 4],
    dg [T, H, D], dbeta [T, H], and -- for the inputs that were given -- dgate, drms_w [D],
    dinitial_state [N, H, D, D] (always returned: the state's gradient at the sequence start)
    and dconv_state_in [N, 3*H*D, 3].
    """
    q = np.asarray(q)
    T, H, D = q.shape
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    qs, ks, vs = (_exact_f32(a, n) for a, n in ((q, "q"), (k, "k"), (v, "v")))
    gs, bs, gts = _exact_f32(g, "g"), _exact_f32(beta, "beta"), _exact_f32(gate, "gate")
    cws = _exact_f32(np.asarray(conv_w).reshape(3, H * D, 4), "conv_w")
    csi = None if conv_state_in is None else _exact_f32(np.asarray(conv_state_in).reshape(N, 3 * H * D, 3),
                                                        "conv_state_in")
    rw = _exact_f32(rms_w, "rms_w")
    s0 = None if initial_state is None else _f64(initial_state)
    dyf = _f64(dy).reshape(T, H, D)
    dsf = None if d_final_state is None else _f64(d_final_state)
    out = {"dq": np.zeros((T, H, D)), "dk": np.zeros((T, H, D)), "dv": np.zeros((T, H, D)),
           "dconv_w": np.zeros((3, H * D, 4)), "dg": np.zeros((T, H, D)), "dbeta": np.zeros((T, H)),
           "dinitial_state": np.zeros((N, H, D, D))}
    dgate = np.zeros((T, H, D)) if gate is not None else None
    drms = np.zeros(D) if rms_w is not None else None
    dcs = np.zeros((N, 3 * H * D, 3)) if conv_state_in is not None else None
    rc = _load().kda_oracle_backward(T, N, H, D, cu, qs, ks, vs, cws, _ptr(csi), gs, bs, _ptr(gts),
                                     _ptr(rw), float(eps_l2), float(eps_rms), float(scale), _ptr(s0),
                                     dyf, _ptr(dsf), out["dq"], out["dk"], out["dv"], out["dconv_w"],
                                     _ptr(dcs), out["dg"], out["dbeta"], _ptr(dgate), _ptr(drms),
                                     _ptr(out["dinitial_state"]), int(n_threads))
    if rc:
        raise ValueError(f"kda_oracle_backward failed ({rc})")
    if dgate is not None:
        out["dgate"] = dgate
    if drms is not None:
        out["drms_w"] = drms
    if dcs is not None:
        out["dconv_state_in"] = dcs
    return out


# --------------------------------------------------------------------------- projections around the layer
# "Kimi K3 / Architecture", KDA panel: the normalized input x_t goes through linear projections
# to q, k, v and to alpha_t / beta_t (channel-wise retention, one write strength per head, the
# log-decay bounded below by -5); the head output y_t leaves through W_o.  The gated-MLA panel of
# the same page writes the output gate as sigmoid(W_g x_t), full rank, one value per channel.
# Readings (the pages give no activation for alpha and beta): g = -5 sigmoid(z) is the plainest
# map onto the bounded range (-5, 0); beta = sigmoid(z) onto the write-strength range (0, 1).

def linear(x, w):
    """x W^T in fp64: x [M, K], w [N, K] (a linear layer's [out, in] weight) -> [M, N]."""
    return _f64(x) @ _f64(w).T


def _sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(-np.abs(z))             # never overflows
    return np.where(z >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def decay_from_logits(z):
    """Bounded log-decay g = -5 sigmoid(z), in (-5, 0)."""
    return -5.0 * _sigmoid(z)


def strength_from_logits(z):
    """Write strength beta = sigmoid(z), in (0, 1)."""
    return _sigmoid(z)


def round_bf16(x):
    """Round to the nearest bf16 value, ties to even (the layer's bf16 interfaces: gate
    pre-activations and y leave their producers in bf16).  Returns fp64 values."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    b = f.view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    out = (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    return np.where(np.isfinite(f), out, f).astype(np.float64)


def projected_layer(x, w_alpha, w_beta, w_gate, w_out, q, k, v, conv_w, cu_seqlens, rms_w=None,
                    eps_l2=1e-6, eps_rms=1e-6, scale=1.0, initial_state=None, conv_state_in=None):
    """The layer with its projections: g = -5 sigmoid(x W_alpha^T), beta = sigmoid(x W_beta^T),
    gate = x W_g^T (rounded to bf16, the prefill's gate input dtype), y = the KDA layer, then
    out = y W_o^T with y rounded to bf16 first (the projection's input dtype).  q, k, v are the
    raw projections (inputs here).  Shapes: x [T, d_model]; w_alpha [H*D, d_model]; w_beta
    [H, d_model]; w_gate [H*D, d_model]; w_out [d_out, H*D].  Returns a dict with g, beta,
    gate, y, out (fp64) and final_state."""
    q = np.asarray(q)
    T, H, D = q.shape
    g = decay_from_logits(linear(x, w_alpha)).reshape(T, H, D)
    beta = strength_from_logits(linear(x, w_beta)).reshape(T, H)
    gate = round_bf16(linear(x, w_gate)).reshape(T, H, D)
    g32 = g.astype(np.float32)           # the prefill takes g and beta in fp32
    b32 = beta.astype(np.float32)
    res = forward(q, k, v, conv_w, cu_seqlens, g32, b32, gate=gate.astype(np.float32), rms_w=rms_w,
                  eps_l2=eps_l2, eps_rms=eps_rms, scale=scale, initial_state=initial_state,
                  conv_state_in=conv_state_in)
    y = res["out"]
    out = linear(round_bf16(y).reshape(T, H * D), w_out)
    return {"g": g, "beta": beta, "gate": gate, "y": y, "out": out,
            "final_state": res["final_state"]}
