"""fp64 CPU oracle for the HYPIC linear-attention state path -- TEST INFRASTRUCTURE.

This module is the checker, not the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it.
It loads ``hypic_oracle.c`` (built here with gcc, never with the CUDA
toolchain) through ctypes and shares no code with the GPU library.

What it computes (sources named in ``hypic_oracle.c``'s header):

* ``build``   -- per (segment, layer, head) the cached pair (T_C, S(C|0)) of
  the aibase article's linear-layer paragraph, by the plain token loop from
  T = I, S = 0.
* ``compose`` -- S(C1.C2) = T(C2) S(C1) + S(C2) along a chain (same
  paragraph), or the naive addition strawman with ``naive=True``.
* ``seam``    -- the seam-window advance of the full-attention paragraph:
  the token loop from a given state, emitting o_t = S_t^T q_t per token.  One
  seam spanning a whole request from zero is the full sequential recurrence.

All arithmetic is double precision; float32 inputs (bf16 inputs upcast
exactly) are widened on read.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FAMILIES = {"gdn": 0, "retnet": 1, "gla": 2, "vanilla": 3, "kda": 4, "mamba2": 5}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hypic_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libhypic_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP); returns the .so path."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            os.makedirs(os.path.dirname(_LIB), exist_ok=True)
            tmp = _LIB + f".tmp{os.getpid()}"
            # -ffp-contract=off keeps each double multiply and add a separate
            # IEEE operation, so the result does not depend on the host's FMA.
            subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC",
                                   "-shared", _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        LL = ctypes.c_longlong
        lib.oracle_build.argtypes = [I, I, I, I, I, I, P, P, LL, P, P, P, P, P, P, P, P, I]
        lib.oracle_compose.argtypes = [I, I, I, I, I, I, P, P, I, P, P, P, P, I, I, P]
        lib.oracle_seam.argtypes = [I, I, I, I, I, I, P, LL, P, P, P, P, P, P, P, P, P, P, I]
        lib.oracle_rope.argtypes = [I, I, I, I, I, I, I, ctypes.c_double, P, P, P]
        lib.oracle_conv.argtypes = [I, I, I, I, P, LL, P, P, P, P, I, P]
        for f in (lib.oracle_build, lib.oracle_compose, lib.oracle_seam, lib.oracle_rope, lib.oracle_conv):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f32(a):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return a


def _i32(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    return os.cpu_count() or 1


def build_pairs(family, k, v, cu_seqlens, *, alpha=None, beta=None, gamma=None, g=None,
                skip=None, n_threads=None):
    """(T_C, S(C|0)) for every (segment, layer, head).

    k: [n_layers][n_tokens][n_heads][dk], v: [..][dv]; gates as in the header.
    Returns (T, S) in float64 with leading [n_seg][n_layers][n_heads]; T is
    None for vanilla, shaped [...][dk][dk] (GDN, KDA), [...] (RetNet, Mamba2)
    or [...][dk] (GLA).
    """
    fam = FAMILIES[family]
    k, v = _f32(k), _f32(v)
    n_layers, n_tokens, n_heads, dk = k.shape
    dv = v.shape[-1]
    cu = _i32(cu_seqlens)
    n_seg = cu.shape[0] - 1
    sk = _i32(skip)
    alpha, beta, gamma, g = _f32(alpha), _f32(beta), _f32(gamma), _f32(g)
    S = np.zeros((n_seg, n_layers, n_heads, dk, dv))
    if fam in (0, 4):
        T = np.zeros((n_seg, n_layers, n_heads, dk, dk))
    elif fam in (1, 5):
        T = np.zeros((n_seg, n_layers, n_heads))
    elif fam == 2:
        T = np.zeros((n_seg, n_layers, n_heads, dk))
    else:
        T = None
    rc = _load().oracle_build(fam, n_layers, n_heads, dk, dv, n_seg, _ptr(cu), _ptr(sk), n_tokens,
                              _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(gamma), _ptr(g),
                              _ptr(T), _ptr(S), n_threads or default_threads())
    if rc:
        raise RuntimeError("oracle_build failed")
    return T, S


def compose(family, T_tab, S_tab, cu_chain, seg_idx, S0=None, *, naive=False, n_threads=None, want_T=False):
    """Chain compose S <- T_i S + S_i (double precision).

    T_tab / S_tab: [n_pairs][n_layers][n_heads]... as returned by build_pairs
    (T with any storage scale already applied).  Returns S_end
    [n_chains][n_layers][n_heads][dk][dv]; with ``want_T`` it returns
    (S_end, T_chain), T_chain being each chain's transition product
    T_{p_n} ... T_{p_1} in the family's T layout.
    """
    fam = FAMILIES[family]
    S_tab = _f64(S_tab)
    n_pairs, n_layers, n_heads, dk, dv = S_tab.shape
    T_tab = _f64(T_tab)
    cu = _i32(cu_chain)
    idx = _i32(seg_idx)
    n_chains = cu.shape[0] - 1
    S0 = _f64(S0)
    out = np.zeros((n_chains, n_layers, n_heads, dk, dv))
    T_out = None
    if want_T:
        shape = {0: (dk, dk), 4: (dk, dk), 1: (), 5: (), 2: (dk,)}[fam]
        T_out = np.zeros((n_chains, n_layers, n_heads) + shape)
    rc = _load().oracle_compose(fam, n_layers, n_heads, dk, dv, n_pairs, _ptr(T_tab), _ptr(S_tab),
                                n_chains, _ptr(cu), _ptr(idx), _ptr(S0), _ptr(out), int(bool(naive)),
                                n_threads or default_threads(), _ptr(T_out))
    if rc:
        raise RuntimeError("oracle_compose failed")
    return (out, T_out) if want_T else out


def seam(family, q, k, v, cu_seam, state_in=None, *, alpha=None, beta=None, gamma=None, g=None,
         n_threads=None):
    """Seam-window advance; returns (state_out, o).

    q, k: [n_layers][n_tok][n_heads][dk], v: [..][dv]; state_in
    [n_seams][n_layers][n_heads][dk][dv] or None (zero start).  o has the
    layout of v; rows outside every seam stay zero.
    """
    fam = FAMILIES[family]
    q, k, v = _f32(q), _f32(k), _f32(v)
    n_layers, n_tokens, n_heads, dk = k.shape
    dv = v.shape[-1]
    cu = _i32(cu_seam)
    n_seams = cu.shape[0] - 1
    alpha, beta, gamma, g = _f32(alpha), _f32(beta), _f32(gamma), _f32(g)
    sin = _f64(state_in)
    sout = np.zeros((n_seams, n_layers, n_heads, dk, dv))
    o = np.zeros((n_layers, n_tokens, n_heads, dv))
    rc = _load().oracle_seam(fam, n_layers, n_heads, dk, dv, n_seams, _ptr(cu), n_tokens,
                             _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(gamma), _ptr(g),
                             _ptr(sin), _ptr(sout), _ptr(o), n_threads or default_threads())
    if rc:
        raise RuntimeError("oracle_seam failed")
    return sout, o


# -------------------------------------------------------------- utilities --

def rope(family, T, S, delta, *, rotary_dim=None, base=10000.0):
    """Cached pairs re-rotated for a shift of delta[p] positions (the state
    re-rotation patch, restated in hypic_oracle.c): returns (R T R^T, R S) in
    float64 (T None for the scalar families and vanilla)."""
    fam = FAMILIES[family]
    S = np.array(S, dtype=np.float64, copy=True, order="C")
    n_pairs, n_layers, n_heads, dk, dv = S.shape
    T = None if T is None else np.array(T, dtype=np.float64, copy=True, order="C")
    d = np.ascontiguousarray(np.asarray(delta, dtype=np.int64))
    rc = _load().oracle_rope(fam, n_layers, n_heads, dk, dv, n_pairs, int(rotary_dim or dk), float(base),
                             _ptr(d), _ptr(T), _ptr(S))
    if rc:
        raise RuntimeError("oracle_rope failed")
    return T, S


def conv(x, cu_seam, w, *, hist=None, bias=None, act=1):
    """Conv-state warm-up (restated in hypic_oracle.c): the depthwise causal
    convolution of each window's inputs x [L][n_tok][C] with the K-1 inputs
    before it taken from hist [n_seams][L][K-1][C] (zeros when None);
    w [L][C][K], bias [L][C].  Returns y [L][n_tok][C] in float64."""
    x, w = _f32(x), _f32(w)
    n_layers, n_tokens, C = x.shape
    K = w.shape[-1]
    cu = _i32(cu_seam)
    y = np.zeros((n_layers, n_tokens, C))
    rc = _load().oracle_conv(n_layers, C, K, cu.shape[0] - 1, _ptr(cu), n_tokens, _ptr(x), _ptr(_f32(hist)),
                             _ptr(w), _ptr(_f32(bias)), int(act), _ptr(y))
    if rc:
        raise RuntimeError("oracle_conv failed")
    return y


def rel_fro(x, ref, axes):
    """Relative Frobenius error ||x - ref|| / ||ref|| per object, in fp64.

    ``axes`` are the trailing axes that make up one object (e.g. (-2, -1) for a
    d x d matrix).  The error is relative however small ||ref|| is (a T_C of
    1e-140 is compared at its own scale); only where ref is exactly zero is
    the absolute error returned.
    """
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref), axis=axes, keepdims=True)
    scale = np.where(scale > 0, scale, 1.0)
    num = np.sqrt(np.sum(((x - ref) / scale) ** 2, axis=axes))
    den = np.sqrt(np.sum((ref / scale) ** 2, axis=axes))
    return np.where(den == 0, num, num / np.where(den == 0, 1.0, den))


def scaled_to_f64(mant, exp):
    """T = mant * 2**exp, mant float32 [..][d][d], exp int32 [..] -> float64."""
    mant = np.asarray(mant, dtype=np.float64)
    exp = np.asarray(exp, dtype=np.int64)
    return np.ldexp(mant, exp[..., None, None])


def f64_to_scaled(T):
    """Split a float64 matrix stack into (float32 mantissa, int32 exponent).

    The exponent of each matrix is that of its largest magnitude entry, so the
    mantissa's largest entry lies in [0.5, 1); an all-zero matrix gets 0.
    This is the storage format the GPU build emits for GDN T_C.
    """
    T = np.asarray(T, dtype=np.float64)
    amax = np.max(np.abs(T), axis=(-2, -1))
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))
    e = np.where(amax > 0, e, 0).astype(np.int32)
    mant = np.ldexp(T, -e.astype(np.int64)[..., None, None]).astype(np.float32)
    return mant, e
