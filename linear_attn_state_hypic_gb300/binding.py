"""Thin ctypes binding of libhypic.so (include/hypic.h).

Argument marshalling only: the ``hypic_*`` functions take the C structs of the
header; the lower-case wrappers take torch CUDA tensors, allocate outputs and
scratch with torch (device memory is all torch is used for) and call the C
ABI on the current torch stream.  Every arithmetic step runs in the
library's kernels.  Importing this module loads the library and raises if it
has not been built (``python -m linear_attn_state_hypic_gb300.build_lib``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libhypic.so")

GDN, RETNET, GLA, VANILLA, KDA, MAMBA2 = 0, 1, 2, 3, 4, 5
FAMILY = {"gdn": GDN, "retnet": RETNET, "gla": GLA, "vanilla": VANILLA, "kda": KDA, "mamba2": MAMBA2}
F32, BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)

_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_int64


class BuildArgs(ctypes.Structure):
    _fields_ = [("family", _I), ("in_dtype", _I), ("n_layers", _I), ("n_heads", _I), ("dk", _I), ("dv", _I),
                ("n_segments", _I), ("n_tokens", _LL),
                ("cu_seqlens", _P), ("cu_seqlens_host", _P), ("seam_skip", _P), ("seam_skip_host", _P),
                ("k", _P), ("v", _P), ("alpha", _P), ("beta", _P), ("gamma", _P), ("g", _P),
                ("T_out", _P), ("T_exp_out", _P), ("S_out", _P)]


class ComposeArgs(ctypes.Structure):
    _fields_ = [("family", _I), ("n_layers", _I), ("n_heads", _I), ("dk", _I), ("dv", _I), ("n_pairs", _I),
                ("T_tab", _P), ("T_exp_tab", _P), ("S_tab", _P), ("n_chains", _I),
                ("cu_chain", _P), ("cu_chain_host", _P), ("seg_idx", _P), ("seg_idx_host", _P),
                ("S0", _P), ("S_out", _P), ("T_out", _P), ("T_exp_out", _P)]


class SeamArgs(ctypes.Structure):
    _fields_ = [("family", _I), ("in_dtype", _I), ("n_layers", _I), ("n_heads", _I), ("dk", _I), ("dv", _I),
                ("n_seams", _I), ("n_tokens", _LL),
                ("cu_seam", _P), ("cu_seam_host", _P), ("q", _P), ("k", _P), ("v", _P),
                ("alpha", _P), ("beta", _P), ("gamma", _P), ("g", _P),
                ("state_in", _P), ("state_out", _P), ("o_out", _P)]


class ChainArgs(ctypes.Structure):
    _fields_ = [("family", _I), ("in_dtype", _I), ("n_layers", _I), ("n_heads", _I), ("dk", _I), ("dv", _I),
                ("n_pairs", _I), ("T_tab", _P), ("T_exp_tab", _P), ("S_tab", _P), ("n_chains", _I),
                ("cu_chain", _P), ("cu_chain_host", _P), ("seg_idx", _P), ("seg_idx_host", _P),
                ("cu_step", _P), ("cu_step_host", _P), ("n_tokens", _LL),
                ("q", _P), ("k", _P), ("v", _P), ("alpha", _P), ("beta", _P), ("gamma", _P), ("g", _P),
                ("S0", _P), ("S_out", _P), ("o_out", _P)]


class RopeArgs(ctypes.Structure):
    _fields_ = [("family", _I), ("n_layers", _I), ("n_heads", _I), ("dk", _I), ("dv", _I), ("n_pairs", _I),
                ("rotary_dim", _I), ("base", ctypes.c_double), ("delta", _P), ("T", _P), ("S", _P)]


class ConvArgs(ctypes.Structure):
    _fields_ = [("n_layers", _I), ("C", _I), ("K", _I), ("n_seams", _I), ("n_tokens", _LL),
                ("cu_seam", _P), ("cu_seam_host", _P), ("x", _P), ("hist", _P), ("w", _P), ("bias", _P),
                ("act", _I), ("y", _P)]


EXPORTS = ["hypic_build_workspace_size", "hypic_segment_build", "hypic_compose", "hypic_seam_advance",
           "hypic_status_string", "hypic_last_error_detail", "hypic_version", "hypic_check_device",
           "hypic_segment_build_noalloc", "hypic_chain_workspace_size", "hypic_reuse_chain", "hypic_rope_rerotate",
           "hypic_conv_warmup"]
NOALLOC_MAX_SEGMENTS = 16384


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: run `python -m linear_attn_state_hypic_gb300.build_lib` "
                           "(or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    lib.hypic_build_workspace_size.argtypes = [ctypes.POINTER(BuildArgs)]
    lib.hypic_build_workspace_size.restype = ctypes.c_size_t
    lib.hypic_segment_build.argtypes = [ctypes.POINTER(BuildArgs), _P, ctypes.c_size_t, _P]
    lib.hypic_segment_build_noalloc.argtypes = [ctypes.POINTER(BuildArgs), _P]
    lib.hypic_segment_build_noalloc.restype = _I
    lib.hypic_compose.argtypes = [ctypes.POINTER(ComposeArgs), _P]
    lib.hypic_seam_advance.argtypes = [ctypes.POINTER(SeamArgs), _P]
    lib.hypic_check_device.argtypes = [_P]
    lib.hypic_chain_workspace_size.argtypes = [ctypes.POINTER(ChainArgs)]
    lib.hypic_chain_workspace_size.restype = ctypes.c_size_t
    lib.hypic_reuse_chain.argtypes = [ctypes.POINTER(ChainArgs), _P, ctypes.c_size_t, _P]
    lib.hypic_rope_rerotate.argtypes = [ctypes.POINTER(RopeArgs), _P]
    lib.hypic_conv_warmup.argtypes = [ctypes.POINTER(ConvArgs), _P]
    for f in (lib.hypic_segment_build, lib.hypic_compose, lib.hypic_seam_advance, lib.hypic_check_device,
              lib.hypic_reuse_chain, lib.hypic_rope_rerotate, lib.hypic_conv_warmup):
        f.restype = _I
    lib.hypic_status_string.argtypes = [_I]
    lib.hypic_status_string.restype = ctypes.c_char_p
    lib.hypic_last_error_detail.argtypes = []
    lib.hypic_last_error_detail.restype = ctypes.c_char_p
    lib.hypic_version.restype = _I
    return lib


lib = _load()


class HypicError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(f"{lib.hypic_status_string(status).decode()}: {lib.hypic_last_error_detail().decode()}")


def _check(status: int):
    if status != OK:
        raise HypicError(status)


# ------------------------------------------------------------ raw C ABI ----

def hypic_build_workspace_size(args: BuildArgs) -> int:
    return lib.hypic_build_workspace_size(ctypes.byref(args))


def hypic_segment_build(args: BuildArgs, workspace: int, workspace_bytes: int, stream: int) -> int:
    return lib.hypic_segment_build(ctypes.byref(args), workspace, workspace_bytes, stream)


def hypic_segment_build_noalloc(args: BuildArgs, stream: int) -> int:
    return lib.hypic_segment_build_noalloc(ctypes.byref(args), stream)


def hypic_compose(args: ComposeArgs, stream: int) -> int:
    return lib.hypic_compose(ctypes.byref(args), stream)


def hypic_seam_advance(args: SeamArgs, stream: int) -> int:
    return lib.hypic_seam_advance(ctypes.byref(args), stream)


def hypic_check_device(stream: int) -> int:
    return lib.hypic_check_device(stream)


def hypic_rope_rerotate(args: RopeArgs, stream: int) -> int:
    return lib.hypic_rope_rerotate(ctypes.byref(args), stream)


def hypic_conv_warmup(args: ConvArgs, stream: int) -> int:
    return lib.hypic_conv_warmup(ctypes.byref(args), stream)


def hypic_version() -> int:
    return lib.hypic_version()


# --------------------------------------------------------- torch wrappers --

def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _host_i32(x):
    """Contiguous host int32 numpy copy (kept alive by the caller's frame)."""
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _hptr(a) -> int | None:
    return None if a is None else a.ctypes.data


def _dev_i32(host, dev, device):
    import torch
    if host is None:
        return None
    if dev is not None:
        return dev
    return torch.from_numpy(host).to(device, non_blocking=False)


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"k/v/q must be float32 or bfloat16, got {t.dtype}")


def build_args(family, k, v, cu_seqlens, *, alpha=None, beta=None, gamma=None, g=None, seam_skip=None,
               T_out=None, T_exp_out=None, S_out=None, cu_seqlens_dev=None, seam_skip_dev=None):
    """Fill a BuildArgs from tensors; returns (args, keepalive)."""
    fam = FAMILY[family] if isinstance(family, str) else family
    cu = _host_i32(cu_seqlens)
    sk = _host_i32(seam_skip)
    cu_d = _dev_i32(cu, cu_seqlens_dev, k.device)
    sk_d = _dev_i32(sk, seam_skip_dev, k.device)
    a = BuildArgs()
    a.family, a.in_dtype = fam, _dtype_code(k)
    a.n_layers, a.n_tokens, a.n_heads, a.dk = k.shape
    a.dv = v.shape[-1]
    a.n_segments = len(cu) - 1
    a.cu_seqlens, a.cu_seqlens_host = _ptr(cu_d), _hptr(cu)
    a.seam_skip, a.seam_skip_host = _ptr(sk_d), _hptr(sk)
    a.k, a.v = _ptr(k), _ptr(v)
    a.alpha, a.beta, a.gamma, a.g = _ptr(alpha), _ptr(beta), _ptr(gamma), _ptr(g)
    a.T_out, a.T_exp_out, a.S_out = _ptr(T_out), _ptr(T_exp_out), _ptr(S_out)
    return a, (cu, sk, cu_d, sk_d)


def alloc_build_outputs(family, n_seg, n_layers, n_heads, dk, dv, device):
    import torch
    fam = FAMILY[family] if isinstance(family, str) else family
    lead = (n_seg, n_layers, n_heads)
    S = torch.empty(lead + (dk, dv), dtype=torch.float32, device=device)
    T = T_exp = None
    if fam in (GDN, KDA):
        T = torch.empty(lead + (dk, dk), dtype=torch.float32, device=device)
        T_exp = torch.empty(lead, dtype=torch.int32, device=device)
    elif fam in (RETNET, MAMBA2):
        T = torch.empty(lead, dtype=torch.float32, device=device)
    elif fam == GLA:
        T = torch.empty(lead + (dk,), dtype=torch.float32, device=device)
    return T, T_exp, S


def segment_build(family, k, v, cu_seqlens, *, alpha=None, beta=None, gamma=None, g=None, seam_skip=None,
                  out=None, workspace=None, stream=None, cu_seqlens_dev=None, seam_skip_dev=None):
    """(T, T_exp, S) per (segment, layer, head) via hypic_segment_build.

    k, v: CUDA tensors [n_layers][n_tokens][n_heads][d]; cu_seqlens (and
    seam_skip) host int arrays.  For GDN and KDA the transition product is
    T_C = T * 2**T_exp.  ``out`` = (T, T_exp, S) preallocated, optional.
    """
    import torch
    n_seg = len(cu_seqlens) - 1
    if out is None:
        out = alloc_build_outputs(family, n_seg, k.shape[0], k.shape[2], k.shape[3], v.shape[3], k.device)
    T, T_exp, S = out
    a, keep = build_args(family, k, v, cu_seqlens, alpha=alpha, beta=beta, gamma=gamma, g=g, seam_skip=seam_skip,
                         T_out=T, T_exp_out=T_exp, S_out=S, cu_seqlens_dev=cu_seqlens_dev,
                         seam_skip_dev=seam_skip_dev)
    need = hypic_build_workspace_size(a)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=k.device)
    _check(hypic_segment_build(a, _ptr(workspace), workspace.numel(), _stream(stream)))
    del keep
    return T, T_exp, S


def compose_args(family, S_tab, cu_chain, seg_idx, *, T_tab=None, T_exp_tab=None, S0=None, S_out=None,
                 T_out=None, T_exp_out=None, cu_chain_dev=None, seg_idx_dev=None):
    fam = FAMILY[family] if isinstance(family, str) else family
    cu = _host_i32(cu_chain)
    idx = _host_i32(seg_idx)
    cu_d = _dev_i32(cu, cu_chain_dev, S_tab.device)
    idx_d = _dev_i32(idx, seg_idx_dev, S_tab.device) if len(idx) else None
    a = ComposeArgs()
    a.family = fam
    a.n_pairs, a.n_layers, a.n_heads, a.dk, a.dv = S_tab.shape
    a.T_tab, a.T_exp_tab, a.S_tab = _ptr(T_tab), _ptr(T_exp_tab), _ptr(S_tab)
    a.n_chains = len(cu) - 1
    a.cu_chain, a.cu_chain_host = _ptr(cu_d), _hptr(cu)
    a.seg_idx, a.seg_idx_host = _ptr(idx_d), _hptr(idx) if len(idx) else None
    a.S0, a.S_out = _ptr(S0), _ptr(S_out)
    a.T_out, a.T_exp_out = _ptr(T_out), _ptr(T_exp_out)
    return a, (cu, idx, cu_d, idx_d)


def compose(family, S_tab, cu_chain, seg_idx, *, T_tab=None, T_exp_tab=None, S0=None, out=None, stream=None,
            cu_chain_dev=None, seg_idx_dev=None, want_T=False):
    """End state of every chain via hypic_compose: [n_chains][L][H][dk][dv].

    With ``want_T`` returns (S_end, T_chain, T_chain_exp): each chain's own
    transition product, laid out like the build's T (T_chain_exp only for the
    dense families, else None)."""
    import torch
    fam = FAMILY[family] if isinstance(family, str) else family
    n_chains = len(cu_chain) - 1
    if out is None:
        out = torch.empty((n_chains,) + tuple(S_tab.shape[1:]), dtype=torch.float32, device=S_tab.device)
    T_out = T_exp_out = None
    if want_T:
        T_out, T_exp_out, _ = alloc_build_outputs(fam, n_chains, S_tab.shape[1], S_tab.shape[2], S_tab.shape[3],
                                                  S_tab.shape[4], S_tab.device)
    a, keep = compose_args(family, S_tab, cu_chain, seg_idx, T_tab=T_tab, T_exp_tab=T_exp_tab, S0=S0, S_out=out,
                           T_out=T_out, T_exp_out=T_exp_out, cu_chain_dev=cu_chain_dev, seg_idx_dev=seg_idx_dev)
    _check(hypic_compose(a, _stream(stream)))
    del keep
    return (out, T_out, T_exp_out) if want_T else out


def seam_args(family, q, k, v, cu_seam, *, alpha=None, beta=None, gamma=None, g=None, state_in=None,
              state_out=None, o_out=None, cu_seam_dev=None):
    fam = FAMILY[family] if isinstance(family, str) else family
    cu = _host_i32(cu_seam)
    cu_d = _dev_i32(cu, cu_seam_dev, k.device)
    a = SeamArgs()
    a.family, a.in_dtype = fam, _dtype_code(k)
    a.n_layers, a.n_tokens, a.n_heads, a.dk = k.shape
    a.dv = v.shape[-1]
    a.n_seams = len(cu) - 1
    a.cu_seam, a.cu_seam_host = _ptr(cu_d), _hptr(cu)
    a.q, a.k, a.v = _ptr(q), _ptr(k), _ptr(v)
    a.alpha, a.beta, a.gamma, a.g = _ptr(alpha), _ptr(beta), _ptr(gamma), _ptr(g)
    a.state_in, a.state_out, a.o_out = _ptr(state_in), _ptr(state_out), _ptr(o_out)
    return a, (cu, cu_d)


def seam_advance(family, q, k, v, cu_seam, *, alpha=None, beta=None, gamma=None, g=None, state_in=None,
                 state_out=None, o_out=None, stream=None, cu_seam_dev=None):
    """(state_out, o) via hypic_seam_advance; state_out may be state_in."""
    import torch
    n_seams = len(cu_seam) - 1
    L, N, H, dk = k.shape
    dv = v.shape[-1]
    if state_out is None:
        state_out = torch.empty((n_seams, L, H, dk, dv), dtype=torch.float32, device=k.device)
    if o_out is None:
        o_out = torch.empty((L, N, H, dv), dtype=torch.float32, device=k.device)
    a, keep = seam_args(family, q, k, v, cu_seam, alpha=alpha, beta=beta, gamma=gamma, g=g, state_in=state_in,
                        state_out=state_out, o_out=o_out, cu_seam_dev=cu_seam_dev)
    _check(hypic_seam_advance(a, _stream(stream)))
    del keep
    return state_out, o_out


def hypic_chain_workspace_size(args: ChainArgs) -> int:
    return lib.hypic_chain_workspace_size(ctypes.byref(args))


def hypic_reuse_chain(args: ChainArgs, workspace, workspace_bytes: int, stream) -> int:
    return lib.hypic_reuse_chain(ctypes.byref(args), workspace, workspace_bytes, stream)


def chain_args(family, S_tab, cu_chain, seg_idx, cu_step, q, k, v, *, T_tab=None, T_exp_tab=None, alpha=None,
               beta=None, gamma=None, g=None, S0=None, S_out=None, o_out=None, cu_chain_dev=None, seg_idx_dev=None,
               cu_step_dev=None):
    fam = FAMILY[family] if isinstance(family, str) else family
    cu = _host_i32(cu_chain)
    idx = _host_i32(seg_idx)
    cs = _host_i32(cu_step)
    dev = S_tab.device
    cu_d = _dev_i32(cu, cu_chain_dev, dev)
    idx_d = _dev_i32(idx, seg_idx_dev, dev) if len(idx) else None
    cs_d = _dev_i32(cs, cu_step_dev, dev)
    a = ChainArgs()
    a.family, a.in_dtype = fam, _dtype_code(k)
    a.n_pairs, a.n_layers, a.n_heads, a.dk, a.dv = S_tab.shape
    a.T_tab, a.T_exp_tab, a.S_tab = _ptr(T_tab), _ptr(T_exp_tab), _ptr(S_tab)
    a.n_chains = len(cu) - 1
    a.cu_chain, a.cu_chain_host = _ptr(cu_d), _hptr(cu)
    a.seg_idx, a.seg_idx_host = _ptr(idx_d), _hptr(idx) if len(idx) else None
    a.cu_step, a.cu_step_host = _ptr(cs_d), _hptr(cs)
    a.n_tokens = int(cs[-1])
    a.q, a.k, a.v = _ptr(q), _ptr(k), _ptr(v)
    a.alpha, a.beta, a.gamma, a.g = _ptr(alpha), _ptr(beta), _ptr(gamma), _ptr(g)
    a.S0, a.S_out, a.o_out = _ptr(S0), _ptr(S_out), _ptr(o_out)
    return a, (cu, idx, cs, cu_d, idx_d, cs_d)


def reuse_chain(family, S_tab, cu_chain, seg_idx, cu_step, q, k, v, *, T_tab=None, T_exp_tab=None, alpha=None,
                beta=None, gamma=None, g=None, S0=None, out=None, o_out=None, stream=None):
    """(end states [n_chains][L][H][dk][dv], seam outputs [L][n_tokens][H][dv]) via
    hypic_reuse_chain; q, k, v: [L][n_tokens][H][d] seam tokens, packed by step."""
    import torch
    n_chains = len(cu_chain) - 1
    L, N, H, dk = k.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((n_chains,) + tuple(S_tab.shape[1:]), dtype=torch.float32, device=S_tab.device)
    if o_out is None:
        o_out = torch.empty((L, N, H, dv), dtype=torch.float32, device=S_tab.device)
    a, keep = chain_args(family, S_tab, cu_chain, seg_idx, cu_step, q, k, v, T_tab=T_tab, T_exp_tab=T_exp_tab,
                         alpha=alpha, beta=beta, gamma=gamma, g=g, S0=S0, S_out=out, o_out=o_out)
    nbytes = hypic_chain_workspace_size(a)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=S_tab.device) if nbytes else None
    _check(hypic_reuse_chain(a, _ptr(ws), nbytes, _stream(stream)))
    del keep
    return out, o_out


def rope_rerotate(family, S, delta, *, T=None, rotary_dim=None, base=10000.0, stream=None):
    """Re-rotate cached pairs in place for position shifts delta[p]
    (hypic_rope_rerotate): S [n_pairs][L][H][dk][dv] and, for GDN, the T
    mantissa [n_pairs][L][H][dk][dk].  delta: host ints."""
    import torch
    fam = FAMILY[family] if isinstance(family, str) else family
    d = torch.as_tensor(np.asarray(delta, dtype=np.int64)).to(S.device)
    a = RopeArgs()
    a.family = fam
    a.n_pairs, a.n_layers, a.n_heads, a.dk, a.dv = S.shape
    a.rotary_dim = int(rotary_dim or S.shape[3])
    a.base = float(base)
    a.delta, a.T, a.S = _ptr(d), _ptr(T), _ptr(S)
    _check(hypic_rope_rerotate(a, _stream(stream)))
    return T, S


def conv_warmup(x, cu_seam, w, *, hist=None, bias=None, act=1, out=None, stream=None):
    """Conv-state warm-up of seam windows (hypic_conv_warmup): x [L][n_tok][C]
    CUDA f32, cu_seam host ints, w [L][C][K], hist [n_seams][L][K-1][C] or
    None, bias [L][C] or None.  Returns y [L][n_tok][C]."""
    import torch
    cu = _host_i32(cu_seam)
    cu_d = _dev_i32(cu, None, x.device)
    if out is None:
        out = torch.empty_like(x)
    a = ConvArgs()
    a.n_layers, a.n_tokens, a.C = x.shape
    a.K = w.shape[-1]
    a.n_seams = len(cu) - 1
    a.cu_seam, a.cu_seam_host = _ptr(cu_d), _hptr(cu)
    a.x, a.hist, a.w, a.bias, a.act, a.y = _ptr(x), _ptr(hist), _ptr(w), _ptr(bias), int(act), _ptr(out)
    _check(hypic_conv_warmup(a, _stream(stream)))
    del cu, cu_d
    return out


def check_device(stream=None):
    """Synchronise and raise HypicError if a bounded device wait ran out."""
    _check(hypic_check_device(_stream(stream)))
