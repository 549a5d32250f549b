"""hypic_segment_build_noalloc, the build for callers that may not allocate
device memory (an engine plugin given only its input and output buffers, a
serving loop whose memory belongs to another allocator).  It must give the
same pairs as hypic_segment_build with a caller workspace, call after call,
although every call reuses the library's one fixed scratch array.

This file is named to be collected after every other test file."""
import numpy as np
import pytest

from linear_attn_state_hypic_gb300 import synth
from tests.helpers import TOL_BF16, TOL_F32, assert_rel, dev, gdn_T64, host


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import build_lib
    build_lib.build()
    from linear_attn_state_hypic_gb300 import binding
    return binding


def run_both(B, inp, dtype):
    """The regular call (torch-allocated workspace) and the no-alloc call on
    the same inputs; returns both (T, T_exp, S)."""
    k, v = dev(inp["k"], dtype), dev(inp["v"], dtype)
    a, b = dev(inp["alpha"]), dev(inp["beta"])
    cu = inp["cu_seqlens"]
    ref = B.segment_build("gdn", k, v, cu, alpha=a, beta=b)
    out = B.alloc_build_outputs("gdn", len(cu) - 1, k.shape[0], k.shape[2], k.shape[3], v.shape[3], k.device)
    args, keep = B.build_args("gdn", k, v, cu, alpha=a, beta=b, T_out=out[0], T_exp_out=out[1], S_out=out[2])
    st = B.hypic_segment_build_noalloc(args, B._stream(None))
    assert st == B.OK, B.lib.hypic_last_error_detail().decode()
    B.check_device()
    del keep
    return ref, out


@pytest.mark.gpu
def test_noalloc_build_matches_workspace_build_on_consecutive_calls(B):
    """Two calls in a row with different segment counts and inputs on the
    tensor-core path (d=128, bf16), then one on the CUDA-core path (d=64,
    fp32): each must match the regular entry point, so nothing left in the
    shared scratch by the previous call leaks into the next."""
    cases = [
        (synth.gdn_ragged(seed=31, H=4, d=128, lengths=[700, 1, 64, 129, 0, 2048, 513]), "bf16", TOL_BF16),
        (synth.gdn_ragged(seed=32, H=3, d=128, lengths=[96, 1500, 7], variant="highret"), "bf16", TOL_BF16),
        (synth.gdn_ragged(seed=33, H=2, d=64, lengths=[65, 300, 0, 1], dtype="f32"), "f32", TOL_F32),
    ]
    for inp, dtype, tol in cases:
        (T, Te, S), (T2, Te2, S2) = run_both(B, inp, dtype)
        assert_rel(host(S2), host(S), tol, what="no-alloc S vs workspace S")
        assert_rel(gdn_T64(T2, Te2), gdn_T64(T, Te), tol, what="no-alloc T vs workspace T")


def test_noalloc_rejects_batches_beyond_its_fixed_scratch(B):
    """More segments than the fixed array can order: refused with
    HYPIC_ERR_WORKSPACE and a message, before any GPU work (runs on CPU)."""
    n = B.NOALLOC_MAX_SEGMENTS + 1
    cu = np.arange(n + 1, dtype=np.int32)
    fake = 0x7F0000000000
    a = B.BuildArgs()
    a.family, a.in_dtype, a.n_layers, a.n_heads, a.dk, a.dv = 0, 1, 1, 1, 128, 128
    a.n_segments, a.n_tokens = n, n
    a.cu_seqlens, a.cu_seqlens_host = fake, cu.ctypes.data
    a.k, a.v, a.alpha, a.beta = fake + 0x100000, fake + 0x200000, fake + 0x300000, fake + 0x400000
    a.T_out, a.T_exp_out, a.S_out = fake + 0x500000, fake + 0x600000, fake + 0x700000
    assert B.hypic_segment_build_noalloc(a, None) == B.ERR_WORKSPACE
    assert str(B.NOALLOC_MAX_SEGMENTS) in B.lib.hypic_last_error_detail().decode()
    a.k = fake + 0x100008  # misaligned: the regular argument checks still apply
    a.n_segments, a.n_tokens = 2, 2
    assert B.hypic_segment_build_noalloc(a, None) == B.ERR_INVALID_ARG
