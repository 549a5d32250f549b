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


@pytest.mark.gpu
def test_noalloc_at_the_segment_limit(B):
    """Exactly HYPIC_NOALLOC_MAX_SEGMENTS short segments (lengths 0..8, one
    layer and head, d=16, fp32): the order fills the fixed array to its end
    and the counter block right after it is used.  The pairs must equal the
    workspace build's; the time of the call (mostly the single-CTA ordering
    of 16,384 segments) is printed."""
    import torch
    n = B.NOALLOC_MAX_SEGMENTS
    rng = np.random.default_rng(77)
    lengths = rng.integers(0, 9, n)
    lengths[:4] = [0, 8, 1, 0]
    inp = synth.gdn_ragged(seed=34, H=1, d=16, lengths=lengths, dtype="f32")
    (T, Te, S), (T2, Te2, S2) = run_both(B, inp, "f32")
    assert_rel(host(S2), host(S), TOL_F32, what="no-alloc S vs workspace S at the segment limit")
    assert_rel(gdn_T64(T2, Te2), gdn_T64(T, Te), TOL_F32, what="no-alloc T vs workspace T at the segment limit")
    k, v = dev(inp["k"], "f32"), dev(inp["v"], "f32")
    a, b = dev(inp["alpha"]), dev(inp["beta"])
    args, keep = B.build_args("gdn", k, v, inp["cu_seqlens"], alpha=a, beta=b, T_out=T2, T_exp_out=Te2, S_out=S2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    assert B.hypic_segment_build_noalloc(args, B._stream(None)) == B.OK
    e1.record()
    torch.cuda.synchronize()
    B.check_device()
    print(f"no-alloc build of {n} segments ({int(lengths.sum())} tokens, d=16): {e0.elapsed_time(e1):.3f} ms")


@pytest.mark.gpu
def test_noalloc_call_allocates_nothing(B):
    """Around a warmed-up call, torch's allocator sees no new allocation or
    segment: the call's only scratch is the library's fixed array."""
    import torch
    inp = synth.gdn_ragged(seed=35, H=2, d=128, lengths=[300, 65, 0])
    k, v = dev(inp["k"], "bf16"), dev(inp["v"], "bf16")
    a, b = dev(inp["alpha"]), dev(inp["beta"])
    cu = inp["cu_seqlens"]
    out = B.alloc_build_outputs("gdn", len(cu) - 1, k.shape[0], k.shape[2], k.shape[3], v.shape[3], k.device)
    args, keep = B.build_args("gdn", k, v, cu, alpha=a, beta=b, T_out=out[0], T_exp_out=out[1], S_out=out[2])
    assert B.hypic_segment_build_noalloc(args, B._stream(None)) == B.OK  # warm-up (module load, first lookup)
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(),
              len(torch.cuda.memory_snapshot()))
    for _ in range(3):
        assert B.hypic_segment_build_noalloc(args, B._stream(None)) == B.OK
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), len(torch.cuda.memory_snapshot()))
    B.check_device()
    assert after == before, f"allocator state changed around the no-alloc call: {before} -> {after}"
    del keep
