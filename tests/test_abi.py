"""C-ABI checks that need no GPU: the library loads, exports every function
include/hypic.h declares, the ctypes structs match the header's layout (as
compiled by gcc), and every host-side validation path returns its status
before any CUDA call is made."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hypic.h")


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import build_lib
    build_lib.build()
    from linear_attn_state_hypic_gb300 import binding
    return binding


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"HYPIC_API\s+[\w\s\*]+?\b(hypic_\w+)\s*\(", src)))


def test_header_declares_the_three_calls():
    fns = declared_functions()
    for f in ("hypic_segment_build", "hypic_compose", "hypic_seam_advance", "hypic_build_workspace_size",
              "hypic_reuse_chain", "hypic_chain_workspace_size"):
        assert f in fns


def test_library_exports_every_declared_symbol(B):
    fns = declared_functions()
    assert fns, "no declarations parsed"
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(hypic_\w+)", out))
    assert set(fns) <= exported, set(fns) - exported
    for f in fns:
        getattr(B.lib, f)  # resolvable through ctypes
    assert set(B.EXPORTS) == set(fns)


def test_struct_layout_matches_header(B, tmp_path):
    """Compile a probe against include/hypic.h with gcc and compare sizeof and
    every field offset with the ctypes mirrors."""
    structs = {"hypic_build_args": B.BuildArgs, "hypic_compose_args": B.ComposeArgs, "hypic_seam_args": B.SeamArgs,
               "hypic_chain_args": B.ChainArgs, "hypic_rope_args": B.RopeArgs, "hypic_conv_args": B.ConvArgs}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "hypic.h"', "int main(void){"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0;}")
    c = tmp_path / "probe.c"
    c.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.check_call(["gcc", "-I", os.path.dirname(HEADER), str(c), "-o", str(exe)])
    got = {}
    for ln in subprocess.check_output([str(exe)], text=True).splitlines():
        s, f, v = ln.split()
        got[(s, f)] = int(v)
    for cname, py in structs.items():
        assert got[(cname, "sizeof")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)


def test_status_strings_and_version(B):
    assert B.hypic_version() == 150
    for code, name in enumerate(["HYPIC_OK", "HYPIC_ERR_INVALID_ARG", "HYPIC_ERR_UNSUPPORTED", "HYPIC_ERR_WORKSPACE",
                                 "HYPIC_ERR_CUDA", "HYPIC_ERR_TIMEOUT"]):
        assert B.lib.hypic_status_string(code).decode() == name


# ------------------------------------------------ host validation (no GPU) --
# Device pointers are fake but 16-byte aligned: validation never dereferences
# them, and every case below is rejected before the first CUDA call.

FAKE = 0x7F0000000000


def fake(i):
    return FAKE + 0x100000 * (i + 1)


def base_build(B, family=0, d=128, n_seg=2, lengths=(64, 80)):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    a = B.BuildArgs()
    a.family, a.in_dtype, a.n_layers, a.n_heads, a.dk, a.dv = family, 1, 1, 2, d, d
    a.n_segments, a.n_tokens = n_seg, int(cu[-1])
    a.cu_seqlens, a.cu_seqlens_host = fake(0), cu.ctypes.data
    a.k, a.v = fake(1), fake(2)
    if family == 0:
        a.alpha, a.beta = fake(3), fake(4)
        a.T_exp_out = fake(6)
    if family == 1:
        a.gamma = fake(3)
    if family == 2:
        a.g = fake(3)
    if family == 4:  # KDA: per-channel gate g and beta; dense T with exponent
        a.g, a.beta = fake(3), fake(4)
        a.T_exp_out = fake(6)
    if family == 5:  # Mamba2: per-token decay in alpha; scalar T
        a.alpha = fake(3)
    if family != 3:
        a.T_out = fake(5)
    a.S_out = fake(7)
    return a, cu


def run_build(B, a, ws=1 << 20, ws_ptr=None):
    return B.hypic_segment_build(a, fake(9) if ws_ptr is None else ws_ptr, ws, None)


def test_build_valid_args_reach_workspace_check(B):
    for fam in range(6):
        a, keep = base_build(B, fam)
        need = B.hypic_build_workspace_size(a)
        assert need >= 256
        assert run_build(B, a, ws=need - 1) == B.ERR_WORKSPACE
        assert run_build(B, a, ws_ptr=0) == B.ERR_WORKSPACE
        assert run_build(B, a, ws_ptr=fake(9) + 16) == B.ERR_WORKSPACE  # not 256-byte aligned


@pytest.mark.parametrize("mutate,status", [
    (lambda a, c: setattr(a, "family", 7), 1),
    (lambda a, c: setattr(a, "in_dtype", 5), 1),
    (lambda a, c: setattr(a, "dk", 96), 2),
    (lambda a, c: (setattr(a, "dk", 64)), 2),          # GDN dk != dv
    (lambda a, c: setattr(a, "n_heads", 0), 1),
    (lambda a, c: setattr(a, "n_segments", -1), 1),
    (lambda a, c: setattr(a, "n_tokens", 10), 1),       # cu_seqlens[-1] > n_tokens
    (lambda a, c: c.__setitem__(1, 200), 1),            # non-monotone
    (lambda a, c: setattr(a, "cu_seqlens_host", None), 1),
    (lambda a, c: setattr(a, "k", None), 1),
    (lambda a, c: setattr(a, "k", fake(1) + 8), 1),     # misaligned
    (lambda a, c: setattr(a, "alpha", None), 1),
    (lambda a, c: setattr(a, "gamma", fake(8)), 1),     # gamma given for GDN
    (lambda a, c: setattr(a, "T_exp_out", None), 1),
    (lambda a, c: setattr(a, "S_out", None), 1),
    (lambda a, c: setattr(a, "seam_skip", fake(8)), 1), # device without host copy
])
def test_build_rejections(B, mutate, status):
    a, cu = base_build(B)
    mutate(a, cu)
    assert run_build(B, a) == status
    assert B.lib.hypic_last_error_detail().decode()
    assert B.hypic_build_workspace_size(a) == 0


def test_build_seam_skip_range(B):
    a, cu = base_build(B)
    sk = np.array([0, 81], np.int32)   # longer than the segment
    a.seam_skip, a.seam_skip_host = fake(8), sk.ctypes.data
    assert run_build(B, a) == B.ERR_INVALID_ARG
    sk[1] = 80
    assert run_build(B, a, ws=1) == B.ERR_WORKSPACE  # valid now; stops at the workspace


def test_build_family_specific_rejections(B):
    a, _ = base_build(B, 3)
    a.T_out = fake(5)
    assert run_build(B, a) == B.ERR_INVALID_ARG   # vanilla stores no T
    a, _ = base_build(B, 1)
    a.beta = fake(4)
    assert run_build(B, a) == B.ERR_INVALID_ARG   # RetNet takes no beta
    a, _ = base_build(B, 2)
    a.g = None
    assert run_build(B, a) == B.ERR_INVALID_ARG
    for mut in (lambda a: setattr(a, "g", None), lambda a: setattr(a, "beta", None),
                lambda a: setattr(a, "alpha", fake(8)), lambda a: setattr(a, "T_exp_out", None),
                lambda a: setattr(a, "dk", 64)):
        a, _ = base_build(B, 4)
        mut(a)
        assert run_build(B, a) != B.OK   # KDA needs g, beta, T_exp_out, dk == dv; takes no alpha
    for mut in (lambda a: setattr(a, "alpha", None), lambda a: setattr(a, "beta", fake(8)),
                lambda a: setattr(a, "T_exp_out", fake(6)), lambda a: setattr(a, "g", fake(8))):
        a, _ = base_build(B, 5)
        mut(a)
        assert run_build(B, a) == B.ERR_INVALID_ARG  # Mamba2 needs alpha only; scalar T, no exponent


def test_build_empty_batch_is_ok_without_gpu(B):
    a, cu = base_build(B, n_seg=0, lengths=())
    assert run_build(B, a, ws=0, ws_ptr=0) == B.OK


def base_compose(B, family=0, d=128, chains=((0, 1), (1,))):
    cu = np.array([0] + list(np.cumsum([len(c) for c in chains])), np.int32)
    idx = np.array([i for c in chains for i in c], np.int32)
    a = B.ComposeArgs()
    a.family, a.n_layers, a.n_heads, a.dk, a.dv, a.n_pairs = family, 2, 2, d, d, 2
    a.T_tab = fake(1) if family != 3 else None
    a.S_tab = fake(2)
    a.n_chains = len(chains)
    a.cu_chain, a.cu_chain_host = fake(3), cu.ctypes.data
    a.seg_idx, a.seg_idx_host = fake(4), idx.ctypes.data
    a.S_out = fake(6)
    return a, (cu, idx)


@pytest.mark.parametrize("mutate,status", [
    (lambda a, k: k[1].__setitem__(0, 2), 1),            # pair index out of range
    (lambda a, k: k[1].__setitem__(0, -1), 1),
    (lambda a, k: k[0].__setitem__(0, 1), 1),            # cu_chain[0] != 0
    (lambda a, k: setattr(a, "T_tab", None), 1),
    (lambda a, k: setattr(a, "S_out", fake(2) + 64), 1), # output overlaps S_tab
    (lambda a, k: setattr(a, "S0", fake(6)), 1),         # output overlaps S0
    (lambda a, k: setattr(a, "dv", 64), 2),
    (lambda a, k: setattr(a, "S_tab", fake(2) + 4), 1),
    (lambda a, k: setattr(a, "T_out", fake(8)), 1),           # GDN T_out needs T_exp_out
    (lambda a, k: setattr(a, "T_exp_out", fake(9)), 1),       # ... and T_exp_out needs T_out
    (lambda a, k: (setattr(a, "T_out", fake(1)), setattr(a, "T_exp_out", fake(9))), 1),  # T_out overlaps T_tab
    (lambda a, k: (setattr(a, "T_out", fake(8)), setattr(a, "T_exp_out", fake(6))), 1),  # T_exp_out overlaps S_out
])
def test_compose_rejections(B, mutate, status):
    a, keep = base_compose(B)
    mutate(a, keep)
    assert B.hypic_compose(a, None) == status


def test_compose_vanilla_rejects_T(B):
    a, keep = base_compose(B, 3)
    a.T_tab = fake(1)
    assert B.hypic_compose(a, None) == B.ERR_INVALID_ARG
    a, keep = base_compose(B, 1)
    a.T_exp_tab = fake(7)
    assert B.hypic_compose(a, None) == B.ERR_INVALID_ARG
    a, keep = base_compose(B, 3)
    a.T_out = fake(8)
    assert B.hypic_compose(a, None) == B.ERR_INVALID_ARG   # vanilla has no transition
    a, keep = base_compose(B, 5)
    a.T_out, a.T_exp_out = fake(8), fake(9)
    assert B.hypic_compose(a, None) == B.ERR_INVALID_ARG   # scalar T: no exponent


def base_seam(B, family=0, d=128, lens=(8, 8)):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    a = B.SeamArgs()
    a.family, a.in_dtype, a.n_layers, a.n_heads, a.dk, a.dv = family, 1, 2, 2, d, d
    a.n_seams, a.n_tokens = len(lens), int(cu[-1])
    a.cu_seam, a.cu_seam_host = fake(0), cu.ctypes.data
    a.q, a.k, a.v = fake(1), fake(2), fake(3)
    if family == 0:
        a.alpha, a.beta = fake(4), fake(5)
    a.state_in, a.state_out, a.o_out = fake(6), fake(6), fake(8)
    return a, cu


@pytest.mark.parametrize("mutate,status", [
    (lambda a, c: setattr(a, "n_tokens", 15), 1),        # cu_seam[-1] != n_tokens
    (lambda a, c: setattr(a, "q", None), 1),
    (lambda a, c: setattr(a, "state_out", None), 1),
    (lambda a, c: setattr(a, "state_out", fake(6) + 64), 1),  # partial overlap
    (lambda a, c: setattr(a, "o_out", fake(6)), 1),      # o_out overlaps the state
    (lambda a, c: setattr(a, "beta", None), 1),
    (lambda a, c: setattr(a, "dk", 48), 2),
])
def test_seam_rejections(B, mutate, status):
    a, cu = base_seam(B)
    mutate(a, cu)
    assert B.hypic_seam_advance(a, None) == status


def base_chain(B, family=0, d=64, chains=((0, 1), (1,)), widths=(8, 0, 3)):
    cu = np.array([0] + list(np.cumsum([len(c) for c in chains])), np.int32)
    idx = np.array([i for c in chains for i in c], np.int32)
    cs = np.concatenate([[0], np.cumsum(widths)]).astype(np.int32)
    a = B.ChainArgs()
    a.family, a.in_dtype, a.n_layers, a.n_heads, a.dk, a.dv, a.n_pairs = family, 1, 2, 2, d, d, 2
    a.T_tab = fake(1) if family != 3 else None
    a.S_tab = fake(2)
    a.n_chains = len(chains)
    a.cu_chain, a.cu_chain_host = fake(3), cu.ctypes.data
    a.seg_idx, a.seg_idx_host = fake(4), idx.ctypes.data
    a.cu_step, a.cu_step_host = fake(5), cs.ctypes.data
    a.n_tokens = int(cs[-1])
    a.q, a.k, a.v = fake(7), fake(8), fake(9)
    if family == 0:
        a.alpha, a.beta = fake(10), fake(11)
    a.S_out, a.o_out = fake(12), fake(13)
    return a, (cu, idx, cs)


@pytest.mark.parametrize("mutate,status", [
    (lambda a, k: setattr(a, "n_tokens", 10), 1),         # cu_step[-1] != n_tokens
    (lambda a, k: k[2].__setitem__(1, -1), 1),            # cu_step decreases
    (lambda a, k: k[1].__setitem__(0, 2), 1),             # pair index out of range
    (lambda a, k: setattr(a, "q", None), 1),
    (lambda a, k: setattr(a, "beta", None), 1),
    (lambda a, k: setattr(a, "o_out", fake(12)), 1),      # o_out overlaps S_out
    (lambda a, k: setattr(a, "dk", 48), 2),
])
def test_chain_rejections(B, mutate, status):
    a, keep = base_chain(B)
    mutate(a, keep)
    assert B.hypic_reuse_chain(a, fake(20), 1 << 24, None) == status
    assert B.hypic_chain_workspace_size(a) == 0


def test_chain_step_by_step_path_needs_its_workspace(B):
    """d = 64 runs step by step through a workspace of two states of one
    chain plus the step indices; without it the call is refused before any
    GPU work."""
    a, keep = base_chain(B)
    need = B.hypic_chain_workspace_size(a)
    assert need >= 2 * 4 * 64 * 64 * 2 * 2
    assert B.hypic_reuse_chain(a, None, 0, None) == B.ERR_WORKSPACE
    assert B.hypic_reuse_chain(a, fake(20), need - 1, None) == B.ERR_WORKSPACE
    assert B.hypic_reuse_chain(a, fake(20) + 16, need, None) == B.ERR_WORKSPACE  # not 256-byte aligned


def base_rope(B, family=0, d=64, n_pairs=3):
    a = B.RopeArgs()
    a.family, a.n_layers, a.n_heads, a.dk, a.dv, a.n_pairs = family, 2, 2, d, d, n_pairs
    a.rotary_dim, a.base = d, 10000.0
    a.delta, a.S = fake(1), fake(2)
    a.T = fake(3) if family == 0 else None
    return a


@pytest.mark.parametrize("mutate,status", [
    (lambda a: setattr(a, "family", 2), 2),            # GLA: gates do not commute with R
    (lambda a: setattr(a, "family", 4), 2),            # KDA: same
    (lambda a: setattr(a, "rotary_dim", 63), 1),       # odd
    (lambda a: setattr(a, "rotary_dim", 0), 1),
    (lambda a: setattr(a, "rotary_dim", 66), 1),       # > dk
    (lambda a: setattr(a, "base", 0.0), 1),
    (lambda a: setattr(a, "base", float("nan")), 1),
    (lambda a: setattr(a, "T", None), 1),              # GDN needs T
    (lambda a: setattr(a, "delta", None), 1),
    (lambda a: setattr(a, "S", fake(3) + 256), 1),     # S overlaps T
    (lambda a: setattr(a, "S", fake(2) + 8), 1),       # misaligned
])
def test_rope_rejections(B, mutate, status):
    a = base_rope(B)
    mutate(a)
    assert B.hypic_rope_rerotate(a, None) == status
    assert B.lib.hypic_last_error_detail().decode()


def test_rope_scalar_family_takes_no_T_and_empty_is_ok(B):
    a = base_rope(B, family=1)
    a.T = fake(3)
    assert B.hypic_rope_rerotate(a, None) == B.ERR_INVALID_ARG
    a = base_rope(B, family=1, n_pairs=0)
    assert B.hypic_rope_rerotate(a, None) == B.OK


def base_conv(B, lens=(8, 8, 0)):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    a = B.ConvArgs()
    a.n_layers, a.C, a.K, a.n_seams, a.n_tokens = 2, 64, 4, len(lens), int(cu[-1])
    a.cu_seam, a.cu_seam_host = fake(0), cu.ctypes.data
    a.x, a.w, a.y, a.act = fake(1), fake(2), fake(3), 1
    return a, cu


@pytest.mark.parametrize("mutate,status", [
    (lambda a, c: setattr(a, "K", 0), 2),
    (lambda a, c: setattr(a, "K", 17), 2),
    (lambda a, c: setattr(a, "act", 2), 1),
    (lambda a, c: setattr(a, "n_tokens", 15), 1),      # cu_seam[-1] != n_tokens
    (lambda a, c: c.__setitem__(0, 1), 1),             # cu_seam[0] != 0
    (lambda a, c: setattr(a, "x", None), 1),
    (lambda a, c: setattr(a, "y", fake(1) + 16), 1),   # y overlaps x
    (lambda a, c: setattr(a, "w", fake(2) + 4), 1),    # misaligned
])
def test_conv_rejections(B, mutate, status):
    a, cu = base_conv(B)
    mutate(a, cu)
    assert B.hypic_conv_warmup(a, None) == status
    assert B.lib.hypic_last_error_detail().decode()


def test_build_workspace_caps_kda_chunk_tables(B):
    """The reported KDA workspace holds at most 4 GiB of chunk tables (128 KB per
    chunk, layer and head), and never fewer than two chunks' tables, so that a
    long request is built in batches and a segment longer than a batch in parts."""
    pair = 128 * 1024
    for L, H, lengths, chunks in (
        (30, 32, (640000, 64), (4 << 30) // (30 * 32 * pair)),   # 10,001 chunks, 34 fit 4 GiB
        (100, 1000, (640, 64), 2),                               # one chunk of tables > 4 GiB
        (1, 2, (64, 80), 3),                                     # everything fits: all 3 chunks
    ):
        a, keep = base_build(B, 4, lengths=lengths)
        a.n_layers, a.n_heads = L, H
        a.in_dtype = 0                    # fp32 inputs: the CUDA-core kernel, plan only
        plan = B.hypic_build_workspace_size(a)
        a.in_dtype = 1
        need = B.hypic_build_workspace_size(a)
        LH = L * H
        assert chunks * LH * pair <= need - plan < (chunks + 1) * LH * pair, (L, H, lengths)
        assert run_build(B, a, ws=need - 1) == B.ERR_WORKSPACE


def test_build_workspace_holds_kda_chunk_tables(B):
    """KDA at d = 128 with bf16 k and v: the reported workspace also holds the
    chunk tables of its tensor-core path (T and S of every 64-token chunk,
    layer and head: 128 KB each); other dims and dtypes need only the plan."""
    plan_args, keep0 = base_build(B, 0)
    plan = B.hypic_build_workspace_size(plan_args)
    a, keep = base_build(B, 4)            # bodies of 64 and 80 tokens: 1 + 2 chunks, 1 layer x 2 heads
    need = B.hypic_build_workspace_size(a)
    tables = 3 * 2 * 128 * 1024
    assert plan + tables <= need < plan + tables + 8192
    assert run_build(B, a, ws=need - 1) == B.ERR_WORKSPACE
    a.in_dtype = 0                        # fp32 inputs: the CUDA-core kernel
    assert B.hypic_build_workspace_size(a) == plan
    a.in_dtype, a.dk, a.dv = 1, 64, 64    # d = 64: the CUDA-core kernel
    assert B.hypic_build_workspace_size(a) == plan
    sk = np.array([64, 80], np.int32)     # every body empty: nothing to tabulate
    a.dk, a.dv = 128, 128
    a.seam_skip, a.seam_skip_host = fake(8), sk.ctypes.data
    assert B.hypic_build_workspace_size(a) == plan
