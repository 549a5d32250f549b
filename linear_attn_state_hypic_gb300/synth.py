"""Seeded synthetic inputs for the HYPIC linear-attention state path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the fp64 oracle (tests) and the CUDA library
(tests, bench) can consume what it makes.  Draw order is fixed per workload
(lengths, k, v, q, alpha, beta / g) from ``numpy.random.default_rng(seed)``,
except for the 100k-token workload, which is drawn on the GPU with a seeded
torch generator one layer at a time.

Workloads (shapes of the pages' serving workloads: segments of 512-2048
tokens, tens to ~100 segments, ~30 linear layers, 128-dim heads):

* ``gdn_tiny``      1 layer, 1 head, d=16, fp32, 2 x 64 tokens.
* ``decay_small``   1 layer, 8 heads, d=64, fp32, 8 x 256 tokens; RetNet
  gamma_h = 1 - 2^(-5-h), GLA g = sigmoid(N(2,1)) per key dim.
* ``gdn_ragged``    1 layer, 32 heads, d=128, bf16 q/k/v, 32 segments with
  lengths uniform in [512, 2048].
* ``compose_table`` 30 layers x 32 heads, d=128, fp32 pair table of 128
  segments, 16 chains of 64 random distinct segments.
* ``long_request``  30 layers x 32 heads, d=128, bf16, 100,000 tokens in
  segments of uniform [512, 2048] length (the last takes the remainder), an
  8-token seam at each internal segment start.

k is drawn N(0,1) and L2-normalised per token and head; q likewise; v is
N(0,1).  GDN gates: alpha ~ U(0.85, 1), beta ~ U(0, 1) ("faithful"), or the
high-retention variant alpha ~ U(0.999, 1), beta ~ U(0, 0.1), whose transition
products keep a norm near 1 so that errors in T are visible downstream.
bf16 values are produced by round-to-nearest-even from float32 and handed to
the oracle as their exact float32 upcast.
"""
from __future__ import annotations

import numpy as np

# alpha range, beta range.  "faithful" and "highret" are the two gate mixes of
# the build workload; "middecay" and "fastdecay" (a chunk of 64 tokens decays
# by ~2^-32 and ~2^-115) reach the builds' renormalisation and strong-decay
# branches.
GATES = {"faithful": (0.85, 1.0, 0.0, 1.0), "highret": (0.999, 1.0, 0.0, 0.1),
         "middecay": (0.5, 1.0, 0.0, 1.0), "fastdecay": (0.05, 0.6, 0.0, 1.0)}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = x.view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    x /= np.linalg.norm(x, axis=-1, keepdims=True)
    return x.astype(np.float32)


def ragged_lengths(rng, n_seg, lo, hi):
    return rng.integers(lo, hi + 1, size=n_seg)


def cu_from_lengths(lengths):
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    return cu


def gdn_tiny(seed=0):
    rng = np.random.default_rng(seed)
    lengths = np.array([64, 64])
    n = int(lengths.sum())
    k = _unit_rows(rng, (1, n, 1, 16))
    v = rng.standard_normal((1, n, 1, 16)).astype(np.float32)
    alpha = rng.uniform(0.9, 1.0, (1, n, 1)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (1, n, 1)).astype(np.float32)
    return dict(family="gdn", dtype="f32", k=k, v=v, alpha=alpha, beta=beta,
                cu_seqlens=cu_from_lengths(lengths))


def decay_small(seed=0, n_seg=8, seg_len=256, H=8, d=64):
    rng = np.random.default_rng(seed)
    lengths = np.full(n_seg, seg_len)
    n = int(lengths.sum())
    k = _unit_rows(rng, (1, n, H, d))
    v = rng.standard_normal((1, n, H, d)).astype(np.float32)
    q = _unit_rows(rng, (1, n, H, d))
    gamma = (1.0 - 2.0 ** (-5.0 - np.arange(H, dtype=np.float64))).astype(np.float32)[None, :]
    g = (1.0 / (1.0 + np.exp(-rng.normal(2.0, 1.0, (1, n, H, d))))).astype(np.float32)
    return dict(dtype="f32", k=k, v=v, q=q, gamma=gamma, g=g,
                cu_seqlens=cu_from_lengths(lengths))


def gdn_gates(rng, shape, variant="faithful"):
    alo, ahi, blo, bhi = GATES[variant]
    alpha = rng.uniform(alo, ahi, shape).astype(np.float32)
    beta = rng.uniform(blo, bhi, shape).astype(np.float32)
    return alpha, beta


def gdn_ragged(seed=0, n_seg=32, H=32, d=128, lo=512, hi=2048, variant="faithful",
               lengths=None, n_layers=1, with_q=False, dtype="bf16"):
    """Ragged batch of GDN segments (bf16 k/v by default)."""
    rng = np.random.default_rng(seed)
    if lengths is None:
        lengths = ragged_lengths(rng, n_seg, lo, hi)
    lengths = np.asarray(lengths)
    n = int(lengths.sum())
    k = _unit_rows(rng, (n_layers, n, H, d))
    v = rng.standard_normal((n_layers, n, H, d)).astype(np.float32)
    q = _unit_rows(rng, (n_layers, n, H, d)) if with_q else None
    if dtype == "bf16":
        k, v = round_bf16(k), round_bf16(v)
        q = round_bf16(q) if q is not None else None
    alpha, beta = gdn_gates(rng, (n_layers, n, H), variant)
    out = dict(family="gdn", dtype=dtype, k=k, v=v, alpha=alpha, beta=beta,
               cu_seqlens=cu_from_lengths(lengths))
    if q is not None:
        out["q"] = q
    return out


def compose_chains(seed=0, n_pairs=128, n_chains=16, steps=64, n_layers=30, H=32, d=128,
                   with_tables=True):
    """Chains of distinct random pair indices, start states, and S_C draws.

    Chains 0..n_chains/2-1 start from zero, the rest from S0 ~ N(0,1)/sqrt(d).
    The T_C of the table are not drawn here: they are the build's outputs on
    segments drawn by ``gdn_ragged``.
    """
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(n_pairs)[:steps] for _ in range(n_chains)]).astype(np.int32)
    cu = (np.arange(n_chains + 1) * steps).astype(np.int32)
    S0 = (rng.standard_normal((n_chains, n_layers, H, d, d)) / np.sqrt(d)).astype(np.float32)
    S0[: n_chains // 2] = 0.0
    S_tab = None
    if with_tables:
        S_tab = (rng.standard_normal((n_pairs, n_layers, H, d, d)) / np.sqrt(d)).astype(np.float32)
    return dict(cu_chain=cu, seg_idx=idx.reshape(-1), S0=S0, S_tab=S_tab,
                zero_start=np.arange(n_chains) < n_chains // 2)


def long_request_lengths(seed=0, n_tokens=100_000, lo=512, hi=2048):
    """Segment lengths drawn U{lo..hi} until the total reaches n_tokens; the
    last segment takes the remainder (it may be shorter than lo)."""
    rng = np.random.default_rng(seed)
    out = []
    total = 0
    while total < n_tokens:
        L = int(rng.integers(lo, hi + 1))
        L = min(L, n_tokens - total)
        out.append(L)
        total += L
    return np.array(out, dtype=np.int64)


def long_request_device(seed=0, n_layers=30, H=32, d=128, n_tokens=100_000, seam_w=8,
                        variant="faithful", device="cuda"):
    """The 100k-token request, drawn on the device layer by layer.

    Returns a dict of torch tensors: k, v bf16 [L][N][H][d]; alpha, beta fp32
    [L][N][H]; q_seam bf16 [L][n_seam_tok][H][d] for the seam tokens only;
    plus host arrays cu_seqlens, seam_skip (0 for the first segment, seam_w
    for the others) and seam_tok (token index of every seam token, in order).
    """
    import torch

    lengths = long_request_lengths(seed, n_tokens)
    cu = cu_from_lengths(lengths)
    n_seg = len(lengths)
    skip = np.full(n_seg, seam_w, dtype=np.int32)
    skip[0] = 0
    skip = np.minimum(skip, lengths.astype(np.int32))
    seam_tok = np.concatenate([np.arange(cu[i], cu[i] + skip[i]) for i in range(1, n_seg)]).astype(np.int64)
    alo, ahi, blo, bhi = GATES[variant]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    k = torch.empty((n_layers, n_tokens, H, d), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    q_seam = torch.empty((n_layers, len(seam_tok), H, d), dtype=torch.bfloat16, device=device)
    alpha = torch.empty((n_layers, n_tokens, H), dtype=torch.float32, device=device)
    beta = torch.empty_like(alpha)
    for layer in range(n_layers):
        x = torch.randn((n_tokens, H, d), generator=gen, device=device)
        k[layer] = (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        v[layer] = torch.randn((n_tokens, H, d), generator=gen, device=device).to(torch.bfloat16)
        x = torch.randn((len(seam_tok), H, d), generator=gen, device=device)
        q_seam[layer] = (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        alpha[layer] = torch.rand((n_tokens, H), generator=gen, device=device) * (ahi - alo) + alo
        beta[layer] = torch.rand((n_tokens, H), generator=gen, device=device) * (bhi - blo) + blo
        del x
    return dict(k=k, v=v, alpha=alpha, beta=beta, q_seam=q_seam, cu_seqlens=cu,
                seam_skip=skip, seam_tok=seam_tok, lengths=lengths)
