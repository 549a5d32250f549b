"""GPU parity of hypic_conv_warmup (the conv-state warm-up of seam windows)
against the fp64 oracle, and its purpose: with the new prefix's last K-1
inputs as history, a window's outputs equal the causal convolution of the
whole sequence."""
import numpy as np
import pytest

from oracle import oracle as orc
from tests.helpers import assert_rel, dev, host

pytestmark = pytest.mark.gpu

TOL = 1e-6  # fp32 sums of K products against fp64 (plus SiLU), per output row


@pytest.fixture(scope="module")
def B():
    from linear_attn_state_hypic_gb300 import binding
    return binding


@pytest.mark.parametrize("K,act,with_bias,with_hist", [(4, 1, True, True), (4, 0, False, True), (2, 1, True, False),
                                                       (1, 0, True, True), (7, 1, False, True)])
def test_conv_warmup_matches_oracle(B, K, act, with_bias, with_hist):
    rng = np.random.default_rng(K * 10 + act)
    L, C = 3, 96
    lens = [8, 0, 1, 8, 13]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = int(cu[-1])
    x = rng.standard_normal((L, n, C)).astype(np.float32)
    w = (rng.standard_normal((L, C, K)) / np.sqrt(K)).astype(np.float32)
    b = rng.standard_normal((L, C)).astype(np.float32) if with_bias else None
    hist = rng.standard_normal((len(lens), L, max(K - 1, 1), C)).astype(np.float32)[:, :, :K - 1] if with_hist else None
    hist = None if hist is None else np.ascontiguousarray(hist)
    y = B.conv_warmup(dev(x), cu, dev(w), hist=None if hist is None or K == 1 else dev(hist), bias=dev(b), act=act)
    B.check_device()
    ref = orc.conv(x, cu, w, hist=None if K == 1 else hist, bias=b, act=act)
    assert_rel(host(y), ref, TOL, axes=(-1,), what="conv warm-up")


def test_warmup_with_prefix_history_equals_whole_sequence(B):
    """Windows of a request at the starts of its segments, each given the
    previous segment's last K-1 inputs as history: outputs equal the conv of
    the whole request at those tokens."""
    rng = np.random.default_rng(3)
    L, C, K, n = 2, 64, 4, 300
    xs = rng.standard_normal((L, n, C)).astype(np.float32)
    w = (rng.standard_normal((L, C, K)) / 2).astype(np.float32)
    b = rng.standard_normal((L, C)).astype(np.float32)
    seg_starts = [0, 70, 150, 151, 240]
    win = 8
    tok = np.concatenate([np.arange(s, min(s + win, n)) for s in seg_starts])
    cu = np.concatenate([[0], np.cumsum([min(win, n - s) for s in seg_starts])]).astype(np.int32)
    hist = np.zeros((len(seg_starts), L, K - 1, C), np.float32)
    for r, s0 in enumerate(seg_starts):
        for j in range(K - 1):
            if s0 - (K - 1) + j >= 0:
                hist[r, :, j] = xs[:, s0 - (K - 1) + j]
    y = B.conv_warmup(dev(np.ascontiguousarray(xs[:, tok])), cu, dev(w), hist=dev(hist), bias=dev(b), act=1)
    B.check_device()
    full = orc.conv(xs, [0, n], w, bias=b, act=1)
    assert_rel(host(y), full[:, tok], TOL, axes=(-1,), what="warm-up vs whole-sequence conv")
