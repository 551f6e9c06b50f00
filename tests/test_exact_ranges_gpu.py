"""Bit-exact index ranges on the production path (bf16, d = 128: the tensor-core
kernels), read off outputs that are exact small integers or exact reciprocals.

Window (papernotes.org note on Lizard, 关键设计: Anchor Window Attention): with q = k = 0
every visible logit is 0, so a query i averages the values of exactly S_i = M meta rows
plus the keys [max(0, i-W+1), i].  With one-hot values the output reveals the set.

Chunk partition ("Lizard", arXiv 2507.09025, Method: the chunkwise form; chunk c covers
tokens [128 c, min(128 (c+1), L))): with log gamma = 0, phi_q = phi_k = e_0 and one-hot
values, the GLA output of token t counts the earlier tokens per value column; a token
dropped, doubled or assigned to the wrong side of a chunk boundary changes an integer.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import NAMES, TOL, gpu_bwd, gpu_fwd, rel_l2

pytestmark = pytest.mark.gpu

L = 300  # three 128-token chunks, the last one ragged
D = 128


def _zero_inputs(M, seed, with_dy=False):
    x = synth.make_fwd_inputs(1, 1, L, D, D, M, "bf16", "plain", seed=seed, with_dy=with_dy)
    for n in ("q", "k", "phi_q", "meta_v"):
        x[n][:] = 0
    return x


def _onehot_rows(n):
    e = np.zeros((n, D), dtype=np.float32)
    e[np.arange(n), np.arange(n) % D] = 1.0
    return e


@pytest.mark.parametrize("M", [0, 4, 16])
@pytest.mark.parametrize("W", [1, 63, 64, 65, 66, 127, 128, 129])
def test_window_range_exact_tensor_core(W, M):
    """rint(y_i (M + |S_i|)) counts, per value column c, the keys j of S_i with
    j mod 128 = c: at most one for W <= 128, two at one column for W = 129."""
    x = _zero_inputs(M, seed=40 + W + M)
    x["v"][0, 0] = _onehot_rows(L)
    y, _ = gpu_fwd(x, W, "bf16")
    for i in range(L):
        lo = max(0, i - W + 1)
        cnt = np.bincount(np.arange(lo, i + 1) % D, minlength=D).astype(np.float64)
        got = y[0, 0, i].astype(np.float64) * (M + i + 1 - lo)
        np.testing.assert_array_equal(np.rint(got), cnt, err_msg=f"query {i}")
        assert np.max(np.abs(got - cnt)) < 0.02, i


@pytest.mark.parametrize("M", [0, 4, 16])
@pytest.mark.parametrize("W", [1, 63, 64, 65])
def test_window_backward_key_range_exact(W, M):
    """One-hot upstream gradients dy_i = e_{i mod 128} and phi_q = 0 (no GLA term): the
    value gradient of key j is sum over the queries i that see j of dy_i / (M + |S_i|),
    so (M + |S_i|) dv_j[i mod 128] is 1 exactly for those queries and 0 elsewhere."""
    x = _zero_inputs(M, seed=60 + W + M, with_dy=True)
    x["dy"][0, 0] = _onehot_rows(L)
    g = gpu_bwd(x, W, "bf16")
    dv = g["d_v"][0, 0].astype(np.float64)
    for j in range(L):
        mult = np.zeros(D)
        for i in range(j, min(L, j + W)):
            mult[i % D] = M + min(i + 1, W)
        got = dv[j] * mult
        np.testing.assert_array_equal(np.rint(got), (mult > 0).astype(np.float64), err_msg=f"key {j}")
        assert np.all(dv[j][mult == 0] == 0), j


@pytest.mark.parametrize("M", [4, 16])
@pytest.mark.parametrize("W", [1, 63, 64, 65])
def test_window_backward_query_range_exact(W, M):
    """Window values e_0, meta values 0, dy_i = e_0, keys k_j = e_{j mod 128}, q = 0: the
    logit gradient is M / n_i^2 for every visible token key (n_i = M + |S_i|), so
    n_i^2 dq_i / (scale M) is the indicator of S_i taken mod 128."""
    x = _zero_inputs(M, seed=80 + W + M, with_dy=True)
    x["k"][0, 0] = _onehot_rows(L)
    x["v"][:] = 0
    x["v"][0, 0, :, 0] = 1.0
    x["meta_k"][:] = 0
    x["dy"][:] = 0
    x["dy"][0, 0, :, 0] = 1.0
    g = gpu_bwd(x, W, "bf16")
    scale = 1.0 / np.sqrt(D)
    dq = g["d_q"][0, 0].astype(np.float64)
    for i in range(L):
        lo = max(0, i - W + 1)
        n = M + i + 1 - lo
        ind = np.bincount(np.arange(lo, i + 1) % D, minlength=D).astype(np.float64)
        got = dq[i] * n * n / (scale * M)
        np.testing.assert_array_equal(np.rint(got), ind, err_msg=f"query {i}")


@pytest.mark.parametrize("W", [40, 100])
def test_window_branch_alone_random(W):
    """phi_q = 0 leaves y = alpha y_win: the window branch compared on its own at the bf16
    tolerance, once per key-band size (W <= 65 and W <= 129)."""
    x = synth.make_fwd_inputs(2, 2, L, D, D, 4, "bf16", "plain", seed=100 + W)
    x["phi_q"][:] = 0
    y, _ = gpu_fwd(x, W, "bf16", alpha=0.7)
    ref = oracle.fwd(*(x[n] for n in NAMES), W=W, alpha=0.7)
    assert rel_l2(y, ref["y"]) <= TOL["bf16"]


def _count_inputs(seed, with_dy=False):
    x = synth.make_fwd_inputs(2, 2, L, D, D, 4, "bf16", "plain", seed=seed, with_dy=with_dy)
    x["log_gamma"][:] = 0
    for n in ("phi_q", "phi_k"):
        x[n][:] = 0
        x[n][..., 0] = 1.0
    x["v"][:] = _onehot_rows(L)
    if with_dy:
        x["dy"][:] = _onehot_rows(L)
    return x


def test_chunk_partition_exact_forward():
    """y_t[c] = #{s <= t : s mod 128 = c} (alpha = 0 drops the window branch): integers,
    exact in bf16, equal to the oracle's element by element."""
    x = _count_inputs(seed=120)
    y, hf = gpu_fwd(x, 64, "bf16", alpha=0.0, want_hf=True)
    ref = oracle.fwd(*(x[n] for n in NAMES), W=64, alpha=0.0, want_state=True)
    t = np.arange(L)
    expect = np.stack([np.bincount(t[: i + 1] % D, minlength=D) for i in range(L)])
    np.testing.assert_array_equal(ref["y"][0, 0], expect)
    np.testing.assert_array_equal(y, ref["y"])
    np.testing.assert_array_equal(hf, ref["h_final"])


def test_chunk_partition_exact_backward():
    """dy_t = e_{t mod 128} as well: every GLA gradient is an integer (d v_s counts later
    tokens per column, d phi_q / d phi_k count matching pairs, d log gamma their suffix
    differences), equal to the oracle's element by element."""
    x = _count_inputs(seed=121, with_dy=True)
    g = gpu_bwd(x, 64, "bf16", alpha=0.0)
    ref = oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=64, alpha=0.0)
    for n in ("d_phi_q", "d_phi_k", "d_v", "d_log_gamma"):
        assert np.all(ref[n] == np.rint(ref[n])), n
        np.testing.assert_array_equal(g[n], ref[n], err_msg=n)
