"""Forward pass: CUDA path vs the fp64 oracle on the same seeded inputs.

Tolerance: max relative-L2 error per output tensor of 1e-5 (fp32 inputs) or 2e-2 (bf16
inputs; fp32 state and accumulation).  Index ranges are checked exactly."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import NAMES, TOL, gpu_fwd, rel_l2

pytestmark = pytest.mark.gpu


def _oracle(x, W, alpha=1.0, h0=None, want_state=False, heads=None):
    if heads is not None:  # sampled (b, h) units, each an independent problem
        outs = []
        for (b, h) in heads:
            sub = {n: x[n][b:b + 1, h:h + 1] for n in NAMES if n not in ("meta_k", "meta_v")}
            r = oracle.fwd(*(sub[n] for n in ("phi_q", "phi_k", "v", "log_gamma", "q", "k")),
                           x["meta_k"][h:h + 1], x["meta_v"][h:h + 1], W=W, alpha=alpha)
            outs.append(r["y"][0, 0])
        return outs
    return oracle.fwd(*(x[n] for n in NAMES), W=W, alpha=alpha, h0=h0, want_state=want_state)


def test_tiny_fp32_workload():
    """The tiny fp32 workload: B=1, H=2, L=256, d=64, W=64, M=4."""
    w = synth.WORKLOADS["tiny_fp32"]
    x = synth.workload_inputs("tiny_fp32")
    y, _ = gpu_fwd(x, w["W"], "f32")
    ref = _oracle(x, w["W"])
    assert rel_l2(y, ref["y"]) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,L,d,W,M,alpha", [
    (2, 3, 777, 128, 64, 4, 1.0),    # several chunks, ragged tail
    (1, 2, 1000, 64, 37, 3, 0.7),    # d = 64, odd window
    (1, 1, 130, 128, 128, 8, 1.0),   # W = 128, M = 8
    (2, 1, 65, 128, 1, 0, 1.5),      # W = 1, no meta
    (1, 2, 40, 64, 64, 2, 1.0),      # W >= L, single partial chunk
    (1, 1, 1, 128, 64, 4, 1.0),      # one token
])
def test_fwd_matches_oracle(dtype, B, H, L, d, W, M, alpha):
    x = synth.make_fwd_inputs(B, H, L, d, d, M, dtype, "plain", seed=100 + L + d + W)
    y, _ = gpu_fwd(x, W, dtype, alpha=alpha)
    ref = _oracle(x, W, alpha)
    err = rel_l2(y, ref["y"])
    assert err <= TOL[dtype], err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fwd_initial_and_final_state(dtype):
    B, H, L, d, W, M = 1, 2, 300, 128, 64, 4
    x = synth.make_fwd_inputs(B, H, L, d, d, M, dtype, "bimodal", seed=7)
    rng = np.random.default_rng(8)
    h0 = (0.1 * rng.standard_normal((B, H, d, d))).astype(np.float32)
    y, hf = gpu_fwd(x, W, dtype, h0=h0, want_hf=True)
    ref = _oracle(x, W, h0=h0, want_state=True)
    assert rel_l2(y, ref["y"]) <= TOL[dtype]
    assert rel_l2(hf, ref["h_final"]) <= TOL[dtype]


def test_fwd_empty_sequence_returns_h0():
    x = synth.make_fwd_inputs(1, 2, 0, 64, 64, 2, "f32", "plain", seed=9)
    h0 = np.random.default_rng(9).standard_normal((1, 2, 64, 64)).astype(np.float32)
    y, hf = gpu_fwd(x, 8, "f32", h0=h0, want_hf=True)
    assert y.size == 0
    np.testing.assert_array_equal(hf, h0)


@pytest.mark.parametrize("W,M", [(1, 0), (5, 2), (64, 4), (100, 1)])
def test_window_index_range_exact(W, M):
    """q = k = 0, meta_v = 0, v_j = e_j and phi_q = 0: y_i * (M + |S_i|) is exactly the
    indicator of S_i = [max(0, i-W+1), i] after rounding to the nearest integer."""
    L, d = 128, 128
    x = synth.make_fwd_inputs(1, 1, L, d, d, M, "f32", "plain", seed=10)
    x["q"][:] = 0
    x["k"][:] = 0
    x["phi_q"][:] = 0
    x["meta_v"][:] = 0
    x["v"][:] = np.eye(L, dtype=np.float32)[None, None]
    y, _ = gpu_fwd(x, W, "f32")
    for i in range(L):
        lo = max(0, i - W + 1)
        ind = np.zeros(L)
        ind[lo:i + 1] = 1
        got = y[0, 0, i] * (M + i + 1 - lo)
        np.testing.assert_array_equal(np.rint(got), ind)
        assert np.max(np.abs(got - ind)) < 1e-5


def test_fwd_is_deterministic():
    x = synth.make_fwd_inputs(1, 4, 513, 128, 128, 4, "bf16", "plain", seed=11)
    a, _ = gpu_fwd(x, 64, "bf16")
    b, _ = gpu_fwd(x, 64, "bf16")
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("name,heads", [
    ("llama3_8b_fwd", [(0, 0), (0, 17), (0, 31)]),
    ("long_ctx_64k", [(0, 5)]),
])
def test_full_size_workload_sampled_heads(name, heads):
    """Full-size workloads in the shipped launch configuration; the oracle recomputes a
    few (batch, head) units, which are independent problems."""
    w = synth.WORKLOADS[name]
    x = synth.workload_inputs(name)
    y, _ = gpu_fwd(x, w["W"], w["dtype"])
    refs = _oracle(x, w["W"], heads=heads)
    for (b, h), ref in zip(heads, refs):
        err = rel_l2(y[b, h], ref)
        assert err <= TOL[w["dtype"]], (b, h, err)
    assert np.all(np.isfinite(y))
