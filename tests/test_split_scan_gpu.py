"""Split state scans: with few (batch, head) units and many chunks, the state and adjoint
scans cut each unit's chunks into segments scanned in parallel and joined with the
associative combine ("Lizard", arXiv 2507.09025, Preliminaries: recurrent form).  These
shapes take that path on the tensor-core kernels (bf16, d = 128); the launch counts
show it."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import NAMES, TOL, gpu_fwd, rel_l2

pytestmark = pytest.mark.gpu

GRADS = ("d_phi_q", "d_phi_k", "d_v", "d_log_gamma", "d_q", "d_k", "d_meta_k", "d_meta_v", "d_h0")


def _run_bwd(x, W, h0, fwd_ws_from_forward):
    import torch
    import hybrid_gated_linear_gb300 as lz
    from gpu_util import code, host, to_dev
    B, H, L, d = x["phi_q"].shape
    M = x["meta_k"].shape[1]
    t = to_dev({n: x[n] for n in NAMES + ("dy",)}, "bf16")
    h0t = torch.from_numpy(h0).cuda()
    dims = lz.lizard_dims(B, H, L, d, d, M, code("bf16"), 0.0)
    wf = None
    if fwd_ws_from_forward:
        wf = torch.zeros(lz.lizard_fwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
        y = torch.empty(B, H, L, d, dtype=torch.bfloat16, device="cuda")
        lz.lizard_attn_fwd(dims, *(t[n] for n in NAMES), W, 1.0, y, h0t, None, wf)
        assert lz.lizard_check_device_errors(wf) == 0
    wb = torch.zeros(lz.lizard_bwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
    g = {n: torch.empty(B, H, L, d, dtype=torch.bfloat16, device="cuda")
         for n in ("d_phi_q", "d_phi_k", "d_v", "d_q", "d_k")}
    g["d_log_gamma"] = torch.empty(B, H, L, d, dtype=torch.float32, device="cuda")
    g["d_meta_k"] = torch.empty(H, M, d, dtype=torch.float32, device="cuda")
    g["d_meta_v"] = torch.empty(H, M, d, dtype=torch.float32, device="cuda")
    g["d_h0"] = torch.empty(B, H, d, d, dtype=torch.float32, device="cuda")
    lz.lizard_attn_bwd(dims, *(t[n] for n in NAMES), W, 1.0, h0t, t["dy"], g["d_phi_q"],
                       g["d_phi_k"], g["d_v"], g["d_log_gamma"], g["d_q"], g["d_k"],
                       g["d_meta_k"], g["d_meta_v"], g["d_h0"], wb, fwd_workspace=wf)
    launches = lz.lizard_last_launch_count()
    assert lz.lizard_check_device_errors(wb) == 0
    return {n: host(v) for n, v in g.items()}, launches


@pytest.mark.parametrize("gate,L", [("slow", 3000), ("bimodal", 3000), ("plain", 2900)])
def test_split_forward_matches_oracle(gate, L):
    """B=1, H=2: L=3000 gives 24 chunks of 128 tokens for 8 scan CTAs, split in 3
    segments of 8; L=2900 gives 23 chunks in segments of 12 and 11 with a ragged last
    chunk.  y and h_final from a nonzero h0 against the oracle."""
    B, H, d, W, M = 1, 2, 128, 64, 4
    x = synth.make_fwd_inputs(B, H, L, d, d, M, "bf16", gate, seed=800, with_dy=False)
    h0 = (0.1 * np.random.default_rng(801).standard_normal((B, H, d, d))).astype(np.float32)
    y, hf = gpu_fwd(x, W, "bf16", h0=h0, want_hf=True)
    ref = oracle.fwd(*(x[n] for n in NAMES), W=W, h0=h0, want_state=True)
    errs = {"y": rel_l2(y, ref["y"]), "h_final": rel_l2(hf, ref["h_final"])}
    assert max(errs.values()) <= TOL["bf16"], errs


def test_split_forward_launches_the_join():
    """the header reset, prep, scan, join, fix-up, the chunk kernel and the wide-chunk
    recomputation: seven launches when split, five not."""
    import torch
    import hybrid_gated_linear_gb300 as lz
    from gpu_util import code, to_dev
    counts = {}
    for H, L in ((2, 3000), (2, 900)):
        x = synth.make_fwd_inputs(1, H, L, 128, 128, 4, "bf16", "plain", seed=802)
        t = to_dev({n: x[n] for n in NAMES}, "bf16")
        dims = lz.lizard_dims(1, H, L, 128, 128, 4, code("bf16"), 0.0)
        ws = torch.zeros(lz.lizard_fwd_workspace_bytes(dims, 64), dtype=torch.uint8, device="cuda")
        y = torch.empty(1, H, L, 128, dtype=torch.bfloat16, device="cuda")
        lz.lizard_attn_fwd(dims, *(t[n] for n in NAMES), 64, 1.0, y, None, None, ws)
        counts[L] = lz.lizard_last_launch_count()
        assert lz.lizard_check_device_errors(ws) == 0
    assert counts == {3000: 7, 900: 5}, counts


@pytest.mark.parametrize("L", [3000, 2900])
def test_split_backward_matches_oracle_with_and_without_the_forward_context(L):
    """The adjoint scan alone (with the forward's context) and both scans (without) split;
    every gradient, d_h0 included, against the oracle, and the two runs bitwise equal."""
    B, H, d, W, M = 1, 2, 128, 64, 4
    x = synth.make_fwd_inputs(B, H, L, d, d, M, "bf16", "slow", seed=810, with_dy=True)
    h0 = (0.1 * np.random.default_rng(811).standard_normal((B, H, d, d))).astype(np.float32)
    a, na = _run_bwd(x, W, h0, fwd_ws_from_forward=False)
    b, nb = _run_bwd(x, W, h0, fwd_ws_from_forward=True)
    ref = oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=W, h0=h0, want_dh0=True)
    errs = {n: rel_l2(b[n], ref[n]) for n in GRADS}
    assert max(errs.values()) <= TOL["bf16"], errs
    for n in GRADS:
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)
    # without the context: prep, the split double scan, join + fix-up per direction, ...
    assert na > nb >= 6, (na, nb)


def test_long_context_split_sampled_head():
    """B=1, H=4, L=65536, W=128, M=8 (the long-context shape with 4 heads): 512 chunks per
    unit in 9 segments; head 1 recomputed by the oracle, and the final states of all."""
    B, H, L, d, W, M = 1, 4, 65536, 128, 128, 8
    x = synth.make_fwd_inputs(B, H, L, d, d, M, "bf16", "bimodal", seed=820)
    y, hf = gpu_fwd(x, W, "bf16", want_hf=True)
    h = 1
    sub = {n: (x[n][:, h:h + 1] if x[n].ndim == 4 else x[n][h:h + 1]) for n in NAMES}
    ref = oracle.fwd(*(sub[n] for n in NAMES), W=W, want_state=True)
    assert rel_l2(y[:, h:h + 1], ref["y"]) <= TOL["bf16"]
    assert rel_l2(hf[:, h:h + 1], ref["h_final"]) <= TOL["bf16"]
