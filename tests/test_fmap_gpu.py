"""Hedgehog feature map phi(x) = [exp(x W), exp(-x W)] and its backward, through the C ABI,
against the fp64 oracle ("Lizard", arXiv 2507.09025, Method: Hedgehog feature map)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import NAMES, TOL, code, gpu_fwd, host, rel_l2, torch_dtype

pytestmark = pytest.mark.gpu


def _run(x, dtype, bwd=True, repeat=1):
    import torch
    import hybrid_gated_linear_gb300 as lz
    td = torch_dtype(dtype)
    B, H, L, D = x["x"].shape
    F = x["w"].shape[-1]
    dims = lz.lizard_fmap_dims(B, H, L, D, F, code(dtype))
    X = torch.from_numpy(x["x"]).cuda().to(td)
    Wt = torch.from_numpy(x["w"]).cuda().to(td)
    ws = torch.zeros(lz.lizard_feature_map_workspace_bytes(dims, bwd), dtype=torch.uint8, device="cuda")
    phi = torch.empty(B, H, L, 2 * F, dtype=td, device="cuda")
    lz.lizard_feature_map_fwd(dims, X, Wt, phi, ws)
    assert lz.lizard_check_device_errors(ws) == 0
    out = {"phi": host(phi)}
    if bwd:
        dp = torch.from_numpy(x["d_phi"]).cuda().to(td)
        dws = []
        for _ in range(repeat):
            dx = torch.full((B, H, L, D), float("nan"), dtype=td, device="cuda")
            dw = torch.full((H, D, F), float("nan"), dtype=torch.float32, device="cuda")
            lz.lizard_feature_map_bwd(dims, X, Wt, dp, dx, dw, ws)
            assert lz.lizard_check_device_errors(ws) == 0
            dws.append(dw.cpu().numpy())
        out["dx"], out["dw"], out["dws"] = host(dx), dws[0], dws
    return out


# tensor-core path: bf16, D = 128, F = 64; tails, several tiles, several tile groups
@pytest.mark.parametrize("B,H,L", [(1, 2, 300), (2, 3, 128), (1, 1, 1), (1, 2, 700), (2, 1, 1100)])
def test_feature_map_tensor_core_path_matches_oracle(B, H, L):
    x = synth.make_fmap_inputs(B, H, L, 128, 64, "bf16", seed=200 + L, with_dphi=True)
    got = _run(x, "bf16")
    ref = oracle.feature_map(x["x"], x["w"])
    dx_ref, dw_ref = oracle.feature_map_bwd(x["x"], x["w"], x["d_phi"])
    errs = {"phi": rel_l2(got["phi"], ref), "dx": rel_l2(got["dx"], dx_ref), "dw": rel_l2(got["dw"], dw_ref)}
    assert max(errs.values()) <= TOL["bf16"], errs
    assert np.isfinite(got["dx"]).all() and np.isfinite(got["dw"]).all()


# CUDA-core path: other sizes and fp32
@pytest.mark.parametrize("dtype,D,F,L", [("f32", 64, 32, 300), ("f32", 128, 64, 129),
                                         ("bf16", 64, 32, 77), ("f32", 5, 3, 40), ("f32", 256, 64, 600)])
def test_feature_map_cuda_core_path_matches_oracle(dtype, D, F, L):
    x = synth.make_fmap_inputs(2, 2, L, D, F, dtype, seed=300 + D + L, with_dphi=True)
    got = _run(x, dtype)
    ref = oracle.feature_map(x["x"], x["w"])
    dx_ref, dw_ref = oracle.feature_map_bwd(x["x"], x["w"], x["d_phi"])
    errs = {"phi": rel_l2(got["phi"], ref), "dx": rel_l2(got["dx"], dx_ref), "dw": rel_l2(got["dw"], dw_ref)}
    assert max(errs.values()) <= TOL[dtype], errs


@pytest.mark.parametrize("D,F,dtype", [(128, 64, "bf16"), (64, 32, "f32")])
def test_feature_map_weight_gradient_is_run_to_run_identical(D, F, dtype):
    x = synth.make_fmap_inputs(2, 2, 900, D, F, dtype, seed=400, with_dphi=True)
    got = _run(x, dtype, repeat=3)
    for dw in got["dws"][1:]:
        np.testing.assert_array_equal(dw, got["dws"][0])


def test_feature_map_empty_sequence_zero_fills_the_weight_gradient():
    import torch
    import hybrid_gated_linear_gb300 as lz
    dims = lz.lizard_fmap_dims(1, 2, 0, 128, 64, lz.LIZARD_BF16)
    w = torch.zeros(2, 128, 64, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((2, 128, 64), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.zeros(lz.lizard_feature_map_workspace_bytes(dims, True), dtype=torch.uint8, device="cuda")
    lz.lizard_feature_map_fwd(dims, None, w, None, ws)
    lz.lizard_feature_map_bwd(dims, None, w, None, None, dw, ws)
    assert lz.lizard_check_device_errors(ws) == 0
    assert float(dw.abs().max()) == 0.0


def test_feature_map_full_size_sampled_heads():
    """B=1, H=32, L=4096 (the attention workload's shape): every head's phi is checked on
    sampled rows, and two heads' dx and dW in full."""
    B, H, L = 1, 32, 4096
    x = synth.make_fmap_inputs(B, H, L, 128, 64, "bf16", seed=500, with_dphi=True)
    got = _run(x, "bf16")
    rng = np.random.default_rng(501)
    rows = rng.choice(L, 64, replace=False)
    sub = x["x"][:, :, rows]
    ref = oracle.feature_map(sub, x["w"])
    assert rel_l2(got["phi"][:, :, rows], ref) <= TOL["bf16"]
    for h in (0, 31):
        dx_ref, dw_ref = oracle.feature_map_bwd(x["x"][:, h:h + 1], x["w"][h:h + 1], x["d_phi"][:, h:h + 1])
        assert rel_l2(got["dx"][:, h:h + 1], dx_ref) <= TOL["bf16"]
        assert rel_l2(got["dw"][h:h + 1], dw_ref) <= TOL["bf16"]


def test_feature_map_output_feeds_the_attention_forward():
    """phi_q, phi_k from the feature map are valid operator inputs: the forward over them
    matches the oracle's forward over the oracle's feature map of the same x."""
    B, H, L, M, W = 1, 2, 300, 4, 64
    base = synth.make_fwd_inputs(B, H, L, 128, 128, M, "bf16", "plain", seed=600)
    fq = synth.make_fmap_inputs(B, H, L, 128, 64, "bf16", seed=601)
    fk = synth.make_fmap_inputs(B, H, L, 128, 64, "bf16", seed=602)
    # a small scale keeps phi_q . phi_k in the range of the pages' normalised features
    fq["w"] = synth.to_storage(fq["w"] * 0.5, "bf16")
    fk["w"] = synth.to_storage(fk["w"] * 0.5, "bf16")
    pq = _run(fq, "bf16", bwd=False)["phi"] / np.sqrt(128)
    pk = _run(fk, "bf16", bwd=False)["phi"] / np.sqrt(128)
    x = dict(base, phi_q=synth.to_storage(pq, "bf16"), phi_k=synth.to_storage(pk, "bf16"))
    y, _ = gpu_fwd(x, W, "bf16")
    ref = oracle.fwd(*(x[n] for n in NAMES), W=W, alpha=1.0)["y"]
    assert rel_l2(y, ref) <= TOL["bf16"]
    ref_phi = oracle.feature_map(fq["x"], fq["w"]) / np.sqrt(128)
    assert rel_l2(pq, ref_phi) <= TOL["bf16"]


# --------------------------------------------------------------------------------------
# forward from the raw projections with the feature map fused into the gate absorption
# --------------------------------------------------------------------------------------
def _fused_inputs(B, H, L, M, seed):
    base = synth.make_fwd_inputs(B, H, L, 128, 128, M, "bf16", "plain", seed=seed, with_dy=True)
    fq = synth.make_fmap_inputs(B, H, L, 128, 64, "bf16", seed=seed + 1)
    fk = synth.make_fmap_inputs(B, H, L, 128, 64, "bf16", seed=seed + 2)
    # W ~ N(0, 1/(4D)) keeps phi_q . phi_k moderate
    x = dict(base, x_q=fq["x"], x_k=fk["x"], w_q=synth.to_storage(fq["w"] * 0.5, "bf16"),
             w_k=synth.to_storage(fk["w"] * 0.5, "bf16"))
    x["phi_q"] = oracle.feature_map(x["x_q"], x["w_q"])
    x["phi_k"] = oracle.feature_map(x["x_k"], x["w_k"])
    return x


def _run_fused(x, W, alpha, h0=None, want_hf=True):
    import torch
    import hybrid_gated_linear_gb300 as lz
    bf = torch.bfloat16
    B, H, L, _ = x["x_q"].shape
    M = x["meta_k"].shape[1]
    t = {n: torch.from_numpy(np.ascontiguousarray(x[n])).cuda() for n in
         ("x_q", "x_k", "w_q", "w_k", "v", "q", "k", "meta_k", "meta_v", "log_gamma")}
    for n in t:
        if n != "log_gamma":
            t[n] = t[n].to(bf)
    dims = lz.lizard_dims(B, H, L, 128, 128, M, lz.LIZARD_BF16, 0.0)
    ws = torch.zeros(lz.lizard_fwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
    y = torch.empty(B, H, L, 128, dtype=bf, device="cuda")
    hf = torch.empty(B, H, 128, 128, dtype=torch.float32, device="cuda") if want_hf else None
    h0t = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, dtype=np.float32)).cuda()
    lz.lizard_attn_fwd_fmap(dims, t["x_q"], t["x_k"], t["w_q"], t["w_k"], t["v"], t["log_gamma"],
                            t["q"], t["k"], t["meta_k"], t["meta_v"], W, alpha, y, h0t, hf, ws)
    return t, dims, ws, y, hf


@pytest.mark.parametrize("B,H,L,W,M,alpha,with_h0", [(1, 2, 300, 64, 4, 1.0, False),
                                                     (2, 2, 129, 100, 0, 0.7, True),
                                                     (1, 1, 1, 64, 4, 1.0, False),
                                                     (1, 3, 700, 37, 8, 1.3, True)])
def test_fused_feature_map_forward_matches_oracle(B, H, L, W, M, alpha, with_h0):
    import hybrid_gated_linear_gb300 as lz
    x = _fused_inputs(B, H, L, M, seed=700 + L)
    h0 = (np.random.default_rng(701).standard_normal((B, H, 128, 128)) * 0.1) if with_h0 else None
    _, _, ws, y, hf = _run_fused(x, W, alpha, h0=h0)
    assert lz.lizard_check_device_errors(ws) == 0
    ref = oracle.fwd(*(x[n] for n in NAMES), W=W, alpha=alpha, h0=h0, want_state=True)
    errs = {"y": rel_l2(host(y), ref["y"]), "h_final": rel_l2(hf.cpu().numpy(), ref["h_final"])}
    assert max(errs.values()) <= TOL["bf16"], errs


def test_fused_forward_agrees_with_the_map_followed_by_the_forward():
    import torch
    import hybrid_gated_linear_gb300 as lz
    x = _fused_inputs(1, 2, 500, 4, seed=710)
    t, dims, ws, y, _ = _run_fused(x, 64, 1.0, want_hf=False)
    fd = lz.lizard_fmap_dims(1, 2, 500, 128, 64, lz.LIZARD_BF16)
    wsf = torch.zeros(lz.lizard_feature_map_workspace_bytes(fd, False), dtype=torch.uint8, device="cuda")
    pq = torch.empty(1, 2, 500, 128, dtype=torch.bfloat16, device="cuda")
    pk = torch.empty_like(pq)
    lz.lizard_feature_map_fwd(fd, t["x_q"], t["w_q"], pq, wsf)
    lz.lizard_feature_map_fwd(fd, t["x_k"], t["w_k"], pk, wsf)
    y2 = torch.empty_like(y)
    ws2 = torch.zeros_like(ws)
    lz.lizard_attn_fwd(dims, pq, pk, t["v"], t["log_gamma"], t["q"], t["k"], t["meta_k"],
                       t["meta_v"], 64, 1.0, y2, None, None, ws2)
    assert lz.lizard_check_device_errors(ws) == 0 and lz.lizard_check_device_errors(ws2) == 0
    assert rel_l2(host(y), host(y2)) <= 1e-2


@pytest.mark.parametrize("L,W", [(300, 64), (129, 100)])
def test_fused_training_step_gradients_match_oracle(L, W):
    """Forward from x, backward with phi = NULL and the forward's workspace, then the
    feature map's backward: every gradient against the oracle chain (attention adjoint,
    then the feature map's adjoint)."""
    import torch
    import hybrid_gated_linear_gb300 as lz
    B, H, M = 2, 2, 4
    x = _fused_inputs(B, H, L, M, seed=720 + L)
    t, dims, ws, y, _ = _run_fused(x, W, 1.0, want_hf=False)
    bf = torch.bfloat16
    dy = torch.from_numpy(x["dy"]).cuda().to(bf)
    wsb = torch.zeros(lz.lizard_bwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
    g = {n: torch.empty(B, H, L, 128, dtype=bf, device="cuda")
         for n in ("d_phi_q", "d_phi_k", "d_v", "d_q", "d_k")}
    g["d_log_gamma"] = torch.empty(B, H, L, 128, dtype=torch.float32, device="cuda")
    g["d_meta_k"] = torch.empty(H, M, 128, dtype=torch.float32, device="cuda")
    g["d_meta_v"] = torch.empty(H, M, 128, dtype=torch.float32, device="cuda")
    lz.lizard_attn_bwd(dims, None, None, t["v"], t["log_gamma"], t["q"], t["k"], t["meta_k"],
                       t["meta_v"], W, 1.0, None, dy, g["d_phi_q"], g["d_phi_k"], g["d_v"],
                       g["d_log_gamma"], g["d_q"], g["d_k"], g["d_meta_k"], g["d_meta_v"], None,
                       wsb, fwd_workspace=ws)
    fd = lz.lizard_fmap_dims(B, H, L, 128, 64, lz.LIZARD_BF16)
    wsf = torch.zeros(lz.lizard_feature_map_workspace_bytes(fd, True), dtype=torch.uint8, device="cuda")
    out = {}
    for s in ("q", "k"):
        dxs = torch.empty(B, H, L, 128, dtype=bf, device="cuda")
        dws = torch.empty(H, 128, 64, dtype=torch.float32, device="cuda")
        lz.lizard_feature_map_bwd(fd, t["x_" + s], t["w_" + s], g["d_phi_" + s], dxs, dws, wsf)
        out["dx_" + s], out["dw_" + s] = host(dxs), dws.cpu().numpy()
    for w in (ws, wsb, wsf):
        assert lz.lizard_check_device_errors(w) == 0
    ref = oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=W, alpha=1.0)
    errs = {n: rel_l2(host(gt), ref[n]) for n, gt in g.items()}
    for s in ("q", "k"):
        dxr, dwr = oracle.feature_map_bwd(x["x_" + s], x["w_" + s], ref["d_phi_" + s])
        errs["dx_" + s] = rel_l2(out["dx_" + s], dxr)
        errs["dw_" + s] = rel_l2(out["dw_" + s], dwr)
    assert max(errs.values()) <= TOL["bf16"], errs


def test_fused_forward_without_tokens_carries_h0():
    import torch
    import hybrid_gated_linear_gb300 as lz
    dims = lz.lizard_dims(1, 2, 0, 128, 128, 4, lz.LIZARD_BF16, 0.0)
    w = torch.zeros(2, 128, 64, dtype=torch.bfloat16, device="cuda")
    mk = torch.zeros(2, 4, 128, dtype=torch.bfloat16, device="cuda")
    h0 = torch.randn(1, 2, 128, 128, dtype=torch.float32, device="cuda")
    hf = torch.empty_like(h0)
    ws = torch.zeros(max(16, lz.lizard_fwd_workspace_bytes(dims, 64)), dtype=torch.uint8, device="cuda")
    lz.lizard_attn_fwd_fmap(dims, None, None, w, w, None, None, None, None, mk, mk, 64, 1.0, None,
                            h0, hf, ws)
    assert lz.lizard_check_device_errors(ws) == 0
    assert torch.equal(hf, h0)
