"""Gate projection log gamma = logsigmoid(x W)/tau and its backward through the C ABI
against the oracle's numpy prologue, alone and chained with the operator (forward and
backward) as in a training step."""
import numpy as np
import pytest
import torch

import hybrid_gated_linear_gb300 as lz
import oracle
import synth
from gpu_util import NAMES, TOL, code, host, rel_l2, torch_dtype

pytestmark = pytest.mark.gpu


def _inputs(B, H, L, D, dk, dtype, seed):
    rng = np.random.default_rng(seed)
    x = synth.to_storage(rng.standard_normal((B, H, L, D)), dtype)
    w = synth.to_storage(rng.standard_normal((H, D, dk)) / np.sqrt(D), dtype)
    g = rng.standard_normal((B, H, L, dk)).astype(np.float32)
    return x, w, g


def _run(x, w, g, dtype, tau, bwd=True):
    B, H, L, D = x.shape
    dk = w.shape[-1]
    td = torch_dtype(dtype)
    dims = lz.lizard_gate_dims(B, H, L, D, dk, code(dtype), tau)
    xt = torch.from_numpy(x).cuda().to(td)
    wt = torch.from_numpy(w).cuda().to(td)
    lg = torch.empty(B, H, L, dk, dtype=torch.float32, device="cuda")
    lz.lizard_gate_fwd(dims, xt, wt, lg)
    out = {"log_gamma": lg.cpu().numpy()}
    if bwd:
        ws = torch.zeros(max(16, lz.lizard_gate_workspace_bytes(dims)), dtype=torch.uint8, device="cuda")
        dx = torch.empty(B, H, L, D, dtype=td, device="cuda")
        dw = torch.full((H, D, dk), float("nan"), dtype=torch.float32, device="cuda")
        lz.lizard_gate_bwd(dims, xt, wt, torch.from_numpy(g).cuda(), dx, dw, ws)
        out["dx"], out["dw"] = host(dx), dw.cpu().numpy()
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,L,D,dk,tau", [
    (2, 3, 300, 128, 128, 0.0),   # tau 16 by default; ragged token tile
    (1, 2, 77, 64, 64, 4.0),
    (1, 1, 1, 5, 64, 16.0),       # one token, tiny input
    (1, 2, 1100, 256, 128, 16.0),  # the widest input, several backward groups
])
def test_gate_matches_oracle(dtype, B, H, L, D, dk, tau):
    x, w, g = _inputs(B, H, L, D, dk, dtype, seed=600 + L + D)
    out = _run(x, w, g, dtype, tau)
    t = tau if tau > 0 else 16.0
    lref = oracle.gate(x, w, t)
    dxr, dwr = oracle.gate_bwd(x, w, g, t)
    errs = {"log_gamma": rel_l2(out["log_gamma"], lref), "dx": rel_l2(out["dx"], dxr),
            "dw": rel_l2(out["dw"], dwr)}
    assert errs["log_gamma"] <= 1e-5 and errs["dw"] <= 1e-5, errs
    assert errs["dx"] <= TOL[dtype], errs


def test_gate_empty_sequence_and_determinism():
    x, w, g = _inputs(1, 2, 0, 64, 64, "f32", seed=610)
    out = _run(x, w, g, "f32", 16.0)
    np.testing.assert_array_equal(out["dw"], 0.0)
    x, w, g = _inputs(2, 2, 700, 128, 128, "bf16", seed=611)
    a, b = _run(x, w, g, "bf16", 16.0), _run(x, w, g, "bf16", 16.0)
    for n in a:
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


def test_gate_chained_with_the_operator():
    """x_g, W_gamma -> log gamma -> lizard_attn_fwd -> y; lizard_attn_bwd -> d log gamma ->
    lizard_gate_bwd -> d x_g, d W_gamma: every output against the oracle's chain."""
    B, H, L, d, M, W = 2, 2, 300, 128, 4, 64
    base = synth.make_fwd_inputs(B, H, L, d, d, M, "bf16", "plain", seed=620, with_dy=True)
    xg, wg, _ = _inputs(B, H, L, 128, d, "bf16", seed=621)
    base["log_gamma"] = oracle.gate(xg, wg, 16.0).astype(np.float32)  # reference chain input
    bf = torch.bfloat16
    gd = lz.lizard_gate_dims(B, H, L, 128, d, lz.LIZARD_BF16, 16.0)
    xt, wt = torch.from_numpy(xg).cuda().to(bf), torch.from_numpy(wg).cuda().to(bf)
    lg = torch.empty(B, H, L, d, dtype=torch.float32, device="cuda")
    lz.lizard_gate_fwd(gd, xt, wt, lg)
    t = {n: torch.from_numpy(base[n]).cuda().to(bf) for n in NAMES + ("dy",) if n != "log_gamma"}
    t["log_gamma"] = lg
    dims = lz.lizard_dims(B, H, L, d, d, M, lz.LIZARD_BF16, 0.0)
    wf = torch.zeros(lz.lizard_fwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
    y = torch.empty(B, H, L, d, dtype=bf, device="cuda")
    lz.lizard_attn_fwd(dims, *(t[n] for n in NAMES), W, 1.0, y, None, None, wf)
    wb = torch.zeros(lz.lizard_bwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
    g = {n: torch.empty(B, H, L, d, dtype=bf, device="cuda") for n in ("d_phi_q", "d_phi_k", "d_v", "d_q", "d_k")}
    g["d_log_gamma"] = torch.empty(B, H, L, d, dtype=torch.float32, device="cuda")
    g["d_meta_k"] = torch.empty(H, M, d, dtype=torch.float32, device="cuda")
    g["d_meta_v"] = torch.empty(H, M, d, dtype=torch.float32, device="cuda")
    lz.lizard_attn_bwd(dims, *(t[n] for n in NAMES), W, 1.0, None, t["dy"], g["d_phi_q"],
                       g["d_phi_k"], g["d_v"], g["d_log_gamma"], g["d_q"], g["d_k"], g["d_meta_k"],
                       g["d_meta_v"], None, wb, fwd_workspace=wf)
    wsg = torch.zeros(lz.lizard_gate_workspace_bytes(gd), dtype=torch.uint8, device="cuda")
    dxg = torch.empty(B, H, L, 128, dtype=bf, device="cuda")
    dwg = torch.empty(H, 128, d, dtype=torch.float32, device="cuda")
    lz.lizard_gate_bwd(gd, xt, wt, g["d_log_gamma"], dxg, dwg, wsg)
    for ws in (wf, wb):
        assert lz.lizard_check_device_errors(ws) == 0
    ref = oracle.fwd(*(base[n] for n in NAMES), W=W)
    rb = oracle.bwd(*(base[n] for n in NAMES), base["dy"], W=W)
    dxr, dwr = oracle.gate_bwd(xg, wg, rb["d_log_gamma"], 16.0)
    errs = {"y": rel_l2(host(y), ref["y"]), "log_gamma": rel_l2(lg.cpu().numpy(), base["log_gamma"]),
            "d_x_g": rel_l2(host(dxg), dxr), "d_W_gamma": rel_l2(dwg.cpu().numpy(), dwr)}
    errs.update({n: rel_l2(host(v), rb[n]) for n, v in g.items()})
    assert max(errs.values()) <= TOL["bf16"], errs
