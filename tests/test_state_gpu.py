"""Segment-state combine and the prefill -> decode handoff, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import NAMES, TOL, code, gpu_fwd, host, rel_l2, to_dev, torch_dtype

pytestmark = pytest.mark.gpu


def test_state_combine_matches_oracle_in_and_out_of_place():
    import torch
    import hybrid_gated_linear_gb300 as lz
    rng = np.random.default_rng(120)
    U, dk, dv = 6, 128, 128
    ga, gb = (-rng.random((U, dk)) * 3).astype(np.float32), (-rng.random((U, dk)) * 3).astype(np.float32)
    ha, hb = rng.standard_normal((U, dk, dv)).astype(np.float32), rng.standard_normal((U, dk, dv)).astype(np.float32)
    g_ref, h_ref = oracle.state_combine(ga, ha, gb, hb)
    t = {n: torch.from_numpy(a).cuda() for n, a in dict(ga=ga, ha=ha, gb=gb, hb=hb).items()}
    go, ho = torch.empty_like(t["ga"]), torch.empty_like(t["ha"])
    lz.lizard_state_combine(U, dk, dv, t["ga"], t["ha"], t["gb"], t["hb"], go, ho)
    assert rel_l2(ho.cpu().numpy(), h_ref) <= 1e-6
    np.testing.assert_allclose(go.cpu().numpy(), g_ref, rtol=1e-6, atol=1e-6)
    lz.lizard_state_combine(U, dk, dv, t["ga"], t["ha"], t["gb"], t["hb"], None, t["hb"])
    assert rel_l2(t["hb"].cpu().numpy(), h_ref) <= 1e-6


def test_sequence_split_on_the_gpu():
    """fwd over two segments from zero, the segment sums from lizard_chunk_cumsum and the
    combine give the whole sequence's final state; the second segment started from the
    first one's state gives the whole sequence's GLA outputs (alpha = 0)."""
    import torch
    import hybrid_gated_linear_gb300 as lz
    B, H, L, d, M, W, cut = 1, 2, 700, 128, 4, 64, 300
    x = synth.make_fwd_inputs(B, H, L, d, d, M, "bf16", "slow", seed=121)

    def part(a, b):
        return {n: (np.ascontiguousarray(x[n][:, :, a:b]) if x[n].ndim == 4 else x[n]) for n in NAMES}

    y_full, h_full = gpu_fwd(x, W, "bf16", alpha=0.0, want_hf=True)
    p1, p2 = part(0, cut), part(cut, L)
    _, h1 = gpu_fwd(p1, W, "bf16", alpha=0.0, want_hf=True)
    _, h2 = gpu_fwd(p2, W, "bf16", alpha=0.0, want_hf=True)
    gam = []
    for p, n in ((p1, cut), (p2, L - cut)):
        lg = torch.from_numpy(np.ascontiguousarray(p["log_gamma"])).cuda()
        b = torch.empty_like(lg)
        gc = torch.empty(B * H, 1, d, dtype=torch.float32, device="cuda")
        lz.lizard_chunk_cumsum(B * H, n, d, n, lg, b, gc)
        gam.append(gc.reshape(B, H, d))
    ho = torch.empty(B, H, d, d, dtype=torch.float32, device="cuda")
    lz.lizard_state_combine(B * H, d, d, gam[0], torch.from_numpy(h1).cuda(), gam[1],
                            torch.from_numpy(h2).cuda(), None, ho)
    assert rel_l2(ho.cpu().numpy(), h_full) <= TOL["bf16"]
    y2, _ = gpu_fwd(p2, W, "bf16", alpha=0.0, h0=h1)
    assert rel_l2(y2, y_full[:, :, cut:]) <= TOL["bf16"]


@pytest.mark.parametrize("L,W", [(150, 64), (20, 64), (0, 8)])
def test_prefill_then_decode_continues_the_sequence(L, W):
    """Prefill L tokens with the forward pass (h_final into the decode state), fill the
    rings with lizard_decode_ring_fill, decode T more tokens: every decoded y equals the
    forward pass over all L + T tokens at that position."""
    import torch
    import hybrid_gated_linear_gb300 as lz
    N, H, d, M, T, alpha = 2, 2, 128, 4, 12, 0.8
    x = synth.make_fwd_inputs(N, H, L + T, d, d, M, "bf16", "plain", seed=122 + L)
    ref = oracle.fwd(*(x[n] for n in NAMES), W=W, alpha=alpha)["y"]
    bf = torch.bfloat16
    dev = to_dev({n: x[n] for n in NAMES}, "bf16")
    h = torch.zeros(N, H, d, d, dtype=torch.float32, device="cuda")
    if L > 0:
        pre = {n: (np.ascontiguousarray(x[n][:, :, :L]) if x[n].ndim == 4 else x[n]) for n in NAMES}
        _, hf = gpu_fwd(pre, W, "bf16", alpha=alpha, want_hf=True)
        h.copy_(torch.from_numpy(hf))
    kr = torch.empty(N, H, W, d, dtype=bf, device="cuda")
    vr = torch.empty(N, H, W, d, dtype=bf, device="cuda")
    pos = torch.full((N,), -7, dtype=torch.int64, device="cuda")
    dd = lz.lizard_decode_dims(N, H, d, d, M, code("bf16"), 0.0)
    k_pre = dev["k"][:, :, :L].contiguous() if L > 0 else None
    v_pre = dev["v"][:, :, :L].contiguous() if L > 0 else None
    lz.lizard_decode_ring_fill(dd, L, W, k_pre, v_pre, kr, vr, pos)
    assert pos.cpu().tolist() == [L] * N
    ws = torch.zeros(lz.lizard_decode_workspace_bytes(dd), dtype=torch.uint8, device="cuda")
    y = torch.empty(N, H, d, dtype=bf, device="cuda")
    ys = []
    for t in range(L, L + T):
        tok = {n: dev[n][:, :, t].contiguous() for n in ("phi_q", "phi_k", "v", "log_gamma", "q", "k")}
        lz.lizard_decode_step(dd, tok["phi_q"], tok["phi_k"], tok["v"], tok["log_gamma"], tok["q"],
                              tok["k"], dev["meta_k"], dev["meta_v"], W, alpha, h, kr, vr, pos, y, ws)
        ys.append(host(y))
    assert lz.lizard_check_device_errors(ws) == 0
    got = np.stack(ys, axis=2)
    assert rel_l2(got, ref[:, :, L:]) <= TOL["bf16"]
