"""Gates far stronger than the workloads' (log gamma = -1, -3, -20 per token, a bimodal
gate whose fast half is -5, and a sequence that turns from mild to -1): every path must
still match the oracle's token recurrence, and no device check may fire.

On the tensor-core path a 128-token chunk whose cumulative log gate leaves [-80, 80]
cannot be factorised into e^{+b} e^{-b}; those chunks are recomputed exactly (the
CUDA-core path is the recurrence itself)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import NAMES, TOK, TOL, gpu_bwd, gpu_fwd, rel_l2

pytestmark = pytest.mark.gpu

GRADS = ("d_phi_q", "d_phi_k", "d_v", "d_log_gamma", "d_q", "d_k", "d_meta_k", "d_meta_v")
# (dtype, d, W): tensor cores (bf16, d = 128, W <= 129); CUDA cores in fp32; CUDA cores in
# bf16 (a window wider than the tensor-core band)
PATHS = [("bf16", 128, 64), ("f32", 64, 64), ("bf16", 128, 200)]


def _inputs(dtype, d, gate, B=1, H=2, L=300, M=4, seed=0, with_dy=False):
    x = synth.make_fwd_inputs(B, H, L, d, d, M, dtype, "plain", seed=seed, with_dy=with_dy)
    x["log_gamma"] = synth.strong_log_gate(gate, B, H, L, d, seed=seed + 1)
    return x


@pytest.mark.parametrize("gate", synth.STRONG_GATES)
@pytest.mark.parametrize("dtype,d,W", PATHS)
def test_fwd_strong_gates_match_oracle(dtype, d, W, gate):
    x = _inputs(dtype, d, gate, seed=900 + d + W)
    rng = np.random.default_rng(901)
    h0 = (0.1 * rng.standard_normal((1, 2, d, d))).astype(np.float32)
    y, hf = gpu_fwd(x, W, dtype, alpha=0.8, h0=h0, want_hf=True)  # asserts status == 0
    ref = oracle.fwd(*(x[n] for n in NAMES), W=W, alpha=0.8, h0=h0, want_state=True)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(hf))
    errs = {"y": rel_l2(y, ref["y"]), "h_final": rel_l2(hf, ref["h_final"])}
    assert max(errs.values()) <= TOL[dtype], errs


@pytest.mark.parametrize("gate", synth.STRONG_GATES)
@pytest.mark.parametrize("dtype,d,W", PATHS)
def test_bwd_strong_gates_match_oracle(dtype, d, W, gate):
    x = _inputs(dtype, d, gate, seed=920 + d + W, with_dy=True)
    h0 = (0.1 * np.random.default_rng(921).standard_normal((1, 2, d, d))).astype(np.float32)
    g = gpu_bwd(x, W, dtype, alpha=0.8, h0=h0, want_dh0=True)  # asserts status == 0
    ref = oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=W, alpha=0.8, h0=h0, want_dh0=True)
    errs = {n: rel_l2(g[n], ref[n]) for n in GRADS + ("d_h0",)}
    assert all(np.all(np.isfinite(v)) for v in g.values())
    assert max(errs.values()) <= TOL[dtype], errs


@pytest.mark.parametrize("gate", ["const3", "mixed"])
def test_strong_gates_split_scan(gate):
    """Few heads and a long sequence: the state scans run as parallel segments joined
    afterwards, with wide chunks among them."""
    x = _inputs("bf16", 128, gate, B=1, H=2, L=3000, seed=940, with_dy=True)
    y, hf = gpu_fwd(x, 64, "bf16", want_hf=True)
    ref = oracle.fwd(*(x[n] for n in NAMES), W=64, want_state=True)
    assert rel_l2(y, ref["y"]) <= TOL["bf16"] and rel_l2(hf, ref["h_final"]) <= TOL["bf16"]
    g = gpu_bwd(x, 64, "bf16", want_dh0=True)
    rb = oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=64, want_dh0=True)
    errs = {n: rel_l2(g[n], rb[n]) for n in GRADS + ("d_h0",)}
    assert max(errs.values()) <= TOL["bf16"], errs


@pytest.mark.parametrize("gate", ["const20", "mixed"])
def test_bwd_from_forward_context_strong_gates(gate):
    """The backward that reuses the forward's workspace reads the wide chunks' features
    where the forward's recomputation left them: bitwise the same gradients as a
    backward that recomputes everything, and both match the oracle."""
    import torch
    import hybrid_gated_linear_gb300 as lz
    from gpu_util import code, host, to_dev
    B, H, L, d, M, W = 2, 2, 300, 128, 4, 64
    x = _inputs("bf16", d, gate, B=B, H=H, L=L, seed=950, with_dy=True)
    t = to_dev({n: x[n] for n in NAMES + ("dy",)}, "bf16")
    dims = lz.lizard_dims(B, H, L, d, d, M, code("bf16"), 0.0)
    wf = torch.zeros(lz.lizard_fwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
    y = torch.empty(B, H, L, d, dtype=torch.bfloat16, device="cuda")
    lz.lizard_attn_fwd(dims, *(t[n] for n in NAMES), W, 1.0, y, None, None, wf)
    assert lz.lizard_check_device_errors(wf) == 0

    def run(fwd_ws):
        wb = torch.zeros(lz.lizard_bwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
        g = {n: torch.empty(B, H, L, d, dtype=torch.bfloat16, device="cuda")
             for n in ("d_phi_q", "d_phi_k", "d_v", "d_q", "d_k")}
        g["d_log_gamma"] = torch.empty(B, H, L, d, dtype=torch.float32, device="cuda")
        g["d_meta_k"] = torch.empty(H, M, d, dtype=torch.float32, device="cuda")
        g["d_meta_v"] = torch.empty(H, M, d, dtype=torch.float32, device="cuda")
        lz.lizard_attn_bwd(dims, *(t[n] for n in NAMES), W, 1.0, None, t["dy"], g["d_phi_q"],
                           g["d_phi_k"], g["d_v"], g["d_log_gamma"], g["d_q"], g["d_k"],
                           g["d_meta_k"], g["d_meta_v"], None, wb, fwd_workspace=fwd_ws)
        assert lz.lizard_check_device_errors(wb) == 0
        return {n: host(v) for n, v in g.items()}

    a, b = run(None), run(wf)
    for n in a:
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)
    ref = oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=W)
    errs = {n: rel_l2(b[n], ref[n]) for n in GRADS}
    assert max(errs.values()) <= TOL["bf16"], errs


@pytest.mark.parametrize("gate", ["const1", "bimodal5"])
def test_fused_feature_map_strong_gates(gate):
    """Forward from the raw projections (feature map fused into the gate absorption) and
    the training step's backward from its context (phi = NULL), with wide chunks."""
    import torch
    import hybrid_gated_linear_gb300 as lz
    from test_fmap_gpu import _fused_inputs, _run_fused
    from gpu_util import host
    B, H, L, M, W = 1, 2, 300, 4, 64
    x = _fused_inputs(B, H, L, M, seed=960)
    x["log_gamma"] = synth.strong_log_gate(gate, B, H, L, 128, seed=961)
    t, dims, ws, y, hf = _run_fused(x, W, 1.0)
    assert lz.lizard_check_device_errors(ws) == 0
    ref = oracle.fwd(*(x[n] for n in NAMES), W=W, want_state=True)
    errs = {"y": rel_l2(host(y), ref["y"]), "h_final": rel_l2(hf.cpu().numpy(), ref["h_final"])}
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
    assert lz.lizard_check_device_errors(wsb) == 0
    rb = oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=W)
    errs.update({n: rel_l2(host(v), rb[n]) for n, v in g.items()})
    assert max(errs.values()) <= TOL["bf16"], errs


@pytest.mark.parametrize("gate", ["const20", "bimodal5"])
def test_decode_strong_gates(gate):
    from test_decode_gpu import GpuDecoder, _oracle_state
    s = synth.DecodeStream(2, 2, 128, 128, 4, 16, "bf16", seed=970, prefill=True)
    g = GpuDecoder(s)
    st = _oracle_state(s, [0, 1], [0, 1])
    for i in range(24):
        tok = s.next_token()
        tok["log_gamma"] = synth.strong_log_gate(gate, 2, 2, 1, 128, seed=971 + i)[:, :, 0]
        y = g.step(tok)
        yr = oracle.decode_step(st, *(tok[n] for n in TOK), s.meta_k, s.meta_v, W=16)
        assert rel_l2(y, yr) <= TOL["bf16"]
    assert rel_l2(g.h.cpu().numpy(), st["h"]) <= TOL["bf16"]
