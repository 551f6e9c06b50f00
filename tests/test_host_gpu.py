"""Host-memory forward + backward (lizard_attn_fwd_bwd_host): results must equal those of
the two device calls bit for bit, since every (batch, head) unit is computed by the same
kernels whatever the head slice it falls in."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import NAMES, TOL, code, gpu_bwd, gpu_fwd, host, rel_l2, to_dev, torch_dtype

pytestmark = pytest.mark.gpu

GRADS = ("d_phi_q", "d_phi_k", "d_v", "d_log_gamma", "d_q", "d_k", "d_meta_k", "d_meta_v")


def _host_step(x, W, dtype, alpha=1.0, h0=None, want_state=False):
    import torch
    import hybrid_gated_linear_gb300 as lz
    B, H, L, dk = x["phi_q"].shape
    dv = x["v"].shape[-1]
    M = x["meta_k"].shape[1]
    td = torch_dtype(dtype)
    dev = to_dev({n: x[n] for n in NAMES + ("dy",)}, dtype)
    hin = {n: t.cpu().pin_memory() for n, t in dev.items()}
    dims = lz.lizard_dims(B, H, L, dk, dv, M, code(dtype), 0.0)
    ws = torch.zeros(lz.lizard_fwd_bwd_host_workspace_bytes(dims, W), dtype=torch.uint8,
                     device="cuda")
    out = {n: torch.empty(B, H, L, dk, dtype=td).pin_memory()
           for n in ("y", "d_phi_q", "d_phi_k", "d_v", "d_q", "d_k")}
    out["d_log_gamma"] = torch.empty(B, H, L, dk, dtype=torch.float32).pin_memory()
    out["d_meta_k"] = torch.empty(H, M, dk, dtype=torch.float32).pin_memory() if M else None
    out["d_meta_v"] = torch.empty(H, M, dv, dtype=torch.float32).pin_memory() if M else None
    h0t = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0)).pin_memory()
    hf = torch.empty(B, H, dk, dv, dtype=torch.float32).pin_memory() if want_state else None
    dh0 = torch.empty(B, H, dk, dv, dtype=torch.float32).pin_memory() if want_state else None
    lz.lizard_attn_fwd_bwd_host(dims, *(hin[n] for n in NAMES), W, alpha, h0t, hin["dy"],
                                out["y"], hf, out["d_phi_q"], out["d_phi_k"], out["d_v"],
                                out["d_log_gamma"], out["d_q"], out["d_k"], out["d_meta_k"],
                                out["d_meta_v"], dh0, ws)
    assert lz.lizard_check_device_errors(ws) == 0
    res = {n: host(t) for n, t in out.items() if t is not None}
    if want_state:
        res["h_final"], res["d_h0"] = hf.numpy(), dh0.numpy()
    return res


@pytest.mark.parametrize("dtype,d,W", [("bf16", 128, 64), ("f32", 64, 37), ("bf16", 128, 100)])
def test_host_step_equals_device_calls(dtype, d, W):
    B, H, L, M = 2, 10, 300, 4
    x = synth.make_fwd_inputs(B, H, L, d, d, M, dtype, "plain", seed=300 + d + W, with_dy=True)
    h0 = (0.1 * np.random.default_rng(301).standard_normal((B, H, d, d))).astype(np.float32)
    got = _host_step(x, W, dtype, alpha=0.8, h0=h0, want_state=True)
    y, hf = gpu_fwd(x, W, dtype, alpha=0.8, h0=h0, want_hf=True)
    g = gpu_bwd(x, W, dtype, alpha=0.8, h0=h0, want_dh0=True)
    np.testing.assert_array_equal(got["y"], y)
    np.testing.assert_array_equal(got["h_final"], hf)
    for n in GRADS + ("d_h0",):
        np.testing.assert_array_equal(got[n], g[n], err_msg=n)


def test_host_step_matches_oracle_one_head():
    B, H, L, d, W, M = 1, 3, 257, 128, 64, 4
    x = synth.make_fwd_inputs(B, H, L, d, d, M, "bf16", "slow", seed=302, with_dy=True)
    got = _host_step(x, W, "bf16")
    ref_y = oracle.fwd(*(x[n] for n in NAMES), W=W)["y"]
    ref = oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=W)
    assert rel_l2(got["y"], ref_y) <= TOL["bf16"]
    errs = {n: rel_l2(got[n], ref[n]) for n in GRADS}
    assert all(e <= TOL["bf16"] for e in errs.values()), errs
