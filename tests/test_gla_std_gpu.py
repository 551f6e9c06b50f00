"""The standard fp32 chunkwise GLA forward (the comparison kernel of "Lizard", Efficiency,
Table 3): its y equals the oracle's GLA branch and its final state the oracle's state."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import NAMES, TOL, code, host, rel_l2, to_dev, torch_dtype

pytestmark = pytest.mark.gpu

# fp32 arithmetic throughout: both input types meet the fp32 tolerance against the
# oracle fed the same (bf16-rounded) inputs, up to the final rounding of y
STD_TOL = {"f32": TOL["f32"], "bf16": 1e-2}


def run_std(x, dtype, h0=None):
    import torch
    import hybrid_gated_linear_gb300 as lz
    t = to_dev({n: x[n] for n in ("phi_q", "phi_k", "v", "log_gamma")}, dtype)
    B, H, L, dk = x["phi_q"].shape
    dv = x["v"].shape[-1]
    dims = lz.lizard_dims(B, H, L, dk, dv, 0, code(dtype), 0.0)
    ws = torch.zeros(lz.lizard_gla_std_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    y = torch.empty(B, H, L, dv, dtype=torch_dtype(dtype), device="cuda")
    hf = torch.empty(B, H, dk, dv, dtype=torch.float32, device="cuda")
    h0t = None if h0 is None else torch.from_numpy(h0).cuda()
    lz.lizard_gla_std_fwd(dims, t["phi_q"], t["phi_k"], t["v"], t["log_gamma"], y, h0t, hf, ws)
    return host(y), hf.cpu().numpy(), lz.lizard_check_device_errors(ws)


def _rounded(x, dtype):
    """The inputs as the kernel sees them (bf16 rounding of the T tensors)."""
    if dtype == "f32":
        return x
    import torch
    out = dict(x)
    for n in ("phi_q", "phi_k", "v"):
        out[n] = torch.from_numpy(x[n]).to(torch.bfloat16).float().numpy()
    return out


def _oracle_gla(x, h0=None):
    r = oracle.fwd(*(x[n] for n in NAMES), W=1, alpha=0.0, h0=h0, want_state=True)
    return r["y"], r["h_final"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,H,L,d,gate", [
    (1, 2, 256, 64, "plain"),     # four whole chunks
    (2, 2, 300, 128, "slow"),     # ragged tail, batch > 1
    (1, 1, 1, 128, "plain"),      # one token
    (1, 3, 65, 128, "bimodal"),   # one chunk and a one-token tail
])
def test_gla_std_matches_oracle(dtype, B, H, L, d, gate):
    x = synth.make_fwd_inputs(B, H, L, d, d, 0, dtype, gate, seed=500 + L)
    y, hf, st = run_std(x, dtype)
    assert st == 0
    yr, hr = _oracle_gla(_rounded(x, dtype))
    assert rel_l2(y, yr) <= STD_TOL[dtype]
    assert rel_l2(hf, hr) <= TOL["f32"]


def test_gla_std_initial_state_and_empty():
    B, H, L, d = 1, 2, 130, 128
    x = synth.make_fwd_inputs(B, H, L, d, d, 0, "f32", "plain", seed=41)
    h0 = (0.1 * np.random.default_rng(42).standard_normal((B, H, d, d))).astype(np.float32)
    y, hf, st = run_std(x, "f32", h0=h0)
    assert st == 0
    yr, hr = _oracle_gla(x, h0=h0)
    assert rel_l2(y, yr) <= TOL["f32"] and rel_l2(hf, hr) <= TOL["f32"]
    # L = 0: nothing but h_final = h0
    x0 = {n: a[:, :, :0] for n, a in x.items() if a.ndim == 4}
    x0.update({n: x[n] for n in ("meta_k", "meta_v")})
    y0, hf0, st0 = run_std(x0, "f32", h0=h0)
    assert st0 == 0 and y0.size == 0
    np.testing.assert_array_equal(hf0, h0)


def test_gla_std_agrees_with_tensor_core_path():
    """The two GLA kernels (fp32 CUDA-core and bf16 tensor-core) on the workload shape's
    head count, same inputs, window branch off (alpha = 0): both near the oracle."""
    from gpu_util import gpu_fwd
    B, H, L, d = 1, 4, 1024, 128
    x = synth.make_fwd_inputs(B, H, L, d, d, 4, "bf16", "plain", seed=43)
    y_std, _, st = run_std(x, "bf16")
    assert st == 0
    y_tc, _ = gpu_fwd(x, 64, "bf16", alpha=0.0)
    yr, _ = _oracle_gla(_rounded(x, "bf16"))
    assert rel_l2(y_std, yr) <= STD_TOL["bf16"]
    assert rel_l2(y_tc, yr) <= TOL["bf16"]


def test_gla_std_flags_gates_beyond_its_range():
    """log gamma = -3 per token: b reaches -192 inside a 64-token chunk, where the standard
    factorised form has no finite value; the call says so through the status word."""
    B, H, L, d = 1, 1, 128, 64
    x = synth.make_fwd_inputs(B, H, L, d, d, 0, "f32", "plain", seed=44)
    x["log_gamma"] = synth.strong_log_gate("const3", B, H, L, d)
    _, _, st = run_std(x, "f32")
    assert st == 5  # LIZARD_ERR_DEVICE_CHECK


def test_gla_std_is_deterministic():
    x = synth.make_fwd_inputs(1, 2, 200, 128, 128, 0, "bf16", "plain", seed=45)
    a, ha, _ = run_std(x, "bf16")
    b, hb, _ = run_std(x, "bf16")
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(ha, hb)
