"""Helpers for the GPU parity tests: move seeded inputs to the device, call the C ABI
through the binding, and compare with the oracle by relative L2 error."""
from __future__ import annotations

import numpy as np

import hybrid_gated_linear_gb300 as lz

NAMES = ("phi_q", "phi_k", "v", "log_gamma", "q", "k", "meta_k", "meta_v")
TOK = ("phi_q", "phi_k", "v", "log_gamma", "q", "k")
TOL = {"f32": 1e-5, "bf16": 2e-2}


def rel_l2(a, b) -> float:
    """||a - b||_2 / ||b||_2 over the whole tensor.  When the reference is exactly zero
    (a degenerate case, e.g. the window gradient of k with a single visible key) the
    ratio is undefined and the RMS absolute error is returned instead."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    num = np.linalg.norm(a - b)
    if den > 0:
        return float(num / den)
    return float(num / np.sqrt(max(1, a.size)))


def torch_dtype(dtype: str):
    import torch
    return torch.float32 if dtype == "f32" else torch.bfloat16


def code(dtype: str) -> int:
    return lz.LIZARD_F32 if dtype == "f32" else lz.LIZARD_BF16


def to_dev(x: dict, dtype: str, dev="cuda"):
    import torch
    out = {}
    for n, a in x.items():
        t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        out[n] = t if n == "log_gamma" else t.to(torch_dtype(dtype))
    return out


def host(t):
    return t.float().cpu().numpy()


def gpu_fwd(x: dict, W: int, dtype: str, alpha=1.0, h0=None, want_hf=False, scale=0.0,
            return_tensors=False):
    import torch
    t = to_dev({n: x[n] for n in NAMES}, dtype)
    B, H, L, dk = x["phi_q"].shape
    dv = x["v"].shape[-1]
    M = x["meta_k"].shape[1]
    dims = lz.lizard_dims(B, H, L, dk, dv, M, code(dtype), scale)
    ws = torch.zeros(max(lz.lizard_fwd_workspace_bytes(dims, W), 16), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty(B, H, L, dv, dtype=torch_dtype(dtype), device="cuda")
    h0t = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, dtype=np.float32)).cuda()
    hf = torch.empty(B, H, dk, dv, dtype=torch.float32, device="cuda") if want_hf else None
    lz.lizard_attn_fwd(dims, *(t[n] for n in NAMES), W, alpha, y, h0t, hf, ws)
    status = lz.lizard_check_device_errors(ws)
    assert status == 0, f"device status {status}"
    if return_tensors:
        return y, hf
    return host(y), (None if hf is None else hf.cpu().numpy())


def gpu_bwd(x: dict, W: int, dtype: str, alpha=1.0, h0=None, want_dh0=False):
    import torch
    t = to_dev({n: x[n] for n in NAMES + ("dy",)}, dtype)
    B, H, L, dk = x["phi_q"].shape
    dv = x["v"].shape[-1]
    M = x["meta_k"].shape[1]
    dims = lz.lizard_dims(B, H, L, dk, dv, M, code(dtype), 0.0)
    ws = torch.zeros(lz.lizard_bwd_workspace_bytes(dims, W), dtype=torch.uint8, device="cuda")
    td = torch_dtype(dtype)
    g = {n: torch.empty(B, H, L, dk, dtype=td, device="cuda")
         for n in ("d_phi_q", "d_phi_k", "d_q", "d_k")}
    g["d_v"] = torch.empty(B, H, L, dv, dtype=td, device="cuda")
    g["d_log_gamma"] = torch.empty(B, H, L, dk, dtype=torch.float32, device="cuda")
    g["d_meta_k"] = torch.empty(H, M, dk, dtype=torch.float32, device="cuda") if M else None
    g["d_meta_v"] = torch.empty(H, M, dv, dtype=torch.float32, device="cuda") if M else None
    g["d_h0"] = torch.empty(B, H, dk, dv, dtype=torch.float32, device="cuda") if want_dh0 else None
    h0t = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, dtype=np.float32)).cuda()
    lz.lizard_attn_bwd(dims, *(t[n] for n in NAMES), W, alpha, h0t, t["dy"], g["d_phi_q"],
                       g["d_phi_k"], g["d_v"], g["d_log_gamma"], g["d_q"], g["d_k"],
                       g["d_meta_k"], g["d_meta_v"], g["d_h0"], ws)
    status = lz.lizard_check_device_errors(ws)
    assert status == 0, f"device status {status}"
    return {n: host(v) for n, v in g.items() if v is not None}
