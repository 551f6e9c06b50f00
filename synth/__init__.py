"""Seeded synthetic inputs for the Lizard-attention operator.

This module is the one piece that both sides of every parity check consume: the
fp64 oracle (``oracle/``) and the CUDA library (``hybrid_gated_linear_gb300``).  It
holds none of the operator's arithmetic -- only random draws, the input recipes of the
named workloads, and rounding to the storage dtype.

Recipes (all draws in float64 from ``numpy.random.default_rng(seed)``, then rounded):
  * q, k, v ~ N(0, 1); meta_k, meta_v ~ N(0, 1)
  * phi_q = (elu(q) + 1) / sqrt(d), phi_k = (elu(k) + 1) / sqrt(d), computed in fp64 from
    the *rounded* q, k and rounded again
  * log_gamma = logsigmoid(g + shift) / 16 with g ~ N(0, 1), fp64 then rounded to fp32
  * dy ~ N(0, 1); decode state h0 ~ N(0, 0.1^2) in fp32; ring buffers ~ N(0, 1)
Draw order: q, k, v, g, meta_k, meta_v, then dy; decode: meta_k, meta_v, h0, k_ring,
v_ring, then per step q, k, v, g.

Rounding: float64 -> float32 (round to nearest even) and, for bf16 tensors, float32 ->
bf16 (round to nearest even).  bf16 tensors are returned as float32 arrays holding
exactly representable bf16 values, so widening to fp64 (oracle) and narrowing to
torch.bfloat16 (GPU) are both exact.
"""
from __future__ import annotations

import numpy as np

# Named workloads.  Shapes follow the Lizard paper's setting (Llama-3-8B attention
# layers, 32 heads of 128; training batch 8 x 2048; long-context evaluation to 64K;
# window w and m meta tokens).
WORKLOADS = {
    "tiny_fp32": dict(kind="fwd", dtype="f32", B=1, H=2, L=256, dk=64, dv=64, W=64, M=4,
                      gate="plain", seed=1000),
    "llama3_8b_fwd": dict(kind="fwd", dtype="bf16", B=1, H=32, L=4096, dk=128, dv=128, W=64,
                          M=4, gate="plain", seed=1001),
    "train_fwd_bwd": dict(kind="fwd_bwd", dtype="bf16", B=8, H=32, L=2048, dk=128, dv=128,
                          W=64, M=4, gate="slow", seed=1002),
    "long_ctx_64k": dict(kind="fwd", dtype="bf16", B=1, H=32, L=65536, dk=128, dv=128, W=128,
                         M=8, gate="bimodal", seed=1003),
    "decode_64x32": dict(kind="decode", dtype="bf16", N=64, H=32, dk=128, dv=128, W=64, M=4,
                         steps=1024, gate="plain", seed=1004),
}


def round_bf16(x) -> np.ndarray:
    """Round to the nearest bf16 (ties to even) via float32; returns float32 values."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return (u & 0xFFFFFFFF).astype(np.uint32).view(np.float32).reshape(f.shape)


def to_storage(x, dtype: str) -> np.ndarray:
    """Round a float64 array to the storage dtype ("f32" or "bf16") as float32 values."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return round_bf16(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def _elu_plus_one(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def feature_map(x_rounded, d: int, dtype: str) -> np.ndarray:
    """phi(x) = (elu(x) + 1) / sqrt(d) from already-rounded x, then rounded."""
    return to_storage(_elu_plus_one(np.asarray(x_rounded, dtype=np.float64)) / np.sqrt(d), dtype)


def _logsigmoid(x):
    return np.where(x >= 0, -np.log1p(np.exp(-x)), x - np.log1p(np.exp(x)))


def gate_shift(gate: str, dk: int) -> np.ndarray:
    """Per-key-dimension shift of the gate pre-activation."""
    if gate == "plain":
        return np.zeros(dk)
    if gate == "slow":
        return np.full(dk, 3.0)
    if gate == "bimodal":  # fast-decaying first half, near-1 second half
        return np.concatenate([np.full(dk // 2, -2.0), np.full(dk - dk // 2, 4.0)])
    raise ValueError(f"unknown gate {gate!r}")


def log_gate(g, shift) -> np.ndarray:
    """log gamma = logsigmoid(g + shift) / 16 in fp64, stored as float32."""
    return (_logsigmoid(np.asarray(g, dtype=np.float64) + shift) / 16.0).astype(np.float32)


def make_fwd_inputs(B, H, L, dk, dv, M, dtype="bf16", gate="plain", seed=0, with_dy=False):
    """Inputs of one forward (and optional backward) call, shapes [B,H,L,d] and [H,M,d]."""
    rng = np.random.default_rng(seed)
    q = to_storage(rng.standard_normal((B, H, L, dk)), dtype)
    k = to_storage(rng.standard_normal((B, H, L, dk)), dtype)
    v = to_storage(rng.standard_normal((B, H, L, dv)), dtype)
    g = rng.standard_normal((B, H, L, dk))
    log_gamma = log_gate(g, gate_shift(gate, dk))
    del g
    meta_k = to_storage(rng.standard_normal((H, M, dk)), dtype)
    meta_v = to_storage(rng.standard_normal((H, M, dv)), dtype)
    out = dict(phi_q=feature_map(q, dk, dtype), phi_k=feature_map(k, dk, dtype), v=v,
               log_gamma=log_gamma, q=q, k=k, meta_k=meta_k, meta_v=meta_v)
    if with_dy:
        out["dy"] = to_storage(rng.standard_normal((B, H, L, dv)), dtype)
    return out


STRONG_GATES = ("const1", "const3", "const20", "bimodal5", "mixed")


def strong_log_gate(kind: str, B, H, L, dk, seed=0) -> np.ndarray:
    """Gates far stronger than the workloads' logsigmoid(g)/16, [B,H,L,dk] float32:
    const1 / const3 / const20: log gamma = -1, -3, -20 for every token and key dimension;
    bimodal5: the first half of the key dimensions -5 per token, the second half
    logsigmoid(g + 4)/16; mixed: logsigmoid(g)/16 for tokens before L/3, then -1."""
    if kind.startswith("const"):
        return np.full((B, H, L, dk), -float(kind[5:]), dtype=np.float32)
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((B, H, L, dk))
    if kind == "bimodal5":
        out = log_gate(g, np.full(dk, 4.0))
        out[..., : dk // 2] = -5.0
        return out
    if kind == "mixed":
        out = log_gate(g, np.zeros(dk))
        out[:, :, L // 3:, :] = -1.0
        return out
    raise ValueError(f"unknown gate {kind!r}")


def make_fmap_inputs(B, H, L, D, F, dtype="bf16", seed=0, with_dphi=False):
    """Inputs of a feature-map call: x [B,H,L,D] ~ N(0,1) and per-head W [H,D,F] ~
    N(0, 1/D) (so that x W is about unit variance), each rounded to the storage dtype;
    with_dphi adds an upstream gradient [B,H,L,2F] ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    x = to_storage(rng.standard_normal((B, H, L, D)), dtype)
    w = to_storage(rng.standard_normal((H, D, F)) / np.sqrt(D), dtype)
    out = dict(x=x, w=w)
    if with_dphi:
        out["d_phi"] = to_storage(rng.standard_normal((B, H, L, 2 * F)), dtype)
    return out


def workload_inputs(name: str, **overrides):
    """Inputs of a named forward/backward workload, optionally with overridden sizes."""
    w = dict(WORKLOADS[name])
    w.update(overrides)
    return make_fwd_inputs(w["B"], w["H"], w["L"], w["dk"], w["dv"], w["M"], w["dtype"],
                           w["gate"], w["seed"], with_dy=(w["kind"] == "fwd_bwd"))


class DecodeStream:
    """Seeded decode workload: meta tensors, initial state and rings, then one token per
    step per sequence.  ``prefill=True`` fills all W ring slots and starts at pos = W;
    otherwise the rings are empty and pos starts at 0."""

    def __init__(self, N, H, dk, dv, M, W, dtype="bf16", gate="plain", seed=0, prefill=True,
                 h0_std=0.1):
        self.N, self.H, self.dk, self.dv, self.M, self.W = N, H, dk, dv, M, W
        self.dtype, self.shift = dtype, gate_shift(gate, dk)
        self.rng = np.random.default_rng(seed)
        r = self.rng
        self.meta_k = to_storage(r.standard_normal((H, M, dk)), dtype)
        self.meta_v = to_storage(r.standard_normal((H, M, dv)), dtype)
        if prefill:
            self.h0 = (h0_std * r.standard_normal((N, H, dk, dv))).astype(np.float32)
            self.k_ring = to_storage(r.standard_normal((N, H, W, dk)), dtype)
            self.v_ring = to_storage(r.standard_normal((N, H, W, dv)), dtype)
            self.pos0 = np.full(N, W, dtype=np.int64)
        else:
            self.h0 = np.zeros((N, H, dk, dv), dtype=np.float32)
            self.k_ring = np.zeros((N, H, W, dk), dtype=np.float32)
            self.v_ring = np.zeros((N, H, W, dv), dtype=np.float32)
            self.pos0 = np.zeros(N, dtype=np.int64)

    def next_token(self):
        """Token inputs of the next step, each [N,H,d]."""
        r, N, H, dk, dv, dt = self.rng, self.N, self.H, self.dk, self.dv, self.dtype
        q = to_storage(r.standard_normal((N, H, dk)), dt)
        k = to_storage(r.standard_normal((N, H, dk)), dt)
        v = to_storage(r.standard_normal((N, H, dv)), dt)
        log_gamma = log_gate(r.standard_normal((N, H, dk)), self.shift)
        return dict(phi_q=feature_map(q, dk, dt), phi_k=feature_map(k, dk, dt), v=v,
                    log_gamma=log_gamma, q=q, k=k)


def decode_stream(name="decode_64x32", prefill=True, **overrides):
    w = dict(WORKLOADS[name])
    w.update(overrides)
    return DecodeStream(w["N"], w["H"], w["dk"], w["dv"], w["M"], w["W"], w["dtype"],
                        w["gate"], w["seed"], prefill=prefill)
