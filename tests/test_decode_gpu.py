"""Decode step: CUDA path vs the oracle's stepwise recurrence, and the invariant that
decoding from an empty state reproduces the forward pass."""
import numpy as np
import pytest
import torch

import hybrid_gated_linear_gb300 as lz
import oracle
import synth
from gpu_util import NAMES, TOK, TOL, code, gpu_fwd, host, rel_l2, torch_dtype

pytestmark = pytest.mark.gpu


class GpuDecoder:
    def __init__(self, stream: synth.DecodeStream, units=None):
        s = stream
        self.s = s
        td = torch_dtype(s.dtype)
        self.dims = lz.lizard_decode_dims(s.N, s.H, s.dk, s.dv, s.M, code(s.dtype), 0.0)
        self.h = torch.from_numpy(s.h0).cuda()
        self.kr = torch.from_numpy(s.k_ring).cuda().to(td)
        self.vr = torch.from_numpy(s.v_ring).cuda().to(td)
        self.pos = torch.from_numpy(s.pos0).cuda()
        self.mk = torch.from_numpy(s.meta_k).cuda().to(td)
        self.mv = torch.from_numpy(s.meta_v).cuda().to(td)
        self.ws = torch.zeros(lz.lizard_decode_workspace_bytes(self.dims), dtype=torch.uint8,
                              device="cuda")
        self.y = torch.empty(s.N, s.H, s.dv, dtype=td, device="cuda")

    def step(self, tok, alpha=1.0):
        td = torch_dtype(self.s.dtype)
        t = {n: torch.from_numpy(tok[n]).cuda() for n in TOK}
        for n in TOK:
            if n != "log_gamma":
                t[n] = t[n].to(td)
        lz.lizard_decode_step(self.dims, *(t[n] for n in TOK), self.mk, self.mv, self.s.W, alpha,
                              self.h, self.kr, self.vr, self.pos, self.y, self.ws)
        return host(self.y)


def _oracle_state(s, sel_n, sel_h):
    return dict(h=s.h0[np.ix_(sel_n, sel_h)].astype(np.float64).copy(),
                k_ring=s.k_ring[np.ix_(sel_n, sel_h)].astype(np.float64).copy(),
                v_ring=s.v_ring[np.ix_(sel_n, sel_h)].astype(np.float64).copy(),
                pos=s.pos0[sel_n].copy())


@pytest.mark.parametrize("dtype,W,M,steps,prefill", [
    ("f32", 8, 2, 20, True),      # ring wraps twice
    ("bf16", 64, 4, 70, True),
    ("bf16", 16, 0, 40, False),   # empty ring at start: min(pos+1, W) keys
    ("f32", 5, 3, 12, False),
])
def test_decode_matches_oracle(dtype, W, M, steps, prefill):
    s = synth.DecodeStream(3, 2, 128, 128, M, W, dtype, seed=300 + W, prefill=prefill)
    g = GpuDecoder(s)
    st = _oracle_state(s, [0, 1, 2], [0, 1])
    for _ in range(steps):
        tok = s.next_token()
        y = g.step(tok, alpha=0.9)
        yr = oracle.decode_step(st, *(tok[n] for n in TOK), s.meta_k, s.meta_v, W=W, alpha=0.9)
        assert rel_l2(y, yr) <= TOL[dtype]
    assert rel_l2(g.h.cpu().numpy(), st["h"]) <= TOL[dtype]
    np.testing.assert_array_equal(g.pos.cpu().numpy(), st["pos"])
    kr_ref = st["k_ring"]
    np.testing.assert_array_equal(g.kr.float().cpu().numpy(), kr_ref.astype(np.float32))


def test_decode_from_empty_equals_forward():
    """Recurrent form == parallel form on the GPU: L decode steps from pos = 0, h = 0 give
    the forward pass's outputs and final state."""
    B, H, L, d, W, M = 2, 2, 150, 128, 16, 3
    x = synth.make_fwd_inputs(B, H, L, d, d, M, "f32", "plain", seed=31)
    yf, hf = gpu_fwd(x, W, "f32", want_hf=True)
    s = synth.DecodeStream(B, H, d, d, M, W, "f32", seed=0, prefill=False)
    s.meta_k, s.meta_v = x["meta_k"], x["meta_v"]
    g = GpuDecoder(s)
    ys = []
    for t in range(L):
        tok = {n: np.ascontiguousarray(x[n][:, :, t]) for n in TOK}
        ys.append(g.step(tok))
    yd = np.stack(ys, axis=2)
    assert rel_l2(yd, yf) <= 1e-5
    assert rel_l2(g.h.cpu().numpy(), hf) <= 1e-5


def test_decode_workload_sampled_units():
    """64 sequences x 32 heads, W = 64, M = 4, 1024 steps in the shipped launch
    configuration; the oracle follows sequences {0, 41} x heads {0, 31} step by step:
    every step's output, and the state at steps 256, 512, 768 and 1024."""
    w = synth.WORKLOADS["decode_64x32"]
    s = synth.decode_stream("decode_64x32")
    g = GpuDecoder(s)
    sel_n, sel_h = [0, 41], [0, 31]
    st = _oracle_state(s, sel_n, sel_h)
    mk, mv = s.meta_k[sel_h], s.meta_v[sel_h]
    worst = 0.0
    for step in range(1, w["steps"] + 1):
        tok = s.next_token()
        y = g.step(tok)
        sub = {n: np.ascontiguousarray(tok[n][np.ix_(sel_n, sel_h)]) for n in TOK}
        yr = oracle.decode_step(st, *(sub[n] for n in TOK), mk, mv, W=w["W"])
        worst = max(worst, rel_l2(y[np.ix_(sel_n, sel_h)], yr))
        if step % 256 == 0:
            hs = g.h[sel_n][:, sel_h].cpu().numpy()
            assert rel_l2(hs, st["h"]) <= TOL["bf16"], step
    assert worst <= TOL["bf16"], worst
    np.testing.assert_array_equal(g.pos.cpu().numpy(), np.full(64, 64 + 1024))
