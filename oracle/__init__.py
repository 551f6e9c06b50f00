"""fp64 CPU oracle for the Lizard-attention operator -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg
of ``bench.py`` may import this module.  The CUDA library (``hybrid_gated_linear_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``lizard_oracle.c`` (plain C, fp64, token-by-token loops);
this module compiles it with gcc and marshals numpy arrays through ctypes.  Inputs of
any float dtype are widened to float64 exactly.

Sources: "Lizard: An Efficient Linearization Framework for Large Language Models"
(arXiv 2507.09025) -- Preliminaries, Method; the papernotes.org note on the same paper
-- 关键设计 (GLA recurrence, Anchor Window Attention) and 整体框架 (weighted merge).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lizard_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblizard_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, -O2, IEEE fp64, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            D, I, P = ctypes.c_double, ctypes.c_int, ctypes.c_void_p
            lib.oracle_fwd.argtypes = [I] * 7 + [D, D] + [P] * 13 + [I]
            lib.oracle_bwd.argtypes = [I] * 7 + [D, D] + [P] * 19 + [I]
            lib.oracle_decode_step.argtypes = [I] * 6 + [D, D] + [P] * 13 + [I]
            lib.oracle_chunk_cumsum.argtypes = [I, I, I, I, P, P, P]
            for f in (lib.oracle_fwd, lib.oracle_bwd, lib.oracle_decode_step,
                      lib.oracle_chunk_cumsum):
                f.restype = I
            lib.oracle_last_threads.restype = I
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def last_threads() -> int:
    """Host threads used by the most recent oracle call."""
    return _load().oracle_last_threads()


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def fwd(phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, W, alpha=1.0, scale=None,
        h0=None, want_branches=False, want_state=False, nthreads=0):
    """y = y_gla + alpha*y_win over [B,H,L,*] inputs; returns a dict of float64 arrays."""
    pq, pk, vv, lg, qq, kk = (_f64(x) for x in (phi_q, phi_k, v, log_gamma, q, k))
    B, H, L, dk = pq.shape
    dv = vv.shape[-1]
    mk, mv = _f64(meta_k), _f64(meta_v)
    M = 0 if mk is None else mk.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    y = np.zeros((B, H, L, dv))
    yg = np.zeros_like(y) if want_branches else None
    yw = np.zeros_like(y) if want_branches else None
    hf = np.zeros((B, H, dk, dv)) if want_state else None
    h0a = _f64(h0)
    rc = _load().oracle_fwd(B, H, L, dk, dv, M, int(W), float(alpha), float(scale),
                            _ptr(pq), _ptr(pk), _ptr(vv), _ptr(lg), _ptr(qq), _ptr(kk),
                            _ptr(mk), _ptr(mv), _ptr(h0a), _ptr(y), _ptr(yg), _ptr(yw),
                            _ptr(hf), int(nthreads))
    _check(rc, "fwd")
    out = {"y": y}
    if want_branches:
        out["y_gla"], out["y_win"] = yg, yw
    if want_state:
        out["h_final"] = hf
    return out


def bwd(phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, dy, W, alpha=1.0, scale=None,
        h0=None, want_dh0=False, nthreads=0):
    """Gradients of sum(y * dy) w.r.t. every input; returns a dict of float64 arrays."""
    pq, pk, vv, lg, qq, kk, dyy = (_f64(x) for x in (phi_q, phi_k, v, log_gamma, q, k, dy))
    B, H, L, dk = pq.shape
    dv = vv.shape[-1]
    mk, mv = _f64(meta_k), _f64(meta_v)
    M = 0 if mk is None else mk.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    g = {n: np.zeros((B, H, L, dk)) for n in ("d_phi_q", "d_phi_k", "d_log_gamma", "d_q", "d_k")}
    g["d_v"] = np.zeros((B, H, L, dv))
    g["d_meta_k"] = np.zeros((H, M, dk))
    g["d_meta_v"] = np.zeros((H, M, dv))
    dh0 = np.zeros((B, H, dk, dv)) if want_dh0 else None
    h0a = _f64(h0)
    rc = _load().oracle_bwd(B, H, L, dk, dv, M, int(W), float(alpha), float(scale),
                            _ptr(pq), _ptr(pk), _ptr(vv), _ptr(lg), _ptr(qq), _ptr(kk),
                            _ptr(mk), _ptr(mv), _ptr(h0a), _ptr(dyy),
                            _ptr(g["d_phi_q"]), _ptr(g["d_phi_k"]), _ptr(g["d_v"]),
                            _ptr(g["d_log_gamma"]), _ptr(g["d_q"]), _ptr(g["d_k"]),
                            _ptr(g["d_meta_k"]) if M else None,
                            _ptr(g["d_meta_v"]) if M else None, _ptr(dh0), int(nthreads))
    _check(rc, "bwd")
    if want_dh0:
        g["d_h0"] = dh0
    return g


def decode_step(state, phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, W, alpha=1.0,
                scale=None, nthreads=0):
    """One decode step over N sequences; ``state`` is a dict with float64 arrays
    ``h`` [N,H,dk,dv], ``k_ring`` [N,H,W,dk], ``v_ring`` [N,H,W,dv] and int64 ``pos`` [N],
    all updated in place.  Token inputs are [N,H,d].  Returns y [N,H,dv]."""
    pq, pk, vv, lg, qq, kk = (_f64(x) for x in (phi_q, phi_k, v, log_gamma, q, k))
    N, H, dk = pq.shape
    dv = vv.shape[-1]
    mk, mv = _f64(meta_k), _f64(meta_v)
    M = 0 if mk is None else mk.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    for name, dt in (("h", np.float64), ("k_ring", np.float64), ("v_ring", np.float64),
                     ("pos", np.int64)):
        a = state[name]
        if a.dtype != dt or not a.flags.c_contiguous:
            raise TypeError(f"state[{name!r}] must be a C-contiguous {dt.__name__} array")
    y = np.zeros((N, H, dv))
    rc = _load().oracle_decode_step(N, H, dk, dv, M, int(W), float(alpha), float(scale),
                                    _ptr(pq), _ptr(pk), _ptr(vv), _ptr(lg), _ptr(qq), _ptr(kk),
                                    _ptr(mk), _ptr(mv), _ptr(state["h"]), _ptr(state["k_ring"]),
                                    _ptr(state["v_ring"]), _ptr(state["pos"]), _ptr(y),
                                    int(nthreads))
    _check(rc, "decode_step")
    return y


def chunk_cumsum(log_gamma, chunk):
    """Chunk-local inclusive cumsum of log gamma over [..., L, dk]; returns (b, Gamma)."""
    lg = _f64(log_gamma)
    L, dk = lg.shape[-2:]
    lead = lg.shape[:-2]
    units = int(np.prod(lead)) if lead else 1
    nchunks = (L + chunk - 1) // chunk
    b = np.zeros_like(lg)
    G = np.zeros(lead + (nchunks, dk))
    rc = _load().oracle_chunk_cumsum(units, L, dk, int(chunk), _ptr(lg), _ptr(b), _ptr(G))
    _check(rc, "chunk_cumsum")
    return b, G


def state_combine(gamma_a, h_a, gamma_b, h_b):
    """Segment a followed by segment b ("Lizard", arXiv 2507.09025, Preliminaries: the
    recurrence h_i = diag(gamma_i) h_{i-1} + phi_k_i v_i^T): a segment with log-gate sum
    Gamma and final state h from a zero start maps h0 to diag(exp(Gamma)) h0 + h, so the
    pair composes as (Gamma_a + Gamma_b, diag(exp(Gamma_b)) h_a + h_b).  fp64 numpy over
    [..., dk] and [..., dk, dv]."""
    ga, ha, gb, hb = (_f64(a) for a in (gamma_a, h_a, gamma_b, h_b))
    return ga + gb, np.exp(gb)[..., :, None] * ha + hb


def feature_map(x, w):
    """Hedgehog feature map ("Lizard", arXiv 2507.09025, Method: the strictly
    non-negative map phi(x) = [exp(x W) (+) exp(-x W)]): x [B,H,L,D], per-head W [H,D,F]
    -> phi [B,H,L,2F], the F features exp(z) followed by the F features exp(-z) with
    z = x W.  fp64 numpy."""
    xx, ww = _f64(x), _f64(w)
    z = np.einsum("bhld,hdf->bhlf", xx, ww)
    return np.concatenate([np.exp(z), np.exp(-z)], axis=-1)


def feature_map_bwd(x, w, d_phi):
    """Adjoint of :func:`feature_map`: with z = x W and the two halves dphi+ (first F
    features) and dphi- (last F) of d_phi, dz = dphi+ exp(z) - dphi- exp(-z),
    dx = dz W^T and dW[h] = sum over batch and tokens of x^T dz.  Returns (dx, dW)."""
    xx, ww, dp = _f64(x), _f64(w), _f64(d_phi)
    F = ww.shape[-1]
    z = np.einsum("bhld,hdf->bhlf", xx, ww)
    dz = dp[..., :F] * np.exp(z) - dp[..., F:] * np.exp(-z)
    dx = np.einsum("bhlf,hdf->bhld", dz, ww)
    dw = np.einsum("bhld,bhlf->hdf", xx, dz)
    return dx, dw


def _logsigmoid(z):
    return np.where(z >= 0, -np.log1p(np.exp(-z)), z - np.log1p(np.exp(z)))


def gate(x, w, tau=16.0):
    """Gate projection ("Lizard", arXiv 2507.09025, Method: the trained gate projection
    W_gamma; papernotes.org note, 关键设计: gamma_i from W_gamma), in the form the library
    takes: log gamma = logsigmoid(x W) / tau with x [B,H,L,D] and per-head W [H,D,dk].
    fp64 numpy."""
    z = np.einsum("bhld,hdk->bhlk", _f64(x), _f64(w))
    return _logsigmoid(z) / tau


def gate_bwd(x, w, d_log_gamma, tau=16.0):
    """Adjoint of :func:`gate`: with z = x W, d logsigmoid(z)/dz = sigmoid(-z), so
    dz = d_log_gamma sigmoid(-z) / tau, dx = dz W^T and dW[h] = sum over batch and tokens
    of x^T dz.  Returns (dx, dW)."""
    xx, ww, dl = _f64(x), _f64(w), _f64(d_log_gamma)
    z = np.einsum("bhld,hdk->bhlk", xx, ww)
    dz = dl / (1.0 + np.exp(z)) / tau
    dx = np.einsum("bhlk,hdk->bhld", dz, ww)
    dw = np.einsum("bhld,bhlk->hdk", xx, dz)
    return dx, dw
