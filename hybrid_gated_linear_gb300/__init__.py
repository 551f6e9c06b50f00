"""GB300 (sm_103a) Lizard-attention operator: a thin Python binding of ``include/lizard.h``.

Every function below has the name of a C entry point and only marshals arguments:
tensors become device pointers, the stream becomes a ``cudaStream_t``, and a non-OK
status raises :class:`LizardError`.  All arithmetic runs in the library's CUDA kernels;
there is no Python or CPU fallback.  Call :func:`build`
once to compile ``_build/liblizard.so``; importing works without it, but every call
raises until the library is present.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build_lib import LIB as LIB_PATH
from .build_lib import build as _build

__all__ = [
    "LizardError", "build", "library", "lizard_dims", "lizard_decode_dims",
    "lizard_attn_fwd", "lizard_attn_bwd", "lizard_decode_step", "lizard_chunk_cumsum",
    "lizard_fwd_workspace_bytes", "lizard_bwd_workspace_bytes", "lizard_decode_workspace_bytes",
    "lizard_workspace_init", "lizard_check_device_errors", "lizard_status_string",
    "lizard_abi_version", "lizard_last_launch_count", "lizard_trace_enable", "lizard_trace_read",
    "lizard_decode_step_noalloc", "LIZARD_NOALLOC_MAX_SEQUENCES",
    "lizard_attn_fwd_bwd_host", "lizard_fwd_bwd_host_workspace_bytes",
    "lizard_decode_ring_fill", "lizard_state_combine", "lizard_fmap_dims",
    "lizard_feature_map_fwd", "lizard_feature_map_bwd", "lizard_feature_map_workspace_bytes",
    "lizard_attn_fwd_fmap", "lizard_selftest_wait_timeout", "lizard_gate_dims",
    "lizard_gate_fwd", "lizard_gate_bwd", "lizard_gate_workspace_bytes", "lizard_gla_std_fwd",
    "lizard_gla_std_workspace_bytes", "LIZARD_F32", "LIZARD_BF16", "EXPORTED_SYMBOLS",
]

LIZARD_F32 = 0
LIZARD_BF16 = 1
LIZARD_NOALLOC_MAX_SEQUENCES = 16384

EXPORTED_SYMBOLS = (
    "lizard_attn_fwd", "lizard_attn_bwd", "lizard_decode_step", "lizard_chunk_cumsum",
    "lizard_fwd_workspace_bytes", "lizard_bwd_workspace_bytes", "lizard_decode_workspace_bytes",
    "lizard_workspace_init", "lizard_check_device_errors", "lizard_status_string",
    "lizard_abi_version", "lizard_last_launch_count", "lizard_trace_enable", "lizard_trace_read",
    "lizard_decode_step_noalloc", "lizard_attn_fwd_bwd_host", "lizard_fwd_bwd_host_workspace_bytes",
    "lizard_decode_ring_fill", "lizard_state_combine", "lizard_feature_map_fwd",
    "lizard_feature_map_bwd", "lizard_feature_map_workspace_bytes", "lizard_attn_fwd_fmap",
    "lizard_selftest_wait_timeout", "lizard_gate_fwd", "lizard_gate_bwd",
    "lizard_gate_workspace_bytes", "lizard_gla_std_fwd", "lizard_gla_std_workspace_bytes",
)

STATUS_NAMES = {0: "LIZARD_OK", 1: "LIZARD_ERR_INVALID_ARG", 2: "LIZARD_ERR_UNSUPPORTED",
                3: "LIZARD_ERR_CUDA", 4: "LIZARD_ERR_TIMEOUT", 5: "LIZARD_ERR_DEVICE_CHECK",
                6: "LIZARD_ERR_WORKSPACE"}


class LizardError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{what}: {name} ({lizard_status_string(status)})")


class lizard_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("M", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float)]


class lizard_decode_dims(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int32), ("H", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("M", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class lizard_gate_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32),
                ("D", ctypes.c_int32), ("dk", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("tau", ctypes.c_float)]


class lizard_fmap_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32),
                ("D", ctypes.c_int32), ("F", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (see build_lib.py)."""
    return _build(force=force)


def library():
    """The loaded ctypes library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {LIB_PATH} is missing: run hybrid_gated_linear_gb300.build()")
            lib = ctypes.CDLL(LIB_PATH)
            P, I32, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            DP, DDP = ctypes.POINTER(lizard_dims), ctypes.POINTER(lizard_decode_dims)
            FMP = ctypes.POINTER(lizard_fmap_dims)
            GDP = ctypes.POINTER(lizard_gate_dims)
            sig = {
                "lizard_attn_fwd": (I32, [DP] + [P] * 8 + [I32, F, P, P, P, P, SZ, P]),
                "lizard_attn_bwd": (I32, [DP] + [P] * 8 + [I32, F] + [P] * 12 + [P, SZ, P]),
                "lizard_decode_step": (I32, [DDP] + [P] * 8 + [I32, F] + [P] * 5 + [P, SZ, P]),
                "lizard_chunk_cumsum": (I32, [I32, I32, I32, I32, P, P, P, P]),
                "lizard_fwd_workspace_bytes": (SZ, [DP, I32]),
                "lizard_bwd_workspace_bytes": (SZ, [DP, I32]),
                "lizard_decode_workspace_bytes": (SZ, [DDP]),
                "lizard_workspace_init": (I32, [P, SZ, P]),
                "lizard_check_device_errors": (I32, [P, P]),
                "lizard_status_string": (ctypes.c_char_p, [I32]),
                "lizard_abi_version": (I32, []),
                "lizard_last_launch_count": (I32, []),
                "lizard_trace_enable": (I32, [I32]),
                "lizard_trace_read": (I32, [ctypes.c_char_p, I32, ctypes.POINTER(F), I32]),
                "lizard_decode_step_noalloc": (I32, [DDP] + [P] * 8 + [I32, F] + [P] * 5 + [P]),
                "lizard_fwd_bwd_host_workspace_bytes": (SZ, [DP, I32]),
                "lizard_decode_ring_fill": (I32, [DDP, I32, I32] + [P] * 5 + [P]),
                "lizard_state_combine": (I32, [I32, I32, I32] + [P] * 6 + [P]),
                "lizard_feature_map_workspace_bytes": (SZ, [FMP, I32]),
                "lizard_attn_fwd_fmap": (I32, [DP] + [P] * 10 + [I32, F, P, P, P, P, SZ, P]),
                "lizard_feature_map_fwd": (I32, [FMP, P, P, P, P, SZ, P]),
                "lizard_feature_map_bwd": (I32, [FMP, P, P, P, P, P, P, SZ, P]),
                "lizard_attn_fwd_bwd_host": (I32, [DP] + [P] * 8 + [I32, F] + [P] * 13 + [P, SZ, P]),
                "lizard_selftest_wait_timeout": (I32, [P, SZ, ctypes.c_int64, P]),
                "lizard_gate_workspace_bytes": (SZ, [GDP]),
                "lizard_gate_fwd": (I32, [GDP, P, P, P, P]),
                "lizard_gate_bwd": (I32, [GDP, P, P, P, P, P, P, SZ, P]),
                "lizard_gla_std_workspace_bytes": (SZ, [DP]),
                "lizard_gla_std_fwd": (I32, [DP] + [P] * 8 + [SZ, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


# ------------------------------------------------------------------------------------
# marshalling helpers
# ------------------------------------------------------------------------------------
def _ptr(t):
    """Device pointer of a tensor (None -> NULL).  Requires a contiguous tensor."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    handle = getattr(stream, "cuda_stream", stream)
    return ctypes.c_void_p(int(handle))


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return LIZARD_F32
    if t.dtype == torch.bfloat16:
        return LIZARD_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(status: int, what: str):
    if status != 0:
        raise LizardError(status, what)


def lizard_status_string(status: int) -> str:
    try:
        return library().lizard_status_string(status).decode()
    except RuntimeError:
        return STATUS_NAMES.get(status, "unknown")


def lizard_abi_version() -> int:
    return library().lizard_abi_version()


def lizard_last_launch_count() -> int:
    return library().lizard_last_launch_count()


def make_dims(B, H, L, dk, dv, M, dtype, scale=0.0) -> lizard_dims:
    return lizard_dims(B, H, L, dk, dv, M, dtype, scale)


def lizard_fwd_workspace_bytes(dims: lizard_dims, W: int) -> int:
    return library().lizard_fwd_workspace_bytes(ctypes.byref(dims), W)


def lizard_bwd_workspace_bytes(dims: lizard_dims, W: int) -> int:
    return library().lizard_bwd_workspace_bytes(ctypes.byref(dims), W)


def lizard_fwd_bwd_host_workspace_bytes(dims: lizard_dims, W: int) -> int:
    return library().lizard_fwd_bwd_host_workspace_bytes(ctypes.byref(dims), W)


def lizard_decode_workspace_bytes(dims: lizard_decode_dims) -> int:
    return library().lizard_decode_workspace_bytes(ctypes.byref(dims))


def lizard_workspace_init(workspace, stream=None):
    _check(library().lizard_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)), "lizard_workspace_init")


def lizard_check_device_errors(workspace, stream=None) -> int:
    """Synchronises the stream and returns the device status (0 = OK); does not raise."""
    return library().lizard_check_device_errors(_ptr(workspace), _stream(stream))


def lizard_selftest_wait_timeout(workspace, wait_cycles: int, stream=None):
    """Makes one bounded device wait run out on purpose (see include/lizard.h)."""
    _check(library().lizard_selftest_wait_timeout(_ptr(workspace), _ws_bytes(workspace),
                                                  int(wait_cycles), _stream(stream)),
           "lizard_selftest_wait_timeout")


def lizard_gate_workspace_bytes(dims: lizard_gate_dims) -> int:
    return library().lizard_gate_workspace_bytes(ctypes.byref(dims))


def lizard_gate_fwd(dims: lizard_gate_dims, x, w, log_gamma, stream=None):
    """log_gamma = logsigmoid(x W) / tau into preallocated ``log_gamma``."""
    _check(library().lizard_gate_fwd(ctypes.byref(dims), _ptr(x), _ptr(w), _ptr(log_gamma),
                                     _stream(stream)), "lizard_gate_fwd")


def lizard_gate_bwd(dims: lizard_gate_dims, x, w, d_log_gamma, d_x, d_w, workspace, stream=None):
    """d_x and d_w of the gate projection from d_log_gamma."""
    _check(library().lizard_gate_bwd(ctypes.byref(dims), _ptr(x), _ptr(w), _ptr(d_log_gamma),
                                     _ptr(d_x), _ptr(d_w), _ptr(workspace), _ws_bytes(workspace),
                                     _stream(stream)), "lizard_gate_bwd")


def _ws_bytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def lizard_attn_fwd(dims: lizard_dims, phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, W: int,
                    alpha: float, y, h0, h_final, workspace, stream=None):
    """Forward pass into preallocated ``y`` (and ``h_final`` if given)."""
    st = library().lizard_attn_fwd(ctypes.byref(dims), _ptr(phi_q), _ptr(phi_k), _ptr(v),
                                   _ptr(log_gamma), _ptr(q), _ptr(k), _ptr(meta_k), _ptr(meta_v),
                                   int(W), float(alpha), _ptr(y), _ptr(h0), _ptr(h_final),
                                   _ptr(workspace), _ws_bytes(workspace), _stream(stream))
    _check(st, "lizard_attn_fwd")


def lizard_gla_std_workspace_bytes(dims: lizard_dims) -> int:
    return library().lizard_gla_std_workspace_bytes(ctypes.byref(dims))


def lizard_gla_std_fwd(dims: lizard_dims, phi_q, phi_k, v, log_gamma, y, h0, h_final, workspace,
                       stream=None):
    """The standard fp32 chunkwise GLA forward (GLA branch only) into preallocated ``y``."""
    st = library().lizard_gla_std_fwd(ctypes.byref(dims), _ptr(phi_q), _ptr(phi_k), _ptr(v),
                                      _ptr(log_gamma), _ptr(y), _ptr(h0), _ptr(h_final),
                                      _ptr(workspace), _ws_bytes(workspace), _stream(stream))
    _check(st, "lizard_gla_std_fwd")


def lizard_attn_bwd(dims: lizard_dims, phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v, W: int,
                    alpha: float, h0, dy, d_phi_q, d_phi_k, d_v, d_log_gamma, d_q, d_k,
                    d_meta_k, d_meta_v, d_h0, workspace, stream=None, fwd_workspace=None):
    """Backward pass into preallocated gradient tensors.  ``fwd_workspace``: the workspace
    of the matching lizard_attn_fwd call, whose chunk features and states are reused."""
    st = library().lizard_attn_bwd(ctypes.byref(dims), _ptr(phi_q), _ptr(phi_k), _ptr(v),
                                   _ptr(log_gamma), _ptr(q), _ptr(k), _ptr(meta_k), _ptr(meta_v),
                                   int(W), float(alpha), _ptr(h0), _ptr(dy), _ptr(d_phi_q),
                                   _ptr(d_phi_k), _ptr(d_v), _ptr(d_log_gamma), _ptr(d_q),
                                   _ptr(d_k), _ptr(d_meta_k), _ptr(d_meta_v), _ptr(d_h0),
                                   _ptr(fwd_workspace), _ptr(workspace), _ws_bytes(workspace),
                                   _stream(stream))
    _check(st, "lizard_attn_bwd")


def lizard_decode_step(dims: lizard_decode_dims, phi_q, phi_k, v, log_gamma, q, k, meta_k,
                       meta_v, W: int, alpha: float, h, k_ring, v_ring, pos, y, workspace,
                       stream=None):
    """One decode step; h, rings and pos are updated in place."""
    st = library().lizard_decode_step(ctypes.byref(dims), _ptr(phi_q), _ptr(phi_k), _ptr(v),
                                      _ptr(log_gamma), _ptr(q), _ptr(k), _ptr(meta_k),
                                      _ptr(meta_v), int(W), float(alpha), _ptr(h), _ptr(k_ring),
                                      _ptr(v_ring), _ptr(pos), _ptr(y), _ptr(workspace),
                                      _ws_bytes(workspace), _stream(stream))
    _check(st, "lizard_decode_step")


def lizard_chunk_cumsum(units: int, L: int, dk: int, chunk: int, log_gamma, b, gamma_chunk=None,
                        stream=None):
    st = library().lizard_chunk_cumsum(int(units), int(L), int(dk), int(chunk), _ptr(log_gamma),
                                       _ptr(b), _ptr(gamma_chunk), _stream(stream))
    _check(st, "lizard_chunk_cumsum")


def lizard_trace_enable(enable: bool = True):
    """Turn per-kernel event timing on or off for the calling host thread."""
    _check(library().lizard_trace_enable(1 if enable else 0), "lizard_trace_enable")


def lizard_trace_read(max_records: int = 4096):
    """Wait for the traced kernels and return [(kernel_name, milliseconds), ...]."""
    name_len = 64
    names = ctypes.create_string_buffer(name_len * max_records)
    ms = (ctypes.c_float * max_records)()
    n = library().lizard_trace_read(names, name_len, ms, max_records)
    raw = names.raw
    return [(raw[i * name_len:(i + 1) * name_len].split(b"\0", 1)[0].decode(), float(ms[i]))
            for i in range(n)]


def lizard_decode_step_noalloc(dims: lizard_decode_dims, phi_q, phi_k, v, log_gamma, q, k,
                               meta_k, meta_v, W: int, alpha: float, h, k_ring, v_ring, pos, y,
                               stream=None):
    """lizard_decode_step without a workspace, for callers that cannot allocate device
    memory: the library's own fixed device array holds the per-sequence counters (N at
    most LIZARD_NOALLOC_MAX_SEQUENCES).  Calls that overlap on the GPU race on that array."""
    st = library().lizard_decode_step_noalloc(ctypes.byref(dims), _ptr(phi_q), _ptr(phi_k),
                                              _ptr(v), _ptr(log_gamma), _ptr(q), _ptr(k),
                                              _ptr(meta_k), _ptr(meta_v), int(W), float(alpha),
                                              _ptr(h), _ptr(k_ring), _ptr(v_ring), _ptr(pos),
                                              _ptr(y), _stream(stream))
    _check(st, "lizard_decode_step_noalloc")


def lizard_attn_fwd_bwd_host(dims: lizard_dims, phi_q, phi_k, v, log_gamma, q, k, meta_k, meta_v,
                             W: int, alpha: float, h0, dy, y, h_final, d_phi_q, d_phi_k, d_v,
                             d_log_gamma, d_q, d_k, d_meta_k, d_meta_v, d_h0, workspace,
                             stream=None):
    """Forward + backward with every tensor in host memory (CPU tensors, pinned for overlap);
    ``workspace`` is a device tensor of lizard_fwd_bwd_host_workspace_bytes bytes.  Returns
    once the work is queued; synchronise the stream before reading the outputs."""
    st = library().lizard_attn_fwd_bwd_host(
        ctypes.byref(dims), _ptr(phi_q), _ptr(phi_k), _ptr(v), _ptr(log_gamma), _ptr(q), _ptr(k),
        _ptr(meta_k), _ptr(meta_v), int(W), float(alpha), _ptr(h0), _ptr(dy), _ptr(y),
        _ptr(h_final), _ptr(d_phi_q), _ptr(d_phi_k), _ptr(d_v), _ptr(d_log_gamma), _ptr(d_q),
        _ptr(d_k), _ptr(d_meta_k), _ptr(d_meta_v), _ptr(d_h0), _ptr(workspace),
        _ws_bytes(workspace), _stream(stream))
    _check(st, "lizard_attn_fwd_bwd_host")


def lizard_decode_ring_fill(dims: lizard_decode_dims, L: int, W: int, k, v, k_ring, v_ring, pos,
                            stream=None):
    """Fills the decode rings and positions from a prefill's last W keys and values."""
    st = library().lizard_decode_ring_fill(ctypes.byref(dims), int(L), int(W), _ptr(k), _ptr(v),
                                           _ptr(k_ring), _ptr(v_ring), _ptr(pos), _stream(stream))
    _check(st, "lizard_decode_ring_fill")


def lizard_state_combine(units: int, dk: int, dv: int, gamma_a, h_a, gamma_b, h_b, gamma_out,
                         h_out, stream=None):
    """(gamma_out, h_out) = (gamma_a, h_a) o (gamma_b, h_b): segment a followed by segment b."""
    st = library().lizard_state_combine(int(units), int(dk), int(dv), _ptr(gamma_a), _ptr(h_a),
                                        _ptr(gamma_b), _ptr(h_b), _ptr(gamma_out), _ptr(h_out),
                                        _stream(stream))
    _check(st, "lizard_state_combine")


def lizard_feature_map_workspace_bytes(dims: lizard_fmap_dims, is_bwd: bool) -> int:
    return int(library().lizard_feature_map_workspace_bytes(ctypes.byref(dims), int(bool(is_bwd))))


def lizard_feature_map_fwd(dims: lizard_fmap_dims, x, w, phi, workspace, stream=None):
    """phi = [exp(x W), exp(-x W)] per head (Hedgehog feature map)."""
    st = library().lizard_feature_map_fwd(ctypes.byref(dims), _ptr(x), _ptr(w), _ptr(phi),
                                          _ptr(workspace), _ws_bytes(workspace), _stream(stream))
    _check(st, "lizard_feature_map_fwd")


def lizard_feature_map_bwd(dims: lizard_fmap_dims, x, w, d_phi, d_x, d_w, workspace, stream=None):
    """Gradients of the feature map: d_x [B,H,L,D] and d_w [H,D,F] (fp32)."""
    st = library().lizard_feature_map_bwd(ctypes.byref(dims), _ptr(x), _ptr(w), _ptr(d_phi),
                                          _ptr(d_x), _ptr(d_w), _ptr(workspace), _ws_bytes(workspace),
                                          _stream(stream))
    _check(st, "lizard_feature_map_bwd")


def lizard_attn_fwd_fmap(dims: lizard_dims, x_q, x_k, w_q, w_k, v, log_gamma, q, k, meta_k,
                         meta_v, W: int, alpha: float, y, h0, h_final, workspace, stream=None):
    """Forward pass from the raw projections with the Hedgehog feature map fused into the
    log-space gate absorption (phi is never formed)."""
    st = library().lizard_attn_fwd_fmap(
        ctypes.byref(dims), _ptr(x_q), _ptr(x_k), _ptr(w_q), _ptr(w_k), _ptr(v), _ptr(log_gamma),
        _ptr(q), _ptr(k), _ptr(meta_k), _ptr(meta_v), int(W), float(alpha), _ptr(y), _ptr(h0),
        _ptr(h_final), _ptr(workspace), _ws_bytes(workspace), _stream(stream))
    _check(st, "lizard_attn_fwd_fmap")
