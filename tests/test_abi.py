"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, it
exports every function ``include/lizard.h`` declares, and argument validation returns
the documented status before anything is enqueued."""
import ctypes
import os
import re

import pytest

import hybrid_gated_linear_gb300 as lz

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lizard.h")

OK, INVALID, UNSUPPORTED, CUDA, TIMEOUT, CHECK, WORKSPACE = range(7)
A = 0x7f0000000000  # fake, 16-byte aligned device addresses: validation never dereferences


@pytest.fixture(scope="module")
def lib():
    lz.build()
    return lz.library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lizard_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert sorted(lz.EXPORTED_SYMBOLS) == _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_abi_version(lib):
    m = re.search(r"#define LIZARD_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.lizard_abi_version() == int(m.group(1))


def test_status_strings(lib):
    for s in range(7):
        assert lib.lizard_status_string(s)
    assert lz.lizard_status_string(OK) == "ok"


def _dims(**kw):
    d = dict(B=1, H=2, L=64, dk=128, dv=128, M=4, dtype=lz.LIZARD_BF16, scale=0.0)
    d.update(kw)
    return lz.lizard_dims(**d)


def _fwd(lib, dims, W=64, alpha=1.0, ptrs=None, ws=A + 0x100000, ws_bytes=1 << 20, meta=True):
    p = [ctypes.c_void_p(A + i * 0x1000000) for i in range(6)] if ptrs is None else ptrs
    mk = ctypes.c_void_p(A + 0x20000000) if meta else None
    mv = ctypes.c_void_p(A + 0x21000000) if meta else None
    y = ctypes.c_void_p(A + 0x30000000)
    return lib.lizard_attn_fwd(ctypes.byref(dims) if dims is not None else None, *p, mk, mv, W,
                               alpha, y, None, None, ctypes.c_void_p(ws) if ws else None,
                               ws_bytes, None)


def test_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, None) == INVALID
    assert _fwd(lib, _dims(), W=0) == INVALID
    assert _fwd(lib, _dims(B=0)) == INVALID
    assert _fwd(lib, _dims(M=17)) == INVALID
    assert _fwd(lib, _dims(M=-1)) == INVALID
    assert _fwd(lib, _dims(dtype=7)) == INVALID
    assert _fwd(lib, _dims(L=-3)) == INVALID
    assert _fwd(lib, _dims(), alpha=float("nan")) == INVALID
    assert _fwd(lib, _dims(M=2), meta=False) == INVALID
    bad = [ctypes.c_void_p(A + i * 0x1000000) for i in range(6)]
    bad[2] = ctypes.c_void_p(A + 8)  # misaligned v
    assert _fwd(lib, _dims(), ptrs=bad) == INVALID
    null = list(bad)
    null[2] = None
    assert _fwd(lib, _dims(), ptrs=null) == INVALID


def test_fwd_unsupported_shapes(lib):
    assert _fwd(lib, _dims(dk=96, dv=96)) == UNSUPPORTED
    assert _fwd(lib, _dims(dk=128, dv=64)) == UNSUPPORTED


def test_fwd_workspace_checks(lib):
    need = lib.lizard_fwd_workspace_bytes(ctypes.byref(_dims()), 64)
    assert need >= 4
    assert _fwd(lib, _dims(), ws=None, ws_bytes=0) == WORKSPACE
    assert _fwd(lib, _dims(), ws_bytes=need - 1) == WORKSPACE


def test_fwd_rejects_output_aliasing_an_input(lib):
    p = [ctypes.c_void_p(A + i * 0x1000000) for i in range(6)]
    dims = _dims()
    y = p[0]  # y == phi_q
    st = lib.lizard_attn_fwd(ctypes.byref(dims), *p, ctypes.c_void_p(A + 0x20000000),
                             ctypes.c_void_p(A + 0x21000000), 64, 1.0, y, None, None,
                             ctypes.c_void_p(A + 0x40000000), 1 << 20, None)
    assert st == INVALID


def test_bwd_workspace_grows_with_problem(lib):
    small = lib.lizard_bwd_workspace_bytes(ctypes.byref(_dims(L=64)), 64)
    big = lib.lizard_bwd_workspace_bytes(ctypes.byref(_dims(L=4096, B=2)), 64)
    assert 0 < small < big
    assert lib.lizard_bwd_workspace_bytes(ctypes.byref(_dims(dk=96, dv=96)), 64) == 0


def test_bwd_rejects_bad_arguments(lib):
    dims = _dims()
    P = lambda i: ctypes.c_void_p(A + i * 0x1000000)
    args = [P(i) for i in range(8)]
    grads = [P(20 + i) for i in range(8)]
    ws = P(40)
    need = lib.lizard_bwd_workspace_bytes(ctypes.byref(dims), 64)
    st = lib.lizard_attn_bwd(ctypes.byref(dims), *args, 64, 1.0, None, P(10), *grads, None, None,
                             ws, need - 1, None)
    assert st == WORKSPACE
    grads2 = list(grads)
    grads2[1] = grads2[0]  # two outputs alias
    st = lib.lizard_attn_bwd(ctypes.byref(dims), *args, 64, 1.0, None, P(10), *grads2, None, None,
                             ws, need, None)
    assert st == INVALID


def test_decode_rejects_bad_arguments(lib):
    d = lz.lizard_decode_dims(4, 2, 128, 128, 4, lz.LIZARD_BF16, 0.0)
    P = lambda i: ctypes.c_void_p(A + i * 0x1000000)
    base = [P(i) for i in range(8)]
    need = lib.lizard_decode_workspace_bytes(ctypes.byref(d))
    assert need > 0

    def call(W=64, ws_bytes=need, dims=d, extra=None):
        outs = [P(20 + i) for i in range(5)] if extra is None else extra
        return lib.lizard_decode_step(ctypes.byref(dims), *base, W, 1.0, *outs, P(40), ws_bytes,
                                      None)

    assert call(W=0) == INVALID
    assert call(W=4096) == INVALID
    assert call(ws_bytes=need - 1) == WORKSPACE
    outs = [P(20 + i) for i in range(5)]
    outs[4] = base[0]  # y aliases phi_q
    assert call(extra=outs) == INVALID
    d2 = lz.lizard_decode_dims(4, 2, 80, 80, 4, lz.LIZARD_BF16, 0.0)
    assert call(dims=d2) == UNSUPPORTED


def test_chunk_cumsum_rejects_bad_arguments(lib):
    P = lambda i: ctypes.c_void_p(A + i * 0x1000000)
    assert lib.lizard_chunk_cumsum(0, 10, 4, 64, P(0), P(1), None, None) == INVALID
    assert lib.lizard_chunk_cumsum(1, 10, 4, 0, P(0), P(1), None, None) == INVALID
    assert lib.lizard_chunk_cumsum(1, 10, 4, 64, P(0), P(0), None, None) == INVALID
    assert lib.lizard_chunk_cumsum(1, 10, 4, 64, P(0), None, None, None) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    # monkeypatch restores the loaded library and its path afterwards
    monkeypatch.setattr(lz, "_lib", None)
    monkeypatch.setattr(lz, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        lz.library()


def test_feature_map_rejects_bad_arguments(lib):
    P = lambda i: ctypes.c_void_p(A + i * 0x1000000)
    d = lz.lizard_fmap_dims(1, 2, 300, 128, 64, lz.LIZARD_BF16)
    ws_f = lz.lizard_feature_map_workspace_bytes(d, False)
    ws_b = lz.lizard_feature_map_workspace_bytes(d, True)
    assert ws_f == 256
    # dW partials: one 128x64 fp32 block per (b, h, group of four 128-token tiles)
    assert ws_b == 256 + 2 * 1 * 128 * 64 * 4
    fwd = lambda dims=d, x=P(0), w=P(1), phi=P(2), ws=P(3), n=ws_f: lib.lizard_feature_map_fwd(
        ctypes.byref(dims), x, w, phi, ws, n, None)
    assert fwd(x=None) == INVALID
    assert fwd(w=ctypes.c_void_p(A + 8)) == INVALID          # misaligned
    assert fwd(phi=P(0)) == INVALID                          # output over the input
    assert fwd(n=ws_f - 1) == WORKSPACE
    assert fwd(ws=None) == WORKSPACE
    for bad in (lz.lizard_fmap_dims(1, 2, 300, 0, 64, 1), lz.lizard_fmap_dims(1, 2, 300, 128, 129, 1),
                lz.lizard_fmap_dims(1, 2, 300, 256, 128, 1), lz.lizard_fmap_dims(0, 2, 300, 128, 64, 1),
                lz.lizard_fmap_dims(1, 2, -1, 128, 64, 1), lz.lizard_fmap_dims(1, 2, 300, 128, 64, 7)):
        assert fwd(dims=bad) == INVALID
        assert lz.lizard_feature_map_workspace_bytes(bad, True) == 0
    bwd = lambda x=P(0), w=P(1), dp=P(2), dx=P(3), dw=P(4), ws=P(5), n=ws_b: lib.lizard_feature_map_bwd(
        ctypes.byref(d), x, w, dp, dx, dw, ws, n, None)
    assert bwd(dw=None) == INVALID
    assert bwd(dx=P(2)) == INVALID
    assert bwd(dw=P(3)) == INVALID
    assert bwd(n=ws_b - 256) == WORKSPACE
    # both paths keep one partial per 512 tokens, whichever one runs
    d32 = lz.lizard_fmap_dims(1, 2, 1100, 64, 32, lz.LIZARD_F32)
    assert lz.lizard_feature_map_workspace_bytes(d32, True) == 256 + 2 * 3 * 64 * 32 * 4


def test_fused_forward_and_phi_free_backward_validation(lib):
    P = lambda i: ctypes.c_void_p(A + i * 0x10000000)
    d = lz.lizard_dims(1, 2, 300, 128, 128, 4, lz.LIZARD_BF16, 0.0)
    ws = lz.lizard_fwd_workspace_bytes(d, 64)

    def fwd(dims=d, xq=P(0), xk=P(1), wq=P(2), wk=P(3), y=P(10)):
        return lib.lizard_attn_fwd_fmap(ctypes.byref(dims), xq, xk, wq, wk, P(4), P(5), P(6), P(7),
                                        P(8), P(9), 64, 1.0, y, None, None, P(11), ws, None)
    assert fwd(xq=None) == INVALID
    assert fwd(wk=None) == INVALID
    assert fwd(wq=ctypes.c_void_p(A + 2 * 0x10000000 + 8)) == INVALID  # misaligned
    # only the tensor-core shape exists fused: fp32 and d = 64 are unsupported
    for bad in (lz.lizard_dims(1, 2, 300, 128, 128, 4, lz.LIZARD_F32, 0.0),
                lz.lizard_dims(1, 2, 300, 64, 64, 4, lz.LIZARD_BF16, 0.0)):
        assert fwd(dims=bad) == UNSUPPORTED
    # the backward needs phi unless the forward's saved context stands in for it
    dh = lambda i: ctypes.c_void_p(A + (20 + i) * 0x10000000)
    wsb = lz.lizard_bwd_workspace_bytes(d, 64)
    rc = lib.lizard_attn_bwd(ctypes.byref(d), None, None, P(4), P(5), P(6), P(7), P(8), P(9), 64,
                             1.0, None, P(12), dh(0), dh(1), dh(2), dh(3), dh(4), dh(5), dh(6),
                             dh(7), None, None, dh(8), wsb, None)
    assert rc == INVALID


def _std(lib, dims, ptrs=None, y=A + 0x30000000, ws=A + 0x40000000, ws_bytes=1 << 30):
    p = [ctypes.c_void_p(A + i * 0x1000000) for i in range(4)] if ptrs is None else ptrs
    return lib.lizard_gla_std_fwd(ctypes.byref(dims) if dims is not None else None, *p,
                                  ctypes.c_void_p(y) if y else None, None, None,
                                  ctypes.c_void_p(ws) if ws else None, ws_bytes, None)


def test_gla_std_workspace_is_every_chunk_state(lib):
    """One fp32 D x D state and one Gamma row per 64-token chunk, after the 256-byte header
    (each part rounded up to 256 bytes)."""
    for B, H, L, d in ((1, 2, 64, 128), (2, 3, 300, 64), (1, 1, 1, 128)):
        nc = (L + 63) // 64
        up = lambda x: (x + 255) // 256 * 256
        want = 256 + up(B * H * nc * d * d * 4) + up(B * H * nc * d * 4)
        got = lib.lizard_gla_std_workspace_bytes(ctypes.byref(_dims(B=B, H=H, L=L, dk=d, dv=d)))
        assert got == want, (B, H, L, d)
    assert lib.lizard_gla_std_workspace_bytes(ctypes.byref(_dims(dk=96, dv=96))) == 0
    assert lib.lizard_gla_std_workspace_bytes(None) == 0


def test_gla_std_rejects_bad_arguments(lib):
    assert _std(lib, None) == INVALID
    assert _std(lib, _dims(B=0)) == INVALID
    assert _std(lib, _dims(dtype=7)) == INVALID
    assert _std(lib, _dims(dk=96, dv=96)) == UNSUPPORTED
    assert _std(lib, _dims(dk=128, dv=64)) == UNSUPPORTED
    assert _std(lib, _dims(B=300, H=300)) == UNSUPPORTED  # B*H above one grid dimension
    bad = [ctypes.c_void_p(A + i * 0x1000000) for i in range(4)]
    bad[1] = ctypes.c_void_p(A + 8)  # misaligned phi_k
    assert _std(lib, _dims(), ptrs=bad) == INVALID
    assert _std(lib, _dims(), y=None) == INVALID
    assert _std(lib, _dims(), y=A) == INVALID  # y over phi_q
    assert _std(lib, _dims(), ws=None, ws_bytes=0) == WORKSPACE
    need = lib.lizard_gla_std_workspace_bytes(ctypes.byref(_dims()))
    assert _std(lib, _dims(), ws_bytes=need - 1) == WORKSPACE
