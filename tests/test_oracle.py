"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks the oracle against something independent: a different formula from
the pages (the quadratic form and the parallel form with the cumulative gate matrix), a
closed form (gamma = 1 gives causal linear attention), a library routine (PyTorch's
causal softmax attention when the window covers everything), exact index-revealing
inputs, central finite differences, and invariants (decode equals the forward pass;
splitting the sequence and carrying the state changes nothing; the log-gate gradient
equals a reverse cumulative sum of a per-token identity).

Sources: "Lizard: An Efficient Linearization Framework for Large Language Models"
(arXiv 2507.09025): Preliminaries (linear attention, recurrent form) and Method
(parallel GLA form, cumulative gate products c_t); papernotes.org note on the same
paper, 关键设计 (GLA recurrence; Anchor Window Attention formula).
"""
import numpy as np
import pytest

import oracle
import synth


def _small(B=1, H=2, L=23, dk=5, dv=6, M=3, dtype="f32", gate="plain", seed=7, with_dy=False):
    return synth.make_fwd_inputs(B, H, L, dk, dv, M, dtype, gate, seed, with_dy=with_dy)


def _gla_only(x, **kw):
    out = oracle.fwd(x["phi_q"], x["phi_k"], x["v"], x["log_gamma"], x["q"], x["k"],
                     x["meta_k"], x["meta_v"], W=kw.pop("W", 4), want_branches=True, **kw)
    return out


# --------------------------------------------------------------------------------------
# GLA branch
# --------------------------------------------------------------------------------------
def test_gla_matches_bruteforce_quadratic_form():
    """y_i = sum_{j<=i} phi_q_i^T (prod_{l=j+1..i} gamma_l (.) phi_k_j) v_j^T."""
    x = _small(L=31, dk=4, dv=3, seed=11)
    out = _gla_only(x)
    pq, pk, v = (x[n].astype(np.float64) for n in ("phi_q", "phi_k", "v"))
    gam = np.exp(x["log_gamma"].astype(np.float64))
    B, H, L, dk = pq.shape
    ref = np.zeros((B, H, L, v.shape[-1]))
    for b in range(B):
        for h in range(H):
            for i in range(L):
                for j in range(i + 1):
                    decay = np.ones(dk)
                    for l in range(j + 1, i + 1):
                        decay = decay * gam[b, h, l]
                    ref[b, h, i] += np.dot(pq[b, h, i], decay * pk[b, h, j]) * v[b, h, j]
    np.testing.assert_allclose(out["y_gla"], ref, rtol=1e-12, atol=1e-13)


def test_gla_matches_parallel_form_with_cumulative_gate_matrix():
    """Y = ((Q (.) C)(K / C)^T (.) causal) V with rows c_t = prod_{j<=t} gamma_j."""
    x = _small(L=40, dk=6, dv=5, seed=12)
    out = _gla_only(x)
    pq, pk, v = (x[n].astype(np.float64) for n in ("phi_q", "phi_k", "v"))
    C = np.cumprod(np.exp(x["log_gamma"].astype(np.float64)), axis=2)
    A = np.einsum("bhid,bhjd->bhij", pq * C, pk / C)
    A = A * np.tril(np.ones(A.shape[-2:]))
    ref = np.einsum("bhij,bhjc->bhic", A, v)
    np.testing.assert_allclose(out["y_gla"], ref, rtol=1e-11, atol=1e-12)


def test_gla_gamma_one_is_causal_linear_attention():
    """log gamma = 0: y_i = phi_q_i^T sum_{j<=i} phi_k_j v_j^T (prefix sums)."""
    x = _small(L=50, dk=7, dv=4, seed=13)
    x["log_gamma"] = np.zeros_like(x["log_gamma"])
    out = _gla_only(x)
    pq, pk, v = (x[n].astype(np.float64) for n in ("phi_q", "phi_k", "v"))
    S = np.cumsum(np.einsum("bhid,bhic->bhidc", pk, v), axis=2)
    ref = np.einsum("bhid,bhidc->bhic", pq, S)
    np.testing.assert_allclose(out["y_gla"], ref, rtol=1e-12, atol=1e-13)


def test_gla_sequence_split_carries_state():
    """fwd(L1) then fwd(L2, h0 = h_final) gives the same GLA output and final state."""
    x = _small(L=37, dk=5, dv=4, seed=14)
    full = oracle.fwd(x["phi_q"], x["phi_k"], x["v"], x["log_gamma"], x["q"], x["k"],
                      x["meta_k"], x["meta_v"], W=3, want_branches=True, want_state=True)
    L1 = 16
    part = lambda a, s: a[:, :, s]
    a = oracle.fwd(*(part(x[n], slice(0, L1)) for n in ("phi_q", "phi_k", "v", "log_gamma", "q", "k")),
                   x["meta_k"], x["meta_v"], W=3, want_branches=True, want_state=True)
    b = oracle.fwd(*(part(x[n], slice(L1, None)) for n in ("phi_q", "phi_k", "v", "log_gamma", "q", "k")),
                   x["meta_k"], x["meta_v"], W=3, h0=a["h_final"], want_branches=True,
                   want_state=True)
    np.testing.assert_allclose(np.concatenate([a["y_gla"], b["y_gla"]], axis=2), full["y_gla"],
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["h_final"], full["h_final"], rtol=1e-12, atol=1e-13)


def test_gla_nonzero_h0_adds_decayed_initial_state():
    """With h0, y_i gains phi_q_i^T diag(prod_{l<=i} gamma_l) h0 (linearity in h0)."""
    x = _small(L=20, dk=4, dv=3, seed=15)
    rng = np.random.default_rng(3)
    h0 = rng.standard_normal((1, 2, 4, 3))
    base = _gla_only(x)
    with_h0 = _gla_only(dict(x), h0=h0)
    C = np.cumprod(np.exp(x["log_gamma"].astype(np.float64)), axis=2)
    extra = np.einsum("bhid,bhdc->bhic", x["phi_q"].astype(np.float64) * C, h0)
    np.testing.assert_allclose(with_h0["y_gla"] - base["y_gla"], extra, rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------------------
# Window branch
# --------------------------------------------------------------------------------------
def test_window_covering_everything_is_causal_softmax_attention():
    """W >= L and M = 0 reduces to causal softmax attention (PyTorch SDPA, fp64)."""
    torch = pytest.importorskip("torch")
    x = _small(L=29, dk=8, dv=5, M=0, seed=21)
    out = _gla_only(x, W=64)
    q = torch.from_numpy(x["q"].astype(np.float64))
    k = torch.from_numpy(x["k"].astype(np.float64))
    v = torch.from_numpy(x["v"].astype(np.float64))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=1.0 / np.sqrt(8))
    np.testing.assert_allclose(out["y_win"], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_window_of_one_without_meta_returns_own_value():
    x = _small(L=17, M=0, seed=22)
    out = _gla_only(x, W=1)
    np.testing.assert_array_equal(out["y_win"], x["v"].astype(np.float64))


def test_window_zero_query_is_uniform_average():
    """q = 0: every logit is 0, so y_win_i is the mean over meta values and window values."""
    x = _small(L=19, M=3, seed=23)
    x["q"] = np.zeros_like(x["q"])
    W = 5
    out = _gla_only(x, W=W)
    v = x["v"].astype(np.float64)
    mv = x["meta_v"].astype(np.float64)
    for i in range(19):
        j0 = max(0, i - W + 1)
        for h in range(2):
            vals = np.concatenate([mv[h], v[0, h, j0:i + 1]], axis=0)
            np.testing.assert_allclose(out["y_win"][0, h, i], vals.mean(axis=0), rtol=1e-13,
                                       atol=1e-14)


@pytest.mark.parametrize("W,M", [(1, 0), (3, 0), (4, 2), (7, 1), (40, 3)])
def test_window_index_range_is_exact(W, M):
    """q = k = 0, meta_v = 0, v_j = e_j: y_win_i * (M + |S_i|) is the indicator of S_i,
    with S_i = {j : max(0, i-W+1) <= j <= i}."""
    L = 24
    x = _small(L=L, dk=4, dv=L, M=M, seed=24)
    x["q"] = np.zeros_like(x["q"])
    x["k"] = np.zeros_like(x["k"])
    x["meta_v"] = np.zeros_like(x["meta_v"])
    x["v"] = np.broadcast_to(np.eye(L, dtype=np.float32), x["v"].shape).copy()
    out = _gla_only(x, W=W)
    for i in range(L):
        lo = max(0, i - W + 1)
        ind = np.zeros(L)
        ind[lo:i + 1] = 1.0
        got = out["y_win"][0, :, i] * (M + (i + 1 - lo))
        np.testing.assert_array_equal(np.rint(got), np.broadcast_to(ind, got.shape))
        np.testing.assert_allclose(got, np.broadcast_to(ind, got.shape), atol=1e-12)


def test_meta_tokens_are_shared_across_batch_and_always_visible():
    """Meta keys/values enter every query's softmax, for every batch entry: a query whose
    window is the single token 0 still attends the meta tokens."""
    x = _small(B=2, L=5, M=2, seed=25)
    out = _gla_only(x, W=1)
    scale = 1.0 / np.sqrt(5)
    for b in range(2):
        for h in range(2):
            qi = x["q"][b, h, 0].astype(np.float64)
            keys = np.concatenate([x["meta_k"][h], x["k"][b, h, :1]]).astype(np.float64)
            vals = np.concatenate([x["meta_v"][h], x["v"][b, h, :1]]).astype(np.float64)
            z = scale * keys @ qi
            p = np.exp(z - z.max())
            p /= p.sum()
            np.testing.assert_allclose(out["y_win"][b, h, 0], p @ vals, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------------------
# Merge
# --------------------------------------------------------------------------------------
def test_merge_weights():
    x = _small(L=21, seed=31)
    args = [x[n] for n in ("phi_q", "phi_k", "v", "log_gamma", "q", "k", "meta_k", "meta_v")]
    ref = oracle.fwd(*args, W=4, want_branches=True)
    a0 = oracle.fwd(*args, W=4, alpha=0.0)
    np.testing.assert_array_equal(a0["y"], ref["y_gla"])
    a2 = oracle.fwd(*args, W=4, alpha=2.5)
    np.testing.assert_allclose(a2["y"], ref["y_gla"] + 2.5 * ref["y_win"], rtol=1e-14, atol=1e-15)
    args[0] = np.zeros_like(x["phi_q"])
    z = oracle.fwd(*args, W=4, alpha=0.75)
    np.testing.assert_allclose(z["y"], 0.75 * ref["y_win"], rtol=1e-14, atol=1e-15)


# --------------------------------------------------------------------------------------
# Backward: central finite differences, and the log-gate identity
# --------------------------------------------------------------------------------------
_FD_NAMES = ("phi_q", "phi_k", "v", "log_gamma", "q", "k", "meta_k", "meta_v")
_GRAD_OF = dict(phi_q="d_phi_q", phi_k="d_phi_k", v="d_v", log_gamma="d_log_gamma", q="d_q",
                k="d_k", meta_k="d_meta_k", meta_v="d_meta_v")


@pytest.mark.parametrize("W,M,alpha,with_h0", [(3, 2, 1.0, False), (2, 0, 0.7, True),
                                               (9, 1, 1.3, False)])
def test_backward_matches_central_finite_differences(W, M, alpha, with_h0):
    rng = np.random.default_rng(40 + W)
    B, H, L, dk, dv = 2, 2, 7, 3, 4
    x = {n: a.astype(np.float64) for n, a in
         _small(B=B, H=H, L=L, dk=dk, dv=dv, M=M, seed=41 + W, with_dy=True).items()}
    # Larger-than-default decays so that the gate terms are well exercised.
    x["log_gamma"] = -np.abs(rng.standard_normal(x["log_gamma"].shape))
    h0 = rng.standard_normal((B, H, dk, dv)) if with_h0 else None
    dy = x.pop("dy")

    def loss(xx):
        y = oracle.fwd(*(xx[n] for n in _FD_NAMES), W=W, alpha=alpha, h0=h0)["y"]
        return float(np.sum(y * dy))

    g = oracle.bwd(*(x[n] for n in _FD_NAMES), dy, W=W, alpha=alpha, h0=h0)
    eps = 1e-6
    for name in _FD_NAMES:
        if M == 0 and name.startswith("meta"):
            continue
        fd = np.zeros_like(x[name])
        it = np.nditer(x[name], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = {n: a.copy() for n, a in x.items()}
            xm = {n: a.copy() for n, a in x.items()}
            xp[name][idx] += eps
            xm[name][idx] -= eps
            fd[idx] = (loss(xp) - loss(xm)) / (2 * eps)
        ana = g[_GRAD_OF[name]]
        scale = max(1.0, np.abs(ana).max())
        np.testing.assert_allclose(ana, fd, rtol=0, atol=1e-6 * scale, err_msg=name)


def test_backward_h0_gradient_matches_finite_differences():
    rng = np.random.default_rng(50)
    x = {n: a.astype(np.float64) for n, a in
         _small(B=1, H=1, L=6, dk=3, dv=2, M=1, seed=51, with_dy=True).items()}
    dy = x.pop("dy")
    h0 = rng.standard_normal((1, 1, 3, 2))
    g = oracle.bwd(*(x[n] for n in _FD_NAMES), dy, W=3, h0=h0, want_dh0=True)
    eps = 1e-6
    fd = np.zeros_like(h0)
    for idx in np.ndindex(h0.shape):
        hp, hm = h0.copy(), h0.copy()
        hp[idx] += eps
        hm[idx] -= eps
        lp = np.sum(oracle.fwd(*(x[n] for n in _FD_NAMES), W=3, h0=hp)["y"] * dy)
        lm = np.sum(oracle.fwd(*(x[n] for n in _FD_NAMES), W=3, h0=hm)["y"] * dy)
        fd[idx] = (lp - lm) / (2 * eps)
    np.testing.assert_allclose(g["d_h0"], fd, rtol=0, atol=1e-7)


def test_log_gate_gradient_is_reverse_cumsum_identity():
    """Parallel-form identity: d log_gamma_t = sum_{t' >= t} (phi_q (.) dphi_q - phi_k (.) dphi_k)_{t'}
    (h0 = 0).  The oracle computes d log_gamma from the recurrence, so agreement ties
    the two derivations together."""
    x = _small(B=2, H=2, L=33, dk=5, dv=4, M=2, seed=52, with_dy=True)
    g = oracle.bwd(*(x[n] for n in _FD_NAMES), x["dy"], W=5)
    t = x["phi_q"] * g["d_phi_q"] - x["phi_k"] * g["d_phi_k"]
    ref = np.flip(np.cumsum(np.flip(t, axis=2), axis=2), axis=2)
    np.testing.assert_allclose(g["d_log_gamma"], ref, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------------------
# Decode
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("W,M,alpha", [(4, 2, 1.0), (1, 0, 1.0), (64, 3, 0.6), (5, 1, 2.0)])
def test_decode_from_empty_reproduces_forward(W, M, alpha):
    """Decoding token by token from pos = 0, h = 0 gives the forward pass's outputs and
    final state (recurrent form == parallel form), including ring wrap-around."""
    B, H, L, dk, dv = 2, 3, 19, 4, 5
    x = _small(B=B, H=H, L=L, dk=dk, dv=dv, M=M, seed=60 + W)
    ref = oracle.fwd(*(x[n] for n in _FD_NAMES), W=W, alpha=alpha, want_state=True)
    st = dict(h=np.zeros((B, H, dk, dv)), k_ring=np.zeros((B, H, W, dk)),
              v_ring=np.zeros((B, H, W, dv)), pos=np.zeros(B, dtype=np.int64))
    ys = []
    for t in range(L):
        tok = [x[n][:, :, t] for n in ("phi_q", "phi_k", "v", "log_gamma", "q", "k")]
        ys.append(oracle.decode_step(st, *tok, x["meta_k"], x["meta_v"], W=W, alpha=alpha))
    np.testing.assert_allclose(np.stack(ys, axis=2), ref["y"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(st["h"], ref["h_final"], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(st["pos"], np.full(B, L))


def test_decode_full_ring_slot_order_does_not_matter():
    """A full ring is a set: rotating its slots (and the position) leaves y unchanged."""
    s = synth.DecodeStream(2, 2, 4, 3, 2, 5, dtype="f32", seed=70)
    tok = s.next_token()

    def run(shift):
        st = dict(h=s.h0.astype(np.float64).copy(),
                  k_ring=np.roll(s.k_ring.astype(np.float64), shift, axis=2).copy(),
                  v_ring=np.roll(s.v_ring.astype(np.float64), shift, axis=2).copy(),
                  pos=(s.pos0 + shift).astype(np.int64))
        return oracle.decode_step(st, *(tok[n] for n in ("phi_q", "phi_k", "v", "log_gamma", "q", "k")),
                                  s.meta_k, s.meta_v, W=5)

    # Slot (pos mod W) is overwritten by the new token; after rolling the ring by s and
    # moving pos by s, the overwritten slot holds the same old token, so the key set is
    # the same and only the summation order changes.
    y0 = run(0)
    for shift in (1, 2, 4):
        np.testing.assert_allclose(run(shift), y0, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------------------
# Chunk-local cumulative sum (the reference point of the reparameterisation)
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("L,chunk", [(256, 64), (200, 64), (1, 64), (130, 128), (7, 3)])
def test_chunk_cumsum_ranges_exact(L, chunk):
    """log gamma = 1: b_t = (t mod chunk) + 1 and Gamma_c = length of chunk c, exactly."""
    lg = np.ones((2, L, 3))
    b, G = oracle.chunk_cumsum(lg, chunk)
    t = np.arange(L)
    np.testing.assert_array_equal(b, np.broadcast_to(((t % chunk) + 1)[None, :, None], b.shape))
    nch = (L + chunk - 1) // chunk
    lens = np.array([min(chunk, L - c * chunk) for c in range(nch)], dtype=np.float64)
    np.testing.assert_array_equal(G, np.broadcast_to(lens[None, :, None], G.shape))


def test_chunk_cumsum_values():
    rng = np.random.default_rng(80)
    lg = rng.standard_normal((3, 150, 4))
    b, G = oracle.chunk_cumsum(lg, 64)
    for c0 in range(0, 150, 64):
        seg = lg[:, c0:c0 + 64]
        np.testing.assert_allclose(b[:, c0:c0 + 64], np.cumsum(seg, axis=1), rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(G[:, c0 // 64], seg.sum(axis=1), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------------------
# Input generator sanity (no operator arithmetic; checks the recipe)
# --------------------------------------------------------------------------------------
def test_bf16_rounding_is_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(90)
    x = (rng.standard_normal(10000) * 10.0 ** rng.integers(-6, 6, 10000)).astype(np.float32)
    ours = synth.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_generator_is_seeded_and_in_range():
    a = synth.make_fwd_inputs(1, 2, 33, 8, 8, 2, "bf16", "bimodal", seed=5, with_dy=True)
    b = synth.make_fwd_inputs(1, 2, 33, 8, 8, 2, "bf16", "bimodal", seed=5, with_dy=True)
    for n in a:
        np.testing.assert_array_equal(a[n], b[n])
    assert np.all(a["phi_q"] > 0) and np.all(a["phi_k"] > 0)
    assert np.all(a["log_gamma"] < 0)
    assert a["log_gamma"][..., :4].mean() < a["log_gamma"][..., 4:].mean()


# --------------------------------------------------------------------------------------
# Segment-state combine (sequence split)
# --------------------------------------------------------------------------------------
def test_state_combine_of_segments_gives_the_full_state_and_is_associative():
    """Final states of consecutive segments computed from zero, combined left to right,
    equal the final state of the whole sequence; the combine is associative; a segment
    started from the combined state of its predecessors reproduces the whole sequence's
    GLA outputs for its tokens."""
    B, H, L, dk, dv = 2, 2, 30, 4, 5
    x = _small(B=B, H=H, L=L, dk=dk, dv=dv, M=2, seed=80, gate="bimodal")
    full = oracle.fwd(*(x[n] for n in _FD_NAMES), W=3, alpha=0.0, want_state=True)
    cuts = [0, 7, 19, 30]
    segs = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = {n: (x[n][:, :, a:b] if x[n].ndim == 4 else x[n]) for n in _FD_NAMES}
        out = oracle.fwd(*(part[n] for n in _FD_NAMES), W=3, alpha=0.0, want_state=True)
        segs.append((x["log_gamma"][:, :, a:b].astype(np.float64).sum(axis=2), out["h_final"]))
    g01, h01 = oracle.state_combine(*segs[0], *segs[1])
    g, h = oracle.state_combine(g01, h01, *segs[2])
    np.testing.assert_allclose(h, full["h_final"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g, x["log_gamma"].astype(np.float64).sum(axis=2), rtol=1e-12, atol=1e-13)
    g12, h12 = oracle.state_combine(*segs[1], *segs[2])
    g_, h_ = oracle.state_combine(*segs[0], g12, h12)
    np.testing.assert_allclose(h_, h, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g_, g, rtol=1e-12, atol=1e-13)
    part = {n: (x[n][:, :, 19:30] if x[n].ndim == 4 else x[n]) for n in _FD_NAMES}
    y = oracle.fwd(*(part[n] for n in _FD_NAMES), W=3, alpha=0.0, h0=h01)["y"]
    np.testing.assert_allclose(y, full["y"][:, :, 19:30], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------------------
# Hedgehog feature map ("Lizard", arXiv 2507.09025, Method: phi(x) = [exp(xW) (+) exp(-xW)])
# --------------------------------------------------------------------------------------
def _fmap_small(B=2, H=2, L=5, D=6, F=4, seed=90):
    x = synth.make_fmap_inputs(B, H, L, D, F, "f32", seed, with_dphi=True)
    return {n: a.astype(np.float64) for n, a in x.items()}


def test_feature_map_kernel_is_a_sum_of_cosh():
    """phi(x) . phi(y) = sum_j [e^{a_j} e^{b_j} + e^{-a_j} e^{-b_j}] = 2 sum_j cosh(a_j + b_j)
    with a = x W, b = y W; the right side is evaluated from (x + y) W with plain loops."""
    x = _fmap_small()
    X, Wt = x["x"], x["w"]
    phi = oracle.feature_map(X, Wt)
    B, H, L, D = X.shape
    F = Wt.shape[-1]
    for b in range(B):
        for h in range(H):
            for i in range(L):
                for j in range(L):
                    s = 0.0
                    for f in range(F):
                        u = sum((X[b, h, i, d] + X[b, h, j, d]) * Wt[h, d, f] for d in range(D))
                        s += 2.0 * np.cosh(u)
                    assert abs(float(phi[b, h, i] @ phi[b, h, j]) - s) <= 1e-12 * abs(s)


def test_feature_map_special_values_and_symmetry():
    """phi(0) is all ones; phi is positive; phi(-x) swaps the two halves; the first half
    of phi(x) for a one-hot x = e_d is exp of row d of W."""
    x = _fmap_small(seed=91)
    X, Wt = x["x"], x["w"]
    F = Wt.shape[-1]
    np.testing.assert_array_equal(oracle.feature_map(np.zeros_like(X), Wt), 1.0)
    phi = oracle.feature_map(X, Wt)
    assert (phi > 0).all()
    neg = oracle.feature_map(-X, Wt)
    np.testing.assert_allclose(neg[..., :F], phi[..., F:], rtol=1e-14)
    np.testing.assert_allclose(neg[..., F:], phi[..., :F], rtol=1e-14)
    D = X.shape[-1]
    one = np.zeros((1, Wt.shape[0], D, D))
    for d in range(D):
        one[0, :, d, d] = 1.0
    p1 = oracle.feature_map(one, Wt)
    for h in range(Wt.shape[0]):
        for d in range(D):
            for f in range(F):
                assert p1[0, h, d, f] == pytest.approx(np.exp(Wt[h, d, f]), rel=1e-15)


def test_feature_map_gradients_match_finite_differences():
    """loss = sum(phi(x; W) * G): central differences in every entry of x and W against
    feature_map_bwd(x, W, G)."""
    x = _fmap_small(B=1, H=2, L=3, D=4, F=3, seed=92)
    X, Wt, G = x["x"], x["w"], x["d_phi"]
    dx, dw = oracle.feature_map_bwd(X, Wt, G)

    def loss(Xa, Wa):
        return float((oracle.feature_map(Xa, Wa) * G).sum())

    eps = 1e-6
    for arr, grad, is_x in ((X, dx, True), (Wt, dw, False)):
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            lp = loss(p, Wt) if is_x else loss(X, p)
            lm = loss(m, Wt) if is_x else loss(X, m)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (is_x, idx, fd, grad[idx])


def _gate_small(B=1, H=2, L=4, D=5, dk=3, seed=95):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, H, L, D)), rng.standard_normal((H, D, dk)) / np.sqrt(D),
            rng.standard_normal((B, H, L, dk)))


def test_gate_special_values():
    """W = 0 gives logsigmoid(0)/tau = -ln 2 / tau everywhere; a one-hot input row e_d
    gives logsigmoid of row d of W; tau only divides; log gamma is negative, tends to 0
    for large positive z and to z / tau for large negative z."""
    X, Wt, _ = _gate_small()
    np.testing.assert_allclose(oracle.gate(X, np.zeros_like(Wt), 16.0), -np.log(2.0) / 16.0,
                               rtol=1e-15)
    D = X.shape[-1]
    one = np.zeros((1, Wt.shape[0], D, D))
    for d in range(D):
        one[0, :, d, d] = 1.0
    g1 = oracle.gate(one, Wt, 1.0)
    for h in range(Wt.shape[0]):
        for d in range(D):
            for k in range(Wt.shape[-1]):
                z = Wt[h, d, k]
                assert g1[0, h, d, k] == pytest.approx(-np.log(1.0 + np.exp(-z)), rel=1e-14)
    np.testing.assert_allclose(oracle.gate(X, Wt, 4.0) * 4.0, oracle.gate(X, Wt, 1.0), rtol=1e-14)
    assert (oracle.gate(X, Wt) < 0).all()
    big = np.full((1, 1, 1, 1), 50.0)
    assert abs(oracle.gate(big, np.ones((1, 1, 1)), 1.0)[0, 0, 0, 0]) < 1e-20
    assert oracle.gate(-big, np.ones((1, 1, 1)), 2.0)[0, 0, 0, 0] == pytest.approx(-25.0, rel=1e-15)


def test_gate_gradients_match_finite_differences():
    """loss = sum(gate(x; W) * G): central differences in every entry of x and W against
    gate_bwd(x, W, G)."""
    X, Wt, G = _gate_small(seed=96)
    dx, dw = oracle.gate_bwd(X, Wt, G, 3.0)

    def loss(Xa, Wa):
        return float((oracle.gate(Xa, Wa, 3.0) * G).sum())

    eps = 1e-6
    for arr, grad, is_x in ((X, dx, True), (Wt, dw, False)):
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            lp = loss(p, Wt) if is_x else loss(X, p)
            lm = loss(m, Wt) if is_x else loss(X, m)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (is_x, idx, fd, grad[idx])
