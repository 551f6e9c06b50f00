"""Multi-process paths on CPU ranks (gloo, world size 2).

The operator shards without a data-path collective; the two places ranks exchange data are
(1) the timing harness (barrier, max over ranks) and (2) a sequence split, whose only
exchange is the associative combine of segment states followed by an exclusive scan over
ranks ("Lizard", arXiv 2507.09025, Preliminaries: recurrent form).  Both run here as two
spawned processes on 127.0.0.1 with the oracle standing in for the device."""
import os
import socket

import numpy as np
import pytest

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    return dist


def _bench_worker(rank, port, q):
    try:
        dist = _init(rank, port)
        import torch

        import bench
        bench._barrier(WORLD)
        m = bench._max_over_ranks(1.5 + rank, WORLD, torch.device("cpu"))
        bench._barrier(WORLD)
        dist.destroy_process_group()
        q.put((rank, m))
    except Exception as e:  # reported to the parent, never hidden
        q.put((rank, repr(e)))


def _split_worker(rank, port, q):
    """Rank r owns tokens [r*L/2, (r+1)*L/2) as two segments; it combines them locally,
    all-gathers the per-rank (Gamma, h), scans the ranks before it into its initial state
    and recomputes its outputs from that state."""
    try:
        dist = _init(rank, port)
        import torch

        import oracle
        import synth
        names = ("phi_q", "phi_k", "v", "log_gamma", "q", "k", "meta_k", "meta_v")
        B, H, L, dk, dv, M = 1, 2, 40, 4, 5, 2
        x = synth.make_fwd_inputs(B, H, L, dk, dv, M, "f32", "bimodal", seed=91)
        half = L // WORLD
        lo, hi = rank * half, (rank + 1) * half

        def seg(a, b, h0=None):
            part = {n: (x[n][:, :, a:b] if x[n].ndim == 4 else x[n]) for n in names}
            out = oracle.fwd(*(part[n] for n in names), W=3, alpha=0.0, h0=h0, want_state=True)
            return x["log_gamma"][:, :, a:b].astype(np.float64).sum(axis=2), out

        mid = lo + 7  # two segments per rank
        ga, oa = seg(lo, mid)
        gb, ob = seg(mid, hi)
        g_r, h_r = oracle.state_combine(ga, oa["h_final"], gb, ob["h_final"])
        gath_g = [torch.zeros(g_r.shape, dtype=torch.float64) for _ in range(WORLD)]
        gath_h = [torch.zeros(h_r.shape, dtype=torch.float64) for _ in range(WORLD)]
        dist.all_gather(gath_g, torch.from_numpy(g_r))
        dist.all_gather(gath_h, torch.from_numpy(h_r))
        # exclusive scan: the state at the start of this rank's range
        g0, h0 = np.zeros((B, H, dk)), np.zeros((B, H, dk, dv))
        for r in range(rank):
            g0, h0 = oracle.state_combine(g0, h0, gath_g[r].numpy(), gath_h[r].numpy())
        _, mine = seg(lo, hi, h0=h0)
        full = oracle.fwd(*(x[n] for n in names), W=3, alpha=0.0, want_state=True)
        err_y = float(np.max(np.abs(mine["y"] - full["y"][:, :, lo:hi])))
        g_all, h_all = np.zeros((B, H, dk)), np.zeros((B, H, dk, dv))
        for r in range(WORLD):
            g_all, h_all = oracle.state_combine(g_all, h_all, gath_g[r].numpy(), gath_h[r].numpy())
        err_h = float(np.max(np.abs(h_all - full["h_final"])))
        dist.destroy_process_group()
        q.put((rank, (err_y, err_h)))
    except Exception as e:
        q.put((rank, repr(e)))


def _run(target):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def test_bench_rank_helpers_take_the_max_over_gloo_ranks():
    pytest.importorskip("torch")
    res = _run(_bench_worker)
    assert res == {0: 2.5, 1: 2.5}, res


def test_sequence_split_combine_over_gloo_ranks():
    pytest.importorskip("torch")
    res = _run(_split_worker)
    for rank, val in res.items():
        assert isinstance(val, tuple), (rank, val)
        err_y, err_h = val
        assert err_y < 1e-12 and err_h < 1e-12, (rank, val)
