"""Chunk-local log-gate cumulative sum (the reparameterisation's reference point):
chunk ranges bit-exact, values against the oracle."""
import numpy as np
import pytest
import torch

import hybrid_gated_linear_gb300 as lz
import oracle
from gpu_util import rel_l2

pytestmark = pytest.mark.gpu


def _run(lg, chunk):
    units, L, dk = lg.shape
    t = torch.from_numpy(lg).cuda()
    b = torch.empty_like(t)
    nch = (L + chunk - 1) // chunk
    G = torch.empty(units, nch, dk, dtype=torch.float32, device="cuda")
    lz.lizard_chunk_cumsum(units, L, dk, chunk, t, b, G)
    torch.cuda.synchronize()
    return b.cpu().numpy(), G.cpu().numpy()


@pytest.mark.parametrize("L,chunk,dk", [(4096, 64, 128), (1000, 64, 128), (1, 64, 64),
                                        (130, 128, 64), (77, 5, 32)])
def test_chunk_ranges_exact(L, chunk, dk):
    lg = np.ones((3, L, dk), dtype=np.float32)
    b, G = _run(lg, chunk)
    t = np.arange(L)
    np.testing.assert_array_equal(b, np.broadcast_to(((t % chunk) + 1)[None, :, None], b.shape))
    lens = np.array([min(chunk, L - c * chunk) for c in range((L + chunk - 1) // chunk)])
    np.testing.assert_array_equal(G, np.broadcast_to(lens[None, :, None], G.shape))


def test_chunk_cumsum_values():
    rng = np.random.default_rng(5)
    lg = (-np.abs(rng.standard_normal((4, 999, 128))) / 16).astype(np.float32)
    b, G = _run(lg, 64)
    rb, rG = oracle.chunk_cumsum(lg, 64)
    assert rel_l2(b, rb) <= 1e-6
    assert rel_l2(G, rG) <= 1e-6
