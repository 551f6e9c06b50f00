"""The allocation-free decode step, for callers that cannot allocate device memory (a
host program or binding with no device allocator of its own, or a runtime whose pool owns
all device memory and may not call cudaMalloc while serving).

lizard_decode_step_noalloc keeps its per-sequence counters in the library's own fixed
device array instead of a caller workspace.  This test drives it through the C ABI for
two decode steps in a row and checks every output against lizard_decode_step (the entry
point with a workspace) on an identical copy of the state.  Both run the same kernels on
the same inputs, so every output must agree bit for bit; the first step is also checked
against the fp64 oracle within the bf16 tolerance of the other tests.  Two calls in a row
also check that the shared array is left in a usable state by the first call.  The file
is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import hybrid_gated_linear_gb300 as lz
import oracle
import synth
from gpu_util import TOK, TOL, host, rel_l2

pytestmark = pytest.mark.gpu


def _state(s, dev):
    bf = torch.bfloat16
    return dict(h=torch.from_numpy(s.h0).to(dev), kr=torch.from_numpy(s.k_ring).to(dev).to(bf),
                vr=torch.from_numpy(s.v_ring).to(dev).to(bf), pos=torch.from_numpy(s.pos0).to(dev),
                y=torch.empty(s.N, s.H, s.dv, dtype=bf, device=dev))


def test_noalloc_decode_matches_workspace_decode_two_calls():
    lz.build()
    dev = torch.device("cuda")
    N, H, d, M, W = 6, 4, 128, 4, 16
    s = synth.DecodeStream(N, H, d, d, M, W, "bf16", seed=77, prefill=True)
    dims = lz.lizard_decode_dims(N, H, d, d, M, lz.LIZARD_BF16, 0.0)
    mk = torch.from_numpy(s.meta_k).to(dev).to(torch.bfloat16)
    mv = torch.from_numpy(s.meta_v).to(dev).to(torch.bfloat16)
    a, b = _state(s, dev), _state(s, dev)
    ws = torch.zeros(lz.lizard_decode_workspace_bytes(dims), dtype=torch.uint8, device=dev)
    st = dict(h=s.h0.astype(np.float64), k_ring=s.k_ring.astype(np.float64),
              v_ring=s.v_ring.astype(np.float64), pos=s.pos0.copy())
    for step in range(2):
        tok = s.next_token()
        t = {n: torch.from_numpy(tok[n]).to(dev) for n in TOK}
        for n in TOK:
            if n != "log_gamma":
                t[n] = t[n].to(torch.bfloat16)
        args = [t[n] for n in TOK] + [mk, mv, W, 1.0]
        lz.lizard_decode_step(dims, *args, a["h"], a["kr"], a["vr"], a["pos"], a["y"], ws)
        lz.lizard_decode_step_noalloc(dims, *args, b["h"], b["kr"], b["vr"], b["pos"], b["y"])
        assert lz.lizard_last_launch_count() >= 1
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(b["y"]), host(a["y"]))
        np.testing.assert_array_equal(b["h"].cpu().numpy(), a["h"].cpu().numpy())
        if step == 0:
            yr = oracle.decode_step(st, *(tok[n] for n in TOK), s.meta_k, s.meta_v, W=W)
            assert rel_l2(host(b["y"]), yr) <= TOL["bf16"]
            assert rel_l2(b["h"].cpu().numpy(), st["h"]) <= TOL["bf16"]
        np.testing.assert_array_equal(host(b["kr"]), host(a["kr"]))
        np.testing.assert_array_equal(host(b["vr"]), host(a["vr"]))
        np.testing.assert_array_equal(b["pos"].cpu().numpy(), a["pos"].cpu().numpy())
    np.testing.assert_array_equal(b["pos"].cpu().numpy(), s.pos0 + 2)


def test_noalloc_decode_rejects_too_many_sequences():
    lz.build()
    N = lz.LIZARD_NOALLOC_MAX_SEQUENCES + 1
    dims = lz.lizard_decode_dims(N, 1, 64, 64, 0, lz.LIZARD_BF16, 0.0)
    bufs = [torch.empty(64, dtype=torch.uint8, device="cuda") for _ in range(11)]
    with pytest.raises(lz.LizardError) as e:
        lz.lizard_decode_step_noalloc(dims, *bufs[:6], None, None, 8, 1.0, *bufs[6:])
    assert e.value.status == 2  # LIZARD_ERR_UNSUPPORTED, before anything is enqueued
