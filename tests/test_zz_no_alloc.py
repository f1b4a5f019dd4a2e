"""moe_dispatch_static: the dispatch for callers that cannot allocate device
memory (an engine plugin handed only its input and output buffers, a loop
that may not allocate after start-up).  Its scratch is a fixed device array
inside the library instead of a caller workspace.

Checked through the C ABI against moe_dispatch (the workspace entry point) on
two calls in a row with different batches, so that the second call runs on
the array as the first one left it.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import WEIGHT_RTOL
from token_level_top_gb300 import build, moe


def _skewed_scores(T, E, seed):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((T, E)).astype(np.float32)
    s[:, 0] += 1.2
    for b in range(0, T, 640):          # runs of identical tokens
        s[b:b + 128] = s[b]
    return s


def _compare(got, want):
    for key in ("assign", "slot", "flags", "counts", "offsets", "n_rerouted", "n_dropped"):
        assert torch.equal(got[key], want[key]), key
    n = int(want["offsets"][-1].item())
    assert torch.equal(got["perm"][:n], want["perm"][:n])
    np.testing.assert_allclose(got["cw"].cpu().numpy(), want["cw"].cpu().numpy(),
                               rtol=WEIGHT_RTOL, atol=1e-7)


@pytest.mark.gpu
def test_static_dispatch_matches_workspace_dispatch_two_calls():
    build.build()
    moe.lib()
    cases = [moe.Config(T=3000, d_model=64, E=16, k=2, d_ff=128, cf=1.0),
             moe.Config(T=777, d_model=64, E=64, k=2, d_ff=128, cf=1.0)]
    for i, cfg in enumerate(cases):
        s = torch.from_numpy(_skewed_scores(cfg.T, cfg.E, 11 + i)).cuda()
        got = moe.dispatch_static(cfg, s)
        ws = moe.workspace(cfg)
        want = moe.dispatch(cfg, ws, s)
        torch.cuda.synchronize()
        assert int(got["status"].item()) == 0
        assert moe.device_status(ws) == 0
        assert int(want["n_rerouted"].item()) > 0        # the capacity path was exercised
        _compare(got, want)


def test_static_dispatch_rejects_batches_beyond_the_array():
    build.build()
    L = moe.lib()
    cfg = moe.Config(T=200000, d_model=64, E=64, k=2, d_ff=128, cf=1.0).c()
    P = ctypes.c_void_p
    fake = [P(0x7f0000000000)] * 10
    # rejected before anything is enqueued
    assert L.moe_dispatch_static(ctypes.byref(cfg), *fake, None, None) == 2
