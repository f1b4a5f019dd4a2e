"""moe_dispatch_static: the dispatch for callers that cannot allocate device
memory (an engine plugin handed only its input and output buffers, a loop
that may not allocate after start-up).  Its scratch is a fixed device array
inside the library instead of a caller workspace.

Checked through the C ABI against the oracle's dispatch (bit for bit) and
against moe_dispatch (the workspace entry point) on a run of calls in a row
with different batches, so that each call after the first runs on the array
as the one before left it.  The outputs start out filled with values the call
must overwrite, so a total or a count the kernels skip shows up.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import WEIGHT_RTOL, assert_dispatch_equal, np_
from token_level_top_gb300 import build, moe


def _skewed_scores(T, E, seed, run=128, every=640, lead=1.2):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((T, E)).astype(np.float32)
    s[:, 0] += lead
    for b in range(0, T, every):          # runs of identical tokens
        s[b:b + run] = s[b]
    return s


# (config, scores seed, identical-token run length, spacing of the runs)
CASES = [
    (moe.Config(T=3000, d_model=64, E=16, k=2, d_ff=128, cf=1.0), 11, 128, 640),
    (moe.Config(T=200, d_model=64, E=8, k=2, d_ff=128, cf=1.0), 12, 64, 100),     # one routing chunk
    (moe.Config(T=777, d_model=64, E=64, k=2, d_ff=128, cf=1.0), 13, 128, 640),
    (moe.Config(T=256, d_model=64, E=200, k=2, d_ff=128, cf=1.0), 14, 40, 128),
    (moe.Config(T=1000, d_model=64, E=16, k=4, d_ff=128, cf=1.0), 15, 128, 320),
    (moe.Config(T=0, d_model=64, E=8, k=2, d_ff=128, cf=1.0), 16, 1, 1),
    (moe.Config(T=300, d_model=64, E=4, k=4, d_ff=128, cf=0.5), 17, 64, 150),     # drops
]


def _compare_oracle(got, ora, T, k):
    assert_dispatch_equal(got, ora, T, k)
    assert int(got["n_rerouted"].item()) == ora["n_rerouted"]
    assert int(got["n_dropped"].item()) == ora["n_dropped"]
    np.testing.assert_allclose(np_(got["cw"]).reshape(T, k), ora["cw"], rtol=WEIGHT_RTOL, atol=1e-7)


def _compare_workspace(got, want):
    for key in ("assign", "slot", "flags", "counts", "offsets", "n_rerouted", "n_dropped"):
        assert torch.equal(got[key], want[key]), key
    n = int(want["offsets"][-1].item())
    assert torch.equal(got["perm"][:n], want["perm"][:n])
    assert torch.equal(got["cw"], want["cw"])


@pytest.mark.gpu
def test_static_dispatch_matches_oracle_and_workspace_dispatch_calls_in_a_row():
    build.build()
    moe.lib()
    seen_reroute = seen_drop = False
    for cfg, seed, run, every in CASES:
        s_np = _skewed_scores(cfg.T, cfg.E, seed, run, every)
        s = torch.from_numpy(s_np).cuda()
        got = moe.dispatch_static(cfg, s)
        torch.cuda.synchronize()
        assert int(got["status"].item()) == 0
        ora = oracle.dispatch(s_np, cfg.k, oracle.capacity(cfg.T, cfg.k, cfg.E, cfg.cf))
        _compare_oracle(got, ora, cfg.T, cfg.k)
        seen_reroute |= ora["n_rerouted"] > 0
        seen_drop |= ora["n_dropped"] > 0
        if cfg.T > 0:
            ws = moe.workspace(cfg)
            want = moe.dispatch(cfg, ws, s)
            torch.cuda.synchronize()
            assert moe.device_status(ws) == 0
            _compare_workspace(got, want)
    assert seen_reroute and seen_drop        # the capacity paths were exercised


def test_static_dispatch_rejects_batches_beyond_the_array_and_bad_shapes():
    build.build()
    L = moe.lib()
    P = ctypes.c_void_p
    fake = [P(0x7f0000000000)] * 10
    # rejected before anything is enqueued (no pointer is touched)
    for cfg, want in ((moe.Config(T=200000, d_model=64, E=64, k=2, d_ff=128, cf=1.0), 2),
                      (moe.Config(T=100, d_model=64, E=256, k=2, d_ff=128, cf=1.0), 2),
                      (moe.Config(T=100, d_model=64, E=16, k=9, d_ff=128, cf=1.0), 2),
                      (moe.Config(T=100, d_model=64, E=4, k=5, d_ff=128, cf=1.0), 1)):
        c = cfg.c()
        assert L.moe_dispatch_static(ctypes.byref(c), *fake, None, None) == want, cfg
