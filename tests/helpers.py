"""Shared helpers for the GPU parity tests (inputs, oracle calls, metrics)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from token_level_top_gb300 import moe, synth

# Tolerances (the pages fix none for the layer; these follow from the
# arithmetic: bf16 inputs, fp32 accumulation, one bf16 rounding of the
# SwiGLU activation and of the output).
LOGIT_MAX_ABS = 1e-3        # router logits vs the oracle's double-accumulated fp32 logits
OUT_REL_FROB = 2e-2         # layer / expert outputs, relative Frobenius error
WEIGHT_RTOL = 1e-5          # softmax probabilities, combine weights, P (fp32 vs double)
MARGIN = 1e-4               # tokens with a smaller top-k score margin are not compared


def rel_frob(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / max(den, 1e-30))


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def make_layer(shape, device="cuda"):
    """Seeded inputs of a workload on the device plus the packed W13."""
    h, wr, bias, usage = synth.router_inputs(shape)
    w1, w3, w2 = synth.expert_weights(shape, device=device)
    d = dict(h=h.to(device), wr=wr.to(device), w1=w1, w3=w3, w2=w2,
             bias=None if bias is None else bias.to(device),
             usage=None if usage is None else usage.to(device))
    d["w13"] = moe.pack_w13(w1, w3)
    return d


def topk_margin(scores: np.ndarray, k: int) -> np.ndarray:
    """min over the first k ranks of (s_(r) - s_(r+1)) of the sorted scores."""
    s = -np.sort(-scores.astype(np.float64), axis=1)
    kk = min(k + 1, s.shape[1])
    gaps = s[:, : kk - 1] - s[:, 1:kk]
    return gaps.min(axis=1) if gaps.shape[1] else np.full(s.shape[0], np.inf)


def sample_tokens(T: int, n: int, seed: int, must=()) -> np.ndarray:
    rng = np.random.default_rng(seed)
    base = {0, 1, T - 2, T - 1} | {int(t) for t in must}
    extra = rng.choice(T, size=min(n, T), replace=False)
    toks = sorted(t for t in (base | set(int(x) for x in extra)) if 0 <= t < T)
    return np.array(toks, np.int32)


def tile_tokens(perm: np.ndarray, offsets: np.ndarray, k: int, seed: int, tile: int = 128) -> np.ndarray:
    """One token per (expert, row tile) of the expert GEMMs: for every 128-slot row tile
    of every expert's slot range, the token of one of its slots (the tile's last slot
    for an expert's tail tile, a seeded random one otherwise), so that a fault confined
    to one row tile or one expert's ragged tail shows in some checked row."""
    rng = np.random.default_rng(seed)
    toks = set()
    for e in range(offsets.shape[0] - 1):
        off, cnt = int(offsets[e]), int(offsets[e + 1] - offsets[e])
        for m0 in range(0, cnt, tile):
            m1 = min(cnt, m0 + tile)
            j = m1 - 1 if m1 == cnt else int(rng.integers(m0, m1))
            toks.add(int(perm[off + j]) // k)
    return np.array(sorted(toks), np.int32)


def assert_rows_close(got: np.ndarray, want: np.ndarray, bound: float = OUT_REL_FROB):
    """The pooled relative Frobenius bound, and a per-row bound of 4x it (rows the
    oracle gives as exact zeros -- every choice dropped -- must be zero)."""
    err = rel_frob(got, want)
    assert err <= bound, f"relative Frobenius error {err:.3e}"
    nw = np.linalg.norm(np.asarray(want, np.float64), axis=1)
    ng = np.linalg.norm(np.asarray(got, np.float64) - np.asarray(want, np.float64), axis=1)
    zero = nw == 0
    assert (ng[zero] == 0).all(), "a row the oracle gives as zero is not zero"
    rows = ng[~zero] / nw[~zero]
    if rows.size:
        i = int(np.argmax(rows))
        assert rows[i] <= 4 * bound, f"row {np.flatnonzero(~zero)[i]}: relative error {rows[i]:.3e}"


def oracle_dispatch_of(scores: np.ndarray, k: int, C: int):
    return oracle.dispatch(scores, k, C)


def assert_dispatch_equal(gpu: dict, ora: dict, T: int, k: int):
    for key in ("assign", "slot", "flags"):
        g = np_(gpu[key]).reshape(T, k)
        o = ora[key].reshape(T, k)
        bad = np.argwhere(g != o)
        assert bad.size == 0, f"{key} differs at {bad[:5].tolist()}: gpu {g[tuple(bad[0])]} oracle {o[tuple(bad[0])]}"
    assert np.array_equal(np_(gpu["counts"]), ora["counts"])
    if "offsets" in gpu:
        assert np.array_equal(np_(gpu["offsets"]), ora["offsets"])
    if "perm" in gpu:
        n = int(ora["offsets"][-1])
        assert np.array_equal(np_(gpu["perm"])[:n], ora["perm"])
