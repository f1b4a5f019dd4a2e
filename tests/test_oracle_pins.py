"""Pins for the CPU oracle: values the pages print, closed forms, invariants,
brute force on tiny inputs and special cases that reduce to library routines.

Every check here is independent of the oracle's own code paths, so that a
plausible mistake in it (a dropped term, a wrong sign or index, a transposed
operand, a rank-minor dispatch order) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from token_level_top_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def bf16(a):
    return synth.bf16_bits(torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def widen(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- capacity

def test_capacity_page_value():
    g = golden("capacity_coreui_5_2.json")
    assert oracle.capacity(g["T"], g["k"], g["E"], g["cf"]) == g["C"]


@pytest.mark.parametrize("T,k,E,cf,C", [
    (256, 2, 8, 1.25, 80), (4096, 2, 8, 1.25, 1280), (64, 2, 8, 1.25, 20),
    (16384, 2, 64, 1.0, 512), (8192, 2, 16, 1.0, 1024),
    (10, 2, 8, 1.0, 3),            # 2.5 rounds up
    (100, 2, 26, 1.3, 10),         # exactly 10: a binary 1.3 would give 10.000...02 -> 11
    (1, 1, 64, 1.0, 1),
])
def test_capacity_closed_form(T, k, E, cf, C):
    assert oracle.capacity(T, k, E, cf) == C


def test_capacity_explicit_override():
    assert oracle.capacity(4096, 2, 8, 1.25, 7) == 7


# --------------------------------------------------------------------------- router

def test_preference_matches_sorted_with_ties():
    rng = np.random.default_rng(1)
    for _ in range(200):
        E = int(rng.integers(1, 12))
        s = rng.integers(-3, 3, E).astype(np.float32)   # many ties
        if rng.random() < 0.3:
            s[rng.integers(0, E)] = -0.0
        want = sorted(range(E), key=lambda e: (-float(s[e]), e))
        assert oracle.preference(s).tolist() == want


def test_preference_signed_zero_and_inf():
    s = np.array([0.0, -0.0, np.inf, -np.inf, 0.0], np.float32)
    assert oracle.preference(s).tolist() == [2, 0, 1, 4, 3]


def test_topk_is_best_subset_brute_force():
    """Top-k set = the k-subset whose sorted score list is lexicographically
    best, ties going to the lexicographically smaller index list."""
    rng = np.random.default_rng(2)
    for _ in range(150):
        E = int(rng.integers(2, 7))
        k = int(rng.integers(1, min(3, E) + 1))
        T = 3
        z = rng.integers(-2, 3, (T, E)).astype(np.float32)
        r = oracle.route(k, logits_in=z)
        for t in range(T):
            best = None
            for sub in itertools.combinations(range(E), k):
                key = tuple(sorted(((-float(z[t, e]), e) for e in sub)))
                if best is None or key < best[0]:
                    best = (key, sub)
            want = [e for _, e in best[0]]
            assert r["ids"][t].tolist() == want


def test_equal_logits_pick_lowest_indices():
    z = np.zeros((4, 8), np.float32)
    r = oracle.route(2, logits_in=z)
    assert (r["ids"] == np.array([0, 1])).all()
    np.testing.assert_allclose(r["topk_p"], 1.0 / 8, rtol=1e-7)


def test_logits_match_float64_matmul():
    rng = np.random.default_rng(3)
    h = bf16(rng.standard_normal((37, 96)))
    wr = bf16(rng.standard_normal((5, 96)) * 0.02)
    bias = rng.standard_normal(5).astype(np.float32)
    r = oracle.route(2, h=h, wr=wr, bias=bias)
    want = widen(h).astype(np.float64) @ widen(wr).astype(np.float64).T + bias.astype(np.float64)
    np.testing.assert_allclose(r["logits"], want.astype(np.float32), rtol=2e-7, atol=1e-7)
    # h is [T,d] and W_r is [E,d]: a transposed operand cannot give this shape
    assert r["logits"].shape == (37, 5)


def test_penalty_is_two_rounded_fp32_ops():
    # z - fl(lambda*u) with values where a fused multiply-add rounds differently
    # z equals fl(lambda*u) for expert 0, so the unfused score is exactly 0
    # while a fused multiply-add leaves the product's rounding error behind.
    lam = np.float32(0.7)
    u = np.array([0.6369616985321045, 1.0 / 3.0, 0.1], np.float32)
    z = np.array([[float(np.float32(lam * u[0])), 1.0, 0.5]], np.float32)
    r = oracle.route(1, logits_in=z, usage=u, lam=float(lam))
    pen = (lam * u).astype(np.float32)
    want = (z - pen).astype(np.float32)
    assert np.array_equal(r["scores"], want)
    fused = (z.astype(np.float64) - lam.astype(np.float64) * u.astype(np.float64)).astype(np.float32)
    assert not np.array_equal(fused, want), "case must separate fused from unfused"


def test_penalty_special_cases():
    rng = np.random.default_rng(4)
    z = rng.standard_normal((50, 6)).astype(np.float32)
    u = rng.random(6).astype(np.float32)
    base = oracle.route(2, logits_in=z)
    zero_lam = oracle.route(2, logits_in=z, usage=u, lam=0.0)
    assert np.array_equal(base["ids"], zero_lam["ids"])
    assert np.array_equal(base["scores"], zero_lam["scores"])
    # a heavily used expert is never picked
    u2 = np.zeros(6, np.float32)
    u2[3] = 1e6
    pen = oracle.route(2, logits_in=z, usage=u2, lam=1.0)
    assert not (pen["ids"] == 3).any()
    # the penalty lowers the score (sign): expert 3 loses exactly lambda*u
    assert np.array_equal(pen["scores"][:, 3], (z[:, 3] - np.float32(1e6)).astype(np.float32))


def test_softmax_and_stats_match_scipy():
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    T, E, k = 300, 7, 2
    z = (rng.standard_normal((T, E)) * 1.3).astype(np.float32)
    u = rng.random(E).astype(np.float32)
    r = oracle.route(k, logits_in=z, usage=u, lam=0.8)
    p = softmax(r["scores"].astype(np.float64), axis=1)
    np.testing.assert_allclose(r["topk_p"], np.take_along_axis(p, r["ids"].astype(np.int64), 1),
                               rtol=1e-6)
    np.testing.assert_allclose(r["P"], p.mean(0), rtol=1e-6)
    assert abs(float(r["P"].astype(np.float64).sum()) - 1.0) < 1e-6
    assert r["counts_pre"].sum() == T * k
    assert abs(float(r["f"].astype(np.float64).sum()) - k) < 1e-5
    want_counts = np.bincount(r["ids"].ravel(), minlength=E)
    assert np.array_equal(r["counts_pre"], want_counts)
    np.testing.assert_allclose(r["f"], want_counts / T, rtol=1e-7)


def test_softmax_limits():
    z = np.array([[np.inf, 1.0, np.inf, 0.0], [-np.inf] * 4], np.float32)
    r = oracle.route(2, logits_in=z)
    assert r["ids"][0].tolist() == [0, 2]
    np.testing.assert_allclose(r["topk_p"][0], [0.5, 0.5])
    np.testing.assert_allclose(r["topk_p"][1], [0.25, 0.25])


def test_nan_score_is_an_error():
    z = np.zeros((3, 4), np.float32)
    z[1, 2] = np.nan
    with pytest.raises(oracle.OracleError) as ei:
        oracle.route(2, logits_in=z)
    assert ei.value.status == 5
    with pytest.raises(oracle.OracleError):
        oracle.dispatch(z, 2, 4)


# --------------------------------------------------------------------------- dispatch

def test_worked_case_128_identical_tokens():
    """128 identical tokens, E=8, k=2, cf=1.0 -> C=32 (closed form)."""
    C = oracle.capacity(128, 2, 8, 1.0)
    assert C == 32
    s = np.tile(np.arange(8, 0, -1, dtype=np.float32), (128, 1))   # prefers 0 > 1 > ... > 7
    d = oracle.dispatch(s, 2, C)
    for t in range(128):
        g = t // 32
        assert d["assign"][t].tolist() == [g, g + 4]
        assert d["slot"][t].tolist() == [t % 32, t % 32]
    assert d["n_rerouted"] == 224 and d["n_dropped"] == 0
    assert (d["counts"] == 32).all()
    assert d["flags"][:32, 0].tolist() == [0] * 32
    assert (d["flags"][32:, 0] == 1).all() and (d["flags"][:, 1] == 1).all()


def test_page_overflow_case():
    g = golden("overflow_mhpn_2_3.json")
    T, E, C = g["T"], g["E"], g["C"]
    s = np.zeros((T, E), np.float32)
    s[:, g["first"]] = 2.0
    s[:, g["second"]] = 1.0
    d = oracle.dispatch(s, g["k"], C)
    assert (d["assign"][:127, 0] == g["first"]).all()
    assert d["counts"][g["first"]] == g["expect_first_count"]
    assert d["assign"][127, 0] == g["expect_token_127"]
    assert d["n_rerouted"] == g["expect_rerouted"] and d["flags"][127, 0] == 1


def test_drop_case():
    s = np.array([[2.0, 1.0], [2.0, 1.0]], np.float32)
    d = oracle.dispatch(s, 2, 1)
    assert d["assign"].tolist() == [[0, -1], [1, -1]]
    assert d["flags"].tolist() == [[0, 2], [1, 2]]
    assert d["n_dropped"] == 2 and d["n_rerouted"] == 1
    assert d["cw"].tolist() == [[1.0, 0.0], [1.0, 0.0]]


def test_capacity_zero_drops_everything():
    s = np.random.default_rng(0).standard_normal((5, 4)).astype(np.float32)
    d = oracle.dispatch(s, 2, 0)
    assert (d["assign"] == -1).all() and d["n_dropped"] == 10 and d["perm"].size == 0


def _greedy_any_position(s, k, C):
    """Each entry takes the first expert in the WHOLE preference list that is
    not full and not already serving the token (rank-major, token-minor)."""
    T, E = s.shape
    pref = [sorted(range(E), key=lambda e: (-float(s[t, e]), e)) for t in range(T)]
    fill = [0] * E
    assign = [[-1] * k for _ in range(T)]
    for r in range(k):
        for t in range(T):
            for e in pref[t]:
                if fill[e] < C and e not in assign[t][:r]:
                    assign[t][r] = e
                    fill[e] += 1
                    break
    return assign


def _queue_simulation(s, k, C):
    """Independent form: arrivals enter per-expert queues in the order
    (rank, token); a queue at its limit bounces the arrival to the token's
    next candidate (cyclic from its own pick, skipping the token's experts)."""
    T, E = s.shape
    queues = {e: [] for e in range(E)}
    assign = [[-1] * k for _ in range(T)]
    for r in range(k):
        for t in range(T):
            cand = sorted(range(E), key=lambda e: (-float(s[t, e]), e))
            for e in cand[r:] + cand[:r]:
                if e in assign[t]:
                    continue
                if len(queues[e]) < C:
                    queues[e].append((t, r))
                    assign[t][r] = e
                    break
    slots = {}
    for e, q in queues.items():
        for i, tr in enumerate(q):
            slots[tr] = i
    return assign, slots


def test_dispatch_brute_force_tiny():
    rng = np.random.default_rng(6)
    for _ in range(400):
        T = int(rng.integers(1, 7))
        E = int(rng.integers(1, 6))
        k = int(rng.integers(1, min(3, E) + 1))
        C = int(rng.integers(0, 4))
        s = rng.integers(-2, 3, (T, E)).astype(np.float32)
        d = oracle.dispatch(s, k, C)
        assert d["assign"].tolist() == _greedy_any_position(s, k, C)
        qa, qs = _queue_simulation(s, k, C)
        assert d["assign"].tolist() == qa
        for t in range(T):
            for r in range(k):
                if qa[t][r] >= 0:
                    assert d["slot"][t, r] == qs[(t, r)]


def _check_dispatch_invariants(s, k, C, d):
    T, E = s.shape
    assign, slot, flags = d["assign"], d["slot"], d["flags"]
    kept = assign >= 0
    assert (d["counts"] <= C).all()
    assert d["counts"].sum() == T * k - d["n_dropped"] == kept.sum()
    assert np.array_equal(d["counts"], np.bincount(assign[kept], minlength=E))
    assert d["offsets"][0] == 0 and np.array_equal(np.diff(d["offsets"]), d["counts"])
    for t in range(T):
        e_t = assign[t][assign[t] >= 0]
        assert len(set(e_t.tolist())) == len(e_t)          # distinct experts per token
    for e in range(E):
        sl = np.sort(slot[assign == e])
        assert np.array_equal(sl, np.arange(d["counts"][e]))
    perm = d["perm"]
    assert sorted(perm.tolist()) == sorted(np.flatnonzero(kept.ravel()).tolist())
    for i, idx in enumerate(perm):
        e = assign.ravel()[idx]
        assert d["offsets"][e] <= i < d["offsets"][e + 1]
        assert slot.ravel()[idx] == i - d["offsets"][e]
    pref = np.array([oracle.preference(s[t]) for t in range(T)])
    for t in range(T):
        for r in range(k):
            if assign[t, r] < 0:
                assert flags[t, r] == 2
                held = set(assign[t][assign[t] >= 0].tolist())
                assert all(d["counts"][e] == C or e in held for e in range(E))
            else:
                assert flags[t, r] == (1 if assign[t, r] != pref[t, r] else 0)
    assert d["n_rerouted"] == int((flags == 1).sum()) and d["n_dropped"] == int((flags == 2).sum())
    cw = d["cw"]
    tot = np.where(kept, cw, 0).sum(1)
    assert np.all(np.abs(tot[kept.any(1)] - 1.0) < 1e-6)
    assert (cw[~kept] == 0).all()


@pytest.mark.parametrize("T,E,k,cf,skew", [(500, 8, 2, 1.0, 0.0), (300, 16, 2, 1.0, 2.0),
                                            (200, 5, 3, 1.0, 1.0), (64, 8, 1, 1.25, 0.5)])
def test_dispatch_invariants_random(T, E, k, cf, skew):
    rng = np.random.default_rng(T + E)
    s = rng.standard_normal((T, E)).astype(np.float32)
    s[:, 0] += skew
    s[T // 3: T // 3 + 40] = s[T // 3]       # a run of identical tokens
    C = oracle.capacity(T, k, E, cf)
    d = oracle.dispatch(s, k, C)
    _check_dispatch_invariants(s, k, C, d)
    assert d["assign"].tolist() == _greedy_any_position(s, k, C)


def test_no_overflow_is_plain_topk_with_stable_slots():
    rng = np.random.default_rng(7)
    T, E, k = 120, 6, 2
    s = rng.standard_normal((T, E)).astype(np.float32)
    d = oracle.dispatch(s, k, T)
    r = oracle.route(k, logits_in=s)
    assert np.array_equal(d["assign"], r["ids"]) and d["n_rerouted"] == 0
    seen = {}
    for r_ in range(k):
        for t in range(T):
            e = int(d["assign"][t, r_])
            assert d["slot"][t, r_] == seen.get(e, 0)
            seen[e] = seen.get(e, 0) + 1


def test_rank_major_order_matters():
    """All rank-0 picks are placed before any rank-1 pick: token 1's first
    choice beats token 0's second choice to the last slot."""
    s = np.array([[3.0, 2.0, 0.0], [2.0, 3.0, 0.0]], np.float32)
    d = oracle.dispatch(s, 2, 1)
    # rank 0: t0 -> 0, t1 -> 1; rank 1: t0 wants 1 (full) -> 2; t1 wants 0 (full), 2 full -> drop
    assert d["assign"].tolist() == [[0, 2], [1, -1]]


# --------------------------------------------------------------------------- combine weights

def test_combine_weight_page_example():
    g = golden("combine_mhpn_4_3.json")
    s = np.log(np.array([g["p"]], np.float64)).astype(np.float32)
    d = oracle.dispatch(s, 2, 10)
    # expert order follows the scores: p[1] > p[0]
    got = {int(e): float(w) for e, w in zip(d["assign"][0], d["cw"][0])}
    assert abs(got[0] - g["w"][0]) <= g["tol"] and abs(got[1] - g["w"][1]) <= g["tol"]
    assert abs(got[0] - 2.1 / 5.8) < 1e-6


def test_reroute_weight_uses_the_expert_actually_used():
    # C=1.  Rank 0: token 0 takes expert 0, token 1 finds 0 full and takes 1.
    # Rank 1: token 0 wants 1 (full) and takes 2; token 1 holds 1, so its next
    # candidate is 3.  Token 1 uses (1, 3) and its weights renormalise p1, p3.
    s = np.log(np.array([[0.5, 0.3, 0.15, 0.05], [0.55, 0.25, 0.05, 0.15]],
                        np.float64)).astype(np.float32)
    d = oracle.dispatch(s, 2, 1)
    assert d["assign"].tolist() == [[0, 2], [1, 3]]
    assert d["flags"].tolist() == [[0, 1], [1, 1]]
    np.testing.assert_allclose(d["cw"][1], [0.25 / 0.4, 0.15 / 0.4], rtol=1e-6)
    np.testing.assert_allclose(d["cw"][0], [0.5 / 0.65, 0.15 / 0.65], rtol=1e-6)


def test_k1_weight_is_one():
    s = np.random.default_rng(8).standard_normal((40, 5)).astype(np.float32)
    d = oracle.dispatch(s, 1, 40)
    assert (d["cw"] == 1.0).all()


# --------------------------------------------------------------------------- experts

def test_dense_swiglu_reduces_to_torch():
    """E=1, k=1, no overflow: the layer is a dense SwiGLU FFN."""
    rng = np.random.default_rng(9)
    T, d, F = 9, 32, 48
    h = bf16(rng.standard_normal((T, d)))
    wr = bf16(rng.standard_normal((1, d)))
    w1 = bf16(rng.standard_normal((1, F, d)) / math.sqrt(d))
    w3 = bf16(rng.standard_normal((1, F, d)) / math.sqrt(d))
    w2 = bf16(rng.standard_normal((1, d, F)) / math.sqrt(F))
    r, dsp, out = oracle.layer_forward(h, wr, w1, w3, w2, k=1, C=T)
    x = torch.from_numpy(widen(h)).double()
    g = x @ torch.from_numpy(widen(w1)[0]).double().T
    u = x @ torch.from_numpy(widen(w3)[0]).double().T
    y = (torch.nn.functional.silu(g) * u) @ torch.from_numpy(widen(w2)[0]).double().T
    np.testing.assert_allclose(out, y.numpy(), rtol=1e-6, atol=1e-6)


def test_gate_and_up_branches_are_not_swapped():
    """x = e_0; W1 rows c_j e_0 and W3 rows e_0 give a_j = silu(c_j);
    swapping the branches gives a_j = silu(1) * c_j instead.  W2 = identity."""
    d = F = 8
    c = np.linspace(-3, 3, F)
    x = np.zeros(d)
    x[0] = 1.0
    w1 = np.zeros((F, d))
    w1[:, 0] = c
    w3 = np.zeros((F, d))
    w3[:, 0] = 1.0
    w2 = np.eye(d, F)
    y = oracle.expert_row(bf16(x), bf16(w1), bf16(w3), bf16(w2))
    cb = widen(bf16(c)).astype(np.float64)
    want = cb / (1.0 + np.exp(-cb))
    np.testing.assert_allclose(y, want, rtol=1e-12)
    swapped = oracle.expert_row(bf16(x), bf16(w3), bf16(w1), bf16(w2))
    assert not np.allclose(swapped, want)


def test_down_projection_orientation():
    """W2 is [d, F] (out x in): a one-hot W2 row picks one activation."""
    d, F = 4, 6
    x = np.zeros(d)
    x[1] = 1.0
    w1 = np.zeros((F, d))
    w1[:, 1] = 1.0
    w3 = np.zeros((F, d))
    w3[:, 1] = np.arange(1, F + 1)
    w2 = np.zeros((d, F))
    w2[2, 5] = 1.0
    y = oracle.expert_row(bf16(x), bf16(w1), bf16(w3), bf16(w2))
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(y, [0, 0, s1 * 6, 0], rtol=1e-12)


def test_combine_rows_weights_and_drops():
    rng = np.random.default_rng(10)
    T, d, E, F, k = 6, 16, 3, 24, 2
    h = bf16(rng.standard_normal((T, d)))
    w1 = bf16(rng.standard_normal((E, F, d)) / 4)
    w3 = bf16(rng.standard_normal((E, F, d)) / 4)
    w2 = bf16(rng.standard_normal((E, d, F)) / 5)
    assign = np.array([[0, 1], [2, -1], [-1, -1], [1, 0], [2, 0], [0, 2]], np.int32)
    cw = np.array([[0.25, 0.75], [1, 0], [0, 0], [0.5, 0.5], [0.1, 0.9], [0.6, 0.4]], np.float32)
    out = oracle.combine_rows(h, w1, w3, w2, assign, cw, np.arange(T))
    assert (out[2] == 0).all()
    for t in range(T):
        want = np.zeros(d)
        for r in range(k):
            e = assign[t, r]
            if e >= 0:
                want += cw[t, r] * oracle.expert_row(h[t], w1[e], w3[e], w2[e])
        np.testing.assert_allclose(out[t], want, rtol=1e-6, atol=1e-7)


def test_expert_slots_follow_perm():
    rng = np.random.default_rng(11)
    T, d, E, F, k = 20, 16, 4, 32, 2
    h = bf16(rng.standard_normal((T, d)))
    w1 = bf16(rng.standard_normal((E, F, d)) / 4)
    w3 = bf16(rng.standard_normal((E, F, d)) / 4)
    w2 = bf16(rng.standard_normal((E, d, F)) / 5)
    s = rng.standard_normal((T, E)).astype(np.float32)
    dsp = oracle.dispatch(s, k, oracle.capacity(T, k, E, 1.0))
    ys = oracle.expert_slots(h, w1, w3, w2, dsp["assign"], dsp["perm"], 0, dsp["perm"].size)
    for i, idx in enumerate(dsp["perm"]):
        t, r = divmod(int(idx), k)
        e = dsp["assign"][t, r]
        np.testing.assert_allclose(ys[i], oracle.expert_row(h[t], w1[e], w3[e], w2[e]),
                                   rtol=1e-6, atol=1e-7)


# --------------------------------------------------------------------------- the five workloads

@pytest.mark.parametrize("name", synth.CONFIG_ORDER)
def test_workload_router_statistics(name):
    """Routing + dispatch of each workload's seeded inputs satisfy the
    invariants, and the skewed workload's expert-0 rank-1 share is the
    calibrated 42.66%."""
    shape = synth.CONFIGS[name]
    C = oracle.capacity(shape.T, shape.k, shape.E, shape.cf, shape.capacity)
    if shape.T * shape.d <= 8192 * 4096:
        h, wr, bias, usage = synth.router_inputs(shape)
        r = oracle.route(shape.k, h=synth.bf16_bits(h), wr=synth.bf16_bits(wr),
                         bias=None if bias is None else bias.numpy(),
                         usage=None if usage is None else usage.numpy(), lam=shape.lam)
        s = r["scores"]
        assert r["counts_pre"].sum() == shape.T * shape.k
    else:
        rng = np.random.default_rng(shape.seed)
        s = (rng.standard_normal((shape.T, shape.E)) * 0.02 * math.sqrt(shape.d)).astype(np.float32)
    d = oracle.dispatch(s, shape.k, C)
    assert (d["counts"] <= C).all()
    assert d["counts"].sum() == shape.T * shape.k - d["n_dropped"]
    if name == "skewed":
        assert abs((oracle.route(2, logits_in=s)["ids"][:, 0] == 0).mean() - 0.4266) < 1e-3


# ----------------------------------------------------------------------------- e4m3 weights

# Codes and values fixed by the e4m3 format: sign bit, exponent bias 7, three
# mantissa bits, subnormals m/8 * 2^-6 at exponent 0, no infinity, 0x7F NaN.
E4M3_KNOWN = [(0x00, 0.0), (0x80, -0.0), (0x38, 1.0), (0xB8, -1.0), (0x3C, 1.5), (0x40, 2.0),
              (0x7E, 448.0), (0xFE, -448.0), (0x77, 240.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9),
              (0x07, 7 * 2.0 ** -9), (0x0F, 1.875 * 2.0 ** -6), (0x30, 0.5), (0x39, 1.125)]


@pytest.mark.parametrize("code,value", E4M3_KNOWN)
def test_e4m3_known_codes(code, value):
    got = oracle.e4m3_value(code)
    assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value)


def test_e4m3_nan_codes():
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    # encoding NaN gives the positive NaN code, as torch's float8_e4m3fn conversion does
    ref = torch.tensor([float("nan")]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    assert oracle.e4m3_encode(float("nan")) == ref == 0x7F


def test_e4m3_all_codes_match_torch():
    """Every code against torch's float8_e4m3fn -> float conversion (a library routine)."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def test_q8_experts_equal_bf16_experts_on_exact_weights():
    """Weights that are e4m3 values times power-of-two row scales are exact in
    bf16 too: the 8-bit path must then give the bf16 path's numbers exactly (a
    dropped scale, a row/column mix-up or a wrong row stride breaks this)."""
    rng = np.random.default_rng(11)
    T, d, F, E, k = 6, 32, 24, 3, 2
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    q1, q3 = (rng.choice(finite, size=(E, F, d)) for _ in range(2))
    q2 = rng.choice(finite, size=(E, d, F))
    s1, s3 = (np.ldexp(1.0, rng.integers(-12, -4, size=(E, F))).astype(np.float32) for _ in range(2))
    s2 = np.ldexp(1.0, rng.integers(-12, -4, size=(E, d))).astype(np.float32)
    val = np.vectorize(oracle.e4m3_value)
    w1 = val(q1) * s1[:, :, None]
    w3 = val(q3) * s3[:, :, None]
    w2 = val(q2) * s2[:, :, None]
    h = bf16(rng.standard_normal((T, d)))
    assign = rng.integers(0, E, size=(T, k)).astype(np.int32)
    assign[2, 1] = -1
    cw = rng.random((T, k)).astype(np.float32)
    toks = np.arange(T, dtype=np.int32)
    got = oracle.combine_rows_q8(h, q1, s1, q3, s3, q2, s2, assign, cw, toks, quant_act=False)
    want = oracle.combine_rows(h, bf16(w1), bf16(w3), bf16(w2), assign, cw, toks)
    assert np.array_equal(got, want)
    # a scale that is off by one row changes the result
    s1_bad = np.roll(s1, 1, axis=1)
    bad = oracle.combine_rows_q8(h, q1, s1_bad, q3, s3, q2, s2, assign, cw, toks, quant_act=False)
    assert not np.array_equal(bad, want)


def test_e4m3_encode_inverts_decode():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c, c


@pytest.mark.parametrize("v,code", [(1.0625, 0x38), (1.1875, 0x3A), (3 * 2.0 ** -10, 0x02),
                                    (2.0 ** -10, 0x00), (-(2.0 ** -10), 0x80), (448.0, 0x7E),
                                    (460.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE),
                                    (0.3, 0x2A)])   # 0.3 = 1.2*2^-2: 0.3125 (1.25*2^-2) is nearest
def test_e4m3_encode_ties_and_saturation(v, code):
    """Halfway values go to the even code; magnitudes past 448 saturate."""
    assert oracle.e4m3_encode(v) == code


def test_e4m3_encode_matches_torch():
    """Round-to-nearest-even against torch's float8_e4m3fn conversion (within range)."""
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-4, 2.6, 20000),
                        rng.uniform(-448, 448, 2000)]).astype(np.float32)
    v = v[np.abs(v) < 464]   # torch turns larger magnitudes into NaN; the encoder saturates
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(x) for x in v], np.uint8)
    assert v.size > 15000 and np.array_equal(got, ref)


def test_quantize_row_matches_torch():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(700) * 3).astype(np.float32)
    codes, sc = oracle.quantize_row(x)
    assert sc == np.float32(np.abs(x).max()) / np.float32(448.0)
    ref = torch.from_numpy(x / np.float32(sc)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    codes0, sc0 = oracle.quantize_row(np.zeros(5, np.float32))
    assert sc0 == 1.0 and not codes0.any()


def _e4m3_codes(values):
    """Codes of values that e4m3 holds exactly (torch's float8_e4m3fn conversion, a
    library routine); checked to decode back to the same values."""
    v = torch.as_tensor(np.asarray(values, np.float64))
    codes = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy(),
                          v.numpy()), "not exact in e4m3"
    return codes


def _q8_rows(w, scales):
    """Weights [.., rows, cols] that are e4m3 values times a per-row scale: (codes, scales)."""
    scales = np.asarray(scales, np.float32)
    return _e4m3_codes(w / scales[..., None]).reshape(np.shape(w)), scales


def test_q8_activation_quantisation_is_identity_on_exact_rows():
    """quant_act=1 against quant_act=0 where both quantisations are lossless.

    Each token row is e4m3 values times 2^p with 7*2^p (= 448 * 2^(p-6)) its largest
    magnitude, so the row scale max/448 is the power of two 2^(p-6) and the codes give the
    row back exactly.  W1 sends column 1 (= 2^p) to every gate, g = 64 * 2^p >= 64, where
    silu(g) = g/(1 + e^-g) equals g in double; W3 scales the same column by an e4m3 value
    over 64, so a = silu(g) u is an e4m3 value times 2^p with 448 * 2^p in every row: exact
    in bf16 and again quantised losslessly.  The two paths must then agree bit for bit.
    A dequantisation that drops the scale, a scale other than max/448, or an activation
    scale taken from g, u or x instead of the bf16 activation row breaks the equality."""
    rng = np.random.default_rng(21)
    T, d, F, E, k = 5, 16, 8, 3, 2
    vals = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = torch.from_numpy(vals).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    small = vals[(np.abs(vals) < 448) & (np.abs(vals) >= 2.0 ** -6)]
    p = rng.integers(0, 3, size=T)
    x = rng.choice(small, size=(T, d)) * 2.0 ** -6
    x[:, 0] = 7.0
    x[:, 1] = 1.0
    x *= (2.0 ** p)[:, None]
    h = bf16(x)
    assert np.array_equal(widen(h), x.astype(np.float32))
    w1 = np.zeros((E, F, d))
    w1[:, :, 1] = 64.0
    w3 = np.zeros((E, F, d))
    w3[:, :, 1] = rng.choice(small[np.abs(small) <= 64], size=(E, F)) / 64.0
    w3[:, 0, 1] = 7.0                       # a = 448 * 2^p in every row
    w2 = rng.choice(small, size=(E, d, F)) * 2.0 ** -9
    q1, s1 = _q8_rows(w1, np.ones((E, F)))
    q3, s3 = _q8_rows(w3, np.full((E, F), 2.0 ** -6))
    q2, s2 = _q8_rows(w2, np.full((E, d), 2.0 ** -9))
    assign = np.array([[0, 1], [2, 0], [1, -1], [2, 1], [0, 2]], np.int32)
    cw = rng.random((T, k)).astype(np.float32)
    toks = np.arange(T, dtype=np.int32)
    exact = oracle.combine_rows_q8(h, q1, s1, q3, s3, q2, s2, assign, cw, toks, quant_act=False)
    quant = oracle.combine_rows_q8(h, q1, s1, q3, s3, q2, s2, assign, cw, toks, quant_act=True)
    assert np.abs(exact).max() > 0
    assert np.array_equal(quant, exact)
    perm = np.array([0, 3, 9, 7, 2, 6, 1, 8, 4], np.int32)     # every kept entry once
    slots = oracle.expert_slots_q8(h, q1, s1, q3, s3, q2, s2, assign, perm, 0, perm.size, quant_act=True)
    slots0 = oracle.expert_slots_q8(h, q1, s1, q3, s3, q2, s2, assign, perm, 0, perm.size, quant_act=False)
    assert np.array_equal(slots, slots0)


def _rounding_case():
    """Two token rows, x_B = 2 x_A, one expert (d = 8, F = 4), worked by hand.

    x_A = (7, 1, 2^-6, 2^-4, 1.15625, 0, 0, 0): max 7, so the row scale is 7/448 = 2^-6;
    x/scale = (448, 64, 1, 4, 74), and 74 lies between the e4m3 values 72 and 80, so the
    quantised row is x'_A = (7, 1, 2^-6, 2^-4, 1.125, 0, 0, 0); x_B has scale 2^-5 and the
    same codes, x'_B = 2 x'_A.
    W1 puts 64 on column 1 in every row: g = 64 (A) and 128 (B), where silu(g) = g in
    double.  W3 rows: 7 e_1; 2^-6 e_1 + 2^-10 e_2 + 2^-6 e_3; (15/1024) e_4; 2^-3 e_1
    (e4m3 codes times a row scale of 1, 2^-14, 2^-8, 1).
      A: u = (7, 2^-6 + 2^-16 + 2^-10, (15/1024) 1.125, 2^-3),
         a = 64 u = (448, 1 + 2^-4 + 2^-10, 1.0546875, 8).
         bf16 rounds a_1 = 1.0634765625 to 1.0625 (7 fraction bits); the row max is 448,
         scale 1; 1.0625 lies halfway between the e4m3 values 1 and 1.125 and ties to the
         even code, 1; 1.0546875 rounds to 1.  a' = (448, 1, 1, 8).
         (Quantising the unrounded a_1 would give 1.125; the unquantised token value
         1.15625 would make a_2 = 1.083984375 and a'_2 = 1.125.)
      B: a = (1792, 4.25390625, 4.21875, 32) -> bf16 (1792, 4.25, 4.21875, 32), scale
         1792/448 = 4, a/4 = (448, 1.0625, 1.0546875, 8) -> (448, 1, 1, 8),
         a' = (1792, 4, 4, 32).
    W2 rows (e4m3 times 2^-8 or 1): 2^-8 e_0; e_1; 2^-3 e_3; 2^-1 e_1 + 2^-4 e_3; e_2; zeros.
      y_A = (448/256, 1, 1, 1/2 + 1/2, 1, 0, 0, 0) = (1.75, 1, 1, 1, 1, 0, 0, 0)
      y_B = (7, 4, 4, 4, 4, 0, 0, 0)."""
    d, F = 8, 4
    x = np.zeros((2, d))
    x[0, :5] = [7, 1, 2.0 ** -6, 2.0 ** -4, 1.15625]
    x[1] = 2 * x[0]
    w1 = np.zeros((1, F, d))
    w1[0, :, 1] = 64
    w3 = np.zeros((1, F, d))
    w3[0, 0, 1] = 7
    w3[0, 1, 1:4] = [2.0 ** -6, 2.0 ** -10, 2.0 ** -6]
    w3[0, 2, 4] = 15 / 1024
    w3[0, 3, 1] = 2.0 ** -3
    w2 = np.zeros((1, d, F))
    w2[0, 0, 0] = 2.0 ** -8
    w2[0, 1, 1] = 1
    w2[0, 2, 3] = 2.0 ** -3
    w2[0, 3, 1] = 0.5
    w2[0, 3, 3] = 2.0 ** -4
    w2[0, 4, 2] = 1
    q1, s1 = _q8_rows(w1, np.ones((1, F)))
    q3, s3 = _q8_rows(w3, [[1, 2.0 ** -14, 2.0 ** -8, 1]])
    q2, s2 = _q8_rows(w2, [[2.0 ** -8, 1, 1, 1, 1, 1, 1, 1]])
    want = np.array([[1.75, 1, 1, 1, 1, 0, 0, 0], [7, 4, 4, 4, 4, 0, 0, 0]], np.float32)
    return bf16(x), (q1, s1, q3, s3, q2, s2), want


def test_q8_activation_rounding_hand_case():
    """The bf16 rounding of a = silu(g) u before its quantisation decides an e4m3 code
    (the tie at 1.0625), and the token row's quantisation decides another (74 -> 72):
    the hand-worked rows of _rounding_case, through both the token-order and the
    slot-order oracle functions."""
    h, q, want = _rounding_case()
    assign = np.array([[0], [0]], np.int32)
    cw = np.ones((2, 1), np.float32)
    got = oracle.combine_rows_q8(h, *q, assign, cw, np.arange(2, dtype=np.int32), quant_act=True)
    np.testing.assert_array_equal(got, want)
    slots = oracle.expert_slots_q8(h, *q, assign, np.array([1, 0], np.int32), 0, 2, quant_act=True)
    np.testing.assert_array_equal(slots, want[::-1])
    # without quantisation of the token and activation rows the unrounded values reach
    # the output: a_1 = 1.0634765625 and a_2 = 64 (15/1024) 1.15625 = 1.083984375
    raw = oracle.combine_rows_q8(h, *q, assign, cw, np.arange(2, dtype=np.int32), quant_act=False)
    assert raw[0, 1] == np.float32(1.0634765625) and raw[1, 1] == np.float32(4 * 1.0634765625)
    assert raw[0, 4] == np.float32(1.083984375) and raw[1, 4] == np.float32(4 * 1.083984375)


# ----------------------------------------------------------------------------- NVFP4 weights
# e2m1 (the OCP microscaling FP4 element): sign, 2-bit exponent with bias 1, 1-bit mantissa,
# exponent 0 the subnormal 0.5; NVFP4 groups 16 elements under one e4m3 block scale
# ([2kiu] §5.1 quantises experts to 4-6 bits; the format choice is this library's).

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_all_codes():
    for c in range(16):
        want = E2M1[c & 7] * (-1.0 if c & 8 else 1.0)
        got = oracle.e2m1_value(c)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), c


def _e2m1_nearest(v):
    """Brute force: the magnitude nearest to |v|, ties to the even code (mantissa bit 0)."""
    a = abs(v)
    best = min(range(8), key=lambda c: (abs(a - E2M1[c]), c & 1))
    return best | (8 if math.copysign(1.0, v) < 0 else 0)


def test_e2m1_encode_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(12)
    grid = np.arange(-64, 65) / 8.0                      # every tie and every code value
    vals = np.concatenate([grid, rng.uniform(-8, 8, 3000), rng.standard_normal(2000) * 3,
                           [1e30, -1e30, 6.0001, -5.9999, 0.2499, 0.2501]]).astype(np.float32)
    for v in vals:
        assert oracle.e2m1_encode(float(v)) == _e2m1_nearest(float(v)), v


def _nvfp4_exact_row(rng, blocks, scale_pow, max_block):
    """A row that NVFP4 represents exactly: block j is e2m1 values times v_j * 2^scale_pow,
    v_j an e4m3 power of two, its largest magnitude 6 (so its block scale is v_j), and block
    `max_block` has v = 448 (so the row scale is 2^scale_pow).  Returns the row and (v_j)."""
    s = 2.0 ** scale_pow
    vs = [2.0 ** int(rng.integers(-6, 8)) for _ in range(blocks)]
    vs[max_block] = 448.0
    row = []
    for v in vs:
        c = rng.choice(E2M1, size=16) * rng.choice([-1.0, 1.0], size=16)
        c[int(rng.integers(16))] = 6.0 * rng.choice([-1.0, 1.0])
        row.append(c * v * s)
    return np.concatenate(row), vs


def test_nvfp4_row_quantisation_is_exact_on_representable_rows():
    """Rows of e2m1 values times power-of-two block scales, with 6 in every block and
    6 * 448 * 2^p as the row's largest magnitude: the scale is 2^p, every block scale
    comes back exactly and every code gives its value back (a dropped factor of 6 or
    448, a block scale taken from the wrong block, or swapped nibbles break this)."""
    rng = np.random.default_rng(13)
    for trial in range(20):
        blocks = int(rng.integers(1, 9))
        p = int(rng.integers(-12, 4))
        row, vs = _nvfp4_exact_row(rng, blocks, p, int(rng.integers(blocks)))
        codes, bs, sc = oracle.quantize_row_nvfp4(row.astype(np.float32))
        assert sc == 2.0 ** p
        assert [oracle.e4m3_value(b) for b in bs] == vs
        vals = [oracle.e2m1_value((codes[i // 2] >> (4 * (i & 1))) & 15) * vs[i // 16] * sc
                for i in range(row.size)]
        assert np.array_equal(np.array(vals), row)


def test_nvfp4_row_quantisation_hand_case():
    """32 elements worked by hand.  max|x| = 21, scale = 21 / 2688 = 2^-7.
    Block 0 = (21, 7, 3.5, 1, zeros): t = 21 / scale = 2688, u = t / 6 = 448 -> block code
    0x7E; den = 448 * scale = 3.5; x / den = (6, 2, 1, 0.2857...) -> codes 7, 4, 2, 1
    (0.2857 is nearer 0.5 than 0).
    Block 1 = (-0.7, 0.35, zeros): t = 0.7 / scale = 89.6, u = 14.93... -> e4m3 15
    (1.875 * 8, code 0x57); den = 15 * scale = 0.1171875; x / den = (-5.9733, 2.9866)
    -> codes 15 (-6) and 5 (3: exponent 2, mantissa 1)."""
    x = np.zeros(32, np.float32)
    x[:4] = [21, 7, 3.5, 1]
    x[16:18] = [-0.7, 0.35]
    codes, bs, sc = oracle.quantize_row_nvfp4(x)
    assert sc == 2.0 ** -7
    assert list(bs) == [0x7E, 0x57]
    nib = [(codes[i // 2] >> (4 * (i & 1))) & 15 for i in range(32)]
    assert nib[:4] == [7, 4, 2, 1] and nib[16:18] == [15, 5]
    assert not any(nib[4:16]) and not any(nib[18:])


def test_nvfp4_zero_row_and_underflowing_block():
    """The two degenerate cases of the row quantisation.  An all-zero row has row scale 1
    and every code and block scale 0.  A block whose maximum is below about 2^-21 of the
    row's maximum gets a block scale that rounds to the e4m3 zero: with max 1e-7 against
    1.0, u = 1e-7 * 2688 / 6 = 4.48e-5, under half the smallest subnormal (2^-10).  Its
    divisor is then 0, and its codes are 0 (not saturated by x / 0), so the block
    decodes to zeros."""
    codes, bs, sc = oracle.quantize_row_nvfp4(np.zeros(32, np.float32))
    assert sc == 1.0 and not codes.any() and not bs.any()
    x = np.zeros(32, np.float32)
    x[0], x[16], x[17] = 1.0, 1e-7, -3e-8
    codes, bs, sc = oracle.quantize_row_nvfp4(x)
    assert sc == np.float32(1.0) / np.float32(2688.0)
    assert bs[0] == 0x7E and bs[1] == 0
    nib = [(codes[i // 2] >> (4 * (i & 1))) & 15 for i in range(32)]
    assert nib[0] == 7 and not any(nib[1:])


def _q4_weights(rng, E, rows, cols, exact=True):
    """NVFP4 weights [E, rows, cols]: random codes, random e4m3 block scales (powers of two
    when `exact`, so that every weight is exact in bf16), power-of-two row scales."""
    codes = rng.integers(0, 16, size=(E, rows, cols)).astype(np.uint8)
    if exact:
        bvals = 2.0 ** rng.integers(-4, 5, size=(E, rows, cols // 16))
        b = np.vectorize(oracle.e4m3_encode)(bvals.astype(np.float32)).astype(np.uint8)
    else:
        b = rng.integers(0x20, 0x60, size=(E, rows, cols // 16)).astype(np.uint8)
    s = (2.0 ** rng.integers(-10, -4, size=(E, rows))).astype(np.float32)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    val = (np.vectorize(oracle.e2m1_value)(codes) * np.vectorize(oracle.e4m3_value)(b).repeat(16, axis=2)
           * s[..., None])
    return (packed, b, s), val


def test_q4_experts_equal_bf16_experts_on_exact_weights():
    """NVFP4 weights whose values are exact in bf16: without activation quantisation the
    4-bit path must give the bf16 path's numbers exactly; a block scale moved to the next
    block changes them."""
    rng = np.random.default_rng(14)
    T, d, F, E, k = 5, 32, 48, 3, 2
    w1, v1 = _q4_weights(rng, E, F, d)
    w3, v3 = _q4_weights(rng, E, F, d)
    w2, v2 = _q4_weights(rng, E, d, F)
    h = bf16(rng.standard_normal((T, d)))
    assign = np.array([[0, 1], [2, 0], [1, -1], [2, 1], [0, 2]], np.int32)
    cw = rng.random((T, k)).astype(np.float32)
    toks = np.arange(T, dtype=np.int32)
    got = oracle.combine_rows_q4(h, w1, w3, w2, assign, cw, toks, quant_act=False)
    want = oracle.combine_rows(h, bf16(v1), bf16(v3), bf16(v2), assign, cw, toks)
    assert np.array_equal(bf16(v1), bf16(v1.astype(np.float32))) and np.array_equal(got, want)
    bad1 = (w1[0], np.roll(w1[1], 1, axis=2), w1[2])
    assert not np.array_equal(oracle.combine_rows_q4(h, bad1, w3, w2, assign, cw, toks, quant_act=False), want)


def _q4_act_case():
    """Token rows A and B = 2A (d = 48: three blocks) and one expert (F = 32), built so that
    both NVFP4 quantisations are exact except where stated.
    x_A: block 0 = (6, 1, 0, ...) (block scale 256, unit 1), block 1 = (10.5, 0, ...) (the
    row's largest: scale 10.5 / 2688 = 2^-8, block scale 448), block 2 = (6 * 2^-9, 2^-9,
    1.25 * 2^-9, 0, ...) (block scale 0.5, unit 2^-9): every code gives its value back
    except x_34, where 1.25 units lie halfway between 1 and 1.5 and tie to 1: x'_34 = 2^-9.
    W1: 64 on column 1 in every row: g = 64 (A), 128 (B); silu(g) = g in double.
    W3 rows: 0: 0.375 e_1; 1: (5/64) e_1 + 2^-5 e_33; 2: 96 e_34; 16: 10.5 e_1; others zero.
      A: u = (0.375, 5/64 + 2^-14, 96 * 2^-9, ..., 10.5 at 16),
         a = 64 u = (24, 5 + 2^-8, 12, 0, ..., 672).
      The activation row's largest is 672: scale 0.25; block 0 max 24: block scale 16, unit 4;
      a_1 rounds to bf16 5 (ulp 2^-5 at 4..8), 5 / 4 = 1.25 is halfway between the e2m1
      values 1 and 1.5 and ties to 1: a'_1 = 4 (unrounded, 1.2509... -> 1.5: 6).  a'_2 = 12
      (3 units; with the unquantised x_34 it would be 15 -> 3.75 units -> 4: 16).  a'_0 = 24,
      a'_16 = 672 exactly.  B: g and u double, so a and its scale quadruple.
    W2 rows: 0: e_1; 1: e_0; 2: 2^-4 e_16; 3: e_2; the others zero.
      y_A = (4, 24, 42, 12, 0, ...), y_B = (16, 96, 168, 48, 0, ...)."""
    d, F = 48, 32
    x = np.zeros((2, d))
    x[0, [0, 1, 16, 32, 33, 34]] = [6, 1, 10.5, 6 * 2.0 ** -9, 2.0 ** -9, 1.25 * 2.0 ** -9]
    x[1] = 2 * x[0]

    def pack(vals, codes_for, bscale_vals, row_scales):
        rows, cols = vals.shape
        codes = np.zeros((rows, cols), np.uint8)
        for r in range(rows):
            for c in range(cols):
                v = vals[r, c] / (bscale_vals[r][c // 16] * row_scales[r])
                codes[r, c] = codes_for[v]
                assert E2M1[codes[r, c] & 7] * (-1 if codes[r, c] & 8 else 1) == v
        b = np.array([[oracle.e4m3_encode(v) for v in bv] for bv in bscale_vals], np.uint8)
        assert all(oracle.e4m3_value(bb) == vv for br, bv in zip(b, bscale_vals) for bb, vv in zip(br, bv))
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        return packed[None], b[None], np.asarray(row_scales, np.float32)[None]

    enc = {v: i for i, v in enumerate(E2M1)}
    enc.update({-v: i | 8 for i, v in enumerate(E2M1) if v})
    w1 = np.zeros((F, d))
    w1[:, 1] = 64
    w3 = np.zeros((F, d))
    w3[0, 1] = 0.375
    w3[1, 1] = 5 / 64
    w3[1, 33] = 2.0 ** -5
    w3[2, 34] = 96
    w3[16, 1] = 10.5
    w2 = np.zeros((d, F))
    w2[0, 1] = 1
    w2[1, 0] = 1
    w2[2, 16] = 2.0 ** -4
    w2[3, 2] = 1
    # block scales and row scales that make every weight an e2m1 value
    w1q = pack(w1, enc, [[64.0] * 3] * F, [0.25] * F)        # 64 = 4 * 64 * 0.25
    w3_b = [[1.0] * 3 for _ in range(F)]
    w3_s = [1.0] * F
    w3_b[0] = [0.25, 1, 1]                     # 0.375 = 1.5 * 0.25
    w3_b[1], w3_s[1] = [5.0, 1, 2.0], 2.0 ** -6     # 5/64 = 1 * 5 * 2^-6; 2^-5 = 1 * 2 * 2^-6
    w3_b[2] = [1, 1, 16.0]                     # 96 = 6 * 16
    w3_b[16] = [1.75, 1, 1]                    # 10.5 = 6 * 1.75
    w3q = pack(w3, enc, w3_b, w3_s)
    w2_b = [[1.0] * 2 for _ in range(d)]
    w2_s = [1.0] * d
    w2_b[2], w2_s[2] = [1, 1.0], 2.0 ** -4
    w2q = pack(w2, enc, w2_b, w2_s)
    want = np.zeros((2, d), np.float32)
    want[0, :4] = [4, 24, 42, 12]
    want[1, :4] = [16, 96, 168, 48]
    return bf16(x), w1q, w3q, w2q, want


def test_q4_activation_quantisation_hand_case():
    """The bf16 rounding of the activation before its NVFP4 quantisation decides a code
    (the tie at 1.25 in units of 4), and the token row's quantisation decides another
    (x_34), through the token-order and slot-order functions; quantising without the
    rounding would give a'_1 = 6, without the token quantisation a'_2 = 16."""
    h, w1, w3, w2, want = _q4_act_case()
    assign = np.array([[0], [0]], np.int32)
    cw = np.ones((2, 1), np.float32)
    got = oracle.combine_rows_q4(h, w1, w3, w2, assign, cw, np.arange(2, dtype=np.int32), quant_act=True)
    np.testing.assert_array_equal(got, want)
    slots = oracle.expert_slots_q4(h, w1, w3, w2, assign, np.array([1, 0], np.int32), 0, 2, quant_act=True)
    np.testing.assert_array_equal(slots, want[::-1])
    raw = oracle.combine_rows_q4(h, w1, w3, w2, assign, cw, np.arange(2, dtype=np.int32), quant_act=False)
    assert raw[0, 0] == np.float32(5 + 2.0 ** -8) and raw[1, 0] == np.float32(4 * (5 + 2.0 ** -8))


# --------------------------------------------------------------------------- router variants
# Temperature ([cnnetsun] §3.1 step 3; [2kiu] §2), normalisation before the
# router ([2kiu] §5.2), the two-layer router silu(x W1) W2 ([cnnetsun] §3.1 step 2).


def _eye(n):
    return bf16(np.eye(n))


def test_layernorm_worked_example():
    # mean 2.5, mean squared deviation 1.25: x = (h - 2.5) / sqrt(1.25)
    z = oracle.router_logits(bf16([[1, 2, 3, 4]]), _eye(4), norm=oracle.NORM_LAYER, eps=0.0)
    s = 1.0 / math.sqrt(1.25)
    np.testing.assert_allclose(z[0], [-1.5 * s, -0.5 * s, 0.5 * s, 1.5 * s], rtol=1e-7)
    # gamma scales and beta shifts each normalised component
    z = oracle.router_logits(bf16([[1, 2, 3, 4]]), _eye(4), gamma=[1, 2, 3, 4], beta=[0.5, 0, 0, -1],
                             norm=oracle.NORM_LAYER, eps=0.0)
    np.testing.assert_allclose(z[0], [-1.5 * s + 0.5, -1.0 * s, 1.5 * s, 6.0 * s - 1.0], rtol=1e-7)


def test_layernorm_shift_and_scale_invariance():
    rng = np.random.default_rng(21)
    h = rng.integers(-20, 20, (6, 16)).astype(np.float32)
    w = bf16(rng.standard_normal((5, 16)))
    a = oracle.router_logits(bf16(h), w, norm=oracle.NORM_LAYER, eps=0.0)
    b = oracle.router_logits(bf16(3 * h + 7), w, norm=oracle.NORM_LAYER, eps=0.0)   # exact in bf16
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-6)


def test_layernorm_router_reduces_to_torch():
    rng = np.random.default_rng(22)
    T, d, E = 11, 64, 6
    h = bf16(rng.standard_normal((T, d)) * 3 + 1)
    w = bf16(rng.standard_normal((E, d)) * 0.1)
    gamma = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    beta = (0.1 * rng.standard_normal(d)).astype(np.float32)
    bias = rng.standard_normal(E).astype(np.float32)
    z = oracle.router_logits(h, w, gamma=gamma, beta=beta, bias=bias, norm=oracle.NORM_LAYER, eps=1e-5)
    x = torch.nn.functional.layer_norm(torch.from_numpy(widen(h)).double(), (d,),
                                       torch.from_numpy(gamma).double(), torch.from_numpy(beta).double(), 1e-5)
    want = x @ torch.from_numpy(widen(w)).double().T + torch.from_numpy(bias).double()
    np.testing.assert_allclose(z, want.numpy().astype(np.float32), rtol=2e-7, atol=1e-6)


def test_l2_norm_worked_example_and_torch():
    z = oracle.router_logits(bf16([[3, 4, 0, 0], [0, 0, 0, 0]]), _eye(4), norm=oracle.NORM_L2, eps=1e-12)
    np.testing.assert_allclose(z, [[0.6, 0.8, 0, 0], [0, 0, 0, 0]], rtol=1e-7)
    rng = np.random.default_rng(23)
    h = bf16(rng.standard_normal((9, 32)) * 50)
    w = bf16(rng.standard_normal((4, 32)))
    z = oracle.router_logits(h, w, norm=oracle.NORM_L2, eps=1e-12)
    x = torch.nn.functional.normalize(torch.from_numpy(widen(h)).double(), p=2.0, dim=1, eps=1e-12)
    want = x @ torch.from_numpy(widen(w)).double().T
    np.testing.assert_allclose(z, want.numpy().astype(np.float32), rtol=2e-7, atol=1e-7)


def test_l2_norm_eps_is_a_floor():
    """eps bounds the divisor from below (h / max(|h|, eps), torch's normalize): a row shorter
    than eps is divided by eps itself, a longer row by its norm; eps is not added to the norm."""
    h = bf16([[0.25, 0.5, 0, 0], [3, 4, 0, 0], [0, 0, 0, 0]])   # norms 0.559, 5, 0
    z = oracle.router_logits(h, _eye(4), norm=oracle.NORM_L2, eps=1.0)
    np.testing.assert_allclose(z, [[0.25, 0.5, 0, 0], [0.6, 0.8, 0, 0], [0, 0, 0, 0]], rtol=1e-7)
    x = torch.nn.functional.normalize(torch.from_numpy(widen(h)).double(), p=2.0, dim=1, eps=1.0)
    np.testing.assert_allclose(z, x.numpy().astype(np.float32), rtol=1e-7)


def test_two_layer_router_identity_is_silu():
    # W1 = W2 = I: z = silu(h); silu(1) = 1 / (1 + e^-1), silu(-1) = -e^-1 / (1 + e^-1)
    z = oracle.router_logits(bf16([[0, 1, -1, 2]]), _eye(4), w2=_eye(4))
    e1 = math.exp(-1.0)
    np.testing.assert_allclose(z[0], [0.0, 1 / (1 + e1), -e1 / (1 + e1), 2 / (1 + math.exp(-2.0))], rtol=1e-7)


def test_two_layer_router_orientation():
    # W1 [H=2, d=3] picks h0 and h2 into the hidden units; W2 [E=2, H=2] swaps them
    w1 = bf16([[1, 0, 0], [0, 0, 1]])
    w2 = bf16([[0, 1], [1, 0]])
    z = oracle.router_logits(bf16([[1, 5, 2]]), w1, w2=w2, bias=[0.25, -0.5])
    silu = lambda u: u / (1 + math.exp(-u))
    np.testing.assert_allclose(z[0], [silu(2.0) + 0.25, silu(1.0) - 0.5], rtol=1e-7)


def test_two_layer_router_reduces_to_torch():
    rng = np.random.default_rng(24)
    T, d, E = 13, 128, 8
    H = 2 * E
    h = bf16(rng.standard_normal((T, d)))
    w1 = bf16(rng.standard_normal((H, d)) * 0.1)
    w2 = bf16(rng.standard_normal((E, H)) * 0.3)
    z = oracle.router_logits(h, w1, w2=w2, norm=oracle.NORM_LAYER, eps=1e-5)
    x = torch.nn.functional.layer_norm(torch.from_numpy(widen(h)).double(), (d,), eps=1e-5)
    a = torch.nn.functional.silu(x @ torch.from_numpy(widen(w1)).double().T)
    want = a @ torch.from_numpy(widen(w2)).double().T
    np.testing.assert_allclose(z, want.numpy().astype(np.float32), rtol=2e-7, atol=1e-7)


def test_temperature_comes_before_the_penalty():
    # z = [1.0, 0.8], usage = [1, 0], lambda = 0.3.  tau = 1: s = [0.7, 0.8], expert 1
    # first; tau = 0.5: s = [2.0 - 0.3, 1.6] = [1.7, 1.6], expert 0 first.  Penalising
    # before dividing would give [1.4, 1.6] and keep expert 1 first.
    z = np.array([[1.0, 0.8]], np.float32)
    u = np.array([1.0, 0.0], np.float32)
    r1 = oracle.route(1, logits_in=z, usage=u, lam=0.3, tau=1.0)
    r2 = oracle.route(1, logits_in=z, usage=u, lam=0.3, tau=0.5)
    assert r1["ids"][0, 0] == 1 and r2["ids"][0, 0] == 0
    pen = np.float32(0.3) * np.float32(1.0)
    assert r2["scores"][0, 0] == np.float32(np.float32(2.0) - pen)
    assert r2["scores"][0, 1] == np.float32(1.6)
    # the logits output is the raw z, not divided
    assert np.array_equal(r2["logits"], z)


def test_temperature_sharpens_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(25)
    z = rng.standard_normal((40, 8)).astype(np.float32)
    for tau in (0.5, 0.7, 2.0):
        r = oracle.route(2, logits_in=z, tau=tau)
        s = (z / np.float32(tau)).astype(np.float32)
        assert np.array_equal(r["scores"], s)
        p = softmax(s.astype(np.float64), axis=1)
        np.testing.assert_allclose(r["topk_p"], np.take_along_axis(p, r["ids"], 1), rtol=1e-6)
        # a positive scale keeps the ranking (no new ties at these values)
        assert np.array_equal(r["ids"], oracle.route(2, logits_in=z)["ids"])
    # a smaller tau gives the top pick more probability
    p5 = oracle.route(1, logits_in=z, tau=0.5)["topk_p"]
    p1 = oracle.route(1, logits_in=z, tau=1.0)["topk_p"]
    assert np.all(p5 >= p1)


@pytest.mark.parametrize("tau", [0.0, -1.0, float("inf"), float("nan")])
def test_temperature_must_be_positive(tau):
    with pytest.raises(oracle.OracleError):
        oracle.route(1, logits_in=np.zeros((2, 3), np.float32), tau=tau)


# --------------------------------------------------------------------------- backward
# The layer's gradients for a fixed dispatch, against torch autograd on a plain
# torch forward (double): the routing decisions are held fixed, the combine
# weights are the renormalised softmax probabilities of the kept experts, and a
# load-balancing term sum_i dP_i * P_i brings in the gradient of an aux loss.

def _torch_backward(h, wr, b, w1, w3, w2, usage, lam, tau, k, C, dout, dP):
    dd = lambda a: torch.from_numpy(np.asarray(a, np.float64)).requires_grad_(True)
    H, WR, B = dd(widen(h)), dd(widen(wr)), dd(b)
    W1, W3, W2 = dd(widen(w1)), dd(widen(w3)), dd(widen(w2))
    z = H @ WR.T + B
    s = z / tau - lam * torch.from_numpy(usage.astype(np.float64))
    s_used = s + (s.detach().float().double() - s.detach())   # the fp32 scores, gradient unchanged
    scores = s_used.detach().float().numpy()
    assign = oracle.dispatch(scores, k, C)["assign"]
    p = torch.softmax(s_used, dim=1)
    T = h.shape[0]
    rows = []
    for t in range(T):
        kept = [int(e) for e in assign[t] if e >= 0]
        acc = torch.zeros(H.shape[1], dtype=torch.float64)
        if kept:
            S = sum(p[t, e] for e in kept)
            for e in kept:
                a = torch.nn.functional.silu(W1[e] @ H[t]) * (W3[e] @ H[t])
                acc = acc + p[t, e] / S * (W2[e] @ a)
        rows.append(acc)
    out = torch.stack(rows)
    L = (out * torch.from_numpy(dout.astype(np.float64))).sum() + (torch.from_numpy(dP.astype(np.float64)) *
                                                                   p.mean(dim=0)).sum()
    grads = torch.autograd.grad(L, [H, WR, B, W1, W3, W2])
    return scores, assign, [g.numpy() for g in grads]


@pytest.mark.parametrize("T,d,E,F,k,C,lam,tau", [(24, 16, 5, 12, 2, 8, 0.3, 0.7),
                                                 (20, 16, 4, 8, 1, 4, 0.0, 1.0),
                                                 (18, 8, 6, 8, 3, 6, 0.5, 2.0),
                                                 (16, 8, 4, 8, 2, 2, 0.0, 0.5)])
def test_backward_matches_torch_autograd(T, d, E, F, k, C, lam, tau):
    tau = float(np.float32(tau))   # the temperature is an fp32 value of the config
    rng = np.random.default_rng(T * 31 + E)
    h = bf16(rng.standard_normal((T, d)))
    wr = bf16(rng.standard_normal((E, d)) * 0.5)
    b = rng.standard_normal(E).astype(np.float32) * 0.1
    w1 = bf16(rng.standard_normal((E, F, d)) / math.sqrt(d))
    w3 = bf16(rng.standard_normal((E, F, d)) / math.sqrt(d))
    w2 = bf16(rng.standard_normal((E, d, F)) / math.sqrt(F))
    usage = rng.random(E).astype(np.float32)
    dout = rng.standard_normal((T, d)).astype(np.float32)
    dP = rng.standard_normal(E).astype(np.float32)
    scores, assign, want = _torch_backward(h, wr, b, w1, w3, w2, usage, lam, tau, k, C, dout, dP)
    # the cases exercise reroutes and drops
    dsp = oracle.dispatch(scores, k, C)
    assert dsp["n_rerouted"] + dsp["n_dropped"] > 0
    g = oracle.layer_backward(h, wr, w1, w3, w2, scores, assign, dout, tau=tau, dP=dP)
    for name, ref in zip(["dh", "dwr", "dbias", "dw1", "dw3", "dw2"], want):
        np.testing.assert_allclose(g[name], ref, rtol=1e-9, atol=1e-12, err_msg=name)


def test_backward_dense_swiglu_is_torch_autograd():
    """E = 1, k = 1, no drops: the combine weight is 1 and the router gets no
    gradient; the expert gradients are those of a dense SwiGLU FFN."""
    rng = np.random.default_rng(40)
    T, d, F = 7, 16, 24
    h = bf16(rng.standard_normal((T, d)))
    wr = bf16(rng.standard_normal((1, d)))
    w1 = bf16(rng.standard_normal((1, F, d)) / 4)
    w3 = bf16(rng.standard_normal((1, F, d)) / 4)
    w2 = bf16(rng.standard_normal((1, d, F)) / 4)
    dout = rng.standard_normal((T, d)).astype(np.float32)
    g = oracle.layer_backward(h, wr, w1, w3, w2, np.zeros((T, 1), np.float32), np.zeros((T, 1), np.int32), dout)
    x = torch.from_numpy(widen(h)).double().requires_grad_(True)
    m1, m3, m2 = (torch.from_numpy(widen(w)[0]).double().requires_grad_(True) for w in (w1, w3, w2))
    y = (torch.nn.functional.silu(x @ m1.T) * (x @ m3.T)) @ m2.T
    gx, g1, g3, g2 = torch.autograd.grad((y * torch.from_numpy(dout).double()).sum(), [x, m1, m3, m2])
    np.testing.assert_allclose(g["dh"], gx.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dw1"][0], g1.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dw3"][0], g3.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dw2"][0], g2.numpy(), rtol=1e-10, atol=1e-12)
    assert np.all(g["dwr"] == 0) and np.all(g["dbias"] == 0)


def test_backward_dropped_token_gets_only_the_aux_gradient():
    # C = 0: every pick is dropped, the output is 0; only dP reaches the router
    rng = np.random.default_rng(41)
    T, d, E, F = 5, 8, 3, 8
    h = bf16(rng.standard_normal((T, d)))
    wr = bf16(rng.standard_normal((E, d)))
    w = bf16(rng.standard_normal((E, F, d)))
    w2 = bf16(rng.standard_normal((E, d, F)))
    s = rng.standard_normal((T, E)).astype(np.float32)
    assign = np.full((T, 2), -1, np.int32)
    dout = rng.standard_normal((T, d)).astype(np.float32)
    g0 = oracle.layer_backward(h, wr, w, w, w2, s, assign, dout)
    assert np.all(g0["dh"] == 0) and np.all(g0["dw1"] == 0) and np.all(g0["dw2"] == 0) and np.all(g0["dwr"] == 0)
    dP = np.array([1.0, -2.0, 0.5], np.float32)
    g1 = oracle.layer_backward(h, wr, w, w, w2, s, assign, dout, dP=dP)
    # dL/dz[t,i] = p_i (dP_i - sum_j p_j dP_j) / T; the bias gradient sums it over t
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    dz = p * (dP - (p * dP).sum(1, keepdims=True)) / T
    np.testing.assert_allclose(g1["dbias"], dz.sum(0), rtol=1e-6)
