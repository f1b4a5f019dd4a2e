"""The capacity replay's fixed-point rounds, modelled on the CPU (no GPU).

The dispatch kernel replays the entries that follow the first capacity overflow
in windows of consecutive entries of one rank.  Each expert has a fill position
in the window (the entry that takes its last slot; -1 when it was full before the
window, none when it does not fill).  In a round every entry picks its expert with
the experts whose fill position lies before it counted as full; the slots follow
from the counts in window order and give new fill positions; rounds repeat until
the positions reproduce themselves.  This model takes the same steps in plain
Python and checks, on random and adversarial batches, that

* the fixed point is the sequential fill of "GPT-4稀疏激活真相" §2.3 (third
  check) -- the oracle's dispatch, bit for bit in assign and slot;
* a window takes at most one round per fill in it plus one, never more than the
  E + 1 rounds after which the kernel stops with a timeout status.

Neither the argument nor the bound depends on the window length, so short
windows (more windows, more fills per window relative to its length) are
checked beside the kernel's 256.
"""
import numpy as np
import pytest

import oracle

NONE = 1 << 30   # "does not fill in this window"


def _choose(pref_row, start, held, fpos, i):
    """The expert entry i of the window picks: the first one of its preference order,
    from its rank's position on, that is not held by its token and not full at i."""
    for e in pref_row[start:]:
        if e in held:
            continue
        if fpos[e] < i:      # -1 (full before the window) or filled earlier in it
            continue
        return int(e)
    return -1


def replay(scores, k, C, W):
    """Rank-major, window-by-window fixed-point replay; returns assign, slot and
    the (rounds, fills) of every window."""
    T, E = scores.shape
    pref = np.array([oracle.preference(scores[t]) for t in range(T)])
    assign = np.full((T, k), -1, np.int64)
    slot = np.full((T, k), -1, np.int64)
    fill = np.zeros(E, np.int64)
    stats = []
    for r in range(k):
        for w0 in range(0, T, W):
            toks = range(w0, min(T, w0 + W))
            held = [set(int(x) for x in assign[t, :r]) for t in toks]
            fpos = np.where(fill >= C, -1, NONE)
            rounds = 0
            while True:
                rounds += 1
                choice = [_choose(pref[t], r, held[i], fpos, i) for i, t in enumerate(toks)]
                count = fill.copy()
                slots = []
                nxt = np.where(fill >= C, -1, NONE)
                for i, e in enumerate(choice):
                    if e < 0:
                        slots.append(-1)
                        continue
                    slots.append(int(count[e]))
                    count[e] += 1
                    if count[e] == C:
                        nxt[e] = i
                if np.array_equal(nxt, fpos):
                    break
                assert rounds <= E + 1, "the kernel would stop here with a timeout status"
                fpos = nxt
            fills = int(((fpos >= 0) & (fpos < NONE)).sum())
            assert rounds <= fills + 1, (rounds, fills)
            stats.append((rounds, fills))
            for i, t in enumerate(toks):
                assign[t, r] = choice[i]
                slot[t, r] = slots[i]
            for e in choice:
                if e >= 0:
                    fill[e] += 1
    return assign, slot, stats


def _cases():
    rng = np.random.default_rng(11)
    out = []
    for i in range(60):
        T = int(rng.integers(1, 700))
        E = int(rng.integers(2, 40))
        k = int(rng.integers(1, min(E, 4) + 1))
        cf = float(rng.choice([0.3, 0.6, 1.0, 1.25]))
        s = rng.standard_normal((T, E)).astype(np.float32)
        s[:, : max(1, E // 4)] += float(rng.uniform(0, 3))     # skew toward a few experts
        if T > 40 and i % 3 == 0:
            s[T // 4: T // 4 + 40] = s[T // 4]                     # a run of identical tokens
        out.append((f"rand{i}", s, k, oracle.capacity(T, k, E, cf)))
    # every expert fills inside one window: E fills, E + 1 rounds at most
    s = np.tile(np.arange(16, dtype=np.float32)[::-1], (200, 1))
    out.append(("all-fill-one-window", s, 2, 3))
    # capacity 1: every pick of a new expert is a fill
    out.append(("capacity-1", rng.standard_normal((300, 12)).astype(np.float32), 3, 1))
    # scores in reverse preference per token half: fills cascade through the order
    s = rng.standard_normal((256, 24)).astype(np.float32)
    s[:128] = np.sort(s[:128], 1)
    s[128:] = np.sort(s[128:], 1)[:, ::-1]
    out.append(("cascade", s, 2, 5))
    return out


CASES = _cases()


@pytest.mark.parametrize("W", [256, 32])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fixed_point_is_the_sequential_fill(case, W):
    name, s, k, C = case
    assign, slot, stats = replay(s, k, C, W)
    o = oracle.dispatch(s, k, C)
    assert np.array_equal(assign, o["assign"]) and np.array_equal(slot, o["slot"])


def test_rounds_reach_the_bound_without_passing_it():
    """A window where every one of E experts fills in turn needs E + 1 rounds in this
    order of events, the most the kernel allows; the model reaches it exactly."""
    E = 16
    s = np.tile(np.arange(E, dtype=np.float32)[::-1], (E * 3, 1))   # everyone prefers 0, 1, 2, ...
    assign, slot, stats = replay(s, 1, 3, 256)
    rounds, fills = stats[0]
    assert fills == E and rounds == E + 1
    assert np.array_equal(assign, oracle.dispatch(s, 1, 3)["assign"])
