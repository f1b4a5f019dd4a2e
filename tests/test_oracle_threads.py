"""The oracle's per-row functions give the same bits whether their rows run on one
thread or are split over several (each part is a call of the same C function on
its own rows).  CPU only."""
import numpy as np
import pytest

import oracle
from test_oracle_pins import _q4_weights, bf16


@pytest.fixture
def threads():
    saved = oracle.THREADS

    def run(n, fn, *a, **kw):
        oracle.THREADS = n
        try:
            return fn(*a, **kw)
        finally:
            oracle.THREADS = saved
    return run


def _case(seed, T=37, d=32, F=48, E=4, k=2):
    rng = np.random.default_rng(seed)
    h = bf16(rng.standard_normal((T, d)))
    w1, w3 = (bf16(rng.standard_normal((E, F, d)) / 6) for _ in range(2))
    w2 = bf16(rng.standard_normal((E, d, F)) / 7)
    s = rng.standard_normal((T, E)).astype(np.float32)
    dsp = oracle.dispatch(s, k, oracle.capacity(T, k, E, 1.0))
    return rng, h, w1, w3, w2, dsp


@pytest.mark.parametrize("n", [2, 3, 8, 64])
def test_bf16_rows_and_slots_do_not_depend_on_threads(threads, n):
    rng, h, w1, w3, w2, dsp = _case(1)
    toks = np.array([5, 0, 36, 7, 7, 19, 2, 30, 11], np.int32)
    one = threads(1, oracle.combine_rows, h, w1, w3, w2, dsp["assign"], dsp["cw"], toks)
    many = threads(n, oracle.combine_rows, h, w1, w3, w2, dsp["assign"], dsp["cw"], toks)
    assert np.array_equal(one, many)
    m = len(dsp["perm"])
    one = threads(1, oracle.expert_slots, h, w1, w3, w2, dsp["assign"], dsp["perm"], 3, m - 2)
    many = threads(n, oracle.expert_slots, h, w1, w3, w2, dsp["assign"], dsp["perm"], 3, m - 2)
    assert one.shape == (m - 5, h.shape[1]) and np.array_equal(one, many)


def test_quantised_rows_do_not_depend_on_threads(threads):
    rng, h, w1, w3, w2, dsp = _case(2)
    toks = np.arange(37, dtype=np.int32)
    E, F, d = w1.shape

    def q8(w):
        rows = w.reshape(-1, w.shape[-1]).view(np.uint16).astype(np.uint32) << 16
        x = rows.view(np.float32)
        codes, scales = zip(*(oracle.quantize_row(r) for r in x))
        return np.array(codes, np.uint8).reshape(w.shape), np.array(scales, np.float32).reshape(w.shape[:-1])
    (q1, s1), (q3, s3), (q2, s2) = q8(w1), q8(w3), q8(w2)
    args = (h, q1, s1, q3, s3, q2, s2, dsp["assign"], dsp["cw"], toks)
    assert np.array_equal(threads(1, oracle.combine_rows_q8, *args), threads(5, oracle.combine_rows_q8, *args))
    m = len(dsp["perm"])
    args = (h, q1, s1, q3, s3, q2, s2, dsp["assign"], dsp["perm"], 1, m)
    assert np.array_equal(threads(1, oracle.expert_slots_q8, *args), threads(3, oracle.expert_slots_q8, *args))
    a1, _ = _q4_weights(rng, E, F, d, exact=False)
    a3, _ = _q4_weights(rng, E, F, d, exact=False)
    a2, _ = _q4_weights(rng, E, d, F, exact=False)
    args = (h, a1, a3, a2, dsp["assign"], dsp["cw"], toks)
    assert np.array_equal(threads(1, oracle.combine_rows_q4, *args), threads(6, oracle.combine_rows_q4, *args))
    args = (h, a1, a3, a2, dsp["assign"], dsp["perm"], 0, m)
    assert np.array_equal(threads(1, oracle.expert_slots_q4, *args), threads(4, oracle.expert_slots_q4, *args))


def test_empty_token_list(threads):
    rng, h, w1, w3, w2, dsp = _case(3)
    out = threads(8, oracle.combine_rows, h, w1, w3, w2, dsp["assign"], dsp["cw"], np.zeros(0, np.int32))
    assert out.shape == (0, h.shape[1])
