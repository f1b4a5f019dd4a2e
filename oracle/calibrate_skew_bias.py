"""Find the router bias beta of the skewed workload with the oracle's router.

The skewed workload adds ``beta`` to expert 0's logit so that expert 0 is the
rank-1 pick (after the load penalty) of about 42% of the tokens.  This script
bisects beta on the seeded hidden states, router weights and usage vector of
that workload, using only the oracle, and prints the value recorded as
``SKEW_BETA`` in ``token_level_top_gb300/synth.py``.

Run:  python -m oracle.calibrate_skew_bias
"""
from __future__ import annotations

import numpy as np

import oracle
from token_level_top_gb300 import synth

TARGET = 0.42


def share_for(beta, h, wr, usage, lam, E):
    bias = np.zeros(E, np.float32)
    bias[0] = beta
    r = oracle.route(2, h=h, wr=wr, bias=bias, usage=usage, lam=lam)
    return float((r["ids"][:, 0] == 0).mean())


def main():
    shape = synth.with_shape(synth.CONFIGS["skewed"], skew_beta=0.0)
    h, wr, _, usage = synth.router_inputs(shape)
    hb, wb = synth.bf16_bits(h), synth.bf16_bits(wr)
    u = usage.numpy()
    # Bisection on the unbiased logits plus the bias (cheap), then one check
    # through the oracle's router with the bias argument.
    base = oracle.route(2, h=hb, wr=wb, usage=None, lam=0.0)["logits"]
    lo, hi = 0.0, 8.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        z = base.copy()
        z[:, 0] += np.float32(mid)
        r = oracle.route(2, logits_in=z, usage=u, lam=shape.lam)
        share = float((r["ids"][:, 0] == 0).mean())
        if share < TARGET:
            lo = mid
        else:
            hi = mid
    beta = float(np.float32(hi))
    share = share_for(beta, hb, wb, u, shape.lam, shape.E)
    print(f"SKEW_BETA = {beta!r}  # expert-0 rank-1 share {share:.4f}")


if __name__ == "__main__":
    main()
