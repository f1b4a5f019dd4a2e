"""GPU parity of the router variants against the CPU oracle.

Temperature ("MoE稀疏激活原理…" §3.1 step 3; 2kiu page §2): scores, picks and
dispatch bit-exact on shared logits.  Normalisation before the router (2kiu
page §5.2) and the two-layer router silu(x W1) W2 ("MoE稀疏激活原理…" §3.1
step 2): logits within a bound that follows from the arithmetic -- the GPU
rounds the normalised rows to bf16 for the router GEMM (relative error at
most 2^-9 per element), so |dz_e| <= 2^-9 * sum_i |x_i W_ei| plus fp32
accumulation error; the two-layer router carries that through silu (slope
at most 1.1) and W2.  The tests allow twice that.  Routing on the GPU's own
logits is bit-exact, and the layer output is within the layer tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (OUT_REL_FROB, WEIGHT_RTOL, assert_dispatch_equal, bits, make_layer, np_, rel_frob,
                     sample_tokens)
from token_level_top_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def router_weights(d, E, H, norm, seed, bias=True):
    return synth.router_variant_weights(d, E, H, norm == moe.NORM_LAYER, seed, bias)


def to_router(rw):
    return moe.Router(**{k: (None if v is None else v.cuda()) for k, v in rw.items()})


def oracle_logits(h, rw, norm, eps):
    return oracle.router_logits(bits(h), bits(rw["w"]), w2=None if rw["w2"] is None else bits(rw["w2"]),
                                bias=None if rw["bias"] is None else rw["bias"].numpy(),
                                gamma=None if rw["gamma"] is None else rw["gamma"].numpy(),
                                beta=None if rw["beta"] is None else rw["beta"].numpy(), norm=norm, eps=eps)


def logit_bound(h, rw, norm, eps):
    """Twice the first-order error bound of rounding the normalised rows to bf16
    (plus a small fp32 floor)."""
    x = h.double()
    if norm == moe.NORM_LAYER:
        x = torch.nn.functional.layer_norm(x, (x.shape[1],), rw["gamma"].double(), rw["beta"].double(), eps)
    elif norm == moe.NORM_L2:
        x = torch.nn.functional.normalize(x, p=2.0, dim=1, eps=eps)
    w = rw["w"].double()
    mag = x.abs() @ w.abs().T                  # sum_i |x_i W_ei| (or W1_ji)
    if rw["w2"] is None:
        return 2 * (2.0 ** -9 * mag + 1e-5 * mag) + 1e-5
    du = 2.0 ** -9 * mag + 1e-5 * mag
    u = x @ w.T
    a = torch.nn.functional.silu(u)
    w2 = rw["w2"].double().abs()
    return 2 * (1.1 * du @ w2.T + 1e-5 * (a.abs() @ w2.T)) + 1e-5


CASES = [  # T, d, E, H, norm
    (300, 512, 8, 0, moe.NORM_LAYER),
    (300, 512, 8, 16, moe.NORM_NONE),
    (1000, 1024, 64, 128, moe.NORM_LAYER),
    (257, 256, 16, 32, moe.NORM_L2),
    (64, 4096, 8, 16, moe.NORM_LAYER),
    (129, 2048, 32, 0, moe.NORM_L2),
    (40, 128, 4, 1, moe.NORM_NONE),
    (600, 16384, 8, 16, moe.NORM_LAYER),
]


@pytest.mark.parametrize("T,d,E,H,norm", CASES)
def test_router_logits_vs_oracle(T, d, E, H, norm):
    eps = 1e-5 if norm == moe.NORM_LAYER else 1e-12
    g = torch.Generator().manual_seed(T + d)
    h = (torch.randn(T, d, generator=g) * 2 + 0.5).to(torch.bfloat16)
    h[min(3, T - 1)] *= 40   # a row of unusually large norm, the case the page normalises for
    rw = router_weights(d, E, H, norm, seed=T * 7 + E)
    cfg = moe.Config(T=T, d_model=d, E=E, k=2, d_ff=0, router_norm=norm, norm_eps=eps, router_hidden=H)
    ws = moe.workspace(cfg)
    z = moe.router_logits(cfg, ws, h.cuda(), to_router(rw))
    assert moe.device_status(ws) == 0
    want = oracle_logits(h, rw, norm, eps)
    err = np.abs(np_(z).astype(np.float64) - want)
    bound = logit_bound(h.float(), rw, norm, eps).numpy()
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"


def test_linear_router_logits_equal_route_logits():
    """router_logits without a front end sums the GEMM's split partials exactly
    as the route step does."""
    T, d, E = 1000, 2048, 16
    g = torch.Generator().manual_seed(5)
    h = torch.randn(T, d, generator=g).to(torch.bfloat16).cuda()
    rw = router_weights(d, E, 0, moe.NORM_NONE, seed=6)
    cfg = moe.Config(T=T, d_model=d, E=E, k=2, d_ff=0)
    ws = moe.workspace(cfg)
    z = moe.router_logits(cfg, ws, h, to_router(rw))
    r = moe.route(cfg, ws, h=h, wr=rw["w"].cuda(), bias=rw["bias"].cuda())
    assert torch.equal(z, r["logits"])


def test_l2_zero_row_gives_bias():
    T, d, E = 8, 256, 8
    h = torch.zeros(T, d, dtype=torch.bfloat16)
    h[1, 5] = 3.0
    rw = router_weights(d, E, 0, moe.NORM_L2, seed=7)
    cfg = moe.Config(T=T, d_model=d, E=E, k=2, d_ff=0, router_norm=moe.NORM_L2, norm_eps=1e-12)
    ws = moe.workspace(cfg)
    z = np_(moe.router_logits(cfg, ws, h.cuda(), to_router(rw)))
    assert np.array_equal(z[0], rw["bias"].numpy())
    # the one nonzero row normalises to the unit vector e_5
    np.testing.assert_allclose(z[1], rw["w"].float().numpy()[:, 5] + rw["bias"].numpy(), rtol=1e-6)


@pytest.mark.parametrize("T,E,k,lam,tau", [(1000, 8, 2, 0.0, 0.5), (1000, 8, 2, 0.8, 0.7),
                                            (3000, 64, 2, 0.3, 1.3), (77, 16, 4, 0.5, 0.1),
                                            (500, 8, 1, 0.8, 3.0)])
def test_temperature_route_shared_logits(T, E, k, lam, tau):
    rng = np.random.default_rng(T + E)
    z = rng.standard_normal((T, E)).astype(np.float32)
    usage = rng.random(E).astype(np.float32)
    cfg = moe.Config(T=T, d_model=64, E=E, k=k, d_ff=0, lam=lam, tau=tau)
    ws = moe.workspace(cfg)
    g = moe.route(cfg, ws, logits_in=torch.from_numpy(z).cuda(), usage=torch.from_numpy(usage).cuda())
    assert moe.device_status(ws) == 0
    o = oracle.route(k, logits_in=z, usage=usage, lam=lam, tau=tau)
    assert np.array_equal(np_(g["scores"]), o["scores"])
    assert np.array_equal(np_(g["ids"]), o["ids"])
    assert np.array_equal(np_(g["counts_pre"]), o["counts_pre"])
    np.testing.assert_allclose(np_(g["topk_w"]), o["topk_p"], rtol=WEIGHT_RTOL, atol=1e-7)
    np.testing.assert_allclose(np_(g["P"]), o["P"], rtol=WEIGHT_RTOL, atol=1e-7)


VARIANTS = [  # name, tau, norm, hidden (0 = linear, -1 = 2E)
    ("tau", 0.7, moe.NORM_NONE, 0),
    ("layernorm", 1.0, moe.NORM_LAYER, 0),
    ("l2", 0.5, moe.NORM_L2, 0),
    ("two_layer", 1.0, moe.NORM_NONE, -1),
    ("layernorm_two_layer_tau", 0.7, moe.NORM_LAYER, -1),
]


@pytest.mark.parametrize("variant", VARIANTS, ids=[v[0] for v in VARIANTS])
@pytest.mark.parametrize("name", ["tiny", "mixtral_decode", "skewed"])
def test_layer_forward_router_variants(name, variant):
    _, tau, norm, hidden = variant
    shape = synth.CONFIGS[name]
    H = 2 * shape.E if hidden < 0 else hidden
    eps = 1e-5 if norm == moe.NORM_LAYER else 1e-12
    Ld = make_layer(shape)
    rw = router_weights(shape.d, shape.E, H, norm, seed=shape.seed + 11)
    cfg = moe.Config.of(shape, tau=tau, router_norm=norm, norm_eps=eps, router_hidden=H)
    ws = moe.workspace(cfg)
    out, aux = moe.layer_forward(cfg, ws, Ld["h"], to_router(rw), Ld["w13"], Ld["w2"], usage=Ld["usage"],
                                 aux=True)
    assert moe.device_status(ws) == 0
    h_cpu = Ld["h"].cpu()
    gl = np_(aux["logits"])
    # (1) the logits within the rounding bound
    err = np.abs(gl.astype(np.float64) - oracle_logits(h_cpu, rw, norm, eps))
    assert np.all(err <= logit_bound(h_cpu.float(), rw, norm, eps).numpy())
    # (2) on the GPU's logits, routing and dispatch are the oracle's, bit for bit
    unp = None if Ld["usage"] is None else np_(Ld["usage"])
    o_r = oracle.route(shape.k, logits_in=gl, usage=unp, lam=shape.lam, tau=tau)
    C = oracle.capacity(shape.T, shape.k, shape.E, shape.cf, shape.capacity)
    o_d = oracle.dispatch(o_r["scores"], shape.k, C)
    assert_dispatch_equal(aux, o_d, shape.T, shape.k)
    np.testing.assert_allclose(np_(aux["P"]), o_r["P"], rtol=WEIGHT_RTOL, atol=1e-7)
    # (3) the output on sampled tokens
    toks = sample_tokens(shape.T, min(shape.T, 24), shape.seed)
    want = oracle.combine_rows(bits(Ld["h"]), bits(Ld["w1"]), bits(Ld["w3"]), bits(Ld["w2"]), o_d["assign"],
                               o_d["cw"], toks)
    assert rel_frob(np_(out.float())[toks], want) <= OUT_REL_FROB


def test_layer_forward_router_fp8_experts():
    from test_gpu_fp8 import quantized
    shape = synth.CONFIGS["tiny"]
    Ld = make_layer(shape)
    rw = router_weights(shape.d, shape.E, 2 * shape.E, moe.NORM_LAYER, seed=3)
    cfg = moe.Config.of(shape, tau=0.7, router_norm=moe.NORM_LAYER, router_hidden=2 * shape.E,
                        flags=moe.FLAG_FP8)
    ws = moe.workspace(cfg)
    w13, w2, o = quantized(Ld, shape)
    out, aux = moe.layer_forward(cfg, ws, Ld["h"], to_router(rw), w13, w2, aux=True)
    assert moe.device_status(ws) == 0
    # the router and the dispatch are those of the bf16 layer with the same router
    cfg16 = moe.Config.of(shape, tau=0.7, router_norm=moe.NORM_LAYER, router_hidden=2 * shape.E)
    _, aux16 = moe.layer_forward(cfg16, moe.workspace(cfg16), Ld["h"], to_router(rw), Ld["w13"], Ld["w2"],
                                 aux=True)
    assert torch.equal(aux["logits"], aux16["logits"])
    assert torch.equal(aux["assign"], aux16["assign"])
    # the output is the e4m3 layer's on that dispatch
    o_r = oracle.route(shape.k, logits_in=np_(aux["logits"]), tau=0.7)
    C = oracle.capacity(shape.T, shape.k, shape.E, shape.cf, shape.capacity)
    o_d = oracle.dispatch(o_r["scores"], shape.k, C)
    assert_dispatch_equal(aux, o_d, shape.T, shape.k)
    toks = np.arange(shape.T, dtype=np.int32)
    want = oracle.combine_rows_q8(bits(Ld["h"]), o["q1"], o["s1"], o["q3"], o["s3"], o["q2"], o["s2"],
                                  o_d["assign"], o_d["cw"], toks)
    assert rel_frob(np_(out.float()), want) <= OUT_REL_FROB


def test_layer_forward_temperature_one_is_the_plain_layer():
    shape = synth.CONFIGS["tiny"]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape)
    a = moe.layer_forward(cfg, moe.workspace(cfg), Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], bias=Ld["bias"])
    cfg1 = moe.Config.of(shape, tau=1.0)
    b = moe.layer_forward(cfg1, moe.workspace(cfg1), Ld["h"], moe.Router(w=Ld["wr"], bias=Ld["bias"]),
                          Ld["w13"], Ld["w2"])
    assert torch.equal(a, b)
