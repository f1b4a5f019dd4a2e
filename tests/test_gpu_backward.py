"""GPU parity of the layer's backward pass (moe_layer_backward) against the oracle.

The oracle takes the forward's penalised scores (re-derived from the GPU's logits, bit-exact)
and its assignment, and computes every gradient in double.  The GPU keeps the gathered rows and
the operands of the weight and input gradients in bf16 (x, dL/dout, cw*a, dg, du) with fp32
accumulation, so those gradients agree within the layer's 2e-2 relative Frobenius bound.  The
router's gradients depend on differences dcw_r - sum_r' cw_r' dcw_r' of dot products that can
cancel, so their inputs stay fp32 (the forward's g and u, W2^T dL/dout): they agree to 1e-3.

At the benchmark sizes, dL/dout is zero outside a sample of tokens (and there is no
load-balancing term): every gradient then comes from the sampled tokens alone, so the oracle run
on those tokens gives all of them exactly -- the weight gradients included.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import OUT_REL_FROB, bits, make_layer, np_, rel_frob, sample_tokens
from token_level_top_gb300 import moe, synth

pytestmark = pytest.mark.gpu

GRAD_REL_FROB = OUT_REL_FROB
ROUTER_REL_FROB = 1e-3


def unpack13(dw13, F):
    E, _, d = dw13.shape
    q = dw13.reshape(E, F // 128, 2, 128, d)
    return q[:, :, 0].reshape(E, F, d), q[:, :, 1].reshape(E, F, d)


def run(shape, dout, dP=None, usage_on=True):
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_BACKWARD)
    ws = moe.workspace(cfg)
    usage = Ld["usage"] if usage_on else None
    _, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], bias=Ld["bias"], usage=usage,
                               aux=True)
    g = moe.layer_backward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], dout.cuda(),
                           dP=None if dP is None else torch.from_numpy(dP).cuda())
    assert moe.device_status(ws) == 0
    unp = None if usage is None else np_(usage)
    o_r = oracle.route(shape.k, logits_in=np_(aux["logits"]), usage=unp, lam=shape.lam, tau=cfg.tau)
    return Ld, aux, g, o_r["scores"]


def check(Ld, shape, aux, g, scores, dout, dP, toks=None):
    assign = np_(aux["assign"])
    h = bits(Ld["h"])
    d32 = dout.float().numpy()
    if toks is not None:
        h, scores, assign, d32 = h[toks], scores[toks], assign[toks], d32[toks]
    want = oracle.layer_backward(h, bits(Ld["wr"]), bits(Ld["w1"]), bits(Ld["w3"]), bits(Ld["w2"]), scores,
                                 assign, d32, dP=dP)
    dh = np_(g["dh"])
    if toks is not None:
        rest = np.setdiff1d(np.arange(shape.T), toks)
        assert np.all(dh[rest] == 0), "tokens with dL/dout = 0 get no gradient"
        dh = dh[toks]
    assert rel_frob(dh, want["dh"]) <= GRAD_REL_FROB
    dw1, dw3 = unpack13(np_(g["dw13"]), shape.F)
    assert rel_frob(dw1, want["dw1"]) <= GRAD_REL_FROB
    assert rel_frob(dw3, want["dw3"]) <= GRAD_REL_FROB
    assert rel_frob(np_(g["dw2"]), want["dw2"]) <= GRAD_REL_FROB
    assert rel_frob(np_(g["dwr"]), want["dwr"]) <= ROUTER_REL_FROB
    assert rel_frob(np_(g["dbias"]), want["dbias"]) <= ROUTER_REL_FROB


SMALL = [  # T, d, E, F, k, cf, lam, tau
    (300, 256, 5, 256, 2, 1.0, 0.3, 0.7),
    (256, 512, 8, 1024, 2, 1.25, 0.0, 1.0),
    (200, 128, 4, 384, 1, 1.0, 0.0, 1.0),
    (150, 256, 6, 256, 3, 0.8, 0.5, 2.0),
    (77, 192, 3, 128, 2, 0.5, 0.0, 0.5),
]


@pytest.mark.parametrize("T,d,E,F,k,cf,lam,tau", SMALL)
def test_layer_backward_vs_oracle(T, d, E, F, k, cf, lam, tau):
    shape = synth.MoEShape("t", T=T, d=d, E=E, F=F, k=k, cf=cf, lam=lam, seed=T + d)
    gen = torch.Generator().manual_seed(T * 3 + F)
    dout = torch.randn(T, d, generator=gen).to(torch.bfloat16)
    dP = np.random.default_rng(T).standard_normal(E).astype(np.float32)
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_BACKWARD, tau=tau)
    ws = moe.workspace(cfg)
    usage = torch.from_numpy(np.random.default_rng(E).random(E).astype(np.float32)).cuda()
    _, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], usage=usage, aux=True)
    g = moe.layer_backward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], dout.cuda(), dP=torch.from_numpy(dP).cuda())
    assert moe.device_status(ws) == 0
    scores = oracle.route(k, logits_in=np_(aux["logits"]), usage=np_(usage), lam=lam, tau=tau)["scores"]
    C = oracle.capacity(T, k, E, cf)
    o_d = oracle.dispatch(scores, k, C)
    assert np.array_equal(np_(aux["assign"]), o_d["assign"])
    want = oracle.layer_backward(bits(Ld["h"]), bits(Ld["wr"]), bits(Ld["w1"]), bits(Ld["w3"]), bits(Ld["w2"]),
                                 scores, o_d["assign"], dout.float().numpy(), tau=tau, dP=dP)
    assert rel_frob(np_(g["dh"]), want["dh"]) <= GRAD_REL_FROB
    dw1, dw3 = unpack13(np_(g["dw13"]), F)
    assert rel_frob(dw1, want["dw1"]) <= GRAD_REL_FROB
    assert rel_frob(dw3, want["dw3"]) <= GRAD_REL_FROB
    assert rel_frob(np_(g["dw2"]), want["dw2"]) <= GRAD_REL_FROB
    assert rel_frob(np_(g["dwr"]), want["dwr"]) <= ROUTER_REL_FROB
    assert rel_frob(np_(g["dbias"]), want["dbias"]) <= ROUTER_REL_FROB


@pytest.mark.parametrize("name", ["mixtral_decode", "mixtral_prefill", "fine_grained"])
def test_layer_backward_full_size_sampled_tokens(name):
    shape = synth.CONFIGS[name]
    toks = sample_tokens(shape.T, 4, shape.seed)[:6]
    gen = torch.Generator().manual_seed(shape.seed + 5)
    dout = torch.zeros(shape.T, shape.d, dtype=torch.bfloat16)
    dout[toks] = torch.randn(len(toks), shape.d, generator=gen).to(torch.bfloat16)
    Ld, aux, g, scores = run(shape, dout)
    check(Ld, shape, aux, g, scores, dout, None, toks=toks)


def test_layer_backward_all_dropped_gets_only_the_aux_gradient():
    shape = synth.MoEShape("t", T=64, d=128, E=4, F=128, k=2, cf=1.0, capacity=0, seed=9)
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_BACKWARD, capacity=0, cf=0.01)   # C = 1
    ws = moe.workspace(cfg)
    _, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], aux=True)
    dout = torch.randn(shape.T, shape.d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    dP = np.array([1.0, -1.0, 0.5, 0.0], np.float32)
    g = moe.layer_backward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], dout.cuda(), dP=torch.from_numpy(dP).cuda())
    scores = oracle.route(2, logits_in=np_(aux["logits"]))["scores"]
    want = oracle.layer_backward(bits(Ld["h"]), bits(Ld["wr"]), bits(Ld["w1"]), bits(Ld["w3"]), bits(Ld["w2"]),
                                 scores, np_(aux["assign"]), dout.float().numpy(), dP=dP)
    assert (np_(aux["assign"]) >= 0).sum() == 4   # one slot per expert
    assert rel_frob(np_(g["dh"]), want["dh"]) <= GRAD_REL_FROB
    assert rel_frob(np_(g["dwr"]), want["dwr"]) <= ROUTER_REL_FROB


def test_layer_backward_deterministic_and_empty():
    shape = synth.CONFIGS["tiny"]
    dout = torch.randn(shape.T, shape.d, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_BACKWARD)
    ws = moe.workspace(cfg)
    moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], bias=Ld["bias"])
    a = moe.layer_backward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], dout.cuda())
    b = moe.layer_backward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], dout.cuda())
    for n in a:
        assert torch.equal(a[n], b[n]), n
    empty = moe.Config.of(synth.with_shape(shape, T=0), flags=moe.FLAG_BACKWARD)
    e = moe.layer_backward(empty, moe.workspace(empty), Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], dout.cuda())
    assert float(e["dw13"].abs().max()) == 0 and float(e["dw2"].abs().max()) == 0
