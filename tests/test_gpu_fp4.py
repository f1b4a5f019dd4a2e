"""GPU parity of the NVFP4 expert path (4-bit weights and activations) against the oracle.

The quantiser is compared bit for bit with the oracle's (codes, e4m3 block scales and
fp32 row scales of every row), including the 128-row packing of W13.  The expert FFN and
the layer (e2m1 codes with block scales on tcgen05.mma.kind::mxf4nvf4, token and activation
rows quantised on the fly) are compared with the oracle run the same way in double
precision on the GPU's quantised weights.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (assert_dispatch_equal, assert_rows_close, bits, make_layer, np_, sample_tokens,
                     tile_tokens)
from token_level_top_gb300.moe import MoEError
from token_level_top_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def oracle_rows(w):
    """The oracle's NVFP4 quantisation of every row of a bf16 tensor [rows, cols]."""
    x = w.float().cpu().numpy()
    out = [oracle.quantize_row_nvfp4(r) for r in x]
    return (np.stack([o[0] for o in out]), np.stack([o[1] for o in out]),
            np.array([o[2] for o in out], np.float32))


def assert_quantised_equal(got, want, cols):
    q, b, s = (np_(t) for t in got)
    wq, wb, ws = want
    rows = wq.shape[0]
    q, b, s = q.reshape(rows, -1), b.reshape(rows, -1), s.reshape(rows)
    assert np.array_equal(s, ws)
    assert np.array_equal(b[:, : cols // 16], wb)
    assert np.array_equal(q, wq)


@pytest.mark.parametrize("rows,cols", [(7, 64), (64, 512), (40, 1408), (16, 4096), (6, 14336), (3, 16384)])
def test_quantize_nvfp4_matches_oracle(rows, cols):
    g = torch.Generator().manual_seed(rows * 7 + cols)
    w = torch.randn(rows, cols, generator=g) * torch.rand(rows, 1, generator=g) * 3
    w[0] = 0                                   # an all-zero row: scale 1, codes 0
    if rows > 2:
        w[1, : cols // 2] *= 1e-4              # blocks far below the row's largest value
        w[2, 16:32] = 0                        # an all-zero block
    if rows > 4:
        w[3] *= 1e-30                          # block divisors below 2^-92: the plain-division path
        w[4, : cols // 2] *= 1e-36             # blocks in bf16's subnormal range beside normal ones
    w = w.to(torch.bfloat16)
    got = moe.quantize_nvfp4(w.cuda())
    assert_quantised_equal(got, oracle_rows(w), cols)


def _bf16_step(x, n):
    """x (bf16-exact float32 values) moved by n bf16 steps away from zero."""
    b = torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16)
    n = torch.from_numpy(np.broadcast_to(np.asarray(n, np.int16), b.shape).copy())
    return (b + n).view(torch.bfloat16).float().numpy()


def test_quantize_nvfp4_rounding_boundaries():
    """Elements exactly on each e2m1 rounding boundary of their block (x / den = 0.25,
    0.75, ..., 5, where the tie goes to the even code) and one bf16 step either side,
    for divisors den = m 2^n with m = 1.75, 1.25, 1.125: 1 / den is inexact, so the
    quotient must be rounded exactly as the oracle's IEEE division rounds it."""
    rng = np.random.default_rng(11)
    ts = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    rows = []
    for k in (-7, 0, 5):                      # row scale 2^k: the row max is 2688 2^k
        for m in (1.75, 1.25, 1.125):
            for j in (-3, 0, 2):              # block scale m 2^j, divisor den = m 2^(j+k)
                den = np.float32(m * 2.0 ** (j + k))
                row = np.zeros(128, np.float32)
                row[0] = 2688 * 2.0 ** k
                for blk in range(1, 8):
                    cand = ts * den
                    pick = rng.integers(0, 7, 15)
                    vals = _bf16_step(cand[pick], rng.integers(-1, 2, 15)) * rng.choice([-1, 1], 15)
                    row[16 * blk] = 6 * den  # the block max: block scale e4m3(m 2^j), exact
                    row[16 * blk + 1: 16 * blk + 16] = vals
                rows.append(row)
    w = torch.from_numpy(np.stack(rows)).to(torch.bfloat16)
    assert torch.equal(w.float(), torch.from_numpy(np.stack(rows)))   # every value bf16-exact
    assert_quantised_equal(moe.quantize_nvfp4(w.cuda()), oracle_rows(w), 128)


def unpack13(q13, b13, s13, F, d):
    """The 4-bit path's W13 packing (128-row blocks: 64 W1 rows, then the matching 64 W3
    rows) back to W1 and W3: codes [E, 2F, d/2], block scales [E, 2F, stride], scales [E*2F]."""
    E = q13.shape[0]
    q = q13.reshape(E, F // 64, 2, 64, d // 2)
    b = b13[:, :, : d // 16].reshape(E, F // 64, 2, 64, d // 16)
    s = s13.reshape(E, F // 64, 2, 64)
    w1 = (q[:, :, 0].reshape(E, F, d // 2), b[:, :, 0].reshape(E, F, d // 16), s[:, :, 0].reshape(E, F))
    w3 = (q[:, :, 1].reshape(E, F, d // 2), b[:, :, 1].reshape(E, F, d // 16), s[:, :, 1].reshape(E, F))
    return w1, w3


def quantized(Ld, shape):
    q13 = moe.quantize_w13_nvfp4(Ld["w13"])
    q2 = moe.quantize_nvfp4(Ld["w2"])
    F, d, E = shape.F, shape.d, shape.E
    w1, w3 = unpack13(*(np_(t) for t in q13), F, d)
    w2 = (np_(q2[0]), np_(q2[1])[:, :, : F // 16], np_(q2[2]).reshape(E, d))
    return q13, q2, (w1, w3, w2)


def test_quantize_w13_nvfp4_packing():
    """Row r of the packed output is the oracle's quantisation of the W1 or W3 row that the
    128-row packing puts there (W1 row 64j + i at 128j + i, W3 row 64j + i at 128j + 64 + i)."""
    shape = synth.MoEShape("t", T=64, d=256, E=3, F=384, k=2, cf=1.0, seed=5)
    Ld = make_layer(shape)
    q13 = moe.quantize_w13_nvfp4(Ld["w13"])
    E, F, d = shape.E, shape.F, shape.d
    w1, w3 = Ld["w1"].cpu(), Ld["w3"].cpu()
    src = torch.empty(E, 2 * F, d, dtype=torch.bfloat16)
    for j in range(F // 64):
        src[:, 128 * j: 128 * j + 64] = w1[:, 64 * j: 64 * j + 64]
        src[:, 128 * j + 64: 128 * j + 128] = w3[:, 64 * j: 64 * j + 64]
    assert_quantised_equal(q13, oracle_rows(src.reshape(E * 2 * F, d)), d)


@pytest.mark.parametrize("T,d,E,F,k,cf", [(300, 256, 5, 256, 2, 1.0), (256, 512, 8, 1024, 2, 1.25),
                                          (64, 1024, 8, 2048, 2, 1.25), (700, 128, 3, 256, 2, 1.0),
                                          (1100, 256, 2, 384, 2, 1.0), (500, 256, 6, 1408, 2, 1.0),
                                          (600, 384, 3, 256, 2, 1.0)])
def test_expert_ffn_nvfp4_vs_oracle(T, d, E, F, k, cf):
    shape = synth.MoEShape("t", T=T, d=d, E=E, F=F, k=k, cf=cf, seed=T + F)
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_NVFP4)
    ws = moe.workspace(cfg)
    s = np.random.default_rng(T).standard_normal((T, E)).astype(np.float32)
    dsp = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    q13, q2, (w1, w3, w2) = quantized(Ld, shape)
    y = moe.expert_ffn(cfg, ws, Ld["h"], dsp["perm"], dsp["offsets"], q13, q2)
    assert moe.device_status(ws) == 0
    n = int(np_(dsp["offsets"])[-1])
    want = oracle.expert_slots_q4(bits(Ld["h"]), w1, w3, w2, np_(dsp["assign"]), np_(dsp["perm"])[:n], 0, n)
    assert_rows_close(np_(y[:n].float()), want)


SAMPLE = {"tiny": 256, "mixtral_decode": 64, "mixtral_prefill": 32}   # >= T: every token


@pytest.mark.parametrize("name", ["tiny", "mixtral_decode", "mixtral_prefill"])
def test_layer_forward_nvfp4_workloads(name):
    shape = synth.CONFIGS[name]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_NVFP4)
    ws = moe.workspace(cfg)
    q13, q2, (w1, w3, w2) = quantized(Ld, shape)
    out, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], q13, q2, bias=Ld["bias"], usage=Ld["usage"],
                                 aux=True)
    assert moe.device_status(ws) == 0
    C = oracle.capacity(shape.T, shape.k, shape.E, shape.cf, shape.capacity)
    o_r = oracle.route(shape.k, logits_in=np_(aux["logits"]))
    o_d = oracle.dispatch(o_r["scores"], shape.k, C)
    assert_dispatch_equal(aux, o_d, shape.T, shape.k)
    # sampled tokens, and one in every (expert, 128-row tile) of the expert GEMMs
    must = tile_tokens(o_d["perm"], o_d["offsets"], shape.k, shape.seed)
    toks = (np.arange(shape.T, dtype=np.int32) if SAMPLE[name] >= shape.T
            else sample_tokens(shape.T, SAMPLE[name], shape.seed, must=must))
    want = oracle.combine_rows_q4(bits(Ld["h"]), w1, w3, w2, o_d["assign"], o_d["cw"], toks)
    assert_rows_close(np_(out.float())[toks], want)


@pytest.mark.parametrize("T,E,k,cap", [(1, 8, 2, 0), (64, 1, 1, 0), (257, 4, 2, 30), (200, 40, 2, 2),
                                       (1200, 16, 4, 0)])
def test_layer_forward_nvfp4_edge_shapes(T, E, k, cap):
    """One token, one expert, forced small capacities with drops, k = 4: every token's row
    against the oracle (all-dropped tokens give zero rows)."""
    shape = synth.MoEShape("edge", T=T, d=128, E=E, F=256, k=k, cf=1.0, capacity=cap, seed=T + E)
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_NVFP4)
    ws = moe.workspace(cfg)
    q13, q2, (w1, w3, w2) = quantized(Ld, shape)
    out, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], q13, q2, aux=True)
    assert moe.device_status(ws) == 0
    C = oracle.capacity(T, k, E, 1.0, cap)
    o_d = oracle.dispatch(oracle.route(k, logits_in=np_(aux["logits"]))["scores"], k, C)
    assert_dispatch_equal(aux, o_d, T, k)
    want = oracle.combine_rows_q4(bits(Ld["h"]), w1, w3, w2, o_d["assign"], o_d["cw"], np.arange(T, dtype=np.int32))
    assert_rows_close(np_(out.float()), want)


def test_layer_forward_nvfp4_deterministic():
    shape = synth.CONFIGS["tiny"]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_NVFP4)
    ws = moe.workspace(cfg)
    q13, q2, _ = quantized(Ld, shape)
    a = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], q13, q2)
    b = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], q13, q2)
    assert torch.equal(a, b)


def test_nvfp4_entry_checks():
    shape = synth.MoEShape("t", T=64, d=192, E=4, F=256, k=2, cf=1.0, seed=3)
    Ld = make_layer(shape)
    q13, q2 = moe.quantize_w13_nvfp4(Ld["w13"]), moe.quantize_nvfp4(Ld["w2"])
    plain = moe.Config.of(shape)   # workspace without the NVFP4 regions
    with pytest.raises(MoEError) as ex:
        moe.layer_forward(plain, moe.workspace(plain), Ld["h"], Ld["wr"], q13, q2)
    assert ex.value.status == 1   # MOE_ERR_INVALID_ARG
    cfg = moe.Config.of(shape, flags=moe.FLAG_NVFP4)   # d = 192 is not a multiple of 128
    with pytest.raises(MoEError) as ex:
        moe.layer_forward(cfg, moe.workspace(cfg), Ld["h"], Ld["wr"], q13, q2)
    assert ex.value.status == 2   # MOE_ERR_UNSUPPORTED
