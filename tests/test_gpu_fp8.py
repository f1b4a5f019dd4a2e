"""GPU parity of the FP8 (e4m3) expert path against the CPU oracle.

The quantiser is compared bit for bit with torch's e4m3 conversion of the same
fp32 quotients.  The expert FFN and the whole layer (e4m3 weights with row
scales, token and activation rows quantised per row on the fly, e4m3 MMAs)
are compared with the oracle run the same way in double precision: decoded
weights, token rows and activation rows (the latter rounded to bf16 first).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (OUT_REL_FROB, assert_dispatch_equal, assert_rows_close, bits, make_layer, np_, rel_frob,
                     sample_tokens, tile_tokens)
from token_level_top_gb300.moe import MoEError
from token_level_top_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def unpack_w13(q13, s13, F):
    """The packed W13 layout (256-row blocks: 128 W1 rows, then the 128 matching
    W3 rows) back to W1 and W3, for codes [E, 2F, d] and scales [E*2F]."""
    E, _, d = q13.shape
    q = q13.reshape(E, F // 128, 2, 128, d)
    s = s13.reshape(E, F // 128, 2, 128)
    return (q[:, :, 0].reshape(E, F, d), s[:, :, 0].reshape(E, F),
            q[:, :, 1].reshape(E, F, d), s[:, :, 1].reshape(E, F))


def quantized(Ld, shape):
    q13, s13 = moe.quantize_fp8(Ld["w13"])
    q2, s2 = moe.quantize_fp8(Ld["w2"])
    q1, s1, q3, s3 = unpack_w13(np_(q13), np_(s13), shape.F)
    ora = dict(q1=q1, s1=s1, q3=q3, s3=s3, q2=np_(q2), s2=np_(s2).reshape(shape.E, shape.d))
    return (q13, s13), (q2, s2), ora


@pytest.mark.parametrize("rows,cols", [(7, 64), (300, 512), (1000, 4096), (3000, 512), (50, 6144),
                                       (20, 8192), (33, 14336), (3, 65664)])
def test_quantize_fp8_matches_torch(rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    w = (torch.randn(rows, cols, generator=g) * torch.rand(rows, 1, generator=g) * 3).to(torch.bfloat16)
    w[1] = 0   # an all-zero row: scale 1, codes 0
    q, s = moe.quantize_fp8(w.cuda())
    wf = w.float()
    amax = wf.abs().amax(dim=1)
    s_ref = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    assert torch.equal(s.cpu(), s_ref)
    q_ref = (wf / s_ref[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(q.cpu(), q_ref)


def test_quantize_fp8_every_bf16_value():
    """Each row holds every finite bf16 value of magnitude at most its maximum
    (both signs; the rest zeros), at scales where some quotients land within a
    few fp32 ulps of an e4m3 rounding midpoint: the codes must still be those
    of the correctly rounded quotient."""
    pos = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    amaxes = [1.0, 3.0, 0.1, 100.5, 7e-3, 448.0, 1e-30, 2.5e5, 0.3, 1e-38]
    cols = 40960
    w = torch.zeros(len(amaxes), cols, dtype=torch.bfloat16)
    for i, a in enumerate(amaxes):
        a = torch.tensor(a).to(torch.bfloat16).float().item()
        x = pos[pos <= a]
        row = torch.from_numpy(np.concatenate([x, -x])).to(torch.bfloat16)
        w[i, :row.numel()] = row
    q, s = moe.quantize_fp8(w.cuda())
    wf = w.float()
    amax = wf.abs().amax(dim=1)
    s_ref = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    assert torch.equal(s.cpu(), s_ref)
    q_ref = (wf / s_ref[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(q.cpu(), q_ref)


@pytest.mark.parametrize("T,d,E,F,k,cf", [(300, 256, 5, 256, 2, 1.0), (256, 512, 8, 1024, 2, 1.25),
                                          (64, 1024, 8, 2048, 2, 1.25), (700, 128, 3, 256, 2, 1.0),
                                          (1100, 256, 2, 384, 2, 1.0)])
def test_expert_ffn_fp8_vs_oracle(T, d, E, F, k, cf):
    shape = synth.MoEShape("t", T=T, d=d, E=E, F=F, k=k, cf=cf, seed=T + F)
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_FP8)
    ws = moe.workspace(cfg)
    s = np.random.default_rng(T).standard_normal((T, E)).astype(np.float32)
    dsp = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    w13, w2, o = quantized(Ld, shape)
    y = moe.expert_ffn(cfg, ws, Ld["h"], dsp["perm"], dsp["offsets"], w13, w2)
    assert moe.device_status(ws) == 0
    n = int(np_(dsp["offsets"])[-1])
    want = oracle.expert_slots_q8(bits(Ld["h"]), o["q1"], o["s1"], o["q3"], o["s3"], o["q2"], o["s2"],
                                  np_(dsp["assign"]), np_(dsp["perm"])[:n], 0, n)
    got = np_(y[:n].float())
    assert rel_frob(got, want) <= OUT_REL_FROB
    rows = np.linalg.norm(got - want, axis=1) / np.maximum(np.linalg.norm(want, axis=1), 1e-12)
    assert rows.max() <= 4 * OUT_REL_FROB


SAMPLE = {"tiny": 256, "mixtral_decode": 64, "mixtral_prefill": 32}   # >= T: every token


@pytest.mark.parametrize("name", ["tiny", "mixtral_decode", "mixtral_prefill"])
def test_layer_forward_fp8_workloads(name):
    shape = synth.CONFIGS[name]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_FP8)
    ws = moe.workspace(cfg)
    w13, w2, o = quantized(Ld, shape)
    out, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], w13, w2, bias=Ld["bias"],
                                 usage=Ld["usage"], aux=True)
    assert moe.device_status(ws) == 0
    C = oracle.capacity(shape.T, shape.k, shape.E, shape.cf, shape.capacity)
    o_r = oracle.route(shape.k, logits_in=np_(aux["logits"]))
    o_d = oracle.dispatch(o_r["scores"], shape.k, C)
    assert_dispatch_equal(aux, o_d, shape.T, shape.k)
    # sampled tokens, and one in every (expert, 128-row tile) of the expert GEMMs
    must = tile_tokens(o_d["perm"], o_d["offsets"], shape.k, shape.seed)
    toks = (np.arange(shape.T, dtype=np.int32) if SAMPLE[name] >= shape.T
            else sample_tokens(shape.T, SAMPLE[name], shape.seed, must=must))
    want = oracle.combine_rows_q8(bits(Ld["h"]), o["q1"], o["s1"], o["q3"], o["s3"], o["q2"], o["s2"],
                                  o_d["assign"], o_d["cw"], toks)
    got = np_(out.float())[toks]
    assert_rows_close(got, want)


@pytest.mark.parametrize("T,E,k,cap", [(1, 8, 2, 0), (64, 1, 1, 0), (257, 4, 2, 30), (200, 40, 2, 2),
                                       (1200, 16, 4, 0)])
def test_layer_forward_fp8_edge_shapes(T, E, k, cap):
    """One token, one expert, forced small capacities with drops, k = 4: every token's row
    against the oracle (all-dropped tokens give zero rows)."""
    shape = synth.MoEShape("edge", T=T, d=128, E=E, F=256, k=k, cf=1.0, capacity=cap, seed=T + E)
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_FP8)
    ws = moe.workspace(cfg)
    w13, w2, o = quantized(Ld, shape)
    out, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], w13, w2, aux=True)
    assert moe.device_status(ws) == 0
    C = oracle.capacity(T, k, E, 1.0, cap)
    o_d = oracle.dispatch(oracle.route(k, logits_in=np_(aux["logits"]))["scores"], k, C)
    assert_dispatch_equal(aux, o_d, T, k)
    want = oracle.combine_rows_q8(bits(Ld["h"]), o["q1"], o["s1"], o["q3"], o["s3"], o["q2"], o["s2"],
                                  o_d["assign"], o_d["cw"], np.arange(T, dtype=np.int32))
    assert_rows_close(np_(out.float()), want)


def test_layer_forward_fp8_deterministic():
    shape = synth.CONFIGS["tiny"]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_FP8)
    ws = moe.workspace(cfg)
    w13, w2, _ = quantized(Ld, shape)
    a = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], w13, w2)
    b = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], w13, w2)
    assert torch.equal(a, b)


def test_fp8_entry_checks():
    shape = synth.MoEShape("t", T=64, d=192, E=4, F=256, k=2, cf=1.0, seed=3)
    Ld = make_layer(shape)
    w13, w2 = moe.quantize_fp8(Ld["w13"]), moe.quantize_fp8(Ld["w2"])
    plain = moe.Config.of(shape)   # workspace without the FP8 regions
    with pytest.raises(MoEError) as ex:
        moe.layer_forward(plain, moe.workspace(plain), Ld["h"], Ld["wr"], w13, w2)
    assert ex.value.status == 1   # MOE_ERR_INVALID_ARG
    cfg = moe.Config.of(shape, flags=moe.FLAG_FP8)   # d = 192 is not a multiple of 128
    with pytest.raises(MoEError) as ex:
        moe.layer_forward(cfg, moe.workspace(cfg), Ld["h"], Ld["wr"], w13, w2)
    assert ex.value.status == 2   # MOE_ERR_UNSUPPORTED
