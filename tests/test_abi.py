"""The C-ABI library without a GPU: it loads, exports every function that
include/moe.h declares, and its host-side logic (capacity, workspace sizing,
synchronous argument checks) behaves as documented.  No call here reaches a
kernel: every case returns before anything is enqueued."""
import ctypes
import math

import numpy as np
import pytest

import oracle
from token_level_top_gb300 import build, moe, synth


@pytest.fixture(scope="module")
def L():
    build.build()
    return moe.lib()


def test_exports_every_declared_symbol(L):
    names = moe.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), f"libmoe.so does not export {n}"
    assert set(names) == set(moe._SIGS), "binding signatures out of sync with include/moe.h"


def test_capacity_matches_oracle(L):
    rng = np.random.default_rng(0)
    for _ in range(500):
        T = int(rng.integers(1, 100000))
        k = int(rng.integers(1, 9))
        E = int(rng.integers(1, 256))
        cf = float(np.round(rng.uniform(0.1, 4.0), int(rng.integers(0, 7))))
        if cf <= 0:
            continue
        assert L.moe_capacity(T, k, E, cf, 0) == oracle.capacity(T, k, E, cf)
    for shape in synth.CONFIGS.values():
        assert L.moe_capacity(shape.T, shape.k, shape.E, shape.cf, 0) == math.ceil(
            round(shape.T * shape.k * shape.cf / shape.E, 9))
    assert L.moe_capacity(32, 2, 64, 1.3, 0) == 2
    assert L.moe_capacity(100, 2, 26, 1.3, 0) == 10
    assert L.moe_capacity(100, 2, 26, 1.3, 7) == 7
    assert L.moe_capacity(0, 2, 8, 1.0, 0) == 0


def _cfg(**kw):
    d = dict(T=256, d_model=512, E=8, k=2, d_ff=1024, cf=1.25, capacity=0, lam=0.0)
    d.update(kw)
    return moe.Config(**d).c()


def test_workspace_size(L):
    sizes = []
    for shape in synth.CONFIGS.values():
        c = moe.Config.of(shape).c()
        n = L.moe_workspace_size(ctypes.byref(c))
        assert n > 0 and n % 256 == 0
        sizes.append(n)
    assert sizes[1] > sizes[0]
    for bad in [dict(E=256), dict(k=9), dict(k=3, E=2), dict(d_model=100), dict(d_ff=200),
                dict(cf=0.0), dict(T=-1)]:
        c = _cfg(**bad)
        assert L.moe_workspace_size(ctypes.byref(c)) == 0, bad
    c = _cfg()
    c.flags = 8   # not a defined flag
    assert L.moe_workspace_size(ctypes.byref(c)) == 0
    # MOE_FLAG_FP8 adds the e4m3 activation rows and the row scales
    c = _cfg()
    base = L.moe_workspace_size(ctypes.byref(c))
    c.flags = moe.FLAG_FP8
    grown = L.moe_workspace_size(ctypes.byref(c))
    assert grown >= base + c.T * c.k * (c.d_ff + 8)
    # MOE_FLAG_BACKWARD adds the per-expert row blocks (each expert's kept rows rounded up
    # to 128, at most E x C' rows) and the forward's g and u
    c.flags = moe.FLAG_BACKWARD
    cap = moe.capacity(c.T, c.k, c.E, c.cf)
    rows = min(c.E * ((min(cap, c.T) + 127) // 128 * 128), c.T * c.k + 127 * c.E)
    assert L.moe_workspace_size(ctypes.byref(c)) >= base + rows * (8 * c.d_model + 10 * c.d_ff) + \
        c.T * c.k * 8 * c.d_ff
    # MOE_FLAG_NVFP4 adds the 4-bit token and activation rows with their scales
    c.flags = moe.FLAG_NVFP4
    assert L.moe_workspace_size(ctypes.byref(c)) >= base + c.T * c.k * (c.d_model // 2 + c.d_ff // 2 + 12)


FAKE = 0x7f0000000000  # never dereferenced: every case below fails validation first


def test_route_argument_checks(L):
    c = _cfg()
    ws_n = L.moe_workspace_size(ctypes.byref(c))
    P = ctypes.c_void_p
    args = lambda **o: [ctypes.byref(o.get("cfg", c)), P(o.get("h", FAKE)), P(o.get("wr", FAKE)),
                        None, None, None, None, None, P(o.get("ids", FAKE)), None, None, None, None,
                        P(o.get("ws", FAKE)), o.get("n", ws_n), None]
    assert L.moe_route(*args(ids=None)) == 1
    assert L.moe_route(*args(h=None)) == 1
    assert L.moe_route(*args(h=FAKE + 8)) == 3
    assert L.moe_route(*args(ws=FAKE + 128)) == 3
    assert L.moe_route(*args(ws=None)) == 1
    assert L.moe_route(*args(n=ws_n - 1)) == 4
    assert L.moe_route(*args(cfg=_cfg(E=300))) == 2
    assert L.moe_route(None, *args()[1:]) == 1


def test_layer_forward_argument_checks(L):
    c = _cfg()
    n = L.moe_workspace_size(ctypes.byref(c))
    P = ctypes.c_void_p
    base = [P(FAKE)] * 2 + [None, None] + [P(FAKE)] * 3 + [None] * 8
    call = lambda cfg, ptrs, ws=FAKE, nb=n: L.moe_layer_forward(ctypes.byref(cfg), *ptrs, P(ws), nb,
                                                                None)
    assert call(c, base, nb=n - 256) == 4
    bad = list(base)
    bad[5] = P(FAKE + 2)                       # w2 misaligned
    assert call(c, bad) == 3
    bad = list(base)
    bad[6] = None                              # out missing
    assert call(c, bad) == 1
    assert call(_cfg(d_ff=192), base) == 2     # d_ff % 128 != 0
    assert call(_cfg(k=0), base) == 1


def test_dispatch_and_ffn_argument_checks(L):
    c = _cfg()
    n = L.moe_workspace_size(ctypes.byref(c))
    P = ctypes.c_void_p
    outs = [P(FAKE)] * 9    # assign, slot, flags, counts, offsets, perm, cw, n_rerouted, n_dropped
    assert L.moe_dispatch(ctypes.byref(c), None, *outs, P(FAKE), n, None) == 1
    assert L.moe_dispatch(ctypes.byref(c), P(FAKE), *outs[:-1], None, P(FAKE), n, None) == 1
    assert L.moe_expert_ffn(ctypes.byref(c), P(FAKE + 4), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                            P(FAKE), P(FAKE), n, None) == 3
    assert L.moe_combine(ctypes.byref(c), None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                         None) == 1
    assert L.moe_pack_w13(8, 100, 512, P(FAKE), P(FAKE), P(FAKE), None) == 2
    assert L.moe_pack_w13(8, 128, 512, P(FAKE), P(FAKE + 1), P(FAKE), None) == 3
    assert L.moe_debug_timeout_probe(P(FAKE), 256, 0, None) == 1
    assert L.moe_workspace_init(P(FAKE + 64), 4096, None) == 3


def test_status_strings(L):
    for code, text in moe.STATUS.items():
        assert L.moe_status_string(code).decode() == text


def test_router_variant_config_checks(L):
    for bad in [dict(tau=-1.0), dict(tau=float("inf")), dict(tau=float("nan")), dict(router_norm=3),
                dict(norm_eps=-1.0), dict(router_hidden=-1), dict(router_hidden=257),
                dict(E=128, router_hidden=256)]:
        c = _cfg(**bad)
        assert L.moe_workspace_size(ctypes.byref(c)) == 0, bad
    base = L.moe_workspace_size(ctypes.byref(_cfg()))
    # tau alone needs no room; the normalised rows and the hidden router add theirs
    assert L.moe_workspace_size(ctypes.byref(_cfg(tau=0.7))) == base
    assert L.moe_workspace_size(ctypes.byref(_cfg(router_norm=1))) > base
    assert L.moe_workspace_size(ctypes.byref(_cfg(router_hidden=16))) > base


def test_router_variant_argument_checks(L):
    P = ctypes.c_void_p
    c = _cfg(router_hidden=16, router_norm=1)
    n = L.moe_workspace_size(ctypes.byref(c))
    r = moe.MoERouter(FAKE, FAKE, None, None, None)
    call = lambda cfg, rt, nb=n, h=FAKE: L.moe_router_logits(ctypes.byref(cfg), P(h), ctypes.byref(rt),
                                                             P(FAKE), P(FAKE), nb, None)
    assert call(c, r, nb=n - 256) == 4
    assert call(c, moe.MoERouter(FAKE, None, None, None, None)) == 1   # the hidden router needs W2
    assert call(_cfg(), moe.MoERouter(FAKE, FAKE, None, None, None)) == 1   # W2 without a hidden width
    assert call(_cfg(), moe.MoERouter(FAKE, None, None, FAKE, None)) == 1   # gamma without LayerNorm
    assert call(c, moe.MoERouter(FAKE, FAKE + 2, None, None, None)) == 3
    assert call(c, r, h=FAKE + 4) == 3
    assert L.moe_router_logits(ctypes.byref(c), P(FAKE), None, P(FAKE), P(FAKE), n, None) == 1
    # the plain entry points do not take these routers' weights
    ids = P(FAKE)
    assert L.moe_route(ctypes.byref(c), P(FAKE), P(FAKE), None, None, None, None, None, ids, None, None,
                       None, None, P(FAKE), n, None) == 1
    base = [P(FAKE)] * 2 + [None, None] + [P(FAKE)] * 3 + [None] * 8
    assert L.moe_layer_forward(ctypes.byref(c), *base, P(FAKE), n, None) == 1
    # layer with the router struct: scales must come in pairs
    lf = lambda s13, s2: L.moe_layer_forward_router(ctypes.byref(c), P(FAKE), ctypes.byref(r), None, P(FAKE),
                                                    s13, P(FAKE), s2, P(FAKE), *([None] * 8), P(FAKE), n, None)
    assert lf(P(FAKE), None) == 1


def test_backward_argument_checks(L):
    P = ctypes.c_void_p
    c = _cfg(flags=moe.FLAG_BACKWARD)
    n = L.moe_workspace_size(ctypes.byref(c))
    ptrs = lambda **o: [P(o.get(k, FAKE)) if o.get(k, FAKE) is not None else None
                        for k in ("h", "wr", "w13", "w2", "dout")] + [None] + \
        [P(o.get(k, FAKE)) if o.get(k, FAKE) is not None else None for k in ("dh", "dwr", "db", "dw13", "dw2")]
    call = lambda cfg, nb=n, **o: L.moe_layer_backward(ctypes.byref(cfg), *ptrs(**o), P(FAKE), nb, None)
    assert call(_cfg()) == 1                       # workspace not sized for the backward
    assert call(c, dout=None) == 1
    assert call(c, dw2=None) == 1
    assert call(c, dh=FAKE + 4) == 3
    assert call(c, nb=n - 256) == 4
    assert call(_cfg(flags=moe.FLAG_BACKWARD, router_hidden=16)) == 2


def test_quantiser_argument_checks(L):
    P = ctypes.c_void_p
    f = P(FAKE)
    # e4m3: cols a multiple of 8, rows >= 0; w 16-byte and q 8-byte aligned
    assert L.moe_quantize_fp8(-1, 64, f, f, f, None) == 1
    assert L.moe_quantize_fp8(10, 60, f, f, f, None) == 1
    assert L.moe_quantize_fp8(0, 64, None, None, None, None) == 0     # nothing to do, nothing enqueued
    assert L.moe_quantize_fp8(10, 64, None, f, f, None) == 1
    assert L.moe_quantize_fp8(10, 64, P(FAKE + 8), f, f, None) == 3
    assert L.moe_quantize_fp8(10, 64, f, P(FAKE + 4), f, None) == 3
    # NVFP4: cols a multiple of 32 and at most 16384; codes and block scales 16-byte aligned
    assert [L.moe_nvfp4_sf_stride(c) for c in (0, 16, 32, 1408, 4096, 14336)] == [0, 16, 16, 96, 256, 896]
    assert L.moe_quantize_nvfp4(10, 48, f, f, f, f, None) == 1
    assert L.moe_quantize_nvfp4(10, 16416, f, f, f, f, None) == 2
    assert L.moe_quantize_nvfp4(0, 64, None, None, None, None, None) == 0
    assert L.moe_quantize_nvfp4(10, 64, f, P(FAKE + 8), f, f, None) == 3
    assert L.moe_quantize_nvfp4(10, 64, f, f, P(FAKE + 8), f, None) == 3
    assert L.moe_quantize_w13_nvfp4(8, 192, 512, f, f, f, f, None) == 1    # d_ff % 128
    assert L.moe_quantize_w13_nvfp4(8, 256, 16416, f, f, f, f, None) == 2  # d > 16384
    assert L.moe_quantize_w13_nvfp4(8, 256, 512, f, f, None, f, None) == 1
    assert L.moe_quantize_w13_nvfp4(8, 256, 512, P(FAKE + 2), f, f, f, None) == 3


def test_quantised_expert_argument_checks(L):
    P = ctypes.c_void_p
    f = P(FAKE)
    plain = _cfg()
    fp8 = _cfg(flags=moe.FLAG_FP8)
    fp4 = _cfg(flags=moe.FLAG_NVFP4)
    n8 = L.moe_workspace_size(ctypes.byref(fp8))
    n4 = L.moe_workspace_size(ctypes.byref(fp4))
    assert n8 > L.moe_workspace_size(ctypes.byref(plain)) and n4 > 0
    # expert FFN: the scales are required; the workspace must be sized for the format
    assert L.moe_expert_ffn_fp8(ctypes.byref(fp8), f, f, f, f, None, f, f, f, f, n8, None) == 1
    assert L.moe_expert_ffn_fp8(ctypes.byref(plain), f, f, f, f, f, f, f, f, f, n8, None) == 1
    assert L.moe_expert_ffn_fp8(ctypes.byref(_cfg(d_model=192, flags=moe.FLAG_FP8)), f, f, f, f, f, f, f, f, f,
                                n8, None) == 2                                       # d % 128
    assert L.moe_expert_ffn_nvfp4(ctypes.byref(fp4), f, f, f, f, None, f, f, f, f, f, f, n4, None) == 1
    assert L.moe_expert_ffn_nvfp4(ctypes.byref(plain), f, f, f, f, f, f, f, f, f, f, f, n4, None) == 1
    assert L.moe_expert_ffn_nvfp4(ctypes.byref(fp4), f, f, f, f, P(FAKE + 8), f, f, f, f, f, f, n4,
                                  None) == 3
    assert L.moe_expert_ffn_nvfp4(ctypes.byref(fp4), f, f, f, f, f, f, f, f, f, f, f, n4 - 256, None) == 4
    # the layer: h, wr, bias, usage, w13 (codes, block scales, row scales), w2 (same), out, 8 optional
    # outputs and the stage events, then the workspace
    lay4 = lambda cfg, n=n4, **o: L.moe_layer_forward_nvfp4(
        ctypes.byref(cfg), f, f, None, None, f, o.get("b13", f), f, f, f, f, o.get("out", f),
        *([None] * 8), f, n, None)
    assert lay4(plain) == 1
    assert lay4(_cfg(d_model=192, flags=moe.FLAG_NVFP4)) == 2
    assert lay4(fp4, b13=P(FAKE + 8)) == 3
    assert lay4(fp4, out=None) == 1
    assert lay4(fp4, n=n4 - 256) == 4
    assert lay4(_cfg(flags=moe.FLAG_NVFP4, router_norm=1)) == 1
    lay8 = lambda cfg, n=n8, s13=f: L.moe_layer_forward_fp8(ctypes.byref(cfg), f, f, None, None, f, s13, f, f,
                                                           f, *([None] * 8), f, n, None)
    assert lay8(plain) == 1
    assert lay8(_cfg(d_model=192, flags=moe.FLAG_FP8)) == 2
    assert lay8(fp8, n=n8 - 256) == 4


def test_backward_static_and_host_argument_checks(L):
    P = ctypes.c_void_p
    f = P(FAKE)
    bw = _cfg(flags=moe.FLAG_BACKWARD)
    nb = L.moe_workspace_size(ctypes.byref(bw))
    # backward: h, wr, w13, w2, dout, dP, dh, dwr, dbias, dw13, dw2, then the workspace
    back = lambda cfg, n=nb, h=f, dw13=f: L.moe_layer_backward(ctypes.byref(cfg), h, f, f, f, f, None, f, None,
                                                               None, dw13, f, f, n, None)
    assert back(_cfg()) == 1                                   # the config lacks MOE_FLAG_BACKWARD
    assert back(_cfg(flags=moe.FLAG_BACKWARD, router_norm=1)) == 2
    assert back(bw, dw13=None) == 1
    assert back(bw, h=P(FAKE + 8)) == 3
    assert back(bw, n=nb - 256) == 4
    # allocation-free dispatch: scores, assign, slot, flags, counts, offsets, perm, cw, totals, status
    st = lambda cfg, scores=f, counts=f: L.moe_dispatch_static(ctypes.byref(cfg), scores, f, f, f, counts, f, f,
                                                               f, f, f, None, None)
    assert st(_cfg(flags=moe.FLAG_FP8)) == 1
    assert st(_cfg(E=300)) == 2
    assert st(_cfg(E=20, k=9)) == 2
    assert st(_cfg(), counts=None) == 1
    assert st(_cfg(), scores=None) == 1
    assert st(_cfg(T=200000, E=64)) == 2                       # scratch beyond the fixed array
    # host buffers: h_host, wr, bias, usage, w13, w2, out_host, then the workspace
    c = _cfg()
    n = L.moe_workspace_size(ctypes.byref(c))
    host = lambda cfg, h=f, out=f, ws=FAKE, nbytes=n: L.moe_layer_forward_host_async(
        ctypes.byref(cfg), h, f, None, None, f, f, out, P(ws), nbytes, None)
    assert host(c, h=None) == 1
    assert host(c, out=None) == 1
    assert host(c, ws=FAKE + 64) == 3
    assert host(c, nbytes=n - 256) == 4
    assert host(_cfg(k=0)) == 1
    assert L.moe_layer_forward_host(ctypes.byref(c), None, f, None, None, f, f, f, f, n, None) == 1
