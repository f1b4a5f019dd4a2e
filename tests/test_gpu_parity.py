"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Routing and dispatch are compared bit for bit when both sides get the same
fp32 logits/scores; floating-point outputs within the tolerances in
helpers.py.  Small cases span several tiles and chunks with ragged tails; the
five workloads run at full size in the launch configuration the benchmark
uses, with the expert FFN compared on sampled token rows."""
import numpy as np
import pytest
import torch

import oracle
from helpers import (LOGIT_MAX_ABS, MARGIN, OUT_REL_FROB, WEIGHT_RTOL, assert_dispatch_equal,
                     assert_rows_close, bits, make_layer, np_, rel_frob, sample_tokens, tile_tokens,
                     topk_margin)
from token_level_top_gb300 import build, moe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    moe.lib()
    yield
    torch.cuda.synchronize()


def _cfg(T, E, k, d=64, F=128, cf=1.0, cap=0, lam=0.0):
    return moe.Config(T=T, d_model=d, E=E, k=k, d_ff=F, cf=cf, capacity=cap, lam=lam)


def _scores(kind, T, E, seed):
    rng = np.random.default_rng(seed)
    if kind == "gauss":
        return (rng.standard_normal((T, E)) * 1.3).astype(np.float32)
    if kind == "ties":
        s = rng.integers(-2, 3, (T, E)).astype(np.float32)
        s[rng.random((T, E)) < 0.1] = -0.0
        return s
    if kind == "skew":
        s = rng.standard_normal((T, E)).astype(np.float32)
        s[:, 0] += 1.5
        s[:, 1] += 0.7
        return s
    if kind == "identical":
        return np.tile(np.arange(E, 0, -1, dtype=np.float32), (T, 1))
    if kind == "runs":
        s = rng.standard_normal((T, E)).astype(np.float32)
        for b in range(0, T, 512):
            s[b:b + 128] = s[b]
        return s
    raise ValueError(kind)


# ----------------------------------------------------------------------------- routing

@pytest.mark.parametrize("T,E,k,lam,kind", [
    (300, 8, 2, 0.0, "gauss"), (777, 64, 2, 0.8, "gauss"), (513, 16, 2, 0.0, "ties"),
    (200, 5, 3, 0.3, "ties"), (64, 200, 1, 0.0, "gauss"), (1, 8, 2, 0.0, "gauss"),
    (1030, 33, 8, 0.5, "gauss"), (100, 1, 1, 0.0, "gauss")])
def test_route_shared_logits(T, E, k, lam, kind):
    z = _scores(kind, T, E, T + E)
    usage = np.random.default_rng(E).random(E).astype(np.float32) if lam else None
    cfg = _cfg(T, E, k, lam=lam)
    ws = moe.workspace(cfg)
    g = moe.route(cfg, ws, logits_in=torch.from_numpy(z).cuda(),
                  usage=None if usage is None else torch.from_numpy(usage).cuda())
    assert moe.device_status(ws) == 0
    o = oracle.route(k, logits_in=z, usage=usage, lam=lam)
    assert np.array_equal(np_(g["logits"]), o["logits"])
    assert np.array_equal(np_(g["scores"]), o["scores"])          # fp32 penalty, no FMA
    assert np.array_equal(np_(g["ids"]), o["ids"])
    assert np.array_equal(np_(g["counts_pre"]), o["counts_pre"])
    np.testing.assert_allclose(np_(g["topk_w"]), o["topk_p"], rtol=WEIGHT_RTOL, atol=1e-7)
    np.testing.assert_allclose(np_(g["P"]), o["P"], rtol=WEIGHT_RTOL, atol=1e-7)
    np.testing.assert_allclose(np_(g["f"]), o["f"], rtol=1e-7)


def test_route_nan_sets_status():
    z = _scores("gauss", 50, 8, 1)
    z[7, 3] = np.nan
    cfg = _cfg(50, 8, 2)
    ws = moe.workspace(cfg)
    g = moe.route(cfg, ws, logits_in=torch.from_numpy(z).cuda())
    assert moe.device_status(ws) == 5
    assert moe.device_status(ws) == 0                 # read clears
    assert 3 not in np_(g["ids"])[7].tolist()          # NaN ranks last


@pytest.mark.parametrize("T,d,E", [(300, 192, 10), (129, 64, 8), (1000, 1024, 64), (5, 128, 3)])
def test_router_gemm_small(T, d, E):
    rng = np.random.default_rng(T)
    h = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    wr = torch.from_numpy((rng.standard_normal((E, d)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    bias = torch.from_numpy(rng.standard_normal(E).astype(np.float32))
    cfg = _cfg(T, E, 2, d=d)
    ws = moe.workspace(cfg)
    g = moe.route(cfg, ws, h=h.cuda(), wr=wr.cuda(), bias=bias.cuda())
    assert moe.device_status(ws) == 0
    o = oracle.route(2, h=bits(h), wr=bits(wr), bias=bias.numpy())
    assert np.abs(np_(g["logits"]) - o["logits"]).max() <= LOGIT_MAX_ABS


@pytest.mark.parametrize("name", synth.CONFIG_ORDER)
def test_router_gemm_workloads(name):
    shape = synth.CONFIGS[name]
    h, wr, bias, usage = synth.router_inputs(shape)
    cfg = moe.Config.of(shape)
    ws = moe.workspace(cfg)
    g = moe.route(cfg, ws, h=h.cuda(), wr=wr.cuda(), bias=None if bias is None else bias.cuda(),
                  usage=None if usage is None else usage.cuda())
    assert moe.device_status(ws) == 0
    bnp = None if bias is None else bias.numpy()
    unp = None if usage is None else usage.numpy()
    o = oracle.route(shape.k, h=bits(h), wr=bits(wr), bias=bnp, usage=unp, lam=shape.lam)
    gl = np_(g["logits"])
    assert np.abs(gl - o["logits"]).max() <= LOGIT_MAX_ABS
    # on the GPU's own logits the routing is exactly the oracle's
    o2 = oracle.route(shape.k, logits_in=gl, usage=unp, lam=shape.lam)
    assert np.array_equal(np_(g["scores"]), o2["scores"])
    assert np.array_equal(np_(g["ids"]), o2["ids"])
    assert np.array_equal(np_(g["counts_pre"]), o2["counts_pre"])
    # against the oracle's own logits: identical picks wherever the margin is clear
    sel = topk_margin(o["scores"], shape.k) >= MARGIN
    assert sel.mean() > 0.95      # one 128-token run of identical tokens is 1.56% alone
    assert np.array_equal(np_(g["ids"])[sel], o["ids"][sel])


# ----------------------------------------------------------------------------- dispatch

DISPATCH_CASES = [
    # name, T, E, k, cf, explicit C, score kind
    ("tiny-shape", 256, 8, 2, 1.25, 0, "gauss"),
    ("overflow", 1000, 8, 2, 1.0, 0, "skew"),
    ("identical-128", 128, 8, 2, 1.0, 0, "identical"),
    ("page-127", 128, 16, 1, 1.0, 127, "identical"),
    ("drops", 5, 2, 2, 1.0, 1, "gauss"),
    ("deep-reroute", 300, 32, 2, 1.0, 10, "identical"),
    ("many-chunks", 5000, 64, 2, 1.0, 0, "gauss"),
    ("runs", 3000, 16, 2, 1.0, 0, "runs"),
    ("k3", 700, 12, 3, 1.0, 0, "skew"),
    ("k8", 513, 20, 8, 1.0, 0, "gauss"),
    ("cap-1", 40, 4, 2, 1.0, 1, "gauss"),
    ("no-overflow", 2000, 8, 2, 8.0, 0, "gauss"),
    ("ties", 1500, 10, 2, 1.0, 0, "ties"),
    ("T1", 1, 8, 2, 1.0, 0, "gauss"),
    ("E1", 77, 1, 1, 1.0, 0, "gauss"),
    ("E200", 4000, 200, 2, 1.1, 0, "skew"),
    # one chunk (T <= 256): route and dispatch run as one block
    ("small-E200", 256, 200, 2, 1.0, 0, "skew"),
    ("small-E255-k8", 250, 255, 8, 1.0, 3, "gauss"),
    ("small-E64-deep", 256, 64, 2, 1.0, 2, "identical"),
    ("small-E128-k4", 199, 128, 4, 1.0, 0, "skew"),
    # capacity well below demand: many fills per replay window, interacting through the
    # reroutes they cause (up to 9 fixed-point rounds in a window), and drops
    ("fills-interact-k8", 3000, 64, 8, 0.5, 0, "skew"),
    ("fills-dense-E255", 6000, 255, 4, 0.4, 0, "gauss"),
    ("small-many-fills", 256, 32, 4, 0.3, 0, "gauss"),
]


@pytest.mark.parametrize("case", DISPATCH_CASES, ids=[c[0] for c in DISPATCH_CASES])
def test_dispatch_shared_scores(case):
    name, T, E, k, cf, cap, kind = case
    s = _scores(kind, T, E, T * 7 + E)
    cfg = _cfg(T, E, k, cf=cf, cap=cap)
    C = moe.capacity(T, k, E, cf, cap)
    assert C == oracle.capacity(T, k, E, cf, cap)
    ws = moe.workspace(cfg)
    g = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    assert moe.device_status(ws) == 0
    o = oracle.dispatch(s, k, C)
    assert_dispatch_equal(g, o, T, k)
    assert int(np_(g["n_rerouted"])[0]) == o["n_rerouted"]
    assert int(np_(g["n_dropped"])[0]) == o["n_dropped"]
    np.testing.assert_allclose(np_(g["cw"]), o["cw"], rtol=WEIGHT_RTOL, atol=1e-7)


def _random_dispatch_case(i):
    rng = np.random.default_rng(1000 + i)
    T = int(rng.choice([1, 7, 64, 200, 256, 257, 700, 1500, 3000]))
    E = int(rng.choice([2, 3, 8, 16, 33, 64, 128, 200, 255]))
    k = int(min(E, rng.choice([1, 2, 2, 3, 4, 8])))
    cf = float(rng.choice([0.2, 0.3, 0.5, 0.8, 1.0, 1.25, 2.0]))
    cap = int(rng.integers(1, 6)) if rng.random() < 0.15 else 0
    kind = str(rng.choice(["gauss", "skew", "ties", "runs", "identical"]))
    return T, E, k, cf, cap, kind


@pytest.mark.parametrize("i", range(40))
def test_dispatch_random_shapes(i):
    """Seeded random shapes and capacities (many fills per replay window, drops, one-chunk
    and multi-chunk batches, k up to 8, E up to 255): the dispatch equals the oracle's."""
    T, E, k, cf, cap, kind = _random_dispatch_case(i)
    s = _scores(kind, T, E, 77 * i + 5)
    cfg = _cfg(T, E, k, cf=cf, cap=cap)
    C = moe.capacity(T, k, E, cf, cap)
    assert C == oracle.capacity(T, k, E, cf, cap)
    ws = moe.workspace(cfg)
    g = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    assert moe.device_status(ws) == 0
    o = oracle.dispatch(s, k, C)
    assert_dispatch_equal(g, o, T, k)
    assert int(np_(g["n_rerouted"])[0]) == o["n_rerouted"]
    assert int(np_(g["n_dropped"])[0]) == o["n_dropped"]
    assert np.array_equal(np_(g["counts"]), o["counts"])


def test_dispatch_repeatable():
    s = _scores("skew", 4000, 16, 3)
    cfg = _cfg(4000, 16, 2, cf=1.0)
    ws = moe.workspace(cfg)
    a = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    b = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    for key in ("assign", "slot", "perm", "cw"):
        assert torch.equal(a[key], b[key])


# ----------------------------------------------------------------------------- experts

# the last three pair row tiles across a 2-CTA cluster (T*k >= 256*E), with odd
# row-tile counts per expert among them
@pytest.mark.parametrize("T,d,E,F,k,cf", [(300, 192, 5, 256, 2, 1.0), (256, 512, 8, 1024, 2, 1.25),
                                          (40, 64, 3, 128, 1, 1.0), (600, 128, 6, 384, 3, 1.0),
                                          (700, 128, 3, 256, 2, 1.0), (1300, 256, 2, 512, 2, 1.25),
                                          (1000, 192, 4, 384, 2, 1.0)])
def test_expert_ffn_vs_oracle(T, d, E, F, k, cf):
    shape = synth.MoEShape("t", T=T, d=d, E=E, F=F, k=k, cf=cf, seed=T + F)
    h, wr, _, _ = synth.router_inputs(shape)
    w1, w3, w2 = synth.expert_weights(shape, device="cuda")
    cfg = moe.Config.of(shape)
    ws = moe.workspace(cfg)
    s = _scores("skew", T, E, T)
    dsp = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    w13 = moe.pack_w13(w1, w3)
    y = moe.expert_ffn(cfg, ws, h.cuda(), dsp["perm"], dsp["offsets"], w13, w2)
    assert moe.device_status(ws) == 0
    n = int(np_(dsp["offsets"])[-1])
    want = oracle.expert_slots(bits(h), bits(w1), bits(w3), bits(w2), np_(dsp["assign"]),
                               np_(dsp["perm"])[:n], 0, n)
    got = np_(y[:n].float())
    assert rel_frob(got, want) <= OUT_REL_FROB
    rows = np.linalg.norm(got - want, axis=1) / np.maximum(np.linalg.norm(want, axis=1), 1e-12)
    assert rows.max() <= 4 * OUT_REL_FROB


# one piece per lane below 2048 tokens, two from there; d = 192 leaves most lanes
# of a row segment past the row's end
@pytest.mark.parametrize("T,d", [(500, 256), (2500, 192), (2048, 4096)])
def test_combine_vs_numpy(T, d):
    E, k = 6, 2
    s = _scores("skew", T, E, 5)
    cfg = _cfg(T, E, k, d=d, cf=1.0)
    ws = moe.workspace(cfg)
    dsp = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    y = torch.randn(T * k, d, device="cuda").to(torch.bfloat16)
    out = moe.combine(cfg, y, dsp["assign"], dsp["slot"], dsp["offsets"], dsp["cw"])
    yf = np_(y.float()).astype(np.float64)
    a, sl, off, cw = (np_(dsp[x]) for x in ("assign", "slot", "offsets", "cw"))
    want = np.zeros((T, d))
    for t in range(T):
        for r in range(k):
            if a[t, r] >= 0:
                want[t] += cw[t, r] * yf[off[a[t, r]] + sl[t, r]]
    assert rel_frob(np_(out.float()), want) <= 1e-2


# ----------------------------------------------------------------------------- fused layer

# sampled tokens besides the per-tile ones (a count >= T checks every token)
SAMPLE = {"tiny": 256, "mixtral_prefill": 64, "mixtral_decode": 64, "fine_grained": 256, "skewed": 128}


@pytest.mark.parametrize("name", synth.CONFIG_ORDER)
def test_layer_forward_workloads(name):
    shape = synth.CONFIGS[name]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape)
    ws = moe.workspace(cfg)
    out, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], bias=Ld["bias"],
                                 usage=Ld["usage"], aux=True)
    assert moe.device_status(ws) == 0
    unp = None if Ld["usage"] is None else np_(Ld["usage"])
    C = oracle.capacity(shape.T, shape.k, shape.E, shape.cf, shape.capacity)
    # (1) routing and dispatch bit-exact on the GPU's logits
    o_r = oracle.route(shape.k, logits_in=np_(aux["logits"]), usage=unp, lam=shape.lam)
    o_d = oracle.dispatch(o_r["scores"], shape.k, C)
    assert_dispatch_equal(aux, o_d, shape.T, shape.k)
    np.testing.assert_allclose(np_(aux["P"]), o_r["P"], rtol=WEIGHT_RTOL, atol=1e-7)
    np.testing.assert_allclose(np_(aux["f"]), o_r["f"], rtol=1e-7)
    # (2) outputs on sampled tokens (all for the tiny layer), incl. rerouted and dropped
    # ones, and one token in every (expert, 128-row tile) of the expert GEMMs
    fl = o_d["flags"]
    special = np.flatnonzero((fl != 0).any(1))[:6]
    special = np.concatenate([special, tile_tokens(o_d["perm"], o_d["offsets"], shape.k, shape.seed)])
    toks = (np.arange(shape.T, dtype=np.int32) if SAMPLE[name] >= shape.T
            else sample_tokens(shape.T, SAMPLE[name], shape.seed, must=special))
    cpu = lambda t: bits(t)
    want = oracle.combine_rows(cpu(Ld["h"]), cpu(Ld["w1"]), cpu(Ld["w3"]), cpu(Ld["w2"]),
                               o_d["assign"], o_d["cw"], toks)
    got = np_(out.float())[toks]
    assert_rows_close(got, want)
    dropped_all = (o_d["assign"] < 0).all(1)
    if dropped_all.any():
        assert (np_(out.float())[dropped_all] == 0).all()


@pytest.mark.parametrize("name", ["tiny", "fine_grained"])
def test_layer_forward_deterministic(name):
    shape = synth.CONFIGS[name]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape)
    ws = moe.workspace(cfg)
    a = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], Ld["bias"], Ld["usage"])
    b = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], Ld["bias"], Ld["usage"])
    assert torch.equal(a, b)


@pytest.mark.parametrize("T,E,k,cap", [(1, 8, 2, 0), (300, 6, 1, 0), (300, 6, 3, 0),
                                       (257, 4, 2, 30), (64, 1, 1, 0), (900, 3, 2, 0),
                                       (1500, 2, 2, 700), (200, 40, 2, 2),
                                       # general k: one choice per token, four per token
                                       (2000, 8, 1, 0), (1200, 16, 4, 0), (600, 12, 4, 40)])
def test_layer_forward_edge_shapes(T, E, k, cap):
    shape = synth.MoEShape("edge", T=T, d=128, E=E, F=256, k=k, cf=1.0, capacity=cap, seed=T + E)
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape)
    ws = moe.workspace(cfg)
    out, aux = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], aux=True)
    assert moe.device_status(ws) == 0
    C = oracle.capacity(T, k, E, 1.0, cap)
    o_r = oracle.route(k, logits_in=np_(aux["logits"]))
    o_d = oracle.dispatch(o_r["scores"], k, C)
    assert_dispatch_equal(aux, o_d, T, k)
    want = oracle.combine_rows(bits(Ld["h"]), bits(Ld["w1"]), bits(Ld["w3"]), bits(Ld["w2"]),
                               o_d["assign"], o_d["cw"], np.arange(T, dtype=np.int32))
    assert rel_frob(np_(out.float()), want) <= OUT_REL_FROB
    dropped_all = (o_d["assign"] < 0).all(1)
    assert (np_(out.float())[dropped_all] == 0).all()


def test_layer_forward_host_matches_device():
    shape = synth.CONFIGS["tiny"]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape)
    ws = moe.workspace(cfg)
    dev = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"])
    h_host = Ld["h"].cpu().pin_memory()
    out_host = torch.empty(shape.T, shape.d, dtype=torch.bfloat16).pin_memory()
    moe.layer_forward_host(cfg, ws, h_host, Ld["wr"], Ld["w13"], Ld["w2"], out_host)
    assert torch.equal(out_host, dev.cpu())


@pytest.mark.parametrize("name", ["tiny", "mixtral_prefill"])
def test_layer_forward_host_async_pipelined(name):
    """Batches alternate over two workspaces and two streams: each output equals the device
    call's on the same input, whatever the overlap."""
    shape = synth.CONFIGS[name]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape)
    wss = [moe.workspace(cfg), moe.workspace(cfg)]
    gen = torch.Generator().manual_seed(11)
    hs = [Ld["h"].cpu()] + [torch.randn(shape.T, shape.d, generator=gen).to(torch.bfloat16) for _ in range(3)]
    want = [moe.layer_forward(cfg, wss[0], h.cuda(), Ld["wr"], Ld["w13"], Ld["w2"]).cpu() for h in hs]
    h_hosts = [h.pin_memory() for h in hs]
    outs = [torch.empty(shape.T, shape.d, dtype=torch.bfloat16).pin_memory() for _ in hs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for i in range(len(hs)):
        with torch.cuda.stream(streams[i % 2]):
            moe.layer_forward_host_async(cfg, wss[i % 2], h_hosts[i], Ld["wr"], Ld["w13"], Ld["w2"], outs[i])
    for st in streams:
        st.synchronize()
    for i in range(len(hs)):
        assert torch.equal(outs[i], want[i]), i


def test_stage_events_recorded():
    shape = synth.CONFIGS["tiny"]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape)
    ws = moe.workspace(cfg)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(moe.NUM_STAGES + 1)]
    moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], stage_events=evs)
    torch.cuda.synchronize()
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(moe.NUM_STAGES)]
    assert all(t >= 0 for t in times)


# ----------------------------------------------------------------------------- failure path

def test_bounded_wait_reports_timeout_and_context_survives():
    cfg = _cfg(10, 4, 2)
    ws = moe.workspace(cfg)
    moe.timeout_probe(ws, 2_000_000)          # ~1 ms of SM clock; nothing ever arrives
    assert moe.device_status(ws) == 6
    assert moe.device_status(ws) == 0
    # the context is still usable
    s = _scores("gauss", 10, 4, 0)
    g = moe.dispatch(cfg, ws, torch.from_numpy(s).cuda())
    o = oracle.dispatch(s, 2, moe.capacity(10, 2, 4, 1.0))
    assert_dispatch_equal(g, o, 10, 2)
