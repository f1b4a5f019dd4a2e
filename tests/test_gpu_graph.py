"""The library's calls are asynchronous on the caller's stream and allocate nothing, so a whole
layer forward (or backward) can be captured in a CUDA graph and replayed: the replay must give
the eager call's results bit for bit."""
import pytest
import torch

from helpers import make_layer
from token_level_top_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()   # warm-up on the side stream: one-time attribute setting and tensor-map encoding
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("name", ["tiny", "mixtral_decode", "skewed"])
def test_layer_forward_graph_replay_matches_eager(name):
    shape = synth.CONFIGS[name]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape)
    ws = moe.workspace(cfg)
    out = torch.empty(shape.T, shape.d, dtype=torch.bfloat16, device="cuda")
    eager = moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], Ld["bias"], Ld["usage"]).clone()
    g = capture(lambda: moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], Ld["bias"], Ld["usage"],
                                          out=out))
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    assert torch.equal(out, eager)
    # new inputs copied into the captured buffers flow through the replay
    h2 = torch.randn(shape.T, shape.d, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16).cuda()
    want = moe.layer_forward(cfg, moe.workspace(cfg), h2, Ld["wr"], Ld["w13"], Ld["w2"], Ld["bias"], Ld["usage"])
    Ld["h"].copy_(h2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, want)


def test_fp8_and_router_variant_forward_graph_replay():
    shape = synth.CONFIGS["mixtral_decode"]
    Ld = make_layer(shape)
    rw = synth.router_variant_weights(shape.d, shape.E, 2 * shape.E, True, seed=5)
    router = moe.Router(**{k: (None if v is None else v.cuda()) for k, v in rw.items()})
    cfg = moe.Config.of(shape, flags=moe.FLAG_FP8, tau=0.7, router_norm=moe.NORM_LAYER,
                        router_hidden=2 * shape.E)
    ws = moe.workspace(cfg)
    w13, w2 = moe.quantize_fp8(Ld["w13"]), moe.quantize_fp8(Ld["w2"])
    out = torch.empty(shape.T, shape.d, dtype=torch.bfloat16, device="cuda")
    eager = moe.layer_forward(cfg, ws, Ld["h"], router, w13, w2).clone()
    g = capture(lambda: moe.layer_forward(cfg, ws, Ld["h"], router, w13, w2, out=out))
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    assert torch.equal(out, eager)


def test_training_step_graph_replay():
    shape = synth.CONFIGS["tiny"]
    Ld = make_layer(shape)
    cfg = moe.Config.of(shape, flags=moe.FLAG_BACKWARD)
    ws = moe.workspace(cfg)
    dout = torch.randn(shape.T, shape.d, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).cuda()
    out = torch.empty(shape.T, shape.d, dtype=torch.bfloat16, device="cuda")
    moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], Ld["bias"], out=out)
    eager = moe.layer_backward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], dout)
    eager = {n: t.clone() for n, t in eager.items()}
    res = {}

    def step():
        moe.layer_forward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], Ld["bias"], out=out)
        res.update(moe.layer_backward(cfg, ws, Ld["h"], Ld["wr"], Ld["w13"], Ld["w2"], dout))

    g = capture(step)
    g.replay()
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    for n in eager:
        assert torch.equal(res[n], eager[n]), n
