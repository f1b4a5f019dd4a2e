"""Thin ctypes binding over libmoe.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (device memory and streams come from
PyTorch); calls are enqueued on the current torch stream.  There is no CPU
fallback: if the library is missing, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe.h")
NUM_STAGES = 6
STAGE_NAMES = ["route", "dispatch", "prep", "gate_up", "down", "combine"]

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "misaligned pointer",
          4: "workspace too small", 5: "non-finite (NaN) score", 6: "bounded device wait timed out",
          7: "CUDA runtime error"}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, 'unknown')} (status {status})")
        self.status = status


class MoEConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("cf", ctypes.c_double),
                ("capacity", ctypes.c_int32), ("lambda_", ctypes.c_float),
                ("flags", ctypes.c_uint32), ("tau", ctypes.c_float), ("router_norm", ctypes.c_uint32),
                ("norm_eps", ctypes.c_float), ("router_hidden", ctypes.c_int32)]


class MoERouter(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("norm_gamma", ctypes.c_void_p), ("norm_beta", ctypes.c_void_p)]


@dataclass
class Config:
    T: int
    d_model: int
    E: int
    k: int
    d_ff: int
    cf: float = 1.25
    capacity: int = 0
    lam: float = 0.0
    flags: int = 0   # FLAG_FP8 / FLAG_NVFP4 / FLAG_BACKWARD: the workspace also serves those entry points
    tau: float = 1.0           # router temperature
    router_norm: int = 0       # NORM_LAYER / NORM_L2: normalise h before the router
    norm_eps: float = 1e-5
    router_hidden: int = 0     # H > 0: the two-layer router silu(x W1^T) W2^T

    def c(self) -> MoEConfig:
        return MoEConfig(self.T, self.d_model, self.E, self.k, self.d_ff, float(self.cf),
                         int(self.capacity), float(self.lam), int(self.flags), float(self.tau),
                         int(self.router_norm), float(self.norm_eps), int(self.router_hidden))

    @classmethod
    def of(cls, shape, **kw):
        d = dict(T=shape.T, d_model=shape.d, E=shape.E, k=shape.k, d_ff=shape.F, cf=shape.cf,
                 capacity=shape.capacity, lam=shape.lam)
        d.update(kw)
        return cls(**d)


FLAG_FP8 = 1   # MOE_FLAG_FP8
FLAG_BACKWARD = 2   # MOE_FLAG_BACKWARD
FLAG_NVFP4 = 4   # MOE_FLAG_NVFP4
NORM_NONE, NORM_LAYER, NORM_L2 = 0, 1, 2   # MOE_ROUTER_NORM_*


@dataclass
class Router:
    """Router weights of the router variants (moe_router_t): w [E,d] bf16, or W1
    [H,d] with w2 = W2 [E,H] for the two-layer router; bias [E] fp32; gamma,
    beta [d] fp32 for the LayerNorm before the router."""
    w: torch.Tensor
    w2: torch.Tensor = None
    bias: torch.Tensor = None
    gamma: torch.Tensor = None
    beta: torch.Tensor = None

    def c(self) -> MoERouter:
        return MoERouter(*[None if t is None else t.data_ptr()
                           for t in (self.w, self.w2, self.bias, self.gamma, self.beta)])

_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
SZ = ctypes.c_size_t
CFG = ctypes.POINTER(MoEConfig)
RTR = ctypes.POINTER(MoERouter)

_SIGS = {
    "moe_capacity": (ctypes.c_int64, [ctypes.c_int64, I32, I32, ctypes.c_double, I32]),
    "moe_workspace_size": (SZ, [CFG]),
    "moe_workspace_init": (I32, [P, SZ, P]),
    "moe_get_device_status": (I32, [P, P]),
    "moe_status_string": (ctypes.c_char_p, [I32]),
    "moe_pack_w13": (I32, [I32, I32, I32, P, P, P, P]),
    "moe_route": (I32, [CFG, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_dispatch": (I32, [CFG, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_expert_ffn": (I32, [CFG, P, P, P, P, P, P, P, SZ, P]),
    "moe_combine": (I32, [CFG, P, P, P, P, P, P, P]),
    "moe_layer_forward": (I32, [CFG, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_layer_forward_host": (I32, [CFG, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_layer_forward_host_async": (I32, [CFG, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_debug_timeout_probe": (I32, [P, SZ, ctypes.c_int64, P]),
    "moe_dispatch_static": (I32, [CFG, P, P, P, P, P, P, P, P, P, P, P, P]),
    "moe_quantize_fp8": (I32, [ctypes.c_int64, I32, P, P, P, P]),
    "moe_expert_ffn_fp8": (I32, [CFG, P, P, P, P, P, P, P, P, P, SZ, P]),
    "moe_layer_forward_fp8": (I32, [CFG] + [P] * 18 + [SZ, P]),
    "moe_nvfp4_sf_stride": (I32, [I32]),
    "moe_quantize_nvfp4": (I32, [ctypes.c_int64, I32, P, P, P, P, P]),
    "moe_quantize_w13_nvfp4": (I32, [I32, I32, I32, P, P, P, P, P]),
    "moe_expert_ffn_nvfp4": (I32, [CFG] + [P] * 10 + [P, SZ, P]),
    "moe_layer_forward_nvfp4": (I32, [CFG] + [P] * 20 + [SZ, P]),
    "moe_router_logits": (I32, [CFG, P, RTR, P, P, SZ, P]),
    "moe_layer_backward": (I32, [CFG] + [P] * 12 + [SZ, P]),
    "moe_layer_forward_router": (I32, [CFG, P, RTR] + [P] * 15 + [SZ, P]),
}


def header_functions():
    """Names of the functions include/moe.h declares."""
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def lib():
    """Load libmoe.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so not found at {LIB_PATH}: run "
                               "`python -m token_level_top_gb300.build` (CUDA path has no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(st: int, where: str):
    if st != 0:
        raise MoEError(st, where)


def capacity(T: int, k: int, E: int, cf: float, explicit: int = 0) -> int:
    return int(lib().moe_capacity(T, k, E, cf, explicit))


def workspace_size(cfg: Config) -> int:
    c = cfg.c()
    return int(lib().moe_workspace_size(ctypes.byref(c)))


def workspace(cfg: Config, device="cuda") -> torch.Tensor:
    """A workspace for ``cfg`` (torch allocation, 512-byte aligned), initialised."""
    n = workspace_size(cfg)
    if n == 0:
        raise MoEError(1, "moe_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(lib().moe_workspace_init(_p(ws), n, _stream()), "moe_workspace_init")
    return ws


def device_status(ws: torch.Tensor) -> int:
    """Synchronises the current stream and returns (and clears) the device status."""
    return int(lib().moe_get_device_status(_p(ws), _stream()))


def check_device(ws: torch.Tensor, where: str = "device"):
    _check(device_status(ws), where)


def pack_w13(w1: torch.Tensor, w3: torch.Tensor) -> torch.Tensor:
    E, F, d = w1.shape
    w13 = torch.empty(E, 2 * F, d, dtype=torch.bfloat16, device=w1.device)
    _check(lib().moe_pack_w13(E, F, d, _p(w1.contiguous()), _p(w3.contiguous()), _p(w13),
                              _stream()), "moe_pack_w13")
    return w13


def quantize_fp8(w: torch.Tensor):
    """Per-row e4m3 quantisation (moe_quantize_fp8) of a bf16 tensor [..., cols]:
    returns (q uint8, same shape; scales fp32, one per row)."""
    w = w.contiguous()
    cols = w.shape[-1]
    rows = w.numel() // cols
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    sc = torch.empty(rows, dtype=torch.float32, device=w.device)
    _check(lib().moe_quantize_fp8(rows, cols, _p(w), _p(q), _p(sc), _stream()), "moe_quantize_fp8")
    return q, sc


def _fp8(w):
    """Expert weights as (q, scales) from quantize_fp8, or None for bf16 weights."""
    return w if isinstance(w, tuple) and len(w) == 2 else None


def _fp4(w):
    """Expert weights as (codes, block scales, row scales) from quantize_nvfp4, or None."""
    return w if isinstance(w, tuple) and len(w) == 3 else None


def quantize_nvfp4(w: torch.Tensor):
    """NVFP4 quantisation (moe_quantize_nvfp4) of a bf16 tensor [..., cols]: returns
    (codes uint8 [..., cols/2], block scales uint8 [..., moe_nvfp4_sf_stride(cols)],
    row scales fp32 [rows])."""
    w = w.contiguous()
    cols = w.shape[-1]
    rows = w.numel() // cols
    sfs = int(lib().moe_nvfp4_sf_stride(cols))
    q = torch.empty(*w.shape[:-1], cols // 2, dtype=torch.uint8, device=w.device)
    b = torch.empty(*w.shape[:-1], sfs, dtype=torch.uint8, device=w.device)
    sc = torch.empty(rows, dtype=torch.float32, device=w.device)
    _check(lib().moe_quantize_nvfp4(rows, cols, _p(w), _p(q), _p(b), _p(sc), _stream()), "moe_quantize_nvfp4")
    return q, b, sc


def quantize_w13_nvfp4(w13: torch.Tensor):
    """moe_quantize_w13_nvfp4: W13 [E, 2F, d] bf16 (moe_pack_w13 layout) to NVFP4 in
    the 4-bit path's 128-row packing (64 W1 rows, then the matching 64 W3 rows)."""
    w13 = w13.contiguous()
    E, F2, d = w13.shape
    sfs = int(lib().moe_nvfp4_sf_stride(d))
    q = torch.empty(E, F2, d // 2, dtype=torch.uint8, device=w13.device)
    b = torch.empty(E, F2, sfs, dtype=torch.uint8, device=w13.device)
    sc = torch.empty(E * F2, dtype=torch.float32, device=w13.device)
    _check(lib().moe_quantize_w13_nvfp4(E, F2 // 2, d, _p(w13), _p(q), _p(b), _p(sc), _stream()),
           "moe_quantize_w13_nvfp4")
    return q, b, sc


def route(cfg: Config, ws, h=None, wr=None, bias=None, usage=None, logits_in=None):
    dev = ws.device
    T, E, k = cfg.T, cfg.E, cfg.k
    out = dict(logits=torch.empty(T, E, dtype=torch.float32, device=dev),
               scores=torch.empty(T, E, dtype=torch.float32, device=dev),
               ids=torch.empty(T, k, dtype=torch.int32, device=dev),
               topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
               counts_pre=torch.empty(E, dtype=torch.int32, device=dev),
               f=torch.empty(E, dtype=torch.float32, device=dev),
               P=torch.empty(E, dtype=torch.float32, device=dev))
    c = cfg.c()
    st = lib().moe_route(ctypes.byref(c), _p(h), _p(wr), _p(bias), _p(usage), _p(logits_in),
                         _p(out["logits"]), _p(out["scores"]), _p(out["ids"]), _p(out["topk_w"]),
                         _p(out["counts_pre"]), _p(out["f"]), _p(out["P"]), _p(ws), ws.numel(),
                         _stream())
    _check(st, "moe_route")
    return out


def router_logits(cfg: Config, ws, h, router: Router):
    """The logits [T, E] fp32 of cfg's router variant (normalisation, two-layer router)."""
    z = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=ws.device)
    c, r = cfg.c(), router.c()
    st = lib().moe_router_logits(ctypes.byref(c), _p(h), ctypes.byref(r), _p(z), _p(ws), ws.numel(),
                                 _stream())
    _check(st, "moe_router_logits")
    return z


def dispatch(cfg: Config, ws, scores):
    dev = ws.device
    T, E, k = cfg.T, cfg.E, cfg.k
    out = dict(assign=torch.empty(T, k, dtype=torch.int32, device=dev),
               slot=torch.empty(T, k, dtype=torch.int32, device=dev),
               flags=torch.empty(T, k, dtype=torch.uint8, device=dev),
               counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               perm=torch.full((max(T * k, 1),), -1, dtype=torch.int32, device=dev),
               cw=torch.empty(T, k, dtype=torch.float32, device=dev),
               n_rerouted=torch.zeros(1, dtype=torch.int32, device=dev),
               n_dropped=torch.zeros(1, dtype=torch.int32, device=dev))
    c = cfg.c()
    st = lib().moe_dispatch(ctypes.byref(c), _p(scores), _p(out["assign"]), _p(out["slot"]),
                            _p(out["flags"]), _p(out["counts"]), _p(out["offsets"]),
                            _p(out["perm"]), _p(out["cw"]), _p(out["n_rerouted"]),
                            _p(out["n_dropped"]), _p(ws), ws.numel(), _stream())
    _check(st, "moe_dispatch")
    return out


def expert_ffn(cfg: Config, ws, h, perm, offsets, w13, w2):
    y = torch.empty(max(cfg.T * cfg.k, 1), cfg.d_model, dtype=torch.bfloat16, device=ws.device)
    c = cfg.c()
    if _fp4(w13):
        (q13, b13, s13), (q2, b2, s2) = w13, w2
        st = lib().moe_expert_ffn_nvfp4(ctypes.byref(c), _p(h), _p(perm), _p(offsets), _p(q13), _p(b13),
                                        _p(s13), _p(q2), _p(b2), _p(s2), _p(y), _p(ws), ws.numel(), _stream())
    elif _fp8(w13):
        (q13, s13), (q2, s2) = w13, w2
        st = lib().moe_expert_ffn_fp8(ctypes.byref(c), _p(h), _p(perm), _p(offsets), _p(q13), _p(s13),
                                      _p(q2), _p(s2), _p(y), _p(ws), ws.numel(), _stream())
    else:
        st = lib().moe_expert_ffn(ctypes.byref(c), _p(h), _p(perm), _p(offsets), _p(w13), _p(w2), _p(y),
                                  _p(ws), ws.numel(), _stream())
    _check(st, "moe_expert_ffn")
    return y


def combine(cfg: Config, y_slots, assign, slot, offsets, cw):
    out = torch.empty(cfg.T, cfg.d_model, dtype=torch.bfloat16, device=y_slots.device)
    c = cfg.c()
    st = lib().moe_combine(ctypes.byref(c), _p(y_slots), _p(assign), _p(slot), _p(offsets), _p(cw),
                           _p(out), _stream())
    _check(st, "moe_combine")
    return out


def layer_forward(cfg: Config, ws, h, wr, w13, w2, bias=None, usage=None, aux=False,
                  stage_events=None, out=None):
    """The fused layer.  Returns out [T, d] bf16 (and a dict of routing outputs when aux).
    wr: the router weight [E, d] bf16, or a Router (any router variant of cfg; its
    bias is the router's, so bias stays None).  w13 / w2: bf16 tensors, (q, scales)
    pairs from quantize_fp8 for e4m3 weights, or (codes, block scales, row scales)
    from quantize_w13_nvfp4 / quantize_nvfp4 for NVFP4 weights."""
    dev = ws.device
    T, E, k = cfg.T, cfg.E, cfg.k
    if out is None:
        out = torch.empty(T, cfg.d_model, dtype=torch.bfloat16, device=dev)
    extras = None
    if aux:
        extras = dict(logits=torch.empty(T, E, dtype=torch.float32, device=dev),
                      assign=torch.empty(T, k, dtype=torch.int32, device=dev),
                      slot=torch.empty(T, k, dtype=torch.int32, device=dev),
                      flags=torch.empty(T, k, dtype=torch.uint8, device=dev),
                      counts=torch.empty(E, dtype=torch.int32, device=dev),
                      f=torch.empty(E, dtype=torch.float32, device=dev),
                      P=torch.empty(E, dtype=torch.float32, device=dev))
    ev_arr = None
    if stage_events is not None:
        for e in stage_events:      # torch creates the CUDA event on its first record
            if e.cuda_event == 0:
                e.record()
        ev_arr = (ctypes.c_void_p * (NUM_STAGES + 1))(*[ctypes.c_void_p(e.cuda_event)
                                                        for e in stage_events])
    g = (lambda n: _p(extras[n]) if extras else None)
    c = cfg.c()
    evp = ctypes.cast(ev_arr, ctypes.c_void_p) if ev_arr is not None else None
    tail = (_p(out), g("logits"), g("assign"), g("slot"), g("flags"), g("counts"), g("f"), g("P"), evp,
            _p(ws), ws.numel(), _stream())
    if isinstance(wr, Router):
        if _fp4(w13):
            raise ValueError("the router variants take bf16 or e4m3 experts")
        if bias is not None:
            raise ValueError("the router's bias belongs in the Router")
        (q13, s13), (q2, s2) = (w13, w2) if _fp8(w13) else ((w13, None), (w2, None))
        r = wr.c()
        st = lib().moe_layer_forward_router(ctypes.byref(c), _p(h), ctypes.byref(r), _p(usage), _p(q13),
                                            _p(s13), _p(q2), _p(s2), *tail)
    elif _fp4(w13):   # NVFP4 expert weights: (codes, block scales, row scales)
        (q13, b13, s13), (q2, b2, s2) = w13, w2
        st = lib().moe_layer_forward_nvfp4(ctypes.byref(c), _p(h), _p(wr), _p(bias), _p(usage), _p(q13),
                                           _p(b13), _p(s13), _p(q2), _p(b2), _p(s2), *tail)
    elif _fp8(w13):   # e4m3 expert weights: (q, scales) pairs from quantize_fp8
        (q13, s13), (q2, s2) = w13, w2
        st = lib().moe_layer_forward_fp8(ctypes.byref(c), _p(h), _p(wr), _p(bias), _p(usage), _p(q13),
                                         _p(s13), _p(q2), _p(s2), *tail)
    else:
        st = lib().moe_layer_forward(ctypes.byref(c), _p(h), _p(wr), _p(bias), _p(usage), _p(w13),
                                     _p(w2), *tail)
    _check(st, "moe_layer_forward")
    return (out, extras) if aux else out


def layer_backward(cfg: Config, ws, h, wr, w13, w2, dout, dP=None, router_grads=True):
    """Gradients of the layer for the forward last run in ws (cfg with FLAG_BACKWARD):
    dict(dh [T,d], dw13 [E,2F,d], dw2 [E,d,F], dwr [E,d], dbias [E]), all fp32.
    dout [T,d] bf16; dP [E] fp32 = dL/dP of a load-balancing loss, or None."""
    dev = ws.device
    T, d, E, F = cfg.T, cfg.d_model, cfg.E, cfg.d_ff
    g = dict(dh=torch.empty(T, d, dtype=torch.float32, device=dev),
             dw13=torch.empty(E, 2 * F, d, dtype=torch.float32, device=dev),
             dw2=torch.empty(E, d, F, dtype=torch.float32, device=dev))
    if router_grads:
        g["dwr"] = torch.empty(E, d, dtype=torch.float32, device=dev)
        g["dbias"] = torch.empty(E, dtype=torch.float32, device=dev)
    c = cfg.c()
    st = lib().moe_layer_backward(ctypes.byref(c), _p(h), _p(wr), _p(w13), _p(w2), _p(dout), _p(dP), _p(g["dh"]),
                                  _p(g.get("dwr")), _p(g.get("dbias")), _p(g["dw13"]), _p(g["dw2"]), _p(ws),
                                  ws.numel(), _stream())
    _check(st, "moe_layer_backward")
    return g


def layer_forward_host(cfg: Config, ws, h_host, wr, w13, w2, out_host, bias=None, usage=None):
    """End-to-end call from pinned host memory; returns after the stream finished."""
    c = cfg.c()
    st = lib().moe_layer_forward_host(ctypes.byref(c), _p(h_host), _p(wr), _p(bias), _p(usage),
                                      _p(w13), _p(w2), _p(out_host), _p(ws), ws.numel(), _stream())
    _check(st, "moe_layer_forward_host")
    return out_host


def layer_forward_host_async(cfg: Config, ws, h_host, wr, w13, w2, out_host, bias=None, usage=None):
    """As layer_forward_host, without the final synchronisation (copies and kernels are enqueued
    on the current stream; synchronise it before reading out_host)."""
    c = cfg.c()
    st = lib().moe_layer_forward_host_async(ctypes.byref(c), _p(h_host), _p(wr), _p(bias), _p(usage),
                                            _p(w13), _p(w2), _p(out_host), _p(ws), ws.numel(), _stream())
    _check(st, "moe_layer_forward_host_async")
    return out_host


def timeout_probe(ws, budget_cycles: int):
    _check(lib().moe_debug_timeout_probe(_p(ws), ws.numel(), int(budget_cycles), _stream()),
           "moe_debug_timeout_probe")


def dispatch_static(cfg: Config, scores, device="cuda"):
    """moe_dispatch_static: the dispatch with the library's fixed scratch array
    instead of a workspace (for callers that cannot allocate).  The output
    tensors are allocated here by torch, as any caller's outputs would be, and
    filled with values the call must overwrite (-1, 0xFF, NaN)."""
    T, E, k = cfg.T, cfg.E, cfg.k

    def full(shape, v, dt):
        return torch.full(shape, v, dtype=dt, device=device)

    out = dict(assign=full((T, k), -1, torch.int32), slot=full((T, k), -1, torch.int32),
               flags=full((T, k), 0xFF, torch.uint8), counts=full((E,), -1, torch.int32),
               offsets=full((E + 1,), -1, torch.int32), perm=full((max(T * k, 1),), -1, torch.int32),
               cw=full((T, k), float("nan"), torch.float32), n_rerouted=full((1,), -1, torch.int32),
               n_dropped=full((1,), -1, torch.int32), status=full((1,), -1, torch.int32))
    c = cfg.c()
    st = lib().moe_dispatch_static(ctypes.byref(c), _p(scores), _p(out["assign"]), _p(out["slot"]),
                                   _p(out["flags"]), _p(out["counts"]), _p(out["offsets"]),
                                   _p(out["perm"]), _p(out["cw"]), _p(out["n_rerouted"]),
                                   _p(out["n_dropped"]), _p(out["status"]), _stream())
    _check(st, "moe_dispatch_static")
    return out
