"""CPU oracle for the MoE layer forward pass -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference leg may import this package.  The product path (the
CUDA library and its binding in ``token_level_top_gb300``) never does.

The arithmetic lives in ``moe_oracle.c`` (plain C, single thread, built with
``-O2 -ffp-contract=off``); this module only builds it, loads it with ctypes
and marshals numpy arrays.  bf16 tensors are passed as their raw 16-bit
patterns (``numpy.uint16``); the C code widens them exactly to fp32.

``THREADS`` (1 unless a caller raises it; the test suite does) lets the
per-row functions (``combine_rows*``, ``expert_slots*``) hand disjoint parts
of their token list or slot range to that many threads, each a call of the
same C function on its own rows.  A row's value depends on nothing but its
inputs, so the results are the same bits for any THREADS.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None
# A library built from an edited copy of moe_oracle.c (the mutation tests plant
# one mistake each and check that some pin fails); unset, the oracle is built here.
_LIB_OVERRIDE = os.environ.get("MOE_ORACLE_LIBRARY")
THREADS = 1


CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -ffp-contract=off)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_LIB_OVERRIDE or build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_capacity.argtypes = [ctypes.c_int64, I, I, ctypes.c_double, ctypes.c_int64]
            lib.oracle_capacity.restype = ctypes.c_int64
            lib.oracle_route.argtypes = [I, I, I, I, P, P, P, P, ctypes.c_float, ctypes.c_float, P,
                                         P, P, P, P, P, P, P]
            lib.oracle_route.restype = I
            lib.oracle_router_logits.argtypes = [I, I, I, I, I, ctypes.c_float, P, P, P, P, P, P, P]
            lib.oracle_router_logits.restype = I
            lib.oracle_layer_backward.argtypes = [I, I, I, I, I, ctypes.c_float] + [P] * 15
            lib.oracle_layer_backward.restype = I
            lib.oracle_preference.argtypes = [I, P, P]
            lib.oracle_preference.restype = I
            lib.oracle_dispatch.argtypes = [I, I, I, ctypes.c_int64, P, P, P, P, P, P, P, P, P, P]
            lib.oracle_dispatch.restype = I
            lib.oracle_expert_row.argtypes = [I, I, P, P, P, P, P]
            lib.oracle_expert_row.restype = None
            lib.oracle_combine_rows.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, I, P]
            lib.oracle_combine_rows.restype = I
            lib.oracle_expert_slots.argtypes = [I, I, I, I, I, P, P, P, P, P, P, I, I, P]
            lib.oracle_expert_slots.restype = I
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_combine_rows_q8.argtypes = [I, I, I, I, I] + [P] * 7 + [I] + [P] * 3 + [I, P]
            lib.oracle_combine_rows_q8.restype = I
            lib.oracle_expert_slots_q8.argtypes = [I, I, I, I, I] + [P] * 7 + [I, P, P, I, I, P]
            lib.oracle_expert_slots_q8.restype = I
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_quantize_row.argtypes = [I, P, P, P]
            lib.oracle_quantize_row.restype = None
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_value.restype = ctypes.c_double
            lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_quantize_row_nvfp4.argtypes = [I, P, P, P, P]
            lib.oracle_quantize_row_nvfp4.restype = None
            lib.oracle_combine_rows_q4.argtypes = [I, I, I, I, I] + [P] * 10 + [I] + [P] * 3 + [I, P]
            lib.oracle_combine_rows_q4.restype = I
            lib.oracle_expert_slots_q4.argtypes = [I, I, I, I, I] + [P] * 10 + [I, P, P, I, I, P]
            lib.oracle_expert_slots_q4.restype = I
            lib.oracle_init_tables.argtypes = []
            lib.oracle_init_tables.restype = None
            lib.oracle_init_tables()   # before any thread of _split_calls runs
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what} returned status {status}")
        self.status = status


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _split_calls(n: int, call, what: str):
    """call(i0, i1) -> status for the parts [i0, i1) of range(n), on up to THREADS threads."""
    _load()
    parts = max(1, min(int(THREADS), n))
    bounds = [n * j // parts for j in range(parts + 1)]
    if parts == 1:
        sts = [call(0, n)]
    else:
        with ThreadPoolExecutor(parts) as ex:
            sts = list(ex.map(lambda j: call(bounds[j], bounds[j + 1]), range(parts)))
    st = next((x for x in sts if x), 0)
    if st:
        raise OracleError(st, what)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def capacity(T: int, k: int, E: int, cf: float, explicit: int = 0) -> int:
    """C = ceil(T*k*cf/E) with cf as an exact decimal (six fractional digits)."""
    return int(_load().oracle_capacity(T, k, E, cf, explicit))


def preference(s_row) -> np.ndarray:
    s_row = _c(s_row, np.float32)
    order = np.empty(s_row.shape[0], np.int32)
    st = _load().oracle_preference(s_row.shape[0], _ptr(s_row), _ptr(order))
    if st:
        raise OracleError(st, "preference")
    return order


def route(k, h=None, wr=None, bias=None, usage=None, lam=0.0, logits_in=None, E=None, tau=1.0):
    """Router step.  h [T,d] / wr [E,d] as uint16 bf16 bits, or logits_in [T,E] fp32;
    tau the temperature (scores s = z / tau - lam * usage).

    Returns dict(logits, scores, ids, topk_p, counts_pre, f, P)."""
    lib = _load()
    if logits_in is not None:
        logits_in = _c(logits_in, np.float32)
        T, E = logits_in.shape
        d = 0
    else:
        h = _c(h, np.uint16)
        wr = _c(wr, np.uint16)
        T, d = h.shape
        E = wr.shape[0]
    bias = _c(bias, np.float32)
    usage = _c(usage, np.float32)
    out = dict(logits=np.empty((T, E), np.float32), scores=np.empty((T, E), np.float32),
               ids=np.empty((T, k), np.int32), topk_p=np.empty((T, k), np.float32),
               counts_pre=np.empty(E, np.int32), f=np.empty(E, np.float32),
               P=np.empty(E, np.float32))
    st = lib.oracle_route(T, d, E, k, _ptr(h), _ptr(wr), _ptr(bias), _ptr(usage), float(lam),
                          float(tau), _ptr(logits_in), _ptr(out["logits"]), _ptr(out["scores"]),
                          _ptr(out["ids"]), _ptr(out["topk_p"]), _ptr(out["counts_pre"]),
                          _ptr(out["f"]), _ptr(out["P"]))
    if st:
        raise OracleError(st, "route")
    return out


NORM_NONE, NORM_LAYER, NORM_L2 = 0, 1, 2


def router_logits(h, w, w2=None, bias=None, gamma=None, beta=None, norm=NORM_NONE, eps=1e-5):
    """Router front end: logits [T,E] fp32 from h [T,d] (bf16 bits), optionally
    normalised per row (NORM_LAYER with gamma/beta [d], or NORM_L2), then either
    x.W^T (w [E,d]) or the two-layer router silu(x.W1^T).W2^T (w = W1 [H,d],
    w2 = W2 [E,H]); bf16 bits for the weights, bias [E] fp32."""
    lib = _load()
    h = _c(h, np.uint16)
    w = _c(w, np.uint16)
    w2 = _c(w2, np.uint16)
    T, d = h.shape
    E = w2.shape[0] if w2 is not None else w.shape[0]
    H = w.shape[0] if w2 is not None else 0
    gamma, beta, bias = _c(gamma, np.float32), _c(beta, np.float32), _c(bias, np.float32)
    out = np.empty((T, E), np.float32)
    st = lib.oracle_router_logits(T, d, E, H, int(norm), float(eps), _ptr(h), _ptr(gamma), _ptr(beta),
                                  _ptr(w), _ptr(w2), _ptr(bias), _ptr(out))
    if st:
        raise OracleError(st, "router_logits")
    return out


def dispatch(scores, k: int, C: int):
    """Capacity-capped dispatch on penalised scores [T,E] fp32.

    Returns dict(assign, slot, flags, counts, offsets, perm, cw, n_rerouted, n_dropped)."""
    lib = _load()
    scores = _c(scores, np.float32)
    T, E = scores.shape
    out = dict(assign=np.empty((T, k), np.int32), slot=np.empty((T, k), np.int32),
               flags=np.empty((T, k), np.uint8), counts=np.empty(E, np.int32),
               offsets=np.empty(E + 1, np.int32), perm=np.full(T * k, -1, np.int32),
               cw=np.empty((T, k), np.float32))
    nre = np.zeros(1, np.int32)
    ndr = np.zeros(1, np.int32)
    st = lib.oracle_dispatch(T, E, k, int(C), _ptr(scores), _ptr(out["assign"]),
                             _ptr(out["slot"]), _ptr(out["flags"]), _ptr(out["counts"]),
                             _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["cw"]),
                             _ptr(nre), _ptr(ndr))
    if st:
        raise OracleError(st, "dispatch")
    out["perm"] = out["perm"][: int(out["offsets"][-1])]
    out["n_rerouted"] = int(nre[0])
    out["n_dropped"] = int(ndr[0])
    return out


def expert_row(x, w1, w3, w2) -> np.ndarray:
    """y = W2 (silu(W1 x) * W3 x) for one token, in double.  bf16 bits in."""
    x, w1, w3, w2 = (_c(a, np.uint16) for a in (x, w1, w3, w2))
    F, d = w1.shape
    y = np.empty(d, np.float64)
    _load().oracle_expert_row(d, F, _ptr(x), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(y))
    return y


def combine_rows(h, w1, w3, w2, assign, cw, tokens) -> np.ndarray:
    """Layer output rows (fp32) for the listed tokens, given a dispatch."""
    h, w1, w3, w2 = (_c(a, np.uint16) for a in (h, w1, w3, w2))
    assign = _c(assign, np.int32)
    cw = _c(cw, np.float32)
    tokens = _c(tokens, np.int32)
    T, d = h.shape
    E, F, _ = w1.shape
    k = assign.shape[1]
    out = np.empty((tokens.shape[0], d), np.float32)
    _split_calls(tokens.shape[0], lambda i0, i1: _lib.oracle_combine_rows(
        T, d, E, k, F, _ptr(h), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(assign), _ptr(cw), _ptr(tokens[i0:i1]),
        i1 - i0, _ptr(out[i0:i1])), "combine_rows")
    return out


def expert_slots(h, w1, w3, w2, assign, perm, row0: int, row1: int) -> np.ndarray:
    """Per-slot expert outputs (fp32) for slots [row0, row1) in slot order."""
    h, w1, w3, w2 = (_c(a, np.uint16) for a in (h, w1, w3, w2))
    assign = _c(assign, np.int32)
    perm = _c(perm, np.int32)
    T, d = h.shape
    E, F, _ = w1.shape
    k = assign.shape[1]
    out = np.empty((row1 - row0, d), np.float32)
    _split_calls(row1 - row0, lambda i0, i1: _lib.oracle_expert_slots(
        T, d, E, k, F, _ptr(h), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(assign), _ptr(perm), row0 + i0, row0 + i1,
        _ptr(out[i0:i1])), "expert_slots")
    return out


def e4m3_value(code: int) -> float:
    """Value of one e4m3 code (sign, 4-bit exponent bias 7, 3-bit mantissa)."""
    return float(_load().oracle_e4m3_value(int(code) & 0xFF))


def e4m3_encode(v: float) -> int:
    """The e4m3 code nearest to v (ties to even), saturating at +-448."""
    return int(_load().oracle_e4m3_encode(float(v)))


def quantize_row(x):
    """Row quantisation: (codes uint8, scale) with scale = max|x| / 448."""
    x = _c(x, np.float32)
    codes = np.empty(x.shape[0], np.uint8)
    sc = np.empty(1, np.float32)
    _load().oracle_quantize_row(x.shape[0], _ptr(x), _ptr(codes), _ptr(sc))
    return codes, float(sc[0])


def _q8(q1, s1, q3, s3, q2, s2):
    return ([_c(a, np.uint8) for a in (q1, q3, q2)], [_c(a, np.float32) for a in (s1, s3, s2)])


def combine_rows_q8(h, q1, s1, q3, s3, q2, s2, assign, cw, tokens, quant_act=True) -> np.ndarray:
    """combine_rows with e4m3 expert weights: q1, q3 [E,F,d] codes with row scales
    s1, s3 [E,F]; q2 [E,d,F] with s2 [E,d].  quant_act: token and activation
    rows also enter the GEMMs as row-quantised e4m3 (the FP8 layer's form)."""
    h = _c(h, np.uint16)
    (q1, q3, q2), (s1, s3, s2) = _q8(q1, s1, q3, s3, q2, s2)
    assign = _c(assign, np.int32)
    cw = _c(cw, np.float32)
    tokens = _c(tokens, np.int32)
    T, d = h.shape
    E, F, _ = q1.shape
    k = assign.shape[1]
    out = np.empty((tokens.shape[0], d), np.float32)
    _split_calls(tokens.shape[0], lambda i0, i1: _lib.oracle_combine_rows_q8(
        T, d, E, k, F, _ptr(h), _ptr(q1), _ptr(s1), _ptr(q3), _ptr(s3), _ptr(q2), _ptr(s2), int(quant_act),
        _ptr(assign), _ptr(cw), _ptr(tokens[i0:i1]), i1 - i0, _ptr(out[i0:i1])), "combine_rows_q8")
    return out


def expert_slots_q8(h, q1, s1, q3, s3, q2, s2, assign, perm, row0: int, row1: int,
                    quant_act=True) -> np.ndarray:
    """expert_slots with e4m3 expert weights (layouts and quant_act as combine_rows_q8)."""
    h = _c(h, np.uint16)
    (q1, q3, q2), (s1, s3, s2) = _q8(q1, s1, q3, s3, q2, s2)
    assign = _c(assign, np.int32)
    perm = _c(perm, np.int32)
    T, d = h.shape
    E, F, _ = q1.shape
    k = assign.shape[1]
    out = np.empty((row1 - row0, d), np.float32)
    _split_calls(row1 - row0, lambda i0, i1: _lib.oracle_expert_slots_q8(
        T, d, E, k, F, _ptr(h), _ptr(q1), _ptr(s1), _ptr(q3), _ptr(s3), _ptr(q2), _ptr(s2), int(quant_act),
        _ptr(assign), _ptr(perm), row0 + i0, row0 + i1, _ptr(out[i0:i1])), "expert_slots_q8")
    return out


def layer_forward(h, wr, w1, w3, w2, k, C, bias=None, usage=None, lam=0.0, tokens=None,
                  logits_in=None):
    """Whole layer: route, dispatch, experts and combine.

    ``tokens`` limits the (expensive) expert part to a sample of token rows.
    ``logits_in`` replaces the router GEMM (shared-logit comparisons)."""
    r = route(k, h=h, wr=wr, bias=bias, usage=usage, lam=lam, logits_in=logits_in)
    dsp = dispatch(r["scores"], k, C)
    T = r["scores"].shape[0]
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    out = combine_rows(h, w1, w3, w2, dsp["assign"], dsp["cw"], tokens)
    return r, dsp, out


def layer_backward(h, wr, w1, w3, w2, scores, assign, dout, tau=1.0, dP=None):
    """Backward pass for a fixed dispatch.  h [T,d], wr [E,d], w1/w3 [E,F,d], w2 [E,d,F]
    as bf16 bits; scores [T,E] fp32 (the forward's penalised scores); assign [T,k];
    dout [T,d] fp32; dP [E] (dL/dP of a load-balancing loss) or None.
    Returns dict(dh, dwr, dbias, dw1, dw3, dw2) in double."""
    lib = _load()
    h, wr, w1, w3, w2 = (_c(a, np.uint16) for a in (h, wr, w1, w3, w2))
    scores = _c(scores, np.float32)
    assign = _c(assign, np.int32)
    dout = _c(dout, np.float32)
    dP = _c(dP, np.float32)
    T, d = h.shape
    E, F, _ = w1.shape
    k = assign.shape[1]
    out = dict(dh=np.empty((T, d)), dwr=np.empty((E, d)), dbias=np.empty(E), dw1=np.empty((E, F, d)),
               dw3=np.empty((E, F, d)), dw2=np.empty((E, d, F)))
    st = lib.oracle_layer_backward(T, d, E, k, F, float(tau), _ptr(h), _ptr(wr), _ptr(w1), _ptr(w3), _ptr(w2),
                                   _ptr(scores), _ptr(assign), _ptr(dout), _ptr(dP), _ptr(out["dh"]),
                                   _ptr(out["dwr"]), _ptr(out["dbias"]), _ptr(out["dw1"]), _ptr(out["dw3"]),
                                   _ptr(out["dw2"]))
    if st:
        raise OracleError(st, "layer_backward")
    return out


def e2m1_value(code: int) -> float:
    """Value of a 4-bit e2m1 code (sign, 2-bit exponent bias 1, 1-bit mantissa)."""
    return float(_load().oracle_e2m1_value(int(code) & 0xF))


def e2m1_encode(v: float) -> int:
    """The e2m1 code nearest to v (ties to the even code), saturating at +-6."""
    return int(_load().oracle_e2m1_encode(float(v)))


def quantize_row_nvfp4(x):
    """NVFP4 row quantisation: (codes uint8 [n/2] packed, element 2m in the low
    nibble; e4m3 block scales uint8 [n/16]; fp32 row scale)."""
    x = _c(x, np.float32)
    n = x.shape[0]
    codes = np.empty(n // 2, np.uint8)
    bs = np.empty(n // 16, np.uint8)
    sc = np.empty(1, np.float32)
    _load().oracle_quantize_row_nvfp4(n, _ptr(x), _ptr(codes), _ptr(bs), _ptr(sc))
    return codes, bs, float(sc[0])


def _q4(w):
    """(codes, block scales, row scales) of the three weight matrices, contiguous."""
    return [(_c(q, np.uint8), _c(b, np.uint8), _c(sc, np.float32)) for q, b, sc in w]


def combine_rows_q4(h, w1, w3, w2, assign, cw, tokens, quant_act=True) -> np.ndarray:
    """combine_rows with NVFP4 expert weights.  w1, w3: (codes [E,F,d/2], block
    scales [E,F,d/16], row scales [E,F]); w2: (codes [E,d,F/2], [E,d,F/16], [E,d]).
    quant_act: token and activation rows NVFP4-quantised per row as well."""
    h = _c(h, np.uint16)
    (q1, b1, s1), (q3, b3, s3), (q2, b2, s2) = _q4((w1, w3, w2))
    assign = _c(assign, np.int32)
    cw = _c(cw, np.float32)
    tokens = _c(tokens, np.int32)
    T, d = h.shape
    E, F = s1.shape
    k = assign.shape[1]
    out = np.empty((tokens.shape[0], d), np.float32)
    _split_calls(tokens.shape[0], lambda i0, i1: _lib.oracle_combine_rows_q4(
        T, d, E, k, F, _ptr(h), _ptr(q1), _ptr(b1), _ptr(s1), _ptr(q3), _ptr(b3), _ptr(s3), _ptr(q2), _ptr(b2),
        _ptr(s2), int(quant_act), _ptr(assign), _ptr(cw), _ptr(tokens[i0:i1]), i1 - i0, _ptr(out[i0:i1])),
        "combine_rows_q4")
    return out


def expert_slots_q4(h, w1, w3, w2, assign, perm, row0: int, row1: int, quant_act=True) -> np.ndarray:
    """expert_slots with NVFP4 expert weights (layouts and quant_act as combine_rows_q4)."""
    h = _c(h, np.uint16)
    (q1, b1, s1), (q3, b3, s3), (q2, b2, s2) = _q4((w1, w3, w2))
    assign = _c(assign, np.int32)
    perm = _c(perm, np.int32)
    T, d = h.shape
    E, F = s1.shape
    k = assign.shape[1]
    out = np.empty((row1 - row0, d), np.float32)
    _split_calls(row1 - row0, lambda i0, i1: _lib.oracle_expert_slots_q4(
        T, d, E, k, F, _ptr(h), _ptr(q1), _ptr(b1), _ptr(s1), _ptr(q3), _ptr(b3), _ptr(s3), _ptr(q2), _ptr(b2),
        _ptr(s2), int(quant_act), _ptr(assign), _ptr(perm), row0 + i0, row0 + i1, _ptr(out[i0:i1])),
        "expert_slots_q4")
    return out
