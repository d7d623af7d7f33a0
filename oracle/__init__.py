"""ctypes wrapper around the C++ oracle of the NVFP4 MoE layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the product library never does, and the two share no code.
Every function here only marshals numpy arrays into the C routines of ``moe_oracle.cpp``.

The source builds twice: ``liboracle_moe.so`` (single-threaded, the oracle proper) and, where the
compiler has OpenMP, ``liboracle_moe_omp.so`` (the same loops spread over independent experts,
rows and tokens; identical bits).  ``use_threads(n)`` routes later calls to the second build.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle_moe.so")
_OMP_PATH = os.path.join(_HERE, "liboracle_moe_omp.so")
_libs = {}          # path -> loaded library
_active = _LIB_PATH


def _compile(path: str, extra) -> bool:
    if os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return True
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           *extra, "-o", tmp, _SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if not extra:
            raise RuntimeError(f"oracle build failed:\n{r.stderr}")
        return False
    os.replace(tmp, path)
    return True


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (-ffp-contract=off: no fused multiply-add anywhere), once
    single-threaded and once with OpenMP (skipped where the compiler has none)."""
    if force:
        for p in (_LIB_PATH, _OMP_PATH):
            if os.path.exists(p):
                os.remove(p)
    _compile(_LIB_PATH, [])
    _compile(_OMP_PATH, ["-fopenmp"])
    return _LIB_PATH


def use_threads(n) -> int:
    """Route later oracle calls to the OpenMP build with n threads (n = None or 0: all host cores;
    n = 1: the single-threaded build).  Returns the thread count in use."""
    global _active
    build()
    if n == 1 or not os.path.exists(_OMP_PATH):
        _active = _LIB_PATH
        return 1
    _active = _OMP_PATH
    L = lib()
    L.orc_set_threads(int(n or 0))
    return int(L.orc_threads())


class Expert(C.Structure):
    _fields_ = [("codes", C.c_void_p * 3), ("sf", C.c_void_p * 3), ("ts", C.c_float * 3)]


class MoeArgs(C.Structure):
    _fields_ = [("T", C.c_int64), ("H", C.c_int32), ("I", C.c_int32), ("E", C.c_int32),
                ("k", C.c_int32), ("has_shared", C.c_int32), ("I_shared", C.c_int32),
                ("ts_h", C.c_float), ("xq", C.c_void_p), ("xsf", C.c_void_p), ("ts_a", C.c_float),
                ("logits", C.c_void_p), ("experts", C.c_void_p), ("y", C.c_void_p),
                ("ids", C.c_void_p), ("w", C.c_void_p), ("counts", C.c_void_p),
                ("offsets", C.c_void_p), ("perm_src", C.c_void_p), ("inv", C.c_void_p),
                ("hq", C.c_void_p), ("hsf", C.c_void_p), ("shq", C.c_void_p), ("shsf", C.c_void_p),
                ("router_mode", C.c_int32), ("router_bias", C.c_void_p),
                ("swiglu_clamp", C.c_int32), ("swiglu_limit", C.c_float),
                ("act_mode", C.c_int32), ("x_bf16", C.c_void_p), ("hb", C.c_void_p),
                ("shb", C.c_void_p), ("hf", C.c_void_p), ("act_kind", C.c_int32),
                ("swiglu_alpha", C.c_float)]


# activation of the expert: SwiGLU (optionally clamped), non-gated squared ReLU, gpt-oss SwiGLU
ACT_KINDS = {"swiglu": 0, "relu2": 1, "swiglu_oai": 2}


ROUTER_MODES = {"softmax": 0, "sqrtsoftplus": 1}
# activation precision of the layer: NVFP4 activations with h requantised to NVFP4, W4A16 (BF16
# activations as they are, h rounded to BF16) or W4A8 (MXFP8 activations and h, MXFP4 weights)
ACT_MODES = {"nvfp4": 0, "bf16": 1, "mxfp8": 2}


def lib():
    if _active not in _libs:
        build()
        L = C.CDLL(_active)
        L.orc_set_threads.restype = None
        L.orc_set_threads.argtypes = [C.c_int]
        L.orc_threads.restype = C.c_int
        L.orc_threads.argtypes = []
        L.orc_bf16_to_f32.restype = C.c_float
        L.orc_bf16_to_f32.argtypes = [C.c_uint16]
        L.orc_f32_to_bf16.restype = C.c_uint16
        L.orc_f32_to_bf16.argtypes = [C.c_float]
        L.orc_e2m1_decode.restype = C.c_float
        L.orc_e2m1_decode.argtypes = [C.c_uint8]
        L.orc_e2m1_encode.restype = C.c_uint8
        L.orc_e2m1_encode.argtypes = [C.c_float]
        L.orc_e4m3_decode.restype = C.c_float
        L.orc_e4m3_decode.argtypes = [C.c_uint8]
        L.orc_e4m3_encode.restype = C.c_uint8
        L.orc_e4m3_encode.argtypes = [C.c_float]
        L.orc_quantize_f32.restype = None
        L.orc_quantize_f32.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_float, C.c_void_p, C.c_void_p]
        L.orc_tensor_scale_bf16.restype = C.c_float
        L.orc_tensor_scale_bf16.argtypes = [C.c_void_p, C.c_int64]
        L.orc_quantize_bf16.restype = C.c_int
        L.orc_quantize_bf16.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]
        L.orc_dequantize.restype = None
        L.orc_dequantize.argtypes = [C.c_void_p, C.c_void_p, C.c_float, C.c_int64, C.c_int64, C.c_void_p]
        L.orc_e8m0_decode.restype = C.c_float
        L.orc_e8m0_decode.argtypes = [C.c_uint8]
        L.orc_mx_scale.restype = C.c_uint8
        L.orc_mx_scale.argtypes = [C.c_float, C.c_int]
        L.orc_mx_quantize_f32.restype = None
        L.orc_mx_quantize_f32.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_int, C.c_void_p,
                                          C.c_void_p]
        L.orc_mx_dequantize.restype = None
        L.orc_mx_dequantize.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_int,
                                        C.c_void_p]
        L.orc_router.restype = None
        L.orc_router.argtypes = [C.c_void_p, C.c_int64, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.orc_router_ex.restype = None
        L.orc_router_ex.argtypes = [C.c_void_p, C.c_int64, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                    C.c_void_p, C.c_void_p]
        L.orc_sqrt_softplus.restype = C.c_float
        L.orc_sqrt_softplus.argtypes = [C.c_float]
        L.orc_sum_squares.restype = C.c_float
        L.orc_sum_squares.argtypes = [C.c_void_p, C.c_int64]
        L.orc_rmsnorm_quantize.restype = C.c_int
        L.orc_rmsnorm_quantize.argtypes = [C.c_void_p, C.c_void_p, C.c_float, C.c_int64, C.c_int64,
                                           C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                           C.c_void_p]
        L.orc_swiglu.restype = C.c_float
        L.orc_swiglu.argtypes = [C.c_float, C.c_float, C.c_int, C.c_float]
        L.orc_activation.restype = C.c_float
        L.orc_activation.argtypes = [C.c_float, C.c_float, C.c_int, C.c_int, C.c_float, C.c_float]
        L.orc_plan.restype = None
        L.orc_plan.argtypes = [C.c_void_p, C.c_int64, C.c_int, C.c_int] + [C.c_void_p] * 4
        L.orc_moe_forward.restype = C.c_int
        L.orc_moe_forward.argtypes = [C.POINTER(MoeArgs)]
        L.orc_moe_forward_bruteforce.restype = C.c_int
        L.orc_moe_forward_bruteforce.argtypes = [C.POINTER(MoeArgs)]
        _libs[_active] = L
    return _libs[_active]


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------------------- scalar codecs
def e2m1_decode(code: int) -> float:
    return float(lib().orc_e2m1_decode(code))


def e2m1_encode(q: float) -> int:
    return int(lib().orc_e2m1_encode(q))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(code))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(v))


def f32_to_bf16_bits(v: float) -> int:
    return int(lib().orc_f32_to_bf16(v))


# ----------------------------------------------------------------------------- quantisation
def as_bf16_bits(x) -> np.ndarray:
    """A torch BF16 tensor or a uint16 array -> contiguous uint16 bit patterns."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint16))


def quantize_bf16(x):
    """BF16 [rows, cols] -> (codes uint8 [rows, cols/2], sf uint8 [rows, cols/16], ts float, status)."""
    xb = as_bf16_bits(x)
    rows, cols = xb.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    ts = C.c_float(0)
    st = lib().orc_quantize_bf16(_p(xb), rows, cols, _p(codes), _p(sf), C.byref(ts))
    return codes, sf, float(np.float32(ts.value)), st


def quantize_f32(x: np.ndarray, ts: float):
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    lib().orc_quantize_f32(_p(x), rows, cols, ts, _p(codes), _p(sf))
    return codes, sf


def tensor_scale_bf16(x) -> float:
    xb = as_bf16_bits(x)
    return float(np.float32(lib().orc_tensor_scale_bf16(_p(xb), xb.size)))


def rmsnorm_quantize(x, gamma, eps: float, want_r: bool = False):
    """RMSNorm of BF16 x [rows, cols] with BF16 gamma [cols] (FP32 arithmetic; the sum of squares
    accumulated in float64 and rounded once to FP32), then NVFP4 with the tensor scale of the
    normalised values.  Returns (codes, sf, ts, status, y) with y the FP32 normalised values, and
    each row's 1/rms as a sixth item when want_r is set."""
    xb = as_bf16_bits(x)
    gb = np.ascontiguousarray(as_bf16_bits(gamma).reshape(-1))
    rows, cols = xb.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    ts = np.zeros(1, np.float32)
    y = np.zeros((rows, cols), np.float32)
    r = np.zeros(rows, np.float32)
    st = lib().orc_rmsnorm_quantize(_p(xb), _p(gb), float(eps), rows, cols, _p(codes), _p(sf),
                                    _p(ts), _p(y), _p(r))
    out = (codes, sf, float(ts[0]), int(st), y)
    return out + (r,) if want_r else out


def sum_squares(v) -> float:
    """The mean-square numerator of rmsnorm_quantize: the squares summed in float64, rounded once
    to FP32."""
    v = np.ascontiguousarray(v, np.float32)
    return float(lib().orc_sum_squares(_p(v), v.size))


def dequantize(codes: np.ndarray, sf: np.ndarray, ts: float) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((rows, cols), np.float32)
    lib().orc_dequantize(_p(codes), _p(sf), ts, rows, cols, _p(out))
    return out


# ----------------------------------------------------------------------------- MX formats
MX_KINDS = {"e4m3": 0, "e2m1": 1}   # MXFP8 / MXFP4 elements


def e8m0_decode(b: int) -> float:
    return float(lib().orc_e8m0_decode(b))


def mx_scale(amax: float, emax: int) -> int:
    return int(lib().orc_mx_scale(amax, emax))


def mx_quantize(x: np.ndarray, kind: str):
    """MX quantisation of FP32 rows [rows, cols] (cols % 32 == 0): element codes (E4M3: one byte
    each, [rows, cols]; E2M1: two per byte, [rows, cols/2]) and E8M0 scales [rows, cols/32]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    codes = np.zeros((rows, cols if kind == "e4m3" else cols // 2), np.uint8)
    sc = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_mx_quantize_f32(_p(x), rows, cols, MX_KINDS[kind], _p(codes), _p(sc))
    return codes, sc


def mx_dequantize(codes: np.ndarray, scales: np.ndarray, kind: str) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    rows = codes.shape[0]
    cols = codes.shape[1] if kind == "e4m3" else codes.shape[1] * 2
    out = np.zeros((rows, cols), np.float32)
    lib().orc_mx_dequantize(_p(codes), _p(scales), rows, cols, MX_KINDS[kind], _p(out))
    return out


# ----------------------------------------------------------------------------- routing
def router(logits: np.ndarray, k: int, mode: str = "softmax", bias=None):
    """Top-k routing.  mode "softmax": selection on the logits, softmax weights renormalised over
    the k; "sqrtsoftplus": scores sqrt(softplus(logit)), selection on score + bias (bias [E] or
    None), weights = chosen unbiased scores / their sum."""
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    lib().orc_router_ex(_p(logits), T, E, k, ROUTER_MODES[mode], _p(b) if b is not None else None,
                        _p(ids), _p(w))
    return ids, w


def sqrt_softplus(x: float) -> float:
    return float(lib().orc_sqrt_softplus(float(x)))


def swiglu(g: float, u: float, limit=None) -> float:
    """silu(g) * u, or silu(min(g, L)) * clamp(u, -L, L) with limit L."""
    return float(lib().orc_swiglu(float(g), float(u), 0 if limit is None else 1,
                                  0.0 if limit is None else float(limit)))


def activation(g: float, u: float, kind: str = "swiglu", limit=None, alpha: float = 1.702) -> float:
    """One feature of h from its gate and up values: "swiglu" silu(g) * u (clamped with limit),
    "relu2" max(u, 0)^2 (g unused), "swiglu_oai" (clamp(u, -L, L) + 1) * g' * sigmoid(alpha * g'),
    g' = min(g, L)."""
    return float(lib().orc_activation(float(g), float(u), ACT_KINDS[kind],
                                      0 if limit is None else 1,
                                      0.0 if limit is None else float(limit), float(alpha)))


def plan(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, np.int32)
    T, k = ids.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm_src = np.zeros(T * k, np.int32)
    inv = np.zeros(T * k, np.int32)
    lib().orc_plan(_p(ids), T, E, k, _p(counts), _p(offsets), _p(perm_src), _p(inv))
    return counts, offsets, perm_src, inv


# ----------------------------------------------------------------------------- the layer
class QuantExpert:
    """Canonical NVFP4 weights of one expert: gate/up [I,H], down [H,I] codes + scales + ts."""

    def __init__(self, codes, sf, ts):
        self.codes = [None if c is None else np.ascontiguousarray(c, np.uint8) for c in codes]
        self.sf = [None if s is None else np.ascontiguousarray(s, np.uint8) for s in sf]
        self.ts = [float(t) for t in ts]

    @classmethod
    def from_bf16(cls, gate, up, down):
        """gate may be None (a non-gated ReLU2 expert)."""
        cs, ss, ts = [], [], []
        for w in (gate, up, down):
            if w is None:
                cs.append(None), ss.append(None), ts.append(0.0)
                continue
            c, s, t, st = quantize_bf16(w)
            if st != 0:
                raise ValueError("non-finite weight")
            cs.append(c), ss.append(s), ts.append(t)
        return cls(cs, ss, ts)


class QuantExpertMX(QuantExpert):
    """MXFP4 weights of one expert (the W4A8 layer): gate/up [I,H], down [H,I] E2M1 codes [N, K/2]
    + E8M0 scales [N, K/32]; no tensor scale (ts = 1)."""

    @classmethod
    def from_bf16(cls, gate, up, down):
        """gate may be None (a non-gated ReLU2 expert)."""
        cs, ss = [], []
        for w in (gate, up, down):
            if w is None:
                cs.append(None), ss.append(None)
                continue
            wf = (np.asarray(as_bf16_bits(w), np.uint32) << 16).view(np.float32)
            c, s = mx_quantize(wf, "e2m1")
            cs.append(c), ss.append(s)
        return cls(cs, ss, [1.0, 1.0, 1.0])


def moe_forward(xq, xsf, ts_a, logits, experts, k, ts_h=1.0, shared=None, bruteforce=False,
                want_debug=False, router_mode="softmax", router_bias=None, swiglu_limit=None,
                act="nvfp4", x_bf16=None, activation="swiglu", swiglu_alpha=1.702):
    """The layer on quantised activations.  ``experts`` is a list of length E whose entries are
    QuantExpert or None (None only for experts no token routes to); ``shared`` a QuantExpert.
    ``router_mode``/``router_bias``: see router(); ``swiglu_limit``: None for plain SwiGLU, else
    the clamp limit L of silu(min(g, L)) * clamp(u, -L, L).  ``act="bf16"`` is the W4A16 layer:
    ``x_bf16`` (BF16 bits or a bfloat16 tensor [T, H]) enters GEMM1 as it is (xq, xsf and ts_a
    are then unused and may be None) and h is rounded to BF16; its debug output holds ``hb`` (and
    ``shb``) instead of the NVFP4 codes.  Debug output ``hf``: h in FP32 before its rounding or
    requantisation (routed rows, permuted order).  ``act="mxfp8"`` is the W4A8 layer: x_bf16 is
    quantised to MXFP8, ``experts`` / ``shared`` are QuantExpertMX (MXFP4), h is requantised to
    MXFP8 (debug ``hq`` [rows, I] E4M3 codes, ``hsf`` [rows, I/32] E8M0 scales).
    ``activation``: "swiglu" (clamped by swiglu_limit when given), "relu2" (non-gated experts:
    their gate entries are None) or "swiglu_oai" (limit swiglu_limit, slope swiglu_alpha)."""
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    if act in ("bf16", "mxfp8"):
        xb = np.ascontiguousarray(as_bf16_bits(x_bf16), np.uint16)
        H = xb.shape[1]
        xq = np.zeros((T, H // 2), np.uint8)
        xsf = np.zeros((T, H // 16), np.uint8)
        ts_a = 0.0
    else:
        xb = None
        xq = np.ascontiguousarray(xq, np.uint8)
        xsf = np.ascontiguousarray(xsf, np.uint8)
        H = xq.shape[1] * 2
    I = None
    for ex in experts:
        if ex is not None:
            I = ex.codes[1].shape[0]
            break
    if I is None:
        I = 16
    Is = shared.codes[1].shape[0] if shared is not None else 0
    table = (Expert * (E + (1 if shared is not None else 0)))()
    keep = []
    for i, ex in enumerate(list(experts) + ([shared] if shared is not None else [])):
        if ex is None:
            continue
        for m in range(3):
            table[i].codes[m] = _p(ex.codes[m])
            table[i].sf[m] = _p(ex.sf[m])
            table[i].ts[m] = ex.ts[m]
        keep.append(ex)
    y = np.zeros((T, H), np.uint16)
    a = MoeArgs()
    a.T, a.H, a.I, a.E, a.k = T, H, I, E, k
    a.has_shared = 1 if shared is not None else 0
    a.I_shared = Is
    a.ts_h = ts_h
    a.xq, a.xsf, a.ts_a = _p(xq), _p(xsf), ts_a
    a.logits = _p(logits)
    a.experts = C.cast(table, C.c_void_p)
    a.y = _p(y)
    a.router_mode = ROUTER_MODES[router_mode]
    rb = None if router_bias is None else np.ascontiguousarray(router_bias, np.float32)
    a.router_bias = _p(rb) if rb is not None else None
    a.swiglu_clamp = 0 if swiglu_limit is None else 1
    a.swiglu_limit = 0.0 if swiglu_limit is None else float(swiglu_limit)
    a.act_kind = ACT_KINDS[activation]
    a.swiglu_alpha = float(swiglu_alpha)
    if activation == "swiglu_oai" and swiglu_limit is None:
        raise ValueError("swiglu_oai needs swiglu_limit")
    a.act_mode = ACT_MODES[act]
    a.x_bf16 = _p(xb) if xb is not None else None
    dbg = {}
    if want_debug and not bruteforce:
        dbg = dict(ids=np.zeros((T, k), np.int32), w=np.zeros((T, k), np.float32),
                   counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
                   perm_src=np.zeros(T * k, np.int32), inv=np.zeros(T * k, np.int32),
                   hf=np.zeros((T * k, I), np.float32))
        if act == "bf16":
            dbg["hb"] = np.zeros((T * k, I), np.uint16)
            if shared is not None:
                dbg["shb"] = np.zeros((T, Is), np.uint16)
        elif act == "mxfp8":
            dbg["hq"] = np.zeros((T * k, I), np.uint8)
            dbg["hsf"] = np.zeros((T * k, I // 32), np.uint8)
            if shared is not None:
                dbg["shq"] = np.zeros((T, Is), np.uint8)
                dbg["shsf"] = np.zeros((T, Is // 32), np.uint8)
        else:
            dbg["hq"] = np.zeros((T * k, I // 2), np.uint8)
            dbg["hsf"] = np.zeros((T * k, I // 16), np.uint8)
            if shared is not None:
                dbg["shq"] = np.zeros((T, Is // 2), np.uint8)
                dbg["shsf"] = np.zeros((T, Is // 16), np.uint8)
        for name, arr in dbg.items():
            setattr(a, name, _p(arr))
    fn = lib().orc_moe_forward_bruteforce if bruteforce else lib().orc_moe_forward
    st = fn(C.byref(a))
    if st != 0:
        raise RuntimeError(f"oracle status {st}")
    return (y, dbg) if want_debug else y


def bf16_bits_to_f32(y: np.ndarray) -> np.ndarray:
    return (np.asarray(y, np.uint32) << 16).view(np.float32)
