"""Fused NVFP4 Mixture-of-Experts layer for GB300 (sm_103a): Python binding.

Thin ctypes marshalling over the C ABI in ``include/nvfp4_moe.h``; every step of the layer runs
in the library's CUDA kernels.  PyTorch only provides device memory and the current stream.  The
library must have been built (``__graft_entry__.build()``); there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvfp4moe.so")
_lib = None

MOE_OK = 0
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED_SHAPE",
          -3: "MOE_ERR_WORKSPACE_TOO_SMALL", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE_TIMEOUT",
          -6: "MOE_ERR_NONFINITE", -7: "MOE_ERR_UNIMPLEMENTED"}

EXPORTED = ["moe_status_string", "moe_config_check", "moe_weights_size", "moe_quantize_weights",
            "moe_weights_export", "moe_act_workspace_size", "moe_quantize_act",
            "moe_plan_workspace_size", "moe_plan", "moe_workspace_size", "moe_run",
            "moe_last_device_status", "moe_plan_static", "moe_run_kernel_count",
            "moe_set_router_bias", "moe_rmsnorm_workspace_size", "moe_rmsnorm_quantize_act",
            "moe_run_quantized"]


class MoeConfig(C.Structure):
    _fields_ = [("num_experts", C.c_int32), ("hidden", C.c_int32), ("inter", C.c_int32),
                ("top_k", C.c_int32), ("shared_inter", C.c_int32), ("h_tensor_scale", C.c_float),
                ("max_tokens", C.c_int32), ("flags", C.c_uint32), ("swiglu_limit", C.c_float),
                ("swiglu_alpha", C.c_float)]

    def __repr__(self):
        return (f"MoeConfig(E={self.num_experts}, H={self.hidden}, I={self.inter}, k={self.top_k}, "
                f"shared_inter={self.shared_inter}, ts_h={self.h_tensor_scale}, "
                f"max_tokens={self.max_tokens})")


# Stages between the library's stage events.  Small batches run the quantiser, router and plan
# as one fused kernel: its time is reported under "act_quant" and "router_plan" is then empty.
STAGES = ("act_quant", "router_plan", "gemm1_swiglu", "gemm2_combine", "bf16_out")
N_STAGE_EVENTS = len(STAGES) + 1


class MoeDebug(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("topk_ids", "topk_w", "counts", "offsets", "perm_src",
                                          "inv", "xq", "xsf", "ts_a", "hq", "hsf",
                                          "stage_events")] + [("inject", C.c_uint32),
                                                              ("hb", C.c_void_p)]


MOE_INJECT_NO_PLAN_FLAG = 1


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import "
                               "__graft_entry__ as g; g.build()')")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
        cfgp = C.POINTER(MoeConfig)
        sig = {
            "moe_status_string": (C.c_char_p, [C.c_int]),
            "moe_config_check": (C.c_int, [cfgp]),
            "moe_weights_size": (sz, [cfgp]),
            "moe_quantize_weights": (C.c_int, [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "moe_weights_export": (C.c_int, [cfgp, vp, i32, i32, vp, vp, vp, vp]),
            "moe_act_workspace_size": (sz, [i64, i64]),
            "moe_quantize_act": (C.c_int, [vp, i64, i64, vp, vp, vp, vp, sz, vp]),
            "moe_plan_workspace_size": (sz, [i32, i32, i32]),
            "moe_plan": (C.c_int, [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "moe_workspace_size": (sz, [cfgp, i32]),
            "moe_run": (C.c_int, [cfgp, vp, vp, vp, i32, i32, vp, vp, sz, vp, C.POINTER(MoeDebug)]),
            "moe_run_quantized": (C.c_int, [cfgp, vp, vp, vp, vp, vp, i32, i32, vp, vp, sz, vp,
                                            C.POINTER(MoeDebug)]),
            "moe_last_device_status": (C.c_int, [vp, C.POINTER(C.c_int32)]),
            "moe_plan_static": (C.c_int, [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]),
            "moe_run_kernel_count": (C.c_int, [cfgp, i32]),
            "moe_set_router_bias": (C.c_int, [cfgp, vp, vp, vp]),
            "moe_rmsnorm_workspace_size": (sz, [i64]),
            "moe_rmsnorm_quantize_act": (C.c_int, [vp, vp, C.c_float, i64, i64, vp, vp, vp, vp, vp, sz,
                                                   vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(st: int) -> str:
    return lib().moe_status_string(st).decode()


def _check(st: int, what: str):
    if st != MOE_OK:
        raise RuntimeError(f"{what} failed: {STATUS.get(st, st)} ({status_string(st)})")


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


FLAG_ROUTER_SQRTSOFTPLUS = 1
FLAG_SWIGLU_CLAMP = 2
FLAG_ACT_RELU2 = 4
FLAG_ACT_SWIGLU_OAI = 8
FLAG_ACT_BF16 = 16
FLAG_ACT_MXFP8 = 32
ACTIVATIONS = ("swiglu", "relu2", "swiglu_oai")


def make_config(num_experts, hidden, inter, top_k, shared_inter=0, h_tensor_scale=1.0,
                max_tokens=0, router="softmax", swiglu_limit=None, activation="swiglu",
                swiglu_alpha=1.702, precision="nvfp4") -> MoeConfig:
    """router: "softmax" (top-k of the logits, softmax over the k) or "sqrtsoftplus" (scores
    sqrt(softplus(logit)), selection on score + the bias set by set_router_bias, weights the
    normalised unbiased scores).  activation: "swiglu" (silu(g)*u, or with swiglu_limit L
    silu(min(g, L)) * clamp(u, -L, L)), "relu2" (non-gated experts, max(u, 0)^2) or "swiglu_oai"
    ((clamp(u, -L, L) + 1) * g' * sigmoid(alpha * g'), g' = min(g, L); needs swiglu_limit).
    precision: "nvfp4" (activations and h quantised to NVFP4), "w4a16" (BF16 activations as
    they are, weights decoded to BF16 in the GEMMs, h rounded to BF16) or "w4a8" (MXFP4 weights,
    MXFP8 activations and h)."""
    if router not in ("softmax", "sqrtsoftplus"):
        raise ValueError(f"unknown router {router!r}")
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}")
    if activation == "swiglu_oai" and swiglu_limit is None:
        raise ValueError("swiglu_oai needs swiglu_limit")
    flags = FLAG_ROUTER_SQRTSOFTPLUS if router == "sqrtsoftplus" else 0
    if activation == "relu2":
        flags |= FLAG_ACT_RELU2
    elif activation == "swiglu_oai":
        flags |= FLAG_ACT_SWIGLU_OAI
    elif swiglu_limit is not None:
        flags |= FLAG_SWIGLU_CLAMP
    if precision == "w4a16":
        flags |= FLAG_ACT_BF16
    elif precision == "w4a8":
        flags |= FLAG_ACT_MXFP8
    elif precision != "nvfp4":
        raise ValueError(f"unknown precision {precision!r}")
    return MoeConfig(num_experts, hidden, inter, top_k, shared_inter, h_tensor_scale, max_tokens,
                     flags, 0.0 if swiglu_limit is None else float(swiglu_limit),
                     float(swiglu_alpha))


def config_check(cfg: MoeConfig) -> int:
    return lib().moe_config_check(C.byref(cfg))


def weights_size(cfg: MoeConfig) -> int:
    return int(lib().moe_weights_size(C.byref(cfg)))


def quantize_weights(cfg: MoeConfig, w_gate, w_up, w_down, shared=None, wbuf=None, stream=None):
    """BF16 expert weights -> packed NVFP4 weight buffer (a uint8 CUDA tensor).  w_gate (and the
    shared expert's gate) may be None for non-gated (relu2) layers; they are not read there."""
    n = weights_size(cfg)
    if n == 0:
        _check(config_check(cfg), "moe_weights_size")
    if wbuf is None:
        wbuf = torch.empty(n, dtype=torch.uint8, device=w_up.device)
    sg, su, sd = shared if shared is not None else (None, None, None)
    _check(lib().moe_quantize_weights(C.byref(cfg), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                      _ptr(sg), _ptr(su), _ptr(sd), _ptr(wbuf), wbuf.numel(),
                                      _stream(stream)), "moe_quantize_weights")
    return wbuf


def set_router_bias(cfg: MoeConfig, wbuf: torch.Tensor, bias: torch.Tensor) -> None:
    """Stores the sqrt-softplus router's per-expert selection bias (FP32 [E]) in wbuf."""
    bias = bias.to(device=wbuf.device, dtype=torch.float32).contiguous()
    if bias.numel() != cfg.num_experts:
        raise ValueError("bias must have num_experts entries")
    _check(lib().moe_set_router_bias(C.byref(cfg), _ptr(wbuf), _ptr(bias), _stream()),
           "moe_set_router_bias")
    torch.cuda.current_stream().synchronize()


def weights_export(cfg: MoeConfig, wbuf, expert: int, matrix: int, stream=None):
    """Canonical (codes [N,K/2], sf [N,K/16] E4M3 - or [N,K/32] E8M0 for a W4A8 layer's MXFP4
    weights - and ts [1]) of one expert matrix (-1 = shared)."""
    Iw = cfg.shared_inter if expert == -1 else cfg.inter   # this expert's intermediate size
    N, K = (Iw, cfg.hidden) if matrix < 2 else (cfg.hidden, Iw)
    dev = wbuf.device
    codes = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(N, K // (32 if cfg.flags & FLAG_ACT_MXFP8 else 16), dtype=torch.uint8,
                     device=dev)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    _check(lib().moe_weights_export(C.byref(cfg), _ptr(wbuf), expert, matrix, _ptr(codes), _ptr(sf),
                                    _ptr(ts), _stream(stream)), "moe_weights_export")
    return codes, sf, ts


def quantize_act(x, workspace=None, stream=None):
    """x [rows, cols] BF16 -> (codes [rows, cols/2], sf [rows, cols/16], ts [1]) on the device."""
    rows, cols = x.shape
    dev = x.device
    codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(rows, cols // 16, dtype=torch.uint8, device=dev)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    nws = int(lib().moe_act_workspace_size(rows, cols))
    if workspace is None:
        workspace = torch.empty(nws, dtype=torch.uint8, device=dev)
    _check(lib().moe_quantize_act(_ptr(x), rows, cols, _ptr(codes), _ptr(sf), _ptr(ts),
                                  _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_quantize_act")
    return codes, sf, ts


def rmsnorm_quantize_act(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6,
                         workspace=None, stream=None, want_rrms: bool = False):
    """RMSNorm of BF16 x [rows, cols] by BF16 gamma [cols], then NVFP4 (codes, sf, ts) on the
    device (+ each row's 1/rms when want_rrms); a non-finite result is reported through the
    device status (last_device_status), not raised here."""
    rows, cols = x.shape
    dev = x.device
    codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(rows, cols // 16, dtype=torch.uint8, device=dev)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    rr = torch.empty(rows, dtype=torch.float32, device=dev) if want_rrms else None
    if workspace is None:
        workspace = torch.empty(lib().moe_rmsnorm_workspace_size(rows), dtype=torch.uint8,
                                device=dev)
    _check(lib().moe_rmsnorm_quantize_act(_ptr(x), _ptr(gamma), float(eps), rows, cols,
                                          _ptr(codes), _ptr(sf), _ptr(ts),
                                          _ptr(rr) if rr is not None else None, _ptr(workspace),
                                          workspace.numel(), _stream(stream)),
           "moe_rmsnorm_quantize_act")
    return (codes, sf, ts, rr) if want_rrms else (codes, sf, ts)


def plan(logits, k: int, workspace=None, stream=None):
    """Router top-k + permutation plan for logits [T, E] FP32 (dict of device tensors)."""
    T, E = logits.shape
    dev = logits.device
    out = dict(topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
               topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
               counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               perm_src=torch.empty(T * k, dtype=torch.int32, device=dev),
               inv=torch.empty(T * k, dtype=torch.int32, device=dev))
    nws = int(lib().moe_plan_workspace_size(T, E, k))
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
    _check(lib().moe_plan(_ptr(logits), T, E, k, _ptr(out["topk_ids"]), _ptr(out["topk_w"]),
                          _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm_src"]),
                          _ptr(out["inv"]), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_plan")
    return out


def plan_static(logits, k: int, out=None, stream=None):
    """moe_plan through moe_plan_static: no workspace argument, for callers that cannot
    allocate device memory (the library's static per-device scratch is used; calls on several
    streams at once race).  ``out`` may pass preallocated output tensors."""
    T, E = logits.shape
    dev = logits.device
    if out is None:
        out = dict(topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
                   topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
                   counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   perm_src=torch.empty(T * k, dtype=torch.int32, device=dev),
                   inv=torch.empty(T * k, dtype=torch.int32, device=dev))
    _check(lib().moe_plan_static(_ptr(logits), T, E, k, _ptr(out["topk_ids"]), _ptr(out["topk_w"]),
                                 _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm_src"]),
                                 _ptr(out["inv"]), _stream(stream)), "moe_plan_static")
    return out


def workspace_size(cfg: MoeConfig, T: int) -> int:
    return int(lib().moe_workspace_size(C.byref(cfg), T))


def run_kernel_count(cfg: MoeConfig, T: int) -> int:
    """Kernels one run() at T tokens launches (host arithmetic, no device needed)."""
    n = int(lib().moe_run_kernel_count(C.byref(cfg), T))
    if n < 0:
        raise RuntimeError(f"moe_run_kernel_count: {status_string(n)}")
    return n


class StageTimer:
    """CUDA events the library records on its launch stream between the layer's stages."""

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(N_STAGE_EVENTS)]
        for e in self.events:      # torch creates the CUDA event on its first record
            e.record()
        self._handles = (C.c_void_p * N_STAGE_EVENTS)(*[e.cuda_event for e in self.events])
        self.c_debug = MoeDebug(*([None] * 11), C.cast(self._handles, C.c_void_p))

    def stage_ms(self):
        """Milliseconds of each stage of the last recorded call (synchronise first)."""
        return {n: self.events[i].elapsed_time(self.events[i + 1]) for i, n in enumerate(STAGES)}


def run(cfg: MoeConfig, wbuf, x, logits, k=None, y=None, workspace=None, debug=False, stream=None,
        timer: StageTimer = None, quantized=None, inject: int = 0):
    """The layer: y [T, H] BF16 (and, with debug=True, a dict of its intermediates).  x is the BF16
    input [T, H]; or pass x=None and quantized=(xq [T, H/2] u8, xsf [T, H/16] u8, ts_a [1] f32),
    already-NVFP4 activations (moe_run_quantized)."""
    if quantized is not None:
        xq, xsf, ts_a = quantized
        T, H = xq.shape[0], xq.shape[1] * 2
        dev = xq.device
    else:
        T, H = x.shape
        dev = x.device
    k = cfg.top_k if k is None else k
    if y is None:
        y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = torch.empty(max(workspace_size(cfg, T), 256), dtype=torch.uint8, device=dev)
    dbg = None
    dbg_c = None
    if debug:
        # h rows are as wide as the layer's widest intermediate (a shared expert of another
        # width than the routed ones: the narrower rows end in zeros)
        E, I = cfg.num_experts, max(cfg.inter, cfg.shared_inter)
        Rt = T * k + (T if cfg.shared_inter else 0)
        dbg = dict(topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
                   topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
                   counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   perm_src=torch.empty(T * k, dtype=torch.int32, device=dev),
                   inv=torch.empty(T * k, dtype=torch.int32, device=dev),
                   xq=torch.empty(T, H // 2, dtype=torch.uint8, device=dev),
                   xsf=torch.empty(T, H // 16, dtype=torch.uint8, device=dev),
                   ts_a=torch.empty(1, dtype=torch.float32, device=dev),
                   hq=torch.empty(Rt, I // 2, dtype=torch.uint8, device=dev),
                   hsf=torch.empty(Rt, I // 16, dtype=torch.uint8, device=dev))
        if cfg.flags & FLAG_ACT_BF16:        # nothing is quantised; h stays BF16 (hb)
            for n in ("hq", "hsf", "xq", "xsf", "ts_a"):
                del dbg[n]
            dbg["hb"] = torch.empty(Rt, I, dtype=torch.bfloat16, device=dev)
        if cfg.flags & FLAG_ACT_MXFP8:       # MXFP8 codes + E8M0 scales of x and h, decoded h
            del dbg["ts_a"]
            dbg["xq"] = torch.empty(T, H, dtype=torch.uint8, device=dev)
            dbg["xsf"] = torch.empty(T, H // 32, dtype=torch.uint8, device=dev)
            dbg["hq"] = torch.empty(Rt, I, dtype=torch.uint8, device=dev)
            dbg["hsf"] = torch.empty(Rt, I // 32, dtype=torch.uint8, device=dev)
            dbg["hb"] = torch.empty(Rt, I, dtype=torch.bfloat16, device=dev)
        dbg_c = MoeDebug(*[dbg[n].data_ptr() if n in dbg else None
                           for n, _ in MoeDebug._fields_[:11]],
                         C.cast(timer._handles, C.c_void_p) if timer is not None else None)
        if "hb" in dbg:
            dbg_c.hb = dbg["hb"].data_ptr()
    elif timer is not None:
        dbg_c = timer.c_debug
    if inject:
        dbg_c = MoeDebug.from_buffer_copy(dbg_c) if dbg_c is not None else MoeDebug()
        dbg_c.inject = inject
    dptr = C.byref(dbg_c) if dbg_c is not None else None
    if quantized is not None:
        _check(lib().moe_run_quantized(C.byref(cfg), _ptr(wbuf), _ptr(xq), _ptr(xsf), _ptr(ts_a),
                                       _ptr(logits), T, k, _ptr(y), _ptr(workspace),
                                       workspace.numel(), _stream(stream), dptr),
               "moe_run_quantized")
    else:
        _check(lib().moe_run(C.byref(cfg), _ptr(wbuf), _ptr(x), _ptr(logits), T, k, _ptr(y),
                             _ptr(workspace), workspace.numel(), _stream(stream), dptr), "moe_run")
    return (y, dbg) if debug else y


def last_device_status(workspace) -> int:
    st = C.c_int32(0)
    _check(lib().moe_last_device_status(_ptr(workspace), C.byref(st)), "moe_last_device_status")
    return int(st.value)


class MoeLayer:
    """Packed weights + a reusable workspace for one layer shape."""

    def __init__(self, cfg: MoeConfig, w_gate, w_up, w_down, shared=None, max_tokens=None):
        self.cfg = cfg
        self.device = w_up.device          # w_gate is None for non-gated (relu2) experts
        self.wbuf = quantize_weights(cfg, w_gate, w_up, w_down, shared)
        self._ws = None
        self._ws_T = -1
        if max_tokens:
            self._ensure_ws(max_tokens)

    def _ensure_ws(self, T):
        if self._ws is None or T > self._ws_T:
            self._ws = torch.empty(max(workspace_size(self.cfg, T), 256), dtype=torch.uint8,
                                   device=self.device)
            self._ws_T = T
        return self._ws

    def __call__(self, x, logits, y=None, debug=False):
        ws = self._ensure_ws(x.shape[0])
        return run(self.cfg, self.wbuf, x, logits, y=y, workspace=ws, debug=debug)

    def status(self) -> int:
        return last_device_status(self._ws)
