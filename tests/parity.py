"""Shared helpers of the GPU parity tests: input construction and the comparison criteria.

Criteria (the layer's correctness contract):
  * router ids, permutation, offsets, quantised codes and block scales: bit-exact;
  * final output: relative L2 error <= 5e-3 and max |error| <= 3e-2 * RMS(reference);
  * requantised intermediate codes: at most 0.1% differ, each by one step of the ordered E2M1
    value list (+-0 counted as one value); block scales likewise at most 0.1%, one E4M3 step.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

Y_REL_L2 = 5e-3
Y_MAX_ABS_RMS = 3e-2
H_CODE_FRAC = 1e-3


def e2m1_rank(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int32)
    m = c & 7
    return np.where((c & 8) != 0, 7 - m, 7 + m)


def unpack_nibbles(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, np.uint8)
    return np.stack([b & 15, b >> 4], -1).reshape(b.shape[0], -1)


def compare_h(gpu_codes, gpu_sf, ref_codes, ref_sf):
    """Returns (fraction of differing codes, max step, fraction of differing scales, max step)."""
    gc, rc = unpack_nibbles(gpu_codes), unpack_nibbles(ref_codes)
    dr = np.abs(e2m1_rank(gc) - e2m1_rank(rc))
    # scales: E4M3 codes of non-negative values are ordered like their bytes
    ds = np.abs(gpu_sf.astype(np.int32) - ref_sf.astype(np.int32))
    return (float(np.mean(dr > 0)) if dr.size else 0.0, int(dr.max()) if dr.size else 0,
            float(np.mean(ds > 0)) if ds.size else 0.0, int(ds.max()) if ds.size else 0)


def assert_h_close(gpu_codes, gpu_sf, ref_codes, ref_sf):
    fc, mc, fs, ms = compare_h(gpu_codes, gpu_sf, ref_codes, ref_sf)
    assert fc <= H_CODE_FRAC and mc <= 1, f"h codes: {fc:.2e} differ, max step {mc}"
    assert fs <= H_CODE_FRAC and ms <= 1, f"h scales: {fs:.2e} differ, max step {ms}"


def y_errors(y_gpu_f32: np.ndarray, y_ref_f32: np.ndarray):
    yg = y_gpu_f32.astype(np.float64)
    yr = y_ref_f32.astype(np.float64)
    rel = np.linalg.norm(yg - yr) / max(np.linalg.norm(yr), 1e-30)
    rms = np.sqrt(np.mean(yr ** 2))
    return rel, np.abs(yg - yr).max() / max(rms, 1e-30)


def assert_y_close(y_gpu_f32, y_ref_f32):
    rel, mx = y_errors(y_gpu_f32, y_ref_f32)
    assert rel <= Y_REL_L2 and mx <= Y_MAX_ABS_RMS, f"y: rel_l2={rel:.3e} max/rms={mx:.3e}"
    return rel, mx


def bf16_to_np_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def stack_experts(cfg: synth.MoeConfig, device):
    """All routed experts generated directly on `device` (counter-based, identical values)."""
    return synth.gen_all_experts(cfg, device=device)


def oracle_experts_from(wg, wu, wd, ids=None):
    """Oracle-quantised experts from BF16 tensors [E,...]; only experts in `ids` (None = all)."""
    E = wg.shape[0]
    want = set(range(E)) if ids is None else set(int(i) for i in np.unique(ids))
    out = []
    for e in range(E):
        if e in want:
            out.append(oracle.QuantExpert.from_bf16(wg[e].cpu(), wu[e].cpu(), wd[e].cpu()))
        else:
            out.append(None)
    return out
