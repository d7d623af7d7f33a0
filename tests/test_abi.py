"""The C-ABI library loads without a GPU, exports every function include/*.h declares, and rejects
bad arguments on the host before touching the device."""
import ctypes as C
import glob
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def moe():
    from nvfp4_mixture_experts_softmax_gb300 import _build
    _build.build()
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_symbols_exported(moe):
    names = declared_functions()
    assert "moe_run" in names and len(names) >= 12
    lib = C.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(moe.EXPORTED)


def test_status_strings(moe):
    for code in range(-7, 1):
        assert moe.status_string(code)
    assert moe.status_string(-99) == "unknown status"


@pytest.mark.parametrize("kw,want", [
    (dict(num_experts=8, hidden=256, inter=512, top_k=2), 0),
    (dict(num_experts=8, hidden=256, inter=512, top_k=9), -1),
    (dict(num_experts=0, hidden=256, inter=512, top_k=1), -1),
    (dict(num_experts=8, hidden=200, inter=512, top_k=2), -2),
    (dict(num_experts=8, hidden=256, inter=100, top_k=2), -2),
    (dict(num_experts=8, hidden=288, inter=160, top_k=2), 0),      # multiples of 32: padded
    (dict(num_experts=8, hidden=32, inter=32, top_k=2), 0),
    (dict(num_experts=8, hidden=2080, inter=1408, top_k=2, shared_inter=1408), 0),
    (dict(num_experts=8, hidden=2 ** 21, inter=256, top_k=2), -2),
    (dict(num_experts=2048, hidden=256, inter=256, top_k=2), -2),
    (dict(num_experts=64, hidden=256, inter=256, top_k=33), -2),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, shared_inter=256), 0),  # own width
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, shared_inter=96), 0),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, shared_inter=100), -2),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, h_tensor_scale=0.0), -1),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, h_tensor_scale=float("nan")), -1),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, router="sqrtsoftplus"), 0),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, swiglu_limit=10.0), 0),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, swiglu_limit=0.0), 0),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, swiglu_limit=-1.0), -1),
    (dict(num_experts=8, hidden=256, inter=512, top_k=2, swiglu_limit=float("inf")), -1),
])
def test_config_check(moe, kw, want):
    assert moe.config_check(moe.make_config(**kw)) == want


def test_sizes(moe):
    cfg = moe.make_config(128, 2048, 768, 8)
    # weights: per expert 3 * H * I * (1/2 + 1/16) bytes, plus the tensor scales
    assert moe.weights_size(cfg) >= 128 * 3 * 2048 * 768 * 9 // 16
    assert moe.weights_size(cfg) < 128 * 3 * 2048 * 768 * 9 // 16 + 4096
    assert moe.workspace_size(cfg, 64) > moe.workspace_size(cfg, 1) > 0
    assert moe.workspace_size(moe.make_config(8, 200, 512, 2), 4) == 0
    shared = moe.make_config(256, 7168, 2048, 8, shared_inter=2048)
    assert moe.weights_size(shared) > moe.weights_size(moe.make_config(256, 7168, 2048, 8))
    # widths that are multiples of 32 only run at the next multiples of 256: the packed weights
    # are those of the padded layer, the workspace adds the padded rows of x and of the output
    pad, full = moe.make_config(8, 288, 160, 2), moe.make_config(8, 512, 256, 2)
    assert moe.weights_size(pad) == moe.weights_size(full)
    assert moe.workspace_size(pad, 10) == moe.workspace_size(full, 10) + 2 * (10 * 512 * 2)
    # a shared expert of its own width: both intermediates at the larger one, rounded up
    assert (moe.weights_size(moe.make_config(8, 512, 256, 2, shared_inter=160)) ==
            moe.weights_size(moe.make_config(8, 512, 256, 2, shared_inter=256)))
    assert (moe.weights_size(moe.make_config(8, 512, 256, 2, shared_inter=640)) ==
            moe.weights_size(moe.make_config(8, 512, 768, 2, shared_inter=768)))


def test_host_side_rejections(moe):
    L = moe.lib()
    cfg = moe.make_config(8, 256, 512, 2)
    # null / undersized buffers are rejected before any device work
    assert L.moe_quantize_act(None, 4, 256, None, None, None, None, 0, None) == -3
    assert L.moe_quantize_act(None, 4, 250, None, None, None, None, 0, None) == -1
    assert L.moe_plan(None, 4, 8, 9, None, None, None, None, None, None, None, 0, None) == -1
    assert L.moe_plan(None, 4, 2048, 2, None, None, None, None, None, None, None, 0, None) == -2
    assert L.moe_run(C.byref(cfg), None, None, None, 4, 2, None, None, 0, None, None) == -1
    assert L.moe_run(C.byref(cfg), None, None, None, 4, 3, None, None, 0, None, None) == -1
    assert L.moe_quantize_weights(C.byref(cfg), None, None, None, None, None, None, None, 0, None) == -1
    assert L.moe_weights_export(C.byref(cfg), None, 0, 0, None, None, None, None) == -1
    st = C.c_int32(0)
    assert L.moe_last_device_status(None, C.byref(st)) == -1
    assert L.moe_plan_static(None, 4, 8, 9, None, None, None, None, None, None, None) == -1
    assert L.moe_plan_static(None, 1 << 24, 1024, 8, None, None, None, None, None, None, None) == -3


def test_run_kernel_count(moe):
    """The launch count follows moe_run's path choice: decode-sized batches take three kernels,
    other small batches five, large ones six (one-kernel plan) or eight (three-kernel plan)."""
    dec = moe.make_config(128, 2048, 768, 8, max_tokens=8192)
    assert [moe.run_kernel_count(dec, T) for T in (1, 8, 32, 64)] == [3, 3, 3, 3]
    assert moe.run_kernel_count(dec, 0) == 0
    assert moe.run_kernel_count(dec, 8192) == 8
    mid = moe.make_config(16, 2048, 256, 4, max_tokens=1024)
    assert moe.run_kernel_count(mid, 100) == 5     # fits the one-block prologue
    assert moe.run_kernel_count(mid, 500) == 6     # 2000 routed rows: one-kernel plan
    assert moe.run_kernel_count(mid, 600) == 8     # 2400 routed rows: three-kernel plan
    with pytest.raises(RuntimeError):
        moe.run_kernel_count(dec, -1)
    with pytest.raises(RuntimeError):
        moe.run_kernel_count(moe.make_config(8, 200, 512, 2), 4)


def test_variant_flags_and_bias_rejections(moe):
    cfg = moe.make_config(8, 256, 512, 2)
    cfg.flags = 64                                 # not a defined variant bit
    assert moe.config_check(cfg) == -1
    cfg.flags = 4 | 8                              # two activations at once
    assert moe.config_check(cfg) == -1
    cfg.flags = 8                                  # SwiGLU-OAI with a limit of 0 and alpha 1.702
    assert moe.config_check(cfg) == 0
    cfg.swiglu_limit = -1.0
    assert moe.config_check(cfg) == -1
    L = moe.lib()
    ok = moe.make_config(8, 256, 512, 2, router="sqrtsoftplus")
    assert L.moe_set_router_bias(C.byref(ok), None, None, None) == -1
    with pytest.raises(ValueError):
        moe.make_config(8, 256, 512, 2, router="sigmoid")
