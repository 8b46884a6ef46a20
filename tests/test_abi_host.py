"""Host-side checks of the C ABI that need no GPU: the library builds, loads
and exports every function include/lmoe.h declares; argument validation and
workspace sizing work without a device."""
import ctypes
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"LMOE_API\s+[\w\s\*]+?\b(lmoe_\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lm():
    import latent_moe_layer_fp32_gb300 as lm
    lm.build()
    lm.load()
    return lm


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ("lmoe_route", "lmoe_pool", "lmoe_experts_mxfp4", "lmoe_norm_combine_unpool", "lmoe_forward",
              "lmoe_workspace_bytes", "lmoe_status_check", "lmoe_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lm):
    lib = lm.load()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_error_strings(lm):
    for code in range(-6, 1):
        assert lm.lmoe_error_string(code)
    assert lm.lmoe_error_string(-99) == "unknown error"


def test_workspace_sizing_without_gpu(lm):
    for name, d in synth.CONFIGS.items():
        n = lm.lmoe_workspace_bytes(lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps))
        # at least the per-route fp32 rows and the bf16 intermediates
        assert n >= 4 * d.T * d.k * d.L + 2 * d.T * d.L, name
        lay = lm.lmoe_workspace_layout(lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps))
        assert lay.total == n
        offs = [lay.status, lay.topk_idx, lay.topk_w, lay.expert_offsets, lay.sorted_rows, lay.row_pos, lay.x_lat,
                lay.y, lay.z]
        assert all(o % 256 == 0 for o in offs) and len(set(offs)) == len(offs)
        assert lay.z + 2 * d.T * d.L <= n


def test_block_workspace_sizing_without_gpu(lm):
    for name, d in synth.CONFIGS.items():
        dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
        n, nb = lm.lmoe_workspace_bytes(dims), lm.lmoe_block_workspace_bytes(dims)
        # the layer's workspace plus the pre-norm output, the split router input and the layer output
        assert nb >= n + 2 * d.T * d.H + 4 * d.T * d.H + 2 * d.T * d.H, name
    assert lm.lmoe_block_workspace_bytes(lm.dims_of(0, 512, 256, 256, 16, 4, 1e-6)) == 0


def test_host_workspace_sizing_without_gpu(lm):
    for name, d in synth.CONFIGS.items():
        dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
        n, nh = lm.lmoe_workspace_bytes(dims), lm.lmoe_host_workspace_bytes(dims)
        # the layer's workspace plus a staging buffer for the tokens and one for the output, 256-byte aligned
        rows = 2 * d.T * d.H
        assert nh >= n + 2 * rows and nh <= n + 2 * rows + 3 * 256, name
    assert lm.lmoe_host_workspace_bytes(lm.dims_of(0, 512, 256, 256, 16, 4, 1e-6)) == 0


def test_host_forward_refuses_bad_arguments_without_gpu(lm):
    """Argument checks run before any device work: no workspace, null buffers."""
    d = synth.CONFIGS["tiny"]
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    lib = lm.load()
    w = lm.LmoeWeights()
    rc = lib.lmoe_forward_host(ctypes.byref(dims), ctypes.byref(w), None, None, None, 0, None)
    assert rc != 0


@pytest.mark.parametrize("field,value", [("T", 0), ("top_k", 9), ("top_k", 0), ("n_experts", 257),
                                         ("hidden", 100), ("latent", 96), ("inter", 0), ("eps", -1.0)])
def test_bad_dims_rejected(lm, field, value):
    d = synth.CONFIGS["tiny"]
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    setattr(dims, field, value)
    assert lm.lmoe_workspace_bytes(dims) == 0
    lib = lm.load()
    rc = lib.lmoe_forward(ctypes.byref(dims), None, None, None, None, 0, None)
    assert rc == -1


def test_unsupported_width(lm):
    # K is streamed in 2048-element chunks above 2048, and in 128-byte planes; a
    # group's activation rows (K <= 8192) sit in shared memory
    for h, l, i in [(8192, 2560, 4096), (8192, 4096, 3328), (8192 + 128, 4096, 4096), (8192, 10240, 4096),
                    (8192, 4096, 10240)]:
        assert lm.lmoe_workspace_bytes(lm.dims_of(1, h, l, i, 256, 8, 1e-6)) == 0
    assert lm.lmoe_workspace_bytes(lm.dims_of(1, 8192, 8192, 8192, 256, 8, 1e-6)) > 0


def test_regime_options_round_trip(lm):
    for key, default in ((lm.LMOE_OPT_DENSE_MIN_TOKENS, 64), (lm.LMOE_OPT_EXPERT_TC_MIN_TOKENS, 352)):
        prev = lm.lmoe_set_option(key, 7)
        assert prev == default
        assert lm.lmoe_set_option(key, 0) == 7  # 0 restores the default
        assert lm.lmoe_set_option(key, prev) == default
    with pytest.raises(lm.LmoeError):
        lm.lmoe_set_option(99, 1)


def test_launch_names_out_of_range(lm):
    assert lm.lmoe_last_launch_name(-1) is None
    assert lm.lmoe_last_launch_name(1 << 20) is None


def test_missing_library_fails_loudly(lm, tmp_path):
    """No CPU fallback: without the built library every entry point refuses to run."""
    import latent_moe_layer_fp32_gb300 as pkg
    saved = pkg._lib
    pkg._lib = None
    try:
        with pytest.raises(ImportError):
            pkg.load(str(tmp_path / "liblmoe.so"))
    finally:
        pkg._lib = saved
