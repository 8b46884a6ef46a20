"""GPU parity of the grouped tensor-core experts (tcgen05, weights dequantised
to bf16 in shared memory) against the oracle.

The regime switch forces the tensor-core path at token counts where the
oracle evaluates every row: the small layer at several T (ragged groups, one
expert over 256 rows so that its rows split into several groups) and the
full layer shape at T = 8 and 64, with and without skewed routing.  The
format check runs the kernels' dequantisation on every code byte under every
scale byte and compares it bit for bit with the oracle's MXFP4 values.
"""
from __future__ import annotations

import contextlib

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (check_out, check_rows_normwise, device_weights, host_weights, to_dev, to_host, ws_for,
                         ws_view)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import latent_moe_layer_fp32_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lm.load()
    return lm


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@contextlib.contextmanager
def experts_tc_from(lm, min_t):
    prev = lm.lmoe_set_option(lm.LMOE_OPT_EXPERT_TC_MIN_TOKENS, min_t)
    try:
        yield
    finally:
        lm.lmoe_set_option(lm.LMOE_OPT_EXPERT_TC_MIN_TOKENS, prev)


def dims_c(lm, d):
    return lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)


def test_dequant_matches_oracle_for_every_code_and_scale(lm, orc):
    # 256 scales x 16 blocks: block j of scale s holds the code bytes 16 j .. 16 j + 15,
    # so every byte value (two codes) meets every scale byte
    scales = np.repeat(np.arange(256, dtype=np.uint8), 16)
    codes = np.tile(np.arange(256, dtype=np.uint8), 256)
    out = torch.empty(scales.size * 32, dtype=torch.int16, device="cuda")
    lm.lmoe_selftest_dequant_bf16(to_dev(codes), to_dev(scales), out)
    got = to_host(out).view(np.uint16).reshape(-1, 32)
    want = np.empty_like(got)
    nan = np.zeros(got.shape, bool)
    for b in range(scales.size):
        s = int(scales[b])
        for i in range(32):
            byte = int(codes[16 * b + i // 2])
            code = (byte >> (4 * (i & 1))) & 15
            v = orc.mxfp4_value(code, s)
            nan[b, i] = np.isnan(v)
            want[b, i] = orc.bf16_rne(v)
    got_nan = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert np.array_equal(got_nan, nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert nan[scales == 255].all() and not nan[scales != 255].any()


CASES = [("tiny", 1), ("tiny", 17), ("tiny", 130), ("tiny", 300), ("tiny", 1100), ("verify_t8", None),
         ("verify_t8_skewed", None), ("batched_t64", None)]


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_tc_experts_stage_and_forward(lm, orc, name, T):
    d = synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    ref = orc.forward(d, x, hw)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    off, rows, _ = orc.table(d, ref["topk_idx"])
    if name == "tiny" and T == 1100:
        assert np.diff(off).max() > 256  # some expert spans more than one 256-row group
    y = torch.empty(d.T * d.k, d.L, dtype=torch.float32, device="cuda")
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    with experts_tc_from(lm, 1):
        lm.lmoe_experts_mxfp4(dims, to_dev(ref["x_lat"]), to_dev(off), to_dev(rows), w["w13_q"], w["w13_s"],
                              w["w2_q"], w["w2_s"], y, ws)
        names = [lm.lmoe_last_launch_name(i) for i in range(lm.lmoe_last_launch_count())]
        assert "expert_gateup_tc" in names and "expert_down_tc" in names, names
        assert lm.lmoe_status_check(ws) == 0
        check_rows_normwise(to_host(y), ref["y"], 2e-3, "y")
        lm.lmoe_forward(dims, lm.weights_of(w), to_dev(x), out, ws)
        assert lm.lmoe_status_check(ws) == 0
    from test_gpu_parity import check_out_routed
    from parity_util import check_indices, router_regime
    lay = lm.lmoe_workspace_layout(dims)
    got_idx = to_host(ws_view(ws, lay.topk_idx, torch.int32, (d.T, d.k)))
    got_w = to_host(ws_view(ws, lay.topk_w, torch.float32, (d.T, d.k)))
    logits, absdot = orc.router_logits(d, x, hw["router_w"], hw["router_bias"], want_absdot=True)
    _, differs = check_indices(d, got_idx, ref["topk_idx"], logits, absdot, regime=router_regime(d))
    # every token: tokens routed differently (near ties) against the oracle on the GPU's routing
    check_out_routed(orc, d, x, hw, to_host(out), ref["out"], differs, got_idx, got_w, "forward[tc experts]")
