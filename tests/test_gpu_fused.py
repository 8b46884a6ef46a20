"""The persistent decode experts (gate/up + SwiGLU and down in one launch, a
device-wide hand-off between them) against the oracle and against the
two-launch streaming kernels: the same per-plane work and the same summation
order, so y is bit-identical between the two, and the layer output too."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check_out, check_rows_normwise, device_weights, host_weights, to_dev, to_host, ws_for

pytestmark = pytest.mark.gpu

CASES = [("tiny", 1), ("tiny", 4), ("tiny", 8), ("tiny", 16), ("decode_t1", None), ("verify_t4", None),
         ("verify_t8", None), ("verify_t8_skewed", None)]


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


def run_experts(lm, d, w, x_lat, off, rows, fused_max):
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    y = torch.full((d.T * d.k, d.L), float("nan"), dtype=torch.float32, device="cuda")
    prev = lm.lmoe_set_option(lm.LMOE_OPT_FUSED_MAX_TOKENS, fused_max)
    try:
        lm.lmoe_experts_mxfp4(dims, x_lat, off, rows, w["w13_q"], w["w13_s"], w["w2_q"], w["w2_s"], y, ws)
        names = [lm.lmoe_last_launch_name(i) for i in range(lm.lmoe_last_launch_count())]
        assert lm.lmoe_status_check(ws) == 0
    finally:
        lm.lmoe_set_option(lm.LMOE_OPT_FUSED_MAX_TOKENS, prev)
    return to_host(y), names


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_fused_experts_match_streaming_and_oracle(lm, orc, name, T):
    d = synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    ref = orc.forward(d, x, hw)
    off, rows, _ = orc.table(d, ref["topk_idx"])
    x_lat, off_d, rows_d = to_dev(ref["x_lat"]), to_dev(off), to_dev(rows)
    y_f, names_f = run_experts(lm, d, w, x_lat, off_d, rows_d, 8)
    y_s, names_s = run_experts(lm, d, w, x_lat, off_d, rows_d, 0)
    fused = d.T <= 8 and d.T * d.k <= 64
    assert ("expert_fused" in names_f) == fused, names_f
    assert "expert_fused" not in names_s and "expert_gateup" in names_s, names_s
    check_rows_normwise(y_f, ref["y"], 2e-3, "y (persistent experts)")
    assert np.array_equal(y_f.view(np.uint32), y_s.view(np.uint32)), "persistent and two-launch experts differ"
    # the whole layer through the persistent experts
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    prev = lm.lmoe_set_option(lm.LMOE_OPT_FUSED_MAX_TOKENS, 8)
    try:
        lm.lmoe_forward(dims, lm.weights_of(w), to_dev(x), out, ws)
        assert lm.lmoe_status_check(ws) == 0
        names = [lm.lmoe_last_launch_name(i) for i in range(lm.lmoe_last_launch_count())]
    finally:
        lm.lmoe_set_option(lm.LMOE_OPT_FUSED_MAX_TOKENS, prev)
    assert ("expert_fused" in names) == fused, names
    if fused:  # the norm and weighted sum run inside the persistent launch: no combine launch
        assert "combine_kernel" not in names, names
    check_out(to_host(out), ref["out"], "forward (persistent experts)")
    # the two-launch path gives the same bits (same sums in the same order)
    out2 = torch.empty_like(out)
    prev = lm.lmoe_set_option(lm.LMOE_OPT_FUSED_MAX_TOKENS, 0)
    try:
        lm.lmoe_forward(dims, lm.weights_of(w), to_dev(x), out2, ws)
        assert lm.lmoe_status_check(ws) == 0
    finally:
        lm.lmoe_set_option(lm.LMOE_OPT_FUSED_MAX_TOKENS, prev)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_fused_experts_repeat_calls(lm):
    """The device-wide counters live in the workspace and are zeroed by every
    call: back-to-back calls on one workspace give the same bits."""
    d = synth.CONFIGS["verify_t8"]
    w = device_weights(d)
    x = to_dev(synth.make_x(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    outs = []
    prev = lm.lmoe_set_option(lm.LMOE_OPT_FUSED_MAX_TOKENS, 8)
    try:
        for _ in range(3):
            o = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
            lm.lmoe_forward(dims, lm.weights_of(w), x, o, ws)
            outs.append(o)
    finally:
        lm.lmoe_set_option(lm.LMOE_OPT_FUSED_MAX_TOKENS, prev)
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
