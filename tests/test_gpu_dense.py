"""GPU parity of the dense projections (pooler H -> L, unpooler L -> H) in
both regimes: the weight-streaming kernel for a few tokens and the tcgen05
tensor-core GEMM for many.  Both are checked against the oracle on the same
inputs, at token counts that leave a ragged last 128-row tile, and the whole
layer is checked once with the tensor-core projections on the small shape.
"""
from __future__ import annotations

import contextlib
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import bf, check_bf16_close, check_out, device_weights, host_weights, sum_err, to_dev, to_host, ws_for

pytestmark = pytest.mark.gpu

TID_TEST_Y = 21
STREAM_ONLY = 1 << 30  # no token count reaches it: always the streaming kernel

CASES = [("tiny", 1), ("tiny", 37), ("tiny", 128), ("tiny", 130), ("tiny", 300), ("verify_t8", 130)]


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
def dense_from(lm, min_t):
    prev = lm.lmoe_set_option(lm.LMOE_OPT_DENSE_MIN_TOKENS, min_t)
    try:
        yield
    finally:
        lm.lmoe_set_option(lm.LMOE_OPT_DENSE_MIN_TOKENS, prev)


def dims_c(lm, d):
    return lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)


@pytest.mark.parametrize("regime", ["stream", "tensor"])
@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_projections(lm, orc, name, T, regime):
    d = synth.with_tokens(synth.CONFIGS[name], T)
    hw = host_weights(d)
    w = device_weights(d)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    x = synth.make_x(d)
    # the routing the unpool stage needs comes from the oracle
    logits = orc.router_logits(d, x, hw["router_w"], hw["router_bias"])
    idx, tw = orc.topk(d, logits)
    yy = synth.normal_f32(0, TID_TEST_Y, (T * d.k, d.L), 0.0, 1.0)
    with dense_from(lm, 1 if regime == "tensor" else STREAM_ONLY):
        x_lat = torch.empty(T, d.L, dtype=torch.bfloat16, device="cuda")
        lm.lmoe_pool(dims, to_dev(x), w["pooler_w"], x_lat, ws)
        out = torch.empty(T, d.H, dtype=torch.bfloat16, device="cuda")
        lm.lmoe_norm_combine_unpool(dims, to_dev(yy), to_dev(idx), to_dev(tw), w["norm_g"], w["unpooler_w"], out, ws)
        assert lm.lmoe_status_check(ws) == 0
    check_bf16_close(to_host(x_lat), orc.pool(d, x, hw["pooler_w"]), "x_lat",
                     sum_err(d.H, np.abs(bf(x)), np.abs(bf(hw["pooler_w"]))))
    z = orc.norm_combine(d, yy, idx, tw, hw["norm_g"])
    check_out(to_host(out), orc.unpool(d, z, hw["unpooler_w"]), f"unpool[{regime}]")


@pytest.mark.parametrize("T", [130, 300])
def test_forward_tensor_projections(lm, orc, T):
    d = synth.with_tokens(synth.CONFIGS["tiny"], T)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    ref = orc.forward(d, x, hw)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    out = torch.empty(T, d.H, dtype=torch.bfloat16, device="cuda")
    with dense_from(lm, 1):
        lm.lmoe_forward(dims, lm.weights_of(w), to_dev(x), out, ws)
        assert lm.lmoe_status_check(ws) == 0
    check_out(to_host(out), ref["out"], "forward[tensor]")


def test_regimes_agree_on_rounding(lm):
    """Both regimes round fp32 dot products to bf16 and differ only in the
    summation order: within one bf16 ulp plus both orders' error bound, and
    identical on nearly every element."""
    d = synth.with_tokens(synth.CONFIGS["verify_t8"], 256)
    hw = host_weights(d)
    w = device_weights(d)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    x = synth.make_x(d)
    x_dev = to_dev(x)
    res = {}
    for regime, min_t in (("stream", STREAM_ONLY), ("tensor", 1)):
        x_lat = torch.empty(d.T, d.L, dtype=torch.bfloat16, device="cuda")
        with dense_from(lm, min_t):
            lm.lmoe_pool(dims, x_dev, w["pooler_w"], x_lat, ws)
        res[regime] = to_host(x_lat)
    bound = 2.0 * sum_err(d.H, np.abs(bf(x)), np.abs(bf(hw["pooler_w"])))
    check_bf16_close(res["tensor"], res["stream"], "tensor vs stream", bound, frac=0.05)


ROUTE_CASES = [("tiny_e32", 200), ("tiny_e32", 1000), ("verify_t8", 300)]


@pytest.mark.parametrize("regime", ["stream", "tensor"])
@pytest.mark.parametrize("name,T", ROUTE_CASES, ids=[f"{n}_T{t}" for n, t in ROUTE_CASES])
def test_router_regimes(lm, orc, name, T, regime):
    """The router's logits on CUDA cores (fp32 FMA) or on the tensor cores
    (x against the three bf16 parts of the fp32 weights, split-K): both give
    the oracle's top-k outside near ties and its renormalised weights."""
    from test_gpu_parity import check_route, run_route
    base = dataclasses.replace(synth.CONFIGS["tiny"], E=32) if name == "tiny_e32" else synth.CONFIGS[name]
    d = synth.with_tokens(base, T)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    with dense_from(lm, 1 if regime == "tensor" else STREAM_ONLY):
        got = run_route(lm, d, to_dev(x), w)
        names = [lm.lmoe_last_launch_name(i) for i in range(lm.lmoe_last_launch_count())]
    assert ("router_tc_gemm" in names) == (regime == "tensor"), names
    check_route(orc, d, x, hw, got, regime="tensor" if regime == "tensor" else "simt",
                label=f"{name} T={T} {regime} router")
