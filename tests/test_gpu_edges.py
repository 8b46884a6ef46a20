"""Edge cases of the layer against the CPU oracle: the widest latent and
intermediate widths the decode kernels hold (8192: the activation panel and
the ring at their limits), degenerate routing (top-1; every expert selected),
and the largest token count the library accepts (65536)."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check_out, to_dev, to_host, ws_for

pytestmark = pytest.mark.gpu

WIDE = synth.Dims(T=4, H=512, L=8192, I=8192, E=16, k=4)


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


def run_forward(lm, d, w, x, nvfp4=False):
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    wd = {k: (None if v is None else to_dev(v)) for k, v in w.items()}
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    if nvfp4:
        lm.lmoe_forward_nvfp4(dims, lm.weights_of(wd), lm.nvfp4_of(wd), to_dev(x), out, ws)
    else:
        lm.lmoe_forward(dims, lm.weights_of(wd), to_dev(x), out, ws)
    assert lm.lmoe_status_check(ws) == 0
    lay = lm.lmoe_workspace_layout(dims)
    idx = ws[lay.topk_idx:lay.topk_idx + 4 * d.T * d.k].view(torch.int32).cpu().numpy().reshape(d.T, d.k)
    return to_host(out), idx


@pytest.mark.parametrize("nvfp4", [False, True], ids=["mxfp4", "nvfp4"])
@pytest.mark.parametrize("T", [1, 4, 37])
def test_widest_expert_widths(lm, orc, T, nvfp4):
    """latent = inter = 8192: each activation row fills a 16 KB panel row and,
    for several-row groups, the ring keeps only its minimum of two slots."""
    d = synth.with_tokens(WIDE, T)
    w = synth.make_weights_nvfp4(d) if nvfp4 else synth.make_weights(d)
    x = synth.make_x(d)
    ref = orc.forward_nvfp4(d, x, w) if nvfp4 else orc.forward(d, x, w)
    out, idx = run_forward(lm, d, w, x, nvfp4)
    assert np.array_equal(idx, ref["topk_idx"])
    check_out(out, ref["out"], f"out (L = I = 8192, {'NVFP4' if nvfp4 else 'MXFP4'})")


DEGENERATE = [(16, 1, 4), (16, 1, 37), (8, 8, 4), (8, 8, 37), (32, 1, 600), (8, 8, 600)]


@pytest.mark.parametrize("E,k,T", DEGENERATE, ids=[f"E{e}_k{k}_T{t}" for e, k, t in DEGENERATE])
def test_degenerate_routing(lm, orc, E, k, T):
    """Top-1 (each token's weight is exactly 1) and k = E (every expert takes
    every token, the weights are the full softmax) in the decode and the
    tensor-core regimes."""
    d = dataclasses.replace(synth.CONFIGS["tiny"], T=T, E=E, k=k)
    w = synth.make_weights(d)
    x = synth.make_x(d)
    ref = orc.forward(d, x, w)
    if k == 1:
        assert np.all(ref["topk_w"] == 1.0)
    if k == E:
        assert np.array_equal(np.sort(ref["topk_idx"], axis=1), np.tile(np.arange(E), (T, 1)))
    out, idx = run_forward(lm, d, w, x)
    assert np.array_equal(idx, ref["topk_idx"])
    check_out(out, ref["out"], f"out (E={E}, k={k})")


def test_largest_token_count(lm, orc):
    """T = 65536, the most the library accepts: the routing table is checked in
    full against the oracle's, the output on sampled tokens (the layer is
    token-independent)."""
    from test_gpu_parity import check_out_routed, check_route, run_route, sample_tokens
    from parity_util import device_weights, host_weights, ws_view
    d = synth.with_tokens(synth.CONFIGS["prefill_t4096"], 65536)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    x_dev = to_dev(x)
    got = run_route(lm, d, x_dev, w)
    _, _, differs = check_route(orc, d, x, hw, got, label="T=65536")
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward(dims, lm.weights_of(w), x_dev, out, ws)
    assert lm.lmoe_status_check(ws) == 0
    lay = lm.lmoe_workspace_layout(dims)
    fidx = to_host(ws_view(ws, lay.topk_idx, torch.int32, (d.T, d.k)))
    fw = to_host(ws_view(ws, lay.topk_w, torch.float32, (d.T, d.k)))
    assert np.array_equal(fidx, got["idx"])
    # sampled tokens, plus every token routed differently from the oracle (checked on its own routing)
    S = np.union1d(sample_tokens(d.T), differs)
    dS = synth.with_tokens(d, len(S))
    ref = orc.forward(dS, np.ascontiguousarray(x[S]), hw)
    check_out_routed(orc, d, x, hw, to_host(out)[S], ref["out"], differs, fidx, fw,
                     "out (T = 65536, sampled tokens)", tokens=S)
