"""lmoe_forward captured in a CUDA graph: the zeroing kernel, the programmatic-launch
chain and the side-stream fork/join all replay.  A replay equals the eager
call bit for bit and matches the CPU oracle, also after new input is copied
into the captured buffer; a two-layer stack captured in one graph (each
layer's bf16 output the next layer's input) matches the oracle layer by
layer and the oracle applied twice; the host-buffer entry point replays
against the same pinned buffers."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (bf, check_indices, check_out, device_weights, host_weights, router_regime, to_dev,
                         to_host, ws_for, ws_view)

pytestmark = pytest.mark.gpu

# decode chain (one launch of routing), many-token routing on the side stream,
# tensor-core projections and experts, and the full decode shape
CASES = [("tiny", 1), ("tiny", 37), ("tiny", 600), ("decode_t1", None)]


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


def check_layer(lm, orc, d, x_u16, out_u16, ws, dims, what):
    """One layer's output against the oracle on the same input: the oracle's
    own routing where the GPU picked the same experts, the oracle on the GPU's
    routing for near-tie tokens (none are expected)."""
    from test_gpu_parity import check_out_routed
    hw = host_weights(d)
    ref = orc.forward(d, x_u16, hw)
    lay = lm.lmoe_workspace_layout(dims)
    gidx = to_host(ws_view(ws, lay.topk_idx, torch.int32, (d.T, d.k)))
    gw = to_host(ws_view(ws, lay.topk_w, torch.float32, (d.T, d.k)))
    logits, absdot = orc.router_logits(d, x_u16, hw["router_w"], hw["router_bias"], want_absdot=True)
    _, differs = check_indices(d, gidx, ref["topk_idx"], logits, absdot, regime=router_regime(d))
    check_out_routed(orc, d, x_u16, hw, out_u16, ref["out"], differs, gidx, gw, what)
    return ref


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_forward_replays_from_a_cuda_graph(lm, orc, name, T):
    d = synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)
    wts = lm.weights_of(device_weights(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    xh, x2h = synth.make_x(d), synth.make_x(d, token0=d.T)  # the next T tokens of the same stream
    x, x2 = to_dev(xh), to_dev(x2h)
    ref = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    ref2 = torch.empty_like(ref)
    lm.lmoe_forward(dims, wts, x, ref, ws)
    lm.lmoe_forward(dims, wts, x2, ref2, ws)
    assert lm.lmoe_status_check(ws) == 0

    out = torch.empty_like(ref)
    xin = x.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first-use setup (attributes, tensor maps, side stream) outside capture
        lm.lmoe_forward(dims, wts, xin, out, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lm.lmoe_forward(dims, wts, xin, out, ws)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    check_layer(lm, orc, d, xh, to_host(out), ws, dims, "graph replay")
    xin.copy_(x2)
    g.replay()
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(out.view(torch.int16), ref2.view(torch.int16))
    check_layer(lm, orc, d, x2h, to_host(out), ws, dims, "graph replay, new input")


@pytest.mark.parametrize("name,T", [("tiny", 4), ("decode_t1", None)], ids=["tiny_T4", "decode_t1"])
def test_two_layer_stack_from_a_cuda_graph(lm, orc, name, T):
    """Two layers back to back in one captured graph, layer 2 reading layer 1's
    bf16 output, each layer with its own device copy of the weights and its
    own workspace (the multi-layer decode loop)."""
    d = synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)
    w1 = device_weights(d)
    w2 = {k: (None if v is None else v.clone()) for k, v in w1.items()}
    wts = [lm.weights_of(w1), lm.weights_of(w2)]
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = [ws_for(lm, dims), ws_for(lm, dims)]
    xh = synth.make_x(d)
    x = to_dev(xh)
    mid = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(mid)

    def stack():
        lm.lmoe_forward(dims, wts[0], x, mid, ws[0])
        lm.lmoe_forward(dims, wts[1], mid, out, ws[1])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        stack()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        stack()
    mid.zero_()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws[0]) == 0 and lm.lmoe_status_check(ws[1]) == 0
    mid_h, out_h = to_host(mid), to_host(out)
    # layer by layer: each layer against the oracle on the same input
    ref1 = check_layer(lm, orc, d, xh, mid_h, ws[0], dims, "layer 1")
    check_layer(lm, orc, d, mid_h, out_h, ws[1], dims, "layer 2 (on the GPU's layer-1 output)")
    # end to end: the oracle applied twice (layer 2 on the oracle's own layer-1 output)
    hw = host_weights(d)
    ref2 = orc.forward(d, ref1["out"], hw)
    lay = lm.lmoe_workspace_layout(dims)
    gidx2 = to_host(ws_view(ws[1], lay.topk_idx, torch.int32, (d.T, d.k)))
    assert np.array_equal(gidx2, ref2["topk_idx"]), "layer 2 routed differently from the oracle applied twice"
    # two layers' errors add: the layer-2 input already differs from the oracle's by layer 1's
    # rounding, so the element-wise bar is twice one layer's; the normwise and cosine bars stay
    g, r = bf(out_h), bf(ref2["out"])
    dd = g - r
    assert np.abs(dd).max() / np.abs(r).max() <= 2e-2
    assert float((g * r).sum() / (np.linalg.norm(g) * np.linalg.norm(r))) >= 0.9999
    assert np.all(np.abs(dd) <= 4e-2 * (np.abs(r) + np.sqrt((r * r).mean())))


@pytest.mark.parametrize("name,T", [("tiny", 4), ("tiny", 600), ("decode_t1", None)],
                         ids=["tiny_T4", "tiny_T600", "decode_t1"])
def test_host_buffer_forward_replays_from_a_cuda_graph(lm, name, T):
    """lmoe_forward_host captured in a graph: the copy kernels (few tokens) or
    the copy-engine transfers (many) replay against the same pinned buffers,
    so new tokens written into the host input give the eager result for them."""
    d = synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)
    wts = lm.weights_of(device_weights(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    x, x2 = to_dev(synth.make_x(d)), to_dev(synth.make_x(d, token0=d.T))
    ref = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    ref2 = torch.empty_like(ref)
    ws_dev = ws_for(lm, dims)
    lm.lmoe_forward(dims, wts, x, ref, ws_dev)
    lm.lmoe_forward(dims, wts, x2, ref2, ws_dev)
    torch.cuda.synchronize()

    ws = torch.empty(lm.lmoe_host_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    x_host = x.cpu().pin_memory()
    out_host = torch.zeros(d.T, d.H, dtype=torch.bfloat16).pin_memory()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first-use setup outside the capture
        lm.lmoe_forward_host(dims, wts, x_host, out_host, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lm.lmoe_forward_host(dims, wts, x_host, out_host, ws)
    out_host.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(out_host.view(torch.int16), ref.cpu().view(torch.int16))
    x_host.copy_(x2.cpu())
    g.replay()
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(out_host.view(torch.int16), ref2.cpu().view(torch.int16))
