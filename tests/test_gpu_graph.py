"""lmoe_forward captured in a CUDA graph: the memset, the programmatic-launch
chain and the side-stream fork/join all replay, and a replay equals the eager
call bit for bit, also after new input is copied into the captured buffer."""
from __future__ import annotations

import pytest
import torch

import synth
from parity_util import device_weights, to_dev, ws_for

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


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_forward_replays_from_a_cuda_graph(lm, name, T):
    d = synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)
    wts = lm.weights_of(device_weights(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    x = to_dev(synth.make_x(d))
    x2 = to_dev(synth.make_x(d, token0=d.T))  # the next T tokens of the same stream
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
    xin.copy_(x2)
    g.replay()
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(out.view(torch.int16), ref2.view(torch.int16))
