"""NVFP4 expert weights (E2M1 codes, E4M3 scale per 16 elements, fp32 global
scale per expert matrix) against the CPU oracle: the expert stage on the
oracle's activations and table, and the whole layer, in the decode kernels
(one-row and several-row groups, one K chunk and several) and the grouped
tensor-core kernels."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check_out, to_dev, to_host, ws_for

pytestmark = pytest.mark.gpu

# tiny shapes (K = 256: one chunk, scales by bulk copy), full shape (K = 4096: two
# chunks, scales by tensor copy); T = 600 runs the grouped tensor-core experts
STAGE_CASES = [("tiny", 1), ("tiny", 4), ("tiny", 37), ("tiny", 600), ("decode_t1", None), ("verify_t8", None),
               ("batched_t64", None)]
FORWARD_CASES = [("tiny", 4), ("tiny", 37), ("tiny", 600), ("decode_t1", None), ("verify_t8", None),
                 ("batched_t64", None)]

_W = {}


def nv_weights(d):
    key = (d.H, d.L, d.I, d.E)
    if key not in _W:
        _W.clear()
        torch.cuda.empty_cache()
        hw = synth.make_weights_nvfp4(d)
        _W[key] = (hw, {k: (None if v is None else to_dev(v)) for k, v in hw.items()})
    return _W[key]


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


def cfg(name, T):
    d = synth.CONFIGS[name]
    return d if T is None else synth.with_tokens(d, T)


def check_y_nvfp4(got, ref):
    """Per-route rows.  The oracle rounds every weight (E2M1 x E4M3) x global in
    fp32 before its dot products; the kernels multiply each dot product by the
    global scale once.  The pre-activations then differ by a few fp32 ulps, and
    where that moves bf16(silu(g) u) across a rounding boundary, one h element
    changes by one bf16 ulp (2^-8 of it).  For one of a row's largest h elements
    (about ten times its rms, over I = 256) that moves y by up to
    10 * 2^-8 / sqrt(256) ~ 2.4e-3 of its norm, so the worst row may reach
    5e-3.  A flip is about as likely for every element (probability ~ the
    relative pre-activation difference / 2^-8), so a row's error is near
    2^-8 * sqrt(that probability) at any width: the 99th percentile must stay
    below 1e-3 (measured 6e-5 at I = 256, 3.6e-4 at I = 4096).  With a global
    scale of one the rows match like the MXFP4 ones."""
    g, r = got.astype(np.float64), ref.astype(np.float64)
    e = np.linalg.norm(g - r, axis=-1) / (np.linalg.norm(r, axis=-1) + 1e-30)
    assert e.max() <= 5e-3, f"worst row normwise error {e.max():.3e}"
    assert np.quantile(e, 0.99) <= 1e-3, f"99th percentile row error {np.quantile(e, 0.99):.3e}"


@pytest.mark.parametrize("name,T", STAGE_CASES, ids=[f"{n}_T{t}" for n, t in STAGE_CASES])
def test_nvfp4_experts_stage(lm, orc, name, T):
    d = cfg(name, T)
    hw, w = nv_weights(d)
    x = synth.make_x(d)
    logits = orc.router_logits(d, x, hw["router_w"], hw["router_bias"])
    idx, _ = orc.topk(d, logits)
    x_lat = orc.pool(d, x, hw["pooler_w"])
    ref = orc.experts_nvfp4(d, x_lat, idx, hw)
    off, rows, _ = orc.table(d, idx)
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    y = torch.empty(d.T * d.k, d.L, dtype=torch.float32, device="cuda")
    lm.lmoe_experts_nvfp4(dims, to_dev(x_lat), to_dev(off), to_dev(rows), w["w13_q"], w["w13_s"], w["w13_gs"],
                          w["w2_q"], w["w2_s"], w["w2_gs"], y, ws)
    assert lm.lmoe_status_check(ws) == 0
    names = [lm.lmoe_last_launch_name(i) for i in range(lm.lmoe_last_launch_count())]
    assert any(n.startswith("expert_gateup") for n in names), names
    check_y_nvfp4(to_host(y), ref)


@pytest.mark.parametrize("name,T", FORWARD_CASES, ids=[f"{n}_T{t}" for n, t in FORWARD_CASES])
def test_nvfp4_forward(lm, orc, name, T):
    d = cfg(name, T)
    hw, w = nv_weights(d)
    x = synth.make_x(d)
    ref = orc.forward_nvfp4(d, x, hw)
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward_nvfp4(dims, lm.weights_of(w), lm.nvfp4_of(w), to_dev(x), out, ws)
    assert lm.lmoe_status_check(ws) == 0
    lay = lm.lmoe_workspace_layout(dims)
    gidx = ws[lay.topk_idx:lay.topk_idx + 4 * d.T * d.k].view(torch.int32).cpu().numpy().reshape(d.T, d.k)
    assert np.array_equal(gidx, ref["topk_idx"])  # the router is the MXFP4 layer's; seeded inputs have no near ties
    check_out(to_host(out), ref["out"], "out (NVFP4)")


def test_nvfp4_scales_differ_from_mxfp4(lm):
    """The NVFP4 entry really reads E4M3 scales per 16 elements: the same bytes
    read as MXFP4 (E8M0 per 32) give a different result."""
    d = cfg("tiny", 4)
    hw, w = nv_weights(d)
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    x = to_dev(synth.make_x(d))
    a = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward_nvfp4(dims, lm.weights_of(w), lm.nvfp4_of(w), x, a, ws)
    assert lm.lmoe_status_check(ws) == 0
    b = torch.empty_like(a)
    lm.lmoe_forward(dims, lm.weights_of(w), x, b, ws)  # the first half of each scale row read as E8M0
    assert lm.lmoe_status_check(ws) == 0
    assert not torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 600), ("decode_t1", None)])
def test_nvfp4_forward_replays_from_a_cuda_graph(lm, name, T):
    d = cfg(name, T)
    _, w = nv_weights(d)
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    wts, nv = lm.weights_of(w), lm.nvfp4_of(w)
    x = to_dev(synth.make_x(d))
    ref = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward_nvfp4(dims, wts, nv, x, ref, ws)
    out = torch.empty_like(ref)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        lm.lmoe_forward_nvfp4(dims, wts, nv, x, out, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lm.lmoe_forward_nvfp4(dims, wts, nv, x, out, ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
