"""The sandwich block (lmoe_block_forward: y = x + post_norm(layer(pre_norm(x))),
the router fed by the pre-norm's fp32 output) against the CPU oracle's block,
in every regime of the layer, plus the in-place form (y = x)."""
from __future__ import annotations

import contextlib
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (bf, check_indices, check_out, device_weights, host_weights, record_route, router_regime,
                         to_dev, to_host, weights_at, ws_view)
from test_gpu_dense import dense_from

pytestmark = pytest.mark.gpu

# (config, T, dense threshold or None): decode chain with one- and several-row groups,
# many-token routing next to the pooler, the tensor-core router, pooler and unpooler
# (32 experts, threshold 1), and the grouped tensor-core experts (T >= 352)
CASES = [("tiny", 4, None), ("tiny", 37, None), ("tiny_e32", 37, 1), ("tiny_e32", 200, None),
         ("tiny", 600, None), ("decode_t1", None, None), ("verify_t8", None, None)]


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
    base = dataclasses.replace(synth.CONFIGS["tiny"], E=32) if name == "tiny_e32" else synth.CONFIGS[name]
    return base if T is None else synth.with_tokens(base, T)


def run_block(lm, d, w, nw_dev, x_dev, y_dev, dense=None):
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = torch.empty(lm.lmoe_block_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    with (dense_from(lm, dense) if dense is not None else contextlib.nullcontext()):
        lm.lmoe_block_forward(dims, lm.weights_of(w), lm.norms_of(nw_dev, d.eps), x_dev, y_dev, ws)
        names = [lm.lmoe_last_launch_name(i) for i in range(lm.lmoe_last_launch_count())]
    assert lm.lmoe_status_check(ws) == 0
    return dims, ws, names


@pytest.mark.parametrize("name,T,dense", CASES, ids=[f"{n}_T{t}" + ("_dense" if c else "") for n, t, c in CASES])
def test_block_matches_oracle(lm, orc, name, T, dense):
    d = cfg(name, T)
    hw = host_weights(d)
    w = device_weights(d)
    nw = synth.make_block_norms(d)
    nw_dev = {k: to_dev(v) for k, v in nw.items()}
    x = synth.make_x(d)
    ref = orc.block_forward(d, x, hw, nw)
    x_dev = to_dev(x)
    y_dev = torch.empty_like(x_dev)
    dims, ws, names = run_block(lm, d, w, nw_dev, x_dev, y_dev, dense)
    assert names[0] == "ws_zero_kernel" and names[1] == "prenorm_kernel", names
    assert names[-1] == "postnorm_residual_kernel", names
    if dense == 1:
        assert "router_tc_gemm" in names, names
    lay = lm.lmoe_workspace_layout(dims)
    # routing: the router reads x * g scaled by the token's rinv, the oracle the rounded fp32
    # pre-norm output; a common positive factor keeps the order, and the two inputs differ by
    # the two roundings of n (2 ulp per term), within the bound below
    gidx = to_host(ws_view(ws, lay.topk_idx, torch.int32, (d.T, d.k)))
    gw = to_host(ws_view(ws, lay.topk_w, torch.float32, (d.T, d.k)))
    regime = router_regime(d, dense if dense is not None else 64)
    # the tensor-core router of the block runs over K = 6H (the input in two bf16 parts)
    extra = 3 + (2 * (3 * d.H // 4) if regime == "tensor" else 0)
    flagged, differs = check_indices(d, gidx, ref["topk_idx"], ref["logits"], ref["absdot"], extra_depth=extra,
                                     regime=regime)
    rec = record_route(f"block {name} T={d.T}", d, regime, ref["logits"], ref["absdot"], flagged, differs, extra)
    print(f"[block {name} T={d.T}] {rec}")
    same = np.ones(d.T, bool)
    same[differs] = False
    assert np.allclose(gw[same], ref["topk_w"][same], rtol=1e-4, atol=2e-6), np.abs(gw[same] - ref["topk_w"][same]).max()
    if differs.size:
        assert np.allclose(gw[differs], weights_at(ref["logits"][differs], gidx[differs]), rtol=1e-4, atol=2e-6)
    off = to_host(ws_view(ws, lay.expert_offsets, torch.int32, (d.E + 1,)))
    rows = to_host(ws_view(ws, lay.sorted_rows, torch.int32, (d.T * d.k,)))
    pos = to_host(ws_view(ws, lay.row_pos, torch.int32, (d.T * d.k,)))
    # the table: bit-exact against the oracle's table of the GPU's picks
    o_off, o_rows, o_pos = orc.table(d, gidx)
    assert np.array_equal(off, o_off) and np.array_equal(rows, o_rows) and np.array_equal(pos, o_pos)
    y = to_host(y_dev)
    want = ref["y"].copy()
    if differs.size:
        # tokens routed differently (near ties): the oracle's block on the GPU's routing
        dS = synth.with_tokens(d, len(differs))
        r = orc.forward_routed(dS, np.ascontiguousarray(ref["nb"][differs]), hw, np.ascontiguousarray(gidx[differs]),
                               np.ascontiguousarray(gw[differs]))
        p = orc.rmsnorm(r["out"], nw["post_g"], d.eps)
        want[differs] = orc.residual_add(np.ascontiguousarray(x[differs]), p)
    check_out(y, want, "y")
    # y minus the residual: the post-norm of the layer output, compared on its own scale
    post_g = bf(nw["post_g"])
    got_p, ref_p = bf(y) - bf(x), bf(want) - bf(x)
    num = np.linalg.norm(got_p - ref_p, axis=1)
    den = np.linalg.norm(ref_p, axis=1) + 1e-30
    assert np.all(num / den <= 2e-2), np.max(num / den)
    assert np.abs(post_g).max() > 0


def test_block_in_place(lm, orc):
    """y = x: the residual stream updated in place gives the same bits."""
    d = cfg("tiny", 37)
    w = device_weights(d)
    nw_dev = {k: to_dev(v) for k, v in synth.make_block_norms(d).items()}
    x = synth.make_x(d)
    y_sep = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    run_block(lm, d, w, nw_dev, to_dev(x), y_sep)
    xy = to_dev(x)
    run_block(lm, d, w, nw_dev, xy, xy)
    assert torch.equal(xy.view(torch.int16), y_sep.view(torch.int16))


def test_block_zero_post_gain_is_identity(lm):
    """A zero post-norm gain leaves the residual stream bit for bit (the same
    identity pins the oracle)."""
    d = cfg("tiny", 9)
    w = device_weights(d)
    nw = synth.make_block_norms(d)
    nw["post_g"] = np.zeros_like(nw["post_g"])
    x = synth.make_x(d)
    y = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    run_block(lm, d, w, {k: to_dev(v) for k, v in nw.items()}, to_dev(x), y)
    assert np.array_equal(to_host(y), x)


@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 37), ("decode_t1", None)])
def test_block_replays_from_a_cuda_graph(lm, name, T):
    """The block (pre-norm, layer, post-norm and residual, with the side stream for
    many tokens) captured in a CUDA graph replays bit for bit."""
    d = cfg(name, T)
    w = device_weights(d)
    nw_dev = {k: to_dev(v) for k, v in synth.make_block_norms(d).items()}
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = torch.empty(lm.lmoe_block_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    wts, norms = lm.weights_of(w), lm.norms_of(nw_dev, d.eps)
    x = to_dev(synth.make_x(d))
    ref = torch.empty_like(x)
    lm.lmoe_block_forward(dims, wts, norms, x, ref, ws)
    y = torch.empty_like(x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        lm.lmoe_block_forward(dims, wts, norms, x, y, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lm.lmoe_block_forward(dims, wts, norms, x, y, ws)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
