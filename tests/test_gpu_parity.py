"""GPU parity: every C-ABI call against the CPU oracle, element by element.

Each stage is checked on its own with the oracle's inputs for that stage
(route, pool, experts, norm+combine+unpool), and the fused lmoe_forward is
checked end to end.  Shapes: the tiny layer (several token counts, ragged
tails) and the full layer at T = 1, 4, 8, 4 and 8 with skewed routing, 64 and
4096.  At T = 4096 the oracle evaluates a sample of tokens (the layer is
token-independent) and stage inputs that the oracle cannot produce for every
token come from the seeded generator.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (bf, check_bf16_close, check_indices, check_out, check_rows_normwise, device_weights,
                         host_weights, record_route, router_regime, sum_err, to_dev, to_host, weights_at, ws_for,
                         ws_view)

pytestmark = pytest.mark.gpu

TID_TEST_XLAT, TID_TEST_Y = 20, 21

SMALL = [("tiny", 4), ("tiny", 1), ("tiny", 3), ("tiny", 7), ("tiny", 16), ("tiny", 37)]
FULL = ["decode_t1", "verify_t4", "verify_t8", "verify_t4_skewed", "verify_t8_skewed", "batched_t64"]


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


def dims_c(lm, d):
    return lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)


def cfg(name, T=None):
    d = synth.CONFIGS[name]
    return d if T is None else synth.with_tokens(d, T)


def sample_tokens(T, n=16, seed=7):
    if T <= 64:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    fixed = np.array([0, 1, T // 2 - 1, T // 2, T - 2, T - 1])
    rest = rng.choice(np.arange(2, T - 2), size=n - fixed.size, replace=False)
    return np.unique(np.concatenate([fixed, rest]))


def run_route(lm, d, x_dev, w):
    T, k, E = d.T, d.k, d.E
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    out = dict(idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
               off=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               rows=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               pos=torch.empty(T * k, dtype=torch.int32, device="cuda"))
    lm.lmoe_route(dims, x_dev, w["router_w"], w["router_bias"], out["idx"], out["w"], out["off"], out["rows"],
                  out["pos"], ws)
    assert lm.lmoe_status_check(ws) == 0
    return {k_: to_host(v) for k_, v in out.items()}


def pool_err(d, x, hw):
    return sum_err(d.H, np.abs(bf(x)), np.abs(bf(hw["pooler_w"])))


def check_route(orc, d, x, hw, got, regime=None, label=None, strict=False):
    """Top-k, weights and table of one routing call against the oracle.

    Indices: bit-exact outside near ties (a valid choice inside).  Weights: the
    oracle's weights at the GPU's picks.  Table: bit-exact against the oracle's
    table of the GPU's picks, always.  The counts of near-tie and differently
    routed tokens are recorded; strict (the layer's workload configs) asserts
    that no token was routed differently.  Returns the oracle's (idx, w), the
    tokens the GPU routed differently and the oracle logits."""
    regime = regime or router_regime(d)
    logits, absdot = orc.router_logits(d, x, hw["router_w"], hw["router_bias"], want_absdot=True)
    idx, tw = orc.topk(d, logits)
    flagged, differs = check_indices(d, got["idx"], idx, logits, absdot, regime=regime)
    rec = record_route(label or f"T={d.T}", d, regime, logits, absdot, flagged, differs)
    print(f"[route {rec['config']}] {rec}")
    same = np.ones(d.T, bool)
    same[differs] = False
    assert np.allclose(got["w"][same], tw[same], rtol=5e-5, atol=1e-6), np.abs(got["w"][same] - tw[same]).max()
    if differs.size:
        ref_w = weights_at(logits[differs], got["idx"][differs])
        assert np.allclose(got["w"][differs], ref_w, rtol=5e-5, atol=1e-6)
    assert np.allclose(got["w"].sum(1), 1.0, atol=1e-5)
    off, rows, pos = orc.table(d, got["idx"])
    assert np.array_equal(got["off"], off)
    assert np.array_equal(got["rows"], rows)
    assert np.array_equal(got["pos"], pos)
    if strict:
        assert differs.size == 0, f"{rec['config']}: tokens routed differently from the oracle: {rec['differing']}"
    return idx, tw, differs


def check_out_routed(orc, d, x, hw, out_u16, ref_out, differs, gpu_idx, gpu_w, what="forward", tokens=None):
    """Layer output of every token: the oracle's own output where the GPU
    routed like the oracle, the oracle run on the GPU's routing
    (forward_routed) where it did not.  tokens: the rows of out_u16 / ref_out
    (default: all T)."""
    tokens = np.arange(d.T) if tokens is None else np.asarray(tokens)
    want = ref_out.copy()
    dt = np.nonzero(np.isin(tokens, differs))[0]
    if dt.size:
        tt = tokens[dt]
        dS = synth.with_tokens(d, len(tt))
        r = orc.forward_routed(dS, np.ascontiguousarray(x[tt]), hw, np.ascontiguousarray(gpu_idx[tt]),
                               np.ascontiguousarray(gpu_w[tt]))
        want[dt] = r["out"]
    return check_out(out_u16, want, what)


# ------------------------------------------------------------------------------------------------
# small shapes: every stage from the oracle's own chain
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name,T", SMALL, ids=[f"{n}_T{t}" for n, t in SMALL])
def test_stages_small(lm, orc, name, T):
    d = cfg(name, T)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    ref = orc.forward(d, x, hw)
    x_dev = to_dev(x)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    # route
    got = run_route(lm, d, x_dev, w)
    check_route(orc, d, x, hw, got, label=f"{name} T={T}", strict=(name == "tiny" and T == 4))
    # pool
    x_lat = torch.empty(T, d.L, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_pool(dims, x_dev, w["pooler_w"], x_lat, ws)
    check_bf16_close(to_host(x_lat), ref["x_lat"], "x_lat", pool_err(d, x, hw))
    # experts on the oracle's x_lat and table
    off, rows, _ = orc.table(d, ref["topk_idx"])
    y = torch.empty(T * d.k, d.L, dtype=torch.float32, device="cuda")
    lm.lmoe_experts_mxfp4(dims, to_dev(ref["x_lat"]), to_dev(off), to_dev(rows), w["w13_q"], w["w13_s"], w["w2_q"],
                          w["w2_s"], y, ws)
    assert lm.lmoe_status_check(ws) == 0
    check_rows_normwise(to_host(y), ref["y"], 2e-3, "y")
    # norm + combine + unpool on the oracle's y and routing
    out = torch.empty(T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_norm_combine_unpool(dims, to_dev(ref["y"]), to_dev(ref["topk_idx"]), to_dev(ref["topk_w"]),
                                w["norm_g"], w["unpooler_w"], out, ws)
    assert lm.lmoe_status_check(ws) == 0
    check_out(to_host(out), ref["out"], "norm_combine_unpool")


@pytest.mark.parametrize("name,T", SMALL, ids=[f"{n}_T{t}" for n, t in SMALL])
def test_forward_small(lm, orc, name, T):
    d = cfg(name, T)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    ref = orc.forward(d, x, hw)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    out = torch.empty(T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward(dims, lm.weights_of(w), to_dev(x), out, ws)
    assert lm.lmoe_status_check(ws) == 0
    check_out(to_host(out), ref["out"])
    lay = lm.lmoe_workspace_layout(dims)
    assert np.array_equal(to_host(ws_view(ws, lay.topk_idx, torch.int32, (T, d.k))), ref["topk_idx"])
    check_bf16_close(to_host(ws_view(ws, lay.x_lat, torch.bfloat16, (T, d.L))), ref["x_lat"], "x_lat",
                     pool_err(d, x, hw))


# ------------------------------------------------------------------------------------------------
# full layer shape
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", FULL)
def test_full_shape(lm, orc, name):
    d = cfg(name)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    x_dev = to_dev(x)
    ref = orc.forward(d, x, hw)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    got = run_route(lm, d, x_dev, w)
    _, _, differs = check_route(orc, d, x, hw, got, label=name, strict=True)
    x_lat = torch.empty(d.T, d.L, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_pool(dims, x_dev, w["pooler_w"], x_lat, ws)
    check_bf16_close(to_host(x_lat), ref["x_lat"], "x_lat", pool_err(d, x, hw))
    off, rows, _ = orc.table(d, ref["topk_idx"])
    y = torch.empty(d.T * d.k, d.L, dtype=torch.float32, device="cuda")
    lm.lmoe_experts_mxfp4(dims, to_dev(ref["x_lat"]), to_dev(off), to_dev(rows), w["w13_q"], w["w13_s"], w["w2_q"],
                          w["w2_s"], y, ws)
    assert lm.lmoe_status_check(ws) == 0
    check_rows_normwise(to_host(y), ref["y"], 2e-3, "y")
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_norm_combine_unpool(dims, to_dev(ref["y"]), to_dev(ref["topk_idx"]), to_dev(ref["topk_w"]),
                                w["norm_g"], w["unpooler_w"], out, ws)
    check_out(to_host(out), ref["out"], "norm_combine_unpool")
    out2 = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward(dims, lm.weights_of(w), x_dev, out2, ws)
    assert lm.lmoe_status_check(ws) == 0
    lay = lm.lmoe_workspace_layout(dims)
    fidx = to_host(ws_view(ws, lay.topk_idx, torch.int32, (d.T, d.k)))
    fw = to_host(ws_view(ws, lay.topk_w, torch.float32, (d.T, d.k)))
    assert np.array_equal(fidx, got["idx"])  # the fused call routes like lmoe_route
    check_out_routed(orc, d, x, hw, to_host(out2), ref["out"], differs, fidx, fw, "forward")
    if d.skewed:
        touched = np.count_nonzero(np.diff(got["off"]))
        assert touched < 40, touched  # routes concentrate on the biased experts


def test_prefill_sampled(lm, orc):
    d = cfg("prefill_t4096")
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    x_dev = to_dev(x)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    S = sample_tokens(d.T)
    dS = synth.with_tokens(d, len(S))
    xS = np.ascontiguousarray(x[S])
    # route: all tokens (indices and tables are checked in full)
    got = run_route(lm, d, x_dev, w)
    idx, tw, differs = check_route(orc, d, x, hw, got, label="prefill_t4096", strict=True)
    # pool: sampled rows
    x_lat = torch.empty(d.T, d.L, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_pool(dims, x_dev, w["pooler_w"], x_lat, ws)
    check_bf16_close(to_host(x_lat)[S], orc.pool(dS, xS, hw["pooler_w"]), "x_lat", pool_err(dS, xS, hw))
    # experts: generator-made x_lat for every token, the oracle's full table
    xl = synth.normal_bf16(0, TID_TEST_XLAT, (d.T, d.L), 0.0, 1.0)
    off, rows, _ = orc.table(d, idx)
    y = torch.empty(d.T * d.k, d.L, dtype=torch.float32, device="cuda")
    lm.lmoe_experts_mxfp4(dims, to_dev(xl), to_dev(off), to_dev(rows), w["w13_q"], w["w13_s"], w["w2_q"], w["w2_s"],
                          y, ws)
    assert lm.lmoe_status_check(ws) == 0
    yS = orc.experts(dS, np.ascontiguousarray(xl[S]), np.ascontiguousarray(idx[S]), hw)
    rS = (S[:, None] * d.k + np.arange(d.k)[None, :]).reshape(-1)
    check_rows_normwise(to_host(y)[rS], yS, 2e-3, "y")
    # norm + combine + unpool: generator-made y for every row, the oracle's routing
    yy = synth.normal_f32(0, TID_TEST_Y, (d.T * d.k, d.L), 0.0, 1.0)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_norm_combine_unpool(dims, to_dev(yy), to_dev(idx), to_dev(tw), w["norm_g"], w["unpooler_w"], out, ws)
    zS = orc.norm_combine(dS, np.ascontiguousarray(yy[rS]), np.ascontiguousarray(idx[S]),
                          np.ascontiguousarray(tw[S]), hw["norm_g"])
    check_out(to_host(out)[S], orc.unpool(dS, zS, hw["unpooler_w"]), "norm_combine_unpool")
    # the whole layer
    out2 = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward(dims, lm.weights_of(w), x_dev, out2, ws)
    assert lm.lmoe_status_check(ws) == 0
    refS = orc.forward(dS, xS, hw)
    lay = lm.lmoe_workspace_layout(dims)
    fidx = to_host(ws_view(ws, lay.topk_idx, torch.int32, (d.T, d.k)))
    fw = to_host(ws_view(ws, lay.topk_w, torch.float32, (d.T, d.k)))
    assert np.array_equal(fidx, got["idx"])
    check_out_routed(orc, d, x, hw, to_host(out2)[S], refS["out"], differs, fidx, fw, "forward", tokens=S)


# ------------------------------------------------------------------------------------------------
# format self-check, determinism, errors
# ------------------------------------------------------------------------------------------------

def test_e2m1_conversion_matches_ocp_table(lm):
    from oracle_pins import golden_e2m1
    tab = golden_e2m1()
    out = torch.empty(512, dtype=torch.float32, device="cuda")
    lm.lmoe_selftest_e2m1(out)
    got = out.cpu().numpy().reshape(256, 2)
    b = np.arange(256)
    assert np.array_equal(got[:, 0], tab[b & 15]), "low nibble -> first element"
    assert np.array_equal(got[:, 1], tab[b >> 4]), "high nibble -> second element"


def test_forward_deterministic(lm):
    d = cfg("verify_t8")
    w = device_weights(d)
    x_dev = to_dev(synth.make_x(d))
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    outs = []
    for _ in range(2):
        o = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
        lm.lmoe_forward(dims, lm.weights_of(w), x_dev, o, ws)
        outs.append(to_host(o))
    assert np.array_equal(outs[0], outs[1])
    assert lm.lmoe_last_launch_count() >= 5  # kernels of the fused chain ran


def test_host_errors(lm):
    d = cfg("tiny")
    w = device_weights(d)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    x = to_dev(synth.make_x(d))
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_forward(dims, lm.weights_of(w), x, out, ws[:1024])
    assert e.value.code == -6
    bad = torch.empty(d.T * d.H + 8, dtype=torch.bfloat16, device="cuda")[1:1 + d.T * d.H].view(d.T, d.H)
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_forward(dims, lm.weights_of(w), bad, out, ws)
    assert e.value.code == -1
    bad_dims = dims_c(lm, d)
    bad_dims.top_k = 9
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_forward(bad_dims, lm.weights_of(w), x, out, ws)
    assert e.value.code == -1


def test_device_checks_report_bad_tables(lm):
    d = cfg("tiny")
    w = device_weights(d)
    dims = dims_c(lm, d)
    ws = ws_for(lm, dims)
    R = d.T * d.k
    x_lat = torch.zeros(d.T, d.L, dtype=torch.bfloat16, device="cuda")
    off = torch.zeros(d.E + 1, dtype=torch.int32, device="cuda")
    off[1:] = R
    rows = torch.arange(R, dtype=torch.int32, device="cuda")
    rows[3] = R + 5  # out of range
    y = torch.zeros(R, d.L, dtype=torch.float32, device="cuda")
    lm.lmoe_experts_mxfp4(dims, x_lat, off, rows, w["w13_q"], w["w13_s"], w["w2_q"], w["w2_s"], y, ws)
    assert lm.lmoe_status_check(ws) == -5
    idx = torch.zeros(d.T, d.k, dtype=torch.int32, device="cuda")
    idx[0, 0] = d.E  # out of range
    tw = torch.full((d.T, d.k), 1.0 / d.k, dtype=torch.float32, device="cuda")
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_norm_combine_unpool(dims, y, idx, tw, w["norm_g"], w["unpooler_w"], out, ws)
    assert lm.lmoe_status_check(ws) == -5
    # a good call afterwards resets the status
    rows[3] = 3
    lm.lmoe_experts_mxfp4(dims, x_lat, off, rows, w["w13_q"], w["w13_s"], w["w2_q"], w["w2_s"], y, ws)
    assert lm.lmoe_status_check(ws) == 0
