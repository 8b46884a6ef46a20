"""The CPU oracle against its pins (see oracle_pins.py), plus planted mistakes."""
import numpy as np
import pytest

import oracle
import synth
from oracle_pins import BLOCK_PINS, NV_PINS, PINS, make_block_case, make_case, make_nv_case


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.fixture(scope="module")
def case(o):
    return make_case(o, T=16)


@pytest.fixture(scope="module")
def case_skewed(o):
    return make_case(o, T=16, skewed=True)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, o, case):
    pin(o, case)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin_skewed(pin, o, case_skewed):
    pin(o, case_skewed)


def test_skewed_routes_concentrate(case_skewed):
    # +3.0 on experts 0..15 (all 16 of the tiny config's experts) changes nothing
    # relative; at full shape it concentrates routes.  Here check the bias is applied.
    assert case_skewed.w["router_bias"] is not None and case_skewed.w["router_bias"][:16].min() == 3.0


def test_forward_is_stage_composition(o, case):
    d = case.d
    r = o.forward(d, case.x, case.w)
    assert np.array_equal(r["topk_idx"], case.idx)
    assert np.array_equal(r["topk_w"], case.tw)
    assert np.array_equal(r["x_lat"], case.x_lat)
    assert np.array_equal(r["y"], case.y)
    assert np.array_equal(r["z"], case.z)
    assert np.array_equal(r["out"], case.out)


def test_forward_routed_with_its_own_routing_is_forward(o, case):
    d = case.d
    r = o.forward_routed(d, case.x, case.w, case.idx, case.tw)
    for key in ("x_lat", "y", "z", "out"):
        assert np.array_equal(r[key], getattr(case, key)), key


def test_forward_routed_duplicate_route_sums_its_weights(o, case):
    # a token naming one expert twice with weights a, b gives the sum of a route
    # with weight a + b plus a route of weight 0 (0.25 + 0.25 = 0.5 and 0 * y are exact)
    d = case.d
    idx = case.idx.copy()
    w = np.full(idx.shape, 1.0 / d.k, np.float32)
    w[:, :2] = 0.25 if d.k == 4 else w[:, :2]
    w[:, 2:] = (1.0 - w[:, :2].sum(1, keepdims=True)) / (d.k - 2)
    dup = idx.copy()
    dup[:, 1] = dup[:, 0]
    single = idx.copy()
    ws = w.copy()
    ws[:, 0] = w[:, 0] + w[:, 1]
    ws[:, 1] = 0.0
    a = o.forward_routed(d, case.x, case.w, dup, w)
    b = o.forward_routed(d, case.x, case.w, single, ws)
    assert np.array_equal(a["z"], b["z"])
    assert np.array_equal(a["out"], b["out"])


def test_thread_count_invariance(case):
    d = case.d
    a = oracle.Oracle(0, threads=1).forward(d, case.x, case.w)
    b = oracle.Oracle(0, threads=7).forward(d, case.x, case.w)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_token_independence(o, case):
    """Each token's output depends only on that token (inputs are prefixes)."""
    d1 = synth.with_tokens(case.d, 3)
    r = o.forward(d1, case.x[:3].copy(), case.w)
    assert np.array_equal(r["out"], case.out[:3])


def test_top1_reduces_to_one_dense_expert(o, case):
    """k = 1: weight 1, z is the single normed expert row."""
    from dataclasses import replace
    d = replace(case.d, k=1)
    r = o.forward(d, case.x, case.w)
    assert np.all(r["topk_w"] == 1.0)
    e = np.argmax(case.logits, axis=1)
    assert np.array_equal(r["topk_idx"][:, 0], e)
    y = o.experts(d, r["x_lat"], r["topk_idx"], case.w)
    z, yhat = o.norm_combine(d, y, r["topk_idx"], r["topk_w"], case.w["norm_g"], want_yhat=True)
    assert np.array_equal(z, yhat)


@pytest.fixture(scope="module")
def block_case(o):
    return make_block_case(o)


@pytest.mark.parametrize("pin", BLOCK_PINS, ids=[p.__name__ for p in BLOCK_PINS])
def test_block_pin(pin, o, block_case):
    pin(o, block_case)


@pytest.fixture(scope="module")
def nv_case(o):
    return make_nv_case(o)


@pytest.mark.parametrize("pin", NV_PINS, ids=[p.__name__ for p in NV_PINS])
def test_nv_pin(pin, o, nv_case):
    pin(o, nv_case)


PLANTS = {1: "nibble order", 2: "gate/up swapped", 3: "W2 transposed", 4: "scale off by one",
          5: "no renormalisation", 6: "ties to higher index", 7: "norm on the sum", 8: "gain dropped",
          9: "row RMSNorm gain dropped", 10: "block residual dropped", 11: "NVFP4 blocks of 32",
          12: "NVFP4 global scale dropped"}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=[PLANTS[k] for k in sorted(PLANTS)])
def test_planted_mistake_is_caught(plant):
    bad = oracle.Oracle(plant)
    failed = []
    try:
        c = make_case(bad, T=16)
    except AssertionError:
        return
    for pin in PINS:
        try:
            pin(bad, c)
        except AssertionError:
            failed.append(pin.__name__)
    bc = make_block_case(bad)
    for pin in BLOCK_PINS:
        try:
            pin(bad, bc)
        except AssertionError:
            failed.append(pin.__name__)
    nc = make_nv_case(bad)
    for pin in NV_PINS:
        try:
            pin(bad, nc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake '{PLANTS[plant]}' passed every pin"


def test_acc64_mode_reports_the_oracles_own_error(o, case):
    """fp64 sums (the diagnostic mode) against the default fp32 sums: the same
    routing, per-stage differences at the level of fp32 rounding and one bf16
    ulp, and the default restored bit for bit afterwards."""
    d = case.d
    rep = o.error_report(d, case.x, case.w)
    assert rep["topk_idx_same"]
    assert rep["x_lat"] <= 2 ** -8 and rep["out"] <= 2 ** -8, rep   # at most bf16 rounding flips
    assert rep["y"] <= 1e-3 and rep["z"] <= 1e-3, rep
    assert 0 < rep["y"]  # the fp32 sums do round
    again = o.forward(d, case.x, case.w)
    assert np.array_equal(again["out"], case.out)
