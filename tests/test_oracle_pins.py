"""The CPU oracle against its pins (see oracle_pins.py), plus planted mistakes."""
import numpy as np
import pytest

import oracle
import synth
from oracle_pins import PINS, make_case


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


PLANTS = {1: "nibble order", 2: "gate/up swapped", 3: "W2 transposed", 4: "scale off by one",
          5: "no renormalisation", 6: "ties to higher index", 7: "norm on the sum", 8: "gain dropped"}


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
    assert failed, f"planted mistake '{PLANTS[plant]}' passed every pin"
