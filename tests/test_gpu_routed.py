"""The layer with caller-supplied routing (lmoe_forward_routed) against the CPU
oracle's stages composed with the same routing, in every regime."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check_out, device_weights, host_weights, to_dev, to_host, ws_for

pytestmark = pytest.mark.gpu

# (config, T): decode with one- and several-row groups, many-token routing next to
# the pooler, tensor-core projections, and the grouped tensor-core experts (T >= 352)
CASES = [("tiny", 4), ("tiny", 37), ("tiny", 300), ("tiny", 600), ("decode_t1", None), ("verify_t8", None)]


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


def random_routing(d, seed):
    """Seeded routing: expert ids drawn with repeats allowed (a token may name an
    expert twice), positive weights summing to 1 per token."""
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, d.E, size=(d.T, d.k), dtype=np.int32)
    w = rng.uniform(0.05, 1.0, size=(d.T, d.k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    return idx, w.astype(np.float32)


def run(lm, d, w, x, idx, tw):
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward_routed(dims, lm.weights_of(w), to_dev(x), to_dev(idx), to_dev(tw), out, ws)
    return out, ws


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_forward_routed_matches_oracle(lm, orc, name, T):
    d = cfg(name, T)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    idx, tw = random_routing(d, seed=17 + d.T)
    ref = orc.forward_routed(d, x, hw, idx, tw)
    out, ws = run(lm, d, w, x, idx, tw)
    assert lm.lmoe_status_check(ws) == 0
    check_out(to_host(out), ref["out"])


def test_forward_routed_with_the_routers_choice_is_forward(lm):
    # the same kernels on the same routing table: bit-identical to lmoe_forward
    d = cfg("tiny", 37)
    w = device_weights(d)
    x = to_dev(synth.make_x(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward(dims, lm.weights_of(w), x, out, ws)
    assert lm.lmoe_status_check(ws) == 0
    lay = lm.lmoe_workspace_layout(dims)
    idx = ws[lay.topk_idx:lay.topk_idx + 4 * d.T * d.k].view(torch.int32).clone()
    tw = ws[lay.topk_w:lay.topk_w + 4 * d.T * d.k].view(torch.float32).clone()
    ws2 = ws_for(lm, dims)
    out2 = torch.empty_like(out)
    lm.lmoe_forward_routed(dims, lm.weights_of(w), x, idx, tw, out2, ws2)
    assert lm.lmoe_status_check(ws2) == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_forward_routed_reports_an_id_out_of_range(lm):
    d = cfg("tiny", 4)
    w = device_weights(d)
    x = synth.make_x(d)
    idx, tw = random_routing(d, seed=3)
    idx[1, 2] = d.E  # one past the last expert
    out, ws = run(lm, d, w, x, idx, tw)
    assert lm.lmoe_status_check(ws) == lm.LMOE_EDEVICE_CHECK
