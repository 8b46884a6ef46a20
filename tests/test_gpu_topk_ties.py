"""Exact ties in the router's logits: experts 2m and 2m+1 get the same weight
row, so their logits are equal to the last bit in every routing path (the
same products summed in the same order).  The selection order of the pages'
router ("Muse Spark Open on Gaudi 2", "What was built": top-k of an fp32
softmax) is silent on ties; the library and the oracle give the lower expert
index first.  So every pick must come with its twin right after it, the two
weights must be equal, and the order of the pairs must match the oracle's
wherever the pairs' own logits are not within the summation error bound."""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check_indices, router_regime, to_dev, weights_at, ws_for

pytestmark = pytest.mark.gpu

CASES = [("tiny", 1), ("tiny", 8), ("tiny", 37), ("decode_t1", None), ("verify_t8", None), ("batched_t64", None)]


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


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_exact_ties_go_to_the_lower_index(lm, orc, name, T):
    d = synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)
    assert d.k % 2 == 0
    wr = synth.normal_f32(7, synth.TID_ROUTER, (d.E, d.H), 0.0, (1.0 / d.H) ** 0.5)
    wr[1::2] = wr[0::2]
    x = synth.make_x(d, 3)
    logits, absdot = orc.router_logits(d, x, wr, None, want_absdot=True)
    assert np.array_equal(logits[:, 0::2], logits[:, 1::2])
    ref_idx, ref_w = orc.topk(d, logits)

    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    idx = torch.empty(d.T, d.k, dtype=torch.int32, device="cuda")
    tw = torch.empty(d.T, d.k, dtype=torch.float32, device="cuda")
    off = torch.empty(d.E + 1, dtype=torch.int32, device="cuda")
    rows = torch.empty(d.T * d.k, dtype=torch.int32, device="cuda")
    pos = torch.empty(d.T * d.k, dtype=torch.int32, device="cuda")
    lm.lmoe_route(dims, to_dev(x), to_dev(wr), None, idx, tw, off, rows, pos, ws)
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    gidx, gw = idx.cpu().numpy(), tw.cpu().numpy()

    # every pick is the lower twin, followed by the upper one with the same weight
    assert (gidx[:, 0::2] % 2 == 0).all(), gidx
    assert np.array_equal(gidx[:, 1::2], gidx[:, 0::2] + 1), gidx
    assert np.array_equal(gw[:, 0::2].view(np.uint32), gw[:, 1::2].view(np.uint32))
    # the order of the pairs: exact wherever the pairs' logits are apart by more than the
    # rigorous bound, a valid top-k choice of pairs within it elsewhere
    regime = router_regime(d)
    dp = replace(d, E=d.E // 2, k=d.k // 2)
    flagged, differs = check_indices(dp, gidx[:, 0::2] // 2, ref_idx[:, 0::2] // 2, logits[:, 0::2],
                                     absdot[:, 0::2], regime=regime)
    if regime == "simt":  # a tight bound: nearly every token is decided
        assert d.T - flagged.size >= max(1, int(0.9 * d.T)), flagged
    assert np.allclose(gw, weights_at(logits, gidx), rtol=5e-5, atol=1e-6)
    # and the table of the GPU's picks is the oracle's table of those picks
    o_off, o_rows, o_pos = orc.table(d, gidx)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(rows.cpu().numpy(), o_rows)
    assert np.array_equal(pos.cpu().numpy(), o_pos)
