"""Per-launch timing events (lmoe_profile_events): each launch is bracketed by
its own pair of events on the stream it runs on, so every launch's device time
is well defined and non-negative, also above 16 tokens where the routing
launches run on a second stream beside the pooler."""
from __future__ import annotations

import pytest
import torch

import synth
from parity_util import to_dev, ws_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import latent_moe_layer_fp32_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lm.load()
    return lm


@pytest.mark.parametrize("T", [4, 64])
def test_launch_event_pairs(lm, T):
    d = synth.with_tokens(synth.CONFIGS["tiny"], T)
    hw = synth.make_weights(d)
    wd = {k: (None if v is None else to_dev(v)) for k, v in hw.items()}
    x = to_dev(synth.make_x(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    ref = torch.empty_like(out)
    lm.lmoe_forward(dims, lm.weights_of(wd), x, ref, ws)
    n = lm.lmoe_last_launch_count()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    lm.lmoe_profile_events(evs)
    try:
        lm.lmoe_forward(dims, lm.weights_of(wd), x, out, ws)
        torch.cuda.synchronize()
    finally:
        lm.lmoe_profile_events(None)
    assert lm.lmoe_last_launch_count() == n
    assert lm.lmoe_status_check(ws) == 0
    times = [evs[2 * j].elapsed_time(evs[2 * j + 1]) for j in range(n)]
    assert all(t >= 0.0 for t in times), times
    assert torch.equal(out, ref)  # timing changes no result
