"""Failure detection on the GPU without a fault: every device-side wait of the
library is bounded and reports LMOE_ETIMEOUT through the workspace status
word.  The self-test kernel waits on a barrier that nothing completes; the
status must report the timeout, and the context must stay usable."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check_out, device_weights, host_weights, to_dev, to_host, ws_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import latent_moe_layer_fp32_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lm.load()
    return lm


def test_bounded_wait_reports_timeout_and_the_context_survives(lm):
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    lm.lmoe_selftest_timeout(ws, 10000)  # 10 ms
    assert lm.lmoe_status_check(ws) == lm.LMOE_ETIMEOUT
    # the next call on the same context runs and matches the oracle
    d = synth.with_tokens(synth.CONFIGS["tiny"], 4)
    hw = host_weights(d)
    w = device_weights(d)
    x = synth.make_x(d)
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws2 = ws_for(lm, dims)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    lm.lmoe_forward(dims, lm.weights_of(w), to_dev(x), out, ws2)
    assert lm.lmoe_status_check(ws2) == 0
    check_out(to_host(out), oracle.get().forward(d, x, hw)["out"])


def test_timeout_self_test_rejects_bad_arguments(lm):
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    for limit in (0, 2_000_000):
        with pytest.raises(lm.LmoeError):
            lm.lmoe_selftest_timeout(ws, limit)
