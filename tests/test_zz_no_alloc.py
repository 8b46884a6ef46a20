"""lmoe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a plugin running inside another runtime's enqueue path, where
that runtime owns all device memory, or an embedded runtime with a fixed
budget) cannot pass the workspace lmoe_route needs; this entry point keeps
its scratch in a fixed array inside the library.  The test calls it through
the C ABI twice in a row, with different inputs, and checks each result
against lmoe_route on the same inputs (indices and tables bit-exact, weights
within the 5e-5 relative tolerance of the parity tests), plus the size limit.
It builds its own inputs so it passes alone in a fresh process as well as
after the other tests.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _outs(d):
    return (torch.empty(d.T, d.k, dtype=torch.int32, device="cuda"),
            torch.empty(d.T, d.k, dtype=torch.float32, device="cuda"),
            torch.empty(d.E + 1, dtype=torch.int32, device="cuda"),
            torch.empty(d.T * d.k, dtype=torch.int32, device="cuda"),
            torch.empty(d.T * d.k, dtype=torch.int32, device="cuda"))


def test_route_noalloc_matches_route():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import latent_moe_layer_fp32_gb300 as lm
    lm.build()
    lm.load()
    base = synth.with_tokens(synth.CONFIGS["tiny"], 64)
    # router, bias and input only (the call touches nothing else); two different problems
    from dataclasses import replace
    cases = [(synth.with_tokens(base, 37), 0), (replace(base, skewed=True), 3)]
    for d, seed in cases:
        wr = _dev(synth.normal_f32(seed, synth.TID_ROUTER, (d.E, d.H), 0.0, (1.0 / d.H) ** 0.5))
        bias = _dev(synth.make_router_bias(d))
        x = _dev(synth.make_x(d, seed))
        dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
        ws = torch.empty(lm.lmoe_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
        ref = _outs(d)
        lm.lmoe_route(dims, x, wr, bias, *ref, ws)
        got = _outs(d)
        for o in got:
            o.fill_(-1)
        lm.lmoe_route_noalloc(dims, x, wr, bias, *got)
        torch.cuda.synchronize()
        assert lm.lmoe_status_check(ws) == 0
        assert torch.equal(got[0], ref[0])
        assert torch.allclose(got[1], ref[1], rtol=5e-5, atol=1e-6)
        for a, b in zip(got[2:], ref[2:]):
            assert torch.equal(a, b)
    # beyond the fixed scratch: a clear error, nothing launched
    d = synth.with_tokens(base, 65)
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    x = torch.zeros(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros(d.E, d.H, dtype=torch.float32, device="cuda")
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_route_noalloc(dims, x, wr, None, *_outs(d))
    assert e.value.code == lm.LMOE_ENOSCRATCH
