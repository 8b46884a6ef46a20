"""lmoe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a plugin running inside another runtime's enqueue path, where
that runtime owns all device memory, or an embedded runtime with a fixed
budget) cannot pass the workspace lmoe_route needs; this entry point keeps
its scratch in a fixed array inside the library.  The tests call it through
the C ABI, twice in a row with different inputs, and check:
  * against lmoe_route on the same inputs: indices and tables bit-exact,
    weights within the 5e-5 relative tolerance of the parity tests;
  * at the full layer width (8192 hidden, 256 experts) against the oracle:
    indices outside near ties and tables bit-exact, weights within the same
    tolerance (lmoe_route takes its tensor-core router from 64 tokens there,
    so the oracle is the common reference);
  * that a call allocates no device memory (torch's allocator and the
    driver's free-memory count unchanged across it);
  * the size limit.
They build their own inputs, so they pass alone in a fresh process as well
as after the other tests.  This file is collected last.
"""
from dataclasses import replace

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


def _router_inputs(d, seed):
    """Router weights, bias and input only: the call touches nothing else."""
    wr = synth.normal_f32(seed, synth.TID_ROUTER, (d.E, d.H), 0.0, (1.0 / d.H) ** 0.5)
    bias = synth.make_router_bias(d)
    x = synth.make_x(d, seed)
    return wr, bias, x


@pytest.fixture(scope="module")
def lm():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import latent_moe_layer_fp32_gb300 as lm
    lm.build()
    lm.load()
    return lm


def test_route_noalloc_matches_route(lm):
    base = synth.with_tokens(synth.CONFIGS["tiny"], 64)
    # two different problems in a row; the second with routes concentrated by a
    # +3 logit bias on experts 0..15 of 32 (a real skew: half the experts biased)
    cases = [(synth.with_tokens(base, 37), 0), (replace(base, E=32, skewed=True), 3)]
    for d, seed in cases:
        wr, bias, x = (_dev(a) for a in _router_inputs(d, seed))
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
        assert lm.lmoe_last_launch_count() == 3
        assert torch.equal(got[0], ref[0])
        assert torch.allclose(got[1], ref[1], rtol=5e-5, atol=1e-6)
        for a, b in zip(got[2:], ref[2:]):
            assert torch.equal(a, b)
        if d.skewed:
            counts = torch.diff(got[2]).cpu().numpy()
            assert counts[:16].sum() > counts[16:].sum()  # the biased half takes most routes


@pytest.mark.parametrize("T", [1, 8, 64])
def test_route_noalloc_full_width_matches_oracle(lm, T):
    import oracle
    from parity_util import check_indices, weights_at
    d = synth.with_tokens(synth.CONFIGS["decode_t1"], T)
    wr_h, bias_h, x_h = _router_inputs(d, 0)
    orc = oracle.get()
    logits, absdot = orc.router_logits(d, x_h, wr_h, bias_h, want_absdot=True)
    idx, tw = orc.topk(d, logits)
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    wr, bias, x = _dev(wr_h), _dev(bias_h), _dev(x_h)
    for call in range(2):  # two calls in a row share the scratch
        got = _outs(d)
        for o in got:
            o.fill_(-1)
        lm.lmoe_route_noalloc(dims, x, wr, bias, *got)
        torch.cuda.synchronize()
        g_idx, g_w = got[0].cpu().numpy(), got[1].cpu().numpy()
        _, differs = check_indices(d, g_idx, idx, logits, absdot, regime="simt")
        assert np.allclose(g_w, weights_at(logits, g_idx), rtol=5e-5, atol=1e-6)
        off, rows, pos = orc.table(d, g_idx)
        assert np.array_equal(got[2].cpu().numpy(), off)
        assert np.array_equal(got[3].cpu().numpy(), rows)
        assert np.array_equal(got[4].cpu().numpy(), pos)
        assert differs.size == 0, differs


def test_route_noalloc_allocates_nothing(lm):
    d = synth.with_tokens(synth.CONFIGS["tiny"], 16)
    wr, bias, x = (_dev(a) for a in _router_inputs(d, 5))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    outs = _outs(d)
    lm.lmoe_route_noalloc(dims, x, wr, bias, *outs)  # first call on the device: set-up
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        lm.lmoe_route_noalloc(dims, x, wr, bias, *outs)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0


def test_route_noalloc_size_limit(lm):
    # beyond the fixed scratch: a clear error, nothing launched
    d = synth.with_tokens(synth.CONFIGS["tiny"], 65)
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    x = torch.zeros(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros(d.E, d.H, dtype=torch.float32, device="cuda")
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_route_noalloc(dims, x, wr, None, *_outs(d))
    assert e.value.code == lm.LMOE_ENOSCRATCH
    # dimensions lmoe_route rejects are rejected the same way
    bad = lm.dims_of(4, 512, 384, 256, 16, 4, 1e-6)  # latent not a multiple of 256
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_route_noalloc(bad, x[:4], wr, None, *_outs(synth.with_tokens(synth.CONFIGS["tiny"], 4)))
    assert e.value.code == lm.LMOE_EUNSUPPORTED
