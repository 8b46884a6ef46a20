"""The post-expert norm and the weighted sum formed inside the down launch
(LMOE_OPT_DOWN_Z_MAX_TOKENS): after a device-wide count of the down CTAs, each
CTA forms z for its 32-column slices with the same arithmetic, in the same
order, as the separate combine launch.  So the layer output is bit-identical
between the two, the combine launch is absent from the decode chain, and the
result agrees with the oracle.  Above 64 route rows the combine launch runs."""
from __future__ import annotations

import pytest
import torch

import oracle
import synth
from parity_util import check_out, device_weights, host_weights, to_dev, to_host, ws_for

pytestmark = pytest.mark.gpu

CASES = [("tiny", 1), ("tiny", 4), ("tiny", 8), ("tiny", 9), ("tiny_k8", 8), ("decode_t1", None),
         ("verify_t8", None), ("verify_t8_skewed", None)]


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


def dims_for(name, T):
    if name == "tiny_k8":  # 64 route rows: the most the down launch takes
        import dataclasses
        return dataclasses.replace(synth.with_tokens(synth.CONFIGS["tiny"], T), k=8)
    return synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)


def forward(lm, d, w, x, zmax):
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    prev = lm.lmoe_set_option(lm.LMOE_OPT_DOWN_Z_MAX_TOKENS, zmax)
    try:
        lm.lmoe_forward(dims, lm.weights_of(w), x, out, ws)
        names = [lm.lmoe_last_launch_name(i) for i in range(lm.lmoe_last_launch_count())]
        assert lm.lmoe_status_check(ws) == 0
    finally:
        lm.lmoe_set_option(lm.LMOE_OPT_DOWN_Z_MAX_TOKENS, prev)
    return out, names


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_down_forms_z(lm, orc, name, T):
    d = dims_for(name, T)
    hw = host_weights(d)
    w = device_weights(d)
    x_h = synth.make_x(d)
    x = to_dev(x_h)
    out_z, names_z = forward(lm, d, w, x, 8)
    out_c, names_c = forward(lm, d, w, x, 0)
    in_down = d.T <= 8 and d.T * d.k <= 64
    assert ("combine_kernel" not in names_z) == in_down, names_z
    # the default: the combine launch
    out_d, names_d = forward(lm, d, w, x, -1)
    assert "combine_kernel" in names_d, names_d
    assert torch.equal(out_d.view(torch.int16), out_c.view(torch.int16))
    assert "combine_kernel" in names_c, names_c
    assert torch.equal(out_z.view(torch.int16), out_c.view(torch.int16)), "z in the down launch differs"
    ref = orc.forward(d, x_h, hw)
    check_out(to_host(out_z), ref["out"], f"forward, z in the down launch ({name})")


def test_down_z_repeat_calls(lm):
    """The CTA counter lives in the workspace and every call zeroes it:
    back-to-back calls on one workspace give the same bits."""
    d = synth.CONFIGS["verify_t8"]
    w = device_weights(d)
    x = to_dev(synth.make_x(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = ws_for(lm, dims)
    outs = []
    prev = lm.lmoe_set_option(lm.LMOE_OPT_DOWN_Z_MAX_TOKENS, 8)
    try:
        for _ in range(3):
            o = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
            lm.lmoe_forward(dims, lm.weights_of(w), x, o, ws)
            outs.append(o)
    finally:
        lm.lmoe_set_option(lm.LMOE_OPT_DOWN_Z_MAX_TOKENS, prev)
    torch.cuda.synchronize()
    assert lm.lmoe_status_check(ws) == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
