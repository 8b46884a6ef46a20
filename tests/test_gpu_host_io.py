"""lmoe_forward_host: the layer with its tokens and output in pinned host
memory.  Two small kernels move them between the host buffers and the
workspace (and the first zeroes the workspace's counters in place of the
memset), so the result must be bit-identical to lmoe_forward on the same
tokens, back to back on one workspace, in the decode chain, the side-stream
fork and the tensor-core regime.  Pointers that are not page-locked host
memory and a short workspace are refused before anything is launched."""
from __future__ import annotations

import pytest
import torch

import synth
from parity_util import device_weights, to_dev

pytestmark = pytest.mark.gpu

CASES = [("tiny", 1), ("tiny", 37), ("tiny", 600), ("decode_t1", None), ("verify_t8", None), ("batched_t64", None)]


@pytest.fixture(scope="module")
def lm():
    import latent_moe_layer_fp32_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lm.load()
    return lm


def dims_for(name, T):
    return synth.CONFIGS[name] if T is None else synth.with_tokens(synth.CONFIGS[name], T)


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}_T{t}" for n, t in CASES])
def test_host_io_matches_device_io(lm, name, T):
    d = dims_for(name, T)
    w = lm.weights_of(device_weights(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    x_np = synth.make_x(d)
    x_dev = to_dev(x_np)
    ref = torch.empty(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    ws_dev = torch.empty(lm.lmoe_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    lm.lmoe_forward(dims, w, x_dev, ref, ws_dev)

    hb = lm.lmoe_host_workspace_bytes(dims)
    assert hb >= lm.lmoe_workspace_bytes(dims) + 2 * d.T * d.H * 2
    ws = torch.full((hb,), 0xA5, dtype=torch.uint8, device="cuda")  # stale contents: the call must zero its counters
    x_host = x_dev.cpu().pin_memory()
    outs = []
    for _ in range(2):  # two calls in a row on one workspace
        out_host = torch.full((d.T, d.H), float("nan"), dtype=torch.bfloat16).pin_memory()
        lm.lmoe_forward_host(dims, w, x_host, out_host, ws)
        names = [lm.lmoe_last_launch_name(i) for i in range(lm.lmoe_last_launch_count())]
        torch.cuda.synchronize()
        assert lm.lmoe_status_check(ws) == 0
        if d.T * d.H * 2 <= 256 * 1024:  # small: the copy kernels, else the copy engines
            assert names[0] == "io_in_kernel" and names[-1] == "io_out_kernel", names
        else:
            assert names[0] == "ws_zero_kernel" and "io_in_kernel" not in names, names
        outs.append(out_host)
    ref_h = ref.cpu()
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref_h.view(torch.int16))


def test_host_io_refuses_other_memory(lm):
    d = synth.with_tokens(synth.CONFIGS["tiny"], 4)
    w = lm.weights_of(device_weights(d))
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws = torch.empty(lm.lmoe_host_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    pinned_x = torch.zeros(d.T, d.H, dtype=torch.bfloat16).pin_memory()
    pinned_out = torch.empty(d.T, d.H, dtype=torch.bfloat16).pin_memory()
    pageable = torch.zeros(d.T, d.H, dtype=torch.bfloat16)
    for x, o in ((pageable, pinned_out), (pinned_x, torch.empty(d.T, d.H, dtype=torch.bfloat16))):
        with pytest.raises(lm.LmoeError) as e:
            lm.lmoe_forward_host(dims, w, x, o, ws)
        assert e.value.code == lm.LMOE_EINVAL
    # device memory in place of host memory (the ctypes layer is bypassed to reach the C check)
    dev_x = torch.zeros(d.T, d.H, dtype=torch.bfloat16, device="cuda")
    import ctypes
    rc = lm.load().lmoe_forward_host(ctypes.byref(dims), ctypes.byref(w), ctypes.c_void_p(dev_x.data_ptr()),
                                     ctypes.c_void_p(pinned_out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                     ws.numel(), None)
    assert rc == lm.LMOE_EINVAL
    # a workspace sized for lmoe_forward is too short
    short = torch.empty(lm.lmoe_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    with pytest.raises(lm.LmoeError) as e:
        lm.lmoe_forward_host(dims, w, pinned_x, pinned_out, short)
    assert e.value.code == lm.LMOE_EWORKSPACE
