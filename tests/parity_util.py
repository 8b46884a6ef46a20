"""Shared helpers for the GPU parity tests: device copies of the seeded inputs,
workspace handling and the comparison rules with their tolerances.

Tolerances (the layer's contract is "bit-exact indices and tables; output
max relative error 2e-2 and cosine >= 0.9999"):

* topk_idx, expert_offsets, sorted_rows, row_pos: bit-exact, except tokens
  whose top-k boundary (or order) lies inside the fp32 summation error bound
  of the router's reduction tree (logit_bounds); for those the GPU's choice
  must be a valid top-k for some logits inside the bounds, and the table must
  satisfy its invariants for the GPU's own choice.
* topk_w: the GPU logits differ from the oracle's correctly rounded ones by
  the fp32 summation error (|dl| <~ 1e-5 here), so w = softmax-renormalised
  differs by |dw| <= 2 |dl| w; the test uses 5e-5 relative + 1e-6 absolute.
* x_lat, z (bf16 results of fp32 sums): at most one bf16 ulp from the oracle,
  a different value in < 2% of the elements (summation order moves a sum
  across a rounding midpoint).
* y (per-route expert rows, fp32): one bf16 ulp flips in h move y by ~1e-4 of
  its norm; per row normwise error <= 2e-3.
* out: normwise max error ||d||_inf / ||ref||_inf <= 2e-2, cosine >= 0.9999,
  and element-wise |d| <= 2e-2 * (|ref| + rms(ref)).
"""
from __future__ import annotations

import numpy as np
import torch

import synth

_HOST_W = {}
_DEV_W = {}


def host_weights(d: synth.Dims) -> dict:
    key = (d.H, d.L, d.I, d.E, d.skewed)
    if key not in _HOST_W:
        _HOST_W.clear()
        _HOST_W[key] = synth.make_weights(d)
    return _HOST_W[key]


def device_weights(d: synth.Dims) -> dict:
    key = (d.H, d.L, d.I, d.E, d.skewed)
    if key not in _DEV_W:
        _DEV_W.clear()
        torch.cuda.empty_cache()
        hw = host_weights(d)
        _DEV_W[key] = {k: (None if v is None else to_dev(v)) for k, v in hw.items()}
    return _DEV_W[key]


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf(a: np.ndarray) -> np.ndarray:
    return synth.bf16_to_f32(a).astype(np.float64)


def ws_for(lm, dims) -> torch.Tensor:
    n = lm.lmoe_workspace_bytes(dims)
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def ws_view(ws: torch.Tensor, off: int, dtype, shape):
    n = int(np.prod(shape))
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).view(*shape)


# ----------------------------------------------------------------------------------------
# comparisons
# ----------------------------------------------------------------------------------------

def logit_bounds(d, absdot, depth=None, extra_depth=0):
    """Rigorous bound on |fp32 GPU logit - correctly rounded logit|: a sum
    evaluated as a tree of depth n has error <= n * u * sum|terms|; the router
    kernel's tree is at most 4*H/128 lane terms + 5 shuffle levels + 16
    split partials deep, plus half an ulp for the oracle's rounding.
    extra_depth adds rounding steps per term (the block's router input)."""
    if depth is None:
        depth = 4 * d.H // 128 + 5 + 16 + extra_depth
    return (depth + 1) * 2.0 ** -24 * absdot


def near_tie_tokens(d, logits, absdot, extra_depth=0):
    """Tokens whose top-k boundary lies within the summation error bound."""
    b = logit_bounds(d, absdot, extra_depth=extra_depth)
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")
    l = logits.astype(np.float64)
    sel = order[:, :d.k]
    rest = order[:, d.k:]
    lo_sel = np.min(np.take_along_axis(l - b, sel, 1), axis=1)
    hi_rest = np.max(np.take_along_axis(l + b, rest, 1), axis=1) if rest.shape[1] else np.full(l.shape[0], -np.inf)
    # also ties inside the top-k (order may swap)
    ls = np.take_along_axis(l, sel, 1)
    bs = np.take_along_axis(b, sel, 1)
    inner = np.any(ls[:, :-1] - ls[:, 1:] <= bs[:, :-1] + bs[:, 1:], axis=1) if d.k > 1 else np.zeros(l.shape[0], bool)
    return np.nonzero((lo_sel <= hi_rest) | inner)[0]


def check_indices(d, gpu_idx, ref_idx, logits, absdot, extra_depth=0):
    """Exact equality outside near-tie tokens; a valid top-k choice inside.
    Returns (flagged tokens, tokens whose GPU choice differs)."""
    flagged = near_tie_tokens(d, logits, absdot, extra_depth)
    ok = np.ones(gpu_idx.shape[0], bool)
    ok[flagged] = False
    bad = np.nonzero((gpu_idx != ref_idx).any(1) & ok)[0]
    assert bad.size == 0, f"index mismatch outside near ties: tokens {bad[:10]}"
    b = logit_bounds(d, absdot, extra_depth=extra_depth)
    l = logits.astype(np.float64)
    for t in flagged:
        S = gpu_idx[t]
        assert len(set(S.tolist())) == d.k and S.min() >= 0 and S.max() < d.E
        notS = np.setdiff1d(np.arange(d.E), S)
        # some logits within the bounds make S the top-k, in this order
        assert np.min(l[t, S] + b[t, S]) >= (np.max(l[t, notS] - b[t, notS]) if notS.size else -np.inf)
        assert np.all(l[t, S[:-1]] + b[t, S[:-1]] >= l[t, S[1:]] - b[t, S[1:]])
    differs = np.nonzero((gpu_idx != ref_idx).any(1))[0]
    return flagged, differs


def check_table_properties(d, idx, off, rows, pos):
    R = d.T * d.k
    flat = idx.reshape(-1)
    assert off[0] == 0 and off[-1] == R and np.array_equal(np.diff(off), np.bincount(flat, minlength=d.E))
    assert np.array_equal(rows, np.argsort(flat, kind="stable"))
    assert np.array_equal(pos[rows], np.arange(R))


def check_bf16_close(got_u16, ref_u16, what, abs_err=None, frac=0.02):
    """bf16 results of fp32 sums: within one bf16 ulp plus `abs_err` (the two
    sides' fp32 summation error bound, which dominates near zero)."""
    g, r = bf(got_u16), bf(ref_u16)
    ulp = np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126))) - 7).astype(np.int64))
    bound = ulp * 1.0001 + (0.0 if abs_err is None else abs_err) + 1e-30
    diff = np.abs(g - r)
    assert np.all(diff <= bound), f"{what}: max diff/bound {np.max(diff / bound)}"
    assert np.mean(got_u16 != ref_u16) < frac, f"{what}: {np.mean(got_u16 != ref_u16):.4f} of elements differ"


def sum_err(K, a_abs, b_abs):
    """Rigorous bound on the difference of two fp32 evaluations of sum_k a*b
    (sequential on one side, a tree on the other): 2 K u sum|a b|."""
    return 2.0 * K * 2.0 ** -24 * (a_abs @ b_abs.T)


def check_rows_normwise(got, ref, tol, what):
    g, r = got.astype(np.float64), ref.astype(np.float64)
    num = np.linalg.norm(g - r, axis=-1)
    den = np.linalg.norm(r, axis=-1) + 1e-30
    assert np.all(num / den <= tol), f"{what}: worst row normwise error {np.max(num / den):.3e}"


def check_out(got_u16, ref_u16, what="out"):
    g, r = bf(got_u16), bf(ref_u16)
    d = g - r
    rel_inf = np.abs(d).max() / max(np.abs(r).max(), 1e-30)
    cos = float((g * r).sum() / (np.linalg.norm(g) * np.linalg.norm(r) + 1e-300))
    rms = np.sqrt((r * r).mean())
    assert rel_inf <= 2e-2, f"{what}: normwise max error {rel_inf:.3e}"
    assert cos >= 0.9999, f"{what}: cosine {cos:.6f}"
    assert np.all(np.abs(d) <= 2e-2 * (np.abs(r) + rms)), f"{what}: element-wise error"
    return rel_inf, cos
