"""Shared helpers for the GPU parity tests: device copies of the seeded inputs,
workspace handling and the comparison rules with their tolerances.

Tolerances (the layer's contract is "bit-exact indices and tables; output
max relative error 2e-2 and cosine >= 0.9999"):

* topk_idx: bit-exact, except tokens whose top-k boundary (or order) lies
  inside the fp32 summation error bound of the router's reduction
  (logit_bounds); for those the GPU's choice must be a valid top-k for some
  logits inside the bounds.  Every such token is counted and recorded
  (record_route), and the configs of the layer's workload list must have
  none.
* expert_offsets, sorted_rows, row_pos: always bit-exact against the
  oracle's table of the GPU's own picks.
* tokens the GPU routed differently are never dropped: their outputs are
  compared with the oracle run on the GPU's routing (forward_routed).
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

def router_regime(d, dense_min_t=64):
    """Which router the library runs for d: the tensor-core GEMM above 16
    tokens from the dense threshold on when the experts fill 32-column
    chunks, else the CUDA-core split-K reduction."""
    return "tensor" if (d.T > 16 and d.T >= dense_min_t and d.E % 32 == 0) else "simt"


def router_depth(d, regime="simt"):
    """Rounding steps per term of the GPU router's fp32 logit sum.
    simt: a lane chain of at most 4*H/128 FMAs, 5 shuffle levels, at most 16
    split partials added in order.  tensor: x against the three bf16 parts of
    each weight, K = 3H split at least four ways; the order inside an MMA is not
    documented, so every product of a split counts as its own step, and each
    step twice (a rounding that truncates), plus at most 16 split partials."""
    if regime == "tensor":
        return 2 * (3 * d.H // 4) + 16
    return 4 * d.H // 128 + 5 + 16


def logit_bounds(d, absdot, depth=None, extra_depth=0, regime="simt"):
    """Rigorous bound on |fp32 GPU logit - correctly rounded logit|: a sum
    evaluated with at most n rounding steps per term has error <= n * u *
    sum|terms|, plus half an ulp for the oracle's rounding.  extra_depth adds
    rounding steps per term (the block's router input)."""
    if depth is None:
        depth = router_depth(d, regime) + extra_depth
    return (depth + 1) * 2.0 ** -24 * absdot


def boundary_gaps(d, logits):
    """Per token: the gap between the k-th and (k+1)-th largest logit (inf
    when k = E) and the smallest gap between consecutive picks."""
    l = np.sort(logits.astype(np.float64), axis=1)[:, ::-1]
    kth = l[:, d.k - 1] - l[:, d.k] if d.k < d.E else np.full(l.shape[0], np.inf)
    inner = np.min(l[:, :d.k - 1] - l[:, 1:d.k], axis=1) if d.k > 1 else np.full(l.shape[0], np.inf)
    return kth, inner


def near_tie_tokens(d, logits, absdot, extra_depth=0, regime="simt"):
    """Tokens whose top-k boundary (or the order inside the top k) lies within
    the summation error bound."""
    b = logit_bounds(d, absdot, extra_depth=extra_depth, regime=regime)
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


def check_indices(d, gpu_idx, ref_idx, logits, absdot, extra_depth=0, regime="simt"):
    """Exact equality outside near-tie tokens; a valid top-k choice inside.
    Returns (flagged tokens, tokens whose GPU choice differs)."""
    flagged = near_tie_tokens(d, logits, absdot, extra_depth, regime)
    ok = np.ones(gpu_idx.shape[0], bool)
    ok[flagged] = False
    bad = np.nonzero((gpu_idx != ref_idx).any(1) & ok)[0]
    assert bad.size == 0, f"index mismatch outside near ties: tokens {bad[:10]}"
    b = logit_bounds(d, absdot, extra_depth=extra_depth, regime=regime)
    l = logits.astype(np.float64)
    differs = np.nonzero((gpu_idx != ref_idx).any(1))[0]
    for t in differs:
        S = gpu_idx[t]
        assert len(set(S.tolist())) == d.k and S.min() >= 0 and S.max() < d.E
        notS = np.setdiff1d(np.arange(d.E), S)
        # some logits within the bounds make S the top-k, in this order
        assert np.min(l[t, S] + b[t, S]) >= (np.max(l[t, notS] - b[t, notS]) if notS.size else -np.inf)
        assert np.all(l[t, S[:-1]] + b[t, S[:-1]] >= l[t, S[1:]] - b[t, S[1:]])
    return flagged, differs


def weights_at(logits, idx):
    """Softmax over all experts renormalised over the picks idx, in fp64, from
    the oracle's logits: the weights the oracle gives when it picks idx."""
    l = logits.astype(np.float64)
    sel = np.take_along_axis(l, idx.astype(np.int64), 1)
    p = np.exp(sel - sel.max(axis=1, keepdims=True))
    return p / p.sum(axis=1, keepdims=True)


def record_route(label, d, regime, logits, absdot, flagged, differs, extra_depth=0):
    """One line per routed config into $LMOE_RECORD_DIR/route_record.jsonl (when
    set): how many tokens lie inside the bound and how many the GPU routed
    differently, with the logit gap at the top-k boundary and the bound there."""
    import json
    import os
    out_dir = os.environ.get("LMOE_RECORD_DIR")
    kth, inner = boundary_gaps(d, logits)
    b = logit_bounds(d, absdot, extra_depth=extra_depth, regime=regime)
    bmax = b.max(axis=1)
    ratio = np.minimum(kth, inner) / np.maximum(bmax, 1e-300)
    t_min = int(np.argmin(ratio))
    rec = {"config": label, "T": int(d.T), "E": int(d.E), "k": int(d.k), "regime": regime,
           "flagged": int(len(flagged)), "differs": int(len(differs)),
           "closest_token": t_min, "closest_gap": float(min(kth[t_min], inner[t_min])),
           "closest_bound": float(bmax[t_min]),
           "differing": [{"t": int(t), "gap": float(min(kth[t], inner[t])), "bound": float(bmax[t])}
                         for t in differs[:32]]}
    if out_dir:
        os.makedirs(out_dir, exist_ok=True)
        with open(os.path.join(out_dir, "route_record.jsonl"), "a") as f:
            f.write(json.dumps(rec) + "\n")
    return rec


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
