"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and the shared tiny-shape
case and raises AssertionError on a mismatch.  ``test_oracle_pins.py`` runs
them on the default oracle (all must pass) and on builds with one planted
mistake each (at least one must fail).

What pins what:
  * E2M1 / E8M0 decode  -> the OCP MX v1.0 tables in tests/golden and the
    closed form of the format (exhaustive over code x scale)
  * bf16 rounding       -> torch's fp32 -> bfloat16 conversion
  * router + top-k      -> fp64 numpy logits, a stable full sort, and the
    identity "softmax over all then renormalise == softmax over the selected"
  * routing table       -> permutation / histogram / order invariants and a
    numpy stable argsort
  * pooler, unpooler    -> fp64 numpy matmuls (textbook GEMMs)
  * experts             -> brute-force dense evaluation of EVERY expert for
    every token in fp64 from an independent numpy dequantiser, then gathered
    per (token, route) row ("each (token, route) pair is its own row")
  * norm / combine      -> RMS of each normed row, an fp64 recomputation of
    the per-route norm, an fp32 re-summation in route order, the
    "norm of a partial sum is wrong" control and "non-local rows are exact
    zeros" ("Muse Spark Open on Gaudi 2", "EP and TP layout")

The sandwich block around the layer ("Soporte de dia 0 ...", "Normalizacion
en sandwich") is pinned by BLOCK_PINS:
  * row RMSNorm         -> with eps = 0: bitwise invariance under a power-of-two
    scale of the row, and RMS(out / g) = 1 for every row
  * fp32-input router   -> bitwise equal to the pinned bf16-input router on
    bf16-representable input; fp64 numpy logits on arbitrary fp32 input
  * block               -> a zero post-norm gain or a zero unpooler gives y = x
    exactly; with eps = 0 the layer output does not change when x is scaled by
    a power of two (the norm comes first); token independence

NVFP4 expert weights (NV_PINS):
  * E4M3 decode         -> torch's float8_e4m3fn conversion over all 256 bytes and
    the OCP FP8 values in tests/golden
  * E2M1 x E4M3         -> exact in fp32 and bf16 for every code and scale byte
  * experts             -> brute-force dense evaluation from an independent numpy
    NVFP4 dequantiser (16-element blocks, per-matrix global scale)
  * global scale        -> doubling an expert's W2 global scale doubles its y rows exactly
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EPS32 = 2.0 ** -24  # unit roundoff of fp32


def golden_e2m1() -> np.ndarray:
    vals = np.zeros(16, np.float64)
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                c, v = line.split()
                vals[int(c)] = float(v)
    return vals


def golden_e8m0() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "e8m0_ocp_mx.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                b, e = line.split()
                out[int(b)] = e
    return out


# --------------------------------------------------------------------------------------
# independent numpy helpers (no oracle code)
# --------------------------------------------------------------------------------------

def bf16_to_f64(a):
    return synth.bf16_to_f32(a).astype(np.float64)


def f32_to_bf16_torch(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits through torch's conversion (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (v given as float64)."""
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def dequant_dense(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """[..., N, K/2] codes + [..., N, K/32] scales -> fp64 [..., N, K], per the
    OCP MX layout: element 2m is the low nibble of byte m, 2m+1 the high one."""
    table = golden_e2m1()
    lo = table[q & 15]
    hi = table[q >> 4]
    codes = np.stack([lo, hi], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    return codes * np.repeat(scale, 32, axis=-1)


class Case:
    """A tiny-shape layer instance with all oracle stages evaluated."""

    def __init__(self, o, d: synth.Dims, x, w):
        self.d, self.x, self.w = d, x, w
        self.logits, self.absdot = o.router_logits(d, x, w["router_w"], w["router_bias"], want_absdot=True)
        self.idx, self.tw = o.topk(d, self.logits)
        self.offsets, self.sorted_rows, self.row_pos = o.table(d, self.idx)
        self.x_lat = o.pool(d, x, w["pooler_w"])
        self.y, self.h, self.gu = o.experts(d, self.x_lat, self.idx, w, want_intermediates=True)
        self.z, self.yhat = o.norm_combine(d, self.y, self.idx, self.tw, w["norm_g"], want_yhat=True)
        self.out = o.unpool(d, self.z, w["unpooler_w"])


def make_case(o, T=16, seed=0, d=None, w=None, skewed=False):
    d = d or synth.with_tokens(synth.CONFIGS["tiny"], T)
    if skewed:
        from dataclasses import replace
        d = replace(d, skewed=True)
    w = w or synth.make_weights(d, seed)
    x = synth.make_x(d, seed)
    return Case(o, d, x, w)


# --------------------------------------------------------------------------------------
# pins
# --------------------------------------------------------------------------------------

def pin_e2m1_golden(o, c):
    table = golden_e2m1()
    for code in range(16):
        v = o.mxfp4_value(code, 127)
        assert v == table[code], (code, v, table[code])
        assert math.copysign(1.0, v) == math.copysign(1.0, table[code]), ("sign", code)
    for b, e in golden_e8m0().items():
        v = o.mxfp4_value(2, b)  # code 2 is 1.0
        if e == "nan":
            assert math.isnan(v)
        else:
            assert v == math.ldexp(1.0, int(e)), (b, v, e)


def pin_mxfp4_closed_form(o, c):
    for s in range(0, 253):
        for code in range(16):
            sign = -1.0 if code & 8 else 1.0
            E, M = (code >> 1) & 3, code & 1
            mag = M * 0.5 if E == 0 else math.ldexp(1.0 + 0.5 * M, E - 1)
            ref = sign * math.ldexp(mag, s - 127)
            v = o.mxfp4_value(code, s)
            assert v == ref, (code, s, v, ref)
            # every product is exactly representable in bf16 (W4A16 dequant is exact)
            bits = np.array([v], np.float32).view(np.uint32)[0]
            assert bits & 0xFFFF == 0, (code, s)


def pin_bf16_rne(o, c):
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2 ** 16, size=4000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    near = (rng.integers(0, 2 ** 16, size=4000, dtype=np.uint64).astype(np.uint32) << 16) | \
        rng.choice(np.array([0x7FFF, 0x8001, 0x0000, 0xFFFF], np.uint32), size=4000)
    special = np.array([0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x00000001, 0x80000000, 0], np.uint32)
    allp = np.concatenate([pats, ties, near, special])
    f = allp.view(np.float32)
    keep = ~np.isnan(f)
    f = f[keep]
    ref = f32_to_bf16_torch(f)
    got = np.array([o.bf16_rne(float(v)) for v in f], np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(hex(f[i:i + 1].view(np.uint32)[0]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def pin_router_fp64(o, c):
    x64 = bf16_to_f64(c.x)
    lg = (x64 @ c.w["router_w"].astype(np.float64).T).astype(np.float32)
    if c.w["router_bias"] is not None:
        lg = lg + c.w["router_bias"]
    assert np.array_equal(lg, c.logits), np.abs(lg - c.logits).max()


def pin_topk_bruteforce(o, c):
    d = c.d
    order = np.argsort(-c.logits.astype(np.float64), axis=1, kind="stable")[:, :d.k]
    assert np.array_equal(order, c.idx)
    sel = np.take_along_axis(c.logits.astype(np.float64), order, axis=1)
    p = np.exp(sel - sel.max(axis=1, keepdims=True))
    ref = p / p.sum(axis=1, keepdims=True)
    assert np.allclose(c.tw, ref, rtol=2.5e-7, atol=0), np.abs(c.tw - ref).max()
    # ties: equal logits keep the lower index first
    tie = np.zeros((1, d.E), np.float32)
    tie[0, [3, 5, 9, 12, 14]] = 2.0
    tie[0, [1, 7, 11]] = 1.0
    idx, _ = o.topk(d, tie)
    assert list(idx[0, :min(d.k, 8)]) == [3, 5, 9, 12, 14, 1, 7, 11][:d.k], idx


def pin_table(o, c):
    d = c.d
    R = d.T * d.k
    flat = c.idx.reshape(-1)
    assert c.offsets[0] == 0 and c.offsets[-1] == R and np.all(np.diff(c.offsets) >= 0)
    assert np.array_equal(np.diff(c.offsets), np.bincount(flat, minlength=d.E))
    assert np.array_equal(np.sort(c.sorted_rows), np.arange(R))
    assert np.array_equal(c.sorted_rows, np.argsort(flat, kind="stable"))
    assert np.array_equal(c.row_pos[c.sorted_rows], np.arange(R))
    for e in range(d.E):
        rows = c.sorted_rows[c.offsets[e]:c.offsets[e + 1]]
        assert np.all(flat[rows] == e) and np.all(np.diff(rows) > 0)


def pin_pool_textbook(o, c):
    ref = bf16_to_f64(c.x) @ bf16_to_f64(c.w["pooler_w"]).T
    got = bf16_to_f64(c.x_lat)
    diff = np.abs(got - ref)
    bound = bf16_ulp(ref) * 0.5 + c.d.H * EPS32 * (np.abs(bf16_to_f64(c.x)) @ np.abs(bf16_to_f64(c.w["pooler_w"])).T)
    assert np.all(diff <= bound), (diff / bound).max()
    assert np.mean(c.x_lat != f32_to_bf16_torch(ref.astype(np.float32))) < 0.02


def pin_experts_dense(o, c):
    """Per-route rows equal a brute-force dense evaluation of all experts."""
    d = c.d
    W13 = dequant_dense(c.w["w13_q"], c.w["w13_s"])   # [E][2I][L]
    W2 = dequant_dense(c.w["w2_q"], c.w["w2_s"])      # [E][L][I]
    xl = bf16_to_f64(c.x_lat)                          # [T][L]
    # every expert, every token (dense), then gather the routed (t, e) pairs
    G_all = np.einsum("tl,efl->tef", xl, W13)          # [T][E][2I]
    A_all = np.einsum("tl,efl->tef", np.abs(xl), np.abs(W13))
    t_of_r = np.arange(d.T * d.k) // d.k
    e_of_r = c.idx.reshape(-1)
    G = G_all[t_of_r, e_of_r]
    A = A_all[t_of_r, e_of_r]
    assert np.all(np.abs(c.gu.astype(np.float64) - G) <= d.L * EPS32 * A + 1e-30), \
        np.max(np.abs(c.gu - G) / (A + 1e-30))
    g, u = G[:, :d.I], G[:, d.I:]
    h_ref = g / (1.0 + np.exp(-g)) * u
    h_got = bf16_to_f64(c.h)
    assert np.all(np.abs(h_got - h_ref) <= bf16_ulp(h_ref) * 0.5 + 1e-4 * np.abs(h_ref) + 1e-30)
    # y from the oracle's own h against the dense W2 of the routed expert
    Y = np.einsum("ri,rli->rl", h_got, W2[e_of_r])
    B = np.einsum("ri,rli->rl", np.abs(h_got), np.abs(W2[e_of_r]))
    assert np.all(np.abs(c.y.astype(np.float64) - Y) <= d.I * EPS32 * B + 1e-30)


def pin_norm_per_route(o, c):
    d = c.d
    R = d.T * d.k
    e_of_r = c.idx.reshape(-1)
    y = c.y.astype(np.float64)
    g = bf16_to_f64(c.w["norm_g"])[e_of_r]
    rinv = 1.0 / np.sqrt((y * y).mean(axis=1, keepdims=True) + d.eps)
    ref = y * rinv * g
    assert np.allclose(c.yhat, ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max()), np.abs(c.yhat - ref).max()
    rms = np.sqrt(((c.yhat / g) ** 2).mean(axis=1))
    assert np.all(np.abs(rms - 1.0) < 1e-5), rms
    # fp32 weighted sum in route order reproduces z bit for bit
    z = np.zeros((d.T, d.L), np.float32)
    for j in range(d.k):
        z = z + c.tw[:, j:j + 1] * c.yhat[np.arange(d.T) * d.k + j]
    assert np.array_equal(z, c.z)
    # negative control: normalising the sum instead of each route is far off
    zs = np.zeros((d.T, d.L), np.float64)
    for j in range(d.k):
        zs += c.tw[:, j:j + 1].astype(np.float64) * y[np.arange(d.T) * d.k + j] * g[np.arange(d.T) * d.k + j]
    zs = zs / np.sqrt((zs * zs).mean(axis=1, keepdims=True) + d.eps)
    assert np.abs(zs - c.z).max() > 1e-2 * np.abs(c.z).max()
    assert R == c.yhat.shape[0]


def pin_sharded_invariants(o, c):
    """EP2 x TP2 emulation: the all-reduce of partial per-route rows (non-local
    rows exact zeros) reproduces the unsharded rows, and a norm taken before the
    all-reduce (of a partial sum) is wrong."""
    d = c.d
    e_of_r = c.idx.reshape(-1)
    W2 = dequant_dense(c.w["w2_q"], c.w["w2_s"])
    h = bf16_to_f64(c.h)
    half = d.I // 2
    parts = []
    for ep in range(2):
        local = (e_of_r // (d.E // 2)) == ep
        for tp in range(2):
            sl = slice(tp * half, (tp + 1) * half)
            p = np.einsum("ri,rli->rl", h[:, sl], W2[e_of_r][:, :, sl])
            p[~local] = 0.0                       # non-local rows are exact zeros
            parts.append(p.astype(np.float32))
    red = np.zeros_like(parts[0])
    for p in parts:
        red = red + p                             # the fp32 all-reduce
    B = np.einsum("ri,rli->rl", np.abs(h), np.abs(W2[e_of_r]))
    assert np.all(np.abs(red.astype(np.float64) - c.y) <= 2 * d.I * EPS32 * B + 1e-30)
    z_red = o.norm_combine(d, red, c.idx, c.tw, c.w["norm_g"])
    assert np.allclose(z_red, c.z, rtol=1e-3, atol=1e-4 * np.abs(c.z).max())
    # control: each card normalises its partial rows before the all-reduce
    g = bf16_to_f64(c.w["norm_g"])[e_of_r]
    wrong = sum(p.astype(np.float64) / np.sqrt((p.astype(np.float64) ** 2).mean(axis=1, keepdims=True) + d.eps)
                for p in parts) * g
    z_wrong = np.zeros((d.T, d.L))
    for j in range(d.k):
        z_wrong += c.tw[:, j:j + 1] * wrong[np.arange(d.T) * d.k + j]
    assert np.abs(z_wrong - c.z).max() > 1e-2 * np.abs(c.z).max()


def pin_unpool_textbook(o, c):
    zb = f32_to_bf16_torch(c.z)
    ref = bf16_to_f64(zb) @ bf16_to_f64(c.w["unpooler_w"]).T
    got = bf16_to_f64(c.out)
    bound = bf16_ulp(ref) * 0.5 + c.d.L * EPS32 * (np.abs(bf16_to_f64(zb)) @ np.abs(bf16_to_f64(c.w["unpooler_w"])).T)
    assert np.all(np.abs(got - ref) <= bound)


def pin_w2_scale_invariance(o, c):
    """+1 on every W2 scale byte doubles y exactly; after the per-route norm
    the layer output moves only through eps."""
    d = c.d
    w2 = dict(c.w)
    w2["w2_s"] = (c.w["w2_s"] + 1).astype(np.uint8)
    y2 = o.experts(d, c.x_lat, c.idx, w2)
    assert np.array_equal(y2, 2.0 * c.y)
    z2 = o.norm_combine(d, y2, c.idx, c.tw, c.w["norm_g"])
    assert np.allclose(z2, c.z, rtol=1e-5, atol=1e-6 * np.abs(c.z).max())


def pin_identical_experts(o, c):
    """With every expert identical, z equals one normed route row (sum w = 1)."""
    d = c.d
    w = dict(c.w)
    for key in ("w13_q", "w13_s", "w2_q", "w2_s", "norm_g"):
        w[key] = np.ascontiguousarray(np.broadcast_to(c.w[key][:1], c.w[key].shape))
    y = o.experts(d, c.x_lat, c.idx, w)
    z, yhat = o.norm_combine(d, y, c.idx, c.tw, w["norm_g"], want_yhat=True)
    first = yhat[np.arange(d.T) * d.k]
    assert np.allclose(z, first, rtol=4 * d.k * EPS32 * 2, atol=4 * d.k * EPS32 * np.abs(first).max())


PINS = [pin_e2m1_golden, pin_mxfp4_closed_form, pin_bf16_rne, pin_router_fp64, pin_topk_bruteforce,
        pin_table, pin_pool_textbook, pin_experts_dense, pin_norm_per_route, pin_sharded_invariants,
        pin_unpool_textbook, pin_w2_scale_invariance, pin_identical_experts]


# --------------------------------------------------------------------------------------
# the sandwich block
# --------------------------------------------------------------------------------------

class BlockCase:
    def __init__(self, o, d, x, w, nw):
        self.d, self.x, self.w, self.nw = d, x, w, nw
        self.r = o.block_forward(d, x, w, nw)


def make_block_case(o, T=12, seed=0):
    d = synth.with_tokens(synth.CONFIGS["tiny"], T)
    return BlockCase(o, d, synth.make_x(d, seed), synth.make_weights(d, seed), synth.make_block_norms(d, seed))


def pin_rmsnorm_invariants(o, c):
    x, g = c.x, c.nw["pre_g"]
    a = o.rmsnorm(x, g, 0.0)
    # a power-of-two scale of a row is exact in bf16 and cancels exactly in the norm
    for k in (-3, 5):
        xs = f32_to_bf16_torch(np.ldexp(bf16_to_f64(x), k).astype(np.float32))
        assert np.array_equal(bf16_to_f64(xs), np.ldexp(bf16_to_f64(x), k))
        assert np.array_equal(o.rmsnorm(xs, g, 0.0), a), k
    # RMS over the row of out / g is one (mean over the W columns, the gain applied per column)
    ratio = a.astype(np.float64) / bf16_to_f64(g)[None, :]
    rms = np.sqrt((ratio * ratio).mean(1))
    assert np.all(np.abs(rms - 1.0) <= (x.shape[1] + 16) * EPS32), np.abs(rms - 1.0).max()
    # eps enters inside the square root
    e = 0.25
    b = o.rmsnorm(x, g, e).astype(np.float64) / bf16_to_f64(g)[None, :]
    x64 = bf16_to_f64(x)
    want = x64 / np.sqrt((x64 * x64).mean(1, keepdims=True) + e)
    assert np.allclose(b, want, rtol=(x.shape[1] + 16) * EPS32, atol=0), np.abs(b - want).max()


def pin_router_f32_input(o, c):
    d, w = c.d, c.w
    # bf16-representable fp32 input: the fp32-input router equals the bf16-input one
    xf = synth.bf16_to_f32(c.x)
    la, aa = o.router_logits(d, c.x, w["router_w"], w["router_bias"], want_absdot=True)
    lb, ab = o.router_logits_f32(d, xf, w["router_w"], w["router_bias"], want_absdot=True)
    assert np.array_equal(la, lb) and np.array_equal(aa, ab)
    # arbitrary fp32 input (the block's pre-norm output): fp64 numpy logits
    n = c.r["n"]
    ref = (n.astype(np.float64) @ w["router_w"].astype(np.float64).T).astype(np.float32)
    if w["router_bias"] is not None:
        ref = ref + w["router_bias"]
    assert np.array_equal(ref, c.r["logits"]), np.abs(ref - c.r["logits"]).max()


def pin_block_identity_paths(o, c):
    d = c.d
    zero_post = dict(c.nw, post_g=np.zeros_like(c.nw["post_g"]))
    r = o.block_forward(d, c.x, c.w, zero_post)
    assert np.array_equal(r["y"], c.x), "post-norm gain 0 must leave the residual stream unchanged"
    w0 = dict(c.w, unpooler_w=np.zeros_like(c.w["unpooler_w"]))
    r = o.block_forward(d, c.x, w0, c.nw)
    assert np.all(r["out"] == 0) and np.array_equal(r["y"], c.x), "a zero layer output must give y = x"
    # the residual is added to the block input, not to the normalised input
    assert not np.array_equal(c.r["y"], o.residual_add(c.r["nb"], np.zeros(c.x.shape, np.float32)))


def pin_block_norm_first(o, c):
    d = c.d
    a = o.block_forward(d, c.x, c.w, c.nw, eps=0.0)
    xs = f32_to_bf16_torch(np.ldexp(bf16_to_f64(c.x), 4).astype(np.float32))
    b = o.block_forward(d, xs, c.w, c.nw, eps=0.0)
    assert np.array_equal(a["n"], b["n"]) and np.array_equal(a["out"], b["out"])
    assert not np.array_equal(a["y"], b["y"])


def pin_block_token_independence(o, c):
    d3 = synth.with_tokens(c.d, 3)
    r = o.block_forward(d3, c.x[:3].copy(), c.w, c.nw)
    assert np.array_equal(r["y"], c.r["y"][:3])


BLOCK_PINS = [pin_rmsnorm_invariants, pin_router_f32_input, pin_block_identity_paths, pin_block_norm_first,
              pin_block_token_independence]


# --------------------------------------------------------------------------------------
# NVFP4 expert weights
# --------------------------------------------------------------------------------------

def golden_e4m3() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "e4m3_ocp_fp8.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                b, v = line.split()
                out[int(b, 16)] = float(v)
    return out


def e4m3_torch(b: np.ndarray) -> np.ndarray:
    """E4M3 bytes -> fp64 through torch's float8_e4m3fn conversion."""
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def dequant_dense_nvfp4(q: np.ndarray, s: np.ndarray, gs: np.ndarray) -> np.ndarray:
    """[E, N, K/2] codes + [E, N, K/16] E4M3 scales + [E] global scales -> fp64
    [E, N, K]: element 2m is the low nibble of byte m, 2m+1 the high one."""
    table = golden_e2m1()
    codes = np.stack([table[q & 15], table[q >> 4]], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    scale = np.repeat(e4m3_torch(s), 16, axis=-1)
    return codes * scale * gs.astype(np.float64)[:, None, None]


class NvCase:
    def __init__(self, o, d, x, w):
        self.d, self.x, self.w = d, x, w
        lg = o.router_logits(d, x, w["router_w"], w["router_bias"])
        self.idx, self.tw = o.topk(d, lg)
        self.x_lat = o.pool(d, x, w["pooler_w"])
        self.y, self.h, self.gu = o.experts_nvfp4(d, self.x_lat, self.idx, w, want_intermediates=True)


def make_nv_case(o, T=16, seed=0):
    d = synth.with_tokens(synth.CONFIGS["tiny"], T)
    return NvCase(o, d, synth.make_x(d, seed), synth.make_weights_nvfp4(d, seed))


def pin_e4m3_decode(o, c):
    ref = e4m3_torch(np.arange(256, dtype=np.uint8))
    for b in range(256):
        v = o.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(v), b
        else:
            assert v == ref[b] and math.copysign(1.0, v) == math.copysign(1.0, ref[b]), (b, v, ref[b])
    for b, v in golden_e4m3().items():
        got = o.e4m3_value(b)
        assert (math.isnan(got) and math.isnan(v)) or (got == v and math.copysign(1, got) == math.copysign(1, v)), b


def pin_nvfp4_products_exact(o, c):
    table = golden_e2m1()
    sc = e4m3_torch(np.arange(256, dtype=np.uint8))
    for b in range(256):
        if math.isnan(sc[b]):
            continue
        for code in range(16):
            v = o.nvfp4_value(code, b)
            assert v == table[code] * sc[b], (code, b)
            bits = np.array([v], np.float32).view(np.uint32)[0]
            assert bits & 0xFFFF == 0, (code, b)  # exact in bf16 as well


def pin_experts_nvfp4_dense(o, c):
    d, w = c.d, c.w
    W13 = dequant_dense_nvfp4(w["w13_q"], w["w13_s"], w["w13_gs"])
    W2 = dequant_dense_nvfp4(w["w2_q"], w["w2_s"], w["w2_gs"])
    xl = bf16_to_f64(c.x_lat)
    t_of_r = np.arange(d.T * d.k) // d.k
    e_of_r = c.idx.reshape(-1)
    G = np.einsum("rl,rfl->rf", xl[t_of_r], W13[e_of_r])
    A = np.einsum("rl,rfl->rf", np.abs(xl[t_of_r]), np.abs(W13[e_of_r]))
    # one more rounding per term: the fp32 product with the global scale
    assert np.all(np.abs(c.gu.astype(np.float64) - G) <= (d.L + 2) * EPS32 * A + 1e-30), \
        np.max(np.abs(c.gu - G) / (A + 1e-30))
    h_got = bf16_to_f64(c.h)
    Y = np.einsum("ri,rli->rl", h_got, W2[e_of_r])
    B = np.einsum("ri,rli->rl", np.abs(h_got), np.abs(W2[e_of_r]))
    assert np.all(np.abs(c.y.astype(np.float64) - Y) <= (d.I + 2) * EPS32 * B + 1e-30)


def pin_nvfp4_global_scale(o, c):
    w2 = dict(c.w, w2_gs=(c.w["w2_gs"] * 2).astype(np.float32))
    y2 = o.experts_nvfp4(c.d, c.x_lat, c.idx, w2)
    assert np.array_equal(y2, c.y * 2)


NV_PINS = [pin_e4m3_decode, pin_nvfp4_products_exact, pin_experts_nvfp4_dense, pin_nvfp4_global_scale]
