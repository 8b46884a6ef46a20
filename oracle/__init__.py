"""ctypes binding of the plain-C CPU oracle (``lmoe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the product path never
does.  The oracle shares no code with the CUDA library.  See the header of
``lmoe_oracle.c`` for what each stage computes and which passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lmoe_oracle.c")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


class OrDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32),
                ("I", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("eps", ctypes.c_float)]


def lib_path(plant: int = 0) -> str:
    return os.path.join(_HERE, "liblmoe_oracle.so" if plant == 0 else f"liblmoe_oracle_plant{plant}.so")


def build(plant: int = 0, force: bool = False) -> str:
    out = lib_path(plant)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".{os.getpid()}.tmp"
        flags = CFLAGS + ([f"-DLMOE_ORACLE_PLANT={plant}"] if plant else [])
        subprocess.check_call(["gcc", *flags, _SRC, "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, out)
    return out


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags.c_contiguous, "oracle wants C-contiguous numpy arrays"
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """One loaded oracle library (the default build, or a planted-mistake variant)."""

    def __init__(self, plant: int = 0, threads: int | None = None):
        self.lib = ctypes.CDLL(build(plant))
        L = self.lib
        vp, dp = ctypes.c_void_p, ctypes.POINTER(OrDims)
        L.oracle_bf16_rne.argtypes = [ctypes.c_float]
        L.oracle_bf16_rne.restype = ctypes.c_uint16
        L.oracle_mxfp4_value.argtypes = [ctypes.c_uint, ctypes.c_uint]
        L.oracle_mxfp4_value.restype = ctypes.c_float
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_get_threads.restype = ctypes.c_int
        L.oracle_router_logits.argtypes = [dp, vp, vp, vp, vp, vp]
        L.oracle_topk.argtypes = [dp, vp, vp, vp]
        L.oracle_table.argtypes = [dp, vp, vp, vp, vp]
        L.oracle_pool.argtypes = [dp, vp, vp, vp]
        L.oracle_experts.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.oracle_norm_combine.argtypes = [dp, vp, vp, vp, vp, vp, vp]
        L.oracle_unpool.argtypes = [dp, vp, vp, vp]
        L.oracle_forward.argtypes = [dp] + [vp] * 16
        L.oracle_router_logits_f32.argtypes = [dp, vp, vp, vp, vp, vp]
        i64 = ctypes.c_int64
        L.oracle_rmsnorm_rows.argtypes = [i64, i64, vp, vp, ctypes.c_float, vp]
        L.oracle_bf16_round.argtypes = [i64, vp, vp]
        L.oracle_residual_add.argtypes = [i64, vp, vp, vp]
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint]
        L.oracle_e4m3_value.restype = ctypes.c_float
        L.oracle_nvfp4_value.argtypes = [ctypes.c_uint, ctypes.c_uint]
        L.oracle_nvfp4_value.restype = ctypes.c_float
        L.oracle_experts_nvfp4.argtypes = [dp] + [vp] * 11
        L.oracle_experts_nvfp4.restype = None
        L.oracle_set_acc64.argtypes = [ctypes.c_int]
        L.oracle_set_acc64.restype = None
        L.oracle_get_acc64.restype = ctypes.c_int
        for f in ("oracle_router_logits", "oracle_topk", "oracle_table", "oracle_pool", "oracle_experts",
                  "oracle_norm_combine", "oracle_unpool", "oracle_forward", "oracle_set_threads",
                  "oracle_router_logits_f32", "oracle_rmsnorm_rows", "oracle_bf16_round", "oracle_residual_add"):
            getattr(L, f).restype = None
        self.set_threads(threads if threads else max(1, min(64, os.cpu_count() or 1)))

    def set_threads(self, n: int):
        self.lib.oracle_set_threads(int(n))

    @property
    def threads(self) -> int:
        return self.lib.oracle_get_threads()

    def set_acc64(self, on: bool):
        """Sums in fp64 instead of fp32 (rounded at the same points): a diagnostic of
        the oracle's own accumulation error, never the reference result."""
        self.lib.oracle_set_acc64(1 if on else 0)

    def error_report(self, d, x, w) -> dict:
        """The oracle's own fp32 accumulation error: normwise relative difference of
        each stage's result between fp32 sums and fp64 sums, on the same input."""
        a = self.forward(d, x, w)
        self.set_acc64(True)
        try:
            b = self.forward(d, x, w)
        finally:
            self.set_acc64(False)

        out = {}
        for key in ("x_lat", "y", "z", "out"):
            u, v = a[key], b[key]
            if u.dtype == np.uint16:
                u = (u.astype(np.uint32) << 16).view(np.float32)
                v = (v.astype(np.uint32) << 16).view(np.float32)
            u, v = u.astype(np.float64), v.astype(np.float64)
            out[key] = float(np.linalg.norm(u - v) / (np.linalg.norm(v) + 1e-300))
        out["topk_idx_same"] = bool(np.array_equal(a["topk_idx"], b["topk_idx"]))
        return out

    @staticmethod
    def dims(d, T: int | None = None) -> OrDims:
        return OrDims(d.T if T is None else T, d.H, d.L, d.I, d.E, d.k, d.eps)

    # -- number formats -------------------------------------------------------------
    def bf16_rne(self, f: float) -> int:
        return int(self.lib.oracle_bf16_rne(f))

    def mxfp4_value(self, code: int, scale: int) -> float:
        return float(self.lib.oracle_mxfp4_value(code, scale))

    def e4m3_value(self, b: int) -> float:
        return float(self.lib.oracle_e4m3_value(b))

    def nvfp4_value(self, code: int, scale_byte: int) -> float:
        return float(self.lib.oracle_nvfp4_value(code, scale_byte))

    # -- stages ---------------------------------------------------------------------
    def router_logits(self, d, x, router_w, router_bias=None, want_absdot=False):
        od = self.dims(d, x.shape[0])
        logits = np.empty((od.T, d.E), np.float32)
        absdot = np.empty((od.T, d.E), np.float64) if want_absdot else None
        self.lib.oracle_router_logits(ctypes.byref(od), _p(x), _p(router_w), _p(router_bias), _p(logits), _p(absdot))
        return (logits, absdot) if want_absdot else logits

    def topk(self, d, logits):
        od = self.dims(d, logits.shape[0])
        idx = np.empty((od.T, d.k), np.int32)
        w = np.empty((od.T, d.k), np.float32)
        self.lib.oracle_topk(ctypes.byref(od), _p(np.ascontiguousarray(logits)), _p(idx), _p(w))
        return idx, w

    def table(self, d, topk_idx):
        od = self.dims(d, topk_idx.shape[0])
        R = od.T * d.k
        offsets = np.empty(d.E + 1, np.int32)
        sorted_rows = np.empty(R, np.int32)
        row_pos = np.empty(R, np.int32)
        self.lib.oracle_table(ctypes.byref(od), _p(np.ascontiguousarray(topk_idx)), _p(offsets), _p(sorted_rows), _p(row_pos))
        return offsets, sorted_rows, row_pos

    def pool(self, d, x, pooler_w):
        od = self.dims(d, x.shape[0])
        x_lat = np.empty((od.T, d.L), np.uint16)
        self.lib.oracle_pool(ctypes.byref(od), _p(x), _p(pooler_w), _p(x_lat))
        return x_lat

    def experts(self, d, x_lat, topk_idx, w, want_intermediates=False):
        od = self.dims(d, x_lat.shape[0])
        R = od.T * d.k
        y = np.empty((R, d.L), np.float32)
        h = np.empty((R, d.I), np.uint16) if want_intermediates else None
        gu = np.empty((R, 2 * d.I), np.float32) if want_intermediates else None
        self.lib.oracle_experts(ctypes.byref(od), _p(x_lat), _p(np.ascontiguousarray(topk_idx)),
                                _p(w["w13_q"]), _p(w["w13_s"]), _p(w["w2_q"]), _p(w["w2_s"]), _p(h), _p(gu), _p(y))
        return (y, h, gu) if want_intermediates else y

    def experts_nvfp4(self, d, x_lat, topk_idx, w, want_intermediates=False):
        """The experts on NVFP4 weights: w holds w13_q, w13_s (E4M3 [E][2I][L/16]),
        w13_gs (fp32 [E]), w2_q, w2_s ([E][L][I/16]) and w2_gs."""
        od = self.dims(d, x_lat.shape[0])
        R = od.T * d.k
        y = np.empty((R, d.L), np.float32)
        h = np.empty((R, d.I), np.uint16) if want_intermediates else None
        gu = np.empty((R, 2 * d.I), np.float32) if want_intermediates else None
        self.lib.oracle_experts_nvfp4(ctypes.byref(od), _p(x_lat), _p(np.ascontiguousarray(topk_idx)),
                                      _p(w["w13_q"]), _p(w["w13_s"]), _p(w["w13_gs"]), _p(w["w2_q"]),
                                      _p(w["w2_s"]), _p(w["w2_gs"]), _p(h), _p(gu), _p(y))
        return (y, h, gu) if want_intermediates else y

    def forward_nvfp4(self, d, x, w):
        """Whole layer with NVFP4 expert weights (the router, pooler, norm and
        unpooler as in forward())."""
        logits = self.router_logits(d, x, w["router_w"], w.get("router_bias"))
        idx, tw = self.topk(d, logits)
        x_lat = self.pool(d, x, w["pooler_w"])
        y = self.experts_nvfp4(d, x_lat, idx, w)
        z = self.norm_combine(d, y, idx, tw, w["norm_g"])
        return {"out": self.unpool(d, z, w["unpooler_w"]), "x_lat": x_lat, "y": y, "z": z, "topk_idx": idx,
                "topk_w": tw}

    def norm_combine(self, d, y, topk_idx, topk_w, norm_g, want_yhat=False):
        T = topk_idx.shape[0]
        od = self.dims(d, T)
        z = np.empty((T, d.L), np.float32)
        yhat = np.empty((T * d.k, d.L), np.float32) if want_yhat else None
        self.lib.oracle_norm_combine(ctypes.byref(od), _p(y), _p(np.ascontiguousarray(topk_idx)),
                                     _p(np.ascontiguousarray(topk_w)), _p(norm_g), _p(yhat), _p(z))
        return (z, yhat) if want_yhat else z

    def unpool(self, d, z, unpooler_w):
        od = self.dims(d, z.shape[0])
        out = np.empty((od.T, d.H), np.uint16)
        self.lib.oracle_unpool(ctypes.byref(od), _p(z), _p(unpooler_w), _p(out))
        return out

    # -- the sandwich block around the layer ----------------------------------------------
    def rmsnorm(self, x, g, eps):
        """Row RMSNorm of bf16 rows x [rows][W] with the bf16 gain g [W] -> fp32."""
        x = np.ascontiguousarray(x)
        out = np.empty(x.shape, np.float32)
        self.lib.oracle_rmsnorm_rows(x.shape[0], x.shape[1], _p(x), _p(np.ascontiguousarray(g)), float(eps), _p(out))
        return out

    def router_logits_f32(self, d, x, router_w, router_bias=None, want_absdot=False):
        """Router logits of fp32 input rows x [T][H] (the pre-norm's output)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        od = self.dims(d, x.shape[0])
        logits = np.empty((od.T, d.E), np.float32)
        absdot = np.empty((od.T, d.E), np.float64) if want_absdot else None
        self.lib.oracle_router_logits_f32(ctypes.byref(od), _p(x), _p(router_w), _p(router_bias), _p(logits),
                                          _p(absdot))
        return (logits, absdot) if want_absdot else logits

    def bf16_round(self, a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        out = np.empty(a.shape, np.uint16)
        self.lib.oracle_bf16_round(a.size, _p(a), _p(out))
        return out

    def residual_add(self, x, p):
        x = np.ascontiguousarray(x)
        p = np.ascontiguousarray(p, dtype=np.float32)
        out = np.empty(x.shape, np.uint16)
        self.lib.oracle_residual_add(x.size, _p(x), _p(p), _p(out))
        return out

    def block_forward(self, d, x, w, nw, eps=None):
        """y = x + post_norm(F(pre_norm(x))) with F the layer; the router reads the
        pre-norm's fp32 output, the pooler that output rounded to bf16.  nw holds
        the bf16 gains "pre_g" and "post_g" [H]; eps defaults to the layer's."""
        eps = d.eps if eps is None else eps
        n = self.rmsnorm(x, nw["pre_g"], eps)
        logits, absdot = self.router_logits_f32(d, n, w["router_w"], w.get("router_bias"), want_absdot=True)
        idx, tw = self.topk(d, logits)
        nb = self.bf16_round(n)
        r = self.forward_routed(d, nb, w, idx, tw)
        p = self.rmsnorm(r["out"], nw["post_g"], eps)
        r.update({"y": self.residual_add(x, p), "n": n, "nb": nb, "logits": logits, "absdot": absdot,
                  "topk_idx": idx, "topk_w": tw})
        return r

    def forward_routed(self, d, x, w, topk_idx, topk_w):
        """Whole layer with the given routing: the pooler, expert, norm-and-sum and
        unpooler stages composed as in forward(), the router and top-k skipped."""
        x_lat = self.pool(d, x, w["pooler_w"])
        y = self.experts(d, x_lat, topk_idx, w)
        z = self.norm_combine(d, y, topk_idx, topk_w, w["norm_g"])
        return {"out": self.unpool(d, z, w["unpooler_w"]), "x_lat": x_lat, "y": y, "z": z}

    def forward(self, d, x, w):
        """Whole layer; returns a dict of the output and every intermediate."""
        T = x.shape[0]
        od = self.dims(d, T)
        R = T * d.k
        res = {
            "out": np.empty((T, d.H), np.uint16),
            "topk_idx": np.empty((T, d.k), np.int32),
            "topk_w": np.empty((T, d.k), np.float32),
            "x_lat": np.empty((T, d.L), np.uint16),
            "y": np.empty((R, d.L), np.float32),
            "z": np.empty((T, d.L), np.float32),
        }
        self.lib.oracle_forward(ctypes.byref(od), _p(x), _p(w["router_w"]), _p(w.get("router_bias")),
                                _p(w["pooler_w"]), _p(w["w13_q"]), _p(w["w13_s"]), _p(w["w2_q"]), _p(w["w2_s"]),
                                _p(w["norm_g"]), _p(w["unpooler_w"]), _p(res["out"]), _p(res["topk_idx"]),
                                _p(res["topk_w"]), _p(res["x_lat"]), _p(res["y"]), _p(res["z"]))
        return res


_default = None


def get(threads: int | None = None) -> Oracle:
    """The default (unplanted) oracle, loaded once."""
    global _default
    if _default is None:
        _default = Oracle(0, threads)
    elif threads:
        _default.set_threads(threads)
    return _default
