"""CPU oracle for paged-attention decode (test infrastructure only).

The oracle is a plain double-precision C implementation of what the decode
computes (``pa_oracle.c`` holds the definition and its sources). Only the
tests, the smoke check and the benchmark's CPU-baseline leg may use it; the
product path never imports this package. It shares no code with the CUDA
library: inputs come from ``pa_workloads`` and results go straight back to the
caller as float64 arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pa_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libpa_oracle.so")

_lock = threading.Lock()
_default = None


class Shape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("query_len", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("max_pages_per_seq", ctypes.c_int),
        ("num_pages", ctypes.c_int),
        ("kv_dtype", ctypes.c_int),
        ("scale_mode", ctypes.c_int),
        ("causal", ctypes.c_int),
        ("window", ctypes.c_int),
        ("has_sinks", ctypes.c_int),
        ("topk", ctypes.c_int),
        ("sm_scale", ctypes.c_double),
        ("q_dtype", ctypes.c_int),
        ("v_layout", ctypes.c_int),
    ]


def build(source: str = SOURCE, out: str = LIB_PATH, force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no CUDA involved)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        self.lib = lib
        lib.pa_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.pa_oracle_e4m3_to_double.restype = ctypes.c_double
        lib.pa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.pa_oracle_bf16_to_double.restype = ctypes.c_double
        lib.pa_oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.pa_oracle_f16_to_double.restype = ctypes.c_double
        lib.pa_oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
        lib.pa_oracle_e2m1_to_double.restype = ctypes.c_double
        lib.pa_oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
        lib.pa_oracle_e8m0_to_double.restype = ctypes.c_double
        lib.pa_oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.pa_oracle_round_bf16.restype = ctypes.c_uint16
        lib.pa_oracle_round_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
        lib.pa_oracle_round_bf16_array.restype = None
        vp = ctypes.c_void_p
        lib.pa_oracle_decode.argtypes = [ctypes.POINTER(Shape)] + [vp] * 11
        lib.pa_oracle_decode.restype = ctypes.c_int
        lib.pa_oracle_row_partial.argtypes = ([ctypes.POINTER(Shape)] + [vp] * 6 +
                                              [ctypes.c_int] * 3 + [vp, ctypes.c_int, vp, vp, vp])
        lib.pa_oracle_row_partial.restype = ctypes.c_int
        lib.pa_oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.c_int,
                                        ctypes.c_double, vp]
        lib.pa_oracle_merge.restype = None
        lib.pa_oracle_mqa_logits.argtypes = [ctypes.c_int] * 4 + [vp] * 6 + [ctypes.c_int] + [vp] * 4
        lib.pa_oracle_mqa_logits.restype = ctypes.c_int

    # --- element codecs ---------------------------------------------------
    def e4m3_to_double(self, codes) -> np.ndarray:
        return np.array([self.lib.pa_oracle_e4m3_to_double(int(c)) for c in np.ravel(codes)])

    def e2m1_to_double(self, codes) -> np.ndarray:
        return np.array([self.lib.pa_oracle_e2m1_to_double(int(c)) for c in np.ravel(codes)])

    def e8m0_to_double(self, codes) -> np.ndarray:
        return np.array([self.lib.pa_oracle_e8m0_to_double(int(c)) for c in np.ravel(codes)])

    def bf16_to_double(self, bits) -> np.ndarray:
        return np.array([self.lib.pa_oracle_bf16_to_double(int(b)) for b in np.ravel(bits)])

    def f16_to_double(self, bits) -> np.ndarray:
        return np.array([self.lib.pa_oracle_f16_to_double(int(b)) for b in np.ravel(bits)])

    def round_bf16(self, x) -> np.ndarray:
        x = np.ascontiguousarray(np.ravel(x), dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.pa_oracle_round_bf16_array(_ptr(x), _ptr(out), x.size)
        return out

    # --- decode -----------------------------------------------------------
    @staticmethod
    def shape_of(w, sm_scale: Optional[float] = None) -> Shape:
        if sm_scale is None:
            sm_scale = 1.0 / np.sqrt(w.head_dim)
        # The GPU receives sm_scale as a binary32; use the same value here.
        sm_scale = float(np.float32(sm_scale))
        return Shape(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.query_len,
                     w.page_size, w.max_pages_per_seq, w.num_pages, w.kv_dtype, w.scale_mode,
                     int(w.causal), int(w.window), int(w.sinks is not None), int(w.topk),
                     sm_scale, int(getattr(w, "q_dtype", 0)), int(getattr(w, "v_layout", 0)))

    @staticmethod
    def _arrays(w):
        c = np.ascontiguousarray
        sdt = np.uint8 if w.kv_dtype == 2 else np.float32  # MXFP4: E8M0 scale bytes
        ks = c(w.k_scale, dtype=sdt) if w.k_scale is not None else None
        vs = c(w.v_scale, dtype=sdt) if w.v_scale is not None else None
        sinks = c(w.sinks, dtype=np.float32) if w.sinks is not None else None
        idx = c(w.topk_idx, dtype=np.int32) if w.topk_idx is not None else None
        return (c(w.q), c(w.k_cache), c(w.v_cache), c(w.block_table, dtype=np.int32),
                c(w.ctx_lens, dtype=np.int32), ks, vs, sinks, idx)

    def decode(self, w, sm_scale: Optional[float] = None,
               unit_mask: Optional[np.ndarray] = None) -> np.ndarray:
        """Exact-ish (float64) decode output [B*QL, Hq, D]; NaN where skipped."""
        sh = self.shape_of(w, sm_scale)
        q, kc, vc, bt, ctx, ks, vs, sinks, idx = self._arrays(w)
        out = np.full((w.batch * w.query_len, w.num_q_heads, w.head_dim), np.nan)
        um = None
        if unit_mask is not None:
            um = np.ascontiguousarray(unit_mask, dtype=np.uint8)
        rc = self.lib.pa_oracle_decode(ctypes.byref(sh), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                       _ptr(ctx), _ptr(ks), _ptr(vs), _ptr(sinks), _ptr(idx),
                                       _ptr(um), _ptr(out))
        if rc != 0:
            raise RuntimeError(f"oracle decode failed with code {rc}")
        return out

    def row_partial(self, w, b: int, i: int, h: int, tokens: Sequence[int],
                    sm_scale: Optional[float] = None):
        """(m, l, O[D]) of one query row over an explicit token list."""
        sh = self.shape_of(w, sm_scale)
        q, kc, vc, bt, ctx, ks, vs, _, _ = self._arrays(w)
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        m = ctypes.c_double()
        l = ctypes.c_double()
        o = np.zeros(w.head_dim)
        rc = self.lib.pa_oracle_row_partial(ctypes.byref(sh), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                            _ptr(ks), _ptr(vs), b, i, h, _ptr(tok), tok.size,
                                            ctypes.byref(m), ctypes.byref(l), _ptr(o))
        if rc != 0:
            raise RuntimeError(f"oracle partial failed with code {rc}")
        return m.value, l.value, o

    def merge(self, parts, sink: Optional[float] = None) -> np.ndarray:
        """Merge [(m, l, O), ...] in list order (natural-log units)."""
        n = len(parts)
        D = len(parts[0][2]) if n else 0
        m = np.ascontiguousarray([p[0] for p in parts], dtype=np.float64)
        l = np.ascontiguousarray([p[1] for p in parts], dtype=np.float64)
        o = np.ascontiguousarray(np.stack([p[2] for p in parts]) if n else np.zeros((0, D)))
        out = np.zeros(D)
        self.lib.pa_oracle_merge(n, D, _ptr(m), _ptr(l), _ptr(o), int(sink is not None),
                                 float(sink) if sink is not None else 0.0, _ptr(out))
        return out


class LogitsCase:
    """Indexer-logits inputs as host arrays (see pa_oracle_mqa_logits)."""

    def __init__(self, q, kv, kv_scale, weights, ks, ke):
        self.q = np.ascontiguousarray(q, dtype=np.uint8)  # [rows, heads, dim] e4m3 codes
        self.kv = np.ascontiguousarray(kv, dtype=np.uint8)  # [num_kv, dim]
        self.kv_scale = np.ascontiguousarray(kv_scale, dtype=np.float32)
        self.weights = np.ascontiguousarray(weights, dtype=np.float32)  # [rows, heads]
        self.ks = np.ascontiguousarray(ks, dtype=np.int32)
        self.ke = np.ascontiguousarray(ke, dtype=np.int32)


def mqa_logits(orc: Oracle, case: LogitsCase, rows_idx, cols_idx):
    """(logits, bound) at the listed (row, token) pairs, float64; -inf outside windows."""
    r = np.ascontiguousarray(rows_idx, dtype=np.int32).ravel()
    j = np.ascontiguousarray(cols_idx, dtype=np.int32).ravel()
    out = np.empty(r.size)
    bound = np.empty(r.size)
    rows, heads, dim = case.q.shape
    rc = orc.lib.pa_oracle_mqa_logits(rows, heads, dim, case.kv.shape[0], _ptr(case.q), _ptr(case.kv),
                                      _ptr(case.kv_scale), _ptr(case.weights), _ptr(case.ks), _ptr(case.ke),
                                      r.size, _ptr(r), _ptr(j), _ptr(out), _ptr(bound))
    if rc != 0:
        raise RuntimeError(f"oracle logits failed with code {rc}")
    return out, bound


def mqa_logits_full(orc: Oracle, case: LogitsCase):
    """The whole [rows, num_kv] logits matrix and its bounds (small cases)."""
    rows = case.q.shape[0]
    n = case.kv.shape[0]
    rr, jj = np.meshgrid(np.arange(rows), np.arange(n), indexing="ij")
    out, bound = mqa_logits(orc, case, rr, jj)
    return out.reshape(rows, n), bound.reshape(rows, n)


def get() -> Oracle:
    """The default oracle (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def visible_rows(w):
    """Per (b, i): number of visible tokens, from the definition (for byte counts)."""
    L = w.ctx_lens.astype(np.int64)
    out = np.zeros((w.batch, w.query_len), dtype=np.int64)
    for i in range(w.query_len):
        p = L - w.query_len + i
        hi = np.minimum(L, p + 1) if w.causal else L
        lo = np.maximum(0, p - w.window + 1) if w.window > 0 else np.zeros_like(L)
        out[:, i] = np.maximum(0, hi - lo)
    return out
