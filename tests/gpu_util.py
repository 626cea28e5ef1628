"""Helpers for GPU parity tests: move a seeded workload to the device, run the
library through its C ABI, compare with the oracle."""

from __future__ import annotations

import os

import numpy as np
import torch

import paged_attention_decode_attn_gb300 as pa
import pa_workloads as pw

ATOL = 5e-3
RTOL = 5e-3


class DeviceWorkload:
    def __init__(self, w: pw.Workload, device="cuda"):
        self.w = w
        t = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        qt = torch.float16 if w.q_dtype == pw.Q_FP16 else torch.bfloat16
        self.q = t(w.q.view(np.int16)).view(qt)
        if w.kv_dtype == pw.KV_BF16:
            self.k = t(w.k_cache.view(np.int16)).view(torch.bfloat16)
            self.v = t(w.v_cache.view(np.int16)).view(torch.bfloat16)
        else:
            self.k = t(w.k_cache)
            self.v = t(w.v_cache)
        self.bt = t(w.block_table.astype(np.int32))
        self.ctx = t(w.ctx_lens.astype(np.int32))
        sdt = np.uint8 if w.kv_dtype == pw.KV_MXFP4 else np.float32  # MXFP4: E8M0 block-scale bytes
        self.ks = t(w.k_scale.astype(sdt)) if w.k_scale is not None else None
        self.vs = t(w.v_scale.astype(sdt)) if w.v_scale is not None else None
        self.sinks = t(w.sinks.astype(np.float32)) if w.sinks is not None else None
        self.idx = t(w.topk_idx.astype(np.int32)) if w.topk_idx is not None else None
        self.out = torch.empty_like(self.q)

    def plan_fields(self, **kw):
        w = self.w
        f = dict(batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                 head_dim=w.head_dim, query_len=w.query_len, page_size=w.page_size,
                 max_pages_per_seq=w.max_pages_per_seq, num_pages=w.num_pages,
                 max_context_len=int(w.ctx_lens.max()) if w.batch else 0, kv_dtype=w.kv_dtype,
                 scale_mode=w.scale_mode, causal=int(w.causal), has_sinks=int(w.sinks is not None),
                 sparse_topk=int(w.topk), q_dtype=int(w.q_dtype), v_layout=int(w.v_layout))
        f.update(kw)
        return f

    def poison_out(self):
        self.out.view(torch.int16).fill_(0x7FC0)  # NaN in BF16 and in FP16

    def run(self, plan: pa.Plan, window=None, stream=None):
        w = self.w
        if window is None:
            window = w.window
        if w.topk:
            plan.decode_sparse(self.out, self.q, self.k, self.v, self.bt, self.ctx, self.idx, self.ks,
                               self.vs, self.sinks, stream=stream)
        else:
            plan.decode(self.out, self.q, self.k, self.v, self.bt, self.ctx, self.ks, self.vs, window,
                        self.sinks, stream=stream)
        return self.out


def decode(dw: DeviceWorkload, **plan_kw):
    plan = pa.Plan(**dw.plan_fields(**plan_kw))
    dw.poison_out()
    dw.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return dw.out.float().cpu().numpy().astype(np.float64), plan


# Worst margin seen per test: max over elements of |gpu - ref| / (atol + rtol |ref|)
# (1.0 is the tolerance edge). tests/conftest.py prints the table at the end.
MARGINS = {}


def parity_ratio(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max |gpu - ref| / (atol + rtol |ref|) over the elements."""
    if gpu.size == 0:
        return 0.0
    return float(np.max(np.abs(gpu - ref) / (ATOL + RTOL * np.abs(ref))))


def record_margin(ratio: float, what: str = ""):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    prev = MARGINS.get(test)
    if prev is None or ratio > prev[0]:
        MARGINS[test] = (ratio, what)


def assert_parity(gpu: np.ndarray, ref: np.ndarray, rows_mask=None, what=""):
    if rows_mask is not None:
        gpu = gpu[rows_mask]
        ref = ref[rows_mask]
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite outputs"
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    ratio = parity_ratio(gpu, ref)
    record_margin(ratio, what)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside atol=rtol=5e-3; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}; "
                           f"worst err/bound {ratio:.3f}")
    return ratio


def unit_rows_mask(w: pw.Workload, unit_mask: np.ndarray) -> np.ndarray:
    """Boolean [B*QL, Hq] mask of output rows that belong to selected units."""
    G = w.group
    m = np.zeros((w.batch * w.query_len, w.num_q_heads), dtype=bool)
    for u in np.nonzero(unit_mask)[0]:
        b, g = divmod(int(u), w.num_kv_heads)
        m[b * w.query_len:(b + 1) * w.query_len, g * G:(g + 1) * G] = True
    return m


def arrival_counters(plan, head_dim: int):
    """View of a last-arriver plan's arrival counters (one 128-byte line per
    unit) inside its workspace."""
    info = plan.info
    rpad = info["row_warps"] * info["rows_per_warp"]
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    off = a(info["partial_slots"] * rpad * head_dim * 4)
    off = a(off + info["partial_slots"] * rpad * 8)
    return plan.workspace[off:off + info["units"] * 32 * 4].view(torch.int32)
