"""Python binding of libpa_decode, the GB300 paged-attention decode library.

This module only marshals arguments: it turns tensors into device pointers and
streams into handles and calls the C ABI declared in ``include/pa_decode.h``.
All computation happens in the CUDA kernels of the library. There is no
fallback: if the compiled library is missing, importing the binding's entry
points raises.

Functions keep the C names (``pa_plan_create``, ``pa_decode``,
``pa_decode_sparse``, ...). ``Plan`` bundles a plan handle with a zero-filled
workspace tensor for convenience.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "PA_OK", "PA_ERR_INVALID_ARG", "PA_ERR_UNSUPPORTED", "PA_ERR_WORKSPACE", "PA_ERR_CUDA",
    "PA_ERR_DEVICE_STATUS", "PA_KV_FP8_E4M3", "PA_KV_BF16", "PA_KV_MXFP4", "PA_SCALE_NONE",
    "PA_SCALE_PER_TENSOR", "PA_SCALE_PER_TOKEN", "PA_SCALE_MX_BLOCK", "PA_MERGE_AUTO", "PA_MERGE_DIRECT", "PA_MERGE_CLUSTER",
    "PA_MERGE_LAST_ARRIVER", "PA_MERGE_REDUCER", "PA_SCHED_AUTO", "PA_SCHED_BALANCED",
    "PA_SCHED_PER_UNIT", "PA_CONSUMER_AUTO", "PA_CONSUMER_TILE", "PA_CONSUMER_TMEM", "PA_Q_BF16",
    "PA_Q_FP16", "PA_V_PLAIN", "PA_V_TRANSPOSED", "PaError", "PlanDesc", "PlanInfo", "Plan", "library", "library_path",
    "pa_plan_create", "pa_plan_workspace_bytes", "pa_plan_set_workspace", "pa_plan_get_info",
    "pa_plan_destroy", "pa_decode", "pa_decode_sparse", "pa_decode_noalloc", "pa_mqa_logits", "pa_strerror",
    "pa_last_error", "EXPORTED_SYMBOLS",
]

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_DEVICE_STATUS = range(6)
PA_KV_FP8_E4M3, PA_KV_BF16, PA_KV_MXFP4 = 0, 1, 2
PA_SCALE_NONE, PA_SCALE_PER_TENSOR, PA_SCALE_PER_TOKEN, PA_SCALE_MX_BLOCK = 0, 1, 2, 3
PA_MERGE_AUTO, PA_MERGE_DIRECT, PA_MERGE_CLUSTER, PA_MERGE_LAST_ARRIVER, PA_MERGE_REDUCER = range(5)
PA_SCHED_AUTO, PA_SCHED_BALANCED, PA_SCHED_PER_UNIT = 0, 1, 2
PA_CONSUMER_AUTO, PA_CONSUMER_TILE, PA_CONSUMER_TMEM = 0, 1, 2
PA_Q_BF16, PA_Q_FP16 = 0, 1
PA_V_PLAIN, PA_V_TRANSPOSED = 0, 1

EXPORTED_SYMBOLS = [
    "pa_plan_create", "pa_plan_workspace_bytes", "pa_plan_set_workspace", "pa_plan_get_info",
    "pa_plan_destroy", "pa_decode", "pa_decode_sparse", "pa_decode_noalloc", "pa_mqa_logits", "pa_strerror",
    "pa_last_error",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpa_decode.so")


class PaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class PlanDesc(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "query_len", "page_size",
        "max_pages_per_seq", "num_pages", "max_context_len", "kv_dtype", "scale_mode", "causal",
        "has_sinks", "sparse_topk")] + [("sm_scale", ctypes.c_float)] + [
        (name, ctypes.c_int) for name in (
            "max_partitions", "merge_mode", "schedule", "sm_count_override",
            "ctas_per_sm_override", "device", "consumer", "q_dtype", "v_layout")]


class PlanInfo(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "merge_mode", "schedule", "num_partitions", "stage_tokens", "num_stages", "rows",
        "rows_per_warp", "row_warps", "token_warps", "block_threads", "grid", "cluster",
        "ctas_per_sm", "sm_count", "launches_per_call", "units", "consumer")] + [
        (name, ctypes.c_size_t) for name in (
            "smem_bytes", "workspace_bytes", "partial_slots", "status_offset")]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None


def library():
    """The loaded libpa_decode (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise ImportError(
                f"{library_path} is missing: build it with "
                "paged_attention_decode_attn_gb300._build.build() (needs nvcc)")
        lib = ctypes.CDLL(library_path)
        vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        lib.pa_plan_create.argtypes = [ctypes.POINTER(PlanDesc), ctypes.POINTER(vp)]
        lib.pa_plan_create.restype = st
        lib.pa_plan_workspace_bytes.argtypes = [vp]
        lib.pa_plan_workspace_bytes.restype = ctypes.c_size_t
        lib.pa_plan_set_workspace.argtypes = [vp, vp, ctypes.c_size_t]
        lib.pa_plan_set_workspace.restype = st
        lib.pa_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        lib.pa_plan_get_info.restype = st
        lib.pa_plan_destroy.argtypes = [vp]
        lib.pa_plan_destroy.restype = None
        lib.pa_decode.argtypes = [vp] * 8 + [i, vp, vp, vp]
        lib.pa_decode.restype = st
        lib.pa_decode_sparse.argtypes = [vp] * 12
        lib.pa_decode_sparse.restype = st
        lib.pa_decode_noalloc.argtypes = [vp] * 8 + [i, vp, vp, vp]
        lib.pa_decode_noalloc.restype = st
        # logits, stride, q, kv, kv_scale, weights, ks, ke, rows, heads, dim, num_kv, clean, status, device, stream
        lib.pa_mqa_logits.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp, i, vp]
        lib.pa_mqa_logits.restype = st
        lib.pa_strerror.argtypes = [st]
        lib.pa_strerror.restype = ctypes.c_char_p
        lib.pa_last_error.argtypes = []
        lib.pa_last_error.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def pa_strerror(status: int) -> str:
    return library().pa_strerror(status).decode()


def pa_last_error() -> str:
    return library().pa_last_error().decode()


def _check(status: int):
    if status != PA_OK:
        raise PaError(status, f"{pa_strerror(status)}: {pa_last_error()}")


def _ptr(x) -> Optional[int]:
    """Device/host address of a tensor-like (torch tensor or int) or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def pa_plan_create(**fields) -> ctypes.c_void_p:
    """Create a plan from pa_plan_desc fields (unset fields are 0)."""
    desc = PlanDesc()
    for k, v in fields.items():
        if not hasattr(desc, k):
            raise TypeError(f"unknown plan field {k}")
        setattr(desc, k, v)
    handle = ctypes.c_void_p()
    _check(library().pa_plan_create(ctypes.byref(desc), ctypes.byref(handle)))
    return handle


def pa_plan_workspace_bytes(plan) -> int:
    return int(library().pa_plan_workspace_bytes(plan))


def pa_plan_set_workspace(plan, workspace, nbytes: int):
    _check(library().pa_plan_set_workspace(plan, _ptr(workspace), nbytes))


def pa_plan_get_info(plan) -> dict:
    info = PlanInfo()
    _check(library().pa_plan_get_info(plan, ctypes.byref(info)))
    return info.as_dict()


def pa_plan_destroy(plan):
    library().pa_plan_destroy(plan)


def pa_decode(out, q, k_cache, v_cache, block_table, ctx_lens, k_scale, v_scale, window, sinks,
              plan, stream=None):
    _check(library().pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                               _ptr(ctx_lens), _ptr(k_scale), _ptr(v_scale), int(window), _ptr(sinks),
                               plan, _stream(stream)))


def pa_decode_noalloc(out, q, k_cache, v_cache, block_table, ctx_lens, k_scale, v_scale, window,
                      sinks, plan, stream=None):
    """Dense decode on the library's built-in scratch: for callers that cannot
    allocate device memory (no workspace has to be bound to `plan`)."""
    _check(library().pa_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_table), _ptr(ctx_lens), _ptr(k_scale),
                                       _ptr(v_scale), int(window), _ptr(sinks), plan,
                                       _stream(stream)))


def pa_decode_sparse(out, q, k_cache, v_cache, block_table, ctx_lens, topk_idx, k_scale, v_scale,
                     sinks, plan, stream=None):
    _check(library().pa_decode_sparse(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(block_table), _ptr(ctx_lens), _ptr(topk_idx),
                                      _ptr(k_scale), _ptr(v_scale), _ptr(sinks), plan,
                                      _stream(stream)))


def pa_mqa_logits(logits, q, kv, kv_scale, weights, ks, ke, clean_logits=True, status=None, stream=None):
    """Indexer logits (FP8 q [rows, heads, 128], FP8 kv [num_kv, 128]) into the
    float32 logits [rows, >= num_kv] tensor; see include/pa_decode.h."""
    rows, heads, dim = q.shape
    num_kv = kv.shape[0]
    _check(library().pa_mqa_logits(_ptr(logits), int(logits.stride(0)), _ptr(q), _ptr(kv), _ptr(kv_scale),
                                   _ptr(weights), _ptr(ks), _ptr(ke), int(rows), int(heads), int(dim), int(num_kv),
                                   int(bool(clean_logits)), _ptr(status), int(logits.device.index or 0),
                                   _stream(stream)))
    return logits


class Plan:
    """A plan handle plus its zero-filled device workspace (a torch tensor)."""

    def __init__(self, device=None, **fields):
        import torch

        if device is None:
            device = torch.device("cuda", torch.cuda.current_device())
        device = torch.device(device)
        fields.setdefault("device", device.index or 0)
        self.fields = dict(fields)
        self.handle = pa_plan_create(**fields)
        self.info = pa_plan_get_info(self.handle)
        nbytes = max(256, pa_plan_workspace_bytes(self.handle))
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        pa_plan_set_workspace(self.handle, self.workspace, nbytes)

    def decode(self, out, q, k_cache, v_cache, block_table, ctx_lens, k_scale=None, v_scale=None,
               window: int = 0, sinks=None, stream=None):
        pa_decode(out, q, k_cache, v_cache, block_table, ctx_lens, k_scale, v_scale, window, sinks,
                  self.handle, stream)
        return out

    def decode_sparse(self, out, q, k_cache, v_cache, block_table, ctx_lens, topk_idx,
                      k_scale=None, v_scale=None, sinks=None, stream=None):
        pa_decode_sparse(out, q, k_cache, v_cache, block_table, ctx_lens, topk_idx, k_scale, v_scale,
                         sinks, self.handle, stream)
        return out

    def device_status(self) -> int:
        """The kernels' status word (synchronises the device)."""
        import torch

        off = self.info["status_offset"]
        return int(self.workspace[off:off + 4].view(torch.int32).item())

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.pa_plan_destroy(h)
            self.handle = None
