"""The C ABI on the host: the library builds, loads and exports every entry
point the header declares; plan sizing matches its restated rule bit for bit;
invalid arguments come back as error codes (no GPU needed)."""

import ctypes
import os
import re
import subprocess

import pytest

import paged_attention_decode_attn_gb300 as pa
from paged_attention_decode_attn_gb300 import _build
import plan_rule

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa_decode.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", src)))


def test_header_declares_binding_names():
    assert declared_functions() == sorted(pa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pa.library_path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None
    # nothing but the C ABI is exported from our code
    ours = {n for n in exported if n.startswith("pa_") or "pa::" in n or n.startswith("_ZN2pa")}
    assert ours == set(declared_functions())


def test_strerror(lib):
    assert pa.pa_strerror(pa.PA_OK) == "success"
    assert "unsupported" in pa.pa_strerror(pa.PA_ERR_UNSUPPORTED)


def desc(**kw):
    d = dict(batch=64, num_q_heads=64, num_kv_heads=8, head_dim=128, query_len=1, page_size=16,
             max_pages_per_seq=512, num_pages=40000, kv_dtype=0, scale_mode=1, causal=1,
             sm_count_override=152, ctas_per_sm_override=2)
    d.update(kw)
    return d


PLAN_CASES = [
    desc(),
    desc(ctas_per_sm_override=1, sm_count_override=132),
    desc(batch=16, num_q_heads=16, num_kv_heads=2, head_dim=256, page_size=64, scale_mode=2,
         query_len=4, max_pages_per_seq=2100),
    desc(batch=16, num_q_heads=16, num_kv_heads=2, head_dim=256, page_size=64, scale_mode=2,
         query_len=3, has_sinks=1),
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128),
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, kv_dtype=1, scale_mode=0),
    desc(batch=64, num_q_heads=16, num_kv_heads=1, sparse_topk=2048, max_pages_per_seq=8192,
         num_pages=4096),
    desc(batch=64, num_q_heads=16, num_kv_heads=1, sparse_topk=2048, max_partitions=16,
         merge_mode=pa.PA_MERGE_CLUSTER),
    desc(batch=64, num_q_heads=16, num_kv_heads=1, sparse_topk=2048, max_partitions=8,
         merge_mode=pa.PA_MERGE_REDUCER),
    desc(batch=3, merge_mode=pa.PA_MERGE_DIRECT),
    desc(batch=3, schedule=pa.PA_SCHED_PER_UNIT, max_context_len=100),
    desc(batch=2, num_q_heads=8, num_kv_heads=1, merge_mode=pa.PA_MERGE_REDUCER),
    desc(batch=0),
    desc(num_q_heads=8, num_kv_heads=8, kv_dtype=1, scale_mode=0, head_dim=256),
    desc(num_q_heads=24, num_kv_heads=8, query_len=4, kv_dtype=1, scale_mode=0),
    desc(batch=5, num_q_heads=12, num_kv_heads=1, query_len=5, schedule=pa.PA_SCHED_PER_UNIT,
         max_partitions=3, merge_mode=pa.PA_MERGE_LAST_ARRIVER),
    desc(batch=241, num_q_heads=16, num_kv_heads=1, sparse_topk=2048, sm_count_override=256),
    desc(batch=4, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, schedule=pa.PA_SCHED_PER_UNIT,
         max_partitions=4, merge_mode=pa.PA_MERGE_CLUSTER, consumer=pa.PA_CONSUMER_TMEM),
    desc(batch=16, num_q_heads=16, num_kv_heads=2, head_dim=256, page_size=64, scale_mode=2, query_len=4,
         merge_mode=pa.PA_MERGE_REDUCER, consumer=pa.PA_CONSUMER_TMEM),
    desc(batch=16, num_q_heads=16, num_kv_heads=2, head_dim=256, page_size=64, scale_mode=2, query_len=3,
         consumer=pa.PA_CONSUMER_TMEM),
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, consumer=pa.PA_CONSUMER_TMEM),
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, kv_dtype=1, scale_mode=0,
         consumer=pa.PA_CONSUMER_TMEM),
    desc(num_q_heads=24, num_kv_heads=8, query_len=4, kv_dtype=1, scale_mode=0, consumer=pa.PA_CONSUMER_TILE),
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, consumer=pa.PA_CONSUMER_TILE),
    # FP16 queries: FP8 caches keep the tensor-memory consumer, BF16 caches take the tile consumer
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, q_dtype=pa.PA_Q_FP16),
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, kv_dtype=1, scale_mode=0,
         q_dtype=pa.PA_Q_FP16),
    desc(num_q_heads=8, num_kv_heads=8, kv_dtype=1, scale_mode=0, head_dim=256, q_dtype=pa.PA_Q_FP16),
    # BF16 head_dim 64 (one 128-byte block per token row)
    desc(num_q_heads=64, num_kv_heads=8, kv_dtype=1, scale_mode=0, head_dim=64),
    desc(num_q_heads=64, num_kv_heads=1, kv_dtype=1, scale_mode=0, head_dim=64, q_dtype=pa.PA_Q_FP16),
    desc(batch=8, num_q_heads=32, num_kv_heads=2, query_len=2, scale_mode=2),  # FP8 per-token, 32 rows: auto
    # MXFP4 (64-byte rows, 16 KiB stages, block scales as per-token scale slots): tile consumer
    desc(kv_dtype=pa.PA_KV_MXFP4, scale_mode=pa.PA_SCALE_MX_BLOCK),
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, kv_dtype=pa.PA_KV_MXFP4,
         scale_mode=pa.PA_SCALE_MX_BLOCK),
    desc(num_q_heads=16, num_kv_heads=8, kv_dtype=pa.PA_KV_MXFP4, scale_mode=pa.PA_SCALE_MX_BLOCK,
         merge_mode=pa.PA_MERGE_CLUSTER, schedule=pa.PA_SCHED_PER_UNIT, max_partitions=4),
    # transposed BF16 V: the tile consumer whatever the row count
    desc(num_q_heads=64, num_kv_heads=8, kv_dtype=1, scale_mode=0, v_layout=pa.PA_V_TRANSPOSED),
    desc(batch=32, num_q_heads=64, num_kv_heads=4, query_len=4, page_size=128, kv_dtype=1, scale_mode=0,
         v_layout=pa.PA_V_TRANSPOSED),
    desc(num_q_heads=16, num_kv_heads=2, kv_dtype=1, scale_mode=0, head_dim=256, page_size=64,
         v_layout=pa.PA_V_TRANSPOSED, q_dtype=pa.PA_Q_FP16),
]


@pytest.mark.parametrize("d", PLAN_CASES)
def test_plan_matches_rule(lib, d):
    h = pa.pa_plan_create(**d)
    try:
        assert pa.pa_plan_get_info(h) == plan_rule.plan(d)
        assert pa.pa_plan_workspace_bytes(h) == plan_rule.plan(d)["workspace_bytes"]
    finally:
        pa.pa_plan_destroy(h)


BAD = [
    (dict(head_dim=64), pa.PA_ERR_UNSUPPORTED),  # FP8 caches: 128 or 256 only
    (dict(head_dim=96, kv_dtype=1, scale_mode=0), pa.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=60), pa.PA_ERR_INVALID_ARG),
    (dict(kv_dtype=1, scale_mode=1), pa.PA_ERR_INVALID_ARG),
    (dict(num_q_heads=64, num_kv_heads=1), pa.PA_ERR_UNSUPPORTED),  # 64 rows * QL1 ok? -> 64 ok
    (dict(num_q_heads=128, num_kv_heads=1), pa.PA_ERR_UNSUPPORTED),
    (dict(page_size=8), pa.PA_ERR_UNSUPPORTED),
    (dict(page_size=48), pa.PA_ERR_UNSUPPORTED),
    (dict(sparse_topk=64, query_len=2), pa.PA_ERR_UNSUPPORTED),
    (dict(sm_scale=-1.0), pa.PA_ERR_INVALID_ARG),
    (dict(sm_scale=float("nan")), pa.PA_ERR_INVALID_ARG),
    (dict(merge_mode=pa.PA_MERGE_CLUSTER, schedule=pa.PA_SCHED_BALANCED), pa.PA_ERR_INVALID_ARG),
    (dict(merge_mode=pa.PA_MERGE_DIRECT, max_partitions=4), pa.PA_ERR_INVALID_ARG),
    (dict(merge_mode=pa.PA_MERGE_CLUSTER, max_partitions=17), pa.PA_ERR_UNSUPPORTED),
    (dict(merge_mode=9), pa.PA_ERR_INVALID_ARG),
    (dict(query_len=0), pa.PA_ERR_INVALID_ARG),
    (dict(batch=-1), pa.PA_ERR_INVALID_ARG),
    (dict(num_pages=2 ** 30), pa.PA_ERR_UNSUPPORTED),
    (dict(max_partitions=300), pa.PA_ERR_INVALID_ARG),
    (dict(head_dim=256, num_q_heads=64, num_kv_heads=1), pa.PA_ERR_UNSUPPORTED),
    (dict(consumer=3), pa.PA_ERR_INVALID_ARG),
    (dict(q_dtype=2), pa.PA_ERR_INVALID_ARG),
    (dict(consumer=pa.PA_CONSUMER_TMEM, num_q_heads=64, num_kv_heads=4, kv_dtype=1, scale_mode=0,
          q_dtype=pa.PA_Q_FP16), pa.PA_ERR_UNSUPPORTED),  # BF16 MMAs need BF16 queries
    (dict(consumer=pa.PA_CONSUMER_TMEM), pa.PA_ERR_UNSUPPORTED),  # 8 rows: tile consumer only
    (dict(consumer=pa.PA_CONSUMER_TMEM, num_q_heads=64, num_kv_heads=4, sparse_topk=64), pa.PA_ERR_UNSUPPORTED),
    (dict(consumer=pa.PA_CONSUMER_TMEM, num_q_heads=32, num_kv_heads=2, head_dim=256, kv_dtype=1, scale_mode=0),
     pa.PA_ERR_UNSUPPORTED),  # BF16 head_dim 256: tile consumer only
    (dict(consumer=pa.PA_CONSUMER_TMEM, num_q_heads=128, num_kv_heads=1), pa.PA_ERR_UNSUPPORTED),  # > 64 rows
    (dict(consumer=pa.PA_CONSUMER_TMEM, num_q_heads=64, num_kv_heads=1, head_dim=256), pa.PA_ERR_UNSUPPORTED),
    (dict(consumer=-1), pa.PA_ERR_INVALID_ARG),
    (dict(kv_dtype=pa.PA_KV_MXFP4, scale_mode=pa.PA_SCALE_PER_TOKEN), pa.PA_ERR_INVALID_ARG),  # MX scales only
    (dict(scale_mode=pa.PA_SCALE_MX_BLOCK), pa.PA_ERR_INVALID_ARG),  # FP8 caches take no MX scales
    (dict(kv_dtype=pa.PA_KV_MXFP4, scale_mode=pa.PA_SCALE_MX_BLOCK, head_dim=256), pa.PA_ERR_UNSUPPORTED),
    (dict(kv_dtype=pa.PA_KV_MXFP4, scale_mode=pa.PA_SCALE_MX_BLOCK, sparse_topk=64), pa.PA_ERR_UNSUPPORTED),
    (dict(kv_dtype=pa.PA_KV_MXFP4, scale_mode=pa.PA_SCALE_MX_BLOCK, consumer=pa.PA_CONSUMER_TMEM,
          num_q_heads=64, num_kv_heads=4), pa.PA_ERR_UNSUPPORTED),  # tile consumer only
    (dict(kv_dtype=3), pa.PA_ERR_INVALID_ARG),
    (dict(v_layout=pa.PA_V_TRANSPOSED), pa.PA_ERR_UNSUPPORTED),  # FP8 caches: plain V only
    (dict(kv_dtype=1, scale_mode=0, v_layout=pa.PA_V_TRANSPOSED, sparse_topk=64), pa.PA_ERR_UNSUPPORTED),
    (dict(kv_dtype=1, scale_mode=0, v_layout=pa.PA_V_TRANSPOSED, consumer=pa.PA_CONSUMER_TMEM, num_q_heads=64,
          num_kv_heads=4), pa.PA_ERR_UNSUPPORTED),
    (dict(v_layout=2), pa.PA_ERR_INVALID_ARG),
    (dict(scale_mode=4), pa.PA_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("kw,status", BAD)
def test_invalid_descriptors(lib, kw, status):
    d = desc(**kw)
    if kw == dict(num_q_heads=64, num_kv_heads=1):
        # 64 rows is the largest supported group*query_len
        h = pa.pa_plan_create(**d)
        pa.pa_plan_destroy(h)
        return
    with pytest.raises(pa.PaError) as ei:
        pa.pa_plan_create(**d)
    assert ei.value.status == status
    assert pa.pa_last_error()


def test_decode_argument_errors_before_any_device_work(lib):
    h = pa.pa_plan_create(**desc(batch=2, num_q_heads=8, num_kv_heads=1))
    try:
        good = 0x10000
        args = [good] * 6 + [good, good, 0, None, h]

        def call(**over):
            a = dict(out=good, q=good, k_cache=good, v_cache=good, block_table=good, ctx_lens=good,
                     k_scale=good, v_scale=good, window=0, sinks=None)
            a.update(over)
            with pytest.raises(pa.PaError) as ei:
                pa.pa_decode(a["out"], a["q"], a["k_cache"], a["v_cache"], a["block_table"],
                             a["ctx_lens"], a["k_scale"], a["v_scale"], a["window"], a["sinks"], h,
                             stream=0)
            return ei.value.status

        assert call(q=None) == pa.PA_ERR_INVALID_ARG
        assert call(out=good + 2) == pa.PA_ERR_INVALID_ARG  # misaligned
        assert call(k_scale=None) == pa.PA_ERR_INVALID_ARG  # FP8 per-tensor needs scales
        assert call(window=-1) == pa.PA_ERR_INVALID_ARG
        assert call() == pa.PA_ERR_WORKSPACE  # no workspace bound yet
        with pytest.raises(pa.PaError) as ei:
            pa.pa_decode_sparse(good, good, good, good, good, good, good, good, good, None, h, stream=0)
        assert ei.value.status == pa.PA_ERR_INVALID_ARG  # dense plan
        with pytest.raises(pa.PaError) as ei:
            pa.pa_plan_set_workspace(h, good + 16, 1 << 20)
        assert ei.value.status == pa.PA_ERR_WORKSPACE  # misaligned
        with pytest.raises(pa.PaError) as ei:
            pa.pa_plan_set_workspace(h, good, 16)
        assert ei.value.status == pa.PA_ERR_WORKSPACE  # too small
    finally:
        pa.pa_plan_destroy(h)


def test_window_with_noncausal_mtp_unsupported(lib):
    h = pa.pa_plan_create(**desc(batch=2, num_q_heads=8, num_kv_heads=1, query_len=2, causal=0))
    try:
        with pytest.raises(pa.PaError) as ei:
            pa.pa_decode(0x100, 0x100, 0x100, 0x100, 0x100, 0x100, 0x100, 0x100, 5, None, h, stream=0)
        assert ei.value.status == pa.PA_ERR_UNSUPPORTED
    finally:
        pa.pa_plan_destroy(h)
