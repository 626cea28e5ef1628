"""pa_decode_noalloc, the decode entry point for callers that cannot allocate
device memory: a plugin inside a framework that owns every device
allocation, or a latency-critical path where cudaMalloc may synchronise the
device. It decodes on a scratch buffer built into the library, so no
workspace is bound to its plan.

Checked through the C ABI against pa_decode on the same plan fields (same
schedule, so the outputs must be bit-identical) and against the CPU oracle,
on two calls in a row (the second reuses the scratch the first left behind),
for each merge mechanism, and for a large plan followed by a smaller one
whose counters and partials sit at other offsets of the shared scratch.
"""

import numpy as np
import pytest

import paged_attention_decode_attn_gb300 as pa
import pa_workloads as pw
from paged_attention_decode_attn_gb300 import _build

ATOL = RTOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def test_rejects_plans_larger_than_the_scratch():
    # 16,000 CTAs x 2 partial slots x 64 rows x 128 dims of f32 is far above
    # the 32 MiB scratch: refused before any device work.
    h = pa.pa_plan_create(batch=4, num_q_heads=64, num_kv_heads=1, head_dim=128, query_len=1,
                          page_size=64, max_pages_per_seq=64, num_pages=1024, kv_dtype=0,
                          scale_mode=1, causal=1, sm_count_override=8000, ctas_per_sm_override=2)
    try:
        assert pa.pa_plan_workspace_bytes(h) > (32 << 20)
        with pytest.raises(pa.PaError) as ei:
            pa.pa_decode_noalloc(0x100, 0x100, 0x100, 0x100, 0x100, 0x100, 0x100, 0x100, 0, None, h,
                                 stream=0)
        assert ei.value.status == pa.PA_ERR_WORKSPACE
        assert "32 MiB" in pa.pa_last_error()
    finally:
        pa.pa_plan_destroy(h)


def _workload(lens, seed):
    return pw.make_dense("noalloc", batch=len(lens), hkv=2, group=8, head_dim=128, query_len=2, page_size=16,
                         ctx_lens=lens, kv_dtype=pw.KV_FP8, scale_mode=pw.SCALE_PER_TENSOR, seed=seed,
                         causal=1, with_sinks=True)


def _fields(w, **kw):
    f = dict(batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
             head_dim=w.head_dim, query_len=w.query_len, page_size=w.page_size,
             max_pages_per_seq=w.max_pages_per_seq, num_pages=w.num_pages,
             max_context_len=int(w.ctx_lens.max()), kv_dtype=w.kv_dtype, scale_mode=w.scale_mode,
             causal=1, has_sinks=1)
    f.update(kw)
    return f


def _check_against_pa_decode(torch, w, fields, calls=2):
    """Run pa_decode (caller workspace) once and pa_decode_noalloc `calls`
    times on plans made from the same fields; every no-alloc output must equal
    the pa_decode output bit for bit and match the oracle."""
    import oracle

    dev = torch.device("cuda", 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    q = t(w.q.view(np.int16)).view(torch.bfloat16)
    k, v = t(w.k_cache), t(w.v_cache)
    bt, ctx = t(w.block_table), t(w.ctx_lens)
    ks, vs, sinks = t(w.k_scale), t(w.v_scale), t(w.sinks)
    plan = pa.Plan(device=dev, **fields)
    ref = torch.full_like(q, float("nan"))
    plan.decode(ref, q, k, v, bt, ctx, ks, vs, 0, sinks)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref_bits = ref.view(torch.int16).cpu().numpy()
    expect = oracle.get().decode(w)
    h = pa.pa_plan_create(device=0, **fields)
    try:
        info = pa.pa_plan_get_info(h)
        for _ in range(calls):
            out = torch.full_like(q, float("nan"))
            pa.pa_decode_noalloc(out, q, k, v, bt, ctx, ks, vs, 0, sinks, h)
            torch.cuda.synchronize()
            assert np.array_equal(out.view(torch.int16).cpu().numpy(), ref_bits)
            got = out.float().cpu().numpy().astype(np.float64)
            assert np.all(np.isfinite(got))
            assert np.all(np.abs(got - expect) <= ATOL + RTOL * np.abs(expect))
        return info
    finally:
        pa.pa_plan_destroy(h)


MERGES = [
    (dict(sm_count_override=5, ctas_per_sm_override=2), pa.PA_MERGE_LAST_ARRIVER),
    (dict(sm_count_override=5, ctas_per_sm_override=2, merge_mode=pa.PA_MERGE_REDUCER), pa.PA_MERGE_REDUCER),
    (dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=4, merge_mode=pa.PA_MERGE_CLUSTER), pa.PA_MERGE_CLUSTER),
]


@pytest.mark.gpu
@pytest.mark.parametrize("kw,merge", MERGES, ids=["last-arriver", "reducer", "cluster"])
def test_matches_pa_decode_on_two_calls(kw, merge):
    torch = pytest.importorskip("torch")
    w = _workload([0, 3, 90, 600, 1300, 2222, 4001], seed=21)
    info = _check_against_pa_decode(torch, w, _fields(w, **kw))
    assert info["merge_mode"] == merge


@pytest.mark.gpu
def test_large_plan_then_small_plan():
    """A plan with many partial slots, then one with few: the second call's
    counters and partials start at other offsets of the shared scratch, which
    the first call left non-zero."""
    torch = pytest.importorskip("torch")
    big = _workload([5000, 7000, 1, 3000, 6500, 4000, 2500, 7999], seed=22)
    small = _workload([0, 3, 90, 600, 1300], seed=23)
    bi = _check_against_pa_decode(torch, big, _fields(big, sm_count_override=40, ctas_per_sm_override=2),
                                  calls=1)
    si = _check_against_pa_decode(torch, small, _fields(small, sm_count_override=3, ctas_per_sm_override=1),
                                  calls=2)
    assert bi["workspace_bytes"] > si["workspace_bytes"]
    assert bi["merge_mode"] == si["merge_mode"] == pa.PA_MERGE_LAST_ARRIVER
