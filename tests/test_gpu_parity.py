"""GPU parity against the CPU oracle on small seeded inputs (every output
element), across cache formats, masks, sinks, sparse lists and all merge
paths. Inputs span several stages and tiles with ragged tails."""

import numpy as np
import pytest

import oracle
import paged_attention_decode_attn_gb300 as pa
import pa_workloads as pw

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import DeviceWorkload, assert_parity, decode  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_attention_decode_attn_gb300 import _build

    _build.build()


EDGE_LENS = [0, 1, 15, 16, 17, 63, 64, 65, 127, 200, 777, 1500, 2049]

MODES = [
    dict(),  # automatic: balanced schedule, last-arriver merge
    dict(sm_count_override=3, ctas_per_sm_override=1),  # few CTAs: units split across CTAs
    dict(sm_count_override=5, ctas_per_sm_override=2, merge_mode=pa.PA_MERGE_REDUCER),
    dict(merge_mode=pa.PA_MERGE_DIRECT),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=3, merge_mode=pa.PA_MERGE_LAST_ARRIVER),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=4, merge_mode=pa.PA_MERGE_CLUSTER),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=5, merge_mode=pa.PA_MERGE_REDUCER),
]
MODE_IDS = ["auto", "balanced3", "reducer", "direct", "unit3-la", "cluster4", "unit5-reducer"]


def test_tiny(orc):
    w = pw.tiny()
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in MODES:
        gpu, _ = decode(dw, **m)
        assert_parity(gpu, ref, what=f"tiny {m}")


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_dense_fp8_edges(orc, mode):
    w = pw.make_dense("edges", batch=len(EDGE_LENS), hkv=2, group=8, head_dim=128, query_len=1,
                      page_size=16, ctx_lens=EDGE_LENS, kv_dtype=pw.KV_FP8,
                      scale_mode=pw.SCALE_PER_TENSOR, seed=7)
    gpu, _ = decode(DeviceWorkload(w), **mode)
    assert_parity(gpu, orc.decode(w), what=f"fp8 edges {mode}")


@pytest.mark.parametrize("mode", MODES[:4], ids=MODE_IDS[:4])
def test_dense_bf16(orc, mode):
    w = pw.make_dense("bf16", batch=6, hkv=2, group=8, head_dim=128, query_len=1, page_size=32,
                      ctx_lens=[0, 5, 33, 300, 1111, 2500], kv_dtype=pw.KV_BF16,
                      scale_mode=pw.SCALE_NONE, seed=8)
    gpu, _ = decode(DeviceWorkload(w), **mode)
    assert_parity(gpu, orc.decode(w), what=f"bf16 {mode}")


@pytest.mark.parametrize("ql", [1, 2, 3, 4])
@pytest.mark.parametrize("window", [0, 1, 17, 257])
def test_d256_per_token_mtp_windows(orc, ql, window):
    lens = [0, 1, 2, 63, 64, 65, 700, 2113, 3001]
    w = pw.make_dense("d256s", batch=len(lens), hkv=2, group=8, head_dim=256, query_len=ql,
                      page_size=64, ctx_lens=lens, kv_dtype=pw.KV_FP8, scale_mode=pw.SCALE_PER_TOKEN,
                      seed=100 + ql, causal=1, window=window, with_sinks=(window % 2 == 1))
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    modes = [dict(), dict(sm_count_override=4, ctas_per_sm_override=1)]
    if 8 * ql > 8:  # tensor-memory consumer (head_dim 256: more than 8 rows)
        modes += [dict(consumer=pa.PA_CONSUMER_TMEM),
                  dict(consumer=pa.PA_CONSUMER_TMEM, sm_count_override=4, ctas_per_sm_override=1)]
    for m in modes:
        gpu, _ = decode(dw, **m)
        assert_parity(gpu, ref, what=f"d256 ql{ql} w{window} {m}")


@pytest.mark.parametrize("consumer", [pa.PA_CONSUMER_TILE, pa.PA_CONSUMER_TMEM], ids=["tile", "tmem"])
@pytest.mark.parametrize("kv", [pw.KV_FP8, pw.KV_BF16], ids=["fp8", "bf16"])
@pytest.mark.parametrize("mode", MODES[:2] + MODES[4:6] + [MODES[2]], ids=MODE_IDS[:2] + MODE_IDS[4:6] + [MODE_IDS[2]])
def test_mtp4_gqa16(orc, kv, mode, consumer):
    lens = [3, 4, 5, 128, 129, 1000, 2600]
    w = pw.make_dense("mtp4s", batch=len(lens), hkv=2, group=16, head_dim=128, query_len=4,
                      page_size=128, ctx_lens=lens, kv_dtype=kv,
                      scale_mode=pw.SCALE_PER_TENSOR if kv == pw.KV_FP8 else pw.SCALE_NONE,
                      seed=30, causal=1)
    gpu, plan = decode(DeviceWorkload(w), consumer=consumer, **mode)
    assert plan.info["consumer"] == consumer
    assert_parity(gpu, orc.decode(w), what=f"mtp4 {mode} consumer {consumer}")


@pytest.mark.parametrize("page", [16, 32, 64, 128, 256])
def test_page_sizes(orc, page):
    w = pw.make_dense("pages", batch=4, hkv=1, group=4, head_dim=128, query_len=2, page_size=page,
                      ctx_lens=[1, 100, 513, 1200], kv_dtype=pw.KV_FP8, scale_mode=pw.SCALE_PER_TOKEN,
                      seed=40 + page, causal=1, window=100)
    gpu, _ = decode(DeviceWorkload(w))
    assert_parity(gpu, orc.decode(w), what=f"page {page}")


@pytest.mark.parametrize("group,ql", [(1, 1), (2, 3), (4, 4), (12, 5), (8, 8), (64, 1)])
def test_group_shapes(orc, group, ql):
    w = pw.make_dense("groups", batch=3, hkv=2, group=group, head_dim=128, query_len=ql,
                      page_size=16, ctx_lens=[ql, 90, 700], kv_dtype=pw.KV_BF16,
                      scale_mode=pw.SCALE_NONE, seed=50 + group, causal=1, with_sinks=True)
    dw = DeviceWorkload(w)
    ref = orc.decode(w)
    for consumer in ([pa.PA_CONSUMER_TILE, pa.PA_CONSUMER_TMEM] if group * ql > 16 else [pa.PA_CONSUMER_TILE]):
        gpu, _ = decode(dw, consumer=consumer)
        assert_parity(gpu, ref, what=f"group {group} ql {ql} consumer {consumer}")


@pytest.mark.parametrize("window,sinks", [(0, False), (37, True)])
def test_fp8_per_token_wide_group(orc, window, sinks):
    """FP8 per-token scales, head_dim 128, 32 rows per KV head: both stage
    consumers (the tensor-memory one runs FP8 MMAs on the stage bytes)."""
    w = pw.make_dense("pt32", batch=4, hkv=2, group=16, head_dim=128, query_len=2, page_size=16,
                      ctx_lens=[2, 77, 400, 1500], kv_dtype=pw.KV_FP8, scale_mode=pw.SCALE_PER_TOKEN,
                      seed=88, causal=1, window=window, with_sinks=sinks)
    dw = DeviceWorkload(w)
    ref = orc.decode(w)
    for consumer in (pa.PA_CONSUMER_TILE, pa.PA_CONSUMER_TMEM):
        for m in (dict(), dict(sm_count_override=5, ctas_per_sm_override=1)):
            gpu, plan = decode(dw, consumer=consumer, **m)
            assert plan.info["consumer"] == consumer
            assert_parity(gpu, ref, what=f"fp8 per-token 32 rows consumer {consumer} {m}")


def test_noncausal_mtp(orc):
    w = pw.make_dense("nc", batch=3, hkv=1, group=8, head_dim=128, query_len=3, page_size=16,
                      ctx_lens=[2, 40, 300], kv_dtype=pw.KV_FP8, scale_mode=pw.SCALE_PER_TENSOR,
                      seed=60, causal=0)
    dw = DeviceWorkload(w)
    ref = orc.decode(w)
    for consumer in (pa.PA_CONSUMER_TILE, pa.PA_CONSUMER_TMEM):
        gpu, _ = decode(dw, consumer=consumer)
        assert_parity(gpu, ref, what=f"non-causal consumer {consumer}")


SPARSE_MODES = [dict()] + [dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=p,
                                merge_mode=pa.PA_MERGE_CLUSTER) for p in (2, 4, 8, 16)] + [
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=8, merge_mode=pa.PA_MERGE_REDUCER),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=8, merge_mode=pa.PA_MERGE_LAST_ARRIVER),
    dict(schedule=pa.PA_SCHED_BALANCED, merge_mode=pa.PA_MERGE_LAST_ARRIVER),
    dict(merge_mode=pa.PA_MERGE_DIRECT),
]


@pytest.mark.parametrize("kv", [pw.KV_FP8, pw.KV_BF16], ids=["fp8", "bf16"])
def test_sparse_small(orc, kv):
    w = pw.small_sparse(kv_dtype=kv, rows=5, topk=300, context=1000)
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in SPARSE_MODES:
        gpu, _ = decode(dw, **m)
        assert_parity(gpu, ref, what=f"sparse {m}")


def test_sparse_per_token_and_sinks(orc):
    base = pw.make_dense("spt", batch=3, hkv=2, group=4, head_dim=128, query_len=1, page_size=16,
                         ctx_lens=[500, 37, 0], kv_dtype=pw.KV_FP8, scale_mode=pw.SCALE_PER_TOKEN,
                         seed=70, causal=0, with_sinks=True)
    rng = np.random.default_rng(3)
    idx = np.stack([rng.permutation(600)[:200] for _ in range(3)]).astype(np.int32)
    w = base.with_(topk=200, topk_idx=idx)
    gpu, _ = decode(DeviceWorkload(w))
    assert_parity(gpu, orc.decode(w), what="sparse per-token sinks")


@pytest.mark.parametrize("kv", [pw.KV_FP8, pw.KV_BF16], ids=["fp8", "bf16"])
def test_sparse_prefill_small(orc, kv):
    """Sparse prefill: row r of a 300-token prompt attends to min(r + 1, 128)
    of its first r + 1 tokens (one-slot plans write their rows directly;
    split rows merge through every mechanism)."""
    w = pw.sparse_prefill(kv_dtype=kv, rows=300, topk=128, pool_pages=64, seed=77)
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in SPARSE_MODES:
        gpu, plan = decode(dw, **m)
        assert_parity(gpu, ref, what=f"sparse prefill {m}")
    gpu, plan = decode(dw)
    assert plan.info["merge_mode"] == pa.PA_MERGE_DIRECT  # rows >> SMs: one slot per row


# FP16 queries (and FP16 output) on every consumer and cache format, with
# whole and split units through the merge paths. FP8 caches convert the
# queries exactly; BF16 caches split each into BF16 hi + lo (two MMAs).
FP16_CASES = [
    # id, kv, scale, group, query_len, head_dim, page, window, sinks, consumer the plan must take
    ("fp8-gqa8", pw.KV_FP8, pw.SCALE_PER_TENSOR, 8, 1, 128, 16, 0, False, pa.PA_CONSUMER_TILE),
    ("bf16-gqa8-mtp2-win", pw.KV_BF16, pw.SCALE_NONE, 8, 2, 128, 32, 37, True, pa.PA_CONSUMER_TILE),
    ("fp8-gqa16-mtp4", pw.KV_FP8, pw.SCALE_PER_TENSOR, 16, 4, 128, 128, 0, False, pa.PA_CONSUMER_TMEM),
    ("fp8-tok-gqa8-mtp4", pw.KV_FP8, pw.SCALE_PER_TOKEN, 8, 4, 128, 64, 0, True, pa.PA_CONSUMER_TMEM),
    ("bf16-gqa16-mtp4", pw.KV_BF16, pw.SCALE_NONE, 16, 4, 128, 64, 0, False, pa.PA_CONSUMER_TILE),
    ("bf16-gqa16-mtp2", pw.KV_BF16, pw.SCALE_NONE, 16, 2, 128, 16, 0, False, pa.PA_CONSUMER_TILE),
    ("fp8-d256-tok-mtp4", pw.KV_FP8, pw.SCALE_PER_TOKEN, 8, 4, 256, 64, 17, True, pa.PA_CONSUMER_TMEM),
    ("bf16-d256", pw.KV_BF16, pw.SCALE_NONE, 8, 1, 256, 64, 0, False, pa.PA_CONSUMER_TILE),
]
FP16_MODES = [
    dict(),
    dict(sm_count_override=5, ctas_per_sm_override=1, merge_mode=pa.PA_MERGE_REDUCER),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=4, merge_mode=pa.PA_MERGE_CLUSTER),
]


@pytest.mark.parametrize("case", FP16_CASES, ids=[c[0] for c in FP16_CASES])
def test_fp16_queries(orc, case):
    name, kv, scale, group, ql, D, page, window, sinks, consumer = case
    lens = [0, 1, 17, 130, 1000, 2300]
    w = pw.make_dense("f16q-" + name, batch=len(lens), hkv=2, group=group, head_dim=D, query_len=ql,
                      page_size=page, ctx_lens=lens, kv_dtype=kv, scale_mode=scale,
                      seed=300 + FP16_CASES.index(case), causal=1, window=window, with_sinks=sinks,
                      q_dtype=pw.Q_FP16)
    # most query values need FP16's extra fraction bits (the BF16 lo term is exercised)
    q32 = w.q.view(np.float16).astype(np.float32)
    back = (pw.bf16_bits(q32).astype(np.uint32) << 16).view(np.float32)
    assert np.mean(back != q32) > 0.5
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    assert dw.out.dtype == torch.float16
    for m in FP16_MODES:
        gpu, plan = decode(dw, **m)
        assert plan.info["consumer"] == consumer, (name, plan.info)
        assert_parity(gpu, ref, what=f"fp16 queries {name} {m}")


@pytest.mark.parametrize("kv", [pw.KV_FP8, pw.KV_BF16], ids=["fp8", "bf16"])
def test_fp16_queries_sparse(orc, kv):
    w = pw.small_sparse(kv_dtype=kv, rows=5, topk=300, context=1000, q_dtype=pw.Q_FP16)
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in SPARSE_MODES:
        gpu, _ = decode(dw, **m)
        assert_parity(gpu, ref, what=f"sparse fp16 queries {m}")


# BF16 caches at head_dim 64 (one 128-byte block per token row), every merge
# path, with BF16 and FP16 queries.
@pytest.mark.parametrize("group,ql,window,sinks", [(8, 1, 0, False), (4, 3, 17, True), (16, 4, 0, False),
                                                   (64, 1, 0, True)], ids=["gqa8", "gqa4-mtp3-win", "gqa16-mtp4",
                                                                           "gqa64"])
@pytest.mark.parametrize("q_dtype", [pw.Q_BF16, pw.Q_FP16], ids=["qbf16", "qfp16"])
def test_bf16_head_dim_64(orc, group, ql, window, sinks, q_dtype):
    lens = [0, 1, 65, 300, 1777]
    w = pw.make_dense("d64", batch=len(lens), hkv=2, group=group, head_dim=64, query_len=ql, page_size=16,
                      ctx_lens=lens, kv_dtype=pw.KV_BF16, scale_mode=pw.SCALE_NONE, seed=400 + group + ql,
                      causal=1, window=window, with_sinks=sinks, q_dtype=q_dtype)
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in MODES:
        gpu, plan = decode(dw, **m)
        assert plan.info["consumer"] == pa.PA_CONSUMER_TILE
        assert_parity(gpu, ref, what=f"head_dim 64 {m}")


def test_bf16_head_dim_64_sparse(orc):
    w = pw.small_sparse(kv_dtype=pw.KV_BF16, rows=5, topk=300, context=1000, head_dim=64)
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in SPARSE_MODES:
        gpu, _ = decode(dw, **m)
        assert_parity(gpu, ref, what=f"sparse head_dim 64 {m}")
