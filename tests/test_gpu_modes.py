"""GPU invariants: bit-exact agreement of the merge paths for one schedule,
bit-exact page-id indexing (window 1 returns the query position's V row),
block-table relocation, CUDA-graph replays with NaN-poisoned outputs and
refreshed lengths, self-resetting arrival counters."""

import numpy as np
import pytest

import oracle
import paged_attention_decode_attn_gb300 as pa
import pa_workloads as pw

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import DeviceWorkload, arrival_counters, assert_parity, decode  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_attention_decode_attn_gb300 import _build

    _build.build()


def _w(seed=5, kv=pw.KV_FP8, sinks=True):
    return pw.make_dense("modes", batch=7, hkv=2, group=8, head_dim=128, query_len=2, page_size=16,
                         ctx_lens=[0, 3, 90, 600, 1300, 2222, 4001], kv_dtype=kv,
                         scale_mode=pw.SCALE_PER_TENSOR if kv == pw.KV_FP8 else pw.SCALE_NONE,
                         seed=seed, causal=1, window=0, with_sinks=sinks)


@pytest.mark.parametrize("kv", [pw.KV_FP8, pw.KV_BF16], ids=["fp8", "bf16"])
def test_merge_paths_bit_identical_per_unit(kv):
    dw = DeviceWorkload(_w(kv=kv))
    outs = []
    for merge in (pa.PA_MERGE_CLUSTER, pa.PA_MERGE_LAST_ARRIVER, pa.PA_MERGE_REDUCER):
        gpu, _ = decode(dw, schedule=pa.PA_SCHED_PER_UNIT, max_partitions=6, merge_mode=merge)
        outs.append(gpu)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_merge_paths_bit_identical_balanced():
    dw = DeviceWorkload(_w())
    a, _ = decode(dw, sm_count_override=7, ctas_per_sm_override=2, merge_mode=pa.PA_MERGE_LAST_ARRIVER)
    b, _ = decode(dw, sm_count_override=7, ctas_per_sm_override=2, merge_mode=pa.PA_MERGE_REDUCER)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("kv", [pw.KV_FP8, pw.KV_BF16], ids=["fp8", "bf16"])
def test_tmem_merge_paths_bit_identical(kv):
    """The tensor-memory consumer feeds the same three merges: one schedule,
    bit-identical outputs."""
    w = pw.make_dense("tmem", batch=5, hkv=2, group=16, head_dim=128, query_len=2, page_size=16,
                      ctx_lens=[0, 70, 600, 1300, 2500], kv_dtype=kv,
                      scale_mode=pw.SCALE_PER_TENSOR if kv == pw.KV_FP8 else pw.SCALE_NONE, seed=14, causal=1)
    dw = DeviceWorkload(w)
    outs = [decode(dw, schedule=pa.PA_SCHED_PER_UNIT, max_partitions=5, merge_mode=m, consumer=pa.PA_CONSUMER_TMEM)[0]
            for m in (pa.PA_MERGE_CLUSTER, pa.PA_MERGE_LAST_ARRIVER, pa.PA_MERGE_REDUCER)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    b1, _ = decode(dw, sm_count_override=7, ctas_per_sm_override=1, merge_mode=pa.PA_MERGE_LAST_ARRIVER,
                   consumer=pa.PA_CONSUMER_TMEM)
    b2, _ = decode(dw, sm_count_override=7, ctas_per_sm_override=1, merge_mode=pa.PA_MERGE_REDUCER,
                   consumer=pa.PA_CONSUMER_TMEM)
    assert np.array_equal(b1, b2)
    assert_parity(b1, oracle.get().decode(w), what="tmem balanced")


def test_sparse_merge_paths_bit_identical():
    dw = DeviceWorkload(pw.small_sparse(rows=4, topk=512, context=3000))
    outs = [decode(dw, schedule=pa.PA_SCHED_PER_UNIT, max_partitions=8, merge_mode=m)[0]
            for m in (pa.PA_MERGE_CLUSTER, pa.PA_MERGE_LAST_ARRIVER, pa.PA_MERGE_REDUCER)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


@pytest.mark.parametrize("kv", [pw.KV_BF16, pw.KV_FP8], ids=["bf16", "fp8"])
@pytest.mark.parametrize("page", [16, 64, 128])
def test_window_one_indexing_bit_exact(kv, page):
    """V rows hold base-16 digits of their logical position and the sequence
    number; with window 1 every output row must decode to exactly (p, b)."""
    lens = [1, 4, 17, 100, 333, 1024, 4097]
    w0 = pw.make_dense("idx", batch=len(lens), hkv=2, group=8, head_dim=128, query_len=4,
                       page_size=page, ctx_lens=lens, kv_dtype=kv, scale_mode=pw.SCALE_NONE,
                       seed=9, causal=1, window=1)
    V = w0.v_cache.copy()
    for b, L in enumerate(lens):
        for g in range(2):
            t = np.arange(L)
            digits = np.stack([(t >> (4 * k)) & 15 for k in range(4)] + [np.full(L, b), np.full(L, g)], 1)
            vals = np.zeros((L, 128), dtype=np.float32)
            vals[:, :6] = digits
            enc = pw.bf16_bits(vals) if kv == pw.KV_BF16 else pw.fp8_codes(vals)
            V[w0.block_table[b, t // page], g, t % page] = enc
    w = w0.with_(v_cache=V)
    gpu, _ = decode(DeviceWorkload(w))
    got = np.rint(gpu).astype(np.int64)
    assert np.array_equal(got, gpu.astype(np.int64)), "outputs must be exact small integers"
    for b, L in enumerate(lens):
        for i in range(4):
            p = L - 4 + i
            rows = got[b * 4 + i]
            if p < 0:
                assert np.all(rows == 0)
                continue
            pos = sum(rows[:, k] << (4 * k) for k in range(4))
            assert np.all(pos == p) and np.all(rows[:, 4] == b)
            assert np.all(rows[:, 5] == np.arange(16) // 8)


def test_relocation_bit_identical():
    w = _w(seed=11)
    rng = np.random.default_rng(2)
    perm = rng.permutation(w.num_pages)
    kc = np.empty_like(w.k_cache)
    vc = np.empty_like(w.v_cache)
    kc[perm] = w.k_cache
    vc[perm] = w.v_cache
    w2 = w.with_(k_cache=kc, v_cache=vc, block_table=perm[w.block_table].astype(np.int32))
    a, _ = decode(DeviceWorkload(w))
    b, _ = decode(DeviceWorkload(w2))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("merge,wide", [(pa.PA_MERGE_LAST_ARRIVER, False), (pa.PA_MERGE_REDUCER, False),
                                        (pa.PA_MERGE_CLUSTER, False), (pa.PA_MERGE_LAST_ARRIVER, True),
                                        (pa.PA_MERGE_CLUSTER, True)])
def test_graph_replay_refresh_and_poison(merge, wide):
    """Capture one decode in a CUDA graph; before each replay poison the output
    with NaN and change the context lengths in place. Every replay must equal
    an eager call on the same lengths bit for bit, and the oracle within
    tolerance; arrival counters end at zero. `wide`: 32 rows per KV head, so
    the captured kernel is the tensor-memory consumer."""
    orc = oracle.get()
    w = _w(seed=12)
    if wide:
        w = pw.make_dense("modes-wide", batch=7, hkv=2, group=16, head_dim=128, query_len=2, page_size=16,
                          ctx_lens=[0, 3, 90, 600, 1300, 2222, 4001], kv_dtype=pw.KV_FP8,
                          scale_mode=pw.SCALE_PER_TENSOR, seed=12, causal=1, window=0, with_sinks=True)
    dw = DeviceWorkload(w)
    kw = dict(sm_count_override=6, ctas_per_sm_override=1) if merge != pa.PA_MERGE_CLUSTER else dict(
        schedule=pa.PA_SCHED_PER_UNIT, max_partitions=4)
    plan = pa.Plan(**dw.plan_fields(merge_mode=merge, max_context_len=8192, **kw))
    assert plan.info["consumer"] == (pa.PA_CONSUMER_TMEM if wide else pa.PA_CONSUMER_TILE)
    stream = torch.cuda.Stream()
    dw.poison_out()
    with torch.cuda.stream(stream):
        dw.run(plan, stream=stream)  # warm-up
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        dw.run(plan, stream=stream)
    rng = np.random.default_rng(4)
    for it in range(6):
        lens = rng.integers(0, w.ctx_lens.astype(np.int64) + 1).astype(np.int32)
        lens[it % w.batch] = 0
        dw.ctx.copy_(torch.from_numpy(lens))
        dw.poison_out()
        g.replay()
        torch.cuda.synchronize()
        replayed = dw.out.float().cpu().numpy().astype(np.float64)
        eager, _ = decode(dw, merge_mode=merge, max_context_len=8192, **kw)
        assert np.array_equal(replayed, eager)
        assert_parity(replayed, orc.decode(w.with_(ctx_lens=lens)), what=f"replay {it}")
    if merge == pa.PA_MERGE_LAST_ARRIVER:
        assert int(arrival_counters(plan, w.head_dim).abs().sum().item()) == 0
    assert plan.device_status() == 0


def test_status_and_counters_stay_clean():
    dw = DeviceWorkload(_w(seed=13))
    plan = pa.Plan(**dw.plan_fields(sm_count_override=4, ctas_per_sm_override=2))
    assert plan.info["merge_mode"] == pa.PA_MERGE_LAST_ARRIVER
    for _ in range(20):
        dw.run(plan)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert int(arrival_counters(plan, 128).abs().sum().item()) == 0
