"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark uses (automatic plan), checked against the oracle
on sampled (sequence, KV head) units; every output must be finite."""

import numpy as np
import pytest

import oracle
import paged_attention_decode_attn_gb300 as pa
import pa_workloads as pw

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import DeviceWorkload, assert_parity, decode, unit_rows_mask  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_attention_decode_attn_gb300 import _build

    _build.build()


def sampled(w, n, seed=0, include=()):
    U = w.batch * w.num_kv_heads
    rng = np.random.default_rng(seed)
    mask = np.zeros(U, dtype=np.uint8)
    mask[rng.choice(U, size=min(n, U), replace=False)] = 1
    for u in include:
        mask[u] = 1
    return mask


def check(orc, w, gpu, n_units, seed=0, include=()):
    mask = sampled(w, n_units, seed, include)
    ref = orc.decode(w, unit_mask=mask)
    assert np.all(np.isfinite(gpu)), "non-finite outputs"
    assert_parity(gpu, ref, rows_mask=unit_rows_mask(w, mask), what=w.name)


def test_tiny_full(orc):
    w = pw.tiny()
    gpu, plan = decode(DeviceWorkload(w))
    assert_parity(gpu, orc.decode(w), what="tiny")


def test_dense_full(orc):
    w = pw.dense()
    gpu, plan = decode(DeviceWorkload(w), max_context_len=8192)
    assert plan.info["merge_mode"] == pa.PA_MERGE_LAST_ARRIVER
    check(orc, w, gpu, 40, include=(0, 511))


@pytest.mark.parametrize("ql,window,sinks,consumer", [
    (1, 0, False, 0), (4, 0, True, 1), (3, 8193, False, 1), (2, 257, True, 0), (4, 17, False, 1), (1, 1, True, 0),
    (4, 0, True, 2), (3, 8193, False, 2), (4, 17, False, 2)])
def test_d256_full(orc, ql, window, sinks, consumer):
    w = pw.d256(query_len=ql, window=window, with_sinks=sinks)
    gpu, plan = decode(DeviceWorkload(w), max_context_len=131135, consumer=consumer)
    # seq 0 is empty; odd seqs 8K, even seqs 128K; always include the empty one
    check(orc, w, gpu, 3 if window == 0 else 8, seed=ql, include=(0, 1, 2 * 3 + 1))


@pytest.mark.parametrize("kv", [pw.KV_FP8, pw.KV_BF16], ids=["fp8", "bf16"])
def test_sparse_full(orc, kv):
    w = pw.sparse(kv_dtype=kv)
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in [dict()] + [dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=p) for p in (2, 4, 8, 16)]:
        gpu, _ = decode(dw, **m)
        assert_parity(gpu, ref, what=f"sparse {m}")


@pytest.mark.parametrize("consumer", [pa.PA_CONSUMER_TILE, pa.PA_CONSUMER_TMEM], ids=["tile", "tmem"])
@pytest.mark.parametrize("kv", [pw.KV_FP8, pw.KV_BF16], ids=["fp8", "bf16"])
def test_mtp4_full(orc, kv, consumer):
    w = pw.mtp4(kv_dtype=kv)
    gpu, plan = decode(DeviceWorkload(w), max_context_len=65536, consumer=consumer)
    check(orc, w, gpu, 6, seed=kv)


@pytest.mark.parametrize("rows,kv", [(1024, pw.KV_FP8), (1024, pw.KV_BF16), (8192, pw.KV_FP8)],
                         ids=["1024-fp8", "1024-bf16", "8192-fp8"])
def test_sparse_prefill_full(orc, rows, kv):
    """Sparse prefill at the pages' row counts, in the benchmark's automatic
    plan; checked on sampled rows, always including the first, the row where
    the 2048-token cap starts, and the last."""
    w = pw.sparse_prefill(kv_dtype=kv, rows=rows)
    gpu, plan = decode(DeviceWorkload(w))
    assert plan.info["launches_per_call"] == 1
    include = [0, 1, min(2047, rows - 1), min(2048, rows - 1), rows - 1]
    check(orc, w, gpu, 48, seed=rows, include=include)
