"""GPU parity of the transposed BF16 V layout ([pages, Hkv, S/8, D, 8]): the
oracle on the same inputs, and bit-identical outputs to the plain layout
holding the same values (the kernel feeds the same values to the same MMA
fragments), at head_dim 64/128/256, with BF16 and FP16 queries and every
merge path."""

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


MODES = [
    dict(),
    dict(sm_count_override=3, ctas_per_sm_override=1),
    dict(sm_count_override=5, ctas_per_sm_override=2, merge_mode=pa.PA_MERGE_REDUCER),
    dict(merge_mode=pa.PA_MERGE_DIRECT),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=3, merge_mode=pa.PA_MERGE_LAST_ARRIVER),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=4, merge_mode=pa.PA_MERGE_CLUSTER),
]
MODE_IDS = ["auto", "balanced3", "reducer", "direct", "unit3-la", "cluster4"]

# (head_dim, group, query_len, page, window, sinks, q_dtype)
CASES = [
    (128, 8, 1, 16, 0, False, pw.Q_BF16),
    (128, 16, 4, 128, 17, True, pw.Q_BF16),
    (64, 8, 1, 16, 0, False, pw.Q_BF16),
    (64, 12, 5, 64, 257, True, pw.Q_FP16),
    (256, 8, 2, 64, 0, True, pw.Q_BF16),
    (256, 4, 1, 32, 9, False, pw.Q_FP16),
]


def pair(case, seed, lens):
    D, group, ql, page, window, sinks, q_dtype = case
    mk = lambda layout: pw.make_dense("tv", batch=len(lens), hkv=2, group=group, head_dim=D, query_len=ql,  # noqa: E731
                                      page_size=page, ctx_lens=lens, kv_dtype=pw.KV_BF16, scale_mode=pw.SCALE_NONE,
                                      seed=seed, causal=1, window=window, with_sinks=sinks, q_dtype=q_dtype,
                                      v_layout=layout)
    return mk(pw.V_PLAIN), mk(pw.V_TRANSPOSED)


@pytest.mark.parametrize("case", CASES, ids=[f"d{c[0]}-g{c[1]}-ql{c[2]}-p{c[3]}-w{c[4]}" for c in CASES])
def test_transposed_v(orc, case):
    plain, tv = pair(case, 600 + CASES.index(case), [0, 1, 17, 130, 1000, 2300])
    ref = orc.decode(tv)
    dp, dt = DeviceWorkload(plain), DeviceWorkload(tv)
    for m in MODES:
        # the plain layout on the same (tile) consumer: AUTO would take the
        # tensor-memory consumer for more than 16 rows (8 at head_dim 256)
        out_p, _ = decode(dp, consumer=pa.PA_CONSUMER_TILE, **m)
        out_t, plan = decode(dt, **m)
        assert plan.info["consumer"] == pa.PA_CONSUMER_TILE
        assert_parity(out_t, ref, what=f"transposed V {case} {m}")
        assert np.array_equal(out_t, out_p), f"transposed V differs from plain V: {case} {m}"


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_transposed_v_edges(orc, mode):
    lens = [0, 1, 7, 8, 9, 15, 16, 17, 63, 64, 65, 127, 200, 777, 1500, 2049]
    plain, tv = pair((128, 8, 1, 16, 0, False, pw.Q_BF16), 620, lens)
    out_t, _ = decode(DeviceWorkload(tv), **mode)
    out_p, _ = decode(DeviceWorkload(plain), consumer=pa.PA_CONSUMER_TILE, **mode)
    assert_parity(out_t, orc.decode(tv), what=f"transposed V edges {mode}")
    assert np.array_equal(out_t, out_p)
