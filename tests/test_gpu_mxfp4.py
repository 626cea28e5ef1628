"""GPU parity of MXFP4 K/V caches (OCP MX: E2M1 elements, one E8M0 scale per
32 head dims of a token row) against the oracle: shapes across the tile
consumer's warp layouts, page sizes, masks, sinks, FP16 queries and every
merge path; widely varying block scales; the full dense workload."""

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


MODES = [
    dict(),
    dict(sm_count_override=3, ctas_per_sm_override=1),
    dict(sm_count_override=5, ctas_per_sm_override=2, merge_mode=pa.PA_MERGE_REDUCER),
    dict(merge_mode=pa.PA_MERGE_DIRECT),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=3, merge_mode=pa.PA_MERGE_LAST_ARRIVER),
    dict(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=4, merge_mode=pa.PA_MERGE_CLUSTER),
]
MODE_IDS = ["auto", "balanced3", "reducer", "direct", "unit3-la", "cluster4"]


def mx_dense(name, seed, lens, group=8, ql=1, page=16, window=0, sinks=False, q_dtype=pw.Q_BF16, hkv=2, **kw):
    return pw.make_dense(name, batch=len(lens), hkv=hkv, group=group, head_dim=128, query_len=ql,
                         page_size=page, ctx_lens=lens, kv_dtype=pw.KV_MXFP4, scale_mode=pw.SCALE_MX_BLOCK,
                         seed=seed, causal=1, window=window, with_sinks=sinks, q_dtype=q_dtype, **kw)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_mxfp4_edges(orc, mode):
    lens = [0, 1, 15, 16, 17, 63, 64, 65, 127, 200, 777, 1500, 2049]
    w = mx_dense("mx-edges", 500, lens)
    gpu, plan = decode(DeviceWorkload(w), **mode)
    assert plan.info["consumer"] == pa.PA_CONSUMER_TILE
    assert_parity(gpu, orc.decode(w), what=f"mxfp4 edges {mode}")


# (group, query_len, page, window, sinks, q_dtype): one row warp with four token
# groups, two and three row warps, eight row warps (64 rows, the wide block)
SHAPES = [
    (8, 1, 64, 17, True, pw.Q_BF16),
    (16, 4, 128, 0, False, pw.Q_BF16),
    (4, 3, 32, 257, True, pw.Q_FP16),
    (12, 5, 16, 0, False, pw.Q_BF16),
    (1, 1, 16, 1, False, pw.Q_BF16),
    (2, 8, 256, 9, True, pw.Q_FP16),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"g{s[0]}-ql{s[1]}-p{s[2]}-w{s[3]}" for s in SHAPES])
def test_mxfp4_shapes(orc, shape):
    group, ql, page, window, sinks, q_dtype = shape
    lens = [0, 3, 130, 1000, 2300]
    w = mx_dense("mx-shape", 510 + SHAPES.index(shape), lens, group=group, ql=ql, page=page, window=window,
                 sinks=sinks, q_dtype=q_dtype)
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in MODES:
        gpu, _ = decode(dw, **m)
        assert_parity(gpu, ref, what=f"mxfp4 {shape} {m}")


def test_mxfp4_varied_block_scales(orc):
    """Block scales spread over 2^-12 .. 2^12 inside a token row and across
    tokens (the per-row normalisation to its largest block), large logits."""
    def spread(used, vals):
        blk = np.arange(vals.shape[-1]) // pw.MX_BLOCK  # 0..3
        return vals * np.exp2(4.0 * blk - 6.0).astype(np.float32)
    lens = [1, 40, 333, 1200]
    w = mx_dense("mx-spread", 530, lens, group=8, ql=2, page=16, vfun=spread, token_sigma=3.0, q_amplitude=4.0)
    ks = w.k_scale[w.k_scale != pw.E8M0_NAN].astype(np.int32)
    assert ks.max() - ks.min() >= 16  # the scales really do vary
    ref = orc.decode(w)
    dw = DeviceWorkload(w)
    for m in MODES[:4]:
        gpu, _ = decode(dw, **m)
        assert_parity(gpu, ref, what=f"mxfp4 varied scales {m}")


def test_mxfp4_dense_full(orc):
    """The dense workload (batch 64, 8 KV heads, GQA8, page 16, U[1024, 8192])
    in MXFP4, automatic plan, sampled units."""
    w = pw.dense(kv_dtype=pw.KV_MXFP4)
    gpu, plan = decode(DeviceWorkload(w), max_context_len=8192)
    assert plan.info["consumer"] == pa.PA_CONSUMER_TILE
    U = w.batch * w.num_kv_heads
    mask = np.zeros(U, dtype=np.uint8)
    mask[np.random.default_rng(5).choice(U, size=32, replace=False)] = 1
    mask[[0, U - 1]] = 1
    ref = orc.decode(w, unit_mask=mask)
    assert np.all(np.isfinite(gpu)), "non-finite outputs"
    assert_parity(gpu, ref, rows_mask=unit_rows_mask(w, mask), what="mxfp4 dense full")
