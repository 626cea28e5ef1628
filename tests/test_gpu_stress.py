"""GPU parity on inputs that stress the online softmax and the scale
handling, against the CPU oracle:

* query amplitudes x8 and x16, so logits spread far beyond the N(0,1)
  default and a row's running max keeps moving inside a segment (the
  tensor-memory consumer then leaves its lazy-max fast path and rescales O
  and L in tensor memory);
* a planted dominant key late in a long context, so the max jumps by tens of
  log2 units in a segment's last stages;
* all-zero query rows (uniform attention; the power-of-two row scale of a
  zero row);
* K and V token magnitudes varied by e^N(0,1) (PR "Merge gfx1250 PA decode
  partitions in the tile kernel and speed up dense decode", Validation:
  per-token magnitudes that fail when a scale is misplaced);
* V amplitudes scaled by 1/16 (PR "Extend packed D256 PA decode pipe to
  page16, transposed V and sliding windows", Validation).

Each case runs every stage consumer that covers its shape, with the
automatic schedule (short segments) and with three CTAs (long segments, many
stages per segment)."""

import numpy as np
import pytest

import oracle
import paged_attention_decode_attn_gb300 as pa
import pa_workloads as pw

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import DeviceWorkload, assert_parity, decode  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_attention_decode_attn_gb300 import _build

    _build.build()


LENS = [0, 1, 130, 1000, 3000, 5000]

# (name, group, query_len, head_dim, page, kv dtype, scale mode)
SHAPES = [
    ("gqa8-d128-fp8", 8, 1, 128, 16, pw.KV_FP8, pw.SCALE_PER_TENSOR),
    ("mtp4-gqa16-fp8", 16, 4, 128, 128, pw.KV_FP8, pw.SCALE_PER_TENSOR),
    ("mtp4-gqa16-bf16", 16, 4, 128, 128, pw.KV_BF16, pw.SCALE_NONE),
    ("mtp2-gqa16-fp8-tok", 16, 2, 128, 16, pw.KV_FP8, pw.SCALE_PER_TOKEN),
    ("mtp4-gqa8-d256-fp8-tok", 8, 4, 256, 64, pw.KV_FP8, pw.SCALE_PER_TOKEN),
]
CONDITIONS = ["q_x8", "q_x16", "planted_key", "zero_q_rows", "token_magnitudes", "v_div16"]


def _consumers(group, ql, head_dim, kv):
    out = [pa.PA_CONSUMER_TILE]
    R = group * ql
    if R > (8 if head_dim == 256 else 16) and (head_dim == 128 or kv == pw.KV_FP8):
        out.append(pa.PA_CONSUMER_TMEM)
    return out


def _build_case(shape, cond, seed):
    name, group, ql, D, page, kv, sm = shape
    kw = {}
    if cond == "q_x8":
        kw["q_amplitude"] = 8.0
    elif cond == "q_x16":
        kw["q_amplitude"] = 16.0
    elif cond == "token_magnitudes":
        kw["token_sigma"] = 1.0
    elif cond == "v_div16":
        kw["v_amplitude"] = 1.0 / 16
    w = pw.make_dense(f"stress-{name}-{cond}", batch=len(LENS), hkv=2, group=group, head_dim=D, query_len=ql,
                      page_size=page, ctx_lens=LENS, kv_dtype=kv, scale_mode=sm, seed=seed, causal=1,
                      with_sinks=(cond == "zero_q_rows"), **kw)
    if cond == "zero_q_rows":
        q = w.q.copy()
        q[1::3, ::3, :] = 0  # every third head of every third row
        w = w.with_(q=q)
    elif cond == "planted_key":
        # Each (sequence, KV head) gets a random sign pattern u; its query rows
        # get +2u added (a shared component), and one late token's key is u at
        # the cache's largest magnitude, so that token's logit dominates every
        # row of the group by tens of log2 units.
        rng = np.random.default_rng(seed + 1)
        qf = (w.q.astype(np.uint32) << 16).view(np.float32).copy()
        kc = w.k_cache.copy()
        for b, L in enumerate(LENS):
            if L < 1000:
                continue
            t = L - ql - 37
            for g in range(2):
                u = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
                qf[b * ql:(b + 1) * ql, g * group:(g + 1) * group, :] += 2.0 * u
                page_id = w.block_table[b, t // page]
                if kv == pw.KV_BF16:
                    kc[page_id, g, t % page] = pw.bf16_bits(3.0 * u)
                else:
                    kc[page_id, g, t % page] = pw.fp8_codes(448.0 * u)  # largest code
        w = w.with_(q=pw.bf16_bits(qf), k_cache=kc)
    return w


@pytest.mark.parametrize("cond", CONDITIONS)
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_stress(shape, cond):
    w = _build_case(shape, cond, seed=300 + CONDITIONS.index(cond))
    ref = oracle.get().decode(w)
    dw = DeviceWorkload(w)
    _, group, ql, D, _, kv, _ = shape
    for consumer in _consumers(group, ql, D, kv):
        for sched in (dict(), dict(sm_count_override=3, ctas_per_sm_override=1)):
            gpu, plan = decode(dw, consumer=consumer, **sched)
            assert plan.info["consumer"] == consumer
            assert_parity(gpu, ref, what=f"{shape[0]} {cond} consumer {consumer} {sched}")


def test_planted_key_output_is_its_value_row():
    """With the planted key dominating, every query row of a long sequence
    returns (within tolerance) that token's V row: the late max jump must
    rescale everything accumulated before it to nothing."""
    shape = SHAPES[1]
    w = _build_case(shape, "planted_key", seed=999)
    ref = oracle.get().decode(w)
    b = LENS.index(5000)
    # the oracle itself: all query positions of the long sequence return
    # (nearly) one V row per KV group
    rows = ref[b * 4:(b + 1) * 4]
    assert np.allclose(rows, rows[:1], atol=1e-3)
    for g in range(2):
        grp = rows[:, g * 16:(g + 1) * 16]
        assert np.allclose(grp, grp[:1, :1], atol=1e-3)
    dw = DeviceWorkload(w)
    for consumer in (pa.PA_CONSUMER_TILE, pa.PA_CONSUMER_TMEM):
        gpu, _ = decode(dw, consumer=consumer, sm_count_override=2, ctas_per_sm_override=1)
        assert_parity(gpu, ref, what=f"planted key consumer {consumer}")
