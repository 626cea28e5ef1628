"""CPU checks of the seeded input generator's byte accounting and encoders:
algorithmic_bytes against a brute-force count over visible tokens and pages,
and the MXFP4 encoder against the properties that define it."""

import numpy as np
import pytest

import pa_workloads as pw


def brute_bytes(w):
    """K/V rows (with block or per-token scales), block-table entries of the
    pages read, lengths, Q and output, sinks, sparse indices: counted by
    enumerating each sequence's visible token set."""
    total = 0
    for b in range(w.batch):
        L = int(w.ctx_lens[b])
        if w.topk:
            idx = w.topk_idx[b]
            toks = {int(t) for t in idx if 0 <= t < L}
            per_tok_extra = 4 * 2  # index + block-table entry per gathered token (as gathered)
            total += len([t for t in idx if 0 <= t < L]) * per_tok_extra
        else:
            toks = set()
            for i in range(w.query_len):
                p = L - w.query_len + i
                for t in range(L):
                    if w.causal and t > p:
                        continue
                    if w.window > 0 and t <= p - w.window:
                        continue
                    toks.add(t)
            # union over rows, with every token of the context the window leaves
            if toks:
                toks = set(range(min(toks), L))
            total += len({t // w.page_size for t in toks}) * 4
        n = len(toks) if not w.topk else len([t for t in w.topk_idx[b] if 0 <= t < L])
        if w.kv_dtype == pw.KV_MXFP4:
            row = w.head_dim // 2 + w.head_dim // 32
        else:
            row = w.head_dim * (1 if w.kv_dtype == pw.KV_FP8 else 2)
        total += n * w.num_kv_heads * row * 2
        if w.scale_mode == pw.SCALE_PER_TOKEN:
            total += n * w.num_kv_heads * 4 * 2
    total += w.batch * 4
    total += 2 * w.batch * w.query_len * w.num_q_heads * w.head_dim * 2
    if w.sinks is not None:
        total += w.num_q_heads * 4
    return total


CASES = [
    dict(kv=pw.KV_FP8, scale=pw.SCALE_PER_TENSOR, D=128, QL=1, S=16, window=0, lens=[0, 5, 16, 17, 300]),
    dict(kv=pw.KV_FP8, scale=pw.SCALE_PER_TOKEN, D=256, QL=4, S=64, window=17, lens=[3, 64, 65, 700]),
    dict(kv=pw.KV_BF16, scale=pw.SCALE_NONE, D=64, QL=2, S=32, window=1, lens=[1, 2, 40]),
    dict(kv=pw.KV_MXFP4, scale=pw.SCALE_MX_BLOCK, D=128, QL=3, S=128, window=0, lens=[0, 129, 1000]),
]


@pytest.mark.parametrize("c", CASES, ids=[f"kv{c['kv']}-d{c['D']}-ql{c['QL']}-w{c['window']}" for c in CASES])
def test_algorithmic_bytes_dense(c):
    w = pw.make_dense("acct", batch=len(c["lens"]), hkv=2, group=4, head_dim=c["D"], query_len=c["QL"],
                      page_size=c["S"], ctx_lens=c["lens"], kv_dtype=c["kv"], scale_mode=c["scale"], seed=3,
                      causal=1, window=c["window"], with_sinks=True)
    assert pw.algorithmic_bytes(w) == brute_bytes(w)


def test_algorithmic_bytes_sparse():
    w = pw.small_sparse(rows=4, topk=200, context=500)
    assert pw.algorithmic_bytes(w) == brute_bytes(w)


def test_mxfp4_encode_properties():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((64, 128)) * np.exp(rng.standard_normal((64, 1)) * 3)).astype(np.float32)
    x[0, :32] = 0.0  # an all-zero block
    packed, X = pw.mxfp4_encode(x)
    assert packed.shape == (64, 64) and X.shape == (64, 4)
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(64, 128)
    mag = pw.E2M1_GRID[codes & 7].astype(np.float64)
    dec = np.where(codes & 8, -mag, mag) * np.repeat(np.exp2(X.astype(np.float64) - 127), 32, axis=1)
    blk = np.abs(x.astype(np.float64)).reshape(64, 4, 32).max(axis=2)
    # the block's largest magnitude lands in [4, 8) units of its scale (exponent floor(log2 amax) - 2)
    unit = np.exp2(X.astype(np.float64) - 127)
    nz = blk > 0
    assert np.all((blk[nz] / unit[nz] >= 4) & (blk[nz] / unit[nz] < 8))
    # each element is the nearest E2M1 value of x / unit (saturated at 6): no grid point is closer
    s = np.repeat(unit, 32, axis=1)
    r = np.abs(x / s)
    err = np.abs(np.abs(dec / s) - np.minimum(r, 6.0))
    best = np.abs(r[..., None] - pw.E2M1_GRID[None, None, :]).min(axis=-1)
    assert np.all(err <= best + 1e-6)
    # signs follow the input (zeros aside), the zero block decodes to zeros
    assert np.all((dec == 0) | (np.sign(dec) == np.sign(x)))
    assert np.all(dec[0, :32] == 0)
    # values already on the grid are kept exactly
    e = np.exp2(rng.integers(-6, 6, size=(8, 1)).astype(np.float64))
    grid = (pw.E2M1_GRID[rng.integers(0, 8, size=(8, 128))] * e).astype(np.float32)
    grid[:, ::32] = (6.0 * e).astype(np.float32)  # each block's largest value: 6 units
    p2, X2 = pw.mxfp4_encode(grid)
    c2 = np.stack([p2 & 0xF, p2 >> 4], axis=-1).reshape(8, 128)
    d2 = pw.E2M1_GRID[c2 & 7] * np.repeat(np.exp2(X2.astype(np.float64) - 127), 32, axis=1)
    assert np.array_equal(d2, np.abs(grid).astype(np.float64))


def test_transpose_v_moves_values():
    rng = np.random.default_rng(1)
    v = rng.integers(0, 1 << 16, size=(3, 2, 32, 64), dtype=np.uint16)
    t = pw.transpose_v(v)
    assert t.shape == (3, 2, 4, 64, 8)
    for p, g, s, d in [(0, 0, 0, 0), (2, 1, 31, 63), (1, 0, 9, 17), (2, 1, 8, 0)]:
        assert t[p, g, s // 8, d, s % 8] == v[p, g, s, d]


def test_bench_names_follow_the_options():
    import argparse

    import bench

    def ns(**kw):
        d = dict(batch=0, page=16, window=0, sinks=False, partitions=0, merge="auto", consumer="auto",
                 workload="dense", rows=1024, kv="fp8", ql=1, v_layout="plain")
        d.update(kw)
        return argparse.Namespace(**d)

    assert bench.profile_name(ns(), "pa_tile") == "pa_tile_dense"
    assert bench.profile_name(ns(kv="mxfp4"), "pa_tile") == "pa_tile_dense_mxfp4"
    assert bench.profile_name(ns(workload="mtp4", kv="bf16"), "pa_mtp") == "pa_mtp_mtp4_bf16"
    assert bench.profile_name(ns(workload="d256", ql=4), "pa_mtp") == "pa_mtp_d256_ql4"
    assert bench.profile_name(ns(kv="bf16"), "pa_tile") is None  # no summary covers dense BF16
    assert bench.profile_name(ns(kv="bf16", v_layout="transposed"), "pa_tile") is None
    assert bench.profile_name(ns(batch=16), "pa_tile") is None  # a non-default size
    assert "MXFP4" in bench.workload_name(ns(kv="mxfp4"))
    assert "transposed" in bench.workload_name(ns(kv="bf16", v_layout="transposed"))
    assert bench.workload_name(ns()) == bench.WORKLOADS["dense"]
