"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with

* a library routine (torch's float8_e4m3fn / bfloat16 casts, scipy's softmax),
* the published FP8 format (golden spot values) and the OCP MX FP4/E8M0
  tables (golden, every code),
* an independent brute-force route (NumPy float64 dense attention on
  contiguous dequantised K/V with an explicit mask and a library softmax),
* closed forms (one and two visible tokens, constant V, a sink with one token),
* invariants fixed by the semantics (window 1 returns the query position's V,
  a causal MTP row equals a single-query decode over its prefix, block-table
  relocation, empty contexts, split/merge in any order, sparse lists that
  enumerate the dense context).

The same functions run against deliberately broken copies of the oracle in
``test_oracle_mutants.py`` to show that each plausible mistake trips one.
"""

from __future__ import annotations

import os

import numpy as np
import scipy.special
import torch

import pa_workloads as pw

HERE = os.path.dirname(os.path.abspath(__file__))


# --- an independent second route ----------------------------------------------

def mx_tables():
    """(E2M1 value per code [16], E8M0 value per code [256]) from the golden
    fixture of the OCP MX tables (E8M0 spot values there; the rest from its
    stated rule 2^(code - 127), NaN at 0xFF)."""
    e2m1 = np.full(16, np.nan)
    e8m0 = np.ldexp(1.0, np.arange(256) - 127)
    e8m0[0xFF] = np.nan
    spot = {}
    for line in open(os.path.join(HERE, "golden", "mx_fp4_e2m1_e8m0.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kind, code, val = line.split()
        if kind == "e2m1":
            e2m1[int(code, 16)] = float(val)
        else:
            spot[int(code, 16)] = float(val)
    for c, v in spot.items():
        assert (np.isnan(v) and np.isnan(e8m0[c])) or e8m0[c] == v, ("E8M0 rule vs fixture", c)
    assert not np.isnan(e2m1).any()
    return e2m1, e8m0


def dequant(w, which: str) -> np.ndarray:
    """Dequantise a whole cache with torch's casts, or the MX tables for
    MXFP4 (float64 [P, Hkv, S, D])."""
    cache = w.k_cache if which == "k" else w.v_cache
    scale = w.k_scale if which == "k" else w.v_scale
    if which == "v" and getattr(w, "v_layout", pw.V_PLAIN) == pw.V_TRANSPOSED:
        # [P, Hkv, S/8, D, 8] back to [P, Hkv, S, D]: swap the last two axes, merge chunks
        P, H, C, D, E = cache.shape
        cache = np.ascontiguousarray(np.swapaxes(cache, 3, 4)).reshape(P, H, C * E, D)
    if w.kv_dtype == pw.KV_MXFP4:
        e2m1, e8m0 = mx_tables()
        lo = e2m1[cache & 0xF]
        hi = e2m1[cache >> 4]
        elems = np.stack([lo, hi], axis=-1).reshape(cache.shape[:-1] + (2 * cache.shape[-1],))
        return elems * np.repeat(e8m0[scale], pw.MX_BLOCK, axis=-1)
    if w.kv_dtype == pw.KV_BF16:
        t = torch.from_numpy(np.ascontiguousarray(cache).view(np.int16)).view(torch.bfloat16)
        return t.double().numpy()
    vals = torch.from_numpy(np.ascontiguousarray(cache)).view(torch.float8_e4m3fn).double().numpy()
    if w.scale_mode == pw.SCALE_PER_TENSOR:
        vals = vals * float(scale[0])
    elif w.scale_mode == pw.SCALE_PER_TOKEN:
        vals = vals * scale.astype(np.float64)[..., None]
    return vals


def q_double(w) -> np.ndarray:
    qt = torch.float16 if getattr(w, "q_dtype", pw.Q_BF16) == pw.Q_FP16 else torch.bfloat16
    t = torch.from_numpy(np.ascontiguousarray(w.q).view(np.int16)).view(qt)
    return t.double().numpy()


def brute_force(w, sm_scale=None) -> np.ndarray:
    """Dense float64 attention over gathered contiguous K/V with a mask matrix."""
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(w.head_dim)
    sm_scale = float(np.float32(sm_scale))
    K = dequant(w, "k")
    V = dequant(w, "v")
    Q = q_double(w)
    B, QL, Hq, D = w.batch, w.query_len, w.num_q_heads, w.head_dim
    G = w.group
    out = np.zeros((B * QL, Hq, D))
    for b in range(B):
        L = int(w.ctx_lens[b])
        if w.topk:
            idx = w.topk_idx[b]
            tok = idx[(idx >= 0) & (idx < L)].astype(np.int64)
        else:
            tok = np.arange(L, dtype=np.int64)
        if tok.size == 0:
            continue
        pages = w.block_table[b, tok // w.page_size]
        slots = tok % w.page_size
        for g in range(w.num_kv_heads):
            Kb = K[pages, g, slots]  # [n, D]
            Vb = V[pages, g, slots]
            for i in range(QL):
                p = L - QL + i
                allowed = np.ones(tok.size, dtype=bool)
                if not w.topk:
                    if w.causal:
                        allowed &= tok <= p
                    if w.window > 0:
                        allowed &= tok > p - w.window
                if not allowed.any():
                    continue
                heads = np.arange(g * G, (g + 1) * G)
                qg = Q[b * QL + i, heads]  # [G, D]
                logits = sm_scale * (qg @ Kb[allowed].T)  # [G, n]
                if w.sinks is not None:
                    logits = np.concatenate([logits, w.sinks[heads, None].astype(np.float64)], axis=1)
                P = scipy.special.softmax(logits, axis=1)
                out[b * QL + i, heads] = P[:, : int(allowed.sum())] @ Vb[allowed]
    return out


def assert_close(a, b, rtol=1e-11, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    bad = ~np.isclose(a, b, rtol=rtol, atol=atol, equal_nan=False)
    assert not bad.any(), f"{what}: {int(bad.sum())} mismatches, max |diff| {np.nanmax(np.abs(a - b))}"


def small(seed, *, hkv=1, group=4, D=32, QL=1, S=16, lens=(5, 23, 40), kv=pw.KV_FP8,
          scale=pw.SCALE_PER_TENSOR, causal=1, window=0, sinks=False, **kw):
    return pw.make_dense("pin", batch=len(lens), hkv=hkv, group=group, head_dim=D,
                         query_len=QL, page_size=S, ctx_lens=list(lens), kv_dtype=kv,
                         scale_mode=scale, seed=seed, causal=causal, window=window,
                         with_sinks=sinks, **kw)


# --- codec pins -----------------------------------------------------------------

def pin_e4m3_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.e4m3_to_double(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib)), "NaN codes differ from torch"
    ok = ~np.isnan(lib)
    assert np.array_equal(mine[ok], lib[ok]), "e4m3 values differ from torch"


def pin_e4m3_golden(orc):
    path = os.path.join(HERE, "golden", "e4m3_spot_values.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val = line.split()
        got = orc.e4m3_to_double([int(code, 16)])[0]
        want = float(val)
        if np.isnan(want):
            assert np.isnan(got), code
        else:
            assert got == want and np.signbit(got) == np.signbit(want), (code, got, want)


def pin_mx_codes(orc):
    """Every E2M1 code and the E8M0 spot codes against the OCP MX tables."""
    e2m1, e8m0 = mx_tables()
    got = orc.e2m1_to_double(np.arange(16))
    assert np.array_equal(got, e2m1) and np.array_equal(np.signbit(got), np.signbit(e2m1)), "E2M1 values"
    got = orc.e8m0_to_double(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(e8m0)), "E8M0 NaN code"
    ok = ~np.isnan(e8m0)
    assert np.array_equal(got[ok], e8m0[ok]), "E8M0 values"


def pin_mx_brute_force(orc):
    """MXFP4 caches: the oracle against dense attention over K/V decoded
    with the MX tables (nibble order, block index, scale row layout)."""
    cases = [
        dict(seed=61, D=64, lens=(5, 23, 40)),
        dict(seed=62, D=32, QL=3, window=17, lens=(0, 2, 19, 64), group=2),
        dict(seed=63, D=128, QL=2, sinks=True, hkv=2, group=2, S=64, lens=(1, 70, 130)),
        dict(seed=64, D=64, q_dtype=pw.Q_FP16, causal=0, QL=2, lens=(9, 33), token_sigma=2.0),
    ]
    for c in cases:
        w = small(kv=pw.KV_MXFP4, scale=pw.SCALE_MX_BLOCK, **c)
        assert_close(orc.decode(w), brute_force(w), what=f"mx brute force {c}")


def pin_mx_constant_v(orc):
    """MXFP4 V whose every element encodes 0.75 gives 0.75 (and blocks of
    different scales in one row stay exact: 3 * 2^-2 and 1.5 * 2^-1)."""
    def vconst(used, vals):
        return np.full_like(vals, 0.75)
    w = small(65, kv=pw.KV_MXFP4, scale=pw.SCALE_MX_BLOCK, D=64, QL=2, lens=(3, 40), vfun=vconst)
    out = orc.decode(w)
    assert_close(out, np.full_like(out, 0.75), what="mx constant V")


def pin_transposed_v(orc):
    """Transposed V (BF16 [P, Hkv, S/8, D, 8]): the oracle against the brute
    force (which undoes the layout with NumPy axis swaps), and equal to the
    same values in the plain layout."""
    cases = [
        dict(seed=71, D=64, S=16, lens=(5, 23, 40)),
        dict(seed=72, D=32, S=64, QL=3, window=17, lens=(0, 2, 19, 130), group=2, sinks=True),
        dict(seed=73, D=128, S=32, QL=2, q_dtype=pw.Q_FP16, lens=(1, 70, 99), hkv=2, group=2),
    ]
    for c in cases:
        w = small(kv=pw.KV_BF16, scale=pw.SCALE_NONE, v_layout=pw.V_TRANSPOSED, **c)
        assert w.v_cache.shape[-1] == pw.V_CHUNK
        out = orc.decode(w)
        assert_close(out, brute_force(w), what=f"transposed V brute force {c}")
        plain = small(kv=pw.KV_BF16, scale=pw.SCALE_NONE, **c)
        assert np.array_equal(plain.k_cache, w.k_cache)
        assert_close(out, orc.decode(plain), rtol=0, atol=0, what=f"transposed V = plain {c}")


def pin_bf16_widen(orc):
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    mine = orc.bf16_to_double(bits)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(mine[ok], lib[ok]), "bf16 widening differs from torch"


def pin_f16_widen(orc):
    """All 65536 binary16 patterns against torch's float16 cast, plus values
    that follow from the format's definition (IEEE 754 binary16: bias 15,
    10 fraction bits, subnormals f * 2^-24)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = orc.f16_to_double(bits)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.float16).double().numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan), "f16 NaN patterns differ from torch"
    assert np.array_equal(mine[~nan], lib[~nan]), "f16 widening differs from torch"
    spot = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0400: 2.0 ** -14, 0x0001: 2.0 ** -24,
            0x03FF: 1023 * 2.0 ** -24, 0x3555: 0.333251953125, 0x7C00: np.inf, 0xFC00: -np.inf, 0x8000: -0.0}
    for b, v in spot.items():
        got = orc.f16_to_double([b])[0]
        assert got == v and np.signbit(got) == np.signbit(v), (hex(b), got, v)


def pin_bf16_round(orc):
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 3000),
        np.float32([1e-40, -3e-39, 3.3e38, 1.0, 0.0]),
    ]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = orc.round_bf16(x.astype(np.float64))
    assert np.array_equal(mine, lib), "bf16 rounding differs from torch on binary32 inputs"
    # ties to even (IEEE 754 roundTiesToEven): 1+2^-8 -> 1.0, 1+3*2^-8 -> 1+2^-6
    assert orc.round_bf16([1.0 + 2.0 ** -8])[0] == 0x3F80
    assert orc.round_bf16([1.0 + 3 * 2.0 ** -8])[0] == 0x3F82
    assert orc.round_bf16([-(1.0 + 2.0 ** -8)])[0] == 0xBF80


# --- attention pins ---------------------------------------------------------------

def pin_brute_force(orc):
    cases = [
        dict(seed=11),
        dict(seed=12, scale=pw.SCALE_PER_TOKEN, QL=3, window=17, lens=(0, 2, 19, 64)),
        dict(seed=13, kv=pw.KV_BF16, QL=4, window=2, sinks=True, hkv=2, group=2),
        dict(seed=14, QL=2, causal=0, sinks=True, S=64, lens=(1, 70, 130)),
        dict(seed=15, scale=pw.SCALE_PER_TOKEN, QL=4, window=1, group=8, lens=(3, 33, 50)),
        dict(seed=16, hkv=3, group=1, QL=1, window=5, lens=(7, 16, 17, 45)),
        dict(seed=17, q_dtype=pw.Q_FP16, QL=2, window=9, lens=(4, 31, 66)),
        dict(seed=18, q_dtype=pw.Q_FP16, kv=pw.KV_BF16, group=8, sinks=True, lens=(2, 47)),
    ]
    for c in cases:
        w = small(**c)
        assert_close(orc.decode(w), brute_force(w), what=f"brute force {c}")


def pin_one_token(orc):
    """L = 1: the single visible token's V, whatever q is; with a sink,
    V / (1 + e^(s - x))."""
    for kv in (pw.KV_FP8, pw.KV_BF16):
        w = small(21, kv=kv, lens=(1, 1), group=2)
        V = dequant(w, "v")
        K = dequant(w, "k")
        Q = q_double(w)
        out = orc.decode(w)
        for b in range(2):
            page = w.block_table[b, 0]
            for h in range(2):
                assert_close(out[b, h], V[page, 0, 0], what="one token")
        ws = w.with_(sinks=np.float32([0.7, -1.3]))
        out = orc.decode(ws)
        sm = float(np.float32(1.0 / np.sqrt(w.head_dim)))
        for b in range(2):
            page = w.block_table[b, 0]
            for h in range(2):
                x = sm * float(Q[b, h] @ K[page, 0, 0])
                want = V[page, 0, 0] / (1.0 + np.exp(float(ws.sinks[h]) - x))
                assert_close(out[b, h], want, what="one token + sink")


def pin_two_tokens(orc):
    """L = 2: sigma(x0 - x1) v0 + sigma(x1 - x0) v1."""
    w = small(22, lens=(2,), group=1, D=16)
    V = dequant(w, "v")
    K = dequant(w, "k")
    Q = q_double(w)
    sm = float(np.float32(1.0 / np.sqrt(16)))
    page = w.block_table[0, 0]
    x0 = sm * float(Q[0, 0] @ K[page, 0, 0])
    x1 = sm * float(Q[0, 0] @ K[page, 0, 1])
    want = scipy.special.expit(x0 - x1) * V[page, 0, 0] + scipy.special.expit(x1 - x0) * V[page, 0, 1]
    assert_close(orc.decode(w)[0, 0], want, what="two tokens")


def pin_constant_v(orc):
    """Constant V rows give that constant; a sink scales it by sum e^x / (sum e^x + e^s)."""
    c = 0.625  # exact in BF16 and in e4m3
    def vconst(used, vals):
        return np.full_like(vals, c)
    w = small(23, kv=pw.KV_BF16, QL=2, window=9, lens=(4, 30, 61), group=2, vfun=vconst)
    out = orc.decode(w)
    assert_close(out, np.full_like(out, c), what="constant V")
    ws = w.with_(sinks=np.float32([0.3, 2.0]))
    outs = orc.decode(ws)
    bf = brute_force(w)  # same logits; derive the sink factor from them independently
    K = dequant(w, "k")
    Q = q_double(w)
    sm = float(np.float32(1.0 / np.sqrt(w.head_dim)))
    for b in range(w.batch):
        L = int(w.ctx_lens[b])
        for i in range(2):
            p = L - 2 + i
            tok = np.arange(max(0, p - 8), p + 1)
            pages = w.block_table[b, tok // w.page_size]
            for h in range(2):
                x = sm * (K[pages, 0, tok % w.page_size] @ Q[b * 2 + i, h])
                lse = scipy.special.logsumexp(x)
                factor = 1.0 / (1.0 + np.exp(float(ws.sinks[h]) - lse))
                assert_close(outs[b * 2 + i, h], c * factor * np.ones(w.head_dim), what="const V sink")
    assert bf.shape == outs.shape


def pin_window_one_position(orc):
    """Window 1 returns the V row of the query's own position. V rows carry
    their logical position in base-16 digits, so the output decodes to p
    exactly: this pins page lookup, slot, window bound and query position."""
    for kv in (pw.KV_BF16, pw.KV_FP8):
        w0 = small(24, QL=4, window=1, lens=(1, 4, 17, 100, 333), S=16, D=16, kv=kv,
                   scale=pw.SCALE_NONE, group=2)
        # rebuild V so that row (b, t) holds digits of t
        V = np.zeros_like(w0.v_cache)
        for b in range(w0.batch):
            L = int(w0.ctx_lens[b])
            for t in range(L):
                page = w0.block_table[b, t // w0.page_size]
                digits = [(t >> (4 * k)) & 15 for k in range(4)] + [b]
                vals = np.zeros(w0.head_dim, dtype=np.float32)
                vals[: len(digits)] = digits
                V[page, 0, t % w0.page_size] = (pw.bf16_bits(vals) if kv == pw.KV_BF16
                                                else pw.fp8_codes(vals))
        w = w0.with_(v_cache=V)
        out = orc.decode(w)
        for b in range(w.batch):
            L = int(w.ctx_lens[b])
            for i in range(4):
                p = L - 4 + i
                for h in range(w.num_q_heads):
                    row = out[b * 4 + i, h]
                    if p < 0:
                        assert np.all(row == 0), "row before the context must be zero"
                        continue
                    got = sum(int(round(row[k])) << (4 * k) for k in range(4))
                    assert got == p and int(round(row[4])) == b, (b, i, got, p)


def pin_causal_prefix(orc):
    """A causal MTP row i is a single-query decode over the first p + 1 tokens."""
    w = small(25, QL=4, lens=(4, 9, 40, 77), group=2, sinks=True, scale=pw.SCALE_PER_TOKEN)
    out = orc.decode(w)
    for i in range(4):
        q1 = w.q.reshape(w.batch, 4, w.num_q_heads, w.head_dim)[:, i].copy()
        w1 = w.with_(query_len=1, q=q1, ctx_lens=np.maximum(0, w.ctx_lens - 4 + 1 + i).astype(np.int32))
        ref = orc.decode(w1)
        assert_close(out.reshape(w.batch, 4, w.num_q_heads, -1)[:, i], ref, rtol=0, atol=0,
                     what=f"prefix row {i}")


def pin_relocation(orc):
    """Moving pages in the pool and rewriting the table changes nothing."""
    w = small(26, QL=2, lens=(3, 50, 17), scale=pw.SCALE_PER_TOKEN, window=20)
    rng = np.random.default_rng(1)
    perm = rng.permutation(w.num_pages)  # new position of old page j is perm[j]
    kc = np.empty_like(w.k_cache)
    vc = np.empty_like(w.v_cache)
    ks = np.empty_like(w.k_scale)
    vs = np.empty_like(w.v_scale)
    kc[perm] = w.k_cache
    vc[perm] = w.v_cache
    ks[perm] = w.k_scale
    vs[perm] = w.v_scale
    w2 = w.with_(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs,
                 block_table=perm[w.block_table].astype(np.int32))
    assert_close(orc.decode(w2), orc.decode(w), rtol=0, atol=0, what="relocation")


def pin_empty(orc):
    """Empty contexts and rows before the context give zeros, sink or not."""
    w = small(27, QL=3, lens=(0, 1, 2), sinks=True)
    out = orc.decode(w)
    assert np.all(out[0:3] == 0)  # L = 0
    assert np.all(out[3:5] == 0)  # L = 1, rows i = 0, 1 have p < 0
    assert np.all(out[6] == 0)  # L = 2, row 0 has p = -1
    assert np.all(np.isfinite(out))
    assert np.any(out[5] != 0) and np.any(out[8] != 0)
    w0 = w.with_(sinks=None)
    assert np.all(orc.decode(w0)[0:3] == 0)


def pin_merge_any_split(orc):
    """Partials over any split of the visible set, merged in any order, equal
    the unsplit result; empty partials change nothing."""
    w = small(28, lens=(90,), group=2, sinks=True)
    full = orc.decode(w)
    rng = np.random.default_rng(3)
    for h in range(2):
        tokens = np.arange(90)
        for trial in range(4):
            cuts = np.sort(rng.choice(np.arange(1, 90), size=trial + 1, replace=False))
            parts = [orc.row_partial(w, 0, 0, h, seg) for seg in np.split(rng.permutation(tokens), cuts)]
            parts.append(orc.row_partial(w, 0, 0, h, []))  # an empty partial
            order = rng.permutation(len(parts))
            merged = orc.merge([parts[k] for k in order], sink=float(w.sinks[h]))
            assert_close(merged, full[0, h], what="merge")
        single = orc.merge([orc.row_partial(w, 0, 0, h, tokens)], sink=float(w.sinks[h]))
        assert_close(single, full[0, h], rtol=1e-14, atol=1e-15, what="single partial")
    assert np.all(orc.merge([orc.row_partial(w, 0, 0, 0, [])]) == 0)


def pin_sparse(orc):
    """Sparse lists: enumerating the whole context equals dense decode;
    indices at or beyond the context are ignored; order does not matter."""
    w = small(29, lens=(37, 64, 5), group=4, scale=pw.SCALE_PER_TOKEN)
    dense = orc.decode(w)
    K = 70
    rng = np.random.default_rng(4)
    idx = np.full((w.batch, K), 0, dtype=np.int32)
    for b in range(w.batch):
        L = int(w.ctx_lens[b])
        junk = rng.integers(L, L + 1000, size=K - L)
        row = np.concatenate([rng.permutation(L), junk])
        idx[b] = rng.permutation(row)
    ws = w.with_(topk=K, topk_idx=idx, causal=0)
    assert_close(orc.decode(ws), dense, rtol=1e-12, atol=1e-14, what="sparse = dense")
    sub = np.sort(rng.choice(37, size=9, replace=False)).astype(np.int32)
    idx2 = np.full((w.batch, 9), 10 ** 6, dtype=np.int32)
    idx2[0] = sub
    w2 = w.with_(topk=9, topk_idx=idx2, causal=0)
    out = orc.decode(w2)
    assert np.all(out[1:] == 0)
    bf = brute_force(w2)
    assert_close(out, bf, what="sparse brute force")


def pin_per_token_uniform(orc):
    """Per-token scales that are all equal to s match a per-tensor scale s."""
    w = small(30, QL=2, lens=(12, 40))
    s_k, s_v = float(w.k_scale[0]), float(w.v_scale[0])
    ks = np.full((w.num_pages, w.num_kv_heads, w.page_size), s_k, dtype=np.float32)
    vs = np.full((w.num_pages, w.num_kv_heads, w.page_size), s_v, dtype=np.float32)
    wt = w.with_(scale_mode=pw.SCALE_PER_TOKEN, k_scale=ks, v_scale=vs)
    assert_close(orc.decode(wt), orc.decode(w), rtol=0, atol=0, what="per-token uniform")


def pin_gqa_heads(orc):
    """Query head h reads KV head h // G: poisoning KV head 1 poisons exactly
    heads G..2G-1."""
    w = small(31, hkv=2, group=3, lens=(20,), kv=pw.KV_BF16)
    kc = w.k_cache.copy()
    kc[:, 1] = pw.BF16_NAN
    out = orc.decode(w.with_(k_cache=kc))
    assert np.all(np.isfinite(out[0, 0:3])) and np.all(np.isnan(out[0, 3:6]))


def pin_poison_unread(orc):
    """Generated workloads poison every entry outside the contexts; the
    oracle's outputs stay finite, so it never reads them."""
    for w in (pw.tiny(), small(32, QL=4, window=3, lens=(0, 1, 15, 16, 17), sinks=True,
                               scale=pw.SCALE_PER_TOKEN)):
        out = orc.decode(w)
        assert np.all(np.isfinite(out)), w.name


# --- indexer-logits pins ------------------------------------------------------------

def _logits_case(w):
    import oracle

    return oracle.LogitsCase(w.q, w.kv, w.kv_scale, w.weights, w.ks, w.ke)


def logits_brute_force(w) -> np.ndarray:
    """Float64 logits from torch's e4m3 casts and NumPy einsums, with an explicit window mask."""
    qf = torch.from_numpy(np.ascontiguousarray(w.q)).view(torch.float8_e4m3fn).double().numpy()
    kf = torch.from_numpy(np.ascontiguousarray(w.kv)).view(torch.float8_e4m3fn).double().numpy()
    s = np.einsum("rhd,jd->rhj", qf, kf) * w.kv_scale.astype(np.float64)[None, None, :]
    out = np.einsum("rh,rhj->rj", w.weights.astype(np.float64), np.maximum(s, 0.0))
    j = np.arange(w.num_kv)[None, :]
    inside = (j >= w.ks[:, None]) & (j < w.ke[:, None])
    return np.where(inside, out, -np.inf)


def pin_logits_brute_force(orc):
    import oracle

    for seed, rows, heads, n, win in [(21, 5, 16, 300, "random"), (22, 7, 32, 260, "chunk"),
                                      (23, 3, 64, 129, "random")]:
        w = pw.indexer(seed=seed, rows=rows, heads=heads, num_kv=n, window=win)
        mine, _ = oracle.mqa_logits_full(orc, _logits_case(w))
        ref = logits_brute_force(w)
        assert np.array_equal(np.isneginf(mine), np.isneginf(ref)), f"window mask differs ({seed})"
        fin = np.isfinite(ref)
        assert_close(mine[fin], ref[fin], rtol=1e-11, atol=1e-9, what=f"logits brute force {seed}")


def pin_logits_closed_forms(orc):
    """One head, weight 1: the logit is max(0, scale * q . k); negative scores
    contribute nothing (ReLU); the window is half-open [ks, ke)."""
    import oracle

    dim = 8
    q = np.zeros((1, 1, dim), dtype=np.uint8)
    q[0, 0, 3] = 0x40  # e4m3 2.0
    kv = np.zeros((4, dim), dtype=np.uint8)
    kv[0, 3] = 0x38   # 1.0   -> 2 * 1 * scale
    kv[1, 3] = 0xB8   # -1.0  -> relu -> 0
    kv[2, 3] = 0x44   # 3.0   -> 6 * scale
    kv[3, 3] = 0x38
    scale = np.array([0.5, 2.0, 0.25, 1.0], dtype=np.float32)
    case = oracle.LogitsCase(q, kv, scale, np.ones((1, 1), np.float32), np.array([0], np.int32),
                             np.array([3], np.int32))
    out, bound = oracle.mqa_logits_full(orc, case)
    assert out[0, 0] == 1.0 and out[0, 1] == 0.0 and out[0, 2] == 1.5, out
    assert np.isneginf(out[0, 3]), "ke is exclusive"
    assert bound[0, 1] == 4.0 and bound[0, 3] == 0.0, bound
    # two heads with weights w1, w2: a weighted sum of the per-head ReLUs
    q2 = np.zeros((1, 2, dim), dtype=np.uint8)
    q2[0, 0, 3] = 0x40   # 2.0
    q2[0, 1, 3] = 0xC0   # -2.0
    case2 = oracle.LogitsCase(q2, kv, np.ones(4, np.float32), np.array([[0.75, -0.5]], np.float32),
                              np.array([0], np.int32), np.array([4], np.int32))
    out2, _ = oracle.mqa_logits_full(orc, case2)
    assert out2[0, 0] == 0.75 * 2.0 and out2[0, 1] == -0.5 * 2.0 and out2[0, 2] == 0.75 * 6.0, out2


ALL_PINS = [
    pin_e4m3_all_codes, pin_e4m3_golden, pin_bf16_widen, pin_f16_widen, pin_bf16_round, pin_brute_force,
    pin_one_token, pin_two_tokens, pin_constant_v, pin_window_one_position, pin_causal_prefix,
    pin_relocation, pin_empty, pin_merge_any_split, pin_sparse, pin_per_token_uniform,
    pin_gqa_heads, pin_poison_unread, pin_logits_brute_force, pin_logits_closed_forms,
    pin_mx_codes, pin_mx_brute_force, pin_mx_constant_v, pin_transposed_v,
]
