"""Seeded synthetic inputs for paged-attention decode.

This module is shared by the CPU oracle's tests, the GPU parity tests and
``bench.py``. It only *generates* inputs: Q rows, paged K/V caches (FP8 e4m3
codes or BF16 bits), block tables, context lengths, scales, sink logits and
sparse index lists. It performs none of the attention arithmetic (no
dequantisation, no scores, no softmax) so that neither implementation under
test borrows anything from the other through it.

Workloads follow the shapes the reference pages measure:

* "tiny": batch 2, 1 KV head, GQA8, D128, page 16, contexts {37, 100}, one
  random permutation of a 16-page pool (PR "Add paged-attention Tile kernel",
  the FP8 per-tensor decode path).
* "dense": batch 64, 8 KV heads, GQA8, D128, page 16, contexts uniform in
  [1024, 8192], pages dealt from one permutation of a 40,000-page pool.
* "d256": batch 16, 2 KV heads, GQA8, D256, page 64, contexts {8K, 128K} plus
  ragged tails and one empty sequence, per-token FP8 scales (PR "Extend packed
  D256 PA decode pipe to page16, transposed V and sliding windows", Validation).
* "sparse": 64 rows, 16 query heads, 1 KV head, D128, page 16, 2048 sorted
  top-k indices per row out of a 131072-token context, block tables into a
  4096-page pool (PR "Merge gfx1250 PA decode partitions in the tile kernel and
  speed up dense decode", Performance).
* "mtp4": batch 32, 4 KV heads, GQA16, D128, QL4 causal, page 128, contexts
  uniform in [4096, 65536] (same PR, "Dense tile kernels": MTP4 at GQA16).
* "sparse_prefill": 1024 (or 8192) prompt rows, 16 query heads, 1 KV head,
  D128, page 16, row r attends to min(r + 1, 2048) of the prompt's first r + 1
  tokens (same PR, Performance: the sparse prefill rows).

Cache layout is ``[num_pages, num_kv_heads, page_size, head_dim]`` (bytes for
FP8, BF16 bit patterns for BF16; MXFP4: ``head_dim / 2`` bytes per row, two
E2M1 codes per byte, the even element in the low nibble, with E8M0 scale bytes
``[num_pages, num_kv_heads, page_size, head_dim / 32]``). Every pool page that
no sequence uses, every slot past a sequence's context in its last page and
every block-table entry past a sequence's extent is poisoned with NaN codes
(MXFP4, whose elements have no NaN: NaN scale bytes), so any read of them shows
up in the output. Per-token scale slots past the context are poisoned too.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

KV_FP8 = 0
KV_BF16 = 1
KV_MXFP4 = 2
SCALE_NONE = 0
SCALE_PER_TENSOR = 1
SCALE_PER_TOKEN = 2
SCALE_MX_BLOCK = 3
MX_BLOCK = 32
Q_BF16 = 0
Q_FP16 = 1
V_PLAIN = 0
V_TRANSPOSED = 1  # BF16 V as [num_pages, num_kv_heads, page_size / 8, head_dim, 8]
V_CHUNK = 8

FP8_MAX = 448.0
FP8_NAN = 0x7F
BF16_NAN = 0x7FC0
E8M0_NAN = 0xFF
# magnitudes of the eight non-negative E2M1 codes, in code order
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


@dataclasses.dataclass
class Workload:
    """One seeded input set. Arrays are host (numpy) arrays."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    query_len: int
    page_size: int
    num_pages: int
    max_pages_per_seq: int
    kv_dtype: int
    scale_mode: int
    q: np.ndarray  # uint16 [B*QL, Hq, D] BF16 or FP16 bits (q_dtype)
    k_cache: np.ndarray  # uint8 [P, Hkv, S, D] codes (MXFP4: [.., D/2] packed), or uint16 BF16 bits
    v_cache: np.ndarray
    block_table: np.ndarray  # int32 [B, max_pages_per_seq]
    ctx_lens: np.ndarray  # int32 [B]
    k_scale: Optional[np.ndarray]  # float32 [1] or [P, Hkv, S]; MXFP4: uint8 E8M0 [P, Hkv, S, D/32]
    v_scale: Optional[np.ndarray]
    causal: int = 1
    window: int = 0
    sinks: Optional[np.ndarray] = None  # float32 [Hq]
    topk: int = 0
    topk_idx: Optional[np.ndarray] = None  # int32 [B, topk]
    seed: int = 0
    q_dtype: int = Q_BF16  # element type of q and of the output
    v_layout: int = V_PLAIN  # V cache layout (V_TRANSPOSED: BF16 only)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def row_bytes(self) -> int:
        """Bytes of one K (or V) token row, block scales included."""
        if self.kv_dtype == KV_MXFP4:
            return self.head_dim // 2 + self.head_dim // MX_BLOCK
        return self.head_dim * (1 if self.kv_dtype == KV_FP8 else 2)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE binary16 (torch's RNE cast) and return the bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)


def q_bits(x: np.ndarray, q_dtype: int) -> np.ndarray:
    return f16_bits(x) if q_dtype == Q_FP16 else bf16_bits(x)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (torch's RNE cast) and return the bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def fp8_codes(x: np.ndarray) -> np.ndarray:
    """Encode float32 values as OCP e4m3fn codes (torch's RNE cast, saturated)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.clamp_(-FP8_MAX, FP8_MAX)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def mxfp4_encode(x: np.ndarray):
    """Encode float32 rows (last axis a multiple of 32) as MXFP4.

    Per block of 32 values: shared exponent X = floor(log2(amax)) - 2 + 127
    (the largest E2M1 exponent is 2), clamped to [0, 254] (127 for an all-zero
    block); elements = the nearest E2M1 value of v / 2^(X - 127), ties to the
    even code, saturated at +-6. Returns (packed codes [..., D/2] uint8 with the
    even element in the low nibble, E8M0 scales [..., D/32] uint8).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    D = x.shape[-1]
    blk = x.reshape(x.shape[:-1] + (D // MX_BLOCK, MX_BLOCK))
    amax = np.abs(blk).max(axis=-1)
    with np.errstate(divide="ignore"):
        ex = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2.0, 0.0)
    X = np.clip(ex + 127.0, 0, 254).astype(np.int32)
    scaled = blk / np.exp2((X - 127).astype(np.float32))[..., None]
    mag = np.abs(scaled)
    dist = np.abs(mag[..., None] - E2M1_GRID)  # [..., 32, 8]
    dist -= 1e-6 * (np.arange(8) % 2 == 0)  # ties go to the even code
    code = np.argmin(dist, axis=-1).astype(np.uint8)
    code |= np.where((scaled < 0) & (code != 0), 8, 0).astype(np.uint8)
    code = code.reshape(x.shape[:-1] + (D,))
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, X.astype(np.uint8)


def transpose_v(v_cache: np.ndarray) -> np.ndarray:
    """A plain [P, Hkv, S, D] BF16 V cache rearranged into the transposed
    layout [P, Hkv, S/8, D, 8] (chunks of 8 tokens per head dim; the same
    values, moved)."""
    P, H, S, D = v_cache.shape
    return np.ascontiguousarray(v_cache.reshape(P, H, S // V_CHUNK, V_CHUNK, D).transpose(0, 1, 2, 4, 3))


def _pool_and_table(rng, ctx_lens, page_size, pool_pages, max_pages):
    """Deal one random permutation of the pool to the sequences in order.

    Returns (block_table, used_pages, poison_page). Entries past a sequence's
    extent point at a page no sequence uses.
    """
    need = [(int(L) + page_size - 1) // page_size for L in ctx_lens]
    total = sum(need)
    if total + 1 > pool_pages:
        raise ValueError("page pool too small")
    perm = rng.permutation(pool_pages).astype(np.int32)
    poison_page = int(perm[-1])
    table = np.full((len(ctx_lens), max_pages), poison_page, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[pos : pos + n]
        pos += n
    used = perm[:total]
    return table, used, poison_page


def _fill_cache(rng, num_pages, hkv, S, D, used_pages, valid_slots, kv_dtype,
                scale_mode, amplitude=1.0, vfun=None, token_sigma=0.0):
    """Generate one paged cache (K or V) plus its scales.

    ``valid_slots[p]`` = number of leading valid slots of physical page p
    (0 for unused pages). Invalid slots are NaN-poisoned. ``token_sigma`` > 0
    multiplies each token's row by e^(token_sigma * N(0,1)), so token
    magnitudes vary (the pages' check that catches a misplaced scale).
    """
    elt = 1 if kv_dtype == KV_FP8 else 2
    shape = (num_pages, hkv, S, D)
    n_used = len(used_pages)
    vals = rng.standard_normal((n_used, hkv, S, D), dtype=np.float32)
    if amplitude != 1.0:
        vals *= np.float32(amplitude)
    if token_sigma > 0:
        vals *= np.exp(np.float32(token_sigma) * rng.standard_normal((n_used, hkv, S, 1), dtype=np.float32))
    if vfun is not None:
        vals = vfun(used_pages, vals)
    slot_ok = np.arange(S)[None, :] < valid_slots[used_pages][:, None]  # [n_used, S]
    mask4 = np.broadcast_to(slot_ok[:, None, :, None], vals.shape)
    scale = None
    if kv_dtype == KV_MXFP4:
        packed, X = mxfp4_encode(vals)
        cache = np.full((num_pages, hkv, S, D // 2), 0x77, dtype=np.uint8)
        cache[used_pages] = packed
        scale = np.full((num_pages, hkv, S, D // MX_BLOCK), E8M0_NAN, dtype=np.uint8)
        X[~np.broadcast_to(slot_ok[:, None, :, None], X.shape)] = E8M0_NAN
        scale[used_pages] = X
        return cache, scale
    if kv_dtype == KV_BF16:
        cache = np.full(shape, BF16_NAN, dtype=np.uint16)
        bits = bf16_bits(vals)
        bits[~mask4] = BF16_NAN
        cache[used_pages] = bits
        return cache, None
    cache = np.full(shape, FP8_NAN, dtype=np.uint8)
    if scale_mode == SCALE_PER_TENSOR:
        amax = float(np.abs(vals[mask4]).max()) if mask4.any() else 0.0
        s = amax / FP8_MAX if amax > 0 else 1.0
        scale = np.array([s], dtype=np.float32)
        codes = fp8_codes(vals / np.float32(scale[0]))
    elif scale_mode == SCALE_PER_TOKEN:
        amax = np.abs(vals).max(axis=3)  # [n_used, hkv, S]
        tok = np.where(amax > 0, amax / FP8_MAX, 1.0).astype(np.float32)
        codes = fp8_codes(vals / tok[..., None])
        scale = np.full((num_pages, hkv, S), np.nan, dtype=np.float32)
        tok_ok = np.broadcast_to(slot_ok[:, None, :], tok.shape)
        scale[used_pages] = np.where(tok_ok, tok, np.float32(np.nan))
    else:
        codes = fp8_codes(vals)
    codes[~mask4] = FP8_NAN
    cache[used_pages] = codes
    return cache, scale


def make_dense(name, *, batch, hkv, group, head_dim, query_len, page_size,
               ctx_lens, kv_dtype, scale_mode, seed, pool_pages=None,
               causal=1, window=0, with_sinks=False, max_pages=None,
               v_amplitude=1.0, vfun=None, q_amplitude=1.0, token_sigma=0.0, q_dtype=Q_BF16,
               v_layout=V_PLAIN):
    """Build a dense paged-decode workload with the given context lengths.

    ``q_amplitude`` scales the N(0,1) query values before rounding to the
    query type ``q_dtype`` (BF16 or FP16; large logits); ``token_sigma`` > 0
    varies K and V token magnitudes by e^(token_sigma * N(0,1));
    ``v_amplitude`` scales V."""
    rng = np.random.default_rng(seed)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
    need = (ctx_lens.astype(np.int64) + page_size - 1) // page_size
    if max_pages is None:
        max_pages = max(1, int(need.max()))
    if pool_pages is None:
        pool_pages = int(need.sum()) + 8
    table, used, _ = _pool_and_table(rng, ctx_lens, page_size, pool_pages, max_pages)
    valid = np.zeros(pool_pages, dtype=np.int64)
    for b in range(batch):
        L = int(ctx_lens[b])
        for j in range(int(need[b])):
            valid[table[b, j]] = min(page_size, L - j * page_size)
    hq = hkv * group
    qv = rng.standard_normal((batch * query_len, hq, head_dim), dtype=np.float32)
    if q_amplitude != 1.0:
        qv *= np.float32(q_amplitude)
    q = q_bits(qv, q_dtype)
    kc, ks = _fill_cache(rng, pool_pages, hkv, page_size, head_dim, used, valid,
                         kv_dtype, scale_mode, token_sigma=token_sigma)
    vc, vs = _fill_cache(rng, pool_pages, hkv, page_size, head_dim, used, valid,
                         kv_dtype, scale_mode, amplitude=v_amplitude, vfun=vfun,
                         token_sigma=token_sigma)
    sinks = rng.standard_normal(hq, dtype=np.float32) if with_sinks else None
    if kv_dtype == KV_BF16:
        scale_mode = SCALE_NONE
    if v_layout == V_TRANSPOSED:
        vc = transpose_v(vc)
    return Workload(name=name, batch=batch, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=head_dim, query_len=query_len, page_size=page_size,
                    num_pages=pool_pages, max_pages_per_seq=max_pages,
                    kv_dtype=kv_dtype, scale_mode=scale_mode, q=q, k_cache=kc,
                    v_cache=vc, block_table=table, ctx_lens=ctx_lens, k_scale=ks,
                    v_scale=vs, causal=causal, window=window, sinks=sinks,
                    seed=seed, q_dtype=q_dtype, v_layout=v_layout)


# --- the five workloads -----------------------------------------------------

def tiny(seed: int = 1001) -> Workload:
    """Batch 2, GQA8, D128, page 16, contexts {37, 100}, 16-page pool, FP8 per tensor."""
    return make_dense("tiny", batch=2, hkv=1, group=8, head_dim=128, query_len=1,
                      page_size=16, ctx_lens=[37, 100], kv_dtype=KV_FP8,
                      scale_mode=SCALE_PER_TENSOR, seed=seed, pool_pages=16)


def dense_lengths(seed: int, batch: int = 64, lo: int = 1024, hi: int = 8192):
    rng = np.random.default_rng(seed + 7)
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def dense(seed: int = 1002, batch: int = 64, lo: int = 1024, hi: int = 8192,
          kv_dtype: int = KV_FP8, page_size: int = 16, v_layout: int = V_PLAIN) -> Workload:
    """Batch 64, 8 KV heads, GQA8, D128, page 16, contexts U[1024, 8192], 40k-page pool
    (page_size other than 16 keeps the pool's bytes: 40000 * 16 / page_size pages)."""
    lens = dense_lengths(seed, batch, lo, hi)
    pool = 40000 * 16 // page_size
    return make_dense("dense", batch=batch, hkv=8, group=8, head_dim=128,
                      query_len=1, page_size=page_size, ctx_lens=lens, kv_dtype=kv_dtype,
                      scale_mode=SCALE_MX_BLOCK if kv_dtype == KV_MXFP4 else SCALE_PER_TENSOR, seed=seed,
                      pool_pages=max(pool, int(((lens + page_size - 1) // page_size).sum()) + 8),
                      max_pages=hi // page_size, v_layout=v_layout)


def d256_lengths(seed: int, batch: int = 16, short: int = 8192, long: int = 131072):
    rng = np.random.default_rng(seed + 11)
    lens = np.zeros(batch, dtype=np.int32)
    for b in range(1, batch):
        base = short if b % 2 == 1 else long
        tail = 0 if b in (1, 2) else int(rng.integers(1, 64))
        lens[b] = base + tail
    return lens


def d256(seed: int = 1003, query_len: int = 1, window: int = 0,
         with_sinks: bool = False, batch: int = 16, short: int = 8192,
         long: int = 131072) -> Workload:
    """Batch 16, 2 KV heads, GQA8, D256, page 64, per-token FP8, {8K,128K}+tails, one empty."""
    lens = d256_lengths(seed, batch, short, long)
    return make_dense("d256", batch=batch, hkv=2, group=8, head_dim=256,
                      query_len=query_len, page_size=64, ctx_lens=lens,
                      kv_dtype=KV_FP8, scale_mode=SCALE_PER_TOKEN, seed=seed,
                      causal=1, window=window, with_sinks=with_sinks)


def mtp4_lengths(seed: int, batch: int = 32, lo: int = 4096, hi: int = 65536):
    rng = np.random.default_rng(seed + 13)
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def mtp4(seed: int = 1005, kv_dtype: int = KV_FP8, batch: int = 32,
         lo: int = 4096, hi: int = 65536, v_layout: int = V_PLAIN) -> Workload:
    """Batch 32, 4 KV heads, GQA16, D128, QL4 causal, page 128, contexts U[4096, 65536]."""
    lens = mtp4_lengths(seed, batch, lo, hi)
    return make_dense("mtp4", batch=batch, hkv=4, group=16, head_dim=128,
                      query_len=4, page_size=128, ctx_lens=lens, kv_dtype=kv_dtype,
                      scale_mode=SCALE_MX_BLOCK if kv_dtype == KV_MXFP4 else SCALE_PER_TENSOR, seed=seed, causal=1,
                      max_pages=(hi + 127) // 128, v_layout=v_layout)


def sparse(seed: int = 1004, kv_dtype: int = KV_FP8, rows: int = 64,
           topk: int = 2048, context: int = 131072, pool_pages: int = 4096,
           page_size: int = 16, head_dim: int = 128, group: int = 16,
           q_dtype: int = Q_BF16) -> Workload:
    """64 rows (QL1), 16 query heads, 1 KV head, D128, page 16, top-2048 of 131072."""
    rng = np.random.default_rng(seed)
    hkv = 1
    max_pages = context // page_size
    # Block tables map logical pages into a small shared pool (aliasing allowed),
    # as in a pool of 4096 physical page16 pages.
    table = rng.integers(0, pool_pages, size=(rows, max_pages), dtype=np.int64).astype(np.int32)
    ctx = np.full(rows, context, dtype=np.int32)
    idx = np.empty((rows, topk), dtype=np.int32)
    for r in range(rows):
        idx[r] = np.sort(rng.choice(context, size=topk, replace=False)).astype(np.int32)
    used = np.arange(pool_pages)
    valid = np.full(pool_pages, page_size, dtype=np.int64)
    hq = hkv * group
    q = q_bits(rng.standard_normal((rows, hq, head_dim), dtype=np.float32), q_dtype)
    smode = SCALE_PER_TENSOR if kv_dtype == KV_FP8 else SCALE_NONE
    kc, ks = _fill_cache(rng, pool_pages, hkv, page_size, head_dim, used, valid, kv_dtype, smode)
    vc, vs = _fill_cache(rng, pool_pages, hkv, page_size, head_dim, used, valid, kv_dtype, smode)
    return Workload(name="sparse", batch=rows, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=head_dim, query_len=1, page_size=page_size,
                    num_pages=pool_pages, max_pages_per_seq=max_pages,
                    kv_dtype=kv_dtype, scale_mode=smode, q=q, k_cache=kc,
                    v_cache=vc, block_table=table, ctx_lens=ctx, k_scale=ks,
                    v_scale=vs, causal=0, window=0, sinks=None, topk=topk,
                    topk_idx=idx, seed=seed, q_dtype=q_dtype)


def sparse_prefill(seed: int = 1006, kv_dtype: int = KV_FP8, rows: int = 1024,
                   topk: int = 2048, pool_pages: int = 4096, page_size: int = 16,
                   head_dim: int = 128, group: int = 16) -> Workload:
    """Sparse prefill: one prompt of ``rows`` tokens, each query row r its own
    decode row (query length 1) whose context is the prompt's first r + 1
    tokens; row r lists min(r + 1, topk) token indices out of [0, r] (all of
    them while r < topk, else a sorted sample without replacement), the rest
    of its index row is -1. The prompt's pages come from one random
    permutation of a ``pool_pages`` page16 pool and every row shares its block
    table (PR "Merge gfx1250 PA decode partitions in the tile kernel and speed
    up dense decode", Performance: prefill rows see min(row + 1, 2048) tokens)."""
    rng = np.random.default_rng(seed)
    hkv = 1
    n_pages = (rows + page_size - 1) // page_size
    if n_pages + 1 > pool_pages:
        raise ValueError("page pool too small")
    perm = rng.permutation(pool_pages).astype(np.int32)
    pages = perm[:n_pages]
    table = np.broadcast_to(pages, (rows, n_pages)).copy()
    ctx = np.arange(1, rows + 1, dtype=np.int32)
    idx = np.full((rows, topk), -1, dtype=np.int32)
    for r in range(rows):
        n = min(r + 1, topk)
        if n == r + 1:
            idx[r, :n] = np.arange(n, dtype=np.int32)
        else:
            idx[r, :n] = np.sort(rng.choice(r + 1, size=n, replace=False)).astype(np.int32)
    valid = np.zeros(pool_pages, dtype=np.int64)
    for j, pg in enumerate(pages):
        valid[pg] = min(page_size, rows - j * page_size)
    hq = hkv * group
    q = bf16_bits(rng.standard_normal((rows, hq, head_dim), dtype=np.float32))
    smode = SCALE_PER_TENSOR if kv_dtype == KV_FP8 else SCALE_NONE
    kc, ks = _fill_cache(rng, pool_pages, hkv, page_size, head_dim, pages, valid, kv_dtype, smode)
    vc, vs = _fill_cache(rng, pool_pages, hkv, page_size, head_dim, pages, valid, kv_dtype, smode)
    return Workload(name="sparse_prefill", batch=rows, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=head_dim, query_len=1, page_size=page_size,
                    num_pages=pool_pages, max_pages_per_seq=n_pages,
                    kv_dtype=kv_dtype, scale_mode=smode, q=q, k_cache=kc,
                    v_cache=vc, block_table=table, ctx_lens=ctx, k_scale=ks,
                    v_scale=vs, causal=0, window=0, sinks=None, topk=topk,
                    topk_idx=idx, seed=seed)


def small_sparse(seed: int = 2004, kv_dtype: int = KV_FP8, rows: int = 3,
                 topk: int = 200, context: int = 1000, pool_pages: int = 40,
                 group: int = 16, head_dim: int = 128, q_dtype: int = Q_BF16) -> Workload:
    """A few sparse rows small enough for per-element oracle parity."""
    w = sparse(seed=seed, kv_dtype=kv_dtype, rows=rows, topk=topk,
               context=context + (-context) % 16, pool_pages=pool_pages,
               group=group, head_dim=head_dim, q_dtype=q_dtype)
    ctx = np.asarray([context, context // 2, 0][:rows] + [context] * max(0, rows - 3),
                     dtype=np.int32)
    return w.with_(ctx_lens=ctx)


def algorithmic_bytes(w: Workload, visible_tokens: Optional[np.ndarray] = None) -> int:
    """Bytes the method must move once per call.

    K and V of visible tokens, their per-token scales, the block-table entries
    of the pages read, context lengths, Q and the BF16 output (and sinks,
    sparse indices). ``visible_tokens[b, i]`` is the visible count of query
    row i of sequence b; the union over rows is what is read once.
    """
    B, QL, hkv, D = w.batch, w.query_len, w.num_kv_heads, w.head_dim
    row = w.row_bytes  # one K or V token row (MXFP4: with its block scales)
    total = 0
    if w.topk:
        L = w.ctx_lens.astype(np.int64)
        n_tok = int(((w.topk_idx >= 0) & (w.topk_idx < L[:, None])).sum())
        total += n_tok * hkv * row * 2
        if w.scale_mode == SCALE_PER_TOKEN:
            total += n_tok * hkv * 4 * 2
        total += n_tok * 4 * 2  # index + block-table entry per gathered token
    else:
        L = w.ctx_lens.astype(np.int64)
        lo = np.zeros_like(L)
        if w.window > 0:
            lo = np.maximum(0, L - QL + 1 - w.window)
        n_tok = np.maximum(0, L - lo)
        total += int(n_tok.sum()) * hkv * row * 2
        if w.scale_mode == SCALE_PER_TOKEN:
            total += int(n_tok.sum()) * hkv * 4 * 2
        S = w.page_size
        pages = np.where(n_tok > 0, (L + S - 1) // S - lo // S, 0)
        total += int(pages.sum()) * 4
    total += B * 4
    total += 2 * B * QL * w.num_q_heads * D * 2
    if w.sinks is not None:
        total += w.num_q_heads * 4
    return int(total)


# --- indexer logits ------------------------------------------------------------

@dataclasses.dataclass
class LogitsWorkload:
    """Inputs of the indexer-logits op (host arrays)."""

    name: str
    q: np.ndarray         # uint8 e4m3 [rows, heads, dim]
    kv: np.ndarray        # uint8 e4m3 [num_kv, dim]
    kv_scale: np.ndarray  # float32 [num_kv]
    weights: np.ndarray   # float32 [rows, heads]
    ks: np.ndarray        # int32 [rows] window start
    ke: np.ndarray        # int32 [rows] window end (exclusive)
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.q.shape[0]

    @property
    def heads(self) -> int:
        return self.q.shape[1]

    @property
    def num_kv(self) -> int:
        return self.kv.shape[0]

    def window_tokens(self) -> int:
        a = np.clip(self.ks.astype(np.int64), 0, self.num_kv)
        e = np.clip(self.ke.astype(np.int64), 0, self.num_kv)
        return int(np.maximum(0, e - a).sum())

    def flops(self) -> int:
        """Multiply-adds of the scores inside the windows, 2 FLOPs each."""
        return 2 * self.window_tokens() * self.heads * self.q.shape[2]


def indexer(seed: int = 1007, rows: int = 1024, heads: int = 64, num_kv: int = 131072, dim: int = 128,
            window: str = "chunk") -> LogitsWorkload:
    """Indexer logits over a prompt chunk: `rows` query rows, `heads` heads,
    FP8 queries and an FP8 KV list of `num_kv` tokens with per-token scales.
    window "chunk": the chunk's rows are the last `rows` positions of the KV
    list (a cached prefix before them), row r sees [0, num_kv - rows + r + 1);
    "random": each row sees a random interval (empty ones included)."""
    rng = np.random.default_rng(seed)
    qv = rng.standard_normal((rows, heads, dim), dtype=np.float32)
    q = fp8_codes(qv)
    kvv = rng.standard_normal((num_kv, dim), dtype=np.float32)
    amax = np.abs(kvv).max(axis=1)
    scale = np.where(amax > 0, amax / FP8_MAX, 1.0).astype(np.float32)
    kv = fp8_codes(kvv / scale[:, None])
    weights = (rng.standard_normal((rows, heads), dtype=np.float32) / np.sqrt(heads)).astype(np.float32)
    if window == "chunk":
        ks = np.zeros(rows, dtype=np.int32)
        ke = (num_kv - rows + np.arange(rows) + 1).clip(0, num_kv).astype(np.int32)
    elif window == "random":
        a = rng.integers(-5, num_kv, size=rows)
        b = a + rng.integers(-3, num_kv // 2 + 3, size=rows)
        ks = a.astype(np.int32)
        ke = b.clip(-10, num_kv + 10).astype(np.int32)
    else:
        raise ValueError(window)
    return LogitsWorkload(name=f"indexer-{window}", q=q, kv=kv, kv_scale=scale, weights=weights, ks=ks, ke=ke,
                          seed=seed)
