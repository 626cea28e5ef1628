"""GPU parity of the indexer-logits kernel against the CPU oracle: every
element on small seeded cases (each head count, ragged row blocks and KV
tiles, random and chunked-prefill windows, clean_logits on and off), and
sampled elements of the long-context chunk shape."""

import numpy as np
import pytest

import oracle
import paged_attention_decode_attn_gb300 as pa
import pa_workloads as pw

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import record_margin  # noqa: E402

# Tolerance derived from the arithmetic: the e4m3 products are exact, the
# kernel sums 128 of them per head in the tensor core's FP32 accumulator and
# then 16-128 weighted ReLUs in FP32, so its error is a few hundred FP32
# roundings of terms bounded by B = sum_h |w| |scale| sum_d |q k| (the
# oracle's `bound`): (D + H) 2^-24 B < 2^-16 B. 2^-12 B leaves 16x for the
# accumulator's internal rounding order.
TOL = 2.0 ** -12


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_attention_decode_attn_gb300 import _build

    _build.build()


def run(w, clean=True, stride=None, fill=None, as_f64=True):
    dev = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    stride = stride or (w.num_kv + 3) // 4 * 4
    logits = torch.full((w.rows, stride), float("nan") if fill is None else fill, dtype=torch.float32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    pa.pa_mqa_logits(logits, t(w.q), t(w.kv), t(w.kv_scale), t(w.weights), t(w.ks), t(w.ke), clean_logits=clean,
                     status=status)
    torch.cuda.synchronize()
    assert int(status[0].item()) == 0
    out = logits.cpu().numpy()
    return out.astype(np.float64) if as_f64 else out


def check(gpu, ref, bound, what):
    inside = np.isfinite(ref)
    assert np.array_equal(np.isneginf(gpu), np.isneginf(ref)), f"{what}: -inf pattern differs"
    assert np.all(np.isfinite(gpu[inside])), f"{what}: non-finite inside the windows"
    ratio = float(np.max(np.abs(gpu[inside] - ref[inside]) / (TOL * bound[inside] + 1e-30))) if inside.any() else 0.0
    record_margin(ratio, what)
    assert ratio <= 1.0, f"{what}: worst |err| / tol = {ratio:.3f}"


@pytest.mark.parametrize("heads", [16, 32, 64, 128])
@pytest.mark.parametrize("window", ["random", "chunk"])
def test_logits_small(orc, heads, window):
    w = pw.indexer(seed=31 + heads, rows=37, heads=heads, num_kv=1111, window=window)
    ref, bound = oracle.mqa_logits_full(orc, oracle.LogitsCase(w.q, w.kv, w.kv_scale, w.weights, w.ks, w.ke))
    gpu = run(w)
    check(gpu[:, : w.num_kv], ref, bound, f"logits H{heads} {window}")


def test_logits_no_clean_leaves_outside_untouched(orc):
    w = pw.indexer(seed=41, rows=9, heads=64, num_kv=700, window="random")
    ref, bound = oracle.mqa_logits_full(orc, oracle.LogitsCase(w.q, w.kv, w.kv_scale, w.weights, w.ks, w.ke))
    gpu = run(w, clean=False, stride=1024, fill=12345.0)
    inside = np.isfinite(ref)
    assert np.all(gpu[:, : w.num_kv][~inside] == 12345.0)
    assert np.all(gpu[:, w.num_kv:] == 12345.0)  # the row padding past num_kv is never written
    ref2 = np.where(inside, ref, -np.inf)
    gpu2 = np.where(inside, gpu[:, : w.num_kv], -np.inf)
    check(gpu2, ref2, bound, "logits no clean")


def test_logits_empty_windows(orc):
    w = pw.indexer(seed=42, rows=5, heads=32, num_kv=300, window="chunk")
    w.ks[:] = 10
    w.ke[:] = 10  # every window empty
    gpu = run(w)
    assert np.all(np.isneginf(gpu[:, : w.num_kv]))


def test_logits_long_chunk_sampled(orc):
    """The long-context chunk shape (1024 rows x 128K KV tokens, 64 heads) on
    20000 sampled elements, plus every -inf outside the windows."""
    w = pw.indexer()
    gpu = run(w, as_f64=False)
    rng = np.random.default_rng(5)
    r = rng.integers(0, w.rows, size=20000)
    j = rng.integers(0, w.num_kv, size=20000)
    j[:2000] = w.ke[r[:2000]] - 1 - rng.integers(0, 200, size=2000)  # near each row's window end
    j = np.clip(j, 0, w.num_kv - 1)
    ref, bound = oracle.mqa_logits(orc, oracle.LogitsCase(w.q, w.kv, w.kv_scale, w.weights, w.ks, w.ke), r, j)
    check(gpu[r, j].astype(np.float64), ref, bound, "logits 1024x128K sampled")
    cols = np.arange(w.num_kv)[None, :]
    outside = cols >= w.ke[:, None]
    assert np.all(np.isneginf(gpu[:, : w.num_kv][outside]))
    assert not np.any(np.isnan(gpu[:, : w.num_kv]))
