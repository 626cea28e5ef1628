"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one of them (CPU only; the shipped oracle is untouched)."""

import os
import tempfile

import pytest

import oracle
from oracle_pins import ALL_PINS

# (what the mistake is, original text, broken text)
MUTANTS = [
    ("causal bound off by one", "if (sh->causal && t > p) continue;",
     "if (sh->causal && t >= p) continue;"),
    ("window bound off by one", "t <= p - sh->window) continue;", "t < p - sh->window) continue;"),
    ("query position reversed", "int p = L - sh->query_len + i;", "int p = L - 1 - i;"),
    ("GQA mapping modulo", "int g = h / G;", "int g = h % sh->num_kv_heads;"),
    ("slot off by one", "kv_element(sh, k_cache, k_scale, page, g, t % sh->page_size, d)",
     "kv_element(sh, k_cache, k_scale, page, g, (t + 1) % sh->page_size, d)"),
    ("block-table row stride", "block_table[(size_t)b * sh->max_pages_per_seq + t / sh->page_size]",
     "block_table[(size_t)b * (sh->max_pages_per_seq - 1) + t / sh->page_size]"),
    ("sm_scale dropped", "x[j] = sh->sm_scale * s;", "x[j] = s;"),
    ("sink dropped", "den = l * a + exp(s - M);", "den = l * a;"),
    ("sink sign", "den = l * a + exp(s - M);", "den = l * a + exp(M - s);"),
    ("e4m3 bias", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("e4m3 subnormal", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    ("per-token scale slot", "v *= (double)((const float*)scale)[row];", "v *= (double)((const float*)scale)[row - slot];"),
    ("V uses K scale", "v_element(sh, v_cache, v_scale,", "v_element(sh, v_cache, k_scale,"),
    ("q operand reversed", "s += q_element(sh, qrow, d) *", "s += q_element(sh, qrow, D - 1 - d) *"),
    ("f16 bias", "ldexp(1024.0 + (double)f, e - 25)", "ldexp(1024.0 + (double)f, e - 24)"),
    ("f16 subnormal", "mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    ("f16 queries read as bf16",
     "return sh->q_dtype == ORACLE_Q_FP16 ? pa_oracle_f16_to_double(qrow[d]) : pa_oracle_bf16_to_double(qrow[d]);",
     "return pa_oracle_bf16_to_double(qrow[d]);"),
    ("sparse context filter", "if (t >= 0 && t < L) tokens[n++] = t;", "if (t >= 0) tokens[n++] = t;"),
    ("merge without rescale", "out[d] += o[(size_t)j * D + d] * a;", "out[d] += o[(size_t)j * D + d];"),
    ("merge without sink", "if (has_sink) L += exp(sink - M);", "if (0) L += exp(sink - M);"),
    ("round ties away", "r = nearbyint(ldexp(a, -qexp));", "r = round(ldexp(a, -qexp));"),
    ("bf16 widen shift", "uint32_t w = (uint32_t)bits << 16;", "uint32_t w = (uint32_t)bits << 15;"),
    ("no empty-row guard", "if (ntok == 0) {", "if (ntok < 0) {"),
    ("exp sign", "double w = exp(x[j] - m);", "double w = exp(m - x[j]);"),
    ("window ignored", "if (sh->window > 0 && t <= p - sh->window) continue;", ""),
    ("logits without ReLU", "acc += w * (s > 0.0 ? s : 0.0);", "acc += w * s;"),
    ("logits window end inclusive", "if (!(j >= ks[r] && j < ke[r])) {", "if (!(j >= ks[r] && j <= ke[r])) {"),
    ("logits scale dropped", "      s *= sc;\n", "      (void)sc;\n"),
    ("logits head weight of the wrong head", "double s = 0.0, a = 0.0, w = (double)weights[(size_t)r * heads + h];",
     "double s = 0.0, a = 0.0, w = (double)weights[(size_t)r * heads + (heads - 1 - h)];"),
    ("mx nibble order", "uint8_t code = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);",
     "uint8_t code = (d & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);"),
    ("mx block of 16 dims", "(size_t)(d / ORACLE_MX_BLOCK)];", "(size_t)(d / 16) % (size_t)(sh->head_dim / ORACLE_MX_BLOCK)];"),
    ("mx scale row stride", "uint8_t x = ((const uint8_t*)scale)[row * (size_t)(sh->head_dim / ORACLE_MX_BLOCK)",
     "uint8_t x = ((const uint8_t*)scale)[(row / 2) * (size_t)(sh->head_dim / ORACLE_MX_BLOCK)"),
    ("e2m1 exponent bias", "ldexp(1.0 + 0.5 * (double)m, e - 1)", "ldexp(1.0 + 0.5 * (double)m, e - 2)"),
    ("e2m1 subnormal", "e == 0 ? 0.5 * (double)m", "e == 0 ? 1.0 * (double)m"),
    ("e8m0 bias", "return ldexp(1.0, (int)code - 127);", "return ldexp(1.0, (int)code - 126);"),
    ("transposed V read as plain", "  if (sh->v_layout == ORACLE_V_TRANSPOSED) {\n    size_t block",
     "  if (0) {\n    size_t block"),
    ("transposed V token in chunk", "* sh->head_dim + d) * ORACLE_V_CHUNK + slot % ORACLE_V_CHUNK;",
     "* sh->head_dim + d) * ORACLE_V_CHUNK + (slot + 1) % ORACLE_V_CHUNK;"),
    ("transposed V dims and tokens swapped",
     "size_t idx = ((block + (size_t)(slot / ORACLE_V_CHUNK)) * sh->head_dim + d)",
     "size_t idx = ((block + (size_t)(slot / ORACLE_V_CHUNK)) * sh->head_dim + (d ^ 1))"),
    ("logits kv row off by one", "pa_oracle_e4m3_to_double(kv[(size_t)j * dim + d]);",
     "pa_oracle_e4m3_to_double(kv[(size_t)(j + 1 < num_kv ? j + 1 : j) * dim + d]);"),
]


def test_mutants_are_well_formed():
    src = open(oracle.SOURCE).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, f"mutation site for '{name}' must occur exactly once"


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new):
    src = open(oracle.SOURCE).read()
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new, 1))
        lib = oracle.build(source=path, out=os.path.join(tmp, "libmutant.so"), force=True)
        mutant = oracle.Oracle(lib)
        caught = []
        for pin in ALL_PINS:
            try:
                pin(mutant)
            except Exception as e:  # AssertionError or an oracle error code
                caught.append((pin.__name__, type(e).__name__))
        assert caught, f"no pin catches the mutant '{name}'"
