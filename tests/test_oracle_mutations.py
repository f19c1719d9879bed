"""Plant one plausible mistake at a time in a copy of the oracle's C source and
check that the pin suite catches it. The mistakes are planted in the oracle, on
the CPU, never in the CUDA path."""
import inspect
import json
import os

import pytest

import oracle
import test_oracle_pins as pins
from conftest import f32_to_bf16_bits

MUTATIONS = {
    "ties_to_higher_index": ("if (best < 0 || zf[e] > zf[best]) best = e;",
                             "if (best < 0 || zf[e] >= zf[best]) best = e;"),
    "ascending_selection": ("if (best < 0 || zf[e] > zf[best]) best = e;",
                            "if (best < 0 || zf[e] < zf[best]) best = e;"),
    "bias_dropped_from_selection": ("s32 = s32 + c->bias[e];", "s32 = s32;"),
    "gate_softmax_sign": ("num[j] = exp(zd[it[j]] - zmax);", "num[j] = exp(zmax - zd[it[j]]);"),
    "silu_on_up_projection": ("hv[f] = sa * (1.0 / (1.0 + exp(-sa))) * sb;",
                              "hv[f] = sb * (1.0 / (1.0 + exp(-sb))) * sa;"),
    "sigmoid_sign": ("hv[f] = sa * (1.0 / (1.0 + exp(-sa))) * sb;",
                     "hv[f] = sa * (1.0 / (1.0 + exp(sa))) * sb;"),
    "w2_transposed": ("for (int f = 0; f < F; ++f) s += hv[f] * bf(w[f]);",
                      "for (int f = 0; f < F; ++f) s += hv[f] * bf(W2[(size_t)f * d + o]);"),
    "w1_w3_swapped": ("const uint16_t *g = W1 + (size_t)f * d, *u = W3 + (size_t)f * d;",
                      "const uint16_t *g = W3 + (size_t)f * d, *u = W1 + (size_t)f * d;"),
    "dispatch_unstable": ("for (long t = 0; t < T; ++t) {\n        for (int j = 0; j < k; ++j) {\n            long s = t * k + j;",
                          "for (long t = T - 1; t >= 0; --t) {\n        for (int j = 0; j < k; ++j) {\n            long s = t * k + j;"),
    "combine_gate_reversed": ("const double g = gate[t * k + j];",
                              "const double g = gate[t * k + (k - 1 - j)];"),
    "layer_gate_reversed": ("const double g = c->gate[t * k + j];",
                            "const double g = c->gate[t * k + (k - 1 - j)];"),
    "dropped_last_feature": ("for (int i = 0; i < d; ++i) {\n            double xi = bf(xr[i]);",
                             "for (int i = 0; i < d - 1; ++i) {\n            double xi = bf(xr[i]);"),
}


def _hand():
    with open(pins.GOLDEN) as f:
        g = json.load(f)
    for key, src in (("xb", "x"), ("wrb", "w_router"), ("w1b", "W1"), ("w3b", "W3"), ("w2b", "W2")):
        g[key] = f32_to_bf16_bits(g[src])
    return g


def _run_pin_suite():
    """Run every pin in test_oracle_pins; return the names of those that fail."""
    failed = []
    hand = _hand()
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        calls = []
        if "hand" in params:
            calls.append({"hand": hand})
        elif "T" in params:
            calls += [dict(T=7, k=3, E=5), dict(T=300, k=6, E=64)]
        else:
            calls.append({})
        for kw in calls:
            try:
                fn(**kw)
            except (AssertionError, ValueError):
                failed.append(name)
                break
    return failed


def test_unmutated_source_passes_every_pin():
    assert _run_pin_suite() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation site for {name} no longer in the oracle source"
    lib = oracle.compile_variant(src.replace(old, new, 1), str(tmp_path / f"mut_{name}.so"))
    with oracle.use_library(lib):
        failed = _run_pin_suite()
    assert failed, f"planted mistake {name} was not caught by any pin"
