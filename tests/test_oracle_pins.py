"""Pins of the fp64 CPU oracle against facts that do not come from the oracle itself:
a hand-worked example solved in closed form, brute force on tiny inputs, exact
integer arithmetic, library routines (numpy matmul / stable argsort / expit),
and the invariants the method fixes (a permutation, gates summing to one,
identity experts reproducing the input)."""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
from conftest import bf16_bits_to_f64, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")


def sigma(v):
    return 1.0 / (1.0 + math.exp(-v))


def _eval(expr):
    return eval(expr, {"__builtins__": {}}, {"sigma": sigma})


@pytest.fixture(scope="module")
def hand():
    with open(GOLDEN) as f:
        g = json.load(f)
    g["xb"] = f32_to_bf16_bits(g["x"])
    g["wrb"] = f32_to_bf16_bits(g["w_router"])
    g["w1b"] = f32_to_bf16_bits(g["W1"])
    g["w3b"] = f32_to_bf16_bits(g["W3"])
    g["w2b"] = f32_to_bf16_bits(g["W2"])
    return g


# ---------------------------------------------------------------- hand example

def test_hand_fixture_is_self_consistent(hand):
    for key in ("gates", "h_by_slot", "out"):
        exprs = hand[key + "_expr"]
        vals = np.array([[_eval(e) for e in row] for row in exprs])
        np.testing.assert_allclose(vals, np.array(hand[key]), atol=1e-9)
    # inputs survive the bf16 round trip exactly
    np.testing.assert_array_equal(bf16_bits_to_f64(hand["xb"]), np.array(hand["x"], float))


def test_hand_route(hand):
    r = oracle.route(hand["xb"], hand["wrb"], None, hand["k"], keep_logits=True)
    np.testing.assert_array_equal(r.z64, np.array(hand["logits"], float))
    np.testing.assert_array_equal(r.z32, np.array(hand["logits"], np.float32))
    np.testing.assert_array_equal(r.idx, np.array(hand["topk_idx"]))
    gates = np.array([[_eval(e) for e in row] for row in hand["gates_expr"]])
    np.testing.assert_allclose(r.gate, gates, rtol=0, atol=1e-15)


def test_hand_dispatch(hand):
    disp = oracle.dispatch(np.array(hand["topk_idx"], np.int32), hand["E"])
    np.testing.assert_array_equal(disp.counts, hand["counts"])
    np.testing.assert_array_equal(disp.offsets, hand["offsets"])
    np.testing.assert_array_equal(disp.slot_of_row, hand["slot_of_row"])
    np.testing.assert_array_equal(disp.row_of_slot, hand["row_of_slot"])


def test_hand_ffn_and_layer(hand):
    T, k, E = hand["T"], hand["k"], hand["E"]
    idx = np.array(hand["topk_idx"], np.int32)
    xin = np.repeat(hand["xb"], k, axis=0)  # slot order: (t, j)
    h, y = oracle.ffn_rows(xin, idx.reshape(-1), hand["w1b"], hand["w3b"], hand["w2b"], E,
                           keep_h=True)
    hexp = np.array([[_eval(e) for e in row] for row in hand["h_by_slot_expr"]]).reshape(-1)
    np.testing.assert_allclose(h[:, 0], hexp, atol=1e-15)
    # y = h W2^T: expert 0 -> (h,0), 1 -> (0,h), 2 -> (h,h)
    w2 = np.array(hand["W2"], float)[:, :, 0]
    np.testing.assert_allclose(y, hexp[:, None] * w2[idx.reshape(-1)], atol=1e-15)
    r = oracle.route(hand["xb"], hand["wrb"], None, k)
    out = oracle.layer_tokens(hand["xb"], r.idx, r.gate, hand["w1b"], hand["w3b"], hand["w2b"],
                              np.arange(T), E)
    oexp = np.array([[_eval(e) for e in row] for row in hand["out_expr"]])
    np.testing.assert_allclose(out, oexp, atol=1e-15)
    np.testing.assert_allclose(out, np.array(hand["out"]), atol=1e-9)
    # the dispatched path (route -> dispatch -> per-row FFN -> combine) gives the same
    disp = oracle.dispatch(r.idx, E)
    xperm = hand["xb"][disp.slot_of_row // k]
    _, yperm = oracle.ffn_rows(xperm, np.repeat(np.arange(E), disp.counts), hand["w1b"],
                               hand["w3b"], hand["w2b"], E)
    np.testing.assert_allclose(oracle.combine(yperm, r.gate, disp.row_of_slot), oexp, atol=1e-15)


# ---------------------------------------------------------------- routing

def _brute_topk(z, k):
    """Exhaustive search: the ordered k-tuple minimising ((-z[e0], e0), (-z[e1], e1), ...)."""
    E = len(z)
    best = min(itertools.permutations(range(E), k), key=lambda tup: [(-z[e], e) for e in tup])
    return list(best)


def test_route_integer_exact_and_brute_force():
    rng = np.random.default_rng(1)
    T, d, E, k = 40, 12, 6, 3
    x = rng.integers(-3, 4, size=(T, d))
    wr = rng.integers(-2, 3, size=(E, d))
    x[5] = 0  # an all-zero token: every logit ties
    r = oracle.route(f32_to_bf16_bits(x), f32_to_bf16_bits(wr), None, k, keep_logits=True)
    zexact = x @ wr.T  # Python-int arithmetic
    np.testing.assert_array_equal(r.z64, zexact)
    np.testing.assert_array_equal(r.z32, zexact.astype(np.float32))
    ties = 0
    for t in range(T):
        assert list(r.idx[t]) == _brute_topk(list(zexact[t]), k)
        combo_best = max(sum(zexact[t][list(c)]) for c in itertools.combinations(range(E), k))
        assert zexact[t][r.idx[t]].sum() == combo_best
        ties += len(set(zexact[t])) < E
    assert ties > 5  # the data really exercises the tie rule
    assert list(r.idx[5]) == [0, 1, 2]


def test_route_bias_integer():
    rng = np.random.default_rng(2)
    T, d, E, k = 30, 8, 5, 2
    x = rng.integers(-2, 3, size=(T, d))
    wr = rng.integers(-2, 3, size=(E, d))
    bias = np.array([0.5, -1.0, 2.0, 0.0, -0.25], np.float32)
    r = oracle.route(f32_to_bf16_bits(x), f32_to_bf16_bits(wr), bias, k, keep_logits=True)
    z = (x @ wr.T).astype(np.float64) + bias
    np.testing.assert_array_equal(r.z64, z)
    for t in range(T):
        assert list(r.idx[t]) == _brute_topk(list(z[t]), k)
        sel = z[t][r.idx[t]]
        np.testing.assert_allclose(r.gate[t], np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum(),
                                   rtol=1e-14)


def test_route_float_logits_vs_library_and_fp32_bound():
    rng = np.random.default_rng(3)
    T, d, E, k = 64, 96, 16, 4
    xb = f32_to_bf16_bits(rng.standard_normal((T, d)))
    wb = f32_to_bf16_bits(rng.standard_normal((E, d)) / math.sqrt(d))
    bias = (rng.standard_normal(E) * 0.3).astype(np.float32)
    r = oracle.route(xb, wb, bias, k, keep_logits=True)
    x, w = bf16_bits_to_f64(xb), bf16_bits_to_f64(wb)
    zlib = x @ w.T + bias.astype(np.float64)
    np.testing.assert_allclose(r.z64, zlib, rtol=1e-13, atol=1e-13)
    # fp32 logits stay inside the forward error bound of recursive summation
    u = 2.0 ** -24
    gam = d * u / (1 - d * u)
    bound = gam * (np.abs(x) @ np.abs(w).T) + u * (np.abs(zlib) + 1e-30) * 2
    assert np.all(np.abs(r.z32.astype(np.float64) - zlib) <= bound)
    # the selection is the ordering of the fp32 logits (descending, ties to lower index)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(r.z32[t, e]), e))[:k]
        assert list(r.idx[t]) == order


def test_route_fp32_logits_are_the_ascending_sequential_sum():
    """Selection precision: fp32 sum in ascending feature order (numpy cumsum is sequential)."""
    rng = np.random.default_rng(4)
    T, d, E = 32, 200, 8
    xb = f32_to_bf16_bits(rng.standard_normal((T, d)))
    wb = f32_to_bf16_bits(rng.standard_normal((E, d)) / math.sqrt(d))
    r = oracle.route(xb, wb, None, 2, keep_logits=True)
    p = (bf16_bits_to_f64(xb)[:, None, :] * bf16_bits_to_f64(wb)[None, :, :]).astype(np.float32)
    seq = np.cumsum(p, axis=-1, dtype=np.float32)[..., -1]
    np.testing.assert_array_equal(r.z32, seq)


def test_gates_invariants():
    rng = np.random.default_rng(5)
    T, d, E = 50, 32, 12
    xb = f32_to_bf16_bits(rng.standard_normal((T, d)))
    wb = f32_to_bf16_bits(rng.standard_normal((E, d)) / math.sqrt(d))
    for k in (1, 2, 5, 8):
        r = oracle.route(xb, wb, None, k, keep_logits=True)
        np.testing.assert_allclose(r.gate.sum(axis=1), 1.0, atol=1e-12)
        assert np.all(np.diff(r.gate, axis=1) <= 1e-15)  # descending logits -> descending gates
        if k == 1:
            assert np.all(r.gate == 1.0)
        else:
            sel = np.take_along_axis(r.z64, r.idx, axis=1)
            np.testing.assert_allclose(r.gate[:, 0] / r.gate[:, 1], np.exp(sel[:, 0] - sel[:, 1]),
                                       rtol=1e-12)
            # softmax over all E experts, renormalised over the selection, is the same gate
            full = np.exp(r.z64 - r.z64.max(axis=1, keepdims=True))
            full /= full.sum(axis=1, keepdims=True)
            ren = np.take_along_axis(full, r.idx, axis=1)
            np.testing.assert_allclose(ren / ren.sum(axis=1, keepdims=True), r.gate, rtol=1e-12)


# ---------------------------------------------------------------- dispatch

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (7, 3, 5), (300, 6, 64), (0, 2, 4)])
def test_dispatch_vs_stable_sort(T, k, E):
    rng = np.random.default_rng(T * 31 + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else \
        np.zeros((0, k), np.int32)
    disp = oracle.dispatch(idx, E)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(disp.counts, np.bincount(flat, minlength=E))
    assert disp.offsets[0] == 0 and disp.offsets[-1] == T * k
    np.testing.assert_array_equal(np.diff(disp.offsets), disp.counts)
    np.testing.assert_array_equal(disp.slot_of_row, np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(disp.row_of_slot[disp.slot_of_row], np.arange(T * k))
    for e in range(E):
        rows = disp.slot_of_row[disp.offsets[e]:disp.offsets[e + 1]]
        assert np.all(flat[rows] == e) and np.all(np.diff(rows) > 0)


# ---------------------------------------------------------------- expert FFN

def _numpy_ffn(xin, er, w1, w3, w2):
    a = np.einsum("ni,nfi->nf", xin, w1[er])
    b = np.einsum("ni,nfi->nf", xin, w3[er])
    h = a * expit(a) * b
    return h, np.einsum("nf,nof->no", h, w2[er])


def test_ffn_vs_library_rectangular():
    rng = np.random.default_rng(6)
    n, d, F, E = 37, 24, 40, 3
    xb = f32_to_bf16_bits(rng.standard_normal((n, d)))
    w1b = f32_to_bf16_bits(rng.standard_normal((E, F, d)) / math.sqrt(d))
    w3b = f32_to_bf16_bits(rng.standard_normal((E, F, d)) / math.sqrt(d))
    w2b = f32_to_bf16_bits(rng.standard_normal((E, d, F)) / math.sqrt(F))
    er = rng.integers(0, E, n).astype(np.int32)
    h, y = oracle.ffn_rows(xb, er, w1b, w3b, w2b, E, keep_h=True)
    hr, yr = _numpy_ffn(bf16_bits_to_f64(xb), er, bf16_bits_to_f64(w1b), bf16_bits_to_f64(w3b),
                        bf16_bits_to_f64(w2b))
    np.testing.assert_allclose(h, hr, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(y, yr, rtol=1e-12, atol=1e-13)
    # linearity in W2: doubling W2 (exact in bf16) doubles y
    w2x2 = f32_to_bf16_bits(2.0 * bf16_bits_to_f64(w2b))
    _, y2 = oracle.ffn_rows(xb, er, w1b, w3b, w2x2, E)
    np.testing.assert_array_equal(y2, 2.0 * y)
    # silu is odd-asymmetric: negating W1 changes h, negating W3 flips its sign
    w3neg = f32_to_bf16_bits(-bf16_bits_to_f64(w3b))
    hneg, _ = oracle.ffn_rows(xb, er, w1b, w3neg, w2b, E, keep_h=True)
    np.testing.assert_array_equal(hneg, -h)


def test_identity_experts_round_trip():
    """Identity experts with k = 1: the gate is exactly 1, so combine(dispatch(x)) = x."""
    rng = np.random.default_rng(7)
    T, d, E = 64, 16, 5
    xb = f32_to_bf16_bits(rng.standard_normal((T, d)))
    wb = f32_to_bf16_bits(rng.standard_normal((E, d)))
    r = oracle.route(xb, wb, None, 1)
    assert np.all(r.gate == 1.0)
    disp = oracle.dispatch(r.idx, E)
    xperm = xb[disp.slot_of_row]
    _, yperm = oracle.ffn_rows(xperm, np.repeat(np.arange(E), disp.counts), None, None, None, E,
                               identity=True)
    out = oracle.combine(yperm, r.gate, disp.row_of_slot)
    np.testing.assert_array_equal(out, bf16_bits_to_f64(xb))
    out2 = oracle.layer_tokens(xb, r.idx, r.gate, None, None, None, np.arange(T), E, identity=True)
    np.testing.assert_array_equal(out2, bf16_bits_to_f64(xb))


def test_combine_vs_library():
    rng = np.random.default_rng(8)
    T, k, d = 20, 3, 10
    y = rng.standard_normal((T * k, d))
    g = rng.random((T, k))
    ros = rng.permutation(T * k).astype(np.int32)
    out = oracle.combine(y, g, ros)
    ref = np.einsum("tj,tjd->td", g, y[ros.reshape(T, k)])
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-14)


def test_full_layer_vs_numpy_tiny():
    """The whole tiny layer against an independent numpy formulation of the definition."""
    import synth
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg)
    xb, wrb = synth.bf16_bits(inp.x), synth.bf16_bits(inp.wr)
    w1b, w3b, w2b = synth.bf16_bits(inp.w1), synth.bf16_bits(inp.w3), synth.bf16_bits(inp.w2)
    r, disp, out = oracle.layer(xb, wrb, None, cfg.k, w1b, w3b, w2b)
    x, wr = bf16_bits_to_f64(xb), bf16_bits_to_f64(wrb)
    p = (x[:, None, :] * wr[None, :, :]).astype(np.float32)
    z32 = np.cumsum(p, axis=-1, dtype=np.float32)[..., -1]
    sel = np.array([sorted(range(cfg.E), key=lambda e: (-float(z32[t, e]), e))[:cfg.k]
                    for t in range(cfg.T)])
    np.testing.assert_array_equal(r.idx, sel)
    z = x @ wr.T
    zs = np.take_along_axis(z, sel, axis=1)
    g = np.exp(zs - zs.max(1, keepdims=True))
    g /= g.sum(1, keepdims=True)
    np.testing.assert_allclose(r.gate, g, rtol=1e-12)
    w1, w3, w2 = bf16_bits_to_f64(w1b), bf16_bits_to_f64(w3b), bf16_bits_to_f64(w2b)
    ref = np.zeros((cfg.T, cfg.d))
    for j in range(cfg.k):
        _, yj = _numpy_ffn(x, sel[:, j], w1, w3, w2)
        ref += g[:, j:j + 1] * yj
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
