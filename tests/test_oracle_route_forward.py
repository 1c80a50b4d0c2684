"""Pins for the oracle's router and MoE forward.

Routing semantics: "CMF v2 -- Format Specification", 2.2 MoE (softmax over all
logits, ties to the lower index, selection-only expert_bias, optional
renormalisation, shared expert weight sigmoid(gate . x) or 1).  The forward is
checked by brute force: an independent numpy dequantiser (unpacking by bit
arithmetic, levels from exact fractions) builds dense fp64 matrices, and the
textbook SwiGLU MoE is evaluated with numpy matmuls.
"""
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle as O
from bit_expert_weight_gb300 import synth as S


def bf16(a):
    return S._f32_to_bf16_rne(np.asarray(a, np.float32))


# ------------------------------------------------------------------ routing

def test_route_ties_go_to_lower_index():
    lg = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.0]], np.float32)
    ids, w = O.route(lg, 3, norm=False)
    assert ids.tolist() == [[1, 2, 4]]
    ids, _ = O.route(lg, 4, norm=False)
    assert ids.tolist() == [[1, 2, 4, 3]]
    allsame = np.zeros((1, 8), np.float32)
    ids, w = O.route(allsame, 5, norm=True)
    assert ids.tolist() == [[0, 1, 2, 3, 4]]
    assert np.allclose(w, 0.2)


def test_route_k_equals_E_is_stable_descending_sort():
    rng = np.random.default_rng(0)
    lg = rng.integers(-3, 4, size=(50, 16)).astype(np.float32)  # many ties
    ids, w = O.route(lg, 16, norm=False)
    ref = np.argsort(-lg, axis=1, kind="stable")
    assert np.array_equal(ids, ref)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)


def test_route_weights_are_softmax_over_all_logits():
    rng = np.random.default_rng(1)
    lg = (rng.standard_normal((40, 64)) * 2).astype(np.float32)
    p = softmax(lg.astype(np.float64), axis=1)
    ids, w = O.route(lg, 6, norm=False)
    assert np.allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-6)
    assert np.all(w.sum(1) <= 1.0 + 1e-6)
    ids2, w2 = O.route(lg, 6, norm=True)
    assert np.array_equal(ids, ids2)
    sel = np.take_along_axis(p, ids, 1)
    assert np.allclose(w2, sel / sel.sum(1, keepdims=True), rtol=1e-6)
    assert np.allclose(w2.sum(1), 1.0, atol=1e-6)
    # selection picks the k largest probabilities
    for t in range(40):
        assert set(ids[t]) == set(np.argsort(-p[t], kind="stable")[:6])


def test_expert_bias_affects_selection_only():
    lg = np.array([[2.0, 1.0, 0.5, 0.0]], np.float32)
    bias = np.array([0.0, 0.0, 5.0, 0.0], np.float32)
    ids, w = O.route(lg, 2, norm=False, bias=bias)
    assert ids.tolist() == [[2, 0]]
    p = softmax(lg.astype(np.float64), axis=1)[0]
    assert np.allclose(w[0], [p[2], p[0]], rtol=1e-6)


def test_route_rejects_bad_k():
    lg = np.zeros((1, 4), np.float32)
    for k in (0, 5, 17):
        with pytest.raises(ValueError):
            O.route(lg, k, norm=False)


# ------------------------------------------------------------------ forward

def np_dequant(q, rows, cols, bits):
    """Independent dequantiser: bit arithmetic + exact level fractions."""
    n = rows * cols
    per = 8 // bits
    idx = np.arange(n)
    c = (q["codes_lsb"][idx // per] >> ((idx % per) * bits)) & ((1 << bits) - 1)
    nl = (1 << bits) - 1
    lv = np.array([float(Fraction(2 * i - nl, nl)) for i in range(nl + 1)])
    s = q["scales_f16"].view(np.float16).astype(np.float64)
    return (lv[c] * s[idx // 64]).reshape(rows, cols)


def make_layer(d, f, E, bits, seed, shared_f=0):
    rng = np.random.default_rng(seed)

    def w(r, c):
        a = (rng.standard_normal((r, c)) * 0.02).astype(np.float32)
        a[rng.random((r, c)) < 0.01] *= 10
        return bf16(a)

    experts = []
    for _ in range(E + (1 if shared_f else 0)):
        ff = f if len(experts) < E else shared_f
        g, u, dn = w(ff, d), w(ff, d), w(d, ff)
        qg, qu, qd = O.quantize(g, bits), O.quantize(u, bits), O.quantize(dn, bits)
        experts.append({
            "blob": O.make_blob(qg, qu, qd), "f": ff,
            "Wg": np_dequant(qg, ff, d, bits), "Wu": np_dequant(qu, ff, d, bits),
            "Wd": np_dequant(qd, d, ff, bits),
        })
    router = w(E, d)
    return experts, router


def swiglu(e, x):
    g = e["Wg"] @ x
    u = e["Wu"] @ x
    return e["Wd"] @ (g * expit(g) * u)


@pytest.mark.parametrize("bits", [2, 4])
def test_forward_matches_dense_brute_force(bits):
    d, f, E, k, T = 128, 64, 6, 2, 5
    experts, router = make_layer(d, f, E, bits, seed=10 + bits)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((T, d)).astype(np.float32)
    y, ids, w, lg = O.moe_forward(d, f, E, k, True, bits, router,
                                  [e["blob"] for e in experts], x)
    Wr = S.bf16_to_f32(router).astype(np.float64)
    assert np.allclose(lg, x.astype(np.float64) @ Wr.T, rtol=1e-5, atol=1e-6)
    for t in range(T):
        ref = sum(float(w[t, j]) * swiglu(experts[ids[t, j]], x[t].astype(np.float64))
                  for j in range(k))
        assert np.allclose(y[t], ref, rtol=1e-4, atol=1e-5 * np.abs(ref).max())


def test_expert_ffn_matches_dense_and_returns_h():
    d, f = 128, 64
    experts, _ = make_layer(d, f, 1, 4, seed=3)
    x = np.random.default_rng(2).standard_normal(d).astype(np.float32)
    out, h = O.expert_ffn(experts[0]["blob"], d, f, 4, x)
    e = experts[0]
    g = e["Wg"] @ x
    u = e["Wu"] @ x
    href = g * expit(g) * u
    assert np.allclose(h, href, rtol=1e-5, atol=1e-7)
    assert np.allclose(out, e["Wd"] @ href, rtol=1e-4, atol=1e-6)


def test_single_expert_reduces_to_swiglu_ffn():
    """E = 1, k = 1 with renormalisation: the layer is one SwiGLU FFN."""
    d, f = 128, 64
    experts, router = make_layer(d, f, 1, 4, seed=4)
    x = np.random.default_rng(3).standard_normal((3, d)).astype(np.float32)
    y, ids, w, _ = O.moe_forward(d, f, 1, 1, True, 4, router, [experts[0]["blob"]], x)
    assert np.all(ids == 0) and np.all(w == 1.0)
    for t in range(3):
        out, _ = O.expert_ffn(experts[0]["blob"], d, f, 4, x[t])
        assert np.array_equal(y[t], out)


def test_combine_is_linear_in_routing_weights():
    d, f, E, k = 128, 64, 4, 2
    experts, _ = make_layer(d, f, E, 4, seed=5)
    blobs = [e["blob"] for e in experts]
    x = np.random.default_rng(4).standard_normal((2, d)).astype(np.float32)
    ids = np.array([[1, 3], [0, 2]], np.int32)
    wa = np.array([[0.25, 0.5], [1.0, 0.125]], np.float32)
    wb = np.array([[0.5, 0.25], [0.0, 2.0]], np.float32)
    ya = O.moe_apply(d, f, E, k, 4, blobs, x, ids, wa)
    yb = O.moe_apply(d, f, E, k, 4, blobs, x, ids, wb)
    yab = O.moe_apply(d, f, E, k, 4, blobs, x, ids, wa + wb)
    assert np.allclose(ya + yb, yab, rtol=1e-5, atol=1e-7)


def test_shared_expert_weight_is_sigmoid_of_gate():
    d, f, E, k, fs = 128, 64, 4, 2, 64
    experts, router = make_layer(d, f, E, 4, seed=6, shared_f=fs)
    blobs = [e["blob"] for e in experts[:E]]
    sh = experts[E]
    gate = bf16((np.random.default_rng(9).standard_normal(d) * 0.3).astype(np.float32))
    x = np.random.default_rng(8).standard_normal((3, d)).astype(np.float32)
    y0, ids, w, _ = O.moe_forward(d, f, E, k, True, 4, router, blobs, x)
    y1, _, _, _ = O.moe_forward(d, f, E, k, True, 4, router, blobs, x,
                                shared_blob=sh["blob"], fs=fs, shared_gate=gate)
    y2, _, _, _ = O.moe_forward(d, f, E, k, True, 4, router, blobs, x,
                                shared_blob=sh["blob"], fs=fs)
    gv = S.bf16_to_f32(gate).astype(np.float64)
    for t in range(3):
        xt = x[t].astype(np.float64)
        s = swiglu(sh, xt)
        sw = expit(gv @ xt)
        assert np.allclose(y1[t] - y0[t], sw * s, rtol=1e-3, atol=1e-5 * np.abs(s).max())
        assert np.allclose(y2[t] - y0[t], s, rtol=1e-3, atol=1e-5 * np.abs(s).max())


def test_forward_missing_blob_is_an_error():
    d, f, E = 128, 64, 3
    experts, router = make_layer(d, f, E, 4, seed=7)
    x = np.random.default_rng(1).standard_normal((1, d)).astype(np.float32)
    _, ids, _, _ = O.moe_forward(d, f, E, 1, True, 4, router, [e["blob"] for e in experts], x)
    blobs = {e: experts[e]["blob"] for e in range(E) if e != ids[0, 0]}
    with pytest.raises(ValueError):
        O.moe_forward(d, f, E, 1, True, 4, router, blobs, x)


def test_mixed_bit_depth_forward_matches_dense_brute_force():
    """Experts at their own depths (Q2 and Q4 in one layer): each expert's
    FFN decodes its own levels; the shared expert at the layer's depth."""
    d, f, E, k, T = 128, 64, 6, 3, 5
    bits_e = [4, 2, 2, 4, 2, 4]
    layers = {b: make_layer(d, f, E, b, seed=30, shared_f=64) for b in (2, 4)}
    experts = [layers[bits_e[e]][0][e] for e in range(E)]
    shared = layers[4][0][E]
    router = layers[4][1]
    rng = np.random.default_rng(8)
    x = rng.standard_normal((T, d)).astype(np.float32)
    y, ids, w, lg = O.moe_forward(d, f, E, k, True, 4, router, [e["blob"] for e in experts], x,
                                  shared_blob=shared["blob"], fs=64, expert_bits=bits_e)
    for t in range(T):
        xt = x[t].astype(np.float64)
        ref = sum(float(w[t, j]) * swiglu(experts[ids[t, j]], xt) for j in range(k))
        ref = ref + swiglu(shared, xt)
        assert np.allclose(y[t], ref, rtol=1e-4, atol=1e-5 * np.abs(ref).max())
    # all experts at one depth: the uniform forward
    y4, _, _, _ = O.moe_forward(d, f, E, k, True, 4, router,
                                [layers[4][0][e]["blob"] for e in range(E)], x,
                                expert_bits=[4] * E)
    y4u, _, _, _ = O.moe_forward(d, f, E, k, True, 4, router,
                                 [layers[4][0][e]["blob"] for e in range(E)], x)
    assert np.array_equal(y4, y4u)


def test_threaded_apply_gives_the_serial_bits():
    """The benchmark's all-cores oracle leg (expert FFNs of the (token, slot)
    items on several threads, the combine serial in rank order) must equal
    the single-threaded oracle bit for bit; also checked against the dense
    brute force so that a shared mistake would still show."""
    d, f, E, k, fs, T = 128, 64, 5, 3, 64, 4
    experts, router = make_layer(d, f, E, 4, seed=21, shared_f=fs)
    blobs = [e["blob"] for e in experts[:E]]
    gate = bf16((np.random.default_rng(5).standard_normal(d) * 0.3).astype(np.float32))
    x = np.random.default_rng(6).standard_normal((T, d)).astype(np.float32)
    _, ids, w, _ = O.moe_forward(d, f, E, k, True, 4, router, blobs, x)
    ref = O.moe_apply(d, f, E, k, 4, blobs, x, ids, w, shared_blob=experts[E]["blob"], fs=fs,
                      shared_gate=gate)
    for nt in (1, 3, 16):
        got = O.moe_apply_threads(d, f, E, k, 4, blobs, x, ids, w, nt,
                                  shared_blob=experts[E]["blob"], fs=fs, shared_gate=gate)
        assert np.array_equal(got, ref), nt
    gv = S.bf16_to_f32(gate).astype(np.float64)
    for t in range(T):
        xt = x[t].astype(np.float64)
        dense = sum(float(w[t, j]) * swiglu(experts[ids[t, j]], xt) for j in range(k))
        dense = dense + expit(gv @ xt) * swiglu(experts[E], xt)
        assert np.allclose(ref[t], dense, rtol=1e-4, atol=1e-5 * np.abs(dense).max())
