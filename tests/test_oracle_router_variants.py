"""Pins of the oracle's router variants ("CMF v2 -- Format Specification",
2.2 MoE): with router_sigmoid each expert is scored by sigmoid(logit) on
its own; the expert_bias only moves the selection; the selected scores are
optionally renormalised, then multiplied by routed_scaling_factor."""
import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle as O


def _brute(logits, k, norm, bias, sigm, rsf):
    """Brute-force reference from the stated semantics (library routines for
    the scores, an explicit key order for the selection)."""
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    for t in range(T):
        l = logits[t].astype(np.float64)
        s = expit(l) if sigm else softmax(l)
        if bias is None:
            key = logits[t]
        elif sigm:
            key = (s.astype(np.float32) + bias).astype(np.float32)
        else:
            key = (logits[t] + bias).astype(np.float32)
        order = sorted(range(E), key=lambda e: (-float(key[e]), e))[:k]
        ids[t] = order
        sel = s[order]
        w[t] = (sel / sel.sum() if norm else sel) * rsf
    return ids, w


@pytest.mark.parametrize("sigm", [False, True])
@pytest.mark.parametrize("norm", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("rsf", [1.0, 2.5])
def test_route_variants_match_their_definition(sigm, norm, with_bias, rsf):
    rng = np.random.default_rng(11)
    T, E, k = 20, 24, 5
    lg = (rng.standard_normal((T, E)) * 2.0).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.3).astype(np.float32) if with_bias else None
    ids, w = O.route(lg, k, norm, bias, router_sigmoid=sigm, routed_scaling_factor=rsf)
    ids_ref, w_ref = _brute(lg, k, norm, bias, sigm, rsf)
    assert np.array_equal(ids, ids_ref)
    assert np.allclose(w, w_ref, rtol=1e-6, atol=0)


def test_sigmoid_weights_without_renorm_are_the_scores():
    lg = np.array([[3.0, -1.0, 0.5, 2.0, -4.0]], np.float32)
    ids, w = O.route(lg, 3, False, router_sigmoid=True)
    assert list(ids[0]) == [0, 3, 2]
    assert np.allclose(w[0], expit(np.array([3.0, 2.0, 0.5])), rtol=1e-7)
    # renormalised they sum to the scaling factor
    _, w2 = O.route(lg, 3, True, router_sigmoid=True, routed_scaling_factor=2.5)
    assert abs(float(w2.sum()) - 2.5) < 1e-6


def test_sigmoid_bias_selects_on_score_plus_bias_and_ties_go_low():
    # equal sigmoid scores + equal bias: ties to the lower index
    lg = np.array([[1.0, 1.0, 1.0, 0.0]], np.float32)
    ids, _ = O.route(lg, 2, False, np.zeros(4, np.float32), router_sigmoid=True)
    assert list(ids[0]) == [0, 1]
    # a bias of +1 lifts expert 3 (score 0.5) above the others (score 0.73)
    b = np.array([0, 0, 0, 1.0], np.float32)
    ids, w = O.route(lg, 2, False, b, router_sigmoid=True)
    assert list(ids[0]) == [3, 0]
    assert np.allclose(w[0], expit(np.array([0.0, 1.0])), rtol=1e-7)  # bias not in weights


def test_scaling_factor_is_linear_and_validated():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((6, 16)).astype(np.float32)
    i1, w1 = O.route(lg, 4, True)
    i2, w2 = O.route(lg, 4, True, routed_scaling_factor=2.5)
    assert np.array_equal(i1, i2)
    assert np.allclose(w2, 2.5 * w1, rtol=1e-6)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(ValueError):
            O.route(lg, 4, True, routed_scaling_factor=bad)


def _mask_bits(routable, E):
    m = np.zeros((E + 7) // 8, np.uint8)
    for e in routable:
        m[e // 8] |= 1 << (e % 8)
    return m


@pytest.mark.parametrize("sigm", [False, True])
def test_routing_mask_restricts_selection_and_softmax(sigm):
    """"CMF v2", 5: bit e of the layer's row set = expert e routable;
    selection over the routable set only, the softmax renormalising over
    it."""
    rng = np.random.default_rng(21)
    T, E, k = 12, 20, 3
    lg = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    allowed = [1, 2, 5, 8, 9, 13, 17, 19]
    mask = _mask_bits(allowed, E)
    ids, w = O.route(lg, k, False, router_sigmoid=sigm, mask=mask)
    for t in range(T):
        sub = lg[t, allowed].astype(np.float64)
        s = expit(sub) if sigm else softmax(sub)
        order = sorted(range(len(allowed)), key=lambda i: (-float(lg[t, allowed[i]]), allowed[i]))[:k]
        assert list(ids[t]) == [allowed[i] for i in order]
        assert np.allclose(w[t], s[order], rtol=1e-6)
    # an all-ones row restricts nothing
    i1, w1 = O.route(lg, k, True)
    i2, w2 = O.route(lg, k, True, mask=_mask_bits(range(E), E))
    assert np.array_equal(i1, i2) and np.array_equal(w1, w2)


def test_routing_mask_is_validated():
    lg = np.zeros((2, 10), np.float32)
    with pytest.raises(ValueError):  # fewer routable experts than k
        O.route(lg, 3, True, mask=_mask_bits([1, 2], 10))
    bad = _mask_bits([1, 2, 3], 10)
    bad[1] |= 0x80  # a tail bit beyond E
    with pytest.raises(ValueError):
        O.route(lg, 2, True, mask=bad)
