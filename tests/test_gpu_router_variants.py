"""GPU parity of the router variants ("CMF v2 -- Format Specification", 2.2
MoE): sigmoid scores and the routed scaling factor, with and without a
selection bias and renormalisation, on every routing code path (the fused
decode kernel for T <= 8, the router kernel for larger streaming batches,
the grouped path's tensor-core logits), against the oracle."""
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from bit_expert_weight_gb300 import synth as Y  # noqa: E402

from helpers import HostLayer, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_expert_weight_gb300 import build
    build.build()
    import bit_expert_weight_gb300.smoe as S
    S.load()
    return S


def _keys(lg, bias, sigm):
    if bias is None:
        return lg
    if sigm:
        s = (1.0 / (1.0 + np.exp(-lg.astype(np.float64)))).astype(np.float32)
        return (s + bias[None, :]).astype(np.float32)
    return (lg + bias[None, :]).astype(np.float32)


def _near_ties(lg, k, bias, sigm, rel=1e-5):
    key = _keys(lg, bias, sigm)
    out = set()
    for t in range(key.shape[0]):
        s = np.sort(key[t])[::-1]
        fin = np.abs(key[t][np.isfinite(key[t])])
        if k < s.size and np.isfinite(s[k]) and abs(s[k - 1] - s[k]) < rel * max(fin.max(), 1e-30):
            out.add(t)
    return out


@pytest.mark.parametrize("E,k", [(8, 2), (64, 6), (128, 8), (256, 8)])
@pytest.mark.parametrize("sigm", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_route_from_logits_variants(S, E, k, sigm, with_bias):
    rng = np.random.default_rng(E * 7 + k + 3 * sigm + with_bias)
    T = 37
    lg = (rng.standard_normal((T, E)) * 1.5).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.2).astype(np.float32) if with_bias else None
    for norm, rsf in ((True, 2.5), (False, 1.0), (False, 0.75)):
        ids_r, w_r = O.route(lg, k, norm, bias, router_sigmoid=sigm, routed_scaling_factor=rsf)
        ids, w = S.route_from_logits(to_dev(lg, DEV), k, norm,
                                     None if bias is None else to_dev(bias, DEV),
                                     router_sigmoid=sigm, routed_scaling_factor=rsf)
        ids, w = ids.cpu().numpy(), w.cpu().numpy()
        ties = _near_ties(lg, k, bias, sigm)
        ok = [t for t in range(T) if t not in ties]
        assert np.array_equal(ids[ok], ids_r[ok])
        assert np.allclose(w[ok], w_r[ok], rtol=2e-6, atol=1e-7)


CFG = {
    # name: (d, f, E, k, norm, x_dtype, shared_f, shared_gate)
    "tiny_f32": (256, 128, 8, 2, True, "f32", 0, False),
    "tiny_bf16": (256, 128, 8, 2, True, "bf16", 0, False),
    "wide_bf16": (512, 128, 32, 6, True, "bf16", 0, False),
    "shared_bf16": (256, 128, 24, 8, False, "bf16", 192, True),
}
_HOST = {}


def _host(name):
    if name not in _HOST:
        d, f, E, k, norm, xd, sf, sg = CFG[name]
        seed = zlib.crc32(f"router-variants/{name}".encode()) & 0xFFFF
        wl = Y.Workload(name, d, f, E, k, norm, [4], [1], 1, seed, x_dtype=xd, shared_f=sf,
                        shared_gate=sg)
        _HOST[name] = (wl, HostLayer(wl, 0, 4))
    return _HOST[name]


@pytest.mark.parametrize("name,T,path", [("tiny_f32", 1, None), ("tiny_f32", 8, None),
                                         ("wide_bf16", 13, None), ("shared_bf16", 5, None),
                                         ("shared_bf16", 40, 2), ("wide_bf16", 96, 2),
                                         ("tiny_bf16", 64, 2), ("tiny_f32", 64, None)])
@pytest.mark.parametrize("sigm,rsf,with_bias", [(True, 1.0, False), (True, 2.5, True),
                                                (False, 2.5, True)])
def test_forward_with_router_variants(S, name, T, path, sigm, rsf, with_bias):
    wl, hl = _host(name)
    bias = None
    if with_bias:
        bias = (np.random.default_rng(4).standard_normal(wl.E) * (0.05 if sigm else 0.5)).astype(
            np.float32)
    lay = hl.device_layer(DEV, expert_bias=bias)
    x, _ = wl.activations(0, T)
    xt = to_dev(x, DEV)
    if wl.x_dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    ws = S.workspace(lay, T)
    ids = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    y = S.forward(lay, xt, ws, ids=ids, w=w, path=path, router_sigmoid=sigm,
                  routed_scaling_factor=rsf)
    torch.cuda.synchronize()
    assert S.device_status() == 0
    y, ids, w = y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()
    y_ref, ids_ref, w_ref, lg = O.moe_forward(
        wl.d, wl.f, wl.E, wl.k, wl.norm, 4, hl.router, hl.blob, x, expert_bias=bias,
        shared_blob=hl.shared_blob, fs=wl.shared_f, shared_gate=hl.shared_gate,
        router_sigmoid=sigm, routed_scaling_factor=rsf)
    ties = _near_ties(lg, wl.k, bias, sigm)
    mism = [t for t in range(T) if not np.array_equal(ids[t], ids_ref[t])]
    assert set(mism) <= ties, sorted(set(mism) - ties)
    if mism:
        y_ref = y_ref.copy()
        y_ref[mism] = hl.oracle_apply(x[mism], ids[mism], w[mism])
    ok = [t for t in range(T) if t not in mism]
    assert np.allclose(w[ok], w_ref[ok], rtol=1e-5, atol=1e-6)
    tol = 2e-2 if (path == 2 or S.path_for(lay, T, xt.dtype) == S.PATH_GROUPED) else 1e-3
    err = float(np.abs(y - y_ref).max())
    assert err <= tol * float(np.abs(y_ref).max()), (err, tol)


def _mask_bits(routable, E):
    m = np.zeros((E + 7) // 8, np.uint8)
    for e in routable:
        m[e // 8] |= 1 << (e % 8)
    return m


@pytest.mark.parametrize("E,k", [(20, 3), (64, 6), (256, 8)])
@pytest.mark.parametrize("sigm", [False, True])
def test_route_from_logits_with_mask(S, E, k, sigm):
    rng = np.random.default_rng(E + k + sigm)
    T = 29
    lg = (rng.standard_normal((T, E)) * 1.5).astype(np.float32)
    allowed = sorted(rng.choice(E, size=max(k, E // 3), replace=False).tolist())
    mask = _mask_bits(allowed, E)
    ids_r, w_r = O.route(lg, k, True, router_sigmoid=sigm, routed_scaling_factor=1.5, mask=mask)
    ids, w = S.route_from_logits(to_dev(lg, DEV), k, True, router_sigmoid=sigm,
                                 routed_scaling_factor=1.5, expert_mask=mask)
    ids, w = ids.cpu().numpy(), w.cpu().numpy()
    masked = np.full_like(lg, -np.inf)
    masked[:, allowed] = lg[:, allowed]
    ties = _near_ties(masked, k, None, sigm)
    ok = [t for t in range(T) if t not in ties]
    assert set(ids.ravel().tolist()) <= set(allowed)
    assert np.array_equal(ids[ok], ids_r[ok])
    assert np.allclose(w[ok], w_r[ok], rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("name,T,path", [("tiny_f32", 3, None), ("wide_bf16", 13, None),
                                         ("wide_bf16", 96, 2), ("shared_bf16", 40, 2)])
def test_forward_with_routing_mask(S, name, T, path):
    wl, hl = _host(name)
    allowed = list(range(0, wl.E, 3))[:max(wl.k, wl.E // 2)]
    if len(allowed) < wl.k:
        allowed = list(range(wl.k))
    mask = _mask_bits(allowed, wl.E)
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, T)
    xt = to_dev(x, DEV)
    if wl.x_dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    ws = S.workspace(lay, T)
    ids = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    y = S.forward(lay, xt, ws, ids=ids, w=w, path=path, expert_mask=mask)
    torch.cuda.synchronize()
    assert S.device_status() == 0
    y, ids, w = y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()
    y_ref, ids_ref, w_ref, lg = O.moe_forward(
        wl.d, wl.f, wl.E, wl.k, wl.norm, 4, hl.router, hl.blob, x, shared_blob=hl.shared_blob,
        fs=wl.shared_f, shared_gate=hl.shared_gate, mask=mask)
    assert set(ids.ravel().tolist()) <= set(allowed)
    masked = np.full_like(lg, -np.inf)
    masked[:, allowed] = lg[:, allowed]
    ties = _near_ties(masked, wl.k, None, False)
    mism = [t for t in range(T) if not np.array_equal(ids[t], ids_ref[t])]
    assert set(mism) <= ties
    if mism:
        y_ref = y_ref.copy()
        y_ref[mism] = hl.oracle_apply(x[mism], ids[mism], w[mism])
    ok = [t for t in range(T) if t not in mism]
    assert np.allclose(w[ok], w_ref[ok], rtol=1e-5, atol=1e-6)
    tol = 2e-2 if (path == 2 or S.path_for(lay, T, xt.dtype) == S.PATH_GROUPED) else 1e-3
    assert float(np.abs(y - y_ref).max()) <= tol * float(np.abs(y_ref).max())
