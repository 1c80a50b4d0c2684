"""GPU parity of layers whose routed experts each have their own depth
(some SMOE-Q2, some SMOE-Q4 in one bank; "CMF v2", 2.2 MoE: every expert
entry carries its own dtype) against the oracle.

Such a layer runs on both paths: the streaming kernel (bar 1e-3 *
||y_ref||_inf), whose units each decode at their expert's depth, and the
grouped tensor-core path (bar 2e-2), one GEMM launch per depth present.
The tests cover one token (fused routing and combine), small batches on
either path, both shared-expert depths, one expert of the minority depth,
m-tile pairing, and bit-equality with the single-depth kernels when every
expert has the same depth.
"""
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_expert_weight_gb300 import synth as Y  # noqa: E402

import oracle as O  # noqa: E402
from helpers import HostLayer, check_forward, near_tie_tokens, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-2

CFG = {
    # name: (d, f, E, k, norm, x_dtype, shared_f, shared_gate, shared bits)
    "tiny_f32": (256, 128, 8, 2, True, "f32", 0, False, 4),
    "half_ntile_bf16": (256, 192, 16, 4, False, "bf16", 0, False, 4),
    "shared_bf16": (256, 128, 24, 8, True, "bf16", 192, True, 2),
    "shared_f32": (384, 64, 12, 3, True, "f32", 64, False, 4),
    # bf16 twins of the fp32 shapes for the grouped path (bf16 tokens only)
    "tiny_bf16": (256, 128, 8, 2, True, "bf16", 0, False, 4),
    "shared_nogate_bf16": (384, 64, 12, 3, True, "bf16", 64, False, 4),
}


def pattern(name, E, wl):
    if name == "alternate":
        return [4 if e % 2 == 0 else 2 for e in range(E)]
    if name == "one_q4":
        return [4 if e == 3 else 2 for e in range(E)]
    if name == "one_q2":
        return [2 if e == E - 1 else 4 for e in range(E)]
    if name == "popular":
        return wl.mixed_bits(0.25)
    raise KeyError(name)


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_expert_weight_gb300 import build
    build.build()
    import bit_expert_weight_gb300.smoe as S
    S.load()
    return S


_HOST = {}


def host_layer(name, pat):
    key = (name, pat)
    if key not in _HOST:
        d, f, E, k, norm, xd, sf, sg, sb = CFG[name]
        seed = zlib.crc32(f"mixed/{name}".encode()) & 0xFFFF
        wl = Y.Workload(name, d, f, E, k, norm, [4, 2], [1], 1, seed, x_dtype=xd,
                        shared_f=sf, shared_gate=sg)
        _HOST[key] = (wl, HostLayer(wl, 0, sb, expert_bits=pattern(pat, E, wl)))
    return _HOST[key]


def run(S, lay, wl, x_host, **router):
    T = x_host.shape[0]
    xt = to_dev(x_host, DEV)
    if wl.x_dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    ws = S.workspace(lay, T)
    ids = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    y = S.forward(lay, xt, ws, ids=ids, w=w, **router)
    torch.cuda.synchronize()
    assert S.device_status() == 0
    return y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


STREAM, GROUPED = 1, 2


@pytest.mark.parametrize("name,pat,T,path", [
    # streaming: fused routing + combine (T <= 8), then the separate stages;
    # fp32 tokens stream at every batch size
    ("tiny_f32", "alternate", 1, None), ("half_ntile_bf16", "alternate", 5, None),
    ("shared_bf16", "alternate", 3, None), ("shared_f32", "alternate", 9, None),
    ("shared_bf16", "one_q2", 40, STREAM), ("tiny_f32", "one_q4", 200, STREAM),
    ("half_ntile_bf16", "popular", 64, STREAM), ("shared_f32", "one_q4", 150, STREAM),
    ("tiny_f32", "one_q2", 700, None),
    # grouped, small batches included
    ("tiny_bf16", "alternate", 1, GROUPED), ("shared_bf16", "popular", 7, GROUPED),
    ("tiny_bf16", "alternate", 16, GROUPED), ("tiny_bf16", "one_q4", 200, GROUPED),
    ("tiny_bf16", "one_q2", 700, None), ("half_ntile_bf16", "one_q4", 333, None),
    ("shared_bf16", "popular", 300, None), ("shared_bf16", "one_q2", 40, GROUPED),
    ("shared_nogate_bf16", "one_q4", 150, GROUPED),
    # >= 256 rows per expert on average: items pair two m-tiles
    ("tiny_bf16", "alternate", 1100, None), ("half_ntile_bf16", "popular", 1030, None),
])
def test_mixed_matches_oracle(S, name, pat, T, path):
    wl, hl = host_layer(name, pat)
    lay = hl.device_layer(DEV)
    xdt = torch.float32 if wl.x_dtype == "f32" else torch.bfloat16
    grouped = path == GROUPED or (path is None and S.path_for(lay, T, xdt) == S.PATH_GROUPED)
    x, _ = wl.activations(0, T)
    y, ids, w = run(S, lay, wl, x, path=path)
    check_forward(y, ids, w, hl, x, tol=TOL if grouped else 1e-3)


def test_mixed_grouped_path_refuses_fp32_tokens(S):
    """The tensor-core path takes bf16 tokens only; a forced grouped forward
    of fp32 tokens is refused with nothing enqueued."""
    wl, hl = host_layer("tiny_f32", "alternate")
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, 64)
    xt = to_dev(x, DEV)
    ws = S.workspace(lay, 64)
    y = torch.full((64, wl.d), 7.0, dtype=torch.float32, device=DEV)
    with pytest.raises(S.SmoeError) as ei:
        S.forward(lay, xt, ws, y=y, path=GROUPED)
    assert ei.value.status == -2
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


def test_repack_mixed_is_the_per_expert_repacks_back_to_back(S):
    """Each expert's tiles are its own-depth repack, at the running sum of
    the sizes before it; the unpack restores every stream byte."""
    wl, hl = host_layer("shared_f32", "alternate")
    lay = hl.device_layer(DEV)
    tiles = lay.expert_tiles.cpu().numpy()
    off = 0
    codes, scales = lay._keep
    for e in range(wl.E):
        b = hl.expert_bits[e]
        one = S.repack(codes[3 * e:3 * e + 3], scales[3 * e:3 * e + 3], wl.d, wl.f, 1, b)
        n = S.expert_tiles_bytes(wl.d, wl.f, b)
        assert np.array_equal(tiles[off:off + n], one.cpu().numpy()), e
        off += n
    assert off == tiles.size == S.repacked_bytes_mixed(wl.d, wl.f, hl.expert_bits)
    c2, s2 = S.unpack_mixed(lay.expert_tiles, wl.d, wl.f, hl.expert_bits)
    for a, b in zip(codes + scales, c2 + s2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("T,path", [(5, STREAM), (40, STREAM), (96, GROUPED)])
def test_one_depth_mixed_equals_the_single_depth_kernels(S, bits, T, path):
    """Every expert at the same depth: the mixed-depth kernels give the
    single-depth kernels' bits on both paths."""
    d, f, E, k, norm, xd, sf, sg, _ = CFG["shared_bf16"]
    wl = Y.Workload("shared_bf16", d, f, E, k, norm, [bits], [1], 1, 77, x_dtype=xd,
                    shared_f=sf, shared_gate=sg)
    hu = HostLayer(wl, 0, bits)
    hm = HostLayer(wl, 0, bits, expert_bits=[bits] * E)
    x, _ = wl.activations(0, T)
    yu, idu, wu = run(S, hu.device_layer(DEV), wl, x, path=path)
    ym, idm, wm = run(S, hm.device_layer(DEV), wl, x, path=path)
    assert np.array_equal(idu, idm) and np.array_equal(wu, wm)
    assert np.array_equal(yu, ym)


@pytest.mark.parametrize("T", [6, 70])
def test_mixed_with_router_options(S, T):
    """Sigmoid scores, a routed scaling factor, a selection bias and a
    routing mask on a mixed layer (the router is independent of depth), on
    the streaming (6 tokens) and the grouped path (70)."""
    wl, hl = host_layer("shared_bf16", "alternate")
    bias = (np.random.default_rng(9).standard_normal(wl.E) * 0.05).astype(np.float32)
    allowed = [e for e in range(wl.E) if e % 3 != 1]
    mask = np.zeros((wl.E + 7) // 8, np.uint8)
    for e in allowed:
        mask[e // 8] |= 1 << (e % 8)
    lay = hl.device_layer(DEV, expert_bias=bias)
    x, _ = wl.activations(0, T)
    y, ids, w = run(S, lay, wl, x, router_sigmoid=True, routed_scaling_factor=2.5,
                    expert_mask=mask)
    y_ref, ids_ref, w_ref, lg = hl.oracle_forward(x, bias, router_sigmoid=True,
                                                  routed_scaling_factor=2.5, mask=mask)
    assert set(ids.ravel().tolist()) <= set(allowed)
    # selection keys of the routable experts: fl32(sigmoid(logit)) + bias
    sig = (1.0 / (1.0 + np.exp(-lg.astype(np.float64)))).astype(np.float32)
    key = (sig[:, allowed] + bias[allowed]).astype(np.float32)
    ties = set(near_tie_tokens(key, wl.k, rel=1e-5))
    mism = [t for t in range(T) if not np.array_equal(ids[t], ids_ref[t])]
    assert set(mism) <= ties
    if mism:
        y_ref = y_ref.copy()
        y_ref[mism] = hl.oracle_apply(x[mism], ids[mism], w[mism])
    ok = [t for t in range(T) if t not in mism]
    assert np.allclose(w[ok], w_ref[ok], rtol=1e-5, atol=1e-6)
    xdt = torch.float32 if wl.x_dtype == "f32" else torch.bfloat16
    tol = TOL if S.path_for(lay, T, xdt) == S.PATH_GROUPED else 1e-3
    assert float(np.abs(y - y_ref).max()) <= tol * float(np.abs(y_ref).max())


def test_mixed_is_deterministic(S):
    wl, hl = host_layer("half_ntile_bf16", "popular")
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, 120)
    y1, _, _ = run(S, lay, wl, x)
    y2, _, _ = run(S, lay, wl, x)
    assert np.array_equal(y1, y2)


@pytest.mark.parametrize("T", [12, 50])
def test_mixed_stages_compose_to_the_whole_forward(S, T):
    """The three launch stages, called one by one, give the forward's bits
    (12 tokens: streaming stages; 50: grouped)."""
    wl, hl = host_layer("shared_bf16", "one_q4")
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, T)
    y_all, _, _ = run(S, lay, wl, x)
    xt = to_dev(x, DEV).to(torch.bfloat16)
    ws = S.workspace(lay, T)
    y = torch.empty((T, wl.d), dtype=torch.float32, device=DEV)
    for st in range(3):
        S.forward_stage(lay, st, xt, ws, y)
    torch.cuda.synchronize()
    assert S.device_status() == 0
    assert np.array_equal(y.cpu().numpy(), y_all)
