"""GPU parity of the expert-sorted grouped (tensor-core) path against the
oracle.

The grouped path takes bf16 tokens, rounds the dequantised weights and h to
bf16 (the tcgen05 kind::f16 operand type) and accumulates in fp32; its bar
for bf16 activations is max-abs-error <= 2e-2 * ||y_ref||_inf.  fp32 tokens
never take it: the forward sends them to the streaming path, whose bar is
1e-3 * ||y_ref||_inf, and a forced grouped forward of fp32 tokens is
refused.  Shapes are chosen so that experts span several 128-row m-tiles
with a ragged last one, gate/up n-tiles end half full (f % 128 == 64), down
n-tiles end half full (d % 256 == 128), and the shared expert (all tokens)
is a segment of its own.
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
    # name: (d, f, E, k, norm, x_dtype, shared_f, shared_gate, p_zero)
    "tiny_bf16": (256, 128, 8, 2, True, "bf16", 0, False, 0.2),
    "half_ntile_bf16": (256, 192, 16, 4, False, "bf16", 0, False, 0.0),
    "wide_bf16": (512, 128, 32, 6, True, "bf16", 0, False, 0.0),
    "shared_bf16": (256, 128, 24, 8, True, "bf16", 192, True, 0.0),
    "shared_nogate_bf16": (384, 64, 12, 3, True, "bf16", 64, False, 0.0),
    # fp32 tokens at grouped-path batch sizes (they stream)
    "tiny_f32": (256, 128, 8, 2, True, "f32", 0, False, 0.2),
    "shared_nogate_f32": (384, 64, 12, 3, True, "f32", 64, False, 0.0),
}
TOL_F32 = 1e-3


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


def host_layer(name, bits):
    key = (name, bits)
    if key not in _HOST:
        d, f, E, k, norm, xd, sf, sg, pz = CFG[name]
        seed = zlib.crc32(f"grouped/{name}/{bits}".encode()) & 0xFFFF
        wl = Y.Workload(name, d, f, E, k, norm, [bits], [1], 1, seed, x_dtype=xd, p_zero=pz,
                        shared_f=sf, shared_gate=sg)
        _HOST[key] = (wl, HostLayer(wl, 0, bits))
    return _HOST[key]


def run(S, lay, wl, x_host, path):
    T = x_host.shape[0]
    xt = to_dev(x_host, DEV)
    if wl.x_dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    ws = S.workspace(lay, T)
    ids = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    y = S.forward(lay, xt, ws, ids=ids, w=w, path=path)
    torch.cuda.synchronize()
    assert S.device_status() == 0
    return y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("name,T", [("tiny_bf16", 16), ("tiny_bf16", 200), ("tiny_bf16", 700),
                                    ("half_ntile_bf16", 64), ("half_ntile_bf16", 333),
                                    ("wide_bf16", 257), ("shared_bf16", 40),
                                    ("shared_bf16", 300), ("shared_nogate_bf16", 150),
                                    # >= 256 rows per expert on average: items pair two
                                    # m-tiles in the gate/up GEMM
                                    ("tiny_bf16", 1100), ("half_ntile_bf16", 1030)])
def test_grouped_matches_oracle(S, name, T, bits):
    wl, hl = host_layer(name, bits)
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, T)
    y, ids, w = run(S, lay, wl, x, S.PATH_GROUPED)
    check_forward(y, ids, w, hl, x, tol=TOL)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("name,T", [("tiny_f32", 200), ("tiny_f32", 1100),
                                    ("shared_nogate_f32", 150)])
def test_fp32_tokens_stream_at_grouped_batch_sizes(S, name, T, bits):
    """Batches whose bf16 twin takes the grouped path: with fp32 tokens the
    forward streams (fp32 accumulation) and holds the fp32 bar, 1e-3."""
    wl, hl = host_layer(name, bits)
    lay = hl.device_layer(DEV)
    assert S.path_for(lay, T, torch.bfloat16) == S.PATH_GROUPED
    assert S.path_for(lay, T, torch.float32) == S.PATH_STREAM
    x, _ = wl.activations(0, T)
    y, ids, w = run(S, lay, wl, x, None)
    check_forward(y, ids, w, hl, x, tol=TOL_F32)


def test_grouped_path_refuses_fp32_tokens(S):
    """A forced grouped forward of fp32 tokens would round them to bf16: it
    is refused (SMOE_ERR_UNSUPPORTED) and enqueues nothing."""
    wl, hl = host_layer("tiny_f32", 4)
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, 200)
    xt = to_dev(x, DEV)
    ws = S.workspace(lay, 200)
    y = torch.full((200, wl.d), 7.0, dtype=torch.float32, device=DEV)
    with pytest.raises(S.SmoeError) as ei:
        S.forward(lay, xt, ws, y=y, path=S.PATH_GROUPED)
    assert ei.value.status == -2
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


def test_grouped_with_expert_bias_skew(S):
    """A selection bias that sends most tokens to a few experts: head
    segments of several m-tiles, tail segments of a handful of rows."""
    wl, hl = host_layer("half_ntile_bf16", 4)
    bias = np.zeros(wl.E, dtype=np.float32)
    bias[[3, 7]] = 4.0
    bias[11] = 2.0
    lay = hl.device_layer(DEV, expert_bias=bias)
    T = 300
    x, _ = wl.activations(0, T)
    y, ids, w = run(S, lay, wl, x, S.PATH_GROUPED)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert counts.max() > 256 and (counts[counts > 0] < 10).any()
    check_forward(y, ids, w, hl, x, expert_bias=bias, tol=TOL)


def test_grouped_agrees_with_streaming_path(S):
    """The two paths make their logits in different summation orders (tensor
    cores vs the streaming router), so ids may differ only on near-tie tokens
    and weights only in rounding."""
    wl, hl = host_layer("wide_bf16", 4)
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, 96)
    yg, idg, wg = run(S, lay, wl, x, S.PATH_GROUPED)
    ys, ids_, ws_ = run(S, lay, wl, x, S.PATH_STREAM)
    ties = set(near_tie_tokens(O.router_logits(hl.router, x), wl.k))
    same = [t for t in range(x.shape[0]) if t not in ties]
    assert np.array_equal(idg[same], ids_[same])
    assert np.allclose(wg[same], ws_[same], rtol=1e-5, atol=1e-6)
    assert float(np.abs(yg[same] - ys[same]).max()) <= TOL * float(np.abs(ys).max())


def test_grouped_is_deterministic(S):
    wl, hl = host_layer("shared_bf16", 4)
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, 100)
    y1, _, _ = run(S, lay, wl, x, S.PATH_GROUPED)
    y2, _, _ = run(S, lay, wl, x, S.PATH_GROUPED)
    assert np.array_equal(y1, y2)


def test_grouped_refuses_small_batches(S):
    wl, hl = host_layer("tiny_bf16", 4)
    lay = hl.device_layer(DEV)
    x, _ = wl.activations(0, 15)
    xt = to_dev(x, DEV).to(torch.bfloat16)
    ws = S.workspace(lay, 15)
    y = torch.full((15, wl.d), 7.0, dtype=torch.float32, device=DEV)
    with pytest.raises(S.SmoeError) as ei:
        S.forward(lay, xt, ws, y=y, path=S.PATH_GROUPED)
    assert ei.value.status == -2
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
