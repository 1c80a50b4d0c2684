"""Failure detection on the GPU, without a GPU fault.

(a) A bounded wait that runs out: smoe_debug_set_waits makes the layer
    kernel's routing step wait for logits that no CTA writes, with a short
    bound.  The launch must end by itself, the host must read
    SMOE_ERR_TIMEOUT from the device status word, the context must stay
    usable, and the next forward -- on the same workspace, and on a
    re-initialised one -- must give the undisturbed result bit for bit.
(b) Host input the kernels reject on the device: a NaN in a token makes NaN
    logits, which the routing code of every path records as
    SMOE_ERR_DEVICE_FAULT (no trap); the status is read once and cleared,
    and the following forward is clean.
"""
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_expert_weight_gb300 import synth as Y  # noqa: E402

from helpers import HostLayer, check_forward, to_dev  # noqa: E402

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
    yield S
    S.debug_set_waits()


@pytest.fixture(scope="module")
def layer():
    name = "failure_bf16"
    seed = zlib.crc32(name.encode()) & 0xFFFF
    wl = Y.Workload(name, 256, 128, 16, 4, True, [4], [1], 1, seed, x_dtype="bf16",
                    shared_f=128, shared_gate=True)
    return wl, HostLayer(wl, 0, 4)


def _x(wl, T, nan_token=None):
    x, _ = wl.activations(0, T)
    x = x.copy()
    if nan_token is not None:
        x[nan_token, 17] = np.nan
    return to_dev(x, DEV).to(torch.bfloat16), x


def _run(S, lay, wl, xt, ws, path=None):
    T = xt.shape[0]
    ids = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    y = S.forward(lay, xt, ws, ids=ids, w=w, path=path)
    return y, ids, w


@pytest.mark.parametrize("T", [1, 5])
def test_routing_wait_runs_out_and_reports_timeout(S, layer, T):
    wl, hl = layer
    lay = hl.device_layer(DEV)
    xt, x = _x(wl, T)
    ws = S.workspace(lay, T)
    y_ref, ids_ref, w_ref = _run(S, lay, wl, xt, ws)
    torch.cuda.synchronize()
    assert S.device_status() == 0
    check_forward(y_ref.cpu().numpy(), ids_ref.cpu().numpy(), w_ref.cpu().numpy(), hl, x)
    S.debug_set_waits(100_000, stall_routing=True)  # ~50 us at 2 GHz
    try:
        y_bad = torch.full((T, wl.d), 5.0, dtype=torch.float32, device=DEV)
        S.forward(lay, xt, ws, y=y_bad)
        torch.cuda.synchronize()           # the launch ends by itself
        assert S.device_status() == -6     # SMOE_ERR_TIMEOUT, read once ...
        assert S.device_status() == 0      # ... and cleared
        assert bool((y_bad == 5.0).all())  # the skipped layer wrote nothing
    finally:
        S.debug_set_waits()
    # the context and the workspace are still good: the same bits as before
    for reinit in (False, True):
        if reinit:
            ws = S.workspace(lay, T)
        y2, ids2, w2 = _run(S, lay, wl, xt, ws)
        torch.cuda.synchronize()
        assert S.device_status() == 0
        assert torch.equal(y2, y_ref) and torch.equal(ids2, ids_ref) and torch.equal(w2, w_ref)


@pytest.mark.parametrize("T,path", [(3, None),      # fused layer kernel (routing inside)
                                    (12, None),     # router kernel, layer kernel, combine
                                    (64, "grouped")])  # tensor-core logits + tile routing
def test_nan_token_is_reported_as_device_fault(S, layer, T, path):
    wl, hl = layer
    lay = hl.device_layer(DEV)
    p = S.PATH_GROUPED if path == "grouped" else None
    xt, _ = _x(wl, T, nan_token=T // 2)
    ws = S.workspace(lay, T)
    _run(S, lay, wl, xt, ws, path=p)
    torch.cuda.synchronize()
    assert S.device_status() == -5   # SMOE_ERR_DEVICE_FAULT
    assert S.device_status() == 0
    xc, x = _x(wl, T)
    y, ids, w = _run(S, lay, wl, xc, ws, path=p)
    torch.cuda.synchronize()
    assert S.device_status() == 0
    check_forward(y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), hl, x,
                  tol=2e-2 if path == "grouped" else 1e-3)
