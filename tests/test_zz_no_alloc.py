"""smoe_moe_forward_noalloc: the forward with the library's built-in device
workspace.  Its y, ids and weights must equal smoe_moe_forward's (own
workspace) bit for bit -- both forwards are deterministic -- on two calls in
a row, also when consecutive calls change the layer shape and the path
(streaming cases, then a batch that takes the grouped tensor-core path in
the same array), and it must refuse, and enqueue nothing for, a batch whose
workspace is larger than the built-in one.

Collected last on purpose: it must pass both in a fresh process and after
every other test has used the device.
"""
import ctypes
import os
import re
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_expert_weight_gb300 import synth as Y  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEV = "cuda:0"


# ------------------------------------------------------------ host side (CPU)

@pytest.fixture(scope="module")
def lib():
    from bit_expert_weight_gb300 import build
    build.build()
    import bit_expert_weight_gb300.smoe as S
    return S, S.load()


def test_scratch_size_constant_matches_header():
    import bit_expert_weight_gb300.smoe as S
    text = open(os.path.join(ROOT, "include", "smoe.h")).read()
    m = re.search(r"#define\s+SMOE_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "SMOE_NOALLOC_SCRATCH_BYTES not found"
    assert int(m.group(1)) << int(m.group(2)) == S.NOALLOC_SCRATCH_BYTES
    assert S.NOALLOC_SCRATCH_BYTES % 256 == 0


def test_noalloc_rejects_bad_args_on_host(lib):
    S, L = lib
    P = ctypes.c_void_p
    desc = S.LayerDesc(d_model=256, ffn_dim=128, num_experts=8, top_k=2, norm_topk_prob=1,
                       bits=4, group_size=64, router_w=256, expert_bias=None, expert_tiles=512,
                       shared_tiles=None, shared_ffn_dim=0, shared_gate_w=None)
    bad = S.LayerDesc(d_model=192, ffn_dim=128, num_experts=8, top_k=2, norm_topk_prob=1,
                      bits=4, group_size=64, router_w=256, expert_bias=None, expert_tiles=512,
                      shared_tiles=None, shared_ffn_dim=0, shared_gate_w=None)
    f = L.smoe_moe_forward_noalloc
    assert f(ctypes.byref(bad), P(4096), 0, 4, P(8192), None, None, None) == -1
    assert f(None, P(4096), 0, 4, P(8192), None, None, None) == -1
    assert f(ctypes.byref(desc), P(4096), 0, -1, P(8192), None, None, None) == -1
    assert f(ctypes.byref(desc), P(4096), 7, 4, P(8192), None, None, None) == -1    # dtype
    assert f(ctypes.byref(desc), None, 0, 4, P(8192), None, None, None) == -1       # null x
    assert f(ctypes.byref(desc), P(4096), 0, 4, None, None, None, None) == -1       # null y
    assert f(ctypes.byref(desc), P(4104), 0, 4, P(8192), None, None, None) == -1    # align
    assert f(ctypes.byref(desc), None, 0, 0, None, None, None, None) == 0           # T = 0


# ------------------------------------------------------------- device (GPU)

# name: (d, f, E, k, norm, x_dtype, shared_f, shared_gate, bits, T)
CASES = [
    ("tiny_f32_q4_T3", (256, 128, 8, 2, True, "f32", 0, False, 4, 3)),
    ("shared_bf16_q2_T8", (256, 128, 24, 8, True, "bf16", 192, True, 2, 8)),
    ("wide_bf16_q4_T1", (512, 128, 32, 6, True, "bf16", 0, False, 4, 1)),
    ("small_bf16_q4_T13", (256, 192, 16, 4, False, "bf16", 0, False, 4, 13)),
    # T * k >= 16 * E: the grouped path, after streaming calls of other shapes
    ("tiny_bf16_q4_T64", (256, 128, 8, 2, True, "bf16", 0, False, 4, 64)),
]


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_expert_weight_gb300 import build
    build.build()
    import bit_expert_weight_gb300.smoe as S
    S.load()
    return S


def _device_layer(S, name, spec):
    """Seeded layer, quantised and repacked on the device (no oracle involved:
    the reference here is the library's own smoe_moe_forward)."""
    d, f, E, k, norm, xd, sf, sg, bits, T = spec
    seed = zlib.crc32(name.encode()) & 0xFFFF
    wl = Y.Workload(name, d, f, E, k, norm, [bits], [T], 1, seed, x_dtype=xd, shared_f=sf,
                    shared_gate=sg)

    def tiles_for(expert_ids, ff):
        codes, scales = [], []
        for e in expert_ids:
            for role in (Y.ROLE_GATE, Y.ROLE_UP, Y.ROLE_DOWN):
                w = torch.from_numpy(wl.expert_weight(0, e, role).view(np.int16)).to(DEV)
                c, s = S.quantize(w.view(torch.bfloat16), bits)
                codes.append(c)
                scales.append(s)
        return S.repack(codes, scales, d, ff, len(expert_ids), bits)

    tiles = tiles_for(range(E), f)
    sh_tiles = tiles_for([Y.SHARED_EXPERT], sf) if sf else None
    sh_gate = None
    if sf and sg:
        sh_gate = torch.from_numpy(wl.shared_gate_weight(0).view(np.int16)).to(DEV).view(
            torch.bfloat16)
    router = torch.from_numpy(wl.router_weight(0).view(np.int16)).to(DEV).view(torch.bfloat16)
    lay = S.MoELayer(d, f, E, k, norm, bits, router, tiles, shared_tiles=sh_tiles, shared_f=sf,
                     shared_gate_w=sh_gate)
    x, _ = wl.activations(0, T)
    xt = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    if xd == "bf16":
        xt = xt.to(torch.bfloat16)
    return lay, xt, k


@pytest.mark.gpu
def test_noalloc_matches_forward_on_consecutive_calls(S):
    prepared = [(name, *_device_layer(S, name, spec)) for name, spec in CASES]
    for name, lay, xt, k in prepared:
        assert lay.workspace_bytes(xt.shape[0]) <= S.NOALLOC_SCRATCH_BYTES, name
    assert S.path_for(prepared[-1][1], prepared[-1][2].shape[0]) == S.PATH_GROUPED
    assert all(S.path_for(lay, xt.shape[0]) == S.PATH_STREAM for _, lay, xt, _ in prepared[:-1])
    # reference outputs through smoe_moe_forward with caller-owned workspaces
    refs = {}
    for name, lay, xt, k in prepared:
        T = xt.shape[0]
        ws = S.workspace(lay, T)
        ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        y = S.forward(lay, xt, ws, ids=ids, w=w)
        torch.cuda.synchronize()
        refs[name] = (y.clone(), ids.clone(), w.clone())
    assert S.device_status() == 0
    # two calls in a row per case; consecutive cases change the layer shape
    for name, lay, xt, k in prepared:
        T = xt.shape[0]
        y_ref, ids_ref, w_ref = refs[name]
        for call in range(2):
            ids = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
            w = torch.full((T, k), float("nan"), dtype=torch.float32, device=DEV)
            y = torch.full((T, lay.d), float("nan"), dtype=torch.float32, device=DEV)
            S.forward_noalloc(lay, xt, y=y, ids=ids, w=w)
            torch.cuda.synchronize()
            assert S.device_status() == 0, (name, call)
            assert torch.equal(ids, ids_ref), (name, call)
            assert torch.equal(w, w_ref), (name, call)
            assert torch.equal(y, y_ref), (name, call)


@pytest.mark.gpu
def test_noalloc_refuses_oversized_batch_and_enqueues_nothing(S):
    name, spec = CASES[0]
    lay, _, k = _device_layer(S, name, spec)
    T = 1024
    while lay.workspace_bytes(T) <= S.NOALLOC_SCRATCH_BYTES:
        T *= 2
    x = torch.zeros((T, lay.d), dtype=torch.float32, device=DEV)
    y = torch.full((T, lay.d), 3.0, dtype=torch.float32, device=DEV)
    with pytest.raises(S.SmoeError) as ei:
        S.forward_noalloc(lay, x, y=y)
    assert ei.value.status == -3
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
    assert S.device_status() == 0
