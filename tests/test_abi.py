"""The C-ABI library loads, exports every symbol the headers declare, and its
host-side validation rejects bad arguments without launching anything (these
run without a GPU: validation happens before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libs():
    from bit_expert_weight_gb300 import build
    paths = build.build()
    import bit_expert_weight_gb300.smoe as S
    return S, paths


def declared(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(smoe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(libs):
    S, paths = libs
    for header, lib in (("smoe.h", "libsmoe.so"), ("smoe_synth.h", "libsmoe_synth.so")):
        names = declared(header)
        assert names, header
        so = ctypes.CDLL(paths[lib])
        for n in names:
            assert hasattr(so, n), f"{lib} does not export {n}"
    assert sorted(S.EXPORTED) == declared("smoe.h")


def test_size_queries_match_the_pages_blob_layout(libs):
    S, _ = libs
    assert S.stream_bytes(4096, 1536, 4) == 3_145_728
    assert S.stream_bytes(4096, 1536, 2) == 1_572_864
    assert S.scales_bytes(4096, 1536) == 196_608
    # one Qwen3-235B-like expert: the tile layout is exactly as large as the blob
    assert S.expert_tiles_bytes(4096, 1536, 4) == 10_027_008
    assert S.expert_tiles_bytes(4096, 1536, 2) == 5_308_416
    assert S.repacked_bytes(2048, 1408, 64, 4) == 64 * 4_595_712
    assert S.expert_tiles_bytes(4096, 1500, 4) == 0   # f % 64
    assert S.expert_tiles_bytes(4000, 1536, 4) == 0   # d % 128
    assert S.expert_tiles_bytes(4096, 1536, 3) == 0   # bits
    assert S.stream_bytes(4, 64, 8) == 0


def test_status_strings(libs):
    S, _ = libs
    L = S.load()
    for code in range(-6, 1):
        assert L.smoe_status_string(code)


def _desc(S, **kw):
    base = dict(d_model=256, ffn_dim=128, num_experts=8, top_k=2, norm_topk_prob=1, bits=4,
                group_size=64, router_w=256, expert_bias=None, expert_tiles=512,
                shared_tiles=None, shared_ffn_dim=0, shared_gate_w=None)
    base.update(kw)
    return S.LayerDesc(**base)


BAD = [
    dict(bits=3), dict(bits=8), dict(group_size=32), dict(group_size=128),
    dict(top_k=0), dict(top_k=17), dict(top_k=9), dict(num_experts=0), dict(num_experts=300),
    dict(d_model=192), dict(ffn_dim=100), dict(d_model=0), dict(router_w=None),
    dict(d_model=4224), dict(ffn_dim=2112), dict(shared_ffn_dim=2112, shared_tiles=1024),
    dict(expert_tiles=None), dict(expert_tiles=520), dict(shared_ffn_dim=64),
    dict(shared_tiles=1024), dict(shared_ffn_dim=-64, shared_tiles=1024),
]


@pytest.mark.parametrize("kw", BAD, ids=[",".join(f"{k}={v}" for k, v in b.items()) for b in BAD])
def test_forward_rejects_bad_layer(libs, kw):
    S, _ = libs
    L = S.load()
    desc = _desc(S, **kw)
    rc = L.smoe_moe_forward(ctypes.byref(desc), ctypes.c_void_p(4096), 0, 4,
                            ctypes.c_void_p(8192), ctypes.c_void_p(1 << 20), 1 << 30, None, None,
                            None)
    assert rc == -1
    assert L.smoe_moe_workspace_bytes(ctypes.byref(desc), 4) == 0


def test_forward_rejects_bad_call_args(libs):
    S, _ = libs
    L = S.load()
    desc = _desc(S)
    P = ctypes.c_void_p
    # negative T, bad dtype, null x / y / workspace, misaligned workspace
    assert L.smoe_moe_forward(ctypes.byref(desc), P(4096), 0, -1, P(8192), P(1 << 20), 1 << 30,
                              None, None, None) == -1
    assert L.smoe_moe_forward(ctypes.byref(desc), P(4096), 7, 4, P(8192), P(1 << 20), 1 << 30,
                              None, None, None) == -1
    assert L.smoe_moe_forward(ctypes.byref(desc), None, 0, 4, P(8192), P(1 << 20), 1 << 30,
                              None, None, None) == -1
    assert L.smoe_moe_forward(ctypes.byref(desc), P(4096), 0, 4, None, P(1 << 20), 1 << 30,
                              None, None, None) == -1
    assert L.smoe_moe_forward(ctypes.byref(desc), P(4096), 0, 4, P(8192), None, 1 << 30,
                              None, None, None) == -1
    assert L.smoe_moe_forward(ctypes.byref(desc), P(4096), 0, 4, P(8192), P((1 << 20) + 16),
                              1 << 30, None, None, None) == -1
    assert L.smoe_moe_forward(None, P(4096), 0, 4, P(8192), P(1 << 20), 1 << 30,
                              None, None, None) == -1
    # zero tokens is a no-op
    assert L.smoe_moe_forward(ctypes.byref(desc), None, 0, 0, None, None, 0, None, None,
                              None) == 0


def test_other_entry_points_reject_bad_args(libs):
    S, _ = libs
    L = S.load()
    P = ctypes.c_void_p
    assert L.smoe_quantize(P(4096), 4, 96, 4, 64, P(8192), P(16384), None) == -1   # cols % 64
    assert L.smoe_quantize(P(4096), 4, 64, 3, 64, P(8192), P(16384), None) == -1   # bits
    assert L.smoe_quantize(P(4096), 4, 64, 4, 32, P(8192), P(16384), None) == -1   # group
    assert L.smoe_quantize(None, 4, 64, 4, 64, P(8192), P(16384), None) == -1
    assert L.smoe_quantize(P(4096), -1, 64, 4, 64, P(8192), P(16384), None) == -1
    assert L.smoe_quantize(P(4096), 0, 64, 4, 64, None, None, None) == 0          # empty
    for k, E in ((0, 8), (17, 32), (9, 8)):
        assert L.smoe_route_from_logits(P(4096), 4, E, k, 1, None, P(8192), P(16384),
                                        None) == -1
    assert L.smoe_route_from_logits(None, 4, 8, 2, 1, None, P(8192), P(16384), None) == -1
    assert L.smoe_route_from_logits(P(4096), 0, 8, 2, 1, None, None, None, None) == 0
    arr = (P * 3)(4096, 4096, 4096)
    assert L.smoe_repack(arr, arr, 192, 128, 1, 4, 64, P(4096), 1 << 20, None) == -1
    assert L.smoe_repack(arr, arr, 256, 100, 1, 4, 64, P(4096), 1 << 20, None) == -1
    assert L.smoe_repack(arr, arr, 256, 128, 1, 4, 64, P(4096), 16, None) == -3   # too small
    assert L.smoe_repack(arr, arr, 256, 128, 1, 4, 64, P(4100), 1 << 20, None) == -1  # align
    assert L.smoe_unpack(P(4096), 256, 128, 1, 5, 64, arr, arr, None) == -1


def test_path_selection_and_path_argument(libs):
    """smoe_moe_path: the streaming path below 16 tokens or below 16 routed
    rows per expert on average, the grouped path from there on (bf16 tokens;
    fp32 tokens always stream); an unknown path is refused before anything
    else."""
    S, _ = libs
    L = S.load()
    P = ctypes.c_void_p
    desc = _desc(S)  # E = 8, k = 2
    assert L.smoe_moe_path(ctypes.byref(desc), 1) == S.PATH_STREAM
    assert L.smoe_moe_path(ctypes.byref(desc), 15) == S.PATH_STREAM
    assert L.smoe_moe_path(ctypes.byref(desc), 63) == S.PATH_STREAM     # 126 < 128 rows
    assert L.smoe_moe_path(ctypes.byref(desc), 64) == S.PATH_GROUPED    # 128 rows
    assert L.smoe_moe_path(ctypes.byref(desc), -1) == -1
    assert L.smoe_moe_path(ctypes.byref(_desc(S, bits=3)), 64) == -1
    # fp32 tokens always stream (the tensor-core path would round them)
    for T in (1, 64, 4096):
        assert L.smoe_moe_path_dtype(ctypes.byref(desc), T, S.SMOE_F32) == S.PATH_STREAM
        assert (L.smoe_moe_path_dtype(ctypes.byref(desc), T, S.SMOE_BF16) ==
                L.smoe_moe_path(ctypes.byref(desc), T))
    assert L.smoe_moe_path_dtype(ctypes.byref(desc), 64, 5) == -1
    for bad_path in (-1, 3, 7):
        assert L.smoe_moe_forward_path(ctypes.byref(desc), P(4096), 0, 64, P(8192), P(1 << 20),
                                       1 << 30, None, None, bad_path, None) == -1
    # the workspace makes room for the sorted rows from 16 tokens on
    w15 = L.smoe_moe_workspace_bytes(ctypes.byref(desc), 15)
    w16 = L.smoe_moe_workspace_bytes(ctypes.byref(desc), 16)
    rows16 = 16 * 2 + 8 * 127
    # per sorted row: bf16 token (d), bf16 h (f), bf16 weighted output (d), its weight
    assert w16 - w15 >= rows16 * (256 * 2 + 128 * 2 + 256 * 2 + 4)


def test_router_options_are_validated_on_the_host(libs):
    """smoe_router_opts: the routed scaling factor must be finite and > 0
    (refused before anything is launched)."""
    S, _ = libs
    L = S.load()
    P = ctypes.c_void_p
    desc = _desc(S)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        o = S.RouterOpts(0, bad)
        assert L.smoe_moe_forward_ex(ctypes.byref(desc), ctypes.byref(o), P(4096), 0, 4, P(8192),
                                     P(1 << 20), 1 << 30, None, None, 0, None) == -1
        assert L.smoe_route_from_logits_ex(P(4096), 4, 8, 2, 1, None, ctypes.byref(o), P(8192),
                                           P(16384), None) == -1
    o = S.RouterOpts(1, 2.5)
    assert L.smoe_moe_forward_ex(ctypes.byref(desc), ctypes.byref(o), P(4096), 0, 4, P(8192),
                                 P(1 << 20), 1 << 30, None, None, 9, None) == -1   # bad path
    assert L.smoe_route_from_logits_ex(P(4096), 0, 8, 2, 1, None, ctypes.byref(o), None, None,
                                       None) == 0                                  # T = 0


def test_routing_mask_is_validated_on_the_host(libs):
    """An expert mask with a tail bit beyond E, or fewer routable experts
    than top_k, is refused before anything is launched."""
    S, _ = libs
    L = S.load()
    P = ctypes.c_void_p
    desc = _desc(S)  # E = 8, k = 2
    o = S._opts(False, 1.0, bytes([0b00000001]))  # one routable expert, k = 2
    assert L.smoe_moe_forward_ex(ctypes.byref(desc), ctypes.byref(o), P(4096), 0, 4, P(8192),
                                 P(1 << 20), 1 << 30, None, None, 0, None) == -1
    assert L.smoe_route_from_logits_ex(P(4096), 4, 8, 2, 1, None, ctypes.byref(o), P(8192),
                                       P(16384), None) == -1
    # E = 10: two bytes, bits 10..15 of the second are tail bits
    o = S._opts(False, 1.0, bytes([0b00000011, 0b00000100]))
    assert L.smoe_route_from_logits_ex(P(4096), 4, 10, 2, 1, None, ctypes.byref(o), P(8192),
                                       P(16384), None) == -1
    o = S._opts(False, 1.0, bytes([0b00000011, 0b00000010]))  # bit 9: valid (3 routable)
    assert L.smoe_route_from_logits_ex(P(4096), 0, 10, 2, 1, None, ctypes.byref(o), None, None,
                                       None) == 0


def test_mixed_depth_entry_points_validate_on_the_host(libs):
    """Per-expert depths: sizes are the sum of each expert's own size; a
    depth that is not 2 or 4, or no depth array, is refused before anything
    is launched; the mixed forward's workspace holds the grouped buffers at
    every token count."""
    S, _ = libs
    L = S.load()
    P = ctypes.c_void_p
    q4, q2 = S.expert_tiles_bytes(256, 128, 4), S.expert_tiles_bytes(256, 128, 2)
    assert S.repacked_bytes_mixed(256, 128, [4, 2, 2, 4, 2]) == 2 * q4 + 3 * q2
    assert S.repacked_bytes_mixed(256, 128, [4] * 3) == S.repacked_bytes(256, 128, 3, 4)
    assert S.repacked_bytes_mixed(256, 128, [4, 3]) == 0
    assert S.repacked_bytes_mixed(192, 128, [4, 2]) == 0
    assert L.smoe_repacked_bytes_mixed(256, 128, 2, None, 64) == 0
    desc = _desc(S)  # E = 8, k = 2
    good = S._bits_array([4, 2] * 4)
    bad = S._bits_array([4, 2, 2, 4, 8, 2, 4, 4])
    arr = (P * 24)(*([4096] * 24))
    assert L.smoe_repack_mixed(arr, arr, 256, 128, 8, bad, 64, P(4096), 1 << 20, None) == -1
    assert L.smoe_repack_mixed(arr, arr, 256, 128, 8, None, 64, P(4096), 1 << 20, None) == -1
    assert L.smoe_repack_mixed(arr, arr, 256, 128, 8, good, 64, P(4096), 16, None) == -3
    assert L.smoe_repack_mixed(arr, arr, 256, 128, 8, good, 64, P(4100), 1 << 20, None) == -1
    assert L.smoe_unpack_mixed(P(4096), 256, 128, 8, bad, 64, arr, arr, None) == -1
    for eb in (bad, None):
        assert L.smoe_moe_forward_mixed(ctypes.byref(desc), eb, None, P(4096), 0, 4, P(8192),
                                        P(1 << 20), 1 << 30, None, None, 0, None) == -1
        assert L.smoe_moe_forward_stage_mixed(ctypes.byref(desc), eb, P(4096), 0, 4, P(8192),
                                              P(1 << 20), 1 << 30, None, None, 0, None) == -1
    assert L.smoe_moe_forward_stage_mixed(ctypes.byref(desc), good, P(4096), 0, 4, P(8192),
                                          P(1 << 20), 1 << 30, None, None, 3, None) == -1
    assert L.smoe_moe_forward_mixed(ctypes.byref(desc), good, None, None, 0, 0, None, None, 0,
                                    None, None, 0, None) == 0                   # T = 0
    assert L.smoe_moe_forward_mixed(ctypes.byref(desc), good, None, P(4096), 0, 4, P(8192),
                                    P(1 << 20), 1 << 30, None, None, 5, None) == -1  # bad path
    w1 = L.smoe_moe_workspace_bytes_mixed(ctypes.byref(desc), 1)
    assert w1 > L.smoe_moe_workspace_bytes(ctypes.byref(desc), 1)
    assert w1 >= 128 * (256 * 2 + 128 * 2 + 256 * 2 + 4)  # one padded 128-row tile per segment
    assert L.smoe_moe_workspace_bytes_mixed(ctypes.byref(desc), 64) == \
        L.smoe_moe_workspace_bytes(ctypes.byref(desc), 64)


def test_binding_refuses_mixed_layers_where_the_abi_has_no_depths(libs):
    """The built-in-workspace entry point takes single-depth layers only; the
    binding says so before any call."""
    S, _ = libs
    torch = pytest.importorskip("torch")
    t = torch.zeros(256 * 8, dtype=torch.int16)  # never read: the binding refuses first
    lay = S.MoELayer(256, 128, 8, 2, True, 4, t, t, expert_bits=[4, 2] * 4)
    assert lay.expert_bits == [4, 2, 4, 2, 4, 2, 4, 2]
    with pytest.raises(ValueError):
        S.forward_noalloc(lay, t)
