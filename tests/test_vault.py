""".smoe vault ingest ("".smoe Binary Format"): the oracle's writer and
reader pinned against the page's field tables and blob sizes; the library's
parser (smoe_vault_parse / smoe_vault_find_expert, host code) against the
oracle on vaults the oracle writes, including every rule the page states for
a vault to be refused; on the GPU, smoe_vault_repack_layer against
smoe_repack of the same streams (bit-exact) and a forward through those
tiles against the oracle.
"""
import os
import struct

import numpy as np
import pytest

from oracle import vault as V

HERE = os.path.dirname(os.path.abspath(__file__))
TYPE_SIZES = {"uint8": 1, "uint32": 4, "uint64": 8, "float32": 4}


def _golden():
    rows = []
    with open(os.path.join(HERE, "golden", "smoe_vault_layout.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            st, off, size, typ, name = line.split()
            rows.append((st, int(off), int(size), typ, name))
    return rows


# ------------------------------------------------------------ oracle pins

def test_oracle_struct_formats_match_the_page_tables():
    fmts = {"header": (V.HEADER_FMT, V.HEADER_FIELDS), "sarc": (V.SARC_FMT, V.SARC_FIELDS),
            "entry": (V.ENTRY_FMT, V.ENTRY_FIELDS), "desc": (V.DESC_FMT, V.DESC_FIELDS)}
    gold = _golden()
    for st, (fmt, names) in fmts.items():
        mine = V.field_layout(fmt, names)
        page = [(n, o, s) for (g, o, s, t, n) in gold if g == st]
        assert mine == page, st
        for (g, o, s, t, n) in gold:
            if g == st:
                base = t.split("[")[0]
                cnt = int(t.split("[")[1].rstrip("]")) if "[" in t else 1
                assert TYPE_SIZES.get(base, 1) * cnt == s, (st, n)
    assert [struct.calcsize(f) for f in (V.HEADER_FMT, V.ENTRY_FMT, V.DESC_FMT, V.SARC_FMT)] == \
        [64, 48, 44, 128]


@pytest.mark.parametrize("bits,blob", [(4, 10_027_008), (2, 5_308_416)])
def test_oracle_blob_of_a_qwen3_expert_is_the_page_size(bits, blob):
    """One Qwen3-235B expert (3 x 4096 x 1536) gives the page's blob sizes
    ("SMOE Quantisation", Why Quantise; ".smoe Binary Format", Expert Blob
    Architecture); both are whole 16 KB pages, so padded = raw."""
    d, f = 4096, 1536
    q = {"codes_lsb": np.zeros(V.stream_bytes(f, d, bits), np.uint8),
         "scales_f16": np.zeros(f * d // 64, np.uint16)}
    qd = {"codes_lsb": np.zeros(V.stream_bytes(d, f, bits), np.uint8),
          "scales_f16": np.zeros(d * f // 64, np.uint16)}
    buf = V.write_vault({(0, 0): (q, q, qd)}, d, f, bits)
    p = V.read_vault(buf)
    assert p["entries"][0]["raw_size"] == blob
    assert p["entries"][0]["padded_size"] == blob
    assert p["entries"][0]["byte_offset"] % 16384 == 0
    assert p["entries"][0]["num_groups"] == 3 * d * f // 64


# ------------------------------------------------------------ small vaults

def _small_experts(bits, d=256, f=128, layers=(0, 1), E=3, seed=5):
    rng = np.random.default_rng(seed)
    out = {}
    for l in layers:
        for e in range(E):
            qs = []
            for rows, cols in ((f, d), (f, d), (d, f)):
                qs.append({"codes_lsb": rng.integers(0, 256, V.stream_bytes(rows, cols, bits),
                                                     dtype=np.uint8),
                           "scales_f16": rng.integers(0, 0x7800, rows * cols // 64,
                                                      dtype=np.uint16)})
            out[(l, e)] = tuple(qs)
    return out


@pytest.fixture(scope="module")
def S():
    from bit_expert_weight_gb300 import build
    build.build()
    import bit_expert_weight_gb300.smoe as S
    S.load()
    return S


def _meta(buf):
    h = V.read_vault(buf)["header"]
    return buf[:h["data_offset"]]


@pytest.mark.parametrize("version", [1, 2])
@pytest.mark.parametrize("bits", [4, 2])
def test_library_parser_matches_the_oracle(S, version, bits):
    buf = V.write_vault(_small_experts(bits), 256, 128, bits, version=version, vocab_size=1000,
                        dense_ffn_dim=512, arch={"moe_top_k": 2, "model_type": b"tiny_moe"})
    p = V.read_vault(buf)
    info = S.vault_parse(_meta(buf), len(buf))
    h = p["header"]
    for k in ("version", "num_moe_layers", "max_experts_per_layer", "total_experts",
              "table_offset", "data_offset", "group_size", "bits", "d_model", "vocab_size",
              "ffn_dim", "reserved_ext"):
        assert getattr(info, k) == h[k], k
    assert info.has_arch == (1 if version == 2 else 0)
    if version == 2:
        a = p["arch"]
        for k in ("num_heads", "num_kv_heads", "head_dim", "moe_top_k", "moe_ffn_dim",
                  "dense_ffn_dim", "shared_expert_ffn_dim", "activation", "num_hidden_layers"):
            assert getattr(info, k) == a[k], k
        assert info.arch_flags == a["flags"]
        assert np.float32(info.rope_theta) == np.float32(a["rope_theta"])
        assert np.float32(info.rms_norm_eps) == np.float32(a["rms_norm_eps"])
        assert info.model_type == a["model_type"].rstrip(b"\0")
    for ent, ds in zip(p["entries"], p["descs"]):
        x = S.vault_find_expert(_meta(buf), len(buf), ent["layer_id"], ent["expert_id"])
        for k in ("byte_offset", "raw_size", "padded_size", "num_groups"):
            assert getattr(x, k) == ent[k], k
        for t in range(3):
            for k in ("rows", "cols", "packed_offset", "packed_size", "scales_offset",
                      "scales_size"):
                assert getattr(x.tensor[t], k) == ds[t][k], (t, k)
        # the located bytes are the streams the oracle wrote
        streams = V.expert_streams(buf, p, ent["layer_id"], ent["expert_id"])
        for t, (codes, scales) in enumerate(streams):
            off = x.byte_offset + x.tensor[t].packed_offset
            assert bytes(codes) == buf[off:off + x.tensor[t].packed_size]


def test_library_refuses_a_missing_expert(S):
    buf = V.write_vault(_small_experts(4), 256, 128, 4)
    with pytest.raises(S.SmoeError):
        S.vault_find_expert(_meta(buf), len(buf), 1, 7)


def _mutations(buf):
    """(name, mutated bytes): each breaks one rule the page states."""
    p = V.read_vault(buf)
    h = p["header"]
    n = h["total_experts"]
    ao = h["reserved_ext"]
    e0, d0 = 64, 64 + 48 * n

    def put(b, off, fmt, val):
        b = bytearray(b)
        struct.pack_into(fmt, b, off, val)
        return bytes(b)
    out = [
        ("magic", put(buf, 4, "<B", 0xDF)),
        ("version 0", put(buf, 8, "<I", 0)),
        ("version 3", put(buf, 8, "<I", 3)),
        ("table_offset", put(buf, 24, "<Q", 65)),
        ("data_offset unaligned", put(buf, 32, "<Q", h["data_offset"] + 8)),
        ("group_size", put(buf, 40, "<I", 32)),
        ("bits", put(buf, 44, "<I", 3)),
        ("total_experts past data", put(buf, 20, "<I", 10_000)),
        ("arch offset unaligned", put(buf, 60, "<I", ao + 4)),
        ("arch magic", put(buf, ao, "<B", 0x54)),
        ("arch block_version", put(buf, ao + 4, "<I", 2)),
        ("arch block_size", put(buf, ao + 8, "<I", 64)),
        ("arch activation", put(buf, ao + 48, "<I", 1)),
        ("arch moe_top_k", put(buf, ao + 32, "<I", 17)),
        ("arch head_dim", put(buf, ao + 28, "<I", 257)),
        ("arch head divisibility", put(buf, ao + 20, "<I", 63)),
        ("arch reserved", put(buf, ao + 100, "<B", 1)),
        ("table order", put(buf, e0 + 48 + 4, "<I", 0)),
        ("entry group_size", put(buf, e0 + 32, "<I", 128)),
        ("entry reserved", put(buf, e0 + 45, "<B", 1)),
        ("entry offset unaligned", put(buf, e0 + 8, "<Q", p["entries"][0]["byte_offset"] + 16)),
        ("entry raw > padded", put(buf, e0 + 16, "<Q", p["entries"][0]["padded_size"] + 16)),
        ("entry past the file", put(buf, e0 + 24, "<Q", (len(buf) + 16383) // 16384 * 16384)),
        ("entry num_groups", put(buf, e0 + 36, "<Q", p["entries"][0]["num_groups"] + 1)),
        ("descriptor type", put(buf, d0, "<B", 1)),
        ("descriptor ndim", put(buf, d0 + 1, "<B", 3)),
        ("descriptor reserved", put(buf, d0 + 2, "<B", 1)),
        ("descriptor packed_size", put(buf, d0 + 20, "<Q", p["descs"][0][0]["packed_size"] + 1)),
        ("descriptor scales past raw", put(buf, d0 + 28, "<Q", p["entries"][0]["raw_size"])),
    ]
    return out


def test_library_refuses_what_the_oracle_refuses(S):
    buf = V.write_vault(_small_experts(4), 256, 128, 4, version=2)
    assert V.read_vault(buf)
    L = S.load()
    import ctypes
    for name, bad in _mutations(buf):
        with pytest.raises(V.VaultError):
            V.read_vault(bad)
        meta = bad[:V.read_vault(buf)["header"]["data_offset"]]
        cb = ctypes.create_string_buffer(meta, len(meta))
        info = S.VaultInfo()
        assert L.smoe_vault_parse(cb, len(meta), len(bad), ctypes.byref(info)) == -1, name
    # short metadata and a file that ends before the blobs
    meta = _meta(buf)
    info = S.VaultInfo()
    cb = ctypes.create_string_buffer(meta, len(meta))
    assert L.smoe_vault_parse(cb, 63, len(buf), ctypes.byref(info)) == -1
    assert L.smoe_vault_parse(cb, len(meta) - 16, len(buf), ctypes.byref(info)) == -1
    assert L.smoe_vault_parse(cb, len(meta), len(buf) - 16384, ctypes.byref(info)) == -1


# ------------------------------------------------------------ GPU

@pytest.mark.gpu
@pytest.mark.parametrize("bits", [4, 2])
def test_vault_repack_matches_repack_and_forward(bits):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_expert_weight_gb300 import build
    from bit_expert_weight_gb300 import synth as Y
    build.build()
    import bit_expert_weight_gb300.smoe as S
    from helpers import HostLayer, check_forward, to_dev, to_dev_bf16
    dev = "cuda:0"
    wl = Y.Workload("vault_tiny", 256, 128, 8, 2, True, [bits], [4], 1, 17, x_dtype="f32",
                    p_zero=0.2)
    hl = HostLayer(wl, 0, bits)
    other = _small_experts(bits, layers=(0,), E=2, seed=9)  # another layer before it
    experts = {(1, e): tuple(hl.q[e]) for e in range(wl.E)}
    experts.update(other)
    buf = V.write_vault(experts, wl.d, wl.f, bits, arch={"moe_top_k": 2})
    vd = torch.from_numpy(np.frombuffer(buf, np.uint8).copy()).to(dev)
    tiles = S.vault_repack_layer(_meta(buf), vd, 1, wl.E, wl.d, wl.f, bits)
    codes = [to_dev(q["codes_lsb"], dev) for e in range(wl.E) for q in hl.q[e]]
    scales = [to_dev(q["scales_f16"].view(np.int16), dev) for e in range(wl.E) for q in hl.q[e]]
    ref = S.repack(codes, scales, wl.d, wl.f, wl.E, bits)
    torch.cuda.synchronize()
    assert torch.equal(tiles, ref)
    lay = S.MoELayer(wl.d, wl.f, wl.E, wl.k, wl.norm, bits, to_dev_bf16(hl.router, dev), tiles)
    x, _ = wl.activations(0, 4)
    xt = to_dev(x, dev)
    ws = S.workspace(lay, 4)
    ids = torch.empty((4, wl.k), dtype=torch.int32, device=dev)
    w = torch.empty((4, wl.k), dtype=torch.float32, device=dev)
    y = S.forward(lay, xt, ws, ids=ids, w=w)
    torch.cuda.synchronize()
    assert S.device_status() == 0
    check_forward(y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), hl, x)
