"""CPU oracle for the `.smoe` vault -- TEST INFRASTRUCTURE ONLY.

Writer and reader of the pages' binary vault (".smoe Binary Format": File
Header, Arch Block "SARC", Expert Table Entry, Tensor Descriptor, Expert Blob
Architecture), written from the page's field tables with Python's `struct`
module.  It shares nothing with the library's parser (csrc/vault.cu); the
tests compare the two on vaults written here and pin these formats against
the page's tables (tests/golden/smoe_vault_layout.txt).

Only ``tests/`` may import this module.
"""
from __future__ import annotations

import struct

import numpy as np

# "File Header -- 64 bytes": magic[8], version, num_moe_layers,
# max_experts_per_layer, total_experts, table_offset (u64), data_offset (u64),
# group_size, bits, d_model, vocab_size, ffn_dim, reserved_ext.
HEADER_FMT = "<8sIIIIQQIIIIII"
# "Arch Block SARC -- 128 bytes": magic[4], block_version, block_size, flags,
# rope_theta (f32), num_heads, num_kv_heads, head_dim, moe_top_k, moe_ffn_dim,
# dense_ffn_dim, shared_expert_ffn_dim, activation, num_hidden_layers,
# rms_norm_eps (f32), model_type char[24], reserved[44].
SARC_FMT = "<4sIIIfIIIIIIIIIf24s44s"
# "Expert Table Entry -- 48 bytes": layer_id, expert_id, byte_offset,
# raw_size, padded_size (u64), group_size, num_groups (u64 at offset 36, so
# the entry is packed), reserved[4].
ENTRY_FMT = "<IIQQQIQ4s"
# "Tensor Descriptor -- 44 bytes": tensor_type (u8), ndim (u8),
# reserved_0[2], rows, cols, packed_offset, packed_size, scales_offset,
# scales_size (u64, from offset 12: packed).
DESC_FMT = "<BB2sIIQQQQ"

HEADER_MAGIC = bytes([0x53, 0x4D, 0x4F, 0x45, 0xDE, 0xEA, 0x00, 0x01])
SARC_MAGIC = b"SARC"
PAGE = 16384  # blob and data_offset alignment ("Immutable Encoding")

HEADER_FIELDS = ["magic", "version", "num_moe_layers", "max_experts_per_layer", "total_experts",
                 "table_offset", "data_offset", "group_size", "bits", "d_model", "vocab_size",
                 "ffn_dim", "reserved_ext"]
SARC_FIELDS = ["magic", "block_version", "block_size", "flags", "rope_theta", "num_heads",
               "num_kv_heads", "head_dim", "moe_top_k", "moe_ffn_dim", "dense_ffn_dim",
               "shared_expert_ffn_dim", "activation", "num_hidden_layers", "rms_norm_eps",
               "model_type", "reserved"]
ENTRY_FIELDS = ["layer_id", "expert_id", "byte_offset", "raw_size", "padded_size", "group_size",
                "num_groups", "reserved"]
DESC_FIELDS = ["tensor_type", "ndim", "reserved_0", "rows", "cols", "packed_offset", "packed_size",
               "scales_offset", "scales_size"]


def field_layout(fmt: str, names: list[str]) -> list[tuple[str, int, int]]:
    """(name, offset, size) of every field of a little-endian struct format."""
    out, off = [], 0
    for name, code in zip(names, _codes(fmt)):
        size = struct.calcsize("<" + code)
        out.append((name, off, size))
        off += size
    return out


def _codes(fmt: str) -> list[str]:
    body, out, num = fmt[1:], [], ""
    for ch in body:
        if ch.isdigit():
            num += ch
        else:
            out.append(num + ch)
            num = ""
    # a count without 's' repeats the code (not used by these formats)
    return out


def _align(v: int, a: int) -> int:
    return (v + a - 1) // a * a


def stream_bytes(rows: int, cols: int, bits: int) -> int:
    """ceil(rows * cols * bits / 8) ("Expert Blob Architecture")."""
    return (rows * cols * bits + 7) // 8


def scale_bytes(rows: int, cols: int, group: int = 64) -> int:
    """ceil(rows * cols / group_size) * 2 ("Expert Blob Architecture")."""
    return (rows * cols + group - 1) // group * 2


def write_vault(experts, d_model: int, ffn_dim: int, bits: int, *, version: int = 2,
                num_layers: int | None = None, vocab_size: int = 151936, dense_ffn_dim: int = 0,
                arch: dict | None = None) -> bytes:
    """A vault holding `experts`: {(layer, expert): (q_gate, q_up, q_down)}
    with each q = {"codes_lsb": uint8 array, "scales_f16": uint16 array} (the
    oracle quantiser's output).  Gate/up are [ffn_dim, d_model], down
    [d_model, ffn_dim].  Table sorted by layer then expert; blobs 16 KB
    aligned; v2 writes the arch block right after the descriptors (64-byte
    aligned)."""
    keys = sorted(experts)
    n = len(keys)
    layers = sorted({k[0] for k in keys})
    per_layer = {}
    for l, e in keys:
        per_layer[l] = per_layer.get(l, 0) + 1
    table_off = 64
    desc_off = table_off + n * 48
    end_desc = desc_off + n * 3 * 44
    arch_off = _align(end_desc, 64) if version >= 2 else 0
    data_off = _align((arch_off + 128) if version >= 2 else end_desc, PAGE)
    shapes = [(ffn_dim, d_model), (ffn_dim, d_model), (d_model, ffn_dim)]
    blobs, entries, descs = [], [], []
    off = data_off
    for (l, e) in keys:
        parts, tdesc, pos = [], [], 0
        for t, (q, (rows, cols)) in enumerate(zip(experts[(l, e)], shapes)):
            codes = np.ascontiguousarray(q["codes_lsb"], dtype=np.uint8).tobytes()
            scales = np.ascontiguousarray(q["scales_f16"]).view(np.uint16).astype("<u2").tobytes()
            assert len(codes) == stream_bytes(rows, cols, bits)
            assert len(scales) == scale_bytes(rows, cols)
            tdesc.append((t, 2, b"\0\0", rows, cols, pos, len(codes), pos + len(codes),
                          len(scales)))
            parts += [codes, scales]
            pos += len(codes) + len(scales)
        raw = b"".join(parts)
        padded = _align(len(raw), PAGE)
        ngroups = sum(r * c // 64 for r, c in shapes)
        entries.append((l, e, off, len(raw), padded, 64, ngroups, b"\0\0\0\0"))
        descs += tdesc
        blobs.append(raw + b"\0" * (padded - len(raw)))
        off += padded
    head = struct.pack(HEADER_FMT, HEADER_MAGIC, version,
                       num_layers if num_layers is not None else len(layers),
                       max(per_layer.values()) if per_layer else 0, n, table_off, data_off, 64,
                       bits, d_model, vocab_size, dense_ffn_dim, arch_off if version >= 2 else 0)
    meta = bytearray(data_off)
    meta[0:64] = head
    for i, ent in enumerate(entries):
        meta[table_off + 48 * i:table_off + 48 * (i + 1)] = struct.pack(ENTRY_FMT, *ent)
    for i, ds in enumerate(descs):
        meta[desc_off + 44 * i:desc_off + 44 * (i + 1)] = struct.pack(DESC_FMT, *ds)
    if version >= 2:
        a = dict(flags=1, rope_theta=1.0e6, num_heads=64, num_kv_heads=4, head_dim=128,
                 moe_top_k=8, moe_ffn_dim=ffn_dim, dense_ffn_dim=dense_ffn_dim,
                 shared_expert_ffn_dim=0, activation=0, num_hidden_layers=94,
                 rms_norm_eps=1.0e-6, model_type=b"qwen3_moe")
        a.update(arch or {})
        mt = a["model_type"]
        mt = mt if isinstance(mt, bytes) else mt.encode()
        meta[arch_off:arch_off + 128] = struct.pack(
            SARC_FMT, SARC_MAGIC, 1, 128, a["flags"], a["rope_theta"], a["num_heads"],
            a["num_kv_heads"], a["head_dim"], a["moe_top_k"], a["moe_ffn_dim"],
            a["dense_ffn_dim"], a["shared_expert_ffn_dim"], a["activation"],
            a["num_hidden_layers"], a["rms_norm_eps"], mt.ljust(24, b"\0")[:24], b"\0" * 44)
    return bytes(meta) + b"".join(blobs)


class VaultError(ValueError):
    pass


def read_vault(buf: bytes) -> dict:
    """Parse and validate a vault (the page's field tables and its stated
    rules); raises VaultError on the first violation."""
    if len(buf) < 64:
        raise VaultError("short header")
    h = dict(zip(HEADER_FIELDS, struct.unpack_from(HEADER_FMT, buf, 0)))
    if h["magic"] != HEADER_MAGIC:
        raise VaultError("magic")
    if not 1 <= h["version"] <= 2:
        raise VaultError("version")
    if h["table_offset"] != 64:
        raise VaultError("table_offset")
    if h["data_offset"] % PAGE or h["data_offset"] > len(buf):
        raise VaultError("data_offset")
    if h["group_size"] != 64:
        raise VaultError("group_size")
    if h["bits"] not in (2, 4):
        raise VaultError("bits")
    n = h["total_experts"]
    end_desc = 64 + n * 48 + n * 3 * 44
    if end_desc > h["data_offset"]:
        raise VaultError("table overlaps data")
    arch = None
    if h["version"] >= 2:
        ao = h["reserved_ext"]
        if ao % 64 or ao < end_desc or ao + 128 > h["data_offset"]:
            raise VaultError("arch offset")
        arch = dict(zip(SARC_FIELDS, struct.unpack_from(SARC_FMT, buf, ao)))
        if arch["magic"] != SARC_MAGIC or arch["block_version"] != 1 or arch["block_size"] != 128:
            raise VaultError("arch block")
        if arch["activation"] != 0:
            raise VaultError("activation")
        if arch["moe_top_k"] > 16 or arch["head_dim"] > 256:
            raise VaultError("arch limits")
        if arch["num_kv_heads"] == 0 or arch["num_heads"] % arch["num_kv_heads"]:
            raise VaultError("head divisibility")
        if any(arch["reserved"]):
            raise VaultError("arch reserved")
    entries, descs, prev = [], [], None
    for i in range(n):
        ent = dict(zip(ENTRY_FIELDS, struct.unpack_from(ENTRY_FMT, buf, 64 + 48 * i)))
        key = (ent["layer_id"], ent["expert_id"])
        if prev is not None and key <= prev:
            raise VaultError("table order")
        prev = key
        if ent["group_size"] != 64 or any(ent["reserved"]):
            raise VaultError("entry fields")
        if (ent["byte_offset"] % PAGE or ent["byte_offset"] < h["data_offset"]
                or ent["padded_size"] % PAGE or ent["raw_size"] > ent["padded_size"]
                or ent["byte_offset"] + ent["padded_size"] > len(buf)):
            raise VaultError("entry extent")
        ds, groups = [], 0
        for t in range(3):
            o = 64 + 48 * n + 44 * (3 * i + t)
            dsc = dict(zip(DESC_FIELDS, struct.unpack_from(DESC_FMT, buf, o)))
            if dsc["tensor_type"] != t or dsc["ndim"] != 2 or any(dsc["reserved_0"]):
                raise VaultError("descriptor fields")
            r, c = dsc["rows"], dsc["cols"]
            if (dsc["packed_size"] != stream_bytes(r, c, h["bits"])
                    or dsc["scales_size"] != scale_bytes(r, c)):
                raise VaultError("descriptor sizes")
            for o2, sz in ((dsc["packed_offset"], dsc["packed_size"]),
                           (dsc["scales_offset"], dsc["scales_size"])):
                if o2 + sz > ent["raw_size"]:
                    raise VaultError("descriptor extent")
            groups += (r * c + 63) // 64
            ds.append(dsc)
        if groups != ent["num_groups"]:
            raise VaultError("num_groups")
        entries.append(ent)
        descs.append(ds)
    return {"header": h, "arch": arch, "entries": entries, "descs": descs}


def expert_streams(buf: bytes, parsed: dict, layer: int, expert: int):
    """(codes, scales) of gate, up, down of one expert, located through its
    descriptors (never a fixed stride)."""
    for ent, ds in zip(parsed["entries"], parsed["descs"]):
        if (ent["layer_id"], ent["expert_id"]) == (layer, expert):
            out = []
            for dsc in ds:
                base = ent["byte_offset"]
                codes = np.frombuffer(buf, np.uint8, dsc["packed_size"], base + dsc["packed_offset"])
                scales = np.frombuffer(buf, "<u2", dsc["scales_size"] // 2,
                                       base + dsc["scales_offset"]).astype(np.uint16)
                out.append((codes, scales))
            return out
    raise KeyError((layer, expert))
