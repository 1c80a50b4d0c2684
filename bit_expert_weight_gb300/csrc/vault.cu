// vault.cu -- the pages' ".smoe Binary Format" vault as the input of the
// repack: parse and validate the file header, the arch block "SARC", the
// expert table and the tensor descriptors from a host buffer, locate an
// expert's three sub-tensors through its descriptors, and repack a whole
// layer from a device copy of the file.
//
// Field offsets follow the page's tables (File Header -- 64 bytes; Arch
// Block "SARC" -- 128 bytes; Expert Table Entry -- 48 bytes; Tensor
// Descriptor -- 44 bytes).  The entry and descriptor have 8-byte fields at
// 4-byte offsets (36 and 12), so every field is read byte by byte,
// little-endian ("Immutable Encoding"), independent of the host's struct
// packing and byte order.  Host code only: nothing here touches the GPU
// except the final call of smoe_repack.
#include <string.h>

#include "smoe.h"
#include "internal.h"

namespace {

constexpr uint64_t kPage = 16384;  // blob and data_offset alignment
constexpr size_t kHeaderBytes = 64, kEntryBytes = 48, kDescBytes = 44, kArchBytes = 128;
const uint8_t kMagic[8] = {0x53, 0x4D, 0x4F, 0x45, 0xDE, 0xEA, 0x00, 0x01};

uint32_t rd32(const uint8_t *p)
{
    return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
           (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24);
}
uint64_t rd64(const uint8_t *p) { return rd32(p) | (static_cast<uint64_t>(rd32(p + 4)) << 32); }
float rdf32(const uint8_t *p)
{
    const uint32_t u = rd32(p);
    float f;
    memcpy(&f, &u, 4);
    return f;
}
bool all_zero(const uint8_t *p, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        if (p[i])
            return false;
    return true;
}
uint64_t stream_bytes(uint64_t rows, uint64_t cols, uint32_t bits) { return (rows * cols * bits + 7) / 8; }
uint64_t scales_bytes(uint64_t rows, uint64_t cols) { return (rows * cols + 63) / 64 * 2; }

// The whole metadata check (header, arch block, every entry and descriptor).
bool parse(const uint8_t *m, size_t mb, uint64_t file_bytes, smoe_vault_info *info)
{
    if (!m || mb < kHeaderBytes)
        return false;
    smoe_vault_info v;
    memset(&v, 0, sizeof v);
    if (memcmp(m, kMagic, 8) != 0)
        return false;
    v.version = rd32(m + 8);
    v.num_moe_layers = rd32(m + 12);
    v.max_experts_per_layer = rd32(m + 16);
    v.total_experts = rd32(m + 20);
    v.table_offset = rd64(m + 24);
    v.data_offset = rd64(m + 32);
    v.group_size = rd32(m + 40);
    v.bits = rd32(m + 44);
    v.d_model = rd32(m + 48);
    v.vocab_size = rd32(m + 52);
    v.ffn_dim = rd32(m + 56);
    v.reserved_ext = rd32(m + 60);
    if (v.version < 1 || v.version > 2 || v.table_offset != kHeaderBytes || v.group_size != 64 ||
        (v.bits != 2 && v.bits != 4))
        return false;
    if (v.data_offset % kPage || v.data_offset > file_bytes || v.data_offset > mb)
        return false;
    const uint64_t n = v.total_experts;
    const uint64_t end_desc = kHeaderBytes + n * kEntryBytes + n * 3 * kDescBytes;
    if (end_desc > v.data_offset)
        return false;
    if (v.version >= 2) {
        const uint64_t ao = v.reserved_ext;
        if (ao % 64 || ao < end_desc || ao + kArchBytes > v.data_offset)
            return false;
        const uint8_t *a = m + ao;
        if (memcmp(a, "SARC", 4) != 0 || rd32(a + 4) != 1 || rd32(a + 8) != kArchBytes)
            return false;
        v.has_arch = 1;
        v.arch_flags = rd32(a + 12);
        v.rope_theta = rdf32(a + 16);
        v.num_heads = rd32(a + 20);
        v.num_kv_heads = rd32(a + 24);
        v.head_dim = rd32(a + 28);
        v.moe_top_k = rd32(a + 32);
        v.moe_ffn_dim = rd32(a + 36);
        v.dense_ffn_dim = rd32(a + 40);
        v.shared_expert_ffn_dim = rd32(a + 44);
        v.activation = rd32(a + 48);
        v.num_hidden_layers = rd32(a + 52);
        v.rms_norm_eps = rdf32(a + 56);
        memcpy(v.model_type, a + 60, 24);
        v.model_type[24] = '\0';
        // the load-time checks the page lists: SiLU, top-k, head geometry
        if (v.activation != 0 || v.moe_top_k > 16 || v.head_dim > 256 || v.num_kv_heads == 0 ||
            v.num_heads % v.num_kv_heads || !all_zero(a + 84, 44))
            return false;
    }
    uint32_t prev_l = 0, prev_e = 0;
    for (uint64_t i = 0; i < n; ++i) {
        const uint8_t *en = m + kHeaderBytes + i * kEntryBytes;
        const uint32_t l = rd32(en), e = rd32(en + 4);
        if (i > 0 && (l < prev_l || (l == prev_l && e <= prev_e)))
            return false;  // table sorted by layer, then expert
        prev_l = l;
        prev_e = e;
        const uint64_t off = rd64(en + 8), raw = rd64(en + 16), padded = rd64(en + 24);
        if (rd32(en + 32) != 64 || !all_zero(en + 44, 4))
            return false;
        if (off % kPage || off < v.data_offset || padded % kPage || raw > padded ||
            off + padded > file_bytes || off + padded < off)
            return false;
        uint64_t groups = 0;
        for (int t = 0; t < 3; ++t) {
            const uint8_t *d = m + kHeaderBytes + n * kEntryBytes + (i * 3 + t) * kDescBytes;
            if (d[0] != t || d[1] != 2 || d[2] || d[3])
                return false;
            const uint64_t rows = rd32(d + 4), cols = rd32(d + 8);
            const uint64_t po = rd64(d + 12), ps = rd64(d + 20), so = rd64(d + 28), ss = rd64(d + 36);
            if (ps != stream_bytes(rows, cols, v.bits) || ss != scales_bytes(rows, cols))
                return false;
            if (po + ps > raw || so + ss > raw || po + ps < po || so + ss < so)
                return false;
            groups += (rows * cols + 63) / 64;
        }
        if (groups != rd64(en + 36))
            return false;
    }
    if (info)
        *info = v;
    return true;
}

bool find(const uint8_t *m, uint64_t n, uint32_t layer, uint32_t expert, smoe_vault_expert *out)
{
    for (uint64_t i = 0; i < n; ++i) {
        const uint8_t *en = m + kHeaderBytes + i * kEntryBytes;
        if (rd32(en) != layer || rd32(en + 4) != expert)
            continue;
        smoe_vault_expert x;
        memset(&x, 0, sizeof x);
        x.layer_id = layer;
        x.expert_id = expert;
        x.byte_offset = rd64(en + 8);
        x.raw_size = rd64(en + 16);
        x.padded_size = rd64(en + 24);
        x.num_groups = rd64(en + 36);
        for (int t = 0; t < 3; ++t) {
            const uint8_t *d = m + kHeaderBytes + n * kEntryBytes + (i * 3 + t) * kDescBytes;
            x.tensor[t].rows = rd32(d + 4);
            x.tensor[t].cols = rd32(d + 8);
            x.tensor[t].packed_offset = rd64(d + 12);
            x.tensor[t].packed_size = rd64(d + 20);
            x.tensor[t].scales_offset = rd64(d + 28);
            x.tensor[t].scales_size = rd64(d + 36);
        }
        *out = x;
        return true;
    }
    return false;
}

}  // namespace

extern "C" {

smoe_status smoe_vault_parse(const void *meta, size_t meta_bytes, uint64_t file_bytes,
                             smoe_vault_info *info)
{
    if (!info)
        return SMOE_ERR_INVALID_ARG;
    return parse(static_cast<const uint8_t *>(meta), meta_bytes, file_bytes, info)
               ? SMOE_OK
               : SMOE_ERR_INVALID_ARG;
}

smoe_status smoe_vault_find_expert(const void *meta, size_t meta_bytes, uint64_t file_bytes,
                                   uint32_t layer, uint32_t expert, smoe_vault_expert *out)
{
    smoe_vault_info v;
    if (!out || !parse(static_cast<const uint8_t *>(meta), meta_bytes, file_bytes, &v))
        return SMOE_ERR_INVALID_ARG;
    return find(static_cast<const uint8_t *>(meta), v.total_experts, layer, expert, out)
               ? SMOE_OK
               : SMOE_ERR_INVALID_ARG;
}

smoe_status smoe_vault_repack_layer(const void *meta, size_t meta_bytes, const void *vault_dev,
                                    uint64_t file_bytes, uint32_t layer, uint32_t num_experts,
                                    void *tiles_out, size_t tiles_bytes, void *cuda_stream)
{
    smoe_vault_info v;
    const uint8_t *m = static_cast<const uint8_t *>(meta);
    if (!vault_dev || !tiles_out || num_experts == 0 || num_experts > 65536 ||
        reinterpret_cast<uintptr_t>(vault_dev) % 16 || !parse(m, meta_bytes, file_bytes, &v))
        return SMOE_ERR_INVALID_ARG;
    const int d = static_cast<int>(v.d_model);
    int f = -1;
    const uint8_t *base = static_cast<const uint8_t *>(vault_dev);
    const size_t ptrs = 3 * static_cast<size_t>(num_experts);
    const uint8_t **codes = new const uint8_t *[ptrs];
    const uint16_t **scales = new const uint16_t *[ptrs];
    smoe_status st = SMOE_OK;
    for (uint32_t e = 0; e < num_experts && st == SMOE_OK; ++e) {
        smoe_vault_expert x;
        if (!find(m, v.total_experts, layer, e, &x)) {
            st = SMOE_ERR_INVALID_ARG;
            break;
        }
        // shapes: gate/up [f, d], down [d, f], f the same for the layer
        const int fe = static_cast<int>(x.tensor[0].rows);
        if (f < 0)
            f = fe;
        if (fe != f || x.tensor[0].cols != v.d_model || x.tensor[1].rows != x.tensor[0].rows ||
            x.tensor[1].cols != v.d_model || x.tensor[2].rows != v.d_model ||
            static_cast<int>(x.tensor[2].cols) != f || (v.has_arch && v.moe_ffn_dim != (uint32_t)f)) {
            st = SMOE_ERR_INVALID_ARG;
            break;
        }
        for (int t = 0; t < 3; ++t) {
            codes[3 * e + t] = base + x.byte_offset + x.tensor[t].packed_offset;
            scales[3 * e + t] = reinterpret_cast<const uint16_t *>(base + x.byte_offset +
                                                                   x.tensor[t].scales_offset);
        }
    }
    if (st == SMOE_OK)
        st = smoe_repack(codes, scales, d, f, static_cast<int32_t>(num_experts),
                         static_cast<int>(v.bits), 64, tiles_out, tiles_bytes, cuda_stream);
    delete[] codes;
    delete[] scales;
    return st;
}

}  // extern "C"
