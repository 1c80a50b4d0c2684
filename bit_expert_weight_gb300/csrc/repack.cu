// repack.cu -- byte permutation between the pages' LSB-first code stream +
// fp16 scale array (".smoe Binary Format", Expert Blob Architecture) and the
// device tile layout described in common.cuh.
//
// One warp per 16 x 64 tile.  Lane t = (gq, tig) gathers rows gq and gq + 8,
// columns 16*tig .. 16*tig + 15 of the group: those are 8 (Q4) or 4 (Q2)
// consecutive stream bytes per row, so the read is one aligned 8- or 4-byte
// load per row.  Unpack writes the same bytes back, whole bytes per lane, so
// no two lanes touch one byte.
#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

// Destination of tile (rb, g) of matrix `kind` (0 gate, 1 up, 2 down):
// strip-major, gate and up interleaved per group.
__device__ __forceinline__ int64_t tile_offset(int kind, int rb, int g, int G, int bits,
                                               int64_t gateup_bytes)
{
    if (kind < 2)
        return (((int64_t)rb * G + g) * 2 + kind) * tile_bytes(bits);
    return gateup_bytes + ((int64_t)rb * G + g) * tile_bytes(bits);
}

__global__ void __launch_bounds__(256) repack_kernel(const uint8_t *__restrict__ codes,
                                                     const uint16_t *__restrict__ scales, int kind,
                                                     int R, int K, int bits, uint8_t *out,
                                                     int64_t gateup_bytes)
{
    const int lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const int64_t ntiles = (int64_t)(R / kTileRows) * G;
    const int64_t tile = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (tile >= ntiles)
        return;
    const int rb = static_cast<int>(tile / G), g = static_cast<int>(tile % G);
    const int gq = lane >> 2, tig = lane & 3;
    uint8_t *dst = out + tile_offset(kind, rb, g, G, bits, gateup_bytes);
    uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
        const int64_t r = (int64_t)rb * kTileRows + gq + 8 * rh;
        const int64_t e0 = r * K + (int64_t)g * kGroup + 16 * tig;  // first element
        if (bits == 4) {
            const uint64_t row = *reinterpret_cast<const uint64_t *>(codes + e0 / 2);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t c = static_cast<uint32_t>(row >> (4 * (4 * j + e))) & 0xFu;
                    words[j] |= c << tile_code_bit(4, j, rh, e);
                }
        } else {
            const uint32_t row = *reinterpret_cast<const uint32_t *>(codes + e0 / 4);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t c = (row >> (2 * (4 * j + e))) & 0x3u;
                    words[j >> 1] |= c << tile_code_bit(2, j, rh, e);
                }
        }
    }
    if (bits == 4)
        reinterpret_cast<uint4 *>(dst)[lane] = make_uint4(words[0], words[1], words[2], words[3]);
    else
        reinterpret_cast<uint2 *>(dst)[lane] = make_uint2(words[0], words[1]);
    if (lane < kTileRows) {
        const int64_t r = (int64_t)rb * kTileRows + lane;
        reinterpret_cast<uint16_t *>(dst + tile_code_bytes(bits))[tile_scale_half(lane)] =
            scales[r * G + g];
    }
}

__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t *__restrict__ in, int kind,
                                                     int R, int K, int bits, int64_t gateup_bytes,
                                                     uint8_t *codes, uint16_t *scales)
{
    const int lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const int64_t ntiles = (int64_t)(R / kTileRows) * G;
    const int64_t tile = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (tile >= ntiles)
        return;
    const int rb = static_cast<int>(tile / G), g = static_cast<int>(tile % G);
    const int gq = lane >> 2, tig = lane & 3;
    const uint8_t *src = in + tile_offset(kind, rb, g, G, bits, gateup_bytes);
    uint32_t words[4];
    if (bits == 4) {
        uint4 v = reinterpret_cast<const uint4 *>(src)[lane];
        words[0] = v.x, words[1] = v.y, words[2] = v.z, words[3] = v.w;
    } else {
        uint2 v = reinterpret_cast<const uint2 *>(src)[lane];
        words[0] = v.x, words[1] = v.y, words[2] = words[3] = 0u;
    }
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
        const int64_t r = (int64_t)rb * kTileRows + gq + 8 * rh;
        const int64_t e0 = r * K + (int64_t)g * kGroup + 16 * tig;
        if (bits == 4) {
            uint64_t row = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint64_t c = (words[j] >> tile_code_bit(4, j, rh, e)) & 0xFu;
                    row |= c << (4 * (4 * j + e));
                }
            *reinterpret_cast<uint64_t *>(codes + e0 / 2) = row;
        } else {
            uint32_t row = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t c = (words[j >> 1] >> tile_code_bit(2, j, rh, e)) & 0x3u;
                    row |= c << (2 * (4 * j + e));
                }
            *reinterpret_cast<uint32_t *>(codes + e0 / 4) = row;
        }
    }
    if (lane < kTileRows) {
        const int64_t r = (int64_t)rb * kTileRows + lane;
        scales[r * G + g] =
            reinterpret_cast<const uint16_t *>(src + tile_code_bytes(bits))[tile_scale_half(lane)];
    }
}

}  // namespace

cudaError_t launch_repack(const uint8_t *codes, const uint16_t *scales, int kind, int R, int K,
                          int bits, uint8_t *expert_base, int64_t gateup_bytes,
                          cudaStream_t stream)
{
    int64_t ntiles = (int64_t)(R / kTileRows) * (K / kGroup);
    if (ntiles == 0)
        return cudaSuccess;
    repack_kernel<<<static_cast<unsigned>((ntiles + 7) / 8), 256, 0, stream>>>(
        codes, scales, kind, R, K, bits, expert_base, gateup_bytes);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t *expert_base, int kind, int R, int K, int bits,
                          int64_t gateup_bytes, uint8_t *codes, uint16_t *scales,
                          cudaStream_t stream)
{
    int64_t ntiles = (int64_t)(R / kTileRows) * (K / kGroup);
    if (ntiles == 0)
        return cudaSuccess;
    unpack_kernel<<<static_cast<unsigned>((ntiles + 7) / 8), 256, 0, stream>>>(
        expert_base, kind, R, K, bits, gateup_bytes, codes, scales);
    return cudaGetLastError();
}

}  // namespace smoe
