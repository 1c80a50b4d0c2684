// grouped.cu -- the expert-sorted batched path of one MoE layer: tokens
// gathered per expert, a grouped GEMM on the fifth-generation tensor cores
// (tcgen05.mma kind::f16, bf16 operands, fp32 accumulators in tensor memory)
// for gate/up with SiLU(g)*u in the epilogue, the same for down, then the
// routing-weighted combine.
//
// The arithmetic is the one of "Model Agnosticism" / "Why Quantise"
// (SMOE-Q4 w = (c - 7.5)/7.5 * s, SMOE-Q2 w = (c - 1.5)/1.5 * s, groups of
// 64 along the input dim) and of "CMF v2 -- Format Specification", 2.2 MoE
// (y = sum_j w_j * FFN_{e_j}(x) over the selected experts, plus the shared
// expert weighted by sigmoid(gate . x)).  Here the weights are dequantised to
// bf16 in shared memory (never written to global memory) and the
// activations and h are rounded to bf16: the tensor-core operand type.
//
// Rows: every segment (a routed expert, then the shared expert) owns a run of
// rows padded to a multiple of 128 in the sorted activation matrix; the
// router's dispatch writes each (token, slot)'s row.  A work item is one
// (segment, n-tile, m-tile): 128 rows times 256 output columns over the
// whole K.  Items are ordered so that the m-tiles of one (segment, n-tile)
// are adjacent: CTAs working at the same time read the same weight tiles.
//
// One persistent CTA per SM, 14 warps:
//   warp 0       producer: TMA of the 128 x 64 bf16 activation tile
//                (128-byte swizzle) and bulk copies of the 16 code tiles of
//                the K block into a 5-stage load ring
//   warp 1       tensor memory allocation; lane 0 issues the MMAs
//   warps 2..9   decoders: code tiles -> bf16 weights in the 128-byte
//                swizzled K-major layout the MMA reads (2-stage ring)
//   warps 10..13 epilogue: tensor memory -> registers -> h (bf16) or o (fp32)
// Two accumulators of 256 columns let the epilogue of one item overlap the
// MMAs of the next.  Every wait is bounded; a timeout records
// SMOE_ERR_TIMEOUT, sets the CTA's fail flag, and the CTA drains its copies
// and MMAs in flight before it frees tensor memory and exits.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

constexpr int kGM = 128;             // rows per item (MMA M)
constexpr int kGN = 256;             // output columns per item (MMA N)
constexpr int kGK = 64;              // K per stage (one quantisation group)
constexpr int kLoadStages = 5;
constexpr int kBStages = 2;
constexpr int kDecWarps = 8;
constexpr int kEpiWarpsG = 4;
constexpr int kGWarps = 2 + kDecWarps + kEpiWarpsG;
constexpr int kGThreads = kGWarps * 32;
constexpr int kTilesPerStage = 16;
constexpr uint32_t kATileBytes = kGM * kGK * 2;   // 16 KB
constexpr uint32_t kBTileBytes = kGN * kGK * 2;   // 32 KB
constexpr int kMaxSeg = kMaxExperts + 1;

__host__ __device__ constexpr uint32_t code_stage_bytes(int bits)
{
    return kTilesPerStage * tile_bytes(bits);
}
__host__ __device__ constexpr uint32_t grouped_smem_bytes(int bits)
{
    return kLoadStages * kATileBytes + kBStages * kBTileBytes + kLoadStages * code_stage_bytes(bits) +
           1024;  // slack for the manual 1024-byte alignment
}

struct GSmem {
    uint64_t load_full[kLoadStages];   // producer: 1 arrival + bytes
    uint64_t load_empty[kLoadStages];  // decoder warps + 1 MMA commit
    uint64_t b_full[kBStages];         // decoder warps
    uint64_t b_empty[kBStages];        // 1 MMA commit
    uint64_t acc_full[2];              // 1 MMA commit
    uint64_t acc_empty[2];             // epilogue warps
    uint64_t drain;                    // final MMA commit
    uint32_t tmem_base;
    uint32_t last_it[kLoadStages];     // producer: 1 + last iteration filled per stage
    int fail;
    int nseg, total_items;
    int ipre[kMaxSeg + 1];             // item prefix per segment
    int off[kMaxSeg + 1];              // first row per segment
    int cnt[kMaxSeg];                  // rows used per segment
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows
// of 128 bytes in 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;               // leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;       // stride between 8-row atoms
    d |= static_cast<uint64_t>(1) << 46;               // descriptor version
    d |= static_cast<uint64_t>(2) << 61;               // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 D,
// M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kGN >> 3) << 17) |
                            ((uint32_t)(kGM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
                 "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns of tensor memory.
__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(addr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Bounded wait that records a timeout in the CTA's fail flag.
__device__ __forceinline__ bool gwait(GSmem &sm, uint64_t *bar, unsigned parity, int *status)
{
    if (*reinterpret_cast<volatile int *>(&sm.fail))
        return false;
    if (mbar_wait_bounded(bar, parity))
        return true;
    set_status(status, kStatusTimeout);
    *reinterpret_cast<volatile int *>(&sm.fail) = 1;
    return false;
}

// ------------------------------------------------------------ work items

struct Item {
    int seg, nt, mt, row0, nvalid;
};

template <int PHASE>
__device__ __forceinline__ int seg_ntiles(const GroupedArgs &a, int s)
{
    const int fsg = s < a.E ? a.f : a.fs;
    return PHASE == 0 ? (fsg + 127) / 128 : (a.d + kGN - 1) / kGN;
}

__device__ __forceinline__ Item item_at(const GSmem &sm, int i)
{
    int lo = 0, hi = sm.nseg - 1;  // last segment with ipre[s] <= i
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.ipre[mid] <= i)
            lo = mid;
        else
            hi = mid - 1;
    }
    Item it;
    it.seg = lo;
    const int local = i - sm.ipre[lo];
    const int mtc = (sm.cnt[lo] + kGM - 1) / kGM;
    it.nt = local / mtc;
    it.mt = local % mtc;
    it.row0 = sm.off[lo] + kGM * it.mt;
    const int left = sm.cnt[lo] - kGM * it.mt;
    it.nvalid = left < kGM ? left : kGM;
    return it;
}

// ------------------------------------------------------------ roles

template <int BITS, int PHASE>
__device__ void producer(const GroupedArgs &a, const CUtensorMap *amap, GSmem &sm, uint8_t *sA,
                         uint8_t *sC)
{
    const int lane = threadIdx.x & 31;
    constexpr uint32_t TB = tile_bytes(BITS);
    uint32_t it = 0;
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x) {
        const Item w = item_at(sm, i);
        const bool routed = w.seg < a.E;
        const int fsg = routed ? a.f : a.fs;
        const uint8_t *wb = routed ? a.tiles_routed + (int64_t)w.seg * a.expert_bytes_routed
                                   : a.tiles_shared;
        const int64_t down_off = routed ? a.down_off_routed : a.down_off_shared;
        const int nkb = PHASE == 0 ? a.d / kGK : fsg / kGK;
        const int r0 = (PHASE == 0 ? 128 * w.nt : kGN * w.nt) / 16;  // first strip
        const int nstrips = PHASE == 0 ? fsg / 16 : a.d / 16;
        const int ncopy = PHASE == 0 ? 8 : 16;
        const uint32_t csize = PHASE == 0 ? 2 * TB : TB;
        int nvalid_copy = nstrips - r0;
        nvalid_copy = nvalid_copy < ncopy ? nvalid_copy : ncopy;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = static_cast<int>(it % kLoadStages);
            const unsigned par = ((it / kLoadStages) & 1u) ^ 1u;
            if (!__all_sync(0xffffffffu, gwait(sm, &sm.load_empty[s], par, a.status)))
                return;
            if (lane == 0)
                mbar_arrive_expect_tx(&sm.load_full[s], kATileBytes + nvalid_copy * csize);
            __syncwarp();
            if (lane == 0)
                tma_load_2d(sA + s * kATileBytes, amap, kb * kGK, w.row0, &sm.load_full[s]);
            if (lane == 0)
                sm.last_it[s] = it + 1;
            if (lane < nvalid_copy) {
                const int r = r0 + lane;
                const uint8_t *src =
                    PHASE == 0 ? wb + (((int64_t)r * (a.d / kGK) + kb) * 2) * TB
                               : wb + down_off + ((int64_t)r * (fsg / kGK) + kb) * TB;
                bulk_g2s(sC + s * code_stage_bytes(BITS) + lane * csize, src, csize,
                         &sm.load_full[s]);
            }
        }
    }
}

// Decode one 16 x 64 code tile into rows rowbase .. rowbase + 15 of a
// 128-byte-swizzled K-major bf16 tile: w = (c - L) * (s / L) with
// c - (L + 1/2) exact in bf16 and one rounding in the fused multiply-add.
template <int BITS>
__device__ __forceinline__ void decode_tile(const uint8_t *tile, uint8_t *sB, int rowbase, int lane)
{
    const int gq = lane >> 2, tig = lane & 3;
    constexpr float kInvL = BITS == 4 ? (1.0f / 7.5f) : (1.0f / 1.5f);
    // bf16 128 + c minus 128 + L + 1/2 (136 for Q4, 130 for Q2), both halves
    constexpr uint32_t kSub = BITS == 4 ? 0x43084308u : 0x43024302u;
    const uint32_t sc = *reinterpret_cast<const uint32_t *>(tile + tile_code_bytes(BITS) + 4 * gq);
    const __half2 sh = *reinterpret_cast<const __half2 *>(&sc);
    uint32_t smul[2], sadd[2];
    {
        const float s0 = __low2float(sh) * kInvL, s1 = __high2float(sh) * kInvL;
        smul[0] = pack_bf16x2(s0, s0);
        smul[1] = pack_bf16x2(s1, s1);
        // half of the rounded scale: exact
        sadd[0] = bf16x2_fma(smul[0], 0x3F003F00u, 0u);
        sadd[1] = bf16x2_fma(smul[1], 0x3F003F00u, 0u);
    }
    uint32_t v[2][8];  // [rh][4*pair-in-row ...]: cols 16 tig + 2 m, +1 for m = 0..7
    if (BITS == 4) {
        const uint4 q = *reinterpret_cast<const uint4 *>(tile + 16 * lane);
        const uint32_t wds[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const uint32_t lo = ((wds[j] >> (4 * rh)) & 0x000F000Fu) | 0x43004300u;
                const uint32_t hi = ((wds[j] >> (8 + 4 * rh)) & 0x000F000Fu) | 0x43004300u;
                v[rh][2 * j] = bf16x2_fma(bf16x2_sub(lo, kSub), smul[rh], sadd[rh]);
                v[rh][2 * j + 1] = bf16x2_fma(bf16x2_sub(hi, kSub), smul[rh], sadd[rh]);
            }
    } else {
        const uint2 q = *reinterpret_cast<const uint2 *>(tile + 8 * lane);
        const uint32_t wds[2] = {q.x, q.y};
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const int sh2 = 8 * (j & 1) + 4 * rh;
                const uint32_t w = wds[j >> 1];
                const uint32_t lo = ((w >> sh2) & 0x00030003u) | 0x43004300u;
                const uint32_t hi = ((w >> (sh2 + 2)) & 0x00030003u) | 0x43004300u;
                v[rh][2 * j] = bf16x2_fma(bf16x2_sub(lo, kSub), smul[rh], sadd[rh]);
                v[rh][2 * j + 1] = bf16x2_fma(bf16x2_sub(hi, kSub), smul[rh], sadd[rh]);
            }
    }
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
        const int n = rowbase + gq + 8 * rh;  // n & 7 == gq
        uint8_t *row = sB + n * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int chunk = (2 * tig + h) ^ gq;
            *reinterpret_cast<uint4 *>(row + chunk * 16) =
                make_uint4(v[rh][4 * h], v[rh][4 * h + 1], v[rh][4 * h + 2], v[rh][4 * h + 3]);
        }
    }
}

template <int BITS, int PHASE>
__device__ void decoders(const GroupedArgs &a, GSmem &sm, uint8_t *sB, const uint8_t *sC, int dw)
{
    const int lane = threadIdx.x & 31;
    constexpr uint32_t TB = tile_bytes(BITS);
    uint32_t it = 0;
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x) {
        const Item w = item_at(sm, i);
        const int fsg = w.seg < a.E ? a.f : a.fs;
        const int nkb = PHASE == 0 ? a.d / kGK : fsg / kGK;
        const int r0 = (PHASE == 0 ? 128 * w.nt : kGN * w.nt) / 16;
        const int nstrips = PHASE == 0 ? fsg / 16 : a.d / 16;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = static_cast<int>(it % kLoadStages);
            const int b = static_cast<int>(it % kBStages);
            if (!__all_sync(0xffffffffu, gwait(sm, &sm.load_full[s], (it / kLoadStages) & 1u, a.status)))
                return;
            if (!__all_sync(0xffffffffu, gwait(sm, &sm.b_empty[b], ((it / kBStages) & 1u) ^ 1u, a.status)))
                return;
            const uint8_t *cs = sC + s * code_stage_bytes(BITS);
            uint8_t *bs = sB + b * kBTileBytes;
#pragma unroll
            for (int qq = 0; qq < kTilesPerStage / kDecWarps; ++qq) {
                const int q = dw + kDecWarps * qq;
                // gate/up: copy q/2 holds strip r0 + q/2, gate tile then up tile
                const int strip = PHASE == 0 ? q >> 1 : q;
                const int rowbase = PHASE == 0 ? (q & 1) * 128 + 16 * (q >> 1) : 16 * q;
                if (r0 + strip < nstrips)
                    decode_tile<BITS>(cs + q * TB, bs, rowbase, lane);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.b_full[b]);
                mbar_arrive(&sm.load_empty[s]);
            }
        }
    }
}

template <int PHASE>
__device__ void mma_issuer(const GroupedArgs &a, GSmem &sm, const uint8_t *sA, const uint8_t *sB)
{
    uint32_t it = 0, ic = 0;
    const uint32_t tbase = sm.tmem_base;
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x, ++ic) {
        const Item w = item_at(sm, i);
        const int fsg = w.seg < a.E ? a.f : a.fs;
        const int nkb = PHASE == 0 ? a.d / kGK : fsg / kGK;
        const int ab = static_cast<int>(ic & 1u);
        if (!gwait(sm, &sm.acc_empty[ab], ((ic >> 1) & 1u) ^ 1u, a.status))
            return;
        tc_fence_after();
        const uint32_t dcol = tbase + static_cast<uint32_t>(ab * kGN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = static_cast<int>(it % kLoadStages);
            const int b = static_cast<int>(it % kBStages);
            if (!gwait(sm, &sm.b_full[b], (it / kBStages) & 1u, a.status))
                return;
            if (!gwait(sm, &sm.load_full[s], (it / kLoadStages) & 1u, a.status))
                return;
            tc_fence_after();
            const uint32_t aaddr = smem_u32(sA + s * kATileBytes);
            const uint32_t baddr = smem_u32(sB + b * kBTileBytes);
#pragma unroll
            for (int ks = 0; ks < kGK / 16; ++ks)
                umma_bf16(dcol, sw128_desc(aaddr + 32 * ks), sw128_desc(baddr + 32 * ks),
                          (kb | ks) != 0 ? 1u : 0u);
            umma_commit(&sm.b_empty[b]);
            umma_commit(&sm.load_empty[s]);
        }
        umma_commit(&sm.acc_full[ab]);
    }
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;
}

template <int PHASE>
__device__ void epilogue(const GroupedArgs &a, GSmem &sm)
{
    const int lane = threadIdx.x & 31;
    const int quarter = (threadIdx.x >> 5) & 3;  // tensor-memory lanes 32 q .. 32 q + 31
    const int r = 32 * quarter + lane;
    const uint32_t tbase = sm.tmem_base;
    uint32_t ic = 0;
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x, ++ic) {
        const Item w = item_at(sm, i);
        const int fsg = w.seg < a.E ? a.f : a.fs;
        const int ab = static_cast<int>(ic & 1u);
        if (!__all_sync(0xffffffffu, gwait(sm, &sm.acc_full[ab], (ic >> 1) & 1u, a.status)))
            return;
        tc_fence_after();
        const uint32_t taddr = tbase + (static_cast<uint32_t>(32 * quarter) << 16) +
                               static_cast<uint32_t>(ab * kGN);
        const bool valid = r < w.nvalid;
        const int64_t row = w.row0 + r;
        if (PHASE == 0) {
            const int n0 = 128 * w.nt;
            for (int c = 0; c < 128 && n0 + c < fsg; c += 16) {
                uint32_t g[16], u[16];
                tmem_ld16(taddr + c, g);
                tmem_ld16(taddr + 128 + c, u);
                tmem_wait_ld();
                uint32_t hv[8];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    hv[m] = pack_bf16x2(silu_mul(__uint_as_float(g[2 * m]), __uint_as_float(u[2 * m])),
                                        silu_mul(__uint_as_float(g[2 * m + 1]), __uint_as_float(u[2 * m + 1])));
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(a.h + row * a.hstride + n0 + c);
                    dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    dst[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
                }
            }
        } else {
            const int n0 = kGN * w.nt;
            for (int c = 0; c < kGN && n0 + c < a.d; c += 16) {
                uint32_t o[16];
                tmem_ld16(taddr + c, o);
                tmem_wait_ld();
                if (valid) {
                    float4 *dst = reinterpret_cast<float4 *>(a.o + row * a.d + n0 + c);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        dst[m] = make_float4(__uint_as_float(o[4 * m]), __uint_as_float(o[4 * m + 1]),
                                             __uint_as_float(o[4 * m + 2]), __uint_as_float(o[4 * m + 3]));
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.acc_empty[ab]);
    }
}

template <int BITS, int PHASE>
__global__ void __launch_bounds__(kGThreads, 1)
    grouped_gemm_kernel(const GroupedArgs a, const __grid_constant__ CUtensorMap amap)
{
    extern __shared__ uint8_t g_smem_raw[];
    __shared__ GSmem sm;
    uint8_t *base = g_smem_raw + ((1024u - (smem_u32(g_smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = base;                                   // kLoadStages x 16 KB
    uint8_t *sB = sA + kLoadStages * kATileBytes;          // kBStages x 32 KB
    uint8_t *sC = sB + kBStages * kBTileBytes;             // kLoadStages code stages
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // segment table -> item prefix (one warp; at most 257 segments)
    if (warp == 0) {
        const int nseg = a.E + (a.has_shared ? 1 : 0);
        int run = 0;
        for (int s0 = 0; s0 < nseg; s0 += 32) {
            const int s = s0 + lane;
            int items = 0;
            if (s < nseg) {
                int c = __ldcg(a.seg + nseg + 1 + s);
                const int o = __ldcg(a.seg + s);
                // a segment must lie inside the sorted matrices
                if (c < 0 || o < 0 || (int64_t)o + (int64_t)(c + kGM - 1) / kGM * kGM > a.rows) {
                    set_status(a.status, kStatusBadArg);
                    c = 0;
                }
                sm.cnt[s] = c;
                sm.off[s] = o;
                items = ((c + kGM - 1) / kGM) * seg_ntiles<PHASE>(a, s);
            }
            int incl = items;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (s < nseg)
                sm.ipre[s] = run + incl - items;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            sm.ipre[nseg] = run;
            sm.nseg = nseg;
            sm.total_items = run;
            sm.fail = 0;
            for (int s = 0; s < kLoadStages; ++s) {
                sm.last_it[s] = 0;
                mbar_init(&sm.load_full[s], 1);
                mbar_init(&sm.load_empty[s], kDecWarps + 1);
            }
            for (int b = 0; b < kBStages; ++b) {
                mbar_init(&sm.b_full[b], kDecWarps);
                mbar_init(&sm.b_empty[b], 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(&sm.acc_full[b], 1);
                mbar_init(&sm.acc_empty[b], kEpiWarpsG);
            }
            mbar_init(&sm.drain, 1);
            fence_mbar_init();
        }
    }
    __syncthreads();
    if (static_cast<int>(blockIdx.x) >= sm.total_items)
        return;  // nothing for this CTA (uniform across the CTA)
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sm.tmem_base)),
                     "r"(2 * kGN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0) {
        producer<BITS, PHASE>(a, &amap, sm, sA, sC);
    } else if (warp == 1) {
        if (lane == 0) {
            mma_issuer<PHASE>(a, sm, sA, sB);
            // every MMA issued so far has completed once this commit lands
            umma_commit(&sm.drain);
            if (!mbar_wait_bounded(&sm.drain, 0)) {
                set_status(a.status, kStatusTimeout);
                *reinterpret_cast<volatile int *>(&sm.fail) = 1;
            }
        }
        __syncwarp();
    } else if (warp < 2 + kDecWarps) {
        decoders<BITS, PHASE>(a, sm, sB, sC, warp - 2);
    } else {
        epilogue<PHASE>(a, sm);
    }
    __syncwarp();
    // After a failure the consumers may have left copies unwaited: the
    // producer waits (bounded) for the last phase it filled on every stage,
    // so no copy is in flight when the CTA exits.
    if (warp == 0 && *reinterpret_cast<volatile int *>(&sm.fail) && lane < kLoadStages) {
        const uint32_t last = sm.last_it[lane];
        if (last > 0 && !mbar_wait_bounded(&sm.load_full[lane], ((last - 1) / kLoadStages) & 1u))
            set_status(a.status, kStatusTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(sm.tmem_base),
                     "r"(2 * kGN)
                     : "memory");
    }
}

// ------------------------------------------------------------ gather, combine

// x_sorted[row(t, j)] = bf16(x[t]) for every slot j (and the shared segment).
template <bool XBF16>
__global__ void __launch_bounds__(256) gather_kernel(const void *x, int64_t T, int d, int k,
                                                     int has_shared, const int32_t *rows,
                                                     int64_t nrows, uint16_t *xs)
{
    const int64_t t = blockIdx.x;
    const int nslot = k + (has_shared ? 1 : 0);
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
        uint4 v;
        if (XBF16) {
            v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + t * d + c));
        } else {
            const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(x) + t * d + c);
            const float4 a0 = __ldg(p), a1 = __ldg(p + 1);
            v = make_uint4(pack_bf16x2(a0.x, a0.y), pack_bf16x2(a0.z, a0.w), pack_bf16x2(a1.x, a1.y),
                           pack_bf16x2(a1.z, a1.w));
        }
        for (int j = 0; j < nslot; ++j) {
            const int32_t r = __ldg(rows + t * (k + 1) + (j < k ? j : k));
            if (r >= 0 && r < nrows)
                *reinterpret_cast<uint4 *>(xs + (int64_t)r * d + c) = v;
        }
    }
}

// y[t] = sum_j w[t, j] o[row(t, j)] in rank order, then + shared weight *
// o[shared row].
__global__ void __launch_bounds__(256) grouped_combine_kernel(const float *o, int64_t T, int d, int k,
                                                              int has_shared, const int32_t *rows,
                                                              int64_t nrows, const float *w,
                                                              const float *sw, float *y)
{
    const int64_t t = blockIdx.x;
    for (int c = threadIdx.x * 4; c < d; c += blockDim.x * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int32_t r = __ldg(rows + t * (k + 1) + j);
            if (r < 0 || r >= nrows)
                continue;
            const float wj = __ldg(w + t * k + j);
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(o + (int64_t)r * d + c));
            acc.x = fmaf(wj, v.x, acc.x);
            acc.y = fmaf(wj, v.y, acc.y);
            acc.z = fmaf(wj, v.z, acc.z);
            acc.w = fmaf(wj, v.w, acc.w);
        }
        const int32_t rs = has_shared ? __ldg(rows + t * (k + 1) + k) : -1;
        if (rs >= 0 && rs < nrows) {
            const int32_t r = rs;
            const float ws = __ldg(sw + t);
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(o + (int64_t)r * d + c));
            acc.x = fmaf(ws, v.x, acc.x);
            acc.y = fmaf(ws, v.y, acc.y);
            acc.z = fmaf(ws, v.z, acc.z);
            acc.w = fmaf(ws, v.w, acc.w);
        }
        *reinterpret_cast<float4 *>(y + t * d + c) = acc;
    }
}

// ------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::mutex mu;
    static EncodeTiledFn fn = nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tensor map of a row-major bf16 matrix [rows, cols] read in 128 x 64 boxes
// with the 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGK), static_cast<cuuint32_t>(kGM)};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BITS, int PHASE>
cudaError_t launch_gemm_t(const GroupedArgs &a, const CUtensorMap &map, cudaStream_t s)
{
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev >= 0 && dev < 64 && !attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<BITS, PHASE>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 grouped_smem_bytes(BITS));
            if (e != cudaSuccess)
                return e;
            attr_set[dev] = true;
        }
    }
    grouped_gemm_kernel<BITS, PHASE>
        <<<device_sm_count(), kGThreads, grouped_smem_bytes(BITS), s>>>(a, map);
    return cudaGetLastError();
}

}  // namespace

int64_t grouped_max_rows(int64_t T, int E, int k, int has_shared)
{
    const int64_t tk = T * k;
    const int64_t segs = tk < E ? tk : E;
    int64_t r = tk + segs * (kGM - 1);
    if (has_shared)
        r += T + kGM - 1;
    return (r + kGM - 1) / kGM * kGM;
}

cudaError_t launch_grouped(const GroupedArgs &a, const void *x, int x_bf16, const float *w,
                           const float *sw, float *y, cudaStream_t s)
{
    if (a.T == 0)
        return cudaSuccess;
    CUtensorMap mx, mh;
    if (!make_map(&mx, a.xs, a.rows, a.d) || !make_map(&mh, a.h, a.rows, a.hstride))
        return cudaErrorInvalidValue;
    const unsigned nt = static_cast<unsigned>(a.T);
    if (x_bf16)
        gather_kernel<true><<<nt, 256, 0, s>>>(x, a.T, a.d, a.k, a.has_shared, a.rows_of, a.rows, a.xs);
    else
        gather_kernel<false><<<nt, 256, 0, s>>>(x, a.T, a.d, a.k, a.has_shared, a.rows_of, a.rows, a.xs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    e = a.bits == 4 ? launch_gemm_t<4, 0>(a, mx, s) : launch_gemm_t<2, 0>(a, mx, s);
    if (e != cudaSuccess)
        return e;
    e = a.bits == 4 ? launch_gemm_t<4, 1>(a, mh, s) : launch_gemm_t<2, 1>(a, mh, s);
    if (e != cudaSuccess)
        return e;
    grouped_combine_kernel<<<nt, 256, 0, s>>>(a.o, a.T, a.d, a.k, a.has_shared, a.rows_of, a.rows, w,
                                              sw, y);
    return cudaGetLastError();
}

}  // namespace smoe
