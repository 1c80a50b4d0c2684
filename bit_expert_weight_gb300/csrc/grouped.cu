// grouped.cu -- the expert-sorted batched path of one MoE layer: tokens
// gathered per expert, a grouped GEMM on the fifth-generation tensor cores
// (tcgen05.mma kind::f16, bf16 operands, fp32 accumulators in tensor memory)
// for gate/up with SiLU(g)*u in the epilogue, the same for down with the
// routing weight applied in its epilogue, then the sum over each token's
// rows.
//
// The arithmetic is the one of "Model Agnosticism" / "Why Quantise"
// (SMOE-Q4 w = (c - 7.5)/7.5 * s, SMOE-Q2 w = (c - 1.5)/1.5 * s, groups of
// 64 along the input dim) and of "CMF v2 -- Format Specification", 2.2 MoE
// (y = sum_j w_j * FFN_{e_j}(x) over the selected experts, plus the shared
// expert weighted by sigmoid(gate . x)).  Here the weights are dequantised to
// bf16 in shared memory (never written to global memory), the activations
// and h are rounded to bf16 (the tensor-core operand type), and so is each
// expert's weighted output row before the fp32 sum.
//
// Rows: every segment (a routed expert, then the shared expert) owns a run of
// rows padded to a multiple of 128 in the sorted activation matrix; the
// router's dispatch writes each (token, slot)'s row.  A work item is one
// (segment, n-tile, m-tile): 128 rows times 256 output columns over the
// whole K, for one or two m-tiles (one decoded weight stage then feeds two
// MMA groups).  Items are ordered so that the m-tiles of one (segment,
// n-tile) are adjacent: CTAs working at the same time read the same weights.
//
// One persistent CTA per SM, 28 warps (warp w issues on sub-partition w % 4):
//   warp 0        code producer: the 16 code tiles of every K block, in
//                 stages of 1 or 4 K blocks (one tensor copy per stage, or
//                 one bulk copy per strip for mixed-depth banks), freed
//                 once decoded
//   warp 1        tensor memory allocation; lane 0 issues the MMAs, one
//                 commit per K block frees that block's stage
//   warp 2        activation producer: TMA of the item's one or two
//                 activation tiles of every K block (boxes of 32, 64 or 128
//                 rows x 64 bf16, 128-byte swizzle)
//   warps 3..6    epilogue: tensor memory -> registers -> h (bf16) or the
//                 row's routing weight x o (bf16)
//   16 warps      decoders (warps 7..27 off sub-partition 1; the others
//                 exit), one code tile each per K block: bf16 weights in the
//                 128-byte-swizzled K-major layout the MMA reads
// A stage holds a K block's activations and decoded weights: 3 stages (two
// activation tiles each when items pair two m-tiles).
// Two accumulators of 256 columns: an item of two m-tiles uses both, an item
// of one m-tile alternates between them so that its epilogue overlaps the
// next item's MMAs.  Every wait is bounded; a timeout records
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
constexpr int kMaxCodeStages = 3;
// Code stages: the tiles of code_kb consecutive K blocks of the item's
// strips.  Banks of one depth fill a stage with one tensor copy (a 4-D map:
// tile bytes x K blocks x strips x experts); banks of mixed depths with one
// bulk copy per strip.  A bulk copy has a fixed cost: copies of one K
// block's tiles (1088 B for a gate/up strip at Q4) cap the weight stream
// near 2 TB/s on this part, copies of 4 K blocks reach about 7 TB/s.  Items
// of one m-tile stream each weight tile once per m-tile and take 2 stages
// of 4 K blocks; items of two m-tiles need 3 activation stages and keep 3
// code stages of one K block (what the shared memory leaves).
__host__ __device__ constexpr int code_kb(bool pair) { return pair ? 1 : 4; }
__host__ __device__ constexpr int code_stages(bool pair) { return pair ? 3 : 2; }
constexpr int kMaxStages = 4;        // activations + decoded weights of one K block each
constexpr int kDecWarps = 16;
constexpr int kEpiWarpsG = 4;
constexpr int kEpiWarp0 = 3;         // warps 0 codes, 1 MMA, 2 activations, 3..6 epilogue
constexpr int kGWarps = 28;          // decoders: warps 7..27 off sub-partition 1

// Warp w issues on sub-partition w % 4.  The MMA warp (1) keeps its
// sub-partition to itself and the idle epilogue quarter: the decoders take
// warps 7..27 except those of sub-partition 1, which exit at once, so the
// single MMA-issuing thread never queues behind decoder instructions.
__device__ __forceinline__ int decoder_index(int w)
{
    if (w < 7 || (w & 3) == 1)
        return -1;
    return (w - 7) - (w > 9 ? (w - 6) / 4 : 0);
}
constexpr int kGThreads = kGWarps * 32;
constexpr int kTilesPerStage = 16;
constexpr uint32_t kATileBytes = kGM * kGK * 2;   // 16 KB
constexpr uint32_t kBTileBytes = kGN * kGK * 2;   // 32 KB
// Stages of activations + decoded weights: 3 for both item kinds, what the
// shared memory holds beside the code ring (two activation tiles per stage
// for items of two m-tiles, code stages of 4 K blocks for items of one).
// 4 stages with code stages of 1 K block measured slower.
__host__ __device__ constexpr int num_stages(bool /* pair */) { return 3; }
__host__ __device__ constexpr uint32_t a_stage_bytes(bool pair)
{
    return pair ? 2 * kATileBytes : kATileBytes;
}
constexpr int kMaxSeg = kMaxExperts + 1;

__host__ __device__ constexpr uint32_t code_stage_bytes(int bits, bool pair)
{
    return code_kb(pair) * kTilesPerStage * tile_bytes(bits);
}
__host__ __device__ constexpr uint32_t grouped_smem_bytes(int bits, bool pair)
{
    return num_stages(pair) * (a_stage_bytes(pair) + kBTileBytes) +
           code_stages(pair) * code_stage_bytes(bits, pair) +
           1024;  // slack for the manual 1024-byte alignment
}

struct GSmem {
    uint64_t code_full[kMaxCodeStages];   // code producer: 1 arrival + bytes
    uint64_t code_empty[kMaxCodeStages];  // decoder warps
    uint64_t a_full[kMaxStages];       // activation producer: 1 arrival + bytes
    uint64_t b_full[kMaxStages];       // decoder warps
    uint64_t stage_empty[kMaxStages];  // 1 MMA commit: activations and weights free
    uint64_t acc_full[2];              // 1 MMA commit
    uint64_t acc_empty[2];             // epilogue warps
    uint64_t drain;                    // final MMA commit
    uint32_t tmem_base;
    uint32_t last_code[kMaxCodeStages];   // 1 + last use filled, per stage (drain
    uint32_t last_a[kMaxStages];       // after a failure)
    int fail;
    int nseg, total_items;
    int ipre[kMaxSeg + 1];             // item prefix per segment
    int off[kMaxSeg + 1];              // first row per segment
    int cnt[kMaxSeg];                  // rows used per segment
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

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

// One item: one (segment, n-tile) and one or two consecutive m-tiles of the
// segment, so that each decoded weight stage feeds up to two MMA groups.
struct Item {
    int seg, nt, nm, row0, nvalid0, nvalid1;
};

// Bit depth of segment s (the shared expert: the layer's depth).
__device__ __forceinline__ int seg_bits(const GroupedArgs &a, int s)
{
    return a.mixed && s < a.E ? mixed_expert_bits(a, s) : a.bits;
}

// Byte offset of routed expert s in the bank.
__device__ __forceinline__ int64_t routed_offset(const GroupedArgs &a, int s)
{
    return a.mixed ? mixed_expert_offset(a, s) : (int64_t)s * a.expert_bytes_routed;
}

template <int PHASE>
__device__ __forceinline__ int seg_ntiles(const GroupedArgs &a, int s)
{
    const int fsg = s < a.E ? a.f : a.fs;
    return PHASE == 0 ? (fsg + 127) / 128 : (a.d + kGN - 1) / kGN;
}

// Items of one segment per n-tile: its m-tiles, in pairs when PAIR.
template <bool PAIR>
__device__ __forceinline__ int seg_items(int cnt)
{
    const int mtc = (cnt + kGM - 1) / kGM;
    return PAIR ? (mtc + 1) / 2 : mtc;
}

template <bool PAIR>
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
    const int c = sm.cnt[lo];
    const int mtc = (c + kGM - 1) / kGM;
    const int per = seg_items<PAIR>(c);
    it.nt = local / per;
    const int mt0 = (PAIR ? 2 : 1) * (local % per);
    it.nm = PAIR && mtc - mt0 >= 2 ? 2 : 1;
    it.row0 = sm.off[lo] + kGM * mt0;
    const int left = c - kGM * mt0;
    it.nvalid0 = left < kGM ? left : kGM;
    it.nvalid1 = left - kGM < kGM ? left - kGM : kGM;
    return it;
}

// ------------------------------------------------------------ roles

// Where an item's code tiles come from: K block kb, copy c (one strip: the
// gate and up tiles of the K block for gate/up, the down tile for down).
template <int BITS, int PHASE>
struct CodeSrc {
    const uint8_t *wb;
    int64_t down_off;
    int nkb, r0, ncopy, fsg, d;
    __device__ CodeSrc(const GroupedArgs &a, const Item &w)
    {
        const bool routed = w.seg < a.E;
        fsg = routed ? a.f : a.fs;
        d = a.d;
        // an item only reaches the instance of its segment's depth (BITS)
        wb = routed ? a.tiles_routed + routed_offset(a, w.seg) : a.tiles_shared;
        down_off = routed ? 2ll * a.d * a.f / 1024 * tile_bytes(BITS) : a.down_off_shared;
        nkb = PHASE == 0 ? a.d / kGK : fsg / kGK;
        r0 = (PHASE == 0 ? 128 * w.nt : kGN * w.nt) / 16;  // first strip
        const int nstrips = PHASE == 0 ? fsg / 16 : a.d / 16;
        const int nc = PHASE == 0 ? 8 : 16;
        ncopy = nstrips - r0 < nc ? nstrips - r0 : nc;
    }
    static constexpr uint32_t csize = PHASE == 0 ? 2 * tile_bytes(BITS) : tile_bytes(BITS);
    __device__ const uint8_t *chunk(int kb, int c) const
    {
        constexpr uint32_t TB = tile_bytes(BITS);
        const int r = r0 + c;
        return PHASE == 0 ? wb + (((int64_t)r * (d / kGK) + kb) * 2) * TB
                          : wb + down_off + ((int64_t)r * (fsg / kGK) + kb) * TB;
    }
};

// Tensor maps of one GEMM launch: the activation matrix (the sorted token
// rows, or h) in boxes of 32, 64 and 128 rows x 64 columns, and the code
// tiles of the routed bank and of the shared expert as 4-D tensors of
// 8-byte elements (tile bytes of one K block of a strip, K blocks, strips,
// experts) read in boxes of one code stage.
struct GMaps {
    CUtensorMap act[3];
    CUtensorMap code[2];  // routed, shared
    int code_tma;         // 1: code stages by tensor copy
};

// Code tiles of every K block, in item order (warp 0).
template <int BITS, int PHASE, bool PAIR>
__device__ void code_producer(const GroupedArgs &a, const GMaps *gm, GSmem &sm, uint8_t *sC)
{
    const int lane = threadIdx.x & 31;
    typedef CodeSrc<BITS, PHASE> Src;
    uint32_t it = 0;
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x) {
        const Item w = item_at<PAIR>(sm, i);
        const Src cs(a, w);
        for (int kb0 = 0; kb0 < cs.nkb; kb0 += code_kb(PAIR), ++it) {
            const int nb = cs.nkb - kb0 < code_kb(PAIR) ? cs.nkb - kb0 : code_kb(PAIR);
            const int s = static_cast<int>(it % code_stages(PAIR));
            const unsigned par = ((it / code_stages(PAIR)) & 1u) ^ 1u;
            if (!__all_sync(0xffffffffu, gwait(sm, &sm.code_empty[s], par, a.status)))
                return;
            if (gm->code_tma) {
                // one box: K blocks kb0 .. kb0 + code_kb - 1 of the item's
                // strips; boxes past the last K block or strip are zero-filled
                // and still count their full size
                if (lane == 0) {
                    const bool routed = w.seg < a.E;
                    mbar_arrive_expect_tx(&sm.code_full[s], code_stage_bytes(BITS, PAIR));
                    sm.last_code[s] = it + 1;
                    tma_load_4d(sC + s * code_stage_bytes(BITS, PAIR), &gm->code[routed ? 0 : 1], 0,
                                kb0, cs.r0, routed ? w.seg : 0, &sm.code_full[s]);
                }
                __syncwarp();
                continue;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&sm.code_full[s], cs.ncopy * nb * Src::csize);
                sm.last_code[s] = it + 1;
            }
            __syncwarp();
            // copy c: the strip's tiles of K blocks kb0 .. kb0 + nb - 1 (contiguous)
            if (lane < cs.ncopy)
                bulk_g2s(sC + s * code_stage_bytes(BITS, PAIR) + lane * code_kb(PAIR) * Src::csize,
                         cs.chunk(kb0, lane), nb * Src::csize, &sm.code_full[s]);
        }
    }
}

// Activation tiles of every K block, in item order (warp 2, lane 0).  Each
// m-tile is loaded in the shortest box that covers its valid rows: the rest
// of the 128-row tile keeps older rows, which only reach accumulator rows
// the epilogue never stores.
template <int PHASE, bool PAIR>
__device__ void act_producer(const GroupedArgs &a, const GMaps *gm, GSmem &sm, uint8_t *sA)
{
    uint32_t it = 0;
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x) {
        const Item w = item_at<PAIR>(sm, i);
        const int fsg = w.seg < a.E ? a.f : a.fs;
        const int nkb = PHASE == 0 ? a.d / kGK : fsg / kGK;
        int bx[2];  // box per m-tile: 0 = 32 rows, 1 = 64, 2 = 128
        uint32_t bytes = 0;
        for (int j = 0; j < w.nm; ++j) {
            const int nv = j == 0 ? w.nvalid0 : w.nvalid1;
            bx[j] = nv <= 32 ? 0 : (nv <= 64 ? 1 : 2);
            bytes += (32u << bx[j]) * (kGK * 2);
        }
        for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = static_cast<int>(it % num_stages(PAIR));
            if (!gwait(sm, &sm.stage_empty[s], ((it / num_stages(PAIR)) & 1u) ^ 1u, a.status))
                return;
            mbar_arrive_expect_tx(&sm.a_full[s], bytes);
            sm.last_a[s] = it + 1;
            for (int j = 0; j < w.nm; ++j)
                tma_load_2d(sA + s * a_stage_bytes(PAIR) + j * kATileBytes, &gm->act[bx[j]],
                            kb * kGK, w.row0 + kGM * j, &sm.a_full[s]);
        }
    }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Decode one 16 x 64 code tile (shared address `tile`) into rows rowbase ..
// rowbase + 15 of a 128-byte-swizzled K-major bf16 tile at `sb`:
// w = (c - L) * (s / L), with c - (L + 1/2) exact in bf16 and one rounding
// in the fused multiply-add.  off[rh][h] = the lane's byte offsets of its
// two 16-byte chunks in rows gq and gq + 8 (swizzle included).
template <int BITS>
__device__ __forceinline__ void decode_tile(uint32_t tile, uint32_t sb, const uint32_t (&off)[2][2],
                                            int lane)
{
    const int gq = lane >> 2;
    constexpr float kInvL = BITS == 4 ? (1.0f / 7.5f) : (1.0f / 1.5f);
    // bf16 128 + c minus 128 + L + 1/2 (136 for Q4, 130 for Q2), both halves
    constexpr uint32_t kSub = BITS == 4 ? 0x43084308u : 0x43024302u;
    const uint32_t sc = lds32(tile + tile_code_bytes(BITS) + 4 * gq);
    uint32_t smul[2], sadd[2];
    {
        const float2 sf = __half22float2(*reinterpret_cast<const __half2 *>(&sc));
        const float s0 = sf.x * kInvL, s1 = sf.y * kInvL;
        smul[0] = pack_bf16x2(s0, s0);
        smul[1] = pack_bf16x2(s1, s1);
        // half of the rounded scale: exact
        sadd[0] = bf16x2_fma(smul[0], 0x3F003F00u, 0x80008000u);
        sadd[1] = bf16x2_fma(smul[1], 0x3F003F00u, 0x80008000u);
    }
    uint32_t v[2][8];  // [rh][m]: columns 16 tig + 2 m, + 1
    if (BITS == 4) {
        const uint4 q = lds128(tile + 16 * lane);
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
        const uint2 q = lds64(tile + 8 * lane);
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
    for (int rh = 0; rh < 2; ++rh)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            sts128(sb + off[rh][h], v[rh][4 * h], v[rh][4 * h + 1], v[rh][4 * h + 2],
                   v[rh][4 * h + 3]);
}

template <int BITS, int PHASE, bool PAIR>
__device__ void decoders(const GroupedArgs &a, GSmem &sm, uint8_t *sB, const uint8_t *sC, int dw)
{
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, tig = lane & 3;
    constexpr uint32_t TB = tile_bytes(BITS);
    uint32_t off[2][2];
#pragma unroll
    for (int rh = 0; rh < 2; ++rh)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            off[rh][h] = (gq + 8 * rh) * 128 + ((((2 * tig + h) ^ gq) & 7) << 4);
    const uint32_t sB0 = smem_u32(sB), sC0 = smem_u32(sC);
    uint32_t it = 0, ic = 0;  // K blocks, code stages
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x) {
        const Item w = item_at<PAIR>(sm, i);
        const int fsg = w.seg < a.E ? a.f : a.fs;
        const int nkb = PHASE == 0 ? a.d / kGK : fsg / kGK;
        const int r0 = (PHASE == 0 ? 128 * w.nt : kGN * w.nt) / 16;
        const int nstrips = PHASE == 0 ? fsg / 16 : a.d / 16;
        // this warp's tile: gate/up copy q/2 holds strip r0 + q/2 (gate tile
        // then up tile per K block), down copy q holds strip r0 + q
        const int q = dw;
        const int strip = PHASE == 0 ? q >> 1 : q;
        const int rowbase = PHASE == 0 ? (q & 1) * 128 + 16 * (q >> 1) : 16 * q;
        constexpr uint32_t csize = PHASE == 0 ? 2 * TB : TB;
        const uint32_t tile_off = strip * code_kb(PAIR) * csize + (PHASE == 0 ? (q & 1) * TB : 0);
        for (int kb0 = 0; kb0 < nkb; kb0 += code_kb(PAIR), ++ic) {
            const int nb = nkb - kb0 < code_kb(PAIR) ? nkb - kb0 : code_kb(PAIR);
            const int s = static_cast<int>(ic % code_stages(PAIR));
            if (!__all_sync(0xffffffffu, gwait(sm, &sm.code_full[s], (ic / code_stages(PAIR)) & 1u, a.status)))
                return;
            const uint32_t cs = sC0 + s * code_stage_bytes(BITS, PAIR) + tile_off;
            for (int j = 0; j < nb; ++j, ++it) {
                const int b = static_cast<int>(it % num_stages(PAIR));
                if (!__all_sync(0xffffffffu, gwait(sm, &sm.stage_empty[b], ((it / num_stages(PAIR)) & 1u) ^ 1u, a.status)))
                    return;
                if (r0 + strip < nstrips)
                    decode_tile<BITS>(cs + j * csize, sB0 + b * kBTileBytes + rowbase * 128, off, lane);
                fence_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sm.b_full[b]);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.code_empty[s]);
        }
    }
}

// Accumulator slots: an item of two m-tiles takes both 256-column slots; an
// item of one m-tile takes the slot after the last single one, so that its
// epilogue overlaps the next item's MMAs.  The MMA issuer and the epilogue
// walk the same item sequence, so they agree on every slot and phase.
struct SlotState {
    uint32_t use0, use1;  // completed uses of slot 0 and 1
    int next;
    __device__ void init()
    {
        use0 = use1 = 0u;
        next = 0;
    }
    __device__ int slot(const Item &w, int j) const { return w.nm == 2 ? j : next; }
    __device__ uint32_t uses(int sl) const { return sl == 0 ? use0 : use1; }
    __device__ void done(const Item &w)
    {
        if (w.nm == 2) {
            ++use0;
            ++use1;
        } else {
            if (next == 0)
                ++use0;
            else
                ++use1;
            next ^= 1;
        }
    }
};

template <int PHASE, bool PAIR>
__device__ void mma_issuer(const GroupedArgs &a, GSmem &sm, const uint8_t *sA, const uint8_t *sB)
{
    uint32_t it = 0;
    SlotState st;
    st.init();
    const uint32_t tbase = sm.tmem_base;
    const uint64_t adesc0 = sw128_desc(smem_u32(sA)), bdesc0 = sw128_desc(smem_u32(sB));
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x) {
        const Item w = item_at<PAIR>(sm, i);
        const int fsg = w.seg < a.E ? a.f : a.fs;
        const int nkb = PHASE == 0 ? a.d / kGK : fsg / kGK;
        const int slot0 = st.slot(w, 0), slot1 = st.slot(w, 1);
        if (!gwait(sm, &sm.acc_empty[slot0], (st.uses(slot0) & 1u) ^ 1u, a.status))
            return;
        if (w.nm == 2 && !gwait(sm, &sm.acc_empty[slot1], (st.uses(slot1) & 1u) ^ 1u, a.status))
            return;
        const uint32_t d0 = tbase + static_cast<uint32_t>(slot0 * kGN);
        const uint32_t d1 = tbase + static_cast<uint32_t>(slot1 * kGN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = static_cast<int>(it % num_stages(PAIR));
            const unsigned par = (it / num_stages(PAIR)) & 1u;
            if (!gwait(sm, &sm.b_full[s], par, a.status))
                return;
            if (!gwait(sm, &sm.a_full[s], par, a.status))
                return;
            tc_fence_after();
            // descriptor start addresses are in 16-byte units: one K step of
            // 16 bf16 is +2, one stage +size/16
            const uint64_t ad = adesc0 + (uint64_t)(s * (a_stage_bytes(PAIR) >> 4));
            const uint64_t bd = bdesc0 + (uint64_t)(s * (kBTileBytes >> 4));
#pragma unroll
            for (int ks = 0; ks < kGK / 16; ++ks)
                umma_bf16(d0, ad + 2 * ks, bd + 2 * ks, (kb | ks) != 0 ? 1u : 0u);
            if (kb == nkb - 1)
                umma_commit(&sm.acc_full[slot0]);  // its epilogue may start now
            if (w.nm == 2) {
#pragma unroll
                for (int ks = 0; ks < kGK / 16; ++ks)
                    umma_bf16(d1, ad + (kATileBytes >> 4) + 2 * ks, bd + 2 * ks,
                              (kb | ks) != 0 ? 1u : 0u);
                if (kb == nkb - 1)
                    umma_commit(&sm.acc_full[slot1]);
            }
            umma_commit(&sm.stage_empty[s]);
        }
        st.done(w);
    }
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;
}

template <int PHASE, bool PAIR>
__device__ void epilogue(const GroupedArgs &a, GSmem &sm)
{
    const int lane = threadIdx.x & 31;
    const int quarter = (threadIdx.x >> 5) & 3;  // tensor-memory lanes 32 q .. 32 q + 31
    const int r = 32 * quarter + lane;
    const uint32_t tbase = sm.tmem_base;
    SlotState st;
    st.init();
    for (int i = blockIdx.x; i < sm.total_items; i += gridDim.x) {
        const Item w = item_at<PAIR>(sm, i);
        const int fsg = w.seg < a.E ? a.f : a.fs;
        for (int j = 0; j < w.nm; ++j) {
            const int sl = st.slot(w, j);
            if (!__all_sync(0xffffffffu, gwait(sm, &sm.acc_full[sl], st.uses(sl) & 1u, a.status)))
                return;
            tc_fence_after();
            const uint32_t taddr = tbase + (static_cast<uint32_t>(32 * quarter) << 16) +
                                   static_cast<uint32_t>(sl * kGN);
            const bool valid = r < (j == 0 ? w.nvalid0 : w.nvalid1);
            const int64_t row = w.row0 + kGM * j + r;
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
                        hv[m] = pack_bf16x2(
                            silu_mul(__uint_as_float(g[2 * m]), __uint_as_float(u[2 * m])),
                            silu_mul(__uint_as_float(g[2 * m + 1]), __uint_as_float(u[2 * m + 1])));
                    if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(a.h + row * a.hstride + n0 + c);
                        dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                        dst[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
                    }
                }
            } else {
                // the row's routing weight applied here, the product stored
                // as bf16: the combine only adds the rows of each token
                const int n0 = kGN * w.nt;
                const float wr = valid ? __ldg(a.roww + row) : 0.f;
                for (int c = 0; c < kGN && n0 + c < a.d; c += 16) {
                    uint32_t o[16];
                    tmem_ld16(taddr + c, o);
                    tmem_wait_ld();
                    if (valid) {
                        uint32_t ov[8];
#pragma unroll
                        for (int m = 0; m < 8; ++m)
                            ov[m] = pack_bf16x2(wr * __uint_as_float(o[2 * m]),
                                                wr * __uint_as_float(o[2 * m + 1]));
                        uint4 *dst = reinterpret_cast<uint4 *>(a.o + row * a.d + n0 + c);
                        dst[0] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                        dst[1] = make_uint4(ov[4], ov[5], ov[6], ov[7]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.acc_empty[sl]);
        }
        st.done(w);
    }
}

template <int BITS, int PHASE, bool PAIR>
__global__ void __launch_bounds__(kGThreads, 1)
    grouped_gemm_kernel(const GroupedArgs a, const __grid_constant__ GMaps maps)
{
    extern __shared__ uint8_t g_smem_raw[];
    __shared__ GSmem sm;
    uint8_t *base = g_smem_raw + ((1024u - (smem_u32(g_smem_raw) & 1023u)) & 1023u);
    constexpr int NS = num_stages(PAIR);
    uint8_t *sA = base;                                // NS activation stages
    uint8_t *sB = sA + NS * a_stage_bytes(PAIR);        // NS x 32 KB decoded weights
    uint8_t *sC = sB + NS * kBTileBytes;                // code_stages(PAIR) code stages
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
                // segments of the other depth belong to the other instance
                if (seg_bits(a, s) == BITS)
                    items = seg_items<PAIR>(c) * seg_ntiles<PHASE>(a, s);
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
            for (int s = 0; s < code_stages(PAIR); ++s) {
                sm.last_code[s] = 0;
                mbar_init(&sm.code_full[s], 1);
                mbar_init(&sm.code_empty[s], kDecWarps);
            }
            for (int s = 0; s < num_stages(PAIR); ++s) {
                sm.last_a[s] = 0;
                mbar_init(&sm.a_full[s], 1);
                mbar_init(&sm.b_full[s], kDecWarps);
                mbar_init(&sm.stage_empty[s], 1);
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
        code_producer<BITS, PHASE, PAIR>(a, &maps, sm, sC);
    } else if (warp == 2) {
        if (lane == 0)
            act_producer<PHASE, PAIR>(a, &maps, sm, sA);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            mma_issuer<PHASE, PAIR>(a, sm, sA, sB);
            // every MMA issued so far has completed once this commit lands
            umma_commit(&sm.drain);
            if (!mbar_wait_bounded(&sm.drain, 0)) {
                set_status(a.status, kStatusTimeout);
                *reinterpret_cast<volatile int *>(&sm.fail) = 1;
            }
        }
        __syncwarp();
    } else if (warp < kEpiWarp0 + kEpiWarpsG) {
        epilogue<PHASE, PAIR>(a, sm);
    } else if (decoder_index(warp) >= 0) {
        decoders<BITS, PHASE, PAIR>(a, sm, sB, sC, decoder_index(warp));
    }
    __syncwarp();
    // After a failure the consumers may have left copies unwaited: the
    // producers wait (bounded) for the last phase they filled on every stage,
    // so no copy is in flight when the CTA exits.
    if (*reinterpret_cast<volatile int *>(&sm.fail)) {
        if (warp == 0 && lane < code_stages(PAIR)) {
            const uint32_t last = sm.last_code[lane];
            if (last > 0 && !mbar_wait_bounded(&sm.code_full[lane], ((last - 1) / code_stages(PAIR)) & 1u))
                set_status(a.status, kStatusTimeout);
        }
        if (warp == 2 && lane < num_stages(PAIR)) {
            const uint32_t last = sm.last_a[lane];
            if (last > 0 && !mbar_wait_bounded(&sm.a_full[lane], ((last - 1) / num_stages(PAIR)) & 1u))
                set_status(a.status, kStatusTimeout);
        }
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

// Inclusive scan of v over a 256-thread block; *total gets the block sum.
// s_w holds 8 ints; the caller syncs before reusing it.
__device__ __forceinline__ int block_scan_incl(int v, int *s_w, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += u;
    }
    if (lane == 31)
        s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = lane < 8 ? s_w[lane] : 0;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, wv, o);
            if (lane >= o)
                wv += u;
        }
        if (lane < 8)
            s_w[lane] = wv;
    }
    __syncthreads();
    total = s_w[7];
    return incl + (warp > 0 ? s_w[warp - 1] : 0);
}

// The counting sort of the (token, slot) selections by expert, stable in
// token order.  The router leaves each 8-token tile's count per expert; one
// CTA per expert turns its column into exclusive bases in tile order (in
// place) and its total; the last CTA to finish writes the segment table:
// first row of every segment (rows padded to 128; the shared expert, all T
// tokens, last) and its row count.
__global__ void __launch_bounds__(256) grp_scan_kernel(const GroupedArgs a)
{
    __shared__ int s_w[8];
    __shared__ int s_last;
    const int e = blockIdx.x, tid = threadIdx.x;
    const int E = a.E, nseg = E + (a.has_shared ? 1 : 0);
    int carry = 0;
    for (int b0 = 0; b0 < a.ntiles; b0 += 256) {
        const int tl = b0 + tid;
        int32_t *p = a.tilecnt + (int64_t)tl * E + e;
        const int c = tl < a.ntiles ? __ldcg(p) : 0;
        int tot;
        const int incl = block_scan_incl(c, s_w, tot);
        if (tl < a.ntiles)
            *p = carry + incl - c;
        carry += tot;
        __syncthreads();
    }
    if (tid == 0)
        a.seg[nseg + 1 + e] = carry;
    __threadfence();
    __syncthreads();
    if (tid == 0)
        s_last = atomicAdd(a.scan_ctr, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    int run = 0;
    for (int s0 = 0; s0 < nseg; s0 += 256) {
        const int sg = s0 + tid;
        const int c = sg < nseg ? (sg < E ? __ldcg(a.seg + nseg + 1 + sg) : static_cast<int>(a.T)) : 0;
        const int padc = (c + kGM - 1) / kGM * kGM;
        int tot;
        const int incl = block_scan_incl(padc, s_w, tot);
        if (sg < nseg) {
            a.seg[sg] = run + incl - padc;
            if (sg == E)
                a.seg[nseg + 1 + E] = static_cast<int>(a.T);
        }
        run += tot;
        __syncthreads();
    }
    if (tid == 0) {
        a.seg[nseg] = run;
        if (run > a.rows) {  // cannot happen with the planned row count
            set_status(a.status, kStatusBadArg);
            for (int sg = 0; sg < nseg; ++sg)
                a.seg[nseg + 1 + sg] = 0;
        }
        *a.scan_ctr = 0u;
    }
}

// Row of every (token, slot): its segment's first row + its tile's base
// inside the expert + its rank among the tile's earlier tokens that chose
// the same expert (a token chooses an expert once).  Then x_sorted[row] =
// bf16(x[t]) for every slot (and the shared segment).
template <bool XBF16>
__global__ void __launch_bounds__(256) gather_kernel(const GroupedArgs a, const void *x)
{
    __shared__ int32_t s_rows[SMOE_MAX_TOPK_DEV + 1];
    const int64_t t = blockIdx.x;
    const int d = a.d, k = a.k, E = a.E;
    const int nslot = k + (a.has_shared ? 1 : 0);
    if (static_cast<int>(threadIdx.x) < nslot) {
        const int j = threadIdx.x;
        int64_t row = -1;
        if (j < k) {
            const int e = __ldg(a.ids + t * k + j);
            if (e >= 0 && e < E) {
                const int64_t tile = t / kPairCols;
                int local = 0;
                for (int64_t t2 = tile * kPairCols; t2 < t; ++t2)
                    for (int j2 = 0; j2 < k; ++j2)
                        local += __ldg(a.ids + t2 * k + j2) == e ? 1 : 0;
                row = (int64_t)__ldg(a.seg + e) + __ldg(a.tilecnt + tile * E + e) + local;
            }
        } else {
            row = (int64_t)__ldg(a.seg + E) + t;
        }
        if (row < 0 || row >= a.rows)
            row = -1;
        s_rows[j] = static_cast<int32_t>(row);
        a.rows_of[t * (k + 1) + j] = static_cast<int32_t>(row);
        if (row >= 0)  // the weight the down GEMM's epilogue applies to this row
            a.roww[row] = j < k ? __ldg(a.w + t * k + j) : __ldg(a.sw + t);
    }
    __syncthreads();
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
            const int32_t r = s_rows[j];
            if (r >= 0)
                *reinterpret_cast<uint4 *>(a.xs + (int64_t)r * d + c) = v;
        }
    }
}

// y[t] = sum of the token's weighted rows o[row(t, j)] (already scaled by
// w[t, j] in the down GEMM) in rank order, then the shared expert's row.
__global__ void __launch_bounds__(256) grouped_combine_kernel(const uint16_t *o, int64_t T, int d, int k,
                                                              int has_shared, const int32_t *rows,
                                                              int64_t nrows, float *y)
{
    const int64_t t = blockIdx.x;
    const int nslot = k + (has_shared ? 1 : 0);
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < nslot; ++j) {
            const int32_t r = __ldg(rows + t * (k + 1) + j);
            if (r < 0 || r >= nrows)
                continue;
            const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(o + (int64_t)r * d + c));
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                acc[2 * m] += bf16lo_to_f32(u[m]);
                acc[2 * m + 1] += bf16hi_to_f32(u[m]);
            }
        }
        float4 *dst = reinterpret_cast<float4 *>(y + t * d + c);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// ------------------------------------------------------------ router logits

// logits[t, e] = sum_i x[t, i] * Wr[e, i] for a batch of bf16 tokens, on the
// tensor cores: one CTA per 128 tokens x 128 experts, both operands by TMA
// (128-byte swizzle, 4 stages), fp32 accumulation in tensor memory ("Model
// Agnosticism": the gate has max_experts_per_layer rows).  Warp 0 lane 0
// loads, warp 1 lane 0 issues the MMAs, all four warps write the logits.
constexpr int kRStages = 4;
constexpr uint32_t kRIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) |
                             ((128u >> 4) << 24);

struct RSmem {
    uint64_t full[kRStages], empty[kRStages], done;
    uint32_t tmem_base;
    uint32_t last[kRStages];
    int fail;
};

__global__ void __launch_bounds__(128, 1)
    tc_logits_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                     int64_t T, int d, int E, int Epad, uint32_t stage_tx, float *logits, int *status)
{
    extern __shared__ uint8_t r_smem_raw[];
    __shared__ RSmem sm;
    uint8_t *base = r_smem_raw + ((1024u - (smem_u32(r_smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = base, *sB = base + kRStages * kATileBytes;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t m0 = (int64_t)blockIdx.x * 128;
    const int n0 = blockIdx.y * 128;
    const int nkb = d / kGK;
    if (tid == 0) {
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
            sm.last[s] = 0;
        }
        mbar_init(&sm.done, 1);
        sm.fail = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sm.tmem_base)),
                     "r"(128)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    volatile int *fail = &sm.fail;
    if (tid == 0) {
        for (int kb = 0; kb < nkb && !*fail; ++kb) {
            const int s = kb % kRStages;
            if (!mbar_wait_bounded(&sm.empty[s], ((kb / kRStages) & 1) ^ 1)) {
                set_status(status, kStatusTimeout);
                *fail = 1;
                break;
            }
            mbar_arrive_expect_tx(&sm.full[s], stage_tx);
            sm.last[s] = kb + 1;
            tma_load_2d(sA + s * kATileBytes, &mx, kb * kGK, static_cast<int>(m0), &sm.full[s]);
            tma_load_2d(sB + s * kATileBytes, &mw, kb * kGK, n0, &sm.full[s]);
        }
    } else if (tid == 32) {
        const uint64_t ad0 = sw128_desc(smem_u32(sA)), bd0 = sw128_desc(smem_u32(sB));
        for (int kb = 0; kb < nkb && !*fail; ++kb) {
            const int s = kb % kRStages;
            if (!mbar_wait_bounded(&sm.full[s], (kb / kRStages) & 1)) {
                set_status(status, kStatusTimeout);
                *fail = 1;
                break;
            }
            tc_fence_after();
            const uint64_t off = (uint64_t)(s * (kATileBytes >> 4));
#pragma unroll
            for (int ks = 0; ks < kGK / 16; ++ks)
                asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                             "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tbase),
                             "l"(ad0 + off + 2 * ks), "l"(bd0 + off + 2 * ks), "r"(kRIdesc),
                             "r"((kb | ks) != 0 ? 1u : 0u)
                             : "memory");
            umma_commit(&sm.empty[s]);
        }
        umma_commit(&sm.done);
    }
    __syncwarp();
    // every warp: its 32 rows of the accumulator
    const bool ok = mbar_wait_bounded(&sm.done, 0);
    if (!ok && lane == 0) {
        set_status(status, kStatusTimeout);
        *fail = 1;
    }
    tc_fence_after();
    if (__all_sync(0xffffffffu, ok) && !*fail) {
        const int64_t row = m0 + 32 * warp + lane;
        for (int c = 0; c < 128 && n0 + c < E; c += 16) {
            uint32_t v[16];
            tmem_ld16(tbase + (static_cast<uint32_t>(32 * warp) << 16) + c, v);
            tmem_wait_ld();
            if (row < T)
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (n0 + c + q < E)
                        logits[row * Epad + n0 + c + q] = __uint_as_float(v[q]);
        }
    }
    // after a failure: no copy of this CTA may still be in flight
    if (*fail && tid < kRStages && sm.last[tid] > 0 &&
        !mbar_wait_bounded(&sm.full[tid], ((sm.last[tid] - 1) / kRStages) & 1))
        set_status(status, kStatusTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(128)
                     : "memory");
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

// Tensor map of a row-major bf16 matrix [rows, cols] read in box_rows x 64
// boxes with the 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int box_rows = kGM)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Code tiles of a bank region as a 4-D tensor of 8-byte elements: csize
// bytes (one K block of a strip), G K blocks, nstr strips, nexp experts
// expert_stride bytes apart; boxes of box_kb K blocks x box_str strips.
// False where the encoder refuses it or a box would exceed the tensor.
bool make_code_map(CUtensorMap *m, const uint8_t *base, uint32_t csize, int G, int nstr, int nexp,
                   int64_t expert_stride, int box_kb, int box_str)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base || box_kb > G || box_str > nstr || csize % 16 || expert_stride % 16)
        return false;
    const cuuint64_t dims[4] = {csize / 8, static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(nstr),
                                static_cast<cuuint64_t>(nexp)};
    const cuuint64_t strides[3] = {csize, static_cast<cuuint64_t>(G) * csize,
                                   static_cast<cuuint64_t>(expert_stride)};
    const cuuint32_t box[4] = {csize / 8, static_cast<cuuint32_t>(box_kb),
                               static_cast<cuuint32_t>(box_str), 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, const_cast<uint8_t *>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The maps of one GEMM launch (phase 0: gate/up, 1: down) over activation
// matrix `act` [rows, cols].
bool make_gemm_maps(GMaps *g, const GroupedArgs &a, int phase, bool pair, const void *act, int cols)
{
    memset(g, 0, sizeof *g);
    for (int b = 0; b < 3; ++b)
        if (!make_map(&g->act[b], act, a.rows, cols, 32 << b))
            return false;
    if (a.mixed)
        return true;  // experts of two sizes: per-strip bulk copies
    const uint32_t TB = tile_bytes(a.bits);
    const uint32_t csize = phase == 0 ? 2 * TB : TB;
    const int kbx = pair ? code_kb(true) : code_kb(false), strips = phase == 0 ? 8 : 16;
    bool ok = make_code_map(&g->code[0],
                            a.tiles_routed + (phase == 0 ? 0 : 2ll * a.d * a.f / 1024 * TB), csize,
                            phase == 0 ? a.d / kGK : a.f / kGK, phase == 0 ? a.f / 16 : a.d / 16,
                            a.E, a.expert_bytes_routed, kbx, strips);
    if (ok && a.has_shared)
        ok = make_code_map(&g->code[1], a.tiles_shared + (phase == 0 ? 0 : a.down_off_shared), csize,
                           phase == 0 ? a.d / kGK : a.fs / kGK, phase == 0 ? a.fs / 16 : a.d / 16, 1,
                           3ll * a.d * a.fs / 1024 * TB, kbx, strips);
    g->code_tma = ok ? 1 : 0;
    return true;
}

template <int BITS, int PHASE, bool PAIR>
cudaError_t launch_gemm_t(const GroupedArgs &a, const GMaps &maps, cudaStream_t s)
{
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev >= 0 && dev < 64 && !attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<BITS, PHASE, PAIR>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 grouped_smem_bytes(BITS, PAIR));
            if (e != cudaSuccess)
                return e;
            attr_set[dev] = true;
        }
    }
    grouped_gemm_kernel<BITS, PHASE, PAIR>
        <<<device_sm_count(), kGThreads, grouped_smem_bytes(BITS, PAIR), s>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_logits(const uint16_t *x, const uint16_t *router_w, int64_t T, int d, int E,
                             int Epad, float *logits, int *status, cudaStream_t s)
{
    if (T == 0)
        return cudaSuccess;
    // boxes never taller than the matrices: rows past the end of a box are
    // left over from earlier stages and only reach accumulator rows/columns
    // that are not written out
    const int bx = T < kGM ? static_cast<int>(T) : kGM;
    const int bw = E < 128 ? E : 128;
    CUtensorMap mx, mw;
    if (!make_map(&mx, x, T, d, bx) || !make_map(&mw, router_w, E, d, bw))
        return cudaErrorInvalidValue;
    const int smem = 2 * kRStages * kATileBytes + 1024;
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev >= 0 && dev < 64 && !attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(tc_logits_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess)
                return e;
            attr_set[dev] = true;
        }
    }
    const dim3 grid(static_cast<unsigned>((T + 127) / 128), static_cast<unsigned>((E + 127) / 128));
    const uint32_t tx = static_cast<uint32_t>(kGK * 2 * (bx + bw));
    tc_logits_kernel<<<grid, 128, smem, s>>>(mx, mw, T, d, E, Epad, tx, logits, status);
    return cudaGetLastError();
}

int64_t grouped_max_rows(int64_t T, int E, int k, int has_shared)
{
    const int64_t tk = T * k;
    const int64_t segs = tk < E ? tk : E;
    int64_t r = tk + segs * (kGM - 1);
    if (has_shared)
        r += T + kGM - 1;
    return (r + kGM - 1) / kGM * kGM;
}

cudaError_t launch_grouped(const GroupedArgs &a, const void *x, int x_bf16, float *y, int stage_mask,
                           cudaStream_t s)
{
    if (a.T == 0)
        return cudaSuccess;
    const unsigned nt = static_cast<unsigned>(a.T);
    cudaError_t e = cudaSuccess;
    if (stage_mask & 1) {  // sort and gather
        grp_scan_kernel<<<a.E, 256, 0, s>>>(a);
        if (x_bf16)
            gather_kernel<true><<<nt, 256, 0, s>>>(a, x);
        else
            gather_kernel<false><<<nt, 256, 0, s>>>(a, x);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    // pairs of m-tiles once the experts average two or more
    const bool pair = a.T * a.k >= 2ll * kGM * a.E;
    // the depths present: one GEMM instance per depth, each taking only the
    // segments of its own depth
    const bool layer_depth = !a.mixed || a.has_shared;  // a segment at a.bits
    bool has4 = layer_depth && a.bits == 4, has2 = layer_depth && a.bits == 2;
    if (a.mixed)
        for (int ex = 0; ex < a.E; ++ex)
            ((a.q4mask[ex >> 5] >> (ex & 31)) & 1u ? has4 : has2) = true;
    if (stage_mask & 2) {  // gate/up GEMM + SiLU(g) * u
        GMaps mx;
        if (!make_gemm_maps(&mx, a, 0, pair, a.xs, a.d))
            return cudaErrorInvalidValue;
        if (has4 && (e = pair ? launch_gemm_t<4, 0, true>(a, mx, s)
                              : launch_gemm_t<4, 0, false>(a, mx, s)) != cudaSuccess)
            return e;
        if (has2 && (e = pair ? launch_gemm_t<2, 0, true>(a, mx, s)
                              : launch_gemm_t<2, 0, false>(a, mx, s)) != cudaSuccess)
            return e;
    }
    if (stage_mask & 4) {  // down GEMM + combine
        GMaps mh;
        if (!make_gemm_maps(&mh, a, 1, pair, a.h, a.hstride))
            return cudaErrorInvalidValue;
        if (has4 && (e = pair ? launch_gemm_t<4, 1, true>(a, mh, s)
                              : launch_gemm_t<4, 1, false>(a, mh, s)) != cudaSuccess)
            return e;
        if (has2 && (e = pair ? launch_gemm_t<2, 1, true>(a, mh, s)
                              : launch_gemm_t<2, 1, false>(a, mh, s)) != cudaSuccess)
            return e;
        grouped_combine_kernel<<<nt, 256, 0, s>>>(a.o, a.T, a.d, a.k, a.has_shared, a.rows_of,
                                                  a.rows, y);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace smoe
