// common.cuh -- device helpers shared by the libsmoe kernels (sm_103a).
//
// Tile layout of a quantised matrix W [R, K] (R = output rows, K = input):
//   tile     = 16 rows x 64 input columns (one quantisation group per row)
//   codes    = 512 B (Q4) or 256 B (Q2) in the register order of the
//              mma.sync m16n8k16 A fragment (see tile_code_bit below)
//   scales   = 16 fp16 right after the codes, row r at halfword 2*(r&7)+(r>>3)
//   strip    = the tiles of 16 output rows over all of K, in group order;
//              gate/up strips interleave the gate and up tile of each group
//   expert   = gate/up strips (f/16 of them, 2*d/64 tiles each), then down
//              strips (d/16 of them, f/64 tiles each)
// so each matrix is one contiguous tile stream and every tile is 16-byte
// aligned.  Within a group the 64 input columns are permuted so that lane
// (gq, tig) of an mma fragment owns columns 16*tig .. 16*tig + 15; the
// activation side reads the same columns, so the permutation cancels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace smoe {

constexpr int kGroup = 64;
constexpr int kTileRows = 16;

__host__ __device__ constexpr int tile_code_bytes(int bits) { return bits * 128; }
__host__ __device__ constexpr int tile_bytes(int bits) { return bits * 128 + 32; }

// Banks whose experts each have their own depth: bit e of Args::q4mask
// (8 words) set = expert e is Q4, clear = Q2; the experts lie back to back
// at their own sizes (3 d f / 1024 tiles each).  Constant indices only, so
// the mask stays in kernel parameter space.
template <class Args>
__device__ __forceinline__ uint32_t q4_word(const Args &a, int w)
{
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v = i == w ? a.q4mask[i] : v;
    return v;
}
template <class Args>
__device__ __forceinline__ int mixed_expert_bits(const Args &a, int e)
{
    return (q4_word(a, e >> 5) >> (e & 31)) & 1u ? 4 : 2;
}
// Byte offset of expert e: the Q2 size of every expert before it plus the
// Q4 surplus of the Q4 ones among them.
template <class Args>
__device__ __forceinline__ int64_t mixed_expert_offset(const Args &a, int e)
{
    int n4 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t m = a.q4mask[i];
        if (i < (e >> 5))
            n4 += __popc(m);
        else if (i == (e >> 5))
            n4 += __popc(m & ((1u << (e & 31)) - 1u));
    }
    const int64_t tiles = 3ll * a.d * a.f / 1024;
    return tiles * ((int64_t)e * tile_bytes(2) + (int64_t)n4 * (tile_bytes(4) - tile_bytes(2)));
}

// Bit position, inside lane t's code word(s) of a tile, of the code for
// W[row gq + 8*rh][column 16*tig + 4*j + e] (j = k-subtile 0..3, e = 0..3).
// Q4: word j of the lane's four 32-bit words; register a_i (i = rh + 2*(e>>1))
//     is (word >> 4i) & 0x000F000F, so the code sits at 4i (e even) or
//     16 + 4i (e odd).
// Q2: word j>>1 of the lane's two words; a_i of k-subtile j comes from the
//     word shifted by v = 8*(j&1) + 4*rh and masked at slot 2*(e>>1), i.e.
//     the code sits at 16*(e&1) + v + 2*(e>>1).  Slot 2 holds codes times 4
//     once decoded, so the matching activations are pre-scaled by 1/4.
__host__ __device__ inline int tile_code_word(int bits, int j) { return bits == 4 ? j : (j >> 1); }
__host__ __device__ inline int tile_code_bit(int bits, int j, int rh, int e)
{
    if (bits == 4)
        return 16 * (e & 1) + 4 * (rh + 2 * (e >> 1));
    return 16 * (e & 1) + 8 * (j & 1) + 4 * rh + 2 * (e >> 1);
}
__host__ __device__ inline int tile_scale_half(int r) { return 2 * (r & 7) + (r >> 3); }

// Device status word codes (one per device, cleared by the host query).
enum : int { kStatusOk = 0, kStatusBadExpert = 1, kStatusTimeout = 2, kStatusBadArg = 3 };

// Bounded waits give up after this many SM cycles (~2 s); in practice a wait
// ends in microseconds, so reaching the bound means a broken pipeline.
constexpr long long kWaitCycles = 4000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Plain arrival (count 1) with release semantics at CTA scope: the thread's
// earlier shared-memory reads of the guarded buffer are done.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Non-blocking: true if the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Returns true once the phase with the given parity has completed.  The
// waiting thread is suspended by the hardware (up to the hint, 0.5 ms) and
// woken when the phase completes, so a waiting warp takes no issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity), "r"(500000u)
                 : "memory");
    return ok != 0;
}

// Bounded wait (about kWaitCycles SM cycles); returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles)
            return false;
    return true;
}

// 1-D bulk copy global -> shared through the TMA engine, completing on an
// mbarrier (transaction bytes).  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// D = A * B + C for one m16n8k16 bf16 tile, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B + C with C in separate registers (the first mma of a chain).
__device__ __forceinline__ void mma_bf16_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                           float c0, float c1, float c2, float c3)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1),
                   "f"(c2), "f"(c3));
}

// bf16x2 with lo = a, hi = b (round to nearest even).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Split two fp32 values into bf16x2 hi + bf16x2 lo with hi + lo ~ x to ~2^-16.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf16x2(x0, x1);
    float r0 = x0 - bf16lo_to_f32(hi);
    float r1 = x1 - bf16hi_to_f32(hi);
    lo = pack_bf16x2(r0, r1);
}

// Multiply both bf16 halves by 1/4 (exact: power of two, no underflow for
// normal activations).
__device__ __forceinline__ uint32_t bf16x2_quarter(uint32_t v)
{
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&v);
    __nv_bfloat162 q = __hmul2(h, __floats2bfloat162_rn(0.25f, 0.25f));
    return *reinterpret_cast<uint32_t *>(&q);
}

__device__ __forceinline__ void set_status(int *status, int code)
{
    if (status)
        atomicCAS(status, 0, code);
}

__device__ __forceinline__ float ld_cg_f32(const float *p) { return __ldcg(p); }

}  // namespace smoe
