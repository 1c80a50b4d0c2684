// expert.cu -- fused dequant-multiply expert GEMV for small token counts
// ("SMOE Quantisation", Decoding: the weight is decoded in registers as
// (code - L) / L * scale and multiplied straight away; the matrix is never
// materialised).
//
// Work: a "pair" is one expert applied to up to 8 tokens.  Phase 0 computes
// h = SiLU(W_gate x) * (W_up x) for every pair, phase 1 computes o = W_down h
// and the routing-weighted combine.  The tiles of all pairs form one stream
// (each pair's matrix is contiguous in the tile layout); the stream is cut
// into equal contiguous ranges, one per warp (stream-K), so every warp reads
// the same number of bytes.  Each warp streams its range through a private
// ring of shared-memory stages filled by TMA bulk copies (cp.async.bulk) and
// completed on mbarriers, so ~140 KB per SM is in flight without registers.
//
// Decode in registers: a code c becomes the bf16 value 128 + c by OR-ing the
// exponent pattern 0x4300 over the masked bits (Q2 slot 2 gives 128 + 4c and
// its activations are pre-scaled by 1/4).  mma.sync m16n8k16 multiplies the
// 16 x 16 code block by the activations (8 token columns) with fp32
// accumulation; the accumulator starts at -(128 + L) * sum(x) per group (Q2:
// -(129.5 X0 + 33.5 X1)) so it ends at sum((c - L) x) exactly up to fp32
// rounding, then one FMA per output applies the group's fp16 scale.
//
// Reductions are deterministic: a block (128 output rows x all K) finished by
// one warp is finalised in registers; a block shared by several warps is
// finalised by the last of them to arrive (an atomic counter), which sums
// the partials in warp order.  The down phase's combine over the k experts
// (and the shared expert) is done per 128-row block by the last pair to
// finish that block, in rank order.  No float atomics anywhere.
#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStageTiles = 4;
constexpr int kStages = 4;

__host__ __device__ constexpr int smem_bytes(int bits)
{
    return kWarps * kStages * kStageTiles * tile_bytes(bits) + kWarps * kStages * 8;
}

__device__ __forceinline__ int64_t warp_of(int64_t u, int64_t W, int64_t U)
{
    return ((u + 1) * W - 1) / U;
}

template <int BITS, bool SPLIT, int PHASE>
__global__ void __launch_bounds__(kThreads) expert_kernel(const ExpertArgs a)
{
    constexpr int TB = tile_bytes(BITS);
    constexpr int CB = tile_code_bytes(BITS);
    constexpr float L = BITS == 4 ? 7.5f : 1.5f;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tig = lane & 3;
    uint8_t *ring = smem + warp * (kStages * kStageTiles * TB);
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(smem + kWarps * kStages * kStageTiles * TB) + warp * kStages;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    pdl_wait();
    pdl_launch_dependents();

    const int P_r = __ldcg(a.meta + 0);
    const int P_t = __ldcg(a.meta + 1);
    const int d = a.d;
    // geometry: rows x K per pair
    const int Kr = PHASE == 0 ? d : a.f;
    const int Ks = PHASE == 0 ? d : a.fs;
    const int rows_r = PHASE == 0 ? 2 * a.f : d;  // gate+up rows count twice
    const int rows_s = PHASE == 0 ? 2 * a.fs : d;
    const int64_t U_r = (int64_t)rows_r * Kr / 1024;
    const int64_t U_s = (P_t > P_r) ? (int64_t)rows_s * Ks / 1024 : 0;
    const int64_t U = (int64_t)P_r * U_r + (int64_t)(P_t - P_r) * U_s;
    const int64_t Wall = (int64_t)gridDim.x * kWarps;
    const int64_t W = U < Wall ? U : Wall;
    const int64_t w = (int64_t)blockIdx.x * kWarps + warp;
    if (w >= W)
        return;
    const int64_t u0 = w * U / W, u1 = (w + 1) * U / W;

    // tile u -> (pair, local tile, geometry)
    auto locate = [&](int64_t u, int &p, int64_t &lt, int &G) {
        if (u < (int64_t)P_r * U_r) {
            p = static_cast<int>(u / U_r);
            lt = u - (int64_t)p * U_r;
            G = Kr / kGroup;
        } else {
            int64_t v = u - (int64_t)P_r * U_r;
            int q = static_cast<int>(v / U_s);
            p = P_r + q;
            lt = v - (int64_t)q * U_s;
            G = Ks / kGroup;
        }
    };
    auto tile_src = [&](int p, int64_t lt) -> const uint8_t * {
        const int32_t *pr = a.pairs + p * kPairInts;
        int e = __ldcg(pr);
        const uint8_t *base;
        if (e >= 0) {
            base = a.tiles_routed + (int64_t)e * a.expert_bytes_routed +
                   (PHASE == 0 ? 0 : a.down_off_routed);
        } else {
            base = a.tiles_shared + (PHASE == 0 ? 0 : a.down_off_shared);
        }
        return base + lt * TB;
    };

    // ---- producer: lane 0 issues stage s (tiles [u0 + s*ST, ...)) into slot s % NS
    const int64_t nst = (u1 - u0 + kStageTiles - 1) / kStageTiles;
    auto issue = [&](int64_t s) {
        if (s >= nst)
            return;
        const int slot = static_cast<int>(s % kStages);
        int64_t ua = u0 + s * kStageTiles;
        int64_t ub = ua + kStageTiles < u1 ? ua + kStageTiles : u1;
        mbar_arrive_expect_tx(&bars[slot], static_cast<unsigned>((ub - ua) * TB));
        uint8_t *dst = ring + slot * (kStageTiles * TB);
        while (ua < ub) {
            int p, G;
            int64_t lt;
            locate(ua, p, lt, G);
            int64_t pair_end = ua + ((p < P_r ? U_r : U_s) - lt);
            int64_t ue = pair_end < ub ? pair_end : ub;
            bulk_g2s(dst, tile_src(p, lt), static_cast<unsigned>((ue - ua) * TB), &bars[slot]);
            dst += (ue - ua) * TB;
            ua = ue;
        }
    };
    if (lane == 0)
        for (int s = 0; s < kStages; ++s)
            issue(s);

    // ---- activation fragments for (pair, group): raw loads + bias
    struct BRaw {
        uint4 v[SPLIT || PHASE == 1 ? 4 : 2];
        float2 xs0, xs1;  // (X0, X1) of columns 2tig, 2tig+1
    };
    auto load_b = [&](int p, int g, int G, BRaw &r) {
        const int32_t *pr = a.pairs + p * kPairInts;
        const int ncols = __ldcg(pr + 1);
        const bool valid = gq < ncols;
        constexpr int NV = SPLIT || PHASE == 1 ? 4 : 2;
        if (PHASE == 0) {
            const int tok = valid ? __ldcg(pr + 2 + gq) : 0;
            if (SPLIT) {
                const float *row = reinterpret_cast<const float *>(a.x) + (int64_t)tok * d +
                                   g * kGroup + 16 * tig;
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    r.v[i] = valid ? __ldg(reinterpret_cast<const uint4 *>(row) + i)
                                   : make_uint4(0, 0, 0, 0);
            } else {
                const uint16_t *row = reinterpret_cast<const uint16_t *>(a.x) + (int64_t)tok * d +
                                      g * kGroup + 16 * tig;
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    r.v[i] = valid ? __ldg(reinterpret_cast<const uint4 *>(row) + i)
                                   : make_uint4(0, 0, 0, 0);
            }
        } else {
            const float *row = a.h + ((int64_t)p * kPairCols + gq) * (a.f > a.fs ? a.f : a.fs) +
                               g * kGroup + 16 * tig;
#pragma unroll
            for (int i = 0; i < NV; ++i)
                r.v[i] = valid ? __ldcg(reinterpret_cast<const uint4 *>(row) + i)
                               : make_uint4(0, 0, 0, 0);
        }
        // bias sums for the two output columns this lane accumulates
        const int c0 = 2 * tig, c1 = 2 * tig + 1;
        float2 z = make_float2(0.f, 0.f);
        if (PHASE == 0) {
            const int t0 = c0 < ncols ? __ldcg(pr + 2 + c0) : -1;
            const int t1 = c1 < ncols ? __ldcg(pr + 2 + c1) : -1;
            r.xs0 = t0 >= 0 ? __ldcg(reinterpret_cast<const float2 *>(a.xsum) +
                                     (int64_t)t0 * (d / kGroup) + g)
                            : z;
            r.xs1 = t1 >= 0 ? __ldcg(reinterpret_cast<const float2 *>(a.xsum) +
                                     (int64_t)t1 * (d / kGroup) + g)
                            : z;
        } else {
            const int fmax64 = (a.f > a.fs ? a.f : a.fs) / kGroup;
            r.xs0 = c0 < ncols ? __ldcg(reinterpret_cast<const float2 *>(a.hsum) +
                                        ((int64_t)p * kPairCols + c0) * fmax64 + g)
                               : z;
            r.xs1 = c1 < ncols ? __ldcg(reinterpret_cast<const float2 *>(a.hsum) +
                                        ((int64_t)p * kPairCols + c1) * fmax64 + g)
                               : z;
        }
        (void)G;
    };

    // fragments ready for the mma
    uint32_t b0[4], b1[4], b0l[4], b1l[4];
    float bias0 = 0.f, bias1 = 0.f;
    auto cook_b = [&](const BRaw &r) {
        if (SPLIT || PHASE == 1) {
            const float *xv = reinterpret_cast<const float *>(r.v);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                split_bf16x2(xv[4 * j + 0], xv[4 * j + 1], b0[j], b0l[j]);
                split_bf16x2(xv[4 * j + 2], xv[4 * j + 3], b1[j], b1l[j]);
            }
        } else {
            const uint32_t *xv = reinterpret_cast<const uint32_t *>(r.v);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                b0[j] = xv[2 * j];
                b1[j] = xv[2 * j + 1];
                b0l[j] = b1l[j] = 0u;
            }
        }
        if (BITS == 2) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                b1[j] = bf16x2_quarter(b1[j]);
                b1l[j] = bf16x2_quarter(b1l[j]);
            }
            bias0 = 129.5f * r.xs0.x + 33.5f * r.xs0.y;
            bias1 = 129.5f * r.xs1.x + 33.5f * r.xs1.y;
        } else {
            bias0 = 135.5f * (r.xs0.x + r.xs0.y);
            bias1 = 135.5f * (r.xs1.x + r.xs1.y);
        }
    };

    float acc[8][4];
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            acc[s][e] = 0.f;

    // ---- block finalisation
    auto finalize = [&](int p, int b, float (&v)[8][4]) {
        const int32_t *pr = a.pairs + p * kPairInts;
        const int ncols = __ldcg(pr + 1);
        const float invL = 1.0f / L;
        const int c0 = 2 * tig;
        if (PHASE == 0) {
            const int fmax = a.f > a.fs ? a.f : a.fs;
            float hs[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [col][class]
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float g = v[2 * i][e] * invL;
                    const float u = v[2 * i + 1][e] * invL;
                    const float hv = g / (1.0f + expf(-g)) * u;
                    const int col = c0 + (e & 1);
                    const int row = 64 * b + 16 * i + gq + 8 * (e >> 1);
                    if (col < ncols)
                        a.h[((int64_t)p * kPairCols + col) * fmax + row] = hv;
                    hs[e & 1][0] += hv;
                }
            // class of row within the 64-row group: (gq >> 1) & 1
            const int cls = (gq >> 1) & 1;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float s = hs[c][0];
                s += __shfl_xor_sync(0xffffffffu, s, 4);
                s += __shfl_xor_sync(0xffffffffu, s, 16);
                hs[c][0] = s;
            }
            if ((gq & 5) == 0) {  // gq in {0, 2}: one lane per (tig, class)
                const int fmax64 = fmax / kGroup;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col = c0 + c;
                    if (col < ncols)
                        a.hsum[(((int64_t)p * kPairCols + col) * fmax64 + b) * 2 + cls] = hs[c][0];
                }
            }
        } else {
#pragma unroll
            for (int s = 0; s < 8; ++s)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int col = c0 + (e & 1);
                    const int row = 128 * b + 16 * s + gq + 8 * (e >> 1);
                    if (col < ncols)
                        a.o[((int64_t)p * kPairCols + col) * d + row] = v[s][e] * invL;
                }
            if (!a.fused_combine)
                return;
            // combine: the last pair to finish block b sums rows 128b..128b+127
            __threadfence();
            __syncwarp();
            unsigned last = 0;
            if (lane == 0) {
                unsigned old = atomicAdd(&a.comb_ctr[b], 1u);
                last = old == static_cast<unsigned>(P_t - 1);
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence();
                const int kk = a.k;
                const bool has_sh = P_t > P_r;
                for (int64_t t = 0; t < a.T; ++t) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int row = 128 * b + 32 * q + lane;
                        float yv = 0.f;
                        for (int j = 0; j < kk; ++j) {
                            const int rm = __ldcg(a.route_map + t * (kk + 1) + j);
                            const float wj = __ldcg(a.weights + t * kk + j);
                            yv = fmaf(wj, __ldcg(a.o + (int64_t)rm * d + row), yv);
                        }
                        if (has_sh) {
                            const int rm = __ldcg(a.route_map + t * (kk + 1) + kk);
                            const float sw = __ldcg(a.shared_w + t);
                            yv = fmaf(sw, __ldcg(a.o + (int64_t)rm * d + row), yv);
                        }
                        a.y[t * d + row] = yv;
                    }
                }
                if (lane == 0)
                    a.comb_ctr[b] = 0u;
            }
        }
    };

    // flush the accumulators of block (p, b) covering global tiles [bs, be)
    auto flush = [&](int p, int b, int64_t bs, int64_t be) {
        const int64_t wf = warp_of(bs, W, U), wl = warp_of(be - 1, W, U);
        if (wf == wl) {
            finalize(p, b, acc);
            return;
        }
        const int myslot = u0 >= bs ? 0 : 1;
        float *mine = a.partial + ((w * 2 + myslot) * 32) * 32;
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                mine[(s * 4 + e) * 32 + lane] = acc[s][e];
        __threadfence();
        __syncwarp();
        unsigned last = 0;
        unsigned *ctr = a.blk_ctr + (int64_t)p * kMaxBlocksPerPair + b;
        if (lane == 0) {
            unsigned old = atomicAdd(ctr, 1u);
            last = old == static_cast<unsigned>(wl - wf);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last)
            return;
        __threadfence();
        float tot[8][4];
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                tot[s][e] = 0.f;
        for (int64_t ww = wf; ww <= wl; ++ww) {
            const int64_t wu0 = ww * U / W;
            const int sl = wu0 >= bs ? 0 : 1;
            const float *src = a.partial + ((ww * 2 + sl) * 32) * 32;
#pragma unroll
            for (int s = 0; s < 8; ++s)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    tot[s][e] += __ldcg(src + (s * 4 + e) * 32 + lane);
        }
        if (lane == 0)
            *ctr = 0u;
        finalize(p, b, tot);
    };

    // ---- main loop: one iteration per (block, group) segment of the range;
    // the 8 tiles of a group are unrolled so the accumulator index is static.
    int cur_p = -1, cur_b = -1, cur_g = -1;
    int64_t cur_bs = 0, cur_be = 0;
    BRaw pre;
    int pre_p = -1, pre_g = -1;
    bool timed_out = false;
    int64_t waited = 0;  // stages whose data has been waited for
    int64_t u = u0;
    while (u < u1 && !timed_out) {
        int p, G;
        int64_t lt;
        locate(u, p, lt, G);
        const int64_t tpb = (int64_t)G * kBlockTiles;
        const int b = static_cast<int>(lt / tpb);
        const int64_t rem = lt - (int64_t)b * tpb;
        const int g = static_cast<int>(rem / kBlockTiles);
        const int s_lo = static_cast<int>(rem % kBlockTiles);
        const int s_hi = static_cast<int>(kBlockTiles < s_lo + (u1 - u) ? kBlockTiles : s_lo + (u1 - u));

        if (p != cur_p || b != cur_b) {
            if (cur_p >= 0)
                flush(cur_p, cur_b, cur_bs, cur_be);
#pragma unroll
            for (int s = 0; s < 8; ++s)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[s][e] = 0.f;
            cur_p = p;
            cur_b = b;
            cur_bs = u - lt + (int64_t)b * tpb;
            cur_be = cur_bs + tpb;
            cur_g = -1;
        }
        if (g != cur_g) {
            BRaw now;
            if (pre_p == p && pre_g == g)
                now = pre;
            else
                load_b(p, g, G, now);
            cook_b(now);
            cur_g = g;
            // prefetch the next group's activations
            const int64_t un = u + (s_hi - s_lo);
            pre_p = -1;
            if (un < u1) {
                int pn, Gn;
                int64_t ltn;
                locate(un, pn, ltn, Gn);
                const int64_t tpbn = (int64_t)Gn * kBlockTiles;
                const int gn = static_cast<int>((ltn - (ltn / tpbn) * tpbn) / kBlockTiles);
                load_b(pn, gn, Gn, pre);
                pre_p = pn;
                pre_g = gn;
            }
        }

#pragma unroll
        for (int s = 0; s < kBlockTiles; ++s) {
            if (s < s_lo || s >= s_hi)
                continue;
            const int64_t uu = u + (s - s_lo);
            const int64_t si = (uu - u0) / kStageTiles;
            const int within = static_cast<int>((uu - u0) - si * kStageTiles);
            const int slot = static_cast<int>(si % kStages);
            if (within == 0) {
                if (!mbar_wait_bounded(&bars[slot], static_cast<unsigned>((si / kStages) & 1))) {
                    timed_out = true;
                    break;
                }
                waited = si + 1;
            }
            const uint8_t *tile = ring + slot * (kStageTiles * TB) + within * TB;
            const uint32_t sc = *reinterpret_cast<const uint32_t *>(tile + CB + 4 * gq);
            const float2 s01 = __half22float2(*reinterpret_cast<const __half2 *>(&sc));
            float dv[4] = {-bias0, -bias1, -bias0, -bias1};
            if (BITS == 4) {
                const uint4 cw = *reinterpret_cast<const uint4 *>(tile + 16 * lane);
                const uint32_t q4[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t q = q4[j];
                    uint32_t A[4];
                    A[0] = (q & 0x000F000Fu) | 0x43004300u;
                    A[1] = ((q >> 4) & 0x000F000Fu) | 0x43004300u;
                    A[2] = ((q >> 8) & 0x000F000Fu) | 0x43004300u;
                    A[3] = ((q >> 12) & 0x000F000Fu) | 0x43004300u;
                    mma_bf16(dv, A, b0[j], b1[j]);
                    if (SPLIT || PHASE == 1)
                        mma_bf16(dv, A, b0l[j], b1l[j]);
                }
            } else {
                const uint2 cw = *reinterpret_cast<const uint2 *>(tile + 8 * lane);
                const uint32_t q2[2] = {cw.x, cw.y};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t q = q2[j >> 1];
                    const int v0 = 8 * (j & 1), v1 = v0 + 4;
                    uint32_t A[4];
                    A[0] = ((q >> v0) & 0x00030003u) | 0x43004300u;
                    A[1] = ((q >> v1) & 0x00030003u) | 0x43004300u;
                    A[2] = ((q >> v0) & 0x000C000Cu) | 0x43004300u;
                    A[3] = ((q >> v1) & 0x000C000Cu) | 0x43004300u;
                    mma_bf16(dv, A, b0[j], b1[j]);
                    if (SPLIT || PHASE == 1)
                        mma_bf16(dv, A, b0l[j], b1l[j]);
                }
            }
            acc[s][0] = fmaf(s01.x, dv[0], acc[s][0]);
            acc[s][1] = fmaf(s01.x, dv[1], acc[s][1]);
            acc[s][2] = fmaf(s01.y, dv[2], acc[s][2]);
            acc[s][3] = fmaf(s01.y, dv[3], acc[s][3]);

            // stage consumed: refill its slot
            if (within == kStageTiles - 1 || uu == u1 - 1) {
                __syncwarp();
                if (lane == 0)
                    issue(si + kStages);
            }
        }
        u += s_hi - s_lo;
    }
    if (timed_out) {
        // record, then wait (bounded) for the copies still in flight so that
        // no bulk copy lands in shared memory after this block has exited
        if (lane == 0) {
            set_status(a.status, kStatusTimeout);
            const int64_t issued = waited + kStages < nst ? waited + kStages : nst;
            for (int64_t s = waited; s < issued; ++s)
                (void)mbar_wait_bounded(&bars[s % kStages], static_cast<unsigned>((s / kStages) & 1));
        }
        __syncwarp();
        return;
    }
    if (cur_p >= 0)
        flush(cur_p, cur_b, cur_bs, cur_be);
}

template <int BITS, bool SPLIT, int PHASE>
cudaError_t launch_one(const ExpertArgs &a, cudaStream_t stream, bool pdl)
{
    auto kern = expert_kernel<BITS, SPLIT, PHASE>;
    const int smem = smem_bytes(BITS);
    static bool attr_done[16] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done[dev & 15]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_done[dev & 15] = true;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        per_sm = 1;
    if (per_sm > 4)
        per_sm = 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(device_sm_count() * per_sm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// y[t] = sum_j w[t,j] * o[pair(t,j)] (rank order) + shared_w[t] * o[shared]
__global__ void __launch_bounds__(256) combine_kernel(const ExpertArgs a)
{
    pdl_wait();
    pdl_launch_dependents();
    const int d = a.d, kk = a.k;
    const bool has_sh = __ldcg(a.meta + 1) > __ldcg(a.meta + 0);
    const int64_t n = a.T * (d / 4);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / (d / 4);
        const int r4 = static_cast<int>(i % (d / 4)) * 4;
        float4 yv = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j <= kk; ++j) {
            if (j == kk && !has_sh)
                break;
            const int rm = __ldcg(a.route_map + t * (kk + 1) + j);
            const float wj = j < kk ? __ldcg(a.weights + t * kk + j) : __ldcg(a.shared_w + t);
            const float4 ov = __ldcg(reinterpret_cast<const float4 *>(a.o + (int64_t)rm * d + r4));
            yv.x = fmaf(wj, ov.x, yv.x);
            yv.y = fmaf(wj, ov.y, yv.y);
            yv.z = fmaf(wj, ov.z, yv.z);
            yv.w = fmaf(wj, ov.w, yv.w);
        }
        *reinterpret_cast<float4 *>(a.y + t * d + r4) = yv;
    }
}

}  // namespace

int expert_grid_warps() { return device_sm_count() * 4 * kWarps; }

cudaError_t launch_combine(const ExpertArgs &a, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    int64_t n = a.T * (a.d / 4);
    int64_t blocks = (n + 255) / 256;
    int64_t cap = (int64_t)device_sm_count() * 8;
    cfg.gridDim = dim3(static_cast<unsigned>(blocks < cap ? blocks : cap));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

cudaError_t launch_expert(const ExpertArgs &a, int phase, cudaStream_t stream, bool pdl)
{
    const bool split = phase == 1 || !a.x_bf16;
    if (a.bits == 4) {
        if (phase == 0)
            return split ? launch_one<4, true, 0>(a, stream, pdl) : launch_one<4, false, 0>(a, stream, pdl);
        return launch_one<4, true, 1>(a, stream, pdl);
    }
    if (phase == 0)
        return split ? launch_one<2, true, 0>(a, stream, pdl) : launch_one<2, false, 0>(a, stream, pdl);
    return launch_one<2, true, 1>(a, stream, pdl);
}

}  // namespace smoe
