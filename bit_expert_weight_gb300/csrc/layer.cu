// layer.cu -- the fused MoE layer kernel: router, top-k, dispatch, fused
// dequant gate/up GEMV + SiLU, fused dequant down GEMV and the routing-
// weighted combine, in one cooperative launch per layer.
//
// Method: "SMOE Quantisation", Decoding: Metal Kernel (the weight is decoded
// in registers as (code - L) / L * scale and multiplied at once, never
// materialised); "CMF v2 -- Format Specification", 2.2 MoE (softmax over all
// logits, top-k with ties to the lower index, selection-only bias,
// renormalisation, y = sum_j w_j FFN_j(x) + the sigmoid-gated shared expert);
// "Model Agnosticism", SmoeModelConfig (router rows = max_experts_per_layer).
//
// Phases (every warp runs them in order; cross-CTA dependencies are flags
// polled with bounded acquire loads; the launch is cooperative so every CTA
// is resident):
//  R  (T <= 8 only) one warp per router row computes that expert's logits
//     for all tokens over the full d (no K split, no partials); T more warps
//     compute the per-group activation sums; each bumps an arrival counter.
//     Every CTA then routes the tokens itself (one warp per token) and builds
//     the pair table in its own shared memory -- the same deterministic code
//     on the same logits gives the same table in every CTA, so nothing is
//     written back and re-read.  For T > 8 a separate router kernel has
//     built the tables in global memory before the launch.
//  G  gate/up: the tiles of all pairs (pair = one expert x <= 8 tokens) form
//     one stream of 16-row strips; each warp takes an equal contiguous range
//     (stream-K), streams it through a private ring of shared-memory stages
//     filled by TMA bulk copies, decodes codes in registers and multiplies
//     with mma.sync.  A strip (16 rows x all of d, gate and up interleaved)
//     finished by one warp is finalised in registers; one shared by several
//     warps is finalised by the last to arrive, summing the partials in warp
//     order.  Finalising writes h = SiLU(g) * u as bf16 hi + lo and the
//     strip's per-class sums of h, then bumps the pair's strip count.
//  D  down: the same streaming over 16-row strips of W_down.  A warp issues
//     its first weight copies before its CTA waits for the strip counts of
//     the pairs it reads, so the weights are in flight while gate/up
//     finishes.  The last pair to
//     finish an output strip (T <= 8) sums sum_j w_j o_j (+ shared) in rank
//     order into y.
// Deterministic throughout: no float atomics.
#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

// 16 streaming warps (decode, mma), 2 epilogue warps (unit sums, SiLU,
// stores, cross-CTA fixups) and one producer warp (the TMA ring): global-
// memory round trips and fences are slow while an SM streams, so the
// streaming warps make none.
constexpr int kStreamWarps = 16;
constexpr int kEpiWarps = 2;
constexpr int kProducerWarp = kStreamWarps + kEpiWarps;
constexpr int kWarps = kStreamWarps + kEpiWarps + 1;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxStripsD = 4096 / 16;  // output strips (d <= 4096)
constexpr long long kSpinCycles = 4000000000ll;  // ~2 s at 2 GHz

__device__ __forceinline__ unsigned atom_add_acqrel(unsigned *p, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Release/acquire fence at GPU scope: orders this thread's (and, through the
// preceding __syncwarp, its warp's) writes before a following signal, or a
// signal observed before the following reads.
__device__ __forceinline__ void fence_acq_rel()
{
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
// Relaxed fire-and-forget add / store: after one release fence these
// pipeline, where a chain of acq_rel atomics would serialise.
__device__ __forceinline__ void red_add_relaxed(unsigned *p, unsigned v)
{
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(unsigned *p, unsigned v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Lane 0 polls until *p >= target (bounded); the result is broadcast.
__device__ bool warp_wait_geq(const unsigned *p, unsigned target, int *status)
{
    const int lane = threadIdx.x & 31;
    int ok = 1;
    if (lane == 0) {
        const long long t0 = clock64();
        unsigned ns = 20;
        while (ld_acquire(p) < target) {
            if (clock64() - t0 > kSpinCycles) {
                ok = 0;
                set_status(status, kStatusTimeout);
                break;
            }
            __nanosleep(ns);
            if (ns < 200)
                ns *= 2;
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// CTA-wide named barrier 1 (all kThreads threads); 2: the streaming warps;
// 3: the epilogue warps.
__device__ __forceinline__ void cta_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}
__device__ __forceinline__ void stream_barrier()
{
    asm volatile("bar.sync 2, %0;" ::"n"(kStreamWarps * 32) : "memory");
}
__device__ __forceinline__ void epi_barrier()
{
    asm volatile("bar.sync 3, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

// Stream-K split of U units over W warps: warp w owns [start(w), start(w+1))
// with start(w) = floor(w * U / W), evaluated exactly in 32 bits as
// w*q + (w*r)/W with q = U / W, r = U % W (W < 2^13 keeps w*r < 2^26).
struct Split {
    int U, W, q, r;
};
__device__ __forceinline__ Split make_split(int U, int W)
{
    Split sp;
    sp.U = U;
    sp.W = W;
    sp.q = W > 0 ? U / W : 0;
    sp.r = W > 0 ? U - sp.q * W : 0;
    return sp;
}
__device__ __forceinline__ int split_start(const Split &sp, int w) { return w * sp.q + (w * sp.r) / sp.W; }
// The warp whose range holds unit u: a float estimate corrected to exact.
__device__ __forceinline__ int split_owner(const Split &sp, int u)
{
    int w = static_cast<int>((static_cast<float>(u) + 0.5f) * (static_cast<float>(sp.W) / static_cast<float>(sp.U)));
    w = w < 0 ? 0 : (w >= sp.W ? sp.W - 1 : w);
    while (w > 0 && split_start(sp, w) > u)
        --w;
    while (w + 1 < sp.W && split_start(sp, w + 1) <= u)
        ++w;
    return w;
}

// --------------------------------------------------------------- routing

// 1 / (1 + e^-x) with the hardware exp and divide; the exponent is capped
// so that the divisor stays finite (the result is then 0 to fp32).
__device__ __forceinline__ float sigmoid_fast(float x)
{
    return __fdividef(1.0f, 1.0f + __expf(fminf(-x, 80.0f)));
}

// Routing from the logits of one CTA's copy in shared memory.  Every CTA
// runs the same code on the same values, so every CTA derives the same
// tables.  Task (token t, chunk c) on one warp: lane L takes expert
// e = 32 c + L, whose rank is the number of experts before it in the order
// (key descending, index ascending) -- ties go to the lower index; ranks
// below k are the selection, stored at their rank with its score: the
// softmax over all E logits, or (sigm) the expert's own sigmoid.  The
// softmax maximum and sum run over all E logits in a fixed order
// (lane-strided, then a shuffle tree), the same in every task; exp and divide
// are the hardware approximations (a few ulp), well inside the weights'
// tolerance.
__device__ __noinline__ void route_chunk(const float *lg, const float *key, int E, int k, int c,
                                         int sigm, int16_t *ids_s, float *p_s)
{
    const int lane = threadIdx.x & 31;
    float m = -INFINITY, z = 1.f;
    if (!sigm) {
        for (int i = lane; i < E; i += 32)
            m = fmaxf(m, lg[i]);
        for (int o = 16; o; o >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        z = 0.f;
        for (int i = lane; i < E; i += 32)
            z += __expf(lg[i] - m);
        for (int o = 16; o; o >>= 1)
            z += __shfl_xor_sync(0xffffffffu, z, o);
    }
    const int e = 32 * c + lane;
    if (e >= E)
        return;
    const float ke = key[e];
    int r = 0;
    const float4 *k4 = reinterpret_cast<const float4 *>(key);
#pragma unroll 2
    for (int j = 0; j < E / 4; ++j) {
        const float4 v = k4[j];
        const int e0 = 4 * j;
        r += (v.x > ke || (v.x == ke && e0 < e)) ? 1 : 0;
        r += (v.y > ke || (v.y == ke && e0 + 1 < e)) ? 1 : 0;
        r += (v.z > ke || (v.z == ke && e0 + 2 < e)) ? 1 : 0;
        r += (v.w > ke || (v.w == ke && e0 + 3 < e)) ? 1 : 0;
    }
    for (int e2 = E & ~3; e2 < E; ++e2) {
        const float v = key[e2];
        r += (v > ke || (v == ke && e2 < e)) ? 1 : 0;
    }
    if (r < k) {
        ids_s[r] = static_cast<int16_t>(e);
        p_s[r] = sigm ? sigmoid_fast(lg[e]) : __fdividef(__expf(lg[e] - m), z);  // z in [1, E]
    }
}

// Phase R work of one warp: unit < E (+1 shared gate row) -> logits of that
// row for all tokens; unit >= rows -> group sums of token (unit - rows).
template <bool XBF16>
__device__ __forceinline__ void router_unit(const LayerArgs &a, int unit)
{
    const int lane = threadIdx.x & 31;
    const int d = a.d, T = static_cast<int>(a.T);
    const int rows = a.E + (a.shared_gate ? 1 : 0);
    if (unit < rows) {
        const uint16_t *wr = unit < a.E ? a.router_w + (int64_t)unit * d : a.shared_gate;
        // per token: four 256-column slices per batch, all loads in flight
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
            float acc = 0.f;
#pragma unroll 1
            for (int c0 = lane * 8; c0 < d; c0 += 1024) {
                uint4 wv[4], xv[4], xw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = c0 + 256 * i;
                    const bool in = c < d;
                    wv[i] = in ? __ldg(reinterpret_cast<const uint4 *>(wr + c)) : make_uint4(0u, 0u, 0u, 0u);
                    if (XBF16) {
                        xv[i] = in ? __ldg(reinterpret_cast<const uint4 *>(
                                         reinterpret_cast<const uint16_t *>(a.x) + (int64_t)t * d + c))
                                   : make_uint4(0u, 0u, 0u, 0u);
                    } else {
                        const uint4 *xr = reinterpret_cast<const uint4 *>(
                            reinterpret_cast<const float *>(a.x) + (int64_t)t * d + c);
                        xv[i] = in ? __ldg(xr) : make_uint4(0u, 0u, 0u, 0u);
                        xw[i] = in ? __ldg(xr + 1) : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
                    float xf[8];
                    if (XBF16) {
                        const uint32_t xx[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            xf[2 * q] = bf16lo_to_f32(xx[q]);
                            xf[2 * q + 1] = bf16hi_to_f32(xx[q]);
                        }
                    } else {
                        xf[0] = __uint_as_float(xv[i].x), xf[1] = __uint_as_float(xv[i].y);
                        xf[2] = __uint_as_float(xv[i].z), xf[3] = __uint_as_float(xv[i].w);
                        xf[4] = __uint_as_float(xw[i].x), xf[5] = __uint_as_float(xw[i].y);
                        xf[6] = __uint_as_float(xw[i].z), xf[7] = __uint_as_float(xw[i].w);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc = fmaf(bf16lo_to_f32(ww[q]), xf[2 * q], acc);
                        acc = fmaf(bf16hi_to_f32(ww[q]), xf[2 * q + 1], acc);
                    }
                }
            }
            for (int o = 16; o; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0)
                a.logits[(int64_t)t * a.Epad + unit] = acc;
        }
    } else {
        // group sums of token t: X0 over columns c % 4 in {0,1}, X1 over {2,3}
        const int t = unit - rows;
        for (int g = lane; g < d / kGroup; g += 32) {
            float s0 = 0.f, s1 = 0.f;
            if (XBF16) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const uint16_t *>(a.x) + (int64_t)t * d + g * kGroup);
                uint4 v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = __ldg(src + i);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    s0 += bf16lo_to_f32(v[i].x) + bf16hi_to_f32(v[i].x);
                    s1 += bf16lo_to_f32(v[i].y) + bf16hi_to_f32(v[i].y);
                    s0 += bf16lo_to_f32(v[i].z) + bf16hi_to_f32(v[i].z);
                    s1 += bf16lo_to_f32(v[i].w) + bf16hi_to_f32(v[i].w);
                }
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(
                    reinterpret_cast<const float *>(a.x) + (int64_t)t * d + g * kGroup);
                float4 v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = __ldg(src + i);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    s0 += v[i].x + v[i].y;
                    s1 += v[i].z + v[i].w;
                }
            }
            reinterpret_cast<float2 *>(a.xsum)[(int64_t)t * (d / kGroup) + g] = make_float2(s0, s1);
        }
    }
}

// Routing tables of a CTA.  On the fused path (T <= 8) every CTA builds its
// own copy in shared memory from the published logits (the same
// deterministic code on the same logits gives the same tables everywhere);
// otherwise they point to the tables the router kernel left in global memory.
constexpr int kFusedPairs = kPairCols * SMOE_MAX_TOPK_DEV + 1;
// route_map, weights and ids are [T][k+1], [T][k], [T][k] with the runtime k
// as the row stride, exactly like the global tables.
struct __align__(16) RouteSmem {
    float lg[kPairCols * kMaxExperts];   // [T][E4] logits, row stride E4 = E rounded up to 4
    float key[kPairCols * kMaxExperts];  // [T][E4] selection keys fl32(logit + bias)
    float prob[kPairCols * SMOE_MAX_TOPK_DEV];  // [T][k] softmax of the rank-j expert
    float warm_p[SMOE_MAX_TOPK_DEV];     // scratch of the instruction-cache warm-up
    int16_t warm_id[SMOE_MAX_TOPK_DEV];
    int32_t pairs[kFusedPairs][kPairInts];
    int32_t route_map[kPairCols * (SMOE_MAX_TOPK_DEV + 1)];
    float weights[kPairCols * SMOE_MAX_TOPK_DEV];
    float shared_w[kPairCols];
    int16_t ids[kPairCols * SMOE_MAX_TOPK_DEV];
    int16_t pair_of[kMaxExperts];
    int meta[2];
};
struct RouteView {
    const int32_t *pairs;      // [P][kPairInts]
    const int32_t *route_map;  // [T][k+1]
    const float *weights;      // [T][k]
    const float *shared_w;     // [T]
};

// One warp of the CTA: pair table from the routed ids (T <= 8).  Pair = one
// selected expert with the ascending tokens that chose it, pairs in order of
// first appearance; then the shared expert's pair.
__device__ __forceinline__ void cta_dispatch(const LayerArgs &a, RouteSmem &r)
{
    const int lane = threadIdx.x & 31;
    const int T = static_cast<int>(a.T), k = a.k, E = a.E;
    for (int e = lane; e < E; e += 32)
        r.pair_of[e] = -1;
    __syncwarp();
    int npairs = 0;
    for (int t = 0; t < T; ++t) {
        int e = -1, p = -1;
        if (lane < k) {
            e = r.ids[t * k + lane];
            p = r.pair_of[e];
        }
        const unsigned newm = __ballot_sync(0xffffffffu, lane < k && p < 0);
        if (lane < k && p < 0) {
            p = npairs + __popc(newm & ((1u << lane) - 1u));
            r.pair_of[e] = static_cast<int16_t>(p);
            r.pairs[p][0] = e;
            r.pairs[p][1] = 0;
        }
        npairs += __popc(newm);
        __syncwarp();
        if (lane < k) {
            const int col = r.pairs[p][1];
            r.pairs[p][2 + col] = t;
            r.pairs[p][1] = col + 1;
            r.route_map[t * (k + 1) + lane] = p * kPairCols + col;
        }
        __syncwarp();
    }
    if (a.has_shared) {
        if (lane == 0) {
            r.pairs[npairs][0] = -1;
            r.pairs[npairs][1] = T;
        }
        if (lane < kPairCols)
            r.pairs[npairs][2 + lane] = lane < T ? lane : 0;
        if (lane < T)
            r.route_map[lane * (k + 1) + k] = npairs * kPairCols + lane;
    }
    if (lane == 0) {
        r.meta[0] = npairs;
        r.meta[1] = npairs + (a.has_shared ? 1 : 0);
    }
    __syncwarp();
}

// ------------------------------------------------------------ streaming

// A chunk is a run of up to kChunkGroups consecutive groups of one strip,
// two per streaming warp (groups w and w + 16 of the chunk); one stage of
// the CTA's ring holds one chunk.  Gate/up: a strip of d/64 groups in 1 or
// 2 chunks (gate and up tile per group); down: the whole strip in one chunk.
constexpr int kChunkGroups = 2 * kStreamWarps;
constexpr int kDownGroupsMax = kChunkGroups;  // ffn_dim <= 2048

__host__ __device__ constexpr int stage_bytes(int bits) { return kChunkGroups * 2 * tile_bytes(bits); }
// Kernel instances: BITS = 4 or 2 for a bank of one depth, BITS = 0 for a
// bank of mixed depths, whose ring is sized for Q4 stages.
__host__ __device__ constexpr int ring_bits(int bits) { return bits == 0 ? 4 : bits; }
// About 100 KB in flight per SM: the full HBM rate needs ~64 KB; deeper
// rings delay every other memory access of the SM, which queues behind them.
__host__ __device__ constexpr int num_stages(int bits) { return bits == 4 ? 3 : 5; }
// kRedSlots slots of per-warp unit sums (gate and up float4 per lane)
constexpr int kRedSlots = 4;
__host__ __device__ constexpr int red_bytes() { return kRedSlots * kStreamWarps * 2 * 32 * 16; }
__host__ __device__ constexpr int smem_bytes(int bits)
{
    return num_stages(bits) * stage_bytes(bits) + red_bytes() + (2 * num_stages(bits) + 2 * kRedSlots) * 8;
}
// Pairs whose finished gate/up strips a CTA counts in shared memory and
// publishes once, at the end of its gate/up range.
constexpr int kMaxSpan = 64;

// Step geometry of one phase.  Units are (pair, strip) in pair order; a
// unit's K groups are cut into ch chunks of gc groups (the last may be
// shorter); the steps (chunks) of all units are split evenly over the CTAs.
// Index [0]: routed pairs, [1]: the shared expert's pair.
// (Scalar fields with select accessors: a runtime-indexed array would live
// in local memory.)
struct Geo {
    int P_r, P_t;
    int nstr0, gk0, ch0, gc0, spp0;  // routed: strips, groups per strip, chunks, groups per chunk, steps
    int nstr1, gk1, ch1, gc1, spp1;  // shared
    int SR, S;                       // steps of the routed pairs, of all pairs
    Split sp;                        // steps over CTAs
    int a0, a1;                      // this CTA's steps
    int ts;                          // the CTA runs [ts, a1) first, then [a0, ts)
};

struct UnitGeo {
    int nstr, gk, ch, gc;
};

__device__ __forceinline__ UnitGeo unit_geo(const Geo &g, int p)
{
    const bool r = p < g.P_r;
    UnitGeo u;
    u.nstr = r ? g.nstr0 : g.nstr1;
    u.gk = r ? g.gk0 : g.gk1;
    u.ch = r ? g.ch0 : g.ch1;
    u.gc = r ? g.gc0 : g.gc1;
    return u;
}

__device__ __forceinline__ Geo make_geo(const LayerArgs &a, int phase, int P_r, int P_t)
{
    Geo g;
    g.P_r = P_r;
    g.P_t = P_t;
    {
        const int rows = phase == 0 ? a.f : a.d, K = phase == 0 ? a.d : a.f;
        g.nstr0 = rows / kTileRows;
        g.gk0 = K / kGroup;
        g.ch0 = phase == 0 ? (g.gk0 + kChunkGroups - 1) / kChunkGroups : 1;
        g.gc0 = g.ch0 > 0 ? (g.gk0 + g.ch0 - 1) / g.ch0 : 0;
        g.spp0 = g.nstr0 * g.ch0;
    }
    {
        const int rows = phase == 0 ? a.fs : a.d, K = phase == 0 ? a.d : a.fs;
        g.nstr1 = rows / kTileRows;
        g.gk1 = K / kGroup;
        g.ch1 = phase == 0 ? (g.gk1 + kChunkGroups - 1) / kChunkGroups : (g.gk1 > 0 ? 1 : 0);
        g.gc1 = g.ch1 > 0 ? (g.gk1 + g.ch1 - 1) / g.ch1 : 0;
        g.spp1 = g.nstr1 * g.ch1;
    }
    g.SR = P_r * g.spp0;
    g.S = g.SR + (P_t - P_r) * g.spp1;
    const int C = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    g.sp = make_split(g.S, C);
    g.a0 = split_start(g.sp, c);
    g.a1 = split_start(g.sp, c + 1);
    // Whole units per CTA when every unit has the same chunk count and the
    // extra unit a CTA may get costs under ~48 KB (about a microsecond of
    // one SM's share of HBM): no unit is then shared between CTAs.
    if (g.ch0 > 1 && (P_t == P_r || g.ch1 == g.ch0)) {
        const int U = g.S / g.ch0;
        const int unit_bytes = g.gk0 * (phase == 0 ? 2 : 1) * (a.bits * 128 + 32);
        const int64_t extra = (int64_t)((U + C - 1) / C) * C - U;  // C x (max - mean) units
        if (extra * unit_bytes < (int64_t)C * 48 * 1024) {
            const Split su = make_split(U, C);
            g.a0 = split_start(su, c) * g.ch0;
            g.a1 = split_start(su, c + 1) * g.ch0;
        }
    }
    g.ts = g.a1;
    return g;
}

struct Pos {
    int p, s, c;  // pair, strip, chunk
};

__device__ __forceinline__ Pos decode(const Geo &g, int i)
{
    Pos q;
    int r, ch;
    if (i < g.SR) {
        q.p = i / g.spp0;
        r = i - q.p * g.spp0;
        ch = g.ch0;
    } else {
        const int j = i - g.SR, pp = j / g.spp1;
        q.p = g.P_r + pp;
        r = j - pp * g.spp1;
        ch = g.ch1;
    }
    q.s = r / ch;
    q.c = r - q.s * ch;
    return q;
}

__device__ __forceinline__ void advance(const UnitGeo &u, Pos &q)
{
    if (++q.c == u.ch) {
        q.c = 0;
        if (++q.s == u.nstr) {
            q.s = 0;
            ++q.p;
        }
    }
}

// The ring's producer (lane 0 of warp 0): the next stage to issue, as a
// phase and a step of that phase.
// Order of a CTA's steps: a unit cut by the end of the range is run first,
// then the range from its start (whose first unit may be cut by the start).
// Both contributors of a shared unit then reach it early, so the fixup that
// joins their sums is off the critical path.
__device__ __forceinline__ void set_order(Geo &g)
{
    g.ts = g.a1;
    if (g.a1 <= g.a0)
        return;
    const Pos ql = decode(g, g.a1 - 1);
    const int ch = ql.p < g.P_r ? g.ch0 : g.ch1;
    const int ustart = (g.a1 - 1) - ql.c;
    if (ql.c != ch - 1 && ustart > g.a0)
        g.ts = ustart;
}
// Step index of position k in that order.
__device__ __forceinline__ int step_at(const Geo &g, int k)
{
    const int nt = g.a1 - g.ts;
    return k < nt ? g.ts + k : g.a0 + (k - nt);
}

// Kept in shared memory, like the geometry of both phases (CTA-uniform).
struct Producer {
    int phase;      // 0 gate/up, 1 down, 2 nothing left
    int k;          // position in the phase's step order
    Pos q;
    uint32_t next;  // stages issued so far
};

__device__ __forceinline__ void producer_seek(const Geo *geo, Producer &pr)
{
    while (pr.phase <= 1 && geo[pr.phase].a0 >= geo[pr.phase].a1)
        ++pr.phase;
    if (pr.phase <= 1) {
        pr.k = 0;
        pr.q = decode(geo[pr.phase], step_at(geo[pr.phase], 0));
    }
}

// Depth of the expert of a pair (e < 0: the shared expert, at the layer's
// depth); a compile-time constant except in the mixed-depth instance.
template <int BITS>
__device__ __forceinline__ int pair_bits(const LayerArgs &a, int e)
{
    if (BITS != 0)
        return BITS;
    return e < 0 ? a.bits : mixed_expert_bits(a, e);
}

// Issue the next stage: 1 issued, 0 not now (slot still in use and
// !block, or nothing left), -1 the bounded wait for the slot ran out.
template <int BITS>
__device__ __forceinline__ int produce(const LayerArgs &a, const RouteView &rv, const Geo *geo,
                                       Producer &pr, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                       bool block)
{
    constexpr int NS = num_stages(ring_bits(BITS)), SB = stage_bytes(ring_bits(BITS));
    if (pr.phase > 1)
        return 0;
    const uint32_t j = pr.next;
    const int slot = static_cast<int>(j % NS);
    if (j >= static_cast<uint32_t>(NS)) {
        const unsigned par = ((j / NS) - 1u) & 1u;
        if (block) {
            if (!mbar_wait_bounded(&empty[slot], par))
                return -1;
        } else if (!mbar_test_wait(&empty[slot], par)) {
            return 0;
        }
    }
    const Geo &g = geo[pr.phase];
    const UnitGeo u = unit_geo(g, pr.q.p);
    const int e = rv.pairs[pr.q.p * kPairInts];
    const int TB = tile_bytes(pair_bits<BITS>(a, e));
    const int GB = pr.phase == 0 ? 2 * TB : TB;
    const int g0 = pr.q.c * u.gc;
    const int ng = min(u.gk - g0, u.gc);
    const uint8_t *base;
    if (e < 0)
        base = a.tiles_shared + (pr.phase ? a.down_off_shared : 0);
    else if (BITS != 0)
        base = a.tiles_routed + (int64_t)e * a.expert_bytes_routed + (pr.phase ? a.down_off_routed : 0);
    else  // the expert's own place and down offset in a bank of mixed depths
        base = a.tiles_routed + mixed_expert_offset(a, e) +
               (pr.phase ? 2ll * a.d * a.f / 1024 * TB : 0);
    const uint8_t *src = base + ((int64_t)pr.q.s * u.gk + g0) * GB;
    mbar_arrive_expect_tx(&full[slot], static_cast<unsigned>(ng * GB));
    bulk_g2s(ring + slot * SB, src, static_cast<unsigned>(ng * GB), &full[slot]);
    pr.next = j + 1;
    if (++pr.k == g.a1 - g.a0) {
        ++pr.phase;
        producer_seek(geo, pr);
    } else if (pr.k == g.a1 - g.ts) {
        pr.q = decode(g, g.a0);
    } else {
        advance(u, pr.q);
    }
    return 1;
}

// The lane's view of a pair record: column count, its token row (gq) and
// the tokens of its two output columns.
struct PairInfo {
    int ncols, tok, t0, t1;
};

__device__ __forceinline__ PairInfo read_pair(const RouteView &rv, int p)
{
    const int lane = threadIdx.x & 31, gq = lane >> 2, tig = lane & 3;
    const int32_t *pr = rv.pairs + p * kPairInts;
    PairInfo pi;
    pi.ncols = pr[1];
    pi.tok = gq < pi.ncols ? pr[2 + gq] : 0;
    pi.t0 = 2 * tig < pi.ncols ? pr[2 + 2 * tig] : -1;
    pi.t1 = 2 * tig + 1 < pi.ncols ? pr[2 + 2 * tig + 1] : -1;
    return pi;
}

// mma B fragments of one group (hi and, for fp32 / h activations, lo) and
// the two column biases -(128 + L) X (Q2: -(129.5 X0 + 33.5 X1)), stored
// negated: they are the C operand of a tile's first mma.
struct BFrag {
    uint32_t b0[4], b1[4], b0l[4], b1l[4];
    float bias0, bias1;
};

template <int BITS>
__device__ __forceinline__ void finish_bias(BFrag &f, float2 x0, float2 x1)
{
    if (BITS == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f.b1[j] = bf16x2_quarter(f.b1[j]);
            f.b1l[j] = bf16x2_quarter(f.b1l[j]);
        }
        // one explicit fma: the same rounding in every kernel instance
        f.bias0 = -fmaf(129.5f, x0.x, 33.5f * x0.y);
        f.bias1 = -fmaf(129.5f, x1.x, 33.5f * x1.y);
    } else {
        f.bias0 = -(135.5f * (x0.x + x0.y));
        f.bias1 = -(135.5f * (x1.x + x1.y));
    }
}

// Raw B operand of one group as loaded: gate/up -- this lane's 16
// activations (columns 64 gi + 16 tig .. +15 of its token; bf16 x: 2
// vectors, fp32 x: 4) and the group sums of its two output columns; down --
// h hi (v[0..1]) and lo (v[2..3]) and the lane's strip of the group sums.
// All through L1: x is read-only, and h, the group sums and xsum were
// published (release / acquire) before the first read of each.
template <int NV>
struct BRaw {
    uint4 v[NV];
    float2 xs0, xs1;
};

template <int PHASE, bool XBF16, int NV>
__device__ __forceinline__ void load_raw(const LayerArgs &a, const PairInfo &pi, int p, int gi, int fmax,
                                         BRaw<NV> &r)
{
    const int lane = threadIdx.x & 31, gq = lane >> 2, tig = lane & 3;
    const int d = a.d;
    const bool valid = gq < pi.ncols;
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    const float2 z2 = make_float2(0.f, 0.f);
    if (PHASE == 0) {
        if (XBF16) {
            const uint4 *row = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const uint16_t *>(a.x) + (int64_t)pi.tok * d + gi * kGroup + 16 * tig);
            r.v[0] = valid ? __ldg(row) : z4;
            r.v[1] = valid ? __ldg(row + 1) : z4;
        } else {
            const uint4 *row = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const float *>(a.x) + (int64_t)pi.tok * d + gi * kGroup + 16 * tig);
#pragma unroll
            for (int i = 0; i < NV; ++i)
                r.v[i] = valid ? __ldg(row + i) : z4;
        }
        const float2 *xs = reinterpret_cast<const float2 *>(a.xsum);
        r.xs0 = pi.t0 >= 0 ? __ldca(xs + (int64_t)pi.t0 * (d / kGroup) + gi) : z2;
        r.xs1 = pi.t1 >= 0 ? __ldca(xs + (int64_t)pi.t1 * (d / kGroup) + gi) : z2;
    } else {
        const int64_t off = ((int64_t)p * kPairCols + gq) * fmax + gi * kGroup + 16 * tig;
        const uint4 *hi = reinterpret_cast<const uint4 *>(a.h_hi + off);
        const uint4 *lo = reinterpret_cast<const uint4 *>(a.h_lo + off);
        r.v[0] = valid ? __ldca(hi) : z4;
        r.v[1] = valid ? __ldca(hi + 1) : z4;
        r.v[2] = valid ? __ldca(lo) : z4;
        r.v[3] = valid ? __ldca(lo + 1) : z4;
        // group sums of h: lane (gq, tig) loads strip 4 gi + (gq & 3) of its
        // two columns; cook_b adds the four strips with shuffles
        const int nstrip = fmax / kTileRows;
        const int c0 = 2 * tig, c1 = c0 + 1;
        const float2 *hp = reinterpret_cast<const float2 *>(a.hs_part);
        const int st = 4 * gi + (gq & 3);
        r.xs0 = c0 < pi.ncols ? __ldca(hp + ((int64_t)p * kPairCols + c0) * nstrip + st) : z2;
        r.xs1 = c1 < pi.ncols ? __ldca(hp + ((int64_t)p * kPairCols + c1) * nstrip + st) : z2;
    }
}

// mma fragments and biases from a BRaw (every lane of the warp calls it).
template <int BITS, int PHASE, bool XBF16, int NV>
__device__ __forceinline__ void cook_b(const BRaw<NV> &r, BFrag &f)
{
    float2 x0 = r.xs0, x1 = r.xs1;
    if (PHASE == 1) {
        const uint32_t *hv = reinterpret_cast<const uint32_t *>(r.v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f.b0[j] = hv[2 * j];
            f.b1[j] = hv[2 * j + 1];
            f.b0l[j] = hv[8 + 2 * j];
            f.b1l[j] = hv[8 + 2 * j + 1];
        }
#pragma unroll
        for (int o = 4; o <= 8; o <<= 1) {
            x0.x += __shfl_xor_sync(0xffffffffu, x0.x, o);
            x0.y += __shfl_xor_sync(0xffffffffu, x0.y, o);
            x1.x += __shfl_xor_sync(0xffffffffu, x1.x, o);
            x1.y += __shfl_xor_sync(0xffffffffu, x1.y, o);
        }
    } else if (!XBF16) {
        const float *xv = reinterpret_cast<const float *>(r.v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            split_bf16x2(xv[4 * j + 0], xv[4 * j + 1], f.b0[j], f.b0l[j]);
            split_bf16x2(xv[4 * j + 2], xv[4 * j + 3], f.b1[j], f.b1l[j]);
        }
    } else {
        const uint32_t *xv = reinterpret_cast<const uint32_t *>(r.v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f.b0[j] = xv[2 * j];
            f.b1[j] = xv[2 * j + 1];
            f.b0l[j] = f.b1l[j] = 0u;
        }
    }
    finish_bias<BITS>(f, x0, x1);
}

// Decode + multiply one tile from shared memory into acc: one mma chain
// over the four k-subtiles (hi then lo fragments when split), started from
// the column biases; the warp's other tiles of the step supply the ILP.
// Codes decode to finite values (128 + c) whatever the bytes, so a disabled
// tile (on == false) is computed branch-free and dropped by a zero scale.
template <int BITS, bool SPLIT>
__device__ __forceinline__ void mac_tile(const uint8_t *tile, const BFrag &f, float (&acc)[4], bool on)
{
    constexpr int CB = tile_code_bytes(BITS);
    const int lane = threadIdx.x & 31, gq = lane >> 2;
    const uint32_t sc = *reinterpret_cast<const uint32_t *>(tile + CB + 4 * gq);
    float2 s01 = __half22float2(*reinterpret_cast<const __half2 *>(&sc));
    // a tile of an absent group (in-bounds stage bytes, zero B fragment)
    // contributes exactly nothing: its scale is replaced, not multiplied
    s01.x = on ? s01.x : 0.f;
    s01.y = on ? s01.y : 0.f;
    float dv[4];
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
            if (j == 0)
                mma_bf16_c(dv, A, f.b0[0], f.b1[0], f.bias0, f.bias1, f.bias0, f.bias1);
            else
                mma_bf16(dv, A, f.b0[j], f.b1[j]);
            if (SPLIT)
                mma_bf16(dv, A, f.b0l[j], f.b1l[j]);
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
            if (j == 0)
                mma_bf16_c(dv, A, f.b0[0], f.b1[0], f.bias0, f.bias1, f.bias0, f.bias1);
            else
                mma_bf16(dv, A, f.b0[j], f.b1[j]);
            if (SPLIT)
                mma_bf16(dv, A, f.b0l[j], f.b1l[j]);
        }
    }
    acc[0] = fmaf(s01.x, dv[0], acc[0]);
    acc[1] = fmaf(s01.x, dv[1], acc[1]);
    acc[2] = fmaf(s01.y, dv[2], acc[2]);
    acc[3] = fmaf(s01.y, dv[3], acc[3]);
}

// Finalise unit (p, s) from its full-K sums, one warp (cold path).
// Phase 0: h = SiLU(g) * u as bf16 hi + lo and the strip's per-class sums of
// h.  Phase 1: o.  The caller counts the finished unit.
// What the epilogue writes, passed by value (registers) to its cold helpers.
struct EpiOut {
    uint16_t *h_hi, *h_lo;
    float *hs_part, *o, *partial;
    unsigned *strip_ctr_g, *strip_ctr_d, *pair_done;
    int d, fmax, max_strips;
};

template <int BITS, int PHASE>
__device__ __noinline__ void finalize_unit(const EpiOut a, int ncols, int p, int s, float4 ag, float4 au)
{
    constexpr float L = BITS == 4 ? 7.5f : 1.5f;
    const int lane = threadIdx.x & 31, gq = lane >> 2, tig = lane & 3;
    const int d = a.d;
    const int fmax = a.fmax;
    const float invL = 1.0f / L;
    const int c0 = 2 * tig;
    const float gv[4] = {ag.x, ag.y, ag.z, ag.w}, uv[4] = {au.x, au.y, au.z, au.w};
    if (PHASE == 0) {
        const int nstrip = fmax / kTileRows;
        float hs[2] = {0.f, 0.f};  // per output column, this lane's rows
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float g = gv[e] * invL, u = uv[e] * invL;
            const float hv = __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;  // SiLU(g) * u
            const int col = c0 + (e & 1);
            const int row = 16 * s + gq + 8 * (e >> 1);
            if (col < ncols) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
                const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
                const int64_t off = ((int64_t)p * kPairCols + col) * fmax + row;
                a.h_hi[off] = *reinterpret_cast<const uint16_t *>(&hi);
                a.h_lo[off] = *reinterpret_cast<const uint16_t *>(&lo);
            }
            hs[e & 1] += hv;
        }
        // class of these rows within their 64-row group: (gq >> 1) & 1; sum
        // over lanes with equal tig and class (lane bits 2 and 4)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            hs[c] += __shfl_xor_sync(0xffffffffu, hs[c], 4);
            hs[c] += __shfl_xor_sync(0xffffffffu, hs[c], 16);
        }
        if ((gq & 5) == 0) {
            const int cls = (gq >> 1) & 1;
#pragma unroll
            for (int c = 0; c < 2; ++c)
                if (c0 + c < ncols)
                    a.hs_part[(((int64_t)p * kPairCols + c0 + c) * nstrip + s) * 2 + cls] = hs[c];
        }
        __syncwarp();  // the caller counts the strip (see count_strip)
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = c0 + (e & 1);
            const int row = 16 * s + gq + 8 * (e >> 1);
            if (col < ncols)
                a.o[((int64_t)p * kPairCols + col) * d + row] = gv[e] * invL;
        }
        __syncwarp();  // the caller counts the output strip
    }
}

// One more finished gate/up strip of pair p: counted in shared memory and
// published at the end of the CTA's gate/up range, or published at once
// (release) when the CTA's range spans too many pairs.
__device__ __forceinline__ void count_strip(const EpiOut &a, const int *pspan, unsigned *pcnt, int p)
{
    if ((threadIdx.x & 31) != 0)
        return;
    const int j = p - pspan[0];
    if (pspan[1] > 0 && j >= 0 && j < pspan[1]) {
        atomicAdd(pcnt + j, 1u);
    } else {
        fence_acq_rel();
        red_add_relaxed(a.pair_done + p, 1u);
    }
}

// A finished unit: a gate/up strip of pair p, or a down unit of output
// strip s (counted per CTA, published after the down phase).
template <int PHASE>
__device__ __forceinline__ void count_unit(const EpiOut &a, const int *pspan, unsigned *pcnt,
                                           unsigned *ccnt, int p, int s)
{
    if (PHASE == 0)
        count_strip(a, pspan, pcnt, p);
    else if ((threadIdx.x & 31) == 0)
        atomicAdd(ccnt + s, 1u);
}

// Unit (p, s) shared with other CTAs (cold path): store this CTA's sums,
// count the contributors; the last one adds all sums in CTA order and
// finalises.  Slot 0 of a CTA holds the unit straddling its first step,
// slot 1 the one straddling its last; each phase has its own slots.
template <int BITS, int PHASE>
__device__ __noinline__ void fixup_unit(const EpiOut a, int ncols, const Geo &g, int p, int s, int ustart,
                                        int uend, float4 tg, float4 tu, unsigned *pcnt, const int *pspan,
                                        unsigned *ccnt)
{
    const int lane = threadIdx.x & 31;
    float4 *part = reinterpret_cast<float4 *>(a.partial) + (size_t)PHASE * gridDim.x * 2 * 64;
    const int my = ustart < g.a0 ? 0 : 1;
    float4 *mine = part + ((size_t)blockIdx.x * 2 + my) * 64;
    mine[lane] = tg;
    if (PHASE == 0)
        mine[32 + lane] = tu;
    __syncwarp();
    const int cf = split_owner(g.sp, ustart), cl = split_owner(g.sp, uend - 1);
    unsigned *ctr = (PHASE == 0 ? a.strip_ctr_g : a.strip_ctr_d) + (int64_t)p * a.max_strips + s;
    unsigned old = 0;
    if (lane == 0)
        old = atom_add_acqrel(ctr, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != static_cast<unsigned>(cl - cf))
        return;
    __syncwarp();
    float4 sg = make_float4(0.f, 0.f, 0.f, 0.f), su = sg;
    for (int c0 = cf; c0 <= cl; c0 += 4) {
        float4 vg[4], vu[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c = c0 + q;
            vg[q] = vu[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c <= cl) {
                const int sl = split_start(g.sp, c) > ustart ? 0 : 1;
                const float4 *src = part + ((size_t)c * 2 + sl) * 64;
                vg[q] = __ldcg(src + lane);
                if (PHASE == 0)
                    vu[q] = __ldcg(src + 32 + lane);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            sg.x += vg[q].x, sg.y += vg[q].y, sg.z += vg[q].z, sg.w += vg[q].w;
            su.x += vu[q].x, su.y += vu[q].y, su.z += vu[q].z, su.w += vu[q].w;
        }
    }
    if (lane == 0)
        *ctr = 0u;
    finalize_unit<BITS, PHASE>(a, ncols, p, s, sg, su);
    count_unit<PHASE>(a, pspan, pcnt, ccnt, p, s);
}

// Shared state of the streaming phases, one per CTA.
struct Stream {
    uint8_t *ring;
    uint64_t *full, *empty;          // [NS]: 1 arrival + bytes / kStreamWarps arrivals
    uint64_t *red_full, *red_empty;  // [kRedSlots]: kStreamWarps arrivals / 1 arrival
    unsigned *pcnt;                  // [kMaxSpan] finished gate/up strips per pair
    const int *pspan;                // [0] first pair, [1] span (0: publish each at once)
    unsigned *ccnt;                  // [d/16] finished down units per output strip
    float4 *red;                     // [kRedSlots][kStreamWarps][2][32]
    volatile int *fail;              // a bounded wait ran out somewhere in the CTA
    Producer *pr;                    // shared; used by lane 0 of warp 0 only
    const Geo *geo;                  // shared, [2]
    uint32_t seq;                    // stages consumed by this (streaming) warp
    int uc;                          // units ended so far
};

__device__ __forceinline__ bool unit_ends(const Geo &g, const UnitGeo &u, const Pos &q, int i)
{
    return q.c == u.ch - 1 || i == g.a1 - 1 || (g.ts < g.a1 && i == g.ts - 1);
}

// The warp's tiles of one stage (chunk c of the unit) at depth B:
// branch-free over the warp's two groups (tiles of absent groups read
// in-bounds stage bytes and are dropped), so the four (down: two) mma
// chains of the step schedule together.
template <int B, int PHASE, int KG, bool kSplit, int NB>
__device__ __forceinline__ void step_tiles(const uint8_t *stage, const BFrag (&bf)[NB], int qc, bool g0,
                                           bool g1, float (&accg)[4], float (&accu)[4],
                                           float (&accg2)[4], float (&accu2)[4])
{
    constexpr int TB = tile_bytes(B), GB = PHASE == 0 ? 2 * TB : TB;
    const int warp = threadIdx.x >> 5;
    if (PHASE == 0) {
#pragma unroll
        for (int c = 0; c < KG; ++c) {
            if (c == qc) {
                mac_tile<B, kSplit>(stage + warp * GB, bf[2 * c], accg, g0);
                mac_tile<B, kSplit>(stage + warp * GB + TB, bf[2 * c], accu, g0);
                mac_tile<B, kSplit>(stage + (warp + kStreamWarps) * GB, bf[2 * c + 1], accg2, g1);
                mac_tile<B, kSplit>(stage + (warp + kStreamWarps) * GB + TB, bf[2 * c + 1], accu2, g1);
            }
        }
    } else {
        mac_tile<B, kSplit>(stage + warp * GB, bf[0], accg, g0);
        mac_tile<B, kSplit>(stage + (warp + kStreamWarps) * GB, bf[1], accu, g1);
    }
}

// One phase (0: gate/up, 1: down) of a streaming warp.  The warp holds the
// B fragments of its groups of the current pair: groups c * gc + w and
// c * gc + w + 16 of each chunk c (gate/up: at most KG chunks; down: one).
// At a unit's end it leaves its sums in a slot for the epilogue warps.
template <int BITS, bool XBF16, int KG, int PHASE>
__device__ __forceinline__ void stream_phase(const LayerArgs &a, const RouteView &rv, Stream &st)
{
    constexpr int NS = num_stages(ring_bits(BITS)), SB = stage_bytes(ring_bits(BITS));
    constexpr int NV = (PHASE == 1 || !XBF16) ? 4 : 2;
    constexpr bool kSplit = PHASE == 1 || !XBF16;
    constexpr int NB = PHASE == 0 ? 2 * KG : 2;  // B fragments held
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = st.geo[PHASE];
    const int a0 = g.a0, a1 = g.a1, n = a1 - a0, ts = g.ts, nt = a1 - ts;
    if (n <= 0)
        return;
    const int fmax = a.f > a.fs ? a.f : a.fs;
    Pos q = decode(g, nt > 0 ? ts : a0);
    UnitGeo u = unit_geo(g, q.p);
    int loaded = -1;
    int pb = ring_bits(BITS);  // depth of the loaded pair
    BFrag bf[NB];
    float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
    float accg2[4] = {0.f, 0.f, 0.f, 0.f}, accu2[4] = {0.f, 0.f, 0.f, 0.f};  // gate/up: second group
#pragma unroll 1
    for (int kk = 0; kk < n; ++kk) {
        const int i = kk < nt ? ts + kk : a0 + (kk - nt);
        if (kk == nt && kk > 0)
            q = decode(g, a0);
        if (q.p != loaded) {
            u = unit_geo(g, q.p);
            if (PHASE == 1) {
                // h of pair q.p is complete once all its gate/up strips are
                // published; one warp polls, the others sleep at the barrier
                stream_barrier();
                if (warp == kStreamWarps - 1 && !*st.fail) {
                    const int fp = q.p < g.P_r ? a.f : a.fs;
                    if (!warp_wait_geq(a.pair_done + q.p, static_cast<unsigned>(fp / kTileRows), a.status) &&
                        lane == 0)
                        *st.fail = 1;
                }
                stream_barrier();
            }
            const PairInfo pi = read_pair(rv, q.p);
            pb = pair_bits<BITS>(a, rv.pairs[q.p * kPairInts]);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const int c = b >> 1, lg = warp + (b & 1) * kStreamWarps;  // chunk, group in chunk
                const int gi = c * u.gc + lg;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    bf[b].b0[j] = bf[b].b1[j] = bf[b].b0l[j] = bf[b].b1l[j] = 0u;
                bf[b].bias0 = bf[b].bias1 = 0.f;
                if (c < u.ch && lg < u.gc && gi < u.gk) {
                    BRaw<NV> raw;
                    load_raw<PHASE, XBF16, NV>(a, pi, q.p, gi, fmax, raw);
                    if (BITS != 0 || pb == 4)
                        cook_b<ring_bits(BITS), PHASE, XBF16, NV>(raw, bf[b]);
                    else
                        cook_b<2, PHASE, XBF16, NV>(raw, bf[b]);
                }
            }
            loaded = q.p;
        }
        const int slot = static_cast<int>(st.seq % NS);
        bool ok = !*st.fail;
        if (ok && !mbar_wait_bounded(&st.full[slot], (st.seq / NS) & 1u)) {
            ok = false;
            if (lane == 0) {
                set_status(a.status, kStatusTimeout);
                *st.fail = 1;
            }
        }
        if (ok) {
            // branch-free over the warp's two groups (tiles of absent groups
            // read in-bounds stage bytes and are dropped), so the four (down:
            // two) mma chains of the step schedule together
            const uint8_t *stage = st.ring + slot * SB;
            const int ng = min(u.gc, u.gk - q.c * u.gc);  // groups in this chunk
            const bool g0 = warp < ng, g1 = warp + kStreamWarps < ng;
            if (BITS != 0 || pb == 4)
                step_tiles<ring_bits(BITS), PHASE, KG, kSplit>(stage, bf, q.c, g0, g1, accg, accu, accg2,
                                                               accu2);
            else
                step_tiles<2, PHASE, KG, kSplit>(stage, bf, q.c, g0, g1, accg, accu, accg2, accu2);
        }
        __syncwarp();
        if (ok && lane == 0)
            mbar_arrive(&st.empty[slot]);
        ++st.seq;
        if (q.c == u.ch - 1 || i == a1 - 1 || (nt > 0 && i == ts - 1)) {
            const int rs = st.uc % kRedSlots;
            const unsigned rph = static_cast<unsigned>(st.uc / kRedSlots);
            if (st.uc >= kRedSlots && !*st.fail &&
                !mbar_wait_bounded(&st.red_empty[rs], (rph - 1u) & 1u) && lane == 0) {
                set_status(a.status, kStatusTimeout);
                *st.fail = 1;
            }
            // the two groups' partial sums of the same output rows
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (PHASE == 1) {
                    accg[e] += accu[e];
                } else {
                    accg[e] += accg2[e];
                    accu[e] += accu2[e];
                }
            }
            float4 *rw = st.red + ((rs * kStreamWarps + warp) * 2) * 32;
            rw[lane] = make_float4(accg[0], accg[1], accg[2], accg[3]);
            if (PHASE == 0)
                rw[32 + lane] = make_float4(accu[0], accu[1], accu[2], accu[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                accg[e] = accu[e] = accg2[e] = accu2[e] = 0.f;
            __syncwarp();
            if (lane == 0 && !*st.fail)
                mbar_arrive(&st.red_full[rs]);
            ++st.uc;
        }
        advance(u, q);
    }
}

// The ring's producer (lane 0 of the producer warp): every stage of both
// phases in the CTA's step order, each as soon as its slot is free.
template <int BITS>
__device__ __forceinline__ void produce_all(const LayerArgs &a, const RouteView &rv, Stream &st)
{
    Producer &pr = *st.pr;
    while (pr.phase <= 1 && !*st.fail) {
        const int r = produce<BITS>(a, rv, st.geo, pr, st.ring, st.full, st.empty, true);
        if (r < 0) {
            set_status(a.status, kStatusTimeout);
            *st.fail = 1;
        }
        if (r <= 0)
            break;
    }
}

// One phase of an epilogue warp: the same walk over the CTA's steps; at
// each unit end it owns (units alternate between the epilogue warps) it adds
// the 16 streaming warps' sums in warp order, frees the slot, and finalises
// the unit or, for a unit shared with another CTA, runs the fixup.
template <int BITS, int PHASE>
__device__ __forceinline__ void epi_phase(const LayerArgs &a, const RouteView &rv, Stream &st)
{
    const int e = (threadIdx.x >> 5) - kStreamWarps, lane = threadIdx.x & 31;
    EpiOut eo;
    eo.h_hi = a.h_hi;
    eo.h_lo = a.h_lo;
    eo.hs_part = a.hs_part;
    eo.o = a.o;
    eo.partial = a.partial;
    eo.strip_ctr_g = a.strip_ctr_g;
    eo.strip_ctr_d = a.strip_ctr_d;
    eo.pair_done = a.pair_done;
    eo.d = a.d;
    eo.fmax = a.f > a.fs ? a.f : a.fs;
    eo.max_strips = a.max_strips;
    const Geo &g = st.geo[PHASE];
    const int a0 = g.a0, a1 = g.a1, nt = g.a1 - g.ts;
    if (a0 >= a1)
        return;
    Pos q = decode(g, step_at(g, 0));
    UnitGeo u = unit_geo(g, q.p);
    int curp = q.p;
    int pb = pair_bits<BITS>(a, rv.pairs[q.p * kPairInts]);
#pragma unroll 1
    for (int kk = 0; kk < a1 - a0; ++kk) {
        const int i = step_at(g, kk);
        if (kk == nt && kk > 0)
            q = decode(g, a0);
        if (q.p != curp) {
            u = unit_geo(g, q.p);
            curp = q.p;
            pb = pair_bits<BITS>(a, rv.pairs[q.p * kPairInts]);
        }
        if (unit_ends(g, u, q, i)) {
            if (st.uc % kEpiWarps == e && !*st.fail) {
                const int rs = st.uc % kRedSlots;
                const unsigned rph = static_cast<unsigned>(st.uc / kRedSlots);
                if (!mbar_wait_bounded(&st.red_full[rs], rph & 1u)) {
                    if (lane == 0) {
                        set_status(a.status, kStatusTimeout);
                        *st.fail = 1;
                    }
                } else {
                    float4 tg = make_float4(0.f, 0.f, 0.f, 0.f), tu = tg;
#pragma unroll 4
                    for (int w2 = 0; w2 < kStreamWarps; ++w2) {
                        const float4 *rr = st.red + ((rs * kStreamWarps + w2) * 2) * 32;
                        const float4 vg = rr[lane];
                        tg.x += vg.x, tg.y += vg.y, tg.z += vg.z, tg.w += vg.w;
                        if (PHASE == 0) {
                            const float4 vu = rr[32 + lane];
                            tu.x += vu.x, tu.y += vu.y, tu.z += vu.z, tu.w += vu.w;
                        }
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&st.red_empty[rs]);
                    const int ustart = i - q.c, uend = ustart + u.ch;
                    const int ncols = rv.pairs[q.p * kPairInts + 1];
                    constexpr int RB = ring_bits(BITS);
                    if (ustart >= a0 && uend <= a1) {
                        if (BITS != 0 || pb == 4)
                            finalize_unit<RB, PHASE>(eo, ncols, q.p, q.s, tg, tu);
                        else
                            finalize_unit<2, PHASE>(eo, ncols, q.p, q.s, tg, tu);
                        count_unit<PHASE>(eo, st.pspan, st.pcnt, st.ccnt, q.p, q.s);
                    } else if (BITS != 0 || pb == 4) {
                        fixup_unit<RB, PHASE>(eo, ncols, g, q.p, q.s, ustart, uend, tg, tu, st.pcnt,
                                              st.pspan, st.ccnt);
                    } else {
                        fixup_unit<2, PHASE>(eo, ncols, g, q.p, q.s, ustart, uend, tg, tu, st.pcnt,
                                             st.pspan, st.ccnt);
                    }
                }
            }
            ++st.uc;
        }
        advance(u, q);
    }
}

template <int BITS, bool XBF16, int KG>
__global__ void __launch_bounds__(kThreads, 1) moe_layer_kernel(const __grid_constant__ LayerArgs a)
{
    constexpr int NS = num_stages(ring_bits(BITS));
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int s_ok;
    __shared__ int s_fail;
    __shared__ unsigned s_pcnt[kMaxSpan];
    __shared__ int s_pspan[2];
    __shared__ unsigned s_ccnt[kMaxStripsD];
    Stream st;
    st.ring = smem;
    st.red = reinterpret_cast<float4 *>(smem + NS * stage_bytes(ring_bits(BITS)));
    st.full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes(ring_bits(BITS)) + red_bytes());
    st.empty = st.full + NS;
    st.red_full = st.empty + NS;
    st.red_empty = st.red_full + kRedSlots;
    st.pcnt = s_pcnt;
    st.pspan = s_pspan;
    st.ccnt = s_ccnt;
    st.fail = &s_fail;
    st.seq = 0;
    st.uc = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&st.full[s], 1);
            mbar_init(&st.empty[s], kStreamWarps);
        }
        for (int s = 0; s < kRedSlots; ++s) {
            mbar_init(&st.red_full[s], kStreamWarps);
            mbar_init(&st.red_empty[s], 1);
        }
        fence_mbar_init();
        s_fail = 0;
    }
    for (int j = threadIdx.x; j < kMaxStripsD; j += kThreads)
        s_ccnt[j] = 0u;
    // Launched with programmatic stream serialization: the previous kernel on
    // the stream may still be finishing.  Wait until it has completed and its
    // writes are visible before any global access (the workspace, x), then
    // let the next kernel's launch begin.
    pdl_wait();
    pdl_launch_dependents();
    cta_barrier();
    bool ok = true;

    // ------------------------------------------------------------ phase R
    __shared__ RouteSmem rs;
    RouteView rv;
    int P_r = 0, P_t = 0;
    if (a.do_route) {
        const int rows = a.E + (a.shared_gate ? 1 : 0);
        const int units = rows + static_cast<int>(a.T);
        // unit i runs on warp i / gridDim.x of CTA i % gridDim.x: one per SM first
        const int64_t unit = (int64_t)warp * gridDim.x + blockIdx.x;
        if (unit < units) {
            router_unit<XBF16>(a, static_cast<int>(unit));
            fence_acq_rel();
            __syncwarp();
            unsigned old = 0;
            if (lane == 0)
                old = atom_add_acqrel(a.route_ctr, 1u);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == static_cast<unsigned>(units - 1)) {
                // the last router unit wakes every CTA through its own flag line
                fence_acq_rel();
                for (unsigned c = lane; c < gridDim.x; c += 32)
                    st_relaxed(a.cta_flags + 32 * c, 1u);
            }
        }
        // one poller per CTA, on the CTA's own flag; meanwhile other warps run
        // the routing code once on scratch (in-bounds, results unused) so its
        // instructions are fetched while the logits are still being made
        cta_barrier();
        if (warp == 0) {
            const int good = warp_wait_geq(a.cta_flags + 32 * blockIdx.x, 1u, a.status) ? 1 : 0;
            if (lane == 0) {
                s_ok = good;
                a.cta_flags[32 * blockIdx.x] = 0u;  // only this CTA reads it
            }
        } else if (warp <= (a.E + 31) / 32) {
            route_chunk(rs.lg, rs.key, a.E, a.k, warp - 1, a.router_sigmoid, rs.warm_id, rs.warm_p);
        }
        cta_barrier();
        ok = s_ok != 0;
        // route: stage logits and keys, rank every expert, then warp t
        // turns token t's selection into weights; the last warp builds the pairs
        const int T = static_cast<int>(a.T), E = a.E, kk = a.k, E4 = (a.E + 3) & ~3;
        if (ok) {
            for (int idx = threadIdx.x; idx < T * E; idx += kThreads) {
                const int t = idx / E, e = idx - t * E;
                float l = __ldcg(a.logits + (int64_t)t * a.Epad + e);
                if (l != l) {
                    set_status(a.status, kStatusBadArg);
                    l = -INFINITY;
                }
                // selection key: the logit; with a bias, logit + bias
                // (softmax) or fl32(sigmoid(logit)) + bias (sigmoid)
                float key = a.expert_bias ? __fadd_rn(a.router_sigmoid ? sigmoid_fast(l) : l,
                                                      __ldg(a.expert_bias + e))
                                          : l;
                if (key != key)
                    key = -INFINITY;
                // outside the routing mask: never selected, no softmax term
                if (a.mask.on && !((a.mask.w[e >> 5] >> (e & 31)) & 1u)) {
                    key = -INFINITY;
                    l = -INFINITY;
                }
                rs.lg[t * E4 + e] = l;
                rs.key[t * E4 + e] = key;
            }
        }
        cta_barrier();
        if (ok) {
            const int nc = (E + 31) / 32;
            for (int task = warp; task < T * nc; task += kWarps) {
                const int t = task / nc, c = task - t * nc;
                route_chunk(rs.lg + t * E4, rs.key + t * E4, E, kk, c, a.router_sigmoid,
                            rs.ids + t * kk, rs.prob + t * kk);
            }
        }
        cta_barrier();
        if (ok && warp < T) {
            const int t = warp;
            float psel = 0.f;
            for (int j = 0; j < kk; ++j)
                psel += rs.prob[t * kk + j];
            if (lane < kk) {
                const float pj = rs.prob[t * kk + lane];
                const float wv = (a.norm ? __fdividef(pj, psel) : pj) * a.rsf;
                rs.weights[t * kk + lane] = wv;
                if (blockIdx.x == 0) {
                    const int id = rs.ids[t * kk + lane];
                    a.ids[t * kk + lane] = id;
                    a.weights[t * kk + lane] = wv;
                    if (a.ids_out)
                        a.ids_out[t * kk + lane] = id;
                    if (a.w_out)
                        a.w_out[t * kk + lane] = wv;
                }
            }
            if (lane == 0)
                rs.shared_w[t] =
                    a.shared_gate ? sigmoid_fast(__ldcg(a.logits + (int64_t)t * a.Epad + a.E)) : 1.0f;
        }
        // the pair table needs only the ids: built while the weights are
        if (ok && warp == kWarps - 1)
            cta_dispatch(a, rs);
        cta_barrier();
        rv.pairs = &rs.pairs[0][0];
        rv.route_map = rs.route_map;
        rv.weights = rs.weights;
        rv.shared_w = rs.shared_w;
        if (ok) {
            P_r = rs.meta[0];
            P_t = rs.meta[1];
        }
    } else {
        rv.pairs = a.pairs;
        rv.route_map = a.route_map;
        rv.weights = a.weights;
        rv.shared_w = a.shared_w;
        P_r = __ldcg(a.meta + 0);
        P_t = __ldcg(a.meta + 1);
    }
    if (!ok && threadIdx.x == 0)
        s_fail = 1;

    // ------------------------------------------------------------ phases G, D
    __shared__ Geo s_geo[2];
    __shared__ Producer s_pr;
    if (lane == 0 && warp < 2) {
        Geo gg = make_geo(a, warp, P_r, P_t);
        set_order(gg);
        s_geo[warp] = gg;
    }
    cta_barrier();
    if (threadIdx.x == 0) {
        if (s_geo[0].ch0 > KG || (P_t > P_r && s_geo[0].ch1 > KG) || s_geo[1].gk0 > kDownGroupsMax ||
            (P_t > P_r && s_geo[1].gk1 > kDownGroupsMax)) {
            // the host checks both limits; never reached
            set_status(a.status, kStatusBadArg);
            s_fail = 1;
        }
    }
    cta_barrier();
    st.geo = s_geo;
    st.pr = &s_pr;
    if (warp < kStreamWarps) {
        stream_phase<BITS, XBF16, KG, 0>(a, rv, st);
        stream_phase<BITS, XBF16, KG, 1>(a, rv, st);
    } else if (warp == kProducerWarp) {
        if (lane == 0) {
            s_pr.phase = 0;
            s_pr.next = 0;
            producer_seek(s_geo, s_pr);
            if (!s_fail)
                produce_all<BITS>(a, rv, st);
        }
        __syncwarp();
    } else {
        if (warp == kStreamWarps) {
            // the pairs of this CTA's gate/up range, for batched strip counts
            if (lane == 0) {
                s_pspan[0] = 0;
                s_pspan[1] = 0;
                if (s_geo[0].a0 < s_geo[0].a1) {
                    const int pf = decode(s_geo[0], s_geo[0].a0).p, pl = decode(s_geo[0], s_geo[0].a1 - 1).p;
                    if (pl - pf + 1 <= kMaxSpan) {
                        s_pspan[0] = pf;
                        s_pspan[1] = pl - pf + 1;
                    }
                }
            }
            for (int j = lane; j < kMaxSpan; j += 32)
                s_pcnt[j] = 0u;
        }
        epi_barrier();
        epi_phase<BITS, 0>(a, rv, st);
        // publish this CTA's finished gate/up strips: the barrier orders the
        // other epilogue warp's h stores before the release fence
        epi_barrier();
        if (warp == kStreamWarps && lane == 0 && !s_fail) {
            bool any = false;
            for (int j = 0; j < s_pspan[1]; ++j)
                any |= s_pcnt[j] != 0u;
            if (any) {
                fence_acq_rel();
                for (int j = 0; j < s_pspan[1]; ++j)
                    if (s_pcnt[j])
                        red_add_relaxed(a.pair_done + s_pspan[0] + j, s_pcnt[j]);
            }
        }
        epi_phase<BITS, 1>(a, rv, st);
        epi_barrier();
        if (a.fused_combine && warp == kStreamWarps && lane == 0 && !s_fail) {
            // publish the finished down units per output strip
            const int ns = a.d / kTileRows;
            bool any = false;
            for (int j = 0; j < ns; ++j)
                any |= s_ccnt[j] != 0u;
            if (any) {
                fence_acq_rel();
                for (int j = 0; j < ns; ++j)
                    if (s_ccnt[j])
                        red_add_relaxed(a.comb_ctr + j, s_ccnt[j]);
            }
        }
    }
    cta_barrier();

    // ------------------------------------------------------------ combine
    // (T <= 8) CTA c owns output strips c, c + grid, ...: once all P_t pairs
    // have published their down unit of a strip, y rows = sum_j w_j o_j
    // (+ shared) in rank order.
    if (a.fused_combine) {
        const int ns = a.d / kTileRows;
        if (warp == 0 && !s_fail) {
            for (int s = blockIdx.x; s < ns; s += gridDim.x)
                if (!warp_wait_geq(a.comb_ctr + s, static_cast<unsigned>(P_t), a.status)) {
                    if (lane == 0)
                        s_fail = 1;
                    break;
                }
        }
        cta_barrier();
        if (!s_fail) {
            const int T = static_cast<int>(a.T), kk = a.k, d = a.d;
            const bool has_sh = P_t > P_r;
            for (int s = blockIdx.x; s < ns; s += gridDim.x) {
                for (int i = threadIdx.x; i < kTileRows * T; i += kThreads) {
                    const int t = i / kTileRows, row = 16 * s + i % kTileRows;
                    float yv = 0.f;
                    for (int j = 0; j < kk; ++j) {
                        const int rm = rv.route_map[t * (kk + 1) + j];
                        yv = fmaf(rv.weights[t * kk + j], __ldcg(a.o + (int64_t)rm * d + row), yv);
                    }
                    if (has_sh) {
                        const int rm = rv.route_map[t * (kk + 1) + kk];
                        yv = fmaf(rv.shared_w[t], __ldcg(a.o + (int64_t)rm * d + row), yv);
                    }
                    a.y[(int64_t)t * d + row] = yv;
                }
                if (threadIdx.x == 0)
                    a.comb_ctr[s] = 0u;
            }
        }
    }

    // ------------------------------------------------------------ exit
    if (warp == 0) {
        if (lane == 0) {
            // every stage issued has been consumed unless a wait ran out;
            // then wait (bounded) for the copies still in flight
            const uint32_t n = s_pr.next;
            for (uint32_t j = n > static_cast<uint32_t>(NS) ? n - NS : 0u; j < n; ++j)
                (void)mbar_wait_bounded(&st.full[j % NS], (j / NS) & 1u);
        }
        // the last CTA out resets the per-launch counters
        unsigned old = 0;
        if (lane == 0)
            old = atom_add_acqrel(a.exit_ctr, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == gridDim.x - 1) {
            for (int p = lane; p < a.max_pairs; p += 32)
                a.pair_done[p] = 0u;
            if (lane == 0) {
                *a.route_ctr = 0u;
                fence_acq_rel();
                *a.exit_ctr = 0u;
            }
        }
    }
}

template <int BITS, bool XBF16, int KG>
cudaError_t launch_t(const LayerArgs &a, cudaStream_t stream)
{
    auto kern = moe_layer_kernel<BITS, XBF16, KG>;
    const int smem = smem_bytes(ring_bits(BITS));
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_done[dev & 63] = 1;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(device_sm_count() * kMaxLayerCtasPerSm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // cooperative (every CTA resident: the phases hand off through global
    // counters) and, where the runtime accepts it, programmatic stream
    // serialization so that the launch overlaps the previous kernel's tail
    static int pdl_refused[64] = {0};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_refused[dev & 63] ? 1 : 2;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess && cfg.numAttrs == 2) {
        (void)cudaGetLastError();
        pdl_refused[dev & 63] = 1;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, a);
    }
    return e;
}

// y[t] = sum_j w[t,j] * o[pair(t,j)] (rank order) + shared_w[t] * o[shared]
__global__ void __launch_bounds__(256) combine_kernel(const LayerArgs a)
{
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

cudaError_t launch_combine(const LayerArgs &a, cudaStream_t stream)
{
    const int64_t n = a.T * (a.d / 4);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    combine_kernel<<<static_cast<unsigned>(blocks < cap ? blocks : cap), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

int layer_grid_ctas_max() { return device_sm_count() * kMaxLayerCtasPerSm; }

cudaError_t launch_layer(const LayerArgs &a, cudaStream_t stream)
{
    // gate/up chunks per strip (d / 2048, rounded up) decide how many B
    // fragments a streaming warp holds
    const int kg = (a.d / kGroup + kChunkGroups - 1) / kChunkGroups;
    if (kg > 2 || a.f / kGroup > kDownGroupsMax || a.fs / kGroup > kDownGroupsMax)
        return cudaErrorInvalidValue;
    if (a.mixed)
        return kg <= 1 ? (a.x_bf16 ? launch_t<0, true, 1>(a, stream) : launch_t<0, false, 1>(a, stream))
                       : (a.x_bf16 ? launch_t<0, true, 2>(a, stream) : launch_t<0, false, 2>(a, stream));
    if (kg <= 1) {
        if (a.bits == 4)
            return a.x_bf16 ? launch_t<4, true, 1>(a, stream) : launch_t<4, false, 1>(a, stream);
        return a.x_bf16 ? launch_t<2, true, 1>(a, stream) : launch_t<2, false, 1>(a, stream);
    }
    if (a.bits == 4)
        return a.x_bf16 ? launch_t<4, true, 2>(a, stream) : launch_t<4, false, 2>(a, stream);
    return a.x_bf16 ? launch_t<2, true, 2>(a, stream) : launch_t<2, false, 2>(a, stream);
}

}  // namespace smoe
