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

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kNS = 8;  // stages per warp ring (one group each)
constexpr long long kSpinCycles = 4000000000ll;  // ~2 s at 2 GHz

__host__ __device__ constexpr int kStageBytes(int bits) { return 2 * tile_bytes(bits); }
__host__ __device__ constexpr int ring_bytes(int bits) { return kNS * kStageBytes(bits); }
__host__ __device__ constexpr int smem_bytes(int bits)
{
    return kWarps * ring_bytes(bits) + kWarps * kNS * 8;
}

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

// CTA-wide named barrier 1 (all kThreads threads).
__device__ __forceinline__ void cta_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
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

constexpr int kPerLane = kMaxExperts / 32;

__device__ __noinline__ void route_one_token(const float *lg, int E, int k, int norm, const float *bias,
                                int16_t *ids_s, float *w_s, int32_t *ids_g, float *w_g,
                                int *status)
{
    const int lane = threadIdx.x & 31;
    float key[kPerLane], lv[kPerLane];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        float l = -INFINITY, kk = -INFINITY;
        if (e < E) {
            l = __ldcg(lg + e);
            if (l != l) {
                set_status(status, kStatusBadArg);
                l = -INFINITY;
            }
            kk = bias ? __fadd_rn(l, __ldg(bias + e)) : l;
            if (kk != kk)
                kk = -INFINITY;
        }
        key[i] = kk;
        lv[i] = l;
        m = fmaxf(m, l);
    }
    for (int o = 16; o; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i)
        if (lane + 32 * i < E)
            z += expf(lv[i] - m);
    for (int o = 16; o; o >>= 1)
        z += __shfl_xor_sync(0xffffffffu, z, o);
    unsigned taken = 0u;
    float psel = 0.f, pj_mine = 0.f;
    int ej_mine = 0;
    for (int j = 0; j < k; ++j) {
        float bk = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u))
                if (bi == 0x7fffffff || key[i] > bk || (key[i] == bk && e < bi)) {
                    bk = key[i];
                    bi = e;
                }
        }
        for (int o = 16; o; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != 0x7fffffff && (bi == 0x7fffffff || ok > bk || (ok == bk && oi < bi))) {
                bk = ok;
                bi = oi;
            }
        }
        if ((bi & 31) == lane)
            taken |= 1u << (bi >> 5);
        float mine = lv[0];
#pragma unroll
        for (int i = 1; i < kPerLane; ++i)
            if ((bi >> 5) == i)
                mine = lv[i];
        const float p = expf(__shfl_sync(0xffffffffu, mine, bi & 31) - m) / z;
        psel += p;
        if (lane == j) {
            pj_mine = p;
            ej_mine = bi;
        }
    }
    if (lane < k) {
        const float wv = norm ? pj_mine / psel : pj_mine;
        ids_s[lane] = static_cast<int16_t>(ej_mine);
        w_s[lane] = wv;
        if (ids_g)
            ids_g[lane] = ej_mine;
        if (w_g)
            w_g[lane] = wv;
    }
}

// Phase R work of one warp: unit < E (+1 shared gate row) -> logits of that
// row for all tokens; unit >= rows -> group sums of token (unit - rows).
template <bool XBF16>
__device__ __noinline__ void router_unit(const LayerArgs &a, int unit)
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
struct RouteSmem {
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

// Warp 0 of the CTA: pair table from the routed ids (T <= 8).  Pair = one
// selected expert with the ascending tokens that chose it, pairs in order of
// first appearance; then the shared expert's pair.
__device__ __noinline__ void cta_dispatch(const LayerArgs &a, RouteSmem &r)
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

// Per-warp constants of one phase (passed by value to the cold helpers).
struct Phase {
    int P_r, P_t, fmax, nstrip;  // pairs, widest f, strips of fmax
    int U_r, U_s, UR, U, W;      // groups per routed / shared pair, totals, warps
    Split sp;                    // the stream-K split of U over W
    int u0, u1;                  // this warp's group range
    int gps_r, gps_s;            // groups per strip
    long long w;                 // global warp index
};

// This lane's 16 activations of one group (bf16 x: 2 vectors; fp32 x: 4;
// h of the down phase: hi in v[0..1], lo in v[2..3]) and the group sums
// (X0, X1) of the two output columns the lane accumulates.
template <int NV>
struct BRaw {
    uint4 v[NV];
    float2 xs0, xs1;
};

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

template <int PHASE, bool XBF16, int NV>
__device__ __forceinline__ void load_b(const LayerArgs &a, const PairInfo &pi, int p, int g,
                                       int fmax, int nstrip, BRaw<NV> &r)
{
    const int lane = threadIdx.x & 31, gq = lane >> 2, tig = lane & 3;
    const int d = a.d;
    const bool valid = gq < pi.ncols;
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    const float2 z2 = make_float2(0.f, 0.f);
    if (PHASE == 0) {
        if (XBF16) {
            const uint4 *row = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const uint16_t *>(a.x) + (int64_t)pi.tok * d + g * kGroup + 16 * tig);
            r.v[0] = valid ? __ldg(row) : z4;
            r.v[1] = valid ? __ldg(row + 1) : z4;
        } else {
            const uint4 *row = reinterpret_cast<const uint4 *>(
                reinterpret_cast<const float *>(a.x) + (int64_t)pi.tok * d + g * kGroup + 16 * tig);
#pragma unroll
            for (int i = 0; i < NV; ++i)
                r.v[i] = valid ? __ldg(row + i) : z4;
        }
        const float2 *xs = reinterpret_cast<const float2 *>(a.xsum);
        r.xs0 = pi.t0 >= 0 ? __ldcg(xs + (int64_t)pi.t0 * (d / kGroup) + g) : z2;
        r.xs1 = pi.t1 >= 0 ? __ldcg(xs + (int64_t)pi.t1 * (d / kGroup) + g) : z2;
    } else {
        const int64_t off = ((int64_t)p * kPairCols + gq) * fmax + g * kGroup + 16 * tig;
        const uint4 *hi = reinterpret_cast<const uint4 *>(a.h_hi + off);
        const uint4 *lo = reinterpret_cast<const uint4 *>(a.h_lo + off);
        r.v[0] = valid ? __ldcg(hi) : z4;
        r.v[1] = valid ? __ldcg(hi + 1) : z4;
        r.v[2] = valid ? __ldcg(lo) : z4;
        r.v[3] = valid ? __ldcg(lo + 1) : z4;
        // group sums of h: lane (gq, tig) loads strip 4g + (gq & 3) of its two
        // columns; cook_b adds the four strips with shuffles
        const int c0 = 2 * tig, c1 = c0 + 1;
        const float2 *hp = reinterpret_cast<const float2 *>(a.hs_part);
        const int st = 4 * g + (gq & 3);
        r.xs0 = c0 < pi.ncols ? __ldcg(hp + ((int64_t)p * kPairCols + c0) * nstrip + st) : z2;
        r.xs1 = c1 < pi.ncols ? __ldcg(hp + ((int64_t)p * kPairCols + c1) * nstrip + st) : z2;
    }
}

// mma B fragments (hi and, for fp32 / h activations, lo) and the two column
// biases -(128 + L) X (Q2: -(129.5 X0 + 33.5 X1)) from a BRaw
struct BFrag {
    uint32_t b0[4], b1[4], b0l[4], b1l[4];
    float bias0, bias1;
};

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
    if (BITS == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f.b1[j] = bf16x2_quarter(f.b1[j]);
            f.b1l[j] = bf16x2_quarter(f.b1l[j]);
        }
        f.bias0 = 129.5f * x0.x + 33.5f * x0.y;
        f.bias1 = 129.5f * x1.x + 33.5f * x1.y;
    } else {
        f.bias0 = 135.5f * (x0.x + x0.y);
        f.bias1 = 135.5f * (x1.x + x1.y);
    }
}

// Decode + multiply one tile from shared memory into acc (two independent
// mma chains: k-subtiles 0,2 and 1,3).
template <int BITS, bool SPLIT>
__device__ __forceinline__ void mac_tile(const uint8_t *tile, const BFrag &f, float (&acc)[4])
{
    constexpr int CB = tile_code_bytes(BITS);
    const int lane = threadIdx.x & 31, gq = lane >> 2;
    const uint32_t sc = *reinterpret_cast<const uint32_t *>(tile + CB + 4 * gq);
    const float2 s01 = __half22float2(*reinterpret_cast<const __half2 *>(&sc));
    float dv[4] = {-f.bias0, -f.bias1, -f.bias0, -f.bias1};
    float dw[4] = {0.f, 0.f, 0.f, 0.f};
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
            float(&dd)[4] = (j & 1) ? dw : dv;
            mma_bf16(dd, A, f.b0[j], f.b1[j]);
            if (SPLIT)
                mma_bf16(dd, A, f.b0l[j], f.b1l[j]);
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
            float(&dd)[4] = (j & 1) ? dw : dv;
            mma_bf16(dd, A, f.b0[j], f.b1[j]);
            if (SPLIT)
                mma_bf16(dd, A, f.b0l[j], f.b1l[j]);
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
        dv[e] += dw[e];
    acc[0] = fmaf(s01.x, dv[0], acc[0]);
    acc[1] = fmaf(s01.x, dv[1], acc[1]);
    acc[2] = fmaf(s01.y, dv[2], acc[2]);
    acc[3] = fmaf(s01.y, dv[3], acc[3]);
}

__device__ __forceinline__ int pair_of(const Phase &ph, int u)
{
    return u < ph.UR ? u / ph.U_r : ph.P_r + (u - ph.UR) / ph.U_s;
}
__device__ __forceinline__ int pair_start(const Phase &ph, int p)
{
    return p < ph.P_r ? p * ph.U_r : ph.UR + (p - ph.P_r) * ph.U_s;
}
__device__ __forceinline__ int pair_units(const Phase &ph, int p) { return p < ph.P_r ? ph.U_r : ph.U_s; }

// Finalise strip s of pair p from its full-K accumulators (cold path).
// Phase 0: h = SiLU(g) * u stored as bf16 hi + lo, the strip's per-class
// sums of h, the pair's strip count (the strip completing the pair wakes the
// CTAs whose down ranges read it).  Phase 1: o, then (T <= 8) the combine of
// output strip s by the last pair to finish it, in rank order.
template <int BITS, int PHASE>
__device__ __noinline__ void finalize_strip(const LayerArgs &a, const RouteView rv, const Phase ph,
                                            int p, int s, float4 ag, float4 au)
{
    constexpr float L = BITS == 4 ? 7.5f : 1.5f;
    const int lane = threadIdx.x & 31, gq = lane >> 2, tig = lane & 3;
    const int d = a.d;
    const int ncols = rv.pairs[p * kPairInts + 1];
    const float invL = 1.0f / L;
    const int c0 = 2 * tig;
    const float gv[4] = {ag.x, ag.y, ag.z, ag.w}, uv[4] = {au.x, au.y, au.z, au.w};
    if (PHASE == 0) {
        float hs[2] = {0.f, 0.f};  // per output column, this lane's rows
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float g = gv[e] * invL, u = uv[e] * invL;
            const float hv = g / (1.0f + expf(-g)) * u;
            const int col = c0 + (e & 1);
            const int row = 16 * s + gq + 8 * (e >> 1);
            if (col < ncols) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
                const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
                const int64_t off = ((int64_t)p * kPairCols + col) * ph.fmax + row;
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
                    a.hs_part[(((int64_t)p * kPairCols + c0 + c) * ph.nstrip + s) * 2 + cls] = hs[c];
        }
        fence_acq_rel();
        __syncwarp();
        unsigned old = 0;
        if (lane == 0)
            old = atom_add_acqrel(a.pair_done + p, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        const int fp = p < ph.P_r ? a.f : a.fs;
        if (old == static_cast<unsigned>(fp / kTileRows - 1)) {
            // down-phase geometry (groups of 16 rows x 64 columns of W_down)
            const int DU_r = (d / kTileRows) * (a.f / kGroup);
            const int DU_s = ph.P_t > ph.P_r ? (d / kTileRows) * (a.fs / kGroup) : 0;
            const int DUR = ph.P_r * DU_r;
            const int DU = DUR + (ph.P_t - ph.P_r) * DU_s;
            const int64_t Wall = (int64_t)gridDim.x * kWarps;
            const int DW = DU < Wall ? DU : static_cast<int>(Wall);
            const int ps = p < ph.P_r ? p * DU_r : DUR + (p - ph.P_r) * DU_s;
            const int pe = ps + (p < ph.P_r ? DU_r : DU_s);
            const Split dsp = make_split(DU, DW);
            const int ca = split_owner(dsp, ps) / kWarps;
            const int cb = split_owner(dsp, pe - 1) / kWarps;
            fence_acq_rel();
            for (int c = ca + lane; c <= cb; c += 32)
                red_add_relaxed(a.cta_flags + 32 * c + 1, 1u);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = c0 + (e & 1);
            const int row = 16 * s + gq + 8 * (e >> 1);
            if (col < ncols)
                a.o[((int64_t)p * kPairCols + col) * d + row] = gv[e] * invL;
        }
        if (!a.fused_combine)
            return;
        fence_acq_rel();
        __syncwarp();
        unsigned old = 0;
        if (lane == 0)
            old = atom_add_acqrel(a.comb_ctr + s, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == static_cast<unsigned>(ph.P_t - 1)) {
            fence_acq_rel();
            const int T = static_cast<int>(a.T), kk = a.k;
            const bool has_sh = ph.P_t > ph.P_r;
            for (int i = lane; i < kTileRows * T; i += 32) {
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
            __syncwarp();
            if (lane == 0)
                a.comb_ctr[s] = 0u;
        }
    }
}

// Flush strip (p, s) = groups [ss, se) (cold path): finalise it if this warp
// covered all of it, else store the partial and let the last contributor
// (arrival counter) sum the partials in warp order and finalise.
template <int BITS, int PHASE>
__device__ __noinline__ void flush_strip(const LayerArgs &a, const RouteView rv, const Phase ph,
                                         int p, int s, int ss, int se, float4 ag, float4 au)
{
    const int lane = threadIdx.x & 31;
    const int wf = split_owner(ph.sp, ss), wl = split_owner(ph.sp, se - 1);
    if (wf == wl) {
        finalize_strip<BITS, PHASE>(a, rv, ph, p, s, ag, au);
        return;
    }
    const int myslot = ph.u0 >= ss ? 0 : 1;
    float4 *mine = reinterpret_cast<float4 *>(a.partial) + ((ph.w * 2 + myslot) * 2) * 32;
    mine[lane] = ag;
    if (PHASE == 0)
        mine[32 + lane] = au;
    fence_acq_rel();
    __syncwarp();
    unsigned *ctr = (PHASE == 0 ? a.strip_ctr_g : a.strip_ctr_d) + (int64_t)p * a.max_strips + s;
    unsigned old = 0;
    if (lane == 0)
        old = atom_add_acqrel(ctr, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != static_cast<unsigned>(wl - wf))
        return;
    fence_acq_rel();
    float4 tg = make_float4(0.f, 0.f, 0.f, 0.f), tu = tg;
    for (int w0 = wf; w0 <= wl; w0 += 4) {
        float4 vg[4], vu[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int ww = w0 + q;
            vg[q] = vu[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ww <= wl) {
                const int sl = split_start(ph.sp, ww) >= ss ? 0 : 1;
                const float4 *src = reinterpret_cast<const float4 *>(a.partial) + ((ww * 2 + sl) * 2) * 32;
                vg[q] = __ldcg(src + lane);
                if (PHASE == 0)
                    vu[q] = __ldcg(src + 32 + lane);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            tg.x += vg[q].x, tg.y += vg[q].y, tg.z += vg[q].z, tg.w += vg[q].w;
            tu.x += vu[q].x, tu.y += vu[q].y, tu.z += vu[q].z, tu.w += vu[q].w;
        }
    }
    if (lane == 0)
        *ctr = 0u;
    finalize_strip<BITS, PHASE>(a, rv, ph, p, s, tg, tu);
}

// One streaming phase (0: gate/up + SiLU, 1: down + combine) of one warp.
// The unit of work is a group: 64 input columns of 16 output rows (phase 0:
// the gate tile and the up tile of those rows, phase 1: one down tile).  A
// pair's groups are contiguous in memory (strip-major), so a warp's range is
// a few contiguous runs; each stage of the warp's ring holds one group.
// Returns false if a bounded wait ran out (the status word is set).
template <int BITS, bool XBF16, int PHASE>
__device__ __forceinline__ bool run_phase(const LayerArgs &a, uint8_t *ring, uint64_t *bars,
                                          uint32_t &ring_seq, int P_r, int P_t, int fmax,
                                          int64_t w, int64_t Wall, bool enabled, int *s_ok,
                                          const RouteView &rv)
{
    constexpr int TB = tile_bytes(BITS);
    constexpr int TPG = PHASE == 0 ? 2 : 1;  // tiles per group
    constexpr int GB = TPG * TB;             // bytes per group
    constexpr int NV = (PHASE == 1 || !XBF16) ? 4 : 2;
    constexpr bool kSplit = PHASE == 1 || !XBF16;
    const int lane = threadIdx.x & 31;
    const int d = a.d;
    bool ok = true;
    Phase ph;
    ph.P_r = P_r;
    ph.P_t = P_t;
    ph.fmax = fmax;
    ph.nstrip = fmax / kTileRows;
    {
        const int Kr = PHASE == 0 ? d : a.f, Ks = PHASE == 0 ? d : a.fs;
        const int Rr = PHASE == 0 ? a.f : d, Rs = PHASE == 0 ? a.fs : d;
        ph.gps_r = Kr / kGroup;
        ph.gps_s = Ks / kGroup;
        ph.U_r = (Rr / kTileRows) * ph.gps_r;
        ph.U_s = P_t > P_r ? (Rs / kTileRows) * ph.gps_s : 0;
        ph.UR = P_r * ph.U_r;
        ph.U = enabled ? ph.UR + (P_t - P_r) * ph.U_s : 0;
        ph.W = ph.U < Wall ? ph.U : static_cast<int>(Wall);
        ph.w = w;
        const bool act = w < ph.W;
        ph.sp = make_split(ph.U, ph.W);
        ph.u0 = act ? split_start(ph.sp, static_cast<int>(w)) : 0;
        ph.u1 = act ? split_start(ph.sp, static_cast<int>(w) + 1) : 0;
    }
    const int u0 = ph.u0, u1 = ph.u1, n = u1 - u0;
    auto pair_base = [&](int p) -> const uint8_t * {
        const int e = rv.pairs[p * kPairInts];
        return e >= 0 ? a.tiles_routed + (int64_t)e * a.expert_bytes_routed +
                            (PHASE == 0 ? 0 : a.down_off_routed)
                      : a.tiles_shared + (PHASE == 0 ? 0 : a.down_off_shared);
    };
    // Issue state, lane 0 only: the pair being copied and the next pair's
    // base, looked up one pair ahead.
    int is_ps = 0, is_end = 0, is_p = 0;
    const uint8_t *is_base = nullptr, *nx_base = nullptr;
    int issued = 0, waited = 0;  // stages issued / consumed, for a bounded drain
    if (lane == 0 && n > 0) {
        is_p = pair_of(ph, u0);
        is_ps = pair_start(ph, is_p);
        is_end = is_ps + pair_units(ph, is_p);
        is_base = pair_base(is_p);
        nx_base = is_end < u1 ? pair_base(is_p + 1) : nullptr;
    }
    auto issue = [&](int i) {  // lane 0: the stage of group u0 + i
        if (i >= n)
            return;
        issued = i + 1;
        const int u = u0 + i;
        if (u == is_end) {
            is_p += 1;
            is_ps = is_end;
            is_end += pair_units(ph, is_p);
            is_base = nx_base;
            nx_base = is_end < u1 ? pair_base(is_p + 1) : nullptr;
        }
        const int slot = static_cast<int>((ring_seq + i) % kNS);
        mbar_arrive_expect_tx(&bars[slot], GB);
        bulk_g2s(ring + slot * kStageBytes(BITS), is_base + (int64_t)(u - is_ps) * GB, GB,
                 &bars[slot]);
    };
    if (lane == 0)
        for (int i = 0; i < kNS; ++i)
            issue(i);

    if (PHASE == 1) {
        // Down needs h of its pairs.  The first weight copies are already in
        // flight; warp 0 waits until the strip-completing gate/up warps have
        // woken this CTA for every pair its warps read, while the other warps
        // sleep at a barrier.  Every warp passes both barriers whatever its
        // state, so a timeout cannot strand a warp.
        cta_barrier();
        if ((threadIdx.x >> 5) == 0) {
            int good = enabled ? 1 : 0;
            const int64_t wa = (int64_t)blockIdx.x * kWarps;
            int64_t wb = wa + kWarps - 1;
            if (wb > ph.W - 1)
                wb = ph.W - 1;
            if (good && wa < ph.W) {
                const int pa = pair_of(ph, split_start(ph.sp, static_cast<int>(wa)));
                const int pb = pair_of(ph, split_start(ph.sp, static_cast<int>(wb) + 1) - 1);
                good = warp_wait_geq(a.cta_flags + 32 * blockIdx.x + 1,
                                     static_cast<unsigned>(pb - pa + 1), a.status)
                           ? 1
                           : 0;
            }
            if (lane == 0) {
                *s_ok = good;
                a.cta_flags[32 * blockIdx.x + 1] = 0u;
            }
        }
        cta_barrier();
        ok = *s_ok != 0;
        if (!enabled)
            return false;
    }

    // ---- main loop over (pair, strip) segments -------------------------
    int cp = n > 0 ? pair_of(ph, u0) : 0;
    int cps = pair_start(ph, cp), cpe = cps + pair_units(ph, cp);
    int pair_read = -1;
    PairInfo pi = {0, 0, -1, -1};
    uint32_t seq = ring_seq;  // ring sequence number of the next stage to consume
    int i = 0;                // stage index within this phase
    int u = u0;
#pragma unroll 1
    while (u < u1 && ok) {
        if (u >= cpe) {
            cp += 1;
            cps = cpe;
            cpe += pair_units(ph, cp);
        }
        const int p = cp;
        const int lt = u - cps;
        const int gps = p < P_r ? ph.gps_r : ph.gps_s;
        const int s = lt / gps;
        const int g0 = lt - s * gps;
        const int ss = u - g0, se = ss + gps;
        const int ue = se < u1 ? se : u1;
        const int g1 = g0 + (ue - u);
        if (p != pair_read) {
            pi = read_pair(rv, p);
            pair_read = p;
        }
        float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
        BRaw<NV> cur, nxt;
        load_b<PHASE, XBF16, NV>(a, pi, p, g0, fmax, ph.nstrip, cur);
#pragma unroll 1
        for (int g = g0; g < g1; ++g) {
            if (g + 1 < g1)
                load_b<PHASE, XBF16, NV>(a, pi, p, g + 1, fmax, ph.nstrip, nxt);
            BFrag f;
            cook_b<BITS, PHASE, XBF16, NV>(cur, f);
            const int slot = static_cast<int>(seq % kNS);
            if (!mbar_wait_bounded(&bars[slot], (seq / kNS) & 1u)) {
                ok = false;
                break;
            }
            waited = i + 1;
            const uint8_t *st = ring + slot * kStageBytes(BITS);
            mac_tile<BITS, kSplit>(st, f, ag);
            if (PHASE == 0)
                mac_tile<BITS, kSplit>(st + TB, f, au);
            __syncwarp();
            if (lane == 0)
                issue(i + kNS);
            ++i;
            ++seq;
            cur = nxt;
        }
        if (!ok)
            break;
        flush_strip<BITS, PHASE>(a, rv, ph, p, s, ss, se, make_float4(ag[0], ag[1], ag[2], ag[3]),
                                 make_float4(au[0], au[1], au[2], au[3]));
        u = ue;
    }
    if (!ok) {
        if (lane == 0) {
            set_status(a.status, kStatusTimeout);
            // drain this warp's copies still in flight (bounded)
            for (int j = waited; j < issued; ++j) {
                const uint32_t sq = ring_seq + static_cast<uint32_t>(j);
                (void)mbar_wait_bounded(&bars[sq % kNS], (sq / kNS) & 1u);
            }
        }
        __syncwarp();
        return false;
    }
    ring_seq += static_cast<uint32_t>(n);
    return true;
}

template <int BITS, bool XBF16>
__global__ void __launch_bounds__(kThreads, 2) moe_layer_kernel(const __grid_constant__ LayerArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *ring = smem + warp * ring_bytes(BITS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kWarps * ring_bytes(BITS)) + warp * kNS;
    if (lane == 0) {
        for (int s = 0; s < kNS; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    __shared__ int s_ok;
    const int64_t w = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t Wall = (int64_t)gridDim.x * kWarps;
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
        // one poller per CTA, on the CTA's own flag; the others sleep
        cta_barrier();
        if (warp == 0) {
            const int good = warp_wait_geq(a.cta_flags + 32 * blockIdx.x, 1u, a.status) ? 1 : 0;
            if (lane == 0) {
                s_ok = good;
                a.cta_flags[32 * blockIdx.x] = 0u;  // only this CTA reads it
            }
        }
        cta_barrier();
        ok = s_ok != 0;
        // route the tokens (one warp each), then warp 0 builds the pair table
        if (ok && warp < a.T) {
            const bool out = blockIdx.x == 0;
            const int t = warp;
            route_one_token(a.logits + (int64_t)t * a.Epad, a.E, a.k, a.norm, a.expert_bias,
                            rs.ids + t * a.k, rs.weights + t * a.k, out ? a.ids + t * a.k : nullptr,
                            out ? a.weights + t * a.k : nullptr, a.status);
            __syncwarp();
            if (out) {
                if (a.ids_out && lane < a.k)
                    a.ids_out[t * a.k + lane] = rs.ids[t * a.k + lane];
                if (a.w_out && lane < a.k)
                    a.w_out[t * a.k + lane] = rs.weights[t * a.k + lane];
            }
            if (lane == 0)
                rs.shared_w[t] =
                    a.shared_gate ? 1.0f / (1.0f + expf(-__ldcg(a.logits + (int64_t)t * a.Epad + a.E)))
                                  : 1.0f;
        }
        cta_barrier();
        if (ok && warp == 0)
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
    const int fmax = a.f > a.fs ? a.f : a.fs;

    // ------------------------------------------------------------ phases G, D
    // Phase D runs in every warp (it holds CTA barriers); a warp that failed
    // earlier passes it with no work.
    uint32_t ring_seq = 0;  // ring stages issued (and consumed) by earlier phases
    if (ok)
        ok = run_phase<BITS, XBF16, 0>(a, ring, bars, ring_seq, P_r, P_t, fmax, w, Wall, true,
                                       &s_ok, rv);
    ok = run_phase<BITS, XBF16, 1>(a, ring, bars, ring_seq, P_r, P_t, fmax, w, Wall, ok, &s_ok,
                                   rv);

    // ------------------------------------------------------------ exit: the
    // last warp out resets the flags (counters of strips reset themselves)
    fence_acq_rel();
    __syncwarp();
    unsigned old = 0;
    if (lane == 0)
        old = atom_add_acqrel(a.exit_ctr, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == static_cast<unsigned>(Wall - 1)) {
        for (int p = lane; p < a.max_pairs; p += 32)
            a.pair_done[p] = 0u;
        if (lane == 0) {
            *a.route_ctr = 0u;
            fence_acq_rel();
            *a.exit_ctr = 0u;
        }
    }
}

template <int BITS, bool XBF16>
cudaError_t launch_t(const LayerArgs &a, cudaStream_t stream)
{
    auto kern = moe_layer_kernel<BITS, XBF16>;
    const int smem = smem_bytes(BITS);
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
    if (per_sm > kMaxLayerCtasPerSm)
        per_sm = kMaxLayerCtasPerSm;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(device_sm_count() * per_sm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
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

int layer_grid_warps_max() { return device_sm_count() * kMaxLayerCtasPerSm * kWarps; }

cudaError_t launch_layer(const LayerArgs &a, cudaStream_t stream)
{
    if (a.bits == 4)
        return a.x_bf16 ? launch_t<4, true>(a, stream) : launch_t<4, false>(a, stream);
    return a.x_bf16 ? launch_t<2, true>(a, stream) : launch_t<2, false>(a, stream);
}

}  // namespace smoe
