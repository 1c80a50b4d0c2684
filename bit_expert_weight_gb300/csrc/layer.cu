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
// Cross-CTA hand-offs are tagged words: every value one CTA passes to
// another (a logit, an h value, a partial sum, a down output) is stored as
// one 64-bit word {payload, tag} with a relaxed store, and the reader polls
// its own words with relaxed loads until they carry this launch's tag.  A
// reader that sees the tag sees the payload stored with it, so no fence,
// counter or atomic sits between the producer and the consumer.  The tag is
// the workspace's launch sequence number plus one; CTA 0 stores it back for
// the next launch once every CTA has read it.
//
// Phases (the launch is cooperative, so every CTA is resident):
//  R  (T <= 8 only) CTA c computes router rows c, c + grid, ... with all its
//     threads (the rows' weights are loaded before the previous kernel has
//     finished) and stores the tagged logits.  Every CTA then polls all the
//     logits into shared memory, ranks every (token, expert) against the
//     keys in (key desc, index asc) order (a quad of lanes per expert over
//     the streaming warps), turns the ranks below k into weights and builds
//     the pair table -- the same deterministic code on the same logits gives
//     the same table in every CTA.  For T > 8 a separate router kernel has built the
//     tables in global memory before the launch.
//  G  gate/up: the tiles of all pairs (pair = one expert x <= 8 tokens) form
//     one stream of 16-row strips, cut into chunks of <= 32 groups; the
//     chunks are split evenly over the CTAs (stream-K), streamed through a
//     ring of shared-memory stages filled by TMA bulk copies, decoded in
//     registers and multiplied with mma.sync by 16 warps.  Two epilogue
//     warps sum the warps' partials, finalise h = SiLU(g) * u (bf16 hi + lo)
//     and store it tagged; a strip split between CTAs is finished by its
//     last contributor, which polls the others' tagged partial sums.
//  D  down: steps of up to 4 whole output strips of one pair (one TMA copy
//     each), so no unit is split; the copies are issued as soon as ring
//     slots free up, while gate/up is still finishing.  Each warp polls the
//     h values its two groups need (tagged) when it reaches a new pair.
//  C  combine (T <= 8): every thread of the grid takes outputs (t, row) and
//     sums sum_j w_j o_j (+ shared) in rank order from the tagged down
//     outputs.  For T > 8 a separate combine kernel reads plain outputs.
// Deterministic throughout: no float atomics, fixed summation orders.
#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

// 16 streaming warps (decode, mma), 2 epilogue warps (unit sums, SiLU,
// stores, split-strip joins) and one producer warp (the TMA ring): global-
// memory round trips are slow while an SM streams, so the streaming warps
// make none except their own B operand loads.
constexpr int kStreamWarps = 16;
constexpr int kEpiWarps = 2;
constexpr int kProducerWarp = kStreamWarps + kEpiWarps;
constexpr int kWarps = kStreamWarps + kEpiWarps + 1;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxDownStrips = 4;  // output strips per down step

// ------------------------------------------------------------ tagged words

typedef unsigned long long u64;

__device__ __forceinline__ u64 tag_word(uint32_t payload, uint32_t tag)
{
    return (static_cast<u64>(tag) << 32) | payload;
}
__device__ __forceinline__ uint32_t word_tag(u64 w) { return static_cast<uint32_t>(w >> 32); }
__device__ __forceinline__ uint32_t word_payload(u64 w) { return static_cast<uint32_t>(w); }

__device__ __forceinline__ void st_word(u64 *p, u64 v)
{
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_word2(u64 *p, u64 a, u64 b)
{
    asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ u64 ld_word(const u64 *p)
{
    u64 v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// Two words of one 16-byte aligned pair; each word is loaded atomically.
__device__ __forceinline__ void ld_word2(const u64 *p, u64 &a, u64 &b)
{
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u32(unsigned *p, unsigned v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Poll one word until it carries `want` (bounded by `limit` SM cycles);
// false if the bound ran out.
__device__ __forceinline__ bool poll_word(const u64 *p, uint32_t want, long long limit, u64 &v)
{
    v = ld_word(p);
    if (word_tag(v) == want)
        return true;
    const long long t0 = clock64();
    unsigned ns = 32;
    for (;;) {
        __nanosleep(ns);
        if (ns < 256)
            ns *= 2;
        v = ld_word(p);
        if (word_tag(v) == want)
            return true;
        if (clock64() - t0 > limit)
            return false;
    }
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

// 1 / (1 + e^-x) with the hardware exp and divide; the exponent is capped
// so that the divisor stays finite (the result is then 0 to fp32).
__device__ __forceinline__ float sigmoid_fast(float x)
{
    return __fdividef(1.0f, 1.0f + __expf(fminf(-x, 80.0f)));
}

// Router rows of one CTA (phase R): rows c, c + grid (E routed rows, then
// the shared gate row), at most two.  Thread i holds columns 8i .. 8i+7 of
// each row.
struct RouterPre {
    uint4 w0, w1;
    int nrows;
};

__device__ __forceinline__ const uint16_t *router_row(const LayerArgs &a, int r)
{
    return r < a.E ? a.router_w + (int64_t)r * a.d : a.shared_gate;
}

__device__ __forceinline__ int router_rows_of_cta(const LayerArgs &a)
{
    const int rows = a.E + (a.shared_gate ? 1 : 0);
    const int C = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return c < rows ? (c + C < rows ? 2 : 1) : 0;
}

// Before the previous kernel on the stream has finished: pull the CTA's
// router rows into L2 (one prefetch per 128-byte line).  Only a prefetch:
// L2 is coherent, so a row that kernel still writes is read correctly after
// the wait, where the rows are loaded.
__device__ __forceinline__ void router_prefetch_l2(const LayerArgs &a)
{
    const int n = router_rows_of_cta(a), i = threadIdx.x;
    const int C = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    if (i < a.d / 64) {
        for (int r = 0; r < n; ++r)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(router_row(a, c + r * C) + 64 * i));
    }
}

__device__ __forceinline__ RouterPre router_load(const LayerArgs &a)
{
    RouterPre pre;
    pre.nrows = router_rows_of_cta(a);
    const int C = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const int i = threadIdx.x;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    pre.w0 = pre.w1 = z;
    if (i < a.d / 8) {
        if (pre.nrows > 0)
            pre.w0 = __ldg(reinterpret_cast<const uint4 *>(router_row(a, c) + 8 * i));
        if (pre.nrows > 1)
            pre.w1 = __ldg(reinterpret_cast<const uint4 *>(router_row(a, c + C) + 8 * i));
    }
    return pre;
}

__device__ __forceinline__ float dot8_bf16(uint4 w, const float (&x)[8])
{
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc = fmaf(bf16lo_to_f32(ww[q]), x[2 * q], acc);
        acc = fmaf(bf16hi_to_f32(ww[q]), x[2 * q + 1], acc);
    }
    return acc;
}

// The CTA's router rows for all tokens (at most TMAX: the token loops are
// unrolled to the instance's bound, which keeps this once-per-launch code
// small): per-thread 8-column dot products,
// a shuffle tree per warp, then the warps' sums in warp order; each logit is
// stored tagged into every CTA's own copy of the logits (so that each CTA
// polls lines no other CTA polls).  red: shared scratch of kWarps x 16
// floats plus 16 logits.  Every thread of the CTA calls it.
template <bool XBF16, int TMAX>
__device__ __forceinline__ void router_rows(const LayerArgs &a, const RouterPre &pre, float *red,
                                            uint32_t tag)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, i = threadIdx.x;
    const int T = static_cast<int>(a.T), d = a.d;
    const int nw = (d / 8 + 31) / 32;  // warps holding columns
    if (pre.nrows > 0 && warp < nw) {
        float acc[2][TMAX];
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
            acc[0][t] = acc[1][t] = 0.f;
            if (t < T && i < d / 8) {
                float xf[8];
                if (XBF16) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(
                        reinterpret_cast<const uint16_t *>(a.x) + (int64_t)t * d + 8 * i));
                    const uint32_t xx[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        xf[2 * q] = bf16lo_to_f32(xx[q]);
                        xf[2 * q + 1] = bf16hi_to_f32(xx[q]);
                    }
                } else {
                    const float4 *xr = reinterpret_cast<const float4 *>(
                        reinterpret_cast<const float *>(a.x) + (int64_t)t * d + 8 * i);
                    const float4 v0 = __ldg(xr), v1 = __ldg(xr + 1);
                    xf[0] = v0.x, xf[1] = v0.y, xf[2] = v0.z, xf[3] = v0.w;
                    xf[4] = v1.x, xf[5] = v1.y, xf[6] = v1.z, xf[7] = v1.w;
                }
                acc[0][t] = dot8_bf16(pre.w0, xf);
                acc[1][t] = pre.nrows > 1 ? dot8_bf16(pre.w1, xf) : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                if (r < pre.nrows && t < T) {  // uniform over the warp
                    float v = acc[r][t];
                    for (int o = 16; o; o >>= 1)
                        v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0)
                        red[warp * 16 + r * kPairCols + t] = v;
                }
            }
    }
    cta_barrier();
    float *lg = red + kWarps * 16;
    if (i < pre.nrows * T) {
        const int r = i / T, t = i - r * T;
        float v = 0.f;
        for (int w = 0; w < nw; ++w)
            v += red[w * 16 + r * kPairCols + t];
        lg[i] = v;
    }
    cta_barrier();
    const int C = static_cast<int>(gridDim.x), n = pre.nrows * T;
    for (int j = i; j < n * C; j += kThreads) {
        const int c = j / n, q = j - c * n, r = q / T, t = q - r * T;
        const int row = static_cast<int>(blockIdx.x) + r * C;
        st_word(a.logit_t + ((int64_t)c * T + t) * a.Epad + row, tag_word(__float_as_uint(lg[q]), tag));
    }
}

// Routing tables of a CTA.  On the fused path (T <= 8) every CTA builds its
// own copy in shared memory from the tagged logits (the same deterministic
// code on the same logits gives the same tables everywhere); otherwise they
// point to the tables the router kernel left in global memory.
constexpr int kFusedPairs = kPairCols * SMOE_MAX_TOPK_DEV + 1;
// route_map, weights and ids are [T][k+1], [T][k], [T][k] with the runtime k
// as the row stride, exactly like the global tables.
struct __align__(16) RouteSmem {
    float lg[kPairCols * kMaxExperts];   // [T][E4] logits, row stride E4 = E rounded up to 4
    float key[kPairCols * kMaxExperts];  // [T][E4] selection keys
    float red[kWarps * 16 + 16];         // router row partial sums, then the CTA's logits
    int32_t pairs[kFusedPairs][kPairInts];
    int32_t route_map[kPairCols * (SMOE_MAX_TOPK_DEV + 1)];
    float smax[kPairCols], ssum[kPairCols];  // softmax statistics per token
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

// Rank of expert e (key ke) among the experts lo .. hi - 1 (lo a multiple of
// 4; key rows 16-byte aligned): how many come before it in the order (key
// descending, index ascending) -- ties go to the lower index.
__device__ __forceinline__ int rank_range(const float *key, int e, float ke, int lo, int hi)
{
    int r = 0, j = lo;
    const float4 *k4 = reinterpret_cast<const float4 *>(key);
#pragma unroll 4
    for (; j + 4 <= hi; j += 4) {
        const float4 v = k4[j >> 2];
        r += (v.x > ke || (v.x == ke && j < e)) ? 1 : 0;
        r += (v.y > ke || (v.y == ke && j + 1 < e)) ? 1 : 0;
        r += (v.z > ke || (v.z == ke && j + 2 < e)) ? 1 : 0;
        r += (v.w > ke || (v.w == ke && j + 3 < e)) ? 1 : 0;
    }
    for (; j < hi; ++j) {
        const float v = key[j];
        r += (v > ke || (v == ke && j < e)) ? 1 : 0;
    }
    return r;
}

// Softmax statistics of one token's E logits, in one warp: the maximum m and
// the sum z of exp(l - m), lane-strided then a shuffle tree (a fixed order).
// exp and divide are the hardware approximations (a few ulp), well inside
// the weights' tolerance.
__device__ __forceinline__ void softmax_stats(const float *lg, int E, float *m_out, float *z_out)
{
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
    for (int i = lane; i < E; i += 32)
        m = fmaxf(m, lg[i]);
    for (int o = 16; o; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
    for (int i = lane; i < E; i += 32)
        z += __expf(lg[i] - m);
    for (int o = 16; o; o >>= 1)
        z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0) {
        *m_out = m;
        *z_out = z;  // in [1, E]
    }
}

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

// Gate/up: a chunk is a run of up to kChunkGroups consecutive groups of one
// strip, two per streaming warp (groups w and w + 16 of the chunk); one
// stage of the CTA's ring holds one chunk (gate and up tile per group).
// Down: a step is up to kMaxDownStrips whole output strips of one pair (all
// f/64 groups each, f <= 2048), in one stage.
constexpr int kChunkGroups = 2 * kStreamWarps;
constexpr int kDownGroupsMax = kChunkGroups;  // ffn_dim <= 2048

__host__ __device__ constexpr int stage_bytes(int bits) { return kChunkGroups * 2 * tile_bytes(bits); }
// Kernel instances: BITS = 4 or 2 for a bank of one depth, BITS = 0 for a
// bank of mixed depths, whose ring is sized for Q4 stages.
__host__ __device__ constexpr int ring_bits(int bits) { return bits == 0 ? 4 : bits; }
// About 100 KB per SM: the full HBM rate needs ~64 KB in flight, and the
// streaming warps consume a Q4 stage in ~1.4 us, so stages land before they
// are needed; 4 Q4 stages (with 3 reduction slots) measured slower, and
// copying from L2 instead of HBM changed the stage rate little.
__host__ __device__ constexpr int num_stages(int bits) { return bits == 4 ? 3 : 5; }
// kRedSlots slots of per-warp unit sums (two float4 per lane: gate and up,
// or two down strips)
constexpr int kRedSlots = 4;
__host__ __device__ constexpr int red_bytes() { return kRedSlots * kStreamWarps * 2 * 32 * 16; }
__host__ __device__ constexpr int smem_bytes(int bits)
{
    return num_stages(bits) * stage_bytes(bits) + red_bytes() + (2 * num_stages(bits) + 2 * kRedSlots) * 8;
}

// Step geometry of one phase.  Gate/up: units are (pair, strip) in pair
// order; a unit's K groups are cut into ch chunks of gc groups (the last may
// be shorter); the steps (chunks) of all units are split evenly over the
// CTAs, so a unit may be shared by neighbouring CTAs.  Down: a step is ms
// consecutive strips of one pair (the last step of a pair may hold fewer);
// nstr counts steps per pair and ch = 1, so no unit is ever split.
// Index [0]: routed pairs, [1]: the shared expert's pair.
// (Scalar fields with select accessors: a runtime-indexed array would live
// in local memory.)
struct Geo {
    int P_r, P_t;
    int nstr0, gk0, ch0, gc0, spp0, ms0;  // routed: strips (steps), groups per strip, chunks,
                                          // groups per chunk, steps per pair, strips per step
    int nstr1, gk1, ch1, gc1, spp1, ms1;  // shared
    int rows;                             // down: output strips (d / 16)
    int SR, S;                            // steps of the routed pairs, of all pairs
    Split sp;                             // steps over CTAs
    int a0, a1;                           // this CTA's steps
    int ts;                               // the CTA runs [ts, a1) first, then [a0, ts)
};

struct UnitGeo {
    int nstr, gk, ch, gc, ms;
};

__device__ __forceinline__ UnitGeo unit_geo(const Geo &g, int p)
{
    const bool r = p < g.P_r;
    UnitGeo u;
    u.nstr = r ? g.nstr0 : g.nstr1;
    u.gk = r ? g.gk0 : g.gk1;
    u.ch = r ? g.ch0 : g.ch1;
    u.gc = r ? g.gc0 : g.gc1;
    u.ms = r ? g.ms0 : g.ms1;
    return u;
}

// Down strips per step: as many whole strips of gk tiles as a stage holds
// (64 tiles at the ring's depth), at most kMaxDownStrips.
__device__ __forceinline__ int down_strips_per_step(int gk)
{
    if (gk <= 0)
        return 1;
    const int m = (kChunkGroups * 2) / gk;
    return m < 1 ? 1 : (m > kMaxDownStrips ? kMaxDownStrips : m);
}

__device__ __forceinline__ Geo make_geo(const LayerArgs &a, int phase, int P_r, int P_t)
{
    Geo g;
    g.P_r = P_r;
    g.P_t = P_t;
    g.rows = a.d / kTileRows;
    if (phase == 0) {
        g.gk0 = a.d / kGroup;
        g.nstr0 = a.f / kTileRows;
        g.ch0 = (g.gk0 + kChunkGroups - 1) / kChunkGroups;
        g.gc0 = (g.gk0 + g.ch0 - 1) / g.ch0;
        g.ms0 = 1;
        g.gk1 = a.d / kGroup;
        g.nstr1 = a.fs / kTileRows;
        g.ch1 = g.ch0;
        g.gc1 = g.gc0;
        g.ms1 = 1;
    } else {
        g.gk0 = a.f / kGroup;
        g.ms0 = down_strips_per_step(g.gk0);
        g.nstr0 = (g.rows + g.ms0 - 1) / g.ms0;
        g.ch0 = 1;
        g.gc0 = g.gk0;
        g.gk1 = a.fs / kGroup;
        g.ms1 = down_strips_per_step(g.gk1);
        g.nstr1 = g.gk1 > 0 ? (g.rows + g.ms1 - 1) / g.ms1 : 0;
        g.ch1 = 1;
        g.gc1 = g.gk1;
    }
    g.spp0 = g.nstr0 * g.ch0;
    g.spp1 = g.nstr1 * g.ch1;
    g.SR = P_r * g.spp0;
    g.S = g.SR + (P_t - P_r) * g.spp1;
    const int C = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    g.sp = make_split(g.S, C);
    g.a0 = split_start(g.sp, c);
    g.a1 = split_start(g.sp, c + 1);
    // Gate/up: whole units per CTA when every unit has the same chunk count
    // and the extra unit a CTA may get costs under ~48 KB (about a
    // microsecond of one SM's share of HBM): no unit is then shared.
    if (phase == 0 && g.ch0 > 1 && (P_t == P_r || g.ch1 == g.ch0)) {
        const int U = g.S / g.ch0;
        const int unit_bytes = g.gk0 * 2 * (a.bits * 128 + 32);
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
    int p, s, c;  // pair, strip (gate/up) or step within the pair (down), chunk
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

// Order of a CTA's gate/up steps: a unit cut by the end of the range is run
// first, then the range from its start (whose first unit may be cut by the
// start).  The CTA then hands its part of the shared tail unit to the next
// CTA early, and finishes its head unit (whose first part the previous CTA
// ran first) last among its contributors.
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

// Output strips of down step (pair, step s): [first, first + count).
__device__ __forceinline__ int down_first(const UnitGeo &u, const Pos &q) { return q.s * u.ms; }
__device__ __forceinline__ int down_count(const Geo &g, const UnitGeo &u, const Pos &q)
{
    const int s0 = q.s * u.ms;
    return min(u.ms, g.rows - s0);
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
    const uint8_t *base;
    if (e < 0)
        base = a.tiles_shared + (pr.phase ? a.down_off_shared : 0);
    else if (BITS != 0)
        base = a.tiles_routed + (int64_t)e * a.expert_bytes_routed + (pr.phase ? a.down_off_routed : 0);
    else  // the expert's own place and down offset in a bank of mixed depths
        base = a.tiles_routed + mixed_expert_offset(a, e) +
               (pr.phase ? 2ll * a.d * a.f / 1024 * TB : 0);
    const uint8_t *src;
    unsigned bytes;
    if (pr.phase == 0) {
        const int g0 = pr.q.c * u.gc;
        const int ng = min(u.gk - g0, u.gc);
        src = base + ((int64_t)pr.q.s * u.gk + g0) * 2 * TB;
        bytes = static_cast<unsigned>(ng * 2 * TB);
    } else {
        src = base + (int64_t)down_first(u, pr.q) * u.gk * TB;
        bytes = static_cast<unsigned>(down_count(g, u, pr.q) * u.gk * TB);
    }
    mbar_arrive_expect_tx(&full[slot], bytes);
    bulk_g2s(ring + slot * SB, src, bytes, &full[slot]);
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

// The lane's view of a pair record: column count, the pair column whose
// activations this lane's row of the B fragment holds, and its token.  The
// B fragment's column n is lane >> 2; with packed columns (pairs of at most
// 4 tokens) columns 2c and 2c + 1 carry the bf16 hi and lo parts of pair
// column c, so that one mma takes both parts and the two output columns are
// added afterwards.
struct PairInfo {
    int ncols, col, tok;
};

template <bool PACK>
__device__ __forceinline__ PairInfo read_pair(const RouteView &rv, int p)
{
    const int lane = threadIdx.x & 31;
    const int32_t *pr = rv.pairs + p * kPairInts;
    PairInfo pi;
    pi.ncols = pr[1];
    pi.col = PACK ? lane >> 3 : lane >> 2;
    pi.tok = pi.col < pi.ncols ? pr[2 + pi.col] : 0;
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

// Class sums of a group for the column biases: s0 over the lane's columns
// 16 tig + i with i % 4 in {0, 1}, s1 over i % 4 in {2, 3} (the halves the
// A fragment's registers 0-1 and 2-3 multiply).  Summed over the group's four
// lanes of token row gq, then fetched for the two output columns this lane's
// accumulators hold (2 tig and 2 tig + 1: lanes 8 tig and 8 tig + 4).
template <int BITS>
__device__ __forceinline__ void bias_from_sums(BFrag &f, float s0, float s1)
{
    const int tig = threadIdx.x & 3;
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    float2 x0, x1;
    x0.x = __shfl_sync(0xffffffffu, s0, 8 * tig);
    x0.y = __shfl_sync(0xffffffffu, s1, 8 * tig);
    x1.x = __shfl_sync(0xffffffffu, s0, 8 * tig + 4);
    x1.y = __shfl_sync(0xffffffffu, s1, 8 * tig + 4);
    finish_bias<BITS>(f, x0, x1);
}

// Gate/up B operand of group gi: the lane's 16 activations of its token
// (pair column pi.col) at columns 64 gi + 16 tig .. +15 (bf16 x: 2 vectors,
// fp32 x: 4, split into bf16 hi + lo -- both parts in b*/b*l, or with PACK
// the part of B column lane >> 2: hi for even, lo for odd), and the column
// biases.  on = the group exists (warp-uniform); an absent group or column
// gives zeros.  Every lane of the warp calls it.
template <int BITS, bool XBF16, bool PACK>
__device__ __forceinline__ void load_b_x(const LayerArgs &a, const PairInfo &pi, int gi, bool on,
                                         BFrag &f)
{
    const int lane = threadIdx.x & 31, tig = lane & 3;
    const bool valid = on && pi.col < pi.ncols;
    const bool lo_part = ((lane >> 2) & 1) != 0;
    float s0 = 0.f, s1 = 0.f;
    if (XBF16) {
        const uint4 *row = reinterpret_cast<const uint4 *>(
            reinterpret_cast<const uint16_t *>(a.x) + (int64_t)pi.tok * a.d + gi * kGroup + 16 * tig);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint4 v0 = valid ? __ldg(row) : z, v1 = valid ? __ldg(row + 1) : z;
        const uint32_t xv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f.b0[j] = xv[2 * j];
            f.b1[j] = xv[2 * j + 1];
            f.b0l[j] = f.b1l[j] = 0u;
            s0 += bf16lo_to_f32(xv[2 * j]) + bf16hi_to_f32(xv[2 * j]);
            s1 += bf16lo_to_f32(xv[2 * j + 1]) + bf16hi_to_f32(xv[2 * j + 1]);
        }
    } else {
        const float4 *row = reinterpret_cast<const float4 *>(
            reinterpret_cast<const float *>(a.x) + (int64_t)pi.tok * a.d + gi * kGroup + 16 * tig);
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 v = valid ? __ldg(row + j) : z;
            split_bf16x2(v.x, v.y, f.b0[j], f.b0l[j]);
            split_bf16x2(v.z, v.w, f.b1[j], f.b1l[j]);
            if (PACK) {
                if (lo_part) {
                    f.b0[j] = f.b0l[j];
                    f.b1[j] = f.b1l[j];
                }
                f.b0l[j] = f.b1l[j] = 0u;
                s0 += bf16lo_to_f32(f.b0[j]) + bf16hi_to_f32(f.b0[j]);
                s1 += bf16lo_to_f32(f.b1[j]) + bf16hi_to_f32(f.b1[j]);
            } else {
                s0 += v.x + v.y;
                s1 += v.z + v.w;
            }
        }
    }
    bias_from_sums<BITS>(f, s0, s1);
}

// Down B operand of group gi of pair p: the lane's 16 h values of its pair
// column (rows 64 gi + 16 tig .. +15), polled until every word carries the
// launch's tag, as the bf16 hi and lo fragments (or with PACK the part of B
// column lane >> 2), and the column biases.  False if the bounded poll ran
// out.  Every lane calls it.
template <int BITS, bool PACK>
__device__ __forceinline__ bool load_b_h(const LayerArgs &a, const PairInfo &pi, int p, int gi, bool on,
                                         int fmax, uint32_t tag, BFrag &f)
{
    const int lane = threadIdx.x & 31, tig = lane & 3;
    const bool valid = on && pi.col < pi.ncols;
    const bool lo_part = ((lane >> 2) & 1) != 0;
    const u64 *src = a.h_t + ((int64_t)p * kPairCols + pi.col) * fmax + gi * kGroup + 16 * tig;
    u64 w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        w[i] = 0ull;
    bool ok = true;
    if (__any_sync(0xffffffffu, valid)) {
        const long long t0 = clock64();
        unsigned ns = 64;
        for (;;) {
            bool mine = true;
            if (valid) {
#pragma unroll
                for (int i = 0; i < 16; i += 2)
                    ld_word2(src + i, w[i], w[i + 1]);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    mine = mine && word_tag(w[i]) == tag;
            }
            if (__all_sync(0xffffffffu, mine))
                break;
            if (clock64() - t0 > a.wait_cycles) {
                ok = false;
                break;
            }
            __nanosleep(ns);
            if (ns < 512)
                ns *= 2;
        }
    }
    if (!valid || !ok) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = 0ull;
    }
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t w0 = word_payload(w[4 * j]), w1 = word_payload(w[4 * j + 1]);
        const uint32_t w2 = word_payload(w[4 * j + 2]), w3 = word_payload(w[4 * j + 3]);
        f.b0[j] = __byte_perm(w0, w1, 0x5410);
        f.b0l[j] = __byte_perm(w0, w1, 0x7632);
        f.b1[j] = __byte_perm(w2, w3, 0x5410);
        f.b1l[j] = __byte_perm(w2, w3, 0x7632);
        if (PACK) {
            if (lo_part) {
                f.b0[j] = f.b0l[j];
                f.b1[j] = f.b1l[j];
            }
            f.b0l[j] = f.b1l[j] = 0u;
            s0 += bf16lo_to_f32(f.b0[j]) + bf16hi_to_f32(f.b0[j]);
            s1 += bf16lo_to_f32(f.b1[j]) + bf16hi_to_f32(f.b1[j]);
        } else {
            s0 += (bf16lo_to_f32(w0) + bf16hi_to_f32(w0)) + (bf16lo_to_f32(w1) + bf16hi_to_f32(w1));
            s1 += (bf16lo_to_f32(w2) + bf16hi_to_f32(w2)) + (bf16lo_to_f32(w3) + bf16hi_to_f32(w3));
        }
    }
    bias_from_sums<BITS>(f, s0, s1);
    return ok;
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

// What the epilogue writes, passed by value (registers) to its cold helpers.
struct EpiOut {
    u64 *h_t, *part_t, *o_t;
    float *o;
    int d, fmax, fused;
    uint32_t tag;
    long long wait_cycles;
    int *status;
};

// Accumulator element e of the lane (rows gq, gq + 8; B columns 2 tig,
// 2 tig + 1) as a value of pair column col: unpacked, element e itself;
// packed, the hi + lo columns of pair column tig added (elements 0 + 1 for
// row gq, 2 + 3 for row gq + 8; valid for e even).
template <bool PACK>
__device__ __forceinline__ float acc_col(const float (&v)[4], int e, int &col)
{
    const int tig = threadIdx.x & 3;
    if (PACK) {
        col = (e & 1) ? kPairCols : tig;  // odd elements are the lo parts: no output of their own
        return v[e & 2] + v[(e & 2) + 1];
    }
    col = 2 * tig + (e & 1);
    return v[e];
}

// Finalise gate/up strip s of pair p from its full-K sums (one warp, cold
// path): h = SiLU(g) * u as bf16 hi + lo, stored tagged.
template <int BITS, bool PACK>
__device__ __forceinline__ void finalize_gateup(const EpiOut a, int ncols, int p, int s, float4 ag, float4 au)
{
    constexpr float L = BITS == 4 ? 7.5f : 1.5f;
    const int lane = threadIdx.x & 31, gq = lane >> 2;
    const float invL = 1.0f / L;
    const float gv[4] = {ag.x, ag.y, ag.z, ag.w}, uv[4] = {au.x, au.y, au.z, au.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int col;
        const float gsum = acc_col<PACK>(gv, e, col), usum = acc_col<PACK>(uv, e, col);
        const int row = 16 * s + gq + 8 * (e >> 1);
        if (col < ncols) {
            const float g = gsum * invL, u = usum * invL;
            const float hv = __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;  // SiLU(g) * u
            const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
            const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
            const uint32_t pay = static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(&hi)) |
                                 (static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(&lo)) << 16);
            st_word(a.h_t + ((int64_t)p * kPairCols + col) * a.fmax + row, tag_word(pay, a.tag));
        }
    }
}

// Finalise down strip s of pair p: o rows, tagged for the in-kernel
// combine or plain for the combine kernel.
template <int BITS, bool PACK>
__device__ __forceinline__ void finalize_down(const EpiOut &a, int ncols, int p, int s, float4 ag)
{
    constexpr float L = BITS == 4 ? 7.5f : 1.5f;
    const int lane = threadIdx.x & 31, gq = lane >> 2;
    const float invL = 1.0f / L;
    const float gv[4] = {ag.x, ag.y, ag.z, ag.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int col;
        const float sum = acc_col<PACK>(gv, e, col);
        const int row = 16 * s + gq + 8 * (e >> 1);
        if (col < ncols) {
            const int64_t off = ((int64_t)p * kPairCols + col) * a.d + row;
            const float ov = sum * invL;
            if (a.fused)
                st_word(a.o_t + off, tag_word(__float_as_uint(ov), a.tag));
            else
                a.o[off] = ov;
        }
    }
}

// Gate/up strip (p, s) shared with other CTAs (cold path).  Slot 0 of a CTA
// holds the unit straddling the start of its range, slot 1 the one
// straddling its end.  A contributor that does not hold the unit's last
// step stores its sums tagged and is done; the one that does (the last
// contributor) polls the others' sums, adds them all in CTA order and
// finalises.  False if a bounded poll ran out.
template <int BITS, bool PACK>
__device__ __forceinline__ bool fixup_gateup(const EpiOut a, int ncols, const Geo &g, int p, int s, int ustart,
                                          int uend, float4 tg, float4 tu)
{
    const int lane = threadIdx.x & 31;
    const int c = static_cast<int>(blockIdx.x);
    const int cf = split_owner(g.sp, ustart), cl = split_owner(g.sp, uend - 1);
    if (c != cl) {
        const int my = ustart < g.a0 ? 0 : 1;
        u64 *mine = a.part_t + (((int64_t)c * 2 + my) * 32 + lane) * 8;
        st_word2(mine, tag_word(__float_as_uint(tg.x), a.tag), tag_word(__float_as_uint(tg.y), a.tag));
        st_word2(mine + 2, tag_word(__float_as_uint(tg.z), a.tag), tag_word(__float_as_uint(tg.w), a.tag));
        st_word2(mine + 4, tag_word(__float_as_uint(tu.x), a.tag), tag_word(__float_as_uint(tu.y), a.tag));
        st_word2(mine + 6, tag_word(__float_as_uint(tu.z), a.tag), tag_word(__float_as_uint(tu.w), a.tag));
        return true;
    }
    float4 sg = make_float4(0.f, 0.f, 0.f, 0.f), su = sg;
    bool ok = true;
    for (int c2 = cf; c2 <= cl; ++c2) {
        float v[8];
        if (c2 == c) {
            v[0] = tg.x, v[1] = tg.y, v[2] = tg.z, v[3] = tg.w;
            v[4] = tu.x, v[5] = tu.y, v[6] = tu.z, v[7] = tu.w;
        } else {
            const int sl = split_start(g.sp, c2) > ustart ? 0 : 1;
            const u64 *src = a.part_t + (((int64_t)c2 * 2 + sl) * 32 + lane) * 8;
            u64 w[8];
            const long long t0 = clock64();
            unsigned ns = 64;
            for (;;) {
                bool mine = true;
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    ld_word2(src + i, w[i], w[i + 1]);
                    mine = mine && word_tag(w[i]) == a.tag && word_tag(w[i + 1]) == a.tag;
                }
                if (__all_sync(0xffffffffu, mine))
                    break;
                if (clock64() - t0 > a.wait_cycles) {
                    ok = false;
                    break;
                }
                __nanosleep(ns);
                if (ns < 512)
                    ns *= 2;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = __uint_as_float(word_payload(w[i]));
        }
        sg.x += v[0], sg.y += v[1], sg.z += v[2], sg.w += v[3];
        su.x += v[4], su.y += v[5], su.z += v[6], su.w += v[7];
    }
    if (!ok)
        return false;
    finalize_gateup<BITS, PACK>(a, ncols, p, s, sg, su);
    return true;
}

// Shared state of the streaming phases, one per CTA.
struct Stream {
    uint8_t *ring;
    uint64_t *full, *empty;          // [NS]: 1 arrival + bytes / kStreamWarps arrivals
    uint64_t *red_full, *red_empty;  // [kRedSlots]: kStreamWarps arrivals / 1 arrival
    float4 *red;                     // [kRedSlots][kStreamWarps][2][32]
    volatile int *fail;              // a bounded wait ran out somewhere in the CTA
    Producer *pr;                    // shared; used by lane 0 of the producer warp only
    const Geo *geo;                  // shared, [2]
    uint32_t seq;                    // stages consumed by this (streaming) warp
    int uc;                          // reduction items so far
    uint32_t tag;                    // this launch's tag
};

// Step i (position q) ends its unit in the CTA's range [.., a1) run from
// ts: the unit's last chunk, or the last step before a cut.  The range
// bounds come in registers, not from the shared geometry.
__device__ __forceinline__ bool unit_ends(int a1, int ts, const UnitGeo &u, const Pos &q, int i)
{
    return q.c == u.ch - 1 || i == a1 - 1 || (ts < a1 && i == ts - 1);
}

// Wait for ring stage `st.seq` (bounded); false if the CTA has failed.  The
// stage is tested first: the failure flag (a shared-memory read) is only
// consulted when the stage is not there yet.
template <int NS>
__device__ __forceinline__ bool wait_stage(const LayerArgs &a, Stream &st, int slot)
{
    const int lane = threadIdx.x & 31;
    if (mbar_try_wait(&st.full[slot], (st.seq / NS) & 1u))
        return true;
    if (*st.fail)
        return false;
    if (!mbar_wait_bounded(&st.full[slot], (st.seq / NS) & 1u)) {
        if (lane == 0) {
            set_status(a.status, kStatusTimeout);
            *st.fail = 1;
        }
        return false;
    }
    return true;
}

// Hand two float4 per lane to the epilogue warps through reduction slot
// st.uc (waiting for the slot to be free; after a failure it is not waited
// for, and the arrival completes a phase nobody takes).
__device__ __forceinline__ void put_red(const LayerArgs &a, Stream &st, float4 v0, float4 v1)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rs = st.uc % kRedSlots;
    const unsigned rph = static_cast<unsigned>(st.uc / kRedSlots);
    if (st.uc >= kRedSlots && !mbar_try_wait(&st.red_empty[rs], (rph - 1u) & 1u) && !*st.fail &&
        !mbar_wait_bounded(&st.red_empty[rs], (rph - 1u) & 1u) && lane == 0) {
        set_status(a.status, kStatusTimeout);
        *st.fail = 1;
    }
    float4 *rw = st.red + ((rs * kStreamWarps + warp) * 2) * 32;
    rw[lane] = v0;
    rw[32 + lane] = v1;
    __syncwarp();
    if (lane == 0)
        mbar_arrive(&st.red_full[rs]);
    ++st.uc;
}

// The warp's tiles of one gate/up stage at depth B: groups w (fragments
// f0) and w + 16 (f1), each a gate and an up tile.
template <int B, bool SPLIT>
__device__ __forceinline__ void gateup_tiles(const uint8_t *stage, const BFrag &f0, const BFrag &f1, bool g0,
                                             bool g1, float (&accg)[4], float (&accu)[4], float (&accg2)[4],
                                             float (&accu2)[4])
{
    constexpr int TB = tile_bytes(B);
    const int warp = threadIdx.x >> 5;
    if (g0) {
        mac_tile<B, SPLIT>(stage + warp * 2 * TB, f0, accg, true);
        mac_tile<B, SPLIT>(stage + warp * 2 * TB + TB, f0, accu, true);
    }
    if (g1) {
        mac_tile<B, SPLIT>(stage + (warp + kStreamWarps) * 2 * TB, f1, accg2, true);
        mac_tile<B, SPLIT>(stage + (warp + kStreamWarps) * 2 * TB + TB, f1, accu2, true);
    }
}

// The warp's two tiles of down strip j of a stage at depth B (groups w and
// w + 16 of the strip's gk groups), added into acc.
template <int B, bool SPLIT>
__device__ __forceinline__ void down_tiles(const uint8_t *stage, int j, int gk, const BFrag (&bf)[2], bool g0,
                                           bool g1, float (&acc)[4])
{
    constexpr int TB = tile_bytes(B);
    const int t0 = j * gk + (threadIdx.x >> 5);
    if (g0)
        mac_tile<B, SPLIT>(stage + t0 * TB, bf[0], acc, true);
    if (g1)
        mac_tile<B, SPLIT>(stage + (t0 + kStreamWarps) * TB, bf[1], acc, true);
}

// The gate/up phase of a streaming warp.  The warp holds the B fragments
// of its groups of the current pair: groups c * gc + w and c * gc + w + 16
// of each chunk c (at most KG chunks).  At a unit's end it hands its sums to
// the epilogue warps.
template <int BITS, bool XBF16, int KG, bool PACK>
__device__ __forceinline__ void stream_gateup(const LayerArgs &a, const RouteView &rv, Stream &st)
{
    constexpr int NS = num_stages(ring_bits(BITS)), SB = stage_bytes(ring_bits(BITS));
    // fp32 tokens enter as bf16 hi + lo: two mmas per k-subtile, or with
    // packed columns (<= 4 tokens) one mma whose column pairs are added later
    constexpr bool PG = PACK && !XBF16;
    constexpr bool kSplit = !XBF16 && !PG;
    constexpr int NB = 2 * KG;  // B fragments held
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = st.geo[0];
    const int a0 = g.a0, a1 = g.a1, n = a1 - a0, ts = g.ts, nt = a1 - ts;
    if (n <= 0)
        return;
    Pos q = decode(g, nt > 0 ? ts : a0);
    UnitGeo u = unit_geo(g, q.p);
    int loaded = -1;
    int pb = ring_bits(BITS);  // depth of the loaded pair
    int ltok = -1, lncols = -1, lpb = -1;  // the token column and depth the fragments hold
    BFrag bf[NB];
    float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
    float accg2[4] = {0.f, 0.f, 0.f, 0.f}, accu2[4] = {0.f, 0.f, 0.f, 0.f};  // second group
#pragma unroll 1
    for (int kk = 0; kk < n; ++kk) {
        const int i = kk < nt ? ts + kk : a0 + (kk - nt);
        if (kk == nt && kk > 0)
            q = decode(g, a0);
        if (q.p != loaded) {
            u = unit_geo(g, q.p);
            const PairInfo pi = read_pair<PG>(rv, q.p);
            pb = pair_bits<BITS>(a, rv.pairs[q.p * kPairInts]);
            // every pair's gate/up has K = d, so the fragments depend only on
            // the tokens and the depth: reloaded only when those change
            const bool same = __all_sync(0xffffffffu, pi.tok == ltok && pi.ncols == lncols && pb == lpb);
            if (!same) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int c = b >> 1, lg = warp + (b & 1) * kStreamWarps;  // chunk, group in chunk
                    const int gi = c * u.gc + lg;
                    const bool on = c < u.ch && lg < u.gc && gi < u.gk;
                    if (BITS != 0 || pb == 4)
                        load_b_x<ring_bits(BITS), XBF16, PG>(a, pi, gi, on, bf[b]);
                    else
                        load_b_x<2, XBF16, PG>(a, pi, gi, on, bf[b]);
                }
                ltok = pi.tok;
                lncols = pi.ncols;
                lpb = pb;
            }
            loaded = q.p;
        }
        const int slot = static_cast<int>(st.seq % NS);
        const bool ok = wait_stage<NS>(a, st, slot);
        if (ok) {
            // the warp's two groups of the chunk; a group past the chunk's
            // end is skipped (the branch is uniform over the warp).  The
            // chunk's fragments are selected by value, so that the tile code
            // exists once (a smaller loop for the instruction cache)
            const uint8_t *stage = st.ring + slot * SB;
            const int ng = min(u.gc, u.gk - q.c * u.gc);  // groups in this chunk
            const bool g0 = warp < ng, g1 = warp + kStreamWarps < ng;
            BFrag f0 = bf[0], f1 = bf[1];
#pragma unroll
            for (int c = 1; c < KG; ++c) {
                if (c == q.c) {
                    f0 = bf[2 * c];
                    f1 = bf[2 * c + 1];
                }
            }
            if (BITS != 0 || pb == 4)
                gateup_tiles<ring_bits(BITS), kSplit>(stage, f0, f1, g0, g1, accg, accu, accg2, accu2);
            else
                gateup_tiles<2, kSplit>(stage, f0, f1, g0, g1, accg, accu, accg2, accu2);
        }
        __syncwarp();
        if (ok && lane == 0)
            mbar_arrive(&st.empty[slot]);
        ++st.seq;
        if (unit_ends(a1, ts, u, q, i)) {
            // the two groups' partial sums of the same output rows
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                accg[e] += accg2[e];
                accu[e] += accu2[e];
            }
            put_red(a, st, make_float4(accg[0], accg[1], accg[2], accg[3]),
                    make_float4(accu[0], accu[1], accu[2], accu[3]));
#pragma unroll
            for (int e = 0; e < 4; ++e)
                accg[e] = accu[e] = accg2[e] = accu2[e] = 0.f;
        }
        advance(u, q);
    }
}

// The down phase of a streaming warp: a step is up to kMaxDownStrips whole
// strips of one pair; the warp's groups w and w + 16 of each strip use the
// same two B fragments (h of the pair, polled when the warp reaches the
// pair).  Items of two strips go to the epilogue warps.
template <int BITS, bool PACK>
__device__ __forceinline__ void stream_down(const LayerArgs &a, const RouteView &rv, Stream &st)
{
    constexpr int NS = num_stages(ring_bits(BITS)), SB = stage_bytes(ring_bits(BITS));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = st.geo[1];
    const int a0 = g.a0, n = g.a1 - g.a0;
    if (n <= 0)
        return;
    const int fmax = a.f > a.fs ? a.f : a.fs;
    Pos q = decode(g, a0);
    UnitGeo u = unit_geo(g, q.p);
    int loaded = -1;
    int pb = ring_bits(BITS);
    BFrag bf[2];
#pragma unroll 1
    for (int kk = 0; kk < n; ++kk) {
        if (q.p != loaded) {
            u = unit_geo(g, q.p);
            const PairInfo pi = read_pair<PACK>(rv, q.p);
            pb = pair_bits<BITS>(a, rv.pairs[q.p * kPairInts]);
            bool okb = true;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int gi = warp + b * kStreamWarps;
                const bool on = gi < u.gk && !*st.fail;
                if (BITS != 0 || pb == 4)
                    okb = load_b_h<ring_bits(BITS), PACK>(a, pi, q.p, gi, on, fmax, st.tag, bf[b]) && okb;
                else
                    okb = load_b_h<2, PACK>(a, pi, q.p, gi, on, fmax, st.tag, bf[b]) && okb;
            }
            if (!okb && lane == 0) {
                set_status(a.status, kStatusTimeout);
                *st.fail = 1;
            }
            loaded = q.p;
        }
        const int slot = static_cast<int>(st.seq % NS);
        const bool ok = wait_stage<NS>(a, st, slot);
        const int ns = down_count(g, u, q);
        // the warp's groups w and w + 16 of each strip of the step (absent
        // groups skipped by uniform branches), strips in pairs -- one
        // reduction item each -- in a rolled loop, so that the tile code
        // exists once (a smaller loop for the instruction cache)
        const uint8_t *stage = st.ring + slot * SB;
        const bool g0 = warp < u.gk, g1 = warp + kStreamWarps < u.gk;
#pragma unroll 1
        for (int j2 = 0; j2 < ns; j2 += 2) {
            float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
            if (ok) {
#pragma unroll 1
                for (int jj = j2; jj < j2 + 2 && jj < ns; ++jj) {
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
                    if (BITS != 0 || pb == 4)
                        down_tiles<ring_bits(BITS), !PACK>(stage, jj, u.gk, bf, g0, g1, c);
                    else
                        down_tiles<2, !PACK>(stage, jj, u.gk, bf, g0, g1, c);
                    const bool first = jj == j2;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        a0[e] = first ? c[e] : a0[e];
                        a1[e] = first ? a1[e] : c[e];
                    }
                }
            }
            if (j2 + 2 >= ns) {  // the stage's last tiles are read: release it
                __syncwarp();
                if (ok && lane == 0)
                    mbar_arrive(&st.empty[slot]);
            }
            put_red(a, st, make_float4(a0[0], a0[1], a0[2], a0[3]), make_float4(a1[0], a1[1], a1[2], a1[3]));
        }
        ++st.seq;
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

// Sum reduction item st.uc over the 16 streaming warps (warp order) into
// (v0, v1) and free its slot; false if the wait ran out or the CTA failed.
__device__ __forceinline__ bool take_red(const LayerArgs &a, Stream &st, float4 &v0, float4 &v1)
{
    const int lane = threadIdx.x & 31;
    const int rs = st.uc % kRedSlots;
    const unsigned rph = static_cast<unsigned>(st.uc / kRedSlots);
    if (*st.fail)
        return false;
    if (!mbar_wait_bounded(&st.red_full[rs], rph & 1u)) {
        if (lane == 0) {
            set_status(a.status, kStatusTimeout);
            *st.fail = 1;
        }
        return false;
    }
    v0 = make_float4(0.f, 0.f, 0.f, 0.f);
    v1 = v0;
#pragma unroll 4
    for (int w2 = 0; w2 < kStreamWarps; ++w2) {
        const float4 *rr = st.red + ((rs * kStreamWarps + w2) * 2) * 32;
        const float4 a0 = rr[lane], a1 = rr[32 + lane];
        v0.x += a0.x, v0.y += a0.y, v0.z += a0.z, v0.w += a0.w;
        v1.x += a1.x, v1.y += a1.y, v1.z += a1.z, v1.w += a1.w;
    }
    __syncwarp();
    if (lane == 0)
        mbar_arrive(&st.red_empty[rs]);
    return true;
}

__device__ __forceinline__ EpiOut epi_out(const LayerArgs &a, uint32_t tag)
{
    EpiOut eo;
    eo.h_t = a.h_t;
    eo.part_t = a.part_t;
    eo.o_t = a.o_t;
    eo.o = a.o;
    eo.d = a.d;
    eo.fmax = a.f > a.fs ? a.f : a.fs;
    eo.fused = a.fused_combine;
    eo.tag = tag;
    eo.wait_cycles = a.wait_cycles;
    eo.status = a.status;
    return eo;
}

// The gate/up phase of an epilogue warp: the same walk over the CTA's
// steps; at each unit end it owns (items alternate between the epilogue
// warps) it sums the warps' partials and finalises the unit, or joins a
// unit shared with other CTAs.
template <int BITS, bool PACK>
__device__ __forceinline__ void epi_gateup(const LayerArgs &a, const RouteView &rv, Stream &st)
{
    const int e = (threadIdx.x >> 5) - kStreamWarps, lane = threadIdx.x & 31;
    const EpiOut eo = epi_out(a, st.tag);
    const Geo &g = st.geo[0];
    const int a0 = g.a0, a1 = g.a1, ts = g.ts, nt = g.a1 - g.ts;
    if (a0 >= a1)
        return;
    Pos q = decode(g, step_at(g, 0));
    UnitGeo u = unit_geo(g, q.p);
#pragma unroll 1
    for (int kk = 0; kk < a1 - a0; ++kk) {
        const int i = step_at(g, kk);
        if (kk == nt && kk > 0)
            q = decode(g, a0);
        u = unit_geo(g, q.p);
        if (unit_ends(a1, ts, u, q, i)) {
            float4 tg, tu;
            if (st.uc % kEpiWarps == e && take_red(a, st, tg, tu)) {
                const int pb = pair_bits<BITS>(a, rv.pairs[q.p * kPairInts]);
                const int ustart = i - q.c, uend = ustart + u.ch;
                const int ncols = rv.pairs[q.p * kPairInts + 1];
                constexpr int RB = ring_bits(BITS);
                if (ustart >= a0 && uend <= a1) {
                    if (BITS != 0 || pb == 4)
                        finalize_gateup<RB, PACK>(eo, ncols, q.p, q.s, tg, tu);
                    else
                        finalize_gateup<2, PACK>(eo, ncols, q.p, q.s, tg, tu);
                } else {
                    const bool ok = (BITS != 0 || pb == 4)
                                        ? fixup_gateup<RB, PACK>(eo, ncols, g, q.p, q.s, ustart, uend, tg, tu)
                                        : fixup_gateup<2, PACK>(eo, ncols, g, q.p, q.s, ustart, uend, tg, tu);
                    if (!ok && lane == 0) {
                        set_status(a.status, kStatusTimeout);
                        *st.fail = 1;
                    }
                }
            }
            ++st.uc;
        }
        advance(u, q);
    }
}

// The down phase of an epilogue warp: items of two strips of one step.
template <int BITS, bool PACK>
__device__ __forceinline__ void epi_down(const LayerArgs &a, const RouteView &rv, Stream &st)
{
    const int e = (threadIdx.x >> 5) - kStreamWarps;
    const EpiOut eo = epi_out(a, st.tag);
    const Geo &g = st.geo[1];
    const int a0 = g.a0, n = g.a1 - g.a0;
    if (n <= 0)
        return;
    Pos q = decode(g, a0);
    UnitGeo u = unit_geo(g, q.p);
#pragma unroll 1
    for (int kk = 0; kk < n; ++kk) {
        u = unit_geo(g, q.p);
        const int ns = down_count(g, u, q), s0 = down_first(u, q);
        for (int it = 0; 2 * it < ns; ++it) {
            float4 v0, v1;
            if (st.uc % kEpiWarps == e && take_red(a, st, v0, v1)) {
                const int pb = pair_bits<BITS>(a, rv.pairs[q.p * kPairInts]);
                const int ncols = rv.pairs[q.p * kPairInts + 1];
                if (BITS != 0 || pb == 4) {
                    finalize_down<ring_bits(BITS), PACK>(eo, ncols, q.p, s0 + 2 * it, v0);
                    if (2 * it + 1 < ns)
                        finalize_down<ring_bits(BITS), PACK>(eo, ncols, q.p, s0 + 2 * it + 1, v1);
                } else {
                    finalize_down<2, PACK>(eo, ncols, q.p, s0 + 2 * it, v0);
                    if (2 * it + 1 < ns)
                        finalize_down<2, PACK>(eo, ncols, q.p, s0 + 2 * it + 1, v1);
                }
            }
            ++st.uc;
        }
        advance(u, q);
    }
}

// Step geometry of one phase for P_r routed pairs of P_t; false if a limit
// the host checks is exceeded (never reached): gate/up chunks per strip (the
// B fragments a warp holds), down groups per strip (two per warp).
template <int KG>
__device__ __forceinline__ bool geo_phase(const LayerArgs &a, int phase, int P_r, int P_t, Geo *out)
{
    Geo gg = make_geo(a, phase, P_r, P_t);
    if (phase == 0)
        set_order(gg);
    *out = gg;
    return phase == 0 ? !(gg.ch0 > KG || (P_t > P_r && gg.ch1 > KG))
                      : !(gg.gk0 > kDownGroupsMax || (P_t > P_r && gg.gk1 > kDownGroupsMax));
}

// Leave this launch's tag as the next launch's sequence number once every
// CTA has marked its start (CTA 0, one warp, early in the launch: the next
// launch reads the number only after this one has completed).  The marks are
// loaded all at once, then any not yet tagged is polled (bounded); false if
// a poll ran out.
__device__ __forceinline__ bool publish_seq(const LayerArgs &a, uint32_t tag)
{
    const int lane = threadIdx.x & 31, C = static_cast<int>(gridDim.x);
    bool all = true;
    for (int c0 = 0; c0 < C; c0 += 8 * 32) {
        u64 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + 32 * i + lane;
            v[i] = c < C ? ld_word(a.started + c) : 0;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + 32 * i + lane;
            if (c < C && word_tag(v[i]) != tag && !poll_word(a.started + c, tag, a.wait_cycles, v[i]))
                all = false;
        }
    }
    all = __all_sync(0xffffffffu, all);
    if (all && lane == 0)
        st_relaxed_u32(a.seq, tag);
    return all;
}

// PACK: every pair holds at most 4 tokens (T <= 4), so the bf16 hi and lo
// parts of h (and of fp32 tokens) share one mma as column pairs.
template <int BITS, bool XBF16, int KG, bool PACK>
__global__ void __launch_bounds__(kThreads, 1) moe_layer_kernel(const __grid_constant__ LayerArgs a)
{
    constexpr int NS = num_stages(ring_bits(BITS));
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int s_fail;
    __shared__ uint32_t s_tag;
    __shared__ int s_spec;  // phases whose geometry was computed during routing
    __shared__ Geo s_geo[2];
    __shared__ Producer s_pr;
    Stream st;
    st.ring = smem;
    st.red = reinterpret_cast<float4 *>(smem + NS * stage_bytes(ring_bits(BITS)));
    st.full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes(ring_bits(BITS)) + red_bytes());
    st.empty = st.full + NS;
    st.red_full = st.empty + NS;
    st.red_empty = st.red_full + kRedSlots;
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
        s_spec = 0;
    }
    // Launched with programmatic stream serialization: the previous kernel on
    // the stream may still be finishing.  Only L2 prefetches of the router
    // rows come before waiting for it; every load (the workspace, x, the
    // rows) comes after it has completed and its writes are visible.  Then
    // the next kernel's launch may begin.
    if (a.do_route)
        router_prefetch_l2(a);
    pdl_wait();
    pdl_launch_dependents();
    RouterPre pre;
    pre.nrows = 0;
    if (a.do_route)
        pre = router_load(a);
    if (threadIdx.x == 0) {
        const uint32_t tag = ld_relaxed_u32(a.seq) + 1u;
        s_tag = tag;
        st_word(a.started + blockIdx.x, tag_word(blockIdx.x, tag));
    }
    cta_barrier();
    const uint32_t tag = s_tag;
    st.tag = tag;

    // ------------------------------------------------------------ phase R
    __shared__ RouteSmem rs;
    RouteView rv;
    int P_r = 0, P_t = 0;
    if (a.do_route) {
        router_rows<XBF16, PACK ? 4 : kPairCols>(a, pre, rs.red, tag);
        // every CTA stages all logits (polled until tagged) and the keys
        const int T = static_cast<int>(a.T), E = a.E, kk = a.k, E4 = (a.E + 3) & ~3;
        const int rows = E + (a.shared_gate ? 1 : 0);
        const uint32_t want = tag + a.tag_stall;
        for (int idx = threadIdx.x; idx < T * rows; idx += kThreads) {
            const int t = idx / rows, e = idx - t * rows;
            u64 v;
            if (!poll_word(a.logit_t + ((int64_t)blockIdx.x * T + t) * a.Epad + e, want, a.wait_cycles,
                           v)) {
                set_status(a.status, kStatusTimeout);
                s_fail = 1;
                break;
            }
            float l = __uint_as_float(word_payload(v));
            if (e == E) {  // the shared expert's gate
                rs.shared_w[t] = sigmoid_fast(l);
                continue;
            }
            if (l != l) {
                set_status(a.status, kStatusBadArg);
                l = -INFINITY;
            }
            // selection key: the logit; with a bias, logit + bias (softmax)
            // or fl32(sigmoid(logit)) + bias (sigmoid)
            float key = a.expert_bias
                            ? __fadd_rn(a.router_sigmoid ? sigmoid_fast(l) : l, __ldg(a.expert_bias + e))
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
        if (!a.shared_gate && threadIdx.x < T)
            rs.shared_w[threadIdx.x] = 1.0f;
        cta_barrier();
        const bool ok = s_fail == 0;
        if (ok && warp < kStreamWarps) {
            // Ranking: a quad of lanes per (token, expert), each lane counting
            // the experts ahead of it in one quarter of the keys; an expert
            // whose rank is below k is stored at its rank.
            const int n = T * E, ql = ((E + 15) / 16) * 4;
            const int qi = lane & 3, lo = qi * ql, hi = min(E, lo + ql);
            for (int base = 8 * warp; base < n; base += 8 * kStreamWarps) {
                const int item = base + (lane >> 2);
                const bool on = item < n;
                const int t = on ? item / E : 0, e = on ? item - t * E : 0;
                const float *key = rs.key + t * E4;
                int r = on && lo < hi ? rank_range(key, e, key[e], lo, hi) : 0;
                r += __shfl_xor_sync(0xffffffffu, r, 1);
                r += __shfl_xor_sync(0xffffffffu, r, 2);
                if (on && qi == 0 && r < kk)
                    rs.ids[t * kk + r] = static_cast<int16_t>(e);
            }
        } else if (ok) {
            // the other three warps: softmax statistics of the tokens; with
            // one token, which selects k distinct experts (k routed pairs and
            // the shared one whatever the selection), the step geometry of
            // the two phases on two of them while the ranking runs
            const int w3 = warp - kStreamWarps;  // 0 .. 2
            if (T == 1) {
                if (w3 == 0 && !a.router_sigmoid)
                    softmax_stats(rs.lg, E, rs.smax, rs.ssum);
                if (w3 > 0 && lane == 0) {
                    const bool good = geo_phase<KG>(a, w3 - 1, kk, kk + (a.has_shared ? 1 : 0), &s_geo[w3 - 1]);
                    if (good)
                        atomicAdd(&s_spec, 1);  // 2: both phases known
                }
            } else if (!a.router_sigmoid) {
                for (int t = w3; t < T; t += 3)
                    softmax_stats(rs.lg + t * E4, E, rs.smax + t, rs.ssum + t);
            }
        }
        cta_barrier();
        if (ok && warp < T) {
            // the weights of token t in rank order: the softmax over all E
            // logits or the expert's own sigmoid, renormalised over the
            // selection (summed in rank order, like the oracle) if norm,
            // times the routed scaling factor
            const int t = warp;
            float sc = 0.f;
            if (lane < kk) {
                const float l = rs.lg[t * E4 + rs.ids[t * kk + lane]];
                sc = a.router_sigmoid ? sigmoid_fast(l) : __fdividef(__expf(l - rs.smax[t]), rs.ssum[t]);
            }
            float psel = 0.f;
            for (int j = 0; j < kk; ++j)
                psel += __shfl_sync(0xffffffffu, sc, j);
            if (lane < kk) {
                const float wv = (a.norm ? __fdividef(sc, psel) : sc) * a.rsf;
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
        }
        // the pair table needs only the ids: built while the weights are
        if (ok && warp == kProducerWarp)
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

    // ------------------------------------------------------------ phases G, D
    // (the geometry computed during routing holds exactly when the routing
    // gave k routed pairs, which one token always does)
    if (!(s_spec == 2 && P_r == a.k)) {
        if (lane == 0 && warp < 2 && !geo_phase<KG>(a, warp, P_r, P_t, &s_geo[warp])) {
            set_status(a.status, kStatusBadArg);
            s_fail = 1;
        }
        cta_barrier();
    }
    st.geo = s_geo;
    st.pr = &s_pr;
    if (warp < kStreamWarps) {
        stream_gateup<BITS, XBF16, KG, PACK>(a, rv, st);
        stream_down<BITS, PACK>(a, rv, st);
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
        // the epilogue's first item is at least one unit away
        if (blockIdx.x == 0 && warp == kStreamWarps + 1 && !publish_seq(a, tag) && lane == 0)
            set_status(a.status, kStatusTimeout);
        epi_gateup<BITS, PACK && !XBF16>(a, rv, st);
        epi_down<BITS, PACK>(a, rv, st);
    }
    cta_barrier();

    // ------------------------------------------------------------ combine
    // (T <= 8) the outputs (t, row) dealt over the CTAs (output o to CTA
    // o mod grid, so every CTA takes its share as soon as its own roles are
    // done): y = sum_j w_j o_j (+ shared) in rank order, from the tagged
    // outputs, polled with short back-off (the last ones land at the end).
    // The slots' words are indexed by constants only (the shared expert's
    // apart), so they stay in registers.
    if (a.fused_combine && !s_fail) {
        const int T = static_cast<int>(a.T), kk = a.k, d = a.d;
        const bool has_sh = P_t > P_r;
        const int nout = T * d;
        const int C = static_cast<int>(gridDim.x);
        for (int o = static_cast<int>(threadIdx.x) * C + static_cast<int>(blockIdx.x); o < nout; o += C * kThreads) {
            const int t = o / d, row = o - t * d;
            u64 v[SMOE_MAX_TOPK_DEV], vs = 0;
            const long long t0 = clock64();
            unsigned ns = 32;
            bool good = true;
            for (;;) {
                bool all = true;
#pragma unroll
                for (int j = 0; j < SMOE_MAX_TOPK_DEV; ++j) {
                    if (j < kk) {
                        const int rm = rv.route_map[t * (kk + 1) + j];
                        v[j] = ld_word(a.o_t + (int64_t)rm * d + row);
                        all = all && word_tag(v[j]) == tag;
                    }
                }
                if (has_sh) {
                    vs = ld_word(a.o_t + (int64_t)rv.route_map[t * (kk + 1) + kk] * d + row);
                    all = all && word_tag(vs) == tag;
                }
                if (all)
                    break;
                if (clock64() - t0 > a.wait_cycles) {
                    good = false;
                    break;
                }
                __nanosleep(ns);
                if (ns < 128)
                    ns *= 2;
            }
            if (!good) {
                set_status(a.status, kStatusTimeout);
                break;
            }
            float yv = 0.f;
#pragma unroll
            for (int j = 0; j < SMOE_MAX_TOPK_DEV; ++j)
                if (j < kk)
                    yv = fmaf(rv.weights[t * kk + j], __uint_as_float(word_payload(v[j])), yv);
            if (has_sh)
                yv = fmaf(rv.shared_w[t], __uint_as_float(word_payload(vs)), yv);
            a.y[(int64_t)t * d + row] = yv;
        }
    }

    // ------------------------------------------------------------ exit
    if (warp == kProducerWarp && lane == 0) {
        // every stage issued has been consumed unless a wait ran out; then
        // wait (bounded) for the copies still in flight
        const uint32_t n = s_pr.next;
        for (uint32_t j = n > static_cast<uint32_t>(NS) ? n - NS : 0u; j < n; ++j)
            (void)mbar_wait_bounded(&st.full[j % NS], (j / NS) & 1u);
    }
}

template <int BITS, bool XBF16, int KG, bool PACK>
cudaError_t launch_t(const LayerArgs &a, cudaStream_t stream)
{
    auto kern = moe_layer_kernel<BITS, XBF16, KG, PACK>;
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
    // cooperative (every CTA resident: the phases hand off through tagged
    // words) and, where the runtime accepts it, programmatic stream
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

template <int BITS, int KG>
cudaError_t launch_depth(const LayerArgs &a, cudaStream_t stream)
{
    if (a.T <= 4)
        return a.x_bf16 ? launch_t<BITS, true, KG, true>(a, stream) : launch_t<BITS, false, KG, true>(a, stream);
    return a.x_bf16 ? launch_t<BITS, true, KG, false>(a, stream) : launch_t<BITS, false, KG, false>(a, stream);
}

cudaError_t launch_layer(const LayerArgs &a, cudaStream_t stream)
{
    // gate/up chunks per strip (d / 2048, rounded up) decide how many B
    // fragments a streaming warp holds
    const int kg = (a.d / kGroup + kChunkGroups - 1) / kChunkGroups;
    if (kg > 2 || a.f / kGroup > kDownGroupsMax || a.fs / kGroup > kDownGroupsMax)
        return cudaErrorInvalidValue;
    if (a.mixed)
        return kg <= 1 ? launch_depth<0, 1>(a, stream) : launch_depth<0, 2>(a, stream);
    if (a.bits == 4)
        return kg <= 1 ? launch_depth<4, 1>(a, stream) : launch_depth<4, 2>(a, stream);
    return kg <= 1 ? launch_depth<2, 1>(a, stream) : launch_depth<2, 2>(a, stream);
}

}  // namespace smoe
