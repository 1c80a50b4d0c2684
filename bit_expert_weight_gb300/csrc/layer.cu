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
//     compute the per-group activation sums.  The last warp to finish (an
//     arrival counter) routes every token and builds the pair table, then
//     releases the route flag.  For T > 8 a separate router kernel has done
//     this before the launch.
//  G  gate/up: the tiles of all pairs (pair = one expert x <= 8 tokens) form
//     one stream of 16-row strips; each warp takes an equal contiguous range
//     (stream-K), streams it through a private ring of shared-memory stages
//     filled by TMA bulk copies, decodes codes in registers and multiplies
//     with mma.sync.  A strip (16 rows x all of d, gate and up interleaved)
//     finished by one warp is finalised in registers; one shared by several
//     warps is finalised by the last to arrive, summing the partials in warp
//     order.  Finalising writes h = SiLU(g) * u as bf16 hi + lo and
//     per-strip class sums; the strip that completes a pair sums those into
//     per-group sums and releases the pair's ready flag.
//  D  down: the same streaming over 16-row strips of W_down.  A warp issues
//     its first weight copies before waiting for its pair's ready flag, so
//     the weights are in flight while gate/up finishes.  The last pair to
//     finish an output strip (T <= 8) sums sum_j w_j o_j (+ shared) in rank
//     order into y.
// Deterministic throughout: no float atomics.
#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kST = 4;  // tiles per stage
constexpr int kNS = 4;  // stages per warp ring
constexpr long long kSpinCycles = 4000000000ll;  // ~2 s at 2 GHz

__host__ __device__ constexpr int ring_bytes(int bits) { return kNS * kST * tile_bytes(bits); }
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
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned *p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

__device__ __forceinline__ int64_t warp_of(int64_t u, int64_t W, int64_t U)
{
    return ((u + 1) * W - 1) / U;
}

// --------------------------------------------------------------- routing

constexpr int kPerLane = kMaxExperts / 32;

__device__ void route_one_token(const float *lg, int E, int k, int norm, const float *bias,
                                int32_t *ids, float *w, int32_t *ids2, float *w2, int *status)
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
        ids[lane] = ej_mine;
        w[lane] = wv;
        if (ids2)
            ids2[lane] = ej_mine;
        if (w2)
            w2[lane] = wv;
    }
}

// Phase R work of one warp: unit < E (+1 shared gate row) -> logits of that
// row for all tokens; unit >= rows -> group sums of token (unit - rows).
template <bool XBF16>
__device__ void router_unit(const LayerArgs &a, int unit)
{
    const int lane = threadIdx.x & 31;
    const int d = a.d, T = static_cast<int>(a.T);
    const int rows = a.E + (a.shared_gate ? 1 : 0);
    if (unit < rows) {
        const uint16_t *wr = unit < a.E ? a.router_w + (int64_t)unit * d : a.shared_gate;
        float acc[kPairCols];
#pragma unroll
        for (int t = 0; t < kPairCols; ++t)
            acc[t] = 0.f;
        for (int c = lane * 8; c < d; c += 256) {
            const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(wr + c));
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
            float wf[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                wf[2 * i] = bf16lo_to_f32(ww[i]);
                wf[2 * i + 1] = bf16hi_to_f32(ww[i]);
            }
#pragma unroll
            for (int t = 0; t < kPairCols; ++t) {
                if (t >= T)
                    break;
                float xf[8];
                if (XBF16) {
                    const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(
                        reinterpret_cast<const uint16_t *>(a.x) + (int64_t)t * d + c));
                    const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        xf[2 * i] = bf16lo_to_f32(xx[i]);
                        xf[2 * i + 1] = bf16hi_to_f32(xx[i]);
                    }
                } else {
                    const float *xr = reinterpret_cast<const float *>(a.x) + (int64_t)t * d + c;
                    const float4 x0 = __ldg(reinterpret_cast<const float4 *>(xr));
                    const float4 x1 = __ldg(reinterpret_cast<const float4 *>(xr) + 1);
                    xf[0] = x0.x, xf[1] = x0.y, xf[2] = x0.z, xf[3] = x0.w;
                    xf[4] = x1.x, xf[5] = x1.y, xf[6] = x1.z, xf[7] = x1.w;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[t] = fmaf(wf[i], xf[i], acc[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < kPairCols; ++t) {
            float v = acc[t];
            for (int o = 16; o; o >>= 1)
                v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0 && t < T)
                a.logits[(int64_t)t * a.Epad + unit] = v;
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

// Route every token and build the pair table (T <= 8): pair = one selected
// expert with the (ascending) tokens that chose it; then the shared pair.
__device__ void route_and_dispatch(const LayerArgs &a)
{
    const int lane = threadIdx.x & 31;
    const int T = static_cast<int>(a.T), k = a.k, E = a.E;
    for (int t = 0; t < T; ++t) {
        route_one_token(a.logits + (int64_t)t * a.Epad, E, k, a.norm, a.expert_bias,
                        a.ids + t * k, a.weights + t * k, a.ids_out ? a.ids_out + t * k : nullptr,
                        a.w_out ? a.w_out + t * k : nullptr, a.status);
        if (lane == 0)
            a.shared_w[t] =
                a.shared_gate ? 1.0f / (1.0f + expf(-__ldcg(a.logits + (int64_t)t * a.Epad + E)))
                              : 1.0f;
    }
    __syncwarp();
    __threadfence_block();
    // pair_of[e] lives in the pair table's scratch area (E ints, zeroed = -1 + 1)
    int32_t *pair_of = a.scratch;
    for (int e = lane; e < E; e += 32)
        pair_of[e] = -1;
    __syncwarp();
    int npairs = 0;
    for (int t = 0; t < T; ++t) {
        int e = -1, p = -1;
        if (lane < k) {
            e = a.ids[t * k + lane];
            p = pair_of[e];
        }
        const unsigned newm = __ballot_sync(0xffffffffu, lane < k && p < 0);
        if (lane < k && p < 0) {
            p = npairs + __popc(newm & ((1u << lane) - 1u));
            pair_of[e] = p;
            int32_t *pr = a.pairs + p * kPairInts;
            pr[0] = e;
            pr[1] = 0;
        }
        npairs += __popc(newm);
        __syncwarp();
        if (lane < k) {
            int32_t *pr = a.pairs + p * kPairInts;
            const int col = pr[1];
            pr[2 + col] = t;
            pr[1] = col + 1;
            a.route_map[t * (k + 1) + lane] = p * kPairCols + col;
        }
        __syncwarp();
    }
    if (a.has_shared) {
        if (lane == 0) {
            int32_t *pr = a.pairs + npairs * kPairInts;
            pr[0] = -1;
            pr[1] = T;
            for (int t = 0; t < kPairCols; ++t)
                pr[2 + t] = t < T ? t : 0;
        }
        if (lane < T)
            a.route_map[lane * (k + 1) + k] = npairs * kPairCols + lane;
    }
    if (lane == 0) {
        a.meta[0] = npairs;
        a.meta[1] = npairs + (a.has_shared ? 1 : 0);
    }
    __syncwarp();
}

// --------------------------------------------------------------- the kernel

// This lane's 16 activations of one group (bf16 x: 2 vectors; fp32 x: 4;
// h of the down phase: hi in v[0..1], lo in v[2..3]) and the group sums
// (X0, X1) of the two output columns the lane accumulates.
template <int NV>
struct BRaw {
    uint4 v[NV];
    float2 xs0, xs1;
};

// One streaming phase (0: gate/up + SiLU, 1: down + combine) of one warp.
// Returns false if a bounded wait ran out (the status word is set).
template <int BITS, bool XBF16, int PHASE>
__device__ __forceinline__ bool run_phase(const LayerArgs &a, uint8_t *ring, uint64_t *bars,
                                          int64_t &seq_base, int P_r, int P_t, int fmax,
                                          int64_t w, int64_t Wall)
{
    constexpr int TB = tile_bytes(BITS);
    constexpr int CB = tile_code_bytes(BITS);
    constexpr float L = BITS == 4 ? 7.5f : 1.5f;
    constexpr int phase = PHASE;
    constexpr int NV = (PHASE == 1 || !XBF16) ? 4 : 2;
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, tig = lane & 3;
    const int d = a.d;
    bool ok = true;
    const int Kr = phase == 0 ? d : a.f;    // K of routed pairs
    const int Ks = phase == 0 ? d : a.fs;   // K of the shared pair
    const int Rr = phase == 0 ? a.f : d;    // output rows of routed pairs
    const int Rs = phase == 0 ? a.fs : d;
    const int tps_r = phase == 0 ? 2 * (Kr / kGroup) : Kr / kGroup;  // tiles per strip
    const int tps_s = phase == 0 ? 2 * (Ks / kGroup) : Ks / kGroup;
    const int64_t U_r = (int64_t)(Rr / kTileRows) * tps_r;
    const int64_t U_s = P_t > P_r ? (int64_t)(Rs / kTileRows) * tps_s : 0;
    const int64_t U = (int64_t)P_r * U_r + (int64_t)(P_t - P_r) * U_s;
    const int64_t W = U < Wall ? U : Wall;
    const bool active = w < W;
    const int64_t u0 = active ? w * U / W : 0, u1 = active ? (w + 1) * U / W : 0;
    const int64_t nst = (u1 - u0 + kST - 1) / kST;

    auto locate = [&](int64_t u, int &p, int64_t &lt) {
        if (u < (int64_t)P_r * U_r) {
            p = static_cast<int>(u / U_r);
            lt = u - (int64_t)p * U_r;
        } else {
            const int64_t v = u - (int64_t)P_r * U_r;
            const int q = static_cast<int>(v / U_s);
            p = P_r + q;
            lt = v - (int64_t)q * U_s;
        }
    };
    auto tile_src = [&](int p, int64_t lt) -> const uint8_t * {
        const int e = __ldcg(a.pairs + p * kPairInts);
        const uint8_t *base = e >= 0 ? a.tiles_routed + (int64_t)e * a.expert_bytes_routed +
                                           (phase == 0 ? 0 : a.down_off_routed)
                                     : a.tiles_shared + (phase == 0 ? 0 : a.down_off_shared);
        return base + lt * TB;
    };
    // lane 0 issues stage i of this phase (tiles u0 + i*ST ..); the two
    // marks let a failing warp drain exactly the copies still in flight
    int64_t issued_upto = 0, waited_upto = 0;
    auto issue = [&](int64_t i) {
        if (i >= nst)
            return;
        issued_upto = i + 1 > issued_upto ? i + 1 : issued_upto;
        const int64_t seq = seq_base + i;
        const int slot = static_cast<int>(seq % kNS);
        int64_t ua = u0 + i * kST;
        const int64_t ub = ua + kST < u1 ? ua + kST : u1;
        mbar_arrive_expect_tx(&bars[slot], static_cast<unsigned>((ub - ua) * TB));
        uint8_t *dst = ring + slot * (kST * TB);
        while (ua < ub) {
            int p;
            int64_t lt;
            locate(ua, p, lt);
            const int64_t pe = ua + ((p < P_r ? U_r : U_s) - lt);
            const int64_t ue = pe < ub ? pe : ub;
            bulk_g2s(dst, tile_src(p, lt), static_cast<unsigned>((ue - ua) * TB), &bars[slot]);
            dst += (ue - ua) * TB;
            ua = ue;
        }
    };
    if (lane == 0)
        for (int i = 0; i < kNS; ++i)
            issue(i);

    // activations of (pair, group): this lane's 16 columns of its token
    // row, and the group sums of the two output columns it accumulates
    // the segment's pair record, read once: its column count, this lane's
    // token row (gq) and the tokens of the lane's two output columns
    int pi_ncols = 0, pi_tok = 0, pi_t0 = -1, pi_t1 = -1;
    auto read_pair = [&](int p) {
        const int32_t *pr = a.pairs + p * kPairInts;
        pi_ncols = __ldcg(pr + 1);
        pi_tok = gq < pi_ncols ? __ldcg(pr + 2 + gq) : 0;
        pi_t0 = 2 * tig < pi_ncols ? __ldcg(pr + 2 + 2 * tig) : -1;
        pi_t1 = 2 * tig + 1 < pi_ncols ? __ldcg(pr + 2 + 2 * tig + 1) : -1;
    };
    auto load_b = [&](int p, int g, BRaw<NV> &r) {
        const bool valid = gq < pi_ncols;
        const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
        const float2 z2 = make_float2(0.f, 0.f);
        if (phase == 0) {
            const int tok = pi_tok;
            if (XBF16) {
                const uint4 *row = reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const uint16_t *>(a.x) + (int64_t)tok * d + g * kGroup + 16 * tig);
                r.v[0] = valid ? __ldg(row) : z4;
                r.v[1] = valid ? __ldg(row + 1) : z4;
            } else {
                const uint4 *row = reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const float *>(a.x) + (int64_t)tok * d + g * kGroup + 16 * tig);
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    r.v[i] = valid ? __ldg(row + i) : z4;
            }
            const float2 *xs = reinterpret_cast<const float2 *>(a.xsum);
            r.xs0 = pi_t0 >= 0 ? __ldcg(xs + (int64_t)pi_t0 * (d / kGroup) + g) : z2;
            r.xs1 = pi_t1 >= 0 ? __ldcg(xs + (int64_t)pi_t1 * (d / kGroup) + g) : z2;
        } else {
            const int64_t off = ((int64_t)p * kPairCols + gq) * fmax + g * kGroup + 16 * tig;
            const uint4 *hi = reinterpret_cast<const uint4 *>(a.h_hi + off);
            const uint4 *lo = reinterpret_cast<const uint4 *>(a.h_lo + off);
            r.v[0] = valid ? __ldcg(hi) : z4;
            r.v[1] = valid ? __ldcg(hi + 1) : z4;
            r.v[2] = valid ? __ldcg(lo) : z4;
            r.v[3] = valid ? __ldcg(lo + 1) : z4;
            const int c0 = 2 * tig, c1 = c0 + 1;
            const float2 *hs = reinterpret_cast<const float2 *>(a.hsum);
            const int64_t base = (int64_t)p * kPairCols * (fmax / kGroup);
            r.xs0 = c0 < pi_ncols ? __ldcg(hs + base + (int64_t)c0 * (fmax / kGroup) + g) : z2;
            r.xs1 = c1 < pi_ncols ? __ldcg(hs + base + (int64_t)c1 * (fmax / kGroup) + g) : z2;
        }
    };
    // B fragments for the mma from a BRaw
    uint32_t b0[4], b1[4], b0l[4], b1l[4];
    float bias0 = 0.f, bias1 = 0.f;
    const bool split = phase == 1 || !XBF16;
    auto cook_b = [&](const BRaw<NV> &r) {
        if (phase == 1) {
            const uint32_t *hv = reinterpret_cast<const uint32_t *>(r.v);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                b0[j] = hv[2 * j];
                b1[j] = hv[2 * j + 1];
                b0l[j] = hv[8 + 2 * j];
                b1l[j] = hv[8 + 2 * j + 1];
            }
        } else if (!XBF16) {
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

    // decode + multiply one tile from shared memory into acc
    auto mac_tile = [&](const uint8_t *tile, float (&acc)[4]) {
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
                if (split)
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
                if (split)
                    mma_bf16(dv, A, b0l[j], b1l[j]);
            }
        }
        acc[0] = fmaf(s01.x, dv[0], acc[0]);
        acc[1] = fmaf(s01.x, dv[1], acc[1]);
        acc[2] = fmaf(s01.y, dv[2], acc[2]);
        acc[3] = fmaf(s01.y, dv[3], acc[3]);
    };

    // ---- strip finalisation -------------------------------------------
    auto finalize = [&](int p, int s, const float (&ag)[4], const float (&au)[4]) {
        const int32_t *pr = a.pairs + p * kPairInts;
        const int ncols = __ldcg(pr + 1);
        const float invL = 1.0f / L;
        const int c0 = 2 * tig;
        if (phase == 0) {
            const int fp = p < P_r ? a.f : a.fs;
            float hs[2] = {0.f, 0.f};  // per output column, this lane's rows
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float g = ag[e] * invL, u = au[e] * invL;
                const float hv = g / (1.0f + expf(-g)) * u;
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
            // class of these rows within their 64-row group: (gq >> 1) & 1;
            // sum over lanes with equal tig and class (lane bits 2 and 4)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                hs[c] += __shfl_xor_sync(0xffffffffu, hs[c], 4);
                hs[c] += __shfl_xor_sync(0xffffffffu, hs[c], 16);
            }
            if ((gq & 5) == 0) {
                const int cls = (gq >> 1) & 1;
                const int nstrip = fmax / kTileRows;
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    if (c0 + c < ncols)
                        a.hs_part[(((int64_t)p * kPairCols + c0 + c) * nstrip + s) * 2 + cls] = hs[c];
            }
            __threadfence();
            __syncwarp();
            unsigned old = 0;
            if (lane == 0)
                old = atom_add_acqrel(a.pair_done + p, 1u);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == static_cast<unsigned>(fp / kTileRows - 1)) {
                // this strip completes the pair: group sums for the down phase
                __threadfence();
                const int ng = fp / kGroup, nstrip = fmax / kTileRows;
                for (int i = lane; i < ncols * ng; i += 32) {
                    const int col = i / ng, g = i % ng;
                    const float *src =
                        a.hs_part + (((int64_t)p * kPairCols + col) * nstrip + 4 * g) * 2;
                    float x0 = 0.f, x1 = 0.f;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        x0 += __ldcg(src + 2 * q);
                        x1 += __ldcg(src + 2 * q + 1);
                    }
                    reinterpret_cast<float2 *>(a.hsum)[((int64_t)p * kPairCols + col) * (fmax / kGroup) + g] =
                        make_float2(x0, x1);
                }
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    st_release(a.pair_ready + p, 1u);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = c0 + (e & 1);
                const int row = 16 * s + gq + 8 * (e >> 1);
                if (col < ncols)
                    a.o[((int64_t)p * kPairCols + col) * d + row] = ag[e] * invL;
            }
            if (!a.fused_combine)
                return;
            __threadfence();
            __syncwarp();
            unsigned old = 0;
            if (lane == 0)
                old = atom_add_acqrel(a.comb_ctr + s, 1u);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == static_cast<unsigned>(P_t - 1)) {
                __threadfence();
                const int T = static_cast<int>(a.T), kk = a.k;
                const bool has_sh = P_t > P_r;
                for (int i = lane; i < kTileRows * T; i += 32) {
                    const int t = i / kTileRows, row = 16 * s + i % kTileRows;
                    float yv = 0.f;
                    for (int j = 0; j < kk; ++j) {
                        const int rm = __ldcg(a.route_map + t * (kk + 1) + j);
                        yv = fmaf(__ldcg(a.weights + t * kk + j), __ldcg(a.o + (int64_t)rm * d + row), yv);
                    }
                    if (has_sh) {
                        const int rm = __ldcg(a.route_map + t * (kk + 1) + kk);
                        yv = fmaf(__ldcg(a.shared_w + t), __ldcg(a.o + (int64_t)rm * d + row), yv);
                    }
                    a.y[(int64_t)t * d + row] = yv;
                }
                __syncwarp();
                if (lane == 0)
                    a.comb_ctr[s] = 0u;
            }
        }
    };

    // flush strip (p, s) covering global tiles [ss, se)
    auto flush = [&](int p, int s, int64_t ss, int64_t se, const float (&ag)[4],
                     const float (&au)[4]) {
        const int64_t wf = warp_of(ss, W, U), wl = warp_of(se - 1, W, U);
        if (wf == wl) {
            finalize(p, s, ag, au);
            return;
        }
        const int myslot = u0 >= ss ? 0 : 1;
        float4 *mine = reinterpret_cast<float4 *>(a.partial) + ((w * 2 + myslot) * 2) * 32;
        mine[lane] = make_float4(ag[0], ag[1], ag[2], ag[3]);
        mine[32 + lane] = make_float4(au[0], au[1], au[2], au[3]);
        __threadfence();
        __syncwarp();
        unsigned *ctr = (phase == 0 ? a.strip_ctr_g : a.strip_ctr_d) +
                        (int64_t)p * a.max_strips + s;
        unsigned old = 0;
        if (lane == 0)
            old = atom_add_acqrel(ctr, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != static_cast<unsigned>(wl - wf))
            return;
        __threadfence();
        float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
        for (int64_t w0 = wf; w0 <= wl; w0 += 4) {
            float4 vg[4], vu[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t ww = w0 + q;
                if (ww <= wl) {
                    const int sl = ww * U / W >= ss ? 0 : 1;
                    const float4 *src = reinterpret_cast<const float4 *>(a.partial) + ((ww * 2 + sl) * 2) * 32;
                    vg[q] = __ldcg(src + lane);
                    vu[q] = phase == 0 ? __ldcg(src + 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (w0 + q <= wl) {
                    tg[0] += vg[q].x, tg[1] += vg[q].y, tg[2] += vg[q].z, tg[3] += vg[q].w;
                    tu[0] += vu[q].x, tu[1] += vu[q].y, tu[2] += vu[q].z, tu[3] += vu[q].w;
                }
            }
        }
        if (lane == 0)
            *ctr = 0u;
        finalize(p, s, tg, tu);
    };

    // ---- main loop over (pair, strip) segments ------------------------
    int waited_p = -1;
    int64_t u = u0;
    BRaw<NV> rA, rB, rC;
#pragma unroll 1
    while (u < u1) {
        int p;
        int64_t lt;
        locate(u, p, lt);
        const int tps = p < P_r ? tps_r : tps_s;
        const int s = static_cast<int>(lt / tps);
        const int pos0 = static_cast<int>(lt - (int64_t)s * tps);
        const int64_t ss = u - pos0, se = ss + tps;
        const int64_t ue = se < u1 ? se : u1;
        const int pos1 = static_cast<int>(pos0 + (ue - u));
        if (phase == 1 && p != waited_p) {
            if (!warp_wait_geq(a.pair_ready + p, 1u, a.status)) {
                ok = false;
                break;
            }
            waited_p = p;
        }
        read_pair(p);
        // groups of this segment: phase 0 has 2 tiles (gate, up) per group
        const int tpg = phase == 0 ? 2 : 1;
        const int g0 = pos0 / tpg, g1 = (pos1 - 1) / tpg + 1;
        float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
        auto do_group = [&](const BRaw<NV> &cur, BRaw<NV> &fill, int g) {
            if (g + 2 < g1)
                load_b(p, g + 2, fill);
            cook_b(cur);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h >= tpg)
                    break;
                const int pos = g * tpg + h;
                if (pos < pos0 || pos >= pos1)
                    continue;
                const int64_t uu = ss + pos;
                const int64_t i = (uu - u0) / kST;
                const int within = static_cast<int>((uu - u0) - i * kST);
                const int64_t seq = seq_base + i;
                const int slot = static_cast<int>(seq % kNS);
                if (within == 0) {
                    if (!mbar_wait_bounded(&bars[slot], static_cast<unsigned>((seq / kNS) & 1))) {
                        ok = false;
                        return;
                    }
                    waited_upto = i + 1;
                }
                const uint8_t *tile = ring + slot * (kST * TB) + within * TB;
                if (h == 0)
                    mac_tile(tile, ag);
                else
                    mac_tile(tile, au);
                if (within == kST - 1 || uu == u1 - 1) {
                    __syncwarp();
                    if (lane == 0)
                        issue(i + kNS);
                }
            }
        };
        load_b(p, g0, rA);
        if (g0 + 1 < g1)
            load_b(p, g0 + 1, rB);
#pragma unroll 1
        for (int g = g0; g < g1 && ok; g += 3) {
            do_group(rA, rC, g);
            if (g + 1 < g1 && ok)
                do_group(rB, rA, g + 1);
            if (g + 2 < g1 && ok)
                do_group(rC, rB, g + 2);
        }
        if (!ok)
            break;
        flush(p, s, ss, se, ag, au);
        u = ue;
    }
    if (!ok) {
        if (lane == 0) {
            set_status(a.status, kStatusTimeout);
            // drain this warp's copies still in flight (bounded)
            for (int64_t i = waited_upto; i < issued_upto; ++i) {
                const int64_t seq = seq_base + i;
                (void)mbar_wait_bounded(&bars[seq % kNS], static_cast<unsigned>((seq / kNS) & 1));
            }
        }
        __syncwarp();
        return false;
    }
    seq_base += nst;
    return true;
}

template <int BITS, bool XBF16>
__global__ void __launch_bounds__(kThreads, 2) moe_layer_kernel(const LayerArgs a)
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

    const int64_t w = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t Wall = (int64_t)gridDim.x * kWarps;
    bool ok = true;

    // ------------------------------------------------------------ phase R
    if (a.do_route) {
        const int rows = a.E + (a.shared_gate ? 1 : 0);
        const int units = rows + static_cast<int>(a.T);
        // unit i runs on warp i / gridDim.x of CTA i % gridDim.x: one per SM first
        const int64_t unit = (int64_t)warp * gridDim.x + blockIdx.x;
        if (unit < units) {
            router_unit<XBF16>(a, static_cast<int>(unit));
            __threadfence();
            __syncwarp();
            unsigned old = 0;
            if (lane == 0)
                old = atom_add_acqrel(a.route_ctr, 1u);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == static_cast<unsigned>(units - 1)) {
                __threadfence();
                route_and_dispatch(a);
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    st_release(a.route_flag, 1u);
            }
        }
        ok = warp_wait_geq(a.route_flag, 1u, a.status);
    }

    const int P_r = ok ? __ldcg(a.meta + 0) : 0;
    const int P_t = ok ? __ldcg(a.meta + 1) : 0;
    const int fmax = a.f > a.fs ? a.f : a.fs;

    // ------------------------------------------------------------ phases G, D
    int64_t seq_base = 0;  // ring stages issued (and consumed) by earlier phases
    if (ok)
        ok = run_phase<BITS, XBF16, 0>(a, ring, bars, seq_base, P_r, P_t, fmax, w, Wall);
    if (ok)
        ok = run_phase<BITS, XBF16, 1>(a, ring, bars, seq_base, P_r, P_t, fmax, w, Wall);

    // ------------------------------------------------------------ exit: the
    // last warp out resets the flags (counters of strips reset themselves)
    __threadfence();
    __syncwarp();
    unsigned old = 0;
    if (lane == 0)
        old = atom_add_acqrel(a.exit_ctr, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == static_cast<unsigned>(Wall - 1)) {
        for (int p = lane; p < a.max_pairs; p += 32) {
            a.pair_done[p] = 0u;
            a.pair_ready[p] = 0u;
        }
        if (lane == 0) {
            *a.route_ctr = 0u;
            *a.route_flag = 0u;
            __threadfence();
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
