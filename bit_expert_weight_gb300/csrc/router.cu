// router.cu -- router GEMV, softmax, top-k, renormalisation and dispatch
// ("Model Agnosticism", SmoeModelConfig: the gate has max_experts_per_layer
// rows; "CMF v2 -- Format Specification", 2.2 MoE: softmax over ALL logits,
// top-k with ties to the lower index, selection-only expert_bias, optional
// renormalisation, the shared expert weighted by sigmoid(gate . x)).
//
// One kernel per layer.  CTA (token tile of 8, K slice) computes partial
// logits of all experts with mma.sync (router rows are the A operand, the 8
// tokens the columns; fp32 activations are split into bf16 hi + lo), plus
// the per-group activation sums the expert kernels need.  The last CTA of a
// token tile (arrival counter) sums the K slices in order, routes its tokens
// (one warp per token) and, if it is the last tile overall, builds the pair
// table: every expert's tokens in token order, cut into pairs of <= 8
// columns, plus the shared expert's pairs.  Counters reset themselves.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace smoe {

namespace {

constexpr int kRWarps = 8;
constexpr int kRThreads = kRWarps * 32;
constexpr int kMaxMt = (kMaxExperts + 1 + 15) / 16;          // m-tiles incl. gate row
constexpr int kMtPerWarp = (kMaxMt + kRWarps - 1) / kRWarps;   // 3 for 256 experts
constexpr int kPerLane = kMaxExperts / 32;

// Route one token with one warp: lg = its E logits (any address space).
// Scores: softmax over all E, or (sigm) each expert's sigmoid; key = the
// logit, or with a bias logit + bias (softmax) / fl32(sigmoid) + bias
// (sigmoid); weights = selected scores, renormalised if norm, times rsf.
__device__ void route_token_warp(const float *lg, int E, int k, int norm, const float *bias,
                                 int sigm, float rsf, const ExpertMask &mask, int32_t *ids,
                                 float *w, int32_t *ids2, float *w2, int *status)
{
    const int lane = threadIdx.x & 31;
    float key[kPerLane], lv[kPerLane];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        float l = -INFINITY, kk = -INFINITY;
        if (e < E) {
            l = lg[e];
            if (l != l) {  // NaN logit: record and treat as -inf
                set_status(status, kStatusBadArg);
                l = -INFINITY;
            }
            if (bias)
                kk = __fadd_rn(sigm ? 1.0f / (1.0f + expf(-l)) : l, __ldg(bias + e));
            else
                kk = l;
            // an expert outside the routing mask: no key, no softmax term
            if (mask.on && !((mask.w[e >> 5] >> (e & 31)) & 1u)) {
                kk = -INFINITY;
                l = -INFINITY;
            }
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
    float psel = 0.f;
    float pj_mine = 0.f;  // lane j keeps slot j's probability
    int ej_mine = 0;
    for (int j = 0; j < k; ++j) {
        float bk = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u)) {
                if (bi == 0x7fffffff || key[i] > bk || (key[i] == bk && e < bi)) {
                    bk = key[i];
                    bi = e;
                }
            }
        }
        for (int o = 16; o; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != 0x7fffffff &&
                (bi == 0x7fffffff || ok > bk || (ok == bk && oi < bi))) {
                bk = ok;
                bi = oi;
            }
        }
        if ((bi & 31) == lane)
            taken |= 1u << (bi >> 5);
        const float p = sigm ? 1.0f / (1.0f + expf(-lg[bi])) : expf(lg[bi] - m) / z;
        psel += p;
        if (lane == j) {
            pj_mine = p;
            ej_mine = bi;
        }
    }
    if (lane < k) {
        const float wv = (norm ? pj_mine / psel : pj_mine) * rsf;
        ids[lane] = ej_mine;
        w[lane] = wv;
        if (ids2)
            ids2[lane] = ej_mine;
        if (w2)
            w2[lane] = wv;
    }
}

__global__ void __launch_bounds__(kRThreads) route_logits_kernel(const float *logits, int64_t T,
                                                                 int E, int k, int norm,
                                                                 const float *bias, int sigm,
                                                                 float rsf, const ExpertMask mask,
                                                                 int32_t *ids, float *w,
                                                                 int *status)
{
    const int64_t t = (int64_t)blockIdx.x * kRWarps + (threadIdx.x >> 5);
    if (t >= T)
        return;
    route_token_warp(logits + t * E, E, k, norm, bias, sigm, rsf, mask, ids + t * k, w + t * k,
                     nullptr, nullptr, status);
}

struct DispatchSmem {
    int cnt[kMaxExperts];
    int pbase[kMaxExperts + 1];
    int run[kMaxExperts];
    unsigned mask[kRWarps][kMaxExperts];
    int wbase[kRWarps][kMaxExperts];
};
struct LogitSmem {
    float lg[kPairCols][kMaxMt * 16];
};
union RouterSmem {
    DispatchSmem dsp;
    LogitSmem lgt;
};

__device__ void dispatch(const RouteArgs &a, DispatchSmem &s)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, k = a.k;
    const int64_t T = a.T;
    for (int e = tid; e < E; e += kRThreads) {
        s.cnt[e] = 0;
        s.run[e] = 0;
    }
    __syncthreads();
    for (int64_t i = tid; i < T * k; i += kRThreads) {
        const int e = __ldcg(a.ids + i);
        if (e >= 0 && e < E)
            atomicAdd(&s.cnt[e], 1);
        else
            set_status(a.status, kStatusBadExpert);
    }
    __syncthreads();
    __shared__ int s_ok, s_pr, s_pt;
    if (tid == 0) {
        int P = 0;
        for (int e = 0; e < E; ++e) {
            s.pbase[e] = P;
            P += (s.cnt[e] + kPairCols - 1) / kPairCols;
        }
        s.pbase[E] = P;
        const int nsh = a.has_shared ? static_cast<int>((T + kPairCols - 1) / kPairCols) : 0;
        s_pr = P;
        s_pt = P + nsh;
        s_ok = s_pt <= a.max_pairs;
        if (!s_ok)
            set_status(a.status, kStatusBadArg);
    }
    __syncthreads();
    if (!s_ok) {
        if (tid == 0) {
            a.meta[0] = 0;
            a.meta[1] = 0;
        }
        return;
    }
    for (int64_t r0 = 0; r0 < T; r0 += kRThreads) {
        for (int i = tid; i < kRWarps * E; i += kRThreads)
            s.mask[i / E][i % E] = 0u;
        __syncthreads();
        const int64_t t = r0 + tid;
        int ev[SMOE_MAX_TOPK_DEV];
        if (t < T) {
            for (int j = 0; j < k; ++j) {
                const int e = __ldcg(a.ids + t * k + j);
                ev[j] = (e >= 0 && e < E) ? e : -1;
                if (ev[j] >= 0)
                    atomicOr(&s.mask[warp][ev[j]], 1u << lane);
            }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kRThreads) {
            int c = s.run[e];
            for (int ww = 0; ww < kRWarps; ++ww) {
                s.wbase[ww][e] = c;
                c += __popc(s.mask[ww][e]);
            }
            s.run[e] = c;
        }
        __syncthreads();
        if (t < T) {
            const unsigned lt_mask = (1u << lane) - 1u;
            for (int j = 0; j < k; ++j) {
                const int e = ev[j];
                if (e < 0) {
                    a.route_map[t * (k + 1) + j] = 0;
                    continue;
                }
                const int pos = s.wbase[warp][e] + __popc(s.mask[warp][e] & lt_mask);
                const int pair = s.pbase[e] + pos / kPairCols, col = pos % kPairCols;
                int32_t *pr = a.pairs + pair * kPairInts;
                pr[2 + col] = static_cast<int32_t>(t);
                if (col == 0) {
                    pr[0] = e;
                    const int left = s.cnt[e] - (pos - col);
                    pr[1] = left < kPairCols ? left : kPairCols;
                }
                a.route_map[t * (k + 1) + j] = pair * kPairCols + col;
            }
        }
        __syncthreads();
    }
    const int P_r = s_pr, P_t = s_pt;
    for (int c = tid; c < P_t - P_r; c += kRThreads) {
        int32_t *pr = a.pairs + (P_r + c) * kPairInts;
        pr[0] = -1;
        const int64_t left = T - (int64_t)c * kPairCols;
        pr[1] = static_cast<int32_t>(left < kPairCols ? left : kPairCols);
        for (int i = 0; i < kPairCols; ++i)
            pr[2 + i] = static_cast<int32_t>((int64_t)c * kPairCols + i < T ? c * kPairCols + i : 0);
    }
    if (a.has_shared)
        for (int64_t t = tid; t < T; t += kRThreads)
            a.route_map[t * (k + 1) + k] = static_cast<int32_t>((P_r + t / kPairCols) * kPairCols + t % kPairCols);
    if (tid == 0) {
        a.meta[0] = P_r;
        a.meta[1] = P_t;
    }
}

template <bool XBF16>
__global__ void __launch_bounds__(kRThreads) router_kernel(const RouteArgs a)
{
    __shared__ RouterSmem sm;
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tig = lane & 3;
    const int nt = blockIdx.x, kc = blockIdx.y;
    const int64_t t0 = (int64_t)nt * kPairCols;
    const int d = a.d, E = a.E;
    const int Erows = E + (a.shared_gate ? 1 : 0);
    const int mtiles = (Erows + 15) / 16;
    const int Epad = mtiles * 16;
    const int Kc = d / a.ksplit;
    const int kb = kc * Kc;

    pdl_wait();
    pdl_launch_dependents();

    const int64_t tok = t0 + gq;
    const bool tvalid = tok < a.T;
    float acc[kMtPerWarp][4];
#pragma unroll
    for (int i = 0; i < kMtPerWarp; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            acc[i][e] = 0.f;
    const uint16_t *rowp[kMtPerWarp][2];
#pragma unroll
    for (int i = 0; i < kMtPerWarp; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = 16 * (warp + kRWarps * i) + gq + 8 * h;
            rowp[i][h] = r < E ? a.router_w + (int64_t)r * d
                               : (r == E && a.shared_gate ? a.shared_gate : nullptr);
        }
    float xs = 0.f;  // per-lane activation sum of the current group (class tig & 1)
    // one quantisation group (4 k-steps of 16) per iteration: every load of
    // the group is issued before its MMAs, so the L2 round trips overlap
    for (int k0 = kb; k0 < kb + Kc; k0 += kGroup) {
        uint32_t b0[4], b1[4], b0l[4], b1l[4];
        float xs4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = k0 + 16 * j;
            b0l[j] = b1l[j] = 0u;
            if (XBF16) {
                const uint16_t *xr = reinterpret_cast<const uint16_t *>(a.x) + tok * d + k + 2 * tig;
                b0[j] = tvalid ? __ldg(reinterpret_cast<const uint32_t *>(xr)) : 0u;
                b1[j] = tvalid ? __ldg(reinterpret_cast<const uint32_t *>(xr + 8)) : 0u;
            } else {
                const float *xr = reinterpret_cast<const float *>(a.x) + tok * d + k + 2 * tig;
                const float2 v0 = tvalid ? __ldg(reinterpret_cast<const float2 *>(xr)) : make_float2(0.f, 0.f);
                const float2 v1 = tvalid ? __ldg(reinterpret_cast<const float2 *>(xr + 8)) : make_float2(0.f, 0.f);
                split_bf16x2(v0.x, v0.y, b0[j], b0l[j]);
                split_bf16x2(v1.x, v1.y, b1[j], b1l[j]);
                xs4[j] = (v0.x + v0.y) + (v1.x + v1.y);
            }
        }
        uint32_t A[kMtPerWarp][4][4];
#pragma unroll
        for (int i = 0; i < kMtPerWarp; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = k0 + 16 * j;
                const bool on = warp + kRWarps * i < mtiles;
                A[i][j][0] = on && rowp[i][0] ? __ldg(reinterpret_cast<const uint32_t *>(rowp[i][0] + k + 2 * tig)) : 0u;
                A[i][j][1] = on && rowp[i][1] ? __ldg(reinterpret_cast<const uint32_t *>(rowp[i][1] + k + 2 * tig)) : 0u;
                A[i][j][2] = on && rowp[i][0] ? __ldg(reinterpret_cast<const uint32_t *>(rowp[i][0] + k + 2 * tig + 8)) : 0u;
                A[i][j][3] = on && rowp[i][1] ? __ldg(reinterpret_cast<const uint32_t *>(rowp[i][1] + k + 2 * tig + 8)) : 0u;
            }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (warp == 0) {
                if (XBF16)
                    xs += bf16lo_to_f32(b0[j]) + bf16hi_to_f32(b0[j]) + bf16lo_to_f32(b1[j]) +
                          bf16hi_to_f32(b1[j]);
                else
                    xs += xs4[j];
            }
#pragma unroll
            for (int i = 0; i < kMtPerWarp; ++i) {
                if (warp + kRWarps * i >= mtiles)
                    continue;
                mma_bf16(acc[i], A[i][j], b0[j], b1[j]);
                if (!XBF16)
                    mma_bf16(acc[i], A[i][j], b0l[j], b1l[j]);
            }
        }
        if (warp == 0) {
            // group complete: lanes tig and tig ^ 2 hold the same class
            const float tot = xs + __shfl_xor_sync(0xffffffffu, xs, 2);
            if (tig < 2 && tvalid)
                a.xsum[(tok * (d / kGroup) + k0 / kGroup) * 2 + tig] = tot;
            xs = 0.f;
        }
    }
    // partial logits [kc][T][Epad]
#pragma unroll
    for (int i = 0; i < kMtPerWarp; ++i) {
        if (warp + kRWarps * i >= mtiles)
            continue;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = 16 * (warp + kRWarps * i) + gq + 8 * (e >> 1);
            const int64_t t = t0 + 2 * tig + (e & 1);
            if (t < a.T && r < Erows)
                a.partial[((int64_t)kc * a.T + t) * Epad + r] = acc[i][e];
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned old = atomicAdd(&a.tile_ctr[nt], 1u);
        s_last = old == static_cast<unsigned>(a.ksplit - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    // sum the K slices in order
    for (int i = tid; i < kPairCols * Erows; i += kRThreads) {
        const int tt = i / Erows, r = i % Erows;
        const int64_t t = t0 + tt;
        float v = 0.f;
        if (t < a.T)
            for (int c = 0; c < a.ksplit; ++c)
                v += __ldcg(a.partial + ((int64_t)c * a.T + t) * Epad + r);
        sm.lgt.lg[tt][r] = v;
    }
    __syncthreads();
    {
        const int64_t t = t0 + warp;
        if (warp < kPairCols && t < a.T) {
            route_token_warp(sm.lgt.lg[warp], E, a.k, a.norm, a.expert_bias, a.router_sigmoid,
                             a.rsf, a.mask, a.ids + t * a.k, a.weights + t * a.k,
                             a.ids_out ? a.ids_out + t * a.k : nullptr,
                             a.w_out ? a.w_out + t * a.k : nullptr, a.status);
            if (lane == 0)
                a.shared_w[t] = a.shared_gate ? 1.0f / (1.0f + expf(-sm.lgt.lg[warp][E])) : 1.0f;
        }
    }
    if (tid == 0)
        a.tile_ctr[nt] = 0u;
    if (a.grp_tilecnt) {
        // grouped path: this tile's selections per expert; the sort's scan
        // and row assignment run in their own kernels
        __syncthreads();  // routing done: the logit buffer is free, ids written
        for (int e = tid; e < E; e += kRThreads)
            sm.dsp.cnt[e] = 0;
        __syncthreads();
        for (int i = tid; i < kPairCols * a.k; i += kRThreads) {
            const int64_t t = t0 + i / a.k;
            if (t < a.T) {
                const int e = __ldcg(a.ids + t * a.k + i % a.k);
                if (e >= 0 && e < E)
                    atomicAdd(&sm.dsp.cnt[e], 1);
            }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kRThreads)
            a.grp_tilecnt[(int64_t)nt * E + e] = sm.dsp.cnt[e];
        return;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned old = atomicAdd(a.done_ctr, 1u);
        s_last = old == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    dispatch(a, sm.dsp);
    if (tid == 0)
        *a.done_ctr = 0u;
}

// Grouped path with bf16 tokens: the logits come from the tensor-core GEMM.
// One CTA per 8-token tile, one warp per token: the shared expert's gate
// logit (sum_i gate[i] * x[t, i], fp32), the routing, then the tile's
// selections per expert for the sort.
__global__ void __launch_bounds__(kRThreads) route_tiles_kernel(const RouteArgs a, const float *logits,
                                                                int Epad)
{
    __shared__ int cnt[kMaxExperts];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E, k = a.k;
    const int64_t t0 = (int64_t)blockIdx.x * kPairCols;
    for (int e = tid; e < E; e += kRThreads)
        cnt[e] = 0;
    const int64_t t = t0 + warp;
    if (warp < kPairCols && t < a.T) {
        route_token_warp(logits + t * Epad, E, k, a.norm, a.expert_bias, a.router_sigmoid, a.rsf,
                         a.mask, a.ids + t * k, a.weights + t * k, a.ids_out ? a.ids_out + t * k : nullptr,
                         a.w_out ? a.w_out + t * k : nullptr, a.status);
        float sw = 1.0f;
        if (a.shared_gate) {
            const uint16_t *xr = static_cast<const uint16_t *>(a.x) + t * a.d;
            float acc = 0.f;
            // the gate vector is 4-byte aligned (API contract): 32-bit loads
            for (int i = 2 * lane; i < a.d; i += 64) {
                const uint32_t xv = __ldg(reinterpret_cast<const uint32_t *>(xr + i));
                const uint32_t gv = __ldg(reinterpret_cast<const uint32_t *>(a.shared_gate + i));
                acc = fmaf(bf16lo_to_f32(xv), bf16lo_to_f32(gv), acc);
                acc = fmaf(bf16hi_to_f32(xv), bf16hi_to_f32(gv), acc);
            }
            for (int o = 16; o; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            sw = 1.0f / (1.0f + expf(-acc));
        }
        if (lane == 0)
            a.shared_w[t] = sw;
    }
    __syncthreads();  // the tile's ids are written
    for (int i = tid; i < kPairCols * k; i += kRThreads) {
        const int64_t tt = t0 + i / k;
        if (tt < a.T) {
            const int e = __ldcg(a.ids + tt * k + i % k);
            if (e >= 0 && e < E)
                atomicAdd(&cnt[e], 1);
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kRThreads)
        a.grp_tilecnt[(int64_t)blockIdx.x * E + e] = cnt[e];
}

}  // namespace

cudaError_t launch_route_tiles(const RouteArgs &a, const float *logits, int Epad, cudaStream_t stream)
{
    if (a.T == 0)
        return cudaSuccess;
    route_tiles_kernel<<<static_cast<unsigned>((a.T + kPairCols - 1) / kPairCols), kRThreads, 0,
                         stream>>>(a, logits, Epad);
    return cudaGetLastError();
}

cudaError_t launch_route_logits(const float *logits, int64_t T, int E, int k, int norm,
                                const float *bias, int router_sigmoid, float rsf,
                                const ExpertMask &mask, int32_t *ids, float *w,
                                cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    route_logits_kernel<<<static_cast<unsigned>((T + kRWarps - 1) / kRWarps), kRThreads, 0, stream>>>(
        logits, T, E, k, norm, bias, router_sigmoid, rsf, mask, ids, w, device_status_word());
    return cudaGetLastError();
}

cudaError_t launch_router(const RouteArgs &a, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a.T + kPairCols - 1) / kPairCols),
                       static_cast<unsigned>(a.ksplit));
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.x_bf16)
        return cudaLaunchKernelEx(&cfg, router_kernel<true>, a);
    return cudaLaunchKernelEx(&cfg, router_kernel<false>, a);
}

}  // namespace smoe
