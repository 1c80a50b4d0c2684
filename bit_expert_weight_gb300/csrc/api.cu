// api.cu -- the C ABI of libsmoe.so (declared in include/smoe.h): argument
// validation, workspace layout and the launch sequence of one MoE layer.
#include <string.h>

#include <atomic>
#include <mutex>

#include "smoe.h"
#include "common.cuh"
#include "internal.h"

namespace smoe {

__device__ int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices] = {0};
int g_major[kMaxDevices] = {0};
int g_minor[kMaxDevices] = {0};
int *g_status_ptr[kMaxDevices] = {nullptr};

int cur_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 0;
    return dev;
}

void ensure_device_info()
{
    const int dev = cur_device();
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) {
            g_sms[dev] = prop.multiProcessorCount;
            g_major[dev] = prop.major;
            g_minor[dev] = prop.minor;
        } else {
            g_sms[dev] = 1;
        }
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess)
            g_status_ptr[dev] = static_cast<int *>(p);
    }
}

}  // namespace

int device_sm_count()
{
    ensure_device_info();
    return g_sms[cur_device()];
}

int device_cc_major()
{
    ensure_device_info();
    return g_major[cur_device()];
}

static int device_cc_minor()
{
    ensure_device_info();
    return g_minor[cur_device()];
}

int *device_status_word()
{
    ensure_device_info();
    return g_status_ptr[cur_device()];
}

}  // namespace smoe

using namespace smoe;

namespace {

// Bound of the layer kernel's tag polls (SM cycles; ~2 s at 2 GHz) and the
// routing-poll stall that smoe_debug_set_waits sets for tests.
std::atomic<long long> g_wait_cycles{kWaitCycles};
std::atomic<unsigned> g_tag_stall{0u};

}  // namespace

namespace {

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool device_supported()
{
    // The library is compiled for sm_103a only.
    return device_cc_major() == 10 && device_cc_minor() == 3;
}

smoe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SMOE_OK : SMOE_ERR_CUDA; }

int64_t expert_bytes(int d, int f, int bits)
{
    return 3ll * d * f / 1024 * tile_bytes(bits);
}

int64_t gateup_bytes(int d, int f, int bits) { return 2ll * d * f / 1024 * tile_bytes(bits); }

bool valid_layer(const smoe_layer_desc *L)
{
    if (!L)
        return false;
    if (L->bits != 2 && L->bits != 4)
        return false;
    if (L->group_size != SMOE_GROUP_SIZE)
        return false;
    if (L->d_model <= 0 || L->d_model % 128 || L->d_model > 4096)
        return false;
    if (L->ffn_dim <= 0 || L->ffn_dim % 64 || L->ffn_dim > 2048)
        return false;
    if (L->num_experts < 1 || L->num_experts > kMaxExperts)
        return false;
    if (L->top_k < 1 || L->top_k > SMOE_MAX_TOP_K || L->top_k > L->num_experts)
        return false;
    if (!L->router_w || !L->expert_tiles || !aligned(L->expert_tiles, 16) ||
        !aligned(L->router_w, 16))
        return false;
    if (L->shared_ffn_dim < 0 || L->shared_ffn_dim % 64 || L->shared_ffn_dim > 2048)
        return false;
    if ((L->shared_ffn_dim > 0) != (L->shared_tiles != nullptr))
        return false;
    if (L->shared_tiles && !aligned(L->shared_tiles, 16))
        return false;
    if (L->shared_gate_w && (!L->shared_tiles || !aligned(L->shared_gate_w, 4)))
        return false;
    return true;
}

struct Plan {
    int64_t T;
    int ntiles, ksplit, Epad, max_pairs, fmax, ctas;
    size_t off_seq, off_ctr_tile, off_ctr_done, off_flags, off_started, off_logit_t, off_h_t, off_part_t,
        off_o_t, off_meta, off_plog, off_logits, off_xsum, off_ids, off_w, off_sw, off_pairs, off_rmap,
        off_o, total;
    // grouped path (T >= kGroupedMinT only)
    bool grouped;
    int64_t grows;
    size_t off_grow, off_gseg, off_gtile, off_gxs, off_gh, off_go, off_grw;
};

// Whether the forward takes the expert-sorted tensor-core path: a token
// batch large enough that an average expert sees a dense block of rows.
// bf16 tokens only: the tensor-core path rounds its operands to bf16, so
// fp32 tokens always take the streaming path (fp32-accurate accumulation).
bool auto_grouped(const smoe_layer_desc *L, int64_t T, smoe_dtype x_dtype)
{
    return x_dtype == SMOE_BF16 && T >= kGroupedMinT && T * L->top_k >= 16ll * L->num_experts;
}

// mixed: a layer with per-expert depths, which always takes the grouped path.
Plan make_plan(const smoe_layer_desc *L, int64_t T, bool mixed = false)
{
    Plan p;
    p.T = T;
    const int d = L->d_model, E = L->num_experts, k = L->top_k;
    p.ntiles = static_cast<int>((T + kPairCols - 1) / kPairCols);
    const int G = d / 64;
    const int target = 2 * device_sm_count();
    int ks = 1;
    while (ks * 2 <= G && G % (ks * 2) == 0 && (int64_t)p.ntiles * ks * 2 <= target)
        ks *= 2;
    p.ksplit = ks;
    const int Erows = E + (L->shared_gate_w ? 1 : 0);
    p.Epad = (Erows + 15) / 16 * 16;
    const int64_t tk = T * k;
    const int64_t active = tk < E ? tk : E;
    int64_t mp = (tk + 7 * active + kPairCols - 1) / kPairCols;
    if (L->shared_ffn_dim > 0)
        mp += p.ntiles;
    if (mp < 1)
        mp = 1;
    p.max_pairs = static_cast<int>(mp);
    p.fmax = L->ffn_dim > L->shared_ffn_dim ? L->ffn_dim : L->shared_ffn_dim;
    p.ctas = layer_grid_ctas_max();
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    // Zeroed prefix (smoe_moe_workspace_init): the launch sequence number
    // first, at the same offset for every layer shape, so that it only ever
    // grows and no tagged word left by an earlier launch (of any shape)
    // carries a later launch's tag; then counters the kernels keep at zero,
    // and the tagged exchange areas of the layer kernel.
    const bool small = T <= kFusedCombineMaxT;
    p.off_seq = take(sizeof(unsigned));
    p.off_ctr_tile = take(sizeof(unsigned) * p.ntiles);
    p.off_ctr_done = take(sizeof(unsigned));
    p.off_flags = take(sizeof(unsigned) * 4);
    p.off_started = take(8 * (size_t)p.ctas);
    p.off_logit_t = take(small ? 8 * (size_t)p.ctas * T * p.Epad : 0);
    p.off_h_t = take(8 * (size_t)p.max_pairs * kPairCols * p.fmax);
    p.off_part_t = take(8 * (size_t)p.ctas * 2 * 32 * 8);
    p.off_o_t = take(small ? 8 * (size_t)p.max_pairs * kPairCols * d : 0);
    p.off_meta = take(sizeof(int32_t) * 2);
    p.off_plog = take(sizeof(float) * p.ksplit * T * p.Epad);
    p.off_logits = take(sizeof(float) * T * p.Epad);
    p.off_xsum = take(sizeof(float) * T * G * 2);
    p.off_ids = take(sizeof(int32_t) * tk);
    p.off_w = take(sizeof(float) * tk);
    p.off_sw = take(sizeof(float) * T);
    p.off_pairs = take(sizeof(int32_t) * kPairInts * p.max_pairs);
    p.off_rmap = take(sizeof(int32_t) * T * (k + 1));
    p.off_o = take(small ? 0 : sizeof(float) * (size_t)p.max_pairs * kPairCols * d);
    p.grouped = T >= kGroupedMinT || mixed;
    p.grows = 0;
    p.off_grow = p.off_gseg = p.off_gtile = p.off_gxs = p.off_gh = p.off_go = p.off_grw = 0;
    if (p.grouped) {
        const int has_sh = L->shared_ffn_dim > 0 ? 1 : 0;
        p.grows = grouped_max_rows(T, E, k, has_sh);
        p.off_grow = take(sizeof(int32_t) * T * (k + 1));
        p.off_gseg = take(sizeof(int32_t) * (2 * (kMaxExperts + 1) + 1));
        p.off_gtile = take(sizeof(int32_t) * (size_t)p.ntiles * E);
        p.off_gxs = take(sizeof(uint16_t) * (size_t)p.grows * d);
        p.off_gh = take(sizeof(uint16_t) * (size_t)p.grows * p.fmax);
        p.off_go = take(sizeof(uint16_t) * (size_t)p.grows * d);
        p.off_grw = take(sizeof(float) * (size_t)p.grows);
    }
    p.total = o;
    return p;
}

template <typename T_>
T_ *at(void *base, size_t off)
{
    return reinterpret_cast<T_ *>(static_cast<uint8_t *>(base) + off);
}

}  // namespace

namespace smoe {

size_t moe_workspace_zero_bytes(const smoe_layer_desc *layer, int64_t num_tokens)
{
    if (!valid_layer(layer) || num_tokens < 0)
        return 0;
    return make_plan(layer, num_tokens).off_meta;
}

}  // namespace smoe

extern "C" {

const char *smoe_status_string(smoe_status s)
{
    switch (s) {
    case SMOE_OK:
        return "ok";
    case SMOE_ERR_INVALID_ARG:
        return "invalid argument";
    case SMOE_ERR_UNSUPPORTED:
        return "unsupported (device or configuration)";
    case SMOE_ERR_WORKSPACE:
        return "workspace or output buffer too small";
    case SMOE_ERR_CUDA:
        return "CUDA error";
    case SMOE_ERR_DEVICE_FAULT:
        return "device-side fault recorded";
    case SMOE_ERR_TIMEOUT:
        return "device-side bounded wait timed out";
    }
    return "unknown status";
}

size_t smoe_stream_bytes(int64_t rows, int64_t cols, int bits)
{
    if (rows < 0 || cols < 0 || (bits != 2 && bits != 4))
        return 0;
    return static_cast<size_t>((rows * cols * bits + 7) / 8);
}

size_t smoe_scales_bytes(int64_t rows, int64_t cols, int group_size)
{
    if (rows < 0 || cols < 0 || group_size <= 0)
        return 0;
    return static_cast<size_t>((rows * cols + group_size - 1) / group_size) * 2;
}

size_t smoe_expert_tiles_bytes(int32_t d_model, int32_t ffn_dim, int bits, int group_size)
{
    if ((bits != 2 && bits != 4) || group_size != SMOE_GROUP_SIZE || d_model <= 0 ||
        d_model % 128 || ffn_dim <= 0 || ffn_dim % 64)
        return 0;
    return static_cast<size_t>(expert_bytes(d_model, ffn_dim, bits));
}

size_t smoe_repacked_bytes(int32_t d_model, int32_t ffn_dim, int32_t n_experts, int bits,
                           int group_size)
{
    if (n_experts < 0)
        return 0;
    return smoe_expert_tiles_bytes(d_model, ffn_dim, bits, group_size) * (size_t)n_experts;
}

smoe_status smoe_quantize(const void *w_bf16, int64_t rows, int64_t cols, int bits, int group_size,
                          uint8_t *codes_lsb, uint16_t *scales_f16, void *cuda_stream)
{
    if ((bits != 2 && bits != 4) || group_size != SMOE_GROUP_SIZE || rows < 0 || cols <= 0 ||
        cols % SMOE_GROUP_SIZE)
        return SMOE_ERR_INVALID_ARG;
    if (rows == 0)
        return SMOE_OK;
    if (!w_bf16 || !codes_lsb || !scales_f16 || !aligned(w_bf16, 4) || !aligned(scales_f16, 2))
        return SMOE_ERR_INVALID_ARG;
    if (!device_supported())
        return SMOE_ERR_UNSUPPORTED;
    return cuda_status(launch_quantize(static_cast<const uint16_t *>(w_bf16), rows, cols, bits,
                                       codes_lsb, scales_f16,
                                       static_cast<cudaStream_t>(cuda_stream)));
}

static smoe_status check_repack_args(int32_t d, int32_t f, int32_t n, int bits, int group_size)
{
    if ((bits != 2 && bits != 4) || group_size != SMOE_GROUP_SIZE || d <= 0 || d % 128 ||
        f <= 0 || f % 64 || n < 0)
        return SMOE_ERR_INVALID_ARG;
    return SMOE_OK;
}

smoe_status smoe_repack(const uint8_t *const *codes_lsb, const uint16_t *const *scales_f16,
                        int32_t d_model, int32_t ffn_dim, int32_t n_experts, int bits,
                        int group_size, void *tiles_out, size_t tiles_bytes, void *cuda_stream)
{
    smoe_status st = check_repack_args(d_model, ffn_dim, n_experts, bits, group_size);
    if (st)
        return st;
    if (n_experts == 0)
        return SMOE_OK;
    if (!codes_lsb || !scales_f16 || !tiles_out || !aligned(tiles_out, 16))
        return SMOE_ERR_INVALID_ARG;
    for (int i = 0; i < 3 * n_experts; ++i) {
        const int64_t cols = (i % 3 == 2) ? ffn_dim : d_model;
        if (!codes_lsb[i] || !scales_f16[i] || !aligned(scales_f16[i], 2) ||
            !aligned(codes_lsb[i], bits == 4 ? 8 : 4) || cols % 64)
            return SMOE_ERR_INVALID_ARG;
    }
    if (tiles_bytes < smoe_repacked_bytes(d_model, ffn_dim, n_experts, bits, group_size))
        return SMOE_ERR_WORKSPACE;
    if (!device_supported())
        return SMOE_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const int64_t eb = expert_bytes(d_model, ffn_dim, bits), gu = gateup_bytes(d_model, ffn_dim, bits);
    for (int e = 0; e < n_experts; ++e) {
        uint8_t *base = static_cast<uint8_t *>(tiles_out) + e * eb;
        for (int kind = 0; kind < 3; ++kind) {
            const int R = kind < 2 ? ffn_dim : d_model, K = kind < 2 ? d_model : ffn_dim;
            cudaError_t ce = launch_repack(codes_lsb[3 * e + kind], scales_f16[3 * e + kind], kind,
                                           R, K, bits, base, gu, s);
            if (ce != cudaSuccess)
                return SMOE_ERR_CUDA;
        }
    }
    return SMOE_OK;
}

smoe_status smoe_unpack(const void *tiles, int32_t d_model, int32_t ffn_dim, int32_t n_experts,
                        int bits, int group_size, uint8_t *const *codes_lsb,
                        uint16_t *const *scales_f16, void *cuda_stream)
{
    smoe_status st = check_repack_args(d_model, ffn_dim, n_experts, bits, group_size);
    if (st)
        return st;
    if (n_experts == 0)
        return SMOE_OK;
    if (!codes_lsb || !scales_f16 || !tiles || !aligned(tiles, 16))
        return SMOE_ERR_INVALID_ARG;
    for (int i = 0; i < 3 * n_experts; ++i)
        if (!codes_lsb[i] || !scales_f16[i] || !aligned(scales_f16[i], 2) ||
            !aligned(codes_lsb[i], bits == 4 ? 8 : 4))
            return SMOE_ERR_INVALID_ARG;
    if (!device_supported())
        return SMOE_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const int64_t eb = expert_bytes(d_model, ffn_dim, bits), gu = gateup_bytes(d_model, ffn_dim, bits);
    for (int e = 0; e < n_experts; ++e) {
        const uint8_t *base = static_cast<const uint8_t *>(tiles) + e * eb;
        for (int kind = 0; kind < 3; ++kind) {
            const int R = kind < 2 ? ffn_dim : d_model, K = kind < 2 ? d_model : ffn_dim;
            cudaError_t ce = launch_unpack(base, kind, R, K, bits, gu, codes_lsb[3 * e + kind],
                                           scales_f16[3 * e + kind], s);
            if (ce != cudaSuccess)
                return SMOE_ERR_CUDA;
        }
    }
    return SMOE_OK;
}

static bool valid_opts(const smoe_router_opts *o)
{
    // a positive, finite scaling factor; NaN fails both comparisons
    return !o || (o->routed_scaling_factor > 0.0f && o->routed_scaling_factor <= 3.0e38f);
}

// The routing mask of the options as kernel words; false if its tail bits
// beyond E are set or fewer than k experts are routable.
static bool make_mask(const smoe_router_opts *o, int E, int k, ExpertMask *m)
{
    memset(m, 0, sizeof *m);
    if (!o || !o->expert_mask)
        return true;
    int n = 0;
    for (int e = 0; e < (E + 7) / 8 * 8; ++e) {
        const bool bit = (o->expert_mask[e >> 3] >> (e & 7)) & 1;
        if (bit && e >= E)
            return false;
        if (bit) {
            m->w[e >> 5] |= 1u << (e & 31);
            ++n;
        }
    }
    m->on = 1;
    return n >= k;
}

smoe_status smoe_route_from_logits_ex(const float *logits, int64_t T, int32_t E, int32_t k,
                                      int norm_topk_prob, const float *expert_bias,
                                      const smoe_router_opts *opts, int32_t *ids,
                                      float *weights, void *cuda_stream)
{
    ExpertMask mask;
    if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > SMOE_MAX_TOP_K || k > E ||
        !valid_opts(opts) || !make_mask(opts, E, k, &mask))
        return SMOE_ERR_INVALID_ARG;
    if (T == 0)
        return SMOE_OK;
    if (!logits || !ids || !weights)
        return SMOE_ERR_INVALID_ARG;
    if (!device_supported())
        return SMOE_ERR_UNSUPPORTED;
    return cuda_status(launch_route_logits(logits, T, E, k, norm_topk_prob ? 1 : 0, expert_bias,
                                           opts && opts->router_sigmoid ? 1 : 0,
                                           opts ? opts->routed_scaling_factor : 1.0f, mask, ids,
                                           weights, static_cast<cudaStream_t>(cuda_stream)));
}

smoe_status smoe_route_from_logits(const float *logits, int64_t T, int32_t E, int32_t k,
                                   int norm_topk_prob, const float *expert_bias, int32_t *ids,
                                   float *weights, void *cuda_stream)
{
    if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > SMOE_MAX_TOP_K || k > E)
        return SMOE_ERR_INVALID_ARG;
    if (T == 0)
        return SMOE_OK;
    if (!logits || !ids || !weights)
        return SMOE_ERR_INVALID_ARG;
    if (!device_supported())
        return SMOE_ERR_UNSUPPORTED;
    ExpertMask none;
    memset(&none, 0, sizeof none);
    return cuda_status(launch_route_logits(logits, T, E, k, norm_topk_prob ? 1 : 0, expert_bias, 0,
                                           1.0f, none, ids, weights,
                                           static_cast<cudaStream_t>(cuda_stream)));
}

size_t smoe_moe_workspace_bytes(const smoe_layer_desc *layer, int64_t num_tokens)
{
    if (!valid_layer(layer) || num_tokens < 0)
        return 0;
    return make_plan(layer, num_tokens).total;
}

smoe_status smoe_moe_workspace_init(void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    if (!workspace && workspace_bytes)
        return SMOE_ERR_INVALID_ARG;
    if (!workspace_bytes)
        return SMOE_OK;
    return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes,
                                       static_cast<cudaStream_t>(cuda_stream)));
}

// The Q4 experts of a per-expert depth array as mask words; false unless
// every entry is 2 or 4.
static bool make_q4mask(const uint8_t *expert_bits, int E, uint32_t q4[8])
{
    memset(q4, 0, 8 * sizeof(uint32_t));
    if (!expert_bits || E < 1 || E > kMaxExperts)
        return false;
    for (int e = 0; e < E; ++e) {
        if (expert_bits[e] != 2 && expert_bits[e] != 4)
            return false;
        if (expert_bits[e] == 4)
            q4[e >> 5] |= 1u << (e & 31);
    }
    return true;
}

// expert_bits: nullable host [E] per-expert depths (a mixed layer).
static smoe_status forward_stages(const smoe_layer_desc *layer, const smoe_router_opts *opts,
                                  const void *x, smoe_dtype x_dtype, int64_t num_tokens, float *y,
                                  void *workspace, size_t workspace_bytes, int32_t *ids_out,
                                  float *w_out, int stage_mask, int path, void *cuda_stream,
                                  const uint8_t *expert_bits = nullptr)
{
    ExpertMask mask;
    uint32_t q4mask[8];
    const bool mixed = expert_bits != nullptr;
    if (!valid_layer(layer) || num_tokens < 0 || (x_dtype != SMOE_F32 && x_dtype != SMOE_BF16) ||
        !valid_opts(opts) || !make_mask(opts, layer->num_experts, layer->top_k, &mask) ||
        (mixed && !make_q4mask(expert_bits, layer->num_experts, q4mask)))
        return SMOE_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return SMOE_OK;
    if (!x || !y || !workspace || !aligned(x, 16) || !aligned(y, 16) || !aligned(workspace, 256))
        return SMOE_ERR_INVALID_ARG;
    if (!device_supported())
        return SMOE_ERR_UNSUPPORTED;
    const Plan P = make_plan(layer, num_tokens, mixed);
    if (workspace_bytes < P.total)
        return SMOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const smoe_layer_desc &L = *layer;
    int *status = device_status_word();
    // the tensor-core path takes bf16 tokens only (it would round fp32 ones)
    if (path == SMOE_PATH_GROUPED && x_dtype != SMOE_BF16)
        return SMOE_ERR_UNSUPPORTED;
    const bool grouped = path == SMOE_PATH_GROUPED ||
                         (path == SMOE_PATH_AUTO && auto_grouped(layer, num_tokens, x_dtype));
    if (grouped && !P.grouped)
        return SMOE_ERR_UNSUPPORTED;
    // T <= 8 with all stages: one fused launch (routing inside the kernel)
    const bool fused = num_tokens <= kFusedCombineMaxT && stage_mask == 7;

    RouteArgs ra;
    memset(&ra, 0, sizeof ra);
    ra.router_w = static_cast<const uint16_t *>(L.router_w);
    ra.shared_gate = static_cast<const uint16_t *>(L.shared_gate_w);
    ra.expert_bias = L.expert_bias;
    ra.x = x;
    ra.x_bf16 = x_dtype == SMOE_BF16;
    ra.T = num_tokens;
    ra.d = L.d_model;
    ra.E = L.num_experts;
    ra.k = L.top_k;
    ra.norm = L.norm_topk_prob ? 1 : 0;
    ra.bits = L.bits;
    ra.has_shared = L.shared_ffn_dim > 0;
    ra.ksplit = P.ksplit;
    ra.partial = at<float>(workspace, P.off_plog);
    ra.xsum = at<float>(workspace, P.off_xsum);
    ra.ids = at<int32_t>(workspace, P.off_ids);
    ra.weights = at<float>(workspace, P.off_w);
    ra.shared_w = at<float>(workspace, P.off_sw);
    ra.ids_out = ids_out;
    ra.w_out = w_out;
    ra.pairs = at<int32_t>(workspace, P.off_pairs);
    ra.route_map = at<int32_t>(workspace, P.off_rmap);
    ra.grp_tilecnt = grouped ? at<int32_t>(workspace, P.off_gtile) : nullptr;
    ra.meta = at<int32_t>(workspace, P.off_meta);
    ra.tile_ctr = at<unsigned>(workspace, P.off_ctr_tile);
    ra.done_ctr = at<unsigned>(workspace, P.off_ctr_done);
    ra.status = status;
    ra.max_pairs = P.max_pairs;
    ra.router_sigmoid = opts && opts->router_sigmoid ? 1 : 0;
    ra.rsf = opts ? opts->routed_scaling_factor : 1.0f;
    ra.mask = mask;

    LayerArgs la;
    memset(&la, 0, sizeof la);
    la.router_w = ra.router_w;
    la.shared_gate = ra.shared_gate;
    la.expert_bias = L.expert_bias;
    la.tiles_routed = static_cast<const uint8_t *>(L.expert_tiles);
    la.tiles_shared = static_cast<const uint8_t *>(L.shared_tiles);
    la.expert_bytes_routed = expert_bytes(L.d_model, L.ffn_dim, L.bits);
    la.down_off_routed = gateup_bytes(L.d_model, L.ffn_dim, L.bits);
    la.down_off_shared =
        L.shared_ffn_dim > 0 ? gateup_bytes(L.d_model, L.shared_ffn_dim, L.bits) : 0;
    la.x = x;
    la.x_bf16 = x_dtype == SMOE_BF16;
    la.T = num_tokens;
    la.d = L.d_model;
    la.f = L.ffn_dim;
    la.fs = L.shared_ffn_dim;
    la.E = L.num_experts;
    la.k = L.top_k;
    la.norm = ra.norm;
    la.bits = L.bits;
    la.Epad = P.Epad;
    la.has_shared = ra.has_shared;
    la.router_sigmoid = ra.router_sigmoid;
    la.rsf = ra.rsf;
    la.mask = mask;
    la.do_route = fused ? 1 : 0;
    la.fused_combine = num_tokens <= kFusedCombineMaxT ? 1 : 0;
    la.max_pairs = P.max_pairs;
    la.ids = ra.ids;
    la.weights = ra.weights;
    la.shared_w = ra.shared_w;
    la.ids_out = ids_out;
    la.w_out = w_out;
    la.pairs = ra.pairs;
    la.route_map = ra.route_map;
    la.meta = ra.meta;
    la.seq = at<unsigned>(workspace, P.off_seq);
    la.started = at<unsigned long long>(workspace, P.off_started);
    la.logit_t = at<unsigned long long>(workspace, P.off_logit_t);
    la.h_t = at<unsigned long long>(workspace, P.off_h_t);
    la.part_t = at<unsigned long long>(workspace, P.off_part_t);
    la.o_t = at<unsigned long long>(workspace, P.off_o_t);
    la.o = at<float>(workspace, P.off_o);
    unsigned *flags = at<unsigned>(workspace, P.off_flags);
    la.wait_cycles = g_wait_cycles.load();
    la.tag_stall = g_tag_stall.load();
    la.y = y;
    la.status = status;
    if (mixed) {
        la.mixed = 1;
        memcpy(la.q4mask, q4mask, sizeof q4mask);
    }

    if (grouped) {
        GroupedArgs ga;
        memset(&ga, 0, sizeof ga);
        ga.tiles_routed = la.tiles_routed;
        ga.tiles_shared = la.tiles_shared;
        ga.expert_bytes_routed = la.expert_bytes_routed;
        ga.down_off_shared = la.down_off_shared;
        ga.T = num_tokens;
        ga.d = L.d_model;
        ga.f = L.ffn_dim;
        ga.fs = L.shared_ffn_dim;
        ga.E = L.num_experts;
        ga.k = L.top_k;
        ga.bits = L.bits;
        ga.has_shared = ra.has_shared;
        ga.seg = at<int32_t>(workspace, P.off_gseg);
        ga.rows_of = at<int32_t>(workspace, P.off_grow);
        ga.rows = P.grows;
        ga.ids = ra.ids;
        ga.tilecnt = ra.grp_tilecnt;
        ga.ntiles = P.ntiles;
        ga.scan_ctr = flags + 2;
        ga.xs = at<uint16_t>(workspace, P.off_gxs);
        ga.h = at<uint16_t>(workspace, P.off_gh);
        ga.hstride = P.fmax;
        ga.o = at<uint16_t>(workspace, P.off_go);
        ga.w = ra.weights;
        ga.sw = ra.shared_w;
        ga.roww = at<float>(workspace, P.off_grw);
        ga.status = status;
        if (mixed) {
            ga.mixed = 1;
            memcpy(ga.q4mask, q4mask, sizeof q4mask);
        }
        if (stage_mask & 1) {
            if (ra.x_bf16) {
                if (launch_tc_logits(static_cast<const uint16_t *>(x), ra.router_w, num_tokens,
                                     L.d_model, L.num_experts, P.Epad,
                                     at<float>(workspace, P.off_logits), status,
                                     s) != cudaSuccess ||
                    launch_route_tiles(ra, at<float>(workspace, P.off_logits), P.Epad, s) !=
                        cudaSuccess)
                    return SMOE_ERR_CUDA;
            } else if (launch_router(ra, s, false) != cudaSuccess) {
                return SMOE_ERR_CUDA;
            }
        }
        return launch_grouped(ga, x, ra.x_bf16, y, stage_mask, s) ==
                       cudaSuccess
                   ? SMOE_OK
                   : SMOE_ERR_CUDA;
    }
    if (fused)
        return launch_layer(la, s) == cudaSuccess ? SMOE_OK : SMOE_ERR_CUDA;
    if ((stage_mask & 1) && launch_router(ra, s, false) != cudaSuccess)
        return SMOE_ERR_CUDA;
    if ((stage_mask & 2) && launch_layer(la, s) != cudaSuccess)
        return SMOE_ERR_CUDA;
    if ((stage_mask & 4) && !la.fused_combine && launch_combine(la, s) != cudaSuccess)
        return SMOE_ERR_CUDA;
    return SMOE_OK;
}

smoe_status smoe_moe_forward(const smoe_layer_desc *layer, const void *x, smoe_dtype x_dtype,
                             int64_t num_tokens, float *y, void *workspace,
                             size_t workspace_bytes, int32_t *ids_out, float *w_out,
                             void *cuda_stream)
{
    return forward_stages(layer, nullptr, x, x_dtype, num_tokens, y, workspace, workspace_bytes,
                          ids_out, w_out, 7, SMOE_PATH_AUTO, cuda_stream);
}

smoe_status smoe_moe_forward_ex(const smoe_layer_desc *layer, const smoe_router_opts *opts,
                                const void *x, smoe_dtype x_dtype, int64_t num_tokens, float *y,
                                void *workspace, size_t workspace_bytes, int32_t *ids_out,
                                float *w_out, int path, void *cuda_stream)
{
    if (path != SMOE_PATH_AUTO && path != SMOE_PATH_STREAM && path != SMOE_PATH_GROUPED)
        return SMOE_ERR_INVALID_ARG;
    return forward_stages(layer, opts, x, x_dtype, num_tokens, y, workspace, workspace_bytes,
                          ids_out, w_out, 7, path, cuda_stream);
}

smoe_status smoe_moe_forward_path(const smoe_layer_desc *layer, const void *x, smoe_dtype x_dtype,
                                  int64_t num_tokens, float *y, void *workspace,
                                  size_t workspace_bytes, int32_t *ids_out, float *w_out, int path,
                                  void *cuda_stream)
{
    if (path != SMOE_PATH_AUTO && path != SMOE_PATH_STREAM && path != SMOE_PATH_GROUPED)
        return SMOE_ERR_INVALID_ARG;
    return forward_stages(layer, nullptr, x, x_dtype, num_tokens, y, workspace, workspace_bytes,
                          ids_out, w_out, 7, path, cuda_stream);
}

int smoe_moe_path(const smoe_layer_desc *layer, int64_t num_tokens)
{
    return smoe_moe_path_dtype(layer, num_tokens, SMOE_BF16);
}

int smoe_moe_path_dtype(const smoe_layer_desc *layer, int64_t num_tokens, smoe_dtype x_dtype)
{
    if (!valid_layer(layer) || num_tokens < 0 || (x_dtype != SMOE_F32 && x_dtype != SMOE_BF16))
        return -1;
    return auto_grouped(layer, num_tokens, x_dtype) ? SMOE_PATH_GROUPED : SMOE_PATH_STREAM;
}

smoe_status smoe_moe_forward_stage(const smoe_layer_desc *layer, const void *x,
                                   smoe_dtype x_dtype, int64_t num_tokens, float *y,
                                   void *workspace, size_t workspace_bytes, int32_t *ids_out,
                                   float *w_out, int stage, void *cuda_stream)
{
    if (stage < 0 || stage > 2)
        return SMOE_ERR_INVALID_ARG;
    return forward_stages(layer, nullptr, x, x_dtype, num_tokens, y, workspace, workspace_bytes,
                          ids_out, w_out, 1 << stage, SMOE_PATH_AUTO, cuda_stream);
}

size_t smoe_repacked_bytes_mixed(int32_t d_model, int32_t ffn_dim, int32_t n_experts,
                                 const uint8_t *expert_bits, int group_size)
{
    if (n_experts < 0 || (n_experts > 0 && !expert_bits))
        return 0;
    size_t total = 0;
    for (int e = 0; e < n_experts; ++e) {
        const size_t b = smoe_expert_tiles_bytes(d_model, ffn_dim, expert_bits[e], group_size);
        if (!b)
            return 0;
        total += b;
    }
    return total;
}

// One repack or unpack of experts at their own depths, back to back.
static smoe_status mixed_pass(bool repack, const uint8_t *const *codes, const uint16_t *const *scales,
                              int32_t d, int32_t f, int32_t n, const uint8_t *expert_bits,
                              int group_size, const void *tiles_in, void *tiles_out,
                              size_t tiles_bytes, void *cuda_stream)
{
    if (n < 0 || group_size != SMOE_GROUP_SIZE || d <= 0 || d % 128 || f <= 0 || f % 64)
        return SMOE_ERR_INVALID_ARG;
    if (n == 0)
        return SMOE_OK;
    if (!expert_bits || !codes || !scales || !(repack ? tiles_out : tiles_in) ||
        !aligned(repack ? tiles_out : tiles_in, 16))
        return SMOE_ERR_INVALID_ARG;
    for (int i = 0; i < 3 * n; ++i) {
        const int bits = expert_bits[i / 3];
        if ((bits != 2 && bits != 4) || !codes[i] || !scales[i] || !aligned(scales[i], 2) ||
            !aligned(codes[i], bits == 4 ? 8 : 4))
            return SMOE_ERR_INVALID_ARG;
    }
    if (repack && tiles_bytes < smoe_repacked_bytes_mixed(d, f, n, expert_bits, group_size))
        return SMOE_ERR_WORKSPACE;
    if (!device_supported())
        return SMOE_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    int64_t off = 0;
    for (int e = 0; e < n; ++e) {
        const int bits = expert_bits[e];
        const int64_t gu = gateup_bytes(d, f, bits);
        for (int kind = 0; kind < 3; ++kind) {
            const int R = kind < 2 ? f : d, K = kind < 2 ? d : f;
            const cudaError_t ce =
                repack ? launch_repack(codes[3 * e + kind], scales[3 * e + kind], kind, R, K, bits,
                                       static_cast<uint8_t *>(tiles_out) + off, gu, s)
                       : launch_unpack(static_cast<const uint8_t *>(tiles_in) + off, kind, R, K,
                                       bits, gu, const_cast<uint8_t *>(codes[3 * e + kind]),
                                       const_cast<uint16_t *>(scales[3 * e + kind]), s);
            if (ce != cudaSuccess)
                return SMOE_ERR_CUDA;
        }
        off += expert_bytes(d, f, bits);
    }
    return SMOE_OK;
}

smoe_status smoe_repack_mixed(const uint8_t *const *codes_lsb, const uint16_t *const *scales_f16,
                              int32_t d_model, int32_t ffn_dim, int32_t n_experts,
                              const uint8_t *expert_bits, int group_size, void *tiles_out,
                              size_t tiles_bytes, void *cuda_stream)
{
    return mixed_pass(true, codes_lsb, scales_f16, d_model, ffn_dim, n_experts, expert_bits,
                      group_size, nullptr, tiles_out, tiles_bytes, cuda_stream);
}

smoe_status smoe_unpack_mixed(const void *tiles, int32_t d_model, int32_t ffn_dim,
                              int32_t n_experts, const uint8_t *expert_bits, int group_size,
                              uint8_t *const *codes_lsb, uint16_t *const *scales_f16,
                              void *cuda_stream)
{
    return mixed_pass(false, const_cast<const uint8_t *const *>(codes_lsb),
                      const_cast<const uint16_t *const *>(scales_f16), d_model, ffn_dim, n_experts,
                      expert_bits, group_size, tiles, nullptr, 0, cuda_stream);
}

size_t smoe_moe_workspace_bytes_mixed(const smoe_layer_desc *layer, int64_t num_tokens)
{
    if (!valid_layer(layer) || num_tokens < 0)
        return 0;
    return make_plan(layer, num_tokens, true).total;
}

smoe_status smoe_moe_forward_mixed(const smoe_layer_desc *layer, const uint8_t *expert_bits,
                                   const smoe_router_opts *opts, const void *x, smoe_dtype x_dtype,
                                   int64_t num_tokens, float *y, void *workspace,
                                   size_t workspace_bytes, int32_t *ids_out, float *w_out, int path,
                                   void *cuda_stream)
{
    if (!expert_bits ||
        (path != SMOE_PATH_AUTO && path != SMOE_PATH_STREAM && path != SMOE_PATH_GROUPED))
        return SMOE_ERR_INVALID_ARG;
    return forward_stages(layer, opts, x, x_dtype, num_tokens, y, workspace, workspace_bytes,
                          ids_out, w_out, 7, path, cuda_stream, expert_bits);
}

smoe_status smoe_moe_forward_stage_mixed(const smoe_layer_desc *layer, const uint8_t *expert_bits,
                                         const void *x, smoe_dtype x_dtype, int64_t num_tokens,
                                         float *y, void *workspace, size_t workspace_bytes,
                                         int32_t *ids_out, float *w_out, int stage,
                                         void *cuda_stream)
{
    if (!expert_bits || stage < 0 || stage > 2)
        return SMOE_ERR_INVALID_ARG;
    return forward_stages(layer, nullptr, x, x_dtype, num_tokens, y, workspace, workspace_bytes,
                          ids_out, w_out, 1 << stage, SMOE_PATH_AUTO, cuda_stream, expert_bits);
}

void smoe_debug_set_waits(long long poll_cycles, int stall_routing)
{
    g_wait_cycles.store(poll_cycles > 0 ? poll_cycles : kWaitCycles);
    g_tag_stall.store(stall_routing ? 1u : 0u);
}

smoe_status smoe_get_device_status(void *cuda_stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
        return SMOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess)
        return SMOE_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
        return SMOE_ERR_CUDA;
    if (v == 0)
        return SMOE_OK;
    return v == kStatusTimeout ? SMOE_ERR_TIMEOUT : SMOE_ERR_DEVICE_FAULT;
}

}  // extern "C"
