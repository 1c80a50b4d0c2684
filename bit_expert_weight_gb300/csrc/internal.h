// internal.h -- launchers and host helpers shared by the libsmoe translation
// units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "smoe.h"

namespace smoe {

// Leading bytes of the forward workspace that must hold zero when a forward
// starts (its counters and flags; 0 on invalid arguments).  Everything after
// them is written before it is read.
size_t moe_workspace_zero_bytes(const smoe_layer_desc *layer, int64_t num_tokens);

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();
// Compute capability major of the current device (cached per device).
int device_cc_major();
// Pointer to the device status word of the current device.
int *device_status_word();

void grid_fractions(float out[64]);

cudaError_t launch_quantize(const uint16_t *w, int64_t rows, int64_t cols, int bits,
                            uint8_t *codes, uint16_t *scales, cudaStream_t stream);

// kind: 0 gate, 1 up, 2 down.  R x K is the matrix shape ([f,d] or [d,f]).
cudaError_t launch_repack(const uint8_t *codes, const uint16_t *scales, int kind, int R, int K,
                          int bits, uint8_t *expert_base, int64_t gateup_bytes,
                          cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t *expert_base, int kind, int R, int K, int bits,
                          int64_t gateup_bytes, uint8_t *codes, uint16_t *scales,
                          cudaStream_t stream);

// ------------------------------------------------------------------ forward

// Pair = one expert applied to up to 8 tokens (the n columns of one mma).
constexpr int kPairCols = 8;
constexpr int kPairInts = 16;          // pair record: [expert, ncols, tok0..tok7, pad]
constexpr int kMaxBlocksPerPair = 64;  // counters per pair: f/64 and d/128 blocks
constexpr int kMaxExperts = 256;       // router / dispatch shared-memory bound

// Routable experts (a routing mask), bit e of w[e / 32]; all ones = none.
struct ExpertMask {
    uint32_t w[kMaxExperts / 32];
    int on;                            // 0: every expert routable
};
#define SMOE_MAX_TOPK_DEV 16
// Token counts up to this many combine inside the down kernel (last pair to
// finish a block); larger batches use a separate combine kernel.
constexpr int kFusedCombineMaxT = 8;

struct RouteArgs {
    const uint16_t *router_w;   // bf16 [E, d]
    const uint16_t *shared_gate; // nullable bf16 [d]
    const float *expert_bias;   // nullable [E]
    const void *x;              // [T, d]
    int x_bf16;
    int64_t T;
    int d, E, k, norm, bits;
    int has_shared;             // shared expert present
    int ksplit;                 // K split of the router GEMV
    int gateup_tiles_routed, gateup_tiles_shared;  // per pair
    // workspace
    float *partial;             // [ksplit][T][Epad]
    float *xsum;                // [T][d/64][2]
    int32_t *ids;               // [T][k]
    float *weights;             // [T][k]
    float *shared_w;            // [T]
    int32_t *ids_out;           // nullable
    float *w_out;               // nullable
    int32_t *pairs;             // pair table (see router.cu)
    int32_t *route_map;         // [T][k+1] -> pair*8 + col
    int32_t *meta;              // [0] pairs_routed, [1] pairs_total
    unsigned *tile_ctr;         // [ceil(T/8)]
    unsigned *done_ctr;         // [1]
    int *status;
    int max_pairs;
    int router_sigmoid;         // 1: per-expert sigmoid scores
    float rsf;                  // routed scaling factor
    ExpertMask mask;            // routable experts
    // grouped path (null: the streaming path's pair table is built instead)
    int32_t *grp_tilecnt;       // [T/8 tiles][E] selections per (token tile, expert)
};

cudaError_t launch_route_logits(const float *logits, int64_t T, int E, int k, int norm,
                                const float *bias, int router_sigmoid, float rsf,
                                const ExpertMask &mask, int32_t *ids, float *w,
                                cudaStream_t stream);
cudaError_t launch_router(const RouteArgs &a, cudaStream_t stream, bool pdl);
// Grouped path, bf16 tokens: routing of tiles of 8 tokens from logits
// [T][Epad] (plus the shared gate and the per-tile expert counts).
cudaError_t launch_route_tiles(const RouteArgs &a, const float *logits, int Epad,
                               cudaStream_t stream);

// The fused layer kernel (layer.cu): one CTA of 16 warps per SM.
constexpr int kMaxLayerCtasPerSm = 1;

struct LayerArgs {
    // layer
    const uint16_t *router_w;      // bf16 [E, d]
    const uint16_t *shared_gate;   // nullable bf16 [d]
    const float *expert_bias;      // nullable [E]
    const uint8_t *tiles_routed;   // bank base
    const uint8_t *tiles_shared;   // nullable
    int64_t expert_bytes_routed;   // stride between experts
    int64_t down_off_routed, down_off_shared;
    const void *x;                 // [T, d]
    int x_bf16;
    int64_t T;
    int d, f, fs, E, k, norm, bits, Epad, has_shared;
    int router_sigmoid;            // 1: per-expert sigmoid scores
    float rsf;                     // routed scaling factor
    ExpertMask mask;               // routable experts
    int do_route;                  // 1: phase R inside the kernel (T <= 8)
    int fused_combine;             // 1: combine inside the kernel (T <= 8)
    int max_pairs;
    // workspace: routing tables (written by the router kernel when do_route
    // is 0, by CTA 0 for the host otherwise)
    int32_t *ids;                  // [T][k]
    float *weights;                // [T][k]
    float *shared_w;               // [T]
    int32_t *ids_out;              // nullable
    float *w_out;                  // nullable
    int32_t *pairs;                // [max_pairs][kPairInts]
    int32_t *route_map;            // [T][k+1]
    int32_t *meta;                 // [0] routed pairs, [1] all pairs
    // Cross-CTA exchange by tagged words: a 64-bit word holds a 32-bit
    // payload (low half) and the launch's tag (high half), written by one
    // relaxed 64-bit store and polled with relaxed loads.  The tag of a
    // launch is *seq + 1; the kernel leaves it in *seq for the next launch.
    unsigned *seq;                 // [1], first word of the workspace
    unsigned long long *started;   // [CTAs] each CTA's start mark
    unsigned long long *logit_t;   // [CTAs][T][Epad] logits, one copy per CTA (routing inside)
    unsigned long long *h_t;       // [max_pairs][8][fmax] h: bf16 hi | bf16 lo << 16
    unsigned long long *part_t;    // [CTAs][2 slots][32 lanes][8] split gate/up unit sums
    unsigned long long *o_t;       // [max_pairs][8][d] down outputs (combine inside)
    float *o;                      // [max_pairs][8][d] down outputs (combine kernel)
    float *y;                      // [T, d]
    int *status;
    long long wait_cycles;         // bound of every tag poll
    unsigned tag_stall;            // testing: the logits poll waits for tag + tag_stall
    // mixed bit depth per routed expert (as in GroupedArgs): the kernel
    // instance for mixed banks takes each pair's depth from q4mask and the
    // expert's place in the bank from the depths before it
    int mixed;
    uint32_t q4mask[8];
};

// The expert-sorted grouped path (grouped.cu): segments = the routed experts,
// then the shared expert (all tokens); rows padded to 128 per segment.
struct GroupedArgs {
    const uint8_t *tiles_routed;   // bank base
    const uint8_t *tiles_shared;   // nullable
    int64_t expert_bytes_routed;
    int64_t down_off_shared;
    int64_t T;
    int d, f, fs, E, k, bits, has_shared;
    int32_t *seg;                  // [nseg+1] first rows, then [nseg] counts
    int32_t *rows_of;              // [T][k+1] sorted row of (token, slot); slot k: shared
    int64_t rows;                  // rows of xs, h and o
    const int32_t *ids;            // [T][k] routing
    int32_t *tilecnt;              // [ntiles][E] from the router; scanned in place
    int ntiles;                    // token tiles of the router (8 tokens each)
    unsigned *scan_ctr;            // zero-initialised arrival counter
    uint16_t *xs;                  // bf16 [rows][d]
    uint16_t *h;                   // bf16 [rows][hstride]
    int hstride;                   // max(f, fs)
    uint16_t *o;                   // bf16 [rows][d]: row weight x (W_down h)
    const float *w, *sw;           // routing weights [T][k], shared weights [T]
    float *roww;                   // [rows] the weight of each sorted row
    int *status;
    // mixed bit depth per routed expert: bit e of q4mask set = expert e is
    // Q4, clear = Q2; the bank holds the experts back to back at their own
    // sizes.  mixed = 0: every expert at `bits`, expert_bytes_routed apart.
    // The shared expert is at `bits` in both cases.
    int mixed;
    uint32_t q4mask[8];
};

// Token batches from this size on may take the grouped path (the workspace
// holds its buffers).
constexpr int64_t kGroupedMinT = 16;
int64_t grouped_max_rows(int64_t T, int E, int k, int has_shared);
// logits[T][Epad] = x Wr^T on the tensor cores (bf16 x, 16-byte aligned rows).
cudaError_t launch_tc_logits(const uint16_t *x, const uint16_t *router_w, int64_t T, int d, int E,
                             int Epad, float *logits, int *status, cudaStream_t stream);
// stage_mask: 1 sort + gather, 2 gate/up GEMM, 4 down GEMM + combine.
cudaError_t launch_grouped(const GroupedArgs &a, const void *x, int x_bf16, float *y, int stage_mask,
                           cudaStream_t stream);

int layer_grid_ctas_max();
cudaError_t launch_layer(const LayerArgs &a, cudaStream_t stream);
cudaError_t launch_combine(const LayerArgs &a, cudaStream_t stream);

}  // namespace smoe
