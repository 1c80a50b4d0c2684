/*
 * smoe.h -- C ABI of libsmoe.so: the SMOE group-quantised routed-expert MoE
 * layer forward on one NVIDIA GB300 (sm_103a).
 *
 * The method (page title, section):
 *   "SMOE Quantisation", Quantisation Levels / L2-MSE Scale Optimiser / Bit
 *     Packing / Decoding: Metal Kernel -- symmetric group-of-64 quantisation,
 *     Q4 w = (code - 7.5) / 7.5 * scale, Q2 w = (code - 1.5) / 1.5 * scale,
 *     codes packed LSB-first, one fp16 scale per group chosen by a 64-point
 *     MSE grid over linspace(0.1, 1.0, 64) * absmax.
 *   ".smoe Binary Format", File Header / Expert Blob Architecture -- the
 *     code stream and scale array of each sub-tensor (gate, up, down), and
 *     the header fields group_size, bits, d_model, ffn_dim.
 *   "Model Agnosticism", SmoeModelConfig -- d_model, ffn_dim,
 *     shared_expert_ffn_dim, max_experts_per_layer (router rows),
 *     norm_topk_prob, moe_top_k; routing width capped at 16; SiLU only.
 *   "CMF v2 -- Format Specification", 2.2 MoE -- softmax over all router
 *     logits (or per-expert sigmoid scores), top-k with ties to the lower
 *     index, selection-only expert_bias, optional renormalisation, a routed
 *     scaling factor, y = sum_e w_e FFN_e(x), shared expert weighted by
 *     sigmoid(shared_expert_gate . x) (else 1); each expert entry with its
 *     own dtype (per-expert depth: smoe_repack_mixed, smoe_moe_forward_mixed).
 *   "CMF v2 -- Format Specification", 5 -- routing masks (expert bitfields,
 *     LSB-first): smoe_router_opts.expert_mask.
 *   ".smoe Binary Format", Expert Table Entry / Tensor Descriptor / Arch
 *     Block "SARC" -- the vault reader (smoe_vault_*).
 *
 * Conventions (all entry points):
 *   - Every pointer argument is DEVICE memory owned by the caller unless the
 *     comment says "host".  The library allocates no device memory and never
 *     synchronises the stream, except smoe_get_device_status.
 *   - `cuda_stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - Arguments are validated synchronously on the host; on any error the
 *     call returns a negative smoe_status and launches nothing.
 *   - A launch failure returns SMOE_ERR_CUDA.  Faults detected on the device
 *     (an out-of-range expert id, a bounded wait that ran out) never trap:
 *     the kernel records a code in a device status word and skips the work;
 *     smoe_get_device_status reports and clears it.
 *   - Weights follow the HF orientation [out, in]: gate and up are
 *     [ffn_dim, d_model], down is [d_model, ffn_dim], the router is
 *     [num_experts, d_model]; all row-major.  Groups of 64 run along the
 *     input dimension (the row), so no group straddles two rows.
 */
#ifndef SMOE_H
#define SMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SMOE_OK = 0,
    SMOE_ERR_INVALID_ARG = -1,  /* a size, pointer or parameter is invalid   */
    SMOE_ERR_UNSUPPORTED = -2,  /* valid per the pages, not built (e.g. GPU)  */
    SMOE_ERR_WORKSPACE = -3,    /* workspace or output buffer too small       */
    SMOE_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed       */
    SMOE_ERR_DEVICE_FAULT = -5, /* a kernel recorded a device-side fault      */
    SMOE_ERR_TIMEOUT = -6       /* a kernel's bounded wait ran out            */
} smoe_status;

typedef enum { SMOE_F32 = 0, SMOE_BF16 = 1 } smoe_dtype;

/* Largest routing width ("Model Agnosticism", Expanding the Frontier: the
 * kernels cap routing at 16 experts per token). */
#define SMOE_MAX_TOP_K 16
/* The only group size the pages use (".smoe Binary Format", File Header:
 * group_size is always 64). */
#define SMOE_GROUP_SIZE 64

/* One MoE layer.  Every pointer is device memory owned by the caller. */
typedef struct {
    int32_t d_model;        /* hidden size d; multiple of 128, <= 4096        */
    int32_t ffn_dim;        /* routed-expert intermediate size f; multiple of
                               64, <= 2048 (one down strip per ring stage)    */
    int32_t num_experts;    /* E = router rows (max_experts_per_layer)        */
    int32_t top_k;          /* k, 1..16 and <= E                              */
    int32_t norm_topk_prob; /* nonzero: renormalise the k selected weights    */
    int32_t bits;           /* 4 (SMOE-Q4) or 2 (SMOE-Q2)                     */
    int32_t group_size;     /* must be 64                                     */
    const void *router_w;   /* bf16 [E, d]                                    */
    const float *expert_bias; /* nullable fp32 [E]: added to the logits for
                                 top-k selection only, never to the weights */
    const void *expert_tiles; /* the bank of E experts written by smoe_repack */
    const void *shared_tiles; /* nullable: the shared expert, written by
                                 smoe_repack with n_experts = 1 and
                                 ffn_dim = shared_ffn_dim                     */
    int32_t shared_ffn_dim;   /* 0 = no shared expert; else multiple of 64,
                                 <= 2048                                      */
    const void *shared_gate_w; /* nullable bf16 [d]: shared-expert weight is
                                  sigmoid(shared_gate_w . x), else 1          */
} smoe_layer_desc;

/* Human-readable name of a status code (static string, never NULL). */
const char *smoe_status_string(smoe_status s);

/* ---------------------------------------------------------------- sizes */

/* Code bytes of one rows x cols sub-tensor: ceil(rows*cols*bits/8)
 * (".smoe Binary Format", Expert Blob Architecture).  0 on bad arguments. */
size_t smoe_stream_bytes(int64_t rows, int64_t cols, int bits);

/* fp16 scale bytes of one sub-tensor: ceil(rows*cols/group_size)*2.  0 on
 * bad arguments. */
size_t smoe_scales_bytes(int64_t rows, int64_t cols, int group_size);

/* Bytes of one expert in the device tile layout (gate+up tiles then down
 * tiles).  The layout keeps each 16-row x 64-column tile's codes and its 16
 * fp16 scales together (544 B for Q4, 288 B for Q2), so the per-expert size
 * equals the code+scale bytes of the pages' blob exactly.  0 on bad args. */
size_t smoe_expert_tiles_bytes(int32_t d_model, int32_t ffn_dim, int bits, int group_size);

/* Bytes of a bank of n_experts experts = n_experts * smoe_expert_tiles_bytes. */
size_t smoe_repacked_bytes(int32_t d_model, int32_t ffn_dim, int32_t n_experts, int bits,
                           int group_size);

/* Bytes of a bank whose experts each have their own depth ("CMF v2", 2.2
 * MoE: every expert declares its own dtype): the sum of
 * smoe_expert_tiles_bytes(d, f, expert_bits[e], 64).  expert_bits is a HOST
 * array of n_experts entries, each 2 or 4.  0 on bad args. */
size_t smoe_repacked_bytes_mixed(int32_t d_model, int32_t ffn_dim, int32_t n_experts,
                                 const uint8_t *expert_bits, int group_size);

/* ----------------------------------------------------------- quantiser */

/* L2-MSE grid-search quantisation of a bf16 [rows, cols] tensor
 * ("SMOE Quantisation", L2-MSE Scale Optimiser and Bit Packing).
 * Per group of 64 consecutive elements of the row-major tensor: absmax a;
 * candidates s_j = fl32(fl32(linspace(0.1,1,64)[j]) * a); codes
 * clamp(rint(((w / s) * L) + L), 0, 2L) in fp32 (L = 7.5 or 1.5); the
 * candidate with the least reconstruction MSE wins (the first on exact
 * ties); an all-zero group gets scale 0 and code round(L).
 *   w_bf16      device, bf16 [rows, cols], finite values
 *   cols        multiple of 64
 *   codes_lsb   device, out: smoe_stream_bytes(rows, cols, bits) bytes,
 *               LSB-first (Q4: 2 codes/byte, Q2: 4 codes/byte)
 *   scales_f16  device, out: rows*cols/64 fp16 scales (RNE of the fp32
 *               winning candidate)
 * Errors: SMOE_ERR_INVALID_ARG (bits not 2/4, group_size != 64, cols % 64,
 * rows < 0, null pointer), SMOE_ERR_CUDA. */
smoe_status smoe_quantize(const void *w_bf16, int64_t rows, int64_t cols, int bits,
                          int group_size, uint8_t *codes_lsb, uint16_t *scales_f16,
                          void *cuda_stream);

/* -------------------------------------------------------- repack/unpack */

/* Repack E experts from the pages' LSB-first code streams and fp16 scale
 * arrays (".smoe Binary Format", Expert Blob Architecture) into the device
 * tile layout read by smoe_moe_forward.
 *   codes_lsb   HOST array of 3*n_experts DEVICE pointers, order
 *               (gate, up, down) per expert; gate/up are [ffn_dim, d_model]
 *               streams, down is [d_model, ffn_dim]
 *   scales_f16  HOST array of 3*n_experts DEVICE pointers, same order
 *   tiles_out   device, smoe_repacked_bytes(...) bytes, 16-byte aligned
 * The result is a byte permutation: smoe_unpack restores every byte.
 * Errors: SMOE_ERR_INVALID_ARG (shape not d % 128 == 0 and f % 64 == 0,
 * bits, group_size, null or misaligned pointer), SMOE_ERR_WORKSPACE
 * (tiles_bytes too small), SMOE_ERR_CUDA. */
smoe_status smoe_repack(const uint8_t *const *codes_lsb, const uint16_t *const *scales_f16,
                        int32_t d_model, int32_t ffn_dim, int32_t n_experts, int bits,
                        int group_size, void *tiles_out, size_t tiles_bytes, void *cuda_stream);

/* Exact inverse of smoe_repack: writes the LSB-first streams and fp16 scale
 * arrays back.  Same argument conventions (host arrays of device pointers). */
smoe_status smoe_unpack(const void *tiles, int32_t d_model, int32_t ffn_dim, int32_t n_experts,
                        int bits, int group_size, uint8_t *const *codes_lsb,
                        uint16_t *const *scales_f16, void *cuda_stream);

/* smoe_repack of a bank whose experts each have their own depth:
 * expert_bits is a HOST array of n_experts entries (2 = SMOE-Q2, 4 =
 * SMOE-Q4); expert e's streams are at its depth and its tiles follow
 * expert e-1's, at offset sum_{j<e} smoe_expert_tiles_bytes(d, f,
 * expert_bits[j], 64).  tiles_out: smoe_repacked_bytes_mixed(...) bytes.
 * Errors as smoe_repack (an entry that is not 2 or 4: SMOE_ERR_INVALID_ARG). */
smoe_status smoe_repack_mixed(const uint8_t *const *codes_lsb, const uint16_t *const *scales_f16,
                              int32_t d_model, int32_t ffn_dim, int32_t n_experts,
                              const uint8_t *expert_bits, int group_size, void *tiles_out,
                              size_t tiles_bytes, void *cuda_stream);

/* Exact inverse of smoe_repack_mixed. */
smoe_status smoe_unpack_mixed(const void *tiles, int32_t d_model, int32_t ffn_dim,
                              int32_t n_experts, const uint8_t *expert_bits, int group_size,
                              uint8_t *const *codes_lsb, uint16_t *const *scales_f16,
                              void *cuda_stream);

/* ------------------------------------------------------------ .smoe vault */

/* The pages' binary vault (".smoe Binary Format"): a 64-byte file header, an
 * expert table (48-byte entries, sorted by layer then expert), three 44-byte
 * tensor descriptors per entry (gate, up, down), in version 2 a 128-byte
 * arch block "SARC" at header.reserved_ext, then 16 KB-aligned expert blobs
 * [gate codes][gate fp16 scales][up codes][up scales][down codes][down
 * scales][padding].  All integers little-endian, all offsets from the start
 * of the file.  Here the vault is the input of smoe_repack: nothing is
 * streamed from disk.
 *
 * The functions below read the metadata from a HOST buffer `meta` holding at
 * least the file's first header.data_offset bytes (header, table,
 * descriptors, arch block); `file_bytes` is the size of the whole file, used
 * to bound the blob extents.  They validate what the page fixes and refuse
 * the vault otherwise (SMOE_ERR_INVALID_ARG): magic 53 4D 4F 45 DE EA 00 01,
 * version 1 or 2, table_offset 64, data_offset 16 KB-aligned and past the
 * descriptors, group_size 64, bits 2 or 4; for version 2 an arch block with
 * magic "SARC", block_version 1, block_size 128, activation 0 (SiLU),
 * moe_top_k <= 16, head_dim <= 256, num_heads divisible by num_kv_heads,
 * zero reserved bytes; table entries in (layer, expert) order, group_size
 * 64, zero reserved bytes, 16 KB-aligned blobs inside the file, raw_size <=
 * padded_size; descriptors typed gate, up, down in order, ndim 2, zero
 * reserved bytes, packed_size = ceil(rows*cols*bits/8), scales_size =
 * ceil(rows*cols/64)*2, both inside the blob's raw bytes, num_groups = the
 * three tensors' groups.  Nothing is allocated; no GPU is used. */
typedef struct {
    uint32_t version, num_moe_layers, max_experts_per_layer, total_experts;
    uint64_t table_offset, data_offset;
    uint32_t group_size, bits, d_model, vocab_size;
    uint32_t ffn_dim;        /* header field: dense/shared FFN dimension */
    uint32_t reserved_ext;   /* v2: byte offset of the arch block */
    int32_t has_arch;        /* 1 for version 2 */
    uint32_t arch_flags;     /* bit 0 norm_topk_prob, bit 1 has_qk_norm, bit 2 has_dense_layer_0 */
    float rope_theta;
    uint32_t num_heads, num_kv_heads, head_dim, moe_top_k, moe_ffn_dim, dense_ffn_dim,
        shared_expert_ffn_dim, activation, num_hidden_layers;
    float rms_norm_eps;
    char model_type[25];     /* NUL-terminated */
} smoe_vault_info;

typedef struct {
    uint32_t rows, cols;
    uint64_t packed_offset, packed_size, scales_offset, scales_size;  /* within the blob */
} smoe_vault_tensor;

typedef struct {
    uint32_t layer_id, expert_id;
    uint64_t byte_offset, raw_size, padded_size, num_groups;
    smoe_vault_tensor tensor[3];  /* gate, up, down */
} smoe_vault_expert;

/* Parse and validate the vault metadata; fills *info.  Errors:
 * SMOE_ERR_INVALID_ARG (null pointer, short buffer, any rule above). */
smoe_status smoe_vault_parse(const void *meta, size_t meta_bytes, uint64_t file_bytes,
                             smoe_vault_info *info);

/* Locate expert (layer, expert) through the table and its descriptors.
 * SMOE_ERR_INVALID_ARG also when the vault has no such entry. */
smoe_status smoe_vault_find_expert(const void *meta, size_t meta_bytes, uint64_t file_bytes,
                                   uint32_t layer, uint32_t expert, smoe_vault_expert *out);

/* smoe_repack of one MoE layer straight from a vault: experts 0 ..
 * num_experts - 1 of `layer`, each found through the table and its
 * descriptors (never a fixed stride), their codes and scales read from
 * `vault_dev`, a DEVICE copy of the whole file (file_bytes bytes, 16-byte
 * aligned).  d_model is the header's; the expert ffn_dim is the descriptors'
 * gate rows, which must be equal for every expert of the layer (and equal
 * the arch block's moe_ffn_dim in version 2).  Writes the same tiles as
 * smoe_repack with the same streams, into tiles_out (device,
 * smoe_repacked_bytes(d, f, num_experts, bits, 64) bytes).  Errors:
 * SMOE_ERR_INVALID_ARG (vault rules, missing expert, mismatched shapes, a
 * stream not aligned for the repack kernel), SMOE_ERR_WORKSPACE (tiles_bytes
 * too small), SMOE_ERR_UNSUPPORTED (device), SMOE_ERR_CUDA. */
smoe_status smoe_vault_repack_layer(const void *meta, size_t meta_bytes, const void *vault_dev,
                                    uint64_t file_bytes, uint32_t layer, uint32_t num_experts,
                                    void *tiles_out, size_t tiles_bytes, void *cuda_stream);

/* ---------------------------------------------------------------- route */

/* Top-k routing from given fp32 logits ("CMF v2", 2.2 MoE).
 *   logits       device fp32 [T, E]
 *   expert_bias  nullable device fp32 [E]; the selection key is
 *                fl32(logit + bias), the weights never see the bias
 *   ids          device out int32 [T, k], rank order (largest key first,
 *                equal keys: lower expert index first)
 *   weights      device out fp32 [T, k]: softmax over all E logits at the
 *                selected experts, divided by their sum if norm_topk_prob
 * Errors: SMOE_ERR_INVALID_ARG (T < 0, E < 1, k < 1, k > 16, k > E, null
 * pointer), SMOE_ERR_CUDA. */
smoe_status smoe_route_from_logits(const float *logits, int64_t T, int32_t E, int32_t k,
                                   int norm_topk_prob, const float *expert_bias, int32_t *ids,
                                   float *weights, void *cuda_stream);

/* Router variants ("CMF v2 -- Format Specification", 2.2 MoE) and routing
 * masks (same page, 5: expert bitfields).  Passing NULL where an entry point
 * takes options means the defaults: softmax, factor 1, no mask (what
 * smoe_route_from_logits and smoe_moe_forward do).
 *   router_sigmoid         0: softmax over all E logits; 1: each expert
 *                          scored by sigmoid(logit) on its own
 *   routed_scaling_factor  multiplies the selected weights after the
 *                          optional renormalisation; finite and > 0
 *   expert_mask            nullable HOST bitfield of ceil(E/8) bytes,
 *                          LSB-first: bit e set = expert e routable.  The
 *                          selection runs over the routable experts only
 *                          and the softmax normalises over them; the tail
 *                          bits beyond E must be zero and at least top_k
 *                          experts routable (else SMOE_ERR_INVALID_ARG).
 *                          Read during the call; not kept.
 * Selection key: the logit without a bias; with an expert_bias, logit + bias
 * (softmax) or fl32(sigmoid(logit)) + bias (sigmoid); ties to the lower
 * expert index.  The shared expert's weight is not scaled. */
typedef struct {
    int32_t router_sigmoid;
    float routed_scaling_factor;
    const uint8_t *expert_mask;
} smoe_router_opts;

/* smoe_route_from_logits with router options (opts nullable).  Errors as
 * smoe_route_from_logits, plus SMOE_ERR_INVALID_ARG for a factor that is not
 * finite and positive. */
smoe_status smoe_route_from_logits_ex(const float *logits, int64_t T, int32_t E, int32_t k,
                                      int norm_topk_prob, const float *expert_bias,
                                      const smoe_router_opts *opts, int32_t *ids,
                                      float *weights, void *cuda_stream);

/* ------------------------------------------------------------- forward */

/* Workspace bytes smoe_moe_forward needs for this layer and token count
 * (0 on invalid arguments). */
size_t smoe_moe_workspace_bytes(const smoe_layer_desc *layer, int64_t num_tokens);

/* Zero a workspace.  Required once after allocation, and again after a call
 * that returned an error; the forward leaves its counters at zero itself. */
smoe_status smoe_moe_workspace_init(void *workspace, size_t workspace_bytes, void *cuda_stream);

/* MoE layer forward for T tokens:
 *   logits = x Wr^T;  top-k routing (see smoe_route_from_logits);
 *   per selected expert: h = SiLU(W_gate x) * (W_up x), o = W_down h, with
 *   W decoded as (code - L) / L * scale (never written to global memory);
 *   y = sum_j w_j o_j (rank order, deterministic) + shared expert.
 * Two execution paths compute this ("Model Agnosticism"; "CMF v2", 2.2 MoE):
 *   streaming  codes decoded in registers, fp32 accumulation with the
 *              activations split into bf16 hi + lo (fp32-accurate); taken
 *              for small batches
 *   grouped    tokens sorted by expert, weights decoded to bf16 in shared
 *              memory, tensor-core GEMMs (tcgen05) with bf16 activations and
 *              bf16 h, fp32 accumulation, each expert's output scaled by its
 *              routing weight and rounded to bf16 before the fp32 sum over
 *              the token's experts; taken for bf16 tokens when T >= 16 and
 *              T * top_k >= 16 * num_experts (smoe_moe_path_dtype tells
 *              which).  fp32 tokens always take the streaming path, so that
 *              their accuracy is never reduced to the bf16 operands'.
 * Both are deterministic: the same inputs give the same bits on every call.
 *   x           device [T, d_model], fp32 or bf16 (x_dtype)
 *   y           device out fp32 [T, d_model]
 *   workspace   device, >= smoe_moe_workspace_bytes, 256-byte aligned,
 *               zeroed once by smoe_moe_workspace_init
 *   ids_out     nullable device out int32 [T, k]
 *   w_out       nullable device out fp32 [T, k]
 * The whole layer is enqueued on cuda_stream; nothing is synchronised.
 * Errors: SMOE_ERR_INVALID_ARG (layer fields, T < 0, null pointer),
 * SMOE_ERR_UNSUPPORTED (device is not a Blackwell sm_10x part),
 * SMOE_ERR_WORKSPACE, SMOE_ERR_CUDA. */
smoe_status smoe_moe_forward(const smoe_layer_desc *layer, const void *x, smoe_dtype x_dtype,
                             int64_t num_tokens, float *y, void *workspace,
                             size_t workspace_bytes, int32_t *ids_out, float *w_out,
                             void *cuda_stream);

/* Execution paths of the forward. */
#define SMOE_PATH_AUTO 0
#define SMOE_PATH_STREAM 1
#define SMOE_PATH_GROUPED 2

/* smoe_moe_forward with the execution path chosen by the caller (path
 * SMOE_PATH_AUTO is smoe_moe_forward itself).  The grouped path needs
 * num_tokens >= 16 (the workspace of smaller batches has no room for it) and
 * bf16 tokens (it would round fp32 ones to bf16): otherwise
 * SMOE_ERR_UNSUPPORTED, nothing enqueued.  Same arguments and errors as
 * smoe_moe_forward, plus SMOE_ERR_INVALID_ARG for an unknown path. */
smoe_status smoe_moe_forward_path(const smoe_layer_desc *layer, const void *x, smoe_dtype x_dtype,
                                  int64_t num_tokens, float *y, void *workspace,
                                  size_t workspace_bytes, int32_t *ids_out, float *w_out, int path,
                                  void *cuda_stream);

/* smoe_moe_forward_path with router options (opts nullable; see
 * smoe_router_opts).  Same arguments and errors, plus SMOE_ERR_INVALID_ARG
 * for a scaling factor that is not finite and positive. */
smoe_status smoe_moe_forward_ex(const smoe_layer_desc *layer, const smoe_router_opts *opts,
                                const void *x, smoe_dtype x_dtype, int64_t num_tokens, float *y,
                                void *workspace, size_t workspace_bytes, int32_t *ids_out,
                                float *w_out, int path, void *cuda_stream);

/* Workspace bytes of smoe_moe_forward_mixed for this layer and token count
 * (0 on invalid arguments). */
size_t smoe_moe_workspace_bytes_mixed(const smoe_layer_desc *layer, int64_t num_tokens);

/* The forward of a layer whose routed experts each have their own depth
 * (some SMOE-Q2, some SMOE-Q4).  layer->expert_tiles is a bank written by
 * smoe_repack_mixed with the same expert_bits (HOST array of num_experts
 * entries, each 2 or 4; read during the call, not kept); layer->bits is the
 * shared expert's depth.  Each expert decodes its own levels (L = 7.5 or
 * 1.5); otherwise the same computation as smoe_moe_forward_ex, on the same
 * two paths, chosen the same way (path as in smoe_moe_forward_path; the
 * grouped path also below 16 tokens):
 *   streaming  one launch; each (expert, token block) unit streams and
 *              decodes its tiles at its expert's depth
 *   grouped    one gate/up and one down GEMM launch per depth present, each
 *              taking the experts of its own depth
 * workspace: >= smoe_moe_workspace_bytes_mixed.  Errors as
 * smoe_moe_forward_ex (expert_bits null or an entry not 2 or 4:
 * SMOE_ERR_INVALID_ARG). */
smoe_status smoe_moe_forward_mixed(const smoe_layer_desc *layer, const uint8_t *expert_bits,
                                   const smoe_router_opts *opts, const void *x, smoe_dtype x_dtype,
                                   int64_t num_tokens, float *y, void *workspace,
                                   size_t workspace_bytes, int32_t *ids_out, float *w_out, int path,
                                   void *cuda_stream);

/* smoe_moe_forward_mixed (without router options, path SMOE_PATH_AUTO) one
 * launch stage at a time, as smoe_moe_forward_stage. */
smoe_status smoe_moe_forward_stage_mixed(const smoe_layer_desc *layer, const uint8_t *expert_bits,
                                         const void *x, smoe_dtype x_dtype, int64_t num_tokens,
                                         float *y, void *workspace, size_t workspace_bytes,
                                         int32_t *ids_out, float *w_out, int stage,
                                         void *cuda_stream);

/* The path smoe_moe_forward takes for this layer and token count with bf16
 * tokens (SMOE_PATH_STREAM or SMOE_PATH_GROUPED), or -1 on invalid
 * arguments; smoe_moe_path_dtype(layer, num_tokens, SMOE_BF16). */
int smoe_moe_path(const smoe_layer_desc *layer, int64_t num_tokens);

/* The path smoe_moe_forward takes for this layer, token count and token
 * dtype (fp32 tokens: always SMOE_PATH_STREAM), or -1 on invalid
 * arguments. */
int smoe_moe_path_dtype(const smoe_layer_desc *layer, int64_t num_tokens, smoe_dtype x_dtype);

/* The same forward as smoe_moe_forward, one launch stage at a time, so that
 * a caller can put its own work or timing events between the stages.  The
 * stages follow the path smoe_moe_forward takes (smoe_moe_path):
 *   streaming path
 *     stage 0  router GEMV, softmax, top-k, renormalisation, dispatch
 *     stage 1  fused dequant gate/up GEMV + SiLU(gate) * up
 *     stage 2  fused dequant down GEMV + routing-weighted combine into y
 *   grouped path
 *     stage 0  router logits, softmax, top-k, renormalisation, sort of the
 *              selections by expert, gather of the tokens as bf16 rows
 *     stage 1  gate/up grouped GEMM (tensor cores) + SiLU(gate) * up
 *     stage 2  down grouped GEMM (tensor cores) + routing-weighted combine
 * Calling stages 0, 1, 2 in order on one stream with the same arguments and
 * workspace is exactly smoe_moe_forward.  Same arguments and errors, plus
 * SMOE_ERR_INVALID_ARG for a stage outside 0..2. */
smoe_status smoe_moe_forward_stage(const smoe_layer_desc *layer, const void *x,
                                   smoe_dtype x_dtype, int64_t num_tokens, float *y,
                                   void *workspace, size_t workspace_bytes, int32_t *ids_out,
                                   float *w_out, int stage, void *cuda_stream);

/* ------------------------------------------------- forward, no allocation */

/* Bytes of the device array that smoe_moe_forward_noalloc uses as its
 * workspace: 32 MiB, a fixed part of the library image on each device.  It
 * holds the workspace of a decode batch of up to 8 tokens for layers up to
 * d_model 4096, ffn_dim 1536, 256 experts and top_k 8;
 * smoe_moe_workspace_bytes(layer, T) <= SMOE_NOALLOC_SCRATCH_BYTES tells
 * whether another shape or batch fits. */
#define SMOE_NOALLOC_SCRATCH_BYTES (32u << 20)

/* smoe_moe_forward without a caller-supplied workspace.  The pages describe
 * no counterpart of this entry point: it exists for library users only.
 *
 * Who needs it: smoe_moe_forward wants a device workspace that the caller
 * allocates.  Some callers cannot do that on the path where they run the
 * layer: a plug-in handed device pointers by a host framework that owns all
 * device memory through its own pool and offers it no allocator, or a
 * serving loop that must not call cudaMalloc or cudaFree, since those can
 * block on or synchronise the whole device.  This entry point allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.  Its
 * workspace is a file-scope device array of SMOE_NOALLOC_SCRATCH_BYTES
 * bytes that the CUDA driver reserves when libsmoe.so's module is loaded
 * on a device.
 *
 * Arguments, outputs and results are those of smoe_moe_forward (bit for bit
 * the same y, ids_out and w_out for the same inputs).  Each call first
 * clears the workspace counters that must start at zero (a
 * cudaMemsetAsync on cuda_stream), then enqueues the forward.
 *
 * Restrictions:
 *   - All calls on one device share the one array.  Calls whose work can
 *     overlap on the device (different streams without an ordering between
 *     them, or several host threads) race on it and give wrong results.
 *     Issue them on one stream, or order them with events.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it with
 *     the device's current context; a later call made in another context of
 *     that device (after cudaDeviceReset, say) looks the address up again.
 *     Make the first call in each context before any stream capture begins.
 *   - layer->expert_tiles must be a single-depth bank from smoe_repack: the
 *     descriptor carries no per-expert depths, so a bank from
 *     smoe_repack_mixed would be read as a uniform bank at layer->bits (past
 *     the end of the caller's allocation).  Mixed-depth layers need
 *     smoe_moe_forward_mixed with a workspace the caller allocates.
 *
 * Errors: those of smoe_moe_forward, and SMOE_ERR_WORKSPACE when
 * smoe_moe_workspace_bytes(layer, num_tokens) exceeds
 * SMOE_NOALLOC_SCRATCH_BYTES (the call then enqueues nothing; use
 * smoe_moe_forward with a workspace of your own, or fewer tokens). */
smoe_status smoe_moe_forward_noalloc(const smoe_layer_desc *layer, const void *x,
                                     smoe_dtype x_dtype, int64_t num_tokens, float *y,
                                     int32_t *ids_out, float *w_out, void *cuda_stream);

/* Testing only: make the layer kernel's bounded waits short and, if
 * stall_routing is nonzero, make its routing step wait for logits that no
 * CTA ever writes.  The layer kernel (the streaming path) hands every value
 * between CTAs over as a tagged word and each reader polls its words for the
 * launch's tag; poll_cycles bounds each such poll in SM cycles (<= 0: the
 * default, about two seconds).  With the stall, each CTA gives up after
 * poll_cycles, records SMOE_ERR_TIMEOUT in the device status word, skips the
 * rest of the layer (waits included) and returns; the next launch is not
 * affected, so a test can check that a wait which runs out ends the launch
 * with a status the host reads while the context stays usable.  Applies to
 * forwards enqueued after the call, in this process; a test restores the
 * defaults with smoe_debug_set_waits(0, 0).  No counterpart in the pages. */
void smoe_debug_set_waits(long long poll_cycles, int stall_routing);

/* Synchronise cuda_stream, then read and clear the device status word of the
 * current device.  Returns SMOE_OK, SMOE_ERR_DEVICE_FAULT, SMOE_ERR_TIMEOUT
 * or SMOE_ERR_CUDA. */
smoe_status smoe_get_device_status(void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SMOE_H */
