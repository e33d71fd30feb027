/*
 * gbmoe.h -- C ABI of the single-GPU fused Mixture-of-Experts FFN forward
 * (routing, top-k, expert-sorted permutation, SwiGLU grouped GEMMs, top-k
 * weight-and-reduce) for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named *device* are device (HBM) pointers owned by the caller;
 *    the library never allocates, frees or copies device memory on its own
 *    and never synchronises the stream (except moe_read_error, which says
 *    so).  All work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and is asynchronous.
 *  - Tensors are dense, row-major, last dimension contiguous.  "bf16" data
 *    is IEEE bfloat16 passed as `const void*` (2-byte elements); every bf16
 *    or fp32 base pointer must be 16-byte aligned.
 *  - Validation of sizes, enums and pointers happens on the host before any
 *    launch and returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE_TOO_SMALL without touching the GPU.  Errors that only
 *    the GPU can see (an expert id out of range, a pipeline wait that ran
 *    out of time) are written to a device error word and read back with
 *    moe_read_error; kernels never trap.
 *  - M == 0 (or an empty batched layout) is a valid no-op returning MOE_OK.
 *  - moe_last_error_detail() returns a short text for the last failing call
 *    on the calling thread.
 *
 * Citations are to the source pages by title and section.
 */
#ifndef GBMOE_H
#define GBMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GBMOE_ABI_VERSION 1

#if defined(__GNUC__)
#define GBMOE_API __attribute__((visibility("default")))
#else
#define GBMOE_API
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,
  MOE_ERR_BAD_EXPERT_ID = 4, /* device-detected: topk_ids / counts out of range */
  MOE_ERR_TIMEOUT = 5,       /* device-detected: a bounded pipeline wait gave up */
  MOE_ERR_CUDA = 6,          /* a CUDA runtime/driver call failed */
  MOE_ERR_NO_DEVICE = 7      /* no usable sm_103 device */
} moe_status_t;

typedef enum { MOE_ROUTE_SOFTMAX = 0, MOE_ROUTE_SIGMOID = 1 } moe_routing_t;

/* Where the top-k weight multiply and the k-sum happen ("Fused MoE Modular
 * Kernel" page, TopKWeightAndReduce section).  Both choices apply bias and
 * routing weight in the down-projection (GEMM2) epilogue.
 * SEPARATE: the epilogue writes one fp32 row per routed item in expert-sorted
 *   order (TMA tensor stores); a vectorised kernel sums each token's k rows
 *   through the inverse permutation and casts to bf16.
 * EPILOGUE_ATOMIC: the epilogue adds each weighted row into the token's fp32
 *   accumulator row with vector atomics (resolved in L2); a cast kernel
 *   writes bf16.
 * AUTO: SEPARATE (faster on every measured workload). */
typedef enum {
  MOE_REDUCE_AUTO = 0,
  MOE_REDUCE_EPILOGUE_ATOMIC = 1,
  MOE_REDUCE_SEPARATE = 2
} moe_reduce_t;

/* GEMM row block: experts' item lists are padded to a multiple of this. */
#define MOE_BLOCK_M 128

/* ---------------------------------------------------------------- route --
 * moe_route: router scores -> top-k experts and weights per token.
 * Defines: "MindIE-SD Fused MoE" page, parameter table (routing_method,
 * renormalize, k_group, group_count, group_select_mode,
 * routed_scaling_factor) and routing section; "FlagGems fused_moe.py
 * analysis", section 1.1 (p_t = softmax(s_t), S_t = TopK(p_t, k)).
 *
 *  router_logits  device fp32 [M, E]
 *  routing_method MOE_ROUTE_SOFTMAX (softmax over E) or MOE_ROUTE_SIGMOID
 *  renormalize    softmax only: divide the k selected weights by their sum.
 *                 Sigmoid weights are always divided by their sum.
 *  group_count    experts split into group_count equal contiguous groups
 *                 (E % group_count == 0); 1 = no grouping
 *  k_group        groups kept, 1 <= k_group <= group_count
 *  group_select_mode 0: group score = max score in the group;
 *                 1: sum of the group's two largest scores (needs >= 2
 *                 experts per group)
 *  top_k          1 <= top_k <= k_group * E / group_count, top_k <= 64
 *  routed_scaling_factor  multiplies every output weight (after renormalising)
 *  topk_weights   device fp32 [M, top_k] out
 *  topk_ids       device int32 [M, top_k] out, by descending score, ties to
 *                 the lower expert id (and groups' ties to the lower group)
 * Limits: 1 <= E <= 1024.
 */
GBMOE_API moe_status_t moe_route(const float* router_logits, int64_t M, int32_t E, int32_t top_k,
                       int32_t routing_method, int32_t renormalize, int32_t k_group,
                       int32_t group_count, int32_t group_select_mode,
                       float routed_scaling_factor, float* topk_weights, int32_t* topk_ids,
                       moe_stream_t stream);

/* moe_route_bf16: moe_route with bf16 router logits (the "MindIE-SD Fused
 * MoE" page accepts bf16 router logits).  Each logit is widened exactly to
 * fp32 first; everything else is as moe_route. */
GBMOE_API moe_status_t moe_route_bf16(const void* router_logits, int64_t M, int32_t E,
                                      int32_t top_k, int32_t routing_method, int32_t renormalize,
                                      int32_t k_group, int32_t group_count,
                                      int32_t group_select_mode, float routed_scaling_factor,
                                      float* topk_weights, int32_t* topk_ids,
                                      moe_stream_t stream);

/* ---------------------------------------------------------- router GEMM --
 * moe_router_logits: the router scores ahead of routing,
 *   s_t = W_g^T x_t + b_g        ("fused_moe.py 分析" (FlagDoc), section 1.1)
 * with fp32 accumulation: for few experts (E <= 32, H % 256 == 0, W_g up to
 * 160 KB as fp32) a warp-per-token kernel with W_g in shared memory,
 * otherwise the tensor-core grouped GEMM with one "expert".
 *  hidden  device bf16 [M, H];  w_gate device bf16 [H, E] (W_g, d x E);
 *  b_gate  device bf16 [E] or NULL;  logits device fp32 [M, E] out
 * Limits: H % 8 == 0; E % 8 == 0 (16-byte weight rows; else
 * MOE_ERR_UNSUPPORTED), 1 <= E <= 1024.
 */
GBMOE_API moe_status_t moe_router_logits(const void* hidden, const void* w_gate,
                                         const void* b_gate, int64_t M, int32_t H, int32_t E,
                                         float* logits, moe_stream_t stream);

/* ---------------------------------------------------------------- align --
 * moe_align: expert-sorted, block-padded permutation of the routed items.
 * Defines: "FlagGems fused_moe.py analysis", section moe_align_block_size
 * (flatten (token, slot) items, sort by expert, pad each expert's count to
 * BLOCK_SIZE_M; sorted_token_ids, per-block expert ids,
 * num_tokens_post_padded).
 *
 *  topk_ids           device int32 [M, top_k]; item index r = t * top_k + j
 *  block_m            padding block, 1 <= block_m <= 1024
 *  sorted_token_ids   device int32 [moe_align_capacity(...)] out: expert e's
 *                     items in ascending r at [expert_offsets[e],
 *                     expert_offsets[e] + expert_num_tokens[e]), then the
 *                     sentinel R = M * top_k up to expert_offsets[e + 1];
 *                     entries past expert_offsets[E] are left untouched
 *  expert_offsets     device int32 [E + 1] out: exclusive scan of the padded
 *                     counts; expert_offsets[E] = num_tokens_post_padded
 *  expert_num_tokens  device int32 [E] out
 *  block_expert_ids   device int32 [moe_align_capacity(...) / block_m] out:
 *                     expert of each block_m-row block, -1 past the last
 *  scratch            device, moe_align_scratch_size(...) bytes, any content
 *  error_word         device int32 or NULL: set to MOE_ERR_BAD_EXPERT_ID if
 *                     an id is outside [0, E) (such items are dropped)
 */
GBMOE_API size_t moe_align_capacity(int64_t M, int32_t top_k, int32_t E, int32_t block_m);
GBMOE_API size_t moe_align_scratch_size(int64_t M, int32_t top_k, int32_t E);
GBMOE_API moe_status_t moe_align(const int32_t* topk_ids, int64_t M, int32_t top_k, int32_t E,
                       int32_t block_m, int32_t* sorted_token_ids, int32_t* expert_offsets,
                       int32_t* expert_num_tokens, int32_t* block_expert_ids, void* scratch,
                       size_t scratch_bytes, int32_t* error_word, moe_stream_t stream);

/* moe_align_static_scratch: moe_align for callers that cannot allocate
 * device memory -- code that runs inside another framework's operator or a
 * plugin with no handle to that framework's allocator, or a latency-critical
 * loop where a cudaMalloc (which can synchronise the device) is not allowed.
 * The pages have no counterpart to this entry point: it is a deployment aid.
 *
 * Same arguments, outputs and errors as moe_align, minus `scratch`: the
 * per-chunk count table lives in a library-owned static device array of
 * MOE_ALIGN_STATIC_SCRATCH_INTS int32 (1 MiB).  The array belongs to the
 * library's device code module: with CUDA's lazy module loading (the default)
 * the module, and with it the array, is loaded on a device by the first
 * call of this entry point (or of any other kernel of the library) there, so
 * THAT first call may allocate; every later call allocates nothing.  Once
 * loaded, every GPU that uses the library holds the array until the process
 * exits.  Sizes with ceil(M * top_k / 256) * E > MOE_ALIGN_STATIC_SCRATCH_INTS
 * are rejected with MOE_ERR_WORKSPACE_TOO_SMALL.  The entry point itself calls
 * no cudaMalloc / cudaFree or allocating library routine.  The first call on
 * each device also looks up the array's device address (set-up) and caches
 * it for that device; make that first call before any stream capture.  A
 * device reset (cudaDeviceReset, or tearing down and re-creating the primary
 * context) invalidates the cached address: do not call this entry point in a
 * process after such a reset.  All calls share the one array and it keeps the
 * last call's contents (every entry a call reads is written earlier in that
 * same call, so nothing has to start at zero); calls that overlap on the GPU,
 * on any streams, race on it.
 */
#define MOE_ALIGN_STATIC_SCRATCH_INTS (1 << 18)
GBMOE_API moe_status_t moe_align_static_scratch(const int32_t* topk_ids, int64_t M,
                                                int32_t top_k, int32_t E, int32_t block_m,
                                                int32_t* sorted_token_ids,
                                                int32_t* expert_offsets,
                                                int32_t* expert_num_tokens,
                                                int32_t* block_expert_ids,
                                                int32_t* error_word, moe_stream_t stream);

/* -------------------------------------------------------------- forward --
 * moe_forward: y_t = sum_j topk_weights[t, j] * f_{topk_ids[t, j]}(x_t) with
 * the SwiGLU expert f_e(x) = (SiLU(x W13_e[:, :I] + b13_e[:I]) *
 * (x W13_e[:, I:] + b13_e[I:])) W2_e + b2_e.
 * Defines: "FlagGems fused_moe.py analysis", sections 1.1 and 1.2
 * (routed items h_r, z_r = phi(h_r), o_r, y_t = sum a(r) o_r), SiLU-and-mul
 * activation; "MindIE-SD Fused MoE" page, function signature (w13 fused
 * gate/up [E, H, 2I], w2 [E, I, H], w13_bias [E, 2I], w2_bias [E, H]);
 * "vLLM FusedMoEModularKernel" page, apply() steps (permute, W1 matmul,
 * activation + mul, W2 matmul, unpermute, top-k weight + reduce).
 *
 *  hidden        device bf16 [M, H]
 *  topk_weights  device fp32 [M, top_k];  topk_ids device int32 [M, top_k]
 *  w13           device bf16 [E, H, 2I]: columns [0, I) gate, [I, 2I) up
 *  w2            device bf16 [E, I, H]
 *  w13_bias      device bf16 [E, 2I] or NULL;  w2_bias device bf16 [E, H] or NULL
 *  workspace     device, >= moe_workspace_size(...) bytes, 256-byte aligned;
 *                contents on entry are ignored.  Its first 4 bytes hold the
 *                call's device error word (see moe_workspace_error_word).
 *  out           device bf16 [M, H]; may equal hidden (in-place)
 * Limits: H % 8 == 0, I % 8 == 0 (16-byte row pitch), 1 <= E <= 1024,
 * 1 <= top_k <= 64.
 * Tokens are processed in chunks of at most MOE_CHUNK_TOKENS, so the
 * workspace is bounded by the chunk, not by M.
 */
#define MOE_CHUNK_TOKENS 16384
GBMOE_API moe_status_t moe_workspace_size(int64_t M, int32_t H, int32_t I, int32_t E, int32_t top_k,
                                int32_t reduce_mode, size_t* bytes);
GBMOE_API moe_status_t moe_forward(const void* hidden, const float* topk_weights,
                         const int32_t* topk_ids, int64_t M, int32_t H, int32_t I,
                         int32_t E, int32_t top_k, const void* w13, const void* w2,
                         const void* w13_bias, const void* w2_bias, void* workspace,
                         size_t workspace_bytes, int32_t reduce_mode, void* out,
                         moe_stream_t stream);

/* moe_forward_opts: moe_forward with options.
 *  reduce_mode   as moe_forward's (moe_reduce_t)
 *  apply_router_weight_on_input  0: y_t = sum_r a(r) (W2^T z_r + b2);
 *                1: the weight multiplies the second layer's input instead,
 *                y_t = sum_r (W2^T (a(r) z_r) + b2) -- the switch of that name
 *                in "fused_moe.py 分析" section 1.2; equal to 0 when b2 = 0.
 *  expert_map    device int32 [num_global_experts] or NULL: topk_ids are then
 *                global expert ids, mapped to the local expert index (into
 *                w13 / w2 / biases, E of them) or -1 for experts held
 *                elsewhere -- those items contribute nothing (expert-parallel
 *                local compute; "fused_moe.py 分析", expert_map /
 *                write_zeros_to_output).  A map entry outside [-1, E) or an id
 *                outside [0, num_global_experts) sets MOE_ERR_BAD_EXPERT_ID.
 */
typedef struct {
  int32_t reduce_mode;
  int32_t apply_router_weight_on_input;
  const int32_t* expert_map;
  int32_t num_global_experts;
} moe_forward_opts_t;
GBMOE_API moe_status_t moe_forward_opts(const void* hidden, const float* topk_weights,
                                        const int32_t* topk_ids, int64_t M, int32_t H,
                                        int32_t I, int32_t E, int32_t top_k, const void* w13,
                                        const void* w2, const void* w13_bias,
                                        const void* w2_bias, void* workspace,
                                        size_t workspace_bytes, const moe_forward_opts_t* opts,
                                        void* out, moe_stream_t stream);

/* ----------------------------------------------- step from host memory --
 * moe_forward_host: one layer step whose inputs and output live in host
 * memory: the routing of moe_route, then moe_forward, with the copies --
 * router logits and hidden rows host -> device, out device -> host -- inside
 * the call.  Defines: "MindIE-SD Fused MoE" page, function signature
 * (hidden_states and router_logits in, the layer's output out, the router's
 * top-k inside the operator); "vLLM FusedMoEModularKernel" page, apply() steps.
 *  io->h_hidden      host bf16 [M, H];  io->h_logits host fp32 [M, E]
 *  io->h_out         host bf16 [M, H], written
 *                    (page-locked host memory gives full copy bandwidth and
 *                    keeps the copies asynchronous)
 *  io->d_hidden      device bf16 [M, H];  io->d_logits device fp32 [M, E]
 *  io->topk_weights  device fp32 [M, top_k];  io->topk_ids device int32 [M, top_k]
 *  io->d_out         device bf16 [M, H]
 *                    (device staging, owned by the caller; 16-byte aligned;
 *                    its contents afterwards are unspecified: the last
 *                    chunk's rows go straight to a mapped io->h_out, see
 *                    moe_set_host_out_direct)
 *  route             routing parameters, with moe_route's meaning and limits
 *  w13, w2, w13_bias, w2_bias, workspace, workspace_bytes, reduce_mode:
 *                    as moe_forward
 * Order: the copies in run on a host-to-device stream and the copies out on
 * a device-to-host stream, both kept by the library per host thread and
 * device and ordered with `stream` by events; routing, the plan, the GEMMs
 * and the reduce run on `stream`, each token chunk's rows awaited right
 * before they are first read.  Layers whose halves still average >= 512
 * routed rows per expert and whose copies are large against their weights
 * (copied bytes x 11 > weight bytes) run as two token chunks (results
 * identical to one pass), so the second chunk's rows are copied in while
 * the first is computed and the first chunk's output is copied out while
 * the second is computed.  The last chunk's output is written by its reduce
 * directly into io->h_out when that is mapped page-locked memory (no copy
 * after the reduce).  Returns after
 * enqueueing; io->h_out holds the result once `stream` has passed the call
 * (cudaStreamSynchronize or an event).  The call can be captured in a CUDA
 * graph.  Errors: as moe_route and moe_forward (checked before anything is
 * enqueued); a failed copy or stream operation returns MOE_ERR_CUDA.
 */
typedef struct {
  const void* h_hidden;
  const float* h_logits;
  void* h_out;
  void* d_hidden;
  float* d_logits;
  float* topk_weights;
  int32_t* topk_ids;
  void* d_out;
} moe_host_io_t;
typedef struct {
  int32_t top_k;
  int32_t routing_method; /* moe_routing_t */
  int32_t renormalize;
  int32_t k_group;
  int32_t group_count;
  int32_t group_select_mode;
  float routed_scaling_factor;
} moe_route_params_t;
GBMOE_API moe_status_t moe_forward_host(const moe_host_io_t* io, int64_t M, int32_t H,
                                        int32_t I, int32_t E, const moe_route_params_t* route,
                                        const void* w13, const void* w2, const void* w13_bias,
                                        const void* w2_bias, void* workspace,
                                        size_t workspace_bytes, int32_t reduce_mode,
                                        moe_stream_t stream);

/* ------------------------------------------------------------ FP8 W8A8 --
 * moe_forward_fp8: the layer with FP8 (E4M3) weights and activations
 * ("fused_moe.py 分析", "FP8 W8A8": the inputs of both GEMMs are quantised
 * to FP8 before the GEMM, and each FP8 dot product is multiplied by the
 * activation scale and the weight scale):
 *   h = (q(x) W13q) s_x s_w13 + b13,  z = SiLU(h_gate) h_up,
 *   o = (q(z) W2q) s_z s_w2 + b2,     y_t = sum_j a(t, j) o.
 * Activations (each routed row of x, and of z as held in bf16) are
 * quantised dynamically per row: scale = fp32(max|row| / 448) (1 for an
 * all-zero row), q = e4m3(fp32(row / scale)), round to nearest even,
 * saturating; the quotient is the correctly rounded fp32 one.  Weight scales
 * are per expert, per output channel, or per 128 x 128 block (scale_mode).
 * Block mode follows the page's block-wise path: within each 128-wide K
 * block the FP8 dot product is multiplied by that block's activation scale
 * and weight scale, and the blocks are summed; activations are then
 * quantised per (row, group of 128 along K) instead of per row.
 *  w13, w2       device E4M3 bytes [E, H, 2I] and [E, I, H]
 *  biases        bf16 as in moe_forward, or NULL
 *  workspace     >= moe_workspace_size_fp8(...) bytes, 256-byte aligned
 * Limits: as moe_forward, and H % 16 == 0, I % 16 == 0 (block mode:
 * H % 128 == 0, I % 128 == 0).
 */
typedef enum {
  MOE_FP8_SCALE_EXPERT = 0,  /* w13_scale, w2_scale [E]                               */
  MOE_FP8_SCALE_CHANNEL = 1, /* [E, 2I] and [E, H], per output channel               */
  MOE_FP8_SCALE_BLOCK = 2    /* [E, H/128, 2I/128] and [E, I/128, H/128], per 128 x 128
                                block of the weights; activations then quantised per
                                (row, group of 128 along K)                           */
} moe_fp8_scale_mode_t;
typedef struct {
  const void* w13;
  const void* w2;
  const float* w13_scale;
  const float* w2_scale;
  int32_t scale_mode; /* moe_fp8_scale_mode_t */
} moe_fp8_weights_t;
GBMOE_API moe_status_t moe_workspace_size_fp8(int64_t M, int32_t H, int32_t I, int32_t E,
                                              int32_t top_k, size_t* bytes);
GBMOE_API moe_status_t moe_forward_fp8(const void* hidden, const float* topk_weights,
                                       const int32_t* topk_ids, int64_t M, int32_t H, int32_t I,
                                       int32_t E, int32_t top_k, const moe_fp8_weights_t* w,
                                       const void* w13_bias, const void* w2_bias,
                                       void* workspace, size_t workspace_bytes, void* out,
                                       moe_stream_t stream);

/* moe_quant_rows_fp8: the per-row activation quantisation of the FP8 layer
 * on its own ("fused_moe.py 分析", the quantisation of each GEMM's input):
 * scale[m] = fp32(max_h |x[m, h]| / 448), 1 for an all-zero row;
 * q8[m, h] = e4m3(fp32(x[m, h] / scale[m])) with round to nearest even and
 * saturation to +-448.
 *  x       device bf16 [M, H], row-major
 *  q8      device E4M3 bytes [M, H] (caller-owned, written)
 *  scale   device fp32 [M] (caller-owned, written)
 * Limits: H % 16 == 0; x and q8 16-byte aligned.  M == 0 is a no-op.
 */
GBMOE_API moe_status_t moe_quant_rows_fp8(const void* x, int64_t M, int32_t H, void* q8,
                                          float* scale, moe_stream_t stream);

/* ---------------------------------------------- weight-only quantised --
 * Expert weights stored quantised, activations bf16.  Defines: "fused_moe.py
 * 分析" (FlagDoc), "WNA16 路径" and "5. 特殊量化格式处理": int8 / int4
 * weights with a group scale and a zero point (GPTQ/AWQ style), and OCP MX
 * weights, are dequantised to the activation dtype and the layer runs as
 * the bf16 one on those weights:
 *   int4, int8  w[e, k, n] = bf16((q[e, k, n] - zp[e, k/G, n]) * s[e, k/G, n])
 *   MX FP4/FP6  w[e, k, n] = bf16(value(q[e, k, n]) * 2^(s[e, k/32, n] - 127)),
 *               value = the E2M1 / E3M2 / E2M3 element of the code
 * each value the exact product rounded once (nearest even).  Layouts, in the
 * [E, K, N] orientation of the bf16 weights (w13: K = H, N = 2I with the
 * gate columns first; w2: K = I, N = H), all row-major:
 *  codes  int4 and MX FP4: uint8 [E, K, N/2], column 2j in the low nibble of
 *         byte j, column 2j+1 in its high nibble; int8: int8 [E, K, N];
 *         MX FP6: uint8 [E, K, N], the 6-bit code in the low bits (not the
 *         packed four-codes-in-three-bytes form)
 *  scale  int4 / int8: bf16 [E, K/G, N]; MX: uint8 (UE8M0) [E, K/32, N]
 *  zero   int4: uint8 [E, K/G, N] holding 0..15; int8: int8 [E, K/G, N];
 *         NULL = symmetric (int4: 8, int8: 0); MX: must be NULL
 *  G      group_size along K: a multiple of 32 dividing K (MX: 32)
 * All pointers device, caller-owned, 16-byte aligned.
 */
typedef enum {
  MOE_WQ_INT4 = 0,
  MOE_WQ_INT8 = 1,
  MOE_WQ_MXFP4 = 2,       /* OCP MX E2M1, two codes per byte */
  MOE_WQ_MXFP6_E3M2 = 3,  /* OCP MX FP6 E3M2, one code per byte (low 6 bits) */
  MOE_WQ_MXFP6_E2M3 = 4   /* OCP MX FP6 E2M3, one code per byte (low 6 bits) */
} moe_wq_format_t;
typedef struct {
  int32_t format;     /* moe_wq_format_t */
  int32_t group_size; /* G */
  const void* w13;
  const void* w2;
  const void* w13_scale;
  const void* w2_scale;
  const void* w13_zero; /* NULL, or both zero-point tensors given */
  const void* w2_zero;
} moe_wq_weights_t;

/* moe_dequant_weights: the dequantisation alone (the pages' path before the
 * bf16 layer): out = bf16 [E, K, N] (written).  Limits: N % 16 == 0,
 * K % G == 0.  Asynchronous on `stream`. */
GBMOE_API moe_status_t moe_dequant_weights(int32_t format, const void* codes, const void* scale,
                                           const void* zero, int32_t E, int32_t K, int32_t N,
                                           int32_t group_size, void* out, moe_stream_t stream);

/* moe_forward_wq: the layer with weight-only quantised w13 and w2.  The
 * weights stay quantised in HBM: each grouped GEMM stages their codes and
 * scales in shared memory and expands them to bf16 there.  Arguments as
 * moe_forward with the separate weight-and-reduce; workspace >=
 * moe_workspace_size(M, H, I, E, top_k, MOE_REDUCE_SEPARATE).
 * Limits: as moe_forward, and H, I multiples of 32, at least 64, divisible
 * by G. */
GBMOE_API moe_status_t moe_forward_wq(const void* hidden, const float* topk_weights,
                                      const int32_t* topk_ids, int64_t M, int32_t H, int32_t I,
                                      int32_t E, int32_t top_k, const moe_wq_weights_t* w,
                                      const void* w13_bias, const void* w2_bias, void* workspace,
                                      size_t workspace_bytes, void* out, moe_stream_t stream);

/* ------------------------------------------------------ forward_batched --
 * moe_forward_batched: the Batched activation format.  Defines: "vLLM
 * FusedMoEModularKernel" page, Introduction (activations (num_experts,
 * max_tokens, K) with expert_num_tokens; not every row is valid; Batched
 * differs from Contiguous only in the permute / unpermute).
 *   out[e, i] = row_weight[e, i] * f_e(x[e, i])   for i < expert_num_tokens[e]
 *
 *  x                  device bf16 [E, T, H]; rows i >= expert_num_tokens[e]
 *                     are never read (they may hold anything, NaN included)
 *  expert_num_tokens  device int32 [E], each in [0, T]; a value outside sets
 *                     MOE_ERR_BAD_EXPERT_ID in the error word and that
 *                     expert is skipped
 *  row_weight         device fp32 [E, T] or NULL (= 1)
 *  out                device bf16 [E, T, H]; rows past the count are not written
 * Limits as moe_forward; 1 <= T.
 */
GBMOE_API moe_status_t moe_batched_workspace_size(int32_t E, int32_t T, int32_t H, int32_t I,
                                        size_t* bytes);
GBMOE_API moe_status_t moe_forward_batched(const void* x, const int32_t* expert_num_tokens, int32_t E,
                                 int32_t T, int32_t H, int32_t I, const void* w13,
                                 const void* w2, const void* w13_bias, const void* w2_bias,
                                 const float* row_weight, void* workspace,
                                 size_t workspace_bytes, void* out, moe_stream_t stream);

/* --------------------------------------------------------------- errors --
 * moe_workspace_error_word: device address of the error word inside a
 * forward workspace (pure pointer arithmetic, no GPU access).
 * moe_read_error: SYNCHRONISES `stream`, copies the device error word to
 * the host and returns it as a status (MOE_OK if zero); if reset != 0 the
 * word is cleared afterwards.
 */
GBMOE_API int32_t* moe_workspace_error_word(void* workspace);
GBMOE_API moe_status_t moe_read_error(const int32_t* error_word, int32_t reset, moe_stream_t stream);

/* moe_workspace_layout: byte offsets, inside a forward workspace sized for
 * (M, H, I, E, top_k), of its regions -- for inspecting intermediate stages
 * in tests.  offsets[0..8] = error word, expert_num_tokens [E],
 * expert_offsets [E+1], block_expert_ids, sorted_token_ids [cap], align
 * scratch, inverse permutation int32 [M*top_k] (sorted position of each
 * routed item, -1 if dropped), permuted token rows bf16 [cap, H],
 * z = SiLU(gate)*up bf16 [cap, I], the item rows of SEPARATE (sorted; fp32
 * [cap, H], or fp16 [cap, H] followed by their exponents [ceil(H/32)][cap]
 * bytes, as moe_set_item_rows picks) / the token accumulator fp32 [M, H] of
 * EPILOGUE_ATOMIC, one region -- all for the
 * first token chunk; offsets[10] = cap (rows of the padded layout).
 * No GPU access.
 */
GBMOE_API moe_status_t moe_workspace_layout(int64_t M, int32_t H, int32_t I, int32_t E,
                                            int32_t top_k, size_t offsets[11]);

/* moe_selftest_wait_timeout: failure-detection self-test.  Launches one CTA
 * that waits on an mbarrier nothing ever arrives at, with a wait limit of
 * limit_us microseconds; the kernel must give up, write MOE_ERR_TIMEOUT to
 * *error_word (device int32) and return.  Read it with moe_read_error.
 */
GBMOE_API moe_status_t moe_selftest_wait_timeout(int32_t* error_word, uint32_t limit_us,
                                                 moe_stream_t stream);

GBMOE_API const char* moe_status_string(moe_status_t status);
GBMOE_API const char* moe_last_error_detail(void);
GBMOE_API int32_t moe_abi_version(void);

/* ------------------------------------------------------------- profiler --
 * Per-kernel timing with CUDA events recorded on the launching stream
 * around every kernel the library launches from the calling thread.
 * moe_profiler_start enables it (and clears previous records);
 * moe_profiler_stop synchronises on the recorded events, fills up to
 * `capacity` entries (kernel name, launches, total milliseconds) and
 * disables it.  Returns the number of distinct kernels in *n.
 */
typedef struct {
  char name[48];
  int64_t launches;
  double total_ms;
} moe_kernel_time_t;
GBMOE_API moe_status_t moe_profiler_start(void);
GBMOE_API moe_status_t moe_profiler_stop(moe_kernel_time_t* out, int32_t capacity, int32_t* n);
/* Grouped-GEMM tile shape (process-wide tuning / testing knob):
 * 0 = automatic (CTA pairs when the routed rows average at least four
 * 128-row blocks per expert), 1 = single-CTA 128x256 tiles, 2 = CTA-pair
 * 256x256 tiles (tcgen05 cta_group::2).  Results are the same up to fp32
 * summation order.  Invalid values return MOE_ERR_INVALID_ARG. */
GBMOE_API moe_status_t moe_set_gemm_tiles(int32_t mode);
/* Programmatic dependent launch (process-wide tuning / testing knob, on by
 * default): 1 = every kernel of the library is launched with programmatic
 * stream serialisation allowed and begins by waiting on the device
 * (griddepcontrol.wait) until the kernel before it has completed; kernels
 * with small grids let their successor be scheduled at once, so the launch
 * gaps between a small layer's kernels are hidden, while kernels with large
 * grids let it be scheduled as their CTAs exit; 0 = plain stream order.
 * Results are identical either way.  Values other than 0 / 1 return
 * MOE_ERR_INVALID_ARG. */
GBMOE_API moe_status_t moe_set_pdl(int32_t enabled);
/* Item-row format of the separate weight-and-reduce (process-wide tuning /
 * testing knob) for moe_forward, moe_forward_opts, moe_forward_host and
 * moe_forward_fp8 with per-expert or per-channel weight scales (the
 * block-scaled FP8 and weight-only forwards keep fp32 rows).  The rows are
 * either fp32, or fp16 values times 2^-e with one exponent e >= 0 per row
 * and 32-column chunk, the least that keeps the chunk finite (half the
 * bytes, 11 significant bits, no overflow).  0 = automatic (fp16 when
 * top_k >= 4, where a token's k rows dominate the reduce's traffic; the
 * default), 1 = fp32, 2 = fp16.  "fused_moe.py 分析" rounds these rows to
 * the compute dtype (bf16) before the k-sum; both formats here are more
 * precise.  Results agree to fp16 rounding of each weighted item row.
 * Values outside 0..2 return MOE_ERR_INVALID_ARG. */
GBMOE_API moe_status_t moe_set_item_rows(int32_t mode);
/* Weight-only decode GEMMs (process-wide tuning / testing knob, on by
 * default): 1 = moe_forward_wq takes, for calls of at most 32 tokens (H a
 * multiple of 64, E <= 1024, int formats with a power-of-two group of at
 * least 32 rows), GEMMs that keep each expert's few rows as the MMA's N and
 * expand the quantised weights in registers, GEMM2's K split into parts
 * that the weight-and-reduce adds; 0 = always the grouped tensor-core GEMMs.
 * Results agree up to fp32 summation order.  Values other than 0 / 1 return
 * MOE_ERR_INVALID_ARG. */
GBMOE_API moe_status_t moe_set_wq_decode(int32_t enabled);
/* Direct output of moe_forward_host (process-wide tuning / testing knob, on
 * by default): 1 = when io->h_out is page-locked host memory mapped into the
 * device's address space (cudaHostAlloc / cudaHostRegister; 16-byte
 * aligned), the last token chunk's reduce writes its rows straight into it
 * over the host link, and io->d_out is left unwritten for those rows;
 * 0 = every chunk's output goes through io->d_out and a device-to-host
 * copy.  Results are identical.  Values other than 0 / 1 return
 * MOE_ERR_INVALID_ARG. */
GBMOE_API moe_status_t moe_set_host_out_direct(int32_t enabled);
/* Small calls (process-wide tuning / testing knob, on by default): 1 =
 * moe_forward / moe_forward_opts / moe_forward_host with MOE_REDUCE_AUTO and
 * no expert map or router weight on the input, at most 256 routed items,
 * M * H <= 2^18, H and I multiples of 64 and expert weights of at most
 * 64 MiB, run the layer in two kernels: GEMM1 finds each expert's items in
 * topk_ids itself and gathers their rows (no align plan and no permuted
 * rows: the workspace's plan regions are left unwritten, and the start of
 * its permuted-rows region holds one completion counter per 64 output
 * columns), and GEMM2 adds the weighted rows into an fp32 token accumulator
 * with atomics, the last CTA of each 64-column block writing that block out.
 * 0 = always the general path.  Results agree up to fp32 summation order
 * (for top_k <= 2 that order cannot change the sum).  Values other than
 * 0 / 1 return MOE_ERR_INVALID_ARG. */
GBMOE_API moe_status_t moe_set_small_path(int32_t enabled);
/* Where moe_forward / moe_forward_opts / moe_forward_host take GEMM1's rows
 * from (process-wide tuning / testing knob): 0 = automatic (fused when the
 * routed rows of a token chunk hold at most 16 MiB), 1 = a separate gather
 * kernel writes the expert-sorted rows first, 2 = GEMM1 copies them from the
 * token rows itself (a gather warp, 16-byte asynchronous copies).
 * Results are identical.  Invalid values return MOE_ERR_INVALID_ARG. */
GBMOE_API moe_status_t moe_set_gather_mode(int32_t mode);

/* Total kernel launches issued by the library on this thread since load. */
GBMOE_API int64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GBMOE_H */
