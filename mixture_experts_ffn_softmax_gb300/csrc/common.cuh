// Shared declarations of the gbmoe CUDA library (kernels + host launchers).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "../../include/gbmoe.h"

namespace gbmoe {

using bf16 = __nv_bfloat16;

// A bounded wait gives up after this long; the kernel then records
// MOE_ERR_TIMEOUT in the error word and returns instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ void record_error(int32_t* error_word, int32_t code) {
  if (error_word != nullptr) atomicCAS(error_word, 0, code);
}

template <typename T>
__host__ __device__ constexpr T ceil_div(T a, T b) {
  return (a + b - 1) / b;
}

// ---- host-side launch bookkeeping (api.cu) ----
// Every kernel launch goes through these so the profiler can bracket it with
// CUDA events on the launching stream and count launches.
void prof_before(const char* name, cudaStream_t s);
void prof_after(const char* name, cudaStream_t s);
moe_status_t set_error(moe_status_t st, const char* fmt, ...);
moe_status_t check_launch(const char* name);

// GEMM tile shape selection: 0 auto, 1 single-CTA tiles, 2 CTA-pair tiles.
int gemm_tile_mode();

// ---- programmatic dependent launch ----
// Every kernel of the library is launched with programmatic stream
// serialisation allowed (launch_kernel) and begins with pdl_begin(): it waits
// until the grid before it in the stream has completed and that grid's
// memory operations are visible (griddepcontrol.wait).  A kernel with a small
// grid then lets the next grid be scheduled at once
// (griddepcontrol.launch_dependents): the next kernel's CTAs are made
// resident, their launch latency spent, while it runs -- the gaps between
// the short kernels of a small layer disappear.  A kernel with a large grid
// does not: resident CTAs of the next kernel (a grouped GEMM's hold 53K
// registers each) would take registers and warp slots from its own, so its
// dependents are scheduled as its CTAs exit (the implicit trigger).  Every
// kernel waits before anything else, so completion order is transitive along
// a chain of launches; a kernel whose predecessor is not such a launch
// (another library's kernel, a copy) waits for it as usual.
constexpr unsigned kPdlEarlyTriggerCtas = 64;
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (gridDim.x * gridDim.y * gridDim.z <= kPdlEarlyTriggerCtas)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Whether launches carry the attribute (moe_set_pdl; on by default).
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// A value computed once per device (function attributes, occupancy), safely
// from several host threads: get(f) returns f()'s result for the current
// device, calling f the first time for that device (again after a failure).
class PerDevice {
 public:
  template <typename F>
  cudaError_t get(F&& f, int* value = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) {
      cudaGetLastError();
      return cudaErrorInvalidDevice;
    }
    std::lock_guard<std::mutex> lock(mutex_);
    if (!have_[dev]) {
      int v = 0;
      const cudaError_t e = f(&v);
      if (e != cudaSuccess) return e;
      value_[dev] = v;
      have_[dev] = true;
    }
    if (value) *value = value_[dev];
    return cudaSuccess;
  }

 private:
  static constexpr int kDevices = 64;
  std::mutex mutex_;
  bool have_[kDevices] = {};
  int value_[kDevices] = {};
};

// ---- launchers (one per .cu file) ----
struct RouteArgs {
  const void* logits;  // fp32 or bf16 [M, E]
  int64_t M;
  int32_t E, top_k, method, renormalize, k_group, group_count, group_select_mode;
  float scale;
  float* weights;
  int32_t* ids;
  int32_t logits_bf16 = 0;
};
moe_status_t launch_route(const RouteArgs& a, cudaStream_t s);

struct AlignArgs {
  const int32_t* ids;   // [R] expert id per item
  int64_t R;            // items
  int32_t E, block_m;
  int32_t* sorted;      // [cap]
  int32_t* offsets;     // [E+1]
  int32_t* counts;      // [E]
  int32_t* block_expert;  // [cap / block_m]
  int32_t* chunk_counts;  // scratch [num_chunks * E]
  int64_t cap;
  int32_t* error_word;
  int32_t* inv = nullptr;  // optional [R]: sorted position of item r (-1 if dropped)
  // optional expert parallelism: ids are global ids in [0, E_global); an id
  // maps to local expert expert_map[id] in [0, E), or -1 (held elsewhere:
  // the item is skipped, not an error)
  const int32_t* expert_map = nullptr;
  int32_t E_global = 0;
  // optional: words cleared before anything of the plan runs (the forward's
  // error word and tile-schedule counters) -- by the one-block plan itself,
  // else by a memset ahead of the four-kernel plan
  int32_t* zero_words = nullptr;
  int32_t zero_count = 0;
};
size_t align_scratch_bytes(int64_t R, int32_t E);
moe_status_t launch_align(const AlignArgs& a, cudaStream_t s);
// Same, with the chunk table in the library's static device array.
moe_status_t launch_align_static_scratch(AlignArgs a, cudaStream_t s);

// Batched layout plan: per expert e, rows e*T + i (i < count_e) in order,
// padded with the sentinel to a multiple of block_m.
struct BatchedPlanArgs {
  const int32_t* counts_in;  // [E]
  int32_t E, T, block_m;
  int32_t* sorted;     // [cap]
  int32_t* offsets;    // [E+1]
  int32_t* block_expert;
  int64_t cap;
  int32_t sentinel;
  int32_t* error_word;  // cleared by the plan before use
};
moe_status_t launch_batched_plan(const BatchedPlanArgs& a, cudaStream_t s);

// A_perm[p, :] = src[index[p] / div, :] for p < offsets[E] (zero row when
// index[p] >= sentinel).
struct GatherArgs {
  const bf16* src;
  const int32_t* index;
  const int32_t* offsets;  // [E+1]; offsets[E] = number of rows to produce
  int32_t E;
  int32_t div;
  int32_t sentinel;
  int32_t H;
  int64_t cap;
  bf16* dst;
  // token-major form (inv != null): token t's row goes to the sorted rows
  // inv[t * div + j] (j < div; -1: dropped) for t < tokens, each token row
  // read once; index, offsets and sentinel are then unused
  const int32_t* inv = nullptr;
  int64_t tokens = 0;
};
moe_status_t launch_gather(const GatherArgs& a, cudaStream_t s);

// FP8 rows: for sorted position p < offsets[E] whose index[p] is a real
// entry, row src[index[p] / div] (index == null: row p) is quantised with
// its own scale = amax / 448: q8[p] = e4m3(row / scale), scale[p] = scale.
// FP8 (E4M3) per-row quantisation of the token rows: each token's row is
// read once, its scale and codes go to every sorted row inv[t*k + j] >= 0,
// and row_amax[pos] (if given) is zeroed for the GEMM1 epilogue's max.
struct QuantTokensArgs {
  const bf16* x;          // [M, H]
  const int32_t* inv;     // [M*k] sorted row of item (t, j), or -1
  int64_t M;
  int32_t k, H;
  uint8_t* q8;            // [cap, H] codes
  float* scale;           // [cap]
  float* row_amax;        // [cap] or null
};
moe_status_t launch_quant_tokens_fp8(const QuantTokensArgs& a, cudaStream_t s);
// FP8 quantisation of the expert-sorted rows of z, whose per-row amax the
// GEMM1 epilogue has already taken: scale_io[p] holds amax on entry and the
// row's scale on exit; padding rows are skipped.
struct QuantSortedArgs {
  const bf16* src;        // [cap, H]
  const int32_t* index;   // [cap] sorted item ids (padding >= sentinel)
  const int32_t* offsets; // [E + 1]
  int32_t E, sentinel, H;
  int64_t cap;
  uint8_t* q8;            // [cap, H]
  float* scale_io;        // [cap]
};
moe_status_t launch_quant_sorted_fp8(const QuantSortedArgs& a, cudaStream_t s);
// The token rows' quantisation per (row, group of 128 columns), scales
// group-major [H/128][ld] (ld = cap; row_amax unused).  z of the block-scaled
// layer is quantised the same way by GEMM1's epilogue.
moe_status_t launch_quant_tokens_group_fp8(const QuantTokensArgs& a, int64_t ld, cudaStream_t s);

// Weight-only quantised weights -> bf16 [E, K, N] (wq.cu).  format: 0 int4,
// 1 int8, 2 MX FP4; codes, scale [E, K/G, N], zero [E, K/G, N] or null.
struct WqDequantArgs {
  int32_t format;
  const void* codes;
  const void* scale;
  const void* zero;
  int32_t E, K, N, G;
  __nv_bfloat16* out;
};
moe_status_t launch_dequant_weights(const WqDequantArgs& a, cudaStream_t s);

// y[t, :] = bf16( sum_j o_sorted[inv[t*k + j], :] ), skipping inv < 0.
moe_status_t launch_reduce_sorted(const float* o_sorted, const int32_t* inv, int64_t M,
                                  int32_t k, int32_t H, bf16* y, cudaStream_t s);
// y = bf16(acc), acc fp32 [M, H].
moe_status_t launch_cast_f32_bf16(const float* acc, int64_t n, bf16* y, cudaStream_t s);

// Grouped GEMMs (gemm.cu).
struct GroupedGemmArgs {
  // operands
  const bf16* a;          // [cap, K] expert-sorted rows
  const bf16* w;          // GEMM1: w13 [E, K=H, 2N]; GEMM2: w2 [E, K=I, N=H]
  const bf16* bias;       // GEMM1: [E, 2N]; GEMM2: [E, N]; or null
  int64_t cap;            // rows of a
  int32_t E, N, K;        // GEMM1: N = I (per half); GEMM2: N = H
  const int32_t* offsets;  // [E+1] padded expert offsets
  // epilogue
  void* out;              // GEMM1: z bf16 [cap, N]; GEMM2: fp32 [*, N] or bf16 [*, N]
  const int32_t* row_index;  // GEMM2: routed item (or batched row) per sorted position
  const float* row_weight;   // GEMM2: weight per item / row, or null (=1)
  int32_t sentinel;          // GEMM2: row_index >= sentinel -> padding
  int32_t div;               // GEMM2 atomic: token of item r is r / div
  int32_t* error_word;
  int32_t num_sms;
  int64_t rows_hint;         // routed rows (before padding), for the tile shape choice
  const float* gemm1_row_weight = nullptr;  // GEMM1: weight per routed item multiplied
                                            // into z (router weight on the input)
  // FP8 operands (a and w are E4M3): acc * a_scale[sorted row] * weight scale
  const float* a_scale = nullptr;
  const float* w_scale = nullptr;       // [E, 2N] / [E, N] per channel, or [E]
  int32_t w_scale_per_channel = 0;
  float* row_amax = nullptr;            // GEMM1 FP8: max |bf16 z| of each sorted row (atomic)
  // GEMM1 with block-scaled FP8 (required there): z leaves as E4M3 codes in
  // `out` ([cap, N] bytes) with one scale per row and 128-column group here,
  // [N / 128][cap] -- the quantisation the second GEMM's A takes
  float* z_group_scale = nullptr;
  // weight-only quantised w (codes in `w`): format (0 int4, 1 int8, 2 MX FP4),
  // group size along K, scales [E, K/G, N'] and zero points (or null)
  int32_t wq_format = -1;
  int32_t wq_group = 0;
  const void* wq_scale = nullptr;
  const void* wq_zero = nullptr;
  // GEMM1 with the gather fused (bf16): the token rows [M, K] that A's rows
  // are copied from (row r = token row_index[r] / div), or null (A = a)
  const bf16* a_rows = nullptr;
  // GEMM2 SortedF16: the exponent e of each row's 32-column chunk (rows
  // stored as fp16 times 2^-e), [ceil(N/32)][cap] bytes
  uint8_t* o_exp = nullptr;
  // bf16 grouped GEMMs: two int32 {next tile, CTAs done}, zero at launch
  // (reset by the kernel itself when it ends), for the dynamic tile
  // schedule; null: static schedule
  int32_t* sched = nullptr;
};
// Whether GEMM1 copies its A rows from the token rows itself: the mode set
// by moe_set_gather_mode (0 auto, 1 separate gather kernel, 2 fused) and,
// for auto, the call's shape.
bool gemm1_fused_gather(int64_t rows, int32_t H, int32_t I, int32_t E);
moe_status_t launch_gemm1_swiglu_fp8(const GroupedGemmArgs& a, cudaStream_t s);
moe_status_t launch_gemm2_sorted_fp8(const GroupedGemmArgs& a, cudaStream_t s);
// Dense GEMM with fp32 output: out [M, N] = a [M, K] @ w [K, N] + bias [N]
// (the router logits), one "expert", single-CTA tiles.
moe_status_t launch_dense_f32(const GroupedGemmArgs& a, cudaStream_t s);
// Router logits for few experts (E <= 32, H % 256 == 0, W_g fits in shared
// memory): SIMT, one warp per token, W_g staged in shared memory.
bool router_small_fits(int H, int E);
moe_status_t launch_router_small(const bf16* x, const bf16* wg, const bf16* bg, int64_t M,
                                 int H, int E, float* s, cudaStream_t st);
moe_status_t launch_gemm1_swiglu(const GroupedGemmArgs& a, cudaStream_t s);
// GEMM2, contiguous layout, SEPARATE reduce: weighted fp32 rows in sorted
// order, out = o_sorted [cap, N], written with TMA tensor stores.
moe_status_t launch_gemm2_sorted_f32(const GroupedGemmArgs& a, cudaStream_t s);
// GEMM2, contiguous layout, ATOMIC reduce: out = acc fp32 [M, N]; each
// weighted row is added into row row_index[p] / div with vector fp32 atomics.
moe_status_t launch_gemm2_atomic_f32(const GroupedGemmArgs& a, cudaStream_t s);
// GEMM2, SEPARATE reduce, item rows as fp16 times 2^-e with e per row and
// 32-column chunk in a.o_exp (out = fp16 [cap, N]); bf16 and FP8 operands.
moe_status_t launch_gemm2_sorted_f16(const GroupedGemmArgs& a, cudaStream_t s);
moe_status_t launch_gemm2_sorted_f16_fp8(const GroupedGemmArgs& a, cudaStream_t s);
// The weight-and-reduce over such rows (exponents [chunk][row], ld rows).
moe_status_t launch_reduce_sorted_f16(const void* o16, const uint8_t* o_exp, int64_t ld,
                                     const int32_t* inv, int64_t M, int32_t k, int32_t H, bf16* y,
                                     cudaStream_t s);
// Item-row format of the separate reduce for a call with top_k items per
// token (moe_set_item_rows): true = fp16 with exponents, false = fp32.
bool item_rows_fp16(int32_t top_k);
// Whether moe_forward_host writes a pinned output buffer directly
// (moe_set_host_out_direct; on by default).
bool direct_host_out();

// The whole layer of a small call in two kernels (small.cu): GEMM1 with the
// plan and the gather folded in, GEMM2 with the weight-and-reduce.
struct SmallArgs {
  const bf16* x;
  const bf16* w13;
  const bf16* w2;
  const bf16* b13;
  const bf16* b2;
  const int32_t* ids;
  const float* weights;
  bf16* z;          // workspace [M * k, I]
  float* acc;       // workspace [M, H]
  int32_t* counter; // workspace [H / 64]: GEMM2 CTAs done per 64 output columns
  int32_t* error_word;
  bf16* y;
  int64_t M;
  int32_t H, I, E, k;
};
bool small_forward_applies(int64_t M, int32_t H, int32_t I, int32_t E, int32_t top_k);
moe_status_t launch_small_forward(const SmallArgs& a, cudaStream_t s);
// moe_set_small_path: whether small calls take it (on by default).
bool small_path_enabled();
moe_status_t launch_gemm2_rows_bf16(const GroupedGemmArgs& a, cudaStream_t s);
// FP8 with block-wise scales: a.w_scale [E, K/128, N'/128] per 128 x 128
// weight block, a.a_scale [K/128][cap] per (sorted row, 128-wide K group),
// a.row_amax (GEMM1) [N/128][cap] z amax per row and 128-column group.
moe_status_t launch_gemm1_swiglu_fp8_block(const GroupedGemmArgs& a, cudaStream_t s);
moe_status_t launch_gemm2_sorted_fp8_block(const GroupedGemmArgs& a, cudaStream_t s);
// bf16 A x weight-only quantised w (a.wq_format), B converted to bf16 in
// shared memory: GEMM1 with the SwiGLU epilogue, GEMM2 with sorted fp32 rows.
moe_status_t launch_gemm1_swiglu_wq(const GroupedGemmArgs& a, cudaStream_t s);
moe_status_t launch_gemm2_sorted_wq(const GroupedGemmArgs& a, cudaStream_t s);
moe_status_t launch_wait_timeout_probe(int32_t* err, uint32_t limit_us, cudaStream_t s);
// A tensor map (cuTensorMapEncodeTiled through the driver entry point);
// dims / strides innermost first, strides in bytes for dims 1..rank-1.
moe_status_t encode_tensor_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                               const uint64_t* strides, const uint32_t* box,
                               CUtensorMapDataType dtype, CUtensorMapSwizzle swz);
// Weight-only quantised GEMMs for few rows per expert (M <= 32 tokens):
// whether the call's shape takes them, the K parts of GEMM2, and the
// launches.  GEMM1 writes z rows like launch_gemm1_swiglu_wq; GEMM2 writes
// `splits` weighted fp32 partial rows per routed item, out[(s * R + r) * H],
// which launch_reduce_parts adds per token.
bool wq_decode_applies(int64_t M, int32_t H, int32_t I, int32_t E, int32_t format, int32_t group);
int wq_decode_splits(int64_t M, int32_t top_k, int32_t H, int32_t I, int32_t E, int64_t cap,
                     int32_t num_sms);
moe_status_t launch_wq_decode_gemm1(const GroupedGemmArgs& a, const int32_t* counts, int64_t M,
                                    cudaStream_t s);
moe_status_t launch_wq_decode_gemm2(const GroupedGemmArgs& a, const int32_t* counts, int64_t M,
                                    int32_t splits, int64_t R, cudaStream_t s);
moe_status_t launch_reduce_parts(const float* parts, const int32_t* inv, int64_t M, int32_t k,
                                 int32_t H, int32_t splits, bf16* y, cudaStream_t s);

}  // namespace gbmoe
