// C-ABI entry points: host-side validation, workspace layout, the token
// chunk loop, launch bookkeeping and the event-based kernel profiler.
//
// The forward follows the "vLLM FusedMoEModularKernel" page's apply() step
// list (permute, W1 matmul, activation + mul, W2 matmul, unpermute, top-k
// weight + reduce) and workspace_shapes() idea (intermediates live in one
// caller-allocated workspace), and the "FlagGems fused_moe.py analysis"
// chunk loop (tokens processed CHUNK_SIZE = 16 * 1024 at a time to bound
// the intermediate caches) and its input validation list.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"

namespace gbmoe {

// ------------------------------------------------------------- errors ---
namespace {
thread_local char g_detail[512] = "";
thread_local int64_t g_launches = 0;

struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
thread_local bool g_prof = false;
thread_local std::vector<ProfRec> g_recs;
thread_local std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

namespace {
std::atomic<int> g_gemm_tile_mode{0};
std::atomic<int> g_gather_mode{0};
std::atomic<int> g_pdl{1};
std::atomic<int> g_wq_decode{1};
std::atomic<int> g_item_rows{0};
std::atomic<int> g_direct_host_out{1};
std::atomic<int> g_small_path{1};
}  // namespace

bool direct_host_out() { return g_direct_host_out.load(std::memory_order_relaxed) != 0; }
bool small_path_enabled() { return g_small_path.load(std::memory_order_relaxed) != 0; }

// Automatic choice: fp16 rows when each token has at least four items.  The
// k item rows a token's reduce reads then outweigh the rest of its traffic
// (Qwen-MoE shape, k = 8: layer 1.27 -> 1.14 ms, the reduce 186 -> 109 us;
// DeepSeek-V3 M=8192: 5.76 -> 5.61 ms); with k = 2 (Mixtral shape) the rows
// are a small part of the tensor-bound layer's bytes and gain nothing.
bool item_rows_fp16(int32_t top_k) {
  const int mode = g_item_rows.load(std::memory_order_relaxed);
  return mode == 2 || (mode == 0 && top_k >= 4);
}

int gemm_tile_mode() { return g_gemm_tile_mode.load(std::memory_order_relaxed); }
bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

// Automatic choice: fused when the routed rows are few (<= 16 MiB of them).
// The gather warp's 16-byte copies move ~16 B per cycle per SM, half of what
// GEMM1's MMAs consume on large shapes (Mixtral prefill GEMM1 1257 -> 2446
// us fused), while on small ones the fused copy saves the gather's launch
// and the padding rows' loads (M=64 test shape 34 -> 29 us, DeepSeek-V3
// M=64 2.90 -> 2.83 ms).
bool gemm1_fused_gather(int64_t rows, int32_t H, int32_t I, int32_t E) {
  const int mode = g_gather_mode.load(std::memory_order_relaxed);
  if (mode != 0) return mode == 2;
  (void)I;
  (void)E;
  return rows * static_cast<int64_t>(H) * 2 <= (int64_t{16} << 20);
}

moe_status_t set_error(moe_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return st;
}

moe_status_t check_launch(const char* name) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "launch of %s failed: %s", name, cudaGetErrorString(e));
  return MOE_OK;
}

void prof_before(const char* name, cudaStream_t s) {
  ++g_launches;
  if (!g_prof) return;
  cudaEvent_t a = take_event();
  cudaEventRecord(a, s);
  g_recs.push_back({name, a, nullptr});
}

void prof_after(const char* /*name*/, cudaStream_t s) {
  if (!g_prof || g_recs.empty()) return;
  cudaEvent_t b = take_event();
  cudaEventRecord(b, s);
  g_recs.back().b = b;
}

namespace {

// ------------------------------------------------------------- device ---
moe_status_t check_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return set_error(MOE_ERR_NO_DEVICE, "no CUDA device");
  }
  // per host thread: the last device asked about (no shared mutable state)
  thread_local int cached_dev = -1, cached_ok = 0, cached_sms = 0;
  if (dev != cached_dev) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    cached_dev = dev;
    cached_ok = (major == 10 && minor == 3);
    cached_sms = sms;
    if (!cached_ok)
      return set_error(MOE_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a",
                       dev, major, minor);
  }
  if (!cached_ok) return set_error(MOE_ERR_NO_DEVICE, "device is not sm_103");
  if (num_sms) *num_sms = cached_sms;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr size_t kRegionAlign = 1024;
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int64_t align_cap(int64_t R, int32_t E, int32_t block_m) {
  const int64_t busy = R < E ? R : E;  // experts that can be non-empty
  const int64_t cap = R + busy * (block_m - 1);
  return round_up(static_cast<size_t>(cap), static_cast<size_t>(block_m));
}

// Workspace of one forward chunk (Rc routed items).
struct FwdLayout {
  int64_t cap = 0;
  size_t err = 0, counts = 0, offsets = 0, block_expert = 0, sorted = 0, scratch = 0,
         a_perm = 0, z = 0, o = 0, inv = 0, total = 0;
};

FwdLayout fwd_layout(int64_t Mc, int32_t H, int32_t I, int32_t E, int32_t k) {
  FwdLayout L;
  const int64_t Rc = Mc * k;
  L.cap = align_cap(Rc, E, MOE_BLOCK_M);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, kRegionAlign);
    return at;
  };
  L.err = take(256);
  L.counts = take(sizeof(int32_t) * E);
  L.offsets = take(sizeof(int32_t) * (E + 1));
  L.block_expert = take(sizeof(int32_t) * (L.cap / MOE_BLOCK_M));
  L.sorted = take(sizeof(int32_t) * L.cap);
  L.scratch = take(align_scratch_bytes(Rc, E));
  L.inv = take(sizeof(int32_t) * Rc);
  L.a_perm = take(sizeof(bf16) * L.cap * H);
  L.z = take(sizeof(bf16) * L.cap * I);
  // fp32 rows: sorted item rows [cap, H] (separate reduce) or the token
  // accumulator [Mc, H] (atomic reduce); cap >= Mc, so one region serves both.
  L.o = take(sizeof(float) * L.cap * H);
  L.total = off;
  return L;
}

// TopKWeightAndReduce choice for MOE_REDUCE_AUTO.  Measured on GB300 for the
// Mixtral (k=2), Qwen (k=8, 16K tokens) and DeepSeek (k=8, 8K tokens)
// shapes, sorted fp32 rows + a separate reduce beat the epilogue atomics on
// every one (the 16-byte atomics into scattered token rows are L2-bound), so
// AUTO selects SEPARATE.
int32_t pick_reduce(int64_t /*Mc*/, int32_t /*H*/, int32_t /*k*/, int32_t mode) {
  return mode == MOE_REDUCE_AUTO ? MOE_REDUCE_SEPARATE : mode;
}

struct BatLayout {
  int64_t cap = 0;
  size_t err = 0, offsets = 0, block_expert = 0, sorted = 0, a_perm = 0, z = 0, total = 0;
};

BatLayout bat_layout(int32_t E, int32_t T, int32_t H, int32_t I) {
  BatLayout L;
  L.cap = static_cast<int64_t>(E) * T + static_cast<int64_t>(E) * (MOE_BLOCK_M - 1);
  L.cap = round_up(static_cast<size_t>(L.cap), MOE_BLOCK_M);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, kRegionAlign);
    return at;
  };
  L.err = take(256);
  L.offsets = take(sizeof(int32_t) * (E + 1));
  L.block_expert = take(sizeof(int32_t) * (L.cap / MOE_BLOCK_M));
  L.sorted = take(sizeof(int32_t) * L.cap);
  L.a_perm = take(sizeof(bf16) * L.cap * H);
  L.z = take(sizeof(bf16) * L.cap * I);
  L.total = off;
  return L;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}

moe_status_t validate_ffn_dims(int32_t H, int32_t I, int32_t E) {
  if (E < 1 || E > 1024) return set_error(MOE_ERR_INVALID_ARG, "E=%d outside [1, 1024]", E);
  if (H < 8 || H % 8 != 0) return set_error(MOE_ERR_INVALID_ARG, "H=%d must be a positive multiple of 8", H);
  if (I < 8 || I % 8 != 0) return set_error(MOE_ERR_INVALID_ARG, "I=%d must be a positive multiple of 8", I);
  if (static_cast<int64_t>(H) > (1 << 24) || static_cast<int64_t>(I) > (1 << 24))
    return set_error(MOE_ERR_INVALID_ARG, "H or I too large");
  return MOE_OK;
}

}  // namespace
}  // namespace gbmoe

using namespace gbmoe;

extern "C" {

int32_t moe_abi_version(void) { return GBMOE_ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_BAD_EXPERT_ID: return "MOE_ERR_BAD_EXPERT_ID";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_NO_DEVICE: return "MOE_ERR_NO_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_error_detail(void) { return g_detail; }

int64_t moe_launch_count(void) { return g_launches; }

moe_status_t moe_set_gemm_tiles(int32_t mode) {
  if (mode < 0 || mode > 2) return set_error(MOE_ERR_INVALID_ARG, "gemm tile mode %d", mode);
  g_gemm_tile_mode.store(mode, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_set_pdl(int32_t enabled) {
  if (enabled != 0 && enabled != 1) return set_error(MOE_ERR_INVALID_ARG, "pdl switch %d", enabled);
  g_pdl.store(enabled, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_set_small_path(int32_t enabled) {
  if (enabled != 0 && enabled != 1)
    return set_error(MOE_ERR_INVALID_ARG, "small-path switch %d", enabled);
  g_small_path.store(enabled, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_set_host_out_direct(int32_t enabled) {
  if (enabled != 0 && enabled != 1)
    return set_error(MOE_ERR_INVALID_ARG, "host output switch %d", enabled);
  g_direct_host_out.store(enabled, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_set_item_rows(int32_t mode) {
  if (mode < 0 || mode > 2) return set_error(MOE_ERR_INVALID_ARG, "item-row format %d", mode);
  g_item_rows.store(mode, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_set_wq_decode(int32_t enabled) {
  if (enabled != 0 && enabled != 1)
    return set_error(MOE_ERR_INVALID_ARG, "weight-only decode switch %d", enabled);
  g_wq_decode.store(enabled, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_set_gather_mode(int32_t mode) {
  if (mode < 0 || mode > 2) return set_error(MOE_ERR_INVALID_ARG, "gather mode %d", mode);
  g_gather_mode.store(mode, std::memory_order_relaxed);
  return MOE_OK;
}

// ---------------------------------------------------------------- route --
static moe_status_t route_check(int64_t M, int32_t E, int32_t top_k, int32_t routing_method,
                                int32_t k_group, int32_t group_count, int32_t group_select_mode,
                                float routed_scaling_factor) {
  if (M < 0) return set_error(MOE_ERR_INVALID_ARG, "M=%lld < 0", (long long)M);
  if (E < 1 || E > 1024) return set_error(MOE_ERR_INVALID_ARG, "E=%d outside [1, 1024]", E);
  if (routing_method != MOE_ROUTE_SOFTMAX && routing_method != MOE_ROUTE_SIGMOID)
    return set_error(MOE_ERR_INVALID_ARG, "routing_method=%d", routing_method);
  if (group_count < 1 || E % group_count != 0)
    return set_error(MOE_ERR_INVALID_ARG, "E=%d not divisible by group_count=%d", E, group_count);
  if (k_group < 1 || k_group > group_count)
    return set_error(MOE_ERR_INVALID_ARG, "k_group=%d outside [1, group_count=%d]", k_group,
                     group_count);
  if (group_select_mode != 0 && group_select_mode != 1)
    return set_error(MOE_ERR_INVALID_ARG, "group_select_mode=%d", group_select_mode);
  if (group_count > 1 && group_select_mode == 1 && E / group_count < 2)
    return set_error(MOE_ERR_INVALID_ARG, "group_select_mode=1 needs >= 2 experts per group");
  const int32_t reachable = (group_count > 1) ? k_group * (E / group_count) : E;
  if (top_k < 1 || top_k > 64 || top_k > reachable)
    return set_error(MOE_ERR_INVALID_ARG, "top_k=%d outside [1, min(64, %d)]", top_k, reachable);
  if (!(routed_scaling_factor == routed_scaling_factor) ||
      routed_scaling_factor > 3.0e38f || routed_scaling_factor < -3.0e38f)
    return set_error(MOE_ERR_INVALID_ARG, "routed_scaling_factor is not finite");
  return MOE_OK;
}

static moe_status_t route_impl(const void* router_logits, int32_t logits_bf16, int64_t M,
                               int32_t E, int32_t top_k, int32_t routing_method,
                               int32_t renormalize, int32_t k_group, int32_t group_count,
                               int32_t group_select_mode, float routed_scaling_factor,
                               float* topk_weights, int32_t* topk_ids, moe_stream_t stream) {
  g_detail[0] = 0;
  if (moe_status_t st = route_check(M, E, top_k, routing_method, k_group, group_count,
                                    group_select_mode, routed_scaling_factor))
    return st;
  if (M == 0) return MOE_OK;
  if (!router_logits || !topk_weights || !topk_ids)
    return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (moe_status_t st = check_device(nullptr)) return st;
  RouteArgs a{router_logits, M, E, top_k, routing_method, renormalize ? 1 : 0, k_group,
              group_count, group_select_mode, routed_scaling_factor, topk_weights, topk_ids,
              logits_bf16};
  return launch_route(a, stream);
}

moe_status_t moe_route(const float* router_logits, int64_t M, int32_t E, int32_t top_k,
                       int32_t routing_method, int32_t renormalize, int32_t k_group,
                       int32_t group_count, int32_t group_select_mode,
                       float routed_scaling_factor, float* topk_weights, int32_t* topk_ids,
                       moe_stream_t stream) {
  return route_impl(router_logits, 0, M, E, top_k, routing_method, renormalize, k_group,
                    group_count, group_select_mode, routed_scaling_factor, topk_weights,
                    topk_ids, stream);
}

moe_status_t moe_route_bf16(const void* router_logits, int64_t M, int32_t E, int32_t top_k,
                            int32_t routing_method, int32_t renormalize, int32_t k_group,
                            int32_t group_count, int32_t group_select_mode,
                            float routed_scaling_factor, float* topk_weights,
                            int32_t* topk_ids, moe_stream_t stream) {
  return route_impl(router_logits, 1, M, E, top_k, routing_method, renormalize, k_group,
                    group_count, group_select_mode, routed_scaling_factor, topk_weights,
                    topk_ids, stream);
}

// ---------------------------------------------------------- router GEMM --
moe_status_t moe_router_logits(const void* hidden, const void* w_gate, const void* b_gate,
                               int64_t M, int32_t H, int32_t E, float* logits,
                               moe_stream_t stream) {
  g_detail[0] = 0;
  if (M < 0) return set_error(MOE_ERR_INVALID_ARG, "M < 0");
  if (H < 8 || H % 8 != 0) return set_error(MOE_ERR_INVALID_ARG, "H=%d must be a positive multiple of 8", H);
  if (E < 1 || E > 1024) return set_error(MOE_ERR_INVALID_ARG, "E=%d outside [1, 1024]", E);
  if (E % 8 != 0)
    return set_error(MOE_ERR_UNSUPPORTED, "E=%d: the router weight rows must be 16-byte multiples (E %% 8 == 0)", E);
  if (M >= (int64_t(1) << 31)) return set_error(MOE_ERR_INVALID_ARG, "M too large");
  if (M == 0) return MOE_OK;
  if (!hidden || !w_gate || !logits) return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(hidden) || !aligned16(w_gate) || !aligned16(logits) ||
      (b_gate && !aligned16(b_gate)))
    return set_error(MOE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  int sms = 0;
  if (moe_status_t st = check_device(&sms)) return st;
  if (router_small_fits(H, E))
    return launch_router_small(static_cast<const bf16*>(hidden), static_cast<const bf16*>(w_gate),
                               static_cast<const bf16*>(b_gate), M, H, E, logits, stream);
  GroupedGemmArgs g{};
  g.a = static_cast<const bf16*>(hidden);
  g.w = static_cast<const bf16*>(w_gate);
  g.bias = static_cast<const bf16*>(b_gate);
  g.cap = M;
  g.E = 1;
  g.N = E;
  g.K = H;
  g.out = logits;
  g.sentinel = static_cast<int32_t>(M);
  g.num_sms = sms;
  g.rows_hint = M;
  return launch_dense_f32(g, stream);
}

// ---------------------------------------------------------------- align --
size_t moe_align_capacity(int64_t M, int32_t top_k, int32_t E, int32_t block_m) {
  if (M < 0 || top_k < 1 || E < 1 || block_m < 1) return 0;
  return static_cast<size_t>(align_cap(M * top_k, E, block_m));
}

size_t moe_align_scratch_size(int64_t M, int32_t top_k, int32_t E) {
  if (M < 0 || top_k < 1 || E < 1) return 0;
  return align_scratch_bytes(M * top_k, E);
}

moe_status_t moe_align(const int32_t* topk_ids, int64_t M, int32_t top_k, int32_t E,
                       int32_t block_m, int32_t* sorted_token_ids, int32_t* expert_offsets,
                       int32_t* expert_num_tokens, int32_t* block_expert_ids, void* scratch,
                       size_t scratch_bytes, int32_t* error_word, moe_stream_t stream) {
  g_detail[0] = 0;
  if (M < 0) return set_error(MOE_ERR_INVALID_ARG, "M < 0");
  if (E < 1 || E > 1024) return set_error(MOE_ERR_INVALID_ARG, "E=%d outside [1, 1024]", E);
  if (top_k < 1 || top_k > 1024) return set_error(MOE_ERR_INVALID_ARG, "top_k=%d", top_k);
  if (block_m < 1 || block_m > 1024)
    return set_error(MOE_ERR_INVALID_ARG, "block_m=%d outside [1, 1024]", block_m);
  const int64_t R = M * top_k;
  if (align_cap(R, E, block_m) >= (int64_t(1) << 31))
    return set_error(MOE_ERR_INVALID_ARG, "too many routed items for int32 indices");
  if (!expert_offsets || !expert_num_tokens || !block_expert_ids || !sorted_token_ids)
    return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (R > 0 && !topk_ids) return set_error(MOE_ERR_INVALID_ARG, "null topk_ids");
  const size_t need = align_scratch_bytes(R, E);
  if (need > 0 && (scratch == nullptr || scratch_bytes < need))
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL, "align scratch needs %zu bytes", need);
  if (moe_status_t st = check_device(nullptr)) return st;
  AlignArgs a{topk_ids, R, E, block_m, sorted_token_ids, expert_offsets, expert_num_tokens,
              block_expert_ids, static_cast<int32_t*>(scratch), align_cap(R, E, block_m),
              error_word};
  return launch_align(a, stream);
}

moe_status_t moe_align_static_scratch(const int32_t* topk_ids, int64_t M, int32_t top_k,
                                      int32_t E, int32_t block_m, int32_t* sorted_token_ids,
                                      int32_t* expert_offsets, int32_t* expert_num_tokens,
                                      int32_t* block_expert_ids, int32_t* error_word,
                                      moe_stream_t stream) {
  g_detail[0] = 0;
  if (M < 0) return set_error(MOE_ERR_INVALID_ARG, "M < 0");
  if (E < 1 || E > 1024) return set_error(MOE_ERR_INVALID_ARG, "E=%d outside [1, 1024]", E);
  if (top_k < 1 || top_k > 1024) return set_error(MOE_ERR_INVALID_ARG, "top_k=%d", top_k);
  if (block_m < 1 || block_m > 1024)
    return set_error(MOE_ERR_INVALID_ARG, "block_m=%d outside [1, 1024]", block_m);
  const int64_t R = M * top_k;
  if (align_cap(R, E, block_m) >= (int64_t(1) << 31))
    return set_error(MOE_ERR_INVALID_ARG, "too many routed items for int32 indices");
  if (!expert_offsets || !expert_num_tokens || !block_expert_ids || !sorted_token_ids)
    return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (R > 0 && !topk_ids) return set_error(MOE_ERR_INVALID_ARG, "null topk_ids");
  if (align_scratch_bytes(R, E) > sizeof(int32_t) * size_t(MOE_ALIGN_STATIC_SCRATCH_INTS))
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL,
                     "ceil(M*top_k/256)*E exceeds the static scratch of %d ints",
                     MOE_ALIGN_STATIC_SCRATCH_INTS);
  if (moe_status_t st = check_device(nullptr)) return st;
  AlignArgs a{topk_ids, R, E, block_m, sorted_token_ids, expert_offsets, expert_num_tokens,
              block_expert_ids, nullptr, align_cap(R, E, block_m), error_word};
  return launch_align_static_scratch(a, stream);
}

// -------------------------------------------------------------- forward --
moe_status_t moe_workspace_size(int64_t M, int32_t H, int32_t I, int32_t E, int32_t top_k,
                                int32_t reduce_mode, size_t* bytes) {
  g_detail[0] = 0;
  if (!bytes) return set_error(MOE_ERR_INVALID_ARG, "null bytes");
  if (M < 0) return set_error(MOE_ERR_INVALID_ARG, "M < 0");
  if (moe_status_t st = validate_ffn_dims(H, I, E)) return st;
  if (top_k < 1 || top_k > 64) return set_error(MOE_ERR_INVALID_ARG, "top_k=%d outside [1, 64]", top_k);
  if (reduce_mode != MOE_REDUCE_AUTO && reduce_mode != MOE_REDUCE_SEPARATE &&
      reduce_mode != MOE_REDUCE_EPILOGUE_ATOMIC)
    return set_error(MOE_ERR_INVALID_ARG, "reduce_mode=%d", reduce_mode);
  const int64_t Mc = M < MOE_CHUNK_TOKENS ? M : MOE_CHUNK_TOKENS;
  *bytes = fwd_layout(Mc, H, I, E, top_k).total;
  return MOE_OK;
}

int32_t* moe_workspace_error_word(void* workspace) { return static_cast<int32_t*>(workspace); }

moe_status_t moe_forward(const void* hidden, const float* topk_weights,
                         const int32_t* topk_ids, int64_t M, int32_t H, int32_t I, int32_t E,
                         int32_t top_k, const void* w13, const void* w2, const void* w13_bias,
                         const void* w2_bias, void* workspace, size_t workspace_bytes,
                         int32_t reduce_mode, void* out, moe_stream_t stream) {
  moe_forward_opts_t o{};
  o.reduce_mode = reduce_mode;
  return moe_forward_opts(hidden, topk_weights, topk_ids, M, H, I, E, top_k, w13, w2, w13_bias,
                          w2_bias, workspace, workspace_bytes, &o, out, stream);
}

// Argument checks of moe_forward_opts (nothing is enqueued); *sms gets the
// device's SM count when M > 0.
static moe_status_t forward_check(const void* hidden, const float* topk_weights,
                                  const int32_t* topk_ids, int64_t M, int32_t H, int32_t I,
                                  int32_t E, int32_t top_k, const void* w13, const void* w2,
                                  const void* w13_bias, const void* w2_bias,
                                  const void* workspace, size_t workspace_bytes,
                                  const moe_forward_opts_t* opts, const void* out, int* sms) {
  if (!opts) return set_error(MOE_ERR_INVALID_ARG, "null opts");
  const int32_t reduce_mode = opts->reduce_mode;
  if (opts->apply_router_weight_on_input != 0 && opts->apply_router_weight_on_input != 1)
    return set_error(MOE_ERR_INVALID_ARG, "apply_router_weight_on_input must be 0 or 1");
  if (opts->expert_map != nullptr &&
      (opts->num_global_experts < 1 || opts->num_global_experts > (1 << 20)))
    return set_error(MOE_ERR_INVALID_ARG, "num_global_experts=%d outside [1, 2^20]",
                     opts->num_global_experts);
  size_t need = 0;
  if (moe_status_t st = moe_workspace_size(M, H, I, E, top_k, reduce_mode, &need)) return st;
  if (M == 0) return MOE_OK;
  if (!hidden || !topk_weights || !topk_ids || !w13 || !w2 || !workspace || !out)
    return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(hidden) || !aligned16(w13) || !aligned16(w2) || !aligned16(out) ||
      !aligned16(topk_weights) || (w13_bias && !aligned16(w13_bias)) ||
      (w2_bias && !aligned16(w2_bias)))
    return set_error(MOE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return set_error(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < need)
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes, got %zu", need,
                     workspace_bytes);
  return check_device(sms);
}

// The forward's launches (arguments already checked, M > 0).  wait_rows: an
// event the stream waits for before the hidden rows are first read (their
// copy on another stream), or null.
static moe_status_t forward_launch(const void* hidden, const float* topk_weights,
                                   const int32_t* topk_ids, int64_t M, int32_t H, int32_t I,
                                   int32_t E, int32_t top_k, const void* w13, const void* w2,
                                   const void* w13_bias, const void* w2_bias, void* workspace,
                                   const moe_forward_opts_t* opts, void* out, int sms,
                                   cudaEvent_t wait_rows, cudaStream_t s,
                                   bool reset_error = true) {
  const int32_t reduce_mode = opts->reduce_mode;
  const bool weight_on_input = opts->apply_router_weight_on_input != 0;
  const int64_t Mc_max = M < MOE_CHUNK_TOKENS ? M : MOE_CHUNK_TOKENS;
  const FwdLayout L = fwd_layout(Mc_max, H, I, E, top_k);
  int32_t* err = at<int32_t>(workspace, L.err);
  // the error word and, after it, the GEMMs' tile-schedule counters
  int32_t* sched1 = err + 16;  // GEMM1 {next tile, CTAs done}
  int32_t* sched2 = err + 24;  // GEMM2
  // (the error word and the counters are cleared by the first chunk's plan)

  const bf16* x = static_cast<const bf16*>(hidden);
  bf16* y = static_cast<bf16*>(out);
  // a small call: the whole layer in two kernels (the plan, gather and
  // reduce folded into the GEMMs; an atomic k-sum, as the automatic choice
  // allows)
  if (small_path_enabled() && reduce_mode == MOE_REDUCE_AUTO && !weight_on_input &&
      opts->expert_map == nullptr && reset_error && small_forward_applies(M, H, I, E, top_k)) {
    if (wait_rows != nullptr && cudaStreamWaitEvent(s, wait_rows, 0) != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "cudaStreamWaitEvent: %s",
                       cudaGetErrorString(cudaGetLastError()));
    SmallArgs sa{};
    sa.x = x;
    sa.w13 = static_cast<const bf16*>(w13);
    sa.w2 = static_cast<const bf16*>(w2);
    sa.b13 = static_cast<const bf16*>(w13_bias);
    sa.b2 = static_cast<const bf16*>(w2_bias);
    sa.ids = topk_ids;
    sa.weights = topk_weights;
    sa.z = at<bf16>(workspace, L.z);
    sa.acc = at<float>(workspace, L.o);
    sa.counter = at<int32_t>(workspace, L.a_perm);  // the gathered rows are not used
    sa.error_word = err;
    sa.y = y;
    sa.M = M;
    sa.H = H;
    sa.I = I;
    sa.E = E;
    sa.k = top_k;
    return launch_small_forward(sa, s);
  }
  for (int64_t c0 = 0; c0 < M; c0 += Mc_max) {
    const int64_t Mc = (M - c0) < Mc_max ? (M - c0) : Mc_max;
    const int64_t Rc = Mc * top_k;
    const int64_t cap = align_cap(Rc, E, MOE_BLOCK_M);
    int32_t* sorted = at<int32_t>(workspace, L.sorted);
    int32_t* offsets = at<int32_t>(workspace, L.offsets);
    int32_t* inv = at<int32_t>(workspace, L.inv);
    AlignArgs al{topk_ids + c0 * top_k, Rc, E, MOE_BLOCK_M, sorted, offsets,
                 at<int32_t>(workspace, L.counts), at<int32_t>(workspace, L.block_expert),
                 at<int32_t>(workspace, L.scratch), cap, err, inv};
    al.expert_map = opts->expert_map;
    al.E_global = opts->num_global_experts;
    if (reset_error && c0 == 0) {
      al.zero_words = err;
      al.zero_count = 32;
    }
    if (moe_status_t st = launch_align(al, s)) return st;

    bf16* a_perm = at<bf16>(workspace, L.a_perm);
    GatherArgs ga{x + c0 * H, sorted, offsets, E, top_k, static_cast<int32_t>(Rc), H, cap,
                  a_perm};
    ga.inv = inv;  // each token row read once
    ga.tokens = Mc;
    if (wait_rows != nullptr && c0 == 0 && cudaStreamWaitEvent(s, wait_rows, 0) != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "cudaStreamWaitEvent: %s",
                       cudaGetErrorString(cudaGetLastError()));
    // GEMM1 copies its A rows from the token rows itself, or they are
    // gathered into a_perm first
    const bool fused_gather = gemm1_fused_gather(Rc, H, I, E);
    if (!fused_gather)
      if (moe_status_t st = launch_gather(ga, s)) return st;

    bf16* z = at<bf16>(workspace, L.z);
    GroupedGemmArgs g1{};
    g1.a = a_perm;
    g1.w = static_cast<const bf16*>(w13);
    g1.bias = static_cast<const bf16*>(w13_bias);
    g1.cap = cap;
    g1.E = E;
    g1.N = I;
    g1.K = H;
    g1.offsets = offsets;
    g1.out = z;
    g1.row_index = sorted;
    g1.sentinel = static_cast<int32_t>(Rc);
    if (weight_on_input) g1.gemm1_row_weight = topk_weights + c0 * top_k;
    g1.error_word = err;
    g1.num_sms = sms;
    g1.rows_hint = Rc;
    if (fused_gather) {
      g1.a_rows = x + c0 * H;
      g1.div = top_k;
    }
    g1.sched = sched1;
    if (moe_status_t st = launch_gemm1_swiglu(g1, s)) return st;

    float* o = at<float>(workspace, L.o);
    const int32_t mode = pick_reduce(Mc, H, top_k, reduce_mode);
    if (mode == MOE_REDUCE_EPILOGUE_ATOMIC &&
        cudaMemsetAsync(o, 0, sizeof(float) * Mc * H, s) != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(cudaGetLastError()));
    GroupedGemmArgs g2{};
    g2.a = z;
    g2.w = static_cast<const bf16*>(w2);
    g2.bias = static_cast<const bf16*>(w2_bias);
    g2.cap = cap;
    g2.E = E;
    g2.N = H;
    g2.K = I;
    g2.offsets = offsets;
    g2.out = o;
    g2.row_index = sorted;
    g2.row_weight = weight_on_input ? nullptr : topk_weights + c0 * top_k;
    g2.sentinel = static_cast<int32_t>(Rc);
    g2.div = top_k;
    g2.sched = sched2;
    g2.error_word = err;
    g2.num_sms = sms;
    g2.rows_hint = Rc;
    if (mode == MOE_REDUCE_EPILOGUE_ATOMIC) {
      if (moe_status_t st = launch_gemm2_atomic_f32(g2, s)) return st;
      if (moe_status_t st = launch_cast_f32_bf16(o, Mc * H, y + c0 * H, s)) return st;
    } else if (item_rows_fp16(top_k)) {
      // fp16 rows [cap, H] and their exponents [ceil(H/32)][cap] share the
      // fp32 rows' region
      g2.o_exp = reinterpret_cast<uint8_t*>(o) + static_cast<size_t>(cap) * H * 2;
      if (moe_status_t st = launch_gemm2_sorted_f16(g2, s)) return st;
      if (moe_status_t st = launch_reduce_sorted_f16(o, g2.o_exp, cap, inv, Mc, top_k, H,
                                                     y + c0 * H, s))
        return st;
    } else {
      if (moe_status_t st = launch_gemm2_sorted_f32(g2, s)) return st;
      if (moe_status_t st = launch_reduce_sorted(o, inv, Mc, top_k, H, y + c0 * H, s)) return st;
    }
  }
  return MOE_OK;
}

moe_status_t moe_forward_opts(const void* hidden, const float* topk_weights,
                              const int32_t* topk_ids, int64_t M, int32_t H, int32_t I,
                              int32_t E, int32_t top_k, const void* w13, const void* w2,
                              const void* w13_bias, const void* w2_bias, void* workspace,
                              size_t workspace_bytes, const moe_forward_opts_t* opts, void* out,
                              moe_stream_t stream) {
  int sms = 0;
  if (moe_status_t st = forward_check(hidden, topk_weights, topk_ids, M, H, I, E, top_k, w13, w2,
                                      w13_bias, w2_bias, workspace, workspace_bytes, opts, out,
                                      &sms))
    return st;
  if (M == 0) return MOE_OK;
  return forward_launch(hidden, topk_weights, topk_ids, M, H, I, E, top_k, w13, w2, w13_bias,
                        w2_bias, workspace, opts, out, sms, nullptr, stream);
}

// ------------------------------------------------------- host-memory step --
namespace {
// Per host thread and device: the stream the hidden rows are copied on and
// the events that fork it from, and join it to, the caller's stream.
constexpr int kMaxHostChunks = 2;
struct CopyLane {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t fork = nullptr, join_in = nullptr, join_out = nullptr;
  cudaEvent_t logits[kMaxHostChunks] = {}, rows[kMaxHostChunks] = {}, out[kMaxHostChunks] = {};
};
constexpr int kMaxDevices = 64;

moe_status_t copy_lane(CopyLane** lane) {
  thread_local CopyLane lanes[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_error(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(cudaGetLastError()));
  CopyLane& l = lanes[dev];
  if (l.h2d == nullptr) {
    bool ok = cudaStreamCreateWithFlags(&l.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&l.d2h, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* ev : {&l.fork, &l.join_in, &l.join_out})
      ok = ok && cudaEventCreateWithFlags(ev, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < kMaxHostChunks; ++i)
      for (cudaEvent_t* ev : {&l.logits[i], &l.rows[i], &l.out[i]})
        ok = ok && cudaEventCreateWithFlags(ev, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      l.h2d = nullptr;
      return set_error(MOE_ERR_CUDA, "copy streams: %s", cudaGetErrorString(cudaGetLastError()));
    }
  }
  *lane = &l;
  return MOE_OK;
}
}  // namespace

moe_status_t moe_forward_host(const moe_host_io_t* io, int64_t M, int32_t H, int32_t I,
                              int32_t E, const moe_route_params_t* route, const void* w13,
                              const void* w2, const void* w13_bias, const void* w2_bias,
                              void* workspace, size_t workspace_bytes, int32_t reduce_mode,
                              moe_stream_t stream) {
  g_detail[0] = 0;
  if (!io || !route) return set_error(MOE_ERR_INVALID_ARG, "null io or route");
  if (moe_status_t st = route_check(M, E, route->top_k, route->routing_method, route->k_group,
                                    route->group_count, route->group_select_mode,
                                    route->routed_scaling_factor))
    return st;
  moe_forward_opts_t o{};
  o.reduce_mode = reduce_mode;
  int sms = 0;
  if (moe_status_t st = forward_check(io->d_hidden, io->topk_weights, io->topk_ids, M, H, I, E,
                                      route->top_k, w13, w2, w13_bias, w2_bias, workspace,
                                      workspace_bytes, &o, io->d_out, &sms))
    return st;
  if (M == 0) return MOE_OK;
  if (!io->h_hidden || !io->h_logits || !io->h_out || !io->d_logits)
    return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  CopyLane* lane = nullptr;
  if (moe_status_t st = copy_lane(&lane)) return st;
  cudaStream_t s = stream;
  auto cuda_fail = [](const char* what) {
    return set_error(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(cudaGetLastError()));
  };
  // Two token chunks -- the second chunk's rows copied in while the first is
  // computed, the first chunk's output copied out while the second is --
  // when each half still averages >= 512 routed rows per expert (the GEMMs
  // keep their tile shape, so the results are those of one pass) and the
  // copies are large against the weights, which each chunk reads again:
  // about half the copy time (host link ~300 GB/s) is hidden, one more
  // pass over the weights (HBM ~6.8 TB/s) is paid.  Measured through this
  // call: Qwen-MoE shape (142 MB copied, 1.2 GB of weights) 1.985 -> 1.870
  // ms in two chunks; Mixtral shape (67 MB, 2.8 GB) 2.111 -> 2.300 ms.
  const int32_t k = route->top_k;
  const int64_t copy_bytes = M * (int64_t{4} * H + int64_t{4} * E);
  const int64_t weight_bytes = int64_t{6} * E * H * I;
  const int chunks =
      ((M / 2) * k >= int64_t{512} * E && copy_bytes * 11 > weight_bytes) ? 2 : 1;
  int64_t m0s[kMaxHostChunks + 1];
  for (int c = 0; c <= chunks; ++c) m0s[c] = M * c / chunks;
  // fork the copy streams off the caller's stream; join them on every way out
  if (cudaEventRecord(lane->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(lane->h2d, lane->fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(lane->d2h, lane->fork, 0) != cudaSuccess)
    return cuda_fail("copy stream fork");
  auto join = [&]() {
    cudaEventRecord(lane->join_in, lane->h2d);
    cudaEventRecord(lane->join_out, lane->d2h);
    cudaStreamWaitEvent(s, lane->join_in, 0);
    cudaStreamWaitEvent(s, lane->join_out, 0);
  };
  const bf16* hx = static_cast<const bf16*>(io->h_hidden);
  bf16* hy = static_cast<bf16*>(io->h_out);
  bf16* dx = static_cast<bf16*>(io->d_hidden);
  bf16* dy = static_cast<bf16*>(io->d_out);
  // The last chunk's output follows its reduce with nothing left to overlap:
  // into a pinned (device-mapped, 16-byte aligned) output buffer the reduce
  // writes it directly over the host link instead of through d_out and a
  // device-to-host copy.  Earlier chunks keep the copy, which runs under the
  // next chunk's compute; pageable memory always takes it.
  // (page-locked under this device: memory pinned while another device was
  // current may not be mapped for this one)
  bf16* y_direct = nullptr;
  if (direct_host_out()) {
    cudaPointerAttributes pa{};
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaPointerGetAttributes(&pa, io->h_out) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.device == dev && pa.devicePointer != nullptr &&
        reinterpret_cast<uintptr_t>(pa.devicePointer) % 16 == 0)
      y_direct = static_cast<bf16*>(pa.devicePointer);
    cudaGetLastError();
  }
  for (int c = 0; c < chunks; ++c) {
    const int64_t m0 = m0s[c], mc = m0s[c + 1] - m0s[c];
    if (cudaMemcpyAsync(io->d_logits + m0 * E, io->h_logits + m0 * E,
                        static_cast<size_t>(mc) * E * sizeof(float), cudaMemcpyHostToDevice,
                        lane->h2d) != cudaSuccess ||
        cudaEventRecord(lane->logits[c], lane->h2d) != cudaSuccess ||
        cudaMemcpyAsync(dx + m0 * H, hx + m0 * H, static_cast<size_t>(mc) * H * sizeof(bf16),
                        cudaMemcpyHostToDevice, lane->h2d) != cudaSuccess ||
        cudaEventRecord(lane->rows[c], lane->h2d) != cudaSuccess) {
      join();
      return cuda_fail("host-to-device copy");
    }
  }
  for (int c = 0; c < chunks; ++c) {
    const int64_t m0 = m0s[c], mc = m0s[c + 1] - m0s[c];
    const bool direct = y_direct != nullptr && c == chunks - 1;
    moe_status_t st = MOE_OK;
    if (cudaStreamWaitEvent(s, lane->logits[c], 0) != cudaSuccess) st = cuda_fail("logits wait");
    if (st == MOE_OK)
      st = route_impl(io->d_logits + m0 * E, 0, mc, E, k, route->routing_method,
                      route->renormalize, route->k_group, route->group_count,
                      route->group_select_mode, route->routed_scaling_factor,
                      io->topk_weights + m0 * k, io->topk_ids + m0 * k, s);
    // the rows' copy overlaps routing and the plan: the forward waits for it
    // right before the rows are first read
    if (st == MOE_OK)
      st = forward_launch(dx + m0 * H, io->topk_weights + m0 * k, io->topk_ids + m0 * k, mc, H,
                          I, E, k, w13, w2, w13_bias, w2_bias, workspace, &o,
                          (direct ? y_direct : dy) + m0 * H, sms, lane->rows[c], s,
                          /*reset_error=*/c == 0);
    if (st == MOE_OK && !direct &&
        (cudaEventRecord(lane->out[c], s) != cudaSuccess ||
         cudaStreamWaitEvent(lane->d2h, lane->out[c], 0) != cudaSuccess ||
         cudaMemcpyAsync(hy + m0 * H, dy + m0 * H, static_cast<size_t>(mc) * H * sizeof(bf16),
                         cudaMemcpyDeviceToHost, lane->d2h) != cudaSuccess))
      st = cuda_fail("device-to-host copy");
    if (st != MOE_OK) {
      cudaStreamWaitEvent(s, lane->rows[c], 0);
      join();
      return st;
    }
  }
  join();
  return MOE_OK;
}

// ------------------------------------------------------------ FP8 W8A8 --
namespace {
struct Fp8Layout {
  int64_t cap = 0;
  size_t err = 0, counts = 0, offsets = 0, block_expert = 0, sorted = 0, scratch = 0, inv = 0,
         a8 = 0, a_scale = 0, z = 0, z8 = 0, z_scale = 0, o = 0, total = 0;
};

Fp8Layout fp8_layout(int64_t Mc, int32_t H, int32_t I, int32_t E, int32_t k) {
  Fp8Layout L;
  const int64_t Rc = Mc * k;
  L.cap = align_cap(Rc, E, MOE_BLOCK_M);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, kRegionAlign);
    return at;
  };
  L.err = take(256);
  L.counts = take(sizeof(int32_t) * E);
  L.offsets = take(sizeof(int32_t) * (E + 1));
  L.block_expert = take(sizeof(int32_t) * (L.cap / MOE_BLOCK_M));
  L.sorted = take(sizeof(int32_t) * L.cap);
  L.scratch = take(align_scratch_bytes(Rc, E));
  L.inv = take(sizeof(int32_t) * Rc);
  L.a8 = take(static_cast<size_t>(L.cap) * H);
  // scales per sorted row, or per (row, 128-wide group) in block mode
  L.a_scale = take(sizeof(float) * L.cap * static_cast<size_t>(ceil_div(H, 128)));
  L.z = take(sizeof(bf16) * L.cap * I);
  L.z8 = take(static_cast<size_t>(L.cap) * I);
  L.z_scale = take(sizeof(float) * L.cap * static_cast<size_t>(ceil_div(I, 128)));
  L.o = take(sizeof(float) * L.cap * H);
  L.total = off;
  return L;
}
}  // namespace

moe_status_t moe_workspace_size_fp8(int64_t M, int32_t H, int32_t I, int32_t E, int32_t top_k,
                                    size_t* bytes) {
  g_detail[0] = 0;
  if (!bytes) return set_error(MOE_ERR_INVALID_ARG, "null bytes");
  if (M < 0) return set_error(MOE_ERR_INVALID_ARG, "M < 0");
  if (moe_status_t st = validate_ffn_dims(H, I, E)) return st;
  if (H % 16 != 0 || I % 16 != 0)
    return set_error(MOE_ERR_INVALID_ARG, "FP8 needs H and I multiples of 16 (16-byte rows)");
  if (top_k < 1 || top_k > 64) return set_error(MOE_ERR_INVALID_ARG, "top_k=%d outside [1, 64]", top_k);
  const int64_t Mc = M < MOE_CHUNK_TOKENS ? M : MOE_CHUNK_TOKENS;
  *bytes = fp8_layout(Mc, H, I, E, top_k).total;
  return MOE_OK;
}

moe_status_t moe_forward_fp8(const void* hidden, const float* topk_weights,
                             const int32_t* topk_ids, int64_t M, int32_t H, int32_t I,
                             int32_t E, int32_t top_k, const moe_fp8_weights_t* w,
                             const void* w13_bias, const void* w2_bias, void* workspace,
                             size_t workspace_bytes, void* out, moe_stream_t stream) {
  size_t need = 0;
  if (moe_status_t st = moe_workspace_size_fp8(M, H, I, E, top_k, &need)) return st;
  if (M == 0) return MOE_OK;
  if (!w || !w->w13 || !w->w2 || !w->w13_scale || !w->w2_scale)
    return set_error(MOE_ERR_INVALID_ARG, "null FP8 weights or scales");
  if (w->scale_mode < MOE_FP8_SCALE_EXPERT || w->scale_mode > MOE_FP8_SCALE_BLOCK)
    return set_error(MOE_ERR_INVALID_ARG, "scale_mode=%d", w->scale_mode);
  const bool block = w->scale_mode == MOE_FP8_SCALE_BLOCK;
  if (block && (H % 128 != 0 || I % 128 != 0 || I > 32768))
    return set_error(MOE_ERR_INVALID_ARG,
                     "block-wise FP8 scales need H and I multiples of 128, I <= 32768 (H=%d I=%d)",
                     H, I);
  if (!hidden || !topk_weights || !topk_ids || !workspace || !out)
    return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(hidden) || !aligned16(w->w13) || !aligned16(w->w2) || !aligned16(out) ||
      !aligned16(w->w13_scale) || !aligned16(w->w2_scale) || (w13_bias && !aligned16(w13_bias)) ||
      (w2_bias && !aligned16(w2_bias)))
    return set_error(MOE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return set_error(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < need)
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes, got %zu", need,
                     workspace_bytes);
  int sms = 0;
  if (moe_status_t st = check_device(&sms)) return st;
  cudaStream_t s = stream;
  const int64_t Mc_max = M < MOE_CHUNK_TOKENS ? M : MOE_CHUNK_TOKENS;
  const Fp8Layout L = fp8_layout(Mc_max, H, I, E, top_k);
  int32_t* err = at<int32_t>(workspace, L.err);
  // the error word and the GEMMs' tile-schedule counters after it
  if (cudaMemsetAsync(err, 0, 32 * sizeof(int32_t), s) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(cudaGetLastError()));
  const bf16* x = static_cast<const bf16*>(hidden);
  bf16* y = static_cast<bf16*>(out);
  for (int64_t c0 = 0; c0 < M; c0 += Mc_max) {
    const int64_t Mc = (M - c0) < Mc_max ? (M - c0) : Mc_max;
    const int64_t Rc = Mc * top_k;
    const int64_t cap = align_cap(Rc, E, MOE_BLOCK_M);
    int32_t* sorted = at<int32_t>(workspace, L.sorted);
    int32_t* offsets = at<int32_t>(workspace, L.offsets);
    int32_t* inv = at<int32_t>(workspace, L.inv);
    AlignArgs al{topk_ids + c0 * top_k, Rc, E, MOE_BLOCK_M, sorted, offsets,
                 at<int32_t>(workspace, L.counts), at<int32_t>(workspace, L.block_expert),
                 at<int32_t>(workspace, L.scratch), cap, err, inv};
    if (moe_status_t st = launch_align(al, s)) return st;
    // quantise each token row once (E4M3, one scale per row, or per row and
    // 128-column group) into its k sorted rows; per row, zero those rows' z
    // amax for GEMM1's epilogue
    uint8_t* a8 = at<uint8_t>(workspace, L.a8);
    float* a_scale = at<float>(workspace, L.a_scale);
    float* z_scale = at<float>(workspace, L.z_scale);
    QuantTokensArgs qa{x + c0 * H, inv, Mc, top_k, H, a8, a_scale, block ? nullptr : z_scale};
    if (block) {
      if (moe_status_t st = launch_quant_tokens_group_fp8(qa, cap, s)) return st;
    } else {
      if (moe_status_t st = launch_quant_tokens_fp8(qa, s)) return st;
    }
    bf16* z = at<bf16>(workspace, L.z);
    uint8_t* z8 = at<uint8_t>(workspace, L.z8);
    GroupedGemmArgs g1{};
    g1.a = reinterpret_cast<const bf16*>(a8);
    g1.w = static_cast<const bf16*>(w->w13);
    g1.bias = static_cast<const bf16*>(w13_bias);
    g1.cap = cap;
    g1.E = E;
    g1.N = I;
    g1.K = H;
    g1.offsets = offsets;
    g1.out = block ? static_cast<void*>(z8) : static_cast<void*>(z);
    g1.row_index = sorted;
    g1.sentinel = static_cast<int32_t>(Rc);
    g1.error_word = err;
    g1.sched = err + 16;  // used by the CTA-pair tiles
    g1.num_sms = sms;
    g1.rows_hint = Rc;
    g1.a_scale = a_scale;
    g1.w_scale = w->w13_scale;
    g1.w_scale_per_channel = w->scale_mode == MOE_FP8_SCALE_CHANNEL;
    // block scales: GEMM1 quantises z itself (its tile's 128 z columns are
    // one group); per row: it takes each row's amax for the pass below
    if (block) g1.z_group_scale = z_scale;
    else g1.row_amax = z_scale;
    if (moe_status_t st = block ? launch_gemm1_swiglu_fp8_block(g1, s) : launch_gemm1_swiglu_fp8(g1, s))
      return st;
    if (!block) {
      // quantise z per row for the second GEMM (amax taken by GEMM1)
      QuantSortedArgs qz{z, sorted, offsets, E, static_cast<int32_t>(Rc), I, cap, z8, z_scale};
      if (moe_status_t st = launch_quant_sorted_fp8(qz, s)) return st;
    }
    float* o = at<float>(workspace, L.o);
    GroupedGemmArgs g2{};
    g2.a = reinterpret_cast<const bf16*>(z8);
    g2.w = static_cast<const bf16*>(w->w2);
    g2.bias = static_cast<const bf16*>(w2_bias);
    g2.cap = cap;
    g2.E = E;
    g2.N = H;
    g2.K = I;
    g2.offsets = offsets;
    g2.out = o;
    g2.row_index = sorted;
    g2.row_weight = topk_weights + c0 * top_k;
    g2.sentinel = static_cast<int32_t>(Rc);
    g2.div = top_k;
    g2.error_word = err;
    g2.sched = err + 24;
    g2.num_sms = sms;
    g2.rows_hint = Rc;
    g2.a_scale = z_scale;
    g2.w_scale = w->w2_scale;
    g2.w_scale_per_channel = w->scale_mode == MOE_FP8_SCALE_CHANNEL;
    if (!block && item_rows_fp16(top_k)) {
      g2.o_exp = reinterpret_cast<uint8_t*>(o) + static_cast<size_t>(cap) * H * 2;
      if (moe_status_t st = launch_gemm2_sorted_f16_fp8(g2, s)) return st;
      if (moe_status_t st = launch_reduce_sorted_f16(o, g2.o_exp, cap, inv, Mc, top_k, H,
                                                     y + c0 * H, s))
        return st;
      continue;
    }
    if (moe_status_t st = block ? launch_gemm2_sorted_fp8_block(g2, s) : launch_gemm2_sorted_fp8(g2, s))
      return st;
    if (moe_status_t st = launch_reduce_sorted(o, inv, Mc, top_k, H, y + c0 * H, s)) return st;
  }
  return MOE_OK;
}

moe_status_t moe_quant_rows_fp8(const void* x, int64_t M, int32_t H, void* q8, float* scale,
                                moe_stream_t stream) {
  g_detail[0] = 0;
  if (M < 0) return set_error(MOE_ERR_INVALID_ARG, "M < 0");
  if (H <= 0 || H % 16 != 0) return set_error(MOE_ERR_INVALID_ARG, "H=%d not a positive multiple of 16", H);
  if (M == 0) return MOE_OK;
  if (!x || !q8 || !scale) return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(q8) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
    return set_error(MOE_ERR_INVALID_ARG, "x and q8 must be 16-byte aligned");
  int sms = 0;
  if (moe_status_t st = check_device(&sms)) return st;
  QuantTokensArgs qa{static_cast<const bf16*>(x), nullptr, M, 1, H, static_cast<uint8_t*>(q8),
                     scale, nullptr};
  return launch_quant_tokens_fp8(qa, stream);
}

// ------------------------------------------- weight-only quantised --
namespace {
moe_status_t validate_wq_format(int32_t format, int32_t G, const void* zero) {
  if (format < MOE_WQ_INT4 || format > MOE_WQ_MXFP6_E2M3)
    return set_error(MOE_ERR_INVALID_ARG, "weight format %d", format);
  if (G < 32 || G % 32 != 0)
    return set_error(MOE_ERR_INVALID_ARG, "group_size=%d must be a positive multiple of 32", G);
  const bool mx = format >= MOE_WQ_MXFP4;
  if (mx && G != 32)
    return set_error(MOE_ERR_INVALID_ARG, "MX scales cover blocks of 32 (group_size=%d)", G);
  if (mx && zero != nullptr) return set_error(MOE_ERR_INVALID_ARG, "MX formats have no zero points");
  return MOE_OK;
}
}  // namespace

moe_status_t moe_dequant_weights(int32_t format, const void* codes, const void* scale,
                                 const void* zero, int32_t E, int32_t K, int32_t N,
                                 int32_t group_size, void* out, moe_stream_t stream) {
  g_detail[0] = 0;
  if (moe_status_t st = validate_wq_format(format, group_size, zero)) return st;
  if (E < 1 || K < 1 || N < 16 || N % 16 != 0)
    return set_error(MOE_ERR_INVALID_ARG, "E=%d K=%d N=%d (N a positive multiple of 16)", E, K, N);
  if (K % group_size != 0)
    return set_error(MOE_ERR_INVALID_ARG, "group_size=%d does not divide K=%d", group_size, K);
  if (static_cast<int64_t>(E) * K * N >= (int64_t(1) << 40))
    return set_error(MOE_ERR_INVALID_ARG, "E*K*N too large");
  if (!codes || !scale || !out) return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(codes) || !aligned16(scale) || !aligned16(out) || (zero && !aligned16(zero)))
    return set_error(MOE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  int sms = 0;
  if (moe_status_t st = check_device(&sms)) return st;
  WqDequantArgs a{format, codes, scale, zero, E, K, N, group_size, static_cast<bf16*>(out)};
  return launch_dequant_weights(a, stream);
}

moe_status_t moe_forward_wq(const void* hidden, const float* topk_weights,
                            const int32_t* topk_ids, int64_t M, int32_t H, int32_t I, int32_t E,
                            int32_t top_k, const moe_wq_weights_t* w, const void* w13_bias,
                            const void* w2_bias, void* workspace, size_t workspace_bytes,
                            void* out, moe_stream_t stream) {
  size_t need = 0;
  if (moe_status_t st = moe_workspace_size(M, H, I, E, top_k, MOE_REDUCE_SEPARATE, &need))
    return st;
  if (!w) return set_error(MOE_ERR_INVALID_ARG, "null weights");
  if (moe_status_t st = validate_wq_format(w->format, w->group_size, w->w13_zero)) return st;
  if (w->format >= MOE_WQ_MXFP4 && w->w2_zero != nullptr)
    return set_error(MOE_ERR_INVALID_ARG, "MX formats have no zero points");
  if (H < 64 || I < 64 || H % 32 != 0 || I % 32 != 0)
    return set_error(MOE_ERR_INVALID_ARG,
                     "quantised weights need H and I multiples of 32, at least 64 (H=%d I=%d)", H, I);
  if (H % w->group_size != 0 || I % w->group_size != 0)
    return set_error(MOE_ERR_INVALID_ARG, "group_size=%d must divide H=%d and I=%d",
                     w->group_size, H, I);
  if ((w->w13_zero == nullptr) != (w->w2_zero == nullptr))
    return set_error(MOE_ERR_INVALID_ARG, "zero points for both w13 and w2, or for neither");
  if (M == 0) return MOE_OK;
  if (!hidden || !topk_weights || !topk_ids || !w->w13 || !w->w2 || !w->w13_scale ||
      !w->w2_scale || !workspace || !out)
    return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(hidden) || !aligned16(out) || !aligned16(w->w13) || !aligned16(w->w2) ||
      !aligned16(w->w13_scale) || !aligned16(w->w2_scale) ||
      (w->w13_zero && !aligned16(w->w13_zero)) || (w->w2_zero && !aligned16(w->w2_zero)) ||
      (w13_bias && !aligned16(w13_bias)) || (w2_bias && !aligned16(w2_bias)))
    return set_error(MOE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return set_error(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < need)
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes, got %zu", need,
                     workspace_bytes);
  int sms = 0;
  if (moe_status_t st = check_device(&sms)) return st;
  cudaStream_t s = stream;
  const int64_t Mc_max = M < MOE_CHUNK_TOKENS ? M : MOE_CHUNK_TOKENS;
  const FwdLayout L = fwd_layout(Mc_max, H, I, E, top_k);
  int32_t* err = at<int32_t>(workspace, L.err);
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(cudaGetLastError()));
  const bf16* x = static_cast<const bf16*>(hidden);
  bf16* y = static_cast<bf16*>(out);
  for (int64_t c0 = 0; c0 < M; c0 += Mc_max) {
    const int64_t Mc = (M - c0) < Mc_max ? (M - c0) : Mc_max;
    const int64_t Rc = Mc * top_k;
    const int64_t cap = align_cap(Rc, E, MOE_BLOCK_M);
    int32_t* sorted = at<int32_t>(workspace, L.sorted);
    int32_t* offsets = at<int32_t>(workspace, L.offsets);
    int32_t* inv = at<int32_t>(workspace, L.inv);
    AlignArgs al{topk_ids + c0 * top_k, Rc, E, MOE_BLOCK_M, sorted, offsets,
                 at<int32_t>(workspace, L.counts), at<int32_t>(workspace, L.block_expert),
                 at<int32_t>(workspace, L.scratch), cap, err, inv};
    if (moe_status_t st = launch_align(al, s)) return st;
    bf16* a_perm = at<bf16>(workspace, L.a_perm);
    GatherArgs ga{x + c0 * H, sorted, offsets, E, top_k, static_cast<int32_t>(Rc), H, cap,
                  a_perm};
    ga.inv = inv;  // each token row read once
    ga.tokens = Mc;
    if (moe_status_t st = launch_gather(ga, s)) return st;
    bf16* z = at<bf16>(workspace, L.z);
    GroupedGemmArgs g1{};
    g1.a = a_perm;
    g1.w = static_cast<const bf16*>(w->w13);
    g1.bias = static_cast<const bf16*>(w13_bias);
    g1.cap = cap;
    g1.E = E;
    g1.N = I;
    g1.K = H;
    g1.offsets = offsets;
    g1.out = z;
    g1.row_index = sorted;
    g1.sentinel = static_cast<int32_t>(Rc);
    g1.error_word = err;
    g1.num_sms = sms;
    g1.rows_hint = Rc;
    g1.wq_format = w->format;
    g1.wq_group = w->group_size;
    g1.wq_scale = w->w13_scale;
    g1.wq_zero = w->w13_zero;
    // a few rows per expert: the decode GEMMs (rows as the MMA's N, weights
    // expanded in registers); otherwise the grouped tensor-core GEMMs
    const bool decode = g_wq_decode.load(std::memory_order_relaxed) != 0 &&
                        wq_decode_applies(Mc, H, I, E, w->format, w->group_size);
    const int32_t* counts = at<int32_t>(workspace, L.counts);
    if (decode) {
      if (moe_status_t st = launch_wq_decode_gemm1(g1, counts, Mc, s)) return st;
    } else {
      if (moe_status_t st = launch_gemm1_swiglu_wq(g1, s)) return st;
    }
    float* o = at<float>(workspace, L.o);
    GroupedGemmArgs g2{};
    g2.a = z;
    g2.w = static_cast<const bf16*>(w->w2);
    g2.bias = static_cast<const bf16*>(w2_bias);
    g2.cap = cap;
    g2.E = E;
    g2.N = H;
    g2.K = I;
    g2.offsets = offsets;
    g2.out = o;
    g2.row_index = sorted;
    g2.row_weight = topk_weights + c0 * top_k;
    g2.sentinel = static_cast<int32_t>(Rc);
    g2.div = top_k;
    g2.error_word = err;
    g2.num_sms = sms;
    g2.rows_hint = Rc;
    g2.wq_format = w->format;
    g2.wq_group = w->group_size;
    g2.wq_scale = w->w2_scale;
    g2.wq_zero = w->w2_zero;
    if (decode) {
      // K split into parts, each a weighted fp32 row per routed item
      const int32_t parts = wq_decode_splits(Mc, top_k, H, I, E, cap, sms);
      if (moe_status_t st = launch_wq_decode_gemm2(g2, counts, Mc, parts, Rc, s)) return st;
      if (moe_status_t st = launch_reduce_parts(o, inv, Mc, top_k, H, parts, y + c0 * H, s))
        return st;
      continue;
    }
    if (moe_status_t st = launch_gemm2_sorted_wq(g2, s)) return st;
    if (moe_status_t st = launch_reduce_sorted(o, inv, Mc, top_k, H, y + c0 * H, s)) return st;
  }
  return MOE_OK;
}

// ------------------------------------------------------ forward_batched --
moe_status_t moe_batched_workspace_size(int32_t E, int32_t T, int32_t H, int32_t I,
                                        size_t* bytes) {
  g_detail[0] = 0;
  if (!bytes) return set_error(MOE_ERR_INVALID_ARG, "null bytes");
  if (moe_status_t st = validate_ffn_dims(H, I, E)) return st;
  if (T < 1) return set_error(MOE_ERR_INVALID_ARG, "T=%d < 1", T);
  if (static_cast<int64_t>(E) * T + static_cast<int64_t>(E) * MOE_BLOCK_M >= (int64_t(1) << 31))
    return set_error(MOE_ERR_INVALID_ARG, "E*T too large for int32 row indices");
  *bytes = bat_layout(E, T, H, I).total;
  return MOE_OK;
}

moe_status_t moe_forward_batched(const void* x, const int32_t* expert_num_tokens, int32_t E,
                                 int32_t T, int32_t H, int32_t I, const void* w13,
                                 const void* w2, const void* w13_bias, const void* w2_bias,
                                 const float* row_weight, void* workspace,
                                 size_t workspace_bytes, void* out, moe_stream_t stream) {
  size_t need = 0;
  if (moe_status_t st = moe_batched_workspace_size(E, T, H, I, &need)) return st;
  if (!x || !expert_num_tokens || !w13 || !w2 || !workspace || !out)
    return set_error(MOE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(out) ||
      (w13_bias && !aligned16(w13_bias)) || (w2_bias && !aligned16(w2_bias)))
    return set_error(MOE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return set_error(MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < need)
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes, got %zu", need,
                     workspace_bytes);
  int sms = 0;
  if (moe_status_t st = check_device(&sms)) return st;
  cudaStream_t s = stream;
  const BatLayout L = bat_layout(E, T, H, I);
  int32_t* err = at<int32_t>(workspace, L.err);  // cleared by the plan kernel
  const int32_t sentinel = E * T;
  int32_t* sorted = at<int32_t>(workspace, L.sorted);
  int32_t* offsets = at<int32_t>(workspace, L.offsets);
  BatchedPlanArgs bp{expert_num_tokens, E, T, MOE_BLOCK_M, sorted, offsets,
                     at<int32_t>(workspace, L.block_expert), L.cap, sentinel, err};
  if (moe_status_t st = launch_batched_plan(bp, s)) return st;

  bf16* a_perm = at<bf16>(workspace, L.a_perm);
  GatherArgs ga{static_cast<const bf16*>(x), sorted, offsets, E, 1, sentinel, H, L.cap, a_perm};
  if (moe_status_t st = launch_gather(ga, s)) return st;

  bf16* z = at<bf16>(workspace, L.z);
  GroupedGemmArgs g1{};
  g1.a = a_perm;
  g1.w = static_cast<const bf16*>(w13);
  g1.bias = static_cast<const bf16*>(w13_bias);
  g1.cap = L.cap;
  g1.E = E;
  g1.N = I;
  g1.K = H;
  g1.offsets = offsets;
  g1.out = z;
  g1.row_index = sorted;
  g1.sentinel = sentinel;
  g1.error_word = err;
  g1.num_sms = sms;
  // the tile shape from the layout's capacity, T rows per expert: CTA pairs
  // when an expert can hold four 128-row blocks (E = 32, T = 512 with ~60 %
  // of the rows valid: 0.443 -> 0.426 ms against single-CTA tiles)
  g1.rows_hint = static_cast<int64_t>(E) * T;
  if (moe_status_t st = launch_gemm1_swiglu(g1, s)) return st;

  GroupedGemmArgs g2{};
  g2.a = z;
  g2.w = static_cast<const bf16*>(w2);
  g2.bias = static_cast<const bf16*>(w2_bias);
  g2.cap = L.cap;
  g2.E = E;
  g2.N = H;
  g2.K = I;
  g2.offsets = offsets;
  g2.out = out;
  g2.row_index = sorted;
  g2.row_weight = row_weight;
  g2.sentinel = sentinel;
  g2.error_word = err;
  g2.num_sms = sms;
  g2.rows_hint = static_cast<int64_t>(E) * T;
  return launch_gemm2_rows_bf16(g2, s);
}

moe_status_t moe_workspace_layout(int64_t M, int32_t H, int32_t I, int32_t E, int32_t top_k,
                                  size_t offsets[11]) {
  size_t need = 0;
  if (!offsets) return set_error(MOE_ERR_INVALID_ARG, "null offsets");
  if (moe_status_t st = moe_workspace_size(M, H, I, E, top_k, MOE_REDUCE_AUTO, &need)) return st;
  const int64_t Mc = M < MOE_CHUNK_TOKENS ? M : MOE_CHUNK_TOKENS;
  const FwdLayout L = fwd_layout(Mc, H, I, E, top_k);
  const size_t v[11] = {L.err, L.counts, L.offsets, L.block_expert, L.sorted, L.scratch,
                        L.inv, L.a_perm, L.z, L.o, static_cast<size_t>(L.cap)};
  for (int i = 0; i < 11; ++i) offsets[i] = v[i];
  return MOE_OK;
}

moe_status_t moe_selftest_wait_timeout(int32_t* error_word, uint32_t limit_us,
                                       moe_stream_t stream) {
  g_detail[0] = 0;
  if (!error_word) return set_error(MOE_ERR_INVALID_ARG, "null error word");
  if (limit_us == 0 || limit_us > 1000000u)
    return set_error(MOE_ERR_INVALID_ARG, "limit_us must be in [1, 1e6]");
  if (moe_status_t st = check_device(nullptr)) return st;
  return launch_wait_timeout_probe(error_word, limit_us, stream);
}

// --------------------------------------------------------------- errors --
moe_status_t moe_read_error(const int32_t* error_word, int32_t reset, moe_stream_t stream) {
  if (!error_word) return set_error(MOE_ERR_INVALID_ARG, "null error word");
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, error_word, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "reading the error word: %s",
                     cudaGetErrorString(cudaGetLastError()));
  if (reset && host != 0) {
    if (cudaMemsetAsync(const_cast<int32_t*>(error_word), 0, sizeof(int32_t), stream) !=
        cudaSuccess)
      return set_error(MOE_ERR_CUDA, "clearing the error word");
  }
  return static_cast<moe_status_t>(host);
}

// ------------------------------------------------------------- profiler --
moe_status_t moe_profiler_start(void) {
  for (auto& r : g_recs) {
    if (r.a) g_pool.push_back(r.a);
    if (r.b) g_pool.push_back(r.b);
  }
  g_recs.clear();
  g_prof = true;
  return MOE_OK;
}

moe_status_t moe_profiler_stop(moe_kernel_time_t* out, int32_t capacity, int32_t* n) {
  g_prof = false;
  struct Agg {
    std::string name;
    int64_t launches;
    double ms;
  };
  std::vector<Agg> agg;
  moe_status_t st = MOE_OK;
  for (auto& r : g_recs) {
    if (!r.a || !r.b) continue;
    if (cudaEventSynchronize(r.b) != cudaSuccess) {
      st = set_error(MOE_ERR_CUDA, "cudaEventSynchronize: %s",
                     cudaGetErrorString(cudaGetLastError()));
      break;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    bool found = false;
    for (auto& a : agg)
      if (a.name == r.name) {
        a.launches++;
        a.ms += ms;
        found = true;
      }
    if (!found) agg.push_back({r.name, 1, ms});
  }
  for (auto& r : g_recs) {
    if (r.a) g_pool.push_back(r.a);
    if (r.b) g_pool.push_back(r.b);
  }
  g_recs.clear();
  if (n) *n = static_cast<int32_t>(agg.size());
  if (out) {
    for (int32_t i = 0; i < capacity && i < static_cast<int32_t>(agg.size()); ++i) {
      std::memset(out[i].name, 0, sizeof(out[i].name));
      std::strncpy(out[i].name, agg[i].name.c_str(), sizeof(out[i].name) - 1);
      out[i].launches = agg[i].launches;
      out[i].total_ms = agg[i].ms;
    }
  }
  return st;
}

}  // extern "C"
