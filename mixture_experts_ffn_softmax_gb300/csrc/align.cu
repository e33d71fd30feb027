// Expert-sorted, block-padded permutation of the routed items.
//
// Follows "FlagGems fused_moe.py analysis", section moe_align_block_size:
// flatten the (token, slot) items, sort them by expert, pad each expert's
// count up to the GEMM block size, and emit sorted_token_ids, the expert of
// every block and the padded total.  Items of one expert keep ascending item
// order (a stable sort); padding slots hold the sentinel R.
//
// Deterministic passes, no atomics in the ranking:
//   1. chunk histogram  -- each warp counts the experts of one 256-item chunk
//   2. column scan      -- one block per expert: prefix of its chunk counts
//   3. offsets          -- one block: padded counts, exclusive scan over
//                          experts, block ids, sentinel fill of the padding
//   4. scatter          -- each warp re-walks its chunk in order and writes
//                          every item at offsets[e] + chunk prefix + rank
// Problems of at most 4096 items and 256 experts run all of it in a single
// block (one launch instead of four).
#include <mutex>

#include "common.cuh"

namespace gbmoe {
namespace {

constexpr int kChunk = 256;        // items per warp chunk
constexpr int kAlignWarps = 8;     // warps (= chunks) per CTA
constexpr int kScanThreads = 1024;

// Expert of an item: the local expert id, or -1 if the item is not counted
// here (expert held elsewhere per expert_map, or a bad id -- `bad` says which).
__device__ __forceinline__ int local_expert(int e, int E, const int32_t* __restrict__ emap,
                                            int E_global, bool& bad) {
  if (emap != nullptr) {
    if (e < 0 || e >= E_global) {
      bad = true;
      return -1;
    }
    e = __ldg(emap + e);
    if (e >= E || e < -1) {
      bad = true;
      return -1;
    }
    return e;
  }
  if (e < 0 || e >= E) {
    bad = true;
    return -1;
  }
  return e;
}

__global__ void __launch_bounds__(kAlignWarps * 32)
    align_hist_kernel(const int32_t* __restrict__ ids, int64_t R, int E, int num_chunks,
                      int32_t* __restrict__ chunk_counts, int32_t* error_word,
                      const int32_t* __restrict__ emap, int E_global) {
  pdl_begin();
  extern __shared__ int32_t hist_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kAlignWarps + warp;
  if (chunk >= num_chunks) return;
  int32_t* cnt = hist_smem + warp * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int64_t r0 = static_cast<int64_t>(chunk) * kChunk;
  bool bad = false;
  for (int it = 0; it < kChunk / 32; ++it) {
    const int64_t r = r0 + it * 32 + lane;
    int e = -1;
    if (r < R) e = local_expert(ids[r], E, emap, E_global, bad);
    const bool ok = e >= 0;
    const int key = ok ? e : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    const int leader = __ffs(grp) - 1;
    if (ok && lane == leader) cnt[e] += __popc(grp);
    __syncwarp();
  }
  if (bad) record_error(error_word, MOE_ERR_BAD_EXPERT_ID);
  // expert-major layout: chunk_counts[e * num_chunks + chunk]
  for (int e = lane; e < E; e += 32)
    chunk_counts[static_cast<int64_t>(e) * num_chunks + chunk] = cnt[e];
}

// Block-wide (kScanThreads threads) end of an align plan, given the item
// count of every expert in s_count: padded counts, exclusive scan over the
// experts (expert_offsets), the expert of every block_m block (-1 past the
// last), and the sentinel in every padding slot.  Leaves the offsets in s_off.
__device__ void finish_plan(int E, int block_m, int32_t sentinel, int64_t cap,
                            const int32_t* s_count, int32_t* s_off, int32_t* s_warp,
                            int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                            int32_t* __restrict__ block_expert, int32_t* __restrict__ sorted) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t padded = 0;
  if (tid < E) padded = ceil_div(s_count[tid], block_m) * block_m;
  int32_t incl = padded;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int32_t w = s_warp[lane];
    int32_t wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += v;
    }
    s_warp[lane] = wi - w;
  }
  __syncthreads();
  const int32_t excl = s_warp[warp] + incl - padded;
  if (tid < E) {
    s_off[tid] = excl;
    if (counts != nullptr) counts[tid] = s_count[tid];
    offsets[tid] = excl;
  }
  if (tid == E - 1) {
    s_off[E] = excl + padded;
    offsets[E] = excl + padded;
  }
  __syncthreads();
  const int64_t nblk_cap = cap / block_m;
  const int32_t nblk = s_off[E] / block_m;
  for (int64_t b = tid; b < nblk_cap; b += kScanThreads) {
    int32_t e = -1;
    if (b < nblk) {
      int lo = 0, hi = E - 1;  // largest e with s_off[e] <= b * block_m
      const int32_t pos = static_cast<int32_t>(b) * block_m;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= pos) lo = mid; else hi = mid - 1;
      }
      e = lo;
    }
    block_expert[b] = e;
  }
  for (int e = warp; e < E; e += kScanThreads / 32)
    for (int32_t pos = s_off[e] + s_count[e] + lane; pos < s_off[e + 1]; pos += 32)
      sorted[pos] = sentinel;
}

// Per expert (one block each): exclusive prefix of its chunk counts over the
// chunks, in place, and its total.
constexpr int kColScanThreads = 256;
__global__ void __launch_bounds__(kColScanThreads)
    align_colscan_kernel(int num_chunks, int32_t* __restrict__ chunk_counts,
                         int32_t* __restrict__ counts) {
  pdl_begin();
  __shared__ int32_t s_warp[kColScanThreads / 32];
  __shared__ int32_t s_carry;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* col = chunk_counts + static_cast<int64_t>(blockIdx.x) * num_chunks;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < num_chunks; base += kColScanThreads * 4) {
    int32_t v[4], part = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = base + tid * 4 + i;
      v[i] = c < num_chunks ? col[c] : 0;
      part += v[i];
    }
    int32_t incl = part;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t x = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += x;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int32_t wbase = 0, total = 0;
    for (int w = 0; w < kColScanThreads / 32; ++w) {
      if (w < warp) wbase += s_warp[w];
      total += s_warp[w];
    }
    int32_t run = s_carry + wbase + incl - part;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = base + tid * 4 + i;
      if (c < num_chunks) col[c] = run;
      run += v[i];
    }
    __syncthreads();
    if (tid == 0) s_carry += total;
    __syncthreads();
  }
  if (tid == 0) counts[blockIdx.x] = s_carry;
}

// Offsets, block ids and sentinels from the per-expert totals (one block).
__global__ void __launch_bounds__(kScanThreads)
    align_offsets_kernel(int E, int block_m, int32_t sentinel, int64_t cap,
                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ block_expert, int32_t* __restrict__ sorted) {
  pdl_begin();
  __shared__ int32_t s_count[1024];
  __shared__ int32_t s_off[1025];
  __shared__ int32_t s_warp[32];
  if (threadIdx.x < E) s_count[threadIdx.x] = counts[threadIdx.x];
  __syncthreads();
  finish_plan(E, block_m, sentinel, cap, s_count, s_off, s_warp, nullptr, offsets, block_expert,
              sorted);
}

// The whole align in one block for small problems (R <= kSmallItems,
// E <= kSmallExperts): warp w owns a contiguous run of items; per-warp
// histograms, a prefix over the warps, the plan, then the stable scatter.
constexpr int kSmallItems = 4096;
constexpr int kSmallExperts = 256;
// With few experts the one-block plan stays cheaper up to more items
// (measured on GB300, E = 8: 15 us against 29 us for the four-kernel plan
// at 8192 items, 20 against 30 at 16384; with 128 or 256 experts it loses
// beyond 4096 items).
constexpr int kSmallItemsFewExperts = 16384;
constexpr int kFewExperts = 16;
__global__ void __launch_bounds__(kScanThreads)
    align_small_kernel(const int32_t* __restrict__ ids, int R, int E, int block_m, int64_t cap,
                       int32_t* __restrict__ sorted, int32_t* __restrict__ offsets,
                       int32_t* __restrict__ counts, int32_t* __restrict__ block_expert,
                       int32_t* __restrict__ inv, int32_t* error_word,
                       const int32_t* __restrict__ emap, int E_global, int32_t* zero_words,
                       int zero_count) {
  pdl_begin();
  if (zero_words != nullptr) {  // before any error can be recorded
    for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero_words[i] = 0;
    __syncthreads();
  }
  __shared__ int32_t s_cnt[32 * kSmallExperts];
  __shared__ int32_t s_count[kSmallExperts];
  __shared__ int32_t s_off[kSmallExperts + 1];
  __shared__ int32_t s_warp[32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per = ceil_div(ceil_div(R, 32), 32) * 32;  // items per warp, multiple of 32
  const int r0 = warp * per;
  int32_t* cnt = s_cnt + warp * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  // The warp's items, one per lane and pass, all loaded before any is used
  // (one memory latency instead of one per pass), kept for both passes.
  constexpr int kMaxPasses = kSmallItemsFewExperts / kScanThreads;
  static_assert(kSmallItems / kScanThreads <= kMaxPasses, "passes of the one-block plan");
  int ev[kMaxPasses];
#pragma unroll
  for (int i = 0; i < kMaxPasses; ++i) {
    const int r = r0 + 32 * i + lane;
    ev[i] = (32 * i < per && r < R) ? ids[r] : -1;
  }
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kMaxPasses; ++i) {
    const int r = r0 + 32 * i + lane;
    if (32 * i < per && r < R) ev[i] = local_expert(ev[i], E, emap, E_global, bad);
  }
#pragma unroll
  for (int i = 0; i < kMaxPasses; ++i) {
    if (32 * i >= per) break;  // warp-uniform
    const int e = ev[i];
    const bool ok = e >= 0;
    const unsigned grp = __match_any_sync(0xffffffffu, ok ? e : -1);
    if (ok && lane == __ffs(grp) - 1) cnt[e] += __popc(grp);
    __syncwarp();
  }
  if (bad) record_error(error_word, MOE_ERR_BAD_EXPERT_ID);
  __syncthreads();
  if (tid < E) {  // exclusive prefix of expert tid over the warps
    int32_t run = 0;
    for (int w = 0; w < 32; ++w) {
      const int32_t v = s_cnt[w * E + tid];
      s_cnt[w * E + tid] = run;
      run += v;
    }
    s_count[tid] = run;
  }
  __syncthreads();
  finish_plan(E, block_m, R, cap, s_count, s_off, s_warp, counts, offsets, block_expert, sorted);
  __syncthreads();
  for (int e = lane; e < E; e += 32) cnt[e] += s_off[e];
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < kMaxPasses; ++i) {
    if (32 * i >= per) break;  // warp-uniform
    const int r = r0 + 32 * i + lane;
    const int e = ev[i];
    const bool ok = e >= 0;
    const unsigned grp = __match_any_sync(0xffffffffu, ok ? e : -1);
    const int32_t pos = ok ? cnt[e] + __popc(grp & lt_mask) : -1;
    if (ok) sorted[pos] = r;
    if (inv != nullptr && r < R) inv[r] = pos;
    __syncwarp();
    if (ok && lane == __ffs(grp) - 1) cnt[e] += __popc(grp);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kAlignWarps * 32)
    align_scatter_kernel(const int32_t* __restrict__ ids, int64_t R, int E, int num_chunks,
                         const int32_t* __restrict__ chunk_prefix,
                         const int32_t* __restrict__ offsets, int32_t* __restrict__ sorted,
                         int32_t* __restrict__ inv, const int32_t* __restrict__ emap,
                         int E_global) {
  pdl_begin();
  extern __shared__ int32_t run_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kAlignWarps + warp;
  if (chunk >= num_chunks) return;
  int32_t* run = run_smem + warp * E;
  for (int e = lane; e < E; e += 32)
    run[e] = offsets[e] + chunk_prefix[static_cast<int64_t>(e) * num_chunks + chunk];
  __syncwarp();
  const int64_t r0 = static_cast<int64_t>(chunk) * kChunk;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int it = 0; it < kChunk / 32; ++it) {
    const int64_t r = r0 + it * 32 + lane;
    int e = -1;
    bool bad = false;
    if (r < R) e = local_expert(ids[r], E, emap, E_global, bad);
    const bool ok = e >= 0;
    const int key = ok ? e : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    const int32_t pos = ok ? run[e] + __popc(grp & lt_mask) : -1;
    if (ok) sorted[pos] = static_cast<int32_t>(r);
    if (inv != nullptr && r < R) inv[r] = pos;
    __syncwarp();
    if (ok && lane == __ffs(grp) - 1) run[e] += __popc(grp);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kScanThreads)
    batched_plan_kernel(const int32_t* __restrict__ counts_in, int E, int T, int block_m,
                        int32_t sentinel, int64_t cap, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ block_expert, int32_t* __restrict__ sorted,
                        int32_t* error_word) {
  pdl_begin();
  if (threadIdx.x == 0 && error_word != nullptr) *error_word = 0;  // before any error is recorded
  __syncthreads();
  __shared__ int32_t s_count[1024];
  __shared__ int32_t s_off[1025];
  __shared__ int32_t s_warp[32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t c = 0;
  if (tid < E) {
    c = counts_in[tid];
    if (c < 0 || c > T) {
      record_error(error_word, MOE_ERR_BAD_EXPERT_ID);
      c = 0;
    }
    s_count[tid] = c;
  }
  const int32_t padded = (tid < E) ? ceil_div(c, block_m) * block_m : 0;
  int32_t incl = padded;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = s_warp[lane];
    int32_t wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += v;
    }
    s_warp[lane] = wi - w;
  }
  __syncthreads();
  const int32_t excl = s_warp[warp] + incl - padded;
  if (tid < E) {
    s_off[tid] = excl;
    offsets[tid] = excl;
  }
  if (tid == E - 1) {
    s_off[E] = excl + padded;
    offsets[E] = excl + padded;
  }
  __syncthreads();
  const int64_t nblk_cap = cap / block_m;
  const int32_t nblk = s_off[E] / block_m;
  for (int64_t b = tid; b < nblk_cap; b += kScanThreads) {
    int32_t e = -1;
    if (b < nblk) {
      int lo = 0, hi = E - 1;
      const int32_t pos = static_cast<int32_t>(b) * block_m;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= pos) lo = mid; else hi = mid - 1;
      }
      e = lo;
    }
    block_expert[b] = e;
  }
  for (int e = warp; e < E; e += kScanThreads / 32) {
    const int32_t base = s_off[e], cnt = s_count[e], end = s_off[e + 1];
    for (int32_t i = lane; base + i < end; i += 32)
      sorted[base + i] = (i < cnt) ? e * T + i : sentinel;
  }
}

}  // namespace

size_t align_scratch_bytes(int64_t R, int32_t E) {
  const int64_t chunks = ceil_div<int64_t>(R, kChunk);
  return static_cast<size_t>(chunks) * static_cast<size_t>(E) * sizeof(int32_t);
}

moe_status_t launch_align(const AlignArgs& a, cudaStream_t s) {
  if ((a.R <= kSmallItems && a.E <= kSmallExperts) ||
      (a.R <= kSmallItemsFewExperts && a.E <= kFewExperts)) {
    prof_before("align_small", s);
    launch_kernel(align_small_kernel, 1, kScanThreads, 0, s, a.ids, static_cast<int>(a.R), a.E,
                  a.block_m, a.cap, a.sorted, a.offsets, a.counts, a.block_expert, a.inv,
                  a.error_word, a.expert_map, a.E_global, a.zero_words, a.zero_count);
    prof_after("align_small", s);
    return check_launch("align_small");
  }
  if (a.zero_words != nullptr &&
      cudaMemsetAsync(a.zero_words, 0, sizeof(int32_t) * a.zero_count, s) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(cudaGetLastError()));
  const int num_chunks = static_cast<int>(ceil_div<int64_t>(a.R, kChunk));
  const size_t smem = static_cast<size_t>(kAlignWarps) * a.E * sizeof(int32_t);
  const unsigned grid = static_cast<unsigned>(ceil_div(num_chunks, kAlignWarps));
  prof_before("align_hist", s);
  launch_kernel(align_hist_kernel, grid, kAlignWarps * 32, smem, s, a.ids, a.R, a.E, num_chunks,
                a.chunk_counts, a.error_word, a.expert_map, a.E_global);
  prof_after("align_hist", s);
  if (moe_status_t st = check_launch("align_hist")) return st;
  prof_before("align_colscan", s);
  launch_kernel(align_colscan_kernel, a.E, kColScanThreads, 0, s, num_chunks, a.chunk_counts,
                a.counts);
  prof_after("align_colscan", s);
  if (moe_status_t st = check_launch("align_colscan")) return st;
  prof_before("align_offsets", s);
  launch_kernel(align_offsets_kernel, 1, kScanThreads, 0, s, a.E, a.block_m,
                static_cast<int32_t>(a.R), a.cap, a.counts, a.offsets, a.block_expert, a.sorted);
  prof_after("align_offsets", s);
  if (moe_status_t st = check_launch("align_offsets")) return st;
  prof_before("align_scatter", s);
  launch_kernel(align_scatter_kernel, grid, kAlignWarps * 32, smem, s, a.ids, a.R, a.E, num_chunks,
                a.chunk_counts, a.offsets, a.sorted, a.inv, a.expert_map, a.E_global);
  prof_after("align_scatter", s);
  return check_launch("align_scatter");
}

moe_status_t launch_batched_plan(const BatchedPlanArgs& a, cudaStream_t s) {
  prof_before("batched_plan", s);
  launch_kernel(batched_plan_kernel, 1, kScanThreads, 0, s, a.counts_in, a.E, a.T, a.block_m,
                a.sentinel, a.cap, a.offsets, a.block_expert, a.sorted, a.error_word);
  prof_after("batched_plan", s);
  return check_launch("batched_plan");
}

// ------------------------------------------------- static scratch variant --
// moe_align without a caller-provided scratch buffer: the per-chunk count
// table lives in this file-scope device array.  In host code the symbol is
// only a host-side stand-in, so its device address is looked up once per
// device with cudaGetSymbolAddress and that address is what the kernels get.
namespace {

static __device__ __align__(256) int32_t g_align_static_scratch[MOE_ALIGN_STATIC_SCRATCH_INTS];

constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
int32_t* g_static_scratch_ptr[kMaxDevices] = {};

moe_status_t static_scratch_for_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return set_error(MOE_ERR_NO_DEVICE, "no usable current device for the static scratch");
  }
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (g_static_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_align_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return set_error(MOE_ERR_CUDA, "cudaGetSymbolAddress(static align scratch): %s",
                       cudaGetErrorString(e));
    }
    g_static_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_static_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

moe_status_t launch_align_static_scratch(AlignArgs a, cudaStream_t s) {
  const size_t need = align_scratch_bytes(a.R, a.E);
  if (need > sizeof(int32_t) * static_cast<size_t>(MOE_ALIGN_STATIC_SCRATCH_INTS))
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL,
                     "static align scratch holds %d ints; ceil(R/256)*E needs %zu",
                     MOE_ALIGN_STATIC_SCRATCH_INTS, need / sizeof(int32_t));
  int32_t* p = nullptr;
  if (moe_status_t st = static_scratch_for_current_device(&p)) return st;
  a.chunk_counts = p;
  return launch_align(a, s);
}

}  // namespace gbmoe
