// Permute (row gather into expert-sorted order), unpermute (top-k reduce
// back to token order through the inverse permutation) and the fp32 -> bf16
// cast that follows the atomic reduce.  All HBM-bound: 16-byte vector
// loads/stores, grid sized to the SMs.
//
// "fused_moe.py 分析" (FlagDoc): A rows are found through the sorted item
// list (the token of item r is r // top_k), and moe_sum adds each token's
// top-k expert outputs.  "Fused MoE Modular Kernel" (vLLM): the permute /
// unpermute steps of apply() and TopKWeightAndReduce.
#include <cuda_fp16.h>

#include "common.cuh"
#include "fp8q.cuh"

namespace gbmoe {
namespace {

constexpr int kGatherWarps = 8;

// A_perm[p, :] = src[index[p] / div, :] for p < offsets[E].  Padding rows
// are left as they are: GEMM rows are independent and padding rows never
// reach an output, so nothing is spent writing them.  One warp per row,
// 16-byte vectors.
__global__ void __launch_bounds__(kGatherWarps * 32)
    gather_rows_kernel(const bf16* __restrict__ src, const int32_t* __restrict__ index,
                       const int32_t* __restrict__ offsets, int E, int div, int32_t sentinel,
                       int H, int64_t cap, bf16* __restrict__ dst) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int64_t rows = min(static_cast<int64_t>(offsets[E]), cap);
  const int nvec = H / 8;  // 16-byte vectors per row
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kGatherWarps;
  for (int64_t p = warp0; p < rows; p += nwarps) {
    const int32_t idx = index[p];
    uint4* d = reinterpret_cast<uint4*>(dst + p * H);
    if (idx >= 0 && idx < sentinel) {
      const uint4* sv = reinterpret_cast<const uint4*>(src + static_cast<int64_t>(idx / div) * H);
      for (int v = lane; v < nvec; v += 32) d[v] = __ldg(sv + v);
    }
  }
}

// The same gather token by token: A_perm[inv[t*k + j], :] = src[t, :] for
// every item j of token t with a sorted row (inv < 0: dropped).  In sorted
// order each token row is read once per item, at random, and falls out of
// L2 under the stream of stores (Qwen shape: 0.80 GB of DRAM traffic for
// 0.54 GB of rows written); here it is read once.  A warp takes a token and
// one segment of up to 32 * kTokVec 16-byte vectors of its row.
constexpr int kTokVec = 8;
__global__ void __launch_bounds__(kGatherWarps * 32)
    gather_tokens_kernel(const bf16* __restrict__ src, const int32_t* __restrict__ inv,
                         int64_t M, int k, int H, int64_t cap, bf16* __restrict__ dst) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int nvec = H / 8;  // 16-byte vectors per row
  const int segs = (nvec + 32 * kTokVec - 1) / (32 * kTokVec);
  const int64_t units = M * segs;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kGatherWarps;
  for (int64_t u = warp0; u < units; u += nwarps) {
    const int64_t t = u / segs;
    const int v0 = static_cast<int>(u - t * segs) * 32 * kTokVec;
    // the token's sorted rows: item j's in lane j % 32 of p[j / 32] (k <= 64)
    const int32_t p0 = lane < k ? __ldg(inv + t * k + lane) : -1;
    const int32_t p1 = lane + 32 < k ? __ldg(inv + t * k + lane + 32) : -1;
    const uint4* sv = reinterpret_cast<const uint4*>(src + t * H);
    uint4 x[kTokVec];
#pragma unroll
    for (int i = 0; i < kTokVec; ++i) {
      const int v = v0 + 32 * i + lane;
      if (v < nvec) x[i] = __ldg(sv + v);
    }
    for (int j = 0; j < k; ++j) {
      const int32_t pos = __shfl_sync(0xffffffffu, j < 32 ? p0 : p1, j & 31);
      if (pos < 0 || pos >= cap) continue;  // warp-uniform
      uint4* d = reinterpret_cast<uint4*>(dst + static_cast<int64_t>(pos) * H);
#pragma unroll
      for (int i = 0; i < kTokVec; ++i) {
        const int v = v0 + 32 * i + lane;
        if (v < nvec) d[v] = x[i];
      }
    }
  }
}

// y[t, :] = bf16(sum_j o_sorted[inv[t*k + j], :]) with V x 4 fp32 columns
// per thread; items with inv < 0 (dropped: bad expert id) contribute
// nothing.  V = 2 for small k (two 16-byte loads per item keep more bytes in
// flight: Mixtral shape, k = 2, 35.3 -> 29.0 us), V = 1 for larger k.
// KMAX > 0 (k <= KMAX): a token's k positions are loaded first and then all
// its k rows at once, so that k * V loads per thread are in flight; the sum
// is taken in the same order either way.
template <int V, int KMAX>
__global__ void __launch_bounds__(256)
    reduce_sorted_kernel(const float* __restrict__ o, const int32_t* __restrict__ inv,
                         int64_t M, int k, int H, bf16* __restrict__ y) {
  pdl_begin();
  const int hv = H / (4 * V);  // H % 8 == 0
  const int64_t total = M * hv;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / hv;
    const int c = static_cast<int>(i - t * hv);
    float4 acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](const float4 (&x)[V]) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        acc[v].x += x[v].x;
        acc[v].y += x[v].y;
        acc[v].z += x[v].z;
        acc[v].w += x[v].w;
      }
    };
    if constexpr (KMAX > 0) {
      int32_t pos[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) pos[j] = j < k ? __ldg(inv + t * k + j) : -1;
      float4 x[KMAX][V];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        const float4* src =
            reinterpret_cast<const float4*>(o + static_cast<int64_t>(pos[j] < 0 ? 0 : pos[j]) * H) +
            V * c;
#pragma unroll
        for (int v = 0; v < V; ++v)
          x[j][v] = pos[j] >= 0 ? __ldg(src + v) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (pos[j] >= 0) add(x[j]);
    } else {
      for (int j = 0; j < k; ++j) {
        const int32_t pos = __ldg(inv + t * k + j);
        if (pos < 0) continue;
        const float4* src = reinterpret_cast<const float4*>(o + static_cast<int64_t>(pos) * H) + V * c;
        float4 x[V];
#pragma unroll
        for (int v = 0; v < V; ++v) x[v] = __ldg(src + v);
        add(x);
      }
    }
    uint32_t w[2 * V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[v].x, acc[v].y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[v].z, acc[v].w);
      w[2 * v] = *reinterpret_cast<uint32_t*>(&lo);
      w[2 * v + 1] = *reinterpret_cast<uint32_t*>(&hi);
    }
    if constexpr (V == 2)
      reinterpret_cast<uint4*>(y + t * H)[c] = make_uint4(w[0], w[1], w[2], w[3]);
    else
      reinterpret_cast<uint2*>(y + t * H)[c] = make_uint2(w[0], w[1]);
  }
}

// As reduce_sorted_kernel for item rows stored as fp16 times 2^-e (e per row
// and 32-column chunk in o_exp [chunk][row], ld rows): y[t, :] =
// bf16(sum_j o16[pos_j, :] * 2^e), 8 x V columns per thread (within one
// chunk: one exponent byte per item).
template <int V, int KMAX>
__global__ void __launch_bounds__(256)
    reduce_sorted_f16_kernel(const __half* __restrict__ o, const uint8_t* __restrict__ o_exp,
                             int64_t ld, const int32_t* __restrict__ inv, int64_t M, int k, int H,
                             bf16* __restrict__ y) {
  pdl_begin();
  const int hv = H / (8 * V);
  const int64_t total = M * hv;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / hv;
    const int c = static_cast<int>(i - t * hv);
    const int col = 8 * V * c;
    float acc[8 * V];
#pragma unroll
    for (int v = 0; v < 8 * V; ++v) acc[v] = 0.f;
    auto add = [&](const uint4 (&x)[V], uint32_t e) {
      const float sc = __uint_as_float((127u + e) << 23);  // 2^e
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const uint32_t w[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
          acc[8 * v + 2 * q] = fmaf(f.x, sc, acc[8 * v + 2 * q]);
          acc[8 * v + 2 * q + 1] = fmaf(f.y, sc, acc[8 * v + 2 * q + 1]);
        }
      }
    };
    const uint8_t* ex_col = o_exp + static_cast<int64_t>(col >> 5) * ld;
    if constexpr (KMAX > 0) {
      // all k positions, then all k rows and exponents in flight at once
      int32_t pos[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) pos[j] = j < k ? __ldg(inv + t * k + j) : -1;
      uint4 x[KMAX][V];
      uint32_t e[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        const int64_t p = pos[j] < 0 ? 0 : pos[j];
        const uint4* src = reinterpret_cast<const uint4*>(o + p * H + col);
#pragma unroll
        for (int v = 0; v < V; ++v) x[j][v] = pos[j] >= 0 ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        e[j] = pos[j] >= 0 ? __ldg(ex_col + p) : 0u;
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (pos[j] >= 0) add(x[j], e[j]);
    } else {
      for (int j = 0; j < k; ++j) {
        const int32_t pos = __ldg(inv + t * k + j);
        if (pos < 0) continue;
        const uint4* src = reinterpret_cast<const uint4*>(o + static_cast<int64_t>(pos) * H + col);
        uint4 x[V];
#pragma unroll
        for (int v = 0; v < V; ++v) x[v] = __ldg(src + v);
        add(x, __ldg(ex_col + pos));
      }
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        __nv_bfloat162 b = __floats2bfloat162_rn(acc[8 * v + 2 * q], acc[8 * v + 2 * q + 1]);
        w[q] = *reinterpret_cast<uint32_t*>(&b);
      }
      reinterpret_cast<uint4*>(y + t * H + col)[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// y = bf16(acc), 8 elements per thread.
__global__ void __launch_bounds__(256)
    cast_f32_bf16_kernel(const float* __restrict__ acc, int64_t n8, bf16* __restrict__ y) {
  pdl_begin();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
    __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&p0);
    packed.y = *reinterpret_cast<uint32_t*>(&p1);
    packed.z = *reinterpret_cast<uint32_t*>(&p2);
    packed.w = *reinterpret_cast<uint32_t*>(&p3);
    reinterpret_cast<uint4*>(y)[i] = packed;
  }
}

int device_sms() {
  static PerDevice sms_per_device;
  int sms = 148;
  sms_per_device.get(
      [](int* v) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            *v <= 0)
          *v = 148;
        cudaGetLastError();
        return cudaSuccess;
      },
      &sms);
  return sms;
}

}  // namespace

moe_status_t launch_gather(const GatherArgs& a, cudaStream_t s) {
  if (a.cap <= 0) return MOE_OK;
  if (a.inv != nullptr) {
    if (a.tokens <= 0) return MOE_OK;
    const int64_t segs = ceil_div<int64_t>(a.H / 8, 32 * kTokVec);
    const int64_t want = ceil_div<int64_t>(a.tokens * segs, kGatherWarps);
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, device_sms() * 8));
    prof_before("gather_rows", s);
    launch_kernel(gather_tokens_kernel, grid, kGatherWarps * 32, 0, s, a.src, a.inv, a.tokens,
                  a.div, a.H, a.cap, a.dst);
    prof_after("gather_rows", s);
    return check_launch("gather_rows");
  }
  const int64_t want = ceil_div<int64_t>(a.cap, kGatherWarps);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, device_sms() * 8));
  prof_before("gather_rows", s);
  launch_kernel(gather_rows_kernel, grid, kGatherWarps * 32, 0, s, a.src, a.index, a.offsets, a.E,
                a.div, a.sentinel, a.H, a.cap, a.dst);
  prof_after("gather_rows", s);
  return check_launch("gather_rows");
}

moe_status_t launch_reduce_sorted(const float* o_sorted, const int32_t* inv, int64_t M,
                                  int32_t k, int32_t H, bf16* y, cudaStream_t s) {
  if (M <= 0) return MOE_OK;
  const int V = k <= 4 ? 2 : 1;
  const int64_t total = M * (H / (4 * V));
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(ceil_div<int64_t>(total, 256), device_sms() * 8));
  prof_before("reduce_sorted", s);
  if (V == 2 && k <= 2)
    launch_kernel(reduce_sorted_kernel<2, 2>, grid, 256, 0, s, o_sorted, inv, M, k, H, y);
  else if (V == 2)
    launch_kernel(reduce_sorted_kernel<2, 4>, grid, 256, 0, s, o_sorted, inv, M, k, H, y);
  else if (k <= 8)
    launch_kernel(reduce_sorted_kernel<1, 8>, grid, 256, 0, s, o_sorted, inv, M, k, H, y);
  else
    launch_kernel(reduce_sorted_kernel<1, 0>, grid, 256, 0, s, o_sorted, inv, M, k, H, y);
  prof_after("reduce_sorted", s);
  return check_launch("reduce_sorted");
}

moe_status_t launch_reduce_sorted_f16(const void* o16, const uint8_t* o_exp, int64_t ld,
                                     const int32_t* inv, int64_t M, int32_t k, int32_t H, bf16* y,
                                     cudaStream_t s) {
  if (M <= 0) return MOE_OK;
  const int V = (k <= 4 && H % 16 == 0) ? 2 : 1;
  const int64_t total = M * (H / (8 * V));
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(ceil_div<int64_t>(total, 256), device_sms() * 8));
  const __half* o = static_cast<const __half*>(o16);
  prof_before("reduce_sorted", s);
  if (V == 2 && k <= 2)
    launch_kernel(reduce_sorted_f16_kernel<2, 2>, grid, 256, 0, s, o, o_exp, ld, inv, M, k, H, y);
  else if (V == 2)
    launch_kernel(reduce_sorted_f16_kernel<2, 4>, grid, 256, 0, s, o, o_exp, ld, inv, M, k, H, y);
  else if (k <= 8)
    launch_kernel(reduce_sorted_f16_kernel<1, 8>, grid, 256, 0, s, o, o_exp, ld, inv, M, k, H, y);
  else
    launch_kernel(reduce_sorted_f16_kernel<1, 0>, grid, 256, 0, s, o, o_exp, ld, inv, M, k, H, y);
  prof_after("reduce_sorted", s);
  return check_launch("reduce_sorted");
}

moe_status_t launch_cast_f32_bf16(const float* acc, int64_t n, bf16* y, cudaStream_t s) {
  if (n <= 0) return MOE_OK;
  const int64_t n8 = n / 8;  // n is a multiple of 8 (H % 8 == 0)
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(ceil_div<int64_t>(n8, 256), device_sms() * 8));
  prof_before("cast_f32_bf16", s);
  launch_kernel(cast_f32_bf16_kernel, grid, 256, 0, s, acc, n8, y);
  prof_after("cast_f32_bf16", s);
  return check_launch("cast_f32_bf16");
}

}  // namespace gbmoe

namespace gbmoe {
namespace {

// Router logits for few experts: s[t, e] = sum_h x[t, h] W_g[h, e] + b_g[e]
// ("fused_moe.py 分析" section 1.1), fp32 accumulate.  W_g [H, E] is staged
// in shared memory (as fp32) once per block; one warp per token streams the
// token's row (16-byte loads) -- x is read once, where a tensor-core tile
// would have only M / 128 blocks of work.
constexpr int kRouterWarps = 32;

template <int EMAX>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_small_kernel(const bf16* __restrict__ x, const bf16* __restrict__ wg,
                        const bf16* __restrict__ bg, int64_t M, int H, int E,
                        float* __restrict__ s) {
  pdl_begin();
  extern __shared__ float4 router_smem[];
  // W_g as fp32 [H][EMAX] (zero past E), 16 bytes of padding after every 8
  // rows so that the 32 lanes, 8 rows apart, hit different banks.
  float* sw = reinterpret_cast<float*>(router_smem);
  constexpr int kRowPad = 4;  // floats per 8 rows
  if (E == EMAX) {
    // 16-byte loads: 8 bf16 weights at a time
    for (int i = threadIdx.x; i < H * EMAX / 8; i += blockDim.x) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(wg) + i);
      const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&v);
      const int h = (i * 8) / EMAX, e0 = (i * 8) % EMAX;
      float* d = sw + h * EMAX + (h >> 3) * kRowPad + e0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(w2[j]);
        d[2 * j] = f.x;
        d[2 * j + 1] = f.y;
      }
    }
  } else {
    for (int i = threadIdx.x; i < H * EMAX; i += blockDim.x) {
      const int h = i / EMAX, e = i - h * EMAX;
      sw[h * EMAX + (h >> 3) * kRowPad + e] =
          e < E ? __bfloat162float(wg[static_cast<int64_t>(h) * E + e]) : 0.f;
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kRouterWarps + (threadIdx.x >> 5);
  for (int64_t t = warp0; t < M; t += static_cast<int64_t>(gridDim.x) * kRouterWarps) {
    float acc[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[e] = 0.f;
    const bf16* row = x + t * H;
    for (int hb = lane * 8; hb < H; hb += 4 * 256) {
      uint4 xs[4];  // four 16-byte loads in flight before the math
#pragma unroll
      for (int u = 0; u < 4; ++u)
        xs[u] = (hb + u * 256 < H) ? __ldg(reinterpret_cast<const uint4*>(row + hb + u * 256))
                                   : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
      const int h0 = hb + u * 256;
      if (h0 >= H) break;
      const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xs[u]);
      const float* wrow = sw + h0 * EMAX + (h0 >> 3) * kRowPad;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 xf = __bfloat1622float2(xp[i]);
        const float4* w0 = reinterpret_cast<const float4*>(wrow + (2 * i) * EMAX);
        const float4* w1 = reinterpret_cast<const float4*>(wrow + (2 * i + 1) * EMAX);
#pragma unroll
        for (int q = 0; q < EMAX / 4; ++q) {
          const float4 a = w0[q], b = w1[q];
          acc[4 * q + 0] = fmaf(xf.x, a.x, fmaf(xf.y, b.x, acc[4 * q + 0]));
          acc[4 * q + 1] = fmaf(xf.x, a.y, fmaf(xf.y, b.y, acc[4 * q + 1]));
          acc[4 * q + 2] = fmaf(xf.x, a.z, fmaf(xf.y, b.z, acc[4 * q + 2]));
          acc[4 * q + 3] = fmaf(xf.x, a.w, fmaf(xf.y, b.w, acc[4 * q + 3]));
        }
      }
      }
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      float v = acc[e];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[e] = v;
    }
    if (lane < E && lane < EMAX) {
      float v = 0.f;
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
        if (e == lane) v = acc[e];
      s[t * E + lane] = v + (bg != nullptr ? __bfloat162float(bg[lane]) : 0.f);
    }
  }
}

template <int EMAX>
moe_status_t launch_router_small_t(const bf16* x, const bf16* wg, const bf16* bg, int64_t M,
                                   int H, int E, float* s, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(H) * EMAX * sizeof(float) + (H / 8) * 16;
  static PerDevice attrs;
  if (attrs.get([](int*) {
        return cudaFuncSetAttribute(router_small_kernel<EMAX>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
      }) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute(router_small)");
  const unsigned grid = static_cast<unsigned>(
      std::min<int64_t>(ceil_div<int64_t>(M, kRouterWarps), device_sms()));
  prof_before("router_small", st);
  launch_kernel(router_small_kernel<EMAX>, grid, kRouterWarps * 32, smem, st, x, wg, bg, M, H, E,
                s);
  prof_after("router_small", st);
  return check_launch("router_small");
}

}  // namespace

bool router_small_fits(int H, int E) {
  const int emax = E <= 8 ? 8 : (E <= 16 ? 16 : 32);
  return E <= 32 && H % 256 == 0 &&
         static_cast<size_t>(H) * emax * 4 + (H / 8) * 16 <= 160 * 1024;
}

moe_status_t launch_router_small(const bf16* x, const bf16* wg, const bf16* bg, int64_t M,
                                 int H, int E, float* s, cudaStream_t st) {
  if (E <= 8) return launch_router_small_t<8>(x, wg, bg, M, H, E, s, st);
  if (E <= 16) return launch_router_small_t<16>(x, wg, bg, M, H, E, s, st);
  return launch_router_small_t<32>(x, wg, bg, M, H, E, s, st);
}

}  // namespace gbmoe

namespace gbmoe {
namespace {

constexpr int kQuantWarps = 8;
constexpr int kQuantUnroll = 4;  // 16-byte loads in flight per lane

// max |v| over 8 bf16 values, as bf16 magnitude bits in both halves
__device__ __forceinline__ uint32_t absmax_bits8(const uint4 u, uint32_t m) {
  m = __vmaxu2(m, u.x & 0x7fff7fffu);
  m = __vmaxu2(m, u.y & 0x7fff7fffu);
  m = __vmaxu2(m, u.z & 0x7fff7fffu);
  return __vmaxu2(m, u.w & 0x7fff7fffu);
}

// Token rows, one warp per token: amax over the row, then the codes are
// written to each of the token's sorted rows (the gather of the permuted
// operand and its quantisation in one pass over x).
__global__ void __launch_bounds__(kQuantWarps * 32)
    quant_tokens_fp8_kernel(const bf16* __restrict__ x, const int32_t* __restrict__ inv,
                            int64_t M, int k, int H, uint8_t* __restrict__ q8,
                            float* __restrict__ scale, float* __restrict__ row_amax) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int nvec = H / 8;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQuantWarps;
  for (int64_t t = warp0; t < M; t += nwarps) {
    const uint4* sv = reinterpret_cast<const uint4*>(x + t * H);
    // loops run the same trip count on every lane (warp-uniform shuffles)
    uint32_t m2 = 0;
    for (int b = 0; b < nvec; b += 32 * kQuantUnroll) {
      uint4 u[kQuantUnroll];
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int v = b + 32 * i + lane;
        u[i] = v < nvec ? __ldg(sv + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) m2 = absmax_bits8(u[i], m2);
    }
    uint32_t mb = max(m2 & 0xffffu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const RowScale rs = row_scale(__uint_as_float(mb << 16));
    // sorted rows of the token's k items (lane j holds item j's, j < 32);
    // without inv the rows are not permuted (k = 1, row t)
    const int32_t mypos =
        lane < k ? (inv != nullptr ? __ldg(inv + t * k + lane) : static_cast<int32_t>(t)) : -1;
    for (int b = 0; b < nvec; b += 32 * kQuantUnroll) {
      uint2 c[kQuantUnroll];
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int v = b + 32 * i + lane;
        c[i] = e4m3x8(v < nvec ? __ldg(sv + v) : make_uint4(0, 0, 0, 0), rs);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t pos = j < 32 ? __shfl_sync(0xffffffffu, mypos, j) : __ldg(inv + t * k + j);
        if (pos < 0) continue;
        uint2* dq = reinterpret_cast<uint2*>(q8 + static_cast<int64_t>(pos) * H);
#pragma unroll
        for (int i = 0; i < kQuantUnroll; ++i) {
          const int v = b + 32 * i + lane;
          if (v < nvec) dq[v] = c[i];
        }
      }
    }
    for (int j = lane; j < k; j += 32) {
      const int32_t pos = inv != nullptr ? inv[t * k + j] : static_cast<int32_t>(t);
      if (pos < 0) continue;
      scale[pos] = rs.s;
      if (row_amax != nullptr) row_amax[pos] = 0.f;
    }
  }
}

// Sorted rows of z, one warp per row, one pass: the row's amax was taken by
// the producing GEMM's epilogue.
__global__ void __launch_bounds__(kQuantWarps * 32)
    quant_sorted_fp8_kernel(const bf16* __restrict__ src, const int32_t* __restrict__ index,
                            const int32_t* __restrict__ offsets, int E, int32_t sentinel, int H,
                            int64_t cap, uint8_t* __restrict__ q8, float* __restrict__ scale_io) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int64_t rows = min(static_cast<int64_t>(offsets[E]), cap);
  const int nvec = H / 8;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQuantWarps;
  for (int64_t p = warp0; p < rows; p += nwarps) {
    const int32_t idx = index[p];
    if (idx < 0 || idx >= sentinel) continue;  // padding row
    float amax = 0.f;
    if (lane == 0) amax = scale_io[p];
    const RowScale rs = row_scale(__shfl_sync(0xffffffffu, amax, 0));
    const uint4* sv = reinterpret_cast<const uint4*>(src + p * H);
    uint2* dq = reinterpret_cast<uint2*>(q8 + p * H);
    for (int b = 0; b < nvec; b += 32 * kQuantUnroll) {
      uint4 u[kQuantUnroll];
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int v = b + 32 * i + lane;
        u[i] = v < nvec ? __ldcs(sv + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int v = b + 32 * i + lane;
        if (v < nvec) dq[v] = e4m3x8(u[i], rs);
      }
    }
    if (lane == 0) scale_io[p] = rs.s;
  }
}

// Per-(row, group of 128) quantisation ("fused_moe.py 分析", FP8 W8A8,
// block-wise activations).  Lane l holds 8 elements; each half-warp covers
// one 128-wide group, reduced over its 16 lanes.  Scales are stored group
// major, scale[g * ld + row], so a warp's 32 rows read one line in the GEMM.

__device__ __forceinline__ float half_warp_amax(uint32_t mb) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
  return __uint_as_float(mb << 16);
}

// Token rows: each token's groups are quantised once and the codes written
// to each of its k sorted rows.
__global__ void __launch_bounds__(kQuantWarps * 32)
    quant_tokens_group_fp8_kernel(const bf16* __restrict__ x, const int32_t* __restrict__ inv,
                                  int64_t M, int k, int H, uint8_t* __restrict__ q8,
                                  float* __restrict__ scale, int64_t ld) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kQuantWarps;
  for (int64_t t = warp0; t < M; t += nwarps) {
    const int32_t mypos = lane < k ? __ldg(inv + t * k + lane) : -1;
    // passes of 256 columns (two groups, the same count on every lane),
    // kQuantUnroll of them per iteration with their loads issued first
    for (int b0 = 0; b0 < H; b0 += 256 * kQuantUnroll) {
      uint4 u[kQuantUnroll];
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int v = b0 + 256 * i + lane * 8;
        u[i] = v < H ? __ldg(reinterpret_cast<const uint4*>(x + t * H + v)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int v = b0 + 256 * i + lane * 8;
        const bool in = v < H;
        uint32_t m2 = absmax_bits8(u[i], 0u);
        const RowScale rs = row_scale(half_warp_amax(max(m2 & 0xffffu, m2 >> 16)));
        const uint2 c = e4m3x8(u[i], rs);
        const int g = v / 128;
        for (int j = 0; j < k; ++j) {
          const int32_t pos = j < 32 ? __shfl_sync(0xffffffffu, mypos, j) : __ldg(inv + t * k + j);
          if (pos < 0 || !in) continue;
          *reinterpret_cast<uint2*>(q8 + static_cast<int64_t>(pos) * H + v) = c;
          if ((lane & 15) == 0) scale[static_cast<int64_t>(g) * ld + pos] = rs.s;
        }
      }
    }
  }
}

// Blocks of `kernel` resident on one SM at once (cached per device): a
// grid-stride kernel launched with more gives every block the same share of
// rows, and the blocks past that run as a thin second wave.
template <typename Kernel>
int resident_blocks(Kernel kernel, int threads, PerDevice& cache) {
  int per_sm = 4;
  cache.get(
      [&](int* v) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kernel, threads, 0) != cudaSuccess ||
            *v <= 0)
          *v = 4;
        cudaGetLastError();
        return cudaSuccess;
      },
      &per_sm);
  return per_sm;
}

}  // namespace

moe_status_t launch_quant_tokens_group_fp8(const QuantTokensArgs& a, int64_t ld, cudaStream_t s) {
  if (a.M <= 0) return MOE_OK;
  static PerDevice blocks_per_sm;
  const int per_sm = resident_blocks(quant_tokens_group_fp8_kernel, kQuantWarps * 32, blocks_per_sm);
  const int64_t want = ceil_div<int64_t>(a.M, kQuantWarps);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, device_sms() * per_sm));
  prof_before("quant_tokens_fp8", s);
  launch_kernel(quant_tokens_group_fp8_kernel, grid, kQuantWarps * 32, 0, s, a.x, a.inv, a.M, a.k,
                a.H, a.q8, a.scale, ld);
  prof_after("quant_tokens_fp8", s);
  return check_launch("quant_tokens_fp8");
}

moe_status_t launch_quant_tokens_fp8(const QuantTokensArgs& a, cudaStream_t s) {
  if (a.M <= 0) return MOE_OK;
  const int64_t want = ceil_div<int64_t>(a.M, kQuantWarps);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, device_sms() * 8));
  prof_before("quant_tokens_fp8", s);
  launch_kernel(quant_tokens_fp8_kernel, grid, kQuantWarps * 32, 0, s, a.x, a.inv, a.M, a.k, a.H,
                a.q8, a.scale, a.row_amax);
  prof_after("quant_tokens_fp8", s);
  return check_launch("quant_tokens_fp8");
}

moe_status_t launch_quant_sorted_fp8(const QuantSortedArgs& a, cudaStream_t s) {
  if (a.cap <= 0) return MOE_OK;
  const int64_t want = ceil_div<int64_t>(a.cap, kQuantWarps);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, device_sms() * 8));
  prof_before("quant_z_fp8", s);
  launch_kernel(quant_sorted_fp8_kernel, grid, kQuantWarps * 32, 0, s, a.src, a.index, a.offsets,
                a.E, a.sentinel, a.H, a.cap, a.q8, a.scale_io);
  prof_after("quant_z_fp8", s);
  return check_launch("quant_z_fp8");
}

}  // namespace gbmoe
