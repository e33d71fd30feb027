// Permute (row gather into expert-sorted order), unpermute (top-k reduce
// back to token order through the inverse permutation) and the fp32 -> bf16
// cast that follows the atomic reduce.  All HBM-bound: 16-byte vector
// loads/stores, grid sized to the SMs.
//
// "fused_moe.py 分析" (FlagDoc): A rows are found through the sorted item
// list (the token of item r is r // top_k), and moe_sum adds each token's
// top-k expert outputs.  "Fused MoE Modular Kernel" (vLLM): the permute /
// unpermute steps of apply() and TopKWeightAndReduce.
#include "common.cuh"

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

// y[t, :] = bf16(sum_j o_sorted[inv[t*k + j], :]) with 4 fp32 columns per
// thread; items with inv < 0 (dropped: bad expert id) contribute nothing.
__global__ void __launch_bounds__(256)
    reduce_sorted_kernel(const float* __restrict__ o, const int32_t* __restrict__ inv,
                         int64_t M, int k, int H, bf16* __restrict__ y) {
  const int hv = H / 4;
  const int64_t total = M * hv;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / hv;
    const int c = static_cast<int>(i - t * hv);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int32_t pos = __ldg(inv + t * k + j);
      if (pos < 0) continue;
      const float4 v = __ldg(reinterpret_cast<const float4*>(o + static_cast<int64_t>(pos) * H) + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(y + t * H)[c] = packed;
  }
}

// y = bf16(acc), 8 elements per thread.
__global__ void __launch_bounds__(256)
    cast_f32_bf16_kernel(const float* __restrict__ acc, int64_t n8, bf16* __restrict__ y) {
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
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return sms;
}

}  // namespace

moe_status_t launch_gather(const GatherArgs& a, cudaStream_t s) {
  if (a.cap <= 0) return MOE_OK;
  const int64_t want = ceil_div<int64_t>(a.cap, kGatherWarps);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, device_sms() * 8));
  prof_before("gather_rows", s);
  gather_rows_kernel<<<grid, kGatherWarps * 32, 0, s>>>(a.src, a.index, a.offsets, a.E, a.div,
                                                        a.sentinel, a.H, a.cap, a.dst);
  prof_after("gather_rows", s);
  return check_launch("gather_rows");
}

moe_status_t launch_reduce_sorted(const float* o_sorted, const int32_t* inv, int64_t M,
                                  int32_t k, int32_t H, bf16* y, cudaStream_t s) {
  if (M <= 0) return MOE_OK;
  const int64_t total = M * (H / 4);
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(ceil_div<int64_t>(total, 256), device_sms() * 8));
  prof_before("reduce_sorted", s);
  reduce_sorted_kernel<<<grid, 256, 0, s>>>(o_sorted, inv, M, k, H, y);
  prof_after("reduce_sorted", s);
  return check_launch("reduce_sorted");
}

moe_status_t launch_cast_f32_bf16(const float* acc, int64_t n, bf16* y, cudaStream_t s) {
  if (n <= 0) return MOE_OK;
  const int64_t n8 = n / 8;  // n is a multiple of 8 (H % 8 == 0)
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(ceil_div<int64_t>(n8, 256), device_sms() * 8));
  prof_before("cast_f32_bf16", s);
  cast_f32_bf16_kernel<<<grid, 256, 0, s>>>(acc, n8, y);
  prof_after("cast_f32_bf16", s);
  return check_launch("cast_f32_bf16");
}

}  // namespace gbmoe
