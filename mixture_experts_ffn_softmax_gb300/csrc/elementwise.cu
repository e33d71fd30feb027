// Permute (row gather into expert-sorted order) and unpermute (top-k
// weight-and-reduce back to token order).  Both are HBM-bound copies:
// 16-byte vector loads/stores, one warp per row, grid sized to the SMs.
//
// "FlagGems fused_moe.py analysis": A rows are found through the sorted item
// list (the token of item r is r // top_k), and moe_sum adds each token's
// top-k expert outputs.  "vLLM FusedMoEModularKernel" page: the permute /
// unpermute steps of apply() and TopKWeightAndReduce.
#include "common.cuh"

namespace gbmoe {
namespace {

constexpr int kGatherWarps = 8;

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
    } else {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = lane; v < nvec; v += 32) d[v] = z;
    }
  }
}

// y[t, :] = bf16(sum_j o[t*k + j, :]) with 4 fp32 columns per thread.
__global__ void __launch_bounds__(256)
    reduce_topk_kernel(const float* __restrict__ o, int64_t M, int k, int H,
                       bf16* __restrict__ y) {
  const int hv = H / 4;
  const int64_t total = M * hv;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / hv;
    const int c = static_cast<int>(i - t * hv);
    const float4* base = reinterpret_cast<const float4*>(o + t * k * H) + c;
    float4 acc = __ldg(base);
    for (int j = 1; j < k; ++j) {
      const float4 v = __ldg(base + static_cast<int64_t>(j) * hv);
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

moe_status_t launch_reduce(const float* o, int64_t M, int32_t k, int32_t H, bf16* y,
                           cudaStream_t s) {
  if (M <= 0) return MOE_OK;
  const int64_t total = M * (H / 4);
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(ceil_div<int64_t>(total, 256), device_sms() * 8));
  prof_before("reduce_topk", s);
  reduce_topk_kernel<<<grid, 256, 0, s>>>(o, M, k, H, y);
  prof_after("reduce_topk", s);
  return check_launch("reduce_topk");
}

}  // namespace gbmoe
