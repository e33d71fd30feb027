// Standalone dequantisation of weight-only quantised expert weights to bf16
// ("fused_moe.py 分析", "5. 特殊量化格式处理": the weights are dequantised to
// the activation dtype before the ordinary path runs).  The fused forward
// does the same conversion inside the grouped GEMM (wq.cuh).
#include <algorithm>

#include "common.cuh"
#include "wq.cuh"

namespace gbmoe {
namespace {

int sm_count() {
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

// One thread per 8 columns of one K row of one expert.
template <Wq WQ>
__global__ void __launch_bounds__(256)
    dequant_weights_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scale,
                           const uint8_t* __restrict__ zero, int E, int K, int N, int G,
                           __nv_bfloat16* __restrict__ out) {
  pdl_begin();
  using F = WqFmt<WQ>;
  const int n8 = N / 8;
  const int64_t units = static_cast<int64_t>(E) * K * n8;
  const int KG = K / G;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c8 = static_cast<int>(u % n8);
    const int64_t ek = u / n8;  // e * K + k
    const int k = static_cast<int>(ek % K);
    const int e = static_cast<int>(ek / K);
    const int n = c8 * 8;
    uint2 c;
    if constexpr (F::CODE_BITS == 4) {
      c.x = __ldg(reinterpret_cast<const uint32_t*>(codes + (ek * N + n) / 2));
      c.y = 0;
    } else {
      c = __ldg(reinterpret_cast<const uint2*>(codes + ek * N + n));
    }
    const int64_t prow = (static_cast<int64_t>(e) * KG + k / G) * N + n;  // param element
    uint4 s8;
    if constexpr (F::SCALE_BYTES == 2) {
      s8 = __ldg(reinterpret_cast<const uint4*>(scale + prow * 2));
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(scale + prow));
      s8 = make_uint4(v.x, v.y, 0, 0);
    }
    uint2 z8 = make_uint2(0, 0);
    if (F::HAS_ZERO && zero != nullptr) z8 = __ldg(reinterpret_cast<const uint2*>(zero + prow));
    WqParams8 p;
    wq_params8<WQ>(s8, z8, zero != nullptr, p);
    reinterpret_cast<uint4*>(out)[u] = wq_dequant8<WQ>(c, p);
  }
}

template <Wq WQ>
moe_status_t launch_dequant_t(const WqDequantArgs& a, cudaStream_t s) {
  const int64_t units = static_cast<int64_t>(a.E) * a.K * (a.N / 8);
  if (units == 0) return MOE_OK;
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(ceil_div<int64_t>(units, 256), sm_count() * 16));
  prof_before("dequant_weights", s);
  launch_kernel(dequant_weights_kernel<WQ>, grid, 256, 0, s, static_cast<const uint8_t*>(a.codes),
                static_cast<const uint8_t*>(a.scale), static_cast<const uint8_t*>(a.zero), a.E, a.K,
                a.N, a.G, a.out);
  prof_after("dequant_weights", s);
  return check_launch("dequant_weights");
}

}  // namespace

moe_status_t launch_dequant_weights(const WqDequantArgs& a, cudaStream_t s) {
  switch (a.format) {
    case 0: return launch_dequant_t<Wq::Int4>(a, s);
    case 1: return launch_dequant_t<Wq::Int8>(a, s);
    case 2: return launch_dequant_t<Wq::Mxfp4>(a, s);
    case 3: return launch_dequant_t<Wq::Mxfp6e3m2>(a, s);
    case 4: return launch_dequant_t<Wq::Mxfp6e2m3>(a, s);
    default: return set_error(MOE_ERR_INVALID_ARG, "weight format %d", a.format);
  }
}

}  // namespace gbmoe
