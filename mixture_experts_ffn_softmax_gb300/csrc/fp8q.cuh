// E4M3 quantisation with a dynamic scale, shared by the quantisation
// passes and the GEMM epilogue that quantises its own output.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace gbmoe {

// x / s rounded to nearest even in fp32, for a divisor fixed along a row, by
// Markstein's correction of the product with the reciprocal (P. Markstein,
// "IA-64 and Elementary Functions", 2000; Handbook of Floating-Point
// Arithmetic, division by FMA): with r = RN(1/s) and q = RN(x r) within an
// ulp of x / s, the remainder x - q s is exact as one FMA and RN(q + rem r)
// is the correctly rounded quotient (no overflow or underflow: the caller
// takes the IEEE division for rows whose scale is not a normal float, and a
// quotient below the normal range is far below E4M3's smallest code).
__device__ __forceinline__ float div_fixed(float x, float s, float r) {
  const float q = __fmul_rn(x, r);
  const float rem = __fmaf_rn(-q, s, x);
  return __fmaf_rn(rem, r, q);
}

// Row scale and its reciprocal; `fast` is false where the correction does
// not apply (subnormal or non-finite scale) and the plain division is used.
struct RowScale {
  float s, r;
  bool fast;
};

// Dynamic per-row quantisation: scale = amax / 448, or 1 for an all-zero row
// ("fused_moe.py 分析": activations are quantised per token before each GEMM).
__device__ __forceinline__ RowScale row_scale(float amax) {
  RowScale rs;
  rs.s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  rs.fast = rs.s >= 1.17549435e-38f && rs.s <= 3.0e38f;
  rs.r = rs.fast ? __frcp_rn(rs.s) : 0.f;
  return rs;
}

// E4M3 codes of 8 bf16 values: q = e4m3(x / scale), the quotient correctly
// rounded in fp32, then round to nearest even with saturation to +-448.
__device__ __forceinline__ uint2 e4m3x8(const uint4 u, const RowScale& rs) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
  uint16_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    const float2 v = rs.fast ? make_float2(div_fixed(f.x, rs.s, rs.r), div_fixed(f.y, rs.s, rs.r))
                             : make_float2(__fdiv_rn(f.x, rs.s), __fdiv_rn(f.y, rs.s));
    b[i] = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
  }
  return make_uint2(static_cast<uint32_t>(b[0]) | (static_cast<uint32_t>(b[1]) << 16),
                    static_cast<uint32_t>(b[2]) | (static_cast<uint32_t>(b[3]) << 16));
}

}  // namespace gbmoe
