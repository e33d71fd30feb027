// Weight-only quantised expert weights: dequantisation of 8 consecutive
// columns of one K row to bf16, shared by the standalone dequantisation
// kernel and the converter warps of the grouped GEMM.
//
// Formats ("fused_moe.py 分析", "WNA16 路径" and "5. 特殊量化格式处理":
// int8 / int4 weights with a group scale and a zero point, and OCP MX
// weights, are dequantised to the activation dtype):
//   Int4   codes 0..15, two per byte (column 2j in the low nibble of byte j),
//          w = bf16((q - zp) * s), s bf16 per (group, column), zp 0..15
//          (default 8)
//   Int8   signed codes, w = bf16((q - zp) * s), zp int8 (default 0)
//   Mxfp4  OCP MX E2M1 codes, two per byte, UE8M0 scale 2^(s - 127) per
//          block of 32 rows of K: w = bf16(value(q) * 2^(s - 127))
//   Mxfp6  OCP MX E3M2 or E2M3 codes, one per byte (low 6 bits), UE8M0
//          scales as MX FP4
// bf16 arithmetic keeps subnormals, so 2^-127 scales and products below the
// normal range round like the exact product does.
// Every value is the exact product rounded once to bf16 (nearest even).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace gbmoe {

enum class Wq : int { None = 0, Int4 = 1, Int8 = 2, Mxfp4 = 3, Mxfp6e3m2 = 4, Mxfp6e2m3 = 5 };

template <Wq WQ>
struct WqFmt {
  static constexpr bool MX = WQ == Wq::Mxfp4 || WQ == Wq::Mxfp6e3m2 || WQ == Wq::Mxfp6e2m3;
  static constexpr int CODE_BITS = (WQ == Wq::Int4 || WQ == Wq::Mxfp4) ? 4 : 8;
  static constexpr int CODE_BYTES8 = CODE_BITS;        // bytes of 8 codes
  static constexpr int SCALE_BYTES = MX ? 1 : 2;
  static constexpr bool HAS_ZERO = !MX;
  // codes come out in the pair order (j, j + 4) (see wq_dequant8)
  static constexpr bool PAIRS = WQ != Wq::Int8;
};

// Per-group parameters of 8 columns, prepared for the conversion.
struct WqParams8 {
  __nv_bfloat162 s2[4];   // Int4 / Mxfp4: scales of columns (j, j + 4) (bf16; MX: 2^(s - 127))
  __nv_bfloat162 zb2[4];  // Int4: 128 + zero points of columns (j, j + 4) (exact bf16 values)
  float sf[8];            // Int8: scale as fp32
  float zf[8];            // Int8: 2^23 + 128 + zero point
};

// Column order of the 8 bf16 values wq_dequant8 returns with PAIR_ORDER:
// position p holds column (p even: p / 2, odd: 4 + p / 2), i.e. the order
// 0 4 1 5 2 6 3 7; wq_pair_pos is its inverse, the position of column i.
__host__ __device__ constexpr int wq_pair_pos(int i) { return i < 4 ? 2 * i : 2 * (i - 4) + 1; }

// scale8: the 8 columns' scales (bf16 bits for Int4/Int8, UE8M0 bytes for
// Mxfp4, packed little-endian in a uint4 / the low 8 bytes); zero8: the 8
// zero-point bytes, or has_zero = false for the default.
template <Wq WQ>
__device__ __forceinline__ void wq_params8(const uint4 scale8, const uint2 zero8, bool has_zero,
                                           WqParams8& p) {
  if constexpr (WQ == Wq::Int4) {
    // pairs of columns (j, j + 4), the order in which wq_dequant8 extracts them
    const uint32_t sw[4] = {scale8.x, scale8.y, scale8.z, scale8.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = (sw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;        // column j
      const uint32_t hi = (sw[2 + (j >> 1)] >> (16 * (j & 1))) & 0xFFFFu;  // column j + 4
      const uint32_t v = lo | (hi << 16);
      p.s2[j] = *reinterpret_cast<const __nv_bfloat162*>(&v);
      const uint32_t zl = has_zero ? (zero8.x >> (8 * j)) & 0xFu : 8u;
      const uint32_t zh = has_zero ? (zero8.y >> (8 * j)) & 0xFu : 8u;
      const uint32_t z = zl | (zh << 16) | 0x43004300u;  // bf16 pair (128 + zl, 128 + zh)
      p.zb2[j] = *reinterpret_cast<const __nv_bfloat162*>(&z);
    }
  } else if constexpr (WQ == Wq::Int8) {
    const uint32_t* s = &scale8.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      p.sf[i] = __uint_as_float(((s[i >> 1] >> (16 * (i & 1))) & 0xFFFFu) << 16);
      const uint32_t zw = i < 4 ? zero8.x : zero8.y;
      const int32_t z = has_zero ? static_cast<int32_t>(static_cast<int8_t>((zw >> (8 * (i & 3))) & 0xFFu)) : 0;
      p.zf[i] = 8388608.0f + static_cast<float>(128 + z);  // exact: integers below 2^24
    }
  } else {
    // bf16 2^(e - 127): exponent field e, or the subnormal 2^-127 for e = 0
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t el = (scale8.x >> (8 * j)) & 0xFFu;  // column j
      const uint32_t eh = (scale8.y >> (8 * j)) & 0xFFu;  // column j + 4
      const uint32_t v = (el == 0 ? 0x0040u : (el << 7)) | ((eh == 0 ? 0x0040u : (eh << 7)) << 16);
      p.s2[j] = *reinterpret_cast<const __nv_bfloat162*>(&v);
    }
  }
}

// 8 codes of one K row -> 8 bf16 values (16 bytes), in column order, or
// with PAIR_ORDER (all but Int8) in the pair order 0 4 1 5 2 6 3 7, which
// saves the final byte permutes.  codes: Int4 / Mxfp4 in c.x (8 nibbles);
// Int8 / Mxfp6 in c.x, c.y (8 bytes).
template <Wq WQ, bool PAIR_ORDER = false>
__device__ __forceinline__ uint4 wq_dequant8(const uint2 c, const WqParams8& p) {
  uint4 r;
  uint32_t* o = &r.x;
  if constexpr (WQ != Wq::Int8) {
    // Int4 / Mxfp4: column i sits at bits 4i; shifted by 4j, one mask takes
    // the nibbles of columns j and j + 4 into the two halves of a bf16 pair.
    // Mxfp6: bytes j of c.x and c.y (columns j, j + 4) into the two halves.
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t t = WqFmt<WQ>::CODE_BITS == 4 ? c.x >> (4 * j)
                                                  : __byte_perm(c.x, c.y, j | ((4 + j) << 8));
      __nv_bfloat162 r2;
      if constexpr (WQ == Wq::Int4) {
        // (128 + q) - (128 + zp) = q - zp exactly; one rounding in the product
        const uint32_t v = (t & 0x000F000Fu) | 0x43004300u;
        r2 = __hmul2(__hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), p.zb2[j]), p.s2[j]);
      } else {
        // The code's exponent and mantissa bits placed as the low exponent
        // and high mantissa bits of a bf16, the sign to bit 15: the value
        // times 2^-(127 - bias) for normal and subnormal codes alike (E2M1:
        // bits 8..6, 2^-126; E3M2: bits 9..5, 2^-124; E2M3: bits 8..4,
        // 2^-126); the power of two back is exact, the block scale rounds once
        uint32_t v, back;
        if constexpr (WQ == Wq::Mxfp4) {
          v = ((t & 0x00070007u) << 6) | ((t & 0x00080008u) << 12);
          back = 0x7E807E80u;  // 2^126
        } else if constexpr (WQ == Wq::Mxfp6e3m2) {
          v = ((t & 0x001F001Fu) << 5) | ((t & 0x00200020u) << 10);
          back = 0x7D807D80u;  // 2^124
        } else {
          v = ((t & 0x001F001Fu) << 4) | ((t & 0x00200020u) << 10);
          back = 0x7E807E80u;  // 2^126
        }
        r2 = __hmul2(__hmul2(*reinterpret_cast<const __nv_bfloat162*>(&v),
                             *reinterpret_cast<const __nv_bfloat162*>(&back)),
                     p.s2[j]);
      }
      h[j] = *reinterpret_cast<const uint32_t*>(&r2);
    }
    if constexpr (PAIR_ORDER) {
      o[0] = h[0];
      o[1] = h[1];
      o[2] = h[2];
      o[3] = h[3];
    } else {
      o[0] = __byte_perm(h[0], h[1], 0x5410);  // columns 0, 1
      o[1] = __byte_perm(h[2], h[3], 0x5410);  // columns 2, 3
      o[2] = __byte_perm(h[0], h[1], 0x7632);  // columns 4, 5
      o[3] = __byte_perm(h[2], h[3], 0x7632);  // columns 6, 7
    }
  } else if constexpr (WQ == Wq::Int8) {
    // 2^23 + (q + 128) built from the offset byte; the difference with
    // 2^23 + 128 + zp is q - zp exactly, the product with the scale is exact
    // in fp32 (at most 17 significant bits) and rounded once to bf16
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b = ((i < 4 ? c.x : c.y) >> (8 * (i & 3))) & 0xFFu;
      f[i] = (__uint_as_float(0x4B000000u | (b ^ 0x80u)) - p.zf[i]) * p.sf[i];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
  return r;
}

}  // namespace gbmoe
