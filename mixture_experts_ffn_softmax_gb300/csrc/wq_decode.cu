// Weight-only quantised expert GEMMs for a few rows per expert (decode).
//
// "fused_moe.py 分析", "WNA16 路径": int4 / int8 expert weights with a scale
// and a zero point per group of K rows (and, "5. 特殊量化格式处理", OCP MX
// FP4 / FP6 weights with a power-of-two scale per 32 rows) are dequantised to
// the activation dtype and multiplied with bf16 activations, fp32 accumulate.
//
// At decode an expert holds a handful of rows (at most M, the call's tokens,
// when a token's experts are distinct), so the layer streams the quantised
// weights once and uses every weight for those few rows only.  The tensor-
// core grouped GEMM expands each weight stage into a bf16 B tile in shared
// memory for a 128-row MMA; at decode that expansion (shared-memory stores,
// proxy fences and barrier hand-offs per stage) bounds it.  Here:
//   - every warp is a worker of its own, with a ring of stages of its own
//     (64 K rows: the expert rows' activations, the codes of its 64 weight
//     columns, their group scales and zero points), filled by TMA copies that
//     its lane 0 issues several stages ahead, across unit boundaries;
//   - each lane expands the codes of 8 columns x 4 K rows per 16-row K step
//     directly into the A-operand registers of mma.sync m16n8k16 (the weight
//     columns as the MMA's M, the expert's rows as its N, 8 per tile; the
//     operands never go back to shared memory);
//   - each weight leaves the expansion as the dequantised bf16 value, the
//     exact (q - zp) * scale (int formats) or code value * 2^(s - 127) (MX)
//     rounded once, as the standalone dequantisation gives it.
// GEMM1 (SwiGLU): a warp unit is 32 gate columns and the same 32 up columns of
// one expert over all of K; lane (g, c) with g < 4 holds gate columns, lane
// (g + 4, c) the matching up columns, and one shuffle pairs them for
// z = SiLU(gate + b_gate) * (up + b_up), stored as bf16 rows of the sorted z.
// GEMM2: a warp unit is 64 output columns of one expert over one of S parts of
// K; part s leaves the weighted fp32 partial rows of the expert's items at
// out[(s * R + item) * H], and the weight-and-reduce adds the parts.  An
// expert with more rows than one pass holds (8 * NT) is taken in row groups.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "wq.cuh"

namespace gbmoe {
namespace {

// eight warps per CTA, one CTA per SM: measured on GB300 the same as sixteen
// for the MX formats and faster for the int ones (whose deferred group sums
// need registers a 16-warp CTA does not have)
constexpr int kDecWarps = 8;
constexpr int kDecKR = 64;        // K rows per stage
constexpr int kDecCols = 64;      // weight columns per warp unit
constexpr int kDecMaxE = 1024;    // experts the touched list holds
constexpr int kDecParamRows = 2;  // parameter rows per stage (groups of >= 32 rows)
constexpr int kDecSmemMax = 232448;

template <Wq WQ, int NT, int WARPS>
struct Dec {
  using F = WqFmt<WQ>;
  static constexpr int XROWS = 8 * NT;                       // expert rows per pass
  static constexpr int XB = kDecKR * 2 * XROWS;              // activations, 128B-swizzled rows
  static constexpr int RB = kDecCols * F::CODE_BITS / 8;     // code bytes per K row
  static constexpr int CB = kDecKR * RB;                     // codes per stage
  static constexpr int SB = (kDecParamRows * kDecCols * F::SCALE_BYTES + 127) / 128 * 128;
  static constexpr int ZB = F::HAS_ZERO ? kDecParamRows * kDecCols : 0;
  static constexpr int STAGE = XB + CB + SB + ZB;
  static constexpr int FIXED = 1024 + (kDecMaxE + 1) * 4 + WARPS * 8 * 8;
  static constexpr int DEPTH = (kDecSmemMax - FIXED) / (WARPS * STAGE);
  static constexpr int D = DEPTH < 6 ? DEPTH : 6;            // stages per warp ring
  static constexpr int X_OFF = 0;
  static constexpr int C_OFF = X_OFF + WARPS * D * XB;
  static constexpr int S_OFF = C_OFF + WARPS * D * CB;
  static constexpr int Z_OFF = S_OFF + WARPS * D * SB;
  static constexpr int BAR_OFF = Z_OFF + WARPS * D * ZB;
  static constexpr int LIST_OFF = BAR_OFF + WARPS * D * 8;
  static constexpr int SMEM = 1024 + LIST_OFF + (kDecMaxE + 1) * 4;
  static_assert(XB % 1024 == 0 && C_OFF % 1024 == 0, "swizzled activation tiles 1024-aligned");
  static_assert(CB % 128 == 0 && SB % 128 == 0 && ZB % 128 == 0, "TMA destinations 128-aligned");
  static_assert(D >= 3 && SMEM <= kDecSmemMax, "shared memory budget");
};

struct DecParams {
  const int32_t* counts;      // expert_num_tokens [E]
  const int32_t* offsets;     // padded expert offsets [E + 1]
  const bf16* bias;           // GEMM1 [E, 2N], GEMM2 [E, N], or null
  void* out;                  // GEMM1: z bf16 [cap, N]; GEMM2: fp32 parts [S, R, N]
  const int32_t* row_index;   // GEMM2: routed item per sorted row
  const float* row_weight;    // GEMM2: weight per routed item, or null (= 1)
  int32_t* error_word;
  int64_t R;                  // GEMM2: routed items (rows of one part)
  int32_t E, N, K;            // N: GEMM1 columns per half (I), GEMM2 output columns (H)
  int32_t ncb;                // column blocks per expert (GEMM1 N / 32, GEMM2 N / 64)
  int32_t splits;             // K parts (GEMM2)
  int32_t gshift;             // log2 of the K rows per parameter row (a group, or 32)
  int32_t has_zero;
};

struct Unit {
  int32_t e, off, n, cb, s, st0, nst, ngr;
};

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}
__device__ __forceinline__ uint2 lds64(const uint8_t* p) {
  return *reinterpret_cast<const uint2*>(p);
}
__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint32_t bf2u(__nv_bfloat162 v) {
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ __nv_bfloat162 u2bf(uint32_t v) {
  return *reinterpret_cast<const __nv_bfloat162*>(&v);
}

// Four 8x8 b16 matrices from shared memory (one row address per lane).
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(ptx::smem_u32(row)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(ptx::smem_u32(row)));
}

// d += a (16x16, row-major) * b (16x8, column-major); bf16 in, fp32 out.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Per-column parameters of the lane's 8 columns for the current group /
// block, in the form the expansion uses.
struct ColParams {
  uint32_t p2[8];  // Int4: bf16 pair (128 + zp, 128 + zp); MX: bf16 pair of the
                   // exact multiplier 2^bias * scale
  uint32_t s2[8];  // Int4: bf16 pair (scale, scale)
  float zf[8];     // Int8: 2^23 + 128 + zp
  float sf[8];     // Int8: the group scale
};

// Parameter row `pr` of a stage: 64 columns, the lane's 8 at column 8g.
template <Wq WQ>
__device__ __forceinline__ void load_params(const uint8_t* ssm, const uint8_t* zsm, int pr, int g,
                                            bool has_zero, ColParams& p) {
  using F = WqFmt<WQ>;
  if constexpr (F::MX) {
    const uint2 sc = lds64(ssm + pr * kDecCols + 8 * g);
    // the expansion leaves value * 2^-126 (E2M1, E2M3) or 2^-124 (E3M2);
    // 2^126 (2^124) * 2^(s - 127) is a power of two, exact in bf16
    const __nv_bfloat162 back = u2bf(WQ == Wq::Mxfp6e3m2 ? 0x7D807D80u : 0x7E807E80u);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t el = ((j < 4 ? sc.x : sc.y) >> (8 * (j & 3))) & 0xFFu;
      const uint32_t h = el == 0 ? 0x0040u : (el << 7);
      p.p2[j] = bf2u(__hmul2(back, u2bf(h | (h << 16))));
    }
  } else {
    const uint4 sc = lds128(ssm + (pr * kDecCols + 8 * g) * 2);
    const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t sb = (sw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
      if constexpr (WQ == Wq::Int4)
        p.s2[j] = sb | (sb << 16);
      else
        p.sf[j] = __uint_as_float(sb << 16);
    }
    const uint2 zw = has_zero ? lds64(zsm + pr * kDecCols + 8 * g) : make_uint2(0u, 0u);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t zb = ((j < 4 ? zw.x : zw.y) >> (8 * (j & 3))) & 0xFFu;
      if constexpr (WQ == Wq::Int4) {
        const uint32_t z = (has_zero ? (zb & 0xFu) : 8u) | 0x4300u;  // bf16 128 + zp
        p.p2[j] = z | (z << 16);
      } else {
        const int32_t z = has_zero ? static_cast<int32_t>(static_cast<int8_t>(zb)) : 0;
        p.zf[j] = 8388608.0f + static_cast<float>(128 + z);
      }
    }
  }
}

// Codes of one column for K rows k and k + 1 -> bf16 pair (row k low).
// `t` holds the row-k code at bits 0.. and the row-(k+1) code at bits 16..
// (nibbles for 4-bit formats, bytes for 8-bit ones).
template <Wq WQ>
__device__ __forceinline__ uint32_t expand_pair(uint32_t t, const ColParams& p, int j) {
  if constexpr (WQ == Wq::Int4) {
    // (128 + q) - (128 + zp) = q - zp exactly; one rounding in the product
    return bf2u(__hmul2(__hsub2(u2bf((t & 0x000F000Fu) | 0x43004300u), u2bf(p.p2[j])),
                        u2bf(p.s2[j])));
  } else if constexpr (WQ == Wq::Int8) {
    // q - zp exactly, times the scale exactly in fp32 (16 significant bits
    // at most), rounded once to bf16
    const float lo = (__uint_as_float(0x4B000000u | ((t ^ 0x80u) & 0xFFu)) - p.zf[j]) * p.sf[j];
    const float hi =
        (__uint_as_float(0x4B000000u | (((t >> 16) ^ 0x80u) & 0xFFu)) - p.zf[j]) * p.sf[j];
    return bf2u(__floats2bfloat162_rn(lo, hi));
  } else {
    // exponent and mantissa bits as the low exponent and high mantissa bits
    // of a bf16, the sign to bit 15, then the exact power-of-two multiplier
    uint32_t v;
    if constexpr (WQ == Wq::Mxfp4)
      v = ((t & 0x00070007u) << 6) | ((t & 0x00080008u) << 12);
    else if constexpr (WQ == Wq::Mxfp6e3m2)
      v = ((t & 0x001F001Fu) << 5) | ((t & 0x00200020u) << 10);
    else
      v = ((t & 0x001F001Fu) << 4) | ((t & 0x00200020u) << 10);
    return bf2u(__hmul2(u2bf(v), u2bf(p.p2[j])));
  }
}

// A-operand registers of the four MMAs of one 16-row K step: MMA i takes the
// lane's columns 2i (M row g) and 2i + 1 (M row g + 8); a[i][0..1] rows
// 2c, 2c + 1 of the step, a[i][2..3] rows 2c + 8, 2c + 9.
template <Wq WQ>
__device__ __forceinline__ void expand_step(const uint8_t* csm, int row, int g, const ColParams& p,
                                            uint32_t (&a)[4][4]) {
  using F = WqFmt<WQ>;
  constexpr int RB = kDecCols * F::CODE_BITS / 8;
  if constexpr (F::CODE_BITS == 4) {
    const uint32_t w0 = lds32(csm + row * RB + 4 * g);
    const uint32_t w1 = lds32(csm + (row + 1) * RB + 4 * g);
    const uint32_t w8 = lds32(csm + (row + 8) * RB + 4 * g);
    const uint32_t w9 = lds32(csm + (row + 9) * RB + 4 * g);
    // bytes b0 b1 of rows k and k + 1: columns 0..3 at nibbles (0, 4, 8, 12)
    // of the low half and (16, 20, 24, 28) of the high half
    const uint32_t x01 = __byte_perm(w0, w1, 0x5410), y01 = __byte_perm(w0, w1, 0x7632);
    const uint32_t x89 = __byte_perm(w8, w9, 0x5410), y89 = __byte_perm(w8, w9, 0x7632);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t s0 = i < 2 ? x01 : y01, s8 = i < 2 ? x89 : y89;
      const int sh = (i & 1) * 8;
      a[i][0] = expand_pair<WQ>(s0 >> sh, p, 2 * i);
      a[i][1] = expand_pair<WQ>(s0 >> (sh + 4), p, 2 * i + 1);
      a[i][2] = expand_pair<WQ>(s8 >> sh, p, 2 * i);
      a[i][3] = expand_pair<WQ>(s8 >> (sh + 4), p, 2 * i + 1);
    }
  } else {
    const uint2 w0 = lds64(csm + row * RB + 8 * g);
    const uint2 w1 = lds64(csm + (row + 1) * RB + 8 * g);
    const uint2 w8 = lds64(csm + (row + 8) * RB + 8 * g);
    const uint2 w9 = lds64(csm + (row + 9) * RB + 8 * g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = 2 * i + h;  // column
        const uint32_t sel = (j & 3) | ((4 + (j & 3)) << 8);
        const uint32_t t01 = j < 4 ? __byte_perm(w0.x, w1.x, sel) : __byte_perm(w0.y, w1.y, sel);
        const uint32_t t89 = j < 4 ? __byte_perm(w8.x, w9.x, sel) : __byte_perm(w8.y, w9.y, sel);
        a[i][h] = expand_pair<WQ>(t01, p, j);
        a[i][2 + h] = expand_pair<WQ>(t89, p, j);
      }
    }
  }
}

// Waits for phase `parity` of `bar`, all lanes; warp-uniform result.  Gives
// up after the wait limit, recording MOE_ERR_TIMEOUT.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                          uint64_t limit_ns = kWaitLimitNs) {
  bool ok = ptx::mbar_try_wait(bar, parity);
  if (!ok) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ok) {
      ok = ptx::mbar_try_wait_suspend(bar, parity, 1000000u);
      if (!ok && ptx::globaltimer_ns() - t0 > limit_ns) break;
    }
  }
  ok = __all_sync(0xFFFFFFFFu, ok);
  if (!ok && (threadIdx.x & 31) == 0) record_error(err, MOE_ERR_TIMEOUT);
  return ok;
}

template <Wq WQ, bool SWI, int NT, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1)
    wq_decode_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                     const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                     const DecParams P) {
  using L = Dec<WQ, NT, WARPS>;
  using F = WqFmt<WQ>;
  constexpr bool INT = !F::MX;
  constexpr int D = L::D;
  extern __shared__ uint8_t dsmem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  pdl_begin();
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int g = lane >> 2, c = lane & 3;
  int32_t* list = reinterpret_cast<int32_t*>(sm + L::LIST_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF) + warp * D;
  if (warp == 0) {
    // the experts that hold rows, in order
    int n = 0;
    for (int e0 = 0; e0 < P.E; e0 += 32) {
      const int e = e0 + lane;
      const bool t = e < P.E && __ldg(P.counts + e) > 0;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, t);
      if (t) list[n + __popc(m & ((1u << lane) - 1u))] = e;
      n += __popc(m);
    }
    if (lane == 0) list[kDecMaxE] = n;
  }
  if (lane == 0) {
    for (int i = 0; i < D; ++i) ptx::mbar_init(&full[i], 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  const int64_t units = static_cast<int64_t>(list[kDecMaxE]) * P.ncb * P.splits;
  const int64_t W = static_cast<int64_t>(gridDim.x) * WARPS;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
  if (first >= units) return;
  if (lane == 0) {
    ptx::prefetch_tmap(&tmX);
    ptx::prefetch_tmap(&tmC);
    ptx::prefetch_tmap(&tmS);
    if (INT && P.has_zero) ptx::prefetch_tmap(&tmZ);
  }
  const int NS = (P.K + kDecKR - 1) / kDecKR;
  const int gsh = INT ? P.gshift : 5;  // K rows per parameter row: 1 << gsh
  const int gmask = (1 << gsh) - 1;
  auto unit_at = [&](int64_t u, Unit& U) {
    U.cb = static_cast<int32_t>(u % P.ncb);
    const int64_t r = u / P.ncb;
    U.s = static_cast<int32_t>(r % P.splits);
    U.e = list[r / P.splits];
    U.off = __ldg(P.offsets + U.e);
    U.n = __ldg(P.counts + U.e);
    U.st0 = U.s * NS / P.splits;
    U.nst = (U.s + 1) * NS / P.splits - U.st0;
    U.ngr = (U.n + L::XROWS - 1) / L::XROWS;
  };
  uint8_t* xs = sm + L::X_OFF + warp * D * L::XB;
  uint8_t* cs = sm + L::C_OFF + warp * D * L::CB;
  uint8_t* ss = sm + L::S_OFF + warp * D * L::SB;
  uint8_t* zs = sm + L::Z_OFF + warp * D * L::ZB;
  const uint32_t prow = gsh == 5 ? 2u : 1u;  // parameter rows per stage copy
  const uint32_t tx = L::XB + L::CB + prow * kDecCols * F::SCALE_BYTES +
                      ((INT && P.has_zero) ? prow * kDecCols : 0u);

  // producer cursor (lane 0 issues, every lane tracks it)
  int64_t pu = first;
  Unit PU;
  unit_at(pu, PU);
  int prg = 0, pst = 0;
  auto issue = [&](int slot) -> bool {
    if (pu >= units) return false;
    if (lane == 0) {
      const int k0 = (PU.st0 + pst) * kDecKR;
      uint64_t* bar = &full[slot];
      ptx::mbar_arrive_expect_tx(bar, tx);
      ptx::tma_load_2d(xs + slot * L::XB, &tmX, bar, k0, PU.off + prg * L::XROWS);
      if constexpr (SWI)
        ptx::tma_load_4d(cs + slot * L::CB, &tmC, bar, PU.cb * (L::RB / 2), 0, k0, PU.e);
      else
        ptx::tma_load_3d(cs + slot * L::CB, &tmC, bar, PU.cb * L::RB, k0, PU.e);
      const int gr = k0 >> gsh;
      if constexpr (SWI)
        ptx::tma_load_4d(ss + slot * L::SB, &tmS, bar, PU.cb * 32, 0, gr, PU.e);
      else
        ptx::tma_load_3d(ss + slot * L::SB, &tmS, bar, PU.cb * 64, gr, PU.e);
      if (INT && P.has_zero) {
        if constexpr (SWI)
          ptx::tma_load_4d(zs + slot * L::ZB, &tmZ, bar, PU.cb * 32, 0, gr, PU.e);
        else
          ptx::tma_load_3d(zs + slot * L::ZB, &tmZ, bar, PU.cb * 64, gr, PU.e);
      }
    }
    if (++pst == PU.nst) {
      pst = 0;
      if (++prg == PU.ngr) {
        prg = 0;
        pu += W;
        if (pu < units) unit_at(pu, PU);
      }
    }
    return true;
  };
  int inflight = 0;  // stages issued and not yet consumed
  while (inflight < D && issue(inflight)) ++inflight;

  float acc[4][NT][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][t][q] = 0.0f;
  ColParams prm;
  int slot = 0;
  uint32_t phase = 0;
  for (int64_t u = first; u < units; u += W) {
    Unit U;
    unit_at(u, U);
    const int kend = min(P.K, (U.st0 + U.nst) * kDecKR);
    for (int rg = 0; rg < U.ngr; ++rg) {
      const int rows_here = min(L::XROWS, U.n - rg * L::XROWS);  // rows of this pass
      for (int st = 0; st < U.nst; ++st) {
        if (!warp_wait(&full[slot], phase, P.error_word)) {
          // give the copies still in flight a bounded time to land, then stop
          for (int i = 0; i < inflight; ++i) {
            const int sl = (slot + i) % D;
            const uint32_t ph = phase ^ (slot + i >= D ? 1u : 0u);
            if (!warp_wait(&full[sl], ph, nullptr, 100000000ull)) break;
          }
          return;
        }
        const int k0 = (U.st0 + st) * kDecKR;
        const uint8_t* xsm = xs + slot * L::XB;
        const uint8_t* csm = cs + slot * L::CB;
        const uint8_t* ssm = ss + slot * L::SB;
        const uint8_t* zsm = zs + slot * L::ZB;
#pragma unroll
        for (int j = 0; j < kDecKR / 16; ++j) {
          const int kk = k0 + 16 * j;
          if (kk < kend) {
            if constexpr (INT) {
              if ((kk & gmask) == 0 || (st == 0 && j == 0))
                load_params<WQ>(ssm, zsm, (kk >> gsh) - (k0 >> gsh), g, P.has_zero != 0, prm);
            } else {
              if ((j & 1) == 0) load_params<WQ>(ssm, zsm, j >> 1, g, false, prm);
            }
            uint32_t a[4][4];
            expand_step<WQ>(csm, 16 * j + 2 * c, g, prm, a);
            // activations: tile t rows 8t..8t+7, K columns 16j.. (chunk 2j)
            // and 16j+8.. (chunk 2j+1) of the 128B-swizzled stage rows
            uint32_t b[NT][2];
            {
              const int q = lane >> 3, rr = lane & 7;
              if constexpr (NT == 1) {
                const uint8_t* p = xsm + rr * 128 + (((2 * j + (q & 1)) ^ rr) << 4);
                ldsm_x2(b[0][0], b[0][1], p);
              } else {
#pragma unroll
                for (int t2 = 0; t2 < NT; t2 += 2) {
                  const int row = 8 * (t2 + (q >> 1)) + rr;
                  const uint8_t* p = xsm + row * 128 + (((2 * j + (q & 1)) ^ rr) << 4);
                  ldsm_x4(b[t2][0], b[t2][1], b[t2 + 1][0], b[t2 + 1][1], p);
                }
              }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (8 * t < rows_here) {
#pragma unroll
                for (int i = 0; i < 4; ++i) mma_bf16(acc[i][t], a[i], b[t][0], b[t][1]);
              }
            }
          }
        }
        __syncwarp();
        if (!issue(slot)) --inflight;  // the stage D ahead takes the slot just read
        if (++slot == D) {
          slot = 0;
          phase ^= 1u;
        }
      }
      // ---- epilogue of one row group of the unit ----
      float (&V)[4][NT][4] = acc;
      if constexpr (SWI) {
        const int zc = U.cb * 32 + 8 * (g & 3);  // z column of the lane's first value
        float bg[8], bu[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) bg[j] = bu[j] = 0.0f;
        if (P.bias != nullptr) {
          const uint4 vg = __ldg(reinterpret_cast<const uint4*>(P.bias + static_cast<int64_t>(U.e) * 2 * P.N + zc));
          const uint4 vu = __ldg(reinterpret_cast<const uint4*>(P.bias + static_cast<int64_t>(U.e) * 2 * P.N + P.N + zc));
          const uint32_t wg[4] = {vg.x, vg.y, vg.z, vg.w}, wu[4] = {vu.x, vu.y, vu.z, vu.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 fg = __bfloat1622float2(u2bf(wg[j])), fu = __bfloat1622float2(u2bf(wu[j]));
            bg[2 * j] = fg.x;
            bg[2 * j + 1] = fg.y;
            bu[2 * j] = fu.x;
            bu[2 * j + 1] = fu.y;
          }
        }
        const bool gate = g < 4;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          // gate lanes finish row 2c of the tile, up lanes row 2c + 1
          float snd[8], rcv[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            snd[2 * i] = gate ? V[i][t][1] : V[i][t][0];
            snd[2 * i + 1] = gate ? V[i][t][3] : V[i][t][2];
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) rcv[j] = __shfl_xor_sync(0xFFFFFFFFu, snd[j], 16);
          const int row = rg * L::XROWS + 8 * t + 2 * c + (gate ? 0 : 1);
          if (row < U.n) {
            uint32_t zw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float g0 = gate ? V[i][t][0] : rcv[2 * i];
              const float g1 = gate ? V[i][t][2] : rcv[2 * i + 1];
              const float u0 = gate ? rcv[2 * i] : V[i][t][1];
              const float u1 = gate ? rcv[2 * i + 1] : V[i][t][3];
              const float z0 = silu(g0 + bg[2 * i]) * (u0 + bu[2 * i]);
              const float z1 = silu(g1 + bg[2 * i + 1]) * (u1 + bu[2 * i + 1]);
              zw[i] = bf2u(__floats2bfloat162_rn(z0, z1));
            }
            bf16* z = static_cast<bf16*>(P.out) + static_cast<int64_t>(U.off + row) * P.N + zc;
            *reinterpret_cast<uint4*>(z) = make_uint4(zw[0], zw[1], zw[2], zw[3]);
          }
        }
      } else {
        const int oc = U.cb * 64 + 8 * g;
        float b8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) b8[j] = 0.0f;
        if (P.bias != nullptr && U.s == 0) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(P.bias + static_cast<int64_t>(U.e) * P.N + oc));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(u2bf(w4[j]));
            b8[2 * j] = f.x;
            b8[2 * j + 1] = f.y;
          }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int row = rg * L::XROWS + 8 * t + 2 * c + h2;
            if (row < U.n) {
              const int32_t item = __ldg(P.row_index + U.off + row);
              const float w = P.row_weight != nullptr ? __ldg(P.row_weight + item) : 1.0f;
              float v[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                v[2 * i] = (V[i][t][h2] + b8[2 * i]) * w;
                v[2 * i + 1] = (V[i][t][2 + h2] + b8[2 * i + 1]) * w;
              }
              float* o = static_cast<float*>(P.out) +
                         (static_cast<int64_t>(U.s) * P.R + item) * P.N + oc;
              reinterpret_cast<float4*>(o)[0] = make_float4(v[0], v[1], v[2], v[3]);
              reinterpret_cast<float4*>(o)[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[i][t][q] = 0.0f;
    }
  }
}

// y[t] = sum over the token's routed items r (those the align placed) and
// the K parts s of parts[(s * R + r) * H]; the parts are weighted already.
// One thread per 4 columns of a token; the (item, part) rows are taken eight
// at a time with their loads issued together (the call is a handful of
// tokens, so the latency of dependent loads would bound it).
__global__ void __launch_bounds__(256)
    reduce_parts_kernel(const float* __restrict__ parts, const int32_t* __restrict__ inv,
                        int64_t M, int k, int H, int S, bf16* __restrict__ y) {
  pdl_begin();
  const int hv = H / 4;
  const int64_t R = M * k;
  const int64_t total = M * hv;
  const int n = k * S;  // (item, part) rows of a token, item-major
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / hv;
    const int cc = static_cast<int>(i - t * hv);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < n; q0 += 8) {
      float4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int qq = q0 + q;
        if (qq < n) {
          const int64_t r = t * k + qq / S;
          if (__ldg(inv + r) >= 0)
            v[q] = __ldg(reinterpret_cast<const float4*>(parts + ((qq % S) * R + r) * H) + cc);
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        acc.x += v[q].x;
        acc.y += v[q].y;
        acc.z += v[q].z;
        acc.w += v[q].w;
      }
    }
    const uint32_t w0 = bf2u(__floats2bfloat162_rn(acc.x, acc.y));
    const uint32_t w1 = bf2u(__floats2bfloat162_rn(acc.z, acc.w));
    *reinterpret_cast<uint2*>(y + t * H + static_cast<int64_t>(cc) * 4) = make_uint2(w0, w1);
  }
}

int dec_nt(int64_t M) { return M <= 8 ? 1 : (M <= 16 ? 2 : 4); }

// Tensor maps and launch of one decode GEMM.
template <Wq WQ, bool SWI, int NT, int WARPS>
moe_status_t launch_dec_nt(const GroupedGemmArgs& a, const int32_t* counts, int32_t splits,
                           int64_t R, const char* name, cudaStream_t s) {
  using L = Dec<WQ, NT, WARPS>;
  using F = WqFmt<WQ>;
  auto kernel = wq_decode_kernel<WQ, SWI, NT, WARPS>;
  static PerDevice attrs;
  if (attrs.get([&](int*) {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
      }) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute(%s): %s", name,
                     cudaGetErrorString(cudaGetLastError()));
  const uint64_t E = static_cast<uint64_t>(a.E), K = static_cast<uint64_t>(a.K),
                 N = static_cast<uint64_t>(a.N), cap = static_cast<uint64_t>(a.cap);
  const int gs = F::MX ? 32 : a.wq_group;
  const uint64_t KG = K / static_cast<uint64_t>(gs);
  const uint32_t prow = gs == 32 ? 2u : 1u;
  const uint64_t sb = F::SCALE_BYTES;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapDataType sdt = sb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : u8;
  const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE;
  CUtensorMap tmX, tmC, tmS, tmZ;
  {
    const uint64_t dims[2] = {K, cap};
    const uint64_t strides[1] = {K * 2};
    const uint32_t box[2] = {kDecKR, static_cast<uint32_t>(L::XROWS)};
    if (moe_status_t st = encode_tensor_map(&tmX, a.a, 2, dims, strides, box,
                                            CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                            CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
  }
  const uint64_t nbytes = N * F::CODE_BITS / 8;  // code bytes of one K row (per half)
  if constexpr (SWI) {
    // w13 [E, K, 2, N]: codes (bytes, half, k, e), parameters (n, half, group, e)
    const uint64_t cd[4] = {nbytes, 2, K, E};
    const uint64_t cst[3] = {nbytes, 2 * nbytes, 2 * nbytes * K};
    const uint32_t cbx[4] = {static_cast<uint32_t>(L::RB / 2), 2, kDecKR, 1};
    if (moe_status_t st = encode_tensor_map(&tmC, a.w, 4, cd, cst, cbx, u8, none)) return st;
    const uint64_t pd[4] = {N, 2, KG, E};
    const uint64_t ps[3] = {N * sb, 2 * N * sb, 2 * N * sb * KG};
    const uint32_t pbx[4] = {32, 2, prow, 1};
    if (moe_status_t st = encode_tensor_map(&tmS, a.wq_scale, 4, pd, ps, pbx, sdt, none)) return st;
    tmZ = tmS;
    if (!F::MX && a.wq_zero != nullptr) {
      const uint64_t zs[3] = {N, 2 * N, 2 * N * KG};
      if (moe_status_t st = encode_tensor_map(&tmZ, a.wq_zero, 4, pd, zs, pbx, u8, none)) return st;
    }
  } else {
    const uint64_t cd[3] = {nbytes, K, E};
    const uint64_t cst[2] = {nbytes, nbytes * K};
    const uint32_t cbx[3] = {static_cast<uint32_t>(L::RB), kDecKR, 1};
    if (moe_status_t st = encode_tensor_map(&tmC, a.w, 3, cd, cst, cbx, u8, none)) return st;
    const uint64_t pd[3] = {N, KG, E};
    const uint64_t ps[2] = {N * sb, N * sb * KG};
    const uint32_t pbx[3] = {64, prow, 1};
    if (moe_status_t st = encode_tensor_map(&tmS, a.wq_scale, 3, pd, ps, pbx, sdt, none)) return st;
    tmZ = tmS;
    if (!F::MX && a.wq_zero != nullptr) {
      const uint64_t zs[2] = {N, N * KG};
      if (moe_status_t st = encode_tensor_map(&tmZ, a.wq_zero, 3, pd, zs, pbx, u8, none)) return st;
    }
  }
  DecParams P{};
  P.counts = counts;
  P.offsets = a.offsets;
  P.bias = a.bias;
  P.out = a.out;
  P.row_index = a.row_index;
  P.row_weight = a.row_weight;
  P.error_word = a.error_word;
  P.R = R;
  P.E = a.E;
  P.N = a.N;
  P.K = a.K;
  P.ncb = SWI ? a.N / 32 : a.N / 64;
  P.splits = SWI ? 1 : splits;
  P.gshift = 31 - __builtin_clz(static_cast<unsigned>(gs));  // gs: a power of two
  P.has_zero = (!F::MX && a.wq_zero != nullptr) ? 1 : 0;
  prof_before(name, s);
  launch_kernel(kernel, static_cast<unsigned>(a.num_sms), WARPS * 32, L::SMEM, s, tmX, tmC, tmS,
                tmZ, P);
  prof_after(name, s);
  return check_launch(name);
}

template <Wq WQ, bool SWI>
moe_status_t launch_dec(const GroupedGemmArgs& a, const int32_t* counts, int64_t M,
                        int32_t splits, int64_t R, const char* name, cudaStream_t s) {
  switch (dec_nt(M)) {
    case 1: return launch_dec_nt<WQ, SWI, 1, kDecWarps>(a, counts, splits, R, name, s);
    case 2: return launch_dec_nt<WQ, SWI, 2, kDecWarps>(a, counts, splits, R, name, s);
    default: return launch_dec_nt<WQ, SWI, 4, kDecWarps>(a, counts, splits, R, name, s);
  }
}

}  // namespace

bool wq_decode_applies(int64_t M, int32_t H, int32_t I, int32_t E, int32_t format, int32_t group) {
  if (M < 1 || M > 32 || E > kDecMaxE) return false;
  if (H % 64 != 0 || I % 32 != 0 || H < 64 || I < 64) return false;
  if (format < MOE_WQ_MXFP4) {
    // int formats: groups of a power of two >= 32 rows (whole 16-row K steps
    // and at most two parameter rows per 64-row stage)
    if (group < 32 || (group & (group - 1)) != 0) return false;
  }
  return true;
}

// K parts of GEMM2: the count that spreads (touched experts x column blocks
// x parts) warp units most evenly over the resident warps, the fewest among
// equals; the parts' rows must fit the fp32 row region (cap rows).
int wq_decode_splits(int64_t M, int32_t top_k, int32_t H, int32_t I, int32_t E, int64_t cap,
                     int32_t num_sms) {
  const int64_t R = M * top_k;
  const int64_t touched = std::min<int64_t>(E, R);
  const int64_t ncb = H / 64;
  const int64_t W = static_cast<int64_t>(num_sms) * kDecWarps;
  const int NS = (I + kDecKR - 1) / kDecKR;
  int best = 1;
  double best_cost = 1e30;
  for (int S = 1; S <= 16 && S <= NS && S * R <= cap; ++S) {
    const int64_t U = touched * ncb * S;
    const double cost = static_cast<double>((U + W - 1) / W) / S;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

moe_status_t launch_wq_decode_gemm1(const GroupedGemmArgs& a, const int32_t* counts, int64_t M,
                                    cudaStream_t s) {
  switch (a.wq_format) {
    case 0: return launch_dec<Wq::Int4, true>(a, counts, M, 1, 0, "gemm1_swiglu_int4_decode", s);
    case 1: return launch_dec<Wq::Int8, true>(a, counts, M, 1, 0, "gemm1_swiglu_int8_decode", s);
    case 2: return launch_dec<Wq::Mxfp4, true>(a, counts, M, 1, 0, "gemm1_swiglu_mxfp4_decode", s);
    case 3: return launch_dec<Wq::Mxfp6e3m2, true>(a, counts, M, 1, 0, "gemm1_swiglu_mxfp6_decode", s);
    case 4: return launch_dec<Wq::Mxfp6e2m3, true>(a, counts, M, 1, 0, "gemm1_swiglu_mxfp6_decode", s);
    default: return set_error(MOE_ERR_INVALID_ARG, "weight format %d", a.wq_format);
  }
}

moe_status_t launch_wq_decode_gemm2(const GroupedGemmArgs& a, const int32_t* counts, int64_t M,
                                    int32_t splits, int64_t R, cudaStream_t s) {
  switch (a.wq_format) {
    case 0: return launch_dec<Wq::Int4, false>(a, counts, M, splits, R, "gemm2_int4_decode", s);
    case 1: return launch_dec<Wq::Int8, false>(a, counts, M, splits, R, "gemm2_int8_decode", s);
    case 2: return launch_dec<Wq::Mxfp4, false>(a, counts, M, splits, R, "gemm2_mxfp4_decode", s);
    case 3: return launch_dec<Wq::Mxfp6e3m2, false>(a, counts, M, splits, R, "gemm2_mxfp6_decode", s);
    case 4: return launch_dec<Wq::Mxfp6e2m3, false>(a, counts, M, splits, R, "gemm2_mxfp6_decode", s);
    default: return set_error(MOE_ERR_INVALID_ARG, "weight format %d", a.wq_format);
  }
}

moe_status_t launch_reduce_parts(const float* parts, const int32_t* inv, int64_t M, int32_t k,
                                 int32_t H, int32_t splits, bf16* y, cudaStream_t s) {
  if (M <= 0) return MOE_OK;
  const int64_t total = M * (H / 4);
  const unsigned grid = static_cast<unsigned>(
      std::max<int64_t>(1, std::min<int64_t>(ceil_div<int64_t>(total, 256), 4096)));
  prof_before("reduce_parts", s);
  launch_kernel(reduce_parts_kernel, grid, 256, 0, s, parts, inv, M, k, H, splits, y);
  prof_after("reduce_parts", s);
  return check_launch("reduce_parts");
}

}  // namespace gbmoe
