// Weight-only int4 decode GEMMs on the tcgen05 tensor cores, the weights as
// the MMA's A operand in tensor memory.
//
// "fused_moe.py 分析", "WNA16 路径": int4 expert weights with a scale and a
// zero point per group of G rows along K, bf16 activations, fp32
// accumulation.  For a group g of weight column n,
//   sum_{k in g} x_k (q_kn - zp_gn) s_gn
//     = s_gn * ( sum_k x_k (128 + q_kn) - (128 + zp_gn) * sum_k x_k ),
// the group's exact contribution.  For calls of at most 32 tokens, with the
// codes repacked once along K (moe_wq_pack_k):
//   - a unit is 128 weight columns of one touched expert (GEMM1: 64 gate and
//     the same 64 up columns; GEMM2: 128 output columns over one of S parts
//     of K), one CTA per SM walking its units;
//   - one thread streams 64-row K stages by TMA into a ring: the expert
//     rows' activations (NR rows, 128-byte swizzle), the 128 columns' codes
//     (32 bytes of K-packed codes each, 32-byte swizzle) and, at a group's
//     first stage, its scales and zero points;
//   - four converter warps, one thread per weight column = TMEM lane, turn
//     the codes of their column into the bf16 values 128 + q (a mask per K
//     pair, exact) and store them with tcgen05.st as the stage's A operand
//     (128 lanes x 32 columns of bf16 pairs);
//   - one thread issues tcgen05.mma (M = 128 columns, N = NR rows, K = 16)
//     with A in tensor memory and the activations in shared memory into the
//     group's accumulator, and the same MMA with A = ones into a second
//     accumulator that collects sum_k x_k; a group's pair of accumulators
//     alternates between two TMEM buffers;
//   - after each group the converter threads read both accumulators of their
//     lane and fold s * (acc - (128 + zp) * xsum) into registers; at the end
//     of a unit GEMM1 pairs the gate and up lanes through shared memory for
//     z = SiLU(gate + b_gate) * (up + b_up), GEMM2 writes the weighted fp32
//     part rows that the weight-and-reduce adds.
// The dequantised weight is never rounded to bf16 here, so results agree
// with the standalone dequantisation path to that rounding.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace gbmoe {
namespace {

constexpr int kTKR = 64;        // K rows per stage
constexpr int kTCols = 128;     // weight columns per unit = TMEM lanes = MMA M
constexpr int kTStages = 16;    // shared-memory ring (also keeps one CTA per SM)
constexpr int kTABufs = 3;      // A operand buffers in TMEM, 32 columns each
constexpr int kTWarps = 6;      // producer, MMA, four converter warps
constexpr int kTMaxE = 1024;    // experts the touched list holds
constexpr uint32_t kTTmemCols = 256;

template <int NR>
struct TLay {
  static constexpr int XB = NR * 128;              // activations: NR rows x 64 bf16
  static constexpr int CB = kTCols * (kTKR / 2);   // codes: 128 columns x 32 bytes
  static constexpr int SB = kTCols * 2;            // scales, bf16
  static constexpr int ZB = kTCols;                // zero points, bytes
  static constexpr int X_OFF = 0;
  static constexpr int C_OFF = XB;
  static constexpr int S_OFF = C_OFF + CB;
  static constexpr int Z_OFF = S_OFF + SB;
  static constexpr int STAGE = (Z_OFF + ZB + 1023) / 1024 * 1024;
  static constexpr int XCH_OFF = kTStages * STAGE;              // gate/up exchange
  static constexpr int LIST_OFF = XCH_OFF + 64 * (NR + 1) * 4;  // touched experts
  static constexpr int SMEM = 1024 + LIST_OFF + (kTMaxE + 1) * 4;
  // TMEM columns
  static constexpr uint32_t A_COL = 0;                  // kTABufs x 32
  static constexpr uint32_t ONES_COL = kTABufs * 32;    // 8 columns of bf16 ones
  static constexpr uint32_t DG_COL = 128;               // group sums: 2 x NR
  static constexpr uint32_t DX_COL = 128 + 2 * NR;      // activation sums: 2 x NR
  static_assert(XB % 1024 == 0 && C_OFF % 1024 == 0, "swizzled tiles 1024-aligned");
  static_assert(DX_COL + 2 * NR <= kTTmemCols, "TMEM budget");
  static_assert(SMEM <= 232448 && 2 * SMEM > 232448, "one CTA per SM within the budget");
};

struct TCtl {
  uint64_t full[kTStages], empty[kTStages];
  uint64_t a_full[kTABufs], a_empty[kTABufs];
  uint64_t d_full[2], d_empty[2];
  uint64_t x_full, x_empty;
  uint64_t done;
  uint32_t tmem_base;
  int32_t abort;
};

struct TParams {
  const int32_t* counts;     // expert_num_tokens [E]
  const int32_t* offsets;    // padded expert offsets [E + 1]
  const bf16* bias;          // GEMM1 [E, 2N], GEMM2 [E, N], or null
  void* out;                 // GEMM1: z bf16 [cap, N]; GEMM2: fp32 parts [S, R, N]
  const int32_t* row_index;  // GEMM2: routed item per sorted row
  const float* row_weight;   // GEMM2: weight per routed item, or null (= 1)
  int32_t* error_word;
  int64_t R;                 // GEMM2: routed items (rows of one part)
  int32_t E, N, K;           // N: GEMM1 columns per half (I), GEMM2 output columns (H)
  int32_t ncb;               // units per expert and part (GEMM1 N / 64, GEMM2 N / 128)
  int32_t splits;            // K parts (GEMM2)
  int32_t gshift;            // log2 G
  int32_t has_zero;
};

struct TUnit {
  int32_t e, off, n, cb, s, st0, nst, ngr;
};

// Waits for phase `parity` of `bar`; gives up (recording MOE_ERR_TIMEOUT and
// raising the CTA's abort flag) after the wait limit, or when another role
// has raised the flag.
__device__ __forceinline__ bool t_wait(uint64_t* bar, uint32_t parity, int32_t* abort,
                                       int32_t* err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait_suspend(bar, parity, 1000000u)) return true;
    if (*reinterpret_cast<volatile int32_t*>(abort)) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      *reinterpret_cast<volatile int32_t*>(abort) = 1;
      record_error(err, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}
// The same for a whole warp: every lane waits, the result is warp-uniform.
__device__ __forceinline__ bool t_wait_warp(uint64_t* bar, uint32_t parity, int32_t* abort,
                                            int32_t* err) {
  return __all_sync(0xFFFFFFFFu, t_wait(bar, parity, abort, err));
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

template <bool SWI, int NR>
__global__ void __launch_bounds__(kTWarps * 32, 1)
    wq_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                 const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                 const TParams P) {
  using L = TLay<NR>;
  extern __shared__ uint8_t dsmem[];
  __shared__ TCtl ctl;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  pdl_begin();
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  int32_t* list = reinterpret_cast<int32_t*>(sm + L::LIST_OFF);
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
    if (lane == 0) list[kTMaxE] = n;
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < kTStages; ++i) {
      ptx::mbar_init(&ctl.full[i], 1);   // the producer's arrival with the bytes
      ptx::mbar_init(&ctl.empty[i], 5);  // four converter warps + the MMA's commit
    }
    for (int b = 0; b < kTABufs; ++b) {
      ptx::mbar_init(&ctl.a_full[b], 4);
      ptx::mbar_init(&ctl.a_empty[b], 1);
    }
    for (int j = 0; j < 2; ++j) {
      ptx::mbar_init(&ctl.d_full[j], 1);
      ptx::mbar_init(&ctl.d_empty[j], 4);
    }
    ptx::mbar_init(&ctl.x_full, 2);   // the two up warps
    ptx::mbar_init(&ctl.x_empty, 2);  // the two gate warps
    ptx::mbar_init(&ctl.done, 1);
    ctl.abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, kTTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  int32_t* abort = &ctl.abort;

  const int64_t units = static_cast<int64_t>(list[kTMaxE]) * P.ncb * P.splits;
  const int NS = P.K / kTKR;
  const int gmask = (1 << P.gshift) - 1;
  auto unit_at = [&](int64_t u, TUnit& U) {
    U.cb = static_cast<int32_t>(u % P.ncb);
    const int64_t r = u / P.ncb;
    U.s = static_cast<int32_t>(r % P.splits);
    U.e = list[r / P.splits];
    U.off = __ldg(P.offsets + U.e);
    U.n = __ldg(P.counts + U.e);
    U.st0 = U.s * NS / P.splits;
    U.nst = (U.s + 1) * NS / P.splits - U.st0;
    U.ngr = (U.n + NR - 1) / NR;
  };
  // the two 64-column boxes of a unit: GEMM1 gate and up, GEMM2 two halves
  auto box_col = [&](const TUnit& U, int h) {
    return SWI ? h * P.N + U.cb * 64 : U.cb * 128 + h * 64;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      ptx::prefetch_tmap(&tmX);
      ptx::prefetch_tmap(&tmC);
      ptx::prefetch_tmap(&tmS);
      if (P.has_zero) ptx::prefetch_tmap(&tmZ);
      int slot = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
        TUnit U;
        unit_at(u, U);
        for (int rg = 0; rg < U.ngr && ok; ++rg) {
          for (int st = 0; st < U.nst; ++st) {
            const int k0 = (U.st0 + st) * kTKR;
            const bool gstart = st == 0 || (k0 & gmask) == 0;
            if (!t_wait(&ctl.empty[slot], ph ^ 1u, abort, P.error_word)) {
              ok = false;
              break;
            }
            uint8_t* stg = sm + slot * L::STAGE;
            uint64_t* bar = &ctl.full[slot];
            const uint32_t bytes =
                L::XB + L::CB + (gstart ? L::SB + (P.has_zero ? L::ZB : 0) : 0);
            ptx::mbar_arrive_expect_tx(bar, bytes);
            ptx::tma_load_2d(stg + L::X_OFF, &tmX, bar, k0, U.off + rg * NR);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              ptx::tma_load_3d(stg + L::C_OFF + h * (L::CB / 2), &tmC, bar, k0 / 2, box_col(U, h),
                               U.e);
            if (gstart) {
              const int gr = k0 >> P.gshift;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                ptx::tma_load_3d(stg + L::S_OFF + h * (L::SB / 2), &tmS, bar, box_col(U, h), gr,
                                 U.e);
                if (P.has_zero)
                  ptx::tma_load_3d(stg + L::Z_OFF + h * (L::ZB / 2), &tmZ, bar, box_col(U, h),
                                   gr, U.e);
              }
            }
            if (++slot == kTStages) {
              slot = 0;
              ph ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(kTCols, NR, /*a_mn=*/false, /*b_mn=*/false);
      int slot = 0, ab = 0, j = 0;
      uint32_t ph = 0, aph = 0;
      uint32_t dbits = 0;  // bit j: parity of the uses of accumulator pair j
      bool ok = true;
      for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
        TUnit U;
        unit_at(u, U);
        for (int rg = 0; rg < U.ngr && ok; ++rg) {
          for (int st = 0; st < U.nst; ++st) {
            const int k0 = (U.st0 + st) * kTKR;
            const bool gstart = st == 0 || (k0 & gmask) == 0;
            const bool gend = st == U.nst - 1 || ((k0 + kTKR) & gmask) == 0;
            if (!t_wait(&ctl.full[slot], ph, abort, P.error_word) ||
                !t_wait(&ctl.a_full[ab], aph, abort, P.error_word) ||
                (gstart && !t_wait(&ctl.d_empty[j], ((dbits >> j) & 1u) ^ 1u, abort,
                                   P.error_word))) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t xaddr = ptx::smem_u32(sm + slot * L::STAGE + L::X_OFF);
#pragma unroll
            for (int kk = 0; kk < kTKR / 16; ++kk) {
              const uint64_t bdesc = ptx::smem_desc_sw128(xaddr + 32 * kk, 16, 1024);
              const uint32_t acc = (gstart && kk == 0) ? 0u : 1u;
              ptx::mma_bf16_tmem_a(tmem + L::DG_COL + j * NR, tmem + L::A_COL + ab * 32 + 8 * kk,
                                   bdesc, idesc, acc);
              ptx::mma_bf16_tmem_a(tmem + L::DX_COL + j * NR, tmem + L::ONES_COL, bdesc, idesc,
                                   acc);
            }
            ptx::mma_commit(&ctl.a_empty[ab]);
            ptx::mma_commit(&ctl.empty[slot]);
            if (gend) {
              ptx::mma_commit(&ctl.d_full[j]);
              dbits ^= 1u << j;
              j ^= 1;
            }
            if (++ab == kTABufs) {
              ab = 0;
              aph ^= 1u;
            }
            if (++slot == kTStages) {
              slot = 0;
              ph ^= 1u;
            }
          }
        }
      }
      // every MMA complete before the accumulators are released
      ptx::mma_commit(&ctl.done);
      t_wait(&ctl.done, 0u, abort, P.error_word);
    }
  } else {
    // ------------------------------------------------ converters (warps 2-5) --
    const int q = warp & 3;          // TMEM lane quadrant
    const int cc = q * 32 + lane;    // the thread's column of the unit = its TMEM lane
    const int half = cc >> 6, jc = cc & 63;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    // A = ones for the activation sums
    ptx::tmem_st_8cols_fill(tmem + lane_base + L::ONES_COL, 0x3F803F80u);
    ptx::tmem_st_wait();
    float acc[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r] = 0.0f;
    int slot = 0, ab = 0, j = 0;
    uint32_t ph = 0;
    uint32_t abits = 0;  // bit b: parity of the uses of A buffer b
    uint32_t dbits = 0;  // bit j: parity of the uses of accumulator pair j
    uint32_t xuse = 0;
    float s_cur = 0.0f, z_cur = 0.0f, s_prev = 0.0f, z_prev = 0.0f;
    bool pending = false;
    int jp = 0;
    bool ok = true;
    // fold the finished group in accumulator pair jj into acc
    auto promote = [&](int jj, float s, float z) -> bool {
      if (!t_wait_warp(&ctl.d_full[jj], (dbits >> jj) & 1u, abort, P.error_word)) return false;
      dbits ^= 1u << jj;
      ptx::tc_fence_after();
      uint32_t g[NR], x[NR];
      if constexpr (NR == 16) {
        ptx::tmem_ld_16cols(tmem + lane_base + L::DG_COL + jj * NR, g);
        ptx::tmem_ld_16cols(tmem + lane_base + L::DX_COL + jj * NR, x);
      } else {
        ptx::tmem_ld_32cols(tmem + lane_base + L::DG_COL + jj * NR, g);
        ptx::tmem_ld_32cols(tmem + lane_base + L::DX_COL + jj * NR, x);
      }
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ctl.d_empty[jj]);
#pragma unroll
      for (int r = 0; r < NR; ++r)
        acc[r] = fmaf(s, fmaf(-z, __uint_as_float(x[r]), __uint_as_float(g[r])), acc[r]);
      return true;
    };
    for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
      TUnit U;
      unit_at(u, U);
      for (int rg = 0; rg < U.ngr && ok; ++rg) {
        for (int st = 0; st < U.nst; ++st) {
          const int k0 = (U.st0 + st) * kTKR;
          const bool gstart = st == 0 || (k0 & gmask) == 0;
          const bool gend = st == U.nst - 1 || ((k0 + kTKR) & gmask) == 0;
          if (!t_wait_warp(&ctl.full[slot], ph, abort, P.error_word)) {
            ok = false;
            break;
          }
          const uint8_t* stg = sm + slot * L::STAGE;
          if (gstart) {
            const uint16_t sb =
                *reinterpret_cast<const uint16_t*>(stg + L::S_OFF + (half * 64 + jc) * 2);
            s_cur = __uint_as_float(static_cast<uint32_t>(sb) << 16);
            const uint32_t zb = P.has_zero ? (stg[L::Z_OFF + half * 64 + jc] & 0xFu) : 8u;
            z_cur = static_cast<float>(128u + zb);
          }
          // the column's 32 code bytes; the 32-byte swizzle swaps the 16-byte
          // halves of rows 4..7 of every 8
          const uint8_t* crow = stg + L::C_OFF + half * (L::CB / 2) + jc * 32;
          const int sw = (jc >> 2) & 1;
          const uint4 c0 = *reinterpret_cast<const uint4*>(crow + ((0 ^ sw) << 4));
          const uint4 c1 = *reinterpret_cast<const uint4*>(crow + ((1 ^ sw) << 4));
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&ctl.empty[slot]);
          // word w holds K rows 8w..8w+7 with rows 8w + 2t at nibble t and
          // 8w + 2t + 1 at nibble t + 4: a mask leaves each K pair as two
          // bf16 128 + q
          const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint32_t v[32];
#pragma unroll
          for (int w = 0; w < 8; ++w) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
              v[4 * w + t] = ((wv[w] >> (4 * t)) & 0x000F000Fu) | 0x43004300u;
          }
          if (!t_wait_warp(&ctl.a_empty[ab], ((abits >> ab) & 1u) ^ 1u, abort, P.error_word)) {
            ok = false;
            break;
          }
          abits ^= 1u << ab;
          ptx::tc_fence_after();
          ptx::tmem_st_32cols(tmem + lane_base + L::A_COL + ab * 32, v);
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&ctl.a_full[ab]);
          if (++ab == kTABufs) ab = 0;
          if (++slot == kTStages) {
            slot = 0;
            ph ^= 1u;
          }
          // the previous group's sums, finished while this stage was expanded
          if (pending) {
            if (!promote(jp, s_prev, z_prev)) {
              ok = false;
              break;
            }
            pending = false;
          }
          if (gend) {
            pending = true;
            jp = j;
            s_prev = s_cur;
            z_prev = z_cur;
            j ^= 1;
          }
        }
        if (!ok) break;
        if (pending) {
          if (!promote(jp, s_prev, z_prev)) {
            ok = false;
            break;
          }
          pending = false;
        }
        // ---- epilogue of one row group ----
        const int rows_here = min(NR, U.n - rg * NR);
        if constexpr (SWI) {
          float* xch = reinterpret_cast<float*>(sm + L::XCH_OFF);
          if (half == 1) {
            // up lanes: hand their sums to the gate lanes of the same columns
            if (!t_wait_warp(&ctl.x_empty, (xuse & 1u) ^ 1u, abort, P.error_word)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) xch[jc * (NR + 1) + r] = acc[r];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ctl.x_full);
          } else {
            if (!t_wait_warp(&ctl.x_full, xuse & 1u, abort, P.error_word)) {
              ok = false;
              break;
            }
            const int zc = U.cb * 64 + jc;
            float bg = 0.0f, bu = 0.0f;
            if (P.bias != nullptr) {
              bg = __bfloat162float(P.bias[static_cast<int64_t>(U.e) * 2 * P.N + zc]);
              bu = __bfloat162float(P.bias[static_cast<int64_t>(U.e) * 2 * P.N + P.N + zc]);
            }
            bf16* z = static_cast<bf16*>(P.out);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
              if (r < rows_here) {
                const float up = xch[jc * (NR + 1) + r];
                const float zv = silu_f(acc[r] + bg) * (up + bu);
                z[static_cast<int64_t>(U.off + rg * NR + r) * P.N + zc] = __float2bfloat16_rn(zv);
              }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ctl.x_empty);
          }
          ++xuse;
        } else {
          const int oc = U.cb * 128 + cc;
          const float b = (P.bias != nullptr && U.s == 0)
                              ? __bfloat162float(P.bias[static_cast<int64_t>(U.e) * P.N + oc])
                              : 0.0f;
          float* o = static_cast<float*>(P.out);
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            if (r < rows_here) {
              const int32_t item = __ldg(P.row_index + U.off + rg * NR + r);
              const float w = P.row_weight != nullptr ? __ldg(P.row_weight + item) : 1.0f;
              o[(static_cast<int64_t>(U.s) * P.R + item) * P.N + oc] = (acc[r] + b) * w;
            }
          }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[r] = 0.0f;
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTTmemCols);
  }
}

// Codes [E, K, N/2] (column 2j in the low nibble of byte j) -> [E, N, K/2]:
// word w of column n holds K rows 8w..8w+7, row 8w + 2t at nibble t and
// row 8w + 2t + 1 at nibble t + 4.  One thread per output word.
__global__ void __launch_bounds__(256)
    pack_k_int4_kernel(const uint8_t* __restrict__ codes, int32_t E, int32_t K, int32_t N,
                       uint32_t* __restrict__ out) {
  pdl_begin();
  const int64_t words = static_cast<int64_t>(E) * N * (K / 8);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    // i = ((e * (K / 8)) + w) * N + n: neighbouring threads read neighbouring codes
    const int n = static_cast<int>(i % N);
    const int64_t r = i / N;
    const int w = static_cast<int>(r % (K / 8));
    const int e = static_cast<int>(r / (K / 8));
    const uint8_t* src = codes + (static_cast<int64_t>(e) * K + 8 * w) * (N / 2) + n / 2;
    const int shift = (n & 1) * 4;
    uint32_t v = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t c = (__ldg(src + static_cast<int64_t>(t) * (N / 2)) >> shift) & 0xFu;
      const int pos = (t & 1) ? 4 + (t >> 1) : (t >> 1);
      v |= c << (4 * pos);
    }
    out[(static_cast<int64_t>(e) * N + n) * (K / 8) + w] = v;
  }
}

int device_sms_tc() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  cudaGetLastError();
  return sms;
}

template <bool SWI, int NR>
moe_status_t launch_tc(const GroupedGemmArgs& a, const void* kpack, const int32_t* counts,
                       int32_t splits, int64_t R, const char* name, cudaStream_t s) {
  using L = TLay<NR>;
  auto kernel = wq_tc_kernel<SWI, NR>;
  static PerDevice attrs;
  if (attrs.get([&](int*) {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
      }) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute(%s): %s", name,
                     cudaGetErrorString(cudaGetLastError()));
  const uint64_t E = static_cast<uint64_t>(a.E), K = static_cast<uint64_t>(a.K),
                 N = static_cast<uint64_t>(a.N), cap = static_cast<uint64_t>(a.cap);
  const uint64_t ncols = SWI ? 2 * N : N;  // weight columns of the matrix
  const uint64_t KG = K / static_cast<uint64_t>(a.wq_group);
  CUtensorMap tmX, tmC, tmS, tmZ;
  {
    const uint64_t dims[2] = {K, cap};
    const uint64_t strides[1] = {K * 2};
    const uint32_t box[2] = {static_cast<uint32_t>(kTKR), static_cast<uint32_t>(NR)};
    if (moe_status_t st = encode_tensor_map(&tmX, a.a, 2, dims, strides, box,
                                            CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                            CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
  }
  {
    // K-packed codes [E, ncols, K/2]
    const uint64_t dims[3] = {K / 2, ncols, E};
    const uint64_t strides[2] = {K / 2, ncols * (K / 2)};
    const uint32_t box[3] = {static_cast<uint32_t>(kTKR / 2), 64, 1};
    if (moe_status_t st = encode_tensor_map(&tmC, kpack, 3, dims, strides, box,
                                            CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                            CU_TENSOR_MAP_SWIZZLE_32B))
      return st;
  }
  {
    const uint64_t dims[3] = {ncols, KG, E};
    const uint64_t strides[2] = {ncols * 2, ncols * 2 * KG};
    const uint32_t box[3] = {64, 1, 1};
    if (moe_status_t st = encode_tensor_map(&tmS, a.wq_scale, 3, dims, strides, box,
                                            CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                            CU_TENSOR_MAP_SWIZZLE_NONE))
      return st;
    tmZ = tmS;
    if (a.wq_zero != nullptr) {
      const uint64_t zstrides[2] = {ncols, ncols * KG};
      if (moe_status_t st = encode_tensor_map(&tmZ, a.wq_zero, 3, dims, zstrides, box,
                                              CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                              CU_TENSOR_MAP_SWIZZLE_NONE))
        return st;
    }
  }
  TParams P{};
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
  P.ncb = SWI ? a.N / 64 : a.N / 128;
  P.splits = SWI ? 1 : splits;
  P.gshift = 31 - __builtin_clz(static_cast<unsigned>(a.wq_group));
  P.has_zero = a.wq_zero != nullptr ? 1 : 0;
  prof_before(name, s);
  launch_kernel(kernel, static_cast<unsigned>(a.num_sms), kTWarps * 32, L::SMEM, s, tmX, tmC,
                tmS, tmZ, P);
  prof_after(name, s);
  return check_launch(name);
}

template <bool SWI>
moe_status_t launch_tc_rows(const GroupedGemmArgs& a, const void* kpack, const int32_t* counts,
                            int64_t M, int32_t splits, int64_t R, const char* name,
                            cudaStream_t s) {
  if (M <= 16) return launch_tc<SWI, 16>(a, kpack, counts, splits, R, name, s);
  return launch_tc<SWI, 32>(a, kpack, counts, splits, R, name, s);
}

}  // namespace

bool wq_tc_applies(int64_t M, int32_t H, int32_t I, int32_t E, int32_t format, int32_t group) {
  if (M < 1 || M > 32 || E > kTMaxE || format != MOE_WQ_INT4) return false;
  if (H % 128 != 0 || I % 64 != 0) return false;
  return group >= 64 && (group & (group - 1)) == 0;
}

// K parts of GEMM2: the count that spreads (touched experts x column blocks
// x parts) units most evenly over the CTAs, the fewest among equals; the
// parts' rows must fit the fp32 row region (cap rows).
int wq_tc_splits(int64_t M, int32_t top_k, int32_t H, int32_t I, int32_t E, int64_t cap,
                 int32_t num_sms) {
  const int64_t R = M * top_k;
  const int64_t touched = std::min<int64_t>(E, R);
  const int64_t ncb = H / 128;
  const int NS = I / kTKR;
  int best = 1;
  double best_cost = 1e30;
  for (int S = 1; S <= 16 && S <= NS && S * R <= cap; ++S) {
    const int64_t U = touched * ncb * S;
    const double cost = static_cast<double>((U + num_sms - 1) / num_sms) / S;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

moe_status_t launch_wq_tc_gemm1(const GroupedGemmArgs& a, const void* kpack,
                                const int32_t* counts, int64_t M, cudaStream_t s) {
  return launch_tc_rows<true>(a, kpack, counts, M, 1, 0, "gemm1_swiglu_int4_tc", s);
}

moe_status_t launch_wq_tc_gemm2(const GroupedGemmArgs& a, const void* kpack,
                                const int32_t* counts, int64_t M, int32_t splits, int64_t R,
                                cudaStream_t s) {
  return launch_tc_rows<false>(a, kpack, counts, M, splits, R, "gemm2_int4_tc", s);
}

moe_status_t launch_pack_k_int4(const void* codes, int32_t E, int32_t K, int32_t N, void* out,
                                cudaStream_t s) {
  const int64_t words = static_cast<int64_t>(E) * N * (K / 8);
  if (words <= 0) return MOE_OK;
  const unsigned grid = static_cast<unsigned>(
      std::min<int64_t>((words + 255) / 256, static_cast<int64_t>(device_sms_tc()) * 16));
  launch_kernel(pack_k_int4_kernel, grid, 256, 0, s, static_cast<const uint8_t*>(codes), E, K, N,
                static_cast<uint32_t*>(out));
  return check_launch("pack_k_int4");
}

}  // namespace gbmoe
