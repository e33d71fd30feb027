// Weight-only int4 decode GEMMs on the tcgen05 tensor cores, the weights as
// the MMA's A operand in tensor memory.
//
// "fused_moe.py 分析", "WNA16 路径": int4 expert weights with a scale and a
// zero point per group of G rows along K, bf16 activations, fp32
// accumulation.  For a group g of weight column n,
//   sum_{k in g} x_k (q_kn - zp_gn) s_gn = s_gn * sum_{k in g} x_k (q_kn - zp_gn),
// the group's exact contribution, with q - zp (an integer of at most 15 in
// magnitude) exact as a bf16 operand.  For calls of at most 32 tokens, with
// the codes repacked once along K (moe_wq_pack_k):
//   - a unit is 128 weight columns of one touched expert (GEMM1: 64 gate and
//     the same 64 up columns; GEMM2: 128 output columns over one of S parts
//     of K), one CTA per SM walking its units;
//   - one thread streams 128-row K stages by TMA into a ring: the expert
//     rows' activations (NR rows, two 64-column boxes, 128-byte swizzle), the
//     128 columns' codes (64 bytes of K-packed codes each, 64-byte swizzle)
//     and their zero points;
//   - two groups of four converter warps, taking the stages in turn, one
//     thread per weight column = TMEM lane, turn
//     the codes of their column into the bf16 values q - zp (a mask per K
//     pair gives 128 + q, one bf16 subtraction of 128 + zp, both exact) and
//     store them with tcgen05.st as the stage's A operand (128 lanes x 64
//     columns of bf16 pairs); an A buffer is stored again once the stage
//     that last used it has been released by the MMA;
//   - one thread issues tcgen05.mma (M = 128 columns, N = NR rows, K = 16)
//     with A in tensor memory and the activations in shared memory into the
//     group's accumulator; groups rotate over eight accumulators;
//   - four promoter warps, again one thread per column, read the
//     accumulator of their lane after each group and add s * acc into
//     registers, the group's scale loaded from global memory while the
//     group runs; at the end
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

constexpr int kTKR = 128;       // K rows per stage
constexpr int kTCols = 128;     // weight columns per unit = TMEM lanes = MMA M
constexpr int kTMaxStages = 12; // shared-memory ring, at most
constexpr int kTABufs = 4;      // A operand buffers in TMEM, 64 columns each
constexpr int kTDBufs = 8;      // group accumulators in TMEM
constexpr int kTWarps = 14;     // producer, MMA, eight converter and four promoter warps
constexpr int kTMaxE = 1024;    // experts the touched list holds
constexpr uint32_t kTTmemCols = 512;

template <int NR>
struct TLay {
  static constexpr int XB = NR * 128;              // activations: NR rows x 64 bf16, per box
  static constexpr int CB = kTCols * (kTKR / 2);   // codes: 128 columns x 64 bytes
  static constexpr int ZBOX = 128;                 // zero points of a 64-column box, 128-aligned
  static constexpr int X_OFF = 0;
  static constexpr int C_OFF = 2 * XB;
  static constexpr int Z_OFF = C_OFF + CB;
  static constexpr int STAGE = (Z_OFF + 2 * ZBOX + 1023) / 1024 * 1024;
  // ring depth: deep enough for the loads in flight, and the shared memory
  // then keeps one CTA per SM
  static constexpr int NSTG = NR <= 16 ? 10 : 8;
  static constexpr int XCH_OFF = NSTG * STAGE;                  // gate/up exchange
  static constexpr int LIST_OFF = XCH_OFF + 64 * (NR + 1) * 4;  // touched experts
  static constexpr int SMEM = 1024 + LIST_OFF + (kTMaxE + 1) * 4;
  // TMEM columns
  static constexpr uint32_t A_COL = 0;                  // kTABufs x 64
  static constexpr uint32_t D_COL = 256;                // accumulator j at + j NR
  static_assert(XB % 1024 == 0 && C_OFF % 1024 == 0 && (CB / 2) % 1024 == 0,
                "swizzled tiles 1024-aligned");
  static_assert(Z_OFF % 128 == 0, "TMA destinations 128-aligned");
  static_assert(A_COL + kTABufs * 64 <= D_COL && D_COL + kTDBufs * NR <= kTTmemCols,
                "TMEM budget");
  static_assert(NSTG <= kTMaxStages, "ring within the barrier arrays");
  static_assert(SMEM <= 232448 && 2 * SMEM > 232448, "one CTA per SM within the budget");
};

struct TCtl {
  uint64_t full[kTMaxStages], empty[kTMaxStages];
  uint64_t a_full[kTABufs];
  uint64_t d_full[kTDBufs], d_empty[kTDBufs];
  uint64_t x_full, x_empty;
  uint64_t done;
  uint32_t tmem_base;
  int32_t abort;
};

struct TParams {
  const int32_t* counts;     // expert_num_tokens [E]
  const int32_t* offsets;    // padded expert offsets [E + 1]
  const bf16* bias;          // GEMM1 [E, 2N], GEMM2 [E, N], or null
  const bf16* scale;         // group scales [E, K/G, ncols]
  const uint8_t* zero;       // zero points [E, K/G, ncols], or null (8)
  void* out;                 // GEMM1: z bf16 [cap, N]; GEMM2: fp32 parts [S, R, N]
  const int32_t* row_index;  // GEMM2: routed item per sorted row
  const float* row_weight;   // GEMM2: weight per routed item, or null (= 1)
  int32_t* error_word;
  int64_t R;                 // GEMM2: routed items (rows of one part)
  int32_t E, N, K;           // N: GEMM1 columns per half (I), GEMM2 output columns (H)
  int32_t ncols;             // weight columns of the matrix (GEMM1 2N, GEMM2 N)
  int32_t ncb;               // units per expert and part (GEMM1 N / 64, GEMM2 N / 128)
  int32_t splits;            // K parts (GEMM2)
  int32_t gshift;            // log2 G
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

// Walks a CTA's stages in order: its units (blockIdx.x, + gridDim.x, ...),
// each unit's row groups, each row group's K stages.  Every role walks the
// same sequence.
struct TCursor {
  int64_t u;
  TUnit U;
  int rg, st;
  bool valid;
};

template <bool SWI, int NR>
__global__ void __launch_bounds__(kTWarps * 32, 1)
    wq_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                 const __grid_constant__ CUtensorMap tmZ, const TParams P) {
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
    for (int i = 0; i < L::NSTG; ++i) {
      ptx::mbar_init(&ctl.full[i], 1);   // the producer's arrival with the bytes
      ptx::mbar_init(&ctl.empty[i], 5);  // four converter warps + the MMA's commit
    }
    for (int b = 0; b < kTABufs; ++b) ptx::mbar_init(&ctl.a_full[b], 4);
    for (int j = 0; j < kTDBufs; ++j) {
      ptx::mbar_init(&ctl.d_full[j], 1);
      ptx::mbar_init(&ctl.d_empty[j], 4);
    }
    ptx::mbar_init(&ctl.x_full, 2);   // the two up promoter warps
    ptx::mbar_init(&ctl.x_empty, 2);  // the two gate promoter warps
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
  auto cursor_begin = [&](TCursor& c) {
    c.u = blockIdx.x;
    c.rg = 0;
    c.st = 0;
    c.valid = c.u < units;
    if (c.valid) unit_at(c.u, c.U);
  };
  auto cursor_next = [&](TCursor& c) {
    if (++c.st == c.U.nst) {
      c.st = 0;
      if (++c.rg == c.U.ngr) {
        c.rg = 0;
        c.u += gridDim.x;
        c.valid = c.u < units;
        if (c.valid) unit_at(c.u, c.U);
      }
    }
  };
  auto k0_of = [&](const TCursor& c) { return (c.U.st0 + c.st) * kTKR; };
  auto gstart_of = [&](const TCursor& c) { return c.st == 0 || (k0_of(c) & gmask) == 0; };
  auto gend_of = [&](const TCursor& c) {
    return c.st == c.U.nst - 1 || ((k0_of(c) + kTKR) & gmask) == 0;
  };
  // the unit's two 64-column boxes: GEMM1 gate and up, GEMM2 two halves
  auto box_col = [&](const TUnit& U, int h) {
    return SWI ? h * P.N + U.cb * 64 : U.cb * 128 + h * 64;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      ptx::prefetch_tmap(&tmX);
      ptx::prefetch_tmap(&tmC);
      if (P.zero != nullptr) ptx::prefetch_tmap(&tmZ);
      int slot = 0;
      uint32_t ph = 0;
      TCursor c;
      for (cursor_begin(c); c.valid; cursor_next(c)) {
        if (!t_wait(&ctl.empty[slot], ph ^ 1u, abort, P.error_word)) break;
        uint8_t* stg = sm + slot * L::STAGE;
        uint64_t* bar = &ctl.full[slot];
        const int k0 = k0_of(c);
        const bool zp = P.zero != nullptr;
        ptx::mbar_arrive_expect_tx(bar, 2 * L::XB + L::CB + (zp ? 2 * 64 : 0));
        ptx::tma_load_2d(stg + L::X_OFF, &tmX, bar, k0, c.U.off + c.rg * NR);
        ptx::tma_load_2d(stg + L::X_OFF + L::XB, &tmX, bar, k0 + 64, c.U.off + c.rg * NR);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          ptx::tma_load_3d(stg + L::C_OFF + h * (L::CB / 2), &tmC, bar, k0 / 2, box_col(c.U, h),
                           c.U.e);
          if (zp)
            ptx::tma_load_3d(stg + L::Z_OFF + h * L::ZBOX, &tmZ, bar, box_col(c.U, h),
                             k0 >> P.gshift, c.U.e);
        }
        if (++slot == L::NSTG) {
          slot = 0;
          ph ^= 1u;
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
      TCursor c;
      for (cursor_begin(c); c.valid; cursor_next(c)) {
        const bool gstart = gstart_of(c), gend = gend_of(c);
        // the converters signal a_full after the stage's copies landed and its
        // A was stored
        if (!t_wait(&ctl.a_full[ab], aph, abort, P.error_word) ||
            (gstart &&
             !t_wait(&ctl.d_empty[j], ((dbits >> j) & 1u) ^ 1u, abort, P.error_word)))
          break;
        ptx::tc_fence_after();
        const uint32_t xaddr = ptx::smem_u32(sm + slot * L::STAGE + L::X_OFF);
        const uint32_t dg = tmem + L::D_COL + j * NR;
#pragma unroll
        for (int kk = 0; kk < kTKR / 16; ++kk) {
          const uint64_t bdesc =
              ptx::smem_desc_sw128(xaddr + (kk >> 2) * L::XB + 32 * (kk & 3), 16, 1024);
          const uint32_t acc = (gstart && kk == 0) ? 0u : 1u;
          ptx::mma_bf16_tmem_a(dg, tmem + L::A_COL + ab * 64 + 8 * kk, bdesc, idesc, acc);
        }
        // the stage's activations, and its A buffer, free once these MMAs are
        ptx::mma_commit(&ctl.empty[slot]);
        if (gend) {
          ptx::mma_commit(&ctl.d_full[j]);
          dbits ^= 1u << j;
          if (++j == kTDBufs) j = 0;
        }
        if (++ab == kTABufs) {
          ab = 0;
          aph ^= 1u;
        }
        if (++slot == L::NSTG) {
          slot = 0;
          ph ^= 1u;
        }
      }
      // every MMA complete before the tensor memory is released
      ptx::mma_commit(&ctl.done);
      t_wait(&ctl.done, 0u, abort, P.error_word);
    }
  } else if (warp < 10) {
    // --------------------------------------------- converters (warps 2-9) --
    // warps 2-5 take the even stages, warps 6-9 the odd ones
    const int cw = (warp - 2) >> 2;
    const int q = warp & 3;          // TMEM lane quadrant
    const int cc = q * 32 + lane;    // the thread's column of the unit = its TMEM lane
    const int half = cc >> 6, jc = cc & 63;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int64_t t = 0;  // the CTA's stage index
    uint32_t v[64];
    TCursor c;
    for (cursor_begin(c); c.valid; cursor_next(c), ++t) {
      if ((t & 1) != cw) continue;
      const int slot = static_cast<int>(t % L::NSTG);
      const uint32_t ph = static_cast<uint32_t>((t / L::NSTG) & 1);
      const int ab = static_cast<int>(t % kTABufs);
      if (!t_wait_warp(&ctl.full[slot], ph, abort, P.error_word)) break;
      const uint8_t* stg = sm + slot * L::STAGE;
      uint32_t zz = 0x43084308u;  // bf16 pair 128 + zp (8 without zero points)
      if (P.zero != nullptr) {
        const uint32_t z = 0x4300u | (stg[L::Z_OFF + half * L::ZBOX + jc] & 0xFu);
        zz = z | (z << 16);
      }
      // the column's 64 code bytes; the 64-byte swizzle permutes the 16-byte
      // quarters of each row by bits 1..2 of its index
      const uint8_t* crow = stg + L::C_OFF + half * (L::CB / 2) + jc * 64;
      const int sw = (jc >> 1) & 3;
      uint4 cq[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) cq[h] = *reinterpret_cast<const uint4*>(crow + ((h ^ sw) << 4));
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ctl.empty[slot]);
      // word w holds K rows 8w..8w+7, row 8w + 2t at nibble t and 8w + 2t + 1
      // at nibble t + 4: a mask leaves each K pair as two bf16 128 + q, and
      // subtracting 128 + zp leaves q - zp (exact)
      const __nv_bfloat162 zb = *reinterpret_cast<const __nv_bfloat162*>(&zz);
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        const uint4& q4 = cq[w >> 2];
        const uint32_t word = (w & 3) == 0 ? q4.x : (w & 3) == 1 ? q4.y : (w & 3) == 2 ? q4.z : q4.w;
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          const uint32_t m = ((word >> (4 * tt)) & 0x000F000Fu) | 0x43004300u;
          const __nv_bfloat162 d = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&m), zb);
          v[4 * w + tt] = *reinterpret_cast<const uint32_t*>(&d);
        }
      }
      // the A buffer is free once stage t - kTABufs, its last user, has been
      // released by its MMAs
      if (t >= kTABufs) {
        const int64_t tb = t - kTABufs;
        if (!t_wait_warp(&ctl.empty[tb % L::NSTG], static_cast<uint32_t>((tb / L::NSTG) & 1), abort,
                         P.error_word))
          break;
      }
      ptx::tc_fence_after();
      const uint32_t ta = tmem + lane_base + L::A_COL + ab * 64;
      ptx::tmem_st_32cols(ta, reinterpret_cast<const uint32_t(&)[32]>(v[0]));
      ptx::tmem_st_32cols(ta + 32, reinterpret_cast<const uint32_t(&)[32]>(v[32]));
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ctl.a_full[ab]);
    }
  } else {
    // ----------------------------------------------- promoters (warps 10-13) --
    const int q = warp & 3;
    const int cc = q * 32 + lane;
    const int half = cc >> 6, jc = cc & 63;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int64_t KG = static_cast<int64_t>(P.K) >> P.gshift;
    float acc[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r] = 0.0f;
    int j = 0;
    uint32_t dbits = 0;
    uint32_t xuse = 0;
    bool ok = true;
    uint16_t s_raw = 0;
    TCursor c;
    for (cursor_begin(c); c.valid && ok; cursor_next(c)) {
      if (gstart_of(c)) {
        // the group's scale of this column, in flight while the group's
        // stages run
        const int64_t pi = (static_cast<int64_t>(c.U.e) * KG + (k0_of(c) >> P.gshift)) * P.ncols +
                           box_col(c.U, half) + jc;
        s_raw = __ldg(reinterpret_cast<const uint16_t*>(P.scale) + pi);
      }
      if (gend_of(c)) {
        if (!t_wait_warp(&ctl.d_full[j], (dbits >> j) & 1u, abort, P.error_word)) {
          ok = false;
          break;
        }
        dbits ^= 1u << j;
        ptx::tc_fence_after();
        uint32_t g[NR];
        const uint32_t da = tmem + lane_base + L::D_COL + j * NR;
        if constexpr (NR == 16)
          ptx::tmem_ld_16cols(da, g);
        else
          ptx::tmem_ld_32cols(da, g);
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ctl.d_empty[j]);
        if (++j == kTDBufs) j = 0;
        const float s = __uint_as_float(static_cast<uint32_t>(s_raw) << 16);
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[r] = fmaf(s, __uint_as_float(g[r]), acc[r]);
      }
      if (c.st != c.U.nst - 1) continue;
      // ---- epilogue of one row group ----
      const TUnit& U = c.U;
      const int rg = c.rg;
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
  CUtensorMap tmX, tmC, tmZ;
  {
    const uint64_t dims[2] = {K, cap};
    const uint64_t strides[1] = {K * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(NR)};
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
                                            CU_TENSOR_MAP_SWIZZLE_64B))
      return st;
  }
  tmZ = tmC;
  if (a.wq_zero != nullptr) {
    // zero points [E, K/G, ncols], one 64-column box per unit half
    const uint64_t KG = K / static_cast<uint64_t>(a.wq_group);
    const uint64_t dims[3] = {ncols, KG, E};
    const uint64_t strides[2] = {ncols, ncols * KG};
    const uint32_t box[3] = {64, 1, 1};
    if (moe_status_t st = encode_tensor_map(&tmZ, a.wq_zero, 3, dims, strides, box,
                                            CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                            CU_TENSOR_MAP_SWIZZLE_NONE))
      return st;
  }
  TParams P{};
  P.counts = counts;
  P.offsets = a.offsets;
  P.bias = a.bias;
  P.scale = static_cast<const bf16*>(a.wq_scale);
  P.zero = static_cast<const uint8_t*>(a.wq_zero);
  P.out = a.out;
  P.row_index = a.row_index;
  P.row_weight = a.row_weight;
  P.error_word = a.error_word;
  P.R = R;
  P.E = a.E;
  P.N = a.N;
  P.K = a.K;
  P.ncols = static_cast<int32_t>(ncols);
  P.ncb = SWI ? a.N / 64 : a.N / 128;
  P.splits = SWI ? 1 : splits;
  P.gshift = 31 - __builtin_clz(static_cast<unsigned>(a.wq_group));
  prof_before(name, s);
  launch_kernel(kernel, static_cast<unsigned>(a.num_sms), kTWarps * 32, L::SMEM, s, tmX, tmC, tmZ,
                P);
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
  if (H % 128 != 0 || I % 128 != 0) return false;
  return group >= 128 && (group & (group - 1)) == 0;
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
