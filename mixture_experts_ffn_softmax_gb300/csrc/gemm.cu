// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA through a 4-stage mbarrier pipeline.
//
// "FlagGems fused_moe.py analysis", section 1.3 / fused_moe_kernel: over the
// expert-sorted, block-padded items, C[r, n] = sum_k A[t(r), k] B[e(r), n, k];
// one program handles one block of rows of one expert and one block of output
// columns; the expert of a row block comes from the align output.  Weights
// are stored as on the "MindIE-SD Fused MoE" page: w13 [E, H, 2I] and
// w2 [E, I, H], i.e. N-contiguous, so B is fed to the MMA as an MN-major
// operand straight from its storage layout.
//
// Kernel shape (persistent, one CTA per SM, 320 threads):
//   warp 0  lane 0 : TMA producer (A tile 128x64, B tile 64x256 per stage)
//   warp 1         : TMEM allocator; lane 0 issues tcgen05.mma (M=128, N=256,
//                    K=16) and commits stage / accumulator barriers
//   warps 2..9     : epilogue, two warps per TMEM lane quadrant (tcgen05.ld),
//                    each owning half of the tile's columns
// The 512 TMEM columns hold two 128x256 fp32 accumulators so the epilogue of
// tile i overlaps the MMAs of tile i+1.
//
// Weight-only quantised B (608 threads): warp 0 lane 0 streams the raw codes,
// scales and zero points into a raw ring; warps 2..9 convert them to bf16 in
// the B tile's layout; warp 10 lane 0 loads A; warps 11..18 are the epilogue.
// On CTA pairs the odd CTA's warp 1 lane 0 relays its converted stages to
// the even CTA's barrier.
//
// Tiles are enumerated expert by expert, column block by column block, with
// the row blocks of one expert innermost, so CTAs running at the same time
// share the same weight columns in L2.  The tile count is read on the device
// from the padded expert offsets: no host synchronisation.
//
// Epilogues:
//   SwiGLU     : GEMM1.  Columns [0,128) of the accumulator are the gate
//                block, [128,256) the matching up block; writes
//                z = SiLU(gate + b_gate) * (up + b_up) as bf16.
//   SortedF32  : GEMM2, contiguous layout, separate reduce.  o = (acc + b2) *
//                w(item) as fp32 rows in sorted order, staged through shared
//                memory and written with TMA tensor stores (coalesced, async).
//   SortedF16  : as SortedF32, the rows stored as fp16 values times 2^-e with
//                e >= 0 per row and 32-column chunk, the least that keeps the
//                chunk finite (exponents in o_exp [chunk][row]): half the
//                bytes, 11 significant bits, no overflow.
//   AtomicF32  : GEMM2, contiguous layout, reduce in the epilogue.  The same
//                weighted row is added into the token's fp32 accumulator row
//                with 16-byte vector atomics (the k-sum happens in L2).
//   RowsBF16   : GEMM2, batched layout.  Written as bf16 into the output row
//                row_index[p] = e * T + i of valid rows only.
//   DenseF32   : the router logits s = x W_g + b_g: one "expert", rows in
//                token order, fp32 output [M, E].
// Every mbarrier wait is bounded; on timeout the CTA records MOE_ERR_TIMEOUT,
// all roles stop, in-flight copies are given time to land, TMEM is freed.
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "fp8q.cuh"
#include "ptx.cuh"
#include "wq.cuh"

namespace gbmoe {
namespace {

constexpr int BM = MOE_BLOCK_M;  // 128 rows per tile (MMA M)
constexpr int MMA_N = 256;       // accumulator columns per tile
constexpr int EPI_WARPS = 8;                // two per TMEM lane quadrant
constexpr int NTHREADS = 64 + EPI_WARPS * 32;  // producer + MMA + epilogue
constexpr int A_STAGE_BYTES = BM * 128;        // 16 KB: 128 rows x one 128-byte swizzle row
constexpr int TMEM_COLS = 2 * MMA_N;           // 512: two accumulators
constexpr int MAX_E = 1024;
constexpr int STAGING_BYTES = 32 * 128;        // per epilogue warp: 32 rows x 128 bytes
constexpr int kMaxRaw = 8;
constexpr uint32_t kRelayBytes = 16;  // CTA-pair stage signal (bulk copy size)
// Slots of the dynamic tile ring: more than the producer can run ahead of the
// slowest reader (at most NSTAGES tiles ahead of the MMA, which is at most
// two tiles ahead of the epilogue).
constexpr int kTileSlots = 16;  // raw ring stages the control block has barriers for

// CG = CTAs cooperating on one MMA tile.  CG = 1: a 128 x 256 tile per CTA,
// 48 KB per pipeline stage.  CG = 2 (a CTA pair, tcgen05 cta_group::2): a
// 256 x 256 tile per pair, each CTA staging its 128 rows of A and its 128
// columns of B -- 32 KB per stage per CTA, a third less shared-memory fill
// per MMA than CG = 1.
// F8 = E4M3 operands (kind::f8f6f4, K = 32 per MMA) instead of bf16
// (kind::f16, K = 16).  Either way a stage holds one 128-byte swizzle row of
// K per A row: 64 bf16 or 128 E4M3; B is staged in chunks of one 128-byte
// row of N (64 or 128 columns) by those K rows.
// Raw ring of the weight-only quantised B operand (no swizzle), staged by
// TMA for the converter warps.  A stage holds, for 64 K rows of the tile's
// 256 columns, the codes, up to two rows of group scales and of zero
// points, in NREG regions of contiguous columns: two (gate, up) for the
// SwiGLU GEMM, one for the other -- so that each TMA box row is as wide as
// the region (fewer, longer rows per stage).
template <Wq WQ, int NREG = 2, int RCOLS_ = 256 / NREG>
struct WqRing {
  using F = WqFmt<WQ>;
  static constexpr int RCOLS = RCOLS_;                      // columns of a region
  static constexpr int ROW_BYTES = RCOLS * F::CODE_BITS / 8; // codes of one K row of a region
  static constexpr int CODES = 64 * ROW_BYTES;               // a region's codes, 64 K rows
  static constexpr int SCALES = 2 * RCOLS * F::SCALE_BYTES;  // a region's scales, two group rows
  static constexpr int ZEROS = F::HAS_ZERO ? 2 * RCOLS : 0;  // a region's zero points
  static constexpr int SC_OFF = NREG * CODES;                // scales of region g at SC_OFF + g*SCALES
  static constexpr int Z_OFF = SC_OFF + NREG * SCALES;       // zeros of region g at Z_OFF + g*ZEROS
  static constexpr int STAGE = Z_OFF + NREG * ZEROS;
  // as many raw stages as fit beside the main ring (int8 / FP6 codes are
  // twice the bytes of int4 / FP4)
  static constexpr int NRAW = NREG * RCOLS == 256 ? (F::CODE_BITS == 8 ? 2 : 5)
                                                  : (F::CODE_BITS == 8 ? 4 : 8);
  static constexpr int BYTES = WQ == Wq::None ? 0 : NRAW * STAGE;
  static_assert(CODES % 128 == 0 && SCALES % 128 == 0 && ZEROS % 128 == 0,
                "raw regions keep 128-byte alignment");
  static_assert(NRAW <= kMaxRaw, "raw ring deeper than its barriers");
};

template <int CG, bool F8 = false, Wq WQ = Wq::None>
struct Geo {
  static constexpr int BKE = F8 ? 128 : 64;       // K elements per stage
  static constexpr int CW = F8 ? 128 : 64;        // B columns per chunk
  static constexpr int CHUNKS = MMA_N / CW;       // B chunks per tile
  static constexpr int CHUNK_BYTES = BKE * 128;   // one chunk: BKE k-rows x 128 bytes
  static constexpr int B_CHUNKS_CTA = CHUNKS / CG;
  // row sub-tiles per tile: quantised B on CTA pairs feeds each converted B
  // stage to two MMAs (rows +0 and +256 of a 512-row tile), one per
  // accumulator, halving the conversion per MMA
  static constexpr int SUB = (WQ != Wq::None && CG == 2) ? 2 : 1;
  static constexpr int B_OFF = SUB * A_STAGE_BYTES;  // B after the stage's A tiles
  static constexpr int STAGE = B_OFF + B_CHUNKS_CTA * CHUNK_BYTES;
  static constexpr int UMMA_K = F8 ? 32 : 16;     // K per tcgen05.mma
  static constexpr int KSTEPS = BKE / UMMA_K;
  static constexpr int B_KSTEP = UMMA_K * 128;    // bytes per MMA K step within a chunk
  static constexpr int NSTAGES = WQ != Wq::None ? 3 : (CG == 1 ? 4 : 5);
  // the pair tile prefix, rounded up so that what follows stays 1024-aligned
  static constexpr size_t PREFIX_BYTES = CG == 1 ? 0 : ((MAX_E + 1) * sizeof(int32_t) + 1023) / 1024 * 1024;
  // raw ring: a CTA of a pair converts one 128-column region per stage
  using Raw = std::conditional_t<CG == 1, WqRing<WQ, 2, 128>, WqRing<WQ, 1, 128>>;
  static constexpr size_t SMEM = 1024 /*alignment slack*/ + NSTAGES * STAGE +
                                 EPI_WARPS * STAGING_BYTES + PREFIX_BYTES + Raw::BYTES;
  static constexpr uint32_t IDESC =
      F8 ? ptx::idesc_e4m3_f32(BM * CG, MMA_N, /*a_mn=*/false, /*b_mn=*/true)
         : ptx::idesc_bf16_f32(BM * CG, MMA_N, /*a_mn=*/false, /*b_mn=*/true);
};
static_assert(Geo<1>::SMEM <= 232448 && Geo<2>::SMEM <= 232448, "shared memory budget");
static_assert(Geo<1, true>::SMEM <= 232448 && Geo<2, true>::SMEM <= 232448,
              "shared memory budget");
static_assert(Geo<1, false, Wq::Int4>::SMEM <= 232448 && Geo<1, false, Wq::Int8>::SMEM <= 232448 &&
                  Geo<1, false, Wq::Mxfp4>::SMEM <= 232448 &&
                  Geo<1, false, Wq::Mxfp6e3m2>::SMEM <= 232448 &&
                  Geo<2, false, Wq::Int4>::SMEM <= 232448 && Geo<2, false, Wq::Int8>::SMEM <= 232448 &&
                  Geo<2, false, Wq::Mxfp4>::SMEM <= 232448 &&
                  Geo<2, false, Wq::Mxfp6e3m2>::SMEM <= 232448,
              "shared memory budget");

// Threads of a CTA: producer + MMA warps, converter warps (weight-only
// quantised B), epilogue warps.
template <Wq WQ>
__host__ __device__ constexpr int conv_warps() { return WQ == Wq::None ? 0 : 8; }
template <Wq WQ>
__host__ __device__ constexpr int cta_threads() {
  return 64 + 32 * conv_warps<WQ>() + (WQ == Wq::None ? 0 : 32) + EPI_WARPS * 32;
}

enum class Epi { SwiGLU = 0, SortedF32 = 1, AtomicF32 = 2, RowsBF16 = 3, DenseF32 = 4, SortedF16 = 5 };

template <int NS>
struct Ctl {
  uint64_t full[NS];
  uint64_t empty[NS];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t raw_full[kMaxRaw];   // weight-only quantised B: raw ring
  uint64_t raw_empty[kMaxRaw];
  uint32_t tmem_base;
  int32_t abort;
  // CTA pairs with converters: the odd CTA signals a converted stage to the
  // even CTA by a 16-byte bulk copy into relay_dst[stage] (completing on the
  // even CTA's full barrier); relay_src is its (ignored) source
  alignas(16) uint8_t relay_dst[NS][16];
  alignas(16) uint8_t relay_src[16];
  // dynamic tile schedule: the tile of the i-th unit of work in slot i % 16
  // (16 bytes each: the odd CTA of a pair receives it by bulk copy), ready
  // when tile_full[i % 16] completes phase (i / 16) & 1
  alignas(16) int32_t tile_slot[kTileSlots][4];
  uint64_t tile_full[kTileSlots];
};

struct KParams {
  const bf16* bias;
  void* out;
  const int32_t* offsets;
  const int32_t* row_index;
  const float* row_weight;
  int32_t* error_word;
  int32_t E, N, K, NB, sentinel, div;
  const void* a_rows;  // gathered A: token rows [M, K] (row r: token row_index[r] / div)
  // dynamic tile schedule (bf16 grouped GEMMs): {next tile, CTAs done}, zero
  // at launch, reset by the last CTA to finish; null: static schedule
  int32_t* sched;
  int32_t dense_rows;             // > 0: one expert, rows [0, dense_rows), no offsets
  const float* gemm1_row_weight;  // SwiGLU: per-item weight multiplied into z, or null
  // FP8 dequantisation: acc * a_scale[row] * w_scale[e, col] (per channel,
  // w_scale_ld columns per expert) or * w_scale[e] (per expert)
  const float* a_scale;
  const float* w_scale;
  int32_t w_scale_per_channel, w_scale_ld;
  float* row_amax;  // SwiGLU FP8: atomic max of |bf16 z| per sorted row, or null
  // block-scaled SwiGLU: z is quantised in the epilogue, E4M3 codes in out
  // and one scale per row and 128-column group here, [N / 128][bs_a_ld]
  float* z_group_scale;
  // weight-only quantised B: group size along K, group rows per 64-row
  // stage (1 or 2), zero points present, bytes per raw stage
  int32_t wq_G, wq_gbox, wq_has_zero, wq_raw_tx;
  // block-scaled FP8: activation scales [K/128][a_ld] (group-major), weight
  // scales [E][K/128][w_scale_ld] per 128 x 128 block
  int64_t bs_a_ld;
  // SortedF16: the exponent e of each row's 32-column chunk, [ceil(N/32)][cap]
  uint8_t* o_exp;
  int64_t o_exp_ld;
  // nonzero: tmB views the weights with the tile's 128-byte column chunks as
  // a dimension of their own (stride 128 bytes), so that one TMA copy fills
  // every chunk of a stage; zero: one copy per chunk
  int32_t b_one_box;
};

// Waits for phase `parity` of `bar` to complete.  Gives up (returns false)
// when another role of the CTA has aborted, or after limit_ns, in which case
// it records MOE_ERR_TIMEOUT and raises the CTA's abort flag.
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, int32_t* abort,
                                             int32_t* err, uint64_t limit_ns = kWaitLimitNs) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    // suspended rather than spinning, so waiting roles leave the issue
    // slots to the working ones; wakes when the phase completes
    if (ptx::mbar_try_wait_suspend(bar, parity, 1000000u)) return true;
    if (*reinterpret_cast<volatile int32_t*>(abort)) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      *reinterpret_cast<volatile int32_t*>(abort) = 1;
      record_error(err, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

// One CTA waits on a barrier that nothing arrives at; the bounded wait must
// end it with MOE_ERR_TIMEOUT.
__global__ void wait_timeout_probe_kernel(int32_t* err, uint64_t limit_ns) {
  pdl_begin();
  __shared__ uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) bounded_wait(&bar, 0, &abort_flag, err, limit_ns);
}

struct Tile {
  int e, row0, nb;
};

// Tile t -> (expert, first padded row, column block).  Row blocks of one
// expert are innermost.  s_off holds the padded expert offsets (read through
// L1: a binary search per tile).
__device__ __forceinline__ Tile map_tile(int t, const int32_t* __restrict__ s_off, int E,
                                         int NB) {
  int lo = 0, hi = E - 1;  // largest e with (s_off[e] / BM) * NB <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((s_off[mid] / BM) * NB <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mblocks = (s_off[e + 1] - s_off[e]) / BM;
  const int local = t - (s_off[e] / BM) * NB;
  Tile tl;
  tl.e = e;
  tl.nb = local / mblocks;
  tl.row0 = s_off[e] + (local % mblocks) * BM;
  return tl;
}

// CTA pairs: pair tile t -> (expert, column block, pair of row blocks).
// s_pp[e] = sum over e' < e of ceil(row blocks of e' / 2).  CTA `rank` of
// the pair takes row block 2 * pair + rank, which may not exist (odd count):
// then it still feeds its half of the MMA (rows past the expert, never
// stored) and skips the epilogue.
struct PairTile {
  int e, row0, nb;
  bool mine;  // this CTA's row block belongs to the expert
};
// Tile t of a CTA pair: expert, column block, and this CTA's row block of
// row sub-tile h (a tile spans 2 * SUB row blocks: sub-tile h holds blocks
// 2 SUB q + 2 h + rank).  s_pp: prefix over the experts of their tiles.
template <int SUB>
__device__ __forceinline__ PairTile map_pair_tile(int t, int h, const int32_t* s_pp,
                                                  const int32_t* __restrict__ off, int E,
                                                  int NB, int rank) {
  int lo = 0, hi = E - 1;  // largest e with s_pp[e] * NB <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pp[mid] * NB <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int pairs = s_pp[e + 1] - s_pp[e];
  const int local = t - s_pp[e] * NB;
  const int mb = 2 * SUB * (local % pairs) + 2 * h + rank;
  PairTile tl;
  tl.e = e;
  tl.nb = local / pairs;
  tl.row0 = off[e] + mb * BM;
  tl.mine = mb < (off[e + 1] - off[e]) / BM;
  return tl;
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Loads 8 bf16 bias values as floats (zeros if bias == null or past n_lim).
__device__ __forceinline__ void load_bias8(const bf16* bias, int64_t off, bool ok, float* f) {
  if (bias != nullptr && ok) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(bias + off));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(h[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = 0.f;
  }
}

// Per-tile values of the SwiGLU epilogue that do not depend on the
// accumulator, loaded before its wait.  Lane = accumulator row; the warp's
// 64 columns n_base + 32 c + lane (c = 0, 1) are spread over the lanes, one
// per lane and array, and broadcast with shuffles when used.
struct SwiRow {
  float sa, zw;          // row: activation scale (FP8), weight multiplied into z
  bool real;             // row holds a routed item (padding rows are not stored)
  float sg[2], su[2];    // weight scales of gate / up columns (FP8)
  float bg[2], bu[2];    // biases of gate / up columns
};

template <bool F8>
__device__ __forceinline__ void swiglu_prefetch(const KParams& P, int e, int n_base, int64_t p,
                                                int lane, SwiRow& r) {
  const int N = P.N;
  const int32_t entry = P.row_index[p];
  r.real = entry >= 0 && entry < P.sentinel;
  r.zw = (r.real && P.gemm1_row_weight != nullptr) ? P.gemm1_row_weight[entry] : 1.0f;
  r.sa = F8 ? P.a_scale[p] : 1.0f;
  const int64_t brow = static_cast<int64_t>(e) * 2 * N;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int n = n_base + 32 * c + lane;
    const bool in = n < N;
    if constexpr (F8) {
      if (P.w_scale == nullptr) {
        r.sg[c] = r.su[c] = 1.f;
      } else if (P.w_scale_per_channel) {
        const float* ws = P.w_scale + static_cast<int64_t>(e) * P.w_scale_ld;
        r.sg[c] = in ? __ldg(ws + n) : 0.f;
        r.su[c] = in ? __ldg(ws + N + n) : 0.f;
      } else {
        r.sg[c] = r.su[c] = __ldg(P.w_scale + e);
      }
    } else {
      r.sg[c] = r.su[c] = 1.f;
    }
    const bool b = P.bias != nullptr && in;
    r.bg[c] = b ? __bfloat162float(P.bias[brow + n]) : 0.f;
    r.bu[c] = b ? __bfloat162float(P.bias[brow + N + n]) : 0.f;
  }
}

template <Epi EPI, int CG, bool F8, Wq WQ = Wq::None, bool BS = false, bool GA = false>
__device__ __forceinline__ void gemm_body(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                          const CUtensorMap* tmO, const CUtensorMap* tmS,
                                          const CUtensorMap* tmZ, const KParams& P) {
  using G = Geo<CG, F8, WQ>;
  // raw ring regions: single CTA, the tile's 256 columns (SwiGLU: gate and
  // up halves); CTA pair, this CTA's 128 columns (SwiGLU: gate for the even
  // CTA, up for the odd one)
  using R = std::conditional_t<CG == 2, WqRing<WQ, 1, 128>,
                               WqRing<WQ, EPI == Epi::SwiGLU ? 2 : 1>>;
  static_assert(R::BYTES == G::Raw::BYTES, "raw ring as sized in the shared-memory budget");
  constexpr bool WQM = WQ != Wq::None;
  constexpr int CONV = conv_warps<WQ>();
  constexpr int AWARP = 2 + CONV;  // quantised B: the warp loading A
  constexpr int EPI0 = WQM ? AWARP + 1 : 2;  // first epilogue warp
  constexpr int NEPI = BS ? 16 : EPI_WARPS;  // epilogue warps
  // GA (gathered A): A rows copied from the token rows by the gather warp
  // that follows the epilogue warps, instead of TMA loads of permuted rows
  constexpr int GWARP = EPI0 + NEPI;
  static_assert(!GA || (!WQM && !BS && !F8 && EPI == Epi::SwiGLU), "gathered A: bf16 GEMM1");
  // Int4 / MX B tiles hold each aligned group of 8 columns in the order
  // 0 4 1 5 2 6 3 7 (wq_pair_pos), and so does the accumulator: the epilogue
  // reads column n of a group from position wq_pair_pos(n)
  constexpr bool PERM = WQ != Wq::None && WqFmt<WQ>::PAIRS;
  auto acc_pos = [](int n) { return PERM ? (n & ~7) + wq_pair_pos(n & 7) : n; };
  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctl<G::NSTAGES> ctl;
  static_assert(G::SMEM + sizeof(Ctl<G::NSTAGES>) <= 232448,
                "dynamic + static shared memory within the per-block limit");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;

  // 1024-byte aligned tile area (128-byte swizzle atoms), staging, prefix.
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* tiles = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* staging = tiles + G::NSTAGES * G::STAGE;  // 1024-byte aligned
  int32_t* s_pp = reinterpret_cast<int32_t*>(staging + EPI_WARPS * STAGING_BYTES);
  uint8_t* rawbuf = staging + EPI_WARPS * STAGING_BYTES + G::PREFIX_BYTES;  // WQ raw ring
  static_assert((EPI_WARPS * STAGING_BYTES + G::PREFIX_BYTES) % 1024 == 0 &&
                    (G::NSTAGES * G::STAGE) % 1024 == 0,
                "staging, prefix and raw ring start 1024-byte aligned");
  const int32_t* off = P.offsets;
  // Block-scaled SwiGLU quantising z: the four epilogue warps of a TMEM lane
  // quadrant each hold 32 of a row's 128 z columns and exchange their rows'
  // partial maxima here, in the staging area (which that epilogue does not
  // use): parts by tile parity, quadrant, warp and row, and one barrier per
  // quadrant that completes when its four warps have written theirs.
  struct ZExchange {
    uint32_t part[2][4][4][32];
    uint64_t bar[4];
  };
  static_assert(sizeof(ZExchange) <= EPI_WARPS * STAGING_BYTES, "exchange within the staging area");
  ZExchange* zx = reinterpret_cast<ZExchange*>(staging);

  if constexpr (CG == 2) {
    // prefix of ceil(row blocks / 2) over the experts: lane chunks + warp scan
    if (warp == 0) {
      const int per = ceil_div(P.E, 32);
      const int e0 = lane * per, e1 = min(P.E, e0 + per);
      int32_t part = 0;
      for (int e = e0; e < e1; ++e) part += ((off[e + 1] - off[e]) / BM + 2 * G::SUB - 1) / (2 * G::SUB);
      int32_t incl = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int32_t run = incl - part;
      for (int e = e0; e < e1; ++e) {
        s_pp[e] = run;
        run += ((off[e + 1] - off[e]) / BM + 2 * G::SUB - 1) / (2 * G::SUB);
      }
      if (lane == 31) s_pp[P.E] = incl;
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < G::NSTAGES; ++i) {
      // the producer's arrive with A's bytes, or (quantised B) the converter
      // warps' arrivals, one of them having raised the count by A's bytes
      // quantised B: the converter warps and the A warp (arrive + bytes);
      // the odd CTA of a pair loads A onto the even CTA's barrier, so its
      // own (read by its relay) counts the converters alone
      // gathered A: the producer's arrival (B's bytes) and the gather warp's
      // 32 lanes; the odd CTA of a pair counts its gather lanes alone (read
      // by its relay)
      ptx::mbar_init(&ctl.full[i], WQM  ? CONV + (CG == 1 || rank == 0 ? 1 : 0)
                                   : GA ? 32 + (CG == 1 || rank == 0 ? 1 : 0)
                                        : 1);
      ptx::mbar_init(&ctl.empty[i], 1);
    }
    if constexpr (WQM) {
      for (int i = 0; i < R::NRAW; ++i) {
        ptx::mbar_init(&ctl.raw_full[i], 1);
        ptx::mbar_init(&ctl.raw_empty[i], CONV);
      }
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&ctl.tmem_full[a], 1);
      ptx::mbar_init(&ctl.tmem_empty[a], CG * NEPI);
    }
    // the producer's arrival (the odd CTA's with the 16 bytes it expects)
    for (int i = 0; i < kTileSlots; ++i) ptx::mbar_init(&ctl.tile_full[i], 1);
    if constexpr (BS && EPI == Epi::SwiGLU)
      for (int i = 0; i < 4; ++i) ptx::mbar_init(&zx->bar[i], 4);
    ctl.abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    if constexpr (!GA) ptx::prefetch_tmap(tmA);
    ptx::prefetch_tmap(tmB);
    if constexpr (EPI == Epi::SortedF32 || EPI == Epi::SortedF16 || EPI == Epi::SwiGLU)
      ptx::prefetch_tmap(tmO);
    if constexpr (WQM) {
      ptx::prefetch_tmap(tmS);
      if (P.wq_has_zero) ptx::prefetch_tmap(tmZ);
    }
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      ptx::tmem_alloc_pair(&ctl.tmem_base, TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&ctl.tmem_base, TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;

  const int dense_blocks = ceil_div(P.dense_rows, BM);
  const int total_tiles = P.dense_rows > 0 ? dense_blocks * P.NB
                          : (CG == 2)      ? s_pp[P.E] * P.NB
                                           : (off[P.E] / BM) * P.NB;
  const int unit = (CG == 2) ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = (CG == 2) ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int KB = ceil_div(P.K, G::BKE);
  // Dynamic tile schedule (bf16 grouped GEMMs with P.sched): the producer
  // claims tiles from a global counter in order as its unit becomes free, so
  // the units working on the row blocks that share a weight tile start it
  // together and find it in L2 (a static round-robin lets them drift up to
  // most of a tile apart).  The producer publishes each claim in the tile
  // ring; the other roles read it from there.  Static: unit + i * units.
  const bool dyn = !WQM && !GA && !BS && P.sched != nullptr;
  auto tile_at = [&](int i) -> int {  // the i-th tile of this unit, or -1 past the last
    if (!dyn) {
      const int t = unit + i * units;
      return t < total_tiles ? t : -1;
    }
    const int slot = i % kTileSlots;
    if (!bounded_wait(&ctl.tile_full[slot], static_cast<uint32_t>(i / kTileSlots) & 1u, &ctl.abort,
                      P.error_word))
      return -1;
    return *reinterpret_cast<volatile int32_t*>(&ctl.tile_slot[slot][0]);
  };

  // (h: row sub-tile, always 0 unless G::SUB = 2)
  auto tile_of = [&](int t, int& e, int& row0, int& nb, bool& mine, int h = 0) {
    if constexpr (CG == 2) {
      const PairTile pt = map_pair_tile<G::SUB>(t, h, s_pp, off, P.E, P.NB, static_cast<int>(rank));
      e = pt.e;
      row0 = pt.row0;
      nb = pt.nb;
      mine = pt.mine;
    } else if (P.dense_rows > 0) {
      e = 0;
      nb = t / dense_blocks;
      row0 = (t % dense_blocks) * BM;
      mine = true;
    } else {
      const Tile tl = map_tile(t, off, P.E, P.NB);
      e = tl.e;
      row0 = tl.row0;
      nb = tl.nb;
      mine = true;
    }
  };

  if (WQM && warp == 0) {
    // ------------------------------------- TMA producer (quantised B) --
    // per 64-row K stage: the raw codes / scales / zero points of the four
    // 64-column chunks into the raw ring, as far ahead as the ring allows
    // (A goes to the main ring from the A warp)
    if (lane == 0) {
      int rstage = 0;
      uint32_t rphase = 0;
      bool ok = true;
      for (int t = unit; t < total_tiles && ok; t += units) {
        int e, row0, nb;
        bool mine;
        tile_of(t, e, row0, nb, mine);
        for (int kb = 0; kb < KB; ++kb) {
          if (!bounded_wait(&ctl.raw_empty[rstage], rphase ^ 1u, &ctl.abort, P.error_word)) {
            ok = false;
            break;
          }
          uint64_t* rf = &ctl.raw_full[rstage];
          ptx::mbar_arrive_expect_tx(rf, P.wq_raw_tx);
          uint8_t* rb = rawbuf + rstage * R::STAGE;
          const int g0 = (kb * G::BKE) / P.wq_G;
          if constexpr (CG == 2) {
            // this CTA's 128 columns: SwiGLU gate (even CTA) or up (odd CTA)
            // columns [nb*128, +128); otherwise [nb*256 + rank*128, +128)
            if constexpr (EPI == Epi::SwiGLU) {
              const int col = nb * (MMA_N / 2);
              const int hf = static_cast<int>(rank);
              ptx::tma_load_4d(rb, tmB, rf, col * R::F::CODE_BITS / 8, hf, kb * G::BKE, e);
              ptx::tma_load_4d(rb + R::SC_OFF, tmS, rf, col, hf, g0, e);
              if (P.wq_has_zero) ptx::tma_load_4d(rb + R::Z_OFF, tmZ, rf, col, hf, g0, e);
            } else {
              const int col = nb * MMA_N + static_cast<int>(rank) * (MMA_N / 2);
              ptx::tma_load_3d(rb, tmB, rf, col * R::F::CODE_BITS / 8, kb * G::BKE, e);
              ptx::tma_load_3d(rb + R::SC_OFF, tmS, rf, col, g0, e);
              if (P.wq_has_zero) ptx::tma_load_3d(rb + R::Z_OFF, tmZ, rf, col, g0, e);
            }
          } else if constexpr (EPI == Epi::SwiGLU) {
            // region 0: gate columns [nb*128, +128); region 1: the same up columns
            const int col = nb * (MMA_N / 2);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              ptx::tma_load_4d(rb + g * R::CODES, tmB, rf, col * R::F::CODE_BITS / 8, g,
                               kb * G::BKE, e);
              ptx::tma_load_4d(rb + R::SC_OFF + g * R::SCALES, tmS, rf, col, g, g0, e);
              if (P.wq_has_zero)
                ptx::tma_load_4d(rb + R::Z_OFF + g * R::ZEROS, tmZ, rf, col, g, g0, e);
            }
          } else {
            const int col = nb * MMA_N;
            ptx::tma_load_3d(rb, tmB, rf, col * R::F::CODE_BITS / 8, kb * G::BKE, e);
            ptx::tma_load_3d(rb + R::SC_OFF, tmS, rf, col, g0, e);
            if (P.wq_has_zero) ptx::tma_load_3d(rb + R::Z_OFF, tmZ, rf, col, g0, e);
          }
          if (++rstage == R::NRAW) {
            rstage = 0;
            rphase ^= 1u;
          }
        }
      }
    }
  } else if (WQM && warp < 2 + CONV && warp >= 2) {
    // ------------------------------------------- converters (quantised B) --
    // The stage's region rows (2 x 64 for the SwiGLU GEMM, 64 otherwise) are
    // split evenly over the converter warps.  A region row is read by LPR
    // lanes of 8 columns each (16 lanes for 128 columns, 32 for 256), so a
    // warp reads whole rows -- no bank conflicts -- and every lane keeps one
    // set of group parameters.  Each lane writes its 8 columns as bf16 in
    // the 128-byte-swizzled layout TMA would have produced (16-byte unit j
    // of K row r of a 64-column chunk at j ^ (r & 7)); then the warp arrives
    // on the stage's barrier.
    // regions of this CTA's B tile (a CTA of a pair converts one: its 128 columns)
    constexpr int NREG = (CG == 1 && EPI == Epi::SwiGLU) ? 2 : 1;
    static_assert(NREG * R::RCOLS == 256 / CG, "converted columns = this CTA's B tile");
    constexpr int LPR = R::RCOLS / 8;                 // lanes per region row
    constexpr int RPI = 32 / LPR;                     // rows per warp instruction
    constexpr int ROWS = NREG * 64 / (CONV > 0 ? CONV : 1);  // region rows per warp
    constexpr int ITERS = ROWS / RPI;
    static_assert(!WQM || (ROWS % RPI == 0 && 32 % ROWS == 0), "converter row split");
    const int cw = warp - 2;
    const int first = cw * ROWS;                      // first region row of this warp
    const int reg = first / 64;                       // region (gate / up)
    const int k0 = first % 64 + lane / LPR;           // this lane's first K row
    const int col = (lane % LPR) * 8;                 // first of its 8 columns in the region
    const int gr = (first % 64) / 32;                 // group row (G = 32) of its rows
    const int chunk = reg * (R::RCOLS / 64) + col / 64;  // 64-column chunk of the B tile
    const int unit8 = (col % 64) / 8;
    int stage = 0, rstage = 0;
    uint32_t phase = 0, rphase = 0;
    bool ok = true;
    for (int t = unit; t < total_tiles && ok; t += units) {
      int e, row0, nb;
      bool mine;
      tile_of(t, e, row0, nb, mine);
      for (int kb = 0; kb < KB; ++kb) {
        bool got = bounded_wait(&ctl.empty[stage], phase ^ 1u, &ctl.abort, P.error_word);
        got = got && bounded_wait(&ctl.raw_full[rstage], rphase, &ctl.abort, P.error_word);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint8_t* rb = rawbuf + rstage * R::STAGE;
        const uint8_t* rc = rb + reg * R::CODES + col * R::F::CODE_BITS / 8;
        uint8_t* dst = tiles + stage * G::STAGE + G::B_OFF + chunk * G::CHUNK_BYTES;
        WqParams8 p;
        {
          const int g = P.wq_gbox == 2 ? gr : 0;
          const uint8_t* rsc = rb + R::SC_OFF + reg * R::SCALES + (g * R::RCOLS + col) * R::F::SCALE_BYTES;
          uint4 s8;
          if constexpr (R::F::SCALE_BYTES == 2) {
            s8 = *reinterpret_cast<const uint4*>(rsc);
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(rsc);
            s8 = make_uint4(v.x, v.y, 0, 0);
          }
          uint2 z8 = make_uint2(0, 0);
          if constexpr (R::F::HAS_ZERO) {
            if (P.wq_has_zero)
              z8 = *reinterpret_cast<const uint2*>(rb + R::Z_OFF + reg * R::ZEROS + g * R::RCOLS + col);
          }
          wq_params8<WQ>(s8, z8, P.wq_has_zero != 0, p);
        }
        uint2 c[ITERS];
#pragma unroll
        for (int i = 0; i < ITERS; ++i) {  // all code loads first
          const int r = k0 + RPI * i;
          if constexpr (R::F::CODE_BITS == 4)
            c[i] = make_uint2(*reinterpret_cast<const uint32_t*>(rc + r * R::ROW_BYTES), 0u);
          else
            c[i] = *reinterpret_cast<const uint2*>(rc + r * R::ROW_BYTES);
        }
#pragma unroll
        for (int i = 0; i < ITERS; ++i) {
          const int r = k0 + RPI * i;
          *reinterpret_cast<uint4*>(dst + r * 128 + ((unit8 ^ (r & 7)) << 4)) =
              wq_dequant8<WQ, PERM>(c[i], p);
        }
        ptx::fence_proxy_async_smem();  // generic writes -> visible to the tensor core
        __syncwarp();
        if (lane == 0) {
          // (pairs: the odd CTA's relay thread forwards its CTA's completed
          // stage to the even CTA's barrier)
          ptx::mbar_arrive(&ctl.full[stage]);
          ptx::mbar_arrive(&ctl.raw_empty[rstage]);
        }
        if (++stage == G::NSTAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++rstage == R::NRAW) {
          rstage = 0;
          rphase ^= 1u;
        }
      }
    }
  } else if (WQM && warp == AWARP) {
    // ----------------------------------------- A producer (quantised B) --
    // each stage's A rows as soon as the stage is free; the arrival carries
    // the bytes, so the phase cannot complete before they are counted
    // (pairs: both CTAs' rows and the odd CTA's relay copy complete on the
    // even CTA's barrier, which counts all their bytes)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = unit; t < total_tiles && ok; t += units) {
        int e, row0, nb;
        bool mine;
        tile_of(t, e, row0, nb, mine);
        for (int kb = 0; kb < KB; ++kb) {
          if (!bounded_wait(&ctl.empty[stage], phase ^ 1u, &ctl.abort, P.error_word)) {
            ok = false;
            break;
          }
          if constexpr (CG == 2) {
            // this CTA's rows of both row sub-tiles (row blocks past the
            // expert's, or past the tensor, load rows of the next expert or
            // zeros: their results are not stored)
            if (rank == 0)
              ptx::mbar_arrive_expect_tx(&ctl.full[stage],
                                         2 * G::SUB * A_STAGE_BYTES + kRelayBytes);
#pragma unroll
            for (int h = 0; h < G::SUB; ++h)
              ptx::tma_load_2d_pair(tiles + stage * G::STAGE + h * A_STAGE_BYTES, tmA,
                                    ptx::mapa_shared(ptx::smem_u32(&ctl.full[stage]), 0),
                                    kb * G::BKE, row0 + h * 2 * BM);
          } else {
            ptx::mbar_arrive_expect_tx(&ctl.full[stage], A_STAGE_BYTES);
            ptx::tma_load_2d(tiles + stage * G::STAGE, tmA, &ctl.full[stage], kb * G::BKE, row0);
          }
          if (++stage == G::NSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const bool claimer = dyn && (CG == 1 || rank == 0);
      int early = -1;  // the next tile's claim, made during this tile's last stages
      for (int i = 0; ok; ++i) {
        int t;
        if (dyn) {
          // claim the next tile and publish it (pairs: the even CTA claims
          // and hands the claim to the odd CTA by a 16-byte bulk copy)
          const int slot = i % kTileSlots;
          if (claimer) {
            const int c = early >= 0 ? early : atomicAdd(P.sched, 1);
            early = -1;
            t = c < total_tiles ? c : -1;
            ctl.tile_slot[slot][0] = t;
            if constexpr (CG == 2) {
              ptx::fence_proxy_async_smem();  // the slot as the copy's source
              ptx::bulk_copy_to_cluster(ptx::mapa_shared(ptx::smem_u32(ctl.tile_slot[slot]), 1),
                                        ctl.tile_slot[slot], 16,
                                        ptx::mapa_shared(ptx::smem_u32(&ctl.tile_full[slot]), 1));
            }
            ptx::mbar_arrive(&ctl.tile_full[slot]);
          } else {
            ptx::mbar_arrive_expect_tx(&ctl.tile_full[slot], 16);
            t = tile_at(i);
          }
        } else {
          t = tile_at(i);
        }
        if (t < 0) break;
        int e, row0, nb;
        bool mine;
        tile_of(t, e, row0, nb, mine);
        for (int kb = 0; kb < KB; ++kb) {
          if (!bounded_wait(&ctl.empty[stage], phase ^ 1u, &ctl.abort, P.error_word)) {
            ok = false;
            break;
          }
          // the next claim's round trip (~1-2 us) overlaps this tile's last
          // four stages (a short tile: all of it)
          if (claimer && kb == (KB > 4 ? KB - 4 : 0)) early = atomicAdd(P.sched, 1);
          uint8_t* sa = tiles + stage * G::STAGE;
          uint8_t* sb = sa + G::B_OFF;
          // (gathered A: the stage's B bytes only)
          if constexpr (CG == 1) {
            ptx::mbar_arrive_expect_tx(&ctl.full[stage], GA ? G::STAGE - G::B_OFF : G::STAGE);
            if constexpr (!GA) ptx::tma_load_2d(sa, tmA, &ctl.full[stage], kb * G::BKE, row0);
            if (P.b_one_box) {
              // (column in chunk, k, chunk, [half,] expert)
              if constexpr (EPI == Epi::SwiGLU)
                ptx::tma_load_5d(sb, tmB, &ctl.full[stage], 0, kb * G::BKE,
                                 nb * (G::CHUNKS / 2), 0, e);
              else
                ptx::tma_load_4d(sb, tmB, &ctl.full[stage], 0, kb * G::BKE, nb * G::CHUNKS, e);
            } else {
#pragma unroll
              for (int c = 0; c < G::CHUNKS; ++c) {
                if constexpr (EPI == Epi::SwiGLU)  // gate cols [nb*128,+128), then the up half
                  ptx::tma_load_4d(sb + c * G::CHUNK_BYTES, tmB, &ctl.full[stage],
                                   nb * (MMA_N / 2) + (c % (G::CHUNKS / 2)) * G::CW,
                                   c / (G::CHUNKS / 2), kb * G::BKE, e);
                else
                  ptx::tma_load_3d(sb + c * G::CHUNK_BYTES, tmB, &ctl.full[stage],
                                   nb * MMA_N + c * G::CW, kb * G::BKE, e);
              }
            }
          } else {
            // both CTAs' copies complete on the even CTA's barrier, which
            // expects the bytes of the whole pair
            const uint32_t full0 = ptx::mapa_shared(ptx::smem_u32(&ctl.full[stage]), 0);
            if (rank == 0)
              ptx::mbar_arrive_expect_tx(&ctl.full[stage],
                                         GA ? 2 * (G::STAGE - G::B_OFF) + kRelayBytes : 2 * G::STAGE);
            if constexpr (!GA) ptx::tma_load_2d_pair(sa, tmA, full0, kb * G::BKE, row0);
            if (P.b_one_box) {
              if constexpr (EPI == Epi::SwiGLU)  // even CTA: gate columns, odd CTA: up columns
                ptx::tma_load_5d_pair(sb, tmB, full0, 0, kb * G::BKE, nb * (G::CHUNKS / 2),
                                      static_cast<int>(rank), e);
              else
                ptx::tma_load_4d_pair(sb, tmB, full0, 0, kb * G::BKE,
                                      nb * G::CHUNKS + static_cast<int>(rank) * G::B_CHUNKS_CTA, e);
            } else {
#pragma unroll
              for (int c = 0; c < G::B_CHUNKS_CTA; ++c) {
                const int gc = static_cast<int>(rank) * G::B_CHUNKS_CTA + c;  // chunk of the tile
                if constexpr (EPI == Epi::SwiGLU)  // even CTA: gate columns, odd CTA: up columns
                  ptx::tma_load_4d_pair(sb + c * G::CHUNK_BYTES, tmB, full0,
                                        nb * (MMA_N / 2) + (gc % (G::CHUNKS / 2)) * G::CW,
                                        gc / (G::CHUNKS / 2), kb * G::BKE, e);
                else
                  ptx::tma_load_3d_pair(sb + c * G::CHUNK_BYTES, tmB, full0,
                                        nb * MMA_N + gc * G::CW, kb * G::BKE, e);
              }
            }
          }
          if (++stage == G::NSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    // (CG = 2: only the even CTA issues; its MMAs read both CTAs' tiles)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int i = 0; ok && tile_at(i) >= 0; ++i) {
        // block-scaled FP8: every K stage is its own accumulation, into the
        // two accumulators in turn, handed to the epilogue stage by stage
        // (two row sub-tiles: both accumulators, sub-tile h in accumulator h)
        if (!BS && !bounded_wait(&ctl.tmem_empty[acc], acc_phase ^ 1u, &ctl.abort, P.error_word)) break;
        if (G::SUB == 2 &&
            !bounded_wait(&ctl.tmem_empty[1], acc_phase ^ 1u, &ctl.abort, P.error_word))
          break;
        ptx::tc_fence_after();
        uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MMA_N);
        for (int kb = 0; kb < KB; ++kb) {
          if constexpr (BS) {
            if (!bounded_wait(&ctl.tmem_empty[acc], acc_phase ^ 1u, &ctl.abort, P.error_word)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            d_tmem = tmem_base + static_cast<uint32_t>(acc * MMA_N);
          }
          if (!bounded_wait(&ctl.full[stage], phase, &ctl.abort, P.error_word)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(tiles + stage * G::STAGE);
          const uint32_t sb = sa + G::B_OFF;
#pragma unroll
          for (int ks = 0; ks < G::KSTEPS; ++ks) {
            // B (MN-major): advance UMMA_K k-rows; column chunks are
            // CHUNK_BYTES apart, 8-row k groups 1024 bytes apart.
            const uint64_t bdesc =
                ptx::smem_desc_sw128(sb + ks * G::B_KSTEP, G::CHUNK_BYTES, 1024);
            const uint32_t accum = (BS ? ks : (kb | ks)) != 0 ? 1u : 0u;
#pragma unroll
            for (int h = 0; h < G::SUB; ++h) {
              // A (K-major): advance UMMA_K elements = 32 bytes along the swizzled row.
              const uint64_t adesc = ptx::smem_desc_sw128(sa + h * A_STAGE_BYTES + ks * 32, 16, 1024);
              const uint32_t d = d_tmem + static_cast<uint32_t>(h * MMA_N);
              if constexpr (CG == 2 && F8) ptx::mma_e4m3_pair(d, adesc, bdesc, G::IDESC, accum);
              else if constexpr (CG == 2) ptx::mma_bf16_pair(d, adesc, bdesc, G::IDESC, accum);
              else if constexpr (F8) ptx::mma_e4m3(d, adesc, bdesc, G::IDESC, accum);
              else ptx::mma_bf16(d, adesc, bdesc, G::IDESC, accum);
            }
          }
          if constexpr (CG == 2) ptx::mma_commit_pair(&ctl.empty[stage], 0x3);
          else ptx::mma_commit(&ctl.empty[stage]);
          if (++stage == G::NSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if constexpr (BS) {
            ptx::mma_commit(&ctl.tmem_full[acc]);
            if (++acc == 2) {
              acc = 0;
              acc_phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        if constexpr (!BS) {
#pragma unroll
          for (int h = 0; h < G::SUB; ++h) {
            if constexpr (CG == 2) ptx::mma_commit_pair(&ctl.tmem_full[acc], 0x3);
            else ptx::mma_commit(&ctl.tmem_full[acc]);
            if (++acc == 2) {
              acc = 0;
              acc_phase ^= 1u;
            }
          }
        }
      }
    } else if (CG == 2 && (WQM || GA) && lane == 0) {
      // ---------------------------------- relay (odd CTA, quantised B) --
      // Once this CTA's converter warps have all arrived for a stage (each
      // after fencing its writes for the async proxy), a 16-byte bulk copy
      // into the even CTA completes on that CTA's full barrier: the
      // converted tile is signalled through the async proxy, the way this
      // CTA's TMA loads signal theirs.  (An arrive with release at cluster
      // scope costs a cluster-wide memory barrier, ~1500 cycles, per stage.)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = unit; t < total_tiles && ok; t += units) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!bounded_wait(&ctl.full[stage], phase, &ctl.abort, P.error_word)) {
            ok = false;
            break;
          }
          ptx::bulk_copy_to_cluster(ptx::mapa_shared(ptx::smem_u32(ctl.relay_dst[stage]), 0),
                                    ctl.relay_src, kRelayBytes,
                                    ptx::mapa_shared(ptx::smem_u32(&ctl.full[stage]), 0));
          if (++stage == G::NSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (GA && warp == GWARP) {
    // ------------------------------------------------ A gatherer (GA) --
    // The stage's A rows straight from the token rows: row r of the tile is
    // item row_index[row0 + r] of token item / top_k; padding slots, rows
    // past the expert and columns past K are zero-filled.  Lane l copies rows
    // l, l + 32, l + 64, l + 96: eight 16-byte cp.async per row into the
    // 128-byte-swizzled K-major layout TMA would have produced (16-byte chunk
    // c of row r at c ^ (r & 7)).  A lane waits for its own copies kGaLag
    // stages behind, fences them for the async proxy and then arrives on
    // that stage's barrier (the odd CTA of a pair: its own, for the relay).
    constexpr int kGaLag = 2;
    static_assert(!GA || kGaLag < G::NSTAGES, "gather lag within the ring");
    const bf16* xa = reinterpret_cast<const bf16*>(P.a_rows);
    int stage = 0, sig = 0;
    uint32_t phase = 0;
    int pending = 0;  // stages copied but not yet signalled (the oldest is `sig`)
    bool ok = true;
    auto signal_oldest = [&]() {
      ptx::fence_proxy_async_smem();  // this lane's completed copies -> the tensor core
      ptx::mbar_arrive(&ctl.full[sig]);
      if (++sig == G::NSTAGES) sig = 0;
      --pending;
    };
    for (int t = unit; t < total_tiles && ok; t += units) {
      int e, row0, nb;
      bool mine;
      tile_of(t, e, row0, nb, mine);
      const bf16* src[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int32_t item = mine ? P.row_index[row0 + lane + 32 * i] : P.sentinel;
        src[i] = (item >= 0 && item < P.sentinel)
                     ? xa + static_cast<int64_t>(item / P.div) * P.K : nullptr;
      }
      for (int kb = 0; kb < KB; ++kb) {
        const bool got = bounded_wait(&ctl.empty[stage], phase ^ 1u, &ctl.abort, P.error_word);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        uint8_t* dst = tiles + stage * G::STAGE;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = lane + 32 * i;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int col = kb * G::BKE + 8 * c;
            const bool live = src[i] != nullptr && col < P.K;  // K % 8 == 0
            ptx::cp_async_16(dst + r * 128 + ((c ^ (r & 7)) << 4), live ? src[i] + col : xa,
                             live ? 16u : 0u);
          }
        }
        ptx::cp_async_commit();
        ++pending;
        if (pending > kGaLag) {
          ptx::cp_async_wait<kGaLag>();
          signal_oldest();
        }
        if (++stage == G::NSTAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    ptx::cp_async_wait<0>();
    while (pending > 0) signal_oldest();
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;               // TMEM lane quadrant this warp may access
    const int half = (warp - EPI0) >> 2;  // which half of the tile's columns it owns
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    // hand the accumulator back to the MMA warp (the even CTA's MMA waits
    // for the epilogue warps of both CTAs)
    auto release_acc = [&](int a) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2)
          ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&ctl.tmem_empty[a]), 0));
        else
          ptx::mbar_arrive(&ctl.tmem_empty[a]);
      }
    };
    if constexpr (BS) {
      // ------------------------------------------- block-scaled FP8 epilogue --
      // "fused_moe.py 分析", FP8 W8A8, block-wise: each K block's dot product
      // (one stage's accumulator) times that block's activation scale (per
      // row and 128-wide K group) and weight scale (per 128 x 128 block),
      // summed over the K blocks in registers.  The SwiGLU GEMM leaves z
      // quantised for the second GEMM (E4M3 codes and one scale per row and
      // 128-column group: its tile's z columns), not as bf16 for a pass of
      // its own.
      // CH accumulator chunks of 32 columns per warp: the quadrant's 8
      // chunks split over its NEPI / 4 warps (SwiGLU: matching gate and up
      // chunks, the gate ones first)
      constexpr int CH = 8 / (NEPI / 4);
      const int sub = (warp - EPI0) >> 2;
      auto chunk_col = [&](int c) {
        if constexpr (EPI == Epi::SwiGLU)
          return c < CH / 2 ? 32 * (sub * (CH / 2) + c) : MMA_N / 2 + 32 * (sub * (CH / 2) + c - CH / 2);
        else
          return 32 * (sub * CH + c);
      };
      bool ok = true;
      int zt = 0;  // tiles done (the z exchange's parity)
      for (int t = unit; t < total_tiles && ok; t += units) {
        int e, row0, nb;
        bool mine;
        tile_of(t, e, row0, nb, mine);
        const int64_t p = row0 + row;
        const int32_t entry = P.row_index[p];
        const bool real = entry >= 0 && entry < P.sentinel;
        const int N = P.N;
        // weight blocks: SwiGLU gate block nb and up block N/128 + nb; the
        // other GEMM's 256-column tile spans blocks 2 nb and 2 nb + 1 (a
        // block past N stores nothing; its scale load is kept in range)
        const int blk_a = (EPI == Epi::SwiGLU) ? nb : min(2 * nb + (sub * CH * 32) / 128, P.w_scale_ld - 1);
        const int blk_b = (EPI == Epi::SwiGLU) ? N / 128 + nb : blk_a;
        const float* wsc = P.w_scale + static_cast<int64_t>(e) * KB * P.w_scale_ld;
        float accv[CH][32];
#pragma unroll
        for (int c = 0; c < CH; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) accv[c][j] = 0.f;
        for (int kb = 0; kb < KB; ++kb) {
          // the block's scales, loaded before the wait for its accumulator
          const float sa = P.a_scale[static_cast<int64_t>(kb) * P.bs_a_ld + p];
          const float swa = __ldg(wsc + kb * P.w_scale_ld + blk_a);
          const float swb = __ldg(wsc + kb * P.w_scale_ld + blk_b);
          const bool got = bounded_wait(&ctl.tmem_full[acc], acc_phase, &ctl.abort, P.error_word);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t taddr =
              tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * MMA_N);
          const float sca = sa * swa, scb = sa * swb;
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            const float sc = (EPI == Epi::SwiGLU && c >= CH / 2) ? scb : sca;
            // the chunk's 32 columns as two 16-column loads behind one wait
            uint32_t v[2][16];
            ptx::tmem_ld_16cols(taddr + chunk_col(c), v[0]);
            ptx::tmem_ld_16cols(taddr + chunk_col(c) + 16, v[1]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
              for (int j = 0; j < 16; j += 2)  // packed pairs: half the FMA issues
                ptx::fma2(accv[c][16 * hh + j], accv[c][16 * hh + j + 1],
                          __uint_as_float(v[hh][j]), __uint_as_float(v[hh][j + 1]), sc);
          }
          release_acc(acc);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        if (!ok) continue;
        if constexpr (EPI == Epi::SwiGLU) {
          {
            // z rounded to bf16 and quantised for the second GEMM as its A
            // rows are: E4M3 codes with one scale per row for the tile's 128
            // z columns (one group), from the row's max |z| over the
            // quadrant's four warps (N is a multiple of 128: every column of
            // the tile exists)
            static_assert(NEPI != 16 || CH == 2, "one gate and one up chunk per warp");
            const int64_t brow = static_cast<int64_t>(e) * 2 * N;
            const int n0 = nb * (MMA_N / 2) + chunk_col(0);
            uint4 zz[4];
            uint32_t zmax2 = 0;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int n = n0 + 8 * v;
              float bg[8], bu[8];
              load_bias8(P.bias, brow + n, true, bg);
              load_bias8(P.bias, brow + N + n, true, bu);
              uint32_t* w = reinterpret_cast<uint32_t*>(&zz[v]);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int j = 8 * v + 2 * i;
                const float z0 = silu_f(accv[0][j] + bg[2 * i]) * (accv[CH / 2][j] + bu[2 * i]);
                const float z1 = silu_f(accv[0][j + 1] + bg[2 * i + 1]) *
                                 (accv[CH / 2][j + 1] + bu[2 * i + 1]);
                w[i] = pack_bf16x2(z0, z1);
                zmax2 = __vmaxu2(zmax2, w[i] & 0x7fff7fffu);
              }
            }
            const int par = zt & 1;
            ++zt;
            zx->part[par][q][sub][lane] = max(zmax2 & 0xffffu, zmax2 >> 16);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&zx->bar[q]);
            const bool got = bounded_wait(&zx->bar[q], static_cast<uint32_t>(par), &ctl.abort,
                                          P.error_word);
            if (!__all_sync(0xffffffffu, got)) {
              ok = false;
              continue;
            }
            uint32_t m = 0;
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) m = max(m, zx->part[par][q][w4][lane]);
            const RowScale rs = row_scale(__uint_as_float(m << 16));
            if (mine && real) {
              uint8_t* zq = reinterpret_cast<uint8_t*>(P.out) + p * N + n0;
#pragma unroll
              for (int v = 0; v < 4; ++v) *reinterpret_cast<uint2*>(zq + 8 * v) = e4m3x8(zz[v], rs);
              if (sub == 0) P.z_group_scale[static_cast<int64_t>(nb) * P.bs_a_ld + p] = rs.s;
            }
          }
        } else {
          if (!mine || !real) continue;
          float* o = reinterpret_cast<float*>(P.out);
          const float wgt = P.row_weight != nullptr ? P.row_weight[entry] : 1.0f;
          const int64_t brow = static_cast<int64_t>(e) * N;
#pragma unroll
          for (int c = 0; c < CH; ++c) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int n = nb * MMA_N + chunk_col(c) + 8 * v;
              if (n >= N) break;
              float b[8];
              load_bias8(P.bias, brow + n, true, b);
              float4* d = reinterpret_cast<float4*>(o + p * N + n);
              d[0] = make_float4((accv[c][8 * v] + b[0]) * wgt, (accv[c][8 * v + 1] + b[1]) * wgt,
                                 (accv[c][8 * v + 2] + b[2]) * wgt, (accv[c][8 * v + 3] + b[3]) * wgt);
              d[1] = make_float4((accv[c][8 * v + 4] + b[4]) * wgt, (accv[c][8 * v + 5] + b[5]) * wgt,
                                 (accv[c][8 * v + 6] + b[6]) * wgt, (accv[c][8 * v + 7] + b[7]) * wgt);
            }
          }
        }
      }
    } else
    // row sub-tile h of tile t (one per tile unless G::SUB = 2)
    for (int i = 0, h = 0, t = tile_at(0); t >= 0;
         (h + 1 == G::SUB) ? (h = 0, t = tile_at(++i)) : ++h) {
      int e, row0, nb;
      bool mine;
      tile_of(t, e, row0, nb, mine, h);
      const int64_t p = row0 + row;
      SwiRow sr;
      const int n_base = nb * (MMA_N / 2) + half * (MMA_N / 4);  // SwiGLU: first z column
      if constexpr (EPI == Epi::SwiGLU) {
        if (mine) swiglu_prefetch<F8>(P, e, n_base, p, lane, sr);
      }
      // The other epilogues: the row's item and weight, and the warp's 128
      // columns' biases (and FP8 scales), four columns per lane, broadcast
      // with shuffles when used -- loaded before the wait, not after it (a
      // short tile cannot hide a chain of loads behind its MMAs otherwise).
      int32_t pf_entry = -1;
      float pf_wgt = 0.f, pf_sa = 1.f;
      float pf_b[4] = {0.f, 0.f, 0.f, 0.f}, pf_s[4] = {1.f, 1.f, 1.f, 1.f};
      if constexpr (EPI != Epi::SwiGLU) {
        if (mine) {
          pf_entry = (EPI == Epi::DenseF32) ? static_cast<int32_t>(p) : P.row_index[p];
          const bool v = pf_entry >= 0 && pf_entry < P.sentinel;
          pf_wgt = v ? (P.row_weight != nullptr ? P.row_weight[pf_entry] : 1.0f) : 0.0f;
          const int N = P.N;
          const int nl = nb * MMA_N + half * (MMA_N / 2) + 4 * lane;  // this lane's 4 columns
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool in = nl + i < N;
            if (P.bias != nullptr && in)
              pf_b[i] = __bfloat162float(P.bias[static_cast<int64_t>(e) * N + nl + i]);
            if constexpr (F8) {
              if (P.w_scale == nullptr) pf_s[i] = 1.f;
              else if (!P.w_scale_per_channel) pf_s[i] = __ldg(P.w_scale + e);
              else pf_s[i] = in ? __ldg(P.w_scale + static_cast<int64_t>(e) * P.w_scale_ld + nl + i)
                                : 0.f;
            }
          }
          if constexpr (F8) pf_sa = P.a_scale[p];
        }
      }
      const bool got = bounded_wait(&ctl.tmem_full[acc], acc_phase, &ctl.abort, P.error_word);
      if (!__all_sync(0xffffffffu, got)) break;
      ptx::tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * MMA_N);
      bool released = false;

      if (!mine) {
        // this CTA's half of a pair tile has no rows of the expert
      } else if constexpr (EPI == Epi::SwiGLU) {
        const int N = P.N;
        // this warp's accumulator columns, gate [c0, c0+64) and up
        // [c0+128, c0+192): read at once and the accumulator freed before the
        // math (or, with converter warps in the CTA, one 32-column chunk at a
        // time for the smaller register budget)
        const int c0 = half * (MMA_N / 4);
        uint32_t g[2][32], u[2][32];
        if constexpr (!WQM) {
          ptx::tmem_ld_32cols(taddr + c0, g[0]);
          ptx::tmem_ld_32cols(taddr + c0 + 32, g[1]);
          ptx::tmem_ld_32cols(taddr + MMA_N / 2 + c0, u[0]);
          ptx::tmem_ld_32cols(taddr + MMA_N / 2 + c0 + 32, u[1]);
          ptx::tmem_ld_wait();
          release_acc(acc);
          released = true;
        }
        uint32_t zmax2 = 0;  // max |z| as bf16 magnitude bits, both halves
        // z is staged as the warp's 32 rows x 64 columns (one 128-byte row
        // each, 16-byte chunk j at j ^ (row & 7)) and written with one TMA
        // store; a warp whose rows are all padding, or whose columns all lie
        // past N, stores nothing (no store starts outside the tensor)
        uint8_t* stage_buf = staging + (warp - EPI0) * STAGING_BYTES;
        const bool any_real = __ballot_sync(0xffffffffu, sr.real) != 0u;
        if (any_real && n_base < N) {
          if (lane == 0) ptx::bulk_wait_read0();  // the buffer's previous store has read it
          __syncwarp();
          const bool has_bias = P.bias != nullptr;
          auto col = [&](float v, int j) { return __shfl_sync(0xffffffffu, v, j); };
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if constexpr (WQM) {
              // fewer registers per thread here: one 32-column chunk at a time
              ptx::tmem_ld_32cols(taddr + c0 + 32 * c, g[c]);
              ptx::tmem_ld_32cols(taddr + MMA_N / 2 + c0 + 32 * c, u[c]);
              ptx::tmem_ld_wait();
              if (c == 1) {
                release_acc(acc);
                released = true;
              }
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 pk;
              uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float zz[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int j = v * 8 + 2 * i + h;  // column within the 32-column chunk
                  const int ja = acc_pos(j);        // its accumulator position
                  float gv = __uint_as_float(g[c][ja]), uv = __uint_as_float(u[c][ja]);
                  if constexpr (F8) {
                    gv *= col(sr.sg[c], j) * sr.sa;
                    uv *= col(sr.su[c], j) * sr.sa;
                  }
                  if (has_bias) {
                    gv += col(sr.bg[c], j);
                    uv += col(sr.bu[c], j);
                  }
                  zz[h] = silu_f(gv) * uv * sr.zw;
                }
                w[i] = pack_bf16x2(zz[0], zz[1]);
              }
              const int chunk = c * 4 + v;
              *reinterpret_cast<uint4*>(stage_buf + lane * 128 + ((chunk ^ (lane & 7)) << 4)) = pk;
              if constexpr (F8) {
                if (sr.real && n_base + 32 * c + v * 8 < N) {
#pragma unroll
                  for (int i = 0; i < 4; ++i) zmax2 = __vmaxu2(zmax2, w[i] & 0x7fff7fffu);
                }
              }
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(tmO, stage_buf, n_base, row0 + q * 32);
            ptx::bulk_commit();
          }
        }
        if constexpr (F8) {
          // the row's amax over this tile's columns, as the stored bf16 value
          // (non-negative floats order like their bit patterns)
          const uint32_t m = max(zmax2 & 0xffffu, zmax2 >> 16) << 16;
          if (m != 0u && P.row_amax != nullptr)
            atomicMax(reinterpret_cast<unsigned int*>(P.row_amax) + p, m);
        }
      } else {
        const int N = P.N;
        const int32_t entry = pf_entry;
        const bool valid = entry >= 0 && entry < P.sentinel;
        const float wgt = pf_wgt;
        uint8_t* stage_buf = staging + (warp - EPI0) * STAGING_BYTES;
        // a warp whose 32 rows are all padding has nothing to store
        const bool any_real = __ballot_sync(0xffffffffu, valid) != 0u;
#pragma unroll 1
        for (int c = half * (MMA_N / 2); c < (half + 1) * (MMA_N / 2); c += 32) {
          const int n0 = nb * MMA_N + c;
          if (n0 >= N || !any_real) break;  // warp-uniform
          uint32_t a[32];
          ptx::tmem_ld_32cols(taddr + c, a);
          ptx::tmem_ld_wait();
          float o[32];
          // column c + j of the warp's 128 is held by lane (c - 128 half + j) / 4
          const int lc0 = (c - half * (MMA_N / 2)) >> 2;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float b = __shfl_sync(0xffffffffu, pf_b[j & 3], lc0 + (j >> 2));
            float sc = 1.f;
            if constexpr (F8) sc = __shfl_sync(0xffffffffu, pf_s[j & 3], lc0 + (j >> 2)) * pf_sa;
            o[j] = (__uint_as_float(a[acc_pos(j)]) * sc + b) * wgt;
          }
          if constexpr (EPI == Epi::SortedF32) {
            // Stage the warp's 32x32 fp32 block in the 128-byte-swizzled layout
            // the tensor map expects (row = lane, 16-byte chunk j stored at
            // chunk j ^ (row & 7): conflict-free), then one TMA store.
            if (lane == 0) ptx::bulk_wait_read0();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(stage_buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                  make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(tmO, stage_buf, n0, row0 + q * 32);
              ptx::bulk_commit();
            }
          } else if constexpr (EPI == Epi::SortedF16) {
            // The row's 32 values as fp16 times 2^-e, e >= 0 the least with
            // max |o| * 2^-e < 2^15 (finite in fp16); e in o_exp, chunk-major
            // so that the warp's 32 rows write 32 consecutive bytes.  Staged
            // as a 32 x 32 fp16 block in the 64-byte-swizzled layout of the
            // tensor map (row = lane, 16-byte chunk j at j ^ ((row >> 1) & 3)),
            // then one TMA store; the warp's staging area holds two such
            // blocks, used in turn, so a chunk is staged while the previous
            // chunk's store still reads the other.
            float m = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(o[j]));
            const int ex = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127;
            const int e = max(0, ex - 14);
            const float sc = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
            uint32_t hw[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const __half2 h2 = __floats2half2_rn(o[2 * j] * sc, o[2 * j + 1] * sc);
              hw[j] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            uint8_t* blk = stage_buf + ((c >> 5) & 1) * 2048;
            if (lane == 0) ptx::bulk_wait_read1();  // the store that used blk is done reading
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(blk + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(hw[4 * j], hw[4 * j + 1], hw[4 * j + 2], hw[4 * j + 3]);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(tmO, blk, n0, row0 + q * 32);
              ptx::bulk_commit();
            }
            P.o_exp[static_cast<int64_t>(n0 >> 5) * P.o_exp_ld + row0 + q * 32 + lane] =
                static_cast<uint8_t>(e);
          } else if constexpr (EPI == Epi::AtomicF32) {
            if (valid) {
              float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(P.out) +
                                                    static_cast<int64_t>(entry / P.div) * N + n0);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                if (n0 + v * 4 < N)
                  atomicAdd(d + v, make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]));
            }
          } else if constexpr (EPI == Epi::DenseF32) {
            if (valid) {
              float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(P.out) +
                                                    static_cast<int64_t>(entry) * N + n0);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                if (n0 + v * 4 < N)
                  d[v] = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
            }
          } else {
            if (valid) {
              bf16* d = reinterpret_cast<bf16*>(P.out) + static_cast<int64_t>(entry) * N + n0;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                if (n0 + v * 8 < N) {
                  uint4 pk;
                  pk.x = pack_bf16x2(o[8 * v], o[8 * v + 1]);
                  pk.y = pack_bf16x2(o[8 * v + 2], o[8 * v + 3]);
                  pk.z = pack_bf16x2(o[8 * v + 4], o[8 * v + 5]);
                  pk.w = pack_bf16x2(o[8 * v + 6], o[8 * v + 7]);
                  *reinterpret_cast<uint4*>(d + v * 8) = pk;
                }
              }
            }
          }
        }
      }
      if (!released) release_acc(acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  if constexpr (EPI == Epi::SortedF32 || EPI == Epi::SortedF16 || EPI == Epi::SwiGLU) {
    if (warp >= EPI0 && lane == 0) ptx::bulk_wait0();  // TMA stores done before smem is released
  }
  __syncwarp();  // lane-0-only roles rejoin their warp before the aligned barriers
  if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
  if (*reinterpret_cast<volatile int32_t*>(&ctl.abort)) {
    // Give TMA copies and MMAs still in flight time to land before the
    // shared memory and TMEM of this CTA are released.
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
  }
  if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
  if (dyn && threadIdx.x == 0 && (CG == 1 || rank == 0)) {
    // the last claiming CTA to finish zeroes the counters for the next
    // launch (every claim precedes its CTA's count)
    __threadfence();
    if (atomicAdd(P.sched + 1, 1) == units - 1) {
      atomicExch(P.sched, 0);
      atomicExch(P.sched + 1, 0);
    }
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (CG == 2) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <Epi EPI, bool F8>
__global__ void __launch_bounds__(NTHREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO, const KParams P) {
  pdl_begin();
  gemm_body<EPI, 1, F8>(&tmA, &tmB, &tmO, nullptr, nullptr, P);
}

template <Epi EPI, bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmO, const KParams P) {
  pdl_begin();
  gemm_body<EPI, 2, F8>(&tmA, &tmB, &tmO, nullptr, nullptr, P);
}

// bf16 GEMM1 with the gather fused: the gather warp after the epilogue
// warps copies A's rows from the token rows.
constexpr int GA_THREADS = NTHREADS + 32;
template <Epi EPI>
__global__ void __launch_bounds__(GA_THREADS, 1)
    grouped_gemm_ga_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmO, const KParams P) {
  pdl_begin();
  gemm_body<EPI, 1, false, Wq::None, false, true>(&tmA, &tmB, &tmO, nullptr, nullptr, P);
}
template <Epi EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GA_THREADS, 1)
    grouped_gemm_ga_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                                const __grid_constant__ CUtensorMap tmB,
                                const __grid_constant__ CUtensorMap tmO, const KParams P) {
  pdl_begin();
  gemm_body<EPI, 2, false, Wq::None, false, true>(&tmA, &tmB, &tmO, nullptr, nullptr, P);
}

// FP8 with block-wise (128 x 128) weight scales and per-(row, 128-group)
// activation scales: single-CTA tiles, one accumulation per K stage.
constexpr int BS_THREADS = 64 + 16 * 32;  // producer + MMA + 16 epilogue warps

template <Epi EPI>
__global__ void __launch_bounds__(BS_THREADS, 1)
    grouped_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const KParams P) {
  pdl_begin();
  gemm_body<EPI, 1, true, Wq::None, true>(&tmA, &tmB, &tmB, nullptr, nullptr, P);
}

// bf16 A x weight-only quantised B (converted to bf16 in shared memory).
template <Epi EPI, Wq WQ>
__global__ void __launch_bounds__(cta_threads<WQ>(), 1)
    grouped_gemm_wq_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmO,
                           const __grid_constant__ CUtensorMap tmS,
                           const __grid_constant__ CUtensorMap tmZ, const KParams P) {
  pdl_begin();
  gemm_body<EPI, 1, false, WQ>(&tmA, &tmB, &tmO, &tmS, &tmZ, P);
}

// The same on CTA pairs: each CTA converts its 128 of the tile's 256
// columns, the even CTA's MMA reads both.
template <Epi EPI, Wq WQ>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(cta_threads<WQ>(), 1)
    grouped_gemm_wq_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                                const __grid_constant__ CUtensorMap tmB,
                                const __grid_constant__ CUtensorMap tmO,
                                const __grid_constant__ CUtensorMap tmS,
                                const __grid_constant__ CUtensorMap tmZ, const KParams P) {
  pdl_begin();
  gemm_body<EPI, 2, false, WQ>(&tmA, &tmB, &tmO, &tmS, &tmZ, P);
}

// ------------------------------------------------------------------ host --
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 tensor map with 128-byte swizzle.  dims/strides innermost first;
// strides are in bytes for dims 1..rank-1.
moe_status_t make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box,
                      CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  const CUresult r = fn(m, dtype, rank, const_cast<void*>(base), gd,
                        gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", r);
  return MOE_OK;
}

// CTA pairs (cta_group::2) pay off when the GEMM is tensor-bound and experts
// have several 128-row blocks each.  Measured on GB300: pairs win for the
// Mixtral- and Qwen-shape layers (~1000 rows per expert) and lose for the
// HBM-bound DeepSeek-shape layer (256 rows per expert), so the automatic
// choice asks for at least four row blocks per expert on average.
bool use_pairs(const GroupedGemmArgs& a) {
  const int mode = gemm_tile_mode();
  if (mode == 1) return false;
  if (mode == 2) return a.num_sms >= 2;
  return a.rows_hint >= static_cast<int64_t>(4 * BM) * a.E && a.num_sms >= 2;
}

// Kernel parameters common to every grouped GEMM launch.
template <Epi EPI>
KParams base_params(const GroupedGemmArgs& a, int NB) {
  KParams P{};
  P.bias = a.bias;
  P.out = a.out;
  P.offsets = a.offsets;
  P.row_index = a.row_index;
  P.row_weight = a.row_weight;
  P.error_word = a.error_word;
  P.E = a.E;
  P.N = a.N;
  P.K = a.K;
  P.NB = NB;
  P.sentinel = a.sentinel;
  P.div = a.div > 0 ? a.div : 1;
  P.a_rows = a.a_rows;
  P.sched = a.sched;
  P.dense_rows = (EPI == Epi::DenseF32) ? static_cast<int32_t>(a.sentinel) : 0;
  P.gemm1_row_weight = a.gemm1_row_weight;
  P.a_scale = a.a_scale;
  P.w_scale = a.w_scale;
  P.w_scale_per_channel = a.w_scale_per_channel;
  P.row_amax = a.row_amax;
  P.z_group_scale = a.z_group_scale;
  P.w_scale_ld = (EPI == Epi::SwiGLU) ? 2 * a.N : a.N;
  P.o_exp = a.o_exp;
  P.o_exp_ld = a.cap;
  return P;
}

// Tensor maps of A (sorted rows, K-major) and B (expert weights, MN-major)
// and the number of column blocks, shared by the grouped GEMM launchers.
// `pairs`: the tiles are split over CTA pairs (each CTA loads half of B's
// chunks).  Where the columns split into whole 128-byte chunks, B is viewed
// with the chunk as a dimension of its own, so that one copy per stage loads
// all of a CTA's chunks (*one_box = 1); otherwise, or where `allow_one_box`
// is false, one copy per chunk.  Measured on GB300, the single copy took the
// bf16 layers 1-3 % faster (Mixtral-shape prefill 1.85 -> 1.83 ms,
// DeepSeek-V3 M = 8192 6.24 -> 6.08 ms) and the block-scaled FP8 GEMMs ~1 %
// slower, so those keep one copy per chunk.
template <Epi EPI, bool F8>
moe_status_t make_ab_maps(const GroupedGemmArgs& a, bool pairs, CUtensorMap* tmA,
                          CUtensorMap* tmB, int* NB, int32_t* one_box,
                          bool allow_one_box = true) {
  using G1 = Geo<1, F8>;
  const CUtensorMapDataType dt =
      F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t eb = F8 ? 1 : 2;  // bytes per operand element
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.cap)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.K) * eb};
    const uint32_t box[2] = {G1::BKE, BM};
    if (moe_status_t st = make_map(tmA, a.a, 2, dims, strides, box, dt)) return st;
  }
  const uint64_t N = static_cast<uint64_t>(a.N), K = static_cast<uint64_t>(a.K),
                 E = static_cast<uint64_t>(a.E);
  const uint64_t chunks = allow_one_box ? N / G1::CW : 0;  // whole 128-byte column chunks
  if constexpr (EPI == Epi::SwiGLU) {
    *NB = ceil_div(a.N, MMA_N / 2);
    // w13 [E, K, 2, N]: a box is a CTA's chunks of the gate half, then (one
    // CTA) the same chunks of the up half
    const uint32_t per_half = G1::CHUNKS / 2;
    if (N % G1::CW == 0 && chunks >= per_half) {
      const uint64_t dims[5] = {G1::CW, K, chunks, 2, E};
      const uint64_t strides[4] = {2 * N * eb, G1::CW * eb, N * eb, 2 * N * eb * K};
      const uint32_t box[5] = {G1::CW, G1::BKE, per_half, pairs ? 1u : 2u, 1};
      *one_box = 1;
      return make_map(tmB, a.w, 5, dims, strides, box, dt);
    }
    // (n, half, k, e)
    const uint64_t dims[4] = {N, 2, K, E};
    const uint64_t strides[3] = {N * eb, N * 2 * eb, N * 2 * eb * K};
    const uint32_t box[4] = {G1::CW, 1, G1::BKE, 1};
    *one_box = 0;
    return make_map(tmB, a.w, 4, dims, strides, box, dt);
  } else {
    *NB = ceil_div(a.N, MMA_N);
    // w2 [E, K, N]
    const uint32_t per_cta = pairs ? G1::CHUNKS / 2 : G1::CHUNKS;
    if (N % G1::CW == 0 && chunks >= per_cta) {
      const uint64_t dims[4] = {G1::CW, K, chunks, E};
      const uint64_t strides[3] = {N * eb, G1::CW * eb, N * eb * K};
      const uint32_t box[4] = {G1::CW, G1::BKE, per_cta, 1};
      *one_box = 1;
      return make_map(tmB, a.w, 4, dims, strides, box, dt);
    }
    // (n, k, e)
    const uint64_t dims[3] = {N, K, E};
    const uint64_t strides[2] = {N * eb, N * eb * K};
    const uint32_t box[3] = {G1::CW, G1::BKE, 1};
    *one_box = 0;
    return make_map(tmB, a.w, 3, dims, strides, box, dt);
  }
}

template <Epi EPI, bool F8 = false>
moe_status_t launch_gemm(const GroupedGemmArgs& a, const char* name, cudaStream_t s) {
  using G1 = Geo<1, F8>;
  using G2 = Geo<2, F8>;
  static PerDevice attrs;
  if (attrs.get([](int*) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, F8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(G1::SMEM));
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<EPI, F8>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(G2::SMEM));
        return e;
      }) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute(%s): %s", name,
                     cudaGetErrorString(cudaGetLastError()));
  const bool pairs = EPI != Epi::DenseF32 && use_pairs(a);
  CUtensorMap tmA, tmB;
  int NB;
  int32_t one_box;
  if (moe_status_t st = make_ab_maps<EPI, F8>(a, pairs, &tmA, &tmB, &NB, &one_box)) return st;
  CUtensorMap tmO;
  if constexpr (EPI == Epi::SortedF16) {
    // fp16 [cap, N] rows, 32 x 32 boxes, 64-byte swizzle (matches staging)
    if (a.o_exp == nullptr) return set_error(MOE_ERR_INVALID_ARG, "%s: no exponent array", name);
    const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.cap)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * 2};
    const uint32_t box[2] = {32, 32};
    if (moe_status_t st = make_map(&tmO, a.out, 2, dims, strides, box,
                                   CU_TENSOR_MAP_DATA_TYPE_FLOAT16, CU_TENSOR_MAP_SWIZZLE_64B))
      return st;
  } else if constexpr (EPI == Epi::SortedF32) {
    // fp32 [cap, N] output, 32 x 32 boxes, 128-byte swizzle (matches staging)
    const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.cap)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * 4};
    const uint32_t box[2] = {32, 32};
    if (moe_status_t st = make_map(&tmO, a.out, 2, dims, strides, box,
                                   CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return st;
  } else if constexpr (EPI == Epi::SwiGLU) {
    // z bf16 [cap, N]: one epilogue warp's 32 rows x 64 columns per store,
    // 128-byte swizzle (matches staging)
    const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.cap)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * 2};
    const uint32_t box[2] = {64, 32};
    if (moe_status_t st = make_map(&tmO, a.out, 2, dims, strides, box,
                                   CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
      return st;
  } else {
    tmO = tmA;  // unused
  }
  KParams P = base_params<EPI>(a, NB);
  P.b_one_box = one_box;
  // grouped operands are padded to whole 128-row blocks; the dense one is not
  const int64_t max_blocks = (EPI == Epi::DenseF32) ? ceil_div<int64_t>(a.cap, BM) : a.cap / BM;
  if (max_blocks <= 0) return MOE_OK;
  if (pairs) {
    // Persistent pairs: no more clusters than can be resident at once (the
    // tiles are split statically among them).
    static PerDevice clusters_per_device;
    int resident = a.num_sms / 2;
    clusters_per_device.get(
        [&](int* v) {
          cudaLaunchConfig_t cfg = {};
          cfg.gridDim = dim3(2 * (a.num_sms / 2));
          cfg.blockDim = dim3(NTHREADS);
          cfg.dynamicSmemBytes = G2::SMEM;
          int n = 0;
          if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<EPI, F8>, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = a.num_sms / 2;
          }
          *v = std::min(n, a.num_sms / 2);
          return cudaSuccess;
        },
        &resident);
    // at most blocks/2 + E/2 pair tiles per column block
    const int64_t max_pairs = (max_blocks / 2 + (a.E + 1) / 2 + 1) * NB;
    const unsigned clusters = static_cast<unsigned>(std::min<int64_t>(max_pairs, resident));
    // the dynamic schedule pays where weight tiles are large (K >= 3072:
    // Mixtral-shape gemm1 DRAM reads 1.99-2.55 -> 1.95 GB, FP8 gemm1 ~620 ->
    // 594 us); with short K (Qwen-MoE shape, K = 2048 / 768) it measured
    // 1-2.5 % slower, so those keep the static round-robin
    if (a.K < 3072) P.sched = nullptr;
    prof_before(name, s);
    launch_kernel(grouped_gemm_pair_kernel<EPI, F8>, 2 * clusters, NTHREADS, G2::SMEM, s, tmA, tmB,
                  tmO, P);
    prof_after(name, s);
    return check_launch(name);
  }
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(max_blocks * NB, a.num_sms));
  // single-CTA tiles keep the static schedule: with two row blocks per weight
  // tile (the shapes that take them) adjacent units already share it, and the
  // dynamic one measured slower there (DeepSeek-V3 M=8192 layer 5.8-6.0 ->
  // 6.0-6.3 ms)
  P.sched = nullptr;
  prof_before(name, s);
  launch_kernel(grouped_gemm_kernel<EPI, F8>, grid, NTHREADS, G1::SMEM, s, tmA, tmB, tmO, P);
  prof_after(name, s);
  return check_launch(name);
}

// bf16 GEMM1 with the gather fused (a.a_rows: the token rows); tiles as
// launch_gemm's.  tmA is built on a.a but not read.
moe_status_t launch_gemm1_ga(const GroupedGemmArgs& a, const char* name, cudaStream_t s) {
  constexpr Epi EPI = Epi::SwiGLU;
  using G1 = Geo<1, false>;
  using G2 = Geo<2, false>;
  static PerDevice attrs;
  if (attrs.get([](int*) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_ga_kernel<EPI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(G1::SMEM));
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(grouped_gemm_ga_pair_kernel<EPI>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(G2::SMEM));
        return e;
      }) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute(%s): %s", name,
                     cudaGetErrorString(cudaGetLastError()));
  if ((a.K & 7) != 0 || (reinterpret_cast<uintptr_t>(a.a_rows) & 15u) != 0)
    return set_error(MOE_ERR_INVALID_ARG, "%s: token rows must be 16-byte aligned rows", name);
  const bool pairs = use_pairs(a);
  CUtensorMap tmA, tmB, tmO;
  int NB;
  int32_t one_box;
  if (moe_status_t st = make_ab_maps<EPI, false>(a, pairs, &tmA, &tmB, &NB, &one_box)) return st;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.cap)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * 2};
    const uint32_t box[2] = {64, 32};
    if (moe_status_t st = make_map(&tmO, a.out, 2, dims, strides, box,
                                   CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
      return st;
  }
  KParams P = base_params<EPI>(a, NB);
  P.b_one_box = one_box;
  const int64_t max_blocks = a.cap / BM;
  if (max_blocks <= 0) return MOE_OK;
  if (pairs) {
    // persistent pairs: no more clusters than can be resident at once
    static PerDevice clusters_per_device;
    int resident = a.num_sms / 2;
    clusters_per_device.get([&](int* v) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (a.num_sms / 2));
      cfg.blockDim = dim3(GA_THREADS);
      cfg.dynamicSmemBytes = G2::SMEM;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_ga_pair_kernel<EPI>, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = a.num_sms / 2;
      }
      *v = std::min(n, a.num_sms / 2);
      return cudaSuccess;
    }, &resident);
    const int64_t max_pairs = (max_blocks / 2 + (a.E + 1) / 2 + 1) * NB;
    const unsigned clusters = static_cast<unsigned>(std::min<int64_t>(max_pairs, resident));
    prof_before(name, s);
    launch_kernel(grouped_gemm_ga_pair_kernel<EPI>, 2 * clusters, GA_THREADS, G2::SMEM, s, tmA, tmB,
                  tmO, P);
    prof_after(name, s);
    return check_launch(name);
  }
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(max_blocks * NB, a.num_sms));
  prof_before(name, s);
  launch_kernel(grouped_gemm_ga_kernel<EPI>, grid, GA_THREADS, G1::SMEM, s, tmA, tmB, tmO, P);
  prof_after(name, s);
  return check_launch(name);
}

// FP8 with block scales: single-CTA 128 x 256 tiles, 128 K per stage.
template <Epi EPI>
moe_status_t launch_gemm_bs(const GroupedGemmArgs& a, const char* name, cudaStream_t s) {
  using G = Geo<1, true>;
  static PerDevice attrs;
  if (attrs.get([&](int*) {
        return cudaFuncSetAttribute(grouped_gemm_bs_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(G::SMEM));
      }) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute(%s): %s", name,
                     cudaGetErrorString(cudaGetLastError()));
  if (EPI == Epi::SwiGLU && (a.z_group_scale == nullptr || a.N % 128 != 0))
    return set_error(MOE_ERR_INVALID_ARG, "%s: z group scales and N %% 128 == 0 required", name);
  CUtensorMap tmA, tmB;
  int NB;
  int32_t one_box;
  if (moe_status_t st = make_ab_maps<EPI, true>(a, false, &tmA, &tmB, &NB, &one_box, false)) return st;
  KParams P = base_params<EPI>(a, NB);
  P.b_one_box = one_box;
  P.w_scale_ld = ((EPI == Epi::SwiGLU) ? 2 * a.N : a.N) / 128;  // weight blocks per K block
  P.bs_a_ld = a.cap;
  const int64_t max_blocks = a.cap / BM;
  if (max_blocks <= 0) return MOE_OK;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(max_blocks * NB, a.num_sms));
  prof_before(name, s);
  launch_kernel(grouped_gemm_bs_kernel<EPI>, grid, BS_THREADS, G::SMEM, s, tmA, tmB, P);
  prof_after(name, s);
  return check_launch(name);
}

// bf16 A x weight-only quantised B.  Single-CTA 128 x 256 tiles; the codes,
// scales and zero points travel by TMA without swizzle into the raw ring.
template <Epi EPI, Wq WQ, int CG>
moe_status_t launch_gemm_wq_cg(const GroupedGemmArgs& a, const char* name, cudaStream_t s) {
  using G = Geo<CG, false, WQ>;
  using R = std::conditional_t<CG == 2, WqRing<WQ, 1, 128>,
                               WqRing<WQ, EPI == Epi::SwiGLU ? 2 : 1>>;
  constexpr int NREG = (CG == 1 && EPI == Epi::SwiGLU) ? 2 : 1;
  auto kernel = CG == 2 ? grouped_gemm_wq_pair_kernel<EPI, WQ> : grouped_gemm_wq_kernel<EPI, WQ>;
  static PerDevice attrs;
  if (attrs.get([&](int*) {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(G::SMEM));
      }) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute(%s): %s", name,
                     cudaGetErrorString(cudaGetLastError()));
  const int gsize = a.wq_group;
  const uint32_t gbox = gsize == 32 ? 2u : 1u;  // group rows per 64-row stage
  const uint64_t KG = static_cast<uint64_t>(a.K / gsize);
  const uint64_t E = static_cast<uint64_t>(a.E), K = static_cast<uint64_t>(a.K);
  const uint64_t N = static_cast<uint64_t>(a.N);
  const uint64_t sb = R::F::SCALE_BYTES;
  const CUtensorMapDataType sdt =
      sb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE;
  CUtensorMap tmA, tmB, tmS, tmZ, tmO;
  {
    const uint64_t dims[2] = {K, static_cast<uint64_t>(a.cap)};
    const uint64_t strides[1] = {K * 2};
    const uint32_t box[2] = {G::BKE, BM};
    if (moe_status_t st = make_map(&tmA, a.a, 2, dims, strides, box)) return st;
  }
  const uint64_t nbytes = N * R::F::CODE_BITS / 8;  // bytes of one K row of codes (per half)
  int NB;
  if constexpr (EPI == Epi::SwiGLU) {
    // [E, K, 2, N'] viewed (n', half, k, e) for codes, (n, half, g, e) for params
    const uint64_t cd[4] = {nbytes, 2, K, E};
    const uint64_t cs[3] = {nbytes, 2 * nbytes, 2 * nbytes * K};
    const uint32_t cbx[4] = {static_cast<uint32_t>(R::ROW_BYTES), 1, static_cast<uint32_t>(G::BKE), 1};
    if (moe_status_t st = make_map(&tmB, a.w, 4, cd, cs, cbx, u8, none)) return st;
    const uint64_t pd[4] = {N, 2, KG, E};
    const uint64_t ps[3] = {N * sb, 2 * N * sb, 2 * N * sb * KG};
    const uint32_t pbx[4] = {static_cast<uint32_t>(R::RCOLS), 1, gbox, 1};
    if (moe_status_t st = make_map(&tmS, a.wq_scale, 4, pd, ps, pbx, sdt, none)) return st;
    tmZ = tmS;
    if (a.wq_zero != nullptr) {
      const uint64_t zs[3] = {N, 2 * N, 2 * N * KG};
      if (moe_status_t st = make_map(&tmZ, a.wq_zero, 4, pd, zs, pbx, u8, none)) return st;
    }
    NB = ceil_div(a.N, MMA_N / 2);
    // z bf16 [cap, N], one epilogue warp's 32 x 64 block per store
    const uint64_t od[2] = {N, static_cast<uint64_t>(a.cap)};
    const uint64_t os[1] = {N * 2};
    const uint32_t obx[2] = {64, 32};
    if (moe_status_t st = make_map(&tmO, a.out, 2, od, os, obx)) return st;
  } else {
    const uint64_t cd[3] = {nbytes, K, E};
    const uint64_t cs[2] = {nbytes, nbytes * K};
    const uint32_t cbx[3] = {static_cast<uint32_t>(R::ROW_BYTES), static_cast<uint32_t>(G::BKE), 1};
    if (moe_status_t st = make_map(&tmB, a.w, 3, cd, cs, cbx, u8, none)) return st;
    const uint64_t pd[3] = {N, KG, E};
    const uint64_t ps[2] = {N * sb, N * sb * KG};
    const uint32_t pbx[3] = {static_cast<uint32_t>(R::RCOLS), gbox, 1};
    if (moe_status_t st = make_map(&tmS, a.wq_scale, 3, pd, ps, pbx, sdt, none)) return st;
    tmZ = tmS;
    if (a.wq_zero != nullptr) {
      const uint64_t zs[2] = {N, N * KG};
      if (moe_status_t st = make_map(&tmZ, a.wq_zero, 3, pd, zs, pbx, u8, none)) return st;
    }
    NB = ceil_div(a.N, MMA_N);
    // fp32 [cap, N] output, 32 x 32 boxes (matches staging)
    const uint64_t od[2] = {N, static_cast<uint64_t>(a.cap)};
    const uint64_t os[1] = {N * 4};
    const uint32_t obx[2] = {32, 32};
    if (moe_status_t st = make_map(&tmO, a.out, 2, od, os, obx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return st;
  }
  KParams P = base_params<EPI>(a, NB);
  P.wq_G = gsize;
  P.wq_gbox = static_cast<int32_t>(gbox);
  P.wq_has_zero = a.wq_zero != nullptr ? 1 : 0;
  P.wq_raw_tx = NREG * (R::CODES + static_cast<int32_t>(R::RCOLS * sb * gbox) +
                        (a.wq_zero != nullptr ? static_cast<int32_t>(R::RCOLS * gbox) : 0));
  const int64_t max_blocks = a.cap / BM;
  if (max_blocks <= 0) return MOE_OK;
  unsigned grid;
  if constexpr (CG == 2) {
    // persistent pairs: no more clusters than can be resident at once
    static PerDevice clusters_per_device;
    int resident = a.num_sms / 2;
    clusters_per_device.get(
        [&](int* v) {
          cudaLaunchConfig_t cfg = {};
          cfg.gridDim = dim3(2 * (a.num_sms / 2));
          cfg.blockDim = dim3(cta_threads<WQ>());
          cfg.dynamicSmemBytes = G::SMEM;
          int n = 0;
          if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = a.num_sms / 2;
          }
          *v = std::min(n, a.num_sms / 2);
          return cudaSuccess;
        },
        &resident);
    const int64_t max_pairs = (max_blocks / 2 + (a.E + 1) / 2 + 1) * NB;
    grid = 2 * static_cast<unsigned>(std::min<int64_t>(max_pairs, resident));
  } else {
    grid = static_cast<unsigned>(std::min<int64_t>(max_blocks * NB, a.num_sms));
  }
  prof_before(name, s);
  launch_kernel(kernel, grid, cta_threads<WQ>(), G::SMEM, s, tmA, tmB, tmO, tmS, tmZ, P);
  prof_after(name, s);
  return check_launch(name);
}

template <Epi EPI, Wq WQ>
moe_status_t launch_gemm_wq(const GroupedGemmArgs& a, const char* name, cudaStream_t s) {
  if (use_pairs(a)) return launch_gemm_wq_cg<EPI, WQ, 2>(a, name, s);
  return launch_gemm_wq_cg<EPI, WQ, 1>(a, name, s);
}

}  // namespace

moe_status_t encode_tensor_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                               const uint64_t* strides, const uint32_t* box,
                               CUtensorMapDataType dtype, CUtensorMapSwizzle swz) {
  return make_map(m, base, rank, dims, strides, box, dtype, swz);
}

moe_status_t launch_wait_timeout_probe(int32_t* err, uint32_t limit_us, cudaStream_t s) {
  prof_before("wait_timeout_probe", s);
  launch_kernel(wait_timeout_probe_kernel, 1, 32, 0, s, err,
                static_cast<uint64_t>(limit_us) * 1000ull);
  prof_after("wait_timeout_probe", s);
  return check_launch("wait_timeout_probe");
}

moe_status_t launch_gemm1_swiglu(const GroupedGemmArgs& a, cudaStream_t s) {
  if (a.a_rows != nullptr) return launch_gemm1_ga(a, "gemm1_swiglu", s);
  return launch_gemm<Epi::SwiGLU>(a, "gemm1_swiglu", s);
}
moe_status_t launch_gemm2_sorted_f32(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm<Epi::SortedF32>(a, "gemm2_sorted", s);
}
moe_status_t launch_gemm2_sorted_f16(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm<Epi::SortedF16>(a, "gemm2_sorted", s);
}
moe_status_t launch_gemm2_sorted_f16_fp8(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm<Epi::SortedF16, true>(a, "gemm2_sorted_fp8", s);
}
moe_status_t launch_gemm2_atomic_f32(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm<Epi::AtomicF32>(a, "gemm2_atomic", s);
}
moe_status_t launch_gemm1_swiglu_fp8(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm<Epi::SwiGLU, true>(a, "gemm1_swiglu_fp8", s);
}
moe_status_t launch_gemm2_sorted_fp8(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm<Epi::SortedF32, true>(a, "gemm2_sorted_fp8", s);
}
moe_status_t launch_dense_f32(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm<Epi::DenseF32>(a, "router_logits", s);
}
moe_status_t launch_gemm2_rows_bf16(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm<Epi::RowsBF16>(a, "gemm2_rows_bf16", s);
}

}  // namespace gbmoe

namespace gbmoe {

moe_status_t launch_gemm1_swiglu_fp8_block(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm_bs<Epi::SwiGLU>(a, "gemm1_swiglu_fp8_block", s);
}
moe_status_t launch_gemm2_sorted_fp8_block(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_gemm_bs<Epi::SortedF32>(a, "gemm2_sorted_fp8_block", s);
}

moe_status_t launch_gemm1_swiglu_wq(const GroupedGemmArgs& a, cudaStream_t s) {
  switch (a.wq_format) {
    case 0: return launch_gemm_wq<Epi::SwiGLU, Wq::Int4>(a, "gemm1_swiglu_int4", s);
    case 1: return launch_gemm_wq<Epi::SwiGLU, Wq::Int8>(a, "gemm1_swiglu_int8", s);
    case 2: return launch_gemm_wq<Epi::SwiGLU, Wq::Mxfp4>(a, "gemm1_swiglu_mxfp4", s);
    case 3: return launch_gemm_wq<Epi::SwiGLU, Wq::Mxfp6e3m2>(a, "gemm1_swiglu_mxfp6", s);
    case 4: return launch_gemm_wq<Epi::SwiGLU, Wq::Mxfp6e2m3>(a, "gemm1_swiglu_mxfp6", s);
    default: return set_error(MOE_ERR_INVALID_ARG, "weight format %d", a.wq_format);
  }
}

moe_status_t launch_gemm2_sorted_wq(const GroupedGemmArgs& a, cudaStream_t s) {
  switch (a.wq_format) {
    case 0: return launch_gemm_wq<Epi::SortedF32, Wq::Int4>(a, "gemm2_sorted_int4", s);
    case 1: return launch_gemm_wq<Epi::SortedF32, Wq::Int8>(a, "gemm2_sorted_int8", s);
    case 2: return launch_gemm_wq<Epi::SortedF32, Wq::Mxfp4>(a, "gemm2_sorted_mxfp4", s);
    case 3: return launch_gemm_wq<Epi::SortedF32, Wq::Mxfp6e3m2>(a, "gemm2_sorted_mxfp6", s);
    case 4: return launch_gemm_wq<Epi::SortedF32, Wq::Mxfp6e2m3>(a, "gemm2_sorted_mxfp6", s);
    default: return set_error(MOE_ERR_INVALID_ARG, "weight format %d", a.wq_format);
  }
}

}  // namespace gbmoe
