// The whole layer for small calls in two kernels.  At a few hundred routed
// items each launch of the general path (align plan, GEMM1 with its gather,
// GEMM2, weight-and-reduce) costs a few microseconds of its own, more than
// the work; here the plan, the gather and the reduce are folded into the two
// GEMMs.
//
// "fused_moe.py 分析", the fused_moe kernel and the reduce after it: routed
// item r (token t = r / k, expert e = topk_ids[r], weight a_r) gives
//   z_r = SiLU(x_t W13[e][:, gate] + b13_gate) * (x_t W13[e][:, up] + b13_up)
//   y_t = sum over t's items of a_r (z_r W2[e] + b2[e])
// with z rounded to bf16 and the sum over a token's items in fp32, as the
// general path computes them.
//   small_gemm1_kernel: one CTA per (expert, 64 z columns).  It finds its
//     expert's items in topk_ids itself, in item order, gathers their token
//     rows and the 64 gate and 64 up weight columns one 64-row K stage at a
//     time (16-byte asynchronous copies, up to four stages in flight), multiplies
//     with mma.sync (32 items per pass as M) and writes z [item, I] in bf16.
//     The CTAs also zero the fp32 token accumulator; CTA 0 zeroes the error
//     word and the completion counters, then records ids outside [0, E)
//     (those items contribute nothing).
//   small_gemm2_kernel: one CTA per (expert, 64 output columns), the same
//     way over z and W2 (up to seven stages in flight); each item's weighted
//     row is added into the token accumulator with fp32 atomics, and of the
//     E CTAs of a 64-column block the last to finish writes that block of y
//     in bf16.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace gbmoe {
namespace {

constexpr int kSThreads = 128;           // four warps
constexpr int kSKC = 64;                 // K rows per stage
// stages in the shared-memory ring: the whole 64-column weight slice of a
// GEMM1 CTA with H = 256 (4 stages) and of a GEMM2 CTA with I = 512 (8) is
// in flight at once; both rings take 110 KB
constexpr int kSStages1 = 5;
constexpr int kSStages2 = 8;
constexpr int kSRows = 32;               // items per pass (two 16-row MMA tiles)
constexpr int kSMaxItems = 256;          // routed items of a call
constexpr int kSXStride = kSKC + 8;      // bf16 per activation row in shared memory (padded)
constexpr int64_t kSMaxAccum = 1 << 18;  // token accumulator elements (M * H) of a call

struct SmallParams {
  const bf16* x;           // hidden [M, H]
  const bf16* w13;         // [E, H, 2I]
  const bf16* w2;          // [E, I, H]
  const bf16* b13;         // [E, 2I] or null
  const bf16* b2;          // [E, H] or null
  const int32_t* ids;      // topk_ids [R]
  const float* weights;    // topk_weights [R]
  bf16* z;                 // [R, I]
  float* acc;              // token accumulator [M, H]
  int32_t* counter;        // [H / 64]: CTAs of small_gemm2 done per 64 output columns
  int32_t* error_word;     // 32 words, zeroed by small_gemm1's CTA 0
  bf16* y;                 // [M, H]
  int32_t M, H, I, E, k, R;
};

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(ptx::smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(ptx::smem_u32(p)));
}
// d += a (16x16, row-major) * b (16x8, column-major); bf16 in, fp32 out.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_s(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// The items routed to expert e, in item order, into s_items; returns their
// count.  Ids outside [0, E) match no expert.
__device__ int expert_items(const int32_t* __restrict__ ids, int R, int e, int32_t* s_items,
                            int32_t* s_warp) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int count = 0;
  for (int base = 0; base < R; base += kSThreads) {
    const int r = base + tid;
    const bool hit = r < R && __ldg(ids + r) == e;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, hit);
    if (lane == 0) s_warp[warp] = __popc(m);
    __syncthreads();
    int before = count, total = 0;
#pragma unroll
    for (int w = 0; w < kSThreads / 32; ++w) {
      const int v = s_warp[w];
      if (w < warp) before += v;
      total += v;
    }
    if (hit) s_items[before + __popc(m & ((1u << lane) - 1u))] = r;
    __syncthreads();
    count += total;
  }
  return count;
}

// One pass of 32 items (rows row0..row0+31 of s_items, n_items in all) over
// the CTA's NCOL weight columns and all of K:
//   acc[m][t][*] = C[row0 + 16 m + (g, g + 8), warp * NCOL / 4 + 8 t + (2c, 2c + 1)]
//   C[row, n] = sum_k A[row, k] * W[k, col(n)]
// A's row for item i is x_rows[a_row(i) * lda], a_row(i) = i / k for token
// rows (GEMM1) or i (GEMM2).  Column n of the CTA in shared memory: NCOL = 64
// -> col0 + n; NCOL = 128 -> 16-column groups alternating gate (col0 + ...)
// and up (col_up + ...), so that warp w holds gate and up of the same 16
// columns (group 2w gate, 2w + 1 up).
template <int NCOL, int STAGES>
__device__ __forceinline__ void small_pass(const bf16* __restrict__ x_rows, int64_t lda,
                                           bool token_rows, int k_top, const int32_t* s_items,
                                           int row0, int n_items, int K,
                                           const bf16* __restrict__ w_e, int64_t w_ld, int col0,
                                           int col_up, uint8_t* smem, float (&acc)[2][NCOL / 32][4]) {
  constexpr int WSTRIDE = NCOL + 8;            // bf16 per weight row in shared memory (padded)
  constexpr int XB = kSRows * kSXStride * 2;   // activation bytes of a stage
  constexpr int WB = kSKC * WSTRIDE * 2;       // weight bytes of a stage
  constexpr int NT = NCOL / 32;                // n8 tiles per warp
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][t][i] = 0.0f;
  const int KS = K / kSKC;
  auto load_stage = [&](int ks, int buf) {
    uint8_t* xs = smem + buf * (XB + WB);
    uint8_t* wsm = xs + XB;
    const int k0 = ks * kSKC;
    // 32 rows x 64 k: 256 16-byte chunks, two per thread
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = i * kSThreads + tid;
      const int r = idx >> 3, ch = idx & 7;
      const int row = row0 + r;
      const bool live = row < n_items;
      const int item = live ? s_items[row] : 0;
      const int64_t arow = token_rows ? item / k_top : item;
      const bf16* src = x_rows + arow * lda + k0 + ch * 8;
      ptx::cp_async_16(xs + (r * kSXStride + ch * 8) * 2, live ? src : x_rows, live ? 16u : 0u);
    }
    // 64 k rows x NCOL columns
    constexpr int CH_PER_ROW = NCOL / 8;
#pragma unroll
    for (int i = 0; i < kSKC * CH_PER_ROW / kSThreads; ++i) {
      const int idx = i * kSThreads + tid;
      const int kr = idx / CH_PER_ROW, n = (idx % CH_PER_ROW) * 8;
      int col;
      if constexpr (NCOL == 128) {
        const int gi = n >> 4;
        col = ((gi & 1) ? col_up : col0) + 16 * (gi >> 1) + (n & 15);
      } else {
        col = col0 + n;
      }
      ptx::cp_async_16(wsm + (kr * WSTRIDE + n) * 2, w_e + static_cast<int64_t>(k0 + kr) * w_ld + col,
                       16u);
    }
  };
  // one commit group per stage (empty past the last), so that stage ks has
  // landed once at most STAGES - 2 groups are pending
#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) {
    if (st < KS) load_stage(st, st);
    ptx::cp_async_commit();
  }
  for (int ks = 0; ks < KS; ++ks) {
    const int buf = ks % STAGES;
    ptx::cp_async_wait<STAGES - 2>();
    __syncthreads();  // stage ks visible to all; stage ks - 1's buffer free
    if (ks + STAGES - 1 < KS) load_stage(ks + STAGES - 1, (ks + STAGES - 1) % STAGES);
    ptx::cp_async_commit();
    const uint8_t* xs = smem + buf * (XB + WB);
    const uint8_t* wsm = xs + XB;
#pragma unroll
    for (int kk = 0; kk < kSKC / 16; ++kk) {
      uint32_t a[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int r = 16 * m + (lane & 15), kc = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(a[m][0], a[m][1], a[m][2], a[m][3], xs + (r * kSXStride + kc) * 2);
      }
#pragma unroll
      for (int t2 = 0; t2 < NT; t2 += 2) {
        // k rows kk*16 + (lane & 15) of n8 tiles t2 (lanes 0-15) and t2 + 1
        const int kr = kk * 16 + (lane & 15);
        const int n = warp * (NCOL / 4) + t2 * 8 + (lane >> 4) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, wsm + (kr * WSTRIDE + n) * 2);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          mma16816(acc[m][t2], a[m], b0, b1);
          mma16816(acc[m][t2 + 1], a[m], b2, b3);
        }
      }
    }
  }
  ptx::cp_async_wait<0>();
  __syncthreads();  // the next pass refills the ring
}

template <int NCOL, int STAGES>
constexpr int small_smem() {
  return STAGES * (kSRows * kSXStride * 2 + kSKC * (NCOL + 8) * 2);
}

__global__ void __launch_bounds__(kSThreads)
    small_gemm1_kernel(const SmallParams P) {
  pdl_begin();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int32_t s_items[kSMaxItems];
  __shared__ int32_t s_warp[kSThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  {
    // the token accumulator, a slice per CTA
    const int64_t total = static_cast<int64_t>(P.M) * P.H;
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t b0 = per * blockIdx.x, b1 = min(total, b0 + per);
    for (int64_t i = b0 + tid; i < b1; i += kSThreads) P.acc[i] = 0.0f;
    if (blockIdx.x == 0) {
      if (tid < 32) P.error_word[tid] = 0;
      for (int i = tid; i < P.H / 64; i += kSThreads) P.counter[i] = 0;
      bool bad = false;
      for (int r = tid; r < P.R; r += kSThreads) {
        const int32_t id = __ldg(P.ids + r);
        bad |= id < 0 || id >= P.E;
      }
      if (__syncthreads_or(bad) && tid == 0) record_error(P.error_word, MOE_ERR_BAD_EXPERT_ID);
    }
  }
  const int ncb = P.I / 64;
  const int e = blockIdx.x / ncb, cb = blockIdx.x % ncb;
  const int n = expert_items(P.ids, P.R, e, s_items, s_warp);
  if (n == 0) return;
  const bf16* w_e = P.w13 + static_cast<int64_t>(e) * P.H * 2 * P.I;
  // warp w: z columns zc0 + 16 w + 8 t + 2c (+1), t = 0, 1
  const int zc0 = cb * 64;
  float bg[2][2], bu[2][2];
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int zc = zc0 + 16 * warp + 8 * t + 2 * c + h;
      bg[t][h] = P.b13 != nullptr ? __bfloat162float(P.b13[static_cast<int64_t>(e) * 2 * P.I + zc]) : 0.f;
      bu[t][h] = P.b13 != nullptr
                     ? __bfloat162float(P.b13[static_cast<int64_t>(e) * 2 * P.I + P.I + zc])
                     : 0.f;
    }
  for (int row0 = 0; row0 < n; row0 += kSRows) {
    float acc[2][4][4];
    small_pass<128, kSStages1>(P.x, P.H, true, P.k, s_items, row0, n, P.H, w_e, 2 * static_cast<int64_t>(P.I),
                    zc0, P.I + zc0, smem, acc);
    // tiles 0, 1: gate; 2, 3: up of the same columns
#pragma unroll
    for (int m = 0; m < 2; ++m) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = row0 + 16 * m + g + 8 * hr;
        if (row >= n) continue;
        bf16* zr = P.z + static_cast<int64_t>(s_items[row]) * P.I + zc0 + 16 * warp + 2 * c;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float z0 = silu_s(acc[m][t][2 * hr] + bg[t][0]) * (acc[m][t + 2][2 * hr] + bu[t][0]);
          const float z1 =
              silu_s(acc[m][t][2 * hr + 1] + bg[t][1]) * (acc[m][t + 2][2 * hr + 1] + bu[t][1]);
          *reinterpret_cast<__nv_bfloat162*>(zr + 8 * t) = __floats2bfloat162_rn(z0, z1);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kSThreads)
    small_gemm2_kernel(const SmallParams P) {
  pdl_begin();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int32_t s_items[kSMaxItems];
  __shared__ int32_t s_warp[kSThreads / 32];
  __shared__ int32_t s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int ncb = P.H / 64;
  const int e = blockIdx.x / ncb, cb = blockIdx.x % ncb;
  const int oc0 = cb * 64;
  const int n = expert_items(P.ids, P.R, e, s_items, s_warp);
  if (n > 0) {
    const bf16* w_e = P.w2 + static_cast<int64_t>(e) * P.I * P.H;
    // warp w: output columns oc0 + 16 w + 8 t + 2c (+1), t = 0, 1
    float bb[2][2];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        bb[t][h] = P.b2 != nullptr
                       ? __bfloat162float(P.b2[static_cast<int64_t>(e) * P.H + oc0 + 16 * warp + 8 * t + 2 * c + h])
                       : 0.f;
    for (int row0 = 0; row0 < n; row0 += kSRows) {
      float acc[2][2][4];
      small_pass<64, kSStages2>(P.z, P.I, false, P.k, s_items, row0, n, P.I, w_e, P.H, oc0, 0, smem, acc);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int row = row0 + 16 * m + g + 8 * hr;
          if (row >= n) continue;
          const int item = s_items[row];
          const float wgt = __ldg(P.weights + item);
          float* dst = P.acc + static_cast<int64_t>(item / P.k) * P.H + oc0 + 16 * warp + 2 * c;
#pragma unroll
          for (int t = 0; t < 2; ++t)
            atomicAdd(reinterpret_cast<float2*>(dst + 8 * t),
                      make_float2((acc[m][t][2 * hr] + bb[t][0]) * wgt,
                                  (acc[m][t][2 * hr + 1] + bb[t][1]) * wgt));
        }
      }
    }
  }
  // of the E CTAs of this 64-column block the last to finish writes the
  // block of y (every CTA's additions precede its count)
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(P.counter + cb, 1) == P.E - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // rows r0 + 8 u + tid / 16, columns oc0 + 4 (tid % 16) .. + 3: eight
  // rows' loads in flight per thread
  const int cq = oc0 + 4 * (tid & 15);
  for (int r0 = 0; r0 < P.M; r0 += 64) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int row = r0 + 8 * u + (tid >> 4);
      if (row < P.M)
        v[u] = __ldcg(reinterpret_cast<const float4*>(P.acc + static_cast<int64_t>(row) * P.H + cq));
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int row = r0 + 8 * u + (tid >> 4);
      if (row < P.M) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v[u].x, v[u].y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v[u].z, v[u].w);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(P.y + static_cast<int64_t>(row) * P.H + cq) = o;
      }
    }
  }
}

}  // namespace

bool small_forward_applies(int64_t M, int32_t H, int32_t I, int32_t E, int32_t top_k) {
  const int64_t R = M * top_k;
  if (M < 1 || R > kSMaxItems || H % 64 != 0 || I % 64 != 0) return false;
  if (M * H > kSMaxAccum) return false;
  // weights small enough that the layer is bound by launches, not by streaming them
  return static_cast<int64_t>(E) * H * I * 6 <= (int64_t{64} << 20);
}

moe_status_t launch_small_forward(const SmallArgs& a, cudaStream_t s) {
  SmallParams P{};
  P.x = a.x;
  P.w13 = a.w13;
  P.w2 = a.w2;
  P.b13 = a.b13;
  P.b2 = a.b2;
  P.ids = a.ids;
  P.weights = a.weights;
  P.z = a.z;
  P.acc = a.acc;
  P.counter = a.counter;
  P.error_word = a.error_word;
  P.y = a.y;
  P.M = static_cast<int32_t>(a.M);
  P.H = a.H;
  P.I = a.I;
  P.E = a.E;
  P.k = a.k;
  P.R = static_cast<int32_t>(a.M * a.k);
  constexpr int S1 = small_smem<128, kSStages1>(), S2 = small_smem<64, kSStages2>();
  static_assert(S1 <= 227 * 1024 - 2048 && S2 <= 227 * 1024 - 2048, "shared memory per CTA");
  static PerDevice attrs;
  if (attrs.get([&](int*) {
        cudaError_t e1 = cudaFuncSetAttribute(small_gemm1_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, S1);
        if (e1 != cudaSuccess) return e1;
        return cudaFuncSetAttribute(small_gemm2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    S2);
      }) != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute(small_gemm): %s",
                     cudaGetErrorString(cudaGetLastError()));
  prof_before("small_gemm1", s);
  launch_kernel(small_gemm1_kernel, static_cast<unsigned>(a.E * (a.I / 64)), kSThreads, S1, s, P);
  prof_after("small_gemm1", s);
  if (moe_status_t st = check_launch("small_gemm1")) return st;
  prof_before("small_gemm2", s);
  launch_kernel(small_gemm2_kernel, static_cast<unsigned>(a.E * (a.H / 64)), kSThreads, S2, s, P);
  prof_after("small_gemm2", s);
  return check_launch("small_gemm2");
}

}  // namespace gbmoe
