// Routing: router logits -> top-k expert ids and weights, one warp per token.
//
// Follows the "MindIE-SD Fused MoE" page (parameter table and routing
// section: softmax / sigmoid scores, optional grouped selection with
// group_count / k_group / group_select_mode, renormalize, routed scaling)
// and "FlagGems fused_moe.py analysis" section 1.1 (S_t = TopK(p_t, k)).
//
// Selection is the exact TopK of the scores p.  Softmax (within a row) and
// sigmoid are strictly increasing in the logit, so the kernel orders by the
// fp32 logits themselves: the decision is exact and ties go to the lower
// expert id.  Group mode 0 (max score) is likewise ordered by each group's
// largest logit; group mode 1 (sum of the two largest scores) compares fp32
// sums of the scores.  Weights are computed in fp32.
#include <cfloat>

#include "common.cuh"

namespace gbmoe {
namespace {

constexpr int kWarpsPerBlock = 4;

struct Cand {
  float key;  // ordering key (logit or group score)
  int idx;    // expert or group id; lower wins ties
  float val;  // carried payload (score p)
};

__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float k2 = __shfl_xor_sync(0xffffffffu, c.key, off);
    int i2 = __shfl_xor_sync(0xffffffffu, c.idx, off);
    float v2 = __shfl_xor_sync(0xffffffffu, c.val, off);
    if (better(k2, i2, c.key, c.idx)) {
      c.key = k2;
      c.idx = i2;
      c.val = v2;
    }
  }
  return c;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Order-preserving map of a float to an unsigned key (larger float ->
// larger key); never 0 for a float, so 0 can mean "no candidate".
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = (f == 0.0f) ? 0u : __float_as_uint(f);  // -0 and +0 compare equal
  const uint32_t k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return k == 0u ? 1u : k;
}

// Best of a lane's slots: largest key, ties to the lower slot (= lower
// expert id, since expert = slot * 32 + lane).
template <int EPL>
__device__ __forceinline__ void local_best(const uint32_t (&key)[EPL], const float (&p)[EPL],
                                           uint32_t& bk, int& bi, float& bp) {
  bk = key[0];
  bi = 0;
  bp = p[0];
#pragma unroll
  for (int i = 1; i < EPL; ++i) {
    if (key[i] > bk) {
      bk = key[i];
      bi = i;
      bp = p[i];
    }
  }
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }

// EPL = experts per lane (expert e = i * 32 + lane); T = fp32 or bf16 logits
// (bf16 is widened exactly to fp32 before anything else).
template <int EPL, typename T>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_kernel(const T* __restrict__ logits, int64_t M, int E, int top_k, int method,
                 int renormalize, int k_group, int group_count, int group_select_mode,
                 float scale, float* __restrict__ out_w, int32_t* __restrict__ out_ids) {
  pdl_begin();
  extern __shared__ float route_smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
  if (t >= M) return;

  const T* row = logits + t * E;
  float l[EPL], p[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = i * 32 + lane;
    l[i] = (e < E) ? to_f32(row[e]) : -FLT_MAX;
  }

  // ---- scores ----
  if (method == MOE_ROUTE_SOFTMAX) {
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i * 32 + lane < E) m = fmaxf(m, l[i]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      p[i] = (i * 32 + lane < E) ? expf(l[i] - m) : 0.f;
      s += p[i];
    }
    s = warp_sum(s);
    const float inv = 1.0f / s;
#pragma unroll
    for (int i = 0; i < EPL; ++i) p[i] *= inv;
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) p[i] = 1.0f / (1.0f + expf(-l[i]));
  }

  // ---- grouped pre-selection ----
  uint32_t allowed = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (i * 32 + lane < E) allowed |= 1u << i;

  if (group_count > 1) {
    const int gs = E / group_count;
    float* sl = route_smem + warp * (2 * E + 2 * group_count);
    float* sp = sl + E;
    float* gkey = sp + E;
    float* gsel = gkey + group_count;  // 1.0f once the group is kept
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E) {
        sl[e] = l[i];
        sp[e] = p[i];
      }
    }
    __syncwarp();
    for (int g = lane; g < group_count; g += 32) {
      float key;
      if (group_select_mode == 0) {
        float mx = -FLT_MAX;
        for (int j = 0; j < gs; ++j) mx = fmaxf(mx, sl[g * gs + j]);
        key = mx;
      } else {
        float b1 = -FLT_MAX, b2 = -FLT_MAX;
        for (int j = 0; j < gs; ++j) {
          const float v = sp[g * gs + j];
          if (v > b1) {
            b2 = b1;
            b1 = v;
          } else if (v > b2) {
            b2 = v;
          }
        }
        key = b1 + b2;
      }
      gkey[g] = key;
      gsel[g] = 0.f;
    }
    __syncwarp();
    for (int r = 0; r < k_group; ++r) {
      Cand c{-INFINITY, 0x7fffffff, 0.f};
      for (int g = lane; g < group_count; g += 32)
        if (gsel[g] == 0.f && better(gkey[g], g, c.key, c.idx)) c = Cand{gkey[g], g, 0.f};
      c = warp_best(c);
      if (lane == 0) gsel[c.idx] = 1.f;
      __syncwarp();
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E && gsel[e / gs] == 0.f) allowed &= ~(1u << i);
    }
  }

  // ---- top-k by logit, ties to the lower expert id ----
  // Each lane keeps its best remaining candidate; a round is one warp-wide
  // max over order-preserving integer keys of the logits (REDUX), a ballot
  // for ties, and -- only when two lanes tie -- a min over their expert ids.
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) key[i] = ((allowed >> i) & 1u) ? order_key(l[i]) : 0u;
  uint32_t bk;
  int bi;
  float bp;
  local_best<EPL>(key, p, bk, bi, bp);
  float wsum = 0.f;
  int my_id0 = 0, my_id1 = 0;
  float my_p0 = 0.f, my_p1 = 0.f;
  for (int j = 0; j < top_k; ++j) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, bk);
    const unsigned holders = __ballot_sync(0xffffffffu, bk == mx);
    int win_lane = __ffs(holders) - 1;
    int win_e = __shfl_sync(0xffffffffu, bi * 32 + lane, win_lane);
    if (__popc(holders) > 1) {  // equal logits in several lanes: lowest expert id wins
      win_e = static_cast<int>(__reduce_min_sync(
          0xffffffffu, bk == mx ? static_cast<unsigned>(bi * 32 + lane) : 0xffffffffu));
      win_lane = win_e & 31;
    }
    const float win_p = __shfl_sync(0xffffffffu, bp, win_lane);
    if (lane == win_lane) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == bi) key[i] = 0u;
      local_best<EPL>(key, p, bk, bi, bp);
    }
    wsum += win_p;
    if (j == lane) {
      my_id0 = win_e;
      my_p0 = win_p;
    } else if (j == lane + 32) {
      my_id1 = win_e;
      my_p1 = win_p;
    }
  }
  const bool norm = (method == MOE_ROUTE_SIGMOID) || renormalize;
  const float f = norm ? scale / wsum : scale;
  if (lane < top_k) {
    out_ids[t * top_k + lane] = my_id0;
    out_w[t * top_k + lane] = norm ? (my_p0 / wsum) * scale : my_p0 * f;
  }
  if (lane + 32 < top_k) {
    out_ids[t * top_k + lane + 32] = my_id1;
    out_w[t * top_k + lane + 32] = norm ? (my_p1 / wsum) * scale : my_p1 * f;
  }
}

template <int EPL>
moe_status_t launch_route_t(const RouteArgs& a, cudaStream_t s) {
  const int64_t blocks = ceil_div<int64_t>(a.M, kWarpsPerBlock);
  size_t smem = 0;
  if (a.group_count > 1)
    smem = static_cast<size_t>(kWarpsPerBlock) * (2 * a.E + 2 * a.group_count) * sizeof(float);
  prof_before("route", s);
  if (a.logits_bf16)
    launch_kernel(route_kernel<EPL, bf16>, static_cast<unsigned>(blocks), kWarpsPerBlock * 32, smem,
                  s, static_cast<const bf16*>(a.logits), a.M, a.E, a.top_k, a.method, a.renormalize,
                  a.k_group, a.group_count, a.group_select_mode, a.scale, a.weights, a.ids);
  else
    launch_kernel(route_kernel<EPL, float>, static_cast<unsigned>(blocks), kWarpsPerBlock * 32,
                  smem, s, static_cast<const float*>(a.logits), a.M, a.E, a.top_k, a.method,
                  a.renormalize, a.k_group, a.group_count, a.group_select_mode, a.scale, a.weights,
                  a.ids);
  prof_after("route", s);
  return check_launch("route");
}

}  // namespace

moe_status_t launch_route(const RouteArgs& a, cudaStream_t s) {
  const int epl = ceil_div(a.E, 32);
  if (epl <= 1) return launch_route_t<1>(a, s);
  if (epl <= 2) return launch_route_t<2>(a, s);
  if (epl <= 4) return launch_route_t<4>(a, s);
  if (epl <= 8) return launch_route_t<8>(a, s);
  if (epl <= 16) return launch_route_t<16>(a, s);
  return launch_route_t<32>(a, s);
}

}  // namespace gbmoe
