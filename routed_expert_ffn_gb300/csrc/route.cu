// Top-k gating (CS349D lecture 8 notes, section 1.2 "MoE 层的结构"): one warp
// per token; k rounds of warp-shuffle argmax over the per-lane candidates,
// ties to the lower expert index, then the variant's gate weights.
//
// Two entry kernels share that step:
//  - topk_gating_kernel sums the tensor-core router's K-split partial logits
//    (router_tc.cu) in a fixed order, so the logits are deterministic;
//  - router_small_kernel serves small batches (T <= kSmallRouteT) in one
//    launch: one CTA per expert computes its fp32 logits for every token
//    (lane-strided products per warp, a shuffle tree, then the eight warps'
//    partials in order: a blocked, deterministic sum), and the last CTA to
//    finish gates every token.
#include <float.h>

#include "gating.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

// Router K-split partials loaded per batch by the gating kernel (measured:
// 8 takes 2-5 us off the route at T = 1024..2048 against 4).
#ifndef MOE_TOPK_BATCH
#define MOE_TOPK_BATCH 8
#endif
constexpr int kTopkSplitBatch = MOE_TOPK_BATCH;

// NV = logits per lane (E <= 32 * NV).
template <int NV>
__global__ void __launch_bounds__(256) topk_gating_kernel(
    const float *__restrict__ partial, int splits, const float *__restrict__ sel_bias, int T,
    int E, int k, int gating, float *__restrict__ logits, int32_t *__restrict__ ids,
    float *__restrict__ wout, float *__restrict__ gap) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;  // whole warp leaves together

  float s[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) s[i] = 0.f;
  // sum the router's K-split partials in split order; kTopkSplitBatch
  // splits' loads are issued together
  constexpr int kB = kTopkSplitBatch;
  for (int z0 = 0; z0 < splits; z0 += kB) {
    float p[NV][kB];
#pragma unroll
    for (int u = 0; u < kB; ++u)
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        p[i][u] = (e < E && z0 + u < splits) ? partial[((size_t)(z0 + u) * T + t) * E + e] : 0.f;
      }
#pragma unroll
    for (int u = 0; u < kB; ++u)
#pragma unroll
      for (int i = 0; i < NV; ++i) s[i] += p[i][u];
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (e < E) logits[(size_t)t * E + e] = s[i];
  }
  select_and_gate<NV>(s, lane, t, E, k, gating, sel_bias, ids, wout, gap);
}

// Small batches: one CTA per expert e; its 8 warps each take an eighth of H
// for all T <= kSmallRouteT tokens, the eight partial sums are added in warp
// order, then the last CTA to finish gates every token.
template <int NV>
__global__ void __launch_bounds__(256) router_small_kernel(
    const __nv_bfloat16 *__restrict__ x, const float *__restrict__ w_router,
    const float *__restrict__ sel_bias, int T, int H, int E, int k, int gating,
    float *__restrict__ logits, int32_t *__restrict__ ids, float *__restrict__ wout,
    float *__restrict__ gap, uint32_t *__restrict__ counter) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_last;
  __shared__ float red[8][kSmallRouteT];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x;
  {
    float acc[kSmallRouteT];
#pragma unroll
    for (int t = 0; t < kSmallRouteT; ++t) acc[t] = 0.f;
    const int hs = H / 8;  // a multiple of 8 (H % 64 == 0)
    const int h1 = (warp + 1) * hs;
    const float *wr = w_router + (size_t)e * H;
#pragma unroll 4
    for (int h = warp * hs + lane * 4; h < h1; h += 128) {
      const float4 wv = *reinterpret_cast<const float4 *>(wr + h);
#pragma unroll
      for (int t = 0; t < kSmallRouteT; ++t) {
        if (t < T) {
          const uint2 raw = *reinterpret_cast<const uint2 *>(x + (size_t)t * H + h);
          const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw);
          const float2 a = __bfloat1622float2(p[0]), b = __bfloat1622float2(p[1]);
          float v = acc[t];
          v = fmaf(wv.x, a.x, v);
          v = fmaf(wv.y, a.y, v);
          v = fmaf(wv.z, b.x, v);
          v = fmaf(wv.w, b.y, v);
          acc[t] = v;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kSmallRouteT; ++t) {
      if (t < T) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) red[warp][t] = v;
      }
    }
    __syncthreads();
    if (warp == 0 && lane < T) {
      float v = 0.f;
#pragma unroll
      for (int ww = 0; ww < 8; ++ww) v += red[ww][lane];
      logits[(size_t)lane * E + e] = v;
    }
  }
  // the last CTA to finish gates every token
  __threadfence();
  __syncthreads();
  // atomicInc wraps to 0 at the last arrival, so the counter is 0 again
  // after every call
  if (threadIdx.x == 0) s_last = (atomicInc(counter, gridDim.x - 1) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = warp; t < T; t += blockDim.x >> 5) {
    float s[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int ee = lane + 32 * i;
      s[i] = (ee < E) ? __ldcg(logits + (size_t)t * E + ee) : 0.f;
    }
    select_and_gate<NV>(s, lane, t, E, k, gating, sel_bias, ids, wout, gap);
  }
}

template <int NV>
cudaError_t launch_gating_nv(const float *partial, int splits, const float *sel_bias, int T, int E,
                             int k, int gating, float *logits, int32_t *ids, float *w, float *gap,
                             cudaStream_t s) {
  return launch_pdl(topk_gating_kernel<NV>, dim3((T + 7) / 8), dim3(256), 0, s, partial, splits,
                    sel_bias, T, E, k, gating, logits, ids, w, gap);
}

template <int NV>
cudaError_t launch_small_nv(const __nv_bfloat16 *x, const float *w_router, const float *sel_bias,
                            int T, int H, int E, int k, int gating, float *logits, int32_t *ids,
                            float *w, float *gap, uint32_t *counter, cudaStream_t s) {
  return launch_pdl(router_small_kernel<NV>, dim3(E), dim3(256), 0, s, x, w_router,
                    sel_bias, T, H, E, k, gating, logits, ids, w, gap, counter);
}

}  // namespace

cudaError_t launch_topk_gating(const float *partial, int splits, const float *sel_bias, int T,
                               int E, int k, int gating, float *logits, int32_t *ids, float *w,
                               float *gap, cudaStream_t s) {
  const int nv = (E + 31) / 32;
  if (nv <= 1)
    return launch_gating_nv<1>(partial, splits, sel_bias, T, E, k, gating, logits, ids, w, gap, s);
  if (nv <= 2)
    return launch_gating_nv<2>(partial, splits, sel_bias, T, E, k, gating, logits, ids, w, gap, s);
  if (nv <= 4)
    return launch_gating_nv<4>(partial, splits, sel_bias, T, E, k, gating, logits, ids, w, gap, s);
  if (nv <= 8)
    return launch_gating_nv<8>(partial, splits, sel_bias, T, E, k, gating, logits, ids, w, gap, s);
  return launch_gating_nv<16>(partial, splits, sel_bias, T, E, k, gating, logits, ids, w, gap, s);
}

cudaError_t launch_route_small(const __nv_bfloat16 *x, const float *w_router,
                               const float *sel_bias, int T, int H, int E, int k, int gating,
                               float *logits, int32_t *ids, float *w, float *gap,
                               uint32_t *counter, cudaStream_t s) {
  const int nv = (E + 31) / 32;
  if (nv <= 1)
    return launch_small_nv<1>(x, w_router, sel_bias, T, H, E, k, gating, logits, ids, w, gap,
                              counter, s);
  if (nv <= 2)
    return launch_small_nv<2>(x, w_router, sel_bias, T, H, E, k, gating, logits, ids, w, gap,
                              counter, s);
  if (nv <= 4)
    return launch_small_nv<4>(x, w_router, sel_bias, T, H, E, k, gating, logits, ids, w, gap,
                              counter, s);
  if (nv <= 8)
    return launch_small_nv<8>(x, w_router, sel_bias, T, H, E, k, gating, logits, ids, w, gap,
                              counter, s);
  return launch_small_nv<16>(x, w_router, sel_bias, T, H, E, k, gating, logits, ids, w, gap,
                             counter, s);
}

}  // namespace moe
