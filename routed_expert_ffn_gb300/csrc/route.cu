// Top-k gating (CS349D lecture 8 notes, section 1.2 "MoE 层的结构"): one warp
// per token; k rounds of warp-shuffle argmax over the per-lane candidates,
// ties to the lower expert index, then the variant's gate weights.  The
// router's K-split partial logits (router_tc.cu) are summed here in a fixed
// order, so the logits are deterministic.
#include <float.h>

#include "moe_internal.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

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

  float s[NV], key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) s[i] = 0.f;
  // sum the router's K-split partials in split order; four splits' loads are
  // issued together
  for (int z0 = 0; z0 < splits; z0 += 4) {
    float p[NV][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        p[i][u] = (e < E && z0 + u < splits) ? partial[((size_t)(z0 + u) * T + t) * E + e] : 0.f;
      }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int i = 0; i < NV; ++i) s[i] += p[i][u];
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    key[i] = -FLT_MAX;
    if (e < E) {
      logits[(size_t)t * E + e] = s[i];
      key[i] = (gating == MOE_GATE_SIGMOID_BIAS_RENORM) ? sigmoidf_(s[i]) + sel_bias[e] : s[i];
    }
  }

  uint32_t taken = 0;
  int my_id = 0;
  float my_s = 0.f, kth_key = 0.f, next_key = 0.f;
  const int rounds = (k < E) ? k + 1 : k;
  for (int j = 0; j < rounds; ++j) {
    float bk = -FLT_MAX;
    int bi = 0x7fffffff;
    float bs = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u)) {
        if (key[i] > bk || (key[i] == bk && e < bi)) {
          bk = key[i];
          bi = e;
          bs = s[i];
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      if (ok > bk || (ok == bk && oi < bi)) {
        bk = ok;
        bi = oi;
        bs = os;
      }
    }
    if (j < k) {
      if (lane == j) {
        my_id = bi;
        my_s = bs;
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      kth_key = bk;
    } else {
      next_key = bk;
    }
  }

  float wv = 0.f;
  const bool mine = lane < k;
  if (gating == MOE_GATE_TOPK_SOFTMAX) {
    const float m = __shfl_sync(0xffffffffu, my_s, 0);  // slot 0 holds the largest kept logit
    const float ev = mine ? expf(my_s - m) : 0.f;
    wv = ev / warp_sum(ev);
  } else if (gating == MOE_GATE_SOFTMAX_TOPK || gating == MOE_GATE_SOFTMAX_TOPK_RENORM) {
    const float m = __shfl_sync(0xffffffffu, my_s, 0);  // largest logit of all E
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (lane + 32 * i < E) part += expf(s[i] - m);
    const float zsum = warp_sum(part);
    const float p = mine ? expf(my_s - m) / zsum : 0.f;
    wv = (gating == MOE_GATE_SOFTMAX_TOPK) ? p : p / warp_sum(p);
  } else {
    const float a = mine ? sigmoidf_(my_s) : 0.f;
    wv = a / warp_sum(a);
  }
  if (mine) {
    ids[(size_t)t * k + lane] = my_id;
    wout[(size_t)t * k + lane] = wv;
  }
  if (gap != nullptr && lane == 0) gap[t] = (k < E) ? kth_key - next_key : 0.f;
}

}  // namespace

cudaError_t launch_topk_gating(const float *partial, int splits, const float *sel_bias, int T,
                               int E, int k, int gating, float *logits, int32_t *ids, float *w,
                               float *gap, cudaStream_t s) {
  const int blocks = (T + 7) / 8;
  const int nv = (E + 31) / 32;
  cudaError_t e;
  if (nv <= 1)
    e = launch_pdl(topk_gating_kernel<1>, dim3(blocks), dim3(256), 0, s, partial, splits, sel_bias, T, E, k, gating, logits,
                                                 ids, w, gap);
  else if (nv <= 2)
    e = launch_pdl(topk_gating_kernel<2>, dim3(blocks), dim3(256), 0, s, partial, splits, sel_bias, T, E, k, gating, logits,
                                                 ids, w, gap);
  else if (nv <= 4)
    e = launch_pdl(topk_gating_kernel<4>, dim3(blocks), dim3(256), 0, s, partial, splits, sel_bias, T, E, k, gating, logits,
                                                 ids, w, gap);
  else if (nv <= 8)
    e = launch_pdl(topk_gating_kernel<8>, dim3(blocks), dim3(256), 0, s, partial, splits, sel_bias, T, E, k, gating, logits,
                                                 ids, w, gap);
  else
    e = launch_pdl(topk_gating_kernel<16>, dim3(blocks), dim3(256), 0, s, partial, splits, sel_bias, T, E, k, gating,
                                                  logits, ids, w, gap);
  return e;
}

}  // namespace moe
