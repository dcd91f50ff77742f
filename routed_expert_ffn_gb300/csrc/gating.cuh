// Top-k selection and gate weights of one token, shared by the gating
// kernels (route.cu) and the persistent decode layer (decode_layer.cu):
// k rounds of warp-shuffle argmax over the per-lane candidates, ties to the
// lower expert index, then the variant's gate weights (CS349D lecture 8
// notes, section 1.2 "MoE 层的结构").
#pragma once

#include <float.h>

#include "moe_internal.cuh"

namespace moe {

static __device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

static __device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// Order-preserving map of a float selection key to an unsigned integer (a
// larger key gives a larger integer; -0 and +0 map alike); 0 lies below the
// image of every finite key and marks an expert out of the running.
static __device__ __forceinline__ uint32_t key_bits(float f) {
  const uint32_t b = __float_as_uint(f + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Selection and gate weights of token t from its fp32 logits s (lane holds
// experts lane, lane+32, ...).  The whole warp calls it.  Each of the k
// (+1, for the boundary gap) rounds takes the largest remaining key: every
// lane's best candidate, then a warp max-reduction of the keys and a
// min-reduction of the indices holding that key (ties to the lower expert
// index), both single redux.sync instructions.
template <int NV>
static __device__ __forceinline__ void select_and_gate(const float (&s)[NV], int lane, int t, int E, int k,
                                                int gating, const float *__restrict__ sel_bias,
                                                int32_t *__restrict__ ids, float *__restrict__ wout,
                                                float *__restrict__ gap) {
  float key[NV];
  uint32_t kb[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    key[i] = -FLT_MAX;
    kb[i] = 0u;
    if (e < E) {
      key[i] = (gating == MOE_GATE_SIGMOID_BIAS_RENORM) ? sigmoidf_(s[i]) + sel_bias[e] : s[i];
      kb[i] = key_bits(key[i]);
    }
  }

  int my_id = 0;
  float my_s = 0.f, kth_key = 0.f, next_key = 0.f;
  const int rounds = (k < E) ? k + 1 : k;
  for (int j = 0; j < rounds; ++j) {
    uint32_t lb = 0u;
    int li = 0x7fffffff;
    float ls = 0.f, lk = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      if (kb[i] > lb) {  // strict: the lowest index among equal keys
        lb = kb[i];
        li = lane + 32 * i;
        ls = s[i];
        lk = key[i];
      }
    }
    const uint32_t gb = __reduce_max_sync(0xffffffffu, lb);
    const int bi = __reduce_min_sync(0xffffffffu, lb == gb ? li : 0x7fffffff);
    const int owner = bi & 31;  // its best candidate is the winner
    const float bs = __shfl_sync(0xffffffffu, ls, owner);
    const float bk = __shfl_sync(0xffffffffu, lk, owner);
    if (j < k) {
      if (lane == j) {
        my_id = bi;
        my_s = bs;
      }
      if (lane == owner) {
#pragma unroll
        for (int i = 0; i < NV; ++i)
          if (lane + 32 * i == bi) kb[i] = 0u;
      }
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

}  // namespace moe
