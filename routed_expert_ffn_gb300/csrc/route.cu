// Router and top-k gating.
//
// Router s = W_r x ("MoE推理优化全景指南", section "从 Dense FFN 到专家集合"):
// an fp32 GEMM [T,H] x [E,H]^T on the CUDA cores, register-tiled 64 tokens x
// 64 experts per CTA, split over H when there are too few tiles to fill the
// GPU (the splits are summed in a fixed order by the gating kernel, so the
// result is deterministic).
//
// Top-k gating (CS349D lecture 8 notes, section 1.2 "MoE 层的结构"): one warp
// per token; k rounds of warp-shuffle argmax over the per-lane candidates,
// ties to the lower expert index, then the variant's gate weights.
#include <float.h>

#include "moe_internal.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16 *__restrict__ x,
                                                            const float *__restrict__ wr, int T,
                                                            int H, int E, int split_len,
                                                            float *__restrict__ partial) {
  __shared__ __align__(16) float xs[kRouteBK][kRouteTT + 4];
  __shared__ __align__(16) float ws[kRouteBK][kRouteTE + 4];
  const int e0 = blockIdx.x * kRouteTE;
  const int t0 = blockIdx.y * kRouteTT;
  const int z = blockIdx.z;
  const int kbeg = z * split_len;
  const int kend = min(H, kbeg + split_len);
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int ld_row = tid >> 2, ld_k = (tid & 3) * 8;  // 64 rows x 32 k, 8 elements per thread

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int kk = kbeg; kk < kend; kk += kRouteBK) {
    {
      const int t = t0 + ld_row;
      float v[8];
      if (t < T) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(x + (size_t)t * H + kk + ld_k);
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(p[i]);
          v[2 * i] = f.x;
          v[2 * i + 1] = f.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[ld_k + i][ld_row] = v[i];
    }
    {
      const int e = e0 + ld_row;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (e < E) {
        const float4 *p = reinterpret_cast<const float4 *>(wr + (size_t)e * H + kk + ld_k);
        a = p[0];
        b = p[1];
      }
      ws[ld_k + 0][ld_row] = a.x;
      ws[ld_k + 1][ld_row] = a.y;
      ws[ld_k + 2][ld_row] = a.z;
      ws[ld_k + 3][ld_row] = a.w;
      ws[ld_k + 4][ld_row] = b.x;
      ws[ld_k + 5][ld_row] = b.y;
      ws[ld_k + 6][ld_row] = b.z;
      ws[ld_k + 7][ld_row] = b.w;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRouteBK; ++k) {
      const float4 a = *reinterpret_cast<const float4 *>(&xs[k][ty * 4]);
      const float4 b = *reinterpret_cast<const float4 *>(&ws[k][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) partial[((size_t)z * T + t) * E + e] = acc[i][j];
    }
  }
}

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
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;  // whole warp leaves together

  float s[NV], key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    s[i] = 0.f;
    key[i] = -FLT_MAX;
    if (e < E) {
      float v = 0.f;
      for (int zz = 0; zz < splits; ++zz) v += partial[((size_t)zz * T + t) * E + e];
      s[i] = v;
      logits[(size_t)t * E + e] = v;
      key[i] = (gating == MOE_GATE_SIGMOID_BIAS_RENORM) ? sigmoidf_(v) + sel_bias[e] : v;
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

int route_splits(int T, int E, int H) {
  const int tiles = ((T + kRouteTT - 1) / kRouteTT) * ((E + kRouteTE - 1) / kRouteTE);
  int want = (512 + tiles - 1) / tiles;
  int cap = H / 256;
  if (cap < 1) cap = 1;
  if (cap > kRouteMaxSplits) cap = kRouteMaxSplits;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  // split length: a multiple of the K chunk; recompute the count it implies
  int len = (H + want - 1) / want;
  len = (len + kRouteBK - 1) / kRouteBK * kRouteBK;
  return (H + len - 1) / len;
}

cudaError_t launch_router_logits(const __nv_bfloat16 *x, const float *w_router, int T, int H, int E,
                                 int splits, float *partial, cudaStream_t s) {
  int len = (H + splits - 1) / splits;
  len = (len + kRouteBK - 1) / kRouteBK * kRouteBK;
  dim3 grid((E + kRouteTE - 1) / kRouteTE, (T + kRouteTT - 1) / kRouteTT, splits);
  router_logits_kernel<<<grid, 256, 0, s>>>(x, w_router, T, H, E, len, partial);
  return cudaGetLastError();
}

cudaError_t launch_topk_gating(const float *partial, int splits, const float *sel_bias, int T,
                               int E, int k, int gating, float *logits, int32_t *ids, float *w,
                               float *gap, cudaStream_t s) {
  const int blocks = (T + 7) / 8;
  const int nv = (E + 31) / 32;
  if (nv <= 1)
    topk_gating_kernel<1><<<blocks, 256, 0, s>>>(partial, splits, sel_bias, T, E, k, gating, logits,
                                                 ids, w, gap);
  else if (nv <= 2)
    topk_gating_kernel<2><<<blocks, 256, 0, s>>>(partial, splits, sel_bias, T, E, k, gating, logits,
                                                 ids, w, gap);
  else if (nv <= 4)
    topk_gating_kernel<4><<<blocks, 256, 0, s>>>(partial, splits, sel_bias, T, E, k, gating, logits,
                                                 ids, w, gap);
  else if (nv <= 8)
    topk_gating_kernel<8><<<blocks, 256, 0, s>>>(partial, splits, sel_bias, T, E, k, gating, logits,
                                                 ids, w, gap);
  else
    topk_gating_kernel<16><<<blocks, 256, 0, s>>>(partial, splits, sel_bias, T, E, k, gating,
                                                  logits, ids, w, gap);
  return cudaGetLastError();
}

}  // namespace moe
