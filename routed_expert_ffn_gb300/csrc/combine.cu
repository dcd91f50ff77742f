// Inverse permutation and gate-weighted sum ("MoE推理优化全景指南", section
// "一个 token 为什么要跨 GPU", last step of the data path, and section
// "Dispatch 并不是一次普通 all-to-all": restore the original token order and
// apply the routing weights):
//
//   y[t,:] = sum_j wt(t,j) * out_perm[inv_pos[t*k+j],:]  (+ out_perm[T*k+t,:])
//
// One thread per 8 columns of a token row; the k fp16 expert rows of a token
// are gathered with 16-byte loads and summed in fp32 in slot order; y is
// rounded to bf16 once.
#include "moe_internal.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(256)
    combine_kernel(const __half *__restrict__ out_perm, const int32_t *__restrict__ inv_pos,
                   const float *__restrict__ topk_w, const int32_t *__restrict__ shared_base,
                   int T, int k, int H, int shared, __nv_bfloat16 *__restrict__ y) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int v = blockIdx.y * blockDim.x + threadIdx.x;
  const int nv = H / 8;
  if (v >= nv) return;
  const int64_t Na = (int64_t)T * k;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  auto add = [&](const uint4 &raw, float wt) {
    const __half2 *p = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(p[i]);
      acc[2 * i] = fmaf(wt, f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(wt, f.y, acc[2 * i + 1]);
    }
  };
  // up to kBatch expert rows in flight, added in slot order
  constexpr int kBatch = 8;
  for (int j0 = 0; j0 < k; j0 += kBatch) {
    uint4 raw[kBatch];
    float wt[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      wt[i] = 0.f;
      raw[i] = make_uint4(0, 0, 0, 0);
      const int j = j0 + i;
      if (j < k) {
        const int64_t a = (int64_t)t * k + j;
        const int32_t p = inv_pos[a];
        if (p >= 0 && p < Na) {
          wt[i] = topk_w != nullptr ? topk_w[a] : 1.0f;
          raw[i] = reinterpret_cast<const uint4 *>(out_perm + (int64_t)p * H)[v];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (j0 + i < k) add(raw[i], wt[i]);
    }
  }
  // the shared expert's row: after the routed rows (at *shared_base when
  // given: the kept rows under a capacity limit end there)
  if (shared) {
    const int64_t sb = shared_base != nullptr ? (int64_t)*shared_base : Na;
    add(reinterpret_cast<const uint4 *>(out_perm + (sb + t) * H)[v], 1.0f);
  }
  uint4 o;
  __nv_bfloat162 *q = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  reinterpret_cast<uint4 *>(y + (int64_t)t * H)[v] = o;
}

}  // namespace

cudaError_t launch_combine(const __half *out_perm, const int32_t *inv_pos,
                           const float *topk_w, int T, int k, int H, int shared, __nv_bfloat16 *y,
                           cudaStream_t s, const int32_t *shared_base) {
  const int nv = H / 8;
  dim3 grid(T, (nv + 255) / 256);
  return launch_pdl(combine_kernel, grid, dim3(256), 0, s, out_perm, inv_pos, topk_w, shared_base,
                    T, k, H, shared, y);
}

}  // namespace moe
