// FP8 (E4M3) expert weights with a power-of-two scale per 128 x 128 block
// ("MoE推理优化全景指南", section "量化与 offload 并非独立开关", "专家权重量化":
// FP8 weights cut the weight bytes the expert GEMMs stream; the scale layout
// is the implementation's choice).
//
// For each block of 128 rows x 128 columns of a matrix: s = the smallest
// integer with max|w| / 2^s <= 448, clamped to [-15, 7], codes =
// round-to-nearest-even of w / 2^s to E4M3 with saturation.  Because the
// scale is a power of two in that range, code * 2^s is exact in fp16 (and in
// bf16): the FP8 layer is the layer over the dequantised weights.  One CTA
// per block: the block's absolute maximum by a warp and block reduction,
// then the codes.
#include <cuda_fp8.h>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kQThreads = 256;
constexpr int kQB = 128;  // block edge
constexpr int kMinExp = -15, kMaxExp = 7;  // block exponents (fp16-exact dequantisation)

__global__ void __launch_bounds__(kQThreads)
    quantize_fp8_kernel(const __nv_bfloat16 *__restrict__ w, int rows, int K, int nrb, int nkb,
                        uint8_t *__restrict__ q, int8_t *__restrict__ scale) {
  __shared__ float s_max[kQThreads / 32];
  __shared__ float s_amax;
  const int blk = blockIdx.x;
  const int c = blk % nkb, r = (blk / nkb) % nrb, i = blk / (nkb * nrb);
  const int r0 = r * kQB, c0 = c * kQB;
  const int nrow = min(kQB, rows - r0), ncol = min(kQB, K - c0);
  const size_t base = ((size_t)i * rows + r0) * K + c0;
  // 16 chunks of 8 bf16 per 128-column row; this thread's chunks
  constexpr int kPer = kQB * kQB / 8 / kQThreads;  // 8
  uint4 raw[kPer];
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int ch = threadIdx.x + u * kQThreads;
    const int rr = ch >> 4, cc = (ch & 15) * 8;
    raw[u] = make_uint4(0, 0, 0, 0);
    if (rr < nrow && cc < ncol)
      raw[u] = *reinterpret_cast<const uint4 *>(w + base + (size_t)rr * K + cc);
    const uint32_t wd[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
      amax = fmaxf(amax, fabsf(__uint_as_float(wd[q2] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(wd[q2] & 0xffff0000u)));
    }
  }
  // non-negative floats order like their bit patterns
  const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(amax));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = __uint_as_float(wm);
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int k = 0; k < kQThreads / 32; ++k) m = fmaxf(m, s_max[k]);
    s_amax = m;
  }
  __syncthreads();
  const float am = s_amax;
  int s = 0;
  if (am > 0.f) {
    int x;
    frexpf(am, &x);
    s = x - 9;
    while (ldexpf(am, -s) > 448.f) ++s;
    while (ldexpf(am, -(s - 1)) <= 448.f) --s;
  }
  // code * 2^s exact in fp16: s in [-15, 7]
  s = max(kMinExp, min(kMaxExp, s));
  if (threadIdx.x == 0) scale[blk] = (int8_t)s;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int ch = threadIdx.x + u * kQThreads;
    const int rr = ch >> 4, cc = (ch & 15) * 8;
    if (rr < nrow && cc < ncol) {
      const uint32_t wd[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
      uint32_t out[2] = {0u, 0u};
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const float2 f = make_float2(ldexpf(__uint_as_float(wd[q2] << 16), -s),
                                     ldexpf(__uint_as_float(wd[q2] & 0xffff0000u), -s));
        const uint32_t two = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
        out[q2 >> 1] |= (two & 0xffffu) << (16 * (q2 & 1));
      }
      *reinterpret_cast<uint2 *>(q + base + (size_t)rr * K + cc) = make_uint2(out[0], out[1]);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const __nv_bfloat16 *w, int n, int rows, int K, uint8_t *q,
                                int8_t *scale, cudaStream_t s) {
  const int nrb = (rows + kQB - 1) / kQB, nkb = (K + kQB - 1) / kQB;
  const int64_t blocks = (int64_t)n * nrb * nkb;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  quantize_fp8_kernel<<<(unsigned)blocks, kQThreads, 0, s>>>(w, rows, K, nrb, nkb, q, scale);
  return cudaGetLastError();
}

}  // namespace moe
