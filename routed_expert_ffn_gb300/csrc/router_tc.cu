// Router s = W_r x ("MoE推理优化全景指南", section "从 Dense FFN 到专家集合")
// on the tensor cores, with fp32-accurate products.
//
// W_r is fp32; x is bf16.  W_r is split exactly into three bf16 terms,
//   hi = bf16(w),  mid = bf16(w - hi),  lo = bf16(w - hi - mid)
// (each subtraction is exact -- Sterbenz -- and the last residual has at most
// 8 significant bits, so hi + mid + lo == w exactly).  A bf16 x bf16 product
// has a 16-bit significand, so every product the tensor core forms is exact,
// and two partial logits are accumulated in fp32 in TMEM, one of the hi
// products and one of the mid and lo products (whose sum is 2^-8 of the hi
// sum, so its rounding is negligible):
//   s = (x.mid + x.lo) + x.hi
// Summation is blocked: the tensor core accumulates one chunk of kChunkKB
// K blocks (512 products per logit and term) in TMEM, and the epilogue adds
// the chunks in fp32 registers.  A plain fp32 chain over H = 7168 terms with
// logits up to |s| ~ 14 is off by up to ~6e-5; the chunked sum keeps the
// error of the long accumulation (and the tensor core's accumulation bias)
// to one chunk.
//
// Tile = 128 experts (MMA M) x up to 128 tokens (MMA N) x one K range of H;
// the K ranges (splits) give the GPU enough CTAs at small T and are summed in
// a fixed order by the gating kernel.  Warp roles as in the expert GEMMs: a
// TMA producer warp, a single-thread MMA issuer, four epilogue warps; two
// TMEM buffers let the epilogue drain one chunk while the next accumulates;
// every wait is bounded.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kRThreads = 192;
constexpr int kRBN = 128;                                  // tokens per tile
constexpr int kChunkKB = 8;                                // K blocks per TMEM accumulation
constexpr uint32_t kRA = kBM * kBK * 2;                    // one 128 x 64 bf16 tile
constexpr uint32_t kRB = kRBN * kBK * 2;
constexpr uint32_t kRStage = 3 * kRA + kRB;                // hi, mid, lo + tokens
constexpr int kRStages = 3;
constexpr uint32_t kRAcc = 2 * kRBN;                       // hi and (mid + lo) accumulators
constexpr uint32_t kRTmemCols = 512;                       // 2 buffers x 2 x 128 columns
constexpr size_t kRSmem = 1024 + (size_t)kRStages * kRStage + 256;

__global__ void __launch_bounds__(256)
    router_split_kernel(const float4 *__restrict__ w, int64_t n4, __nv_bfloat16 *__restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t n = n4 * 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = w[i];
    const float f[4] = {v.x, v.y, v.z, v.w};
    __nv_bfloat16 hi[4], mid[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hi[j] = __float2bfloat16_rn(f[j]);
      const float r1 = f[j] - __bfloat162float(hi[j]);
      mid[j] = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid[j]);
      lo[j] = __float2bfloat16_rn(r2);
    }
    uint2 a, b, c;
    memcpy(&a, hi, 8);
    memcpy(&b, mid, 8);
    memcpy(&c, lo, 8);
    reinterpret_cast<uint2 *>(out)[i] = a;
    reinterpret_cast<uint2 *>(out + n)[i] = b;
    reinterpret_cast<uint2 *>(out + 2 * n)[i] = c;
  }
}

__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_w,   // [3][E][H] bf16 (3D)
                     const __grid_constant__ CUtensorMap tm_x,   // [T][H] bf16, 16-row box
                     const __grid_constant__ CUtensorMap tm_x128,  // the same, 128-row box
                     int T, int E, int kb_per_split, int nkb, float *__restrict__ partial,
                     uint32_t *__restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;                                   // [stage][3][kRA]
  uint8_t *sB = sA + (size_t)kRStages * 3 * kRA;        // [stage][kRB]
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + (size_t)kRStages * kRB);
  uint64_t *empty = full + kRStages;
  uint64_t *tfull = empty + kRStages;
  uint64_t *tempty = tfull + 2;
  uint64_t *fin = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * kBM, t0 = blockIdx.y * kRBN, z = blockIdx.z;
  const int kb0 = z * kb_per_split;
  const int kb1 = min(nkb, kb0 + kb_per_split);
  const int nrows = min(kRBN, T - t0);
  const int N = (nrows + 15) & ~15;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kRTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_x128);
  }
  pdl_wait();
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      const int nb16 = (nrows + 15) >> 4;
      const uint32_t bytes = 3 * kRA + (uint32_t)nb16 * 16 * kBK * 2;
      uint32_t it = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int st = (int)(it % kRStages);
        if (!mbar_wait(&empty[st], ((it / kRStages) & 1u) ^ 1u, abort_flag, status,
                       kStatusTimeoutRouter))
          break;
        mbar_arrive_expect_tx(&full[st], bytes);
        uint8_t *a0 = sA + (size_t)st * 3 * kRA;
        for (int p = 0; p < 3; ++p) tma_load_3d(a0 + p * kRA, &tm_w, &full[st], kb * kBK, e0, p);
        uint8_t *b0 = sB + (size_t)st * kRB;
        if (nrows == kRBN) {
          tma_load_2d(b0, &tm_x128, &full[st], kb * kBK, t0);
        } else {
          for (int q = 0; q < nb16; ++q)
            tma_load_2d(b0 + q * 16 * kBK * 2, &tm_x, &full[st], kb * kBK, t0 + q * 16);
        }
      }
      const uint32_t first = it > (uint32_t)kRStages ? it - kRStages : 0u;
      for (uint32_t i = first; i < it; ++i) mbar_wait_drain(&full[i % kRStages], (i / kRStages) & 1u);
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, N);
      bool ok = true;
      uint32_t it = 0;
      for (int kb = kb0; kb < kb1 && ok; ++kb, ++it) {
        const int c = (kb - kb0) / kChunkKB;           // chunk index
        const bool chunk_first = ((kb - kb0) % kChunkKB) == 0;
        const bool chunk_last = ((kb - kb0) % kChunkKB) == kChunkKB - 1 || kb == kb1 - 1;
        const uint32_t buf = c & 1, use = c >> 1;
        if (chunk_first) {
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, status, kStatusTimeoutRouter)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const int st = (int)(it % kRStages);
        if (!mbar_wait(&full[st], (it / kRStages) & 1u, abort_flag, status, kStatusTimeoutRouter)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sA + (size_t)st * 3 * kRA);
        const uint64_t bdesc = sdesc_k_sw128(smem_u32(sB + (size_t)st * kRB));
        const uint32_t d0 = tmem_base + buf * kRAcc;
        const uint64_t a_hi = sdesc_k_sw128(a_addr), a_mid = sdesc_k_sw128(a_addr + kRA),
                       a_lo = sdesc_k_sw128(a_addr + 2 * kRA);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint32_t acc = (!chunk_first || ks != 0) ? 1u : 0u;
          umma_bf16(d0, a_hi + 2 * ks, bdesc + 2 * ks, idesc, acc);
          umma_bf16(d0 + kRBN, a_mid + 2 * ks, bdesc + 2 * ks, idesc, acc);
          umma_bf16(d0 + kRBN, a_lo + 2 * ks, bdesc + 2 * ks, idesc, 1u);
        }
        umma_commit(&empty[st]);
        if (chunk_last) umma_commit(&tfull[buf]);
      }
      umma_commit(fin);
      mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else {
    // acc[n]: this thread's expert (TMEM lane) against token column n
    float acc[kRBN];
#pragma unroll
    for (int n = 0; n < kRBN; ++n) acc[n] = 0.f;
    const int nchunks = (kb1 - kb0 + kChunkKB - 1) / kChunkKB;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t buf = c & 1, use = c >> 1;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&tfull[buf], use & 1u, abort_flag, status, kStatusTimeoutRouter))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(warp * 32) << 16) + buf * kRAcc;
#pragma unroll
      for (int n0 = 0; n0 < kRBN; n0 += 16) {
        if (n0 < N) {
          uint32_t hi[16], ml[16];
          tmem_ld16(tb + n0, hi);
          tmem_ld16(tb + kRBN + n0, ml);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 16; ++q) acc[n0 + q] += __uint_as_float(ml[q]) + __uint_as_float(hi[q]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
    const int e = e0 + warp * 32 + lane;
    if (ok && e < E) {
#pragma unroll
      for (int n = 0; n < kRBN; ++n)
        if (n < nrows) partial[((size_t)z * T + t0 + n) * E + e] = acc[n];
    }
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kRTmemCols);
  }
}

}  // namespace

int route_splits(int T, int E, int H, int nsm) {
  const int tiles = ((E + kBM - 1) / kBM) * ((T + kRBN - 1) / kRBN);
  const int nkb = H / kBK;
  // at most one CTA per SM (each holds all of TMEM): one wave
  int want = nsm / tiles;
  // at least 4 K blocks per split, 8 once there are 8 or more output tiles
  // (measured: 3-4 us less route time at T = 512 and 1024 than 2 K blocks;
  // smaller batches lose about 1 us with 8)
  int cap = nkb / (tiles >= 8 ? 8 : 4);
  if (cap > kRouteMaxSplits) cap = kRouteMaxSplits;
  if (cap < 1) cap = 1;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  const int per = (nkb + want - 1) / want;
  return (nkb + per - 1) / per;
}

cudaError_t launch_router_logits(const __nv_bfloat16 *x, const float *w_router, int T, int H, int E,
                                 int splits, __nv_bfloat16 *w_split, float *partial,
                                 uint32_t *status, cudaStream_t s) {
  const int64_t n4 = (int64_t)E * H / 4;
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
  cudaError_t e = launch_pdl(router_split_kernel, dim3(blocks), dim3(256), 0, s,
                             reinterpret_cast<const float4 *>(w_router), n4, w_split);
  if (e != cudaSuccess) return e;

  CUtensorMap mw, mx;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)E, 3};
    const cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)H * 2 * E};
    const cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)kBM, 1};
    if (!encode_bf16_map(&mw, w_split, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  CUtensorMap mx128;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, 16};
    if (!encode_bf16_map(&mx, x, 2, dims, strides, box)) return cudaErrorInvalidValue;
    const cuuint32_t box128[2] = {(cuuint32_t)kBK, (cuuint32_t)kRBN};
    if (!encode_bf16_map(&mx128, x, 2, dims, strides, box128)) return cudaErrorInvalidValue;
  }
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kRSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int nkb = H / kBK;
  const int per = (nkb + splits - 1) / splits;
  dim3 grid((E + kBM - 1) / kBM, (T + kRBN - 1) / kRBN, splits);
  return launch_pdl(router_tc_kernel, grid, dim3(kRThreads), kRSmem, s, mw, mx, mx128, T, E, per, nkb,
                    partial, status);
}

}  // namespace moe
