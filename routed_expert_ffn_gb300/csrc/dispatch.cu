// Count / prefix sum / permute dispatch ("MoE推理优化全景指南", section
// "Dispatch 并不是一次普通 all-to-all"), and the gather of the permuted token
// rows plus the tile plan the grouped GEMMs read.
//
// The flat assignment list a = t*k + j is cut into per-block chunks:
//   1. hist:    per-block expert histogram in shared memory (atomics only
//               count; they never decide a position);
//   2. scan:    one CTA sums the block histograms per expert, scans them into
//               the expert offsets and gives every (block, expert) its base;
//   3. scatter: each block re-reads its assignments in order and ranks them
//               stably: __match_any_sync groups equal experts inside a warp,
//               per-warp counts in shared memory order the warps, and a
//               running per-expert base orders the block's sub-chunks.
// The result is bit-exact: expert e owns positions [offsets[e], offsets[e+1])
// in ascending assignment (hence token) order.
#include "dispatch_block.cuh"

namespace moe {

namespace {

constexpr int kWarps = kDispatchThreads / 32;

__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_hist_kernel(const int32_t *__restrict__ ids, int64_t Na, int64_t chunk, int E,
                         int32_t *__restrict__ blk_counts, uint32_t *__restrict__ status) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int cnt[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int64_t beg = (int64_t)blockIdx.x * chunk;
  const int64_t end = min(Na, beg + chunk);
  bool bad = false;
  for (int64_t a = beg + threadIdx.x; a < end; a += blockDim.x) {
    const int e = ids[a];
    if (e >= 0 && e < E)
      atomicAdd(&cnt[e], 1);
    else
      bad = true;
  }
  if (bad) atomicOr(status, kStatusBadExpertId);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blk_counts[(size_t)blockIdx.x * E + e] = cnt[e];
}

__global__ void __launch_bounds__(kMaxE)
    dispatch_scan_kernel(const int32_t *__restrict__ blk_counts, int nblk, int E,
                         int32_t *__restrict__ blk_base, int32_t *__restrict__ counts,
                         int32_t *__restrict__ offsets, PlanArgs pa) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int e = threadIdx.x;
  int tot = 0;
  if (e < E)
    for (int b = 0; b < nblk; ++b) tot += blk_counts[(size_t)b * E + e];
  const int excl = block_exclusive_scan(tot, warp_tot, &total);
  if (e < E) {
    counts[e] = tot;
    offsets[e] = excl;
    int run = excl;
    for (int b = 0; b < nblk; ++b) {
      blk_base[(size_t)b * E + e] = run;
      run += blk_counts[(size_t)b * E + e];
    }
  }
  if (e == 0) offsets[E] = total;
  if (pa.plan != nullptr) {
    __syncthreads();
    write_tile_plan(offsets, pa.T, pa.k, E, pa.H, pa.I, pa.shared, pa.plan, pa.num_sms, pa.status);
  }
}

__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_scatter_kernel(const int32_t *__restrict__ ids, const float *__restrict__ topk_w,
                            int64_t Na, int64_t chunk, int E,
                            const int32_t *__restrict__ blk_base,
                            int32_t *__restrict__ perm_src, int32_t *__restrict__ inv_pos,
                            float *__restrict__ w_perm) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int base[kMaxE];
  __shared__ int wcnt[kWarps][kMaxE];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] = blk_base[(size_t)blockIdx.x * E + e];
  const int64_t beg = (int64_t)blockIdx.x * chunk;
  const int64_t end = min(Na, beg + chunk);
  for (int64_t sub = beg; sub < end; sub += kDispatchThreads) {
    for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int64_t a = sub + threadIdx.x;
    int e = (a < end) ? ids[a] : -1;
    if (e < 0 || e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const uint32_t below = peers & lanemask_lt();
    const int rank = __popc(below);
    const bool leader = (below == 0);
    if (e >= 0 && leader) wcnt[w][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int ww = 0; ww < w; ++ww) before += wcnt[ww][e];
      const int pos = base[e] + before + rank;
      perm_src[pos] = (int32_t)a;
      inv_pos[a] = pos;
      if (w_perm != nullptr) w_perm[pos] = topk_w[a];
    }
    __syncthreads();
    if (e >= 0 && leader) atomicAdd(&base[e], __popc(peers));
    __syncthreads();
  }
  (void)lane;
}

// Eight bf16 values to eight fp16 values (round to nearest even; exact for
// |x| in fp16's normal range, which covers the layers' activations).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h2 = __floats2half2_rn(__uint_as_float(w[i] << 16),
                                         __uint_as_float(w[i] & 0xffff0000u));
    o[i] = *reinterpret_cast<const uint32_t *>(&h2);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Rows [0, Na): x_perm[p] = x[perm_src[p] / k]; rows [Na, Na+T) (shared
// expert): x_perm[Na+t] = x[t].  16-byte vectors (to_fp16: converted to
// fp16, the token operand of the FP8-weight GEMMs).  With inv_pos (the layer
// forward) one warp per token reads its row of x once and writes it to the
// token's k positions (and its shared-expert row), so x is read once even
// when it does not fit in L2; without (the standalone FFN call) one warp per
// x_perm row.  The last block instead writes the tile plan of the grouped
// GEMMs (with_plan: when no earlier kernel wrote it).
__global__ void __launch_bounds__(256)
    gather_plan_kernel(const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ perm_src,
                       const int32_t *__restrict__ inv_pos, const int32_t *__restrict__ offsets,
                       int T, int k, int E, int H, int I, int shared,
                       __nv_bfloat16 *__restrict__ x_perm, __nv_bfloat16 *__restrict__ h,
                       int32_t *__restrict__ plan, int with_plan, int num_sms,
                       uint32_t *__restrict__ status, int to_fp16) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t Na = (int64_t)T * k;
  const int64_t R = Na + (shared ? T : 0);
  if (with_plan && blockIdx.x == gridDim.x - 1) {
    write_tile_plan(offsets, T, k, E, H, I, shared, plan, num_sms, status);
    return;
  }
  {
    // Rows past the last segment exist only when the segments end before
    // T*k (a capacity limit, or caller-given offsets): the down GEMM's tiles
    // read up to 256 h rows past their start, so the first 256 such rows of
    // h are zeroed here (gate/up writes only segment rows).
    const int64_t end = (int64_t)offsets[E] + (shared ? T : 0);
    const int64_t tail = min(R, end + 256);
    const int64_t nvh = (tail > end ? tail - end : 0) * (I / 8);
    const int64_t nb = gridDim.x - with_plan;  // the gather blocks (not the plan block)
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvh;
         v += nb * blockDim.x)
      reinterpret_cast<uint4 *>(h + end * I)[v] = make_uint4(0, 0, 0, 0);
  }
  // ---- gather ----
  // the shared expert's rows start at offsets[E] (= Na without a capacity
  // limit, else the number of kept assignments)
  const int64_t sb = offsets[E];
  const int lane = threadIdx.x & 31;
  constexpr int kBatch = 8;  // 16-byte loads in flight per lane before their stores
  const int nv = H / 8;
  if (inv_pos != nullptr) {
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    // lane j < k holds the destination of assignment t*k+j (checked against
    // perm_src: only a position the dispatch gave this assignment is written)
    int32_t myp = -1;
    if (lane < k) {
      const int64_t a = t * k + lane;
      const int32_t p = inv_pos[a];
      if (p >= 0 && p < Na && perm_src[p] == a) myp = p;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(x + t * H);
    for (int v0 = lane; v0 < nv; v0 += 32 * kBatch) {
      uint4 r[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (v0 + 32 * i < nv) r[i] = src[v0 + 32 * i];
      if (to_fp16) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) r[i] = bf16x8_to_f16x8(r[i]);
      }
      for (int j = 0; j <= k; ++j) {
        int64_t row;
        if (j < k) {
          const int32_t p = __shfl_sync(0xffffffffu, myp, j < 32 ? j : 0);
          if (p < 0) continue;
          row = p;
        } else {
          if (!shared) break;
          row = sb + t;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(x_perm + row * H);
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          if (v0 + 32 * i < nv) dst[v0 + 32 * i] = r[i];
      }
    }
    return;
  }
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= R) return;
  int64_t src = -1;
  if (row < sb) {
    const int32_t a = perm_src[row];
    if (a >= 0 && a < Na) src = a / k;
  } else if (shared && row < sb + T) {
    src = row - sb;
  }
  uint4 *dst = reinterpret_cast<uint4 *>(x_perm + row * H);
  if (src < 0) {
    for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4 *s = reinterpret_cast<const uint4 *>(x + src * H);
  for (int v0 = lane; v0 < nv; v0 += 32 * kBatch) {
    uint4 r[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (v0 + 32 * i < nv) r[i] = s[v0 + 32 * i];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (v0 + 32 * i < nv) dst[v0 + 32 * i] = to_fp16 ? bf16x8_to_f16x8(r[i]) : r[i];
  }
}

// Small batches (N_a <= kSmallDispatch): histogram, scan and stable scatter
// in one block (dispatch_block), so the dispatch is one launch; the block
// then writes the tile plan.
constexpr int kSmallThreads = 512;

__global__ void __launch_bounds__(kSmallThreads)
    dispatch_small_kernel(const int32_t *__restrict__ ids, const float *__restrict__ topk_w,
                          int64_t Na, int E, int32_t *__restrict__ counts,
                          int32_t *__restrict__ offsets, int32_t *__restrict__ perm_src,
                          int32_t *__restrict__ inv_pos, float *__restrict__ w_perm,
                          uint32_t *__restrict__ status, PlanArgs pa) {
  pdl_wait();
  pdl_launch_dependents();
  dispatch_block<kSmallThreads>(ids, topk_w, Na, E, counts, offsets, perm_src, inv_pos, w_perm,
                                status);
  if (pa.plan != nullptr) write_tile_plan(offsets, pa.T, pa.k, E, pa.H, pa.I, pa.shared, pa.plan,
                                          pa.num_sms, pa.status);
}

// Capacity limit ("MoE推理优化全景指南", "Capacity、padding 与 token
// dropping": an expert takes at most C assignments, the rest are dropped).
// From the dropless layout, keep the first C positions of every expert's
// segment (its first C tokens in token order) in a compact layout: every
// block computes the kept counts' prefix sum over E (E <= 512), then moves its
// positions.  A dropped assignment gets inv_pos -1 (the combine skips it);
// positions past the kept rows get perm_src -1 (the gather zeroes them).
constexpr int kCapThreads = 256;

__global__ void __launch_bounds__(kCapThreads)
    capacity_kernel(const int32_t *__restrict__ counts, const int32_t *__restrict__ offsets,
                    const int32_t *__restrict__ perm_src, const float *__restrict__ w_perm,
                    int64_t Na, int E, int C, int32_t *__restrict__ counts_c,
                    int32_t *__restrict__ offsets_c, int32_t *__restrict__ perm_c,
                    int32_t *__restrict__ inv_c, float *__restrict__ w_perm_c) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_off[kMaxE + 1], s_offc[kMaxE + 1];
  __shared__ int warp_tot[32];
  __shared__ int total;
  constexpr int kPer = (kMaxE + kCapThreads - 1) / kCapThreads;  // experts per thread
  int kept[kPer], sum = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int e = threadIdx.x * kPer + q;
    kept[q] = (e < E) ? min(counts[e], C) : 0;
    sum += kept[q];
  }
  int run = block_exclusive_scan(sum, warp_tot, &total);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int e = threadIdx.x * kPer + q;
    if (e < E) {
      s_offc[e] = run;
      s_off[e] = offsets[e];
      if (blockIdx.x == 0) {
        counts_c[e] = kept[q];
        offsets_c[e] = run;
      }
    }
    run += kept[q];
  }
  if (threadIdx.x == 0) {
    s_off[E] = offsets[E];
    s_offc[E] = total;
    if (blockIdx.x == 0) offsets_c[E] = total;
  }
  __syncthreads();
  const int64_t p = (int64_t)blockIdx.x * kCapThreads + threadIdx.x;
  if (p >= Na) return;
  if (p >= total) perm_c[p] = -1;  // past the kept rows
  if (p >= s_off[E]) return;       // (a layout with dropped bad ids ends early)
  int lo = 0, hi = E;              // s_off[lo] <= p < s_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] <= p)
      lo = mid;
    else
      hi = mid;
  }
  const int r = (int)(p - s_off[lo]);
  const int32_t a = perm_src[p];
  if (a < 0 || a >= Na) return;
  if (r < C) {
    const int np = s_offc[lo] + r;
    perm_c[np] = a;
    inv_c[a] = np;
    if (w_perm != nullptr) w_perm_c[np] = w_perm[p];
  } else {
    inv_c[a] = -1;
  }
}

}  // namespace

cudaError_t launch_capacity(const int32_t *counts, const int32_t *offsets, const int32_t *perm_src,
                            const float *w_perm, int T, int k, int E, int C, int32_t *counts_c,
                            int32_t *offsets_c, int32_t *perm_c, int32_t *inv_c, float *w_perm_c,
                            cudaStream_t s) {
  const int64_t Na = (int64_t)T * k;
  const int blocks = (int)((Na + kCapThreads - 1) / kCapThreads);
  return launch_pdl(capacity_kernel, dim3(blocks), dim3(kCapThreads), 0, s, counts, offsets,
                    perm_src, w_perm, Na, E, C, counts_c, offsets_c, perm_c, inv_c, w_perm_c);
}

cudaError_t launch_dispatch(const int32_t *ids, const float *topk_w, int T, int k, int E,
                            int32_t *blk_counts, int32_t *blk_base, int32_t *counts,
                            int32_t *offsets, int32_t *perm_src, int32_t *inv_pos, float *w_perm,
                            uint32_t *status, int32_t *plan, int H, int I, int shared,
                            cudaStream_t s) {
  const int64_t Na = (int64_t)T * k;
  PlanArgs pa;
  pa.plan = plan;
  pa.T = T;
  pa.k = k;
  pa.H = H;
  pa.I = I;
  pa.shared = shared;
  pa.num_sms = plan != nullptr ? num_sms() : 1;
  pa.status = status;
  if (Na <= kSmallDispatch) {
    return launch_pdl(dispatch_small_kernel, dim3(1), dim3(kSmallThreads), 0, s, ids, topk_w, Na, E,
                      counts, offsets, perm_src, inv_pos, w_perm, status, pa);
  }
  const int64_t chunk = dispatch_chunk(Na);
  const int nblk = (int)((Na + chunk - 1) / chunk);
  cudaError_t e = launch_pdl(dispatch_hist_kernel, dim3(nblk), dim3(kDispatchThreads), 0, s, ids,
                             Na, chunk, E, blk_counts, status);
  if (e == cudaSuccess)
    e = launch_pdl(dispatch_scan_kernel, dim3(1), dim3(kMaxE), 0, s, blk_counts, nblk, E, blk_base,
                   counts, offsets, pa);
  if (e == cudaSuccess)
    e = launch_pdl(dispatch_scatter_kernel, dim3(nblk), dim3(kDispatchThreads), 0, s, ids, topk_w,
                   Na, chunk, E, blk_base, perm_src, inv_pos, w_perm);
  return e;
}

cudaError_t launch_gather_plan(const __nv_bfloat16 *x, const int32_t *perm_src,
                               const int32_t *inv_pos, const int32_t *offsets, int T, int k, int E,
                               int H, int I, int shared, __nv_bfloat16 *x_perm, __nv_bfloat16 *h,
                               int32_t *plan, uint32_t *status, cudaStream_t s, bool to_fp16) {
  // eight warps per block: one per token (with inv_pos) or per x_perm row;
  // one more block writes the tile plan when `plan` is given
  const int64_t units = inv_pos != nullptr ? (int64_t)T : (int64_t)T * k + (shared ? T : 0);
  const int with_plan = plan != nullptr ? 1 : 0;
  const int blocks = (int)((units + 7) / 8) + with_plan;
  return launch_pdl(gather_plan_kernel, dim3(blocks), dim3(256), 0, s, x, perm_src, inv_pos,
                    offsets, T, k, E, H, I, shared, x_perm, h, plan, with_plan, num_sms(), status,
                    to_fp16 ? 1 : 0);
}

}  // namespace moe
