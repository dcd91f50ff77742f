// Block-level pieces of the dispatch shared by the dispatch kernels and the
// small-batch router (which dispatches in its last CTA): a block scan, the
// one-block counting dispatch, and the tile plan of the grouped GEMMs.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Exclusive scan of one value per thread over a block of up to 1024 threads.
static __device__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int t = (lane < nw) ? warp_tot[lane] : 0;
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += u;
    }
    if (lane < nw) warp_tot[lane] = ti - t;  // exclusive prefix of warp totals
    if (lane == nw - 1) *total = ti;
  }
  __syncthreads();
  const int r = warp_tot[w] + incl - v;
  __syncthreads();
  return r;
}

// Split-K of one GEMM, as the number of K blocks per piece: nkb (no split)
// or an even number below nkb (the GEMM streams K in steps of two blocks).
// With `total` tiles on `num_sms` SMs it minimises the K blocks the busiest
// SM streams.  Only small batches split (every tile has at most
// kSplitMaxRows token rows).  Cost model, in K blocks streamed by the busiest
// SM: each piece also pays a fixed epilogue cost (partial store, fence,
// arrival, barriers) worth kSplitPieceCost K blocks, and the last piece reads
// the partials.  A split is taken only if it saves at least a fifth.
static __device__ int choose_split(int total, int nkb, int num_sms, int max_m) {
  // 32-bit arithmetic throughout: total*pieces <= kMaxSplitTiles is checked
  // before any product that could grow, nkb <= 512
  constexpr int kSplitPieceCost = 8;  // measured: 2 and 4 split too eagerly
  if (total <= 0 || max_m > kSplitMaxRows || total > kMaxSplitTiles / 2) return nkb;
  const int base = (total + num_sms - 1) / num_sms * nkb;
  int best = nkb, best_cost = base;
  for (int S = 2; S <= kMaxSplit; ++S) {
    const int kbs = 2 * ((nkb + 2 * S - 1) / (2 * S));  // even, >= 2
    if (kbs >= nkb) continue;
    const int pieces = (nkb + kbs - 1) / kbs;  // no empty piece
    if (total * pieces > kMaxSplitTiles) break;
    const int cost = (total * pieces + num_sms - 1) / num_sms * (kbs + kSplitPieceCost) + pieces;
    if (cost < best_cost) {
      best = kbs;
      best_cost = cost;
    }
  }
  return (best_cost * 5 <= base * 4) ? best : nkb;
}

// The tile plan of the grouped GEMMs from the dispatch offsets (see the
// workspace layout's `plan` field): segment row offsets, the gate/up and down
// tile prefix sums, split-K pieces and pipeline layouts.  Called by every
// thread of one block of 171..1024 threads (each thread owns up to three
// consecutive segments; nseg <= 513).
static __device__ void write_tile_plan(const int32_t *__restrict__ offsets, int T, int k, int E, int H,
                                int I, int shared, int32_t *__restrict__ plan, int num_sms,
                                uint32_t *__restrict__ status) {
  const int64_t Na = (int64_t)T * k;
  __shared__ int warp_tot[32];
  __shared__ int tot_gu, tot_dn, bad, max_m, n_chunks, n_wide, st_narrow, st_wide;
  const int nseg = E + (shared ? 1 : 0);
  const int nj_dn = (H + kBM - 1) / kBM;
  if (threadIdx.x == 0) {
    bad = 0;
    max_m = 0;
    n_chunks = 0;
    n_wide = 0;
    st_narrow = 0;
    st_wide = 0;
  }
  __syncthreads();
  // validate the offsets (caller-provided in the standalone call)
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (offsets[e] < 0 || offsets[e + 1] < offsets[e] || offsets[e + 1] > Na) bad = 1;
  if (threadIdx.x == 0 && offsets[0] != 0) bad = 1;
  __syncthreads();
  if (threadIdx.x == 0 && bad) atomicOr(status, kStatusBadOffsets);
  int32_t *seg_row = plan, *pref_gu = plan + nseg + 1, *pref_dn = plan + 2 * (nseg + 1);
  // each thread owns up to 3 consecutive segments (nseg <= 513 < 3*256)
  constexpr int kPer = 3;
  const int s0 = threadIdx.x * kPer;
  int ms[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int s = s0 + q;
    int m = 0;
    if (!bad && s < nseg) m = (s < E) ? offsets[s + 1] - offsets[s] : T;
    ms[q] = m;
    if (m > 0) {
      atomicMax(&max_m, m);
      // 256-row token chunks; "wide" ones have more than 128 rows
      atomicAdd(&n_chunks, (m + kTileRowsDown - 1) / kTileRowsDown);
      atomicAdd(&n_wide, m / kTileRowsDown + (m % kTileRowsDown > 128 ? 1 : 0));
      // gate/up pipeline stages per 128 weight rows and K step: narrow tiles
      // (128 + 128 rows by <= 128 tokens) vs wide (64 + 64 rows by <= 256)
      atomicAdd(&st_narrow, (m + kTileRowsGateUp - 1) / kTileRowsGateUp);
      atomicAdd(&st_wide, 2 * ((m + kTileRowsDown - 1) / kTileRowsDown));
    }
    // the shared expert's rows follow the routed rows: at offsets[E] (= T*k
    // without a capacity limit)
    if (s < nseg) seg_row[s] = bad ? 0 : offsets[s < E ? s : E];
  }
  __syncthreads();
  // Pipeline layouts.  Down: "wide" (stages of 256 token rows) when most
  // 256-row chunks have more than 128 rows.  Gate/up: wide tiles (64 gate +
  // 64 up rows by <= 256 token rows, one N <= 256 MMA per K16 step) when
  // they need at most 9/8 the stages of narrow tiles (128 + 128 rows by
  // <= 128 token rows, two MMAs per K16 step).  Measured: a wide stage costs
  // about 0.9 of a narrow one (Mixtral T=4096, ratio 1.04: wide 7% faster;
  // DeepSeek-V3 T=8192, ratio 1.29: wide 10% slower).
  const bool wide_dn = n_wide > 0 && 2 * n_wide >= n_chunks;
  const bool wide_gu = st_narrow > 0 && 8 * st_wide <= 9 * st_narrow;
  const bool thin_all = max_m <= kThinRows;
  const bool medium_all = max_m <= kMediumRows;
  // down, where it would otherwise be narrow or medium: "pair" tiles of 256
  // W2 rows by <= 128 token rows (H >= 256)
  // (measured in place of wide as well: Mixtral T=4096 down 744 -> 827 us;
  // in place of medium: Qwen3 TP-8 slice T=128 down 61 -> 47 us, T=256
  // 63 -> 49 us, Mixtral T=64 160 -> 155 us, Qwen3 T=128 unchanged)
  const bool pair_dn = kDownPair && !thin_all && !wide_dn && H >= 2 * kBM;
  // thin (decode) pairing only for a short down K (I <= 4096); measured:
  // Qwen3 TP-8 slice (I = 192) down 3.6-10.6 us faster at T = 2..16, Qwen3
  // (I = 1536) 1.5 us at T = 1, Mixtral (I = 14336) 3.5 us slower at T = 1
  const bool thin_pair_dn = kDownThinPair && thin_all && H >= 2 * kBM && I <= 4096;
  // gate/up segments above this many rows take wide tiles
  const int wide_above = wide_gu ? 0 : (thin_all ? (1 << 30) : kGateUpWideAbove);
  int gu[kPer], dn[kPer], sum_gu = 0, sum_dn = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    gu[q] = ms[q] > wide_above
                ? (ms[q] + kTileRowsDown - 1) / kTileRowsDown *
                      ((I + kGateUpColsWide - 1) / kGateUpColsWide)
                : (ms[q] + kTileRowsGateUp - 1) / kTileRowsGateUp * ((I + kBM - 1) / kBM);
    dn[q] = (pair_dn || thin_pair_dn) ? (ms[q] + kBM - 1) / kBM * ((H + 2 * kBM - 1) / (2 * kBM))
                    : (ms[q] + kTileRowsDown - 1) / kTileRowsDown * nj_dn;
    sum_gu += gu[q];
    sum_dn += dn[q];
  }
  int run_gu = block_exclusive_scan(sum_gu, warp_tot, &tot_gu);
  int run_dn = block_exclusive_scan(sum_dn, warp_tot, &tot_dn);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int s = s0 + q;
    if (s < nseg) {
      pref_gu[s] = run_gu;
      pref_dn[s] = run_dn;
    }
    run_gu += gu[q];
    run_dn += dn[q];
  }
  if (threadIdx.x == 0) {
    seg_row[nseg] = bad ? 0 : offsets[E] + (shared ? T : 0);
    pref_gu[nseg] = tot_gu;
    pref_dn[nseg] = tot_dn;
    plan[3 * (nseg + 1)] = choose_split(tot_gu, H / kBK, num_sms, max_m);
    plan[3 * (nseg + 1) + 1] = choose_split(tot_dn, I / kBK, num_sms, max_m);
    // layouts: 2 = thin (every tile <= kThinRows token rows: stages of
    // weights + kThinRows token rows, more of them in flight), 1 = wide, 0 =
    // narrow;
    const bool thin = max_m <= kThinRows;
    plan[3 * (nseg + 1) + 2] = thin ? 2 : (wide_gu ? 1 : 0);
    // down only: 3 = medium (every tile <= 64 token rows: stages of 64 rows,
    // four in flight; measured 2% faster than narrow there, and far slower
    // once hot experts reload their weights per 64-row unit), taken only
    // where pair tiles are not (H < 256); 4 = pair; 5 = thin pair
    plan[3 * (nseg + 1) + 3] =
        thin ? (thin_pair_dn ? 5 : 2) : (pair_dn ? 4 : (medium_all ? 3 : (wide_dn ? 1 : 0)));
  }
}

// One-block dispatch of N_a assignments ("MoE推理优化全景指南", dispatch
// example: histogram, prefix sum, stable permutation): counts[E],
// offsets[E+1], perm_src / inv_pos / w_perm.  The ranking is stable: chunks
// of NT assignments in order, warps in order inside a chunk (per-warp
// counts), lanes in order inside a warp (__match_any_sync) -- the same order
// as the multi-block path.  Called by every thread of one block of NT
// threads.
template <int NT>
static __device__ void dispatch_block(const int32_t *__restrict__ ids,
                                      const float *__restrict__ topk_w, int64_t Na, int E,
                                      int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                      int32_t *__restrict__ perm_src,
                                      int32_t *__restrict__ inv_pos, float *__restrict__ w_perm,
                                      uint32_t *__restrict__ status) {
  constexpr int kW = NT / 32;
  constexpr int kPer = (kMaxE + NT - 1) / NT;  // experts per thread in the scan
  __shared__ int base[kMaxE];
  __shared__ int wcnt[kW][kMaxE];
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int w = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += NT) base[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int64_t a = threadIdx.x; a < Na; a += NT) {
    const int e = ids[a];
    if (e >= 0 && e < E)
      atomicAdd(&base[e], 1);
    else
      bad = true;
  }
  if (bad) atomicOr(status, kStatusBadExpertId);
  __syncthreads();
  // thread i owns experts [i*kPer, i*kPer + kPer)
  int cnt[kPer], sum = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int e = threadIdx.x * kPer + q;
    cnt[q] = (e < E) ? base[e] : 0;
    sum += cnt[q];
  }
  int run = block_exclusive_scan(sum, warp_tot, &total);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int e = threadIdx.x * kPer + q;
    if (e < E) {
      counts[e] = cnt[q];
      offsets[e] = run;
      base[e] = run;
    }
    run += cnt[q];
  }
  if (threadIdx.x == 0) offsets[E] = total;
  __syncthreads();
  for (int64_t sub = 0; sub < Na; sub += NT) {
    for (int i = threadIdx.x; i < kW * E; i += NT) wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int64_t a = sub + threadIdx.x;
    int e = (a < Na) ? ids[a] : -1;
    if (e < 0 || e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const uint32_t below = peers & lanemask_lt();
    const bool leader = (below == 0);
    if (e >= 0 && leader) wcnt[w][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int ww = 0; ww < w; ++ww) before += wcnt[ww][e];
      const int pos = base[e] + before + __popc(below);
      perm_src[pos] = (int32_t)a;
      inv_pos[a] = pos;
      if (w_perm != nullptr) w_perm[pos] = topk_w[a];
    }
    __syncthreads();
    if (e >= 0 && leader) atomicAdd(&base[e], __popc(peers));
    __syncthreads();
  }
}

}  // namespace moe
