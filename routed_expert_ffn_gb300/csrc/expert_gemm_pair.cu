// Grouped expert GEMMs for prefill batches on CTA pairs
// (tcgen05.mma.cta_group::2, sm_103a).
//
// The same two GEMMs as the one-SM kernel ("MoE推理优化全景指南", section
// "Expert GEMM 为什么经常不够大": one scheduled launch runs [m_e, hidden] @ W_e
// for every expert; CS349D lecture 8 notes, section 2.4: with a few hundred
// token rows per expert the expert GEMMs become compute-bound):
//
//   gate/up:  h[p, i]   = SiLU(sum_c W13[e][i][c] x[p][c]) * sum_c W13[e][I+i][c] x[p][c]
//   down:     out[p, r] = w_perm[p] * sum_i W2[e][r][i] h[p][i]
//
// A cluster of two CTAs on two SMs computes one tile of 256 weight rows by up
// to 256 token rows.  Each CTA's shared memory holds 128 of the weight rows
// and half of the token rows; one thread of the even CTA issues the MMAs for
// both (M = 256), and each CTA's TMEM receives the fp32 accumulator of its
// own 128 weight rows for all token columns.  Per SM and K block that is
// 32 KB of operands for 128 x 256 x 64 multiply-adds, 1.5x the FLOPs per byte
// of the one-SM 128 x 256 tile, and three 64 KB stages fit where the one-SM
// kernel keeps two of 96 KB.
//
// Tiles: gate/up = (segment, 128 h columns, 256-row token chunk), the even
// CTA taking the 64 gate rows and the 64 up rows of the first 64 columns,
// the odd CTA those of the next 64; down = (segment, 256 W2 rows, chunk).
// Tiles of one weight block are adjacent (chunk innermost); cluster c walks
// tiles c, c + clusters, ...  Token rows of a tile are padded to N (a
// multiple of 32); the even CTA loads rows [0, N/2), the odd CTA [N/2, N).
//
// CTA = 6 warps, in both CTAs of the pair:
//   warp 4     TMA producer: its CTA's weight rows and token rows per stage,
//              completion counted on the even CTA's `full` barrier (whose
//              producer expects the bytes of both CTAs);
//   warp 5     TMEM allocation for the pair; in the even CTA one thread
//              issues the MMAs and commits to both CTAs' `empty` (stage
//              free) and `tfull` (accumulator done) barriers;
//   warps 0-3  epilogue over the CTA's own TMEM lanes: SiLU(gate)*up with
//              the up values passed through shared memory, or the gate
//              weighting; then an arrival on the even CTA's `tempty`.
// Every wait is bounded; on expiry the CTA latches MOE_ERR_TIMEOUT's status
// bit and leaves its loops, and both CTAs meet at a cluster barrier before
// the pair's TMEM is freed.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kPThreads = 192;
constexpr int kPStages = 3;
constexpr int kPRows = 256;                                 // token rows per tile
constexpr uint32_t kPA = kStageKB * kBM * kBK * 2;          // 32 KB: 128 weight rows
constexpr uint32_t kPB = kStageKB * (kPRows / 2) * kBK * 2;  // <= 32 KB: <= 128 token rows
constexpr uint32_t kPStage = kPA + kPB;
constexpr uint32_t kPTmemCols = 512;  // two accumulators of 256 columns
constexpr int kPWide = 64;            // gate/up: h columns per CTA
static_assert(kStageKB == 2, "stages are pairs of K blocks");

constexpr size_t pair_smem_bytes(int nseg) {
  return 1024 + (size_t)kPStages * kPStage   // ring
         + 2 * 16 * kPWide * 4               // up-value exchange [2][16][64] floats
         + 2 * 8 * kBM * 4                   // output slices [2][8][128] words
         + (size_t)kPRows * 4                // gate weights of a tile
         + (2 * kPStages + 5) * 8 + 16       // barriers, TMEM slot, flags
         + (size_t)2 * (nseg + 1) * 4;       // segment rows, tile prefix sums
}
static_assert(pair_smem_bytes(kMaxE + 1) <= 232448, "shared memory per CTA");

// ---- cluster / CTA-pair primitives ----
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_u32(p)), "r"(rank));
  return d;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
               : "memory");
}
// Tensor copies into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_5d_pair(void *dst, const CUtensorMap *m, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *m, uint32_t bar,
                                                 int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (+)= A * B^T over the pair: M = 256 (128 rows from each CTA's shared
// memory), N token columns (N/2 from each CTA).
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` (same offset) in every CTA of `mask` when all tcgen05
// ops issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void epi_sync_p() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_all_p(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, 128, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}

struct PTile {
  int seg, j, row0, nrows;
};

// tile -> (segment, weight block j, token chunk); tp = tile prefix sums
__device__ __forceinline__ PTile pair_tile(int tile, const int32_t *seg_row, const int32_t *tp,
                                           int nseg) {
  int lo = 0, hi = nseg;  // tp[lo] <= tile < tp[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tp[mid] <= tile)
      lo = mid;
    else
      hi = mid;
  }
  PTile t;
  t.seg = lo;
  const int m = seg_row[lo + 1] - seg_row[lo];
  const int chunks = (m + kPRows - 1) / kPRows;
  const int local = tile - tp[lo];
  t.j = local / chunks;
  const int c = local - t.j * chunks;
  t.row0 = seg_row[lo] + c * kPRows;
  t.nrows = min(kPRows, m - c * kPRows);
  return t;
}

template <bool kGateUp>
__global__ void __launch_bounds__(kPThreads, 1)
    expert_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a,     // this CTA's weight rows
                            const __grid_constant__ CUtensorMap tm_a_sh,  // shared expert
                            const __grid_constant__ TokenMaps tm_b,       // token rows [R, K]
                            const int32_t *__restrict__ plan, int nseg, int E, int K, int out_cols,
                            int64_t Na, const float *__restrict__ w_perm, void *__restrict__ out_,
                            uint32_t *__restrict__ status) {
  uint16_t *out = static_cast<uint16_t *>(out_);
  constexpr uint32_t kCode = kGateUp ? kStatusTimeoutGateUp : kStatusTimeoutDown;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *ring = smem;                                                    // [stage][A | B]
  float *sUp = reinterpret_cast<float *>(ring + kPStages * kPStage);      // [2][16][64]
  uint32_t *sOut = reinterpret_cast<uint32_t *>(sUp + 2 * 16 * kPWide);   // [2][8][128]
  float *sW = reinterpret_cast<float *>(sOut + 2 * 8 * kBM);              // [256]
  uint64_t *full = reinterpret_cast<uint64_t *>(sW + kPRows);             // [stages]
  uint64_t *empty = full + kPStages;
  uint64_t *tfull = empty + kPStages;
  uint64_t *tempty = tfull + 2;
  uint64_t *fin = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int32_t *seg_row = reinterpret_cast<int32_t *>(tmem_slot + 4);
  int32_t *tp = seg_row + nseg + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: issues the MMAs
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);  // 4 epilogue warps in each CTA
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc_pair(tmem_slot, kPTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_a_sh);
    for (int i = 0; i < 8; ++i) tma_prefetch_desc(&tm_b.m[i]);
  }
  pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i <= nseg; i += blockDim.x) seg_row[i] = __ldcg(plan + i);
  __syncthreads();
  // tiles per segment -> prefix sums (warp 0: each lane a run of segments)
  if (warp == 0) {
    const int I_or_H = out_cols;
    const int nj = kGateUp ? I_or_H / (2 * kPWide) : I_or_H / (2 * kBM);
    const int per = (nseg + 31) / 32;
    const int s0 = lane * per, s1 = min(nseg, s0 + per);
    int sum = 0;
    for (int s = s0; s < s1; ++s) sum += (seg_row[s + 1] - seg_row[s] + kPRows - 1) / kPRows * nj;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int s = s0; s < s1; ++s) {
      tp[s] = run;
      run += (seg_row[s + 1] - seg_row[s] + kPRows - 1) / kPRows * nj;
    }
    if (lane == 31) tp[nseg] = incl;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tp[nseg];
  const int nkb = K / kBK;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      uint32_t st = 0, ph = 0, issued = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl) {
        const PTile t = pair_tile(tile, seg_row, tp, nseg);
        const bool sh = t.seg >= E;
        const CUtensorMap *ma = sh ? &tm_a_sh : &tm_a;
        const int ecoord = sh ? 0 : t.seg;
        const int arow = kGateUp ? t.j * 2 * kPWide + (int)rank * kPWide
                                 : t.j * 2 * kBM + (int)rank * kBM;
        const int half = ((t.nrows + 31) & ~31) >> 1;  // token rows per CTA (16..128)
        const CUtensorMap *mb = &tm_b.m[(half >> 4) - 1];
        const int brow = t.row0 + (int)rank * half;
        const uint32_t bytes_b = (uint32_t)half * (kStageKB * kBK * 2);
        for (int kb = 0; kb < nkb; kb += kStageKB) {
          if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, status, kCode)) {
            ok = false;
            break;
          }
          const uint32_t bar = cluster_addr(&full[st], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[st], 2 * (kPA + bytes_b));
          uint8_t *dst = ring + st * kPStage;
          tma_load_5d_pair(dst, ma, bar, 0, arow, 0, kb, ecoord);
          tma_load_3d_pair(dst + kPA, mb, bar, 0, brow, kb);
          ++issued;
          if (++st == kPStages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (rank == 0) {
        // every copy of both CTAs completes on these barriers
        const uint32_t n = issued < kPStages ? issued : kPStages;
        for (uint32_t i = 0; i < n; ++i) {
          st = st == 0 ? kPStages - 1 : st - 1;
          if (st == kPStages - 1) ph ^= 1u;
          mbar_wait_drain(&full[st], ph);
        }
      } else if (!ok) {
        // the odd CTA's copies complete on the even CTA's barriers: after an
        // abort give copies in flight time to land before leaving
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------- MMA issuer --
    if (rank == 0 && lane == 0) {
      uint32_t st = 0, ph = 0, tl = 0;
      const uint64_t desc0 = sdesc_k_sw128(smem_u32(ring));
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl, ++tl) {
        const PTile t = pair_tile(tile, seg_row, tp, nseg);
        const int n32 = (t.nrows + 31) & ~31;
        const int half = n32 >> 1;
        const uint32_t idesc = idesc_bf16_f32(2 * kBM, n32);
        const uint32_t buf = tl & 1u, use = tl >> 1;
        if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, status, kCode)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * (kPTmemCols / 2);
        for (int kb = 0; kb < nkb; kb += kStageKB) {
          if (!mbar_wait(&full[st], ph, abort_flag, status, kCode)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = desc0 + st * (kPStage >> 4);
          const uint64_t bdesc = adesc + (kPA >> 4);
#pragma unroll
          for (int c = 0; c < kStageKB; ++c) {
            const uint64_t ac = adesc + c * ((kBM * kBK * 2) >> 4);
            const uint64_t bc = bdesc + c * (((uint32_t)half * kBK * 2) >> 4);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              umma_bf16_pair(d0, ac + 2 * q, bc + 2 * q, idesc, (kb | c | q) != 0 ? 1u : 0u);
          }
          umma_commit_pair(&empty[st], 3);  // both CTAs' stage is free
          if (++st == kPStages) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[buf], 3);  // both CTAs' accumulators are complete
      }
      umma_commit_pair(fin, 1);
      mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    const int r = warp * 32 + lane;  // TMEM lane = weight row of this CTA's half
    uint32_t tl = 0, slice = 0;
    float vmax = 0.f;  // down: largest magnitude written (NaN-propagating)
    for (int tile = cid; tile < total; tile += ncl, ++tl) {
      const PTile t = pair_tile(tile, seg_row, tp, nseg);
      const uint32_t buf = tl & 1u, use = tl >> 1;
      const bool waited = mbar_wait(&tfull[buf], use & 1u, abort_flag, status, kCode);
      if (!epi_all_p(waited && !*abort_flag)) break;
      tc_fence_after();
      if (!kGateUp) {
        for (int n = r; n < kPRows; n += 128) {
          const int64_t row = (int64_t)t.row0 + n;
          sW[n] = (n < t.nrows && w_perm != nullptr && t.seg < E && row < Na) ? w_perm[row] : 1.0f;
        }
        epi_sync_p();
      }
      const uint32_t tb = tmem_base + ((uint32_t)(warp * 32) << 16) + buf * (kPTmemCols / 2);
      const int N = (t.nrows + 15) & ~15;
      for (int n0 = 0; n0 < N; n0 += 16) {
        uint32_t v0[16];
        tmem_ld16(tb + n0, v0);
        tmem_ld_wait();
        if (kGateUp) {
          // lanes [0, 64): gate rows, [64, 128): the up rows of the same h
          // columns; the up values pass through shared memory
          constexpr int W = kPWide;
          float *su = sUp + (slice & 1u) * (16 * W);
          uint16_t *so = reinterpret_cast<uint16_t *>(sOut) + (slice & 1u) * (16 * W);
          if (r >= W) {
#pragma unroll
            for (int q = 0; q < 16; ++q) su[q * W + (r - W)] = __uint_as_float(v0[q]);
          }
          epi_sync_p();
          if (r < W) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float g = __uint_as_float(v0[q]), u = su[q * W + r];
              so[q * W + r] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * u));
            }
          }
          epi_sync_p();
          // 16 token rows x 64 columns x 2 bytes = 128 chunks of 16 bytes
          const int q = r >> 3, ch = r & 7;
          const int n = n0 + q, col = t.j * 2 * W + (int)rank * W + ch * 8;
          if (n < t.nrows && col < out_cols)
            *reinterpret_cast<uint4 *>(out + ((int64_t)t.row0 + n) * out_cols + col) =
                *reinterpret_cast<const uint4 *>(so + q * W + ch * 8);
        } else {
          // token pairs packed per conversion (fp16, saturating), words
          // [8 pairs][128 columns], then 16-byte stores to each token's row
          uint32_t *so = sOut + (slice & 1u) * (8 * kBM);
          float wv[16];
#pragma unroll
          for (int q = 0; q < 16; q += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(sW + n0 + q);
            wv[q] = a.x;
            wv[q + 1] = a.y;
            wv[q + 2] = a.z;
            wv[q + 3] = a.w;
          }
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const float x0 = __uint_as_float(v0[2 * p]) * wv[2 * p];
            const float x1 = __uint_as_float(v0[2 * p + 1]) * wv[2 * p + 1];
            vmax = fmax_nan(vmax, fabsf(x0));
            vmax = fmax_nan(vmax, fabsf(x1));
            so[p * kBM + r] = pack_f16x2_satfinite(x0, x1);
          }
          epi_sync_p();
          const int p = r >> 4, ch = r & 15;
          const uint4 lo = *reinterpret_cast<const uint4 *>(so + p * kBM + ch * 8);
          const uint4 hi = *reinterpret_cast<const uint4 *>(so + p * kBM + ch * 8 + 4);
          const uint4 a =
              make_uint4(__byte_perm(lo.x, lo.y, 0x5410), __byte_perm(lo.z, lo.w, 0x5410),
                         __byte_perm(hi.x, hi.y, 0x5410), __byte_perm(hi.z, hi.w, 0x5410));
          const uint4 b =
              make_uint4(__byte_perm(lo.x, lo.y, 0x7632), __byte_perm(lo.z, lo.w, 0x7632),
                         __byte_perm(hi.x, hi.y, 0x7632), __byte_perm(hi.z, hi.w, 0x7632));
          const int n = n0 + 2 * p, col = t.j * 2 * kBM + (int)rank * kBM + ch * 8;
          if (col < out_cols) {
            uint16_t *o = out + ((int64_t)t.row0 + n) * out_cols + col;
            if (n < t.nrows) *reinterpret_cast<uint4 *>(o) = a;
            if (n + 1 < t.nrows) *reinterpret_cast<uint4 *>(o + out_cols) = b;
          }
        }
        ++slice;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(&tempty[buf], 0));
    }
    if (!kGateUp && !(vmax <= 65504.0f)) atomicOr(status, kStatusRange);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal it
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPTmemCols);
  }
}

}  // namespace

bool gemm_pair_supported(const moe_layer_desc_t &d, bool gate_up) {
  const int K = gate_up ? d.H : d.I;
  const int cols = gate_up ? d.I : d.H;
  // Rows per routed expert (on average) from which pair tiles pay, measured
  // against the one-SM tiles: gate/up from 256 (at 64, Qwen3 T=1024 gate/up
  // 521 -> 537 us); down from 64 when its K (= I) is at least 2048
  // (DeepSeek-V3 T=2048 down 1210 -> 1132 us, Mixtral T=512 237 -> 172 us),
  // else from 256 (Qwen3, I = 1536: no gain at 64).
  const int min_rows = gate_up ? kPRows : (d.I >= 2048 ? 64 : kPRows);
  // whole stages of K and whole pair tiles of output columns
  return num_sms() >= 2 && K % (kStageKB * kBK) == 0 &&
         cols % (gate_up ? 2 * kPWide : 2 * kBM) == 0 &&
         (int64_t)d.T * d.k >= (int64_t)min_rows * d.E;
}

cudaError_t launch_expert_gemm_pair(bool gate_up, const CUtensorMap &a, const CUtensorMap &a_sh,
                                    const TokenMaps &b, const int32_t *plan, int nseg, int E,
                                    int K, int out_cols, int64_t Na, const float *w_perm,
                                    void *out, uint32_t *status, cudaStream_t s) {
  const size_t smem = pair_smem_bytes(nseg);
  auto kern = gate_up ? expert_gemm_pair_kernel<true> : expert_gemm_pair_kernel<false>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static size_t configured[2][64] = {};
  static int clusters[2][64] = {};
  const int g = gate_up ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  if (smem > configured[g][dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[g][dev] = smem;
    clusters[g][dev] = 0;
  }
  if (clusters[g][dev] == 0) {
    // as many pairs as can be resident at once (one CTA per SM): the
    // persistent tile loop assumes every cluster runs from the start
    cfg.gridDim = dim3((unsigned)(num_sms() / 2 * 2));
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    clusters[g][dev] = std::min(n, num_sms() / 2);
  }
  cfg.gridDim = dim3((unsigned)(2 * clusters[g][dev]));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a, a_sh, b, plan, nseg, E, K, out_cols, Na, w_perm, out,
                            status);
}

}  // namespace moe
